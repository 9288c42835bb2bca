"""GPU parity of kda_decode_step against the fp64 oracle (called through the C ABI)."""
import numpy as np
import pytest
import torch

from gated_delta_rule_43_gb300 import inputs, kda
from oracle import oracle as orc
from tests.gpu_util import TOL, gpu_prefill, oracle_prefill, rel_l2, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _decode_and_score(N, H, dk, dv, dtype, steps, seed=0):
    """`steps` in-place decode steps of N sequences against the fp64 oracle: rel-L2 of the
    outputs of every step (concatenated) and of the state after the last step, both over
    the whole tensor; the worst single (sequence, head) within three times the tolerance."""
    ds = inputs.DecodeStream(N, H, dk, dv, dtype, seed=seed, h0_sigma=0.1, device=DEV)
    state = ds.state0.clone()
    ref_state = state.cpu().numpy().astype(np.float64)
    A = ds.A_log.cpu().numpy().astype(np.float64)
    e2 = np.zeros((N, H))
    r2 = np.zeros((N, H))
    for _ in range(steps):
        x = ds.step()
        o = kda.decode_step(x["q"], x["k"], x["v"], x["z"], x["beta"], ds.A_log, state)
        h = {k: inputs.host_array(x[k]) for k in x}
        ref = orc.decode(h["q"], h["k"], h["v"], h["z"], h["beta"], A, ref_state)
        e2 += ((to_f64(o) - ref) ** 2).sum(axis=2)
        r2 += (ref ** 2).sum(axis=2)
    torch.cuda.synchronize()
    e_o = float(np.sqrt(e2.sum() / r2.sum()))
    s64 = to_f64(state)
    e_s = rel_l2(s64, ref_state)
    worst_o = float(np.sqrt((e2 / r2).max()))
    worst_s = float(np.sqrt((((s64 - ref_state) ** 2).sum(axis=(2, 3)) /
                             (ref_state ** 2).sum(axis=(2, 3))).max()))
    tol = TOL[dtype]
    print(f"decode rel-L2 o {e_o:.3e} state {e_s:.3e}; worst per (seq, head) o {worst_o:.3e} "
          f"state {worst_s:.3e}")
    assert e_o <= tol, f"decode o rel-L2 {e_o:.3e} > {tol}"
    assert e_s <= tol, f"decode state rel-L2 {e_s:.3e} > {tol}"
    assert worst_o <= 3 * tol and worst_s <= 3 * tol, (worst_o, worst_s)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(32, 32), (32, 128), (64, 64), (128, 32), (128, 128)])
def test_decode_small(dtype, dk, dv):
    _decode_and_score(5, 3, dk, dv, dtype, steps=6, seed=dk + dv)


@pytest.mark.timeout(1800)
def test_decode_256_workload():
    """256 sequences, H=32, 128 steps in place: every sequence and head scored over every
    step, and the whole state after step 128."""
    _decode_and_score(256, 32, 128, 128, "bf16", steps=128, seed=3)


def test_tiny_workload_as_decode_steps():
    """The tiny fp32 workload run as 64 decode steps equals its 64-token prefill."""
    d = inputs.make_workload(inputs.WORKLOADS["tiny_fp32"], device=DEV)
    o_pre, s_pre = gpu_prefill(d)
    H, dk, dv = 2, 32, 32
    state = torch.zeros(1, H, dk, dv, device=DEV)
    outs = []
    for t in range(64):
        sl = slice(t, t + 1)
        outs.append(kda.decode_step(d["q"][sl], d["k"][sl], d["v"][sl], d["z"][sl],
                                    d["beta"][sl], d["A_log"], state))
    o_dec = torch.cat(outs)
    assert rel_l2(to_f64(o_dec), to_f64(o_pre)) <= TOL["f32"]
    assert rel_l2(to_f64(state), to_f64(s_pre)) <= TOL["f32"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_prefill_then_decode_handoff(dtype):
    """Prefill 50 tokens, then decode 10 more from the emitted state = one 60-token pass."""
    d = inputs.make_prefill([60], H=2, dk=128, dv=128, dtype=dtype, seed=5, h0_sigma=0.1,
                            device=DEV)
    o_all, s_all = gpu_prefill(d)
    a = {k: (v[:50] if k in ("q", "k", "v", "z", "beta") else v) for k, v in d.items()}
    a["cu_seqlens"] = torch.tensor([0, 50], dtype=torch.int32, device=DEV)
    o_a, S = gpu_prefill(a)
    outs = [o_a]
    for t in range(50, 60):
        sl = slice(t, t + 1)
        outs.append(kda.decode_step(d["q"][sl], d["k"][sl], d["v"][sl], d["z"][sl],
                                    d["beta"][sl], d["A_log"], S))
    tol = TOL[dtype]
    assert rel_l2(to_f64(torch.cat(outs)), to_f64(o_all)) <= tol
    assert rel_l2(to_f64(S), to_f64(s_all)) <= tol


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_indexed_state_pool(dtype):
    """Sequence n advances slot idx[n] of a state pool: outputs and the advanced slots match
    the fp64 oracle run on those slots' states, the result is bit-identical to dense decode
    on the gathered states, and the other slots are untouched."""
    N, H, dk, dv, P = 4, 3, 128, 64, 7
    ds = inputs.DecodeStream(N, H, dk, dv, dtype, seed=12, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(13)
    pool = torch.randn(P, H, dk, dv, device=DEV, generator=g) * 0.1
    idx = torch.tensor([5, 0, 3, 6], dtype=torch.int32, device=DEV)
    dense = pool.index_select(0, idx.long()).clone()
    ref_state = dense.cpu().numpy().astype(np.float64)
    A = ds.A_log.cpu().numpy().astype(np.float64)
    before = pool.clone()
    outs, refs = [], []
    for _ in range(3):
        x = ds.step()
        o_pool = kda.decode_step_indexed(x["q"], x["k"], x["v"], x["z"], x["beta"], ds.A_log,
                                         pool, idx, check=True)
        o_dense = kda.decode_step(x["q"], x["k"], x["v"], x["z"], x["beta"], ds.A_log, dense)
        assert torch.equal(o_pool, o_dense)
        h = {k: inputs.host_array(x[k]) for k in x}
        refs.append(orc.decode(h["q"], h["k"], h["v"], h["z"], h["beta"], A, ref_state))
        outs.append(to_f64(o_pool))
    tol = TOL[dtype]
    assert rel_l2(np.stack(outs), np.stack(refs)) <= tol
    assert rel_l2(to_f64(pool.index_select(0, idx.long())), ref_state) <= tol
    assert torch.equal(pool.index_select(0, idx.long()), dense)
    untouched = [s for s in range(P) if s not in idx.tolist()]
    assert torch.equal(pool[untouched], before[untouched])


def test_decode_indexed_rejects_bad_slot():
    ds = inputs.DecodeStream(2, 1, 32, 32, "f32", seed=14, device=DEV)
    pool = torch.zeros(3, 1, 32, 32, device=DEV)
    idx = torch.tensor([1, 3], dtype=torch.int32, device=DEV)   # 3 is outside [0, 3)
    x = ds.step()
    with pytest.raises(kda.KdaError) as ei:
        kda.decode_step_indexed(x["q"], x["k"], x["v"], x["z"], x["beta"], ds.A_log, pool, idx,
                                check=True)
    assert ei.value.code == kda.KDA_ERR_INVALID_ARG and ei.value.info == 1


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_multi_token_decode_through_chunk_fwd(dtype):
    """k tokens per sequence against the resident state in one in-place chunked call
    (initial_state aliasing final_state): outputs and advanced states match the fp64
    oracle on the same packed k-token sequences, and equal k single-token decode steps."""
    N, H, dk, dv, kt = 6, 2, 128, 128, 5
    d = inputs.make_prefill([kt] * N, H=H, dk=dk, dv=dv, dtype=dtype, seed=15, h0_sigma=0.1,
                            device=DEV)
    S_multi = d["h0"].clone()
    o_multi, _ = kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["beta"], d["A_log"],
                               d["cu_seqlens"], S_multi, final_state=S_multi, check=True)
    tol = TOL[dtype]
    ref, _, _ = oracle_prefill(d)
    assert rel_l2(to_f64(o_multi), ref["o"]) <= tol
    assert rel_l2(to_f64(S_multi), ref["state"]) <= tol
    S_step = d["h0"].clone()
    outs = []
    for t in range(kt):
        rows = torch.arange(N, device=DEV) * kt + t
        sel = {n_: d[n_].index_select(0, rows) for n_ in ("q", "k", "v", "z", "beta")}
        outs.append(kda.decode_step(sel["q"], sel["k"], sel["v"], sel["z"], sel["beta"],
                                    d["A_log"], S_step))
    o_step = torch.stack(outs, 1).reshape(N * kt, H, dv)
    assert rel_l2(to_f64(o_multi), to_f64(o_step)) <= tol
    assert rel_l2(to_f64(S_multi), to_f64(S_step)) <= tol
