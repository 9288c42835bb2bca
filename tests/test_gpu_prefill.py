"""GPU parity of kda_chunk_fwd against the fp64 oracle (called through the C ABI)."""
import pytest
import torch

from gated_delta_rule_43_gb300 import inputs, kda
from tests.gpu_util import (LAST_WORST, TOL, gpu_prefill, record_windows, rel_l2,
                            score_prefill, score_prefill_whole, to_f64)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run_and_score(d, dtype, seqs=None, heads=None, final=True):
    """Whole-tensor rel-L2 within the tolerance; the worst single (sequence, head) within
    three times it (a short sequence's few outputs are a noisier ratio)."""
    o, hT = gpu_prefill(d, final=final)
    torch.cuda.synchronize()
    e_o, e_s = score_prefill(d, o, hT, seqs, heads)
    tol = TOL[dtype]
    w = dict(LAST_WORST)
    assert e_o <= tol, f"o rel-L2 {e_o:.3e} > {tol}"
    assert w["o"] <= 3 * tol, f"worst per-(sequence, head) o rel-L2 {w['o']:.3e}"
    if final:
        assert e_s <= tol, f"state rel-L2 {e_s:.3e} > {tol}"
        assert w["state"] <= 3 * tol, f"worst per-(sequence, head) state rel-L2 {w['state']:.3e}"
    print(f"rel-L2 o {e_o:.3e} state {e_s} worst per (seq, head): o {w['o']:.3e} "
          f"state {w['state']:.3e}")
    return e_o, e_s


def test_tiny_fp32_workload():
    """B=1, H=2, T=64, dk=dv=32, fp32, zero initial state, seed 0: rel-L2 <= 1e-4."""
    w = inputs.WORKLOADS["tiny_fp32"]
    d = inputs.make_workload(w, device=DEV)
    _run_and_score(d, "f32")


SHAPES = [(32, 32), (64, 128), (128, 64), (128, 128)]
LENS = [[1], [15], [16], [17], [33], [100, 0, 37], [0], [64, 64, 1, 129]]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("dk,dv", SHAPES)
@pytest.mark.parametrize("lens", LENS, ids=lambda l: "-".join(map(str, l)))
def test_small_shapes_and_ragged_tails(dtype, dk, dv, lens):
    d = inputs.make_prefill(lens, H=3, dk=dk, dv=dv, dtype=dtype, seed=sum(lens) + dk + dv,
                            h0_sigma=0.1 if len(lens) > 1 else 0.0, device=DEV)
    _run_and_score(d, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_in_place_state_and_no_final_state(dtype):
    d = inputs.make_prefill([40, 70], H=2, dk=64, dv=64, dtype=dtype, seed=7, h0_sigma=0.1,
                            device=DEV)
    ref_o, ref_s = gpu_prefill(d)
    S = d["h0"].clone()
    o, s_out = kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["beta"], d["A_log"],
                             d["cu_seqlens"], S, final_state=S, check=True)
    assert s_out.data_ptr() == S.data_ptr()
    assert torch.equal(o, ref_o) and torch.equal(S, ref_s)
    o2, none = kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["beta"], d["A_log"],
                             d["cu_seqlens"], d["h0"], output_final_state=False, check=True)
    assert none is None and torch.equal(o2, ref_o)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_split_and_resume(dtype):
    """Prefill [0, t) then [t, T) from the carried state matches one pass."""
    T = 300
    d = inputs.make_prefill([T], H=2, dk=128, dv=128, dtype=dtype, seed=11, h0_sigma=0.1,
                            device=DEV)
    o_all, s_all = gpu_prefill(d)
    for t in (1, 64, 100):
        a = {k: (v[:t] if k in ("q", "k", "v", "z", "beta") else v) for k, v in d.items()}
        a["cu_seqlens"] = torch.tensor([0, t], dtype=torch.int32, device=DEV)
        oa, sa = gpu_prefill(a)
        b = {k: (v[t:] if k in ("q", "k", "v", "z", "beta") else v) for k, v in d.items()}
        b["cu_seqlens"] = torch.tensor([0, T - t], dtype=torch.int32, device=DEV)
        b["h0"] = sa
        ob, sb = gpu_prefill(b)
        tol = TOL[dtype]
        assert rel_l2(to_f64(torch.cat([oa, ob])), to_f64(o_all)) <= tol
        assert rel_l2(to_f64(sb), to_f64(s_all)) <= tol


def test_prefill_8k_workload():
    """B=1, H=32, T=8192, dk=dv=128, bf16: full oracle comparison."""
    d = inputs.make_workload(inputs.WORKLOADS["prefill_8k"], device=DEV)
    _run_and_score(d, "bf16")


def _score_whole(d, tol):
    o, hT = gpu_prefill(d)
    torch.cuda.synchronize()
    e_o, e_s = score_prefill_whole(d, o, hT)
    w = dict(LAST_WORST)
    print(f"whole-tensor rel-L2 o {e_o:.3e} state {e_s:.3e}; worst per (seq, head): "
          f"o {w['o']:.3e} state {w['state']:.3e}")
    assert e_o <= tol, f"o rel-L2 {e_o:.3e} > {tol}"
    assert e_s <= tol, f"state rel-L2 {e_s:.3e} > {tol}"
    assert w["o"] <= 3 * tol and w["state"] <= 3 * tol, w


@pytest.mark.timeout(1800)
def test_varlen_64_workload():
    """64 packed sequences U[512, 4096], H=32, h0 ~ N(0, 0.01): every sequence and every
    head scored, rel-L2 over the whole o and final-state tensors."""
    d = inputs.make_workload(inputs.WORKLOADS["varlen_64"], device=DEV)
    _score_whole(d, TOL["bf16"])


@pytest.mark.timeout(3600)
def test_prefill_1m_workload():
    """B=1, H=16, T=1,048,576: all 16 heads over the whole length scored, rel-L2 over the
    whole o and final-state tensors."""
    d = inputs.make_workload(inputs.WORKLOADS["prefill_1m"], device=DEV)
    _score_whole(d, TOL["bf16"])


def _chain_shape(N, H):
    """Which chain kernel the library runs for N sequences of H heads (dk = dv = 128, bf16):
    32-column items while N*H*4 fits in two waves of the device's SMs, else 128-column."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return 32 if N * H * 4 <= 2 * sms else 128


@pytest.mark.parametrize("z_shift", [-4.0, -6.0])
@pytest.mark.parametrize("dtype,dk,dv", [("bf16", 128, 128), ("f32", 64, 64)])
def test_long_memory_gates(z_shift, dtype, dk, dv):
    """Gates near g = 0 keep the state for hundreds of tokens, so every chunk's output leans
    on the state carried across many chunks (with the default gates it is forgotten within
    a chunk); an error in the inter-chunk recurrence shows here."""
    d = inputs.make_prefill([2000, 700, 65], H=4, dk=dk, dv=dv, dtype=dtype, seed=int(-z_shift),
                            h0_sigma=0.1, z_shift=z_shift, device=DEV)
    _run_and_score(d, dtype)


@pytest.mark.parametrize("lens", [[130, 257], [130, 257, 64, 3] * 3],
                         ids=["few-seqs", "many-seqs"])
def test_both_chain_shapes(lens):
    """The narrow (32-column) and wide (128-column) chain kernels, with initial states and
    ragged chunks; the two cases are chosen so that they select different kernels."""
    H = 32
    shapes = {_chain_shape(len(l), H) for l in [[130, 257], [130, 257, 64, 3] * 3]}
    assert shapes == {32, 128}
    d = inputs.make_prefill(lens, H=H, dk=128, dv=128, dtype="bf16", seed=len(lens),
                            h0_sigma=0.1, device=DEV)
    _run_and_score(d, "bf16")


def test_many_short_sequences():
    """1200 packed sequences of 0-150 tokens (one in ten empty) with initial states: the
    chunk plan of a large batch and the 128-column chain walking many more items than it
    has CTAs."""
    import numpy as np
    rng = np.random.default_rng(55)
    lens = [0 if rng.random() < 0.1 else int(rng.integers(1, 151)) for _ in range(1200)]
    d = inputs.make_prefill(lens, H=4, dk=128, dv=128, dtype="bf16", seed=56, h0_sigma=0.1,
                            device=DEV)
    _run_and_score(d, "bf16")


@pytest.mark.timeout(900)
def test_windows_one_head_chain_slower_than_prep():
    """One head, about a million tokens: three windows, each window's prep far shorter than
    the previous window's chain, so that a window's chain must wait for the previous chain
    (its start state) as well as for its own prep, and the next prep must not overwrite the
    records of a chain still running."""
    T = 1_000_000
    assert record_windows(T, 1, 1) >= 3
    d = inputs.make_prefill([T], H=1, dk=128, dv=128, dtype="bf16", seed=41, h0_sigma=0.1,
                            z_shift=-4.0, device=DEV)
    _run_and_score(d, "bf16")


@pytest.mark.timeout(900)
def test_windows_beside_the_chain_long_memory():
    """One sequence long enough for several double-buffered windows of chunk records: the
    prep of window w + 1 runs beside the chain of window w; long-memory gates carry the
    state across every window boundary."""
    assert record_windows(30000, 1, 32) >= 2
    d = inputs.make_prefill([30000], H=32, dk=128, dv=128, dtype="bf16", seed=31, h0_sigma=0.1,
                            z_shift=-4.0, device=DEV)
    _run_and_score(d, "bf16")


def test_profiled_entry_pairs_and_stream_order():
    """kda_chunk_fwd_profiled brackets each kernel with an event pair and gives the same
    results as kda_chunk_fwd; inputs written on a side stream just before the call, and
    outputs read on it right after, see the call's work in order (the call may run
    kernels on the library's own streams)."""
    # more than one window of chunk records (451 chunk slots of 32 heads), so that the
    # double-buffered schedule with its own streams runs
    # (the empty sequence in the middle owns no chunk: its final state is its initial one)
    assert record_windows(34000, 3, 32) >= 2
    d = inputs.make_prefill([26000, 0, 8000], H=32, dk=128, dv=128, dtype="bf16", seed=77,
                            h0_sigma=0.1, device=DEV)
    T, H, dk = d["q"].shape
    N = 3
    ws_bytes = kda.chunk_fwd_workspace_size(T, N, H, dk, 128, torch.bfloat16)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        q2 = torch.empty_like(d["q"])
        ws = kda.alloc_workspace(ws_bytes, DEV)
        o = torch.full((T, H, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
        hT = torch.empty(N, H, dk, 128, dtype=torch.float32, device=DEV)
        o2, hT2 = torch.empty_like(o), torch.empty_like(hT)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(256)]
        for _ in range(3):          # a slow producer of the input on the side stream
            q2.copy_(d["q"] * 1.0)
        used = kda.chunk_fwd_profiled(q2, d["k"], d["v"], d["z"], d["beta"], d["A_log"],
                                      d["cu_seqlens"], d["h0"], o, hT, ws, ev, stream=side)
        o_host = o.float().cpu()    # ordered after the call on the side stream
        kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["beta"], d["A_log"], d["cu_seqlens"],
                      d["h0"], o=o2, final_state=hT2, workspace=ws, stream=side)
    side.synchronize()
    assert used >= 2 * (2 + 2 * 2) and used % 2 == 0   # plan, init, two (prep, chain) pairs
    assert all(ev[j].elapsed_time(ev[j + 1]) >= 0.0 for j in range(0, used, 2))
    assert not torch.isnan(o_host).any()
    assert torch.equal(o, o2) and torch.equal(hT, hT2)
    assert torch.equal(hT[1], d["h0"][1])
    e_o, e_s = score_prefill(d, o, hT, None, [0, 17, 31])
    assert e_o <= TOL["bf16"] and e_s <= TOL["bf16"]
