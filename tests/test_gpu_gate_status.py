"""The standalone gate kernel and device-side error reporting (GPU).

Errors are provoked with bad INPUT values (NaN in z, inconsistent
cu_seqlens) that the kernels check themselves, or with the library's test hook
that leaves out one record load so that a bounded device wait (1 ms) expires;
nothing here faults or hangs a GPU.
"""
import numpy as np
import pytest
import torch

from gated_delta_rule_43_gb300 import inputs, kda
from oracle import oracle as orc

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("chunk", [16, 64])
def test_gate_cumsum_matches_oracle(dtype, chunk):
    d = inputs.make_prefill([100, 0, 33, 64], H=3, dk=64, dv=32, dtype=dtype, seed=9,
                            device=DEV)
    G, ws = kda.gate_cumsum(d["z"], d["A_log"], d["cu_seqlens"], chunk=chunk, check=True)
    _, Gref, bad = orc.gate(inputs.host_array(d["z"]), d["A_log"].cpu().numpy(),
                            d["cu_seqlens"].cpu().numpy(), tile=chunk)
    assert bad == 0 or chunk > 16
    err = np.abs(G.cpu().numpy().astype(np.float64) - Gref)
    assert float(err.max()) <= 1e-5 * max(1.0, float(np.abs(Gref).max()))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_nan_decay_is_reported(dtype):
    d = inputs.make_prefill([40, 40], H=2, dk=32, dv=32, dtype=dtype, seed=1, device=DEV)
    d["z"][45, 1, 3] = float("nan")
    with pytest.raises(kda.KdaError) as ei:
        kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["beta"], d["A_log"], d["cu_seqlens"],
                      check=True)
    assert ei.value.code == kda.KDA_ERR_DECAY_RANGE
    assert ei.value.info == 45 * 2 + 1
    with pytest.raises(kda.KdaError) as eg:
        kda.gate_cumsum(d["z"], d["A_log"], d["cu_seqlens"], chunk=64, check=True)
    assert eg.value.code == kda.KDA_ERR_DECAY_RANGE


def test_bad_cu_seqlens_are_reported():
    d = inputs.make_prefill([10, 10, 10], H=1, dk=32, dv=32, dtype="f32", seed=2, device=DEV)
    for bad in ([0, 10, 5, 30], [0, 10, 20, 25], [1, 10, 20, 30]):
        cu = torch.tensor(bad, dtype=torch.int32, device=DEV)
        with pytest.raises(kda.KdaError) as ei:
            kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["beta"], d["A_log"], cu, check=True)
        assert ei.value.code == kda.KDA_ERR_SEQLENS
    # the status word is cleared by the next good call
    o, s = kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["beta"], d["A_log"],
                         d["cu_seqlens"], check=True)
    assert torch.isfinite(o).all()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_softplus_baseline_gate_and_the_bound(dtype):
    """A/B of the lower bound: on the same z, the unbounded -Softplus gate pushes 16-token
    tile sums below -80 (flagged) while the bounded gate stays inside [-80, 0]."""
    d = inputs.make_prefill([100, 37], H=2, dk=32, dv=32, dtype=dtype, seed=21, device=DEV)
    d["z"][:16] = 20.0         # strong gates on the first tile of sequence 0
    host_z = inputs.host_array(d["z"])
    A = d["A_log"].cpu().numpy()
    cu = d["cu_seqlens"].cpu().numpy()
    Gs, _ = kda.gate_cumsum(d["z"], d["A_log"], d["cu_seqlens"], chunk=16, softplus=True)
    code, _ = kda.query_status(_)
    _, Gs_ref, bad_s = orc.gate(host_z, A, cu, tile=16, softplus=True)
    assert bad_s > 0 and code == kda.KDA_ERR_DECAY_RANGE
    err = np.abs(Gs.cpu().numpy().astype(np.float64) - Gs_ref)
    assert float(err.max()) <= 1e-5 * max(1.0, float(np.abs(Gs_ref).max()))
    Gb, wsb = kda.gate_cumsum(d["z"], d["A_log"], d["cu_seqlens"], chunk=16, check=True)
    _, Gb_ref, bad_b = orc.gate(host_z, A, cu, tile=16)
    assert bad_b == 0
    assert float(Gb.min()) >= -80.0


def test_tensor_core_path_nan_is_reported_and_isolated():
    """On the tensor-core path (bf16, 128/128): a NaN z in the second sequence is reported
    with its (token, head), and the first sequence -- whose last chunk's tile loads also
    bring in the second sequence's rows -- still matches the oracle."""
    from tests.gpu_util import TOL, rel_l2, to_f64
    d = inputs.make_prefill([100, 100], H=2, dk=128, dv=128, dtype="bf16", seed=11,
                            h0_sigma=0.1, device=DEV)
    d["z"][130, 1, 7] = float("nan")
    ws = kda.alloc_workspace(kda.chunk_fwd_workspace_size(200, 2, 2, 128, 128, torch.bfloat16),
                             DEV)
    o, hT = kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["beta"], d["A_log"],
                          d["cu_seqlens"], d["h0"], workspace=ws)
    code, info = kda.query_status(ws)
    assert code == kda.KDA_ERR_DECAY_RANGE and info == 130 * 2 + 1
    # sequence 0 alone through the oracle
    h = {n: inputs.host_array(d[n][:100]) for n in ("q", "k", "v", "z", "beta")}
    ref = orc.forward(h["q"], h["k"], h["v"], h["z"], h["beta"],
                      d["A_log"].cpu().numpy().astype(np.float64), np.array([0, 100]),
                      d["h0"][:1].cpu().numpy().astype(np.float64))
    assert rel_l2(to_f64(o[:100]), ref["o"]) <= TOL["bf16"]
    assert rel_l2(to_f64(hT[:1]), ref["state"]) <= TOL["bf16"]


def test_tensor_core_path_bad_cu_seqlens_are_reported():
    d = inputs.make_prefill([70, 70, 70], H=1, dk=128, dv=128, dtype="bf16", seed=12,
                            device=DEV)
    for bad in ([0, 70, 35, 210], [0, 70, 140, 150], [1, 70, 140, 210]):
        cu = torch.tensor(bad, dtype=torch.int32, device=DEV)
        with pytest.raises(kda.KdaError) as ei:
            kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["beta"], d["A_log"], cu, check=True)
        assert ei.value.code == kda.KDA_ERR_SEQLENS
    o, s = kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["beta"], d["A_log"],
                         d["cu_seqlens"], check=True)
    assert torch.isfinite(o).all() and torch.isfinite(s).all()


@pytest.mark.parametrize("lens", [[500, 300], [130, 257, 64, 3] * 4],
                         ids=["32-column-chain", "128-column-chain"])
def test_expired_chain_wait_is_reported_and_the_next_call_is_clean(lens):
    """The test hook leaves out the first record load of chain CTA 0 and gives every wait of
    the chain a 1 ms limit: that CTA's wait expires before it has issued any product, it
    reports KDA_ERR_TIMEOUT (info = its first item, sequence 0 / head 0 / column block 0),
    lets everything it issued finish and leaves.  The next call on the same workspace,
    without the hook, matches the oracle."""
    from tests.gpu_util import TOL, score_prefill
    H = 2 if len(lens) == 2 else 32
    d = inputs.make_prefill(lens, H=H, dk=128, dv=128, dtype="bf16", seed=50 + len(lens),
                            h0_sigma=0.1, device=DEV)
    T, _, dk = d["q"].shape
    N = len(lens)
    ws = kda.alloc_workspace(kda.chunk_fwd_workspace_size(T, N, H, dk, 128, torch.bfloat16),
                             DEV)
    lib = kda.load()
    assert lib.kda_test_chain_fault(1_000_000, 0) == kda.KDA_OK
    kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["beta"], d["A_log"], d["cu_seqlens"],
                  d["h0"], workspace=ws)
    code, info = kda.query_status(ws)
    assert code == kda.KDA_ERR_TIMEOUT and info == 0, (kda.status_string(code), info)
    o, hT = kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["beta"], d["A_log"],
                          d["cu_seqlens"], d["h0"], workspace=ws, check=True)
    e_o, e_s = score_prefill(d, o, hT, heads=[0, H - 1])
    assert e_o <= TOL["bf16"] and e_s <= TOL["bf16"], (e_o, e_s)
