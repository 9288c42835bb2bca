"""Every write of a call lands inside the buffers it was given.

Each output (o, the final state, the decode state, the workspace) is a view into
a larger device buffer whose bands before and after it are filled with a sentinel
byte; after the call (and a synchronize) the bands must be unchanged.  The cases
cover both prefill paths with ragged tails and an empty sequence, the no-alloc
entry, and dense and indexed decode.  This is the out-of-bounds-write check that
stands in for a memory sanitizer.
"""
import pytest
import torch

from gated_delta_rule_43_gb300 import inputs, kda
from tests.gpu_util import record_windows

pytestmark = pytest.mark.gpu
DEV = "cuda"
GUARD = 4096          # bytes on each side; keeps every view 256-byte aligned
SENTINEL = 0xA5


class Banded:
    """A device buffer of `nbytes` with sentinel bands on both sides."""

    def __init__(self, nbytes: int):
        self.nbytes = int(nbytes)
        self.full = torch.full((self.nbytes + 2 * GUARD,), SENTINEL, dtype=torch.uint8,
                               device=DEV)
        self.mid = self.full[GUARD:GUARD + self.nbytes]

    def view(self, dtype, shape):
        return self.mid.view(dtype).view(*shape)

    def check(self, what: str):
        torch.cuda.synchronize()
        lo = self.full[:GUARD]
        hi = self.full[GUARD + self.nbytes:]
        bad_lo = int((lo != SENTINEL).sum())
        bad_hi = int((hi != SENTINEL).sum())
        assert bad_lo == 0 and bad_hi == 0, f"{what}: {bad_lo} bytes before, {bad_hi} after"


def _esize(dtype):
    return torch.empty(0, dtype=dtype).element_size()


def _prefill_banded(d, noalloc=False):
    T, H, dk = d["q"].shape
    dv = d["v"].shape[-1]
    N = d["cu_seqlens"].numel() - 1
    bo = Banded(T * H * dv * _esize(d["q"].dtype))
    bs = Banded(N * H * dk * dv * 4)
    o = bo.view(d["q"].dtype, (T, H, dv))
    hT = bs.view(torch.float32, (N, H, dk, dv))
    if noalloc:
        bst = Banded(16)
        kda.chunk_fwd_noalloc(d["q"], d["k"], d["v"], d["z"], d["beta"], d["A_log"],
                              d["cu_seqlens"], d["h0"], o, hT, bst.mid)
        bst.check("status copy")
        code, info = kda.query_status(bst.mid)
        assert code == kda.KDA_OK, (kda.status_string(code), info)
    else:
        nws = kda.chunk_fwd_workspace_size(T, N, H, dk, dv, d["q"].dtype)
        bw = Banded(nws)
        kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["beta"], d["A_log"], d["cu_seqlens"],
                      d["h0"], o=o, final_state=hT, workspace=bw.mid)
        bw.check("workspace")
        code, info = kda.query_status(bw.mid)
        assert code == kda.KDA_OK, (kda.status_string(code), info)
    bo.check("o")
    bs.check("final state")
    # the views hold real results: compare with a call on plain buffers
    o_ref, s_ref = kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["beta"], d["A_log"],
                                 d["cu_seqlens"], d["h0"], check=True)
    assert torch.equal(o, o_ref) and torch.equal(hT, s_ref)


@pytest.mark.parametrize("dtype,dk,dv", [("bf16", 128, 128), ("f32", 64, 32), ("bf16", 32, 64)])
def test_prefill_writes_stay_in_bounds(dtype, dk, dv):
    d = inputs.make_prefill([100, 0, 37, 129, 1], H=4, dk=dk, dv=dv, dtype=dtype, seed=61,
                            h0_sigma=0.1, device=DEV)
    _prefill_banded(d)


def test_prefill_many_windows_writes_stay_in_bounds():
    # enough chunk slots x heads that the tensor-core path runs its double-buffered windows
    assert record_windows(74100, 4, 32) >= 2
    d = inputs.make_prefill([70000, 3, 0, 4097], H=32, dk=128, dv=128, dtype="bf16", seed=62,
                            h0_sigma=0.1, device=DEV)
    _prefill_banded(d)


def test_noalloc_writes_stay_in_bounds():
    d = inputs.make_prefill([300, 0, 65], H=4, dk=128, dv=128, dtype="bf16", seed=63,
                            h0_sigma=0.1, device=DEV)
    _prefill_banded(d, noalloc=True)


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 32)])
def test_decode_writes_stay_in_bounds(dk, dv):
    N, H = 5, 3
    d = inputs.make_prefill([1] * N, H=H, dk=dk, dv=dv, dtype="bf16", seed=64, device=DEV)
    bS = Banded(N * H * dk * dv * 4)
    S = bS.view(torch.float32, (N, H, dk, dv))
    S.copy_(torch.randn(N, H, dk, dv, device=DEV) * 0.1)
    S_ref = S.clone()
    bo = Banded(N * H * dv * 2)
    o = bo.view(torch.bfloat16, (N, H, dv))
    step = {k: d[k] for k in ("q", "k", "v", "z", "beta")}
    kda.decode_step(step["q"], step["k"], step["v"], step["z"], step["beta"], d["A_log"], S,
                    o=o)
    bS.check("state")
    bo.check("o")
    o_ref = kda.decode_step(step["q"], step["k"], step["v"], step["z"], step["beta"],
                            d["A_log"], S_ref)
    assert torch.equal(o, o_ref) and torch.equal(S, S_ref)


def test_indexed_decode_writes_stay_in_bounds():
    N, H, dk, dv, P = 4, 2, 128, 128, 9
    d = inputs.make_prefill([1] * N, H=H, dk=dk, dv=dv, dtype="bf16", seed=65, device=DEV)
    bP = Banded(P * H * dk * dv * 4)
    pool = bP.view(torch.float32, (P, H, dk, dv))
    pool.copy_(torch.randn(P, H, dk, dv, device=DEV) * 0.1)
    before = pool.clone()
    idx = torch.tensor([8, 0, 3, 5], dtype=torch.int32, device=DEV)
    bo = Banded(N * H * dv * 2)
    o = bo.view(torch.bfloat16, (N, H, dv))
    kda.decode_step_indexed(d["q"], d["k"], d["v"], d["z"], d["beta"], d["A_log"], pool, idx,
                            o=o)
    bP.check("state pool")
    bo.check("o")
    untouched = [p for p in range(P) if p not in idx.tolist()]
    assert torch.equal(pool[untouched], before[untouched])
