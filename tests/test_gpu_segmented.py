"""GPU parity of kda_chunk_fwd_segmented (segment-parallel prefill) against the oracle.

Each sequence's chunks in a window of records are cut into up to `segments`
segments: segment 0 runs from the sequence's state, every later segment's affine
map S_end = M S_start + B is computed in parallel, a scan composes the maps into
start states and a second pass produces the later segments' outputs.  The
results must match the fp64 oracle within the bf16 tolerance, for ragged
sequences, empty ones, initial states, more segments than chunks, and a problem
large enough to run in several windows.
"""
import pytest
import torch

from gated_delta_rule_43_gb300 import inputs, kda
from tests.gpu_util import (LAST_WORST, TOL, gpu_prefill, record_windows, rel_l2,
                            score_prefill, to_f64)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _seg(d, segments, **kw):
    return kda.chunk_fwd_segmented(d["q"], d["k"], d["v"], d["z"], d["beta"], d["A_log"],
                                   d["cu_seqlens"], d["h0"], segments=segments, check=True, **kw)


def _score(d, o, hT, heads=None):
    torch.cuda.synchronize()
    e_o, e_s = score_prefill(d, o, hT, None, heads)
    w = dict(LAST_WORST)
    tol = TOL["bf16"]
    assert e_o <= tol and e_s <= tol, (e_o, e_s)
    assert w["o"] <= 3 * tol and w["state"] <= 3 * tol, w
    print(f"rel-L2 o {e_o:.3e} state {e_s:.3e} worst o {w['o']:.3e} state {w['state']:.3e}")


@pytest.mark.parametrize("segments", [2, 3, 5])
def test_one_long_sequence(segments):
    d = inputs.make_prefill([1100], H=2, dk=128, dv=128, dtype="bf16", seed=70 + segments,
                            h0_sigma=0.1, device=DEV)
    o, hT = _seg(d, segments)
    _score(d, o, hT)


@pytest.mark.parametrize("segments", [2, 4, 64])
def test_ragged_packed_sequences(segments):
    # lengths below, at and above the segment count in chunks (1, 3, 5 and 17 chunks), an
    # empty sequence and a ragged last chunk
    d = inputs.make_prefill([1000, 0, 130, 300, 64, 1], H=3, dk=128, dv=128, dtype="bf16",
                            seed=80 + segments, h0_sigma=0.1, device=DEV)
    o, hT = _seg(d, segments)
    _score(d, o, hT)


def test_zero_initial_state_and_in_place():
    d = inputs.make_prefill([700, 450], H=2, dk=128, dv=128, dtype="bf16", seed=90, device=DEV)
    o, hT = _seg(d, 3)
    _score(d, o, hT)
    # in place: the initial state buffer receives the final state
    d2 = inputs.make_prefill([700, 450], H=2, dk=128, dv=128, dtype="bf16", seed=91,
                             h0_sigma=0.1, device=DEV)
    ref_o, ref_s = _seg(d2, 3)
    S = d2["h0"].clone()
    o2, s2 = kda.chunk_fwd_segmented(d2["q"], d2["k"], d2["v"], d2["z"], d2["beta"],
                                     d2["A_log"], d2["cu_seqlens"], S, segments=3,
                                     final_state=S, check=True)
    assert s2.data_ptr() == S.data_ptr()
    assert torch.equal(o2, ref_o) and torch.equal(S, ref_s)


def test_one_segment_is_the_plain_call():
    d = inputs.make_prefill([500, 77], H=2, dk=128, dv=128, dtype="bf16", seed=92,
                            h0_sigma=0.1, device=DEV)
    o1, s1 = _seg(d, 1)
    o0, s0 = gpu_prefill(d)
    assert torch.equal(o1, o0) and torch.equal(s1, s0)


def test_two_windows():
    # 4 heads x 3750 chunk slots of records (74,240 bytes each) exceed one 1 GiB window
    # (3615 slots): windows of 1807 slots, each after the first starting from the running
    # state the previous one's last segment left (long-memory gates, so that the state
    # carried across the window boundaries matters)
    T = 240_000
    assert record_windows(T, 1, 4) >= 2
    d = inputs.make_prefill([T], H=4, dk=128, dv=128, dtype="bf16", seed=93, h0_sigma=0.1,
                            z_shift=-6.0, device=DEV)
    o, hT = _seg(d, 4)
    o0, s0 = gpu_prefill(d)
    e_o = rel_l2(to_f64(o), to_f64(o0))
    e_s = rel_l2(to_f64(hT), to_f64(s0))
    assert e_o <= TOL["bf16"] and e_s <= TOL["bf16"], (e_o, e_s)
    _score(d, o, hT, heads=[1])


@pytest.mark.parametrize("segments", [3, 6])
def test_long_memory_maps(segments):
    """Gates near g = 0: a later segment's outputs depend on its start state, so the
    composed maps (M, B) are exercised, not just segment 0's walk."""
    d = inputs.make_prefill([3000, 900], H=2, dk=128, dv=128, dtype="bf16", seed=95,
                            h0_sigma=0.1, z_shift=-6.0, device=DEV)
    o, hT = _seg(d, segments)
    _score(d, o, hT)
    o0, s0 = gpu_prefill(d)
    assert rel_l2(to_f64(o), to_f64(o0)) <= TOL["bf16"]
    assert rel_l2(to_f64(hT), to_f64(s0)) <= TOL["bf16"]


def test_nan_decay_is_reported_and_isolated():
    """A NaN z in the second sequence is reported with its (token, head); the first
    sequence, cut into segments, still matches the oracle."""
    import numpy as np
    from oracle import oracle as orc
    d = inputs.make_prefill([900, 400], H=2, dk=128, dv=128, dtype="bf16", seed=96,
                            h0_sigma=0.1, z_shift=-4.0, device=DEV)
    d["z"][1000, 1, 9] = float("nan")
    nbytes = kda.load().kda_chunk_fwd_segmented_workspace_size(1300, 2, 2, 128, 128,
                                                               kda.KDA_BF16, 4)
    ws = kda.alloc_workspace(nbytes, DEV)
    o, hT = kda.chunk_fwd_segmented(d["q"], d["k"], d["v"], d["z"], d["beta"], d["A_log"],
                                    d["cu_seqlens"], d["h0"], segments=4, workspace=ws)
    code, info = kda.query_status(ws)
    assert code == kda.KDA_ERR_DECAY_RANGE and info == 1000 * 2 + 1
    h = {n: inputs.host_array(d[n][:900]) for n in ("q", "k", "v", "z", "beta")}
    ref = orc.forward(h["q"], h["k"], h["v"], h["z"], h["beta"],
                      d["A_log"].cpu().numpy().astype(np.float64), np.array([0, 900]),
                      d["h0"][:1].cpu().numpy().astype(np.float64))
    assert rel_l2(to_f64(o[:900]), ref["o"]) <= TOL["bf16"]
    assert rel_l2(to_f64(hT[:1]), ref["state"]) <= TOL["bf16"]


def _auto_segments(T, N, H):
    """The count kda_chunk_fwd picks by itself (include/kda.h): the largest s <= 16 whose
    first pass fits one wave of 32-column CTAs, with >= 64 chunks per segment."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    chunks = T // (64 * N)
    best = 1
    for s in range(2, 17):
        if N * H * (4 + 8 * (s - 1)) > sms or chunks < 64 * s:
            break
        best = s
    return best


def test_plain_call_picks_segments_for_few_long_sequences():
    T, H = 300_000, 2
    segs = _auto_segments(T, 1, H)
    assert segs >= 2
    d = inputs.make_prefill([T], H=H, dk=128, dv=128, dtype="bf16", seed=97, h0_sigma=0.1,
                            z_shift=-6.0, device=DEV)
    o, hT = gpu_prefill(d)
    o_s, hT_s = _seg(d, segs)
    assert torch.equal(o, o_s) and torch.equal(hT, hT_s)   # the same schedule
    _score(d, o, hT, heads=[0])
    # a workspace sized for the plain schedule makes the call fall back to it
    nplain = kda.load().kda_chunk_fwd_segmented_workspace_size(T, 1, H, 128, 128,
                                                               kda.KDA_BF16, 1)
    ws = kda.alloc_workspace(nplain, DEV)
    o1, h1 = kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["beta"], d["A_log"],
                           d["cu_seqlens"], d["h0"], workspace=ws, check=True)
    o_p, h_p = _seg(d, 1)
    assert torch.equal(o1, o_p) and torch.equal(h1, h_p)


def test_benchmark_shapes_stay_plain():
    for T, N, H in ((8192, 1, 32), (1 << 20, 1, 16), (158_000, 64, 32)):
        assert _auto_segments(T, N, H) == 1, (T, N, H)


def test_bad_segment_counts_are_refused():
    d = inputs.make_prefill([100], H=1, dk=128, dv=128, dtype="bf16", seed=94, device=DEV)
    for bad in (0, 65):
        with pytest.raises(kda.KdaError):
            _seg(d, bad)
