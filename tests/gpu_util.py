"""Shared helpers of the GPU parity tests: run the CUDA path, run the oracle, score."""
from __future__ import annotations

import numpy as np
import torch

from gated_delta_rule_43_gb300 import inputs, kda
from oracle import oracle as orc

# Relative L2 tolerances: fp32 storage 1e-4, bf16 storage 1e-2 (outputs and final states).
TOL = {"f32": 1e-4, "bf16": 1e-2}
DTYPE_NAME = {torch.float32: "f32", torch.bfloat16: "bf16"}


def rel_l2(x, ref) -> float:
    return orc.rel_l2(x, ref)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def gpu_prefill(d, *, final=True, check=True):
    return kda.chunk_fwd(d["q"], d["k"], d["v"], d["z"], d["beta"], d["A_log"], d["cu_seqlens"],
                         d["h0"], output_final_state=final, check=check)


def host_inputs(d, seqs=None, heads=None):
    """Host arrays (exact storage precision) of a packed input dict, optionally sub-sampled.

    seqs: indices of sequences to keep (re-packed); heads: indices of heads to keep.
    Returns (arrays dict, A_log fp64, cu int64, h0 fp64 or None, token index array).
    """
    cu = d["cu_seqlens"].cpu().numpy().astype(np.int64)
    N = len(cu) - 1
    seqs = list(range(N)) if seqs is None else list(seqs)
    tok = np.concatenate([np.arange(cu[n], cu[n + 1]) for n in seqs]) if seqs else np.zeros(0,
                                                                                           int)
    lens = [int(cu[n + 1] - cu[n]) for n in seqs]
    cu_sub = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    H = d["q"].shape[1]
    hsel = list(range(H)) if heads is None else list(heads)
    tok_t = torch.as_tensor(tok, device=d["q"].device, dtype=torch.long)
    hs_t = torch.as_tensor(hsel, device=d["q"].device, dtype=torch.long)
    all_tokens = len(seqs) == N
    arrs = {}
    for name in ("q", "k", "v", "z", "beta"):
        t = d[name] if all_tokens else d[name].index_select(0, tok_t)
        arrs[name] = inputs.host_array(t.index_select(1, hs_t))
    A = d["A_log"].index_select(0, hs_t.to(d["A_log"].device)).cpu().numpy().astype(np.float64)
    h0 = None
    if d["h0"] is not None:
        sel = torch.as_tensor(seqs, device=d["h0"].device, dtype=torch.long)
        h0 = d["h0"].index_select(0, sel).index_select(1, hs_t).cpu().numpy().astype(np.float64)
    return arrs, A, cu_sub, h0, tok, hsel


def oracle_prefill(d, seqs=None, heads=None, o_cmp=None):
    arrs, A, cu, h0, tok, hsel = host_inputs(d, seqs, heads)
    return orc.forward(arrs["q"], arrs["k"], arrs["v"], arrs["z"], arrs["beta"], A, cu, h0,
                       o_cmp=o_cmp), tok, hsel


# The tensor-core path's chunk records, as the library lays them out (74,240 bytes per chunk
# slot and head, at most 2^30 bytes for one window or a double-buffered pair): tests meant
# to cross window boundaries assert that their problem does, so that a change of either
# number cannot quietly make them single-window.
RECORD_BYTES = 74240
RECORD_BUDGET = 1 << 30


def record_windows(T: int, N: int, H: int) -> int:
    """Windows of chunk records the tensor-core path runs for T tokens in N sequences."""
    slots = -(-T // 64) + N
    w = RECORD_BUDGET // (RECORD_BYTES * H)
    if slots <= w:
        return 1
    half = max(1, w // 2)
    return -(-slots // half)


# the last score_prefill call's worst per-(sequence, head) relative L2 errors (o, state)
LAST_WORST = {"o": 0.0, "state": 0.0}
# Sequences shorter than a 16-token tile are left out of the worst per-(sequence, head)
# output error (they stay in the whole-tensor score): a handful of output rows can be
# near zero by cancellation in q.k, and their bf16 rounding error is then a large ratio
# of a small norm (seen on a one-token sequence: 0.26 with the whole tensor at 4e-3).
WORST_MIN_LEN = 16


def _rel(x, ref):
    den = float(np.linalg.norm(ref))
    return float(np.linalg.norm(x - ref)) / den if den > 0 else float(np.linalg.norm(x))


def score_prefill(d, o, hT, seqs=None, heads=None):
    """(rel-L2 of o, rel-L2 of the final state) against the oracle on the selected slice,
    over the whole slice; the worst per-(sequence, head) values go to LAST_WORST."""
    ref, tok, hsel = oracle_prefill(d, seqs, heads)
    dev = o.device
    o_sel = o.index_select(0, torch.as_tensor(tok, device=dev, dtype=torch.long)).index_select(
        1, torch.as_tensor(hsel, device=dev, dtype=torch.long))
    o64 = to_f64(o_sel)
    e_o = rel_l2(o64, ref["o"])
    cu = d["cu_seqlens"].cpu().numpy().astype(np.int64)
    N = len(cu) - 1
    seqs = list(range(N)) if seqs is None else list(seqs)
    lens = [int(cu[n + 1] - cu[n]) for n in seqs]
    bounds = np.concatenate([[0], np.cumsum(lens)])
    worst_o = 0.0
    for i in range(len(seqs)):
        for j in range(len(hsel)):
            a, b = bounds[i], bounds[i + 1]
            if b - a >= WORST_MIN_LEN:
                worst_o = max(worst_o, _rel(o64[a:b, j], ref["o"][a:b, j]))
    e_s, worst_s = None, 0.0
    if hT is not None:
        s_sel = hT.index_select(0, torch.as_tensor(seqs, device=dev, dtype=torch.long))
        s_sel = s_sel.index_select(1, torch.as_tensor(hsel, device=dev, dtype=torch.long))
        s64 = to_f64(s_sel)
        e_s = rel_l2(s64, ref["state"])
        for i in range(len(seqs)):
            for j in range(len(hsel)):
                worst_s = max(worst_s, _rel(s64[i, j], ref["state"][i, j]))
    LAST_WORST["o"], LAST_WORST["state"] = worst_o, worst_s
    return e_o, e_s


def score_prefill_whole(d, o, hT, head_group: int = 4):
    """Whole-tensor (rel-L2 of o, rel-L2 of the final state) against the oracle over every
    sequence and every head, with the worst per-(sequence, head) values in LAST_WORST.

    Heads are scored `head_group` at a time: the GPU result of the group is copied to the
    host and the oracle scores it as it runs (fp64 sums of squared differences per
    (sequence, head)), so no fp64 output tensor is ever materialised and host memory stays
    at one group's inputs."""
    T, H, _ = d["q"].shape
    dev = o.device
    e2o = r2o = e2s = r2s = 0.0
    worst_o = worst_s = 0.0
    for h0 in range(0, H, head_group):
        heads = list(range(h0, min(H, h0 + head_group)))
        arrs, A, cu, h0s, _, _ = host_inputs(d, None, heads)
        hs_t = torch.as_tensor(heads, device=dev, dtype=torch.long)
        o_cmp = inputs.host_array(o.index_select(1, hs_t))
        ref = orc.forward(arrs["q"], arrs["k"], arrs["v"], arrs["z"], arrs["beta"], A, cu, h0s,
                          want_o=False, want_state=hT is not None, o_cmp=o_cmp)
        del arrs, o_cmp
        err2, ref2 = ref["err2"], ref["ref2"]          # [N, len(heads)]
        e2o += float(err2.sum())
        r2o += float(ref2.sum())
        long_seq = (np.diff(cu) >= WORST_MIN_LEN)[:, None]
        nz = (ref2 > 0) & long_seq
        if nz.any():
            worst_o = max(worst_o, float(np.sqrt((err2[nz] / ref2[nz]).max())))
        if hT is not None:
            s64 = to_f64(hT.index_select(1, hs_t))
            diff2 = ((s64 - ref["state"]) ** 2).sum(axis=(2, 3))
            rs2 = (ref["state"] ** 2).sum(axis=(2, 3))
            e2s += float(diff2.sum())
            r2s += float(rs2.sum())
            nzs = rs2 > 0
            if nzs.any():
                worst_s = max(worst_s, float(np.sqrt((diff2[nzs] / rs2[nzs]).max())))
    LAST_WORST["o"], LAST_WORST["state"] = worst_o, worst_s
    e_o = float(np.sqrt(e2o / r2o)) if r2o > 0 else float(np.sqrt(e2o))
    e_s = None if hT is None else (float(np.sqrt(e2s / r2s)) if r2s > 0 else float(np.sqrt(e2s)))
    return e_o, e_s
