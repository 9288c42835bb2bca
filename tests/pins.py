"""Pins for the fp64 oracle: checks against facts fixed by the pages and by mathematics.

Every pin takes an ``Oracle`` instance, so the same checks run against the real
oracle (test_oracle_pins.py) and against deliberately broken builds of it
(test_oracle_mutants.py), which shows that a plausible mistake fails a pin.

Source of the method: "Kimi K3 Architecture: Scaling 2.8T Parameters for
Long-Context Multimodal MoE" (dev.to), section "The Sequence Bottleneck":
g = g_min Sigmoid(e^{A^h} z) in (g_min, 0), alpha = e^g > e^{g_min} ~ 6.7e-3,
g_min = -5, 16-token cumulative decay in (-80, 0); "Kimi K3 - Sparsity
Mechanics..." section 2 "Temporal Sequence (KDA)": a fixed dk x dv state
updated by Householder delta updates and channel-wise forget gates.  The
update S_t = (I - b k k^T) Diag(alpha) S_{t-1} + b k v^T, o_t = S_t^T q_t.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

from oracle import chunked

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _inputs(rng, T, H, dk, dv, *, unit_k=True):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    z = rng.standard_normal((T, H, dk)) * 1.5
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    A = rng.uniform(-1.0, 1.0, H)
    return q, k, v, z, beta, A


def _close(x, ref, tol, what=""):
    x, ref = np.asarray(x, np.float64), np.asarray(ref, np.float64)
    den = max(float(np.abs(ref).max()), 1e-300)
    err = float(np.abs(x - ref).max()) / den
    assert err <= tol, f"{what}: max rel err {err:.3e} > {tol:.1e}"


# ---------------------------------------------------------------- gate

def pin_gate_closed_forms(orc):
    """g at hand-picked z: Sigmoid(0) = 1/2, Sigmoid(ln 3) = 3/4, the two limits."""
    z = np.array([[[0.0, 800.0, -800.0, math.log(3.0), 1.5, -1.5]]])
    g, _, _ = orc.gate(z, [0.0], [0, 1])
    g = g[0, 0]
    assert g[0] == -2.5, g[0]
    assert g[1] == -5.0, g[1]
    assert g[2] == 0.0, g[2]
    assert abs(g[3] - (-3.75)) < 1e-14, g[3]
    # Sigmoid(x) + Sigmoid(-x) = 1  =>  g(z) + g(-z) = g_min
    assert abs(g[4] + g[5] - (-5.0)) < 1e-14
    # exp(A) multiplies z: with A = ln 3, z = 1/3 behaves like z = 1 at A = 0
    g3, _, _ = orc.gate(np.array([[[1.0 / 3.0]]]), [math.log(3.0)], [0, 1])
    g1, _, _ = orc.gate(np.array([[[1.0]]]), [0.0], [0, 1])
    assert abs(g3[0, 0, 0] - g1[0, 0, 0]) < 1e-14


def pin_gate_bounds(orc):
    """g in [g_min, 0], alpha >= e^{g_min}; the page's printed constants."""
    gold = json.load(open(os.path.join(GOLDEN, "gate_bounds.json")))
    g_min = float(gold["g_min"])
    assert round(math.exp(g_min), 4) == gold["alpha_lower_bound_printed"]
    assert gold["tile_tokens"] * g_min == gold["tile_cumulative_log_decay_open"][0]
    rng = np.random.default_rng(1)
    z = rng.standard_normal((50, 3, 16)) * 20.0
    g, _, _ = orc.gate(z, [-1.0, 0.0, 1.0], [0, 50])
    assert np.all(g >= g_min) and np.all(g <= 0.0)
    assert np.all(np.exp(g) >= math.exp(g_min))
    # strictly inside for moderate z (the open interval)
    gm, _, _ = orc.gate(rng.standard_normal((20, 3, 8)), [-1.0, 0.0, 1.0], [0, 20])
    assert np.all(gm > g_min) and np.all(gm < 0.0)
    # monotone decreasing in z
    zs = np.linspace(-6, 6, 97)[:, None, None]
    gs, _, _ = orc.gate(zs, [0.3], [0, 97])
    assert np.all(np.diff(gs[:, 0, 0]) < 0)


def pin_tile_cumsum(orc):
    """In-tile cumulative decay: restarts every 16 tokens and at each sequence start."""
    z = np.full((40, 1, 2), 800.0)  # g = -5 exactly everywhere
    g, G, bad = orc.gate(z, [0.0], [0, 10, 40])
    assert bad == 0, "the closed interval [-80, 0] must accept -80 exactly"
    assert G[9, 0, 0] == -50.0            # sequence 0 ends after 10 tokens
    assert G[10, 0, 0] == -5.0            # sequence 1 restarts
    assert G[25, 0, 0] == -80.0           # 16th token of sequence 1's first tile
    assert G[26, 0, 0] == -5.0            # next tile restarts
    assert G[39, 0, 0] == -70.0
    _, _, bad6 = orc.gate(z, [0.0], [0, 10, 40], g_min=-6.0)
    assert bad6 > 0, "tile sums of -96 must be flagged"
    zn = z.copy()
    zn[3, 0, 1] = np.nan
    _, _, badn = orc.gate(zn, [0.0], [0, 10, 40])
    assert badn > 0, "NaN must be flagged"


def pin_softplus_baseline(orc):
    """The unbounded baseline: -Softplus(0) = -ln 2, -> 0 for large negative arguments,
    -> -x for large positive ones; below g_min where the bounded gate saturates."""
    z = np.array([[[0.0, -60.0, 50.0, 10.0, 2.0]]])
    g, _, _ = orc.gate(z, [0.0], [0, 1], softplus=True)
    g = g[0, 0]
    assert abs(g[0] + math.log(2.0)) < 1e-15
    assert -1e-25 < g[1] < 0.0
    assert g[2] == -50.0
    assert abs(g[3] + (10.0 + math.log1p(math.exp(-10.0)))) < 1e-12
    assert abs(g[4] + math.log1p(math.exp(2.0))) < 1e-14
    # 16 tokens at z = 10 leave the bounded gate at the -80 edge and the baseline far below it
    zt = np.full((16, 1, 1), 10.0)
    _, Gb, bad_b = orc.gate(zt, [0.0], [0, 16])
    _, Gs, bad_s = orc.gate(zt, [0.0], [0, 16], softplus=True)
    assert bad_b == 0 and Gb[-1, 0, 0] >= -80.0
    assert bad_s > 0 and Gs[-1, 0, 0] < -160.0


# ---------------------------------------------------------------- recurrence

def pin_single_step(orc):
    """From a zero state: S_1 = b k v^T and o_1 = b (q.k) v (output after the update)."""
    rng = np.random.default_rng(2)
    q, k, v, z, beta, A = _inputs(rng, 1, 2, 5, 3, unit_k=False)
    out = orc.forward(q, k, v, z, beta, A, [0, 1])
    for h in range(2):
        S1 = beta[0, h] * np.outer(k[0, h], v[0, h])
        _close(out["state"][0, h], S1, 1e-14, "S_1")
        _close(out["o"][0, h], beta[0, h] * (q[0, h] @ k[0, h]) * v[0, h], 1e-14, "o_1")


def pin_dense_bruteforce(orc):
    """Explicit dense (I - b k k^T) and Diag(alpha) matrices, multiplied out."""
    rng = np.random.default_rng(3)
    H, dk, dv = 2, 5, 4
    lens = [3, 5]
    T = sum(lens)
    q, k, v, z, beta, A = _inputs(rng, T, H, dk, dv, unit_k=False)
    h0 = rng.standard_normal((2, H, dk, dv))
    cu = [0, 3, 8]
    g, _, _ = orc.gate(z, A, cu)
    out = orc.forward(q, k, v, z, beta, A, cu, h0)
    for n in range(2):
        for h in range(H):
            S = h0[n, h].copy()
            for t in range(cu[n], cu[n + 1]):
                house = np.eye(dk) - beta[t, h] * np.outer(k[t, h], k[t, h])
                S = house @ np.diag(np.exp(g[t, h])) @ S + beta[t, h] * np.outer(k[t, h], v[t, h])
                _close(out["o"][t, h], S.T @ q[t, h], 1e-12, "o")
            _close(out["state"][n, h], S, 1e-12, "state")


def pin_noop(orc):
    """beta = 0 and alpha = 1: the state never changes and o_t = S_0^T q_t."""
    rng = np.random.default_rng(4)
    q, k, v, z, beta, A = _inputs(rng, 7, 2, 4, 6)
    z[:] = -1e4      # Sigmoid -> 0, g -> -0, alpha = 1
    beta[:] = 0.0
    h0 = rng.standard_normal((1, 2, 4, 6))
    out = orc.forward(q, k, v, z, beta, A, [0, 7], h0)
    assert np.array_equal(out["state"], h0)
    for t in range(7):
        for h in range(2):
            _close(out["o"][t, h], h0[0, h].T @ q[t, h], 1e-14, "o")


def pin_pure_decay(orc):
    """beta = 0: S_T = Diag(exp(sum_t g_t)) S_0, rows (key channels) scaled, dk != dv."""
    rng = np.random.default_rng(5)
    T, H, dk, dv = 6, 2, 7, 3
    q, k, v, z, beta, A = _inputs(rng, T, H, dk, dv)
    beta[:] = 0.0
    h0 = rng.standard_normal((1, H, dk, dv))
    g, _, _ = orc.gate(z, A, [0, T], tile=64)
    out = orc.forward(q, k, v, z, beta, A, [0, T], h0)
    Gc = np.cumsum(g, axis=0)
    for h in range(H):
        _close(out["state"][0, h], np.exp(Gc[-1, h])[:, None] * h0[0, h], 1e-12, "S_T")
        for t in range(T):
            _close(out["o"][t, h], (np.exp(Gc[t, h])[:, None] * h0[0, h]).T @ q[t, h], 1e-12,
                   "o_t")


def pin_householder(orc):
    """beta = 1, |k| = 1: (I - k k^T) projects, so k_t^T S_t = v_t^T; with q = k, o_t = v_t."""
    rng = np.random.default_rng(6)
    T, H, dk, dv = 12, 2, 6, 5
    q, k, v, z, beta, A = _inputs(rng, T, H, dk, dv)
    beta[:] = 1.0
    h0 = rng.standard_normal((1, H, dk, dv))
    out = orc.forward(k.copy(), k, v, z, beta, A, [0, T], h0)
    _close(out["o"], v, 1e-12, "k^T S_t vs v_t")


def pin_contraction(orc):
    """v = 0, |k| = 1, beta in (0, 1), alpha <= 1: ||S_t||_F never grows."""
    rng = np.random.default_rng(7)
    T, H, dk, dv = 24, 2, 6, 4
    q, k, v, z, beta, A = _inputs(rng, T, H, dk, dv)
    v[:] = 0.0
    S = rng.standard_normal((1, H, dk, dv))
    prev = np.linalg.norm(S.reshape(H, -1), axis=1)
    for t in range(T):
        sl = slice(t, t + 1)
        S = orc.forward(q[sl], k[sl], v[sl], z[sl], beta[sl], A, [0, 1], S, want_o=False)["state"]
        cur = np.linalg.norm(S.reshape(H, -1), axis=1)
        assert np.all(cur <= prev * (1 + 1e-13)), (t, cur, prev)
        prev = cur


def pin_split_resume(orc):
    """Prefill [0, t) then [t, T) from the carried state equals one pass (bit for bit)."""
    rng = np.random.default_rng(8)
    T, H, dk, dv = 37, 2, 5, 4
    q, k, v, z, beta, A = _inputs(rng, T, H, dk, dv)
    h0 = rng.standard_normal((1, H, dk, dv))
    whole = orc.forward(q, k, v, z, beta, A, [0, T], h0)
    for ts in (0, 1, 15, 16, 17, 36, 37):
        a = orc.forward(q[:ts], k[:ts], v[:ts], z[:ts], beta[:ts], A, [0, ts], h0)
        b = orc.forward(q[ts:], k[ts:], v[ts:], z[ts:], beta[ts:], A, [0, T - ts], a["state"])
        assert np.array_equal(np.concatenate([a["o"], b["o"]]), whole["o"]), ts
        assert np.array_equal(b["state"], whole["state"]), ts


def pin_varlen_independence(orc):
    """Packed sequences do not interact; an empty sequence returns its initial state."""
    rng = np.random.default_rng(9)
    lens = [5, 0, 7, 3]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, H, dk, dv = int(cu[-1]), 2, 4, 3
    q, k, v, z, beta, A = _inputs(rng, T, H, dk, dv)
    h0 = rng.standard_normal((4, H, dk, dv))
    packed = orc.forward(q, k, v, z, beta, A, cu, h0)
    for n in range(4):
        s = slice(cu[n], cu[n + 1])
        one = orc.forward(q[s], k[s], v[s], z[s], beta[s], A, [0, lens[n]], h0[n:n + 1])
        assert np.array_equal(one["o"], packed["o"][s])
        assert np.array_equal(one["state"][0], packed["state"][n])
    assert np.array_equal(packed["state"][1], h0[1])


def pin_decode_matches_prefill(orc):
    """T single-token decode steps carrying the state equal one T-token prefill."""
    rng = np.random.default_rng(10)
    T, H, dk, dv = 20, 2, 6, 5
    q, k, v, z, beta, A = _inputs(rng, T, H, dk, dv)
    h0 = rng.standard_normal((1, H, dk, dv))
    whole = orc.forward(q, k, v, z, beta, A, [0, T], h0)
    S = h0.copy()
    for t in range(T):
        o = orc.decode(q[t:t + 1], k[t:t + 1], v[t:t + 1], z[t:t + 1], beta[t:t + 1], A, S)
        assert np.array_equal(o[0], whole["o"][t])
    assert np.array_equal(S, whole["state"])


def pin_chunk_algebra(orc):
    """The chunkwise form (W/U/T, decay-masked products) equals the sequential definition."""
    rng = np.random.default_rng(11)
    lens = [70, 33]
    cu = [0, 70, 103]
    T, H, dk, dv = 103, 2, 8, 6
    q, k, v, z, beta, A = _inputs(rng, T, H, dk, dv)
    h0 = rng.standard_normal((2, H, dk, dv)) * 0.1
    ref = orc.forward(q, k, v, z, beta, A, cu, h0)
    for C in (16, 32, 64):
        for tile_ref in (False, True):
            got = chunked.forward(q, k, v, z, beta, A, cu, h0, chunk=C, tile_ref=tile_ref)
            _close(got["o"], ref["o"], 1e-10, f"o C={C} tile_ref={tile_ref}")
            _close(got["state"], ref["state"], 1e-10, f"S C={C} tile_ref={tile_ref}")


def pin_column_blocks(orc):
    """Columns of S evolve independently: any column split gives identical bits."""
    rng = np.random.default_rng(12)
    T, H, dk, dv = 9, 2, 5, 7
    q, k, v, z, beta, A = _inputs(rng, T, H, dk, dv)
    h0 = rng.standard_normal((1, H, dk, dv))
    outs = [orc.forward(q, k, v, z, beta, A, [0, T], h0, col_block=cb) for cb in (1, 3, 7)]
    for o in outs[1:]:
        assert np.array_equal(o["o"], outs[0]["o"])
        assert np.array_equal(o["state"], outs[0]["state"])


def pin_bf16_reader(orc):
    """bf16 bit patterns widen to the values IEEE fixes."""
    bits = np.array([0x3F80, 0xC000, 0x7F80, 0x0001, 0x3EAB], np.uint16)
    x = orc.widen(bits)
    assert x[0] == 1.0 and x[1] == -2.0 and math.isinf(x[2])
    assert x[3] == 2.0 ** -133
    assert x[4] == 0.25 * (1.0 + 43.0 / 128.0)  # exponent 125, mantissa 0x2B


def pin_score_sums(orc):
    """The in-oracle scoring path (o_cmp) sums the same squares as a direct comparison."""
    rng = np.random.default_rng(13)
    T, H, dk, dv = 11, 2, 4, 5
    q, k, v, z, beta, A = _inputs(rng, T, H, dk, dv)
    ref = orc.forward(q, k, v, z, beta, A, [0, 4, 11])
    pert = ref["o"] + rng.standard_normal(ref["o"].shape) * 1e-3
    sc = orc.forward(q, k, v, z, beta, A, [0, 4, 11], want_o=False, o_cmp=pert)
    for n, s in enumerate((slice(0, 4), slice(4, 11))):
        for h in range(H):
            e2 = np.sum((ref["o"][s, h] - pert[s, h]) ** 2)
            r2 = np.sum(ref["o"][s, h] ** 2)
            assert abs(sc["err2"][n, h] - e2) <= 1e-12 * e2
            assert abs(sc["ref2"][n, h] - r2) <= 1e-12 * r2


def pin_segment_maps(orc):
    """The final state is affine in the initial one, S_T = M S_0 + B: M is the final state
    from S_0 = I with v = 0 (the state's evolution without values) and B the final state
    from S_0 = 0.  The maps of consecutive segments compose into the whole sequence's; this
    is the algebra the segment-parallel prefill relies on."""
    rng = np.random.default_rng(12)
    T, H, dk, dv = 30, 2, 5, 4
    q, k, v, z, beta, A = _inputs(rng, T, H, dk, dv)
    h0 = rng.standard_normal((1, H, dk, dv))
    whole = orc.forward(q, k, v, z, beta, A, [0, T], h0)["state"][0]

    def seg_map(a, b):
        n = b - a
        eye = np.broadcast_to(np.eye(dk), (1, H, dk, dk)).copy()
        M = orc.forward(q[a:b], k[a:b], np.zeros((n, H, dk)), z[a:b], beta[a:b], A, [0, n],
                        eye)["state"][0]
        B = orc.forward(q[a:b], k[a:b], v[a:b], z[a:b], beta[a:b], A, [0, n])["state"][0]
        return M, B

    M, B = seg_map(0, T)
    _close(np.einsum("hij,hjk->hik", M, h0[0]) + B, whole, 1e-12, "S_T = M S_0 + B")
    for t in (7, 16, 23):
        M1, B1 = seg_map(0, t)
        M2, B2 = seg_map(t, T)
        s1 = np.einsum("hij,hjk->hik", M1, h0[0]) + B1
        _close(np.einsum("hij,hjk->hik", M2, s1) + B2, whole, 1e-12, f"composed at {t}")


PINS = [pin_gate_closed_forms, pin_gate_bounds, pin_tile_cumsum, pin_softplus_baseline,
        pin_single_step,
        pin_dense_bruteforce, pin_noop, pin_pure_decay, pin_householder, pin_contraction,
        pin_split_resume, pin_varlen_independence, pin_decode_matches_prefill,
        pin_chunk_algebra, pin_column_blocks, pin_bf16_reader, pin_score_sums,
        pin_segment_maps]
