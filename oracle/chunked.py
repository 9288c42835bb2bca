"""fp64 chunkwise restatement of the KDA recurrence (numpy).

TEST INFRASTRUCTURE ONLY.  This is not the oracle the GPU is scored against
(that is the sequential definition in kda_oracle.c); it restates the
chunkwise-parallel form so that a test can show, in fp64, that the chunk
algebra reaches the same result as the token-by-token definition.  It shares
nothing with the CUDA code.

The dev.to page "Kimi K3 Architecture: Scaling 2.8T Parameters for
Long-Context Multimodal MoE", section "The Sequence Bottleneck", says the
model runs KDA in a chunkwise-parallel form whose diagonal and off-diagonal
16-token tiles are dense matrix products, kept in range by the bound on the
cumulative log-decay.  The pages print no chunk equations; the ones below are
derived from the recurrence
    S_t = (I - b_t k_t k_t^T) Diag(a_t) S_{t-1} + b_t k_t v_t^T,  o_t = S_t^T q_t.
Within a chunk with start state S0, G_r = sum_{m<=r} g_m (a dk-vector),
Gam_r = exp(G_r):
    A_rj = b_r (k_r * Gam_r) . (k_j / Gam_j)   for j < r   (strictly lower)
    T    = (I + A)^-1
    W    = T diag(b) (K * Gam),   Ut = T diag(b) V,   U = Ut - W S0
    O    = (Q * Gam) S0 + tril_incl((Q * Gam)(K / Gam)^T) U
    S_C  = Diag(Gam_C) S0 + (K * Gam_C / Gam)^T U
Substituting S_r = Diag(Gam_r)[S0 + sum_{j<=r} (k_j/Gam_j) u_j^T] into the
recurrence and matching the k_r term gives
    u_r + sum_{j<r} A_rj u_j = b_r (v_r - (k_r*Gam_r)^T S0),
i.e. (I + A) U = diag(b)(V - (K*Gam) S0), which is the W/Ut/U line; reading
o_r = S_r^T q_r and S_C off the same expression gives the last two lines.

With ``tile_ref=True`` the decay factor exp(G_r - G_j) inside A and P is split
per 16-row tile a as exp(G_r - ref_a) * exp(ref_a - G_j), ref_a the cumulative
sum at the end of the previous tile: the factorisation that keeps every factor
within e^{+-80} in reduced precision.  In fp64 both ways agree.
"""
from __future__ import annotations

import numpy as np

from . import oracle as _orc


def _tile_ref_factor(G: np.ndarray, tile: int) -> np.ndarray:
    """ref[r] = cumulative decay at the end of the tile before row r's tile (0 in tile 0)."""
    C = G.shape[0]
    ref = np.zeros_like(G)
    for r in range(C):
        a = r // tile
        ref[r] = G[a * tile - 1] if a > 0 else 0.0
    return ref


def _decay_products(Xr, Kc, G, tile_ref: bool, tile: int):
    """M_rj = sum_c Xr_rc Kc_jc exp(G_rc - G_jc) for all r, j (j <= r used)."""
    if not tile_ref:
        return (Xr * np.exp(G)) @ (Kc / np.exp(G)).T
    C = G.shape[0]
    ref = _tile_ref_factor(G, tile)
    M = np.zeros((C, C))
    for r in range(C):
        row = Xr[r] * np.exp(G[r] - ref[r])
        cols = Kc * np.exp(ref[r][None, :] - G)
        M[r] = cols @ row
    return M


def forward(q, k, v, z, beta, A_log, cu_seqlens, h0=None, *, chunk: int = 64,
            tile_ref: bool = False, tile: int = 16, g_min: float = _orc.G_MIN):
    """Chunkwise fp64 KDA forward.  Same arguments and shapes as oracle.forward."""
    q, k, v, z, beta = (_orc.widen(np.ascontiguousarray(x)) for x in (q, k, v, z, beta))
    T, H, dk = q.shape
    dv = v.shape[2]
    cu = np.asarray(cu_seqlens, np.int64)
    N = len(cu) - 1
    g, _, _ = _orc.gate(z, A_log, cu, tile=tile, g_min=g_min)
    o = np.zeros((T, H, dv))
    hT = np.zeros((N, H, dk, dv))
    for n in range(N):
        for h in range(H):
            S = np.zeros((dk, dv)) if h0 is None else np.array(h0[n, h], np.float64)
            for c0 in range(cu[n], cu[n + 1], chunk):
                c1 = min(c0 + chunk, cu[n + 1])
                Q, K, V = q[c0:c1, h], k[c0:c1, h], v[c0:c1, h]
                b = beta[c0:c1, h]
                G = np.cumsum(g[c0:c1, h], axis=0)
                Gam = np.exp(G)
                C = c1 - c0
                A = np.tril(b[:, None] * _decay_products(K, K, G, tile_ref, tile), -1)
                Tm = np.linalg.solve(np.eye(C) + A, np.eye(C))
                W = Tm @ (b[:, None] * (K * Gam))
                Ut = Tm @ (b[:, None] * V)
                U = Ut - W @ S
                P = np.tril(_decay_products(Q, K, G, tile_ref, tile))
                o[c0:c1, h] = (Q * Gam) @ S + P @ U
                S = Gam[-1][:, None] * S + (K * (Gam[-1][None, :] / Gam)).T @ U
            hT[n, h] = S
    return {"o": o, "state": hT}
