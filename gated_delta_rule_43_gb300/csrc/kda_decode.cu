// kda_decode.cu -- one KDA decode step against a resident fp32 state (memory-bound).
//
// Per (sequence n, head h) and value column j, with s = Diag(alpha) S[:, j]:
//   a_j = k . s,   b_j = q . s,   u_j = beta (v_j - a_j)
//   S[:, j] <- s + k u_j                       (= (I - beta k k^T) s + beta k v_j)
//   o_j     = b_j + (q . k) u_j                (= q . S[:, j] after the update)
// which is the update of the dev.to page "Kimi K3 Architecture...", section
// "The Sequence Bottleneck" (state S_t, retention alpha_t, delta strength
// beta_t) for a single token.  The state is read once and written once: one
// CTA per (n, h, block of value columns; two 64-column blocks at dv = 128), each
// thread holding R rows x 4 columns of S in registers between the read and the
// write, so no column is fetched twice.
//
// With a slot index, sequence n reads and writes slot slot_idx[n] of a state
// pool [P, H, dk, dv] instead of state n (the fixed-size KDA states of the
// paged hybrid cache, dev.to page "Kimi K3 Architecture...", section
// "Infrastructure and Training/Inference Mechanics", serving engine).
#include "kda_common.cuh"

namespace kda {

constexpr int kDecodeThreads = 128;   // measured: 128 threads (16 rows x 4 columns each at dk = 128) beat 256 by 5%
constexpr int kDecodeSplit128 = 64;   // value columns per CTA at dv = 128

// One CTA per (n, h, block of DVC value columns); DV / DVC CTAs share one (n, h).
template <int DK, int DV, int DVC, typename T>
__global__ void __launch_bounds__(kDecodeThreads)
decode_step_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                   const T *__restrict__ z, const T *__restrict__ beta,
                   const float *__restrict__ A_log, float *__restrict__ state,
                   T *__restrict__ o, int H, const int32_t *__restrict__ slot_idx, int P,
                   StatusWord *st) {
    constexpr int TPR = DVC / 4;                // threads covering one row (float4 each)
    constexpr int RPP = kDecodeThreads / TPR;   // rows covered per pass
    constexpr int R = DK / RPP;                 // rows per thread
    constexpr int NCB = DV / DVC;
    static_assert(DVC % 4 == 0 && DV % DVC == 0 && kDecodeThreads % TPR == 0 && DK % RPP == 0,
                  "shape");

    __shared__ float s_k[DK], s_q[DK], s_alpha[DK];
    __shared__ float s_v[DVC], s_u[DVC];
    __shared__ __align__(16) float s_pa[RPP][DVC];
    __shared__ __align__(16) float s_pb[RPP][DVC];
    __shared__ float s_qk, s_beta;

    const int nh = blockIdx.x / NCB;
    const int j0 = (blockIdx.x % NCB) * DVC;
    const int h = nh % H;
    const int n = nh / H;
    const int tid = threadIdx.x;
    const int64_t kb = (int64_t)nh * DK;
    const int64_t vb = (int64_t)nh * DV + j0;
    const int slot = slot_idx ? slot_idx[n] : n;
    if (slot < 0 || slot >= P) {
        if (tid == 0 && h == 0 && j0 == 0) report(st, KDA_ERR_INVALID_ARG, n, 20);
        return;
    }

    // Issue the state loads first: they are the bulk of the traffic.
    const int c4 = tid % TPR;
    const int rg = tid / TPR;
    float4 *S4 = reinterpret_cast<float4 *>(state + ((int64_t)slot * H + h) * DK * DV + j0);
    float4 s[R];
#pragma unroll
    for (int p = 0; p < R; ++p) s[p] = __ldcs(S4 + (int64_t)(rg + p * RPP) * (DV / 4) + c4);

    const float expA = expf(A_log[h]);
    for (int i = tid; i < DK; i += kDecodeThreads) {
        s_alpha[i] = expf(gate(to_f(z[kb + i]), expA));
        s_k[i] = to_f(k[kb + i]);
        s_q[i] = to_f(q[kb + i]);
    }
    for (int j = tid; j < DVC; j += kDecodeThreads) s_v[j] = to_f(v[vb + j]);
    if (tid == 0) s_beta = to_f(beta[nh]);
    __syncthreads();
    if (tid < 32) {
        float acc = 0.f;
        for (int i = tid; i < DK; i += 32) acc += s_q[i] * s_k[i];
        acc = warp_sum(acc);
        if (tid == 0) s_qk = acc;
    }

    float pa[4] = {0.f, 0.f, 0.f, 0.f}, pb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int p = 0; p < R; ++p) {
        const int row = rg + p * RPP;
        const float al = s_alpha[row], kr = s_k[row], qr = s_q[row];
        s[p].x *= al; s[p].y *= al; s[p].z *= al; s[p].w *= al;
        pa[0] += kr * s[p].x; pa[1] += kr * s[p].y; pa[2] += kr * s[p].z; pa[3] += kr * s[p].w;
        pb[0] += qr * s[p].x; pb[1] += qr * s[p].y; pb[2] += qr * s[p].z; pb[3] += qr * s[p].w;
    }
    // one 16-byte store per thread: consecutive threads fill consecutive columns
    *reinterpret_cast<float4 *>(&s_pa[rg][c4 * 4]) = make_float4(pa[0], pa[1], pa[2], pa[3]);
    *reinterpret_cast<float4 *>(&s_pb[rg][c4 * 4]) = make_float4(pb[0], pb[1], pb[2], pb[3]);
    __syncthreads();
    for (int j = tid; j < DVC; j += kDecodeThreads) {
        float a = 0.f, b = 0.f;
#pragma unroll 8
        for (int g = 0; g < RPP; ++g) {
            a += s_pa[g][j];
            b += s_pb[g][j];
        }
        const float u = s_beta * (s_v[j] - a);
        s_u[j] = u;
        o[vb + j] = from_f<T>(b + s_qk * u);
    }
    __syncthreads();
    const float u0 = s_u[c4 * 4 + 0], u1 = s_u[c4 * 4 + 1];
    const float u2 = s_u[c4 * 4 + 2], u3 = s_u[c4 * 4 + 3];
#pragma unroll
    for (int p = 0; p < R; ++p) {
        const int row = rg + p * RPP;
        const float kr = s_k[row];
        float4 w = s[p];
        w.x += kr * u0; w.y += kr * u1; w.z += kr * u2; w.w += kr * u3;
        S4[(int64_t)row * (DV / 4) + c4] = w;   // plain store: measured ~1% faster than .cs
    }
}

template <int DK, int DV, typename T>
static cudaError_t launch_decode_t(const void *q, const void *k, const void *v, const void *z,
                                   const void *beta, const float *A_log, float *state, void *o,
                                   int N, int H, const int32_t *slot_idx, int P, StatusWord *st,
                                   cudaStream_t stream) {
    // dv = 128 splits into two 64-column CTAs: half the registers per thread, so more CTAs
    // (and more of the state) in flight per SM
    constexpr int DVC = DV == 128 ? kDecodeSplit128 : DV;
    decode_step_kernel<DK, DV, DVC, T>
        <<<(unsigned)((int64_t)N * H * (DV / DVC)), kDecodeThreads, 0, stream>>>(
        (const T *)q, (const T *)k, (const T *)v, (const T *)z, (const T *)beta, A_log, state,
        (T *)o, H, slot_idx, P, st);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_decode_dt(int dk, int dv, const void *q, const void *k, const void *v,
                                    const void *z, const void *beta, const float *A_log,
                                    float *state, void *o, int N, int H,
                                    const int32_t *slot_idx, int P, StatusWord *st,
                                    cudaStream_t s) {
#define KDA_DEC(DK_, DV_)                                                                    \
    if (dk == DK_ && dv == DV_)                                                              \
        return launch_decode_t<DK_, DV_, T>(q, k, v, z, beta, A_log, state, o, N, H, slot_idx, \
                                            P, st, s);
    KDA_DEC(32, 32) KDA_DEC(32, 64) KDA_DEC(32, 128)
    KDA_DEC(64, 32) KDA_DEC(64, 64) KDA_DEC(64, 128)
    KDA_DEC(128, 32) KDA_DEC(128, 64) KDA_DEC(128, 128)
#undef KDA_DEC
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode(int dtype, int dk, int dv, const void *q, const void *k,
                          const void *v, const void *z, const void *beta, const float *A_log,
                          float *state, void *o, int N, int H, const int32_t *slot_idx, int P,
                          StatusWord *st, cudaStream_t s) {
    if (dtype == KDA_BF16)
        return launch_decode_dt<__nv_bfloat16>(dk, dv, q, k, v, z, beta, A_log, state, o, N, H,
                                               slot_idx, P, st, s);
    return launch_decode_dt<float>(dk, dv, q, k, v, z, beta, A_log, state, o, N, H, slot_idx, P,
                                   st, s);
}

}  // namespace kda
