// kda_chunk_simt.cu -- chunked KDA forward on CUDA cores in fp32, 16-token chunks.
//
// This is the fp32 path (and the path for head sizes the tensor-core kernels
// do not build).  The chunk is exactly the 16-token tile of the dev.to page
// "Kimi K3 Architecture...", section "The Sequence Bottleneck": inside one
// tile the cumulative log-decay G lies in [-80, 0], so exp(G) and exp(-G) are
// both representable in fp32 and the decay-scaled products below can be
// formed directly.  Per chunk with start state S (derived from the recurrence
// S_t = (I - b k k^T) Diag(alpha) S_{t-1} + b k v^T, o_t = S_t^T q_t):
//   A  = strict_lower( diag(b) (K*Gam)(K/Gam)^T ),   T = (I + A)^-1
//   W  = T diag(b) (K*Gam),   U = T diag(b) V - W S
//   O  = (Q*Gam) S + lower_incl( (Q*Gam)(K/Gam)^T ) U
//   S <- Diag(Gam_last) S + (K*Gam_last/Gam)^T U
// One CTA owns one (sequence, head, 32-column block of dv); columns of S
// evolve independently, so the blocks never communicate.
#include "kda_common.cuh"

namespace kda {

constexpr int kSimtThreads = 256;
constexpr int kSimtC = 16;
constexpr int kSimtDVB = 32;

template <int DK>
constexpr size_t simt_smem_floats() {
    return (size_t)DK * kSimtDVB + 5 * kSimtC * (DK + 1) + DK + 2 * kSimtC * kSimtDVB +
           2 * kSimtC * (kSimtC + 1) + kSimtC;
}

template <int DK, typename T>
__global__ void __launch_bounds__(kSimtThreads)
chunk_fwd_simt_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                      const T *__restrict__ z, const T *__restrict__ beta,
                      const float *__restrict__ A_log, const int32_t *__restrict__ cu, int N,
                      int64_t T_tot, int H, int dv, const float *h0, float *hT,
                      T *__restrict__ o, StatusWord *st) {
    constexpr int C = kSimtC, DVB = kSimtDVB, NT = kSimtThreads;
    constexpr int LD = DK + 1;      // padded row stride of the [C][DK] tiles
    constexpr int LC = C + 1;       // padded row stride of the [C][C] tiles
    static_assert(C * C == NT, "one thread per (r, j) of a CxC tile");
    extern __shared__ float smem[];
    float *S = smem;                 // [DK][DVB] state block
    float *Kg = S + DK * DVB;        // [C][LD] k * Gam
    float *Ki = Kg + C * LD;         // [C][LD] k / Gam
    float *Qg = Ki + C * LD;         // [C][LD] q * Gam
    float *Kt = Qg + C * LD;         // [C][LD] k * Gam_last / Gam
    float *W = Kt + C * LD;          // [C][LD]
    float *Gl = W + C * LD;          // [DK]    Gam_last
    float *Vt = Gl + DK;             // [C][DVB]
    float *Ut = Vt + C * DVB;        // [C][DVB] U~, then U
    float *Am = Ut + C * DVB;        // [C][LC] A, then T diag(b)
    float *Pm = Am + C * LC;         // [C][LC]
    float *bt = Pm + C * LC;         // [C]

    const int nblk = dv / DVB;
    const int blk = blockIdx.x % nblk;
    const int h = (blockIdx.x / nblk) % H;
    const int n = blockIdx.x / (nblk * H);
    const int tid = threadIdx.x;
    if (n == 0 && h == 0 && blk == 0 && tid == 0 && (cu[0] != 0 || (int64_t)cu[N] != T_tot))
        report(st, KDA_ERR_SEQLENS, N, 1);
    const int64_t bos = cu[n], eos = cu[n + 1];
    if (bos < 0 || eos < bos || eos > T_tot) {
        if (tid == 0) report(st, KDA_ERR_SEQLENS, n, 2);
        return;
    }
    const int j0 = blk * DVB;
    const int64_t sb = ((int64_t)n * H + h) * (int64_t)DK * dv;
    for (int e = tid; e < DK * DVB; e += NT) {
        const int i = e / DVB, j = e % DVB;
        S[e] = h0 ? h0[sb + (int64_t)i * dv + j0 + j] : 0.f;
    }
    const float expA = expf(A_log[h]);

    for (int64_t t0 = bos; t0 < eos; t0 += C) {
        const int L = (int)min((int64_t)C, eos - t0);
        __syncthreads();
        // (1) gate, in-tile cumulative decay, decay-scaled operands
        if (tid < DK) {
            const int c = tid;
            float run = 0.f;
            float kr[C], gr[C];
#pragma unroll
            for (int r = 0; r < C; ++r) {
                float kk = 0.f, qq = 0.f, g = 0.f;
                if (r < L) {
                    const int64_t idx = ((t0 + r) * H + h) * (int64_t)DK + c;
                    kk = to_f(k[idx]);
                    qq = to_f(q[idx]);
                    g = gate(to_f(z[idx]), expA);
                }
                run += g;
                if (r < L && !decay_ok(run)) report(st, KDA_ERR_DECAY_RANGE, (t0 + r) * H + h, 4);
                const float gam = expf(run);
                Kg[r * LD + c] = kk * gam;
                Ki[r * LD + c] = kk / gam;
                Qg[r * LD + c] = qq * gam;
                kr[r] = kk;
                gr[r] = run;
            }
            Gl[c] = expf(run);
#pragma unroll
            for (int r = 0; r < C; ++r) Kt[r * LD + c] = kr[r] * expf(run - gr[r]);
        } else {
            for (int e = tid - DK; e < C * DVB; e += NT - DK) {
                const int r = e / DVB, j = e % DVB;
                Vt[e] = r < L ? to_f(v[((t0 + r) * H + h) * (int64_t)dv + j0 + j]) : 0.f;
            }
            const int r = tid - DK;
            if (r < C) bt[r] = r < L ? to_f(beta[(t0 + r) * H + h]) : 0.f;
        }
        __syncthreads();
        // (2) A (strictly lower, b-weighted) and P (lower incl.)
        {
            const int r = tid / C, j = tid % C;
            float a = 0.f, p = 0.f;
            if (j <= r) {
#pragma unroll 8
                for (int c = 0; c < DK; ++c) {
                    const float ki = Ki[j * LD + c];
                    a += Kg[r * LD + c] * ki;
                    p += Qg[r * LD + c] * ki;
                }
            }
            Am[r * LC + j] = (j < r) ? bt[r] * a : 0.f;
            Pm[r * LC + j] = (j <= r) ? p : 0.f;
        }
        __syncthreads();
        // (3) T = (I + A)^-1 by forward substitution; lane j owns column j
        if (tid < 32) {
            const int j = tid;
            float tc[C];
#pragma unroll
            for (int r = 0; r < C; ++r) {
                float s = (r == j) ? 1.f : 0.f;
#pragma unroll
                for (int m = 0; m < r; ++m) s -= Am[r * LC + m] * tc[m];
                tc[r] = s;
            }
            __syncwarp();
            if (j < C) {
                const float bj = bt[j];
#pragma unroll
                for (int r = 0; r < C; ++r) Am[r * LC + j] = tc[r] * bj;
            }
        }
        __syncthreads();
        // (4) W = T diag(b) (K*Gam),  U~ = T diag(b) V
        for (int e = tid; e < C * DK; e += NT) {
            const int r = e / DK, c = e % DK;
            float s = 0.f;
            for (int j = 0; j <= r; ++j) s += Am[r * LC + j] * Kg[j * LD + c];
            W[r * LD + c] = s;
        }
        for (int e = tid; e < C * DVB; e += NT) {
            const int r = e / DVB, jv = e % DVB;
            float s = 0.f;
            for (int j = 0; j <= r; ++j) s += Am[r * LC + j] * Vt[j * DVB + jv];
            Ut[e] = s;
        }
        __syncthreads();
        // (5) U = U~ - W S
        for (int e = tid; e < C * DVB; e += NT) {
            const int r = e / DVB, jv = e % DVB;
            float s = Ut[e];
#pragma unroll 8
            for (int c = 0; c < DK; ++c) s -= W[r * LD + c] * S[c * DVB + jv];
            Ut[e] = s;
        }
        __syncthreads();
        // (6) O = (Q*Gam) S + P U
        for (int e = tid; e < C * DVB; e += NT) {
            const int r = e / DVB, jv = e % DVB;
            if (r < L) {
                float s = 0.f;
#pragma unroll 8
                for (int c = 0; c < DK; ++c) s += Qg[r * LD + c] * S[c * DVB + jv];
                for (int j = 0; j <= r; ++j) s += Pm[r * LC + j] * Ut[j * DVB + jv];
                o[((t0 + r) * H + h) * (int64_t)dv + j0 + jv] = from_f<T>(s);
            }
        }
        __syncthreads();
        // (7) S <- Diag(Gam_last) S + (K*Gam_last/Gam)^T U
        for (int e = tid; e < DK * DVB; e += NT) {
            const int c = e / DVB, jv = e % DVB;
            float s = Gl[c] * S[e];
#pragma unroll
            for (int r = 0; r < C; ++r) s += Kt[r * LD + c] * Ut[r * DVB + jv];
            S[e] = s;
        }
    }
    __syncthreads();
    if (hT)
        for (int e = tid; e < DK * DVB; e += NT) {
            const int i = e / DVB, j = e % DVB;
            hT[sb + (int64_t)i * dv + j0 + j] = S[e];
        }
}

template <int DK, typename T>
static cudaError_t launch_simt_t(const void *q, const void *k, const void *v, const void *z,
                                 const void *beta, const float *A_log, const int32_t *cu, int N,
                                 int64_t T_tot, int H, int dv, const float *h0, float *hT,
                                 void *o, StatusWord *st, cudaStream_t s, EventRec *rec) {
    const size_t smem = simt_smem_floats<DK>() * sizeof(float);
    auto kern = chunk_fwd_simt_kernel<DK, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t grid = (int64_t)N * H * (dv / kSimtDVB);
    if (grid <= 0) return cudaSuccess;
    if (rec) rec->mark(s);
    kern<<<(unsigned)grid, kSimtThreads, smem, s>>>((const T *)q, (const T *)k, (const T *)v,
                                                    (const T *)z, (const T *)beta, A_log, cu, N,
                                                    T_tot, H, dv, h0, hT, (T *)o, st);
    if (rec) rec->mark(s);
    return cudaGetLastError();
}

cudaError_t launch_chunk_simt(int dtype, int dk, int dv, const void *q, const void *k,
                              const void *v, const void *z, const void *beta,
                              const float *A_log, const int32_t *cu, int N, int64_t T_tot, int H,
                              const float *h0, float *hT, void *o, StatusWord *st,
                              cudaStream_t s, EventRec *rec) {
#define KDA_SIMT(DK_)                                                                          \
    if (dk == DK_) {                                                                           \
        if (dtype == KDA_BF16)                                                                 \
            return launch_simt_t<DK_, __nv_bfloat16>(q, k, v, z, beta, A_log, cu, N, T_tot, H, \
                                                     dv, h0, hT, o, st, s, rec);               \
        return launch_simt_t<DK_, float>(q, k, v, z, beta, A_log, cu, N, T_tot, H, dv, h0, hT, \
                                         o, st, s, rec);                                       \
    }
    KDA_SIMT(32) KDA_SIMT(64) KDA_SIMT(128)
#undef KDA_SIMT
    return cudaErrorInvalidValue;
}

}  // namespace kda
