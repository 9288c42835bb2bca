// kda_gate.cu -- chunk plan of packed sequences and the standalone gate kernel.
//
// Gate (dev.to page "Kimi K3 Architecture...", section "The Sequence
// Bottleneck", display equation): g = -5 Sigmoid(exp(A_h) z) per channel.
// The paragraph after it bounds every 16-token tile's cumulative log-decay to
// (-80, 0); the kernel below checks that bound tile by tile while it forms the
// in-chunk inclusive cumulative sum the chunked form consumes.
#include "kda_common.cuh"

namespace kda {

// chunk_off[n] = sum over m < n of ceil(len_m / C), for n = 0..N (CTA 0).
// Validates cu_seqlens (0-based, non-decreasing, ending at T_tot); an invalid
// sequence is recorded as KDA_ERR_SEQLENS and given zero chunks.  With
// clear_status the grid's single CTA first zeroes the status word (it is the first
// kernel of a call, so nothing has reported yet).  With S_run != NULL every CTA also
// gives each sequence that owns no chunk (empty or invalid) its final state: h0's
// (zeros when h0 is NULL) -- the chunk kernels only write states of sequences they walk.
constexpr int PLAN_THREADS = 256;
__global__ void __launch_bounds__(PLAN_THREADS)
plan_chunks_kernel(const int32_t *__restrict__ cu, int N, int64_t T_tot, int C,
                   int32_t *__restrict__ chunk_off, StatusWord *st, int clear_status,
                   const float *__restrict__ h0, float *__restrict__ S_run, int H,
                   int64_t dkdv4) {
    if (S_run) {   // grid-stride over (sequence, head) pairs of chunk-less sequences
        for (int64_t nh = blockIdx.x; nh < (int64_t)N * H; nh += gridDim.x) {
            const int n = (int)(nh / H);
            const int64_t b = cu[n], e = cu[n + 1];
            if (b < e && b >= 0 && e <= T_tot) continue;
            float4 *dst = reinterpret_cast<float4 *>(S_run) + nh * dkdv4;
            const float4 *src = h0 ? reinterpret_cast<const float4 *>(h0) + nh * dkdv4 : nullptr;
            for (int64_t i = threadIdx.x; i < dkdv4; i += blockDim.x)
                dst[i] = src ? src[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    if (blockIdx.x != 0) return;
    constexpr int NW = PLAN_THREADS / 32;
    __shared__ int32_t s_warp[NW];
    __shared__ int32_t s_carry;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (clear_status && tid == 0) {
        st->code = 0u;
        st->site = 0u;
        st->info = 0ull;
    }
    __syncthreads();
    if (tid == 0) {
        s_carry = 0;
        if (cu[0] != 0 || (int64_t)cu[N] != T_tot) report(st, KDA_ERR_SEQLENS, N, 1);
    }
    __syncthreads();
    for (int base = 0; base < N; base += PLAN_THREADS) {
        const int n = base + tid;
        int32_t cnt = 0;
        if (n < N) {
            const int64_t b = cu[n], e = cu[n + 1];
            if (b < 0 || e < b || e > T_tot) {
                report(st, KDA_ERR_SEQLENS, n, 2);
            } else {
                cnt = (int32_t)((e - b + C - 1) / C);
            }
        }
        int32_t x = cnt;  // inclusive warp scan
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) s_warp[wid] = x;
        __syncthreads();
        if (wid == 0) {
            int32_t w = lane < NW ? s_warp[lane] : 0;
#pragma unroll
            for (int o = 1; o < NW; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            if (lane < NW) s_warp[lane] = w;
        }
        __syncthreads();
        const int32_t incl = x + (wid > 0 ? s_warp[wid - 1] : 0) + s_carry;
        if (n < N) chunk_off[n] = incl - cnt;
        __syncthreads();
        if (tid == PLAN_THREADS - 1) s_carry = incl;
        __syncthreads();
    }
    if (tid == 0) chunk_off[N] = s_carry;
}

// Sequence owning global chunk `slot` (chunk_off is non-decreasing): the
// largest n with chunk_off[n] <= slot, or -1 when slot >= chunk_off[N].
__device__ __forceinline__ int find_seq(const int32_t *chunk_off, int N, int32_t slot) {
    if (slot >= chunk_off[N]) return -1;
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (chunk_off[mid] <= slot) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// The unbounded baseline the lower-bounded gate replaces (same section of the
// dev.to page: "replaces unbounded negative Softplus decay"): g = -Softplus(e^A z).
__device__ __forceinline__ float gate_softplus(float z, float expA) {
    const float x = expA * z;
    return x > 40.f ? -x : -log1pf(expf(x));
}

// One CTA per (chunk slot, head); thread c walks channel c of the chunk.
// mode 0: the lower-bounded gate; mode 1: the Softplus baseline.
template <typename T>
__global__ void gate_cumsum_kernel(const T *__restrict__ z, const float *__restrict__ A_log,
                                   const int32_t *__restrict__ cu,
                                   const int32_t *__restrict__ chunk_off, int N, int H, int dk,
                                   int C, int mode, float *__restrict__ G, StatusWord *st) {
    const int32_t slot = blockIdx.x;
    const int h = blockIdx.y;
    const int n = find_seq(chunk_off, N, slot);
    if (n < 0) return;
    const int64_t t0 = (int64_t)cu[n] + (int64_t)(slot - chunk_off[n]) * C;
    const int64_t t1 = min(t0 + C, (int64_t)cu[n + 1]);
    const float expA = expf(A_log[h]);
    for (int c = threadIdx.x; c < dk; c += blockDim.x) {
        float run = 0.f, tile = 0.f;
        for (int64_t t = t0; t < t1; ++t) {
            const int64_t idx = (t * H + h) * (int64_t)dk + c;
            const float zz = to_f(z[idx]);
            const float g = mode == 1 ? gate_softplus(zz, expA) : gate(zz, expA);
            if (((t - t0) % kTile) == 0) tile = 0.f;
            run += g;
            tile += g;
            if (!decay_ok(tile)) report(st, KDA_ERR_DECAY_RANGE, t * H + h, 3);
            G[idx] = run;
        }
    }
}

cudaError_t launch_plan(const int32_t *cu, int N, int64_t T_tot, int C, int32_t *chunk_off,
                        StatusWord *st, cudaStream_t s) {
    plan_chunks_kernel<<<1, PLAN_THREADS, 0, s>>>(cu, N, T_tot, C, chunk_off, st, 0, nullptr, nullptr,
                                          0, 0);
    return cudaGetLastError();
}

// The plan of the tensor-core path: also clears the status word and writes the final
// states of chunk-less sequences into S_run (skipped when S_run is h0, an in-place update).
cudaError_t launch_plan_tc(const int32_t *cu, int N, int64_t T_tot, int C, int32_t *chunk_off,
                           StatusWord *st, const float *h0, float *S_run, int H, int64_t dkdv,
                           int grid, cudaStream_t s) {
    const bool init = S_run != h0;
    plan_chunks_kernel<<<init ? grid : 1, PLAN_THREADS, 0, s>>>(cu, N, T_tot, C, chunk_off, st, 1, h0,
                                                       init ? S_run : nullptr, H, dkdv / 4);
    return cudaGetLastError();
}

int64_t chunk_slots(int64_t T_tot, int N, int C) { return (T_tot + C - 1) / C + N; }

cudaError_t launch_gate(int dtype, const void *z, const float *A_log, const int32_t *cu,
                        const int32_t *chunk_off, int N, int64_t T_tot, int H, int dk, int C,
                        int mode, float *G, StatusWord *st, cudaStream_t s) {
    const int64_t slots = chunk_slots(T_tot, N, C);
    if (slots <= 0) return cudaSuccess;
    dim3 grid((unsigned)slots, (unsigned)H);
    if (dtype == KDA_BF16)
        gate_cumsum_kernel<__nv_bfloat16><<<grid, dk, 0, s>>>(
            (const __nv_bfloat16 *)z, A_log, cu, chunk_off, N, H, dk, C, mode, G, st);
    else
        gate_cumsum_kernel<float><<<grid, dk, 0, s>>>((const float *)z, A_log, cu, chunk_off, N,
                                                      H, dk, C, mode, G, st);
    return cudaGetLastError();
}

}  // namespace kda
