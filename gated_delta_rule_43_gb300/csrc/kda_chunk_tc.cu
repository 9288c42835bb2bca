// kda_chunk_tc.cu -- chunked KDA forward on the sm_103a tensor cores (bf16 operands,
// fp32 accumulation in TMEM), dk = dv = 128, 64-token chunks.
//
// The chunkwise-parallel form of the dev.to page "Kimi K3 Architecture...",
// section "The Sequence Bottleneck": within a chunk of C tokens with start
// state S, cumulative log-decay G_r = sum_{m<=r} g_m and Gam_r = exp(G_r)
// (all derived from S_t = (I - b k k^T) Diag(alpha) S_{t-1} + b k v^T,
// o_t = S_t^T q_t):
//   A  = strict_lower( diag(b) [(k_r*Gam_r).(k_j/Gam_j)] ),  T = (I + A)^-1
//   W  = T diag(b) (K*Gam),  Ut = T diag(b) V,  U = Ut - W S
//   O  = (Q*Gam) S + P U,    P = lower_incl( [(q_r*Gam_r).(k_j/Gam_j)] )
//   S <- Diag(Gam_C) S + (K*Gam_C/Gam)^T U
// Everything but the last three products is independent of S, so it runs in
// a parallel "prep" kernel over all (chunk, head) pairs; a "chain" kernel per
// (sequence, head, 32-column block of dv) then walks the chunks in order.
//
// Numerics (the page's point about 16-token tiles): exp(G_r - G_j) is never
// formed from a chunk-global exp(-G).  For row r in 16-token tile a, with
// ref_a the cumulative decay at the end of tile a-1 (0 for a = 0),
//   exp(G_r - G_j) = exp(G_r - ref_a) * exp(ref_a - G_j),
// the row factor lies in (e^-80, 1] and the column factor in [1, e^80) for
// j in tile a (the page's bound) and in (0, 1] for earlier tiles, where
// underflow only drops terms below e^-80.  Each tile a therefore multiplies
// the same row-scaled [K;Q] tile block by its own column-scaled K block.
// W, Q*Gam and K*Gam_C/Gam use exp(G) <= 1 directly.
//
// Prep output per (chunk slot, head): one record of smem images (128-byte
// swizzle) that the chain kernel copies with 1-D bulk TMA:
//   WQ  K-major [128 rows][128 K]: rows 0-63 W, rows 64-127 Q*Gam
//   KT  MN-major [64 k-rows][128 m]: K*Gam_C/Gam, read as the M=dk x K=C operand
//   P   K-major [64][64]
//   Ut  fp32 [4 column blocks][64][32]
//   GC  fp32 [128] Gam_C
#include <algorithm>

#include "kda_common.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace tc {

using namespace sm100;

constexpr int C = 64;            // chunk length (four 16-token tiles)
constexpr int DK = 128, DV = 128;
constexpr int DVB = 32;          // value columns per chain CTA
constexpr int NBLK = DV / DVB;

// record layout (bytes)
constexpr uint32_t REC_WQ = 0;
constexpr uint32_t REC_KT = 32768;
constexpr uint32_t REC_P = 49152;
constexpr uint32_t REC_U = 57344;
constexpr uint32_t REC_G = 90112;
constexpr uint32_t REC_BYTES = 90624;

// ---------------------------------------------------------------- prep kernel
constexpr int PREP_THREADS = 256;
// shared-memory map of the prep kernel (offsets from a 1024-aligned base)
constexpr uint32_t P_KRQR = 0;          // K-major [128][128] row-scaled K/Q, tile a -> rows 32a..32a+31
constexpr uint32_t P_KC = 32768;        // column-scaled K images, a = 0..3: [16(a+1)][128]
constexpr uint32_t P_RAW = 32768;       // (before them) raw bf16 tiles q, k, z: 3 x [64][128]
constexpr uint32_t P_AS = 0;            // (after the A/P products) fp32 A [64][65]
constexpr uint32_t P_TS = 16640;        //   fp32 T [64][65]
constexpr uint32_t P_XS = 33280;        //   fp32 scratch [4][16][17]
constexpr uint32_t P_UST = 37888;       //   fp32 Ut staging [4][64][32]
constexpr uint32_t P_KF = 81920;        // fp32 [64][128] k / exp(G - ref)
constexpr uint32_t P_KGV = 114688;      // MN-major [64][256]: K*Gam (n < 128) | V (n >= 128)
constexpr uint32_t P_WQ = 147456;       // K-major [128][128]
constexpr uint32_t P_KT = 180224;       // MN-major [64][128]
constexpr uint32_t P_TB = 196608;       // K-major [64][64] T diag(b); rows 64..127 of the M=128
constexpr uint32_t P_P = 204800;        //   operand read the P image that follows (ignored rows)
constexpr uint32_t P_REF = 212992;      // fp32 [5][128]: ref_0..ref_3, G_C
constexpr uint32_t P_RT = 215552;       // fp32 [10][128]: exp(ref_a - ref_b) (b<a), exp(G_C - ref_b)
constexpr uint32_t P_BETA = 220672;     // fp32 [64]
constexpr uint32_t P_HALF = 220928;     // fp32 [128] g-sum of rows 0..31 per channel
constexpr uint32_t P_BAR = 221440;      // 2 mbarriers + TMEM slot
constexpr uint32_t P_SMEM = 221504 + 1024;
static_assert(P_UST + 4 * 64 * 32 * 4 <= P_KF, "prep smem reuse overlaps");
static_assert(P_KC + 4096 + 8192 + 12288 + 16384 <= P_KF, "column-scaled K images overflow");
static_assert(P_RAW + 3 * 16384 <= P_KF, "raw tiles overflow");
static_assert(P_XS >= P_TS + 64 * 65 * 4 && P_UST >= P_XS + 4 * 16 * 17 * 4, "solve scratch");
static_assert(P_P == P_TB + 8192, "rows 64..127 of the T diag(b) operand must be valid smem");
static_assert(P_SMEM <= 232448, "prep kernel exceeds 227 KB of shared memory");

__device__ __forceinline__ void st_bf16(uint8_t *base, uint32_t off, float x) {
    *reinterpret_cast<__nv_bfloat16 *>(base + off) = __float2bfloat16_rn(x);
}

// chunk slot -> (sequence, first token, valid rows); false when the slot is unused
__device__ __forceinline__ bool slot_chunk(const int32_t *cu, const int32_t *chunk_off, int N,
                                           int32_t slot, int &n, int64_t &t0, int &L) {
    if (slot >= chunk_off[N]) return false;
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (chunk_off[mid] <= slot) lo = mid; else hi = mid - 1;
    }
    n = lo;
    t0 = (int64_t)cu[n] + (int64_t)(slot - chunk_off[n]) * C;
    L = (int)min((int64_t)C, (int64_t)cu[n + 1] - t0);
    return L > 0;
}

__global__ void __launch_bounds__(PREP_THREADS, 1)
prep_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
            const __nv_bfloat16 *__restrict__ v, const __nv_bfloat16 *__restrict__ z,
            const __nv_bfloat16 *__restrict__ beta, const float *__restrict__ A_log,
            const int32_t *__restrict__ cu, const int32_t *__restrict__ chunk_off, int N, int H,
            int32_t slot0, uint8_t *__restrict__ records, StatusWord *st) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t slot = slot0 + (int32_t)blockIdx.x;
    const int h = blockIdx.y;
    int n = 0, L = 0;
    int64_t t0 = 0;
    if (!slot_chunk(cu, chunk_off, N, slot, n, t0, L)) return;
    uint8_t *rec = records + ((size_t)blockIdx.x * H + h) * REC_BYTES;

    float *KF = reinterpret_cast<float *>(sm + P_KF);
    float *REF = reinterpret_cast<float *>(sm + P_REF);
    float *RT = reinterpret_cast<float *>(sm + P_RT);
    float *BETA = reinterpret_cast<float *>(sm + P_BETA);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + P_BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + P_BAR + 16);

    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, 256);
        tmem_relinquish();
        tc_fence_before();
    }

    // ---- (0) stage the chunk's q, k, z tiles (row-major bf16) and V (into the MN-major
    //          [K*Gam | V] image) with 16-byte loads; rows past the sequence end are zero
    {
        uint8_t *raw = sm + P_RAW;
        for (int e = tid; e < 4 * C * 16; e += PREP_THREADS) {
            const int tsel = e / (C * 16), rem = e % (C * 16);
            const int r = rem / 16, c8 = (rem % 16) * 8;
            const __nv_bfloat16 *src = tsel == 0 ? q : tsel == 1 ? k : tsel == 2 ? z : v;
            uint4 val = make_uint4(0, 0, 0, 0);
            if (r < L) val = *reinterpret_cast<const uint4 *>(src + ((t0 + r) * H + h) * (int64_t)DK + c8);
            if (tsel < 3)
                *reinterpret_cast<uint4 *>(raw + tsel * 16384 + r * 256 + c8 * 2) = val;
            else
                *reinterpret_cast<uint4 *>(sm + P_KGV + sw128_offset(r, 128 + c8, 64)) = val;
        }
        if (tid < C) BETA[tid] = tid < L ? __bfloat162float(beta[(t0 + tid) * H + h]) : 0.f;
    }
    __syncthreads();

    // ---- (1) gate, tile references and decay-scaled operands: thread (c, half) walks
    //          rows 32*half .. 32*half+31 of channel c
    {
        const int c = tid & (DK - 1), half = tid >> 7;
        const __nv_bfloat16 *rq = reinterpret_cast<const __nv_bfloat16 *>(sm + P_RAW);
        const __nv_bfloat16 *rk = rq + C * DK;
        const __nv_bfloat16 *rz = rk + C * DK;
        float *HALF = reinterpret_cast<float *>(sm + P_HALF);
        const float expA = expf(A_log[h]);
        float g[32];
        float part = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int r = 32 * half + i;
            g[i] = r < L ? gate(__bfloat162float(rz[r * DK + c]), expA) : 0.f;
            part += g[i];
        }
        if (half == 0) HALF[c] = part;
        __syncthreads();
        float run = half ? HALF[c] : 0.f;   // chunk cumsum before this thread's first row
        float ref = run, trun = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int r = 32 * half + i;
            const int a = r >> 4;
            if ((i & 15) == 0) {
                ref = run;
                trun = 0.f;
                REF[a * DK + c] = ref;
            }
            run += g[i];
            trun += g[i];
            if (r < L && !decay_ok(trun)) report(st, KDA_ERR_DECAY_RANGE, (t0 + r) * H + h, 5);
            const float kk = __bfloat162float(rk[r * DK + c]);
            const float qq = __bfloat162float(rq[r * DK + c]);
            const float F = expf(trun);          // exp(G_r - ref_a) in [e^-80, 1]
            const float Gm = expf(run);          // exp(G_r) <= 1 (may underflow)
            const uint32_t row = 32 * a + (r & 15);
            st_bf16(sm + P_KRQR, sw128_offset(row, c, 128), kk * F);
            st_bf16(sm + P_KRQR, sw128_offset(row + 16, c, 128), qq * F);
            KF[r * DK + c] = kk / F;             // k_r exp(ref_a - G_r), <= e^80 |k|
            st_bf16(sm + P_WQ, sw128_offset(64 + r, c, 128), qq * Gm);
            st_bf16(sm + P_KGV, sw128_offset(r, c, 64), kk * Gm);
        }
        if (half == 1) {
            REF[4 * DK + c] = run;
            *reinterpret_cast<float *>(rec + REC_G + 4 * c) = expf(run);
        }
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    // ---- (2) factor tables: exp(ref_a - ref_b) for b < a (6 pairs), exp(G_C - ref_b)
    for (int e = tid; e < 10 * DK; e += PREP_THREADS) {
        const int p = e / DK, c = e % DK;
        float x;
        if (p < 6) {
            const int a = (p < 1) ? 1 : (p < 3) ? 2 : 3;
            const int b = p - (a * (a - 1)) / 2;
            x = expf(REF[a * DK + c] - REF[b * DK + c]);
        } else {
            x = expf(REF[4 * DK + c] - REF[(p - 6) * DK + c]);
        }
        RT[p * DK + c] = x;
    }
    __syncthreads();
    // column-scaled K images: Kc_a[j] = k_j exp(ref_a - G_j), j < 16(a+1)
    {
        uint32_t img = P_KC;
        for (int a = 0; a < 4; ++a) {
            const int rows = 16 * (a + 1);
            for (int e = tid; e < rows * DK; e += PREP_THREADS) {
                const int j = e / DK, c = e % DK, b = j >> 4;
                float x = KF[j * DK + c];
                if (b < a) x *= RT[((a * (a - 1)) / 2 + b) * DK + c];
                st_bf16(sm + img, sw128_offset(j, c, rows), x);
            }
            img += rows * 256;
        }
    }
    fence_proxy_async();
    __syncthreads();
    if (tid == 0) {
        tc_fence_after();
        const uint32_t base = smem_u32(sm);
        uint32_t img = base + P_KC;
        for (int a = 0; a < 4; ++a) {
            const int rows = 16 * (a + 1);
            const uint32_t idesc = idesc_bf16(128, rows, false, false);
            const uint32_t dcol = 8 * a * (a + 1);
            for (int s = 0; s < DK / 16; ++s) {
                const uint32_t koff = ((s * 16) % 64) * 2;
                const uint64_t ad = sdesc_sw128(base + P_KRQR + (s >> 2) * 16384 + koff, 16, 1024);
                const uint64_t bd = sdesc_sw128(img + (s >> 2) * rows * 128 + koff, 16, 1024);
                umma_bf16(tmem + dcol, ad, bd, idesc, s > 0);
            }
            img += rows * 256;
        }
        umma_commit(&bar[0]);
    }
    // K*Gam_C/Gam as the MN-major [64 k-rows][128 m] image (overlaps the MMAs)
    for (int e = tid; e < C * DK; e += PREP_THREADS) {
        const int r = e / DK, c = e % DK;
        st_bf16(sm + P_KT, sw128_offset(r, c, 64), KF[r * DK + c] * RT[(6 + (r >> 4)) * DK + c]);
    }
    bool ok = mbar_wait(&bar[0], 0);
    tc_fence_after();

    // ---- (3) A and P from TMEM: warp a reads its own lane quarter (tile a)
    float *AS = reinterpret_cast<float *>(sm + P_AS);
    float *TS = reinterpret_cast<float *>(sm + P_TS);
    if (warp < 4) {
        const int a = warp;
        const bool isA = lane < 16;
        const int r = 16 * a + (lane & 15);
        const float br = BETA[r];
        const uint32_t dcol = 8 * a * (a + 1);
        for (int m = 0; m < a + 1; ++m) {
            float val[16];
            tmem_ld16(tmem + ((uint32_t)(32 * a) << 16) + dcol + 16 * m, val);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int j = 16 * m + i;
                if (isA) AS[r * 65 + j] = (j < r) ? br * val[i] : 0.f;
                else st_bf16(sm + P_P, sw128_offset(r, j, 64), (j <= r) ? val[i] : 0.f);
            }
        }
        for (int j = 16 * (a + 1); j < C; ++j) {
            if (isA) AS[r * 65 + j] = 0.f;
            else st_bf16(sm + P_P, sw128_offset(r, j, 64), 0.f);
        }
    }
    tc_fence_before();
    __syncthreads();

    // ---- (4) T = (I + A)^-1, blocked over 16x16 tiles, fp32
    if (warp < 4 && lane < 16) {  // diagonal blocks by forward substitution
        const int a = warp, j = lane;
        float tcol[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float s = (r == j) ? 1.f : 0.f;
#pragma unroll
            for (int m = 0; m < r; ++m) s -= AS[(16 * a + r) * 65 + 16 * a + m] * tcol[m];
            tcol[r] = s;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) TS[(16 * a + r) * 65 + 16 * a + j] = tcol[r];
    }
    __syncthreads();
    float *XS = reinterpret_cast<float *>(sm + P_XS);
    for (int d = 1; d < 4; ++d) {
        // blocks (a, a-d): X = sum_{m=a-d}^{a-1} A_{a,m} T_{m,a-d};  T_{a,a-d} = -T_aa X
        const int a = d + warp;
        if (warp < 4 - d) {
            const int b = a - d;
            float *X = XS + warp * 16 * 17;
            for (int e = lane; e < 256; e += 32) {
                const int i = e >> 4, jj = e & 15;
                float s = 0.f;
                for (int m = b; m < a; ++m)
                    for (int t = 0; t < 16; ++t)
                        s += AS[(16 * a + i) * 65 + 16 * m + t] * TS[(16 * m + t) * 65 + 16 * b + jj];
                X[i * 17 + jj] = s;
            }
            __syncwarp();
            for (int e = lane; e < 256; e += 32) {
                const int i = e >> 4, jj = e & 15;
                float s = 0.f;
                for (int t = 0; t <= i; ++t) s += TS[(16 * a + i) * 65 + 16 * a + t] * X[t * 17 + jj];
                TS[(16 * a + i) * 65 + 16 * b + jj] = -s;
            }
        }
        __syncthreads();
    }
    // T diag(b) as the K-major [64][64] A image (upper part zero)
    for (int e = tid; e < C * C; e += PREP_THREADS) {
        const int r = e / C, j = e % C;
        const float x = (j <= r) ? TS[r * 65 + j] * BETA[j] : 0.f;
        st_bf16(sm + P_TB, sw128_offset(r, j, 64), x);
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    // ---- (5) [W | Ut] = T diag(b) [K*Gam | V]  (M = 128: rows 64.. are ignored)
    if (tid == 0) {
        tc_fence_after();
        const uint32_t base = smem_u32(sm);
        const uint32_t idesc = idesc_bf16(128, 256, false, true);
        for (int s = 0; s < C / 16; ++s) {
            const uint64_t ad = sdesc_sw128(base + P_TB + s * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(base + P_KGV + s * 2048, 64 * 128, 1024);
            umma_bf16(tmem, ad, bd, idesc, s > 0);
        }
        umma_commit(&bar[1]);
        // the finished images can leave while the MMA runs
        bulk_s2g(rec + REC_KT, sm + P_KT, 16384);
        bulk_s2g(rec + REC_P, sm + P_P, 8192);
        bulk_commit();
    }
    ok = mbar_wait(&bar[1], 0) && ok;
    tc_fence_after();

    // ---- (6) W rows -> WQ image rows 0..63 (warps 0-1); Ut -> fp32 staging (warps 4-5)
    float *UST = reinterpret_cast<float *>(sm + P_UST);
    if (warp == 0 || warp == 1 || warp == 4 || warp == 5) {
        const int quarter = warp & 3;            // TMEM lane quarter 0 or 1
        const int r = 32 * quarter + lane;       // row of W / Ut
        const bool isW = warp < 4;
        for (int cb = 0; cb < 4; ++cb) {
            float val[32];
            tmem_ld32(tmem + ((uint32_t)(32 * quarter) << 16) + (isW ? 0 : 128) + 32 * cb, val);
            tmem_ld_wait();
            if (isW) {
#pragma unroll
                for (int i8 = 0; i8 < 4; ++i8) {
                    __align__(16) __nv_bfloat16 pk[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) pk[i] = __float2bfloat16_rn(val[8 * i8 + i]);
                    *reinterpret_cast<uint4 *>(sm + P_WQ + sw128_offset(r, 32 * cb + 8 * i8, 128)) =
                        *reinterpret_cast<uint4 *>(pk);
                }
            } else {
                float4 *dst = reinterpret_cast<float4 *>(UST + (cb * 64 + r) * 32);
#pragma unroll
                for (int i4 = 0; i4 < 8; ++i4)
                    dst[i4] = make_float4(val[4 * i4], val[4 * i4 + 1], val[4 * i4 + 2], val[4 * i4 + 3]);
            }
        }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        bulk_s2g(rec + REC_WQ, sm + P_WQ, 32768);
        bulk_s2g(rec + REC_U, sm + P_UST, 32768);
        bulk_commit();
        bulk_wait_all();
    }
    if (!ok && tid == 0) report(st, KDA_ERR_TIMEOUT, slot, 10);
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// ---------------------------------------------------------------- chain kernel
constexpr int CHAIN_THREADS = 128;
constexpr uint32_t B_WQ = 0, B_KT = 32768, B_ZP = 49152, B_U = 65536, B_G = 73728;
constexpr uint32_t BUF_BYTES = 74752;
constexpr uint32_t C_S = 2 * BUF_BYTES;              // S image K-major [32][128]
constexpr uint32_t C_UI = C_S + 8192;                // U image K-major [32][64]
constexpr uint32_t C_BAR = C_UI + 4096;              // full[2], m1, m2, TMEM slot
constexpr uint32_t C_SMEM = C_BAR + 64 + 1024;
constexpr uint32_t LOAD_BYTES = 32768 + 16384 + 8192 + 8192 + 512;
static_assert(B_G + 512 <= BUF_BYTES && BUF_BYTES % 1024 == 0, "chain buffer layout");
static_assert(C_SMEM <= 232448, "chain kernel exceeds 227 KB of shared memory");

__device__ __forceinline__ void chain_load(uint8_t *buf, const uint8_t *rec, int blk,
                                           uint64_t *full) {
    mbar_arrive_expect_tx(full, LOAD_BYTES);
    bulk_g2s(buf + B_WQ, rec + REC_WQ, 32768, full);
    bulk_g2s(buf + B_KT, rec + REC_KT, 16384, full);
    bulk_g2s(buf + B_ZP + 8192, rec + REC_P, 8192, full);
    bulk_g2s(buf + B_U, rec + REC_U + blk * 8192, 8192, full);
    bulk_g2s(buf + B_G, rec + REC_G, 512, full);
}

// largest n in [0, N) with chunk_off[n] <= slot (the owner of a used slot)
__device__ __forceinline__ int slot_owner(const int32_t *chunk_off, int N, int32_t slot) {
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (chunk_off[mid] <= slot) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Persistent over work items (sequence, head, 32-column block) of the sequences
// that own chunks in the slot window [slot0, slot1); each item walks its
// chunks in order, carrying its block of S in registers (fp32) and as the bf16
// B operand image in shared memory.
__global__ void __launch_bounds__(CHAIN_THREADS, 1)
chain_kernel(const int32_t *__restrict__ cu, const int32_t *__restrict__ chunk_off, int N, int H,
             int32_t slot0, int32_t slot1, const uint8_t *__restrict__ records,
             float *__restrict__ state, __nv_bfloat16 *__restrict__ o, StatusWord *st) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int32_t used = min(slot1, chunk_off[N]);
    if (slot0 >= used) return;
    const int n_first = slot_owner(chunk_off, N, slot0);
    const int n_last = slot_owner(chunk_off, N, used - 1);
    const int items = (n_last - n_first + 1) * H * NBLK;
    if ((int)blockIdx.x >= items) return;

    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + C_BAR);  // full0, full1, m1, m2
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + C_BAR + 32);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C_BAR + 40);
    if (tid == 0) {
        for (int x = 0; x < 4; ++x) mbar_init(&bar[x], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    // zero rows 0..63 of both [0; P] operand images
    for (int e = tid; e < 2 * 512; e += CHAIN_THREADS) {
        uint8_t *b = sm + (e / 512) * BUF_BYTES + B_ZP;
        reinterpret_cast<uint4 *>(b)[e % 512] = make_uint4(0, 0, 0, 0);
    }
    if (warp == 0) {
        tmem_alloc(tslot, 64);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t D1 = tmem, D2 = tmem + 32;
    const uint32_t base = smem_u32(sm);
    const uint32_t id_kk = idesc_bf16(128, DVB, false, false);
    const uint32_t id_mk = idesc_bf16(128, DVB, true, false);
    const int i = tid;  // this thread's state row
    uint32_t gi = 0;    // chunks processed by this CTA (drives buffer and barrier parity)

    for (int item = blockIdx.x; item < items && !*abort_flag; item += gridDim.x) {
        const int blk = item % NBLK;
        const int h = (item / NBLK) % H;
        const int n = n_first + item / (NBLK * H);
        const int32_t c_begin = max(chunk_off[n], slot0);
        const int32_t c_end = min(chunk_off[n + 1], slot1);
        if (c_begin >= c_end) continue;
        const int64_t bos = cu[n];
        const int64_t eos = cu[n + 1];
        const int j0 = blk * DVB;
        float S[DVB];
        float *srow = state + (((int64_t)n * H + h) * DK + i) * DV + j0;
#pragma unroll
        for (int j4 = 0; j4 < DVB / 4; ++j4) {
            const float4 x = reinterpret_cast<const float4 *>(srow)[j4];
            S[4 * j4] = x.x; S[4 * j4 + 1] = x.y; S[4 * j4 + 2] = x.z; S[4 * j4 + 3] = x.w;
        }
#pragma unroll
        for (int j = 0; j < DVB; ++j) st_bf16(sm + C_S, sw128_offset(j, i, 32), S[j]);
        fence_proxy_async();
        __syncthreads();
        if (tid == 0)
            chain_load(sm + (gi & 1) * BUF_BYTES,
                       records + ((size_t)(c_begin - slot0) * H + h) * REC_BYTES, blk,
                       &bar[gi & 1]);

        for (int32_t cs = c_begin; cs < c_end; ++cs, ++gi) {
            const uint32_t b = gi & 1;
            uint8_t *buf = sm + b * BUF_BYTES;
            const uint32_t bufa = base + b * BUF_BYTES;
            bool ok = mbar_wait(&bar[b], (gi >> 1) & 1);
            if (tid == 0 && ok) {
                // D1 = [W; Q*Gam] S
                tc_fence_after();
                for (int s = 0; s < DK / 16; ++s) {
                    const uint32_t koff = ((s * 16) % 64) * 2;
                    const uint64_t ad = sdesc_sw128(bufa + B_WQ + (s >> 2) * 16384 + koff, 16, 1024);
                    const uint64_t bd = sdesc_sw128(base + C_S + (s >> 2) * 4096 + koff, 16, 1024);
                    umma_bf16(D1, ad, bd, id_kk, s > 0);
                }
                umma_commit(&bar[2]);
                // prefetch the next chunk into the other buffer (its last reader finished)
                if (cs + 1 < c_end)
                    chain_load(sm + (b ^ 1) * BUF_BYTES,
                               records + ((size_t)(cs + 1 - slot0) * H + h) * REC_BYTES, blk,
                               &bar[b ^ 1]);
            }
            ok = ok && mbar_wait(&bar[2], gi & 1);
            tc_fence_after();
            // U = Ut - W S  (rows 0..63 live in TMEM lane quarters 0 and 1)
            if (warp < 2 && ok) {
                const int r = tid;
                float acc[32];
                tmem_ld32(D1 + ((uint32_t)(32 * warp) << 16), acc);
                tmem_ld_wait();
                const float4 *ut = reinterpret_cast<const float4 *>(buf + B_U + r * 128);
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const float4 u4 = ut[j4];
                    st_bf16(sm + C_UI, sw128_offset(4 * j4 + 0, r, 32), u4.x - acc[4 * j4 + 0]);
                    st_bf16(sm + C_UI, sw128_offset(4 * j4 + 1, r, 32), u4.y - acc[4 * j4 + 1]);
                    st_bf16(sm + C_UI, sw128_offset(4 * j4 + 2, r, 32), u4.z - acc[4 * j4 + 2]);
                    st_bf16(sm + C_UI, sw128_offset(4 * j4 + 3, r, 32), u4.w - acc[4 * j4 + 3]);
                }
            }
            if (!ok) *abort_flag = 1;
            fence_proxy_async();
            tc_fence_before();
            __syncthreads();
            if (*abort_flag) break;
            if (tid == 0) {
                tc_fence_after();
                for (int s = 0; s < C / 16; ++s) {
                    // D2 = (K*Gam_C/Gam)^T U ;  D1 += [0; P] U
                    const uint64_t bd = sdesc_sw128(base + C_UI + s * 32, 16, 1024);
                    const uint64_t akt = sdesc_sw128(bufa + B_KT + s * 2048, 64 * 128, 1024);
                    umma_bf16(D2, akt, bd, id_mk, s > 0);
                    const uint64_t azp = sdesc_sw128(bufa + B_ZP + s * 32, 16, 1024);
                    umma_bf16(D1, azp, bd, id_kk, 1);
                }
                umma_commit(&bar[3]);
            }
            ok = mbar_wait(&bar[3], gi & 1);
            tc_fence_after();
            if (ok) {
                // S <- Diag(Gam_C) S + D2 (row i = tid)
                const float gc = reinterpret_cast<const float *>(buf + B_G)[i];
                float acc[32];
                tmem_ld32(D2 + ((uint32_t)(32 * warp) << 16), acc);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < DVB; ++j) {
                    S[j] = gc * S[j] + acc[j];
                    st_bf16(sm + C_S, sw128_offset(j, i, 32), S[j]);
                }
                if (warp >= 2) {
                    // O rows live in TMEM lane quarters 2 and 3 of D1
                    const int r = tid - 64;
                    const int64_t t = bos + (int64_t)(cs - chunk_off[n]) * C + r;
                    float oacc[32];
                    tmem_ld32(D1 + ((uint32_t)(32 * warp) << 16), oacc);
                    tmem_ld_wait();
                    if (t < eos) {
                        uint4 *dst = reinterpret_cast<uint4 *>(o + (t * H + h) * (int64_t)DV + j0);
#pragma unroll
                        for (int i8 = 0; i8 < 4; ++i8) {
                            __align__(16) __nv_bfloat16 pk[8];
#pragma unroll
                            for (int x = 0; x < 8; ++x) pk[x] = __float2bfloat16_rn(oacc[8 * i8 + x]);
                            dst[i8] = *reinterpret_cast<uint4 *>(pk);
                        }
                    }
                }
            } else {
                *abort_flag = 1;
            }
            fence_proxy_async();
            tc_fence_before();
            __syncthreads();
            if (*abort_flag) break;
        }
        if (*abort_flag) {
            if (tid == 0) report(st, KDA_ERR_TIMEOUT, ((int64_t)n * H + h) * NBLK + blk, 11);
        } else {
#pragma unroll
            for (int j4 = 0; j4 < DVB / 4; ++j4)
                reinterpret_cast<float4 *>(srow)[j4] =
                    make_float4(S[4 * j4], S[4 * j4 + 1], S[4 * j4 + 2], S[4 * j4 + 3]);
        }
        __syncthreads();
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 64);
    }
}

// Copy (or zero) the initial state into the running-state buffer.
__global__ void state_init_kernel(const float *__restrict__ h0, float *__restrict__ S,
                                  int64_t n4) {
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n4;
         e += (int64_t)gridDim.x * blockDim.x)
        reinterpret_cast<float4 *>(S)[e] =
            h0 ? reinterpret_cast<const float4 *>(h0)[e] : make_float4(0.f, 0.f, 0.f, 0.f);
}

}  // namespace tc

size_t tc_record_bytes() { return tc::REC_BYTES; }

cudaError_t launch_chunk_tc(const void *q, const void *k, const void *v, const void *z,
                            const void *beta, const float *A_log, const int32_t *cu,
                            const int32_t *chunk_off, int N, int64_t slots, int H,
                            const float *h0, float *S_run, void *o, uint8_t *records,
                            int64_t window, StatusWord *st, cudaStream_t s, EventRec *rec) {
    using namespace tc;
    cudaError_t e = cudaFuncSetAttribute(prep_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)P_SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C_SMEM);
    if (e != cudaSuccess) return e;
    int dev = 0, sm_count = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t n4 = (int64_t)N * H * DK * DV / 4;
    if (h0 != S_run) {
        const int64_t blocks = std::min<int64_t>((n4 + 255) / 256, (int64_t)sm_count * 16);
        state_init_kernel<<<(unsigned)blocks, 256, 0, s>>>(h0, S_run, n4);
        if (rec) rec->mark();
    }
    for (int64_t s0 = 0; s0 < slots; s0 += window) {
        const int64_t s1 = std::min(slots, s0 + window);
        dim3 pg((unsigned)(s1 - s0), (unsigned)H);
        prep_kernel<<<pg, PREP_THREADS, P_SMEM, s>>>(
            (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v,
            (const __nv_bfloat16 *)z, (const __nv_bfloat16 *)beta, A_log, cu, chunk_off, N, H,
            (int32_t)s0, records, st);
        if (rec) rec->mark();
        // items of a window: at most min(N, window) sequences x H x NBLK
        const int64_t items = std::min<int64_t>(N, s1 - s0) * H * NBLK;
        const int64_t grid = std::min<int64_t>(items, sm_count);
        chain_kernel<<<(unsigned)grid, CHAIN_THREADS, C_SMEM, s>>>(
            cu, chunk_off, N, H, (int32_t)s0, (int32_t)s1, records, S_run, (__nv_bfloat16 *)o,
            st);
        if (rec) rec->mark();
    }
    return cudaGetLastError();
}

}  // namespace kda
