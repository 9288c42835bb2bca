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
// a parallel "prep" kernel over all (chunk, head) pairs; a "chain" kernel then walks
// the chunks in order, one CTA per (sequence, head, 32-column block of dv) or, when
// there are many sequences, per (sequence, head) with all 128 columns.
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
//   Ut  bf16 [4 column blocks][64][32], 16-byte piece j of row r holds columns 8 (j ^ ((r / 2) % 4))
//   GC  fp32 [128] Gam_C
#include <cuda.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "kda_common.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace tc {

using namespace sm100;

constexpr int C = 64;            // chunk length (four 16-token tiles)
constexpr int DK = 128, DV = 128;

// record layout (bytes)
constexpr uint32_t REC_WQ = 0;
constexpr uint32_t REC_KT = 32768;
constexpr uint32_t REC_P = 49152;
constexpr uint32_t REC_U = 57344;
constexpr uint32_t REC_G = 73728;
constexpr uint32_t REC_BYTES = 74240;
constexpr uint32_t UT_BLK = 64 * 32 * 2;   // bytes of one 32-column block of Ut (bf16)

// Byte offset of the 16-byte piece j (columns 8j .. 8j+7) of row r in a 32-column block of
// Ut: rows are 64 bytes, pieces swizzled so that 8 consecutive rows reading the same piece
// hit 8 distinct 16-byte bank groups.
__host__ __device__ __forceinline__ uint32_t ut_piece(uint32_t r, uint32_t j) {
    return r * 64 + ((j ^ ((r >> 1) & 3)) << 4);
}

// ---------------------------------------------------------------- prep kernel
constexpr int PREP_THREADS = 256;
constexpr int PREP_WARPS = PREP_THREADS / 32;
constexpr int NU = 32 / PREP_WARPS;     // 8-channel units per thread in the element-wise passes
constexpr int SOLVE_W = (384 + 128 + PREP_THREADS - 1) / PREP_THREADS;   // solve tasks per thread
static_assert(PREP_WARPS == 8 && NU == 4, "row-wise passes map 8 warps x 32 lanes onto 16 rows x 16 chunks, one unit per tile");
constexpr int LDA = 68;                 // row stride (floats) of the fp32 A and T tiles
// Shared-memory map of the prep kernel (offsets from a 1024-aligned base).  Two
// CTAs fit on one SM.  Regions are reused once the A/P products have completed.
constexpr uint32_t P_BAR = 0;           // 2 mbarriers, TMEM slot
constexpr uint32_t P_TOT = 1024;        // fp32 [4][128]  per-tile sums of g
constexpr uint32_t P_ER = 5632;         // fp32 [4][128]  exp(ref_a)
constexpr uint32_t P_RT = 7680;         // fp32 [6][128]  exp(ref_a' - ref_a), a < a'
constexpr uint32_t P_KTF = 10752;       // fp32 [4][128]  exp(G_C - ref_a)
constexpr uint32_t P_BETA = 12800;      // fp32 [64]
constexpr uint32_t P_KRQR = 13312;      // K-major [128][128] row-scaled K/Q: tile a -> rows 32a..32a+31
constexpr uint32_t P_G = 13312;         // (before pass B) fp32 G scratch [64][GLD]
constexpr int GLD = 132;                //   padded row stride: conflict-free row and column access
constexpr uint32_t P_KC = 46080;        // column-scaled K images, a = 0..3, stacked: [160][128]
constexpr uint32_t KC_ROWS = 160;       //   image a = rows 8a(a+1) .. 8a(a+1) + 16(a+1) - 1
constexpr uint32_t P_KGV = 13312;       // (after the A/P products) MN-major [64][256]: K*Gam | V
constexpr uint32_t P_AS = 46080;        //   fp32 A [64][68]
constexpr uint32_t P_TS = 63488;        //   fp32 T [64][68]
constexpr uint32_t P_XS = 80896;        //   fp32 [4][16][XLD] N^2 / N^3 blocks
constexpr int XLD = 20;                 //   padded row stride: conflict-free row-wise reads
constexpr uint32_t P_ZT = 47104;        // (until pass A) z tile, TMA, [2][64][128 B] swizzled
constexpr uint32_t P_KT = 63488;        // (until the table pass) k tile, likewise
constexpr uint32_t P_QT = 79872;        // (until the table pass) q tile, likewise
constexpr uint32_t P_PST = 1024;        // (A/P epilogue) P staging, K-major [64][64], over the dead tables
constexpr uint32_t P_WST = 13312;       // (epilogue) W staging, K-major [2][64][128 B]
constexpr uint32_t P_UST = 46080;       // (epilogue) Ut staging, bf16 [4][64][32]
// The A operand of step E, [T diag(b), 0; 0, T diag(b)] (K-major, 128 rows, K = 2C), in two
// 64-column halves: half 0 over the dead fp32 A, half 1 at the end
constexpr uint32_t P_A0 = P_AS;         //   half 0: T diag(b) in rows 0..63, zeros below
constexpr uint32_t P_TB = 87040;        //   half 1: zeros in rows 0..63, T diag(b) below
constexpr uint32_t P_END = 103424;
constexpr uint32_t P_SMEM = P_END + 1024;
static_assert(P_KC + 4096 + 8192 + 12288 + 16384 <= P_TB, "column-scaled K images overflow");
static_assert(P_KGV + 32768 <= P_AS && P_AS + 64 * LDA * 4 <= P_TS, "prep smem reuse overlaps");
static_assert(P_TS + 64 * LDA * 4 <= P_XS && P_XS + 4 * 16 * XLD * 4 <= P_TB, "solve scratch");
static_assert(P_G + 64 * GLD * 4 <= P_TB, "G scratch overlaps the T diag(b) image");
static_assert(P_ZT >= P_G + 64 * GLD * 4 && P_QT + 16384 <= P_END && P_ZT % 1024 == 0 &&
                  P_KT % 1024 == 0 && P_QT % 1024 == 0, "raw tiles");
static_assert(P_WST + 16384 <= P_AS && P_UST + 16384 <= P_TB &&
                  P_PST + 8192 <= P_BETA,
              "solve / epilogue staging overlaps live data");
static_assert(P_KRQR % 1024 == 0 && P_KC % 1024 == 0 && P_TB % 1024 == 0 && P_A0 % 1024 == 0 &&
                  P_A0 + 16384 <= P_TS, "image alignment");
static_assert(P_TB + 16384 == P_END && 2 * (P_SMEM + 1024) <= 233472, "two CTAs per SM");

__device__ __forceinline__ uint4 pack8(const float (&x)[8]) {
    uint4 r;
    __nv_bfloat162 *p = reinterpret_cast<__nv_bfloat162 *>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
    return r;
}
__device__ __forceinline__ void unpack8(const uint4 &u, float (&x)[8]) {
    const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(p[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void ld8(const float *src, float (&x)[8]) {
    const float4 a = reinterpret_cast<const float4 *>(src)[0];
    const float4 b = reinterpret_cast<const float4 *>(src)[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// The special-function unit's 2^x and 1/x (relative errors near 2^-22 and one ulp; both
// flush subnormals).  Measured on this part, a 64 x 128 gate tile costs about a third of
// the time with these as with the library's fast exponential and division.
constexpr float kLog2e = 1.4426950408889634f;
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// e^x as 2^(x log2 e); results below the normal range flush to 0
__device__ __forceinline__ float exp_decay(float x) { return ex2_approx(x * kLog2e); }

// Per-channel fp32 rows in shared memory (the gate scratch and the factor tables) keep
// channel c = 64 h + 8 j + 4 g + e (h, g in {0, 1}, j < 8, e < 4) at position
// 64 h + 32 g + 4 j + e, so that the 8 lanes reading channels 64 h + 8 j .. + 7 for
// j = 0..7 read two contiguous 128-byte lines.
__host__ __device__ __forceinline__ int chan_pos(int c) {
    return (c & 64) + ((c & 4) << 3) + ((c >> 1) & 28) + (c & 3);
}
__host__ __device__ __forceinline__ int pos_chan(int p) {
    return (p & 64) + ((p & 28) << 1) + ((p >> 3) & 4) + (p & 3);
}
// the 8 values of channels c .. c + 7 (c a multiple of 8) from a position-ordered row
__device__ __forceinline__ void ld8p(const float *row, int c, float (&x)[8]) {
    const int p = chan_pos(c);
    const float4 a = *reinterpret_cast<const float4 *>(row + p);
    const float4 b = *reinterpret_cast<const float4 *>(row + p + 32);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
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

// Window-relative chunk slot of the prep CTA at position y of the launch's slot
// dimension: the last slots first, so that the records of a window's first chunks, which
// the chain kernel reads first, are the most recently written (still in L2).
__device__ __forceinline__ int32_t prep_slot(int32_t y, int32_t nslots) { return nslots - 1 - y; }

// One CTA per (chunk slot, head).  The gate and the in-tile cumulative sums take one
// (tile, channel) column per thread; the row-wise element passes that follow give each
// thread 8 channels of one row in each 16-token tile.
__global__ void __launch_bounds__(PREP_THREADS, 2)
prep_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
            const __nv_bfloat16 *__restrict__ v, const __nv_bfloat16 *__restrict__ z,
            const __nv_bfloat16 *__restrict__ beta, const float *__restrict__ A_log,
            const int32_t *__restrict__ cu, const int32_t *__restrict__ chunk_off, int N,
            int64_t T_tot, int H, int32_t slot0, uint8_t *__restrict__ records, StatusWord *st,
            const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
            const __grid_constant__ CUtensorMap tmap_z, const __grid_constant__ CUtensorMap tmap_v) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + P_BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + P_BAR + 16);
    uint64_t *vbar = reinterpret_cast<uint64_t *>(sm + P_BAR + 32);   // the V tile's TMA
    uint64_t *zbar = reinterpret_cast<uint64_t *>(sm + P_BAR + 40);   // the z tile's TMA
    uint64_t *kqbar = reinterpret_cast<uint64_t *>(sm + P_BAR + 48);  // the k and q tiles' TMA
    uint64_t *drain = reinterpret_cast<uint64_t *>(sm + P_BAR + 56);  // products, after a timeout
    if (tid == 0) {
        // the barriers and the tensor maps, while the chunk's place is looked up
        tma_prefetch_map(&tmap_z);
        tma_prefetch_map(&tmap_k);
        tma_prefetch_map(&tmap_q);
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        mbar_init(vbar, 1);
        mbar_init(zbar, 1);
        mbar_init(kqbar, 1);
        mbar_init(drain, 1);
        fence_mbar_init();
    }
    // launch order is slot-major (all heads of a chunk slot, then the previous slot): the
    // CTAs of a wave read whole token rows of q, k, z and v
    const int32_t xs = prep_slot((int32_t)blockIdx.y, (int32_t)gridDim.y);
    const int32_t slot = slot0 + xs;
    const int h = blockIdx.x;
    int n = 0, L = 0;
    int64_t t0 = 0;
    if (N == 1) {
        // one sequence, tokens 0 .. T_tot - 1 (cu = [0, T_tot]; other cu values are
        // reported by the plan kernel): no lookup
        t0 = (int64_t)slot * C;
        if (t0 >= T_tot) return;
        L = (int)min((int64_t)C, T_tot - t0);
    } else if (!slot_chunk(cu, chunk_off, N, slot, n, t0, L)) {
        return;
    }
    uint8_t *rec = records + ((size_t)xs * H + h) * REC_BYTES;

    float *TOT = reinterpret_cast<float *>(sm + P_TOT);
    float *ER = reinterpret_cast<float *>(sm + P_ER);
    float *RT = reinterpret_cast<float *>(sm + P_RT);
    float *KTF = reinterpret_cast<float *>(sm + P_KTF);
    float *BETA = reinterpret_cast<float *>(sm + P_BETA);

    // The z, k and q tiles (64 tokens x 128 channels each) arrive by TMA in the 128-byte
    // swizzled layout, element (r, c) at sw128_offset(r, c, 64), in shared memory that the
    // element passes overwrite only after reading them.
    if (tid == 0) {
        mbar_arrive_expect_tx(zbar, 2 * 8192);
        tma_load_3d(sm + P_ZT, &tmap_z, 0, h, (int32_t)t0, zbar);
        tma_load_3d(sm + P_ZT + 8192, &tmap_z, 64, h, (int32_t)t0, zbar);
        mbar_arrive_expect_tx(kqbar, 4 * 8192);
        tma_load_3d(sm + P_KT, &tmap_k, 0, h, (int32_t)t0, kqbar);
        tma_load_3d(sm + P_KT + 8192, &tmap_k, 64, h, (int32_t)t0, kqbar);
        tma_load_3d(sm + P_QT, &tmap_q, 0, h, (int32_t)t0, kqbar);
        tma_load_3d(sm + P_QT + 8192, &tmap_q, 64, h, (int32_t)t0, kqbar);
    }

    // Row-wise element passes: thread (row-in-tile rl, 8-channel chunk c .. c + 7) owns
    // unit u = row 16u + rl of tile u, u = 0..3, so that every thread writes the same
    // number of column-scaled key images (tile a's rows appear in images a..3).  A warp
    // covers 4 rows x 64 channels (one 128-byte line of each row of a K half): its
    // 16-byte stores fill whole lines, in shared and in global memory.
    const int rl = 4 * (warp & 3) + (lane >> 3);
    const int c = 64 * (warp >> 2) + 8 * (lane & 7);
    const float alog = A_log[h];
    const float beta_v = tid < L ? __bfloat162float(beta[(t0 + min(tid, C - 1)) * H + h]) : 0.f;
    const float nl2e = -expf(alog) * kLog2e;   // -e^A log2(e)
    if (tid < C) BETA[tid] = beta_v;
    __syncthreads();                           // the barriers' initialisation is visible
    bool ok = mbar_wait(zbar, 0);
    // ---- (A) gate and in-tile inclusive cumsums, fused: thread (tile ta, position p) reads
    //          its column of z from the swizzled tile (a warp's 32 positions share one
    //          128-byte line of a row), forms each g, accumulates G down the tile's 16 rows
    //          in a register and writes it into the fp32 G scratch; the tile sum goes to
    //          TOT.  Every g lies in [g_min, 0] (NaN aside), so a tile's cumulative decay
    //          falls monotonically from 0 and stays in [-80, 0] iff its last value does; a
    //          NaN reaches the last value too.  Only a tile whose last value fails is
    //          searched for its first bad row.
    float *GS = reinterpret_cast<float *>(sm + P_G);
    {
        const int p = tid & (DK - 1);
        const int ch = pos_chan(p);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int ta = (tid >> 7) + 2 * half;
            float zz[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint32_t bits = *reinterpret_cast<const uint16_t *>(
                    sm + P_ZT + sw128_offset(16 * ta + i, ch, 64));
                zz[i] = __uint_as_float(bits << 16);
            }
            float run = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {   // g = -5 / (1 + 2^(-e^A log2(e) z)); NaN stays NaN
                const int r = 16 * ta + i;
                run += r < L ? kGMin * rcp_approx(1.0f + ex2_approx(nl2e * zz[i])) : 0.f;
                GS[r * GLD + p] = run;
            }
            TOT[ta * DK + p] = run;
            if (!decay_ok(run)) {
                int bad_row = -1;
                for (int i = 0; i < 16 && bad_row < 0; ++i)
                    if (16 * ta + i < L && !decay_ok(GS[(16 * ta + i) * GLD + p])) bad_row = 16 * ta + i;
                if (bad_row >= 0) report(st, KDA_ERR_DECAY_RANGE, (t0 + bad_row) * H + h, 5);
            }
        }
    }
    __syncthreads();
    // this thread's G values and k, q chunks, read before pass B reuses their space
    float trun[NU][8];
#pragma unroll
    for (int u = 0; u < NU; ++u) ld8p(GS + (16 * u + rl) * GLD, c, trun[u]);
    ok = mbar_wait(kqbar, 0) && ok;
    uint4 kraw[NU], qraw[NU];
#pragma unroll
    for (int u = 0; u < NU; ++u) {
        const int r = 16 * u + rl;
        const uint4 zero = make_uint4(0, 0, 0, 0);
        kraw[u] = r < L ? *reinterpret_cast<const uint4 *>(sm + P_KT + sw128_offset(r, c, 64)) : zero;
        qraw[u] = r < L ? *reinterpret_cast<const uint4 *>(sm + P_QT + sw128_offset(r, c, 64)) : zero;
    }
    if (warp == PREP_THREADS / 32 - 1) {   // idle during the table pass
        tmem_alloc(tslot, 256);
        tmem_relinquish();
        tc_fence_before();
    }
    // tile references, Gam_C and the per-(tile, channel) factor tables (thread = position)
    if (tid < DK) {
        const int c = tid;
        float run = 0.f, ref[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            ref[t] = run;
            ER[t * DK + c] = exp_decay(run);
            run += TOT[t * DK + c];
        }
        *reinterpret_cast<float *>(rec + REC_G + 4 * pos_chan(c)) = exp_decay(run);
#pragma unroll
        for (int t = 0; t < 4; ++t) KTF[t * DK + c] = exp_decay(run - ref[t]);
        int p = 0;
#pragma unroll
        for (int a2 = 1; a2 < 4; ++a2)
#pragma unroll
            for (int b = 0; b < a2; ++b, ++p) RT[p * DK + c] = exp_decay(ref[a2] - ref[b]);
    }
    __syncthreads();

    // ---- (B) decay-scaled operands, 16-byte stores: [Kr; Qr] (smem), column-scaled K
    //          images (smem), Q*Gam and K*Gam_C/Gam (straight into the record)
    uint4 kgam[NU];   // K*Gam chunks, written into the [K*Gam | V] image after the A/P products
#pragma unroll
    for (int u = 0; u < NU; ++u) {
        const int a = u, r = 16 * u + rl;   // this unit's tile and row of the chunk
        float kk[8], qq[8], er[8], ktf[8];
        unpack8(kraw[u], kk);
        unpack8(qraw[u], qq);
        ld8p(ER + a * DK, c, er);
        ld8p(KTF + a * DK, c, ktf);
        float kr[8], qr[8], kf[8], qg[8], kt[8], kg[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float F = exp_decay(trun[u][i]);    // exp(G_r - ref_a) in [e^-80, 1]
            const float iF = exp_decay(-trun[u][i]);  // exp(ref_a - G_r) in [1, e^80]
            const float Gm = er[i] * F;               // exp(G_r)
            kr[i] = kk[i] * F;
            qr[i] = qq[i] * F;
            kf[i] = kk[i] * iF;                       // k_r exp(ref_a - G_r)
            qg[i] = qq[i] * Gm;                       // q_r exp(G_r)
            kg[i] = kk[i] * Gm;                       // k_r exp(G_r)
            kt[i] = kf[i] * ktf[i];                   // k_r exp(G_C - G_r)
        }
        kgam[u] = pack8(kg);
        const uint32_t row = 32 * a + rl;
        *reinterpret_cast<uint4 *>(sm + P_KRQR + sw128_offset(row, c, 128)) = pack8(kr);
        *reinterpret_cast<uint4 *>(sm + P_KRQR + sw128_offset(row + 16, c, 128)) = pack8(qr);
        *reinterpret_cast<uint4 *>(rec + REC_WQ + sw128_offset(64 + r, c, 128)) = pack8(qg);
        *reinterpret_cast<uint4 *>(rec + REC_KT + sw128_offset(r, c, 64)) = pack8(kt);
        // image a2 >= a holds row r scaled by exp(ref_a2 - G_r) = kf * exp(ref_a2 - ref_a);
        // image a2 occupies rows 8 a2 (a2 + 1) .. of the stacked [160][128] B operand
        *reinterpret_cast<uint4 *>(sm + P_KC + sw128_offset(8 * a * (a + 1) + r, c, KC_ROWS)) = pack8(kf);
#pragma unroll
        for (int a2 = a + 1; a2 < 4; ++a2) {
            float rt[8], x[8];
            ld8p(RT + ((a2 * (a2 - 1)) / 2 + a) * DK, c, rt);
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = kf[i] * rt[i];
            *reinterpret_cast<uint4 *>(sm + P_KC + sw128_offset(8 * a2 * (a2 + 1) + r, c, KC_ROWS)) = pack8(x);
        }
    }
    fence_proxy_async();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t base = smem_u32(sm);

    // ---- A and P: D = [Kr; Qr] x [Kc_0; Kc_1; Kc_2; Kc_3]^T (M = 128, N = 160, K = dk);
    //      tile a's block D_a = [Kr; Qr] x Kc_a^T sits in columns 8 a (a + 1) .. + 16 (a + 1)
    if (warp == 0) {
        const uint32_t idesc = idesc_bf16(128, KC_ROWS, false, false);
        const uint64_t ad = sdesc_sw128(base + P_KRQR, 16, 1024);
        const uint64_t bd = sdesc_sw128(base + P_KC, 16, 1024);
        if (elect_one()) {
#pragma unroll
            for (int s = 0; s < DK / 16; ++s)
                umma_bf16(tmem, desc_add(ad, (s >> 2) * 16384 + (s & 3) * 32),
                          desc_add(bd, (s >> 2) * KC_ROWS * 128 + (s & 3) * 32), idesc, s > 0);
            umma_commit(&bar[0]);
        }
        __syncwarp();
    }
    // while the products run: the zero rows 0..63 of step E's operand half 1 (the q tile
    // that held this region has been read)
#pragma unroll
    for (int e = tid; e < 512; e += PREP_THREADS)
        *reinterpret_cast<uint4 *>(sm + P_TB + 16 * e) = make_uint4(0, 0, 0, 0);
    ok = mbar_wait(&bar[0], 0) && ok;
    tc_fence_after();
    // ---- (C) MN-major [K*Gam | V] image in the freed [Kr; Qr] region: the V half arrives
    //          by TMA (two 64-channel boxes of 64 tokens, 128-byte swizzle, which is the
    //          operand layout) and is not needed before step E; K*Gam from registers
    if (tid == 0) {
        mbar_arrive_expect_tx(vbar, 2 * 64 * 128);
        tma_load_3d(sm + P_KGV + 2 * 8192, &tmap_v, 0, h, (int32_t)t0, vbar);
        tma_load_3d(sm + P_KGV + 3 * 8192, &tmap_v, 64, h, (int32_t)t0, vbar);
    }
#pragma unroll
    for (int u = 0; u < NU; ++u)
        *reinterpret_cast<uint4 *>(sm + P_KGV + sw128_offset(16 * u + rl, c, 64)) = kgam[u];
    // A (fp32, smem) and P (bf16 image, straight into the record) from TMEM:
    // warp w reads its own lane quarter t = w & 3 (rows 32t.. of D_t: 16 Kr rows, then
    // 16 Qr rows), column blocks m = 2 (w >> 2) and 2 (w >> 2) + 1 of D_t
    float *AS = reinterpret_cast<float *>(sm + P_AS);
    float *TS = reinterpret_cast<float *>(sm + P_TS);
    if (warp < 8) {   // eight warps: lane quarter t, two of the four column blocks
        const int t = warp & 3, m0 = 2 * (warp >> 2);
        const bool isA = lane < 16;
        const int rr = 16 * t + (lane & 15);
        const float br = BETA[rr];
        const uint32_t src = tmem + ((uint32_t)(32 * t) << 16) + 8 * t * (t + 1) + 16 * m0;
        float val[2][16];
        if (m0 <= t) tmem_ld16(src, val[0]);
        if (m0 + 1 <= t) tmem_ld16(src + 16, val[1]);
        tmem_ld_wait();
#pragma unroll
        for (int mm = 0; mm < 2; ++mm) {
            const int m = m0 + mm;
            if (m > t) {
#pragma unroll
                for (int i = 0; i < 16; ++i) val[mm][i] = 0.f;
            }
            if (isA) {
#pragma unroll
                for (int i4 = 0; i4 < 4; ++i4) {
                    float x[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int j = 16 * m + 4 * i4 + i;
                        x[i] = (j < rr) ? br * val[mm][4 * i4 + i] : 0.f;
                    }
                    *reinterpret_cast<float4 *>(AS + rr * LDA + 16 * m + 4 * i4) =
                        make_float4(x[0], x[1], x[2], x[3]);
                }
            } else {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float x[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int j = 16 * m + 8 * half + i;
                        x[i] = (j <= rr) ? val[mm][8 * half + i] : 0.f;
                    }
                    *reinterpret_cast<uint4 *>(sm + P_PST + sw128_offset(rr, 16 * m + 8 * half, 64)) = pack8(x);
                }
            }
        }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {                       // P -> the record
        bulk_s2g(rec + REC_P, sm + P_PST, 8192);
        bulk_commit();
    }

    // ---- (D) T = (I + A)^-1 in fp32 over 16x16 blocks.  With D = blockdiag(I + A_aa) and
    //          N = D^-1 (A - blockdiag(A_aa)) (block strictly lower, so N^4 = 0):
    //          T = (I + N)^-1 D^-1 = (I - N + N^2 - N^3) D^-1.
    // T diag(b) (K-major [64][64] bf16) goes into both diagonal blocks of step E's operand:
    // zero blocks above the diagonal in the N^3 step, the other blocks in the last step of
    // the solve; the zero block under half 0's copy in the N^2 step.
    uint8_t *TBI0 = sm + P_A0;
    uint8_t *TBI1 = sm + P_TB + 8192;   // rows 64.. of half 1 share the swizzle of rows 0..
    // off-diagonal block pairs (a, b), a > b, numbered (1,0) (2,1) (3,2) (2,0) (3,1) (3,0).
    auto pair_a = [](int pr) { return pr < 3 ? pr + 1 : (pr == 3 ? 2 : 3); };
    auto pair_b = [](int pr) { return pr < 3 ? pr : (pr == 4 ? 1 : 0); };
    // One step for D^-1 and N: forward substitution down a 16-row column through
    // (I + A_aa), 64 columns e_j (giving T_aa = (I + A_aa)^-1 on the diagonal of TS) and
    // 96 columns of A_ab (giving N_ab = T_aa A_ab in block (a, b) of TS, which T itself
    // never uses: its off-diagonal blocks go straight to the T diag(b) image).
    if (tid < 64 + 96) {
        const bool diag = tid < 64;
        const int pr = diag ? 0 : (tid - 64) >> 4;
        const int a2 = diag ? tid >> 4 : pair_a(pr);
        const int b = diag ? a2 : pair_b(pr);
        const int j = tid & 15;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float s = diag ? ((i == j) ? 1.f : 0.f) : AS[(16 * a2 + i) * LDA + 16 * b + j];
#pragma unroll
            for (int m = 0; m < i; ++m) s -= AS[(16 * a2 + i) * LDA + 16 * a2 + m] * x[m];
            x[i] = s;   // T_aa: zero above the diagonal
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) TS[(16 * a2 + i) * LDA + 16 * b + j] = x[i];
    }
    __syncthreads();
    // The diagonal blocks of T hold explicit zeros above the diagonal, so every product
    // below runs over all 16 terms (fixed trip counts, fully unrolled).
    // dst += X[16 x 16 block rows] (row i) times Y (16 x 4 column group)
    auto acc16 = [](float4 &x, const float *xrow, const float *ycol, int ystride) {
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            const float xv = xrow[t];
            const float4 y = *reinterpret_cast<const float4 *>(ycol + t * ystride);
            x.x += xv * y.x; x.y += xv * y.y; x.z += xv * y.z; x.w += xv * y.w;
        }
    };
    float *XS = reinterpret_cast<float *>(sm + P_XS);   // [0] N2_20 [1] N2_31 [2] N2_30 [3] N3_30
    // N_ab row i, and the 4-column group jq of N_ab (row stride LDA), for pair numbers p
    auto nrow = [&](int p, int i) { return TS + (16 * pair_a(p) + i) * LDA + 16 * pair_b(p); };
    auto ncol = [&](int p, int jq) { return TS + (16 * pair_a(p)) * LDA + 16 * pair_b(p) + 4 * jq; };
    if (tid < 192) {
        // N^2 blocks: (2,0) = N21 N10, (3,1) = N32 N21, (3,0) = N31 N10 + N32 N20 (warp-uniform q)
        const int q = tid >> 6, i = (tid >> 2) & 15, jq = tid & 3;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (q == 0) {
            acc16(x, nrow(1, i), ncol(0, jq), LDA);
        } else if (q == 1) {
            acc16(x, nrow(2, i), ncol(1, jq), LDA);
        } else {
            acc16(x, nrow(4, i), ncol(0, jq), LDA);
            acc16(x, nrow(2, i), ncol(3, jq), LDA);
        }
        *reinterpret_cast<float4 *>(XS + q * 16 * XLD + i * XLD + 4 * jq) = x;
    } else {
        // rows 64..127 of half 0 (over the fp32 A, which the diagonal step has consumed)
#pragma unroll
        for (int e = tid - 192; e < 512; e += PREP_THREADS - 192)
            *reinterpret_cast<uint4 *>(sm + P_A0 + 8192 + 16 * e) = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    if (tid < 64) {  // N^3_30 = N32 N^2_20
        const int i = tid >> 2, jq = tid & 3;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        acc16(x, nrow(2, i), XS + 4 * jq, XLD);
        *reinterpret_cast<float4 *>(XS + 3 * 16 * XLD + i * XLD + 4 * jq) = x;
    } else if (tid < 64 + 192) {
        // zero blocks (a, b > a): (0,1) (0,2) (0,3) (1,2) (1,3) (2,3), 16 rows x two 16-byte chunks
        const int e = tid - 64, ub = e >> 5, rc = e & 31;
        const int ua = ub < 3 ? 0 : (ub < 5 ? 1 : 2);
        const int uc = ub < 3 ? ub + 1 : (ub < 5 ? ub - 1 : 3);
        const uint32_t off = sw128_offset(16 * ua + (rc >> 1), 16 * uc + 8 * (rc & 1), 64);
        *reinterpret_cast<uint4 *>(TBI0 + off) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4 *>(TBI1 + off) = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    // T_ab = M_ab T_bb with M = -N + N^2 - N^3 (blockwise), scaled by b and written to the image
#pragma unroll
    for (int w = 0; w < SOLVE_W; ++w) {
        const int task = tid + w * PREP_THREADS;
        if (task < 384) {
            const int pr = task >> 6, i = (task >> 2) & 15, jq = task & 3;
            const int a2 = pair_a(pr), b = pair_b(pr);
            const int n2 = pr == 3 ? 0 : pr == 4 ? 1 : pr == 5 ? 2 : -1;
            float mrow[16];
            const float *nr = nrow(pr, i);
#pragma unroll
            for (int t = 0; t < 16; ++t) mrow[t] = -nr[t];
            if (n2 >= 0) {
#pragma unroll
                for (int t = 0; t < 16; ++t) mrow[t] += XS[n2 * 16 * XLD + i * XLD + t];
            }
            if (n2 == 2) {
#pragma unroll
                for (int t = 0; t < 16; ++t) mrow[t] -= XS[3 * 16 * XLD + i * XLD + t];
            }
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            acc16(x, mrow, TS + (16 * b) * LDA + 16 * b + 4 * jq, LDA);
            const float4 bb = *reinterpret_cast<const float4 *>(BETA + 16 * b + 4 * jq);
            uint2 pk;
            *reinterpret_cast<__nv_bfloat162 *>(&pk.x) = __floats2bfloat162_rn(x.x * bb.x, x.y * bb.y);
            *reinterpret_cast<__nv_bfloat162 *>(&pk.y) = __floats2bfloat162_rn(x.z * bb.z, x.w * bb.w);
            const uint32_t off = sw128_offset(16 * a2 + i, 16 * b + 4 * jq, 64);
            *reinterpret_cast<uint2 *>(TBI0 + off) = pk;
            *reinterpret_cast<uint2 *>(TBI1 + off) = pk;
        } else if (task < 384 + 128) {
            // diagonal blocks: (block tb, row i, 8-column half) -> one 16-byte chunk
            const int e = task - 384, tb = e >> 5, i = (e >> 1) & 15, hf = e & 1;
            float x[8], bt[8], tt[8];
            ld8(TS + (16 * tb + i) * LDA + 16 * tb + 8 * hf, tt);
            ld8(BETA + 16 * tb + 8 * hf, bt);
#pragma unroll
            for (int c = 0; c < 8; ++c) x[c] = tt[c] * bt[c];
            const uint32_t off = sw128_offset(16 * tb + i, 16 * tb + 8 * hf, 64);
            *reinterpret_cast<uint4 *>(TBI0 + off) = pack8(x);
            *reinterpret_cast<uint4 *>(TBI1 + off) = pack8(x);
        }
    }
    if (L < C) {
        // a sequence's last chunk: the V box also holds the next rows of the tensor; zero the
        // rows past the sequence end so that nothing of another sequence reaches U~
        ok = mbar_wait(vbar, 0) && ok;
        for (int e = tid; e < (C - L) * 16; e += PREP_THREADS) {
            const int rr = L + (e >> 4), c8 = e & 15;
            *reinterpret_cast<uint4 *>(sm + P_KGV + sw128_offset(rr, 128 + 8 * c8, 64)) =
                make_uint4(0, 0, 0, 0);
        }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();

    // ---- (E) [W; Ut] = [T diag(b), 0; 0, T diag(b)] [K*Gam; V]  (M = 128, N = 128, K = 2C):
    //          W in TMEM lanes 0..63, Ut in lanes 64..127, so that all eight warps share
    //          the epilogue.  K steps 0..3 read K*Gam and operand half 0, steps 4..7 V and half 1.
    if (warp == 0) {
        ok = mbar_wait(vbar, 0) && ok;
        tc_fence_after();
        const uint32_t idesc = idesc_bf16(128, DK, false, true);
        const uint64_t a0 = sdesc_sw128(base + P_A0, 16, 1024);
        const uint64_t a1 = sdesc_sw128(base + P_TB, 16, 1024);
        const uint64_t bd = sdesc_sw128(base + P_KGV, 64 * 128, 1024);
        if (elect_one()) {
#pragma unroll
            for (int s = 0; s < 2 * C / 16; ++s)
                umma_bf16(tmem, desc_add(s < 4 ? a0 : a1, (s & 3) * 32),
                          desc_add(bd, (s >> 2) * 16384 + (s & 3) * 2048), idesc, s > 0);
            umma_commit(&bar[1]);
        }
        __syncwarp();
    }
    ok = mbar_wait(&bar[1], 0) && ok;
    tc_fence_after();

    // ---- (F) W (lanes 0..63; K-major, rows 0..63 of the record's WQ image) and Ut (lanes
    //          64..127, bf16) are staged in the freed shared memory and leave in three bulk
    //          copies.  Warp w takes lane quarter w & 3 and the 32-column blocks 2 (w >> 2) and
    //          2 (w >> 2) + 1, two 16-column TMEM loads in flight per wait; W's copies leave
    //          once its four warps have staged it, Ut's once its four have.
    uint8_t *WST = sm + P_WST;   // [2 K halves][64 rows][128 B]
    uint8_t *UST = sm + P_UST;   // [4 column blocks][64 rows][32] bf16, pieces swizzled
    {
        const int quarter = warp & 3;
        const bool isW = quarter < 2;
        const int rr = 32 * (quarter & 1) + lane;
        const uint32_t src = tmem + ((uint32_t)(32 * quarter) << 16);
#pragma unroll
        for (int t2 = 0; t2 < 2; ++t2) {
            const int cb = 2 * (warp >> 2) + t2;
            float lo[16], hi[16];
            tmem_ld16(src + 32 * cb, lo);
            tmem_ld16(src + 32 * cb + 16, hi);
            tmem_ld_wait();
            if (isW) {
#pragma unroll
                for (int i8 = 0; i8 < 4; ++i8) {
                    float x[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) x[i] = i8 < 2 ? lo[8 * i8 + i] : hi[8 * (i8 - 2) + i];
                    *reinterpret_cast<uint4 *>(WST + sw128_offset(rr, 32 * cb + 8 * i8, 64)) = pack8(x);
                }
            } else {
                // row rr of column block cb, bf16, pieces swizzled so that the chain
                // kernels' row-per-thread reads hit distinct banks
                uint8_t *dst = UST + cb * UT_BLK;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float x[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) x[i] = j < 2 ? lo[8 * j + i] : hi[8 * (j - 2) + i];
                    *reinterpret_cast<uint4 *>(dst + ut_piece(rr, j)) = pack8(x);
                }
            }
        }
        fence_proxy_async();
        if (isW) named_bar_sync(1, 128);   // the four W warps
        else named_bar_sync(2, 128);       // the four Ut warps
        if (tid == 0) {
            bulk_s2g(rec + REC_WQ, WST, 8192);                 // W, K half 0
            bulk_s2g(rec + REC_WQ + 16384, WST + 8192, 8192);  // W, K half 1
            bulk_commit();
        } else if (tid == 64) {
            bulk_s2g(rec + REC_U, UST, REC_G - REC_U);         // Ut
            bulk_commit();
        }
    }
    fence_proxy_async();
    tc_fence_before();
    if (!__syncthreads_and(ok)) {
        // an expired wait: every product this CTA issued and every tile load finishes
        // (each wait bounded again) before the tensor memory is released
        if (warp == 0) {
            tc_fence_after();
            if (elect_one()) umma_commit(drain);
            __syncwarp();
            mbar_wait(drain, 0);
        }
        if (tid == 0) {
            mbar_wait(zbar, 0);
            mbar_wait(kqbar, 0);
            mbar_wait(vbar, 0);
            report(st, KDA_ERR_TIMEOUT, slot, 10);
        }
        __syncthreads();
    }
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
    // the CTA may leave once its staging has been read (threads 0 and 64 issued the copies);
    // the writes complete with the kernel, before anything ordered after it reads the records
    if (tid == 0 || tid == 64) bulk_wait_read_all();
}

// ---------------------------------------------------------------- chain kernels
// Records of chunks this far ahead of the one being walked are pulled into L2.
constexpr int kPrefetchAhead = 3;
// largest n in [0, N) with chunk_off[n] <= slot (the owner of a used slot)
__device__ __forceinline__ int slot_owner(const int32_t *chunk_off, int N, int32_t slot) {
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (chunk_off[mid] <= slot) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Segment-parallel passes (the pages' KDA context parallelism, P2 "Infrastructure and
// Training/Inference Mechanics", applied to segments of one window instead of ranks):
// mode 1 walks segment 0 of every sequence from its state and, at the same time, every
// later segment from [I | 0] with [0 | Ut], which yields that segment's affine map
// S_end = M S_start + B (M evolves like S with V = 0); a scan composes the maps into each
// later segment's start state; mode 2 then walks the later segments from those states.
// Mode 0 is the plain walk.
struct SegArgs {
    int mode;       // 0 plain, 1 first pass, 2 second pass
    int segs;       // segments per sequence and window (>= 2 in modes 1 and 2)
    float *start;   // [N][H][segs][DK][DV]      start state of segment k >= 1
    float *maps;    // [N][H][segs][DK][DK + DV] [M | B] of segment k >= 1
};
// Chunks [b, e) of segment k when a sequence's L chunks of the window, starting at c0,
// are cut into s_eff = min(segs, L) near-equal segments.
__device__ __forceinline__ void seg_range(int32_t c0, int32_t L, int segs, int k, int32_t &b,
                                          int32_t &e, int &s_eff) {
    s_eff = min(segs, (int)L);
    b = c0 + (int32_t)(((int64_t)k * L) / s_eff);
    e = c0 + (int32_t)(((int64_t)(k + 1) * L) / s_eff);
}

// Test hook: a bounded wait limit and a record load to leave out (so that the wait for it
// expires), given per launch of a chain kernel.
struct Fault {
    uint64_t wait_ns;    // limit of every bounded wait of the chain kernel
    int skip_cta;        // CTA whose first record load is not issued (-1: none)
};

// ------------------------------------------------ chain kernel, 32-column blocks
// The latency-bound shape: one CTA per (sequence, head, 32-column block of dv).  The
// N = 32 products finish sooner than N = 128 ones, so a lone long sequence walks its
// chunks fastest with four narrow CTAs per head.
namespace c32 {

constexpr int DVB = 32;          // value columns per CTA
constexpr int DK_ROWS = DK;      // threads of the scan kernel (one per state row)
constexpr int NBLK = DV / DVB;
// warps 0-7: row 32 (w % 4) + lane of S, columns 16 (w / 4) .. + 15 of the block; warp 8
// issues [x; P] U
constexpr int CHAIN_THREADS = 288;
constexpr int ROW_WARPS = 8;
constexpr int HCOLS = DVB / 2;   // columns a thread holds
// a record buffer mirrors the record's first 57344 bytes (WQ, KT, P), then this CTA's U
// block and Gam_C
constexpr uint32_t B_WQ = 0, B_KT = 32768, B_P = 49152, B_U = 57344, B_G = B_U + UT_BLK;
constexpr uint32_t BUF_BYTES = (B_G + 512 + 1023) / 1024 * 1024;
constexpr uint32_t C_S = 2 * BUF_BYTES;              // S image, MN-major 64B-swizzle [128 k][32 n]
constexpr uint32_t C_UI = C_S + 8192;                // U images of even / odd chunks, MN-major 64B-swizzle [64 k][32 n]
constexpr uint32_t C_BAR = C_UI + 8192;              // full[2], m1, m2, m3, drain, d2i; TMEM slot, flag
constexpr uint32_t C_SMEM = C_BAR + 128 + 1024;
constexpr uint32_t LOAD_BYTES = REC_U + UT_BLK + 512;
static_assert(B_G + 512 <= BUF_BYTES && BUF_BYTES % 1024 == 0 && B_P == REC_P && B_KT == REC_KT,
              "chain buffer layout");
static_assert(C_S % 1024 == 0 && C_UI % 1024 == 0, "operand image alignment");
static_assert(C_SMEM <= 232448, "chain kernel exceeds 227 KB of shared memory");

__device__ __forceinline__ void chain_load(uint8_t *buf, const uint8_t *rec, int blk,
                                           uint64_t *full) {
    mbar_arrive_expect_tx(full, LOAD_BYTES);
    bulk_g2s(buf, rec, REC_U, full);   // WQ, KT, P in one copy
    bulk_g2s(buf + B_U, rec + REC_U + blk * UT_BLK, UT_BLK, full);
    bulk_g2s(buf + B_G, rec + REC_G, 512, full);
}

// 16 fp32 values -> the two 16-byte chunks of row r, columns c0 .. c0 + 15, of a
// 64B-swizzled MN-major image
__device__ __forceinline__ void store_half_sw64(uint8_t *img, int r, int c0,
                                                const float (&x)[HCOLS]) {
#pragma unroll
    for (int c8 = 0; c8 < 2; ++c8) {
        float y[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) y[i] = x[8 * c8 + i];
        *reinterpret_cast<uint4 *>(img + sw64_offset(r, c0 + 8 * c8, 1)) = pack8(y);
    }
}

// Persistent over work items (sequence, head, 32-column block) of the sequences
// that own chunks in the slot window [slot0, slot1); each item walks its chunks
// in order, carrying its block of S in registers (fp32; thread (i, half) holds 16
// columns of row i) and as
// the bf16 B operand image.  Per chunk, on the critical path:
//   D1 = [W; Q*Gam] S  ->  U = Ut - D1[0:64]  ->  D2 = (K*Gam_C/Gam)^T U,
//   D1 += [x; P] U     ->  S = Diag(Gam_C) S + D2.
// D1 is double-buffered in TMEM so that the output rows of chunk c (D1[64:128])
// are stored by the warps of lane quarters 2-3 while those of quarters 0-1 form U of
// chunk c+1.  In the segment-parallel
// modes (SegArgs) an item is one segment of a sequence's chunks in the window, and a map
// item walks a 32-column block of [M | B] from [I | 0] (Ut = 0 for the M columns)
// without storing outputs.
__global__ void __launch_bounds__(CHAIN_THREADS, 1)
chain_kernel(const int32_t *__restrict__ cu, const int32_t *__restrict__ chunk_off, int N, int H,
             int32_t slot0, int32_t slot1, const uint8_t *__restrict__ records,
             const float *h0, float *__restrict__ state, __nv_bfloat16 *__restrict__ o,
             StatusWord *st, SegArgs sa, Fault flt) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t used = min(slot1, chunk_off[N]);
    if (slot0 >= used) return;
    const int n_first = slot_owner(chunk_off, N, slot0);
    const int n_last = slot_owner(chunk_off, N, used - 1);
    // items per (sequence, head): the column blocks, and in mode 1 the 2 NBLK blocks of
    // [M | B] of every later segment, in mode 2 the blocks of every later segment
    const int ipp = sa.mode == 0 ? NBLK
                  : sa.mode == 1 ? NBLK + 2 * NBLK * (sa.segs - 1) : NBLK * (sa.segs - 1);
    const int items = (n_last - n_first + 1) * H * ipp;
    if ((int)blockIdx.x >= items) return;

    // full0, full1, m1 (D1), m2 (D2), m3 ([x; P] U), drain, d2i (D2 issued)
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + C_BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + C_BAR + 56);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C_BAR + 60);
    // record loads issued into / seen complete in buffers 0 and 1: kept in registers by
    // thread 64, which issues every load (shared-memory counters beside the barriers
    // measured 0.5 us a chunk slower)
    uint32_t iss0 = 0, iss1 = 0, don0 = 0, don1 = 0;
    const uint64_t lim = flt.wait_ns;
    if (tid == 0) {
        for (int x = 0; x < 5; ++x) mbar_init(&bar[x], 1);
        mbar_init(&bar[5], 2);   // one commit from each issuing warp (0 and 8)
        mbar_init(&bar[6], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, 128);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t D2 = tmem + 64;                     // D1 buffers at columns 0 and 32
    const int qr = warp & 3;                           // TMEM lane quarter of this warp
    const int jc = HCOLS * ((warp >> 2) & 1);          // first column of this thread's half
    const uint32_t lane_base = ((uint32_t)(32 * qr) << 16) + (uint32_t)jc;
    const uint32_t base = smem_u32(sm);
    const uint32_t id_km = idesc_bf16(128, DVB, false, true);   // A K-major, B MN-major
    const uint32_t id_mm = idesc_bf16(128, DVB, true, true);    // A MN-major, B MN-major
    const uint64_t bd_s = sdesc_sw64(base + C_S, 128 * 64, 512);    // S image, K step 0
    const uint64_t bd_u = sdesc_sw64(base + C_UI, 64 * 64, 512);    // U image 0, K step 0
    const int i = 32 * qr + lane;  // this thread's state row
    uint32_t gi = 0;    // chunks processed by this CTA (drives buffer and barrier parity)

    for (int item = blockIdx.x; item < items && !*abort_flag; item += gridDim.x) {
        const int r_it = item % ipp;
        const int h = (item / ipp) % H;
        const int n = n_first + item / (ipp * H);
        int blk = r_it, seg = 0;
        bool map = false, mpart = false;   // an [M | B] item, and of the M columns
        if (sa.mode == 1 && r_it >= NBLK) {
            const int x = r_it - NBLK;
            seg = 1 + x / (2 * NBLK);
            map = true;
            mpart = x % (2 * NBLK) < NBLK;
            blk = x % NBLK;
        } else if (sa.mode == 2) {
            seg = 1 + r_it / NBLK;
            blk = r_it % NBLK;
        }
        const int32_t cfirst = chunk_off[n];
        const int32_t w_begin = max(cfirst, slot0);
        int32_t c_begin = w_begin;
        int32_t c_end = min(chunk_off[n + 1], slot1);
        if (c_begin >= c_end) continue;
        int s_eff = 1;
        if (sa.mode != 0) {
            int32_t sb = 0, se = 0;
            seg_range(w_begin, c_end - w_begin, sa.segs, seg, sb, se, s_eff);
            if (seg >= s_eff) continue;
            c_begin = sb;
            c_end = se;
        }
        const int64_t bos = cu[n];
        const int64_t eos = cu[n + 1];
        const int j0 = blk * DVB;
        float S[HCOLS];
        const int64_t pairoff = (int64_t)n * H + h;
        const int64_t soff = (pairoff * DK + i) * DV + j0 + jc;
        float *srow = state + soff;
        // the sequence's first chunk starts from h0 (zeros when absent), later windows from
        // the running state, a later segment from its composed start state, a map from
        // the identity (M columns) or zeros (B columns)
        const float *s_in = map ? nullptr
                          : seg > 0 ? sa.start + ((pairoff * sa.segs + seg) * DK + i) * DV + j0 + jc
                          : w_begin == cfirst ? (h0 ? h0 + soff : nullptr) : srow;
        if (warp < ROW_WARPS) {
#pragma unroll
            for (int j4 = 0; j4 < HCOLS / 4; ++j4) {
                const float4 x = s_in ? reinterpret_cast<const float4 *>(s_in)[j4]
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
                S[4 * j4] = x.x; S[4 * j4 + 1] = x.y; S[4 * j4 + 2] = x.z; S[4 * j4 + 3] = x.w;
            }
            if (mpart) {
#pragma unroll
                for (int j = 0; j < HCOLS; ++j) S[j] = (i == j0 + jc + j) ? 1.f : 0.f;
            }
            store_half_sw64(sm + C_S, i, jc, S);
            fence_proxy_async();
        }
        __syncthreads();
        if (tid == 64 && !(item == (int)blockIdx.x && (int)blockIdx.x == flt.skip_cta)) {
            chain_load(sm + (gi & 1) * BUF_BYTES,
                       records + ((size_t)(c_begin - slot0) * H + h) * REC_BYTES, blk,
                       &bar[gi & 1]);
            iss0 += (gi & 1) == 0;
            iss1 += (gi & 1) == 1;
        }

        // output rows of chunk number `gprev` of this CTA, whose D1 buffer is gprev & 1
        // (the warps of lane quarters 2-3); waits for that chunk's [x; P] U product
        // (barrier m3)
        auto store_o = [&](int32_t cprev, uint32_t gprev) -> bool {
            const uint32_t pb = gprev & 1;
            if (!mbar_wait(&bar[4], gprev & 1, lim)) return false;
            tc_fence_after();
            const int r = i - 64;
            const int64_t t = bos + (int64_t)(cprev - cfirst) * C + r;
            float oacc[HCOLS];
            tmem_ld16(tmem + 32 * pb + lane_base, oacc);
            tmem_ld_wait();
            if (t < eos && !map) {
                uint4 *dst = reinterpret_cast<uint4 *>(o + (t * H + h) * (int64_t)DV + j0 + jc);
#pragma unroll
                for (int i8 = 0; i8 < 2; ++i8) {
                    float y[8];
#pragma unroll
                    for (int x = 0; x < 8; ++x) y[x] = oacc[8 * i8 + x];
                    dst[i8] = pack8(y);
                }
            }
            return true;
        };

        bool aborted = false;
        for (int32_t cs = c_begin; cs < c_end; ++cs, ++gi) {
            const uint32_t b = gi & 1;
            uint8_t *buf = sm + b * BUF_BYTES;
            const uint32_t bufa = base + b * BUF_BYTES;
            if (warp == ROW_WARPS) {
                // D1[b] += [x; P] U (outputs only), issued as soon as D2 has been: the
                // in-order tensor pipe runs it right behind D2, while S is updated and well
                // before the next D1.  This warp joins no per-chunk barrier.  [x; P] reads the
                // 64 rows in front of P (the tail of KT) as its first half; those rows of D1
                // hold W S, which the U epilogue has consumed by then.
                const bool ok4 = __all_sync(0xffffffffu, mbar_wait(&bar[6], gi & 1, lim));
                if (ok4) {
                    tc_fence_after();
                    const uint64_t azp = sdesc_sw128(bufa + B_P - 8192, 16, 1024);
                    if (elect_one()) {
#pragma unroll
                        for (int s = 0; s < C / 16; ++s)
                            umma_bf16(tmem + 32 * b, desc_add(azp, s * 32),
                                      desc_add(bd_u, b * 4096 + s * 1024), id_km, 1);
                        umma_commit(&bar[4]);
                    }
                    __syncwarp();
                } else {
                    if (lane == 0) *abort_flag = 1;
                    aborted = true;
                    break;
                }
                continue;
            }
            bool ok = mbar_wait(&bar[b], (gi >> 1) & 1, lim);
            don0 += ok && b == 0;
            don1 += ok && b == 1;
            if (warp == 0 && __all_sync(0xffffffffu, ok)) {
                // D1[b] = [W; Q*Gam] S
                tc_fence_after();
                const uint64_t ad = sdesc_sw128(bufa + B_WQ, 16, 1024);
                if (elect_one()) {
#pragma unroll
                    for (int s = 0; s < DK / 16; ++s)
                        umma_bf16(tmem + 32 * b, desc_add(ad, (s >> 2) * 16384 + (s & 3) * 32),
                                  desc_add(bd_s, s * 1024), id_km, s > 0);
                    umma_commit(&bar[2]);
                }
                __syncwarp();
            }
            if (qr < 2) {
                // U = Ut - W S  (rows 0..63 live in TMEM lane quarters 0 and 1).  While the
                // product runs: this thread's row of Ut into registers.  The U image of this
                // parity was last read two chunks ago, by products the outputs of the
                // previous chunk waited for.
                const int r = i;
                uint4 ur[2];
#pragma unroll
                for (int j = 0; j < 2; ++j)   // the M columns of a map see Ut = 0
                    ur[j] = mpart ? make_uint4(0, 0, 0, 0)
                                  : *reinterpret_cast<const uint4 *>(buf + B_U + ut_piece(r, jc / 8 + j));
                ok = ok && mbar_wait(&bar[2], gi & 1, lim);
                tc_fence_after();
                if (ok) {
                    float acc[HCOLS];
                    tmem_ld16(tmem + 32 * b + lane_base, acc);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        float u[8];
                        unpack8(ur[j], u);
#pragma unroll
                        for (int x = 0; x < 8; ++x) acc[8 * j + x] = u[x] - acc[8 * j + x];
                    }
                    store_half_sw64(sm + C_UI + b * 4096, r, jc, acc);
                }
                fence_proxy_async();
                tc_fence_before();
                // the U image is complete: D2 = (K*Gam_C/Gam)^T U (only the warps of lane
                // quarters 0-1 wait here)
                ok = bar_and(1, 128, ok);
                if (warp == 0 && ok) {
                    tc_fence_after();
                    const uint64_t akt = sdesc_sw128(bufa + B_KT, 64 * 128, 1024);
                    if (elect_one()) {
#pragma unroll
                        for (int s = 0; s < C / 16; ++s)
                            umma_bf16(D2, desc_add(akt, s * 2048), desc_add(bd_u, b * 4096 + s * 1024),
                                      id_mm, s > 0);
                        umma_commit(&bar[3]);
                        mbar_arrive(&bar[6]);   // the issuing warp may queue [x; P] U behind D2
                    }
                    __syncwarp();
                }
            } else {
                // previous chunk's outputs, off the critical path; its [x; P] U product was
                // the last reader of the other buffer, which then takes the next chunk
                if (cs > c_begin) ok = store_o(cs - 1, gi - 1) && ok;
                if (tid == 64 && ok && cs + 1 < c_end) {
                    chain_load(sm + (b ^ 1) * BUF_BYTES,
                               records + ((size_t)(cs + 1 - slot0) * H + h) * REC_BYTES, blk,
                               &bar[b ^ 1]);
                    iss0 += b == 1;
                    iss1 += b == 0;
                }
                // and the parts of the record kPrefetchAhead chunks on that this CTA reads
                if (tid == 64 && cs + kPrefetchAhead < c_end) {
                    const uint8_t *r2 = records + ((size_t)(cs + kPrefetchAhead - slot0) * H + h) * REC_BYTES;
                    bulk_prefetch_l2(r2 + REC_WQ, REC_U - REC_WQ);
                    bulk_prefetch_l2(r2 + REC_U + blk * UT_BLK, UT_BLK);
                    bulk_prefetch_l2(r2 + REC_G, REC_BYTES - REC_G);
                }
            }
            // S <- Diag(Gam_C) S + D2 (row i = tid)
            const float gc = reinterpret_cast<const float *>(buf + B_G)[i];
            ok = mbar_wait(&bar[3], gi & 1, lim) && ok;
            tc_fence_after();
            if (ok) {
                float acc[HCOLS];
                tmem_ld16(D2 + lane_base, acc);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < HCOLS; ++j) S[j] = gc * S[j] + acc[j];
                store_half_sw64(sm + C_S, i, jc, S);
            }
            fence_proxy_async();
            tc_fence_before();
            // the row warps: S image complete and this chunk's record reads done; the AND
            // makes the decision to stop the same for all of them
            if (!bar_and(2, 32 * ROW_WARPS, ok && !*abort_flag)) {
                if (tid == 0) *abort_flag = 1;
                aborted = true;
                break;
            }
        }
        if (aborted) {
            if (tid == 0) report(st, KDA_ERR_TIMEOUT, ((int64_t)n * H + h) * NBLK + blk, 11);
        } else {
            tc_fence_after();
            bool ok_o = true;
            if (qr >= 2 && warp < ROW_WARPS) ok_o = store_o(c_end - 1, gi - 1);   // the item's last chunk
            if (!ok_o) *abort_flag = 1;
            // where the walk's end state goes: the running state, segment 1's start (first
            // pass, segment 0), the map, or nowhere (second pass, all but the last segment:
            // their ends are the next segments' composed starts)
            float *dst = srow;
            if (map)
                dst = sa.maps + ((pairoff * sa.segs + seg) * DK + i) * (DK + DV) + (mpart ? 0 : DK) + j0 + jc;
            else if (sa.mode == 1 && s_eff > 1)
                dst = sa.start + ((pairoff * sa.segs + 1) * DK + i) * DV + j0 + jc;
            else if (sa.mode == 2 && seg != s_eff - 1)
                dst = nullptr;
            if (warp < ROW_WARPS && dst) {
#pragma unroll
                for (int j4 = 0; j4 < HCOLS / 4; ++j4)
                    reinterpret_cast<float4 *>(dst)[j4] =
                        make_float4(S[4 * j4], S[4 * j4 + 1], S[4 * j4 + 2], S[4 * j4 + 3]);
            }
        }
        tc_fence_before();
        __syncthreads();
    }
    __syncthreads();
    if (*abort_flag) {
        // an expired wait: the products both issuing warps committed and the record loads
        // still in flight finish (each wait bounded again) before the tensor memory is
        // released and the CTA leaves
        if (warp == 0 || warp == ROW_WARPS) {
            tc_fence_after();
            if (elect_one()) umma_commit(&bar[5]);
            __syncwarp();
        }
        if (warp == 0) mbar_wait(&bar[5], 0, lim);
        if (tid == 64) {   // a buffer holds at most one load no wait has seen: its last one
            if (iss0 > don0) mbar_wait(&bar[0], (iss0 - 1) & 1, lim);
            if (iss1 > don1) mbar_wait(&bar[1], (iss1 - 1) & 1, lim);
        }
        __syncthreads();
    }
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 128);
    }
}


// The scan of the segment-parallel schedule: for every (sequence, head, 32-column block)
// of the window, start(k + 1) = M_k start(k) + B_k for k = 1 .. s_eff - 2 (start(1) is
// segment 0's end state from the first pass).  fp32; thread i = row i.
__global__ void __launch_bounds__(DK)
seg_scan_kernel(const int32_t *__restrict__ cu, const int32_t *__restrict__ chunk_off, int N,
                int H, int32_t slot0, int32_t slot1, SegArgs sa) {
    __shared__ __align__(16) float Ss[DK][DVB];
    const int i = threadIdx.x;
    const int32_t used = min(slot1, chunk_off[N]);
    if (slot0 >= used) return;
    const int n_first = slot_owner(chunk_off, N, slot0);
    const int n_last = slot_owner(chunk_off, N, used - 1);
    const int items = (n_last - n_first + 1) * H * NBLK;
    for (int item = blockIdx.x; item < items; item += gridDim.x) {
        const int blk = item % NBLK;
        const int h = (item / NBLK) % H;
        const int n = n_first + item / (NBLK * H);
        const int32_t c_begin = max(chunk_off[n], slot0);
        const int32_t c_end = min(chunk_off[n + 1], slot1);
        const int L = c_end - c_begin;
        const int s_eff = min(sa.segs, L);
        if (s_eff < 3) continue;
        const int j0 = blk * DVB;
        const int64_t pairoff = (int64_t)n * H + h;
        float S[DVB];
        {
            const float4 *src = reinterpret_cast<const float4 *>(
                sa.start + ((pairoff * sa.segs + 1) * DK + i) * DV + j0);
#pragma unroll
            for (int j4 = 0; j4 < DVB / 4; ++j4) {
                const float4 x = src[j4];
                S[4 * j4] = x.x; S[4 * j4 + 1] = x.y; S[4 * j4 + 2] = x.z; S[4 * j4 + 3] = x.w;
            }
        }
        for (int k = 1; k + 1 < s_eff; ++k) {
            __syncthreads();   // the previous step's reads of Ss are done
#pragma unroll
            for (int j = 0; j < DVB; ++j) Ss[i][j] = S[j];
            __syncthreads();
            const float *mrow = sa.maps + ((pairoff * sa.segs + k) * DK + i) * (DK + DV);
            float acc[DVB];
#pragma unroll
            for (int j = 0; j < DVB; ++j) acc[j] = mrow[DK + j0 + j];
            for (int m4 = 0; m4 < DK / 4; ++m4) {
                const float4 mv = reinterpret_cast<const float4 *>(mrow)[m4];
                const float mm[4] = {mv.x, mv.y, mv.z, mv.w};
#pragma unroll
                for (int t = 0; t < 4; ++t) {
#pragma unroll
                    for (int j = 0; j < DVB; ++j) acc[j] += mm[t] * Ss[4 * m4 + t][j];
                }
            }
            float4 *dst = reinterpret_cast<float4 *>(
                sa.start + ((pairoff * sa.segs + k + 1) * DK + i) * DV + j0);
#pragma unroll
            for (int j4 = 0; j4 < DVB / 4; ++j4) {
                dst[j4] = make_float4(acc[4 * j4], acc[4 * j4 + 1], acc[4 * j4 + 2], acc[4 * j4 + 3]);
                S[4 * j4] = acc[4 * j4]; S[4 * j4 + 1] = acc[4 * j4 + 1];
                S[4 * j4 + 2] = acc[4 * j4 + 2]; S[4 * j4 + 3] = acc[4 * j4 + 3];
            }
        }
    }
}

}  // namespace c32

// ----------------------------------------------- chain kernel, all 128 columns
namespace c128 {

// One CTA per work item (sequence, head) owns all dv = 128 columns of S: the
// products below are M = 128, N = 128, which cost the tensor core about as much
// per instruction as N = 32, so one CTA does the work four narrower ones would.
constexpr int CHAIN_THREADS = 512;
constexpr uint32_t C_S = 0;                          // S image, MN-major SW128 [128 k][128 n]
constexpr uint32_t C_UI = 32768;                     // U image, MN-major SW128 [64 k][128 n]
constexpr uint32_t C_BUF0 = 49152;                   // record buffer 0 (REC_BYTES)
constexpr uint32_t C_BAR = C_BUF0 + REC_BYTES;       // full[2], m1, m2, m3, drain; TMEM slot, flags
constexpr uint32_t C_BUF1 = (C_BAR + 72 + 1023) / 1024 * 1024;   // record buffer 1
constexpr uint32_t C_SMEM = C_BUF1 + REC_BYTES + 1024;
static_assert(C_BAR + 72 <= C_BUF1 && C_BUF1 % 1024 == 0 && C_BUF0 % 1024 == 0,
              "chain buffer layout");
static_assert(REC_P % 1024 == 0 && REC_KT % 1024 == 0 && REC_U % 1024 == 0, "record alignment");
static_assert(C_SMEM <= 232448, "chain kernel exceeds 227 KB of shared memory");

__device__ __forceinline__ void chain_load(uint8_t *buf, const uint8_t *rec, uint64_t *full) {
    mbar_arrive_expect_tx(full, REC_BYTES);
    bulk_g2s(buf, rec, REC_BYTES, full);   // the whole record, one copy
}

// 32 fp32 values -> four 16-byte chunks of row r, columns j0.., of a 128B-swizzled
// MN-major image whose 64-column groups are `rows` * 128 bytes apart
__device__ __forceinline__ void store_row_sw128(uint8_t *img, int r, int j0, uint32_t rows,
                                                const float (&x)[32]) {
#pragma unroll
    for (int c8 = 0; c8 < 4; ++c8) {
        float y[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) y[i] = x[8 * c8 + i];
        *reinterpret_cast<uint4 *>(img + sw128_offset(r, j0 + 8 * c8, rows)) = pack8(y);
    }
}

// Persistent over work items (sequence, head) of the sequences that own chunks in
// the slot window [slot0, slot1); each item walks its chunks in order.  Warp w
// holds lane quarter q = w & 3 and column block cb = w >> 2: thread (row 32q +
// lane, columns 32cb..32cb+31) keeps its piece of S in registers (fp32), and S is
// mirrored as the bf16 B operand image.  Per chunk, on the critical path:
//   D1 = [W; Q*Gam] S  ->  U = Ut - D1[0:64]  ->  D2 = (K*Gam_C/Gam)^T U,
//   D1 += [x; P] U     ->  S = Diag(Gam_C) S + D2.
// ([x; P] reads the 64 rows in front of P as its first half; those rows of D1
// hold W S, which has been consumed by then.)  D1 is double-buffered in TMEM so
// that the output rows of chunk c (D1[64:128], lane quarters 2-3) are stored while
// lane quarters 0-1 form U of chunk c+1.
__global__ void __launch_bounds__(CHAIN_THREADS, 1)
chain_kernel(const int32_t *__restrict__ cu, const int32_t *__restrict__ chunk_off, int N, int H,
             int32_t slot0, int32_t slot1, const uint8_t *__restrict__ records,
             const float *h0, float *__restrict__ state, __nv_bfloat16 *__restrict__ o,
             StatusWord *st, Fault flt) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t used = min(slot1, chunk_off[N]);
    if (slot0 >= used) return;
    const int n_first = slot_owner(chunk_off, N, slot0);
    const int n_last = slot_owner(chunk_off, N, used - 1);
    const int items = (n_last - n_first + 1) * H;
    if ((int)blockIdx.x >= items) return;

    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + C_BAR);  // full0, full1, m1, m2, m3, drain
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + C_BAR + 48);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C_BAR + 52);
    // record loads issued into / seen complete in buffers 0 and 1: kept in registers by
    // thread 64, which issues every load (shared-memory counters beside the barriers
    // measured 0.5 us a chunk slower)
    uint32_t iss0 = 0, iss1 = 0, don0 = 0, don1 = 0;
    const uint64_t lim = flt.wait_ns;
    if (tid == 0) {
        for (int x = 0; x < 6; ++x) mbar_init(&bar[x], 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tslot, 512);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t D2 = tmem + 256;                    // D1 buffers at columns 0 and 128
    const int q4 = warp & 3, cb = warp >> 2;
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    const uint32_t base = smem_u32(sm);
    const uint32_t id_km = idesc_bf16(128, DV, false, true);   // A K-major, B MN-major
    const uint32_t id_mm = idesc_bf16(128, DV, true, true);    // A MN-major, B MN-major
    const uint64_t bd_s = sdesc_sw128(base + C_S, DK * 128, 1024);   // S image, K step 0
    const uint64_t bd_u = sdesc_sw128(base + C_UI, C * 128, 1024);   // U image, K step 0
    const int i = 32 * q4 + lane;   // this thread's state row
    const int j0 = 32 * cb;         // and first column
    uint32_t gi = 0;                // chunks processed by this CTA (drives buffer and barrier parity)
    auto buf_off = [](uint32_t b) { return b ? C_BUF1 : C_BUF0; };

    for (int item = blockIdx.x; item < items && !*abort_flag; item += gridDim.x) {
        const int h = item % H;
        const int n = n_first + item / H;
        const int32_t cfirst = chunk_off[n];
        const int32_t c_begin = max(cfirst, slot0);
        const int32_t c_end = min(chunk_off[n + 1], slot1);
        if (c_begin >= c_end) continue;
        const int64_t bos = cu[n];
        const int64_t eos = cu[n + 1];
        float S[32];
        const int64_t soff = (((int64_t)n * H + h) * DK + i) * DV + j0;
        float *srow = state + soff;
        // the sequence's first chunk starts from h0 (zeros when absent), later windows from
        // the running state
        const float *s_in = c_begin == cfirst ? (h0 ? h0 + soff : nullptr) : srow;
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
            const float4 x = s_in ? reinterpret_cast<const float4 *>(s_in)[j4]
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
            S[4 * j4] = x.x; S[4 * j4 + 1] = x.y; S[4 * j4 + 2] = x.z; S[4 * j4 + 3] = x.w;
        }
        store_row_sw128(sm + C_S, i, j0, DK, S);
        fence_proxy_async();
        __syncthreads();
        if (tid == 64 && !(item == (int)blockIdx.x && (int)blockIdx.x == flt.skip_cta)) {
            chain_load(sm + buf_off(gi & 1),
                       records + ((size_t)(c_begin - slot0) * H + h) * REC_BYTES, &bar[gi & 1]);
            iss0 += (gi & 1) == 0;
            iss1 += (gi & 1) == 1;
        }

        // output rows of chunk number `gprev` of this CTA, whose D1 buffer is gprev & 1
        // (lane quarters 2-3); waits for that chunk's [x; P] U product (barrier m3)
        auto store_o = [&](int32_t cprev, uint32_t gprev) -> bool {
            const uint32_t pb = gprev & 1;
            if (!mbar_wait(&bar[4], gprev & 1, lim)) return false;
            tc_fence_after();
            const int r = i - 64;
            const int64_t t = bos + (int64_t)(cprev - cfirst) * C + r;
            float oacc[32];
            tmem_ld32(tmem + 128 * pb + lane_base + j0, oacc);
            tmem_ld_wait();
            if (t < eos) {
                uint4 *dst = reinterpret_cast<uint4 *>(o + (t * H + h) * (int64_t)DV + j0);
#pragma unroll
                for (int i8 = 0; i8 < 4; ++i8) {
                    float y[8];
#pragma unroll
                    for (int x = 0; x < 8; ++x) y[x] = oacc[8 * i8 + x];
                    dst[i8] = pack8(y);
                }
            }
            return true;
        };

        for (int32_t cs = c_begin; cs < c_end; ++cs, ++gi) {
            const uint32_t b = gi & 1;
            uint8_t *buf = sm + buf_off(b);
            const uint32_t bufa = base + buf_off(b);
            bool ok = mbar_wait(&bar[b], (gi >> 1) & 1, lim);
            don0 += ok && b == 0;
            don1 += ok && b == 1;
            if (warp == 0 && __all_sync(0xffffffffu, ok)) {
                // D1[b] = [W; Q*Gam] S
                tc_fence_after();
                const uint64_t ad = sdesc_sw128(bufa + REC_WQ, 16, 1024);
                if (elect_one()) {
#pragma unroll
                    for (int s = 0; s < DK / 16; ++s)
                        umma_bf16(tmem + 128 * b, desc_add(ad, (s >> 2) * 16384 + (s & 3) * 32),
                                  desc_add(bd_s, s * 2048), id_km, s > 0);
                    umma_commit(&bar[2]);
                }
                __syncwarp();
            }
            if (q4 < 2) {
                // U = Ut - W S  (rows 0..63 live in TMEM lane quarters 0 and 1)
                ok = ok && mbar_wait(&bar[2], gi & 1, lim);
                tc_fence_after();
                if (ok) {
                    const int r = i;
                    float acc[32];
                    tmem_ld32(tmem + 128 * b + lane_base + j0, acc);
                    tmem_ld_wait();
                    const uint8_t *ut = buf + REC_U + cb * UT_BLK;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        float u[8];
                        unpack8(*reinterpret_cast<const uint4 *>(ut + ut_piece(r, j)), u);
#pragma unroll
                        for (int x = 0; x < 8; ++x) acc[8 * j + x] = u[x] - acc[8 * j + x];
                    }
                    store_row_sw128(sm + C_UI, r, j0, C, acc);
                }
            } else {
                // previous chunk's outputs, off the critical path; its [x; P] U product was
                // the last reader of the other buffer, which then takes the next chunk
                if (cs > c_begin) ok = store_o(cs - 1, gi - 1) && ok;
                if (tid == 64 && ok && cs + 1 < c_end) {
                    chain_load(sm + buf_off(b ^ 1),
                               records + ((size_t)(cs + 1 - slot0) * H + h) * REC_BYTES,
                               &bar[b ^ 1]);
                    iss0 += b == 1;
                    iss1 += b == 0;
                }
                // and the record kPrefetchAhead chunks on
                if (tid == 64 && cs + kPrefetchAhead < c_end)
                    bulk_prefetch_l2(records + ((size_t)(cs + kPrefetchAhead - slot0) * H + h) * REC_BYTES,
                                     REC_BYTES);
            }
            if (!ok) *abort_flag = 1;
            fence_proxy_async();
            tc_fence_before();
            __syncthreads();
            if (*abort_flag) break;
            if (warp == 0) {
                tc_fence_after();
                // D2 = (K*Gam_C/Gam)^T U  (on the recurrence) ...
                const uint64_t akt = sdesc_sw128(bufa + REC_KT, C * 128, 1024);
                const uint64_t azp = sdesc_sw128(bufa + REC_P - 8192, 16, 1024);
                if (elect_one()) {
#pragma unroll
                    for (int s = 0; s < C / 16; ++s)
                        umma_bf16(D2, desc_add(akt, s * 2048), desc_add(bd_u, s * 2048), id_mm, s > 0);
                    umma_commit(&bar[3]);
                    // ... then D1[b] += [x; P] U (outputs only), which runs while S is updated
#pragma unroll
                    for (int s = 0; s < C / 16; ++s)
                        umma_bf16(tmem + 128 * b, desc_add(azp, s * 32), desc_add(bd_u, s * 2048), id_km, 1);
                    umma_commit(&bar[4]);
                }
                __syncwarp();
            }
            ok = mbar_wait(&bar[3], gi & 1, lim);
            tc_fence_after();
            if (ok) {
                // S <- Diag(Gam_C) S + D2 (row i, columns j0..)
                const float gc = reinterpret_cast<const float *>(buf + REC_G)[i];
                float acc[32];
                tmem_ld32(D2 + lane_base + j0, acc);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) S[j] = gc * S[j] + acc[j];
                store_row_sw128(sm + C_S, i, j0, DK, S);
            } else {
                *abort_flag = 1;
            }
            fence_proxy_async();
            tc_fence_before();
            __syncthreads();
            if (*abort_flag) break;
        }
        if (*abort_flag) {
            if (tid == 0) report(st, KDA_ERR_TIMEOUT, (int64_t)n * H + h, 11);
        } else {
            tc_fence_after();
            bool ok_o = true;
            if (q4 >= 2) ok_o = store_o(c_end - 1, gi - 1);   // the item's last chunk
            if (!ok_o) *abort_flag = 1;
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4)
                reinterpret_cast<float4 *>(srow)[j4] =
                    make_float4(S[4 * j4], S[4 * j4 + 1], S[4 * j4 + 2], S[4 * j4 + 3]);
        }
        tc_fence_before();
        __syncthreads();
    }
    __syncthreads();
    if (*abort_flag) {
        // an expired wait: the issued products and the record loads still in flight finish
        // (each wait bounded again) before the tensor memory is released
        if (warp == 0) {
            tc_fence_after();
            if (elect_one()) umma_commit(&bar[5]);
            __syncwarp();
            mbar_wait(&bar[5], 0, lim);
        }
        if (tid == 64) {   // a buffer holds at most one load no wait has seen: its last one
            if (iss0 > don0) mbar_wait(&bar[0], (iss0 - 1) & 1, lim);
            if (iss1 > don1) mbar_wait(&bar[1], (iss1 - 1) & 1, lim);
        }
        __syncthreads();
    }
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace c128

}  // namespace tc

size_t tc_record_bytes() { return tc::REC_BYTES; }

namespace {

// Streams and events of the double-buffered schedule, created once per device and
// kept for the life of the process.  Two low-priority streams take the prep
// kernels of even and odd windows, one high-priority stream the chain kernels; the
// block scheduler then hands freed SMs to a waiting chain CTA first.
struct Pipe {
    bool ready = false;
    cudaStream_t prep[2] = {nullptr, nullptr};
    cudaStream_t chain = nullptr;
    cudaEvent_t start = nullptr, end = nullptr;
    cudaEvent_t prep_done[2] = {nullptr, nullptr}, chain_done[2] = {nullptr, nullptr};
};
constexpr int kMaxDevices = 64;
std::mutex g_pipe_mutex;     // held while a call enqueues its schedule
Pipe g_pipe[kMaxDevices];

cudaError_t pipe_setup(int dev, Pipe *&out) {
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    Pipe &P = g_pipe[dev];
    out = &P;
    if (P.ready) return cudaSuccess;
    int least = 0, greatest = 0;
    cudaError_t e = cudaDeviceGetStreamPriorityRange(&least, &greatest);
    for (int i = 0; i < 2 && e == cudaSuccess; ++i)
        e = cudaStreamCreateWithPriority(&P.prep[i], cudaStreamNonBlocking, least);
    if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&P.chain, cudaStreamNonBlocking, greatest);
    cudaEvent_t *evs[6] = {&P.start, &P.end, &P.prep_done[0], &P.prep_done[1],
                           &P.chain_done[0], &P.chain_done[1]};
    for (int i = 0; i < 6 && e == cudaSuccess; ++i)
        e = cudaEventCreateWithFlags(evs[i], cudaEventDisableTiming);
    if (e == cudaSuccess) P.ready = true;
    return e;
}

// cuTensorMapEncodeTiled, reached through the runtime's entry-point query (the library
// links no driver library)
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

}  // namespace

// Tensor map of a [T_tot, H, 128] bf16 tensor read in boxes of 64 tokens x 1 head x 64
// channels with the 128-byte swizzle (the MN-major operand layout of the prep kernel).
static cudaError_t tmap_thd(CUtensorMap *m, const void *x, int64_t T_tot, int H) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)T_tot};
    const cuuint64_t strides[2] = {128 * 2, (cuuint64_t)H * 128 * 2};
    const cuuint32_t box[3] = {64, 1, 64};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(x), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {

// The four tensor maps of one call, cached by (device, pointers, T_tot, H): encoding them
// costs host time that matters for short calls (a few tokens per sequence).  A map holds
// only the pointer and the shape, so a hit is exact.
struct TmapEntry {
    int dev;
    const void *ptr[4];
    int64_t T;
    int H;
    CUtensorMap m[4];
};
constexpr int kTmapCache = 16;
std::mutex g_tmap_mutex;
TmapEntry g_tmap[kTmapCache];
int g_tmap_used = 0, g_tmap_next = 0;

cudaError_t tensor_maps(int dev, const void *const (&ptr)[4], int64_t T, int H,
                        CUtensorMap (&out)[4]) {
    std::lock_guard<std::mutex> lock(g_tmap_mutex);
    for (int e = 0; e < g_tmap_used; ++e) {
        const TmapEntry &x = g_tmap[e];
        if (x.dev == dev && x.T == T && x.H == H && x.ptr[0] == ptr[0] && x.ptr[1] == ptr[1] &&
            x.ptr[2] == ptr[2] && x.ptr[3] == ptr[3]) {
            memcpy(out, x.m, sizeof out);
            return cudaSuccess;
        }
    }
    TmapEntry x{};
    x.dev = dev;
    x.T = T;
    x.H = H;
    for (int j = 0; j < 4; ++j) {
        x.ptr[j] = ptr[j];
        const cudaError_t e = tmap_thd(&x.m[j], ptr[j], T, H);
        if (e != cudaSuccess) return e;
    }
    g_tmap[g_tmap_next] = x;
    g_tmap_next = (g_tmap_next + 1) % kTmapCache;
    if (g_tmap_used < kTmapCache) ++g_tmap_used;
    memcpy(out, x.m, sizeof out);
    return cudaSuccess;
}

// Kernel attributes (dynamic shared memory above 48 KB), set once per device.
std::mutex g_attr_mutex;
bool g_attr_set[kMaxDevices] = {};

cudaError_t kernel_attributes(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_attr_mutex);
    if (g_attr_set[dev]) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(tc::prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)tc::P_SMEM);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tc::c32::chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)tc::c32::C_SMEM);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tc::c128::chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)tc::c128::C_SMEM);
    if (e == cudaSuccess) g_attr_set[dev] = true;
    return e;
}

// Test hook (kda_test_chain_fault): the next call's chain launches get this wait limit and
// leave out the first record load of one CTA.
constexpr uint64_t kWaitNs = 1000000000ull;   // the default limit of a bounded wait: 1 s
std::mutex g_fault_mutex;
tc::Fault g_fault_next = {kWaitNs, -1};
bool g_fault_armed = false;

tc::Fault take_fault() {
    std::lock_guard<std::mutex> lock(g_fault_mutex);
    const tc::Fault f = g_fault_armed ? g_fault_next : tc::Fault{kWaitNs, -1};
    g_fault_armed = false;
    return f;
}

}  // namespace

// Records: nbuf (1 or 2) buffers of `window` chunk slots x H records each.  With one
// buffer the windows run prep, chain, prep, chain ... on `s`.  With two, prep of
// window w + 1 runs beside chain of window w (see Pipe); the call's work is still
// ordered after everything enqueued on `s` before it and before everything after it.
cudaError_t launch_chunk_tc(const void *q, const void *k, const void *v, const void *z,
                            const void *beta, const float *A_log, const int32_t *cu,
                            const int32_t *chunk_off, int N, int64_t T_tot, int64_t slots, int H,
                            const float *h0, float *S_run, void *o, uint8_t *records,
                            int64_t window, int nbuf, StatusWord *st, cudaStream_t s,
                            EventRec *rec) {
    using namespace tc;
    if (window > 65535) return cudaErrorInvalidValue;   // the prep grid's slot dimension
    int dev = 0, sm_count = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = kernel_attributes(dev);
    if (e != cudaSuccess) return e;
    const Fault flt = take_fault();
    CUtensorMap tm[4];
    if (T_tot > 0) {
        const void *const ptrs[4] = {q, k, z, v};
        e = tensor_maps(dev, ptrs, T_tot, H, tm);
        if (e != cudaSuccess) return e;
    } else {
        memset(tm, 0, sizeof tm);
    }
    const bool piped = nbuf == 2 && slots > window;
    Pipe *P = nullptr;
    std::unique_lock<std::mutex> lock(g_pipe_mutex, std::defer_lock);
    if (piped) {
        lock.lock();
        e = pipe_setup(dev, P);
        if (e != cudaSuccess) return e;
        e = cudaEventRecord(P->start, s);
        for (int i = 0; i < 2 && e == cudaSuccess; ++i) e = cudaStreamWaitEvent(P->prep[i], P->start, 0);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(P->chain, P->start, 0);
        if (e != cudaSuccess) return e;
    }
    const size_t buf_bytes = (size_t)window * H * REC_BYTES;
    int64_t w = 0;
    for (int64_t s0 = 0; s0 < slots; s0 += window, ++w) {
        const int64_t s1 = std::min(slots, s0 + window);
        const int par = (int)(w & 1);
        uint8_t *recs = records + (piped ? par * buf_bytes : 0);
        cudaStream_t sp = piped ? P->prep[par] : s;
        cudaStream_t sc = piped ? P->chain : s;
        // prep of window w; with two buffers, after the chain of window w - 2 has read
        // this buffer
        if (piped && w >= 2) {
            e = cudaStreamWaitEvent(sp, P->chain_done[par], 0);
            if (e != cudaSuccess) return e;
        }
        dim3 pg((unsigned)H, (unsigned)(s1 - s0));   // slot-major; a window holds < 65536 slots
        if (rec) rec->mark(sp);
        prep_kernel<<<pg, PREP_THREADS, P_SMEM, sp>>>(
            (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v,
            (const __nv_bfloat16 *)z, (const __nv_bfloat16 *)beta, A_log, cu, chunk_off, N, T_tot,
            H, (int32_t)s0, recs, st, tm[0], tm[1], tm[2], tm[3]);
        if (rec) rec->mark(sp);
        if (piped) {
            e = cudaEventRecord(P->prep_done[par], sp);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(sc, P->prep_done[par], 0);
            if (e != cudaSuccess) return e;
        }
        // A window holds at most min(N, window) sequences.  While their 32-column items
        // fit in about two waves the chain is latency-bound and the narrow kernel walks
        // the chunks fastest; with more items the 128-column kernel, which does the same
        // work in about half the SM time, finishes first.  Beside a prep kernel the
        // narrow one is kept only while it leaves at least half of the SMs to the prep.
        const int64_t seqs = std::min<int64_t>(N, s1 - s0);
        const int64_t items32 = seqs * H * c32::NBLK;
        if (rec) rec->mark(sc);
        if (items32 <= (piped ? (int64_t)sm_count / 2 : 2 * (int64_t)sm_count)) {
            const int64_t grid = std::min<int64_t>(seqs * H * c32::NBLK, sm_count);
            c32::chain_kernel<<<(unsigned)grid, c32::CHAIN_THREADS, c32::C_SMEM, sc>>>(
                cu, chunk_off, N, H, (int32_t)s0, (int32_t)s1, recs, h0, S_run,
                (__nv_bfloat16 *)o, st, SegArgs{0, 1, nullptr, nullptr}, flt);
        } else {
            const int64_t grid = std::min<int64_t>(seqs * H, sm_count);
            c128::chain_kernel<<<(unsigned)grid, c128::CHAIN_THREADS, c128::C_SMEM, sc>>>(
                cu, chunk_off, N, H, (int32_t)s0, (int32_t)s1, recs, h0, S_run,
                (__nv_bfloat16 *)o, st, flt);
        }
        if (rec) rec->mark(sc);
        if (piped) {
            e = cudaEventRecord(P->chain_done[par], sc);
            if (e != cudaSuccess) return e;
        }
    }
    if (piped) {
        e = cudaEventRecord(P->end, P->chain);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, P->end, 0);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

// The segment-parallel schedule (see SegArgs): per window of records, on `s` alone: prep,
// first pass (segment 0 walked, later segments' maps), scan, second pass.  Always the
// 32-column chain; `start` and `maps` hold N x H x segs blocks of the shapes in SegArgs.
cudaError_t launch_chunk_tc_segmented(const void *q, const void *k, const void *v,
                                      const void *z, const void *beta, const float *A_log,
                                      const int32_t *cu, const int32_t *chunk_off, int N,
                                      int64_t T_tot, int64_t slots, int H, const float *h0,
                                      float *S_run, void *o, uint8_t *records, int64_t window,
                                      int segs, float *start, float *maps, StatusWord *st,
                                      cudaStream_t s) {
    using namespace tc;
    if (window > 65535 || segs < 2) return cudaErrorInvalidValue;
    if (T_tot <= 0) return cudaSuccess;
    int dev = 0, sm_count = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = kernel_attributes(dev);
    if (e != cudaSuccess) return e;
    const Fault flt = take_fault();
    CUtensorMap tm[4];
    const void *const ptrs[4] = {q, k, z, v};
    e = tensor_maps(dev, ptrs, T_tot, H, tm);
    if (e != cudaSuccess) return e;
    for (int64_t s0 = 0; s0 < slots; s0 += window) {
        const int64_t s1 = std::min(slots, s0 + window);
        dim3 pg((unsigned)H, (unsigned)(s1 - s0));
        prep_kernel<<<pg, PREP_THREADS, P_SMEM, s>>>(
            (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v,
            (const __nv_bfloat16 *)z, (const __nv_bfloat16 *)beta, A_log, cu, chunk_off, N, T_tot,
            H, (int32_t)s0, records, st, tm[0], tm[1], tm[2], tm[3]);
        const int64_t pairs = std::min<int64_t>(N, s1 - s0) * H;
        const int64_t items1 = pairs * (c32::NBLK + 2 * c32::NBLK * (segs - 1));
        c32::chain_kernel<<<(unsigned)std::min<int64_t>(items1, sm_count), c32::CHAIN_THREADS,
                            c32::C_SMEM, s>>>(cu, chunk_off, N, H, (int32_t)s0, (int32_t)s1,
                                              records, h0, S_run, (__nv_bfloat16 *)o, st,
                                              SegArgs{1, segs, start, maps}, flt);
        c32::seg_scan_kernel<<<(unsigned)std::min<int64_t>(pairs * c32::NBLK, 4 * sm_count),
                               c32::DK_ROWS, 0, s>>>(cu, chunk_off, N, H, (int32_t)s0,
                                                      (int32_t)s1, SegArgs{1, segs, start, maps});
        const int64_t items2 = pairs * c32::NBLK * (segs - 1);
        c32::chain_kernel<<<(unsigned)std::min<int64_t>(items2, sm_count), c32::CHAIN_THREADS,
                            c32::C_SMEM, s>>>(cu, chunk_off, N, H, (int32_t)s0, (int32_t)s1,
                                              records, h0, S_run, (__nv_bfloat16 *)o, st,
                                              SegArgs{2, segs, start, maps}, flt);
    }
    return cudaGetLastError();
}

}  // namespace kda

// Test hook declared in kda.h: the next kda_chunk_fwd (tensor-core path) on this process
// gets `wait_ns` as the limit of every bounded wait of its chain kernels and leaves out
// the first record load of chain CTA `skip_cta`, whose wait for it then expires.
extern "C" kda_status kda_test_chain_fault(int64_t wait_ns, int32_t skip_cta) {
    if (wait_ns <= 0) return KDA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(kda::g_fault_mutex);
    kda::g_fault_next = kda::tc::Fault{(uint64_t)wait_ns, skip_cta};
    kda::g_fault_armed = true;
    return KDA_OK;
}
