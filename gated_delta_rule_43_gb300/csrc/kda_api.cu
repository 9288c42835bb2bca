// kda_api.cu -- the C ABI of libkda.so (declared in include/kda.h): argument
// validation, workspace layout and kernel dispatch.  No device memory is
// allocated here; every buffer comes from the caller.
#include <stdint.h>
#include <string.h>

#include "kda_common.cuh"

namespace kda {
cudaError_t launch_decode(int dtype, int dk, int dv, const void *q, const void *k,
                          const void *v, const void *z, const void *beta, const float *A_log,
                          float *state, void *o, int N, int H, const int32_t *slot_idx, int P,
                          StatusWord *st, cudaStream_t s);
cudaError_t launch_chunk_simt(int dtype, int dk, int dv, const void *q, const void *k,
                              const void *v, const void *z, const void *beta,
                              const float *A_log, const int32_t *cu, int N, int64_t T_tot, int H,
                              const float *h0, float *hT, void *o, StatusWord *st,
                              cudaStream_t s, EventRec *rec);
cudaError_t launch_plan(const int32_t *cu, int N, int64_t T_tot, int C, int32_t *chunk_off,
                        StatusWord *st, cudaStream_t s);
cudaError_t launch_plan_tc(const int32_t *cu, int N, int64_t T_tot, int C, int32_t *chunk_off,
                           StatusWord *st, const float *h0, float *S_run, int H, int64_t dkdv,
                           int grid, cudaStream_t s);
size_t tc_record_bytes();
cudaError_t launch_chunk_tc(const void *q, const void *k, const void *v, const void *z,
                            const void *beta, const float *A_log, const int32_t *cu,
                            const int32_t *chunk_off, int N, int64_t T_tot, int64_t slots, int H,
                            const float *h0, float *S_run, void *o, uint8_t *records,
                            int64_t window, int nbuf, StatusWord *st, cudaStream_t s,
                            EventRec *rec);
cudaError_t launch_chunk_tc_segmented(const void *q, const void *k, const void *v,
                                      const void *z, const void *beta, const float *A_log,
                                      const int32_t *cu, const int32_t *chunk_off, int N,
                                      int64_t T_tot, int64_t slots, int H, const float *h0,
                                      float *S_run, void *o, uint8_t *records, int64_t window,
                                      int segs, float *start, float *maps, StatusWord *st,
                                      cudaStream_t s);
int64_t chunk_slots(int64_t T_tot, int N, int C);
cudaError_t launch_gate(int dtype, const void *z, const float *A_log, const int32_t *cu,
                        const int32_t *chunk_off, int N, int64_t T_tot, int H, int dk, int C,
                        int mode, float *G, StatusWord *st, cudaStream_t s);
}  // namespace kda

using namespace kda;

namespace {

constexpr int32_t kAbiVersion = 1;

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }
inline bool head_ok(int32_t d) { return d == 32 || d == 64 || d == 128; }

// Chunk length of the tensor-core path and the byte budget of the chunk records.
// A window of records is produced by the prep kernel and consumed by the chain
// kernel.  Every window costs a ramp and a tail of both kernels, which measured
// more than the DRAM round trip of the records, so windows are large: a problem
// whose records fit the budget runs as one window; a larger one is cut into
// windows of half the budget, double-buffered so that the prep of window w + 1
// runs beside the chain of window w.
constexpr int kTcChunk = 64;
constexpr size_t kTcRecordBudget = 1u << 30;

bool use_tc(int32_t dtype, int32_t dk, int32_t dv) {
    return dtype == KDA_BF16 && dk == 128 && dv == 128;
}

struct ChunkLayout {
    size_t plan_off, plan_bytes;
    size_t state_off, state_bytes;   // running state of the tensor-core path
    size_t rec_off, rec_bytes;       // one or two windows of chunk records
    int64_t slots, window;
    int nbuf;                        // record buffers: 2 when there is more than one window
    size_t seg_off, seg_bytes;       // segmented schedule: segment start states
    size_t map_off, map_bytes;       //   and [M | B] maps
    int segs;                        // segments per sequence and window (1: plain schedule)
    size_t total;
};

ChunkLayout chunk_layout(int64_t T, int32_t N, int32_t H, int32_t dk, int32_t dv,
                         int32_t dtype) {
    ChunkLayout L{};
    L.plan_off = kHeaderBytes;
    L.plan_bytes = round_up(sizeof(int32_t) * ((size_t)N + 1), 1024);
    L.state_off = L.plan_off + L.plan_bytes;
    L.rec_off = L.state_off;
    if (use_tc(dtype, dk, dv)) {
        L.state_bytes = round_up((size_t)N * H * dk * dv * sizeof(float), 1024);
        L.rec_off = L.state_off + L.state_bytes;
        L.slots = chunk_slots(T, N, kTcChunk);
        const size_t rec = tc_record_bytes() * (size_t)H;
        int64_t w = (int64_t)(kTcRecordBudget / rec);
        if (w < 1) w = 1;
        if (L.slots <= w) {
            L.window = L.slots;
            L.nbuf = 1;
        } else {
            L.window = w / 2 > 0 ? w / 2 : 1;
            L.nbuf = 2;
        }
        L.rec_bytes = (size_t)L.nbuf * L.window * rec;
    }
    L.segs = 1;
    L.seg_off = L.map_off = L.rec_off + L.rec_bytes;
    L.seg_bytes = L.map_bytes = 0;
    L.total = L.rec_off + L.rec_bytes;
    return L;
}

// The segment-parallel schedule runs its windows one after the other (one record
// buffer) and adds the start states and maps of the later segments.
ChunkLayout chunk_layout_seg(int64_t T, int32_t N, int32_t H, int32_t dk, int32_t dv,
                             int32_t dtype, int32_t segs) {
    ChunkLayout L = chunk_layout(T, N, H, dk, dv, dtype);
    if (segs <= 1 || !use_tc(dtype, dk, dv)) return L;
    const size_t rec = tc_record_bytes() * (size_t)H;
    int64_t w = (int64_t)(kTcRecordBudget / rec);
    if (w < 1) w = 1;
    L.window = L.slots < w ? L.slots : w;
    L.nbuf = 1;
    L.rec_bytes = (size_t)L.window * rec;
    L.segs = segs;
    const size_t pairs = (size_t)N * H * segs;
    L.seg_off = L.rec_off + L.rec_bytes;
    L.seg_bytes = round_up(pairs * dk * dv * sizeof(float), 1024);
    L.map_off = L.seg_off + L.seg_bytes;
    L.map_bytes = round_up(pairs * dk * (dk + dv) * sizeof(float), 1024);
    L.total = L.map_off + L.map_bytes;
    return L;
}

// The segment count kda_chunk_fwd picks by itself on the tensor-core path: the largest
// s <= 16 whose first pass, N H (4 + 8 (s - 1)) 32-column CTAs, still fits one wave of
// the current device's SMs while the average sequence keeps >= 64 chunks per segment;
// 1 (the plain schedule) when even s = 2 does not qualify.  Measured: one 1M-token
// sequence with 4 heads runs in 10.1 ms with 5 segments against 16.0 ms plain; the
// benchmark workloads (8K with 32 heads, 1M with 16, 64 packed sequences) stay plain.
int32_t auto_segments(int64_t T, int32_t N, int32_t H, int32_t dk, int32_t dv, int32_t dtype) {
    if (!use_tc(dtype, dk, dv) || N <= 0 || T <= 0) return 1;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 1;
    const int64_t pairs = (int64_t)N * H;
    const int64_t chunks = T / ((int64_t)kTcChunk * N);   // whole chunks of the average sequence
    int32_t best = 1;
    for (int32_t s = 2; s <= 16; ++s) {
        if (pairs * (4 + 8 * (s - 1)) > sms || chunks < 64 * (int64_t)s) break;
        best = s;
    }
    return best;
}

kda_status cuda_status(cudaError_t e) { return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA; }

// Grids over chunk slots use gridDim.x, which is limited to 2^31 - 1.
bool chunk_slots_overflow(int64_t T, int32_t N, int32_t C) {
    return (T + C - 1) / C + N > 0x7fffffffLL;
}

// The chunked forward behind kda_chunk_fwd and kda_chunk_fwd_profiled; `rec`
// (optional) records timing events around every kernel it launches.
kda_status chunk_fwd_impl(const void *q, const void *k, const void *v, const void *z,
                          const void *beta, const float *A_log, const int32_t *cu_seqlens,
                          int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t dk,
                          int32_t dv, int32_t dtype, const float *initial_state,
                          float *final_state, void *o, void *workspace, size_t workspace_bytes,
                          void *stream, EventRec *rec, int32_t segs = 1) {
    if (dtype != KDA_F32 && dtype != KDA_BF16) return KDA_ERR_UNSUPPORTED;
    if (!head_ok(dk) || !head_ok(dv)) return KDA_ERR_UNSUPPORTED;
    if (num_seqs < 0 || total_tokens < 0 || H <= 0) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && num_seqs == 0) return KDA_ERR_INVALID_ARG;
    if (total_tokens > ((int64_t)1 << 40) / ((int64_t)H * (dk > dv ? dk : dv)))
        return KDA_ERR_INVALID_ARG;
    if (!A_log || !cu_seqlens || !workspace) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q || !k || !v || !z || !beta || !o)) return KDA_ERR_INVALID_ARG;
    const void *al16[] = {q, k, v, z, o, initial_state, final_state};
    for (const void *p : al16)
        if (!aligned(p, 16)) return KDA_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return KDA_ERR_INVALID_ARG;
    if (o && (o == q || o == k || o == v || o == z || o == beta)) return KDA_ERR_INVALID_ARG;
    if (segs < 1 || segs > 64) return KDA_ERR_INVALID_ARG;
    const ChunkLayout L = chunk_layout_seg(total_tokens, num_seqs, H, dk, dv, dtype, segs);
    if (workspace_bytes < L.total) return KDA_ERR_INVALID_ARG;
    if (chunk_slots_overflow(total_tokens, num_seqs, kTcChunk)) return KDA_ERR_INVALID_ARG;
    // token coordinates of the tensor-core path's tile loads are 32-bit
    if (use_tc(dtype, dk, dv) && total_tokens >= ((int64_t)1 << 31)) return KDA_ERR_INVALID_ARG;

    cudaStream_t s = (cudaStream_t)stream;
    StatusWord *st = (StatusWord *)workspace;
    cudaError_t e = cudaSuccess;
    if (num_seqs > 0 && use_tc(dtype, dk, dv)) {
        // the plan kernel clears the status word and gives chunk-less sequences their
        // final state; the chain kernels read the initial state themselves
        uint8_t *ws = (uint8_t *)workspace;
        int32_t *chunk_off = (int32_t *)(ws + L.plan_off);
        float *S_run = final_state ? final_state : (float *)(ws + L.state_off);
        const int64_t nh = (int64_t)num_seqs * H;
        if (rec) rec->mark(s);
        e = launch_plan_tc(cu_seqlens, num_seqs, total_tokens, kTcChunk, chunk_off, st,
                           initial_state, S_run, H, (int64_t)dk * dv, (int)(nh < 256 ? nh : 256),
                           s);
        if (e != cudaSuccess) return KDA_ERR_CUDA;
        if (rec) rec->mark(s);
        if (L.segs > 1)
            e = launch_chunk_tc_segmented(q, k, v, z, beta, A_log, cu_seqlens, chunk_off,
                                          num_seqs, total_tokens, L.slots, H, initial_state,
                                          S_run, o, ws + L.rec_off, L.window, L.segs,
                                          (float *)(ws + L.seg_off), (float *)(ws + L.map_off),
                                          st, s);
        else
            e = launch_chunk_tc(q, k, v, z, beta, A_log, cu_seqlens, chunk_off, num_seqs,
                                total_tokens, L.slots, H,
                                initial_state, S_run, o, ws + L.rec_off, L.window, L.nbuf, st, s,
                                rec);
        return cuda_status(e);
    }
    e = cudaMemsetAsync(st, 0, sizeof(StatusWord), s);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    if (num_seqs == 0) return KDA_OK;
    e = launch_chunk_simt(dtype, dk, dv, q, k, v, z, beta, A_log, cu_seqlens, num_seqs,
                          total_tokens, H, initial_state, final_state, o, st, s, rec);
    return cuda_status(e);
}

}  // namespace

extern "C" {

int32_t kda_abi_version(void) { return kAbiVersion; }

const char *kda_status_string(int32_t s) {
    switch (s) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: invalid argument";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: unsupported head size or dtype";
        case KDA_ERR_DECAY_RANGE:
            return "KDA_ERR_DECAY_RANGE: 16-token cumulative log-decay not finite or outside [-80, 0]";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT: a bounded device wait expired";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA: CUDA runtime error";
        case KDA_ERR_SEQLENS: return "KDA_ERR_SEQLENS: inconsistent cu_seqlens";
        default: return "KDA_ERR_UNKNOWN";
    }
}

size_t kda_chunk_fwd_workspace_size(int64_t total_tokens, int32_t num_seqs, int32_t H,
                                    int32_t dk, int32_t dv, int32_t dtype) {
    if (total_tokens < 0 || num_seqs < 0 || H <= 0 || !head_ok(dk) || !head_ok(dv) ||
        (dtype != KDA_F32 && dtype != KDA_BF16))
        return 0;
    return chunk_layout_seg(total_tokens, num_seqs, H, dk, dv, dtype,
                            auto_segments(total_tokens, num_seqs, H, dk, dv, dtype)).total;
}

size_t kda_chunk_fwd_segmented_workspace_size(int64_t total_tokens, int32_t num_seqs, int32_t H,
                                              int32_t dk, int32_t dv, int32_t dtype,
                                              int32_t segments) {
    if (total_tokens < 0 || num_seqs < 0 || H <= 0 || !head_ok(dk) || !head_ok(dv) ||
        (dtype != KDA_F32 && dtype != KDA_BF16) || segments < 1 || segments > 64)
        return 0;
    return chunk_layout_seg(total_tokens, num_seqs, H, dk, dv, dtype, segments).total;
}

size_t kda_decode_workspace_size(void) { return kHeaderBytes; }

kda_status kda_chunk_fwd(const void *q, const void *k, const void *v, const void *z,
                         const void *beta, const float *A_log, const int32_t *cu_seqlens,
                         int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t dk,
                         int32_t dv, int32_t dtype, const float *initial_state,
                         float *final_state, void *o, void *workspace, size_t workspace_bytes,
                         void *stream) {
    // the segment-parallel schedule when it pays and the workspace holds it
    int32_t segs = auto_segments(total_tokens, num_seqs, H, dk, dv, dtype);
    if (segs > 1 &&
        workspace_bytes < chunk_layout_seg(total_tokens, num_seqs, H, dk, dv, dtype, segs).total)
        segs = 1;
    return chunk_fwd_impl(q, k, v, z, beta, A_log, cu_seqlens, num_seqs, total_tokens, H, dk, dv,
                          dtype, initial_state, final_state, o, workspace, workspace_bytes, stream,
                          nullptr, segs);
}

kda_status kda_chunk_fwd_segmented(const void *q, const void *k, const void *v, const void *z,
                                   const void *beta, const float *A_log,
                                   const int32_t *cu_seqlens, int32_t num_seqs,
                                   int64_t total_tokens, int32_t H, int32_t dk, int32_t dv,
                                   int32_t dtype, const float *initial_state, float *final_state,
                                   void *o, int32_t segments, void *workspace,
                                   size_t workspace_bytes, void *stream) {
    return chunk_fwd_impl(q, k, v, z, beta, A_log, cu_seqlens, num_seqs, total_tokens, H, dk, dv,
                          dtype, initial_state, final_state, o, workspace, workspace_bytes, stream,
                          nullptr, segments);
}

kda_status kda_chunk_fwd_profiled(const void *q, const void *k, const void *v, const void *z,
                                  const void *beta, const float *A_log,
                                  const int32_t *cu_seqlens, int32_t num_seqs,
                                  int64_t total_tokens, int32_t H, int32_t dk, int32_t dv,
                                  int32_t dtype, const float *initial_state, float *final_state,
                                  void *o, void *workspace, size_t workspace_bytes, void *stream,
                                  void *const *events, int32_t n_events, int32_t *n_recorded) {
    if (!events || n_events < 1 || !n_recorded) return KDA_ERR_INVALID_ARG;
    EventRec rec;
    rec.ev = (cudaEvent_t *)events;
    rec.cap = n_events;
    const kda_status r = chunk_fwd_impl(q, k, v, z, beta, A_log, cu_seqlens, num_seqs,
                                        total_tokens, H, dk, dv, dtype, initial_state,
                                        final_state, o, workspace, workspace_bytes, stream, &rec);
    *n_recorded = rec.used;
    return r;
}

// Shared body of kda_decode_step (slot_idx NULL: sequence n owns state n) and
// kda_decode_step_indexed (sequence n owns slot slot_idx[n] of a pool of P).
static kda_status decode_impl(const void *q, const void *k, const void *v, const void *z,
                              const void *beta, const float *A_log, float *state,
                              const int32_t *slot_idx, int32_t P, void *o, int32_t N,
                              int32_t H, int32_t dk, int32_t dv, int32_t dtype, void *workspace,
                              size_t workspace_bytes, void *stream) {
    if (dtype != KDA_F32 && dtype != KDA_BF16) return KDA_ERR_UNSUPPORTED;
    if (!head_ok(dk) || !head_ok(dv)) return KDA_ERR_UNSUPPORTED;
    if (N < 0 || H <= 0 || P < 0) return KDA_ERR_INVALID_ARG;
    if ((int64_t)N * H > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < kHeaderBytes || !aligned(workspace, 256))
        return KDA_ERR_INVALID_ARG;
    if (N > 0 && (!q || !k || !v || !z || !beta || !A_log || !state || !o))
        return KDA_ERR_INVALID_ARG;
    const void *al16[] = {q, k, v, z, o, state};
    for (const void *p : al16)
        if (!aligned(p, 16)) return KDA_ERR_INVALID_ARG;
    if (o && (o == q || o == k || o == v || o == z || o == beta || o == (void *)state))
        return KDA_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    StatusWord *st = (StatusWord *)workspace;
    cudaError_t e = cudaMemsetAsync(st, 0, sizeof(StatusWord), s);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    if (N == 0) return KDA_OK;
    return cuda_status(launch_decode(dtype, dk, dv, q, k, v, z, beta, A_log, state, o, N, H,
                                     slot_idx, P, st, s));
}

kda_status kda_decode_step(const void *q, const void *k, const void *v, const void *z,
                           const void *beta, const float *A_log, float *state, void *o,
                           int32_t N, int32_t H, int32_t dk, int32_t dv, int32_t dtype,
                           void *workspace, size_t workspace_bytes, void *stream) {
    return decode_impl(q, k, v, z, beta, A_log, state, nullptr, N, o, N, H, dk, dv, dtype,
                       workspace, workspace_bytes, stream);
}

kda_status kda_decode_step_indexed(const void *q, const void *k, const void *v, const void *z,
                                   const void *beta, const float *A_log, float *state_pool,
                                   const int32_t *state_idx, int32_t P, void *o, int32_t N,
                                   int32_t H, int32_t dk, int32_t dv, int32_t dtype,
                                   void *workspace, size_t workspace_bytes, void *stream) {
    if (N > 0 && !state_idx) return KDA_ERR_INVALID_ARG;
    return decode_impl(q, k, v, z, beta, A_log, state_pool, state_idx, P, o, N, H, dk, dv,
                       dtype, workspace, workspace_bytes, stream);
}

kda_status kda_gate_cumsum(const void *z, const float *A_log, const int32_t *cu_seqlens,
                           int32_t num_seqs, int64_t total_tokens, int32_t H, int32_t dk,
                           int32_t dtype, int32_t chunk, int32_t gate_mode, float *g_cumsum,
                           void *workspace, size_t workspace_bytes, void *stream) {
    if (dtype != KDA_F32 && dtype != KDA_BF16) return KDA_ERR_UNSUPPORTED;
    if (gate_mode != 0 && gate_mode != 1) return KDA_ERR_INVALID_ARG;
    if (!head_ok(dk)) return KDA_ERR_UNSUPPORTED;
    if (num_seqs < 0 || total_tokens < 0 || H <= 0 || chunk <= 0 || chunk % kTile != 0)
        return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && num_seqs == 0) return KDA_ERR_INVALID_ARG;
    if (!A_log || !cu_seqlens || !workspace || (total_tokens > 0 && (!z || !g_cumsum)))
        return KDA_ERR_INVALID_ARG;
    if (!aligned(z, 16) || !aligned(g_cumsum, 16) || !aligned(workspace, 256))
        return KDA_ERR_INVALID_ARG;
    if ((const void *)g_cumsum == z && g_cumsum) return KDA_ERR_INVALID_ARG;
    const ChunkLayout L = chunk_layout(total_tokens, num_seqs, H, dk, dk, dtype);
    if (workspace_bytes < L.total) return KDA_ERR_INVALID_ARG;
    if (chunk_slots_overflow(total_tokens, num_seqs, chunk)) return KDA_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    StatusWord *st = (StatusWord *)workspace;
    int32_t *chunk_off = (int32_t *)((char *)workspace + L.plan_off);
    cudaError_t e = cudaMemsetAsync(st, 0, sizeof(StatusWord), s);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    if (num_seqs == 0) return KDA_OK;
    e = launch_plan(cu_seqlens, num_seqs, total_tokens, chunk, chunk_off, st, s);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    e = launch_gate(dtype, z, A_log, cu_seqlens, chunk_off, num_seqs, total_tokens, H, dk, chunk,
                    gate_mode, g_cumsum, st, s);
    return cuda_status(e);
}

kda_status kda_query_status(const void *workspace, void *stream, int64_t *info) {
    if (!workspace) return KDA_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
    StatusWord w;
    if (cudaMemcpy(&w, workspace, sizeof w, cudaMemcpyDeviceToHost) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (info) *info = (int64_t)w.info;
    return (kda_status)w.code;
}

}  // extern "C"
