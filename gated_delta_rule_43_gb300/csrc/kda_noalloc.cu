// kda_noalloc.cu -- kda_chunk_fwd_noalloc: the chunked forward for callers that cannot
// allocate device memory.
//
// Some callers are handed their input and output buffers and nothing else: a
// plug-in running inside a host application that owns every device
// allocation, or a serving loop that must not call cudaMalloc after start-up
// (it synchronises the device and can fail under memory pressure).  They
// cannot provide the workspace kda_chunk_fwd asks for.  This entry point runs
// the same kernels with their scratch (status word, chunk plan, running state,
// one window of chunk records) in a fixed-size array that the library owns.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds KDA_NOALLOC_SCRATCH_BYTES of it until the process exits.
// Host code cannot use its name as a device address, so every call looks the
// address up with cudaGetSymbolAddress on the current device (no allocation, and no
// cached pointer that a cudaDeviceReset could leave stale); the first call on a device
// also loads the library's device code there, so it should happen before any stream
// capture.  All calls share the one array: calls whose work
// overlaps on the GPU (different streams, or different host threads without
// ordering) race on it and must be serialised by the caller.  Nothing in the
// array has to start at zero: the status word is cleared by every call and
// every other byte read by a kernel is written earlier in the same call.
#include "kda_common.cuh"

namespace kda {
cudaError_t launch_plan_tc(const int32_t *cu, int N, int64_t T_tot, int C, int32_t *chunk_off,
                           StatusWord *st, const float *h0, float *S_run, int H, int64_t dkdv,
                           int grid, cudaStream_t s);
cudaError_t launch_chunk_tc(const void *q, const void *k, const void *v, const void *z,
                            const void *beta, const float *A_log, const int32_t *cu,
                            const int32_t *chunk_off, int N, int64_t T_tot, int64_t slots, int H,
                            const float *h0, float *S_run, void *o, uint8_t *records,
                            int64_t window, int nbuf, StatusWord *st, cudaStream_t s,
                            EventRec *rec);
cudaError_t launch_chunk_simt(int dtype, int dk, int dv, const void *q, const void *k,
                              const void *v, const void *z, const void *beta,
                              const float *A_log, const int32_t *cu, int N, int64_t T_tot, int H,
                              const float *h0, float *hT, void *o, StatusWord *st,
                              cudaStream_t s, EventRec *rec);
size_t tc_record_bytes();
int64_t chunk_slots(int64_t T_tot, int N, int C);
}  // namespace kda

using namespace kda;

namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on the current device.
cudaError_t scratch_address(void **out) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    *out = p;
    return cudaSuccess;
}

inline size_t up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline bool al(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }
inline bool head_ok(int32_t d) { return d == 32 || d == 64 || d == 128; }

constexpr int kChunk = 64;                    // tensor-core chunk length

}  // namespace

extern "C" kda_status kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                                            const void *z, const void *beta, const float *A_log,
                                            const int32_t *cu_seqlens, int32_t num_seqs,
                                            int64_t total_tokens, int32_t H, int32_t dk,
                                            int32_t dv, int32_t dtype,
                                            const float *initial_state, float *final_state,
                                            void *o, void *status_out, void *stream) {
    if (dtype != KDA_F32 && dtype != KDA_BF16) return KDA_ERR_UNSUPPORTED;
    if (!head_ok(dk) || !head_ok(dv)) return KDA_ERR_UNSUPPORTED;
    if (num_seqs < 0 || total_tokens < 0 || H <= 0) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && num_seqs == 0) return KDA_ERR_INVALID_ARG;
    if (total_tokens > ((int64_t)1 << 40) / ((int64_t)H * (dk > dv ? dk : dv)))
        return KDA_ERR_INVALID_ARG;
    if (!A_log || !cu_seqlens) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q || !k || !v || !z || !beta || !o)) return KDA_ERR_INVALID_ARG;
    const void *al16[] = {q, k, v, z, o, initial_state, final_state, status_out};
    for (const void *p : al16)
        if (!al(p, 16)) return KDA_ERR_INVALID_ARG;
    if (o && (o == q || o == k || o == v || o == z || o == beta)) return KDA_ERR_INVALID_ARG;
    if ((total_tokens + kChunk - 1) / kChunk + num_seqs > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    const bool tc = dtype == KDA_BF16 && dk == 128 && dv == 128;
    // token coordinates of the tensor-core path's tile loads are 32-bit
    if (tc && total_tokens >= ((int64_t)1 << 31)) return KDA_ERR_INVALID_ARG;

    // Scratch layout inside the fixed array; reject what does not fit.  The window of
    // chunk records is whatever the array has left after the plan and the running state.
    const size_t plan_off = kHeaderBytes;
    const size_t plan_bytes = up(sizeof(int32_t) * ((size_t)num_seqs + 1), 1024);
    size_t state_off = plan_off + plan_bytes, state_bytes = 0, rec_off = state_off;
    int64_t slots = 0, window = 0;
    if (tc) {
        if (!final_state) state_bytes = up((size_t)num_seqs * H * dk * dv * sizeof(float), 1024);
        rec_off = state_off + state_bytes;
        if (rec_off > KDA_NOALLOC_SCRATCH_BYTES) return KDA_ERR_INVALID_ARG;
        const size_t rec = tc_record_bytes() * (size_t)H;
        slots = chunk_slots(total_tokens, num_seqs, kChunk);
        const int64_t fit = (int64_t)((KDA_NOALLOC_SCRATCH_BYTES - rec_off) / rec);
        if (fit < 1 && slots > 0) return KDA_ERR_INVALID_ARG;
        window = slots < fit ? slots : fit;
    } else if (plan_off + plan_bytes > KDA_NOALLOC_SCRATCH_BYTES) {
        return KDA_ERR_INVALID_ARG;
    }

    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return KDA_ERR_CUDA;
    uint8_t *ws = (uint8_t *)scratch;
    StatusWord *st = (StatusWord *)ws;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaMemsetAsync(st, 0, sizeof(StatusWord), s);
    if (e == cudaSuccess && num_seqs > 0) {
        if (tc) {
            int32_t *chunk_off = (int32_t *)(ws + plan_off);
            float *S_run = final_state ? final_state : (float *)(ws + state_off);
            const int64_t nh = (int64_t)num_seqs * H;
            e = launch_plan_tc(cu_seqlens, num_seqs, total_tokens, kChunk, chunk_off, st,
                               initial_state, S_run, H, (int64_t)dk * dv,
                               (int)(nh < 256 ? nh : 256), s);
            if (e == cudaSuccess)
                e = launch_chunk_tc(q, k, v, z, beta, A_log, cu_seqlens, chunk_off, num_seqs,
                                    total_tokens, slots, H, initial_state, S_run, o, ws + rec_off, window, 1,
                                    st, s, nullptr);
        } else {
            e = launch_chunk_simt(dtype, dk, dv, q, k, v, z, beta, A_log, cu_seqlens, num_seqs,
                                  total_tokens, H, initial_state, final_state, o, st, s,
                                  nullptr);
        }
    }
    if (e == cudaSuccess && status_out)
        e = cudaMemcpyAsync(status_out, st, sizeof(StatusWord), cudaMemcpyDeviceToDevice, s);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
