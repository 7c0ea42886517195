// kda_chunk_fwd_split_noalloc: the segment-split prefill with its scratch in
// a buffer the library owns, for callers that cannot allocate device memory
// themselves (see include/kda.h).  The buffer is a file-scope device array
// of KDA_SPLIT_SCRATCH_BYTES; every GPU that loads the library holds it
// until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "kda.h"

namespace {

static __device__ __align__(256) unsigned char g_split_scratch[KDA_SPLIT_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code
// the array's name is only a stand-in, so the address is looked up once per
// device (with that device current) and cached.
cudaError_t scratch_address(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_split_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" kda_status kda_chunk_fwd_split_noalloc(kda_dtype dt, int B, int T, int H, int dk, int dv,
                                                  const void *q, const void *k, const void *v,
                                                  const void *g_raw, const void *beta,
                                                  const float *init_state,
                                                  const int32_t *cu_seqlens, int N, int segment_tokens,
                                                  void *out, float *final_state,
                                                  const kda_params *p, kda_stream_t stream) {
    const unsigned long long need =
        kda_chunk_fwd_split_workspace(B, T, H, dk, dv, N > 0 ? N : 1, segment_tokens);
    if (need == 0)   // sizes the split rejects: it reports which, before enqueuing anything
        return kda_chunk_fwd_split(dt, B, T, H, dk, dv, q, k, v, g_raw, beta, init_state, cu_seqlens, N,
                                   segment_tokens, out, final_state, nullptr, 0, p, stream);
    if (need > KDA_SPLIT_SCRATCH_BYTES) return KDA_ERR_SCRATCH;
    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return KDA_ERR_LAUNCH;
    return kda_chunk_fwd_split(dt, B, T, H, dk, dv, q, k, v, g_raw, beta, init_state, cu_seqlens, N,
                               segment_tokens, out, final_state, scratch, KDA_SPLIT_SCRATCH_BYTES, p,
                               stream);
}
