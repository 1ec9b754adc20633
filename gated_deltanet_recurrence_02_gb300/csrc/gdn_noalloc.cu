// gdn_noalloc.cu -- gdn_prefill_chunked_noalloc: the chunked prefill for
// callers that cannot allocate device memory.
//
// The tensor-core prefill needs a scratch workspace (one record per chunk and
// value head).  gdn_prefill_chunked takes it from the caller; this entry point
// instead uses a fixed buffer compiled into the library: the file-scope device
// array below, GDN_NOALLOC_SCRATCH_BYTES long.  Every device that loads the
// library holds that buffer until the process exits.
//
// Host code must not pass `g_prefill_scratch` itself to a kernel: in host code
// that name denotes a host-side shadow object, not device memory.  Its device
// address is looked up with cudaGetSymbolAddress, once per device, with that
// device current, on the first call made on that device; the address is then
// cached.  That first call therefore makes a CUDA runtime query and should be
// made before any stream capture begins.
//
// Every call shares the one buffer, and the buffer keeps whatever the last
// call left in it.  The prefill writes every scratch byte it later reads, so
// nothing needs clearing between calls.  Two calls whose work overlaps on the
// GPU (for example on two streams without ordering between them) race on the
// buffer; callers must serialise them.
//
// No allocation happens here or below: no cudaMalloc / cudaFree, no torch, no
// allocating library routine.  A problem whose workspace would exceed the
// buffer is rejected with GDN_ERR_WORKSPACE before anything is launched.
#include <mutex>

#include "gdn_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_prefill_scratch[GDN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of the scratch buffer on the current device (set-up on the
// first use per device).
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_prefill_scratch) != cudaSuccess || ptr == nullptr)
            return GDN_ERR_CUDA;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return GDN_OK;
}

}  // namespace

extern "C" int gdn_prefill_chunked_noalloc(const void *q, const void *k, const void *v,
                                           const void *alpha, const void *beta,
                                           const int32_t *cu_seqlens, const float *initial_state,
                                           const int32_t *initial_state_indices,
                                           int num_initial_states, float *final_state, void *out,
                                           int B, int T, int Hq, int Hk, int Hv, int dk, int dv,
                                           int chunk, float scale, int dtype_qkv, int dtype_gate,
                                           void *stream) {
    const size_t need =
        gdn_prefill_workspace_size(B, T, Hk, Hv, dk, dv, chunk, dtype_qkv, cu_seqlens != nullptr);
    if (need == (size_t)-1) return GDN_ERR_INVALID_ARG;
    if (need > (size_t)GDN_NOALLOC_SCRATCH_BYTES) return GDN_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (need > 0) {
        const int st = scratch_address(&scratch);
        if (st != GDN_OK) return st;
    }
    return gdn_prefill_chunked(q, k, v, alpha, beta, cu_seqlens, initial_state, initial_state_indices,
                               num_initial_states, final_state, out, B, T, Hq, Hk, Hv, dk, dv, chunk,
                               scale, dtype_qkv, dtype_gate, scratch,
                               scratch ? (size_t)GDN_NOALLOC_SCRATCH_BYTES : 0, stream);
}
