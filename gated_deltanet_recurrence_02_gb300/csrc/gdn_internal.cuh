// gdn_internal.cuh -- parameter blocks, launchers and small device helpers
// shared by the libgdn kernels.  Not part of the public ABI (include/gdn.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/gdn.h"

namespace gdn {

// Every parameter block carries `err`: the device address of the library's
// error word (GDN_DEVERR_* bits), resolved by the host layer per device, and
// `wait_ns`: the limit of waits on another warp's work (kDefaultWaitNs unless
// a test lowered it with gdn_set_wait_limit_ns).  Waits for a CTA's own copies
// in flight, before it exits, always use kDefaultWaitNs.
constexpr uint64_t kDefaultWaitNs = 1000000000ull;

// ---------------------------------------------------------------- params --

struct RecurrentParams {
    const void *q, *k, *v, *alpha, *beta;
    const int32_t *cu_seqlens;
    const float *s0;
    const int32_t *s0_idx;
    int n_s0;
    float *s_final;
    void *out;
    int B, T, Hk, Hv, dk, dv;
    float scale;
    int dt_qkv, dt_gate;
    int conv;  // GDN_QK_L2NORM | GDN_ALPHA_LOG | GDN_BETA_LOGIT bits
    int capacity;
    const int32_t *capture_count;
    const int32_t *active;
    float *su;
    // Fused replay + verify: before the tokens, replay the first
    // clamp(rp_accepted[b], 0, rp_capacity) slots of rp_su onto the state and
    // write the result to s_commit.  rp_capacity == 0 and s_commit == nullptr
    // for the plain recurrent path.
    const float *rp_su;
    int rp_capacity;
    const int32_t *rp_accepted;
    float *s_commit;
    uint64_t wait_ns;
    uint32_t *err;
};

struct ReplayParams {
    const float *s_in;
    float *s_out;
    const float *su;
    int capacity;
    const int32_t *accepted;
    int B, Hk, Hv, dk, dv;
    uint64_t wait_ns;
    uint32_t *err;
};

struct PrefillParams {
    const void *q, *k, *v, *alpha, *beta;
    const int32_t *cu_seqlens;
    const float *s0;
    const int32_t *s0_idx;
    int n_s0;
    float *s_final;
    void *out;
    int B, T, Hk, Hv, dk, dv, chunk;
    float scale;
    int dt_qkv, dt_gate;
    int conv;  // GDN_QK_L2NORM | GDN_ALPHA_LOG | GDN_BETA_LOGIT bits
    void *ws;
    size_t ws_bytes;
    // Chunk-boundary checkpoints (nullptr: none): slot j of row b receives the
    // state after (j + 1) * ckpt_every chunks, for j < ckpt_cap, when that
    // boundary lies inside the row.  Layout [B, ckpt_cap, Hv, dv, dk].
    float *ckpt;
    int ckpt_cap, ckpt_every;
    // Compact capture as on the recurrent path (capacity 0: none): tokens
    // t < n_b of row b write decay, shared key and delta into slot t; while
    // inactive the whole [B, capacity, slot] buffer is zeroed instead.
    int capacity;
    const int32_t *capture_count;
    const int32_t *active;
    float *su;
    // Packed rows on the tensor-core path: the first global chunk index of
    // every row (B + 1 entries), written into the head of the workspace by a
    // prologue kernel; nullptr for uniform rows.
    const int32_t *chunk_table;
    uint64_t wait_ns;
    uint32_t *err;
};

// Captured tokens of row b (row length len): n_b = clamp(count, 0, min(capacity, len)),
// 0 when capture is off or inactive.
__device__ __forceinline__ int prefill_ncap(const PrefillParams &p, int b, int len) {
    if (p.capacity <= 0 || (p.active != nullptr && *p.active == 0)) return 0;
    const int c = p.capture_count[b];
    const int lim = p.capacity < len ? p.capacity : len;
    return c < 0 ? 0 : (c > lim ? lim : c);
}

// Inactive capture: CTA `cta` of `ncta` zeroes its share of the whole buffer.
__device__ __forceinline__ void prefill_capture_clear(const PrefillParams &p, long slot, long cta, long ncta,
                                                      int tid, int nthreads) {
    if (p.capacity <= 0 || p.active == nullptr || *p.active != 0) return;
    const long total = (long)p.B * p.capacity * slot;
    const long per = (total + ncta - 1) / ncta;
    const long e0 = cta * per;
    const long e1 = (e0 + per < total) ? e0 + per : total;
    for (long e = e0 + tid; e < e1; e += nthreads) p.su[e] = 0.0f;
}

// Checkpoint slot written at the end of chunk cc (0-based) of a row of len
// tokens, or -1.
__host__ __device__ __forceinline__ int ckpt_slot(const PrefillParams &p, int cc, int len) {
    if (p.ckpt == nullptr) return -1;
    const int done = cc + 1;
    if (done % p.ckpt_every != 0 || (long)done * p.chunk > len) return -1;
    const int j = done / p.ckpt_every - 1;
    return j < p.ckpt_cap ? j : -1;
}

// Launchers: enqueue on `stream`, return cudaGetLastError().
cudaError_t launch_recurrent(const RecurrentParams &p, cudaStream_t stream);
cudaError_t launch_replay(const ReplayParams &p, cudaStream_t stream);
cudaError_t launch_prefill_simt(const PrefillParams &p, cudaStream_t stream);
bool prefill_simt_supported(int dk, int dv, int chunk);
cudaError_t launch_prefill_tc(const PrefillParams &p, cudaStream_t stream);
bool prefill_tc_supported(int dk, int dv, int chunk, int dt_qkv);
size_t prefill_tc_workspace_bytes(int B, int T, int Hk, int Hv, bool varlen);

// Raises kernel Kern's dynamic shared-memory limit to `bytes`, once per device
// (function attributes belong to the device's context): later calls make no
// CUDA call, so launches captured into a CUDA graph carry none.
template <auto Kern>
inline cudaError_t set_smem_once(int bytes) {
    static std::atomic<uint64_t> done{0};  // one bit per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
    e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// Multiprocessor count of the current device, cached per device (0..63) so
// that calls after the first make no CUDA call.
inline int sm_count_of_current_device() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) return 1;
    if (dev >= 0 && dev < 64) cache[dev].store(v, std::memory_order_relaxed);
    return v;
}

// ------------------------------------------------------------- helpers --

__device__ __forceinline__ float ld_f(const float *p) { return *p; }
__device__ __forceinline__ float ld_f(const __half *p) { return __half2float(*p); }
__device__ __forceinline__ float ld_f(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

// Four consecutive elements widened to fp32 (p 16-byte aligned for float,
// 8-byte aligned for the 16-bit types).
__device__ __forceinline__ float4 ld4(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
__device__ __forceinline__ float4 ld4(const __half *p) {
    uint2 u = *reinterpret_cast<const uint2 *>(p);
    float2 a = __half22float2(*reinterpret_cast<__half2 *>(&u.x));
    float2 b = __half22float2(*reinterpret_cast<__half2 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ float4 ld4(const __nv_bfloat16 *p) {
    uint2 u = *reinterpret_cast<const uint2 *>(p);
    float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&u.x));
    float2 b = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

// Store fp32 as the output type, round-to-nearest-even.
__device__ __forceinline__ void st_out(float *p, float x) { *p = x; }
__device__ __forceinline__ void st_out(__half *p, float x) { *p = __float2half_rn(x); }
__device__ __forceinline__ void st_out(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

// The same, as a volatile read-only load: it is issued where it is written,
// so that a load meant to run ahead of its use is not moved next to it.
__device__ __forceinline__ float ld_gate_early(const void *p, long idx, int dt) {
    if (dt == GDN_F32) {
        float x;
        asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(x) : "l"(reinterpret_cast<const float *>(p) + idx));
        return x;
    }
    unsigned short u;
    asm volatile("ld.global.nc.b16 %0, [%1];" : "=h"(u) : "l"(reinterpret_cast<const unsigned short *>(p) + idx));
    if (dt == GDN_F16) return __half2float(__ushort_as_half(u));
    return __bfloat162float(__ushort_as_bfloat16(u));
}

// Gate value (alpha / beta) of runtime dtype `dt` at element `idx`.
__device__ __forceinline__ float ld_gate(const void *p, long idx, int dt) {
    if (dt == GDN_F32) return reinterpret_cast<const float *>(p)[idx];
    if (dt == GDN_F16) return __half2float(reinterpret_cast<const __half *>(p)[idx]);
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[idx]);
}

// Token range [tok0, tok0 + len) of row b.  With cu_seqlens, T is the
// total token count the host validated the buffers for, and the bounds read
// from the device are clamped to [0, T] so that no access leaves the inputs.
__device__ __forceinline__ void row_range(const int32_t *cu, int b, int T,
                                          long &tok0, int &len) {
    if (cu == nullptr) {
        tok0 = (long)b * T;
        len = T;
        return;
    }
    const long total = T;
    long a = cu[b], e = cu[b + 1];
    a = a < 0 ? 0 : (a > total ? total : a);
    e = e < a ? a : (e > total ? total : e);
    tok0 = a;
    len = (int)(e - a);
}

// Initial-state matrix of (row b, head h) or nullptr for zeros.
__device__ __forceinline__ const float *initial_state_ptr(const float *s0, const int32_t *idx,
                                                          int n_s0, int b, int h, int Hv,
                                                          int dv, int dk, uint32_t *err) {
    if (s0 == nullptr) return nullptr;
    long src = b;
    if (idx != nullptr) {
        src = idx[b];
        if (src < 0 || src >= n_s0) {
            atomicOr(err, (uint32_t)GDN_DEVERR_BAD_INDEX);
            return nullptr;
        }
    }
    return s0 + ((src * Hv + h) * (long)dv) * dk;
}

// Input conventions: the decay and the write strength from the stored gates,
// and the L2-normalisation factor of a q or k vector with squared norm ss.
__device__ __forceinline__ float conv_alpha(float x, int conv) {
    return (conv & GDN_ALPHA_LOG) ? expf(x) : x;
}
__device__ __forceinline__ float conv_log_alpha(float x, int conv) {
    return (conv & GDN_ALPHA_LOG) ? x : logf(x);
}
__device__ __forceinline__ float conv_beta(float x, int conv) {
    return (conv & GDN_BETA_LOGIT) ? 1.0f / (1.0f + expf(-x)) : x;
}
__device__ __forceinline__ float l2norm_factor(float ss) { return rsqrtf(ss + 1e-6f); }

template <int W>
__device__ __forceinline__ float group_sum(float x) {
    // butterfly sum over aligned groups of W lanes (W a power of two <= 32)
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

}  // namespace gdn
