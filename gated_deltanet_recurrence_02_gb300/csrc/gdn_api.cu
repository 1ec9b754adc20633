// gdn_api.cu -- the C ABI of libgdn (include/gdn.h): argument validation,
// buffer-overlap checks and kernel dispatch.  Host code only; every check
// runs before anything is launched, so a rejected call has no side effects.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "gdn_internal.cuh"

namespace gdn {

// The library's device error word (GDN_DEVERR_* bits).  Its device address is
// resolved once per device and handed to kernels in their parameter blocks.
__device__ uint32_t g_device_errors = 0;

namespace {

constexpr int kMaxDevices = 64;
// Per-device cache of the error word's address.  Filled under the mutex by
// the first call on a device; read lock-free afterwards (acquire pairs with
// the release store), so concurrent first calls from several host threads
// are safe.
std::atomic<uint32_t *> g_err_addr[kMaxDevices] = {};
std::mutex g_err_mutex;

cudaError_t error_word(uint32_t **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    uint32_t *a = g_err_addr[dev].load(std::memory_order_acquire);
    if (a == nullptr) {
        std::lock_guard<std::mutex> lock(g_err_mutex);
        a = g_err_addr[dev].load(std::memory_order_relaxed);
        if (a == nullptr) {
            void *ptr = nullptr;
            e = cudaGetSymbolAddress(&ptr, g_device_errors);
            if (e != cudaSuccess) return e;
            a = static_cast<uint32_t *>(ptr);
            g_err_addr[dev].store(a, std::memory_order_release);
        }
    }
    *out = a;
    return cudaSuccess;
}

// Limit of the kernels' waits on work of another warp (see
// gdn_set_wait_limit_ns); the waits for the CTA's own copies in flight keep
// the full limit.
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};

size_t dtype_bytes(int dt) {
    switch (dt) {
        case GDN_F32: return 4;
        case GDN_F16: return 2;
        case GDN_BF16: return 2;
        default: return 0;
    }
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

struct Span {
    const void *p;
    size_t bytes;
    bool is_output;
};

bool overlaps(const Span &a, const Span &b) {
    if (a.p == nullptr || b.p == nullptr || a.bytes == 0 || b.bytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

// GDN_ERR_ALIAS if an output overlaps anything else, except the exact
// in-place pair (same start, same size) `allow_a`/`allow_b` when given.
int check_alias(const Span *s, int n, int allow_a, int allow_b) {
    for (int i = 0; i < n; ++i)
        for (int j = i + 1; j < n; ++j) {
            if (!s[i].is_output && !s[j].is_output) continue;
            if (!overlaps(s[i], s[j])) continue;
            const bool pair = (i == allow_a && j == allow_b) || (i == allow_b && j == allow_a);
            if (pair && s[i].p == s[j].p && s[i].bytes == s[j].bytes) continue;
            return GDN_ERR_ALIAS;
        }
    return GDN_OK;
}

// Splits a dtype argument into the storage type and its convention bits;
// false if it carries bits outside `allowed`.
bool split_dtype(int code, int allowed, int *dt, int *conv) {
    const int flags = code & ~0xFF;
    if (flags & ~allowed) return false;
    *dt = code & 0xFF;
    *conv |= flags;
    return true;
}

bool mul_ok(size_t a, size_t b, size_t *out) {
    if (a != 0 && b > SIZE_MAX / a) return false;
    *out = a * b;
    return true;
}

// Sizes shared by prefill and recurrent calls.
struct Shapes {
    size_t total_T, qk_bytes, v_bytes, gate_bytes, s0_bytes, sf_bytes;
};

int check_common(const void *q, const void *k, const void *v, const void *alpha,
                 const void *beta, const int32_t *cu, const float *s0,
                 const int32_t *s0_idx, int n_s0, const float *sf, const void *out,
                 int B, int T, int Hq, int Hk, int Hv, int dk, int dv, int dt_qkv,
                 int dt_gate, Shapes *sh) {
    if (B < 0 || T < 0 || Hk <= 0 || Hv <= 0 || dk <= 0 || dv <= 0) return GDN_ERR_INVALID_ARG;
    if (Hq != Hk || Hv % Hk != 0) return GDN_ERR_INVALID_ARG;
    if (dtype_bytes(dt_qkv) == 0 || dtype_bytes(dt_gate) == 0) return GDN_ERR_INVALID_ARG;
    if (!(dk == 32 || dk == 64 || dk == 128) || !(dv == 32 || dv == 64 || dv == 128))
        return GDN_ERR_UNSUPPORTED;
    if (B > 65535 || Hv > 65535) return GDN_ERR_UNSUPPORTED;
    size_t total_T = (cu == nullptr) ? (size_t)B * (size_t)T : (size_t)T;
    if (B > 0 && total_T > 0) {
        if (!q || !k || !v || !alpha || !beta || !out) return GDN_ERR_INVALID_ARG;
    }
    if (s0_idx != nullptr && s0 == nullptr) return GDN_ERR_INVALID_ARG;
    if (s0 != nullptr) {
        if (s0_idx == nullptr && n_s0 < B) return GDN_ERR_INVALID_ARG;
        if (n_s0 < 0) return GDN_ERR_INVALID_ARG;
    }
    const void *a16[] = {q, k, v, alpha, beta, out, s0, sf};
    for (const void *p : a16)
        if (p && !aligned(p, 16)) return GDN_ERR_ALIGN;
    if ((cu && !aligned(cu, 4)) || (s0_idx && !aligned(s0_idx, 4))) return GDN_ERR_ALIGN;

    const size_t st = (size_t)Hv * dv * dk * sizeof(float);
    sh->total_T = total_T;
    if (!mul_ok(total_T, (size_t)Hk * dk * dtype_bytes(dt_qkv), &sh->qk_bytes)) return GDN_ERR_INVALID_ARG;
    if (!mul_ok(total_T, (size_t)Hv * dv * dtype_bytes(dt_qkv), &sh->v_bytes)) return GDN_ERR_INVALID_ARG;
    if (!mul_ok(total_T, (size_t)Hv * dtype_bytes(dt_gate), &sh->gate_bytes)) return GDN_ERR_INVALID_ARG;
    sh->s0_bytes = s0 ? (size_t)(s0_idx ? n_s0 : (n_s0 > B ? n_s0 : B)) * st : 0;
    sh->sf_bytes = sf ? (size_t)B * st : 0;
    return GDN_OK;
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" {

const char *gdn_status_string(int status) {
    switch (status) {
        case GDN_OK: return "ok";
        case GDN_ERR_INVALID_ARG: return "invalid argument";
        case GDN_ERR_UNSUPPORTED: return "unsupported size, chunk or dtype";
        case GDN_ERR_ALIAS: return "an output buffer overlaps another buffer";
        case GDN_ERR_ALIGN: return "misaligned pointer";
        case GDN_ERR_CUDA: return "CUDA launch or runtime error";
        case GDN_ERR_TIMEOUT: return "a kernel abandoned a bounded wait";
        case GDN_ERR_WORKSPACE: return "workspace missing or too small";
        default: return "unknown status";
    }
}

int gdn_recurrent_capture(const void *q, const void *k, const void *v, const void *alpha,
                          const void *beta, const int32_t *cu_seqlens,
                          const float *initial_state, const int32_t *initial_state_indices,
                          int num_initial_states, float *final_state, void *out, int B, int T,
                          int Hq, int Hk, int Hv, int dk, int dv, float scale, int dtype_qkv,
                          int dtype_gate, int state_update_capacity,
                          const int32_t *capture_count, const int32_t *state_update_active,
                          float *state_update, void *stream) {
    int conv = 0, dtq = 0, dtg = 0;
    if (!split_dtype(dtype_qkv, GDN_QK_L2NORM, &dtq, &conv) ||
        !split_dtype(dtype_gate, GDN_ALPHA_LOG | GDN_BETA_LOGIT, &dtg, &conv))
        return GDN_ERR_INVALID_ARG;
    dtype_qkv = dtq;
    dtype_gate = dtg;
    Shapes sh;
    int st = check_common(q, k, v, alpha, beta, cu_seqlens, initial_state, initial_state_indices,
                          num_initial_states, final_state, out, B, T, Hq, Hk, Hv, dk, dv,
                          dtype_qkv, dtype_gate, &sh);
    if (st != GDN_OK) return st;
    const int cap = state_update_capacity;
    if (cap < 0) return GDN_ERR_INVALID_ARG;
    if (cap > 0 && (capture_count == nullptr || state_update == nullptr)) return GDN_ERR_INVALID_ARG;
    if (state_update && !aligned(state_update, 16)) return GDN_ERR_ALIGN;
    if ((capture_count && !aligned(capture_count, 4)) ||
        (state_update_active && !aligned(state_update_active, 4)))
        return GDN_ERR_ALIGN;
    if (final_state != nullptr && final_state == initial_state && initial_state_indices != nullptr)
        return GDN_ERR_ALIAS;
    size_t su_bytes = 0;
    if (cap > 0 && !mul_ok((size_t)B * cap, GDN_STATE_UPDATE_SLOT(Hk, Hv, dk, dv) * sizeof(float), &su_bytes))
        return GDN_ERR_INVALID_ARG;
    const size_t sf_in_place = (final_state == initial_state) ? sh.sf_bytes : 0;
    Span spans[] = {
        {q, sh.qk_bytes, false},                        // 0
        {k, sh.qk_bytes, false},                        // 1
        {v, sh.v_bytes, false},                         // 2
        {alpha, sh.gate_bytes, false},                  // 3
        {beta, sh.gate_bytes, false},                   // 4
        {cu_seqlens, cu_seqlens ? (size_t)(B + 1) * 4 : 0, false},
        {initial_state, sf_in_place ? sf_in_place : sh.s0_bytes, false},  // 6
        {initial_state_indices, initial_state_indices ? (size_t)B * 4 : 0, false},
        {capture_count, cap > 0 ? (size_t)B * 4 : 0, false},
        {state_update_active, state_update_active ? 4u : 0u, false},
        {final_state, sh.sf_bytes, true},               // 10
        {out, sh.v_bytes, true},
        {state_update, su_bytes, true},
    };
    st = check_alias(spans, (int)(sizeof(spans) / sizeof(spans[0])), 6, 10);
    if (st != GDN_OK) return st;
    if (B == 0) return GDN_OK;

    RecurrentParams p{};
    p.q = q; p.k = k; p.v = v; p.alpha = alpha; p.beta = beta;
    p.cu_seqlens = cu_seqlens;
    p.s0 = initial_state; p.s0_idx = initial_state_indices; p.n_s0 = num_initial_states;
    p.s_final = final_state; p.out = out;
    p.B = B; p.T = T; p.Hk = Hk; p.Hv = Hv; p.dk = dk; p.dv = dv;
    p.scale = scale; p.dt_qkv = dtype_qkv; p.dt_gate = dtype_gate; p.conv = conv;
    p.capacity = cap; p.capture_count = capture_count; p.active = state_update_active;
    p.su = cap > 0 ? state_update : nullptr;
    p.rp_su = nullptr; p.rp_capacity = 0; p.rp_accepted = nullptr; p.s_commit = nullptr;
    p.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    if (error_word(&p.err) != cudaSuccess) return GDN_ERR_CUDA;
    return launch_recurrent(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int gdn_replay_verify(const void *q, const void *k, const void *v, const void *alpha,
                      const void *beta, const int32_t *cu_seqlens, const float *state_in,
                      float *state_out, const float *prev_state_update, int prev_capacity,
                      const int32_t *accepted_count, float *draft_final_state, void *out, int B,
                      int T, int Hq, int Hk, int Hv, int dk, int dv, float scale, int dtype_qkv,
                      int dtype_gate, int state_update_capacity, const int32_t *capture_count,
                      const int32_t *state_update_active, float *state_update, void *stream) {
    int conv = 0, dtq = 0, dtg = 0;
    if (!split_dtype(dtype_qkv, GDN_QK_L2NORM, &dtq, &conv) ||
        !split_dtype(dtype_gate, GDN_ALPHA_LOG | GDN_BETA_LOGIT, &dtg, &conv))
        return GDN_ERR_INVALID_ARG;
    dtype_qkv = dtq;
    dtype_gate = dtg;
    Shapes sh;
    int st = check_common(q, k, v, alpha, beta, cu_seqlens, state_in, nullptr, B, draft_final_state,
                          out, B, T, Hq, Hk, Hv, dk, dv, dtype_qkv, dtype_gate, &sh);
    if (st != GDN_OK) return st;
    const int cap = state_update_capacity;
    if (cap < 0 || prev_capacity < 0) return GDN_ERR_INVALID_ARG;
    if (cap > 0 && (capture_count == nullptr || state_update == nullptr)) return GDN_ERR_INVALID_ARG;
    if (prev_capacity > 0 && (prev_state_update == nullptr || accepted_count == nullptr))
        return GDN_ERR_INVALID_ARG;
    if (B > 0 && state_out == nullptr) return GDN_ERR_INVALID_ARG;
    if ((state_out && !aligned(state_out, 16)) || (state_update && !aligned(state_update, 16)) ||
        (prev_state_update && !aligned(prev_state_update, 16)))
        return GDN_ERR_ALIGN;
    if ((capture_count && !aligned(capture_count, 4)) ||
        (state_update_active && !aligned(state_update_active, 4)) ||
        (accepted_count && !aligned(accepted_count, 4)))
        return GDN_ERR_ALIGN;
    const size_t slot_bytes = GDN_STATE_UPDATE_SLOT(Hk, Hv, dk, dv) * sizeof(float);
    size_t su_bytes = 0, prev_bytes = 0;
    if (cap > 0 && !mul_ok((size_t)B * cap, slot_bytes, &su_bytes)) return GDN_ERR_INVALID_ARG;
    if (prev_capacity > 0 && !mul_ok((size_t)B * prev_capacity, slot_bytes, &prev_bytes))
        return GDN_ERR_INVALID_ARG;
    const size_t sbytes = (size_t)B * Hv * dv * dk * sizeof(float);
    Span spans[] = {
        {q, sh.qk_bytes, false},                        // 0
        {k, sh.qk_bytes, false},                        // 1
        {v, sh.v_bytes, false},                         // 2
        {alpha, sh.gate_bytes, false},                  // 3
        {beta, sh.gate_bytes, false},                   // 4
        {cu_seqlens, cu_seqlens ? (size_t)(B + 1) * 4 : 0, false},
        {state_in, state_in ? sbytes : 0, false},       // 6
        {prev_state_update, prev_bytes, false},
        {accepted_count, prev_capacity > 0 ? (size_t)B * 4 : 0, false},
        {capture_count, cap > 0 ? (size_t)B * 4 : 0, false},
        {state_update_active, state_update_active ? 4u : 0u, false},
        {state_out, sbytes, true},                      // 11
        {draft_final_state, sh.sf_bytes, true},
        {out, sh.v_bytes, true},
        {state_update, su_bytes, true},
    };
    st = check_alias(spans, (int)(sizeof(spans) / sizeof(spans[0])), 6, 11);
    if (st != GDN_OK) return st;
    if (B == 0) return GDN_OK;

    RecurrentParams p{};
    p.q = q; p.k = k; p.v = v; p.alpha = alpha; p.beta = beta;
    p.cu_seqlens = cu_seqlens;
    p.s0 = state_in; p.s0_idx = nullptr; p.n_s0 = B;
    p.s_final = draft_final_state; p.out = out;
    p.B = B; p.T = T; p.Hk = Hk; p.Hv = Hv; p.dk = dk; p.dv = dv;
    p.scale = scale; p.dt_qkv = dtype_qkv; p.dt_gate = dtype_gate; p.conv = conv;
    p.capacity = cap; p.capture_count = capture_count; p.active = state_update_active;
    p.su = cap > 0 ? state_update : nullptr;
    p.rp_su = prev_capacity > 0 ? prev_state_update : nullptr;
    p.rp_capacity = prev_capacity;
    p.rp_accepted = prev_capacity > 0 ? accepted_count : nullptr;
    p.s_commit = state_out;
    p.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    if (error_word(&p.err) != cudaSuccess) return GDN_ERR_CUDA;
    return launch_recurrent(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

int gdn_replay_state_updates(const float *state_in, float *state_out, const float *state_update,
                             int state_update_capacity, const int32_t *accepted_count, int B,
                             int Hk, int Hv, int dk, int dv, void *stream) {
    if (B < 0 || Hk <= 0 || Hv <= 0 || dk <= 0 || dv <= 0 || Hv % Hk != 0) return GDN_ERR_INVALID_ARG;
    if (state_update_capacity < 0) return GDN_ERR_INVALID_ARG;
    if (!(dk == 32 || dk == 64 || dk == 128) || !(dv == 32 || dv == 64 || dv == 128))
        return GDN_ERR_UNSUPPORTED;
    if (B > 65535 || Hv > 65535) return GDN_ERR_UNSUPPORTED;
    if (B > 0 && (!state_in || !state_out || !accepted_count)) return GDN_ERR_INVALID_ARG;
    if (B > 0 && state_update_capacity > 0 && !state_update) return GDN_ERR_INVALID_ARG;
    if ((state_in && !aligned(state_in, 16)) || (state_out && !aligned(state_out, 16)) ||
        (state_update && !aligned(state_update, 16)) ||
        (accepted_count && !aligned(accepted_count, 4)))
        return GDN_ERR_ALIGN;
    const size_t sbytes = (size_t)B * Hv * dv * dk * sizeof(float);
    const size_t su_bytes = (size_t)B * state_update_capacity *
                            GDN_STATE_UPDATE_SLOT(Hk, Hv, dk, dv) * sizeof(float);
    Span spans[] = {
        {state_in, sbytes, false},
        {state_update, su_bytes, false},
        {accepted_count, (size_t)B * 4, false},
        {state_out, sbytes, true},
    };
    int st = check_alias(spans, 4, 0, 3);
    if (st != GDN_OK) return st;
    if (B == 0) return GDN_OK;
    ReplayParams p{};
    p.s_in = state_in; p.s_out = state_out; p.su = state_update;
    p.capacity = state_update_capacity; p.accepted = accepted_count;
    p.B = B; p.Hk = Hk; p.Hv = Hv; p.dk = dk; p.dv = dv;
    p.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    if (error_word(&p.err) != cudaSuccess) return GDN_ERR_CUDA;
    return launch_replay(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

size_t gdn_prefill_workspace_size(int B, int T, int Hk, int Hv, int dk, int dv, int chunk,
                                  int dtype_qkv, int varlen) {
    // the storage type decides; the GDN_QK_L2NORM convention bit changes nothing here
    int conv = 0, dt = 0;
    if (!split_dtype(dtype_qkv, GDN_QK_L2NORM, &dt, &conv)) return (size_t)-1;
    if (B < 0 || T < 0 || Hk <= 0 || Hv <= 0 || dk <= 0 || dv <= 0 || chunk <= 0 || dtype_bytes(dt) == 0)
        return (size_t)-1;
    if (prefill_tc_supported(dk, dv, chunk, dt)) return prefill_tc_workspace_bytes(B, T, Hk, Hv, varlen != 0);
    return 0;
}

void gdn_set_wait_limit_ns(uint64_t ns) {
    g_wait_ns.store(ns == 0 ? kDefaultWaitNs : ns, std::memory_order_relaxed);
}

}  // extern "C"

namespace {

// Every prefill entry point: validation, overlap checks, then one of the two
// prefill kernels.  Checkpoints and capture are optional extras.
int prefill_call(const void *q, const void *k, const void *v, const void *alpha, const void *beta,
                 const int32_t *cu_seqlens, const float *initial_state,
                 const int32_t *initial_state_indices, int num_initial_states, float *final_state,
                 void *out, int B, int T, int Hq, int Hk, int Hv, int dk, int dv, int chunk,
                 float scale, int dtype_qkv, int dtype_gate, float *checkpoints,
                 int checkpoint_capacity, int checkpoint_interval, int capacity,
                 const int32_t *capture_count, const int32_t *state_update_active,
                 float *state_update, void *workspace, size_t workspace_bytes, void *stream) {
    int conv = 0, dtq = 0, dtg = 0;
    if (!split_dtype(dtype_qkv, GDN_QK_L2NORM, &dtq, &conv) ||
        !split_dtype(dtype_gate, GDN_ALPHA_LOG | GDN_BETA_LOGIT, &dtg, &conv))
        return GDN_ERR_INVALID_ARG;
    dtype_qkv = dtq;
    dtype_gate = dtg;
    Shapes sh;
    int st = check_common(q, k, v, alpha, beta, cu_seqlens, initial_state, initial_state_indices,
                          num_initial_states, final_state, out, B, T, Hq, Hk, Hv, dk, dv,
                          dtype_qkv, dtype_gate, &sh);
    if (st != GDN_OK) return st;
    if (!(chunk == 16 || chunk == 32 || chunk == 64)) return GDN_ERR_UNSUPPORTED;
    const bool use_tc = prefill_tc_supported(dk, dv, chunk, dtype_qkv);
    if (!use_tc && !prefill_simt_supported(dk, dv, chunk)) return GDN_ERR_UNSUPPORTED;
    if (final_state != nullptr && final_state == initial_state && initial_state_indices != nullptr)
        return GDN_ERR_ALIAS;
    const size_t need =
        gdn_prefill_workspace_size(B, T, Hk, Hv, dk, dv, chunk, dtype_qkv, cu_seqlens != nullptr);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return GDN_ERR_WORKSPACE;
    if (workspace && !aligned(workspace, 16)) return GDN_ERR_ALIGN;
    if (checkpoint_capacity < 0 || checkpoint_interval < 1) return GDN_ERR_INVALID_ARG;
    if (checkpoint_capacity > 0 && checkpoints == nullptr) return GDN_ERR_INVALID_ARG;
    if (checkpoints && !aligned(checkpoints, 16)) return GDN_ERR_ALIGN;
    size_t ck_bytes = 0;
    if (checkpoint_capacity > 0 &&
        !mul_ok((size_t)B * checkpoint_capacity, (size_t)Hv * dv * dk * sizeof(float), &ck_bytes))
        return GDN_ERR_INVALID_ARG;
    if (capacity < 0) return GDN_ERR_INVALID_ARG;
    if (capacity > 0 && (capture_count == nullptr || state_update == nullptr)) return GDN_ERR_INVALID_ARG;
    if (state_update && !aligned(state_update, 16)) return GDN_ERR_ALIGN;
    if ((capture_count && !aligned(capture_count, 4)) ||
        (state_update_active && !aligned(state_update_active, 4)))
        return GDN_ERR_ALIGN;
    size_t su_bytes = 0;
    if (capacity > 0 &&
        !mul_ok((size_t)B * capacity, GDN_STATE_UPDATE_SLOT(Hk, Hv, dk, dv) * sizeof(float), &su_bytes))
        return GDN_ERR_INVALID_ARG;
    const size_t sf_in_place = (final_state == initial_state) ? sh.sf_bytes : 0;
    Span spans[] = {
        {q, sh.qk_bytes, false},
        {k, sh.qk_bytes, false},
        {v, sh.v_bytes, false},
        {alpha, sh.gate_bytes, false},
        {beta, sh.gate_bytes, false},
        {cu_seqlens, cu_seqlens ? (size_t)(B + 1) * 4 : 0, false},
        {initial_state, sf_in_place ? sf_in_place : sh.s0_bytes, false},  // 6
        {initial_state_indices, initial_state_indices ? (size_t)B * 4 : 0, false},
        {capture_count, capacity > 0 ? (size_t)B * 4 : 0, false},
        {state_update_active, (capacity > 0 && state_update_active) ? 4u : 0u, false},
        {final_state, sh.sf_bytes, true},                                  // 10
        {out, sh.v_bytes, true},
        {workspace, need, true},
        {checkpoints, ck_bytes, true},
        {state_update, su_bytes, true},
    };
    st = check_alias(spans, (int)(sizeof(spans) / sizeof(spans[0])), 6, 10);
    if (st != GDN_OK) return st;
    if (B == 0) return GDN_OK;

    PrefillParams p{};
    p.q = q; p.k = k; p.v = v; p.alpha = alpha; p.beta = beta;
    p.cu_seqlens = cu_seqlens;
    p.s0 = initial_state; p.s0_idx = initial_state_indices; p.n_s0 = num_initial_states;
    p.s_final = final_state; p.out = out;
    p.B = B; p.T = T; p.Hk = Hk; p.Hv = Hv; p.dk = dk; p.dv = dv; p.chunk = chunk;
    p.scale = scale; p.dt_qkv = dtype_qkv; p.dt_gate = dtype_gate; p.conv = conv;
    p.ws = workspace; p.ws_bytes = workspace_bytes;
    p.ckpt = checkpoint_capacity > 0 ? checkpoints : nullptr;
    p.ckpt_cap = checkpoint_capacity; p.ckpt_every = checkpoint_interval;
    p.capacity = capacity;
    p.capture_count = capacity > 0 ? capture_count : nullptr;
    p.active = capacity > 0 ? state_update_active : nullptr;
    p.su = capacity > 0 ? state_update : nullptr;
    p.chunk_table = nullptr;  // set by the tensor-core launcher for packed rows
    p.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    if (error_word(&p.err) != cudaSuccess) return GDN_ERR_CUDA;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t e = use_tc ? launch_prefill_tc(p, s) : launch_prefill_simt(p, s);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

extern "C" {

int gdn_prefill_chunked(const void *q, const void *k, const void *v, const void *alpha,
                        const void *beta, const int32_t *cu_seqlens, const float *initial_state,
                        const int32_t *initial_state_indices, int num_initial_states,
                        float *final_state, void *out, int B, int T, int Hq, int Hk, int Hv,
                        int dk, int dv, int chunk, float scale, int dtype_qkv, int dtype_gate,
                        void *workspace, size_t workspace_bytes, void *stream) {
    return prefill_call(q, k, v, alpha, beta, cu_seqlens, initial_state, initial_state_indices,
                        num_initial_states, final_state, out, B, T, Hq, Hk, Hv, dk, dv, chunk,
                        scale, dtype_qkv, dtype_gate, nullptr, 0, 1, 0, nullptr, nullptr, nullptr,
                        workspace, workspace_bytes, stream);
}

int gdn_prefill_chunked_checkpoints(const void *q, const void *k, const void *v,
                                    const void *alpha, const void *beta,
                                    const int32_t *cu_seqlens, const float *initial_state,
                                    const int32_t *initial_state_indices, int num_initial_states,
                                    float *final_state, void *out, int B, int T, int Hq, int Hk,
                                    int Hv, int dk, int dv, int chunk, float scale, int dtype_qkv,
                                    int dtype_gate, float *checkpoints, int checkpoint_capacity,
                                    int checkpoint_interval, void *workspace,
                                    size_t workspace_bytes, void *stream) {
    return prefill_call(q, k, v, alpha, beta, cu_seqlens, initial_state, initial_state_indices,
                        num_initial_states, final_state, out, B, T, Hq, Hk, Hv, dk, dv, chunk,
                        scale, dtype_qkv, dtype_gate, checkpoints, checkpoint_capacity,
                        checkpoint_interval, 0, nullptr, nullptr, nullptr, workspace,
                        workspace_bytes, stream);
}

int gdn_prefill_chunked_capture(const void *q, const void *k, const void *v, const void *alpha,
                                const void *beta, const int32_t *cu_seqlens,
                                const float *initial_state, const int32_t *initial_state_indices,
                                int num_initial_states, float *final_state, void *out, int B, int T,
                                int Hq, int Hk, int Hv, int dk, int dv, int chunk, float scale,
                                int dtype_qkv, int dtype_gate, int state_update_capacity,
                                const int32_t *capture_count, const int32_t *state_update_active,
                                float *state_update, void *workspace, size_t workspace_bytes,
                                void *stream) {
    return prefill_call(q, k, v, alpha, beta, cu_seqlens, initial_state, initial_state_indices,
                        num_initial_states, final_state, out, B, T, Hq, Hk, Hv, dk, dv, chunk,
                        scale, dtype_qkv, dtype_gate, nullptr, 0, 1, state_update_capacity,
                        capture_count, state_update_active, state_update, workspace,
                        workspace_bytes, stream);
}

int gdn_device_errors(void *stream, uint32_t *flags) {
    if (flags == nullptr) return GDN_ERR_INVALID_ARG;
    *flags = 0;
    uint32_t *addr = nullptr;
    if (error_word(&addr) != cudaSuccess) return GDN_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_CUDA;
    uint32_t host = 0;
    if (cudaMemcpy(&host, addr, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess) return GDN_ERR_CUDA;
    const uint32_t zero = 0;
    if (cudaMemcpy(addr, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return GDN_ERR_CUDA;
    *flags = host;
    return (host & GDN_DEVERR_TIMEOUT) ? GDN_ERR_TIMEOUT : GDN_OK;
}

}  // extern "C"
