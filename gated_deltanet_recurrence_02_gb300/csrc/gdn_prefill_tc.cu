// gdn_prefill_tc.cu -- chunked prefill on the 5th-generation tensor cores
// (tcgen05 MMA, TMEM accumulators, TMA), for dk = dv = 128, chunk 64, bf16 or
// fp16 inputs.
//
// "Enable the native Kev example on NVIDIA GPUs through ExecuTorch's AOTI CUDA
// backend" (executorch issue 23097), work list: a chunked GDN prefill with an
// explicit initial and final state and an FP32 recurrence under 16-bit
// weights.  Chunk form (per chunk of n <= 64 tokens, start state S0, local
// log-decay sums g_t, gamma_t = e^{g_t}, w_t = e^{g_last - g_t}):
//   A[t][i] = beta_t e^{g_t - g_i} k_t.k_i (i < t),   T = (I + A)^{-1}
//   U = T diag(beta) V,   W = T diag(beta gamma) K,   P'[t][i] = e^{g_t - g_i} q_t.k_i (i <= t)
//   Delta = U - W S0^T
//   O     = diag(gamma) Q S0^T + P' Delta   (Q: scale * q; the scale is folded into
//                                           P' and into the gamma of the output)
//   S_end = gamma_last S0 + Delta^T diag(w) K
//
// Phase A (prefill_intra_kernel, one CTA per (chunk, value head), all chunks in
// parallel): [K;Q] K^T on the tensor cores, A and P' from it, T by a blocked
// (16 x 16 tiles) unit-lower-triangular inverse in fp32, then U and W on the
// tensor cores with T rounded to the 16-bit input type (its rounding is of
// the same size as the rounding of U and W themselves).  V is loaded into
// Q's shared-memory slot once [K;Q]K^T has consumed Q; 71 KB of shared
// memory and 128 TMEM columns per CTA let three CTAs share an SM.  Writes W,
// P' and U as ready-made shared-memory operand images plus gamma / w into
// the workspace.
//
// Phase B (prefill_carry_kernel, one CTA per (value head, 32-row dv tile,
// row), serial over chunks; a 64-row-tile instance with a two-stage ring
// takes over when the 32-row grid is larger than the SM count, where
// throughput rather than the chain's latency decides; it is launched as a
// programmatic dependent of phase A): per chunk two dependent tensor-core
// steps,
//   D1 = [Q; W] S^T                       (M=128: Q S^T and W S^T at once)
//   Delta = U - (W S^T)                   (threads, fp32)
//   D2 = K^T diag(w) Delta,  D3 = P' Delta (tensor cores)
//   S <- gamma_last S + D2,  O = gamma (Q S^T) + D3
// The state tile lives in fp32 registers (thread j owns column j of S, i.e.
// row j of S^T, for half of the tile's rows) and is re-packed to bf16/fp16 in
// shared memory as the next chunk's MMA operand.  Chunk operands stream in
// through a TMA / bulk-copy ring, with L2 prefetches further
// ahead; the output MMA (P' Delta) is committed separately so the state
// update never waits for it, and the next chunk's first MMA is issued as soon
// as the state image is written.  At a requested chunk boundary the fp32
// state in the registers is also streamed out as a checkpoint.  Capture: the
// rows of Delta are the tokens' deltas, so the carry phase writes the first
// n_b tokens' deltas and phase A their decay and shared key (and clears the
// whole buffer while capture is inactive).
//
// Ragged chunks: tokens t >= n get alpha = 1 and beta = 0, which makes their
// rows of T the identity rows and their U, W, Delta rows zero, so whatever the
// loads bring into those rows (zeros past the end of the tensor, the next row's
// tokens otherwise) never reaches S or a stored output.  Precondition: every
// alpha in (0, 1].
//
// Every mbarrier wait is bounded; on timeout the CTA raises
// GDN_DEVERR_TIMEOUT, waits (bounded) for its copies in flight, releases its
// TMEM and exits.
#include <cstring>
#include <mutex>

#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int C = 64;    // chunk
constexpr int D = 128;   // dk = dv
constexpr uint64_t kWaitNs = kDefaultWaitNs;  // drains of the CTA's own copies

// Workspace record per (chunk, value head), bytes.
constexpr uint32_t REC_W = 0;         // W image: 2 SW128 blocks (dk 0-63, 64-127) x 64 rows
constexpr uint32_t REC_P = 16384;     // P' image: 1 SW128 block, 64 rows
constexpr uint32_t REC_U = 24576;     // U: 4 dv tiles of [64 t][32 i], 4 KB each
constexpr uint32_t REC_VEC = 40960;   // gamma[64], w[64], gamma_last
constexpr uint32_t REC_BYTES = 41984;

template <typename E>
struct Elem;
template <>
struct Elem<__nv_bfloat16> {
    static constexpr bool kBf16 = true;
    __device__ static uint32_t pack2(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __device__ static float2 unpack2(uint32_t u) {
        return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&u));
    }
    __device__ static float round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }
};
template <>
struct Elem<__half> {
    static constexpr bool kBf16 = false;
    __device__ static uint32_t pack2(float a, float b) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __device__ static float2 unpack2(uint32_t u) { return __half22float2(*reinterpret_cast<__half2 *>(&u)); }
    __device__ static float round(float x) { return __half2float(__float2half_rn(x)); }
};

// Eight fp32 values -> eight 16-bit elements in one 16-byte vector.
template <typename E>
__device__ __forceinline__ uint4 pack8(const float *v) {
    return make_uint4(Elem<E>::pack2(v[0], v[1]), Elem<E>::pack2(v[2], v[3]), Elem<E>::pack2(v[4], v[5]),
                      Elem<E>::pack2(v[6], v[7]));
}
template <typename E>
__device__ __forceinline__ void unpack8(uint4 u, float *v) {
    float2 a = Elem<E>::unpack2(u.x), b = Elem<E>::unpack2(u.y), c = Elem<E>::unpack2(u.z),
           d = Elem<E>::unpack2(u.w);
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y; v[4] = c.x; v[5] = c.y; v[6] = d.x; v[7] = d.y;
}

// Byte offset of the 16-byte chunk holding elements [8*q, 8*q+8) of row r.
__device__ __forceinline__ uint32_t sw128_chunk(int r, int q) {
    return (uint32_t)(r * 128 + (((q ^ (r & 7)) & 7) << 4));
}
// Same for the 64-byte rows of a 32-column U tile (chunks swizzled by row % 4).
__device__ __forceinline__ uint32_t u32_chunk(int r, int q) {
    return (uint32_t)(r * 64 + (((q ^ (r & 3)) & 3) << 4));
}

// ---- chunk bookkeeping ------------------------------------------------------

__device__ __forceinline__ int n_chunks(int len) { return (len + C - 1) / C; }

// Bytes at the head of the workspace that hold the per-row chunk table
// (packed rows only).
__host__ __device__ constexpr size_t chunk_table_bytes(int B) { return ((size_t)(B + 1) * 4 + 1023) / 1024 * 1024; }

// First global chunk index of row b (uniform rows: b * chunks per row; packed
// rows: the table).
__device__ __forceinline__ long chunk_base(const PrefillParams &p, int b) {
    if (p.chunk_table == nullptr) return (long)b * n_chunks(p.T);
    return p.chunk_table[b];
}

// Global chunk index -> (row, chunk in row); false past the last chunk.  With
// packed rows a binary search over the table (rows without chunks have equal
// neighbouring entries and are skipped by taking the last row that starts at
// or before gc).
__device__ __forceinline__ bool chunk_of(const PrefillParams &p, long gc, int &b, int &c) {
    if (p.chunk_table == nullptr) {
        const int nc = n_chunks(p.T);
        if (nc == 0) return false;
        b = (int)(gc / nc);
        c = (int)(gc % nc);
        return b < p.B;
    }
    const int32_t *tbl = p.chunk_table;
    if (gc >= tbl[p.B]) return false;
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tbl[mid] <= gc) lo = mid; else hi = mid - 1;
    }
    b = lo;
    c = (int)(gc - tbl[lo]);
    return true;
}

// The records follow the chunk table (if any) in the workspace.
__device__ __forceinline__ uint8_t *records(const PrefillParams &p) {
    return reinterpret_cast<uint8_t *>(p.ws) + (p.chunk_table ? chunk_table_bytes(p.B) : 0);
}

// Prologue for packed rows: table[b] = chunks of rows 0 .. b-1 (table[0] = 0,
// table[B] = all chunks), one CTA scanning the rows 1024 at a time.
__global__ void __launch_bounds__(1024) chunk_table_kernel(const int32_t *cu, int B, int T, int32_t *table) {
    __shared__ int32_t warp_incl[32];
    __shared__ int32_t carry;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        carry = 0;
        table[0] = 0;
    }
    __syncthreads();
    for (int r0 = 0; r0 < B; r0 += 1024) {
        const int r = r0 + tid;
        int x = 0;
        if (r < B) {
            long tok0;
            int len;
            row_range(cu, r, T, tok0, len);
            x = n_chunks(len);
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_incl[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = warp_incl[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            warp_incl[lane] = w;
        }
        __syncthreads();
        const int incl = carry + (warp ? warp_incl[warp - 1] : 0) + x;
        if (r < B) table[r + 1] = incl;
        __syncthreads();
        if (tid == 1023) carry = incl;
        __syncthreads();
    }
}

struct TcMaps {
    CUtensorMap q, k, v;
};

// ============================================================ phase A ====

constexpr uint32_t A_KQ = 0;          // [K;Q] image, 2 K-blocks of 128 rows (32 KB); V replaces Q
constexpr uint32_t A_V0 = 8192;       //   V dv 0-63 (rows of the first K-block's Q half)
constexpr uint32_t A_V1 = 24576;      //   V dv 64-127 (second K-block's Q half)
constexpr uint32_t A_IMG = 32768;     // [T*beta ; T*beta*gamma] bf16 image (16 KB) ...
constexpr uint32_t A_AT = A_IMG;      //   ... aliasing, before it exists, A^T fp32 [64][68]
constexpr uint32_t A_X = A_IMG + 64 * 68 * 4;  //   and the blocked-inverse scratch, 3 x 16 x 16 fp32
constexpr uint32_t A_T = A_X + 3 * 256 * 4;    // T fp32 [64][68]
constexpr uint32_t A_VEC = A_T + 64 * 68 * 4;  // g, beta, gamma, 1/|k|, 1/|q|: 5 x 64 floats
constexpr uint32_t A_BAR = A_VEC + 1536;
constexpr uint32_t A_SMEM = A_BAR + 64 + 1024;  // + alignment slack
constexpr uint32_t A_TMEM_COLS = 128;
constexpr int LD = 68;                           // fp32 row stride of A^T and T

// T = (I + A)^{-1} for the strictly lower 64 x 64 matrix A (A[r][c] = At[c*LD + r]),
// blocked in 16 x 16 tiles: the four diagonal tiles D_J = (I + A_JJ)^{-1} by
// forward substitution, then the off-diagonal tiles by increasing distance,
// T_JI = -D_J (sum_{I <= K < J} A_JK T_KI).  In the level stages each thread
// computes a 1 x 4 piece of a tile (row r, columns c0 .. c0 + 3), fed by one
// float4 of T per step, with four partial sums; the diagonal solves load each
// row of A one step ahead.  256 threads; T written to sT.
constexpr int kIntraThreads = 256;
__device__ __forceinline__ void blocked_unit_lower_inverse(const float *At, float *sT, float *X, int tid) {
    if (tid < 64) {
        const int bb = tid >> 4, cl = tid & 15, o = 16 * bb;
        float acc[16], row[16];  // row: A[o+t][o+r], loaded one step ahead
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            acc[r] = 0.f;
            row[r] = At[o * LD + o + r];
        }
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            float nxt[16];
            if (t + 1 < 16) {
#pragma unroll
                for (int r = 0; r < 16; ++r) nxt[r] = (r > t + 1) ? At[(o + t + 1) * LD + o + r] : 0.f;
            }
            const float x = (t < cl) ? 0.f : ((t == cl) ? 1.f : -acc[t]);
            sT[(o + t) * LD + o + cl] = x;
#pragma unroll
            for (int r = t + 1; r < 16; ++r) acc[r] = fmaf(row[r], x, acc[r]);
            if (t + 1 < 16) {
#pragma unroll
                for (int r = 0; r < 16; ++r) row[r] = nxt[r];
            }
        }
    } else {
        // zero the tiles above the diagonal
        for (int e = tid - 64; e < 6 * 64; e += kIntraThreads - 64) {
            const int blk = e >> 6, r = (e >> 2) & 15, c4 = (e & 3) * 4;
            const int I = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
            const int J = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
            *reinterpret_cast<float4 *>(sT + (16 * I + r) * LD + 16 * J + c4) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    __syncthreads();
    // four partial sums per dot product (independent chains hide the
    // shared-memory latency), added at the end
    auto sum4 = [](const float4 (&a)[4]) {
        return make_float4((a[0].x + a[1].x) + (a[2].x + a[3].x), (a[0].y + a[1].y) + (a[2].y + a[3].y),
                           (a[0].z + a[1].z) + (a[2].z + a[3].z), (a[0].w + a[1].w) + (a[2].w + a[3].w));
    };
    const int q = tid & 63, r = q >> 2, c0 = (q & 3) * 4;
#pragma unroll
    for (int d = 1; d < 4; ++d) {
        const int nb = 4 - d;
        const int blk = tid >> 6, I = blk, J = blk + d;
        if (blk < nb) {
            float4 a[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) a[u] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int kk = 0; kk < d; ++kk) {
                const int K = I + kk;
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const float x = At[(16 * K + m) * LD + 16 * J + r];
                    const float4 t4 = *reinterpret_cast<const float4 *>(sT + (16 * K + m) * LD + 16 * I + c0);
                    float4 &acc = a[m & 3];
                    acc.x = fmaf(x, t4.x, acc.x); acc.y = fmaf(x, t4.y, acc.y);
                    acc.z = fmaf(x, t4.z, acc.z); acc.w = fmaf(x, t4.w, acc.w);
                }
            }
            *reinterpret_cast<float4 *>(X + blk * 256 + r * 16 + c0) = sum4(a);
        }
        __syncthreads();
        if (blk < nb) {
            float4 a[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) a[u] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const float dd = sT[(16 * J + r) * LD + 16 * J + m];
                const float4 x4 = *reinterpret_cast<const float4 *>(X + blk * 256 + m * 16 + c0);
                float4 &acc = a[m & 3];
                acc.x = fmaf(dd, x4.x, acc.x); acc.y = fmaf(dd, x4.y, acc.y);
                acc.z = fmaf(dd, x4.z, acc.z); acc.w = fmaf(dd, x4.w, acc.w);
            }
            const float4 s4 = sum4(a);
            *reinterpret_cast<float4 *>(sT + (16 * J + r) * LD + 16 * I + c0) = make_float4(-s4.x, -s4.y, -s4.z, -s4.w);
        }
        __syncthreads();
    }
}

// XO: the call also writes capture or checkpoints; NORM: q and k are
// L2-normalised in the kernel.  Separate instances, so that the plain prefill
// carries none of that code.  The norms enter as per-token scalars:
// A gets r_t r_i, P' rq_t r_i, the W image beta gamma r, and the record's
// gamma (output) and w (state update) rq_t and r_t, with r = 1/|k|, rq = 1/|q|.
template <typename E, bool XO, bool NORM>
__global__ void __launch_bounds__(kIntraThreads, 3)
prefill_intra_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap mq,
                     const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sKQ = sm + A_KQ;
    uint8_t *sImg = sm + A_IMG;
    float *At = reinterpret_cast<float *>(sm + A_AT);
    float *X = reinterpret_cast<float *>(sm + A_X);
    float *sT = reinterpret_cast<float *>(sm + A_T);
    float *vg = reinterpret_cast<float *>(sm + A_VEC);
    float *vbeta = vg + 64, *vgam = vg + 128, *vkn = vg + 192, *vqn = vg + 256;
    uint64_t *bar_ld = reinterpret_cast<uint64_t *>(sm + A_BAR);
    uint64_t *bar_mma = bar_ld + 1;
    uint64_t *bar_v = bar_ld + 2;
    uint32_t *slot = reinterpret_cast<uint32_t *>(bar_ld + 3);

    // the carry kernel may start its prologue once every CTA here has started
    grid_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.y, Hv = p.Hv, Hk = p.Hk;
    const int hk = h / (Hv / Hk);
    int b, c;
    if (!chunk_of(p, blockIdx.x, b, c)) return;
    long rtok0;
    int len;
    row_range(p.cu_seqlens, b, p.T, rtok0, len);
    const long tok0 = rtok0 + (long)c * C;
    const int n = min(C, len - c * C);
    uint8_t *rec = records(p) + ((size_t)(chunk_base(p, b) + c) * Hv + h) * REC_BYTES;

    if (tid == 0) {
        prefetch_tensormap(&mq);
        prefetch_tensormap(&mk);
        prefetch_tensormap(&mv);
        mbar_init(bar_ld, 1);
        mbar_init(bar_mma, 1);
        mbar_init(bar_v, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0) {
        tmem_alloc(slot, A_TMEM_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_arrive_expect_tx(bar_ld, 32768);
        tma_load_3d(sKQ, &mk, 0, hk, (int)tok0, bar_ld);
        tma_load_3d(sKQ + 16384, &mk, 64, hk, (int)tok0, bar_ld);
        tma_load_3d(sKQ + 8192, &mq, 0, hk, (int)tok0, bar_ld);
        tma_load_3d(sKQ + 24576, &mq, 64, hk, (int)tok0, bar_ld);
    }
    // capture: clear the whole buffer when inactive (every CTA a share), else
    // this chunk's captured tokens' decay and (once per key head) shared key;
    // their deltas come from the carry phase
    const long su_slot = (long)Hv + (long)Hk * D + (long)Hv * D;
    int ncap = 0;
    float *su0 = nullptr;
    if constexpr (XO) {
        prefill_capture_clear(p, su_slot, (long)blockIdx.y * gridDim.x + blockIdx.x,
                              (long)gridDim.x * gridDim.y, tid, kIntraThreads);
        ncap = prefill_ncap(p, b, len) - c * C;
        if (ncap > 0) su0 = p.su + ((long)b * p.capacity + (long)c * C) * su_slot;
    }
    if (tid < C) {
        const long gi = (tok0 + tid) * Hv + h;
        const float a = (tid < n) ? ld_gate(p.alpha, gi, p.dt_gate) : 0.f;
        vg[tid] = (tid < n) ? conv_log_alpha(a, p.conv) : 0.f;
        vbeta[tid] = (tid < n) ? conv_beta(ld_gate(p.beta, gi, p.dt_gate), p.conv) : 0.f;
        if (tid < ncap) su0[tid * su_slot + h] = conv_alpha(a, p.conv);
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = *slot;
    const uint32_t lane_base = tbase + ((uint32_t)(32 * (warp & 3)) << 16);
    const bool kbf = Elem<E>::kBf16;
    bool ok = true;
    if (tid == 0) {
        // [K; Q] K^T -> TMEM cols [0, 64): rows 0-63 K K^T, rows 64-127 Q K^T
        ok = mbar_wait(bar_ld, 0, p.wait_ns);
        if (ok) {
            fence_after_sync();
            const uint64_t d0 = desc_sw128(smem_u32(sKQ), 16, 1024);
            const uint32_t id = idesc_f16(128, 64, false, false, kbf);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint64_t d = desc_add(d0, (k >> 2) * 16384 + (k & 3) * 32);
                mma_f16(tbase, d, d, id, k > 0);
            }
            mma_commit(bar_mma);
        }
    }
    // warp 1: cumulative log-decay g, gamma, w while the MMA runs
    float g0 = 0.f, g1 = 0.f, w0 = 0.f, w1 = 0.f, glast = 0.f;
    if (warp == 1) {
        float x0 = vg[lane], x1 = vg[lane + 32];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            float y0 = __shfl_up_sync(0xffffffffu, x0, o);
            float y1 = __shfl_up_sync(0xffffffffu, x1, o);
            if (lane >= o) { x0 += y0; x1 += y1; }
        }
        x1 += __shfl_sync(0xffffffffu, x0, 31);
        glast = __shfl_sync(0xffffffffu, x1, 31);
        g0 = expf(x0); g1 = expf(x1); w0 = expf(glast - x0); w1 = expf(glast - x1);
        vg[lane] = x0;
        vg[lane + 32] = x1;
        vgam[lane] = g0; vgam[lane + 32] = g1;
    }
    // record: gamma for the output gamma (scale q) S^T, w for the state update
    float *rv = reinterpret_cast<float *>(rec + REC_VEC);
    if constexpr (NORM) {
        // 1/|k_t| and 1/|q_t| from the staged tiles (rows 0-63 K, 64-127 Q;
        // two threads per row, one per 64-column block), before V replaces Q
        if (!mbar_wait(bar_ld, 0, p.wait_ns)) ok = false;
        const int r = tid >> 1, kb = tid & 1;
        float ss = 0.f;
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) {
            float x[8];
            unpack8<E>(*reinterpret_cast<const uint4 *>(sKQ + kb * 16384 + sw128_chunk(r, q8)), x);
#pragma unroll
            for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
        }
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        if (kb == 0) (r < C ? vkn[r] : vqn[r - C]) = l2norm_factor(ss);
        __syncthreads();
        if (warp == 1) {
            rv[lane] = p.scale * g0 * vqn[lane]; rv[lane + 32] = p.scale * g1 * vqn[lane + 32];
            rv[64 + lane] = w0 * vkn[lane]; rv[96 + lane] = w1 * vkn[lane + 32];
            if (lane == 0) rv[128] = expf(glast);
        }
    } else {
        if (warp == 1) {
            rv[lane] = p.scale * g0; rv[lane + 32] = p.scale * g1; rv[64 + lane] = w0; rv[96 + lane] = w1;
            if (lane == 0) rv[128] = expf(glast);
        }
    }
    __syncthreads();
    if (ncap > 0 && h % (Hv / Hk) == 0) {
        // captured keys: the (normalised) key the recurrence used
        const E *kg = reinterpret_cast<const E *>(p.k);
        const int nk = ncap < n ? ncap : n;
        for (int e = tid; e < nk * D; e += kIntraThreads) {
            const int t = e / D, j = e % D;
            su0[t * su_slot + Hv + (long)hk * D + j] =
                ld_f(kg + ((tok0 + t) * Hk + hk) * D + j) * (NORM ? vkn[t] : 1.f);
        }
    }
    ok = ok && mbar_wait(bar_mma, 0, p.wait_ns);
    fence_after_sync();
    const bool v_issued = ok;  // the same for every thread (ok is uniform after the wait)
    if (ok && tid == 0) {
        // Q has been consumed: V takes its place (the load overlaps A, P' and T)
        mbar_arrive_expect_tx(bar_v, 16384);
        tma_load_3d(sm + A_V0, &mv, 0, h, (int)tok0, bar_v);
        tma_load_3d(sm + A_V1, &mv, 64, h, (int)tok0, bar_v);
    }
    if (ok) {
        // warp w reads TMEM lane quarter (w % 4); warps w and w + 4 split the 64 columns
        const int quarter = warp & 3, half = warp >> 2;
        if (quarter < 2) {
            // A, stored transposed: At[i][t] = A[t][i] = beta_t e^{g_t - g_i} k_t.k_i  (i < t)
            const int t = 32 * quarter + lane;
            const float gt = vg[t], bt = vbeta[t] * (NORM ? vkn[t] : 1.f);
            float v[32];
            tmem_ld32(lane_base + 32 * half, v);
#pragma unroll
            for (int ii = 0; ii < 32; ++ii) {
                const int i = 32 * half + ii;
                At[i * LD + t] = (i < t) ? bt * __expf(gt - vg[i]) * (NORM ? v[ii] * vkn[i] : v[ii]) : 0.f;
            }
        } else {
            // P'[t][i] = e^{g_t - g_i} (scale q_t).k_i (i <= t), image straight to the workspace
            const int t = 32 * (quarter - 2) + lane;
            const float gt = vg[t], sc = p.scale * (NORM ? vqn[t] : 1.f);
            uint8_t *dst = rec + REC_P;
            float v[32];
            tmem_ld32(lane_base + 32 * half, v);
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8) {
                float pv[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int i = 32 * half + 8 * q8 + e;
                    pv[e] = (i <= t) ? __expf(gt - vg[i]) * (sc * (NORM ? v[8 * q8 + e] * vkn[i] : v[8 * q8 + e]))
                                     : 0.f;
                }
                *reinterpret_cast<uint4 *>(dst + sw128_chunk(t, 4 * half + q8)) = pack8<E>(pv);
            }
        }
    }
    __syncthreads();

    // ---- T = (I + A)^{-1}
    if (ok) blocked_unit_lower_inverse(At, sT, X, tid);
    else {
        __syncthreads(); __syncthreads(); __syncthreads(); __syncthreads(); __syncthreads(); __syncthreads();
        __syncthreads();
    }

    // ---- operand image [T diag(beta) ; T diag(beta gamma)] in the 16-bit input type
    if (ok) {
        const int t = tid & 63, which = (tid >> 6) & 1, part = tid >> 7, r = which * 64 + t;
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
            const int q8 = 4 * part + qq;
            float val[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int s = 8 * q8 + e;
                val[e] = sT[t * LD + s] * (which ? vbeta[s] * vgam[s] * (NORM ? vkn[s] : 1.f) : vbeta[s]);
            }
            *reinterpret_cast<uint4 *>(sImg + sw128_chunk(r, q8)) = pack8<E>(val);
        }
    }
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();

    // ---- U = [T b ; T b g] V (rows 0-63 used) -> TMEM cols [0, 128)
    if (ok && tid == 0) {
        fence_after_sync();
        ok = mbar_wait(bar_v, 0, p.wait_ns);
        if (ok) {
            const uint64_t a0 = desc_sw128(smem_u32(sImg), 16, 1024), b0 = desc_sw128(smem_u32(sm + A_V0), 16384, 1024);
            const uint32_t id = idesc_f16(128, 128, false, true, kbf);
#pragma unroll
            for (int k = 0; k < 4; ++k) mma_f16(tbase, desc_add(a0, k * 32), desc_add(b0, k * 2048), id, k > 0);
            mma_commit(bar_mma);
        }
    }
    ok = ok && mbar_wait(bar_mma, 1, p.wait_ns);
    fence_after_sync();
    if (ok && (warp & 3) < 2) {
        // U as four thread-read tiles of 32 dv columns: [64 t][32 i], 16-byte chunks swizzled by t
        const int t = 32 * (warp & 3) + lane, half = warp >> 2;
#pragma unroll
        for (int qq = 0; qq < 2; ++qq) {
            const int q4 = 2 * half + qq;
            float v[32];
            tmem_ld32(lane_base + 32 * q4, v);
            uint8_t *dst = rec + REC_U + q4 * 4096;
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8)
                *reinterpret_cast<uint4 *>(dst + u32_chunk(t, q8)) = pack8<E>(v + 8 * q8);
        }
    }
    fence_before_sync();
    __syncthreads();

    // ---- W = [T b ; T b g] K (rows 64-127 used) -> TMEM cols [0, 128)
    if (ok && tid == 0) {
        fence_after_sync();
        const uint64_t a0 = desc_sw128(smem_u32(sImg), 16, 1024), b0 = desc_sw128(smem_u32(sKQ), 16384, 1024);
        const uint32_t id = idesc_f16(128, 128, false, true, kbf);
#pragma unroll
        for (int k = 0; k < 4; ++k) mma_f16(tbase, desc_add(a0, k * 32), desc_add(b0, k * 2048), id, k > 0);
        mma_commit(bar_mma);
    }
    ok = ok && mbar_wait(bar_mma, 0, p.wait_ns);
    fence_after_sync();
    if (ok && (warp & 3) >= 2) {
        const int t = 32 * ((warp & 3) - 2) + lane, half = warp >> 2;
#pragma unroll
        for (int qq = 0; qq < 2; ++qq) {
            const int q4 = 2 * half + qq;
            float v[32];
            tmem_ld32(lane_base + 32 * q4, v);
            uint8_t *dst = rec + REC_W + (q4 >> 1) * 8192;
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8)
                *reinterpret_cast<uint4 *>(dst + sw128_chunk(t, (q4 & 1) * 4 + q8)) = pack8<E>(v + 8 * q8);
        }
    }
    if (!ok) {
        if (tid == 0) atomicOr(p.err, (uint32_t)GDN_DEVERR_TIMEOUT);
        // copies in flight must land before the CTA exits
        mbar_wait(bar_ld, 0, kWaitNs);
        if (v_issued) mbar_wait(bar_v, 0, kWaitNs);
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, A_TMEM_COLS);
}

// ============================================================ phase B ====

// One carry CTA owns TV rows of one (row, value head) state: TV = 32 (the
// latency instance: the most CTAs, three stages) or TV = 64 (the throughput
// instance, for grids of many rows: twice the work per MMA for about the same
// issue time, two stages).
template <int TV>
struct CarryCfg {
    static constexpr int kCols = TV / 2;             // state columns per compute thread
    static constexpr int NS = TV == 32 ? 3 : 2;      // stages in the ring
    static constexpr uint32_t ST_A1 = 0;             // [Q ; W] image, 2 K-blocks of 128 rows
    static constexpr uint32_t ST_K = 32768;          // K image, 2 dk blocks of 64 rows
    static constexpr uint32_t ST_P = 49152;          // P' image (rows 0-63 of the [P'; X] operand)
    static constexpr uint32_t ST_U = 57344;          // U tiles, TV / 32 of [64 t][32 i]
    static constexpr uint32_t kUBytes = TV * 128;
    static constexpr uint32_t ST_VEC = ST_U + kUBytes;  // gamma, w, gamma_last
    static constexpr uint32_t ST_BYTES = ST_VEC + 1024;
    static constexpr uint32_t B_S = NS * ST_BYTES;   // S^T image (MN-major, 128 K-rows, TV N used)
    static constexpr uint32_t B_DW = B_S + 16384;    // diag(w) Delta image (64 K-rows)
    static constexpr uint32_t B_DD = B_DW + 8192;    // Delta image
    static constexpr uint32_t B_BAR = B_DD + 8192;
    static constexpr uint32_t B_SMEM = B_BAR + 128 + 1024;
    static constexpr uint32_t STAGE_TX = 16384 + 16384 + 16384 + 8192 + kUBytes + 1024;
    // TMEM columns: D1 = [Q; W] S^T at 0 / TV (by chunk parity), D2 = K^T w Delta
    // at 2 TV, D3 = P' Delta at 3 TV / 4 TV (by chunk parity)
    static constexpr uint32_t T_D2 = 2 * TV, T_D3 = 3 * TV;
    static constexpr uint32_t T_COLS = TV == 32 ? 256 : 512;
    static_assert(B_SMEM <= 232448, "carry CTA exceeds the shared memory of an SM");
};
// 8 compute warps: warp w reads TMEM lane quarter w % 4, warps w and w + 4
// split the tile's TV columns.  Warp 8 issues every MMA; warp 9 refills the
// stage ring, each stage once the output MMA of its chunk has retired (that
// MMA's commit arrives on the stage's `empty` barrier).
constexpr int kCarryComputeWarps = 8;
constexpr int kIssuerWarp = kCarryComputeWarps;          // issues every MMA
constexpr int kCopierWarp = kCarryComputeWarps + 1;      // issues every copy; no named barriers
constexpr int kCarryThreads = (kCarryComputeWarps + 2) * 32;
constexpr int kBarThreads = (kCarryComputeWarps + 1) * 32;  // compute warps + issuer
constexpr uint32_t kBarDelta = 1;  // named barrier: Delta images written (all warps)
constexpr uint32_t kBarState = 2;  // named barrier: S image written (all warps)

// The calling warp's N consecutive TMEM columns (N = 16 or 32), see tmem_ld16.
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[N]) {
    if constexpr (N == 16) tmem_ld16(taddr, v);
    else tmem_ld32(taddr, v);
}

template <typename E, bool XO, int TV>
__global__ void __launch_bounds__(kCarryThreads, 1)
prefill_carry_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap mq,
                     const __grid_constant__ CUtensorMap mk) {
    using Cfg = CarryCfg<TV>;
    constexpr int NS = Cfg::NS, NC = Cfg::kCols, Q8 = NC / 8;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sS = sm + Cfg::B_S, *sDw = sm + Cfg::B_DW, *sDd = sm + Cfg::B_DD;
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + Cfg::B_BAR);  // [NS]
    uint64_t *empty = full + NS;                                       // [NS]
    uint64_t *bar1 = full + 2 * NS, *bar2 = bar1 + 1, *bar3 = bar1 + 2;
    uint32_t *slot = reinterpret_cast<uint32_t *>(bar1 + 3);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = (warp >> 2) & 1;
    const int vt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int Hv = p.Hv, Hk = p.Hk;
    const int hk = h / (Hv / Hk);
    const int i0 = vt * TV;
    long rtok0;
    int len;
    row_range(p.cu_seqlens, b, p.T, rtok0, len);
    const int nc = n_chunks(len);
    const long su_slot = (long)Hv + (long)Hk * D + (long)Hv * D;
    const int ncap = XO ? prefill_ncap(p, b, len) : 0;
    const uint8_t *rec0 = records(p) + (size_t)chunk_base(p, b) * Hv * REC_BYTES +
                          (size_t)h * REC_BYTES;
    const size_t rec_stride = (size_t)Hv * REC_BYTES;

    if (tid == 0) {
        if (nc > 0) {  // with no token at all the maps are left unencoded
            prefetch_tensormap(&mq);
            prefetch_tensormap(&mk);
        }
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(bar1, 1);
        mbar_init(bar2, 1);
        mbar_init(bar3, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0) {
        tmem_alloc(slot, Cfg::T_COLS);
        tmem_relinquish();
    }
    const bool kbf = Elem<E>::kBf16;
    bool ok = true;

    if (warp == kCopierWarp) {
        // ======================= copier warp ============================
        auto issue_stage = [&](int cc) {
            const int s = cc % NS;
            uint8_t *st = sm + s * Cfg::ST_BYTES;
            const uint8_t *rec = rec0 + (size_t)cc * rec_stride;
            const int t0 = (int)(rtok0 + (long)cc * C);
            mbar_arrive_expect_tx(&full[s], Cfg::STAGE_TX);
            tma_load_3d(st + Cfg::ST_A1, &mq, 0, hk, t0, &full[s]);
            tma_load_3d(st + Cfg::ST_A1 + 16384, &mq, 64, hk, t0, &full[s]);
            bulk_load(st + Cfg::ST_A1 + 8192, rec + REC_W, 8192, &full[s]);
            bulk_load(st + Cfg::ST_A1 + 24576, rec + REC_W + 8192, 8192, &full[s]);
            tma_load_3d(st + Cfg::ST_K, &mk, 0, hk, t0, &full[s]);
            tma_load_3d(st + Cfg::ST_K + 8192, &mk, 64, hk, t0, &full[s]);
            bulk_load(st + Cfg::ST_P, rec + REC_P, 8192, &full[s]);
            bulk_load(st + Cfg::ST_U, rec + REC_U + vt * Cfg::kUBytes, Cfg::kUBytes, &full[s]);
            bulk_load(st + Cfg::ST_VEC, rec + REC_VEC, 1024, &full[s]);
        };
        auto prefetch_chunk = [&](int cc) {
            const uint8_t *rec = rec0 + (size_t)cc * rec_stride;
            const int t0 = (int)(rtok0 + (long)cc * C);
            tma_prefetch_l2_3d(&mq, 0, hk, t0);
            tma_prefetch_l2_3d(&mq, 64, hk, t0);
            tma_prefetch_l2_3d(&mk, 0, hk, t0);
            tma_prefetch_l2_3d(&mk, 64, hk, t0);
            bulk_prefetch_l2(rec + REC_W, 16384 + 8192);
            bulk_prefetch_l2(rec + REC_U + vt * Cfg::kUBytes, Cfg::kUBytes);
            bulk_prefetch_l2(rec + REC_VEC, 1024);
        };
        if (lane == 0) {
            grid_dependency_wait();  // the records are the chunk-parallel kernel's output
            for (int cc = 0; cc < NS && cc < nc; ++cc) issue_stage(cc);
            for (int cc = NS; cc < NS + 2 && cc < nc; ++cc) prefetch_chunk(cc);
            for (int cc = NS; cc < nc; ++cc) {
                // chunk cc reuses the stage of chunk cc - NS
                if (!mbar_wait(&empty[cc % NS], (cc / NS - 1) & 1, p.wait_ns)) {
                    ok = false;
                    break;
                }
                issue_stage(cc);
                if (cc + 2 < nc) prefetch_chunk(cc + 2);
            }
        }
    } else if (warp == kIssuerWarp) {
        // ======================= issuer warp ============================
        fence_before_sync();
        named_bar(kBarState, kBarThreads);  // initial S image written
        fence_after_sync();
        const uint32_t tbase = *slot;
        const uint32_t id1 = idesc_f16(128, TV, false, true, kbf);
        const uint32_t id2 = idesc_f16(128, TV, true, true, kbf);
        const uint32_t id3 = idesc_f16(128, TV, false, true, kbf);
        const uint64_t bS0 = desc_sw128(smem_u32(sS), 8192, 1024);
        const uint64_t bDw0 = desc_sw128(smem_u32(sDw), 8192, 1024);
        const uint64_t bDd0 = desc_sw128(smem_u32(sDd), 8192, 1024);
        for (int cc = 0; cc < nc; ++cc) {
            const int s = cc % NS;
            uint8_t *st = sm + s * Cfg::ST_BYTES;
            if (lane == 0) {
                ok = mbar_wait(&full[s], (cc / NS) & 1, p.wait_ns);
                if (ok) {
                    // D1 = [Q; W] S^T
                    const uint64_t a0 = desc_sw128(smem_u32(st + Cfg::ST_A1), 16, 1024);
                    const uint32_t d1 = (cc & 1) ? (uint32_t)TV : 0u;
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mma_f16(tbase + d1, desc_add(a0, (k >> 2) * 16384 + (k & 3) * 32), desc_add(bS0, k * 2048),
                                id1, k > 0);
                    mma_commit(bar1);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            fence_before_sync();
            named_bar(kBarDelta, kBarThreads);  // Delta images written
            fence_after_sync();
            if (lane == 0 && ok) {
                const uint64_t k0 = desc_sw128(smem_u32(st + Cfg::ST_K), 8192, 1024);
                const uint64_t p0 = desc_sw128(smem_u32(st + Cfg::ST_P), 16, 1024);
                const uint32_t d3 = Cfg::T_D3 + ((cc & 1) ? (uint32_t)TV : 0u);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_f16(tbase + Cfg::T_D2, desc_add(k0, k * 2048), desc_add(bDw0, k * 2048), id2, k > 0);
                mma_commit(bar2);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_f16(tbase + d3, desc_add(p0, k * 32), desc_add(bDd0, k * 2048), id3, k > 0);
                mma_commit(bar3);
                mma_commit(&empty[s]);  // every MMA reading this chunk's stage has retired
            }
            fence_before_sync();
            named_bar(kBarState, kBarThreads);  // S image written
            fence_after_sync();
        }
        if (lane == 0 && nc > 0) {
            // drain: the last output MMA and any copy still in flight
            mbar_wait(bar3, (nc - 1) & 1, kWaitNs);
        }
    } else {
        // ======================= compute warps ==========================
        // state tile: thread (quarter, lane) owns dk row j = 32 * quarter + lane of
        // S^T for the NC columns [NC * half, NC * half + NC) of the tile
        const int j = 32 * quarter + lane;
        const int c0 = NC * half;
        float S[NC];
        const float *s0 = initial_state_ptr(p.s0, p.s0_idx, p.n_s0, b, h, Hv, D, D, p.err);
#pragma unroll
        for (int i = 0; i < NC; ++i) S[i] = s0 ? s0[(size_t)(i0 + c0 + i) * D + j] : 0.f;
#pragma unroll
        for (int q8 = 0; q8 < Q8; ++q8)
            *reinterpret_cast<uint4 *>(sS + sw128_chunk(j, c0 / 8 + q8)) = pack8<E>(S + 8 * q8);
        fence_proxy_async();
        grid_dependency_wait();  // global writes below follow the chunk-parallel kernel's
        fence_before_sync();
        named_bar(kBarState, kBarThreads);
        fence_after_sync();
        const uint32_t tbase = *slot;
        const uint32_t lane_base = tbase + ((uint32_t)(32 * quarter) << 16);
        E *ob = reinterpret_cast<E *>(p.out);

        for (int cc = 0; cc < nc; ++cc) {
            const int s = cc % NS;
            uint8_t *st = sm + s * Cfg::ST_BYTES;
            const uint32_t d1 = (cc & 1) ? (uint32_t)TV : 0u;
            const uint32_t d3 = Cfg::T_D3 + ((cc & 1) ? (uint32_t)TV : 0u);
            const int n = min(C, len - cc * C);
            if (ok) ok = mbar_wait(&full[s], (cc / NS) & 1, p.wait_ns);
            const float *vec = reinterpret_cast<const float *>(st + Cfg::ST_VEC);
            const float gC = ok ? vec[128] : 0.f;
            if (quarter >= 2) {
                // Delta = U - W S^T for token t, NC of the TV columns
                const int t = 32 * (quarter - 2) + lane;
                const float wt = ok ? vec[64 + t] : 0.f;
                if (ok) ok = mbar_wait(bar1, cc & 1, p.wait_ns);
                if (ok) {
                    fence_after_sync();
                    float ws[NC];
                    tmem_ld_cols<NC>(lane_base + d1 + c0, ws);
                    // captured tokens: Delta's row t is token t's delta
                    float *cap = (cc * C + t < ncap)
                                     ? p.su + ((size_t)b * p.capacity + cc * C + t) * su_slot + Hv + (size_t)Hk * D +
                                           (size_t)h * D + i0 + c0
                                     : nullptr;
#pragma unroll
                    for (int q8 = 0; q8 < Q8; ++q8) {
                        // column c0 + 8 q8 of the tile: U tile (c / 32), chunk (c % 32) / 8
                        const int c = c0 + 8 * q8;
                        const uint8_t *su = st + Cfg::ST_U + (c >> 5) * 4096;
                        float u[8], dd[8], dw[8];
                        unpack8<E>(*reinterpret_cast<const uint4 *>(su + u32_chunk(t, (c & 31) >> 3)), u);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            dd[e] = u[e] - ws[8 * q8 + e];
                            dw[e] = wt * dd[e];
                        }
                        *reinterpret_cast<uint4 *>(sDd + sw128_chunk(t, c >> 3)) = pack8<E>(dd);
                        *reinterpret_cast<uint4 *>(sDw + sw128_chunk(t, c >> 3)) = pack8<E>(dw);
                        if (cap != nullptr)
#pragma unroll
                            for (int e = 0; e < 8; ++e) cap[8 * q8 + e] = dd[e];
                    }
                    fence_proxy_async();
                }
            }
            const float gt = (quarter < 2 && ok) ? vec[32 * quarter + lane] : 0.f;
            fence_before_sync();
            named_bar(kBarDelta, kBarThreads);
            fence_after_sync();
            // S <- gamma_last S + K^T diag(w) Delta   (TMEM lane j = dk index)
            if (ok) ok = mbar_wait(bar2, cc & 1, p.wait_ns);
            if (ok) {
                fence_after_sync();
                float v[NC];
                tmem_ld_cols<NC>(lane_base + Cfg::T_D2 + c0, v);
#pragma unroll
                for (int i = 0; i < NC; ++i) S[i] = fmaf(gC, S[i], v[i]);
#pragma unroll
                for (int q8 = 0; q8 < Q8; ++q8)
                    *reinterpret_cast<uint4 *>(sS + sw128_chunk(j, c0 / 8 + q8)) = pack8<E>(S + 8 * q8);
                fence_proxy_async();
                if constexpr (XO) {
                    // chunk-boundary checkpoint: the fp32 state after this chunk
                    const int ck = ckpt_slot(p, cc, len);
                    if (ck >= 0) {
                        float *dst = p.ckpt + ((((size_t)b * p.ckpt_cap + ck) * Hv + h) * D + i0 + c0) * D;
#pragma unroll
                        for (int i = 0; i < NC; ++i) __stcs(dst + (size_t)i * D + j, S[i]);
                    }
                }
            }
            fence_before_sync();
            named_bar(kBarState, kBarThreads);
            fence_after_sync();
            if (quarter < 2 && ok) {
                // O = gamma_t (Q S^T) + P' Delta for token t, NC columns
                const int t = 32 * quarter + lane;
                ok = mbar_wait(bar3, cc & 1, p.wait_ns);
                if (ok) {
                    fence_after_sync();
                    float qs[NC], pd[NC];
                    tmem_ld_cols<NC>(lane_base + d1 + c0, qs);
                    tmem_ld_cols<NC>(lane_base + d3 + c0, pd);
                    if (t < n) {
                        E *dst = ob + ((rtok0 + (long)cc * C + t) * Hv + h) * (long)D + i0 + c0;
#pragma unroll
                        for (int q8 = 0; q8 < Q8; ++q8) {
                            float o[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) o[e] = fmaf(gt, qs[8 * q8 + e], pd[8 * q8 + e]);
                            *reinterpret_cast<uint4 *>(dst + 8 * q8) = pack8<E>(o);
                        }
                    }
                }
            }
        }
        if (ok && p.s_final != nullptr) {
            float *sf = p.s_final + (((size_t)b * Hv + h) * D + i0 + c0) * D;
#pragma unroll
            for (int i = 0; i < NC; ++i) sf[(size_t)i * D + j] = S[i];
        }
    }
    if (!ok && tid == 0) atomicOr(p.err, (uint32_t)GDN_DEVERR_TIMEOUT);
    fence_before_sync();
    __syncthreads();
    if (!ok && tid == 0)
        for (int s = 0; s < NS; ++s) mbar_wait(&full[s], 0, kWaitNs / 8);  // copies must land first
    __syncthreads();
    if (warp == 0) tmem_dealloc(*slot, Cfg::T_COLS);
}

// ============================================================== host =====

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// [total_T, H, 128] 16-bit tensor, box {64 features, 1 head, 64 tokens}, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *ptr, int H, long total_T, bool bf16) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)total_T};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
               const_cast<void *>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename E, bool XO>
cudaError_t launch_e(const PrefillParams &p, long total_T, long max_chunks, cudaStream_t stream) {
    const bool bf = Elem<E>::kBf16;
    CUtensorMap mq, mk, mv;
    memset(&mq, 0, sizeof(mq));
    memset(&mk, 0, sizeof(mk));
    memset(&mv, 0, sizeof(mv));
    // With no tokens at all no chunk exists and the maps are never used.
    if (total_T > 0 && (!make_map(&mq, p.q, p.Hk, total_T, bf) || !make_map(&mk, p.k, p.Hk, total_T, bf) ||
                        !make_map(&mv, p.v, p.Hv, total_T, bf)))
        return cudaErrorInvalidValue;
    const bool norm = (p.conv & GDN_QK_L2NORM) != 0;
    auto intra = norm ? prefill_intra_kernel<E, XO, true> : prefill_intra_kernel<E, XO, false>;
    cudaError_t e = norm ? set_smem_once<prefill_intra_kernel<E, XO, true>>((int)A_SMEM)
                         : set_smem_once<prefill_intra_kernel<E, XO, false>>((int)A_SMEM);
    if (e != cudaSuccess) return e;
    // carry instance: 32-row tiles while one wave of them fits the GPU (the
    // chain's latency decides), 64-row tiles for more rows (throughput decides)
    const bool wide = (long)(D / 32) * p.Hv * p.B > (long)sm_count_of_current_device();
    e = wide ? set_smem_once<prefill_carry_kernel<E, XO, 64>>((int)CarryCfg<64>::B_SMEM)
             : set_smem_once<prefill_carry_kernel<E, XO, 32>>((int)CarryCfg<32>::B_SMEM);
    if (e != cudaSuccess) return e;
    if (max_chunks > 0) {
        dim3 ga((unsigned)max_chunks, p.Hv);
        intra<<<ga, kIntraThreads, A_SMEM, stream>>>(p, mq, mk, mv);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    // The carry kernel is a programmatic dependent of the chunk-parallel one:
    // its prologue (barriers, TMEM, the initial state) overlaps that kernel's
    // tail, and it waits for that kernel's records before reading them.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(D / (wide ? 64 : 32), p.Hv, p.B);
    cfg.blockDim = dim3(kCarryThreads);
    cfg.dynamicSmemBytes = wide ? CarryCfg<64>::B_SMEM : CarryCfg<32>::B_SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = max_chunks > 0 ? 1 : 0;
    return wide ? cudaLaunchKernelEx(&cfg, prefill_carry_kernel<E, XO, 64>, p, mq, mk)
                : cudaLaunchKernelEx(&cfg, prefill_carry_kernel<E, XO, 32>, p, mq, mk);
}

long max_chunks_of(int B, int T, bool varlen) {
    return varlen ? (long)T / C + B : (long)B * ((T + C - 1) / C);
}

}  // namespace

bool prefill_tc_supported(int dk, int dv, int chunk, int dt_qkv) {
    return dk == D && dv == D && chunk == C && (dt_qkv == GDN_BF16 || dt_qkv == GDN_F16);
}

size_t prefill_tc_workspace_bytes(int B, int T, int /*Hk*/, int Hv, bool varlen) {
    return (varlen ? chunk_table_bytes(B) : 0) + (size_t)max_chunks_of(B, T, varlen) * (size_t)Hv * REC_BYTES;
}

cudaError_t launch_prefill_tc(const PrefillParams &p_in, cudaStream_t stream) {
    PrefillParams p = p_in;
    const bool varlen = p.cu_seqlens != nullptr;
    const long total_T = varlen ? (long)p.T : (long)p.B * p.T;
    const long mc = max_chunks_of(p.B, p.T, varlen);
    const bool xo = p.ckpt != nullptr || p.capacity > 0;
    p.chunk_table = nullptr;
    if (varlen && p.B > 0) {
        // packed rows: per-row chunk table at the head of the workspace
        int32_t *tbl = reinterpret_cast<int32_t *>(p.ws);
        chunk_table_kernel<<<1, 1024, 0, stream>>>(p.cu_seqlens, p.B, p.T, tbl);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        p.chunk_table = tbl;
    }
    if (p.dt_qkv == GDN_BF16)
        return xo ? launch_e<__nv_bfloat16, true>(p, total_T, mc, stream)
                  : launch_e<__nv_bfloat16, false>(p, total_T, mc, stream);
    return xo ? launch_e<__half, true>(p, total_T, mc, stream) : launch_e<__half, false>(p, total_T, mc, stream);
}

}  // namespace gdn
