// gdn_prefill_tc.cu -- chunked prefill on the 5th-generation tensor cores
// (tcgen05 MMA, TMEM accumulators, TMA), for dk, dv in {32, 64, 128}, chunk
// 64, bf16 or fp16 inputs.  The kernels work on 128-wide tiles: a smaller
// head is read as zero-padded to 128 (the tensor maps' out-of-bounds fill),
// which changes no product with the real features, and only its real rows
// and columns are written.
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
// Phase A (prefill_intra_kernel, persistent: two CTAs per SM walk the
// (chunk, value head) units, the next unit's tiles in flight while the
// current one is solved): [K;Q] K^T on the tensor cores, A and P' from it,
// then [U | W] = (I + A)^{-1} [diag(beta) V | diag(beta gamma) K] by block
// forward substitution over four 16-token blocks on warp-level MMAs (the
// 16 x 16 diagonal blocks inverted in fp32 by substitution); U, W and P'
// leave as ready-made operand images, staged in shared memory and
// bulk-stored to the workspace with gamma / w.
//
// Phase B (prefill_carry_kernel, one CTA per (value head, 32-row dv tile,
// row), serial over chunks; 128-row-tile (64-row at dv = 64) instances with a
// two-stage ring take over when the 32-row grid is larger than the SM count,
// where throughput rather than the chain's latency decides; it is launched
// as a programmatic dependent of phase A): per chunk two dependent
// tensor-core steps,
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
#include <type_traits>
#include <mutex>

#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int C = 64;    // chunk
constexpr int D = 128;   // tile width of dk and of dv (smaller heads are zero-padded to it)
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
    __device__ static __nv_bfloat16 from(float x) { return __float2bfloat16_rn(x); }
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
    __device__ static __half from(float x) { return __float2half_rn(x); }
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

// 2^x by the PTX ISA's base-2 exponential instruction, flushing subnormal
// results to zero.  Phase A evaluates e^{g_t - g_i} as 2^{(g_t - g_i) log2 e}
// with both terms pre-scaled by log2 e; every argument it keeps is <= 0, so
// the values lie in (0, 1], and results below 2^-126 (flushed) are negligible
// against the other terms.  Its accuracy is covered by the parity tests
// (per chunk and head against the fp64 oracle).  The accurate library paths
// (expf, exp2f) handle subnormals and cost this kernel ~6 us at T=4100.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
constexpr float kLog2e = 1.4426950408889634f;

// The 1024-byte aligned start of a kernel's dynamic shared memory, found by
// pointer arithmetic on the __shared__ array itself: through an integer round
// trip the compiler no longer sees that the pointer, and every pointer derived
// from it, addresses shared memory, and each access becomes a generic one
// (slower, and a measured ~1.3k cycles of every chunk-parallel unit).
__device__ __forceinline__ uint8_t *smem_align1k(uint8_t *raw) {
    return raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
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

// Bytes at the head of the workspace that hold the per-row chunk table and
// the carry's row order (packed rows only): table[B + 1], then order[B].
__host__ __device__ constexpr size_t chunk_table_bytes(int B) { return ((size_t)(2 * B + 1) * 4 + 1023) / 1024 * 1024; }
constexpr int kOrderMaxRows = 1024;  // rows the prologue can sort (one CTA, one row per thread)

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
        // 32-bit division: the launcher keeps every chunk index below 2^31
        const unsigned q = (unsigned)gc / (unsigned)nc;
        b = (int)q;
        c = (int)((unsigned)gc - q * (unsigned)nc);
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
// table[B] = all chunks), one CTA scanning the rows 1024 at a time; then
// order = table + B + 1, the order in which the carry grid takes the rows:
// with `sort` (at most kOrderMaxRows rows) by decreasing chunk count, ties by
// index, else as given.  The carry's CTAs start in grid order as SMs free up,
// so when its grid is a few waves the longest chains start first and the
// short ones fill in behind them, instead of a long row starting last and
// running on alone.
__global__ void __launch_bounds__(1024) chunk_table_kernel(const int32_t *cu, int B, int T, int32_t *table,
                                                           int sort) {
    __shared__ int32_t warp_incl[32];
    __shared__ int32_t carry;
    __shared__ unsigned long long key[kOrderMaxRows];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int my_chunks = 0;  // chunks of row tid (the first pass)
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
        if (r0 == 0) my_chunks = x;
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
    int32_t *order = table + B + 1;
    if (!sort || B > kOrderMaxRows) {
        for (int r = tid; r < B; r += 1024) order[r] = r;
        return;
    }
    // bitonic sort, ascending, of (~chunks, row): decreasing chunk count,
    // ties by increasing row; the slots past B sort last
    key[tid] = tid < B ? ((unsigned long long)(~(uint32_t)my_chunks) << 32) | (uint32_t)tid : ~0ull;
    __syncthreads();
    for (int k = 2; k <= kOrderMaxRows; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            const int l = tid ^ j;
            if (l > tid) {
                const unsigned long long a = key[tid], c = key[l];
                if (((tid & k) == 0) == (a > c)) {
                    key[tid] = c;
                    key[l] = a;
                }
            }
            __syncthreads();
        }
    }
    if (tid < B) order[tid] = (int32_t)(key[tid] & 0xffffffffu);
}

struct TcMaps {
    CUtensorMap q, k, v;
};

// ============================================================ phase A ====
//
// Persistent: a grid of up to two CTAs per SM (256 threads each) walks the
// (chunk, value head) units u = blockIdx.x, blockIdx.x + gridDim.x, ...; unit
// u is global chunk u / Hv of value head u % Hv.  The next unit's K, Q and V
// tiles are issued as soon as the current ones have been read (the current
// unit's right-hand sides are taken into registers at its start, so the copies
// overlap the whole unit) and its gates are loaded into registers one unit
// ahead.  (An L2 prefetch of the unit after it gained nothing at T = 4100 and
// cost 2% on many packed rows.)
//
// Per unit:
//  1. [K;Q] K^T: one tcgen05 MMA group (M = 128) into TMEM.
//  2. From TMEM: -A (16-bit, row-major) and its four 16 x 16 diagonal blocks
//     (fp32); P' as its operand image, staged and bulk-stored to the record.
//     Rows 0-31 of A and of P' go to one warp each (they end at column 31),
//     rows 32-63 to two warps each.
//  3. D_J = (I + A_JJ)^{-1} for the diagonal blocks (fp32 substitution, one
//     block per warp, each column on two lanes), stored 16-bit.
//  4. [U | W] = (I + A)^{-1} [diag(beta) V | diag(beta gamma) K] by block
//     forward substitution over the four 16-token blocks, on warp-level MMAs
//     in registers: each warp owns 32 of the 256 right-hand-side columns and
//     computes, transposed, X_J^T = (R_J^T - sum_{K<J} X_K^T A_JK^T) D_J^T.
//     Operands are 16-bit (the inputs' type) with fp32 accumulation, as the
//     carry phase's own MMAs use.  X_J leaves through stmatrix (transposed)
//     in the record's U tile / W image layout, and is bulk-stored.
// Warp 4, which builds no row of A or P' and handles no gate, issues every
// copy, [K;Q] K^T MMA and U / W store (kIssueThread), so that none of that
// waits on, or delays, the warps on the unit's critical path.  The kernel is
// kept small (one code path for A and P', rolled bounded waits): at 88 KB of
// code its instruction cache missed a third of its fetches.

constexpr uint32_t A_KQ = 0;        // [K;Q] image: K-block 0 (K rows 0-63 | Q rows 64-127), K-block 1 at 16384
constexpr uint32_t A_V = 32768;     // V image: dv 0-63 | 64-127, 8 KB each
constexpr uint32_t A_NA = 49152;    // -A, 16-bit, 64 rows of 128 B, 16-byte chunks swizzled by row % 8
constexpr uint32_t A_AD = A_NA + 8192;            // diagonal blocks, fp32, transposed: [J][col][row], J stride 272
constexpr uint32_t A_D = A_AD + 4 * 272 * 4;      // D_J, 16-bit row-major, 32 B rows (chunks swizzled), 512 B each
constexpr uint32_t A_VEC = A_D + 4 * 512;         // g, beta, beta gamma (r), 1/|k|, 1/|q|, g log2(e): 6 x 64 floats
constexpr uint32_t A_PS = 65536;                  // P' image on its way out (8 KB)
constexpr uint32_t A_US = A_PS + 8192;            // U tiles on their way out (16 KB)
constexpr uint32_t A_WS = A_US + 16384;           // W image on its way out (16 KB)
constexpr uint32_t A_BAR = A_WS + 16384;
constexpr uint32_t A_SMEM = A_BAR + 64 + 1024;    // + alignment slack
constexpr uint32_t A_TMEM_COLS = 128;  // [K;Q] K^T of this unit and of the next, by unit parity
constexpr int kIntraThreads = 256;
constexpr int kIntraCtasPerSm = 2;
constexpr uint32_t kBarDiag01 = 1;    // named barrier: diagonal blocks 0, 1 written (warps 0, 4)
constexpr uint32_t kBarDiag23 = 3;    // named barrier: diagonal blocks 2, 3 written (warps 2, 5, 6)
constexpr uint32_t kBarPImage = 2;    // named barrier of the P' warps (2, 3, 6, 7)
constexpr int kPStoreThread = 64;     // issues (and drains) the P' image stores
constexpr int kIssueThread = 128;     // issues every copy, [K;Q]K^T MMA and U / W record store (warp 4
                                      // builds no row of A / P' and none of the gates)
static_assert(A_VEC + 6 * 256 <= A_PS, "phase A shared-memory layout overlaps");
static_assert(A_SMEM * kIntraCtasPerSm + 2048 <= 232448, "two chunk-parallel CTAs must fit an SM");

// Row r, 16-byte chunk q of -A (rows of 128 B).
__device__ __forceinline__ uint32_t na_off(int r, int q) { return (uint32_t)(r * 128 + (((q ^ r) & 7) << 4)); }
// Row r, 16-byte chunk q (0, 1) of D_J (rows of 32 B).
__device__ __forceinline__ uint32_t d_off(int r, int q) { return (uint32_t)(r * 32 + ((q ^ (r >> 2)) & 1) * 16); }

// D = (I + A_JJ)^{-1} for one 16 x 16 diagonal block (A_JJ strictly lower
// triangular) by forward substitution, (I + A_JJ) x = e_c column by column,
// on one warp: lane (c = lane % 16, h = lane / 16) keeps the partial sums of
// rows 8h .. 8h + 7 of column c, and each x_l of rows 0-7 reaches the lanes
// of rows 8-15 by a shuffle.  Aj[l * 16 + r] = A_JJ[r][l] in fp32, zero for
// r <= l, so every lane adds every column's term.  Each lane's eight values
// of D leave 16-bit, in the D_J layout, once the column is solved.
template <typename E>
__device__ __forceinline__ void solve_diag_block(const float *Aj, uint8_t *Dj, int lane) {
    const int c = lane & 15, h = lane >> 4;
    // this lane's rows of column l of A_JJ, loaded one step ahead of their use
    // (in step order, so that the sixteen columns are never all held in
    // registers at once)
    auto load_col = [&](int l, float (&av)[8]) {
        const uint32_t src = smem_u32(Aj + l * 16 + 8 * h);
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(av[0]), "=f"(av[1]), "=f"(av[2]), "=f"(av[3]) : "r"(src) : "memory");
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(av[4]), "=f"(av[5]), "=f"(av[6]), "=f"(av[7]) : "r"(src + 16) : "memory");
    };
    float acc[8], xs[8], av[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    load_col(0, av);
#pragma unroll
    for (int l = 0; l < 16; ++l) {
        float nx[8];
        if (l + 1 < 16) load_col(l + 1, nx);
        const float own = (l < c) ? 0.f : ((l == c) ? 1.f : -acc[l & 7]);  // D[l][c] in the lanes of row l's half
        const float x = (l < 8) ? __shfl_sync(0xffffffffu, own, c) : own;
        if ((l >> 3) == h) xs[l & 7] = x;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(av[i], x, acc[i]);
        if (l + 1 < 16) {
#pragma unroll
            for (int i = 0; i < 8; ++i) av[i] = nx[i];
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) reinterpret_cast<E *>(Dj + d_off(8 * h + i, c >> 3))[c & 7] = Elem<E>::from(xs[i]);
}

// XO: the call also writes capture or checkpoints; NORM: q and k are
// L2-normalised in the kernel.  Separate instances, so that the plain prefill
// carries none of that code.  The norms enter as per-token scalars:
// A gets r_t r_i, P' rq_t r_i, W's right-hand side beta gamma r, and the
// record's gamma (output) and w (state update) rq_t and r_t, with r = 1/|k|,
// rq = 1/|q|.
template <typename E, bool XO, bool NORM>
__global__ void __launch_bounds__(kIntraThreads, kIntraCtasPerSm)
prefill_intra_kernel(const PrefillParams p, long max_chunks, const __grid_constant__ CUtensorMap mq,
                     const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_align1k(smem_raw);
    uint8_t *sKQ = sm + A_KQ;
    uint8_t *sNA = sm + A_NA;
    float *Adt = reinterpret_cast<float *>(sm + A_AD);
    uint8_t *sD = sm + A_D;
    float *vg = reinterpret_cast<float *>(sm + A_VEC);
    float *vbeta = vg + 64, *vbw = vg + 128, *vkn = vg + 192, *vqn = vg + 256;
    float *vgl = vg + 320;  // g log2(e): e^{g_t - g_i} = 2^{vgl_t - vgl_i}
    uint64_t *bar_kq = reinterpret_cast<uint64_t *>(sm + A_BAR);
    uint64_t *bar_v = bar_kq + 1;
    uint64_t *bar_mma = bar_kq + 2;
    uint32_t *slot = reinterpret_cast<uint32_t *>(bar_kq + 3);

    // the carry kernel may start its prologue once every CTA here has started
    grid_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int Hv = p.Hv, Hk = p.Hk, G = Hv / Hk;
    const int ksteps = p.dk > 64 ? 8 : 4;  // K = 16 steps of the products over dk
    const long su_slot = (long)Hv + (long)Hk * p.dk + (long)Hv * p.dv;
    constexpr bool kbf = Elem<E>::kBf16;
    // L2 priorities: V is read here only; the records are read by the carry
    // kernel next, and the footprint of one call's inputs and records exceeds L2
    const uint64_t pol_read_once = l2_evict_first_policy(), pol_keep = l2_evict_last_policy();

    // Units are (global chunk gc, value head h), unit index gc * Hv + h; this
    // CTA's units advance by gridDim.x, i.e. by (gridDim.x / Hv) chunks and
    // (gridDim.x % Hv) heads (no division inside the loop).
    struct Unit {
        long gc;
        int h;
        bool valid;
        int b, c, n, len;
        long tok0;
    };
    const int step_gc = (int)(gridDim.x / Hv), step_h = (int)(gridDim.x % Hv);
    auto unit_at = [&](long gc, int h) {
        Unit x;
        x.gc = gc;
        x.h = h;
        x.valid = gc < max_chunks && chunk_of(p, gc, x.b, x.c);
        if (x.valid) {
            long rtok0;
            row_range(p.cu_seqlens, x.b, p.T, rtok0, x.len);
            x.tok0 = rtok0 + (long)x.c * C;
            x.n = min(C, x.len - x.c * C);
        }
        return x;
    };
    auto next_unit = [&](const Unit &x) {
        int h = x.h + step_h;
        long gc = x.gc + step_gc;
        if (h >= Hv) {
            h -= Hv;
            gc += 1;
        }
        return unit_at(gc, h);
    };
    // the issuing thread, for a valid unit x: its Q and K tiles (on bar_kq) and
    // its V tiles (on bar_v), once the unit before has no more use for its own
    // (its [K; Q] K^T is done and its right-hand sides are in registers)
    auto issue_q = [&](const Unit &x) {
        const int hk = x.h / G;
        mbar_arrive_expect_tx(bar_kq, 32768);
        tma_load_3d(sKQ + 8192, &mq, 0, hk, (int)x.tok0, bar_kq);
        tma_load_3d(sKQ + 24576, &mq, 64, hk, (int)x.tok0, bar_kq);
    };
    auto issue_kv = [&](const Unit &x) {
        const int h = x.h, hk = h / G;
        tma_load_3d(sKQ, &mk, 0, hk, (int)x.tok0, bar_kq);
        tma_load_3d(sKQ + 16384, &mk, 64, hk, (int)x.tok0, bar_kq);
        mbar_arrive_expect_tx(bar_v, 16384);
        tma_load_3d_hint(sm + A_V, &mv, 0, h, (int)x.tok0, bar_v, pol_read_once);
        tma_load_3d_hint(sm + A_V + 8192, &mv, 64, h, (int)x.tok0, bar_v, pol_read_once);
    };
    // the issuing thread: [K; Q] K^T of the unit with loop index `ui` into TMEM buffer ui % 2
    // (rows 0-63 K K^T, rows 64-127 Q K^T), once its tiles have landed
    auto issue_kq_mma = [&](int ui, uint32_t tb) -> bool {
        if (!mbar_wait(bar_kq, (uint32_t)ui & 1u, p.wait_ns)) return false;
        fence_after_sync();
        const uint64_t d0 = desc_sw128(smem_u32(sKQ), 16, 1024);
        const uint32_t id = idesc_f16(128, 64, false, false, kbf);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (k >= ksteps) break;  // a head of <= 64 features: its second K-block is all zeros
            const uint64_t d = desc_add(d0, (k >> 2) * 16384 + (k & 3) * 32);
            mma_f16(tb + (ui & 1) * 64, d, d, id, k > 0);
        }
        mma_commit(bar_mma);
        return true;
    };
    // gates of unit x for token `tid` (threads < C); identity past the chunk's end.
    // Issued as volatile loads so that they stay a unit ahead of their use.
    auto load_gates = [&](const Unit &x, float &ga, float &gb) {
        ga = 1.f;
        gb = 0.f;
        if (tid < C && x.valid && tid < x.n) {
            const long gi = (x.tok0 + tid) * Hv + x.h;
            ga = ld_gate_early(p.alpha, gi, p.dt_gate);
            gb = ld_gate_early(p.beta, gi, p.dt_gate);
        }
    };

    if (tid == 0) {
        prefetch_tensormap(&mq);
        prefetch_tensormap(&mk);
        prefetch_tensormap(&mv);
        mbar_init(bar_kq, 1);
        mbar_init(bar_v, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0) {
        tmem_alloc(slot, A_TMEM_COLS);
        tmem_relinquish();
    }
    // the issuing thread's view of its copies and MMAs in flight, for the drain
    // on timeout
    bool kq_pending = false, v_pending = false, mma_pending = false, kq_pending_fail = false;
    Unit cur = unit_at(blockIdx.x / Hv, blockIdx.x % Hv);
    Unit nxt = next_unit(cur);
    if (tid == kIssueThread && cur.valid) {
        issue_q(cur);
        issue_kv(cur);
        kq_pending = v_pending = true;
    }
    if constexpr (XO) {
        // inactive capture: every CTA clears a share of the whole buffer
        prefill_capture_clear(p, su_slot, blockIdx.x, gridDim.x, tid, kIntraThreads);
    }
    float ga, gb;
    load_gates(cur, ga, gb);
    {
        // columns 32-63 of P' rows 0-31 are zero in every unit: written once into
        // the staging image (four threads per row, one of its chunks 4-7 each)
        const int r = tid >> 2, q = 4 + (tid & 3);
        if (r < 32) *reinterpret_cast<uint4 *>(sm + A_PS + sw128_chunk(r, q)) = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async();  // (read by the bulk stores)
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = *slot;
    const uint32_t lane_base = tbase + ((uint32_t)(32 * (warp & 3)) << 16);
    const int quarter = warp & 3, half = warp >> 2;
    // the first unit's [K; Q] K^T (later units': issued by the unit before)
    if (tid == kIssueThread && cur.valid) {
        const bool ok0 = issue_kq_mma(0, tbase);
        kq_pending = !ok0;
        mma_pending = ok0;
    }
    // this warp's 32 right-hand-side columns: V columns (U) for warps 0-3, K columns (W) for 4-7
    const bool isW = warp >= 4;
    const int cc0 = 32 * (warp & 3);                    // first column within V or K
    const int t4 = lane & 3;                            // fragment column-pair index
    bool failed = false;

    int it = 0;
    // (packed rows: every unit after an invalid one is past the end too)
    for (; cur.valid; cur = nxt, nxt = next_unit(nxt), ++it) {
        const int b = cur.b, c = cur.c, h = cur.h, n = cur.n, len = cur.len;
        const long tok0 = cur.tok0;
        const int hk = h / G;
        const uint32_t ph = (uint32_t)it & 1u;
        uint8_t *rec = records(p) + ((size_t)cur.gc * Hv + h) * REC_BYTES;
        int ncap = 0;
        float *su0 = nullptr;
        if constexpr (XO) {
            ncap = prefill_ncap(p, b, len) - c * C;
            if (ncap > 0) su0 = p.su + ((long)b * p.capacity + (long)c * C) * su_slot;
        }
        // ---- gates (loaded one unit ahead); start the next unit's gate loads
        if (tid < C) {
            vg[tid] = (tid < n) ? conv_log_alpha(ga, p.conv) : 0.f;
            vbeta[tid] = (tid < n) ? conv_beta(gb, p.conv) : 0.f;
            if (tid < ncap) su0[tid * su_slot + h] = conv_alpha(ga, p.conv);
        }
        load_gates(nxt, ga, gb);
        bool ok = !(tid == kIssueThread && (kq_pending_fail || (it == 0 && kq_pending)));  // this unit's [K; Q] K^T issued
        if constexpr (NORM) {
            // 1/|k_t| and 1/|q_t| from the staged tiles (rows 0-63 K, 64-127 Q;
            // two threads per row, one per 64-column block)
            if (!mbar_wait(bar_kq, ph, p.wait_ns)) ok = false;
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
        }
        if (__syncthreads_or(!ok)) { failed = true; break; }
        // warp 1: cumulative log-decay g, gamma, w; W's right-hand-side scale; the record's vectors
        if (warp == 1) {
            float x0 = vg[lane], x1 = vg[lane + 32];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                float y0 = __shfl_up_sync(0xffffffffu, x0, o);
                float y1 = __shfl_up_sync(0xffffffffu, x1, o);
                if (lane >= o) { x0 += y0; x1 += y1; }
            }
            x1 += __shfl_sync(0xffffffffu, x0, 31);
            const float glast = __shfl_sync(0xffffffffu, x1, 31);
            const float g0 = expf(x0), g1 = expf(x1), w0 = expf(glast - x0), w1 = expf(glast - x1);
            vg[lane] = x0;
            vg[lane + 32] = x1;
            vgl[lane] = x0 * kLog2e;
            vgl[lane + 32] = x1 * kLog2e;
            const float rk0 = NORM ? vkn[lane] : 1.f, rk1 = NORM ? vkn[lane + 32] : 1.f;
            const float rq0 = NORM ? vqn[lane] : 1.f, rq1 = NORM ? vqn[lane + 32] : 1.f;
            vbw[lane] = vbeta[lane] * g0 * rk0;
            vbw[lane + 32] = vbeta[lane + 32] * g1 * rk1;
            float *rv = reinterpret_cast<float *>(rec + REC_VEC);
            rv[lane] = p.scale * g0 * rq0;
            rv[lane + 32] = p.scale * g1 * rq1;
            rv[64 + lane] = w0 * rk0;
            rv[96 + lane] = w1 * rk1;
            if (lane == 0) rv[128] = expf(glast);
        }
        if (ncap > 0 && h % G == 0) {
            // captured keys: the (normalised) key the recurrence used
            const E *kg = reinterpret_cast<const E *>(p.k);
            const int nk = ncap < n ? ncap : n;
            const int dk = p.dk;
            for (int e = tid; e < nk * dk; e += kIntraThreads) {
                const int t = e / dk, j = e % dk;
                su0[t * su_slot + Hv + (long)hk * dk + j] =
                    ld_f(kg + ((tok0 + t) * Hk + hk) * dk + j) * (NORM ? vkn[t] : 1.f);
            }
        }
        // every warp: its right-hand-side columns, transposed, for all four token
        // blocks (fragment of R^T, rows = its columns, cols = tokens; scaled when
        // used), taken into registers now, so that once this unit's [K; Q] K^T is
        // done its K, Q and V tiles are free and the next unit's copies have the
        // whole unit to land
        ok = mbar_wait(bar_v, ph, p.wait_ns);
        // (W's right-hand sides are K's columns: the K copy has landed, as the
        // issuing thread saw before the barrier above; the wait makes it
        // explicit for this thread)
        if (ok && isW) ok = mbar_wait(bar_kq, ph, p.wait_ns);
        uint32_t rf[4][2][4];
        if (ok) {
            const uint8_t *srcb = isW ? sKQ + 16384 * (cc0 >> 6) : sm + A_V + 8192 * (cc0 >> 6);
            const int mi_l = (lane >> 3) & 1, ti_l = lane >> 4, r8 = lane & 7;
#pragma unroll
            for (int J = 0; J < 4; ++J)
#pragma unroll
                for (int mi = 0; mi < 2; ++mi) {
                    const int t = 16 * J + 8 * ti_l + r8;
                    const int q = ((cc0 & 63) + 16 * mi + 8 * mi_l) >> 3;
                    ldsm_x4_trans(rf[J][mi], srcb + sw128_chunk(t, q));
                }
        }
        if (ok) ok = mbar_wait(bar_mma, ph, p.wait_ns);  // this unit's [K; Q] K^T
        if (tid == kIssueThread || tid == kPStoreThread) bulk_wait_read_all();  // the last unit's staged images have been read
        if (__syncthreads_or(!ok)) { failed = true; break; }
        fence_after_sync();
        if (tid == kIssueThread) {
            mma_pending = false;
            if (nxt.valid) {
                // this unit's K, Q and V tiles have been read: the next unit's may land
                issue_q(nxt);
                issue_kv(nxt);
                kq_pending = v_pending = true;
            }
        }
        const uint32_t lane_buf = lane_base + (uint32_t)(it & 1) * 64;  // this unit's [K; Q] K^T
        // ---- -A (16-bit) and its diagonal blocks (fp32), P' (image, staged) from TMEM.
        // Warp w reads TMEM lane quarter w % 4 (rows 0-63: K K^T, 64-127: Q K^T):
        // rows 0-31 of A / P' have nothing right of column 31 and go to warp w
        // alone (w < 4); rows 32-63 use all 64 columns, 32 to each of w and w + 4.
        {
            // A[t][i] = beta_t e^{g_t - g_i} k_t.k_i (i < t), stored negated, and
            // P'[t][i] = e^{g_t - g_i} (scale q_t).k_i (i <= t) take the same steps
            // with their own row factor (-beta_t, or the query scale), last column
            // (t - 1 or t) and image (-A, or P' staged for a bulk store; both of
            // 128-byte rows, 16-byte chunks swizzled by row % 8); A's diagonal
            // block (J, J), J = t / 16, also goes out in fp32 for D_J.  One code
            // path for both halves keeps the kernel's instruction footprint small.
            const bool aside = quarter < 2;  // A (K rows) or P' (Q rows)
            const int t = 32 * (quarter & 1) + lane;
            const int c_lo = (quarter & 1) ? 32 * half : 0;
            const float gtl = vgl[t];
            const float f = aside ? -vbeta[t] * (NORM ? vkn[t] : 1.f) : p.scale * (NORM ? vqn[t] : 1.f);
            const int ilast = aside ? t - 1 : t;
            uint8_t *img = aside ? sNA : sm + A_PS;
            const int J = t >> 4;
            // every column first (broadcast reads of their g), then every
            // store, so that no shared-memory read waits behind a store
            auto emit = [&](const float *v, auto ncols) {
                constexpr int NCOL = decltype(ncols)::value;
                float a[NCOL];
#pragma unroll
                for (int e = 0; e < NCOL; ++e) {
                    const int i = c_lo + e;
                    const float kk = NORM ? v[e] * vkn[i] : v[e];
                    a[e] = (i <= ilast) ? ex2_approx(gtl - vgl[i]) * (f * kk) : 0.f;
                }
                if (aside) {
#pragma unroll
                    for (int blk = 0; blk < NCOL / 16; ++blk) {
                        if ((c_lo >> 4) + blk == J) {
                            float *dst = Adt + J * 272 + (t & 15);  // column e of the block at e * 16
#pragma unroll
                            for (int e = 0; e < 16; ++e) dst[e * 16] = -a[16 * blk + e];
                        }
                    }
                }
#pragma unroll
                for (int q8 = 0; q8 < NCOL / 8; ++q8)
                    *reinterpret_cast<uint4 *>(img + sw128_chunk(t, (c_lo >> 3) + q8)) = pack8<E>(a + 8 * q8);
            };
            // rows 0-31 need columns 0-31 (warp half 0; half 1 has nothing to
            // build), rows 32-63 columns 0-63 in two halves of 32
            if ((quarter & 1) != 0 || half == 0) {
                float v[32];
                tmem_ld32(lane_buf + c_lo, v);
                emit(v, std::integral_constant<int, 32>{});
            }
        }
        fence_before_sync();
        if (quarter >= 2) {
            // P' warps: the image is staged; one of them stores it
            fence_proxy_async();
            named_bar(kBarPImage, 128);
            if (tid == kPStoreThread) {
                bulk_store_hint(rec + REC_P, sm + A_PS, 8192, pol_keep);
                bulk_commit();
            }
        }
        // ---- D_J = (I + A_JJ)^{-1}, one warp per block: warp 0 built blocks 0
        // and 1 and solves block 0, warp 4 solves block 1 behind a named barrier
        // with it; blocks 2 and 3 (built by warp 5) go to P' warps 2 and 6
        {
            int J = -1;
            if (warp == 0) {
                named_bar_arrive(kBarDiag01, 64);
                __syncwarp();  // (its own lanes wrote block 0)
                J = 0;
            } else if (warp == 5) {
                named_bar_arrive(kBarDiag23, 96);
            } else if (warp == 4) {
                named_bar(kBarDiag01, 64);
                J = 1;
            } else if (quarter == 2) {
                named_bar(kBarDiag23, 96);
                J = 2 + half;
            }
            if (J >= 0) solve_diag_block<E>(Adt + J * 272, sD + J * 512, lane);
        }
        __syncthreads();  // -A and D_J written
        // ---- block substitution: X_J^T = (R_J^T - sum_{K<J} X_K^T A_JK^T) D_J^T
        {
            const float *scl = isW ? vbw : vbeta;
            uint32_t xa[4][2][4];  // X_K^T as A fragments, per block K and m-tile
#pragma unroll
            for (int J = 0; J < 4; ++J) {
                float acc[2][2][4];
#pragma unroll
                for (int ni = 0; ni < 2; ++ni) {
                    const float2 s0 = *reinterpret_cast<const float2 *>(scl + 16 * J + 8 * ni + 2 * t4);
#pragma unroll
                    for (int mi = 0; mi < 2; ++mi) {
                        const float2 lo = Elem<E>::unpack2(rf[J][mi][2 * ni]);      // row g
                        const float2 hi = Elem<E>::unpack2(rf[J][mi][2 * ni + 1]);  // row g + 8
                        acc[mi][ni][0] = lo.x * s0.x;
                        acc[mi][ni][1] = lo.y * s0.y;
                        acc[mi][ni][2] = hi.x * s0.x;
                        acc[mi][ni][3] = hi.y * s0.y;
                    }
                }
#pragma unroll
                for (int K = 0; K < J; ++K) {
                    uint32_t bq[4];  // (-A_JK)^T as B fragments: n-tile 0 (b0, b1), n-tile 1 (b0, b1)
                    const int row = 16 * J + (lane & 7) + 8 * (lane >> 4);
                    ldsm_x4(bq, sNA + na_off(row, 2 * K + ((lane >> 3) & 1)));
#pragma unroll
                    for (int mi = 0; mi < 2; ++mi) {
                        mma16816<kbf>(acc[mi][0], xa[K][mi], bq[0], bq[1]);
                        mma16816<kbf>(acc[mi][1], xa[K][mi], bq[2], bq[3]);
                    }
                }
                uint32_t ya[2][4];
#pragma unroll
                for (int mi = 0; mi < 2; ++mi) {
                    ya[mi][0] = Elem<E>::pack2(acc[mi][0][0], acc[mi][0][1]);
                    ya[mi][1] = Elem<E>::pack2(acc[mi][0][2], acc[mi][0][3]);
                    ya[mi][2] = Elem<E>::pack2(acc[mi][1][0], acc[mi][1][1]);
                    ya[mi][3] = Elem<E>::pack2(acc[mi][1][2], acc[mi][1][3]);
                }
                uint32_t bd[4];  // D_J^T as B fragments
                {
                    const int row = (lane & 7) + 8 * (lane >> 4);
                    ldsm_x4(bd, sD + J * 512 + d_off(row, (lane >> 3) & 1));
                }
#pragma unroll
                for (int mi = 0; mi < 2; ++mi) {
                    float o0[4] = {0.f, 0.f, 0.f, 0.f}, o1[4] = {0.f, 0.f, 0.f, 0.f};
                    mma16816<kbf>(o0, ya[mi], bd[0], bd[1]);
                    mma16816<kbf>(o1, ya[mi], bd[2], bd[3]);
                    xa[J][mi][0] = Elem<E>::pack2(o0[0], o0[1]);
                    xa[J][mi][1] = Elem<E>::pack2(o0[2], o0[3]);
                    xa[J][mi][2] = Elem<E>::pack2(o1[0], o1[1]);
                    xa[J][mi][3] = Elem<E>::pack2(o1[2], o1[3]);
                    // X_J rows (tokens) 16J .. 16J+15, this m-tile's 16 columns, to the staged record
                    const int t = 16 * J + 8 * (lane >> 4) + (lane & 7);
                    const int ccol = cc0 + 16 * mi + 8 * ((lane >> 3) & 1);
                    uint8_t *dst = isW ? sm + A_WS + (ccol >> 6) * 8192 + sw128_chunk(t, (ccol & 63) >> 3)
                                       : sm + A_US + (ccol >> 5) * 4096 + u32_chunk(t, (ccol & 31) >> 3);
                    stsm_x4_trans(dst, xa[J][mi]);
                }
            }
        }
        fence_proxy_async();
        fence_before_sync();
        __syncthreads();
        if (tid == kIssueThread) {
            bulk_store_hint(rec + REC_U, sm + A_US, 16384, pol_keep);
            bulk_store_hint(rec + REC_W, sm + A_WS, 16384, pol_keep);
            bulk_commit();
            // the next unit's [K; Q] K^T, into the other TMEM buffer
            if (nxt.valid && !kq_pending_fail) {
                if (issue_kq_mma(it + 1, tbase)) {
                    kq_pending = false;
                    mma_pending = true;
                } else {
                    kq_pending_fail = true;  // reported at the next unit's first check
                }
            }
        }
    }
    if (failed) {
        if (tid == kIssueThread) {
            atomicOr(p.err, (uint32_t)GDN_DEVERR_TIMEOUT);
            // copies and MMAs in flight must finish before the CTA exits
            // (copies of this unit or of the next, whichever were issued last)
            for (uint32_t ph = 0; ph < 2; ++ph) {
                if (kq_pending) mbar_wait(bar_kq, ph, kWaitNs / 4);
                if (v_pending) mbar_wait(bar_v, ph, kWaitNs / 4);
                if (mma_pending) mbar_wait(bar_mma, ph, kWaitNs / 4);
            }
        }
    }
    // (without a timeout nothing is in flight here: no copy is issued past the last unit)
    if (tid == kIssueThread || tid == kPStoreThread) bulk_wait_all();  // the records have been written
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, A_TMEM_COLS);
}

// ============================================================ phase B ====

// One carry CTA owns TV rows of one (row, value head) state: TV = 32 (the
// latency instance: the most CTAs, three stages) or TV = 64 / 128 (the
// throughput instances, for grids of many rows: two and four times the work
// per MMA for about the same issue time, two stages).  Operand images wider
// than 64 columns are stored as 64-column blocks (N-blocks of the MN-major
// 128-byte-swizzled layout, one after the other).
template <int TV>
struct CarryCfg {
    static constexpr int kCols = TV / 2;             // state columns per compute thread
    static constexpr int kGroup = kCols < 32 ? kCols : 32;  // columns a thread handles at a time
    static constexpr int NS = TV == 32 ? 3 : 2;      // stages in the ring
    static constexpr uint32_t ST_A1 = 0;             // [Q ; W] image, 2 K-blocks of 128 rows
    static constexpr uint32_t ST_K = 32768;          // K image, 2 dk blocks of 64 rows
    static constexpr uint32_t ST_P = 49152;          // P' image (rows 0-63 of the [P'; X] operand)
    static constexpr uint32_t ST_U = 57344;          // U tiles, TV / 32 of [64 t][32 i]
    static constexpr uint32_t kUBytes = TV * 128;
    static constexpr uint32_t ST_VEC = ST_U + kUBytes;  // gamma, w, gamma_last
    static constexpr uint32_t ST_BYTES = ST_VEC + 1024;
    static constexpr uint32_t kNBlocks = TV > 64 ? 2 : 1;  // 64-column blocks of the images
    static constexpr uint32_t SIMG_BLOCK = 16384;    // S^T image block: 128 K-rows (dk)
    static constexpr uint32_t DIMG_BLOCK = 8192;     // Delta image block: 64 K-rows (tokens)
    static constexpr uint32_t B_S = NS * ST_BYTES;   // S^T image (MN-major, TV N used)
    static constexpr uint32_t B_DW = B_S + kNBlocks * SIMG_BLOCK;  // diag(w) Delta image
    static constexpr uint32_t B_DD = B_DW + kNBlocks * DIMG_BLOCK;  // Delta image
    static constexpr uint32_t B_BAR = B_DD + kNBlocks * DIMG_BLOCK;
    static constexpr uint32_t B_SMEM = B_BAR + 128 + 1024;
    static constexpr uint32_t STAGE_TX = 16384 + 16384 + 16384 + 8192 + kUBytes + 1024;
    // TMEM columns: D1 = [Q; W] S^T at 0 / TV (by chunk parity), D2 = K^T w Delta
    // at 2 TV, D3 = P' Delta at 3 TV / 4 TV (by chunk parity; one buffer at
    // TV = 128, where the output warps read D3 of a chunk before they reach
    // the next chunk's Delta barrier, after which its D3 is issued)
    static constexpr uint32_t T_D2 = 2 * TV, T_D3 = 3 * TV;
    static constexpr uint32_t T_D3_ODD = TV == 128 ? 0u : (uint32_t)TV;
    static constexpr uint32_t T_COLS = TV == 32 ? 256 : 512;
    static_assert(T_D3 + T_D3_ODD + TV <= T_COLS, "carry TMEM columns");
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
    static_assert(N == 16 || N == 32, "16 or 32 columns");
    if constexpr (N == 16) tmem_ld16(taddr, v);
    else tmem_ld32(taddr, v);
}
// Byte offset of the 16-byte chunk holding columns [c, c + 8) of row r of an
// operand image stored as 64-column SW128 blocks `block` bytes apart.
__device__ __forceinline__ uint32_t img_chunk(int r, int c, uint32_t block) {
    return (uint32_t)(c >> 6) * block + sw128_chunk(r, (c & 63) >> 3);
}

template <typename E, bool XO, int TV>
__global__ void __launch_bounds__(kCarryThreads, 1)
prefill_carry_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap mq,
                     const __grid_constant__ CUtensorMap mk) {
    using Cfg = CarryCfg<TV>;
    constexpr int NS = Cfg::NS, NC = Cfg::kCols, Q8 = NC / 8, CG = Cfg::kGroup;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_align1k(smem_raw);
    uint8_t *sS = sm + Cfg::B_S, *sDw = sm + Cfg::B_DW, *sDd = sm + Cfg::B_DD;
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + Cfg::B_BAR);  // [NS]
    uint64_t *empty = full + NS;                                       // [NS]
    uint64_t *bar1 = full + 2 * NS, *bar2 = bar1 + 1, *bar3 = bar1 + 2;
    uint32_t *slot = reinterpret_cast<uint32_t *>(bar1 + 3);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = (warp >> 2) & 1;
    // packed rows: the grid takes the rows in the prologue's order
    const int vt = blockIdx.x, h = blockIdx.y, b = p.chunk_table ? p.chunk_table[p.B + 1 + blockIdx.z] : blockIdx.z;
    const int Hv = p.Hv, Hk = p.Hk;
    const int ksteps = p.dk > 64 ? 8 : 4;  // K = 16 steps of D1 (over dk)
    const int hk = h / (Hv / Hk);
    const int i0 = vt * TV;
    long rtok0;
    int len;
    row_range(p.cu_seqlens, b, p.T, rtok0, len);
    const int nc = n_chunks(len);
    const long su_slot = (long)Hv + (long)Hk * p.dk + (long)Hv * p.dv;
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
        const uint64_t pol_read_once = l2_evict_first_policy();  // the records are read once
        auto issue_stage = [&](int cc) {
            const int s = cc % NS;
            uint8_t *st = sm + s * Cfg::ST_BYTES;
            const uint8_t *rec = rec0 + (size_t)cc * rec_stride;
            const int t0 = (int)(rtok0 + (long)cc * C);
            mbar_arrive_expect_tx(&full[s], Cfg::STAGE_TX);
            tma_load_3d(st + Cfg::ST_A1, &mq, 0, hk, t0, &full[s]);
            tma_load_3d(st + Cfg::ST_A1 + 16384, &mq, 64, hk, t0, &full[s]);
            bulk_load_hint(st + Cfg::ST_A1 + 8192, rec + REC_W, 8192, &full[s], pol_read_once);
            bulk_load_hint(st + Cfg::ST_A1 + 24576, rec + REC_W + 8192, 8192, &full[s], pol_read_once);
            tma_load_3d(st + Cfg::ST_K, &mk, 0, hk, t0, &full[s]);
            tma_load_3d(st + Cfg::ST_K + 8192, &mk, 64, hk, t0, &full[s]);
            bulk_load_hint(st + Cfg::ST_P, rec + REC_P, 8192, &full[s], pol_read_once);
            bulk_load_hint(st + Cfg::ST_U, rec + REC_U + vt * Cfg::kUBytes, Cfg::kUBytes, &full[s],
                           pol_read_once);
            bulk_load_hint(st + Cfg::ST_VEC, rec + REC_VEC, 1024, &full[s], pol_read_once);
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
        // (LBO: the distance between 64-column blocks of an MN-major operand)
        const uint64_t bS0 = desc_sw128(smem_u32(sS), Cfg::kNBlocks > 1 ? Cfg::SIMG_BLOCK : 8192u, 1024);
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
                    for (int k = 0; k < 8; ++k) {
                        if (k >= ksteps) break;  // a head of <= 64 features: its second K-block is all zeros
                        mma_f16(tbase + d1, desc_add(a0, (k >> 2) * 16384 + (k & 3) * 32), desc_add(bS0, k * 2048),
                                id1, k > 0);
                    }
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
                const uint32_t d3 = Cfg::T_D3 + ((cc & 1) ? Cfg::T_D3_ODD : 0u);
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
        // (columns j >= dk of a smaller head stay zero: so do K's and Q's there)
        const int dk = p.dk, dv = p.dv;
        const bool jin = j < dk;
        const float *s0 = initial_state_ptr(p.s0, p.s0_idx, p.n_s0, b, h, Hv, dv, dk, p.err);
#pragma unroll
        for (int i = 0; i < NC; ++i) S[i] = (s0 && jin) ? s0[(size_t)(i0 + c0 + i) * dk + j] : 0.f;
#pragma unroll
        for (int q8 = 0; q8 < Q8; ++q8)
            *reinterpret_cast<uint4 *>(sS + img_chunk(j, c0 + 8 * q8, Cfg::SIMG_BLOCK)) = pack8<E>(S + 8 * q8);
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
            const uint32_t d3 = Cfg::T_D3 + ((cc & 1) ? Cfg::T_D3_ODD : 0u);
            const int n = min(C, len - cc * C);
            if (ok) ok = mbar_wait(&full[s], (cc / NS) & 1, p.wait_ns);
            const float *vec = reinterpret_cast<const float *>(st + Cfg::ST_VEC);
            const float gC = ok ? vec[128] : 0.f;
            if (quarter >= 2) {
                // Delta = U - W S^T for token t, NC of the TV columns
                const int t = 32 * (quarter - 2) + lane;
                const float wt = ok ? vec[64 + t] : 0.f;
                // this row's U chunks, read while D1 runs
                uint4 uraw[Q8];
#pragma unroll
                for (int q8 = 0; q8 < Q8; ++q8) {
                    const int c = c0 + 8 * q8;  // column of the tile: U tile (c / 32), chunk (c % 32) / 8
                    uraw[q8] = ok ? *reinterpret_cast<const uint4 *>(st + Cfg::ST_U + (c >> 5) * 4096 +
                                                                      u32_chunk(t, (c & 31) >> 3))
                                  : make_uint4(0u, 0u, 0u, 0u);
                }
                if (ok) ok = mbar_wait(bar1, cc & 1, p.wait_ns);
                if (ok) {
                    fence_after_sync();
                    // captured tokens: Delta's row t is token t's delta
                    float *cap = (cc * C + t < ncap)
                                     ? p.su + ((size_t)b * p.capacity + cc * C + t) * su_slot + Hv +
                                           (size_t)Hk * p.dk + (size_t)h * p.dv + i0 + c0
                                     : nullptr;
#pragma unroll
                    for (int gq = 0; gq < NC / CG; ++gq) {
                        float ws[CG];
                        tmem_ld_cols<CG>(lane_base + d1 + c0 + gq * CG, ws);
#pragma unroll
                        for (int q8 = 0; q8 < CG / 8; ++q8) {
                            const int qq = gq * (CG / 8) + q8;
                            const int c = c0 + 8 * qq;
                            float u[8], dd[8], dw[8];
                            unpack8<E>(uraw[qq], u);
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                dd[e] = u[e] - ws[8 * q8 + e];
                                dw[e] = wt * dd[e];
                            }
                            *reinterpret_cast<uint4 *>(sDd + img_chunk(t, c, Cfg::DIMG_BLOCK)) = pack8<E>(dd);
                            *reinterpret_cast<uint4 *>(sDw + img_chunk(t, c, Cfg::DIMG_BLOCK)) = pack8<E>(dw);
                            if (cap != nullptr)
#pragma unroll
                                for (int e = 0; e < 8; ++e) cap[8 * qq + e] = dd[e];
                        }
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
#pragma unroll
                for (int gq = 0; gq < NC / CG; ++gq) {
                    float v[CG];
                    tmem_ld_cols<CG>(lane_base + Cfg::T_D2 + c0 + gq * CG, v);
#pragma unroll
                    for (int i = 0; i < CG; ++i) S[gq * CG + i] = fmaf(gC, S[gq * CG + i], v[i]);
                }
#pragma unroll
                for (int q8 = 0; q8 < Q8; ++q8)
                    *reinterpret_cast<uint4 *>(sS + img_chunk(j, c0 + 8 * q8, Cfg::SIMG_BLOCK)) = pack8<E>(S + 8 * q8);
                fence_proxy_async();
                if constexpr (XO) {
                    // chunk-boundary checkpoint: the fp32 state after this chunk
                    const int ck = ckpt_slot(p, cc, len);
                    if (ck >= 0 && jin) {
                        float *dst = p.ckpt + ((((size_t)b * p.ckpt_cap + ck) * Hv + h) * dv + i0 + c0) * dk;
#pragma unroll
                        for (int i = 0; i < NC; ++i) __stcs(dst + (size_t)i * dk + j, S[i]);
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
                    E *dst = ob + ((rtok0 + (long)cc * C + t) * Hv + h) * (long)dv + i0 + c0;
#pragma unroll
                    for (int gq = 0; gq < NC / CG; ++gq) {
                        float qs[CG], pd[CG];
                        tmem_ld_cols<CG>(lane_base + d1 + c0 + gq * CG, qs);
                        tmem_ld_cols<CG>(lane_base + d3 + c0 + gq * CG, pd);
                        if (t < n) {
#pragma unroll
                            for (int q8 = 0; q8 < CG / 8; ++q8) {
                                float o[8];
#pragma unroll
                                for (int e = 0; e < 8; ++e) o[e] = fmaf(gt, qs[8 * q8 + e], pd[8 * q8 + e]);
                                *reinterpret_cast<uint4 *>(dst + gq * CG + 8 * q8) = pack8<E>(o);
                            }
                        }
                    }
                }
            }
        }
        if (ok && p.s_final != nullptr && jin) {
            float *sf = p.s_final + (((size_t)b * Hv + h) * dv + i0 + c0) * dk;
#pragma unroll
            for (int i = 0; i < NC; ++i) sf[(size_t)i * dk + j] = S[i];
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

// Rows of the carry tiles for grids of many rows (64 or 128).
constexpr int kWideRows = 128;

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

// [total_T, H, width] 16-bit tensor, box {64 features, 1 head, 64 tokens},
// 128-byte swizzle.  A head narrower than 128 features reads as zero-padded
// to 128: the box parts past `width` are out of bounds and come back as zeros.
bool make_map(CUtensorMap *m, const void *ptr, int H, long total_T, bool bf16, int width) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return false;
    cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)H, (cuuint64_t)total_T};
    cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)H * width * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
               const_cast<void *>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Carry instance: 32-row tiles while one wave of them fits the GPU (the
// chain's latency decides), wider tiles for more rows (throughput decides).
int carry_rows(const PrefillParams &p) {
    if ((long)(p.dv / 32) * p.Hv * p.B > (long)sm_count_of_current_device() && p.dv >= 64)
        return p.dv >= kWideRows ? kWideRows : 64;
    return 32;
}

template <typename E, bool XO>
cudaError_t launch_e(const PrefillParams &p, long total_T, long max_chunks, cudaStream_t stream) {
    const bool bf = Elem<E>::kBf16;
    CUtensorMap mq, mk, mv;
    memset(&mq, 0, sizeof(mq));
    memset(&mk, 0, sizeof(mk));
    memset(&mv, 0, sizeof(mv));
    // With no tokens at all no chunk exists and the maps are never used.
    if (total_T > 0 && (!make_map(&mq, p.q, p.Hk, total_T, bf, p.dk) || !make_map(&mk, p.k, p.Hk, total_T, bf, p.dk) ||
                        !make_map(&mv, p.v, p.Hv, total_T, bf, p.dv)))
        return cudaErrorInvalidValue;
    const bool norm = (p.conv & GDN_QK_L2NORM) != 0;
    auto intra = norm ? prefill_intra_kernel<E, XO, true> : prefill_intra_kernel<E, XO, false>;
    cudaError_t e = norm ? set_smem_once<prefill_intra_kernel<E, XO, true>>((int)A_SMEM)
                         : set_smem_once<prefill_intra_kernel<E, XO, false>>((int)A_SMEM);
    if (e != cudaSuccess) return e;
    const int tv = carry_rows(p);
    e = tv == 32 ? set_smem_once<prefill_carry_kernel<E, XO, 32>>((int)CarryCfg<32>::B_SMEM)
        : tv == 64 ? set_smem_once<prefill_carry_kernel<E, XO, 64>>((int)CarryCfg<64>::B_SMEM)
                   : set_smem_once<prefill_carry_kernel<E, XO, 128>>((int)CarryCfg<128>::B_SMEM);
    if (e != cudaSuccess) return e;
    if (max_chunks > 0) {
        // persistent: at most two CTAs per SM walk the (chunk, value head) units
        const long n_units = max_chunks * p.Hv;
        const long cap = (long)kIntraCtasPerSm * sm_count_of_current_device();
        const unsigned grid = (unsigned)(n_units < cap ? n_units : cap);
        intra<<<grid, kIntraThreads, A_SMEM, stream>>>(p, max_chunks, mq, mk, mv);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    // The carry kernel is a programmatic dependent of the chunk-parallel one:
    // its prologue (barriers, TMEM, the initial state) overlaps that kernel's
    // tail, and it waits for that kernel's records before reading them.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.dv / tv, p.Hv, p.B);
    cfg.blockDim = dim3(kCarryThreads);
    cfg.dynamicSmemBytes = tv == 32 ? CarryCfg<32>::B_SMEM : tv == 64 ? CarryCfg<64>::B_SMEM : CarryCfg<128>::B_SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = max_chunks > 0 ? 1 : 0;
    if (tv == 32) return cudaLaunchKernelEx(&cfg, prefill_carry_kernel<E, XO, 32>, p, mq, mk);
    if (tv == 64) return cudaLaunchKernelEx(&cfg, prefill_carry_kernel<E, XO, 64>, p, mq, mk);
    return cudaLaunchKernelEx(&cfg, prefill_carry_kernel<E, XO, 128>, p, mq, mk);
}

long max_chunks_of(int B, int T, bool varlen) {
    return varlen ? (long)T / C + B : (long)B * ((T + C - 1) / C);
}

}  // namespace

bool prefill_tc_supported(int dk, int dv, int chunk, int dt_qkv) {
    auto width_ok = [](int d) { return d == 32 || d == 64 || d == D; };
    return width_ok(dk) && width_ok(dv) && chunk == C && (dt_qkv == GDN_BF16 || dt_qkv == GDN_F16);
}

size_t prefill_tc_workspace_bytes(int B, int T, int /*Hk*/, int Hv, bool varlen) {
    return (varlen ? chunk_table_bytes(B) : 0) + (size_t)max_chunks_of(B, T, varlen) * (size_t)Hv * REC_BYTES;
}

cudaError_t launch_prefill_tc(const PrefillParams &p_in, cudaStream_t stream) {
    PrefillParams p = p_in;
    const bool varlen = p.cu_seqlens != nullptr;
    const long total_T = varlen ? (long)p.T : (long)p.B * p.T;
    const long mc = max_chunks_of(p.B, p.T, varlen);
    if (mc >= 0x7fffffffL) return cudaErrorInvalidValue;  // chunk indices stay 32-bit
    const bool xo = p.ckpt != nullptr || p.capacity > 0;
    p.chunk_table = nullptr;
    if (varlen && p.B > 0) {
        // packed rows: per-row chunk table at the head of the workspace
        int32_t *tbl = reinterpret_cast<int32_t *>(p.ws);
        // longest rows first while the carry grid is a few waves (there the
        // last wave decides); for many waves the given order, which keeps the
        // rows' records nearer in L2 (measured: +2% on 64 rows when sorted)
        const long ctas = (long)(p.dv / carry_rows(p)) * p.Hv * p.B;
        const int sort = ctas <= 4L * sm_count_of_current_device() ? 1 : 0;
        chunk_table_kernel<<<1, 1024, 0, stream>>>(p.cu_seqlens, p.B, p.T, tbl, sort);
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
