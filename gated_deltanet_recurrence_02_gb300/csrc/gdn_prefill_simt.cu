// gdn_prefill_simt.cu -- chunked prefill for the general shapes, fp32
// arithmetic throughout: CUDA cores, with the two large products on the
// warp-level tensor cores at fp32 accuracy (each operand split into two tf32
// parts, three products).
//
// "Enable the native Kev example on NVIDIA GPUs through ExecuTorch's AOTI CUDA
// backend" (executorch issue 23097), work list: chunked GDN prefill with an
// explicit initial and final state and an FP32 recurrence.  This is the
// general-shape path (any dk, dv in {32, 64, 128}, chunk in {16, 32, 64}, any
// storage dtype); the tensor-core kernels take chunk 64 with 16-bit inputs,
// so this one runs fp32 inputs and chunks of 16 and 32.
//
// One CTA (256 threads) carries a 32-row tile of one (row b, value head h)
// state through all chunks of that row.  Inside a chunk of n tokens with start
// state S0 and local log-decay sums g_t (gamma_t = e^{g_t}):
//   A[t][i] = beta_t e^{g_t - g_i} k_t.k_i  (i < t),  P[t][i] = e^{g_t - g_i} q_t.k_i  (i <= t)
//   R       = diag(beta) (V - diag(gamma) K S0^T)          [n x 32]
//   Delta   = (I + A)^{-1} R                               forward substitution
//   O       = diag(gamma) Q S0^T + P Delta
//   S_end   = gamma_n S0 + Delta^T diag(e^{g_n - g}) K
// S_end of a chunk that ends on a requested boundary is also written out as a
// checkpoint (the state after that many tokens of the row).  With capture on,
// the rows of Delta are the tokens' deltas (the delta rule's delta, formed
// with the decayed state), so the first n_b tokens' decay, key and delta go to
// the capture buffer exactly as on the recurrent path.
// (the UT/WY form; Delta equals U - W S0^T with U = T diag(beta) V and
// W = T diag(beta gamma) K).  A ragged last chunk is padded with identity
// tokens (k = q = v = 0, alpha = 1, beta = 0), which leave S unchanged and
// whose outputs are not stored.  Precondition: every alpha in (0, 1].
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kDVT = 32;  // state rows per CTA

// fp32 products on the warp-level tensor cores at fp32 accuracy: each operand
// x is split into two tf32 parts x = big + small (big = x rounded to tf32,
// small = the rest rounded to tf32), and a b is taken as
// a_small b_big + a_big b_small + a_big b_big, dropping a_small b_small
// (relative size ~2^-22); products accumulate in fp32.
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void split_tf32(float x, uint32_t &big, uint32_t &small) {
    big = to_tf32(x);
    small = to_tf32(x - __uint_as_float(big));
}
// m16n8k8, tf32 inputs, fp32 accumulate.  Fragments (g = lane / 4, t = lane % 4):
// A a0 = (g, t), a1 = (g + 8, t), a2 = (g, t + 4), a3 = (g + 8, t + 4);
// B b0 = (k = t, n = g), b1 = (k = t + 4, n = g);
// C c0, c1 = (g, 2t), (g, 2t + 1); c2, c3 = (g + 8, 2t), (g + 8, 2t + 1).
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
struct SplitA {
    uint32_t big[4], small[4];
};
struct SplitB {
    uint32_t big[2], small[2];
};
// d[n] += a b[n] for N fragments, each of the three terms issued for all N
// before the next (consecutive MMAs then go to different accumulators)
template <int N>
__device__ __forceinline__ void mma_3xtf32_n(float (&d)[N][4], const SplitA &a, const SplitB (&b)[N]) {
#pragma unroll
    for (int n = 0; n < N; ++n) mma_tf32(d[n], a.small, b[n].big[0], b[n].big[1]);
#pragma unroll
    for (int n = 0; n < N; ++n) mma_tf32(d[n], a.big, b[n].small[0], b[n].small[1]);
#pragma unroll
    for (int n = 0; n < N; ++n) mma_tf32(d[n], a.big, b[n].big[0], b[n].big[1]);
}
// A fragment of rows r0 .. r0 + 15, columns k0 .. k0 + 7 of a row-major fp32
// matrix with row stride `ld` (floats).
__device__ __forceinline__ SplitA load_a(const float *m, int ld, int r0, int k0, int g, int t) {
    SplitA a;
    split_tf32(m[(r0 + g) * ld + k0 + t], a.big[0], a.small[0]);
    split_tf32(m[(r0 + g + 8) * ld + k0 + t], a.big[1], a.small[1]);
    split_tf32(m[(r0 + g) * ld + k0 + t + 4], a.big[2], a.small[2]);
    split_tf32(m[(r0 + g + 8) * ld + k0 + t + 4], a.big[3], a.small[3]);
    return a;
}
// B fragment (k = k0 .. k0 + 7, n = n0 .. n0 + 7) of B = M^T for a row-major
// M with rows n and row stride `ld`: B[k][n] = M[n][k].
__device__ __forceinline__ SplitB load_bt(const float *m, int ld, int n0, int k0, int g, int t) {
    SplitB b;
    split_tf32(m[(n0 + g) * ld + k0 + t], b.big[0], b.small[0]);
    split_tf32(m[(n0 + g) * ld + k0 + t + 4], b.big[1], b.small[1]);
    return b;
}

template <int DK, int C>
struct SimtSmem {
    static constexpr int KS = DK + 4;   // row stride of S, K, Q
    static constexpr int DS = kDVT + 4; // row stride of V/R/Delta, O
    static constexpr int AS = C + 1;    // row stride of A, P
    static constexpr int kFloats = kDVT * KS + 2 * C * KS + 2 * C * DS + 2 * C * AS + 4 * C;
    static constexpr size_t kBytes = sizeof(float) * kFloats;
};

template <int DK, int C, typename TQ>
__global__ void __launch_bounds__(kThreads, 1) prefill_simt_kernel(const PrefillParams p) {
    using L = SimtSmem<DK, C>;
    constexpr int KS = L::KS, DS = L::DS, AS = L::AS;
    extern __shared__ float4 smem4[];
    float *Ss = reinterpret_cast<float *>(smem4);  // [32][KS]
    float *Ks = Ss + kDVT * KS;                    // [C][KS]
    float *Qs = Ks + C * KS;                       // [C][KS]  (scaled q)
    float *Vs = Qs + C * KS;                       // [C][DS]  V tile -> R -> Delta
    float *Os = Vs + C * DS;                       // [C][DS]  diag(gamma) Q S0^T
    float *As = Os + C * DS;                       // [C][AS]
    float *Ps = As + C * AS;                       // [C][AS]
    float *lg = Ps + C * AS;                       // [C] log alpha, then g
    float *bt = lg + C;                            // [C] beta
    float *eg = bt + C;                            // [C] e^{g_t}
    float *wg = eg + C;                            // [C] e^{g_last - g_t}

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int Hv = p.Hv, Hk = p.Hk, dv = p.dv;
    const int hk = h / (Hv / Hk);
    const int row0 = tile * kDVT;
    long tok0;
    int Tb;
    row_range(p.cu_seqlens, b, p.T, tok0, Tb);

    const TQ *qb = reinterpret_cast<const TQ *>(p.q);
    const TQ *kb = reinterpret_cast<const TQ *>(p.k);
    const TQ *vb = reinterpret_cast<const TQ *>(p.v);
    TQ *ob = reinterpret_cast<TQ *>(p.out);
    const float scale = p.scale;

    const long slot = (long)Hv + (long)Hk * DK + (long)Hv * dv;
    prefill_capture_clear(p, slot, ((long)b * gridDim.y + h) * gridDim.x + tile,
                          (long)gridDim.x * gridDim.y * gridDim.z, tid, kThreads);
    const int ncap = prefill_ncap(p, b, Tb);

    const float *s0 = initial_state_ptr(p.s0, p.s0_idx, p.n_s0, b, h, Hv, dv, DK, p.err);
    for (int e = tid; e < kDVT * DK / 4; e += kThreads) {
        const int i = e / (DK / 4), j = (e % (DK / 4)) * 4;
        float4 x = s0 ? *reinterpret_cast<const float4 *>(s0 + (long)(row0 + i) * DK + j)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4 *>(Ss + i * KS + j) = x;
    }

    // The next chunk's k, q, v and gates are loaded into registers while the
    // current chunk is computed, and written to shared memory at the start of
    // the next iteration (identity tokens past the row's end).
    constexpr int NKQ = (C * DK / 4 + kThreads - 1) / kThreads;  // float4 of k (and of q) per thread
    constexpr int NV = (C * kDVT + kThreads - 1) / kThreads;      // v elements per thread
    float4 kr[NKQ], qr[NKQ];
    float vr[NV], ga = 1.f, gb = 0.f;
    auto load_chunk = [&](int cs) {
        const int nn = (Tb - cs < C) ? (Tb - cs) : C;
#pragma unroll
        for (int u = 0; u < NKQ; ++u) {
            const int e = tid + u * kThreads, t = e / (DK / 4), j = (e % (DK / 4)) * 4;
            kr[u] = qr[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e < C * DK / 4 && t < nn) {
                const long off = ((tok0 + cs + t) * Hk + hk) * DK + j;
                kr[u] = ld4(kb + off);
                qr[u] = ld4(qb + off);
            }
        }
#pragma unroll
        for (int u = 0; u < NV; ++u) {
            const int e = tid + u * kThreads, t = e / kDVT, i = e % kDVT;
            vr[u] = (e < C * kDVT && t < nn) ? ld_f(vb + ((tok0 + cs + t) * Hv + h) * (long)dv + row0 + i) : 0.f;
        }
        ga = 1.f;
        gb = 0.f;
        if (tid < nn) {
            const long g = (tok0 + cs + tid) * Hv + h;
            ga = ld_gate(p.alpha, g, p.dt_gate);
            gb = ld_gate(p.beta, g, p.dt_gate);
        }
    };
    if (Tb > 0) load_chunk(0);

    for (int c0 = 0; c0 < Tb; c0 += C) {
        const int n = (Tb - c0 < C) ? (Tb - c0) : C;
        // ---- 1. stage the chunk (identity tokens past n) -------------------
#pragma unroll
        for (int u = 0; u < NKQ; ++u) {
            const int e = tid + u * kThreads, t = e / (DK / 4), j = (e % (DK / 4)) * 4;
            if (e < C * DK / 4) {
                float4 qq = qr[u];
                if (!(p.conv & GDN_QK_L2NORM)) {
                    qq.x *= scale; qq.y *= scale; qq.z *= scale; qq.w *= scale;
                }
                *reinterpret_cast<float4 *>(Ks + t * KS + j) = kr[u];
                *reinterpret_cast<float4 *>(Qs + t * KS + j) = qq;
            }
        }
#pragma unroll
        for (int u = 0; u < NV; ++u) {
            const int e = tid + u * kThreads, t = e / kDVT, i = e % kDVT;
            if (e < C * kDVT) Vs[t * DS + i] = vr[u];
        }
        if (tid < C) {
            lg[tid] = (tid < n) ? conv_log_alpha(ga, p.conv) : 0.f;
            bt[tid] = (tid < n) ? conv_beta(gb, p.conv) : 0.f;
        }
        __syncthreads();
        if (c0 + C < Tb) load_chunk(c0 + C);  // in flight while this chunk is computed
        if (p.conv & GDN_QK_L2NORM) {
            // q and k normalised in the kernel, one warp per row; q then scaled
            for (int r = warp; r < 2 * C; r += kThreads / 32) {
                float *row = (r < C) ? Ks + r * KS : Qs + (r - C) * KS;
                float ss = 0.f;
                for (int j = lane; j < DK; j += 32) ss += row[j] * row[j];
                ss = group_sum<32>(ss);
                const float f = l2norm_factor(ss) * ((r < C) ? 1.f : scale);
                for (int j = lane; j < DK; j += 32) row[j] *= f;
            }
            __syncthreads();
        }

        // ---- 2. cumulative log decay (warp 0) ------------------------------
        if (warp == 0) {
            float x0 = (lane < C) ? lg[lane] : 0.f;
            float x1 = (lane + 32 < C) ? lg[lane + 32] : 0.f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                float y0 = __shfl_up_sync(0xffffffffu, x0, o);
                float y1 = __shfl_up_sync(0xffffffffu, x1, o);
                if (lane >= o) { x0 += y0; x1 += y1; }
            }
            x1 += __shfl_sync(0xffffffffu, x0, 31);
            const float glast = (C > 32) ? __shfl_sync(0xffffffffu, x1, (C - 33) & 31)
                                         : __shfl_sync(0xffffffffu, x0, (C - 1) & 31);
            if (lane < C) { lg[lane] = x0; eg[lane] = expf(x0); wg[lane] = expf(glast - x0); }
            if (lane + 32 < C) { lg[lane + 32] = x1; eg[lane + 32] = expf(x1); wg[lane + 32] = expf(glast - x1); }
        }
        __syncthreads();

        // ---- 3. [K; Q] [K^T | S^T] on the warp-level tensor cores (3 x tf32):
        // warp w < C / 8 takes rows 16w .. 16w + 15 of [K; Q] (K rows, then Q
        // rows); its fragments give A or P (decay and mask applied) and R (in
        // place over V) or the readout from the chunk's start state.
        if (warp < C / 8) {
            const int g = lane >> 2, t4 = lane & 3;
            const bool krows = 16 * warp < C;
            const int r0 = krows ? 16 * warp : 16 * warp - C;  // first row within K or Q
            const float *M = krows ? Ks : Qs;
            constexpr int NA = C / 8, NS8 = kDVT / 8;  // n-tiles of K^T and of S^T
            float acc[NA + NS8][4];
#pragma unroll
            for (int n = 0; n < NA + NS8; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
            for (int k0 = 0; k0 < DK; k0 += 8) {
                const SplitA a = load_a(M, KS, r0, k0, g, t4);
                SplitB bf[NA + NS8];
#pragma unroll
                for (int n = 0; n < NA; ++n) bf[n] = load_bt(Ks, KS, 8 * n, k0, g, t4);
#pragma unroll
                for (int n = 0; n < NS8; ++n) bf[NA + n] = load_bt(Ss, KS, 8 * n, k0, g, t4);
                mma_3xtf32_n<NA + NS8>(acc, a, bf);
            }
            // element e of a fragment: row r0 + g + 8 (e / 2), column 8 n + 2 t4 + e % 2
#pragma unroll
            for (int n = 0; n < NA; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int t = r0 + g + 8 * (e >> 1), i = 8 * n + 2 * t4 + (e & 1);
                    const float decay = (i <= t) ? expf(lg[t] - lg[i]) : 0.f;
                    if (krows) As[t * AS + i] = (i < t) ? bt[t] * decay * acc[n][e] : 0.f;
                    else Ps[t * AS + i] = (i <= t) ? decay * acc[n][e] : 0.f;
                }
#pragma unroll
            for (int n = 0; n < NS8; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int t = r0 + g + 8 * (e >> 1), i = 8 * n + 2 * t4 + (e & 1);
                    if (krows) Vs[t * DS + i] = bt[t] * (Vs[t * DS + i] - eg[t] * acc[NA + n][e]);
                    else Os[t * DS + i] = eg[t] * acc[NA + n][e];
                }
        }
        __syncthreads();

        // ---- 4. Delta = (I + A)^{-1} R by forward substitution in registers:
        // warp w owns columns 4w .. 4w+3, lane 8 ci + rg rows rg, rg + 8, ... of
        // column 4w + ci.  Row s is final once the rows above it have been
        // folded in; its owner broadcasts it to the column's 8 lanes, which
        // subtract A[t][s] x_s from their rows (A[t][s] = 0 for t <= s).
        {
            constexpr int RPL = C / 8;  // rows per lane
            const int rg = lane & 7, i = warp * 4 + (lane >> 3);
            float x[RPL];
#pragma unroll
            for (int k = 0; k < RPL; ++k) x[k] = Vs[(rg + 8 * k) * DS + i];
#pragma unroll
            for (int s = 0; s < C - 1; ++s) {
                const float xs = __shfl_sync(0xffffffffu, x[s >> 3], (lane & ~7) | (s & 7));
#pragma unroll
                for (int k = s >> 3; k < RPL; ++k) x[k] = fmaf(-As[(rg + 8 * k) * AS + s], xs, x[k]);
            }
#pragma unroll
            for (int k = 0; k < RPL; ++k) Vs[(rg + 8 * k) * DS + i] = x[k];
        }
        __syncthreads();

        // ---- 4b. capture: delta of the tile's rows, decay and shared key -----
        if (c0 < ncap) {
            const int nc = (ncap - c0 < n) ? (ncap - c0) : n;
            float *su0 = p.su + ((long)b * p.capacity + c0) * slot;
            for (int e = tid; e < nc * kDVT; e += kThreads) {
                const int t = e / kDVT, i = e % kDVT;
                su0[t * slot + Hv + (long)Hk * DK + (long)h * dv + row0 + i] = Vs[t * DS + i];
            }
            if (tile == 0) {
                for (int t = tid; t < nc; t += kThreads)
                    su0[t * slot + h] = conv_alpha(ld_gate(p.alpha, (tok0 + c0 + t) * Hv + h, p.dt_gate), p.conv);
                if (h % (Hv / Hk) == 0)
                    for (int e = tid; e < nc * DK; e += kThreads) {
                        const int t = e / DK, j = e % DK;
                        su0[t * slot + Hv + (long)hk * DK + j] = Ks[t * KS + j];
                    }
            }
        }

        // ---- 5a. outputs O = Os + P Delta: 2 tokens x 4 columns per thread ---
        for (int blk = tid; blk < (C / 2) * (kDVT / 4); blk += kThreads) {
            const int t0 = (blk / (kDVT / 4)) * 2, i0 = (blk % (kDVT / 4)) * 4;
            float4 acc[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) acc[r] = *reinterpret_cast<const float4 *>(Os + (t0 + r) * DS + i0);
            for (int s = 0; s <= t0 + 1; ++s) {  // P[t][s] = 0 for s > t
                const float4 d = *reinterpret_cast<const float4 *>(Vs + s * DS + i0);
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const float pr = Ps[(t0 + r) * AS + s];
                    acc[r].x += pr * d.x;
                    acc[r].y += pr * d.y;
                    acc[r].z += pr * d.z;
                    acc[r].w += pr * d.w;
                }
            }
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                if (t0 + r < n) {
                    TQ *o = ob + ((tok0 + c0 + t0 + r) * Hv + h) * (long)dv + row0 + i0;
                    st_out(o, acc[r].x);
                    st_out(o + 1, acc[r].y);
                    st_out(o + 2, acc[r].z);
                    st_out(o + 3, acc[r].w);
                }
            }
        }
        // ---- 5b. S <- e^{g_last} S + Delta^T diag(e^{g_last - g}) K (3 x tf32):
        // the 32 x DK state as 2 x DK / 8 fragment tiles, DK / 32 per warp
        {
            const int g = lane >> 2, t4 = lane & 3;
            const float glast = eg[C - 1];
            // warp w: state rows 16 m .. (m = w / 4), columns 8 n .. for its NP n-tiles
            constexpr int NP = DK / 32;
            const int m = warp >> 2, nb = (warp & 3) * NP;
            float acc[NP][4];
#pragma unroll
            for (int pi = 0; pi < NP; ++pi)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[pi][e] = 0.f;
            for (int k0 = 0; k0 < C; k0 += 8) {
                // A = (diag(w) Delta)^T: A[i][s] = w_s Delta[s][i]; B = K: B[s][j] = K[s][j]
                SplitA a;
                split_tf32(wg[k0 + t4] * Vs[(k0 + t4) * DS + 16 * m + g], a.big[0], a.small[0]);
                split_tf32(wg[k0 + t4] * Vs[(k0 + t4) * DS + 16 * m + g + 8], a.big[1], a.small[1]);
                split_tf32(wg[k0 + t4 + 4] * Vs[(k0 + t4 + 4) * DS + 16 * m + g], a.big[2], a.small[2]);
                split_tf32(wg[k0 + t4 + 4] * Vs[(k0 + t4 + 4) * DS + 16 * m + g + 8], a.big[3], a.small[3]);
                SplitB bk[NP];
#pragma unroll
                for (int pi = 0; pi < NP; ++pi) {
                    split_tf32(Ks[(k0 + t4) * KS + 8 * (nb + pi) + g], bk[pi].big[0], bk[pi].small[0]);
                    split_tf32(Ks[(k0 + t4 + 4) * KS + 8 * (nb + pi) + g], bk[pi].big[1], bk[pi].small[1]);
                }
                mma_3xtf32_n<NP>(acc, a, bk);
            }
#pragma unroll
            for (int pi = 0; pi < NP; ++pi)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float *sp = Ss + (16 * m + g + 8 * (e >> 1)) * KS + 8 * (nb + pi) + 2 * t4 + (e & 1);
                    *sp = fmaf(glast, *sp, acc[pi][e]);
                }
        }
        __syncthreads();
        // ---- 6. chunk-boundary checkpoint ------------------------------------
        const int ck = ckpt_slot(p, c0 / C, Tb);
        if (ck >= 0) {
            float *dst = p.ckpt + ((((long)b * p.ckpt_cap + ck) * Hv + h) * dv + row0) * DK;
            for (int e = tid; e < kDVT * DK / 4; e += kThreads) {
                const int i = e / (DK / 4), j = (e % (DK / 4)) * 4;
                __stcs(reinterpret_cast<float4 *>(dst + (long)i * DK + j),
                       *reinterpret_cast<const float4 *>(Ss + i * KS + j));
            }
        }
    }

    if (p.s_final != nullptr) {
        float *sf = p.s_final + (((long)b * Hv + h) * dv + row0) * DK;
        for (int e = tid; e < kDVT * DK / 4; e += kThreads) {
            const int i = e / (DK / 4), j = (e % (DK / 4)) * 4;
            *reinterpret_cast<float4 *>(sf + (long)i * DK + j) =
                *reinterpret_cast<const float4 *>(Ss + i * KS + j);
        }
    }
}

template <int DK, int C, typename TQ>
cudaError_t launch_t(const PrefillParams &p, cudaStream_t stream) {
    auto kern = prefill_simt_kernel<DK, C, TQ>;
    const size_t bytes = SimtSmem<DK, C>::kBytes;
    cudaError_t e = set_smem_once<prefill_simt_kernel<DK, C, TQ>>((int)bytes);
    if (e != cudaSuccess) return e;
    dim3 grid(p.dv / kDVT, p.Hv, p.B);
    kern<<<grid, kThreads, bytes, stream>>>(p);
    return cudaGetLastError();
}

template <int DK, int C>
cudaError_t launch_c(const PrefillParams &p, cudaStream_t stream) {
    switch (p.dt_qkv) {
        case GDN_F32: return launch_t<DK, C, float>(p, stream);
        case GDN_F16: return launch_t<DK, C, __half>(p, stream);
        default: return launch_t<DK, C, __nv_bfloat16>(p, stream);
    }
}

template <int DK>
cudaError_t launch_dk(const PrefillParams &p, cudaStream_t stream) {
    switch (p.chunk) {
        case 16: return launch_c<DK, 16>(p, stream);
        case 32: return launch_c<DK, 32>(p, stream);
        default: return launch_c<DK, 64>(p, stream);
    }
}

}  // namespace

bool prefill_simt_supported(int dk, int dv, int chunk) {
    return (dk == 32 || dk == 64 || dk == 128) && (dv == 32 || dv == 64 || dv == 128) &&
           (chunk == 16 || chunk == 32 || chunk == 64);
}

cudaError_t launch_prefill_simt(const PrefillParams &p, cudaStream_t stream) {
    switch (p.dk) {
        case 32: return launch_dk<32>(p, stream);
        case 64: return launch_dk<64>(p, stream);
        default: return launch_dk<128>(p, stream);
    }
}

}  // namespace gdn
