// gdn_recurrent.cu -- per-token recurrent / decode path with compact capture.
//
// One CTA owns 32 rows of one state matrix (row b, value head h): 4 warps,
// each warp 2 passes of 4 rows, each row split over 8 lanes that hold dk/8
// consecutive-in-groups-of-4 columns as float4 registers.  The state is read
// once from HBM with 128-bit streaming loads, stays in registers across all
// tokens of the call, and is written back once with 128-bit streaming stores,
// so a decode step moves exactly the state's bytes plus the token vectors.
// S k and S q are 8-lane butterfly reductions; the key/query head is shared by
// the G = Hv / Hk value heads that read it (inverse GQA).
//
// Per token (gated delta rule): delta = beta (v - alpha S_old k) is the delta
// formed with the decayed state, S <- alpha S_old + delta k^T, and the
// readout with the updated state is alpha (S_old q) + delta (k . q).
//
// Capture ("[WebGPU EP] adds state update capacity support for GatedDeltaNet",
// onnxruntime PR 32767, "Changes"): tokens t < n_b of row b write decay,
// shared key and delta into slot t; with state_update_active == 0 the whole
// buffer is zeroed instead and nothing else is written to it.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kLanesPerRow = 8;
constexpr int kWarps = 4;
constexpr int kPasses = 2;
constexpr int kRowsPerWarp = (32 / kLanesPerRow) * kPasses;  // 8
constexpr int kRowsPerCta = kWarps * kRowsPerWarp;            // 32
constexpr int kThreads = kWarps * 32;

__device__ __forceinline__ float dot4(float4 a, float4 b) {
    return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

template <int DK, typename TQ>
__global__ void __launch_bounds__(kThreads)
recurrent_kernel(const RecurrentParams p) {
    constexpr int F4 = DK / (4 * kLanesPerRow);  // float4 per lane per row
    const int tile = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = lane / kLanesPerRow, l8 = lane % kLanesPerRow;
    const int Hv = p.Hv, Hk = p.Hk, dv = p.dv;
    const int G = Hv / Hk, hk = h / G;

    long tok0;
    int Tb;
    row_range(p.cu_seqlens, b, p.T, tok0, Tb);

    // ---- capture bookkeeping ------------------------------------------
    const long slot = (long)Hv + (long)Hk * DK + (long)Hv * dv;
    const bool active = (p.active == nullptr) || (*p.active != 0);
    int ncap = 0;
    if (p.capacity > 0) {
        if (!active) {
            // Inactive: this CTA zeroes its share of the whole buffer.
            const long total = (long)p.B * p.capacity * slot;
            const long ncta = (long)gridDim.x * gridDim.y * gridDim.z;
            const long cid = blockIdx.x + (long)gridDim.x * (blockIdx.y + (long)gridDim.y * blockIdx.z);
            const long per = (total + ncta - 1) / ncta;
            const long e0 = cid * per;
            const long e1 = (e0 + per < total) ? e0 + per : total;
            for (long e = e0 + threadIdx.x; e < e1; e += kThreads) p.su[e] = 0.0f;
        } else {
            int c = p.capture_count[b];
            int lim = p.capacity < Tb ? p.capacity : Tb;
            ncap = c < 0 ? 0 : (c > lim ? lim : c);
        }
    }
    float *su_row = (p.capacity > 0) ? p.su + (long)b * p.capacity * slot : nullptr;

    // ---- load the state rows ------------------------------------------
    int row[kPasses];
#pragma unroll
    for (int r = 0; r < kPasses; ++r)
        row[r] = tile * kRowsPerCta + warp * kRowsPerWarp + r * (32 / kLanesPerRow) + grp;

    const float *s0 = initial_state_ptr(p.s0, p.s0_idx, p.n_s0, b, h, Hv, dv, DK, p.err);
    float4 S[kPasses][F4];
#pragma unroll
    for (int r = 0; r < kPasses; ++r)
#pragma unroll
        for (int f = 0; f < F4; ++f) {
            const int col = (f * kLanesPerRow + l8) * 4;
            S[r][f] = s0 ? __ldcs(reinterpret_cast<const float4 *>(s0 + (long)row[r] * DK + col))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }

    const TQ *qb = reinterpret_cast<const TQ *>(p.q);
    const TQ *kb = reinterpret_cast<const TQ *>(p.k);
    const TQ *vb = reinterpret_cast<const TQ *>(p.v);
    TQ *ob = reinterpret_cast<TQ *>(p.out);
    const float scale = p.scale;

    // ---- token loop -----------------------------------------------------
    for (int t = 0; t < Tb; ++t) {
        const long tok = tok0 + t;
        const TQ *kt = kb + (tok * Hk + hk) * DK;
        const TQ *qt = qb + (tok * Hk + hk) * DK;
        float4 kv[F4], qv[F4];
        float kq = 0.f;
#pragma unroll
        for (int f = 0; f < F4; ++f) {
            const int col = (f * kLanesPerRow + l8) * 4;
            kv[f] = ld4(kt + col);
            float4 qq = ld4(qt + col);
            qv[f] = make_float4(qq.x * scale, qq.y * scale, qq.z * scale, qq.w * scale);
            kq += dot4(kv[f], qv[f]);
        }
        kq = group_sum<kLanesPerRow>(kq);
        const float a = ld_gate(p.alpha, tok * Hv + h, p.dt_gate);
        const float bt = ld_gate(p.beta, tok * Hv + h, p.dt_gate);
        const bool cap = t < ncap;
        float *su_t = cap ? su_row + (long)t * slot : nullptr;

#pragma unroll
        for (int r = 0; r < kPasses; ++r) {
            float sk = 0.f, sq = 0.f;
#pragma unroll
            for (int f = 0; f < F4; ++f) {
                sk += dot4(S[r][f], kv[f]);
                sq += dot4(S[r][f], qv[f]);
            }
            sk = group_sum<kLanesPerRow>(sk);
            sq = group_sum<kLanesPerRow>(sq);
            const float vi = ld_f(vb + (tok * Hv + h) * (long)dv + row[r]);
            const float delta = bt * (vi - a * sk);
#pragma unroll
            for (int f = 0; f < F4; ++f) {
                S[r][f].x = fmaf(a, S[r][f].x, delta * kv[f].x);
                S[r][f].y = fmaf(a, S[r][f].y, delta * kv[f].y);
                S[r][f].z = fmaf(a, S[r][f].z, delta * kv[f].z);
                S[r][f].w = fmaf(a, S[r][f].w, delta * kv[f].w);
            }
            if (l8 == 0) {
                st_out(ob + (tok * Hv + h) * (long)dv + row[r], fmaf(a, sq, delta * kq));
                if (cap) su_t[Hv + (long)Hk * DK + (long)h * dv + row[r]] = delta;
            }
        }
        if (cap && tile == 0) {
            if (threadIdx.x == 0) su_t[h] = a;
            // the first value head of the group stores the shared key once
            if (h % G == 0 && warp == 0 && grp == 0) {
                float *kd = su_t + Hv + (long)hk * DK;
#pragma unroll
                for (int f = 0; f < F4; ++f) {
                    const int col = (f * kLanesPerRow + l8) * 4;
                    kd[col + 0] = kv[f].x;
                    kd[col + 1] = kv[f].y;
                    kd[col + 2] = kv[f].z;
                    kd[col + 3] = kv[f].w;
                }
            }
        }
    }

    // ---- write the state back -------------------------------------------
    if (p.s_final != nullptr) {
        float *sf = p.s_final + (((long)b * Hv + h) * dv) * DK;
#pragma unroll
        for (int r = 0; r < kPasses; ++r)
#pragma unroll
            for (int f = 0; f < F4; ++f) {
                const int col = (f * kLanesPerRow + l8) * 4;
                __stcs(reinterpret_cast<float4 *>(sf + (long)row[r] * DK + col), S[r][f]);
            }
    }
}

template <int DK>
cudaError_t launch_dk(const RecurrentParams &p, cudaStream_t stream) {
    dim3 grid(p.dv / kRowsPerCta, p.Hv, p.B);
    switch (p.dt_qkv) {
        case GDN_F32: recurrent_kernel<DK, float><<<grid, kThreads, 0, stream>>>(p); break;
        case GDN_F16: recurrent_kernel<DK, __half><<<grid, kThreads, 0, stream>>>(p); break;
        default: recurrent_kernel<DK, __nv_bfloat16><<<grid, kThreads, 0, stream>>>(p); break;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_recurrent(const RecurrentParams &p, cudaStream_t stream) {
    switch (p.dk) {
        case 32: return launch_dk<32>(p, stream);
        case 64: return launch_dk<64>(p, stream);
        default: return launch_dk<128>(p, stream);
    }
}

}  // namespace gdn
