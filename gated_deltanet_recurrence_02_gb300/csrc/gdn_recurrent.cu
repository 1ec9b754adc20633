// gdn_recurrent.cu -- per-token recurrent / decode path with compact capture.
//
// Work unit: a tile of 32 rows of one state matrix (row b, value head h),
// processed by 4 warps -- each warp 2 passes of 4 rows, each row split over 8
// lanes that hold dk/8 columns as float4s.  The 32 rows are contiguous in HBM,
// so one bulk (1-D TMA) copy stages a tile in shared memory.  The kernel is
// persistent and warp-specialised: a grid of (SMs x 4) CTAs walks the tiles
// with a grid stride; in each CTA a producer warp stages three tiles ahead --
// the state tile, the first token's k, q and v slice (bulk copies) and a
// header with its gates, capture count and row bounds -- and four compute
// warps work from shared memory only, so neither HBM nor L2 latency sits on
// their path.  A tile stays on chip
// across all tokens of the call and the last token writes it back with
// 128-bit streaming stores -- a decode step moves exactly the state's bytes
// plus the token vectors.
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
#include "tc_ptx.cuh"

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

constexpr int kStages = 3;       // tiles in flight per CTA
constexpr int kCtasPerSm = 4;    // persistent CTAs per SM
constexpr int kComputeWarps = kWarps;
constexpr int kCtaThreads = kThreads + 32;  // + one producer warp

// Per-stage header, written by the producer before it arrives on the stage.
struct TileHeader {
    long tok0;
    int b, h, tt, Tb, ncap, has_state;
    float alpha0, beta0;  // gates of the tile's first token
};

template <int DK, typename TQ>
struct StageLayout {
    static constexpr uint32_t kState = kRowsPerCta * DK * sizeof(float);
    static constexpr uint32_t kVec = DK * sizeof(TQ);         // k or q of one token
    static constexpr uint32_t kV = kRowsPerCta * sizeof(TQ);  // the tile's slice of v
    static constexpr uint32_t oK = kState, oQ = oK + kVec, oV = oQ + kVec;
    static constexpr uint32_t oH = (oV + kV + 15) / 16 * 16;
    static constexpr uint32_t kBytes = (oH + sizeof(TileHeader) + 127) / 128 * 128;
};

template <int DK, typename TQ>
__global__ void __launch_bounds__(kCtaThreads, kCtasPerSm)
recurrent_kernel(const RecurrentParams p) {
    using L = StageLayout<DK, TQ>;
    constexpr int F4 = DK / (4 * kLanesPerRow);  // float4 per lane per row
    constexpr uint32_t kTileFloats = kRowsPerCta * DK;
    extern __shared__ float4 smem4[];
    uint8_t *sbase = reinterpret_cast<uint8_t *>(smem4);
    uint64_t *full = reinterpret_cast<uint64_t *>(sbase + kStages * L::kBytes);
    uint64_t *empty = full + kStages;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hv = p.Hv, Hk = p.Hk, dv = p.dv;
    const int G = Hv / Hk;
    const int tiles_per_head = dv / kRowsPerCta;
    const long n_tiles = (long)p.B * Hv * tiles_per_head;
    const long slot = (long)Hv + (long)Hk * DK + (long)Hv * dv;
    const bool active = (p.active == nullptr) || (*p.active != 0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], kComputeWarps);
        }
        tc::fence_mbar_init();
    }
    __syncthreads();

    // ======================= producer warp ================================
    if (warp == kComputeWarps) {
        if (lane != 0) return;
        int it = 0;
        for (long id = blockIdx.x; id < n_tiles; id += gridDim.x, ++it) {
            const int stage = it % kStages;
            if (it >= kStages && !tc::mbar_wait(&empty[stage], ((it / kStages) - 1) & 1, 1000000000ull)) {
                atomicOr(p.err, (uint32_t)GDN_DEVERR_TIMEOUT);
                return;
            }
            uint8_t *st = sbase + stage * L::kBytes;
            TileHeader hd;
            hd.tt = (int)(id % tiles_per_head);
            const long bh = id / tiles_per_head;
            hd.h = (int)(bh % Hv);
            hd.b = (int)(bh / Hv);
            row_range(p.cu_seqlens, hd.b, p.T, hd.tok0, hd.Tb);
            hd.ncap = 0;
            if (p.capacity > 0 && active) {
                const int c = p.capture_count[hd.b];
                const int lim = p.capacity < hd.Tb ? p.capacity : hd.Tb;
                hd.ncap = c < 0 ? 0 : (c > lim ? lim : c);
            }
            const float *s0 = initial_state_ptr(p.s0, p.s0_idx, p.n_s0, hd.b, hd.h, Hv, dv, DK, p.err);
            hd.has_state = s0 != nullptr;
            hd.alpha0 = hd.Tb > 0 ? ld_gate(p.alpha, hd.tok0 * Hv + hd.h, p.dt_gate) : 0.f;
            hd.beta0 = hd.Tb > 0 ? ld_gate(p.beta, hd.tok0 * Hv + hd.h, p.dt_gate) : 0.f;
            *reinterpret_cast<TileHeader *>(st + L::oH) = hd;
            uint32_t tx = 0;
            if (s0 != nullptr) tx += L::kState;
            if (hd.Tb > 0) tx += 2 * L::kVec + L::kV;
            // the arrive releases the header; the copies complete the phase
            tc::mbar_arrive_expect_tx(&full[stage], tx);
            if (s0 != nullptr) tc::bulk_load(st, s0 + (long)hd.tt * kTileFloats, L::kState, &full[stage]);
            if (hd.Tb > 0) {
                const int hk = hd.h / G;
                const TQ *kt = reinterpret_cast<const TQ *>(p.k) + (hd.tok0 * Hk + hk) * DK;
                const TQ *qt = reinterpret_cast<const TQ *>(p.q) + (hd.tok0 * Hk + hk) * DK;
                const TQ *vt = reinterpret_cast<const TQ *>(p.v) + (hd.tok0 * Hv + hd.h) * (long)dv +
                               hd.tt * kRowsPerCta;
                tc::bulk_load(st + L::oK, kt, L::kVec, &full[stage]);
                tc::bulk_load(st + L::oQ, qt, L::kVec, &full[stage]);
                tc::bulk_load(st + L::oV, vt, L::kV, &full[stage]);
            }
        }
        // drain: the copies of the last tiles must land before this warp exits
        for (int s = 0; s < kStages && it - 1 - s >= 0; ++s) {
            const int j = it - 1 - s;
            tc::mbar_wait(&full[j % kStages], (j / kStages) & 1, 1000000000ull);
        }
        return;
    }

    // ======================= compute warps ================================
    const int grp = lane / kLanesPerRow, l8 = lane % kLanesPerRow;
    // Inactive capture: every CTA zeroes its share of the whole buffer.
    if (p.capacity > 0 && !active) {
        const long total = (long)p.B * p.capacity * slot;
        const long per = (total + gridDim.x - 1) / gridDim.x;
        const long e0 = (long)blockIdx.x * per;
        const long e1 = (e0 + per < total) ? e0 + per : total;
        for (long e = e0 + threadIdx.x; e < e1; e += kThreads) p.su[e] = 0.0f;
    }
    const TQ *qb = reinterpret_cast<const TQ *>(p.q);
    const TQ *kb = reinterpret_cast<const TQ *>(p.k);
    const TQ *vb = reinterpret_cast<const TQ *>(p.v);
    TQ *ob = reinterpret_cast<TQ *>(p.out);
    const float scale = p.scale;
    int lrow[kPasses];  // row inside the tile
#pragma unroll
    for (int r = 0; r < kPasses; ++r) lrow[r] = warp * kRowsPerWarp + r * (32 / kLanesPerRow) + grp;

    int it = 0;
    for (long id = blockIdx.x; id < n_tiles; id += gridDim.x, ++it) {
        const int stage = it % kStages;
        uint8_t *st = sbase + stage * L::kBytes;
        float *sS = reinterpret_cast<float *>(st);
        if (!tc::mbar_wait(&full[stage], (it / kStages) & 1, 1000000000ull)) {
            if (threadIdx.x == 0) atomicOr(p.err, (uint32_t)GDN_DEVERR_TIMEOUT);
            break;
        }
        const TileHeader hd = *reinterpret_cast<const TileHeader *>(st + L::oH);
        const int b = hd.b, h = hd.h, hk = h / G, row0 = hd.tt * kRowsPerCta, Tb = hd.Tb;
        float *su_row = (p.capacity > 0) ? p.su + (long)b * p.capacity * slot : nullptr;
        float *sf = (p.s_final != nullptr) ? p.s_final + (((long)b * Hv + h) * dv + row0) * DK : nullptr;
        if (!hd.has_state) {
#pragma unroll
            for (int r = 0; r < kPasses; ++r)
#pragma unroll
                for (int f = 0; f < F4; ++f)
                    *reinterpret_cast<float4 *>(sS + lrow[r] * DK + (f * kLanesPerRow + l8) * 4) =
                        make_float4(0.f, 0.f, 0.f, 0.f);
        }

        if (Tb == 0 && sf != nullptr) {
#pragma unroll
            for (int r = 0; r < kPasses; ++r)
#pragma unroll
                for (int f = 0; f < F4; ++f) {
                    const int col = (f * kLanesPerRow + l8) * 4;
                    __stcs(reinterpret_cast<float4 *>(sf + (long)lrow[r] * DK + col),
                           *reinterpret_cast<const float4 *>(sS + lrow[r] * DK + col));
                }
        }

        for (int t = 0; t < Tb; ++t) {
            const long tok = hd.tok0 + t;
            const bool last = (t == Tb - 1);
            // token 0 comes from the stage; later tokens (T > 1) straight from memory
            const TQ *kt = (t == 0) ? reinterpret_cast<const TQ *>(st + L::oK) : kb + (tok * Hk + hk) * DK;
            const TQ *qt = (t == 0) ? reinterpret_cast<const TQ *>(st + L::oQ) : qb + (tok * Hk + hk) * DK;
            float kq = 0.f;
#pragma unroll
            for (int f = 0; f < F4; ++f) {
                const int col = (f * kLanesPerRow + l8) * 4;
                kq += dot4(ld4(kt + col), ld4(qt + col));
            }
            kq = group_sum<kLanesPerRow>(kq) * scale;
            const float a = (t == 0) ? hd.alpha0 : ld_gate(p.alpha, tok * Hv + h, p.dt_gate);
            const float bt = (t == 0) ? hd.beta0 : ld_gate(p.beta, tok * Hv + h, p.dt_gate);
            const bool cap = t < hd.ncap;
            float *su_t = cap ? su_row + (long)t * slot : nullptr;

#pragma unroll
            for (int r = 0; r < kPasses; ++r) {
                float4 Sr[F4], kv[F4];
                float sk = 0.f, sq = 0.f;
#pragma unroll
                for (int f = 0; f < F4; ++f) {
                    const int col = (f * kLanesPerRow + l8) * 4;
                    Sr[f] = *reinterpret_cast<const float4 *>(sS + lrow[r] * DK + col);
                    kv[f] = ld4(kt + col);
                    sk += dot4(Sr[f], kv[f]);
                    sq += dot4(Sr[f], ld4(qt + col));
                }
                sk = group_sum<kLanesPerRow>(sk);
                sq = group_sum<kLanesPerRow>(sq) * scale;
                const float vi = (t == 0) ? ld_f(reinterpret_cast<const TQ *>(st + L::oV) + lrow[r])
                                          : ld_f(vb + (tok * Hv + h) * (long)dv + row0 + lrow[r]);
                const float delta = bt * (vi - a * sk);
#pragma unroll
                for (int f = 0; f < F4; ++f) {
                    const int col = (f * kLanesPerRow + l8) * 4;
                    float4 n;
                    n.x = fmaf(a, Sr[f].x, delta * kv[f].x);
                    n.y = fmaf(a, Sr[f].y, delta * kv[f].y);
                    n.z = fmaf(a, Sr[f].z, delta * kv[f].z);
                    n.w = fmaf(a, Sr[f].w, delta * kv[f].w);
                    if (!last)
                        *reinterpret_cast<float4 *>(sS + lrow[r] * DK + col) = n;
                    else if (sf != nullptr)
                        __stcs(reinterpret_cast<float4 *>(sf + (long)lrow[r] * DK + col), n);
                }
                if (l8 == 0) {
                    st_out(ob + (tok * Hv + h) * (long)dv + row0 + lrow[r], fmaf(a, sq, delta * kq));
                    if (cap) su_t[Hv + (long)Hk * DK + (long)h * dv + row0 + lrow[r]] = delta;
                }
            }
            if (cap && hd.tt == 0) {
                if (threadIdx.x == 0) su_t[h] = a;
                // the first value head of the group stores the shared key once
                if (h % G == 0 && warp == 0 && grp == 0) {
                    float *kd = su_t + Hv + (long)hk * DK;
#pragma unroll
                    for (int f = 0; f < F4; ++f) {
                        const int col = (f * kLanesPerRow + l8) * 4;
                        const float4 kk = ld4(kt + col);
                        kd[col + 0] = kk.x;
                        kd[col + 1] = kk.y;
                        kd[col + 2] = kk.z;
                        kd[col + 3] = kk.w;
                    }
                }
            }
        }
        // this warp is done with the stage (the proxy fence orders its shared
        // writes before the copy that will overwrite them)
        tc::fence_proxy_async();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&empty[stage]);
    }
}

int sm_count() {
    static int n = 0;
    if (n == 0) {
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
            n = v;
        else
            n = 132;
    }
    return n;
}

template <int DK, typename TQ>
cudaError_t launch_t(const RecurrentParams &p, cudaStream_t stream) {
    auto kern = recurrent_kernel<DK, TQ>;
    const size_t bytes = (size_t)kStages * StageLayout<DK, TQ>::kBytes + 2 * kStages * sizeof(uint64_t);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    const long tiles = (long)p.B * p.Hv * (p.dv / kRowsPerCta);
    const long cap = (long)sm_count() * kCtasPerSm;
    const unsigned grid = (unsigned)(tiles < cap ? tiles : cap);
    kern<<<grid, kCtaThreads, bytes, stream>>>(p);
    return cudaGetLastError();
}

template <int DK>
cudaError_t launch_dk(const RecurrentParams &p, cudaStream_t stream) {
    switch (p.dt_qkv) {
        case GDN_F32: return launch_t<DK, float>(p, stream);
        case GDN_F16: return launch_t<DK, __half>(p, stream);
        default: return launch_t<DK, __nv_bfloat16>(p, stream);
    }
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
