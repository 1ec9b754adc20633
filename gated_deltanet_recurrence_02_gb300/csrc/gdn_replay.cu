// gdn_replay.cu -- replay of captured state updates after an accepted prefix.
//
// "[WebGPU EP] adds state update capacity support for GatedDeltaNet"
// (onnxruntime PR 32767), "Changes" / "DFlash2 Prerequisite": the captured
// factors replay S = decay * S + outer(key, delta).  With S stored [dv, dk],
// entry (i, j) becomes decay * S[i][j] + delta[i] * key[j], for the first m_b
// slots of row b, m_b = clamp(accepted_count[b], 0, capacity).
//
// Same register layout as the recurrent kernel: a CTA owns 32 rows of one
// (row, value head) state, each row spread over 8 lanes as float4s.  There is
// no reduction: the state streams HBM -> registers -> HBM once, and the
// factors (a few KB per row) come through L1/L2.  Slots are not 16-byte
// aligned in general (slot width Hv + Hk*dk + Hv*dv floats), so the factors
// are read as scalars.  In place with m_b == 0 the rows are left untouched.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kLanesPerRow = 8;
constexpr int kWarps = 4;
constexpr int kPasses = 2;
constexpr int kRowsPerWarp = (32 / kLanesPerRow) * kPasses;
constexpr int kRowsPerCta = kWarps * kRowsPerWarp;
constexpr int kThreads = kWarps * 32;

template <int DK>
__global__ void __launch_bounds__(kThreads) replay_kernel(const ReplayParams p) {
    constexpr int F4 = DK / (4 * kLanesPerRow);
    const int tile = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = lane / kLanesPerRow, l8 = lane % kLanesPerRow;
    const int Hv = p.Hv, Hk = p.Hk, dv = p.dv;
    const int hk = h / (Hv / Hk);
    const long slot = (long)Hv + (long)Hk * DK + (long)Hv * dv;

    int m = p.accepted[b];
    m = m < 0 ? 0 : (m > p.capacity ? p.capacity : m);
    if (m == 0 && p.s_out == p.s_in) return;

    const long base = (((long)b * Hv + h) * dv) * DK;
    const float *si = p.s_in + base;
    float *so = p.s_out + base;
    int row[kPasses];
    float4 S[kPasses][F4];
#pragma unroll
    for (int r = 0; r < kPasses; ++r) {
        row[r] = tile * kRowsPerCta + warp * kRowsPerWarp + r * (32 / kLanesPerRow) + grp;
#pragma unroll
        for (int f = 0; f < F4; ++f) {
            const int col = (f * kLanesPerRow + l8) * 4;
            S[r][f] = __ldcs(reinterpret_cast<const float4 *>(si + (long)row[r] * DK + col));
        }
    }

    const float *su_row = p.su + (long)b * p.capacity * slot;
    for (int t = 0; t < m; ++t) {
        const float *s = su_row + (long)t * slot;
        const float decay = s[h];
        const float *key = s + Hv + (long)hk * DK;
        const float *delta = s + Hv + (long)Hk * DK + (long)h * dv;
        float4 kv[F4];
#pragma unroll
        for (int f = 0; f < F4; ++f) {
            const int col = (f * kLanesPerRow + l8) * 4;
            kv[f] = make_float4(key[col], key[col + 1], key[col + 2], key[col + 3]);
        }
#pragma unroll
        for (int r = 0; r < kPasses; ++r) {
            const float d = delta[row[r]];
#pragma unroll
            for (int f = 0; f < F4; ++f) {
                S[r][f].x = fmaf(decay, S[r][f].x, d * kv[f].x);
                S[r][f].y = fmaf(decay, S[r][f].y, d * kv[f].y);
                S[r][f].z = fmaf(decay, S[r][f].z, d * kv[f].z);
                S[r][f].w = fmaf(decay, S[r][f].w, d * kv[f].w);
            }
        }
    }

#pragma unroll
    for (int r = 0; r < kPasses; ++r)
#pragma unroll
        for (int f = 0; f < F4; ++f) {
            const int col = (f * kLanesPerRow + l8) * 4;
            __stcs(reinterpret_cast<float4 *>(so + (long)row[r] * DK + col), S[r][f]);
        }
}

}  // namespace

cudaError_t launch_replay(const ReplayParams &p, cudaStream_t stream) {
    dim3 grid(p.dv / kRowsPerCta, p.Hv, p.B);
    switch (p.dk) {
        case 32: replay_kernel<32><<<grid, kThreads, 0, stream>>>(p); break;
        case 64: replay_kernel<64><<<grid, kThreads, 0, stream>>>(p); break;
        default: replay_kernel<128><<<grid, kThreads, 0, stream>>>(p); break;
    }
    return cudaGetLastError();
}

}  // namespace gdn
