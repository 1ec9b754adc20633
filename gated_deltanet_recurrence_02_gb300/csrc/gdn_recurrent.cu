// gdn_recurrent.cu -- per-token recurrent path (decode, verify, per-token
// prefill) with compact capture, and the fused replay + verify step.
//
// Work unit: a tile of 32 rows of one state matrix (row b, value head h),
// processed by CW compute warps (4 in both instances launched: each lane
// holds its dk/8 columns of two rows).  The
// 32 rows are contiguous in HBM, so one bulk (1-D TMA) copy stages a tile in
// shared memory.  The kernel is persistent and warp-specialised: a grid of
// (SMs x CTAs-per-SM) walks the tiles with a grid stride; in each CTA a
// producer warp stages three tiles ahead -- the state tile and the first TS
// tokens' k, q and v slice (bulk copies), their gates, the first RS replayed
// slots' factors and a header -- and the compute warps work from shared
// memory only, so neither HBM nor L2 latency sits on their path.  The compute
// lanes keep their state columns in registers (float2 pairs for the packed
// fp32x2 FMA) across all tokens of the call and write them back once with
// 128-bit streaming stores: a decode step moves the state's bytes plus the
// token vectors.  S k, S q and k q are 8-lane butterfly reductions; the
// key/query head is shared by the G = Hv / Hk value heads that read it
// (inverse GQA).
//
// Per token (gated delta rule): delta = beta (v - alpha S_old k) is the delta
// formed with the decayed state, S <- alpha S_old + delta k^T, and the
// readout with the updated state is alpha (S_old q) + delta (k . q).
//
// Capture ("[WebGPU EP] adds state update capacity support for GatedDeltaNet",
// onnxruntime PR 32767, "Changes"): tokens t < n_b of row b write decay,
// shared key and delta into slot t; with state_update_active == 0 the whole
// buffer is zeroed instead and nothing else is written to it.
//
// Fused replay + verify (same page, "DFlash2 Prerequisite": replay after
// partial acceptance): before the tokens, the first m_b slots of the previous
// capture are replayed on the registers, S <- decay S + delta key^T, with the
// same fp32 operations as the token update, and the committed state is
// written out; the drafts then run from it.
#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

constexpr int kLanesPerRow = 8;
constexpr int kRowsPerCta = 32;

__device__ __forceinline__ void split4(float4 v, float2 &lo, float2 &hi) {
    lo = make_float2(v.x, v.y);
    hi = make_float2(v.z, v.w);
}

// The lane's F4 float4 column groups of a dk-vector, widened to fp32 pairs.
template <int F4, typename TQ>
__device__ __forceinline__ void load_pairs(const TQ *p, int l8, float2 (&out)[2 * F4]) {
#pragma unroll
    for (int f = 0; f < F4; ++f) split4(ld4(p + (f * kLanesPerRow + l8) * 4), out[2 * f], out[2 * f + 1]);
}

// Partial dot product over the lane's columns (packed fp32x2 FMAs).
template <int F2>
__device__ __forceinline__ float dot_pairs(const float2 (&x)[F2], const float2 (&y)[F2]) {
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < F2; ++i) acc = __ffma2_rn(x[i], y[i], acc);
    return acc.x + acc.y;
}

// The lane's columns of one row, written with 128-bit streaming stores.
template <int DK, int F4>
__device__ __forceinline__ void store_row(float *dst, const float2 (&Sr)[2 * F4], int lrow, int l8) {
#pragma unroll
    for (int f = 0; f < F4; ++f)
        __stcs(reinterpret_cast<float4 *>(dst + (long)lrow * DK + (f * kLanesPerRow + l8) * 4),
               make_float4(Sr[2 * f].x, Sr[2 * f].y, Sr[2 * f + 1].x, Sr[2 * f + 1].y));
}

constexpr int kStages = 3;       // tiles in flight per CTA

// Per-stage header, written by the producer before it arrives on the stage.
struct TileHeader {
    long tok0;
    int b, h, tt, Tb, ncap, has_state;
    int m;  // replayed slots (fused replay + verify), 0 otherwise
};

constexpr uint32_t up16(uint32_t x) { return (x + 15u) / 16u * 16u; }

// One pipeline stage: the state tile, the first TS tokens' k, q and the
// tile's slice of v, the first RS replayed slots' key (fp32), the tile's
// slice of delta and the decay, then the TS tokens' gates and the header.
template <int DK, typename TQ, int TS, int RS>
struct StageLayout {
    static constexpr uint32_t kState = kRowsPerCta * DK * sizeof(float);
    static constexpr uint32_t kVec = DK * sizeof(TQ);         // k or q of one token
    static constexpr uint32_t kV = kRowsPerCta * sizeof(TQ);  // the tile's slice of v
    static constexpr uint32_t oK = kState;
    static constexpr uint32_t oQ = oK + TS * kVec;
    static constexpr uint32_t oV = oQ + TS * kVec;
    static constexpr uint32_t oRK = up16(oV + TS * kV);       // [RS][DK] replay keys
    static constexpr uint32_t oRD = oRK + RS * DK * 4;        // [RS][32] replay deltas
    static constexpr uint32_t oRA = oRD + RS * kRowsPerCta * 4;  // [RS] replay decays
    static constexpr uint32_t oG = up16(oRA + RS * 4);        // [TS] alpha, then [TS] beta
    static constexpr uint32_t oH = up16(oG + 2 * TS * 4);
    static constexpr uint32_t kBytes = (oH + sizeof(TileHeader) + 127) / 128 * 128;
};

// TS tokens and RS replayed slots per tile are staged in shared memory by the
// producer; later ones (long rows, large acceptance counts) are read by the
// compute warps straight from memory.  CPS = resident CTAs per SM.
template <int DK, typename TQ, int TS, int RS, int CPS, int CW>
__global__ void __launch_bounds__(CW * 32 + 32, CPS)
recurrent_kernel(const RecurrentParams p) {
    using L = StageLayout<DK, TQ, TS, RS>;
    // CW compute warps share the tile's 32 rows: each 8-lane group of a warp
    // holds NP rows (CW = 4: two rows, CW = 8: one row)
    constexpr int NP = 32 / (CW * 4);
    constexpr int kRowsW = 4 * NP;  // rows per compute warp
    constexpr int F4 = DK / (4 * kLanesPerRow);  // float4 per lane per row
    constexpr int F2 = 2 * F4;                   // the same columns as float2 pairs
    constexpr int KPL = DK / 32;                 // replay-key floats per producer lane
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
            tc::mbar_init(&empty[s], CW);
        }
        tc::fence_mbar_init();
    }
    __syncthreads();

    // ======================= producer warp ================================
    // Lane 0 issues the bulk copies; the lanes load the gates and the replay
    // factors (plain loads: slots are not 16-byte aligned in general) and
    // store them into the stage; lane 0's arrive then releases the stage.
    if (warp == CW) {
        int it = 0;
        for (long id = blockIdx.x; id < n_tiles; id += gridDim.x, ++it) {
            const int stage = it % kStages;
            if (it >= kStages && !tc::mbar_wait(&empty[stage], ((it / kStages) - 1) & 1, p.wait_ns)) {
                if (lane == 0) atomicOr(p.err, (uint32_t)GDN_DEVERR_TIMEOUT);
                break;
            }
            uint8_t *st = sbase + stage * L::kBytes;
            // every lane derives the header (same values; loads are broadcasts)
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
            hd.m = 0;
            if (p.rp_capacity > 0) {
                const int a = p.rp_accepted[hd.b];
                hd.m = a < 0 ? 0 : (a > p.rp_capacity ? p.rp_capacity : a);
            }
            const float *s0 = initial_state_ptr(p.s0, p.s0_idx, p.n_s0, hd.b, hd.h, Hv, dv, DK, p.err);
            hd.has_state = s0 != nullptr;
            const int hk = hd.h / G;
            const int nts = hd.Tb < TS ? hd.Tb : TS;
            if (lane == 0) {
                const uint32_t tx = (s0 != nullptr ? L::kState : 0u) + (uint32_t)nts * (2 * L::kVec + L::kV);
                tc::mbar_expect_tx(&full[stage], tx);
                if (s0 != nullptr) tc::bulk_load(st, s0 + (long)hd.tt * kTileFloats, L::kState, &full[stage]);
                for (int t = 0; t < nts; ++t) {
                    const long tok = hd.tok0 + t;
                    const TQ *kt = reinterpret_cast<const TQ *>(p.k) + (tok * Hk + hk) * DK;
                    const TQ *qt = reinterpret_cast<const TQ *>(p.q) + (tok * Hk + hk) * DK;
                    const TQ *vt = reinterpret_cast<const TQ *>(p.v) + (tok * Hv + hd.h) * (long)dv +
                                   hd.tt * kRowsPerCta;
                    tc::bulk_load(st + L::oK + t * L::kVec, kt, L::kVec, &full[stage]);
                    tc::bulk_load(st + L::oQ + t * L::kVec, qt, L::kVec, &full[stage]);
                    tc::bulk_load(st + L::oV + t * L::kV, vt, L::kV, &full[stage]);
                }
            }
            float *sg = reinterpret_cast<float *>(st + L::oG);
            if (lane < nts) {
                const long gi = (hd.tok0 + lane) * Hv + hd.h;
                sg[lane] = conv_alpha(ld_gate(p.alpha, gi, p.dt_gate), p.conv);
                sg[TS + lane] = conv_beta(ld_gate(p.beta, gi, p.dt_gate), p.conv);
            }
            if constexpr (RS > 0) {
                // the first RS replayed slots (all loads issued, then stored)
                const int nrs = hd.m < RS ? hd.m : RS;
                if (nrs > 0) {
                    const float *su_b = p.rp_su + (long)hd.b * p.rp_capacity * slot;
                    float kf[RS][KPL], df[RS], af[RS];
#pragma unroll
                    for (int j = 0; j < RS; ++j) {
                        if (j < nrs) {
                            const float *s = su_b + (long)j * slot;
#pragma unroll
                            for (int i = 0; i < KPL; ++i) kf[j][i] = __ldg(s + Hv + (long)hk * DK + lane + 32 * i);
                            df[j] = __ldg(s + Hv + (long)Hk * DK + (long)hd.h * dv + hd.tt * kRowsPerCta + lane);
                            af[j] = __ldg(s + hd.h);
                        }
                    }
                    float *rk = reinterpret_cast<float *>(st + L::oRK);
                    float *rd = reinterpret_cast<float *>(st + L::oRD);
                    float *ra = reinterpret_cast<float *>(st + L::oRA);
#pragma unroll
                    for (int j = 0; j < RS; ++j) {
                        if (j < nrs) {
#pragma unroll
                            for (int i = 0; i < KPL; ++i) rk[j * DK + lane + 32 * i] = kf[j][i];
                            rd[j * kRowsPerCta + lane] = df[j];
                            if (lane == 0) ra[j] = af[j];
                        }
                    }
                }
            }
            if (lane == 0) *reinterpret_cast<TileHeader *>(st + L::oH) = hd;
            // lane 0's arrive releases every lane's shared-memory writes (the
            // warp barrier orders them before it); the copies complete the phase
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&full[stage]);
        }
        // drain: the copies of the last tiles must land before this warp exits
        if (lane == 0)
            for (int s = 0; s < kStages && it - 1 - s >= 0; ++s) {
                const int j = it - 1 - s;
                tc::mbar_wait(&full[j % kStages], (j / kStages) & 1, kDefaultWaitNs);
            }
        return;
    }

    // ======================= compute warps ================================
    // Each lane holds its dk/8 columns of two state rows in registers for the
    // whole tile, as float2 pairs for the packed fp32x2 FMA: the state is read
    // from the stage once and never goes back to shared memory.
    const int grp = lane / kLanesPerRow, l8 = lane % kLanesPerRow;
    // Inactive capture: every CTA zeroes its share of the whole buffer.
    if (p.capacity > 0 && !active) {
        const long total = (long)p.B * p.capacity * slot;
        const long per = (total + gridDim.x - 1) / gridDim.x;
        const long e0 = (long)blockIdx.x * per;
        const long e1 = (e0 + per < total) ? e0 + per : total;
        for (long e = e0 + threadIdx.x; e < e1; e += CW * 32) p.su[e] = 0.0f;
    }
    const TQ *qb = reinterpret_cast<const TQ *>(p.q);
    const TQ *kb = reinterpret_cast<const TQ *>(p.k);
    const TQ *vb = reinterpret_cast<const TQ *>(p.v);
    TQ *ob = reinterpret_cast<TQ *>(p.out);
    const float scale = p.scale;
    const bool commit_in_place = (p.s_commit == p.s0);
    int lrow[NP];  // row inside the tile
#pragma unroll
    for (int r = 0; r < NP; ++r) lrow[r] = warp * kRowsW + r * (32 / kLanesPerRow) + grp;

    int it = 0;
    for (long id = blockIdx.x; id < n_tiles; id += gridDim.x, ++it) {
        const int stage = it % kStages;
        const uint8_t *st = sbase + stage * L::kBytes;
        if (!tc::mbar_wait(&full[stage], (it / kStages) & 1, p.wait_ns)) {
            if (threadIdx.x == 0) atomicOr(p.err, (uint32_t)GDN_DEVERR_TIMEOUT);
            break;
        }
        const TileHeader hd = *reinterpret_cast<const TileHeader *>(st + L::oH);
        const int b = hd.b, h = hd.h, hk = h / G, row0 = hd.tt * kRowsPerCta, Tb = hd.Tb;
        float *su_row = (p.capacity > 0) ? p.su + (long)b * p.capacity * slot : nullptr;
        float *sf = (p.s_final != nullptr) ? p.s_final + (((long)b * Hv + h) * dv + row0) * DK : nullptr;

        // Inputs of token t shared by the tile's rows: k and q widened to
        // fp32 pairs, the gates, from the stage or (past TS) from memory.
        auto token_in = [&](int t, float2(&kf)[F2], float2(&qf)[F2], float &a, float &bt) {
            if (t < TS) {
                load_pairs<F4>(reinterpret_cast<const TQ *>(st + L::oK + t * L::kVec), l8, kf);
                load_pairs<F4>(reinterpret_cast<const TQ *>(st + L::oQ + t * L::kVec), l8, qf);
                const float *sg = reinterpret_cast<const float *>(st + L::oG);
                a = sg[t];
                bt = sg[TS + t];
            } else {
                const long tok = hd.tok0 + t;
                load_pairs<F4>(kb + (tok * Hk + hk) * DK, l8, kf);
                load_pairs<F4>(qb + (tok * Hk + hk) * DK, l8, qf);
                a = conv_alpha(ld_gate(p.alpha, tok * Hv + h, p.dt_gate), p.conv);
                bt = conv_beta(ld_gate(p.beta, tok * Hv + h, p.dt_gate), p.conv);
            }
            if (p.conv & GDN_QK_L2NORM) {
                // q and k normalised in the kernel (8-lane sums of squares)
                const float nk = l2norm_factor(group_sum<kLanesPerRow>(dot_pairs<F2>(kf, kf)));
                const float nq = l2norm_factor(group_sum<kLanesPerRow>(dot_pairs<F2>(qf, qf)));
                const float2 rk = make_float2(nk, nk), rq = make_float2(nq, nq);
#pragma unroll
                for (int i = 0; i < F2; ++i) {
                    kf[i] = __fmul2_rn(kf[i], rk);
                    qf[i] = __fmul2_rn(qf[i], rq);
                }
            }
        };
        // One row, one token: delta with the decayed state, the rank-1
        // update, the readout with the updated state and the captured delta.
        auto row_step = [&](float2(&Sr)[F2], int r, int t, const float2(&kf)[F2], const float2(&qf)[F2],
                            float a, float bt, float kq, float *su_t) {
            const float sk = group_sum<kLanesPerRow>(dot_pairs<F2>(Sr, kf));
            const float sq = group_sum<kLanesPerRow>(dot_pairs<F2>(Sr, qf)) * scale;
            const long tok = hd.tok0 + t;
            const float vi = (t < TS) ? ld_f(reinterpret_cast<const TQ *>(st + L::oV + t * L::kV) + lrow[r])
                                      : ld_f(vb + (tok * Hv + h) * (long)dv + row0 + lrow[r]);
            const float delta = bt * (vi - a * sk);
            const float2 a2 = make_float2(a, a), d2 = make_float2(delta, delta);
#pragma unroll
            for (int i = 0; i < F2; ++i) Sr[i] = __ffma2_rn(a2, Sr[i], __fmul2_rn(d2, kf[i]));
            if (l8 == 0) {
                st_out(ob + (tok * Hv + h) * (long)dv + row0 + lrow[r], fmaf(a, sq, delta * kq));
                if (su_t != nullptr) su_t[Hv + (long)Hk * DK + (long)h * dv + row0 + lrow[r]] = delta;
            }
        };
        // The token's decay and (once per key head) its key, in slot su_t.
        auto capture_token = [&](float *su_t, float a, const float2(&kf)[F2]) {
            if (hd.tt != 0) return;
            if (threadIdx.x == 0) su_t[h] = a;
            if (h % G == 0 && warp == 0 && grp == 0) {
                float *kd = su_t + Hv + (long)hk * DK;
#pragma unroll
                for (int f = 0; f < F4; ++f) {
                    const int col = (f * kLanesPerRow + l8) * 4;
                    kd[col + 0] = kf[2 * f].x;
                    kd[col + 1] = kf[2 * f].y;
                    kd[col + 2] = kf[2 * f + 1].x;
                    kd[col + 3] = kf[2 * f + 1].y;
                }
            }
        };
        auto load_row = [&](int r, float2(&Sr)[F2]) {
            if (hd.has_state) {
                const float *sS = reinterpret_cast<const float *>(st);
#pragma unroll
                for (int f = 0; f < F4; ++f)
                    split4(*reinterpret_cast<const float4 *>(sS + lrow[r] * DK + (f * kLanesPerRow + l8) * 4),
                           Sr[2 * f], Sr[2 * f + 1]);
            } else {
#pragma unroll
                for (int i = 0; i < F2; ++i) Sr[i] = make_float2(0.f, 0.f);
            }
        };

        if constexpr (TS == 1) {
            // Single-token variant (the launcher sends it rows of at most one
            // token and no replay): one row at a time, straight to memory.
            float2 kf[F2], qf[F2];
            float a = 0.f, bt = 0.f, kq = 0.f;
            float *su_t = nullptr;
            if (Tb > 0) {
                token_in(0, kf, qf, a, bt);
                kq = group_sum<kLanesPerRow>(dot_pairs<F2>(kf, qf)) * scale;
                if (hd.ncap > 0) su_t = su_row;
            }
#pragma unroll
            for (int r = 0; r < NP; ++r) {
                float2 Sr[F2];
                load_row(r, Sr);
                if (Tb > 0) row_step(Sr, r, 0, kf, qf, a, bt, kq, su_t);
                if (sf != nullptr) store_row<DK, F4>(sf, Sr, lrow[r], l8);
            }
            if (su_t != nullptr) capture_token(su_t, a, kf);
        } else {
            float2 S[NP][F2];
#pragma unroll
            for (int r = 0; r < NP; ++r) load_row(r, S[r]);

            // Replay of the accepted prefix, S <- decay S + delta key^T per
            // slot, then the committed state (skipped in place when nothing
            // changed).
            if (hd.m > 0) {
                const float *su_b = p.rp_su + (long)b * p.rp_capacity * slot;
                for (int j = 0; j < hd.m; ++j) {
                    float dec, dl[NP];
                    float2 kk[F2];
                    if (j < RS) {
                        const float *rk = reinterpret_cast<const float *>(st + L::oRK) + j * DK;
                        const float *rd = reinterpret_cast<const float *>(st + L::oRD) + j * kRowsPerCta;
                        dec = reinterpret_cast<const float *>(st + L::oRA)[j];
#pragma unroll
                        for (int r = 0; r < NP; ++r) dl[r] = rd[lrow[r]];
#pragma unroll
                        for (int f = 0; f < F4; ++f)
                            split4(*reinterpret_cast<const float4 *>(rk + (f * kLanesPerRow + l8) * 4), kk[2 * f],
                                   kk[2 * f + 1]);
                    } else {
                        const float *s = su_b + (long)j * slot;
                        const float *key = s + Hv + (long)hk * DK;
                        const float *del = s + Hv + (long)Hk * DK + (long)h * dv + row0;
                        dec = __ldg(s + h);
#pragma unroll
                        for (int r = 0; r < NP; ++r) dl[r] = __ldg(del + lrow[r]);
#pragma unroll
                        for (int f = 0; f < F4; ++f) {
                            const int col = (f * kLanesPerRow + l8) * 4;
                            kk[2 * f] = make_float2(__ldg(key + col), __ldg(key + col + 1));
                            kk[2 * f + 1] = make_float2(__ldg(key + col + 2), __ldg(key + col + 3));
                        }
                    }
                    const float2 dec2 = make_float2(dec, dec);
#pragma unroll
                    for (int r = 0; r < NP; ++r) {
                        const float2 d2 = make_float2(dl[r], dl[r]);
#pragma unroll
                        for (int i = 0; i < F2; ++i) S[r][i] = __ffma2_rn(dec2, S[r][i], __fmul2_rn(d2, kk[i]));
                    }
                }
            }
            if (p.s_commit != nullptr && (hd.m > 0 || !commit_in_place)) {
                float *sc = p.s_commit + (((long)b * Hv + h) * dv + row0) * DK;
#pragma unroll
                for (int r = 0; r < NP; ++r) store_row<DK, F4>(sc, S[r], lrow[r], l8);
            }

            for (int t = 0; t < Tb; ++t) {
                float2 kf[F2], qf[F2];
                float a, bt, vi[NP];
                token_in(t, kf, qf, a, bt);
                const long tok = hd.tok0 + t;
                if (t < TS) {
                    const TQ *vs = reinterpret_cast<const TQ *>(st + L::oV + t * L::kV);
#pragma unroll
                    for (int r = 0; r < NP; ++r) vi[r] = ld_f(vs + lrow[r]);
                } else {
                    const TQ *vg = vb + (tok * Hv + h) * (long)dv + row0;
#pragma unroll
                    for (int r = 0; r < NP; ++r) vi[r] = ld_f(vg + lrow[r]);
                }
                // every row's dot products first, then all reductions together
                // (independent shuffle chains), then the updates
                float kq = dot_pairs<F2>(kf, qf), sk[NP], sq[NP];
#pragma unroll
                for (int r = 0; r < NP; ++r) {
                    sk[r] = dot_pairs<F2>(S[r], kf);
                    sq[r] = dot_pairs<F2>(S[r], qf);
                }
                kq = group_sum<kLanesPerRow>(kq) * scale;
#pragma unroll
                for (int r = 0; r < NP; ++r) {
                    sk[r] = group_sum<kLanesPerRow>(sk[r]);
                    sq[r] = group_sum<kLanesPerRow>(sq[r]) * scale;
                }
                float *su_t = (t < hd.ncap) ? su_row + (long)t * slot : nullptr;
                const float2 a2 = make_float2(a, a);
#pragma unroll
                for (int r = 0; r < NP; ++r) {
                    const float delta = bt * (vi[r] - a * sk[r]);
                    const float2 d2 = make_float2(delta, delta);
#pragma unroll
                    for (int i = 0; i < F2; ++i) S[r][i] = __ffma2_rn(a2, S[r][i], __fmul2_rn(d2, kf[i]));
                    if (l8 == 0) {
                        st_out(ob + (tok * Hv + h) * (long)dv + row0 + lrow[r], fmaf(a, sq[r], delta * kq));
                        if (su_t != nullptr) su_t[Hv + (long)Hk * DK + (long)h * dv + row0 + lrow[r]] = delta;
                    }
                }
                if (su_t != nullptr) capture_token(su_t, a, kf);
            }
            if (sf != nullptr)
#pragma unroll
                for (int r = 0; r < NP; ++r) store_row<DK, F4>(sf, S[r], lrow[r], l8);
        }
        // this warp is done reading the stage
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&empty[stage]);
    }
}

template <int DK, typename TQ, int TS, int RS, int CPS, int CW>
cudaError_t launch_v(const RecurrentParams &p, cudaStream_t stream) {
    auto kern = recurrent_kernel<DK, TQ, TS, RS, CPS, CW>;
    const size_t bytes = (size_t)kStages * StageLayout<DK, TQ, TS, RS>::kBytes + 2 * kStages * sizeof(uint64_t);
    cudaError_t e = set_smem_once<recurrent_kernel<DK, TQ, TS, RS, CPS, CW>>((int)bytes);
    if (e != cudaSuccess) return e;
    const long tiles = (long)p.B * p.Hv * (p.dv / kRowsPerCta);
    const long cap = (long)sm_count_of_current_device() * CPS;
    const unsigned grid = (unsigned)(tiles < cap ? tiles : cap);
    kern<<<grid, CW * 32 + 32, bytes, stream>>>(p);
    return cudaGetLastError();
}

// Single-token decode without replay: one staged token, small stages, four
// CTAs per SM.  Anything else (several tokens per row, replayed slots):
// four tokens and four slots staged, three CTAs per SM.
template <int DK, typename TQ>
cudaError_t launch_t(const RecurrentParams &p, cudaStream_t stream) {
    if (p.rp_capacity == 0 && p.cu_seqlens == nullptr && p.T <= 1)
        return launch_v<DK, TQ, 1, 0, 4, 4>(p, stream);
    return launch_v<DK, TQ, 4, 4, 3, 4>(p, stream);
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
