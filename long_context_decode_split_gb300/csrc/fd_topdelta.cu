// fd_topdelta.cu -- the sparse decode of the "Faster Flash Decoding" summary
// (PaperDaily) for sm_103a: the key encoder (section 5) and one fused pass
// per cache chunk that scans the 2-bit keys, takes the pseudo-max over the
// sink and window anchors (section 4), keeps keys with s~ >= m^ - delta
// (section 3), corrects the kept keys with their int8 residual and attends
// over them exactly (section 5, Fig. 2), with the stages fused as section 6
// asks: nothing but the per-chunk (m_i, l_i, O_i) leaves the chip.
//
// Fused pass, one CTA per (chunk, KV head, sequence), 1 producer + 4
// consumer warps, 64-token tiles (the same tile grid as the dense path):
//   * anchor pass: the consumer warps score the tiles that hold anchors and
//     take m^ per query head.  Every CTA of a (sequence, head) computes the
//     same m^ bit for bit: the anchor scores are produced by the same code,
//     lanes and operation order as the main scan.
//   * scan ring (2-bit codes + fp16 min/scale, 48 B per token at d=128) is
//     filled LA+1 tiles ahead by bulk copies.  Consumers score tile k,
//     store s~ in shared memory and flag whether any query head of the
//     group selected a token of the tile.
//   * detail ring (int8 residual + fp16 scales + bf16 V, 392 B per token):
//     the producer issues a tile's copies only once the consumers flagged it,
//     LA tiles before the consumers attend to it, so the residual and V of
//     tiles without candidates are never read from HBM.
//   * attend: exact scores s = s~ + scale * sum_g rs_g <q_g, rq_g> for the
//     candidates, online softmax and P.V as in the dense pass, then the same
//     warp combine and chunk merge.
#include <cmath>
#include <cuda_fp16.h>

#include "fd_device.cuh"
#include "fd_internal.h"

namespace fd {

__device__ unsigned int g_status_topdelta;

namespace {

constexpr int kMaxDevices = 64;
constexpr int CW = 4;           // consumer warps
constexpr int LA = 2;           // tiles scanned ahead of the attend step
constexpr int DS = LA + 1;      // detail ring depth (= decision slots)
constexpr int SS = LA + 2;      // scan ring depth

// ============================================================== encoder

// One warp encodes 32/(D/4) token rows; lane owns 4 channels, 8 lanes form
// a 32-channel group.  Same binary32 operation order as the definition in
// fd.h, with explicitly rounded intrinsics so nothing is fused.
template <int D>
__global__ void __launch_bounds__(256)
quantize_kernel(const uint16_t* __restrict__ k, const int32_t* __restrict__ seq_lens, int Hkv, int L_max,
                long long rows, uint8_t* __restrict__ codes, uint16_t* __restrict__ mn_scale,
                int8_t* __restrict__ res, uint16_t* __restrict__ res_scale) {
    constexpr int LPRQ = D / 4;     // lanes per row
    constexpr int RPW = 32 / LPRQ;  // rows per warp
    constexpr int NG = D / 32;
    const int lane = threadIdx.x & 31;
    const int sub = lane / LPRQ;
    const int c4 = lane % LPRQ;
    const int grp = c4 / 8;
    const long long warp_id = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long r0 = warp_id * RPW; r0 < rows; r0 += nwarps * RPW) {
        const long long row = r0 + sub;
        bool valid = row < rows;
        if (valid) {
            const int t = (int)(row % L_max);
            const int b = (int)(row / ((long long)Hkv * L_max));
            valid = t < clamped_len(seq_lens, b, L_max, &g_status_topdelta);
        }
        float x[4] = {0.f, 0.f, 0.f, 0.f};
        if (valid) {
            const uint2 w = *reinterpret_cast<const uint2*>(k + row * D + 4 * c4);
            const float2 a = bf16x2_to_float2(w.x), bb = bf16x2_to_float2(w.y);
            x[0] = a.x;
            x[1] = a.y;
            x[2] = bb.x;
            x[3] = bb.y;
        }
        float mn = fminf(fminf(x[0], x[1]), fminf(x[2], x[3]));
        float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
        mn = __fadd_rn(mn, 0.0f);  // a zero extreme is +0 whatever its sign
        mx = __fadd_rn(mx, 0.0f);
        const __half mn16 = __float2half_rn(mn);
        const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), 3.0f));
        const float mnf = __half2float(mn16);
        const float sf = __half2float(s16);
        int code[4];
        float r[4];
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            int q2 = 0;
            if (sf != 0.f) {
                const int rr = __float2int_rn(__fdiv_rn(__fsub_rn(x[i], mnf), sf));
                q2 = min(max(rr, 0), 3);
            }
            code[i] = q2;
            const float dq = __fadd_rn(mnf, __fmul_rn((float)q2, sf));
            r[i] = __fsub_rn(x[i], dq);
            amax = fmaxf(amax, fabsf(r[i]));
        }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const __half rs16 = __float2half_rn(__fdiv_rn(amax, 127.0f));
        const float rsf = __half2float(rs16);
        uint32_t packed = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            int q8 = 0;
            if (rsf != 0.f) q8 = min(max(__float2int_rn(__fdiv_rn(r[i], rsf)), -127), 127);
            packed |= (uint32_t)(q8 & 0xff) << (8 * i);
        }
        if (valid) {
            codes[row * (D / 4) + c4] = (uint8_t)(code[0] | (code[1] << 2) | (code[2] << 4) | (code[3] << 6));
            *reinterpret_cast<uint32_t*>(res + row * D + 4 * c4) = packed;
            if ((c4 & 7) == 0) {
                mn_scale[(row * NG + grp) * 2 + 0] = __half_as_ushort(mn16);
                mn_scale[(row * NG + grp) * 2 + 1] = __half_as_ushort(s16);
                res_scale[row * NG + grp] = __half_as_ushort(rs16);
            }
        }
    }
}

// ============================================================ fused pass

template <int D>
struct TGeo {
    static constexpr int LPR = D / 8;      // lanes per row, 8 channels each
    static constexpr int RPI = 32 / LPR;   // rows per warp-wide step
    static constexpr int TPW = kTile / CW; // rows of a tile per warp
    static constexpr int NIT = TPW / RPI;
    static constexpr int LOG_LPR = D == 128 ? 4 : 3;
    static constexpr int LOG_NIT = NIT == 8 ? 3 : NIT == 4 ? 2 : NIT == 2 ? 1 : 0;
    static constexpr int SH = LOG_LPR - LOG_NIT;
    static constexpr int CODES_ROW = D / 4;   // bytes
    static constexpr int MS_ROW = D / 8;      // (mn16, s16) per 32 channels
    static constexpr int RES_ROW = D;
    static constexpr int RS_ROW = D / 16;     // rs16 per 32 channels
    static constexpr int V_ROW = 2 * D;
    static constexpr int SCAN_STAGE = kTile * (CODES_ROW + MS_ROW);
    static constexpr int DET_STAGE = kTile * (RES_ROW + RS_ROW + V_ROW);
};

template <int D, int GP>
struct TLayout {
    using Gm = TGeo<D>;
    static constexpr int SCAN_OFF = 0;
    static constexpr int DET_OFF = SCAN_OFF + SS * Gm::SCAN_STAGE;
    static constexpr int DEC_OFF = DET_OFF + DS * Gm::DET_STAGE;                // s~ [DS][64][GP] f32
    static constexpr int FLAG_OFF = DEC_OFF + DS * kTile * GP * 4;              // need[DS][CW], loaded[DS], scan_rows[SS]
    static constexpr int BAR_OFF = (FLAG_OFF + (DS * CW + DS + SS) * 4 + 15) / 16 * 16;
    static constexpr int MH_OFF = BAR_OFF + (2 * SS + 3 * DS) * 8;               // anchor maxima [CW][GP]
    static constexpr int BYTES = MH_OFF + CW * GP * 4;
    static_assert(DEC_OFF >= CW * GP * D * 4 + 2 * CW * GP * 4, "epilogue scratch must fit in the rings");
};

struct TDParams {
    const uint16_t* q;
    const uint8_t* codes;
    const uint16_t* mn_scale;
    const int8_t* res;
    const uint16_t* res_scale;
    const uint16_t* v;
    const int32_t* seq_lens;
    int Hq, Hkv, L_max, G;
    float scale, delta;
    int n_sink, window;
    int splits, chunk_fixed;
    uint32_t* sel_mask;
    int32_t* sel_count;
    StoreTarget st;
};

// The 2-bit score's contribution of one lane's 8 channels of one row, for
// every query of the group: s * <q, code> + mn * sum(q) over those channels.
// Codes are turned into floats exactly: (w & 3<<2i) | 0x4B000000 is the
// binary32 value 2^23 + code * 4^i; subtracting 2^23 leaves code * 4^i, and
// the query weights carry the matching 4^-i.  Every operation is an
// explicitly rounded intrinsic, so all call sites round identically.
template <int GP>
__device__ __forceinline__ void scan_partial(uint32_t w16, uint32_t ms_bits, const float2 (&qs)[GP][4],
                                             const float (&qsum)[GP], float (&out)[GP]) {
    const float2 magic = make_float2(-8388608.f, -8388608.f);
    float2 cf[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const uint32_t lo = (w16 & (3u << (4 * e))) | 0x4B000000u;
        const uint32_t hi = (w16 & (3u << (4 * e + 2))) | 0x4B000000u;
        cf[e] = __fadd2_rn(make_float2(__uint_as_float(lo), __uint_as_float(hi)), magic);
    }
    const float mn = __half2float(__ushort_as_half((unsigned short)(ms_bits & 0xffffu)));
    const float sc = __half2float(__ushort_as_half((unsigned short)(ms_bits >> 16)));
#pragma unroll
    for (int g = 0; g < GP; ++g) {
        float2 acc = __fmul2_rn(qs[g][0], cf[0]);
        acc = __ffma2_rn(qs[g][1], cf[1], acc);
        acc = __ffma2_rn(qs[g][2], cf[2], acc);
        acc = __ffma2_rn(qs[g][3], cf[3], acc);
        out[g] = __fmaf_rn(sc, __fadd_rn(acc.x, acc.y), __fmul_rn(mn, qsum[g]));
    }
}

// Scores s~ (natural-log units) of the warp's 16 rows of one tile.  `codes`
// and `ms` point at the tile's first row, in shared or global memory;
// rows >= `rows` are not read when `guard` is set.  On return lane l holds
// the score of row warp*16 + RPI*((l >> SH) & (NIT-1)) + l / LPR.
template <int D, int GP>
__device__ __forceinline__ void score_tile_rows(const uint8_t* codes, const uint16_t* ms, int warp, int lane,
                                                int rows, bool guard, const float2 (&qs)[GP][4],
                                                const float (&qsum)[GP], float scale, float (&s)[GP]) {
    using Gm = TGeo<D>;
    const int c = lane % Gm::LPR;
    const int rg = lane / Gm::LPR;
    float part[GP][Gm::NIT];
#pragma unroll
    for (int i = 0; i < Gm::NIT; ++i) {
        const int row = warp * Gm::TPW + Gm::RPI * i + rg;
        uint32_t w16 = 0, msb = 0;
        if (!guard || row < rows) {
            w16 = *reinterpret_cast<const uint16_t*>(codes + row * Gm::CODES_ROW + c * 2);
            msb = *reinterpret_cast<const uint32_t*>(ms + row * (Gm::MS_ROW / 2) + (c / 4) * 2);
        }
        float pg[GP];
        scan_partial<GP>(w16, msb, qs, qsum, pg);
#pragma unroll
        for (int g = 0; g < GP; ++g) part[g][i] = pg[g];
    }
#pragma unroll
    for (int g = 0; g < GP; ++g) s[g] = __fmul_rn(transpose_reduce<Gm::NIT, Gm::LPR>(part[g], lane), scale);
}

template <int D, int GP>
// two CTAs per SM (168 registers) up to groups of 4; groups of 8 need the registers of one
__global__ void __launch_bounds__((CW + 1) * 32, GP >= 8 ? 1 : 2)
topdelta_kernel(const TDParams p) {
    using Gm = TGeo<D>;
    using Ly = TLayout<D, GP>;
    extern __shared__ __align__(128) unsigned char smem[];
    float* dec_s = reinterpret_cast<float*>(smem + Ly::DEC_OFF);
    int* need = reinterpret_cast<int*>(smem + Ly::FLAG_OFF);
    int* loaded = need + DS * CW;
    int* scan_rows = loaded + DS;
    uint64_t* scan_full = reinterpret_cast<uint64_t*>(smem + Ly::BAR_OFF);
    uint64_t* scan_empty = scan_full + SS;
    uint64_t* det_full = scan_empty + SS;
    uint64_t* det_empty = det_full + DS;
    uint64_t* decided = det_empty + DS;
    float* mh_red = reinterpret_cast<float*>(smem + Ly::MH_OFF);

    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = clamped_len(p.seq_lens, b, p.L_max, &g_status_topdelta);
    int chunk = p.chunk_fixed;
    if (chunk <= 0) {
        chunk = (L + p.splits - 1) / p.splits;
        chunk = (chunk + kTile - 1) / kTile * kTile;
        if (chunk <= 0) chunk = kTile;
    }
    const int t0 = split * chunk;
    const int t1 = min(L, t0 + chunk);
    const int hq0 = h * p.G;
    const size_t head_row0 = ((size_t)b * p.Hkv + h) * (size_t)p.L_max;

    if (t0 >= t1) {
        pdl_launch_dependents();
        if (p.st.direct && split == 0) {
            for (int i = threadIdx.x; i < p.G * D; i += blockDim.x) {
                const size_t o = (size_t)(b * p.Hq + hq0 + i / D) * D + (i % D);
                if (p.st.out_bf16) static_cast<uint16_t*>(p.st.out)[o] = 0;
                else static_cast<float*>(p.st.out)[o] = 0.f;
            }
            if (p.st.lse && threadIdx.x < p.G) p.st.lse[b * p.Hq + hq0 + threadIdx.x] = -INFINITY;
        }
        return;
    }
    const int ntiles = (t1 - t0 + kTile - 1) / kTile;

    if (threadIdx.x == 0) {
        for (int s = 0; s < SS; ++s) {
            mbar_init(&scan_full[s], 1);
            mbar_init(&scan_empty[s], CW);
        }
        for (int s = 0; s < DS; ++s) {
            mbar_init(&det_full[s], 1);
            mbar_init(&det_empty[s], CW);
            mbar_init(&decided[s], CW);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == CW) {
        // ----------------------------- producer --------------------------------
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            auto rows_of = [&](int t) { return min(kTile, t1 - (t0 + t * kTile)); };
            auto copy_rows = [&](int t) { return (rows_of(t) + 3) & ~3; };  // L_max % 4 == 0 keeps this in bounds
            auto issue_scan = [&](int k) -> bool {
                const int s = k % SS;
                if (!mbar_wait(&scan_empty[s], ((uint32_t)(k / SS) & 1u) ^ 1u)) return false;
                const size_t row0 = head_row0 + t0 + (size_t)k * kTile;
                const uint32_t rc = (uint32_t)copy_rows(k);
                unsigned char* dst = smem + Ly::SCAN_OFF + s * Gm::SCAN_STAGE;
                scan_rows[s] = rows_of(k);
                mbar_arrive_expect_tx(&scan_full[s], rc * (Gm::CODES_ROW + Gm::MS_ROW));
                bulk_g2s(dst, p.codes + row0 * Gm::CODES_ROW, rc * Gm::CODES_ROW, &scan_full[s], pol);
                bulk_g2s(dst + kTile * Gm::CODES_ROW, reinterpret_cast<const uint8_t*>(p.mn_scale) + row0 * Gm::MS_ROW,
                         rc * Gm::MS_ROW, &scan_full[s], pol);
                return true;
            };
            bool ok = true;
            for (int k = 0; k <= LA && k < ntiles && ok; ++k) ok = issue_scan(k);
            for (int t = 0; t < ntiles && ok; ++t) {
                const int s = t % DS;
                const uint32_t ph = (uint32_t)(t / DS) & 1u;
                if (!mbar_wait(&decided[s], ph) || !mbar_wait(&det_empty[s], ph ^ 1u)) {
                    ok = false;
                    break;
                }
                int any = 0;
                for (int w = 0; w < CW; ++w) any |= need[s * CW + w];
                if (any) {
                    const size_t row0 = head_row0 + t0 + (size_t)t * kTile;
                    const uint32_t rc = (uint32_t)copy_rows(t);
                    unsigned char* dst = smem + Ly::DET_OFF + s * Gm::DET_STAGE;
                    loaded[s] = 1;
                    mbar_arrive_expect_tx(&det_full[s], rc * (Gm::RES_ROW + Gm::RS_ROW + Gm::V_ROW));
                    bulk_g2s(dst, p.res + row0 * Gm::RES_ROW, rc * Gm::RES_ROW, &det_full[s], pol);
                    bulk_g2s(dst + kTile * Gm::RES_ROW,
                             reinterpret_cast<const uint8_t*>(p.res_scale) + row0 * Gm::RS_ROW, rc * Gm::RS_ROW,
                             &det_full[s], pol);
                    bulk_g2s(dst + kTile * (Gm::RES_ROW + Gm::RS_ROW), p.v + row0 * D, rc * Gm::V_ROW, &det_full[s],
                             pol);
                } else {
                    loaded[s] = 0;
                    mbar_arrive(&det_full[s]);
                }
                if (t + LA + 1 < ntiles) ok = issue_scan(t + LA + 1);
            }
            if (!ok) atomicOr(&g_status_topdelta, kStatusTimeout);
        }
        pdl_launch_dependents();
        return;
    }

    // ------------------------------- consumers -----------------------------------
    const int c = lane % Gm::LPR;
    const int rg = lane / Gm::LPR;
    const int my_i = (lane >> Gm::SH) & (Gm::NIT - 1);
    const int my_row = warp * Gm::TPW + Gm::RPI * my_i + rg;
    const bool my_dup = (lane & ((1 << Gm::SH) - 1)) != 0;

    // query weights for my 8 channels: exact (for the residual and V passes)
    // and scaled by 4^-i (for the 2-bit codes), plus their sum
    float2 qv[GP][4], qs[GP][4];
    float qsum[GP];
#pragma unroll
    for (int g = 0; g < GP; ++g) {
        float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (g < p.G) {
            const uint4 w = *reinterpret_cast<const uint4*>(p.q + (size_t)(b * p.Hq + hq0 + g) * D + c * 8);
            const float2 a0 = bf16x2_to_float2(w.x), a1 = bf16x2_to_float2(w.y);
            const float2 a2 = bf16x2_to_float2(w.z), a3 = bf16x2_to_float2(w.w);
            f[0] = a0.x; f[1] = a0.y; f[2] = a1.x; f[3] = a1.y;
            f[4] = a2.x; f[5] = a2.y; f[6] = a3.x; f[7] = a3.y;
        }
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) sum = __fadd_rn(sum, f[i]);
        qsum[g] = sum;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            qv[g][e] = make_float2(f[2 * e], f[2 * e + 1]);
            // channel 2e at bits 4e: weight 4^-(2e); channel 2e+1 at bits 4e+2: 4^-(2e+1)
            const float w0 = __int_as_float((127 - 4 * e) << 23);  // 4^-(2e), exact
            const float w1 = __int_as_float((125 - 4 * e) << 23);  // 4^-(2e+1)
            qs[g][e] = make_float2(__fmul_rn(f[2 * e], w0), __fmul_rn(f[2 * e + 1], w1));
        }
    }

    // ---------------- anchor pass: pseudo-max per query head --------------------
    float mh[GP];
#pragma unroll
    for (int g = 0; g < GP; ++g) mh[g] = -INFINITY;
    {
        const int sink_end = min(p.n_sink, L);              // anchors [0, sink_end)
        const int win_beg = max(0, L - p.window);            // anchors [win_beg, L)
        const int ts_end = (sink_end + kTile - 1) / kTile;   // sink tiles [0, ts_end)
        const int tw_beg = win_beg < L ? win_beg / kTile : (L + kTile - 1) / kTile;
        const int tw_end = (L + kTile - 1) / kTile;          // window tiles [tw_beg, tw_end)
        for (int T = 0; T < tw_end; ++T) {
            if (T >= ts_end && T < tw_beg) T = tw_beg;
            if (T >= tw_end) break;
            const int tb = T * kTile;
            const int rows = min(kTile, L - tb);
            float s[GP];
            score_tile_rows<D, GP>(p.codes + (head_row0 + tb) * Gm::CODES_ROW,
                                   p.mn_scale + (head_row0 + tb) * (Gm::MS_ROW / 2), warp, lane, rows, true, qs,
                                   qsum, p.scale, s);
            const int j = tb + my_row;
            const bool anchor = my_row < rows && (j < sink_end || j >= win_beg);
#pragma unroll
            for (int g = 0; g < GP; ++g)
                if (anchor) mh[g] = fmaxf(mh[g], s[g]);
        }
#pragma unroll
        for (int g = 0; g < GP; ++g) {
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) mh[g] = fmaxf(mh[g], __shfl_xor_sync(0xffffffffu, mh[g], off));
            if (lane == 0) mh_red[warp * GP + g] = mh[g];
        }
        named_barrier(1, CW * 32);
#pragma unroll
        for (int g = 0; g < GP; ++g) {
            float m = -INFINITY;
#pragma unroll
            for (int w = 0; w < CW; ++w) m = fmaxf(m, mh_red[w * GP + g]);
            mh[g] = m;
        }
    }
    float thr[GP];
#pragma unroll
    for (int g = 0; g < GP; ++g) thr[g] = __fsub_rn(mh[g], p.delta);  // delta = inf keeps every key

    float m_run[GP], l_lane[GP];
    float2 o[GP][4];
    int cnt[GP];
#pragma unroll
    for (int g = 0; g < GP; ++g) {
        m_run[g] = -INFINITY;
        l_lane[g] = 0.f;
        cnt[g] = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) o[g][e] = make_float2(0.f, 0.f);
    }
    bool failed = false;

    // scan one tile: s~ to the decision slot, flag the tile if any key passes
    auto scan_step = [&](int k) {
        const int s = k % SS;
        if (!warp_wait(&scan_full[s], (uint32_t)(k / SS) & 1u)) {
            failed = true;
            return;
        }
        const int rows = scan_rows[s];
        const unsigned char* base = smem + Ly::SCAN_OFF + s * Gm::SCAN_STAGE;
        float sc[GP];
        score_tile_rows<D, GP>(base, reinterpret_cast<const uint16_t*>(base + kTile * Gm::CODES_ROW), warp, lane,
                               rows, false, qs, qsum, p.scale, sc);
        const int ds = k % DS;
        bool any = false;
#pragma unroll
        for (int g = 0; g < GP; ++g) {
            if (!my_dup) dec_s[(ds * kTile + my_row) * GP + g] = sc[g];
            any |= (g < p.G) && (my_row < rows) && (sc[g] >= thr[g]);
        }
        any = __any_sync(0xffffffffu, any);
        __syncwarp();
        if (lane == 0) {
            need[ds * CW + warp] = any ? 1 : 0;
            mbar_arrive(&scan_empty[s]);
            mbar_arrive(&decided[ds]);
        }
    };

    const int pro = min(LA, ntiles);
    for (int k = 0; k < pro && !failed; ++k) scan_step(k);
    for (int t = 0; t < ntiles && !failed; ++t) {
        if (t + LA < ntiles) {
            scan_step(t + LA);
            if (failed) break;
        }
        const int ds = t % DS;
        if (!warp_wait(&det_full[ds], (uint32_t)(t / DS) & 1u)) {
            failed = true;
            break;
        }
        if (loaded[ds]) {
            const int tok0 = t0 + t * kTile;
            const int rows = min(kTile, t1 - tok0);
            const unsigned char* rb = smem + Ly::DET_OFF + ds * Gm::DET_STAGE;
            const unsigned char* rsb = rb + kTile * Gm::RES_ROW;
            const unsigned char* vb = rsb + kTile * Gm::RS_ROW;
            // residual term per row: rs * <q, rq> over my 8 channels, then butterfly
            float part[GP][Gm::NIT];
#pragma unroll
            for (int i = 0; i < Gm::NIT; ++i) {
                const int row = warp * Gm::TPW + Gm::RPI * i + rg;
                const uint2 w = *reinterpret_cast<const uint2*>(rb + row * Gm::RES_ROW + c * 8);
                const float rsf = __half2float(__ushort_as_half(
                    *reinterpret_cast<const unsigned short*>(rsb + row * Gm::RS_ROW + (c / 4) * 2)));
                float2 rf[4];
                rf[0] = make_float2((float)(int8_t)(w.x & 0xff), (float)(int8_t)((w.x >> 8) & 0xff));
                rf[1] = make_float2((float)(int8_t)((w.x >> 16) & 0xff), (float)(int8_t)(w.x >> 24));
                rf[2] = make_float2((float)(int8_t)(w.y & 0xff), (float)(int8_t)((w.y >> 8) & 0xff));
                rf[3] = make_float2((float)(int8_t)((w.y >> 16) & 0xff), (float)(int8_t)(w.y >> 24));
#pragma unroll
                for (int g = 0; g < GP; ++g) {
                    float2 acc = f2mul(qv[g][0], rf[0]);
                    acc = f2fma(qv[g][1], rf[1], acc);
                    acc = f2fma(qv[g][2], rf[2], acc);
                    acc = f2fma(qv[g][3], rf[3], acc);
                    part[g][i] = rsf * (acc.x + acc.y);
                }
            }
            float sx[GP];
            bool sel[GP];
            const bool my_valid = my_row < rows;
#pragma unroll
            for (int g = 0; g < GP; ++g) {
                const float rterm = transpose_reduce<Gm::NIT, Gm::LPR>(part[g], lane) * p.scale;
                const float st = dec_s[(ds * kTile + my_row) * GP + g];
                sel[g] = my_valid && (g < p.G) && (st >= thr[g]);
                sx[g] = sel[g] ? (st + rterm) * kLog2e : -INFINITY;
                if (sel[g] && !my_dup) {
                    ++cnt[g];
                    if (p.sel_mask) {
                        const int j = tok0 + my_row;
                        const int words = (p.L_max + 31) / 32;
                        atomicOr(&p.sel_mask[(size_t)(b * p.Hq + hq0 + g) * words + j / 32], 1u << (j % 32));
                    }
                }
            }
            // online softmax over the candidates of this tile
            float pr[GP];
#pragma unroll
            for (int g = 0; g < GP; ++g) {
                float mx = sx[g];
#pragma unroll
                for (int off = 16; off >= (1 << Gm::SH); off >>= 1)
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                const float m_new = fmaxf(m_run[g], mx);
                if (m_new == -INFINITY) {
                    pr[g] = 0.f;
                    continue;
                }
                const float alpha = exp2_approx(m_run[g] - m_new);
                m_run[g] = m_new;
                pr[g] = exp2_approx(sx[g] - m_new);
                l_lane[g] = l_lane[g] * alpha + (my_dup ? 0.f : pr[g]);
                const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                for (int e = 0; e < 4; ++e) o[g][e] = f2mul(o[g][e], a2);
            }
#pragma unroll
            for (int i = 0; i < Gm::NIT; ++i) {
                const int row = warp * Gm::TPW + Gm::RPI * i + rg;
                const int src = rg * Gm::LPR + (i << Gm::SH);
                float pi[GP];
                bool anyp = false;
#pragma unroll
                for (int g = 0; g < GP; ++g) {
                    pi[g] = __shfl_sync(0xffffffffu, pr[g], src);
                    anyp |= pi[g] != 0.f;
                }
                if (row < rows && anyp) {
                    const uint4 w = lds128(vb + (row * D + c * 8) * 2);
                    const float2 v0 = bf16x2_to_float2(w.x), v1 = bf16x2_to_float2(w.y);
                    const float2 v2 = bf16x2_to_float2(w.z), v3 = bf16x2_to_float2(w.w);
#pragma unroll
                    for (int g = 0; g < GP; ++g) {
                        const float2 p2 = make_float2(pi[g], pi[g]);
                        o[g][0] = f2fma(p2, v0, o[g][0]);
                        o[g][1] = f2fma(p2, v1, o[g][1]);
                        o[g][2] = f2fma(p2, v2, o[g][2]);
                        o[g][3] = f2fma(p2, v3, o[g][3]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&det_empty[ds]);
    }
    if (failed) atomicOr(&g_status_topdelta, kStatusTimeout);
    pdl_launch_dependents();

    if (p.sel_count) {
#pragma unroll
        for (int g = 0; g < GP; ++g) {
            int n = cnt[g];
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) n += __shfl_xor_sync(0xffffffffu, n, off);
            if (lane == 0 && g < p.G && n) atomicAdd(&p.sel_count[b * p.Hq + hq0 + g], n);
        }
    }
    combine_warps_and_store<D, GP, CW>(smem, warp, lane, p.G, b * p.Hq + hq0, split, m_run, l_lane, o, failed,
                                       p.st);
}

template <int D, int GP>
struct TDLauncher {
    static constexpr int SMEM = TLayout<D, GP>::BYTES;
    static cudaError_t prepare() {
        static bool done[kMaxDevices] = {};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < kMaxDevices && done[dev]) return cudaSuccess;
        e = cudaFuncSetAttribute(topdelta_kernel<D, GP>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (e == cudaSuccess && dev < kMaxDevices) done[dev] = true;
        return e;
    }
    static int ctas_per_sm() {
        static int cache[kMaxDevices] = {};
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return 1;
        if (dev < kMaxDevices && cache[dev] > 0) return cache[dev];
        if (prepare() != cudaSuccess) return 1;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, topdelta_kernel<D, GP>, (CW + 1) * 32, SMEM) !=
                cudaSuccess ||
            n <= 0)
            return 1;
        if (dev < kMaxDevices) cache[dev] = n;
        return n;
    }
    static cudaError_t launch(const TDParams& pp, dim3 grid, cudaStream_t st) {
        cudaError_t e = prepare();
        if (e != cudaSuccess) return e;
        topdelta_kernel<D, GP><<<grid, (CW + 1) * 32, SMEM, st>>>(pp);
        return cudaGetLastError();
    }
};

template <int D>
int td_ctas(int G) {
    if (G <= 1) return TDLauncher<D, 1>::ctas_per_sm();
    if (G <= 2) return TDLauncher<D, 2>::ctas_per_sm();
    if (G <= 4) return TDLauncher<D, 4>::ctas_per_sm();
    return TDLauncher<D, 8>::ctas_per_sm();
}

template <int D>
cudaError_t td_launch(int G, const TDParams& pp, dim3 grid, cudaStream_t st) {
    if (G <= 1) return TDLauncher<D, 1>::launch(pp, grid, st);
    if (G <= 2) return TDLauncher<D, 2>::launch(pp, grid, st);
    if (G <= 4) return TDLauncher<D, 4>::launch(pp, grid, st);
    return TDLauncher<D, 8>::launch(pp, grid, st);
}

}  // namespace

int topdelta_ctas_per_sm(int D, int G) { return D == 128 ? td_ctas<128>(G) : td_ctas<64>(G); }

cudaError_t launch_quantize(const QuantArgs& a, cudaStream_t stream) {
    const long long rows = (long long)a.B * a.Hkv * a.L_max;
    if (rows == 0) return cudaSuccess;
    const int rows_per_block = 8 * (a.D == 128 ? 1 : 2);
    long long blocks = (rows + rows_per_block - 1) / rows_per_block;
    if (blocks > 152 * 16) blocks = 152 * 16;
    const unsigned g = (unsigned)blocks;
    if (a.D == 128)
        quantize_kernel<128><<<g, 256, 0, stream>>>(
            static_cast<const uint16_t*>(a.k), a.seq_lens, a.Hkv, a.L_max, rows, a.codes,
            static_cast<uint16_t*>(a.mn_scale), a.res, static_cast<uint16_t*>(a.res_scale));
    else
        quantize_kernel<64><<<g, 256, 0, stream>>>(
            static_cast<const uint16_t*>(a.k), a.seq_lens, a.Hkv, a.L_max, rows, a.codes,
            static_cast<uint16_t*>(a.mn_scale), a.res, static_cast<uint16_t*>(a.res_scale));
    return cudaGetLastError();
}

cudaError_t launch_topdelta(const TopDeltaArgs& a, cudaStream_t stream) {
    if (a.B == 0) return cudaSuccess;
    const int words = (a.L_max + 31) / 32;
    cudaError_t e;
    if (a.sel_mask) {
        e = cudaMemsetAsync(a.sel_mask, 0, (size_t)a.B * a.Hq * words * sizeof(uint32_t), stream);
        if (e != cudaSuccess) return e;
    }
    if (a.sel_count) {
        e = cudaMemsetAsync(a.sel_count, 0, (size_t)a.B * a.Hq * sizeof(int32_t), stream);
        if (e != cudaSuccess) return e;
    }
    TDParams pp;
    pp.q = static_cast<const uint16_t*>(a.q);
    pp.codes = a.codes;
    pp.mn_scale = static_cast<const uint16_t*>(a.mn_scale);
    pp.res = a.res;
    pp.res_scale = static_cast<const uint16_t*>(a.res_scale);
    pp.v = static_cast<const uint16_t*>(a.v);
    pp.seq_lens = a.seq_lens;
    pp.Hq = a.Hq;
    pp.Hkv = a.Hkv;
    pp.L_max = a.L_max;
    pp.G = a.Hq / a.Hkv;
    pp.scale = a.scale;
    pp.delta = a.delta;
    pp.n_sink = a.n_sink;
    pp.window = a.window;
    pp.splits = a.splits;
    pp.chunk_fixed = a.chunk_fixed;
    pp.sel_mask = a.sel_mask;
    pp.sel_count = a.sel_count;
    pp.st.out = a.out;
    pp.st.out_bf16 = a.out_bf16;
    pp.st.lse = a.lse;
    pp.st.part_o = a.part_o;
    pp.st.part_ml = a.part_ml;
    pp.st.direct = a.splits == 1 ? 1 : 0;
    pp.st.splits = a.splits;
    const dim3 grid((unsigned)a.splits, (unsigned)a.Hkv, (unsigned)a.B);
    e = a.D == 128 ? td_launch<128>(pp.G, pp, grid, stream) : td_launch<64>(pp.G, pp, grid, stream);
    if (e != cudaSuccess || a.splits == 1) return e;
    return launch_merge(a.part_o, a.part_ml, a.seq_lens, a.B, a.Hq, a.L_max, a.D, a.splits, a.chunk_fixed, a.out,
                        a.out_bf16, a.lse, stream);
}

cudaError_t topdelta_status_read(unsigned* bits, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(bits, g_status_topdelta, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_status_topdelta, &zero, sizeof(unsigned));
}

}  // namespace fd
