// fd_fp8.cu -- split-KV decode attention ("Flash Decoding" tutorial, sections
// 1-3) over an 8-bit floating-point KV cache, and the cache encoder, for
// sm_103a.  The benchmarking blog on a hosted 1M-context model (section 1)
// names a narrow-float KV cache as the way to cut the bytes a decode step
// reads; this file defines one such cache:
//
//   per cache row (token, KV head): s = max_c |x_c| / 448 (binary32) and
//   codes e4m3(x_c / s) (round to nearest even, saturating; all zero if s = 0).
//
// A row then costs d + 4 bytes instead of 2d, so K and V together stream
// about half the bytes of the bf16 cache.
//
// Partial pass, one CTA per (chunk, KV head, sequence), warp-specialised as
// the bf16 pass: warp 4 issues the tile copies (two 64-row code boxes and two
// 68-entry scale boxes per 64-token tile, through a STAGES-deep mbarrier
// ring), warps 0..3 each own 16 tokens of every tile, take NT tiles per step
// (one online-softmax update per step) and run both products on the tensor
// cores with fp16 operands (every e4m3 value is exact in fp16):
//   S = K Q^T   A = the warp's 16 K rows: codes fetched by ldmatrix (4 bytes
//               = 4 channels per lane) and widened with cvt.rn.f16x2.e4m3x2;
//               B = the query group (up to 8 columns) in fp16, scaled per
//               query by a power of two so that |q| < 1 (exact).  The channel
//               order inside each 16-channel k-step is permuted identically
//               on Q, so the dot products are unchanged.  The row scale of K
//               and the power of two of Q are applied to the fp32 scores.
//   O^T += V^T P^T
//               A = V codes: lane group gid reads channels D/8 * gid ..
//               + D/8 - 1 of its four tokens in one shared load each, and
//               byte permutes pair the tokens up before widening (row gid +
//               8r of output tile j is channel D/8 * gid + 2j + r);
//               B = P * s_V / s_ref in fp16, transposed from the S layout by
//               movmatrix, where s_ref, the largest V scale the warp has
//               seen, keeps the operand in [0, 1]; a growing s_ref rescales O
//               like a growing running max.  O is multiplied by s_ref at the
//               end.
// The chunk's (m_i, l_i, O_i) then go through the same combine and merge as
// the bf16 pass.
#include <cmath>
#include <cstdio>

#include "fd_device.cuh"
#include "fd_internal.h"
#include "fd_tma.h"

namespace fd {

__device__ unsigned int g_status_fp8;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kScaleBox = 68;     // scales per copy: a 64-token tile + up to 3 of alignment slack
constexpr int kScaleSlot = 384;   // bytes reserved per scale copy in shared memory (128-byte multiple)

// Four e4m3 codes (bytes 0..3 of w) -> two fp16x2 words: lo = (byte 0, byte 1),
// hi = (byte 2, byte 3), the lower byte in the lower half.  Exact.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 a, b;\n\t"
        "mov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// Two fp32 -> two e4m3 codes (round to nearest even, saturating to +-448),
// `lo` in the low byte of the result.
__device__ __forceinline__ uint32_t e4m3x2_from_f32(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b16 t;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n\t"
        "cvt.u32.u16 %0, t;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}

// ---------------------------------------------------------------------------
// Encoder: one warp per cache row; lane l holds channels D/32 * l ...
template <int D>
__global__ void __launch_bounds__(256)
fp8_quantize_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ seq_lens, int H, int L_max,
                    long long rows, uint8_t* __restrict__ codes, float* __restrict__ scales) {
    constexpr int E = D / 32;  // channels per lane: 4 or 2
    const int lane = threadIdx.x & 31;
    const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
         row += nwarps) {
        const int t = (int)(row % L_max);
        const int b = (int)(row / ((long long)H * L_max));
        const int L = clamped_len(seq_lens, b, L_max, &g_status_fp8);
        if (t >= L) continue;  // warp-uniform: rows past the sequence are not written
        float v[E];
        if constexpr (E == 4) {
            const uint2 w = *reinterpret_cast<const uint2*>(x + row * D + lane * 4);
            const float2 a = bf16x2_to_float2(w.x), c = bf16x2_to_float2(w.y);
            v[0] = a.x; v[1] = a.y; v[2] = c.x; v[3] = c.y;
        } else {
            const uint32_t w = *reinterpret_cast<const uint32_t*>(x + row * D + lane * 2);
            const float2 a = bf16x2_to_float2(w);
            v[0] = a.x; v[1] = a.y;
        }
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(v[e]));
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const float s = amax / 448.0f;
        uint32_t packed = 0;
#pragma unroll
        for (int e = 0; e < E; e += 2) {
            const uint32_t pair = s != 0.f ? e4m3x2_from_f32(v[e] / s, v[e + 1] / s) : 0u;
            packed |= pair << (8 * e);
        }
        if constexpr (E == 4) *reinterpret_cast<uint32_t*>(codes + row * D + lane * 4) = packed;
        else *reinterpret_cast<uint16_t*>(codes + row * D + lane * 2) = (uint16_t)packed;
        if (lane == 0) scales[row] = s;
    }
}

// ---------------------------------------------------------------------------
// Partial pass.
struct Fp8Params {
    const uint16_t* q;
    const int32_t* seq_lens;
    const int32_t* page_table;
    int max_pages, num_pages;
    int Hq, Hkv, L_max, G;
    float scale_log2;
    int splits, chunk_fixed;
    StoreTarget st;
};

// Byte offset of 16-byte chunk `ch` of code row `row` in a 64-row box
// (128-byte rows: 128-byte swizzle; 64-byte rows: 64-byte swizzle).
template <int D>
__device__ __forceinline__ uint32_t code_off(int row, int ch) {
    if constexpr (D == 128) return swz(row, ch);
    else return swz64(row, ch);
}

// Resident CTAs per SM the partial pass is compiled for: 3 for the paged pool
// (4 stages, 128 registers), 2 for the contiguous cache (6 stages).
template <bool PAGED>
constexpr int fp8_min_ctas() { return PAGED ? 3 : 2; }

template <int D, int STAGES, int NT, bool PAGED>
__global__ void __launch_bounds__(5 * 32, fp8_min_ctas<PAGED>())
fp8_partial_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                   const __grid_constant__ CUtensorMap tmks, const __grid_constant__ CUtensorMap tmvs,
                   const Fp8Params p) {
    constexpr int CW = 4;
    constexpr int CB = 64 * D;        // bytes of one code tile (64 rows of D bytes)
    constexpr int STAGE = 2 * CB;     // K tile + V tile
    constexpr int SSTAGE = 2 * kScaleSlot;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char* scl = smem + STAGES * STAGE;
    uint64_t* full = reinterpret_cast<uint64_t*>(scl + STAGES * SSTAGE);
    uint64_t* empty = full + STAGES;
    int* stage_rows = reinterpret_cast<int*>(empty + STAGES);
    int* stage_off = stage_rows + STAGES;

    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait_primary();  // the previous kernel in the stream may still be running
    const int L = clamped_len(p.seq_lens, b, p.L_max, &g_status_fp8);
    const int chunk = chunk_len(L, p.splits, p.chunk_fixed);
    const int t0 = split * chunk;
    const int t1 = min(L, t0 + chunk);
    const int hq0 = h * p.G;

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
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CW);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == CW) {
        // ---------------- producer: one lane issues all tile copies --------
        if (lane == 0) {
            prefetch_tmap(&tmk);
            prefetch_tmap(&tmv);
            prefetch_tmap(&tmks);
            prefetch_tmap(&tmvs);
            const uint64_t pol = l2_evict_first_policy();
            const int head_row0 = PAGED ? 0 : (b * p.Hkv + h) * p.L_max;
            for (int t = 0; t < ntiles; ++t) {
                const int s = t % STAGES;
                const uint32_t ph = (uint32_t)(t / STAGES) & 1u;
                if (!mbar_wait(&empty[s], ph ^ 1u)) {
                    atomicOr(&g_status_fp8, kStatusTimeout);
                    break;
                }
                const int tok = t0 + t * kTile;
                const int rows = min(kTile, t1 - tok);
                int y;
                bool ok = true;
                if (PAGED) {
                    const int pg = p.page_table[(size_t)b * p.max_pages + tok / kTile];
                    ok = pg >= 0 && pg < p.num_pages;
                    y = (pg * p.Hkv + h) * kTile;
                } else {
                    y = head_row0 + tok;
                }
                unsigned char* sk = smem + s * STAGE;
                unsigned char* ss = scl + s * SSTAGE;
                if (ok) {
                    stage_rows[s] = rows;
                    stage_off[s] = y & 3;
                    mbar_arrive_expect_tx(&full[s], STAGE + 2 * kScaleBox * 4);
                    if constexpr (D == 128) {
                        tma_load_box(sk, &tmk, 0, y, &full[s], pol);
                        tma_load_box(sk + CB, &tmv, 0, y, &full[s], pol);
                    } else {
                        tma_load_box64(sk, &tmk, y, &full[s], pol);
                        tma_load_box64(sk + CB, &tmv, y, &full[s], pol);
                    }
                    // the scale copies start on the 16-byte boundary at or below the tile
                    tma_load_1d(ss, &tmks, y & ~3, &full[s], pol);
                    tma_load_1d(ss + kScaleSlot, &tmvs, y & ~3, &full[s], pol);
                } else {
                    atomicOr(&g_status_fp8, kStatusBadPage);
                    stage_rows[s] = 0;
                    stage_off[s] = 0;
                    mbar_arrive(&full[s]);
                }
            }
        }
        pdl_launch_dependents();
        return;
    }

    // ------------------------------ consumers ------------------------------
    const int gid = lane >> 2, tig = lane & 3, mi = lane >> 3;
    // Q as the B fragment of S = K Q^T: channels 16c + 4*tig + {0,1} (qa0) and
    // {2,3} (qa2) of query gid, times 2^-e with e the exponent of the query's
    // largest |q|.  The accumulators hold rows (tokens) gid, gid + 8 and
    // columns (queries) 2 tig, 2 tig + 1.
    uint32_t qa0[D / 16], qa2[D / 16];
    float2 qmul;  // columns 2 tig, 2 tig + 1
    {
        float qv[D / 16][4];
        float amax = 0.f;
        const uint16_t* qrow = p.q + (size_t)(b * p.Hq + hq0 + gid) * D;
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
            if (gid < p.G) {
                const uint2 w = *reinterpret_cast<const uint2*>(qrow + 16 * c + 4 * tig);
                const float2 a = bf16x2_to_float2(w.x), d2 = bf16x2_to_float2(w.y);
                qv[c][0] = a.x; qv[c][1] = a.y; qv[c][2] = d2.x; qv[c][3] = d2.y;
            } else {
                qv[c][0] = qv[c][1] = qv[c][2] = qv[c][3] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fabsf(qv[c][e]));
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        int ex = 0;
        if (amax > 0.f && amax <= 3.4e38f) (void)frexpf(amax, &ex);
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
            qa0[c] = pack_f16(ldexpf(qv[c][0], -ex), ldexpf(qv[c][1], -ex));
            qa2[c] = pack_f16(ldexpf(qv[c][2], -ex), ldexpf(qv[c][3], -ex));
        }
        const float qm = ldexpf(p.scale_log2, ex);  // query gid's; lane 4q holds query q
        qmul = make_float2(__shfl_sync(0xffffffffu, qm, 8 * tig), __shfl_sync(0xffffffffu, qm, 8 * tig + 4));
    }

    float o[D / 16][4];
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) o[mt][i] = 0.f;
    float2 m_run = make_float2(-INFINITY, -INFINITY), l_run = make_float2(0.f, 0.f);  // columns 2 tig, 2 tig + 1
    float vref = 0.f;
    bool failed = false;
    const int ld_row = warp * 16 + 8 * (mi >> 1) + (lane & 7);  // row this lane addresses for ldmatrix
    const int r0 = warp * 16 + 2 * tig;                         // V^T P^T: tokens r0, r0+1, r0+8, r0+9
    const int srow[2] = {warp * 16 + gid, warp * 16 + gid + 8};  // S = K Q^T: the lane's accumulator rows
    constexpr int VW = D / 32;                                  // V words per token and lane (D/8 channels)
    // byte offset of this lane's V channels D/8 * gid .. within a code row
    const uint32_t vofs_lo = D == 128 ? 0u : 8u * (uint32_t)(gid & 1);
    const int vch = D == 128 ? gid : gid >> 1;

    const int tok[4] = {r0, r0 + 1, r0 + 8, r0 + 9};
    for (int t = 0; t < ntiles; t += NT) {
        // NT consecutive stages per step; a step past the last tile reuses the
        // first stage's buffers with no valid rows (everything masked)
        int st[NT], rows[NT];
        bool have[NT];
#pragma unroll
        for (int k = 0; k < NT; ++k) {
            have[k] = t + k < ntiles;
            st[k] = have[k] ? (t + k) % STAGES : t % STAGES;
            rows[k] = 0;
            if (have[k]) {
                if (!warp_wait(&full[st[k]], (uint32_t)((t + k) / STAGES) & 1u)) failed = true;
                else rows[k] = stage_rows[st[k]];
            }
        }
        if (failed) {
            atomicOr(&g_status_fp8, kStatusTimeout);
            break;
        }

        // ---- S = K Q^T over this warp's 16 tokens of each stage ---------------
        float sacc[NT][4];
#pragma unroll
        for (int k = 0; k < NT; ++k) {
#pragma unroll
            for (int i = 0; i < 4; ++i) sacc[k][i] = 0.f;
            const uint32_t kt = smem_u32(smem + st[k] * STAGE);
#pragma unroll
            for (int kk = 0; kk < D / 32; ++kk) {
                // w0 / w2: rows gid / gid + 8, channels 32 kk + 4 tig ..; w1 / w3: the next 16 channels
                uint32_t w0, w1, w2, w3, a0, a1, a2, a3;
                ldsm_x4(kt + code_off<D>(ld_row, 2 * kk + (mi & 1)), w0, w1, w2, w3);
                e4m3x4_to_f16x4(w0, a0, a2);
                e4m3x4_to_f16x4(w2, a1, a3);
                mma_f16(sacc[k], a0, a1, a2, a3, qa0[2 * kk], qa2[2 * kk]);
                e4m3x4_to_f16x4(w1, a0, a2);
                e4m3x4_to_f16x4(w3, a1, a3);
                mma_f16(sacc[k], a0, a1, a2, a3, qa0[2 * kk + 1], qa2[2 * kk + 1]);
            }
        }
        float sc[NT][4], vs[NT][2];  // scores (rows gid, gid + 8 x columns); V scales of rows gid, gid + 8
#pragma unroll
        for (int k = 0; k < NT; ++k) {
            const float* ksc = reinterpret_cast<const float*>(scl + st[k] * SSTAGE) + stage_off[st[k]];
            const float* vsc = reinterpret_cast<const float*>(scl + st[k] * SSTAGE + kScaleSlot) + stage_off[st[k]];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const bool ok = srow[r] < rows[k];
                const float ks = ok ? ksc[srow[r]] : 0.f;
                sc[k][2 * r] = ok ? sacc[k][2 * r] * ks * qmul.x : -INFINITY;
                sc[k][2 * r + 1] = ok ? sacc[k][2 * r + 1] * ks * qmul.y : -INFINITY;
                vs[k][r] = ok ? vsc[srow[r]] : 0.f;
            }
        }

        // ---- online softmax per column and the V reference scale ---------------
        float mx0 = -INFINITY, mx1 = -INFINITY, vmax = 0.f;
#pragma unroll
        for (int k = 0; k < NT; ++k) {
            mx0 = fmaxf(mx0, fmaxf(sc[k][0], sc[k][2]));
            mx1 = fmaxf(mx1, fmaxf(sc[k][1], sc[k][3]));
            vmax = fmaxf(vmax, fmaxf(vs[k][0], vs[k][1]));
        }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {  // over the 16 rows: the lanes of equal tig
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, off));
        }
        const float vref_new = fmaxf(vref, vmax);
        const float vinv = vref_new > 0.f ? __fdividef(1.f, vref_new) : 0.f;
        const float vf = vref_new > 0.f ? vref * vinv : 1.f;
        vref = vref_new;
        const float m0 = fmaxf(m_run.x, mx0), m1 = fmaxf(m_run.y, mx1);
        const bool none0 = m0 == -INFINITY, none1 = m1 == -INFINITY;
        const float alpha0 = none0 ? 1.f : exp2_approx(m_run.x - m0);
        const float alpha1 = none1 ? 1.f : exp2_approx(m_run.y - m1);
        m_run = make_float2(m0, m1);
        float lsum0 = 0.f, lsum1 = 0.f;
        uint32_t pb[NT][2];
#pragma unroll
        for (int k = 0; k < NT; ++k) {
            float pr[4];
            pr[0] = none0 ? 0.f : exp2_approx(sc[k][0] - m0);
            pr[1] = none1 ? 0.f : exp2_approx(sc[k][1] - m1);
            pr[2] = none0 ? 0.f : exp2_approx(sc[k][2] - m0);
            pr[3] = none1 ? 0.f : exp2_approx(sc[k][3] - m1);
            lsum0 += pr[0] + pr[2];
            lsum1 += pr[1] + pr[3];
            // P * s_V / s_ref of rows gid and gid + 8, then each 8x8 block transposed into P^T
            const float v0 = vs[k][0] * vinv, v1 = vs[k][1] * vinv;
            pb[k][0] = movmatrix_trans(pack_f16(pr[0] * v0, pr[1] * v0));
            pb[k][1] = movmatrix_trans(pack_f16(pr[2] * v1, pr[3] * v1));
        }
        l_run.x = l_run.x * alpha0 + lsum0;
        l_run.y = l_run.y * alpha1 + lsum1;
        if (!__all_sync(0xffffffffu, alpha0 == 1.f && alpha1 == 1.f && vf == 1.f)) {
            // accumulator columns are the lane's own queries 2*tig and 2*tig+1
            const float a_even = alpha0 * vf, a_odd = alpha1 * vf;
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                o[mt][0] *= a_even;
                o[mt][1] *= a_odd;
                o[mt][2] *= a_even;
                o[mt][3] *= a_odd;
            }
        }

        // ---- O^T += V^T P^T ----------------------------------------------------
#pragma unroll
        for (int k = 0; k < NT; ++k) {
            const uint32_t vt = smem_u32(smem + st[k] * STAGE) + CB;
            uint32_t vw[4][VW];  // [token r0, r0+1, r0+8, r0+9][word]
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t a = vt + code_off<D>(tok[i], vch) + vofs_lo;
                if constexpr (VW == 4) {
                    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                                 : "=r"(vw[i][0]), "=r"(vw[i][1]), "=r"(vw[i][2]), "=r"(vw[i][3])
                                 : "r"(a));
                } else {
                    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(vw[i][0]), "=r"(vw[i][1]) : "r"(a));
                }
            }
            if (warp * 16 + 16 > rows[k]) {  // rows past the tile's end may hold any bytes (0 * NaN = NaN)
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int w = 0; w < VW; ++w) vw[i][w] = tok[i] < rows[k] ? vw[i][w] : 0u;
            }
#pragma unroll
            for (int j = 0; j < D / 16; ++j) {
                // channels D/8 * gid + 2j + {0, 1}: tokens (r0, r0+1) and (r0+8, r0+9)
                const uint32_t sel = (j & 1) ? 0x7362u : 0x5140u;
                uint32_t a0, a1, a2, a3;
                e4m3x4_to_f16x4(__byte_perm(vw[0][j >> 1], vw[1][j >> 1], sel), a0, a1);
                e4m3x4_to_f16x4(__byte_perm(vw[2][j >> 1], vw[3][j >> 1], sel), a2, a3);
                mma_f16(o[j], a0, a1, a2, a3, pb[k][0], pb[k][1]);
            }
        }
        __syncwarp();
        if (lane == 0) {
#pragma unroll
            for (int k = 0; k < NT; ++k)
                if (have[k]) mbar_arrive(&empty[st[k]]);
        }
    }
    pdl_launch_dependents();

    // ---- combine the consumer warps and store --------------------------------
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {  // exp-sums over the 16 rows (the lanes of equal tig)
        l_run.x += __shfl_xor_sync(0xffffffffu, l_run.x, off);
        l_run.y += __shfl_xor_sync(0xffffffffu, l_run.y, off);
    }
    named_barrier(1, CW * 32);  // every consumer is done with the stage ring
    float* red_o = reinterpret_cast<float*>(smem);  // [CW][8][D]
    float* red_m = red_o + CW * 8 * D;              // [CW][8]
    float* red_l = red_m + CW * 8;                  // [CW][8]
#pragma unroll
    for (int jj = 0; jj < D / 32; ++jj) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            // query 2*tig + i, channels D/8 * gid + 4*jj .. + 3
            const int qi = 2 * tig + i;
            const float4 val = make_float4(o[2 * jj][i] * vref, o[2 * jj][i + 2] * vref, o[2 * jj + 1][i] * vref,
                                           o[2 * jj + 1][i + 2] * vref);
            *reinterpret_cast<float4*>(red_o + (warp * 8 + qi) * D + (D / 8) * gid + 4 * jj) = val;
        }
    }
    if (gid == 0) {
        red_m[warp * 8 + 2 * tig] = failed ? -INFINITY : m_run.x;
        red_m[warp * 8 + 2 * tig + 1] = failed ? -INFINITY : m_run.y;
        red_l[warp * 8 + 2 * tig] = failed ? 0.f : l_run.x;
        red_l[warp * 8 + 2 * tig + 1] = failed ? 0.f : l_run.y;
    }
    named_barrier(1, CW * 32);
    store_combined<D, 8, CW>(smem, threadIdx.x, p.G, b * p.Hq + hq0, split, p.st);
}

template <int D, bool PAGED>
struct Fp8Launcher {
    // two stages per consumer step share the softmax bookkeeping and give each
    // warp two independent MMA chains.  Contiguous cache: six stages keep ~100
    // KiB per CTA in flight at 2 CTAs/SM.  Paged pool (ragged batches, where
    // more resident CTAs shorten the tail): four stages at 3 CTAs/SM.
    static constexpr int STAGES = PAGED ? 4 : 6;
    static constexpr int NT = 2;  // stages a consumer warp takes per step
    static_assert(STAGES >= 2 * NT, "the producer needs stages to fill while NT are consumed");
    static constexpr int STAGE = 2 * 64 * D;
    static constexpr int SMEM = 1024 + STAGES * STAGE + STAGES * 2 * kScaleSlot + STAGES * 16 + STAGES * 8 + 64;
    static constexpr int RED = 4 * 8 * D * 4 + 2 * 4 * 8 * 4;
    static_assert(STAGES * STAGE >= RED, "reduction scratch must fit in the ring");
    static constexpr auto kernel = fp8_partial_kernel<D, STAGES, NT, PAGED>;

    static cudaError_t prepare() {
        static bool done[kMaxDevices] = {};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < kMaxDevices && done[dev]) return cudaSuccess;
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
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
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, 5 * 32, SMEM) != cudaSuccess || n <= 0)
            return 1;
        if (dev < kMaxDevices) cache[dev] = n;
        return n;
    }
    static cudaError_t launch(const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tks,
                              const CUtensorMap& tvs, const Fp8Params& pp, dim3 grid, cudaStream_t st) {
        cudaError_t e = prepare();
        if (e != cudaSuccess) return e;
        return launch_pdl(kernel, grid, dim3(5 * 32), SMEM, st, tk, tv, tks, tvs, pp);
    }
};

}  // namespace

int fp8_ctas_per_sm(int D, bool paged) {
    if (D == 128) return paged ? Fp8Launcher<128, true>::ctas_per_sm() : Fp8Launcher<128, false>::ctas_per_sm();
    return paged ? Fp8Launcher<64, true>::ctas_per_sm() : Fp8Launcher<64, false>::ctas_per_sm();
}

cudaError_t launch_quantize_fp8(const Fp8QuantArgs& a, cudaStream_t stream) {
    const long long rows = (long long)a.B * a.H * a.L_max;
    if (rows == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long long want = (rows + 7) / 8;  // 8 rows (warps) per block
    const long long cap = (long long)sms * 8;
    const unsigned grid = (unsigned)(want < cap ? want : cap);
    const uint16_t* x = static_cast<const uint16_t*>(a.x);
    if (a.D == 128)
        fp8_quantize_kernel<128><<<grid, 256, 0, stream>>>(x, a.seq_lens, a.H, a.L_max, rows, a.codes, a.scales);
    else
        fp8_quantize_kernel<64><<<grid, 256, 0, stream>>>(x, a.seq_lens, a.H, a.L_max, rows, a.codes, a.scales);
    return cudaGetLastError();
}

cudaError_t launch_decode_fp8(const DecodeArgs& a, cudaStream_t stream) {
    if (a.B == 0) return cudaSuccess;
    const bool paged = a.page_table != nullptr;
    const uint64_t rows = paged ? (uint64_t)a.num_pages * a.Hkv * kTile : (uint64_t)a.B * a.Hkv * a.L_max;
    CUtensorMap tk, tv, tks, tvs;
    if (rows == 0) {
        // nothing can be read (an empty pool or cache): any well-formed map will do
        if (!make_row_map(&tk, a.q, 1, (uint32_t)a.D * 2) || !make_row_map(&tv, a.q, 1, (uint32_t)a.D * 2) ||
            !make_vec_map(&tks, a.q, 1, kScaleBox) || !make_vec_map(&tvs, a.q, 1, kScaleBox))
            return cudaErrorInvalidValue;
    } else if (!make_row_map(&tk, a.k, rows, (uint32_t)a.D) || !make_row_map(&tv, a.v, rows, (uint32_t)a.D) ||
               !make_vec_map(&tks, a.k_scales, rows, kScaleBox) || !make_vec_map(&tvs, a.v_scales, rows, kScaleBox)) {
        return cudaErrorInvalidValue;
    }
    Fp8Params pp;
    pp.q = static_cast<const uint16_t*>(a.q);
    pp.seq_lens = a.seq_lens;
    pp.page_table = a.page_table;
    pp.max_pages = a.max_pages;
    pp.num_pages = a.num_pages;
    pp.Hq = a.Hq;
    pp.Hkv = a.Hkv;
    pp.L_max = a.L_max;
    pp.G = a.Hq / a.Hkv;
    pp.scale_log2 = a.scale * kLog2e;
    pp.splits = a.splits;
    pp.chunk_fixed = a.chunk_fixed;
    pp.st.part_o = a.part_o;
    pp.st.part_ml = a.part_ml;
    pp.st.out = a.out;
    pp.st.out_bf16 = a.out_bf16;
    pp.st.lse = a.lse;
    pp.st.direct = a.splits == 1 ? 1 : 0;
    pp.st.splits = a.splits;
    const dim3 grid((unsigned)a.splits, (unsigned)a.Hkv, (unsigned)a.B);
    cudaError_t e;
    if (a.D == 128)
        e = paged ? Fp8Launcher<128, true>::launch(tk, tv, tks, tvs, pp, grid, stream)
                  : Fp8Launcher<128, false>::launch(tk, tv, tks, tvs, pp, grid, stream);
    else
        e = paged ? Fp8Launcher<64, true>::launch(tk, tv, tks, tvs, pp, grid, stream)
                  : Fp8Launcher<64, false>::launch(tk, tv, tks, tvs, pp, grid, stream);
    if (e != cudaSuccess || a.splits == 1) return e;
    return launch_merge(a.part_o, a.part_ml, a.seq_lens, a.B, a.Hq, a.L_max, a.D, a.splits, a.chunk_fixed,
                        a.out, a.out_bf16, a.lse, stream);
}

cudaError_t fp8_status_read(unsigned* bits, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(bits, g_status_fp8, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_status_fp8, &zero, sizeof(unsigned));
}

}  // namespace fd
