// fd_fp4.cu -- split-KV decode attention ("Flash Decoding" tutorial, sections
// 1-3) over a 4-bit floating-point KV cache, and its encoder, for sm_103a.
// The benchmarking blog on a hosted 1M-context model (section 1) names an
// "FP4" KV cache; this file implements this library's definition of one:
//
//   per cache row (token, KV head) and 32-channel block b:
//     e_b  = the smallest integer in [-126, 127] with 6 * 2^e_b >= max |x|
//     code = e2m1(x * 2^-e_b)      (round to nearest even; |x * 2^-e_b| <= 6)
//   one byte e_b + 127 per block; key codes two channels per byte (the low
//   nibble holds the even channel), value codes two tokens per byte (the low
//   nibble holds the even token, rows of pairs [(L_max + 1) / 2, D]).
//
// A row costs d/2 + d/32 bytes per operand (68 at d = 128), a quarter of the
// bf16 cache.  The partial pass has the shape of the fp8 pass (fd_fp8.cu):
// warp 4 copies per 64-token tile one K and one V code box and two scale
// boxes into a STAGES-deep ring; warps 0..3 each own 16 tokens of every tile.
// Both products run on fp16 tensor cores (every e2m1 value is exact in fp16):
//   S = K Q^T   the warp's 16 K rows are the A operand, the query group
//               (up to 8 columns) the B operand; one ldmatrix word per lane
//               holds 8 channels of one block of one row, each of its bytes
//               widens (cvt.rn.f16x2.e2m1x2) to one A register, Q's channel
//               order inside each block permuted alike; every block
//               accumulates on its own and is scaled by 2^e_b of its token
//               before the blocks are summed.
//   O^T += V^T P^T
//               the value cache is stored one channel of two consecutive
//               tokens per byte (token pairs), so ldmatrix.trans of a tile's
//               pair rows hands each lane bytes (pair, channel) that widen
//               (one cvt each) straight into A fragments of V^T: output tile
//               j holds channels 16j + 2*gid (row gid) and 16j + 2*gid + 1
//               (row gid + 8), its k index 2*tig + i / 8 + 2*tig + i is token
//               4*tig + i / 4*tig + 2 + i.  The score rows of S = K Q^T are
//               ordered to match (accumulator row m is token sigma(m)), so
//               movmatrix of P gives the B fragments directly, once per
//               tile; block b's operand multiplies them (mul.rn.f16x2) by
//               the fp16 pairs 2^e_b(token) / s_ref of their tokens, s_ref
//               the largest V block scale the warp has seen.  The block
//               scales are decoded once per row and step into a per-warp
//               buffer (K as floats, V as those fp16 pairs), and the query
//               fragments are read from shared memory where they are used:
//               the registers they free are worth more at 3 CTAs per SM.
#include <cmath>
#include <cstdio>

#include "fd_device.cuh"
#include "fd_internal.h"
#include "fd_tma.h"

namespace fd {

__device__ unsigned int g_status_fp4;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kScaleSlot = 384;  // bytes reserved per scale copy in shared memory (128-byte multiple)
constexpr int kStepTiles = 3;    // tiles a consumer warp takes per step
// per consumer warp and step, for each tile: the K block scales of its 16 rows
// (4 floats per row) and the V block scales of its 8 token pairs relative to
// the running reference (4 fp16x2 per pair)
constexpr int kScaleTileBytes = 16 * 4 * 4 + 8 * 4 * 4;
constexpr int kScaleBufBytes = 4 * kStepTiles * kScaleTileBytes;

// Geometry per head size: code bytes per row, scale bytes per row, and the
// scale copy (elements of SB bytes, a 64-token tile plus alignment slack).
template <int D>
struct F4Geo {
    static constexpr int RB = D / 2;                 // code bytes per row
    static constexpr int NB = D / 32;                // blocks per row = scale bytes per row
    static constexpr int SB = NB;                    // scale element: one row's scale bytes (4 or 2)
    static constexpr int ALIGN = 16 / SB;            // rows per 16 bytes of scales
    static constexpr int SBOX = 64 + ALIGN;          // scale elements per copy
    static constexpr int CB = 64 * RB;               // bytes of one code tile
    static_assert(SBOX * SB <= kScaleSlot, "scale copy must fit its slot");
};

// Byte offset of 16-byte chunk `ch` of code row `row` in a 64-row box
// (64-byte rows: 64-byte swizzle; 32-byte rows: no swizzle).
template <int D>
__device__ __forceinline__ uint32_t code4_off(int row, int ch) {
    if constexpr (D == 128) return swz64(row, ch);
    else return (uint32_t)(row * 32 + ch * 16);
}

// Four bytes of e2m1 pairs -> four fp16x2 words (byte i -> h[i], the low
// nibble in the low half).  Exact.
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t (&h)[4]) {
    asm("{\n\t.reg .b8 a, b, c, d;\n\t"
        "mov.b32 {a, b, c, d}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, a;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, c;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, d;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
}

// Two fp32 -> one byte of e2m1 codes (round to nearest even, saturating to
// +-6), `lo` in the low nibble.
__device__ __forceinline__ uint32_t e2m1x2_from_f32(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u32.u8 %0, t;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}

// Element-wise fp16x2 product, round to nearest even.
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// 2^(E - 127) for a scale byte E in [1, 254] (a normal binary32, exact).
__device__ __forceinline__ float scale_value(uint32_t E) { return __uint_as_float(E << 23); }



// ---------------------------------------------------------------------------
// Encoder: one warp per cache row; lane l holds channels D/32 * l ...
template <int D>
__global__ void __launch_bounds__(256)
fp4_quantize_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ seq_lens, int H, int L_max,
                    long long rows, uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
    constexpr int E = D / 32;       // channels per lane: 4 or 2
    constexpr int LPB = 32 / E;     // lanes per 32-channel block: 8 or 16
    const int lane = threadIdx.x & 31;
    const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
         row += nwarps) {
        const int t = (int)(row % L_max);
        const int b = (int)(row / ((long long)H * L_max));
        const int L = clamped_len(seq_lens, b, L_max, &g_status_fp4);
        if (t >= L) continue;  // warp-uniform: rows past the sequence are not written
        float v[E];
        if constexpr (E == 4) {
            const uint2 w = *reinterpret_cast<const uint2*>(x + row * D + lane * 4);
            const float2 a = bf16x2_to_float2(w.x), c = bf16x2_to_float2(w.y);
            v[0] = a.x; v[1] = a.y; v[2] = c.x; v[3] = c.y;
        } else {
            const float2 a = bf16x2_to_float2(*reinterpret_cast<const uint32_t*>(x + row * D + lane * 2));
            v[0] = a.x; v[1] = a.y;
        }
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(v[e]));
#pragma unroll
        for (int off = LPB / 2; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        // smallest e with 6 * 2^e >= amax: amax = 1.m * 2^k needs k - 2 when 1.m <= 1.5, else k - 1
        int eb = -126;
        const uint32_t bits = __float_as_uint(amax);
        if ((bits >> 23) != 0u) {
            const int k = (int)(bits >> 23) - 127;
            eb = max(-126, k - 2 + ((bits & 0x7fffffu) > 0x400000u ? 1 : 0));
        }
        const float inv = __uint_as_float((uint32_t)(127 - eb) << 23);  // 2^-eb, exact
        uint32_t packed = 0;
#pragma unroll
        for (int e = 0; e < E; e += 2) packed |= e2m1x2_from_f32(v[e] * inv, v[e + 1] * inv) << (4 * e);
        if constexpr (E == 4) *reinterpret_cast<uint16_t*>(codes + row * (D / 2) + lane * 2) = (uint16_t)packed;
        else codes[row * (D / 2) + lane] = (uint8_t)packed;
        if (lane % LPB == 0) scales[row * (D / 32) + lane / LPB] = (uint8_t)(eb + 127);
    }
}

// The same encoding for the value cache, stored in token pairs: one warp per
// pair of rows (tokens 2p, 2p + 1 of one head); lane l encodes channels
// D/32 * l ... of both rows, and channel c of the pair is one byte (the even
// token in the low nibble).  Pairs whose first token is past the sequence are
// not written; a second token past it encodes as code 0 with its scale
// byte not written.
template <int D>
__global__ void __launch_bounds__(256)
fp4_quantize_pairs_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ seq_lens, int H, int L_max,
                          long long pair_rows, uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
    constexpr int E = D / 32;       // channels per lane: 4 or 2
    constexpr int LPB = 32 / E;     // lanes per 32-channel block: 8 or 16
    const int Lp = (L_max + 1) / 2;
    const int lane = threadIdx.x & 31;
    const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long pr = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); pr < pair_rows;
         pr += nwarps) {
        const long long bh = pr / Lp;
        const int t0 = 2 * (int)(pr % Lp);
        const int b = (int)(bh / H);
        const int L = clamped_len(seq_lens, b, L_max, &g_status_fp4);
        if (t0 >= L) continue;  // warp-uniform
        const bool has1 = t0 + 1 < L;
        float v[2][E];
        int eb[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const long long row = bh * L_max + t0 + r;
            if (r == 1 && !has1) {
#pragma unroll
                for (int e = 0; e < E; ++e) v[r][e] = 0.f;
            } else if constexpr (E == 4) {
                const uint2 w = *reinterpret_cast<const uint2*>(x + row * D + lane * 4);
                const float2 a = bf16x2_to_float2(w.x), c = bf16x2_to_float2(w.y);
                v[r][0] = a.x; v[r][1] = a.y; v[r][2] = c.x; v[r][3] = c.y;
            } else {
                const float2 a = bf16x2_to_float2(*reinterpret_cast<const uint32_t*>(x + row * D + lane * 2));
                v[r][0] = a.x; v[r][1] = a.y;
            }
            float amax = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(v[r][e]));
#pragma unroll
            for (int off = LPB / 2; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
            eb[r] = -126;
            const uint32_t bits = __float_as_uint(amax);
            if ((bits >> 23) != 0u) {
                const int k = (int)(bits >> 23) - 127;
                eb[r] = max(-126, k - 2 + ((bits & 0x7fffffu) > 0x400000u ? 1 : 0));
            }
        }
        const float inv0 = __uint_as_float((uint32_t)(127 - eb[0]) << 23);  // 2^-eb, exact
        const float inv1 = __uint_as_float((uint32_t)(127 - eb[1]) << 23);
        uint32_t packed = 0;
#pragma unroll
        for (int e = 0; e < E; ++e) packed |= e2m1x2_from_f32(v[0][e] * inv0, v[1][e] * inv1) << (8 * e);
        if constexpr (E == 4) *reinterpret_cast<uint32_t*>(codes + pr * D + lane * 4) = packed;
        else *reinterpret_cast<uint16_t*>(codes + pr * D + lane * 2) = (uint16_t)packed;
        if (lane % LPB == 0) {
            scales[(bh * L_max + t0) * (D / 32) + lane / LPB] = (uint8_t)(eb[0] + 127);
            if (has1) scales[(bh * L_max + t0 + 1) * (D / 32) + lane / LPB] = (uint8_t)(eb[1] + 127);
        }
    }
}

// Byte offset of 16-byte chunk `ch` of a value pair row (D bytes: the
// 128-byte swizzle at D = 128, the 64-byte swizzle at D = 64).
template <int D>
__device__ __forceinline__ uint32_t vpair_off(int row, int ch) {
    if constexpr (D == 128) return swz(row, ch);
    else return swz64(row, ch);
}

// Token of the warp's 16-row slice that accumulator row m of S = K Q^T
// holds: rows 0..7 are tokens 0,1,4,5,8,9,12,13 and rows 8..15 tokens
// 2,3,6,7,10,11,14,15, so that the movmatrix transposes of P (k = 2*tig + i
// and 8 + 2*tig + i) meet the token order of the value pairs (4*tig + i and
// 4*tig + 2 + i).
__device__ __forceinline__ int score_row_token(int m) { return 2 * (m & 7) - (m & 1) + ((m >> 3) << 1); }

// ---------------------------------------------------------------------------
// Partial pass.
struct Fp4Params {
    const uint16_t* q;
    const int32_t* seq_lens;
    const int32_t* page_table;
    int max_pages, num_pages;
    int Hq, Hkv, L_max, G;
    float scale_log2;
    int splits, chunk_fixed;
    StoreTarget st;
};

template <int D, int STAGES, bool PAGED>
__global__ void __launch_bounds__(5 * 32, 3)
fp4_partial_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                   const __grid_constant__ CUtensorMap tmks, const __grid_constant__ CUtensorMap tmvs,
                   const Fp4Params p) {
    using Gm = F4Geo<D>;
    constexpr int CW = 4;
    constexpr int NT = kStepTiles;        // stages a consumer warp takes per step
    static_assert(STAGES >= 2 * NT, "the producer needs stages to fill while NT are consumed");
    constexpr int CB = Gm::CB;
    constexpr int STAGE = 2 * CB;         // K tile + V tile
    constexpr int SSTAGE = 2 * kScaleSlot;
    constexpr int NB = Gm::NB;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    unsigned char* scl = smem + STAGES * STAGE;
    uint64_t* full = reinterpret_cast<uint64_t*>(scl + STAGES * SSTAGE + kScaleBufBytes);
    uint64_t* empty = full + STAGES;
    int* stage_rows = reinterpret_cast<int*>(empty + STAGES);
    int* stage_off = stage_rows + STAGES;
    uint4* qsm = reinterpret_cast<uint4*>((reinterpret_cast<uintptr_t>(stage_off + STAGES) + 15) &
                                          ~static_cast<uintptr_t>(15));  // Q fragments [NB][32]

    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait_primary();  // the previous kernel in the stream may still be running
    const int L = clamped_len(p.seq_lens, b, p.L_max, &g_status_fp4);
    const int Lp = (p.L_max + 1) / 2;  // value pair rows per head
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
                    atomicOr(&g_status_fp4, kStatusTimeout);
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
                    stage_off[s] = y & (Gm::ALIGN - 1);
                    mbar_arrive_expect_tx(&full[s], STAGE + 2 * Gm::SBOX * Gm::SB);
                    // the value pair rows of the tile: 32 rows of D bytes
                    const int yv = PAGED ? y / 2 : (b * p.Hkv + h) * Lp + tok / 2;
                    tma_load_box64(sk, &tmk, y, &full[s], pol);  // one box of 64 rows (x = 0)
                    tma_load_box64(sk + CB, &tmv, yv, &full[s], pol);
                    // the scale copies start on the 16-byte boundary at or below the tile
                    tma_load_1d(ss, &tmks, y & ~(Gm::ALIGN - 1), &full[s], pol);
                    tma_load_1d(ss + kScaleSlot, &tmvs, y & ~(Gm::ALIGN - 1), &full[s], pol);
                } else {
                    atomicOr(&g_status_fp4, kStatusBadPage);
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
    // Q as the B fragment of S = K Q^T, query gid, per block c: qa[c][0] =
    // channels 32c + 8*tig + {0,1}, [1] = {2,3}, [2] = {4,5}, [3] = {6,7}, as
    // fp16 times 2^-e (e the exponent of the query's largest |q|; exact).  The
    // accumulators hold rows (tokens) gid, gid + 8 and columns (queries)
    // 2 tig, 2 tig + 1.
    float2 qmul;  // columns 2 tig, 2 tig + 1
    {
        uint32_t qa[NB][4];
        const uint16_t* qrow = p.q + (size_t)(b * p.Hq + hq0 + gid) * D;
        float amax = 0.f;
        uint4 qw[NB];
#pragma unroll
        for (int c = 0; c < NB; ++c) {
            qw[c] = gid < p.G ? *reinterpret_cast<const uint4*>(qrow + 32 * c + 8 * tig) : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t wv[4] = {qw[c].x, qw[c].y, qw[c].z, qw[c].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = bf16x2_to_float2(wv[i]);
                amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        int ex = 0;
        if (amax > 0.f && amax <= 3.4e38f) (void)frexpf(amax, &ex);
#pragma unroll
        for (int c = 0; c < NB; ++c) {
            const uint32_t wv[4] = {qw[c].x, qw[c].y, qw[c].z, qw[c].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = bf16x2_to_float2(wv[i]);
                qa[c][i] = pack_f16(ldexpf(f.x, -ex), ldexpf(f.y, -ex));
            }
        }
        const float qm = ldexpf(p.scale_log2, ex);  // query gid's; lane 4q holds query q
        qmul = make_float2(__shfl_sync(0xffffffffu, qm, 8 * tig), __shfl_sync(0xffffffffu, qm, 8 * tig + 4));
        // every consumer warp holds the same fragments: one copy in shared memory,
        // [block][lane] so that a warp's 16-byte reads hit distinct banks
        if (warp == 0)
#pragma unroll
            for (int c = 0; c < NB; ++c) qsm[c * 32 + lane] = make_uint4(qa[c][0], qa[c][1], qa[c][2], qa[c][3]);
        named_barrier(1, CW * 32);
    }

    float o[D / 16][4];
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) o[mt][i] = 0.f;
    float2 m_run = make_float2(-INFINITY, -INFINITY), l_run = make_float2(0.f, 0.f);  // columns 2 tig, 2 tig + 1
    float vref = 0.f;
    bool failed = false;
    // S = K Q^T: the token each lane addresses for ldmatrix (accumulator row
    // 8 * (mi / 2) + lane % 8) and the tokens of the lane's accumulator rows
    const int ld_row = warp * 16 + score_row_token(8 * (mi >> 1) + (lane & 7));
    const int srl[2] = {score_row_token(gid), score_row_token(gid + 8)};  // within the warp's 16 rows
    const int srow[2] = {warp * 16 + srl[0], warp * 16 + srl[1]};
    float* kbuf = reinterpret_cast<float*>(scl + STAGES * SSTAGE + warp * NT * kScaleTileBytes);  // [NT][16][4]
    uint32_t* vbuf = reinterpret_cast<uint32_t*>(kbuf + NT * 16 * 4);                              // [NT][8][NB]
    const int pv = NB == 4 ? lane >> 2 : (lane >> 1) & 7;  // the token pair whose V scales the lane turns into fp16
    const int cv = NB == 4 ? lane & 3 : lane & 1;          // and the block

    for (int t = 0; t < ntiles; t += NT) {
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
            atomicOr(&g_status_fp4, kStatusTimeout);
            break;
        }
        // the scale copies start this many rows before the tile (a page starts on a
        // 64-row boundary: none)
        auto soff = [&](int s) { return PAGED ? 0 : stage_off[s]; };

        // ---- key block scales ----------------------------------------------------
        // Lane l decodes blocks 2(l % 2), 2(l % 2) + 1 (block l % 2 at d = 64) of
        // row l / 2 of the warp's 16 (natural token order) as 2^(E - 127) into
        // kbuf[k][row][block].  Rows past the tile read as scale byte 0 (scale 0).
#pragma unroll
        for (int k = 0; k < NT; ++k) {
            const unsigned char* ksrc = scl + st[k] * SSTAGE + soff(st[k]) * Gm::SB;
            const int lr = lane >> 1;
            uint32_t kw = 0u;
            if (warp * 16 + lr < rows[k]) {
                if constexpr (NB == 4) kw = *reinterpret_cast<const uint32_t*>(ksrc + 4 * (warp * 16 + lr));
                else kw = *reinterpret_cast<const uint16_t*>(ksrc + 2 * (warp * 16 + lr));
            }
            float* kdst = kbuf + (k * 16 + lr) * 4;
            if constexpr (NB == 4) {
                const int c0 = 2 * (lane & 1);
                *reinterpret_cast<float2*>(kdst + c0) =
                    make_float2(scale_value((kw >> (8 * c0)) & 0xffu), scale_value((kw >> (8 * c0 + 8)) & 0xffu));
            } else {
                kdst[lane & 1] = scale_value((kw >> (8 * (lane & 1))) & 0xffu);
            }
        }
        __syncwarp();

        // ---- scores, block by block -------------------------------------------
        float sc[NT][4];  // rows gid, gid + 8 x columns 2 tig, 2 tig + 1
#pragma unroll
        for (int k = 0; k < NT; ++k) {
            const uint32_t kt = smem_u32(smem + st[k] * STAGE);
            float kf[2][NB];  // the K block scales of rows gid, gid + 8
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const float* src = kbuf + (k * 16 + srl[r]) * 4;
                if constexpr (NB == 4) {
                    const float4 f = *reinterpret_cast<const float4*>(src);
                    kf[r][0] = f.x; kf[r][1] = f.y; kf[r][2] = f.z; kf[r][3] = f.w;
                } else {
                    const float2 f = *reinterpret_cast<const float2*>(src);
                    kf[r][0] = f.x; kf[r][1] = f.y;
                }
            }
            float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);  // rows gid, gid + 8
#pragma unroll
            for (int cp = 0; cp < NB / 2; ++cp) {
                // (rows gid, block 2cp), (gid, 2cp+1), (gid + 8, 2cp), (gid + 8, 2cp+1)
                uint32_t w[4];
                ldsm_x4(kt + code4_off<D>(ld_row, 2 * cp + (mi & 1)), w[0], w[1], w[2], w[3]);
#pragma unroll
                for (int hb = 0; hb < 2; ++hb) {
                    const int c = 2 * cp + hb;
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
                    uint32_t ha[4], hb8[4];
                    e2m1x8_to_f16x8(w[hb], ha);       // row gid: channels 32c + 8 tig ..
                    e2m1x8_to_f16x8(w[2 + hb], hb8);  // row gid + 8
                    const uint4 qf = qsm[c * 32 + lane];
                    mma_f16(acc, ha[0], hb8[0], ha[1], hb8[1], qf.x, qf.y);
                    mma_f16(acc, ha[2], hb8[2], ha[3], hb8[3], qf.z, qf.w);
                    s0 = __ffma2_rn(make_float2(acc[0], acc[1]), make_float2(kf[0][c], kf[0][c]), s0);
                    s1 = __ffma2_rn(make_float2(acc[2], acc[3]), make_float2(kf[1][c], kf[1][c]), s1);
                }
            }
            const bool ok0 = srow[0] < rows[k], ok1 = srow[1] < rows[k];
            sc[k][0] = ok0 ? s0.x * qmul.x : -INFINITY;
            sc[k][1] = ok0 ? s0.y * qmul.y : -INFINITY;
            sc[k][2] = ok1 ? s1.x * qmul.x : -INFINITY;
            sc[k][3] = ok1 ? s1.y * qmul.y : -INFINITY;
        }

        // ---- online softmax per column and the V reference scale ---------------
        // V: lane l reads the scale bytes of block cv of the token pair pv = l / 4
        // (l / 2 mod 8 at d = 64), rows 2 pv and 2 pv + 1 (byte 0 past the tile); the
        // warp's largest byte is the step's largest scale (one redux), and the bytes
        // become fp16 pairs over the reference below.
        float mx0 = -INFINITY, mx1 = -INFINITY;
        uint32_t ev[NT][2];
        uint32_t emax = 0u;
#pragma unroll
        for (int k = 0; k < NT; ++k) {
            mx0 = fmaxf(mx0, fmaxf(sc[k][0], sc[k][2]));
            mx1 = fmaxf(mx1, fmaxf(sc[k][1], sc[k][3]));
            const unsigned char* vsrc = scl + st[k] * SSTAGE + soff(st[k]) * Gm::SB + kScaleSlot;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int r = warp * 16 + 2 * pv + h;
                ev[k][h] = r < rows[k] ? (uint32_t)vsrc[Gm::SB * r + cv] : 0u;
                emax = max(emax, ev[k][h]);
            }
        }
        emax = __reduce_max_sync(0xffffffffu, emax);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {  // over the 16 rows: the lanes of equal tig
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float vref_new = fmaxf(vref, scale_value(emax));
        const float vinv = vref_new > 0.f ? __fdividef(1.f, vref_new) : 0.f;
        const float vf = vref_new > 0.f ? vref * vinv : 1.f;
        vref = vref_new;
        // V block scales over the reference as fp16 pairs: lane l writes block cv of
        // its token pair pv, (s(2 pv) / s_ref, s(2 pv + 1) / s_ref), both <= 1
#pragma unroll
        for (int k = 0; k < NT; ++k)
            vbuf[(k * 8 + pv) * NB + cv] = pack_f16(scale_value(ev[k][0]) * vinv, scale_value(ev[k][1]) * vinv);
        __syncwarp();
        const float m0 = fmaxf(m_run.x, mx0), m1 = fmaxf(m_run.y, mx1);
        const bool none0 = m0 == -INFINITY, none1 = m1 == -INFINITY;
        const float alpha0 = none0 ? 1.f : exp2_approx(m_run.x - m0);
        const float alpha1 = none1 ? 1.f : exp2_approx(m_run.y - m1);
        m_run = make_float2(m0, m1);
        float lsum0 = 0.f, lsum1 = 0.f;
        float pr[NT][4];  // p, same layout as sc
#pragma unroll
        for (int k = 0; k < NT; ++k) {
            pr[k][0] = none0 ? 0.f : exp2_approx(sc[k][0] - m0);
            pr[k][1] = none1 ? 0.f : exp2_approx(sc[k][1] - m1);
            pr[k][2] = none0 ? 0.f : exp2_approx(sc[k][2] - m0);
            pr[k][3] = none1 ? 0.f : exp2_approx(sc[k][3] - m1);
            lsum0 += pr[k][0] + pr[k][2];
            lsum1 += pr[k][1] + pr[k][3];
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

        // ---- O^T += V^T P^T -------------------------------------------------
#pragma unroll
        for (int k = 0; k < NT; ++k) {
            const uint32_t vt = smem_u32(smem + st[k] * STAGE + CB);
            // P^T for each V block c: p * 2^e_c(token) / s_ref of accumulator rows gid and
            // gid + 8 (the scale is 0 past the tile, where the codes may be anything
            // finite), each 8x8 block transposed from the score layout
            // P^T of the tile (transposed from the score layout by movmatrix): b0 holds
            // tokens 4 tig, 4 tig + 1 (pair 2 tig), b1 tokens 4 tig + 2, 4 tig + 3
            // (pair 2 tig + 1), query gid; block c's operand scales each token by
            // its block scale over the reference
            const uint32_t p0 = movmatrix_trans(pack_f16(pr[k][0], pr[k][1]));
            const uint32_t p1 = movmatrix_trans(pack_f16(pr[k][2], pr[k][3]));
            uint32_t sv0[NB], sv1[NB];
            if constexpr (NB == 4) {
                const uint4 a = *reinterpret_cast<const uint4*>(vbuf + (k * 8 + 2 * tig) * NB);
                const uint4 c = *reinterpret_cast<const uint4*>(vbuf + (k * 8 + 2 * tig + 1) * NB);
                sv0[0] = a.x; sv0[1] = a.y; sv0[2] = a.z; sv0[3] = a.w;
                sv1[0] = c.x; sv1[1] = c.y; sv1[2] = c.z; sv1[3] = c.w;
            } else {
                const uint2 a = *reinterpret_cast<const uint2*>(vbuf + (k * 8 + 2 * tig) * NB);
                const uint2 c = *reinterpret_cast<const uint2*>(vbuf + (k * 8 + 2 * tig + 1) * NB);
                sv0[0] = a.x; sv0[1] = a.y;
                sv1[0] = c.x; sv1[1] = c.y;
            }
            uint32_t pb[NB][2];
#pragma unroll
            for (int c = 0; c < NB; ++c) {
                pb[c][0] = hmul2_u32(p0, sv0[c]);
                pb[c][1] = hmul2_u32(p1, sv1[c]);
            }
#pragma unroll
            for (int x = 0; x < D / 64; ++x) {
                // matrix j: the warp's 8 pair rows x channels 16 (4x + j) .. + 15; lane (gid, tig)
                // receives pairs 2 tig, 2 tig + 1 of channels 2 gid, 2 gid + 1 (one byte each)
                uint32_t w[4];
                ldsm_x4_t(vt + vpair_off<D>(warp * 8 + (lane & 7), 4 * x + (lane >> 3)), w[0], w[1], w[2], w[3]);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int ch = 4 * x + j;
                    uint32_t a[4];  // (ch 2gid: tokens 4tig, +1), (2gid+1: same), (2gid: 4tig+2, +3), (2gid+1: same)
                    e2m1x8_to_f16x8(w[j], a);
                    mma_f16(o[ch], a[0], a[1], a[2], a[3], pb[ch >> 1][0], pb[ch >> 1][1]);
                }
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
    for (int ch = 0; ch < D / 16; ++ch) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            // query 2*tig + i; output tile ch: channels 16 ch + 2 gid (row gid) and + 1 (row gid + 8)
            *reinterpret_cast<float2*>(red_o + (warp * 8 + 2 * tig + i) * D + 16 * ch + 2 * gid) =
                make_float2(o[ch][i] * vref, o[ch][i + 2] * vref);
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
struct Fp4Launcher {
    static constexpr int STAGES = 7;
    static constexpr int STAGE = 2 * F4Geo<D>::CB;
    static constexpr int SMEM =
        1024 + STAGES * STAGE + STAGES * 2 * kScaleSlot + kScaleBufBytes + STAGES * 16 + STAGES * 8 + 16 +
        F4Geo<D>::NB * 32 * 16 + 64;
    static constexpr int RED = 4 * 8 * D * 4 + 2 * 4 * 8 * 4;
    static_assert(STAGES * STAGE >= RED, "reduction scratch must fit in the ring");
    // three CTAs per SM: 228 KB of shared memory per SM, 1 KB of it reserved per CTA
    static_assert(3 * (SMEM + 1024) <= 228 * 1024, "three CTAs per SM must fit in shared memory");
    static constexpr auto kernel = fp4_partial_kernel<D, STAGES, PAGED>;

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
                              const CUtensorMap& tvs, const Fp4Params& pp, dim3 grid, cudaStream_t st) {
        cudaError_t e = prepare();
        if (e != cudaSuccess) return e;
        return launch_pdl(kernel, grid, dim3(5 * 32), SMEM, st, tk, tv, tks, tvs, pp);
    }
};

}  // namespace

int fp4_ctas_per_sm(int D, bool paged) {
    if (D == 128) return paged ? Fp4Launcher<128, true>::ctas_per_sm() : Fp4Launcher<128, false>::ctas_per_sm();
    return paged ? Fp4Launcher<64, true>::ctas_per_sm() : Fp4Launcher<64, false>::ctas_per_sm();
}

cudaError_t launch_quantize_fp4(const Fp4QuantArgs& a, cudaStream_t stream) {
    const long long rows = (long long)a.B * a.H * a.L_max;
    if (rows == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long long units = a.token_pairs ? (long long)a.B * a.H * ((a.L_max + 1) / 2) : rows;
    const long long want = (units + 7) / 8;  // 8 rows or pair rows (warps) per block
    const long long cap = (long long)sms * 8;
    const unsigned grid = (unsigned)(want < cap ? want : cap);
    const uint16_t* x = static_cast<const uint16_t*>(a.x);
    if (a.token_pairs) {
        if (a.D == 128)
            fp4_quantize_pairs_kernel<128><<<grid, 256, 0, stream>>>(x, a.seq_lens, a.H, a.L_max, units, a.codes,
                                                                     a.scales);
        else
            fp4_quantize_pairs_kernel<64><<<grid, 256, 0, stream>>>(x, a.seq_lens, a.H, a.L_max, units, a.codes,
                                                                    a.scales);
    } else if (a.D == 128) {
        fp4_quantize_kernel<128><<<grid, 256, 0, stream>>>(x, a.seq_lens, a.H, a.L_max, rows, a.codes, a.scales);
    } else {
        fp4_quantize_kernel<64><<<grid, 256, 0, stream>>>(x, a.seq_lens, a.H, a.L_max, rows, a.codes, a.scales);
    }
    return cudaGetLastError();
}

template <int D>
static bool fp4_maps(const DecodeArgs& a, uint64_t rows, uint64_t pair_rows, CUtensorMap& tk, CUtensorMap& tv,
                     CUtensorMap& tks, CUtensorMap& tvs) {
    using Gm = F4Geo<D>;
    if (rows == 0) {
        // nothing can be read (an empty pool or cache): any well-formed map will do
        return make_row_map(&tk, a.q, 1, Gm::RB) && make_row_map(&tv, a.q, 1, D, 32) &&
               make_vec_map(&tks, a.q, 1, Gm::SBOX, Gm::SB) && make_vec_map(&tvs, a.q, 1, Gm::SBOX, Gm::SB);
    }
    // keys: rows of D/2 bytes in 64-row boxes; values: pair rows of D bytes in 32-row boxes
    return make_row_map(&tk, a.k, rows, Gm::RB) && make_row_map(&tv, a.v, pair_rows, D, 32) &&
           make_vec_map(&tks, a.k_scales, rows, Gm::SBOX, Gm::SB) &&
           make_vec_map(&tvs, a.v_scales, rows, Gm::SBOX, Gm::SB);
}

cudaError_t launch_decode_fp4(const DecodeArgs& a, cudaStream_t stream) {
    if (a.B == 0) return cudaSuccess;
    const bool paged = a.page_table != nullptr;
    const uint64_t rows = paged ? (uint64_t)a.num_pages * a.Hkv * kTile : (uint64_t)a.B * a.Hkv * a.L_max;
    CUtensorMap tk, tv, tks, tvs;
    const uint64_t pair_rows =
        paged ? (uint64_t)a.num_pages * a.Hkv * (kTile / 2) : (uint64_t)a.B * a.Hkv * ((a.L_max + 1) / 2);
    const bool ok = a.D == 128 ? fp4_maps<128>(a, rows, pair_rows, tk, tv, tks, tvs)
                               : fp4_maps<64>(a, rows, pair_rows, tk, tv, tks, tvs);
    if (!ok) return cudaErrorInvalidValue;
    Fp4Params pp;
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
        e = paged ? Fp4Launcher<128, true>::launch(tk, tv, tks, tvs, pp, grid, stream)
                  : Fp4Launcher<128, false>::launch(tk, tv, tks, tvs, pp, grid, stream);
    else
        e = paged ? Fp4Launcher<64, true>::launch(tk, tv, tks, tvs, pp, grid, stream)
                  : Fp4Launcher<64, false>::launch(tk, tv, tks, tvs, pp, grid, stream);
    if (e != cudaSuccess || a.splits == 1) return e;
    return launch_merge(a.part_o, a.part_ml, a.seq_lens, a.B, a.Hq, a.L_max, a.D, a.splits, a.chunk_fixed,
                        a.out, a.out_bf16, a.lse, stream);
}

cudaError_t fp4_status_read(unsigned* bits, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(bits, g_status_fp4, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_status_fp4, &zero, sizeof(unsigned));
}

}  // namespace fd
