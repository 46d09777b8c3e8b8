// fd_topdelta.cu -- the sparse decode of the "Faster Flash Decoding" summary
// (PaperDaily) for sm_103a: the key encoder (section 5) and one fused pass
// per cache chunk that scans the 2-bit keys, takes the pseudo-max over the
// sink and window anchors (section 4), keeps keys with s~ >= m^ - delta
// (section 3), corrects the kept keys with their int8 residual and attends
// over them exactly (section 5, Fig. 2), with the stages fused as section 6
// asks: nothing but the per-chunk (m_i, l_i, O_i) leaves the chip.
//
// Fused pass, one CTA per (chunk, KV head, sequence), 2 producer + 4
// consumer warps, 64-token tiles (the same tile grid as the dense path):
//   * anchor pass: the consumer warps score the tiles that hold anchors and
//     take m^ per query head.  Every CTA of a (sequence, head) computes the
//     same m^ bit for bit: the anchor scores are produced by the same code,
//     lanes and operation order as the main scan.
//   * scan ring (2-bit codes + fp16 min/scale, 48 B per token at d=128, SS
//     stages): its own producer warp refills a stage with bulk copies as soon
//     as the consumers have scored the tile in it, so on a sparse cache
//     (few tiles with candidates, the pass reduced to the scan) the copies
//     run SS tiles ahead.  Consumers score tile k, store s~ in shared memory
//     and flag whether any query head of the group selected a token of it.
//   * detail ring (int8 residual + fp16 scales + bf16 V, 392 B per token):
//     the detail producer warp issues a tile's copies only once the
//     consumers flagged it, LA tiles before the consumers attend to it, so
//     the residual and V of tiles without candidates are never read.
//   * attend: exact scores s = s~ + scale * sum_g rs_g <q_g, rq_g> for the
//     candidates, online softmax and O^T += V^T P^T, then the same warp
//     combine and chunk merge as the dense pass.  With `group_union` every
//     query head of a KV group attends to the union of the group's candidate
//     sets (the tiles loaded are the same: a tile is loaded when any head of
//     the group selected one of its tokens).
// Both dot stages put the warp's 16 tokens in the MMA's M dimension and the
// group's query heads in N (S = K Q^T), so no accumulator is spent on
// padding query rows; movmatrix turns the P values into P^T fragments.
#include <cmath>
#include <cuda_fp16.h>

#include "fd_device.cuh"
#include "fd_internal.h"
#include "fd_tma.h"

namespace fd {

__device__ unsigned int g_status_topdelta;

namespace {

constexpr int kMaxDevices = 64;
constexpr int CW = 4;           // consumer warps
constexpr int NW = CW + 2;      // + the detail producer warp (CW) and the scan producer warp (CW + 1)
constexpr int LA = 2;           // tiles scanned ahead of the attend step
constexpr int DS = LA + 1;      // detail ring depth (= decision slots)
constexpr int SS = 8;           // scan ring depth: the scan producer keeps it full on its own

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
    static constexpr int NG = D / 32;          // 32-channel groups
    static constexpr int KS = D / 16;          // 16-channel k-steps
    static constexpr int CODES_ROW = D / 4;    // bytes per token row
    static constexpr int MS_ROW = D / 8;       // (mn16, s16) per group
    static constexpr int RES_ROW = D;
    static constexpr int RS_ROW = D / 16;      // rs16 per group
    static constexpr int SCAN_STAGE = kTile * (CODES_ROW + MS_ROW);
    static constexpr int RES_BYTES = kTile * RES_ROW;        // one box
    static constexpr int V_BYTES = kTile * 2 * D;            // D/64 boxes
    static constexpr int RS_BYTES = kTile * RS_ROW;
    static constexpr int DET_STAGE = (RES_BYTES + V_BYTES + RS_BYTES + 1023) / 1024 * 1024;
};

template <int D>
struct TLayout {
    using Gm = TGeo<D>;
    static constexpr int DET_OFF = 0;                                          // 1024-aligned boxes
    static constexpr int SCAN_OFF = DET_OFF + DS * Gm::DET_STAGE;
    static constexpr int DEC_OFF = SCAN_OFF + SS * Gm::SCAN_STAGE;             // s~ [DS][CW][32][4] f32
    static constexpr int FLAG_OFF = DEC_OFF + DS * CW * 32 * 16;               // need[DS][CW], loaded[DS], scan_rows[SS]
    static constexpr int BAR_OFF = (FLAG_OFF + (DS * CW + DS + SS) * 4 + 15) / 16 * 16;
    static constexpr int MH_OFF = BAR_OFF + (2 * SS + 3 * DS) * 8;             // anchor maxima [CW][8]
    static constexpr int QV = 3 * Gm::NG;                                      // query vectors per lane
    static constexpr int Q_OFF = (MH_OFF + CW * 8 * 4 + 15) / 16 * 16;         // [QV][32] x 16 B
    static constexpr int BYTES = 1024 + Q_OFF + QV * 32 * 16;
    static_assert(DS * Gm::DET_STAGE >= CW * 8 * D * 4 + 2 * CW * 8 * 4, "epilogue scratch must fit in the rings");
    static_assert(Gm::DET_STAGE >= Gm::SCAN_STAGE, "anchor staging must fit in one detail stage");
    // two CTAs per SM: 228 KB of shared memory per SM, 1 KB of it reserved per CTA
    static_assert(2 * (BYTES + 1024) <= 228 * 1024, "two CTAs per SM must fit in shared memory");
};

struct TDParams {
    const uint16_t* q;
    const uint8_t* codes;
    const uint8_t* mn_scale;
    const uint8_t* res_scale;
    const int32_t* seq_lens;
    int Hq, Hkv, L_max, G;
    float scale, delta;
    int n_sink, window;
    int splits, chunk_fixed;
    int group_union;  // every head of a KV group attends to the union of the group's candidates
    uint32_t* sel_mask;
    int32_t* sel_count;
    StoreTarget st;
};


// Both dot stages run as S = K Q^T on m16n8k16: the 16 token rows of a
// warp's slice are M, the (up to 8) query heads of the group are N, so every
// accumulator a lane holds belongs to a real token.  Lane (gid, tig) holds
// the B fragment of query gid and, in the accumulators, rows gid and gid + 8
// (tokens) x columns 2 tig, 2 tig + 1 (queries).
//
// B fragments of query gid per 16-channel k-step.  The k order inside a
// step is permuted to match how the A operands are unpacked (the same
// permutation on both sides leaves every dot product unchanged):
//   2-bit codes: k = 2t, 2t+1, 8+2t, 9+2t <-> channels 2t, 2t+8, 2t+1, 2t+9,
//                the last two unpacked as 4 * code and weighted by q / 4; the
//                codes enter as bf16 subnormals code * 2^-133 (the tensor
//                cores keep subnormal operands), so qc0 / qc2 carry the query
//                scaled by 2^(sq + 126), sq a per-query power of two with
//                max |q| * 2^sq in [1, 2): every product is exact and the dot
//                products are those of the plain codes times 2^(sq - 7) (up to
//                the tensor cores' fp32 accumulation order).
//   int8 residual (ldmatrix of 16-byte chunks): k = 2t, 2t+1, 8+2t, 9+2t <->
//   channels 4t, 4t+1, 4t+2, 4t+3          (t = tig, relative to 16*kk)
// The per-query constants are held for the lane's accumulator columns,
// queries 2 tig (.x) and 2 tig + 1 (.y).
template <int D>
struct TDQuery {
    uint32_t qc0[D / 16], qc2[D / 16];  // bf16, for the 2-bit scan (scaled, see above)
    uint32_t qr0[D / 16], qr2[D / 16];  // fp16, for the residual
    float2 qsum[D / 32];                // sum of the query over each 32-channel group, times 2^(sq - 7)
    float2 off[D / 32];                 // 1152 times the same sum over the query's fp16 values
    float2 scan_scale;                  // softmax scale times 2^(7 - sq)
};

// Scores s~ (natural-log units) of the warp's 16 rows of a tile whose codes
// and (mn16, s16) rows sit in shared memory (plain row-major).  st[i] is the
// score of row warp*16 + gid + 8*(i >> 1) for query 2*tig + (i & 1).
//   s~ = scale * sum_g ( s_g * <q, code>_g + mn_g * sum_g(q) )
// The per-group dots run on the tensor cores with the codes as exact bf16
// subnormals; the group sums are combined with explicitly rounded operations
// in group order.
template <int D>
__device__ __forceinline__ void scan_tile(const unsigned char* codes, const unsigned char* ms, int warp, int lane,
                                          const uint4* qv, float2 scan_scale, float (&st)[4]) {
    using Gm = TGeo<D>;
    const int gid = lane >> 2, tig = lane & 3;
    const int r0 = warp * 16 + gid, r1 = r0 + 8;
    // (mn16, s16) of every group for rows r0 and r1
    uint32_t ma[Gm::NG], mb[Gm::NG];
    if constexpr (Gm::NG == 4) {
        const uint4 a = *reinterpret_cast<const uint4*>(ms + r0 * Gm::MS_ROW);
        const uint4 bq = *reinterpret_cast<const uint4*>(ms + r1 * Gm::MS_ROW);
        ma[0] = a.x; ma[1] = a.y; ma[2] = a.z; ma[3] = a.w;
        mb[0] = bq.x; mb[1] = bq.y; mb[2] = bq.z; mb[3] = bq.w;
    } else {
        const uint2 a = *reinterpret_cast<const uint2*>(ms + r0 * Gm::MS_ROW);
        const uint2 bq = *reinterpret_cast<const uint2*>(ms + r1 * Gm::MS_ROW);
        ma[0] = a.x; ma[1] = a.y;
        mb[0] = bq.x; mb[1] = bq.y;
    }
    const uint4* ca = reinterpret_cast<const uint4*>(codes + r0 * Gm::CODES_ROW);
    const uint4* cb = reinterpret_cast<const uint4*>(codes + r1 * Gm::CODES_ROW);
    float2 v0 = make_float2(0.f, 0.f), v1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int kq = 0; kq < Gm::KS / 4; ++kq) {
        const uint4 wa4 = ca[kq], wb4 = cb[kq];
        const uint32_t wa[4] = {wa4.x, wa4.y, wa4.z, wa4.w};
        const uint32_t wb[4] = {wb4.x, wb4.y, wb4.z, wb4.w};
#pragma unroll
        for (int hg = 0; hg < 2; ++hg) {  // the two 32-channel groups of this 16-byte word
            const int g = 2 * kq + hg;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            const uint4 qg = qv[g * 32];  // qc0, qc2 of k-steps 2g and 2g + 1
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
                const uint32_t ua = wa[2 * hg + e2] >> (4 * tig), ub = wb[2 * hg + e2] >> (4 * tig);
                // bits 0-1 / 16-17: codes of the even pair as bf16 subnormals code * 2^-133; bits 2-3 /
                // 18-19: the odd pair as 4 * code * 2^-133 (qc2 carries the 1/4)
                mma_bf16(acc, ua & 0x00030003u, ub & 0x00030003u, ua & 0x000C000Cu, ub & 0x000C000Cu,
                         e2 ? qg.z : qg.x, e2 ? qg.w : qg.y);
            }
            const float4 qs4 = *reinterpret_cast<const float4*>(&qv[(2 * Gm::NG + g / 2) * 32]);
            const float2 qsum = (g & 1) ? make_float2(qs4.z, qs4.w) : make_float2(qs4.x, qs4.y);
            // group g of rows r0 / r1, queries 2 tig and 2 tig + 1: s_g * <q, code>_g + mn_g * sum_g(q),
            // added in g order
            const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&ma[g]));  // (mn, s) of row r0
            const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&mb[g]));  // (mn, s) of row r1
            v0 = __fadd2_rn(v0, __ffma2_rn(make_float2(fa.y, fa.y), make_float2(acc[0], acc[1]),
                                           __fmul2_rn(make_float2(fa.x, fa.x), qsum)));
            v1 = __fadd2_rn(v1, __ffma2_rn(make_float2(fb.y, fb.y), make_float2(acc[2], acc[3]),
                                           __fmul2_rn(make_float2(fb.x, fb.x), qsum)));
        }
    }
    // v is the group sum times 2^(sq - 7) exactly; scan_scale undoes the power of two
    st[0] = __fmul_rn(v0.x, scan_scale.x);
    st[1] = __fmul_rn(v0.y, scan_scale.y);
    st[2] = __fmul_rn(v1.x, scan_scale.x);
    st[3] = __fmul_rn(v1.y, scan_scale.y);
}

// Residual term sum_g rs_g * <q, rq>_g of the warp's 16 rows (same layout as
// scan_tile).  The int8 residual tile is one swizzled box; each lane's
// ldmatrix word holds 4 consecutive bytes of one row, which prmt with 0x64
// high bytes turns into the exact fp16 values 1152 + x.  The offset is
// removed from the fp32 sums afterwards; its rounding error (~1e-3 in units
// of rq) is scaled down by rs (~1e-2) and the softmax scale before it
// reaches a score.  Each group is folded into the running sum right after
// its two k-steps, in group order.
template <int D>
__device__ __forceinline__ void residual_tile(uint32_t res_s, const unsigned char* rs, int warp, int lane,
                                              const uint4* qv, float (&rt)[4]) {
    using Gm = TGeo<D>;
    const int gid = lane >> 2;
    const int mi = lane >> 3;
    const int ld_row = warp * 16 + 8 * (mi >> 1) + (lane & 7);
    const int r0 = warp * 16 + gid, r1 = r0 + 8;
    // rs16 of every group for rows r0 and r1
    __half2 ra[Gm::NG / 2], rb[Gm::NG / 2];
    if constexpr (Gm::NG == 4) {
        const uint2 a = *reinterpret_cast<const uint2*>(rs + r0 * Gm::RS_ROW);
        const uint2 bq = *reinterpret_cast<const uint2*>(rs + r1 * Gm::RS_ROW);
        ra[0] = *reinterpret_cast<const __half2*>(&a.x);
        ra[1] = *reinterpret_cast<const __half2*>(&a.y);
        rb[0] = *reinterpret_cast<const __half2*>(&bq.x);
        rb[1] = *reinterpret_cast<const __half2*>(&bq.y);
    } else {
        const uint32_t a = *reinterpret_cast<const uint32_t*>(rs + r0 * Gm::RS_ROW);
        const uint32_t bq = *reinterpret_cast<const uint32_t*>(rs + r1 * Gm::RS_ROW);
        ra[0] = *reinterpret_cast<const __half2*>(&a);
        rb[0] = *reinterpret_cast<const __half2*>(&bq);
    }
    float2 v0 = make_float2(0.f, 0.f), v1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int g = 0; g < Gm::NG; ++g) {
        const int chunk = 2 * g + (mi & 1);
        const uint32_t addr = res_s + (D == 128 ? swz(ld_row, chunk) : swz64(ld_row, chunk));
        uint32_t r[4];
        ldsm_x4(addr, r[0], r[1], r[2], r[3]);  // (row r0, kk 2g), (r0, 2g+1), (r1, 2g), (r1, 2g+1)
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const uint4 qg = qv[(Gm::NG + g) * 32];  // qr0, qr2 of k-steps 2g and 2g + 1
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            // fp16 0x64uu is 1024 + uu exactly; with uu = x + 128 the operand is 1152 + x and
            // the offset leaves the sum as 1152 * (sum of q over the group), removed below
            const uint32_t ua = r[e] ^ 0x80808080u, ub = r[e + 2] ^ 0x80808080u;
            mma_f16(acc, __byte_perm(ua, 0x64646464u, 0x4140), __byte_perm(ub, 0x64646464u, 0x4140),
                    __byte_perm(ua, 0x64646464u, 0x4342), __byte_perm(ub, 0x64646464u, 0x4342), e ? qg.z : qg.x,
                    e ? qg.w : qg.y);
        }
        const float4 of4 = *reinterpret_cast<const float4*>(&qv[(2 * Gm::NG + Gm::NG / 2 + g / 2) * 32]);
        const float2 off = (g & 1) ? make_float2(of4.z, of4.w) : make_float2(of4.x, of4.y);
        const float2 fa = __half22float2(ra[g >> 1]), fb = __half22float2(rb[g >> 1]);
        const float rsa = (g & 1) ? fa.y : fa.x, rsb = (g & 1) ? fb.y : fb.x;
        v0 = __ffma2_rn(make_float2(rsa, rsa), make_float2(acc[0] - off.x, acc[1] - off.y), v0);
        v1 = __ffma2_rn(make_float2(rsb, rsb), make_float2(acc[2] - off.x, acc[3] - off.y), v1);
    }
    rt[0] = v0.x;
    rt[1] = v0.y;
    rt[2] = v1.x;
    rt[3] = v1.y;
}

template <int D>
__global__ void __launch_bounds__(NW * 32, 2)
topdelta_kernel(const __grid_constant__ CUtensorMap tm_res, const __grid_constant__ CUtensorMap tm_v,
                const TDParams p) {
    using Gm = TGeo<D>;
    using Ly = TLayout<D>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
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
    pdl_wait_primary();  // the previous kernel in the stream may still be running
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
    const int head_row0 = (b * p.Hkv + h) * p.L_max;

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

    auto rows_of = [&](int t) { return min(kTile, t1 - (t0 + t * kTile)); };
    auto copy_rows = [&](int t) { return (rows_of(t) + 3) & ~3; };  // L_max % 4 == 0 keeps this in bounds
    if (warp == CW + 1) {
        // --------------------------- scan producer ------------------------------
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            int k = 0;
            for (; k < ntiles; ++k) {
                const int s = k % SS;
                if (!mbar_wait(&scan_empty[s], ((uint32_t)(k / SS) & 1u) ^ 1u)) {
                    atomicOr(&g_status_topdelta, kStatusTimeout);
                    break;
                }
                const size_t row0 = (size_t)head_row0 + t0 + (size_t)k * kTile;
                const uint32_t rc = (uint32_t)copy_rows(k);
                unsigned char* dst = smem + Ly::SCAN_OFF + s * Gm::SCAN_STAGE;
                scan_rows[s] = rows_of(k);
                mbar_arrive_expect_tx(&scan_full[s], rc * (Gm::CODES_ROW + Gm::MS_ROW));
                bulk_g2s(dst, p.codes + row0 * Gm::CODES_ROW, rc * Gm::CODES_ROW, &scan_full[s], pol);
                bulk_g2s(dst + kTile * Gm::CODES_ROW, p.mn_scale + row0 * Gm::MS_ROW, rc * Gm::MS_ROW, &scan_full[s],
                         pol);
            }
            // the consumers may stop early (a time-out): let every copy started
            // land before the CTA can exit (the last tile of each stage)
            for (int u = k - 1; u >= 0 && u >= k - SS; --u) mbar_wait(&scan_full[u % SS], (uint32_t)(u / SS) & 1u);
        }
        pdl_launch_dependents();
        return;
    }
    if (warp == CW) {
        // -------------------------- detail producer -----------------------------
        if (lane == 0) {
            prefetch_tmap(&tm_res);
            prefetch_tmap(&tm_v);
            const uint64_t pol = l2_evict_first_policy();
            bool ok = true;
            int t = 0;
            for (; t < ntiles; ++t) {
                const int s = t % DS;
                const uint32_t ph = (uint32_t)(t / DS) & 1u;
                if (!mbar_wait(&decided[s], ph) || !mbar_wait(&det_empty[s], ph ^ 1u)) {
                    ok = false;
                    break;
                }
                int any = 0;
                for (int w = 0; w < CW; ++w) any |= need[s * CW + w];
                if (any) {
                    const int y = head_row0 + t0 + t * kTile;
                    const uint32_t rc = (uint32_t)copy_rows(t);
                    unsigned char* dst = smem + Ly::DET_OFF + s * Gm::DET_STAGE;
                    loaded[s] = 1;
                    mbar_arrive_expect_tx(&det_full[s], Gm::RES_BYTES + Gm::V_BYTES + rc * Gm::RS_ROW);
                    if (D == 128) tma_load_box(dst, &tm_res, 0, y, &det_full[s], pol);
                    else tma_load_box64(dst, &tm_res, y, &det_full[s], pol);
#pragma unroll
                    for (int bx = 0; bx < D / 64; ++bx)
                        tma_load_box(dst + Gm::RES_BYTES + bx * kBoxBytes, &tm_v, 64 * bx, y, &det_full[s], pol);
                    bulk_g2s(dst + Gm::RES_BYTES + Gm::V_BYTES, p.res_scale + (size_t)y * Gm::RS_ROW,
                             rc * Gm::RS_ROW, &det_full[s], pol);
                } else {
                    loaded[s] = 0;
                    mbar_arrive(&det_full[s]);
                }
            }
            if (!ok) atomicOr(&g_status_topdelta, kStatusTimeout);
            for (int u = t - 1; u >= 0 && u >= t - DS; --u) mbar_wait(&det_full[u % DS], (uint32_t)(u / DS) & 1u);
        }
        pdl_launch_dependents();
        return;
    }

    // ------------------------------- consumers -----------------------------------
    const int gid = lane >> 2, tig = lane & 3;
    const bool q_real = gid < p.G;                                // the lane's B-fragment query
    const bool c_real[2] = {2 * tig < p.G, 2 * tig + 1 < p.G};    // its accumulator columns' queries
    // the query fragments of every consumer warp are the same: one copy in
    // shared memory, [vector][lane], read where they are used (the registers
    // they would hold are worth more to the dot stages)
    const uint4* qv = reinterpret_cast<const uint4*>(smem + Ly::Q_OFF) + lane;
    float2 scan_scale;
    TokAcc<D> ac;
    {
        TDQuery<D> tq;
        const uint16_t* qrow = p.q + (size_t)(b * p.Hq + hq0 + gid) * D;
        auto qf = [&](int c) { return q_real ? __uint_as_float((uint32_t)qrow[c] << 16) : 0.f; };
        // sq: max |q| * 2^sq in [1, 2) over the query's channels (a quad shares a query)
        float amax = 0.f;
        for (int c = tig; c < D; c += 4) amax = fmaxf(amax, fabsf(qf(c)));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        int ex = 0;  // amax = m * 2^ex, m in [0.5, 1)
        if (amax > 0.f && amax <= 3.4e38f) (void)frexpf(amax, &ex);
        const int sq = 1 - ex;
        auto qs = [&](int c) { return ldexpf(qf(c), sq + 126); };  // exact: |q| 2^(sq+126) < 2^127
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const int c0 = 16 * kk;
            tq.qc0[kk] = pack_bf16(qs(c0 + 2 * tig), qs(c0 + 2 * tig + 8));                  // exact
            tq.qc2[kk] = pack_bf16(0.25f * qs(c0 + 2 * tig + 1), 0.25f * qs(c0 + 2 * tig + 9));  // exact
            tq.qr0[kk] = pack_f16(qf(c0 + 4 * tig), qf(c0 + 4 * tig + 1));
            tq.qr2[kk] = pack_f16(qf(c0 + 4 * tig + 2), qf(c0 + 4 * tig + 3));
        }
        // per-query constants of query gid, then moved to the lanes whose
        // accumulator columns hold that query (lane 4q holds query q)
#pragma unroll
        for (int g = 0; g < D / 32; ++g) {
            float sum = 0.f, sumh = 0.f;
            for (int c = 0; c < 32; ++c) {
                sum = __fadd_rn(sum, qf(32 * g + c));
                sumh += __half2float(__float2half_rn(qf(32 * g + c)));
            }
            const float qsum = ldexpf(sum, sq - 7);  // exact
            const float off = 1152.f * sumh;
            tq.qsum[g] = make_float2(__shfl_sync(0xffffffffu, qsum, 8 * tig), __shfl_sync(0xffffffffu, qsum, 8 * tig + 4));
            tq.off[g] = make_float2(__shfl_sync(0xffffffffu, off, 8 * tig), __shfl_sync(0xffffffffu, off, 8 * tig + 4));
        }
        const float ssc = ldexpf(p.scale, 7 - sq);
        scan_scale = make_float2(__shfl_sync(0xffffffffu, ssc, 8 * tig), __shfl_sync(0xffffffffu, ssc, 8 * tig + 4));
        if (warp == 0) {
            // vectors: [g] scan qc0/qc2 of k-steps 2g, 2g+1; [NG + g] residual qr0/qr2 of
            // the same; [2 NG + i] qsum of groups 2i, 2i+1; [2 NG + NG/2 + i] off of the same
            uint4* qw = reinterpret_cast<uint4*>(smem + Ly::Q_OFF) + lane;
#pragma unroll
            for (int g = 0; g < Gm::NG; ++g) {
                qw[g * 32] = make_uint4(tq.qc0[2 * g], tq.qc2[2 * g], tq.qc0[2 * g + 1], tq.qc2[2 * g + 1]);
                qw[(Gm::NG + g) * 32] = make_uint4(tq.qr0[2 * g], tq.qr2[2 * g], tq.qr0[2 * g + 1], tq.qr2[2 * g + 1]);
            }
#pragma unroll
            for (int i = 0; i < Gm::NG / 2; ++i) {
                *reinterpret_cast<float4*>(&qw[(2 * Gm::NG + i) * 32]) =
                    make_float4(tq.qsum[2 * i].x, tq.qsum[2 * i].y, tq.qsum[2 * i + 1].x, tq.qsum[2 * i + 1].y);
                *reinterpret_cast<float4*>(&qw[(2 * Gm::NG + Gm::NG / 2 + i) * 32]) =
                    make_float4(tq.off[2 * i].x, tq.off[2 * i].y, tq.off[2 * i + 1].x, tq.off[2 * i + 1].y);
            }
        }
        named_barrier(1, CW * 32);  // the query vectors are in place
        tok_acc_init(ac);
    }

    // ---------------- anchor pass: pseudo-max per query head --------------------
    // Anchor tiles are staged in the first detail stage (untouched until the
    // first tile is flagged) in the scan ring's layout and scored by the same
    // code, so m^ equals the scan's s~ of the best anchor bit for bit.
    float mh[2] = {-INFINITY, -INFINITY};  // queries 2 tig, 2 tig + 1
    {
        unsigned char* stage = smem + Ly::DET_OFF;
        const int sink_end = min(p.n_sink, L);
        const int win_beg = max(0, L - p.window);
        const int ts_end = (sink_end + kTile - 1) / kTile;
        const int tw_beg = win_beg < L ? win_beg / kTile : (L + kTile - 1) / kTile;
        const int tw_end = (L + kTile - 1) / kTile;
        const int tid = warp * 32 + lane;
        // the anchor tiles: [0, ts_end) and [tw_lo, tw_end), each once, staged
        // NBA at a time (one round of loads for all of them on common settings)
        const int tw_lo = max(ts_end, tw_beg);
        const int na = ts_end + max(0, tw_end - tw_lo);
        auto anchor_tile = [&](int i) { return i < ts_end ? i : tw_lo + (i - ts_end); };
        constexpr int NBA = Gm::DET_STAGE / Gm::SCAN_STAGE;
        constexpr int CV = kTile * Gm::CODES_ROW / 16, MV = kTile * Gm::MS_ROW / 16;
        for (int a0 = 0; a0 < na; a0 += NBA) {
            const int nb = min(NBA, na - a0);
            named_barrier(1, CW * 32);  // the staging area is free
            for (int i = tid; i < nb * (CV + MV); i += CW * 32) {
                const int j = i / (CV + MV), e = i % (CV + MV);
                const int tb = anchor_tile(a0 + j) * kTile;
                const int rows = min(kTile, L - tb);
                unsigned char* sj = stage + j * Gm::SCAN_STAGE;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (e < CV) {
                    const int r = e * 16 / Gm::CODES_ROW;  // first row this 16-byte vector covers
                    if (r < rows) v = reinterpret_cast<const uint4*>(p.codes + (size_t)(head_row0 + tb) * Gm::CODES_ROW)[e];
                    reinterpret_cast<uint4*>(sj)[e] = v;
                } else {
                    const int k = e - CV;
                    const int r = k * 16 / Gm::MS_ROW;  // first row this 16-byte vector covers
                    if (r < rows) v = reinterpret_cast<const uint4*>(p.mn_scale + (size_t)(head_row0 + tb) * Gm::MS_ROW)[k];
                    reinterpret_cast<uint4*>(sj + kTile * Gm::CODES_ROW)[k] = v;
                }
            }
            named_barrier(1, CW * 32);
            for (int j = 0; j < nb; ++j) {
                const int tb = anchor_tile(a0 + j) * kTile;
                const int rows = min(kTile, L - tb);
                const unsigned char* sj = stage + j * Gm::SCAN_STAGE;
                float st[4];
                scan_tile<D>(sj, sj + kTile * Gm::CODES_ROW, warp, lane, qv, scan_scale, st);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = warp * 16 + gid + 8 * (i >> 1);
                    const int jt = tb + r;
                    if (r < rows && (jt < sink_end || jt >= win_beg)) mh[i & 1] = fmaxf(mh[i & 1], st[i]);
                }
            }
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            mh[0] = fmaxf(mh[0], __shfl_xor_sync(0xffffffffu, mh[0], o));
            mh[1] = fmaxf(mh[1], __shfl_xor_sync(0xffffffffu, mh[1], o));
        }
        if (gid == 0) {
            mh_red[warp * 8 + 2 * tig] = mh[0];
            mh_red[warp * 8 + 2 * tig + 1] = mh[1];
        }
        // staging stores must be ordered before the tile copies that reuse the area
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        named_barrier(1, CW * 32);
#pragma unroll
        for (int w = 0; w < CW; ++w) {
            mh[0] = fmaxf(mh[0], mh_red[w * 8 + 2 * tig]);
            mh[1] = fmaxf(mh[1], mh_red[w * 8 + 2 * tig + 1]);
        }
    }
    // delta = inf keeps every key
    const float thr[2] = {__fsub_rn(mh[0], p.delta), __fsub_rn(mh[1], p.delta)};
    int cnt[2] = {0, 0};
    bool failed = false;

    auto scan_step = [&](int k) {
        const int s = k % SS;
        if (!warp_wait(&scan_full[s], (uint32_t)(k / SS) & 1u)) {
            failed = true;
            return;
        }
        const int rows = scan_rows[s];
        const unsigned char* base = smem + Ly::SCAN_OFF + s * Gm::SCAN_STAGE;
        float st[4];
        scan_tile<D>(base, base + kTile * Gm::CODES_ROW, warp, lane, qv, scan_scale, st);
        const int ds = k % DS;
        reinterpret_cast<float4*>(dec_s)[(ds * CW + warp) * 32 + lane] = make_float4(st[0], st[1], st[2], st[3]);
        bool any = false;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = warp * 16 + gid + 8 * (i >> 1);
            any |= c_real[i & 1] && r < rows && st[i] >= thr[i & 1];
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
            unsigned char* st_base = smem + Ly::DET_OFF + ds * Gm::DET_STAGE;
            float rt[4];
            residual_tile<D>(smem_u32(st_base), st_base + Gm::RES_BYTES + Gm::V_BYTES, warp, lane, qv, rt);
            const float4 sv = reinterpret_cast<const float4*>(dec_s)[(ds * CW + warp) * 32 + lane];
            const float stv[4] = {sv.x, sv.y, sv.z, sv.w};
            bool selv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = warp * 16 + gid + 8 * (i >> 1);
                selv[i] = c_real[i & 1] && r < rows && stv[i] >= thr[i & 1];
            }
            if (p.group_union) {
                // a token some head of the group selected is attended by every head
                // (the lanes of a quad hold the 8 query columns of the same two rows)
                uint32_t any = (selv[0] || selv[1] ? 1u : 0u) | (selv[2] || selv[3] ? 2u : 0u);
                any |= __shfl_xor_sync(0xffffffffu, any, 1);
                any |= __shfl_xor_sync(0xffffffffu, any, 2);
#pragma unroll
                for (int i = 0; i < 4; ++i) selv[i] = c_real[i & 1] && ((any >> (i >> 1)) & 1u);
            }
            float sc[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = warp * 16 + gid + 8 * (i >> 1);
                const bool sel = selv[i];
                sc[i] = sel ? fmaf(p.scale, rt[i], stv[i]) * kLog2e : -INFINITY;
                if (sel) {
                    ++cnt[i & 1];
                    if (p.sel_mask) {
                        const int j = tok0 + r;
                        const int words = (p.L_max + 31) / 32;
                        const int qh = hq0 + 2 * tig + (i & 1);
                        atomicOr(&p.sel_mask[(size_t)(b * p.Hq + qh) * words + j / 32], 1u << (j % 32));
                    }
                }
            }
            mma_softmax_pv<D>(ac, sc, smem_u32(st_base + Gm::RES_BYTES), st_base + Gm::RES_BYTES, warp, lane, rows);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&det_empty[ds]);
    }
    if (failed) atomicOr(&g_status_topdelta, kStatusTimeout);
    pdl_launch_dependents();

    // per column: selected counts over the 16 rows (lanes of equal tig)
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        cnt[0] += __shfl_xor_sync(0xffffffffu, cnt[0], o);
        cnt[1] += __shfl_xor_sync(0xffffffffu, cnt[1], o);
    }
    if (p.sel_count && gid == 0) {
        if (c_real[0] && cnt[0]) atomicAdd(&p.sel_count[b * p.Hq + hq0 + 2 * tig], cnt[0]);
        if (c_real[1] && cnt[1]) atomicAdd(&p.sel_count[b * p.Hq + hq0 + 2 * tig + 1], cnt[1]);
    }
    combine_tok_warps_and_store<D, CW>(smem, warp, lane, p.G, b * p.Hq + hq0, split, ac, failed, p.st);
}

template <int D>
struct TDLauncher {
    static constexpr int SMEM = TLayout<D>::BYTES;
    static cudaError_t prepare() {
        static bool done[kMaxDevices] = {};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < kMaxDevices && done[dev]) return cudaSuccess;
        e = cudaFuncSetAttribute(topdelta_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
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
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, topdelta_kernel<D>, NW * 32, SMEM) !=
                cudaSuccess ||
            n <= 0)
            return 1;
        if (dev < kMaxDevices) cache[dev] = n;
        return n;
    }
    static cudaError_t launch(const CUtensorMap& tr, const CUtensorMap& tv, const TDParams& pp, dim3 grid,
                              cudaStream_t st) {
        cudaError_t e = prepare();
        if (e != cudaSuccess) return e;
        return launch_pdl(topdelta_kernel<D>, grid, dim3(NW * 32), SMEM, st, tr, tv, pp);
    }
};

}  // namespace

int topdelta_ctas_per_sm(int D, int) { return D == 128 ? TDLauncher<128>::ctas_per_sm() : TDLauncher<64>::ctas_per_sm(); }

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
    const uint64_t rows = (uint64_t)a.B * a.Hkv * a.L_max;
    CUtensorMap tr, tv;
    if (!make_row_map(&tr, a.res, rows, (uint32_t)a.D) || !make_row_map(&tv, a.v, rows, (uint32_t)a.D * 2))
        return cudaErrorInvalidValue;
    TDParams pp;
    pp.q = static_cast<const uint16_t*>(a.q);
    pp.codes = a.codes;
    pp.mn_scale = static_cast<const uint8_t*>(a.mn_scale);
    pp.res_scale = static_cast<const uint8_t*>(a.res_scale);
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
    pp.group_union = a.group_union;
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
    e = a.D == 128 ? TDLauncher<128>::launch(tr, tv, pp, grid, stream) : TDLauncher<64>::launch(tr, tv, pp, grid, stream);
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
