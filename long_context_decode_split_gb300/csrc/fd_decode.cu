// fd_decode.cu -- split-KV decode attention ("Flash Decoding" tutorial,
// sections 1-3) for sm_103a: the per-chunk partial pass over a contiguous or
// paged bf16 KV cache, and the exact log-sum-exp merge of the chunks.
//
// Partial pass, one CTA per (chunk, KV head, sequence):
//   * warp CW (the producer) streams the chunk's K and V through a STAGES-deep
//     ring of 64-token shared-memory tiles with bulk asynchronous copies
//     (cp.async.bulk + mbarrier transaction counts).  A tile is one contiguous
//     64-row slab in both layouts: a slice of [L, d] rows, or one cache page.
//   * warps 0..CW-1 (the consumers) each own 64/CW rows of every tile and
//     keep, for every query head of the GQA group, a running max m, exp-sum l
//     and output accumulator o in registers (online softmax in base 2).  So
//     every K/V byte is read from HBM once per KV head, whatever the group
//     size.  For one query head (MHA) the dot products run on packed fp32x2
//     FMAs and per-row partial sums are combined by a transposing butterfly
//     (one shuffle per token); for a group of 2..8 they run on mma.sync as
//     S = K Q^T (the warp's 16 tokens as M, the group as N) and O^T += V^T P^T
//     with P^T formed by movmatrix.
//   * at the end the consumer warps combine their states through shared
//     memory and write either the final output (one chunk) or the chunk's
//     (m_i, l_i, O_i / l_i) to the workspace.
// Merge, one CTA per (sequence, query head): m = max_i m_i,
//   w_i = 2^(m_i - m) l_i, out = sum_i w_i O_i / sum_i w_i, lse = m + log sum w.
// Both kernels are launched with programmatic dependent launch: the merge's
// launch overlaps the tail of the partial pass, and the next call's partial
// pass is scheduled while this call's merge runs (each waits on the grid
// dependency before its first global memory access).
#include <atomic>
#include <cmath>
#include <cstdio>

#include "fd_device.cuh"
#include "fd_internal.h"
#include "fd_tma.h"

namespace fd {

__device__ unsigned int g_status_decode;

namespace {

constexpr int kMaxDevices = 64;

// Static geometry of the partial pass for head dim D, padded group GP and CW
// consumer warps.
template <int D, int GP, int CW>
struct Geo {
    static constexpr int LPR = D / 8;           // lanes per K/V row (16 B each)
    static constexpr int RPI = 32 / LPR;        // rows per warp-wide load
    static constexpr int TPW = kTile / CW;      // rows of a tile owned by one warp
    static constexpr int NIT = TPW / RPI;       // loads per warp per tile
    static constexpr int LOG_LPR = D == 128 ? 4 : 3;
    static constexpr int LOG_NIT = NIT == 16 ? 4 : NIT == 8 ? 3 : NIT == 4 ? 2 : NIT == 2 ? 1 : 0;
    static constexpr int SH = LOG_LPR - LOG_NIT;  // low lane bits that hold copies
    static_assert(NIT >= 1 && NIT <= LPR, "bad warp split");
    static_assert((1 << LOG_NIT) == NIT, "NIT must be a power of two");
};

struct PartialParams {
    const uint16_t* q;
    const int32_t* seq_lens;
    const int32_t* page_table;
    int max_pages, num_pages;
    int Hq, Hkv, L_max, G;
    float scale_log2;
    int splits, chunk_fixed;
    float phi2, lo2;  // unified-max variant: phi and phi - kUnifiedRange, log2 units
    unsigned long long wait_limit_ns;  // time limit of every pipeline wait
    int withhold_tile;                 // >= 0: fault injection, that tile of each chunk is never copied
    StoreTarget st;
};

// Fault injection for the tests of the time-out path (fd_debug_inject_wait_timeout).
std::atomic<unsigned long long> g_inject_wait_limit_ns{0};
std::atomic<int> g_inject_withhold_tile{-1};

// Unified-max variant (FlashDecoding++ summary, sections 1, 3 and 5: one
// fixed max value phi for every chunk, so no chunk reduces its scores to a
// max; a fallback to the running-max computation when the scores leave the
// range in which that is exact).  A warp stays on the fixed reference while
// every score it attends lies in [phi - R, phi] (R = kUnifiedRange nats):
// then each weight 2^(s - phi) is a normal binary32 number in [e^-R, 1] and
// no sum can overflow.  At the first tile with a score outside that range it
// rebases its O and l from phi to the largest score it has attended so far
// (the exact state the running-max computation would hold) and continues on
// the running-max path.  Every result is the one the plain path computes, up
// to fp32 rounding.
constexpr float kUnifiedRange = 60.f;

// Tensor-core consumer, one warp, 16 rows of a 64-token tile: S = K Q^T on
// mma.sync (A = the warp's K rows by ldmatrix from the swizzled tile, B = Q
// fragments in registers; accumulator rows gid, gid + 8 are tokens, columns
// 2 tig, 2 tig + 1 query heads), then the shared online-softmax / P.V step.
template <int D>
__device__ __forceinline__ void mma_consume_tile(TokAcc<D>& ac, const uint32_t (&qa0)[D / 16],
                                                 const uint32_t (&qa2)[D / 16], uint32_t ks, uint32_t vs,
                                                 unsigned char* vgen, int warp, int lane, int rows, float scale_log2) {
    const int gid = lane >> 2;
    const int mi = lane >> 3;
    const int a_row = warp * 16 + 8 * (mi & 1) + (lane & 7);  // K row this lane addresses (A fragment)
    float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(ks + swz(a_row, 2 * kk + (mi >> 1)), a0, a1, a2, a3);
        mma_bf16(sacc, a0, a1, a2, a3, qa0[kk], qa2[kk]);
    }
    const int r0 = warp * 16 + gid;
    float sc[4];
    sc[0] = r0 < rows ? sacc[0] * scale_log2 : -INFINITY;
    sc[1] = r0 < rows ? sacc[1] * scale_log2 : -INFINITY;
    sc[2] = r0 + 8 < rows ? sacc[2] * scale_log2 : -INFINITY;
    sc[3] = r0 + 8 < rows ? sacc[3] * scale_log2 : -INFINITY;
    mma_softmax_pv<D>(ac, sc, vs, vgen, warp, lane, rows);
}

// The same tile step through the unified-max variant.
template <int D>
__device__ __forceinline__ void mma_consume_tile_unified(TokAcc<D>& ac, bool& unified, float2& seen,
                                                         const uint32_t (&qa0)[D / 16], const uint32_t (&qa2)[D / 16],
                                                         uint32_t ks, uint32_t vs, unsigned char* vgen, int warp,
                                                         int lane, int rows, float scale_log2, float phi2, float lo2) {
    const int gid = lane >> 2;
    const int mi = lane >> 3;
    const int a_row = warp * 16 + 8 * (mi & 1) + (lane & 7);
    float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(ks + swz(a_row, 2 * kk + (mi >> 1)), a0, a1, a2, a3);
        mma_bf16(sacc, a0, a1, a2, a3, qa0[kk], qa2[kk]);
    }
    const int r0 = warp * 16 + gid;
    float sc[4];
    sc[0] = r0 < rows ? sacc[0] * scale_log2 : -INFINITY;
    sc[1] = r0 < rows ? sacc[1] * scale_log2 : -INFINITY;
    sc[2] = r0 + 8 < rows ? sacc[2] * scale_log2 : -INFINITY;
    sc[3] = r0 + 8 < rows ? sacc[3] * scale_log2 : -INFINITY;
    fixed_ref_softmax_pv<D>(ac, unified, seen, sc, vs, vgen, warp, lane, rows, make_float2(phi2, phi2),
                            make_float2(lo2, lo2));
}

template <int D, int GP, int CW, int STAGES, bool PAGED, bool MMA, bool UMAX>
__global__ void __launch_bounds__((CW + 1) * 32, (MMA || GP < 8) ? 2 : 1)
partial_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
               const PartialParams p) {
    using Gm = Geo<D, GP, CW>;
    constexpr int BOXES = D / 64;                // boxes per K (or V) tile
    constexpr int STAGE = 2 * BOXES * kBoxBytes;  // K tile + V tile
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE);
    uint64_t* empty = full + STAGES;
    int* stage_rows = reinterpret_cast<int*>(empty + STAGES);

    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait_primary();  // the previous kernel in the stream may still be running
    const int L = clamped_len(p.seq_lens, b, p.L_max, &g_status_decode);
    const int chunk = chunk_len(L, p.splits, p.chunk_fixed);
    const int t0 = split * chunk;
    const int t1 = min(L, t0 + chunk);
    const int hq0 = h * p.G;

    if (t0 >= t1) {
        pdl_launch_dependents();
        // An empty chunk writes nothing, except that the only chunk of an
        // empty sequence writes out = 0, lse = -inf.
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
            const uint64_t pol = l2_evict_first_policy();
            const int head_row0 = PAGED ? 0 : (b * p.Hkv + h) * p.L_max;
            int t = 0;
            for (; t < ntiles; ++t) {
                const int s = t % STAGES;
                const uint32_t ph = (uint32_t)(t / STAGES) & 1u;
                if (!mbar_wait(&empty[s], ph ^ 1u, p.wait_limit_ns)) {
                    atomicOr(&g_status_decode, kStatusTimeout);
                    break;
                }
                if (t == p.withhold_tile) continue;  // fault injection: no copy, no arrival
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
                if (ok) {
                    stage_rows[s] = rows;
                    mbar_arrive_expect_tx(&full[s], STAGE);
#pragma unroll
                    for (int bx = 0; bx < BOXES; ++bx) {
                        tma_load_box(sk + bx * kBoxBytes, &tmk, 64 * bx, y, &full[s], pol);
                        tma_load_box(sk + (BOXES + bx) * kBoxBytes, &tmv, 64 * bx, y, &full[s], pol);
                    }
                } else {
                    atomicOr(&g_status_decode, kStatusBadPage);
                    stage_rows[s] = 0;
                    mbar_arrive(&full[s]);
                }
            }
            if (t < ntiles || p.withhold_tile >= 0) {
                // the consumers may have stopped early: before the CTA exits, let
                // every copy this loop started land (the last tile of each stage)
                for (int u = t - 1; u >= 0 && u >= t - STAGES; --u) {
                    if (u == p.withhold_tile) continue;
                    mbar_wait(&full[u % STAGES], (uint32_t)(u / STAGES) & 1u, p.wait_limit_ns);
                }
            }
        }
        pdl_launch_dependents();
        return;
    }

    bool failed = false;
    if constexpr (MMA) {
        // ------------------- tensor-core consumers (groups of 2..8) --------
        const int gid = lane >> 2, tig = lane & 3;
        uint32_t qa0[D / 16], qa2[D / 16];  // B fragments of query gid
        TokAcc<D> ac;
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(p.q + (size_t)(b * p.Hq + hq0 + gid) * D);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            qa0[kk] = gid < p.G ? qrow[8 * kk + tig] : 0u;
            qa2[kk] = gid < p.G ? qrow[8 * kk + 4 + tig] : 0u;
        }
        tok_acc_init(ac);
        bool unified = UMAX;
        float2 seen = make_float2(-INFINITY, -INFINITY);
        for (int t = 0; t < ntiles; ++t) {
            const int s = t % STAGES;
            if (!warp_wait(&full[s], (uint32_t)(t / STAGES) & 1u, p.wait_limit_ns)) {
                atomicOr(&g_status_decode, kStatusTimeout);
                failed = true;
                break;
            }
            const int rows = stage_rows[s];
            unsigned char* sk = smem + s * STAGE;
            if constexpr (UMAX)
                mma_consume_tile_unified<D>(ac, unified, seen, qa0, qa2, smem_u32(sk), smem_u32(sk + BOXES * kBoxBytes),
                                            sk + BOXES * kBoxBytes, warp, lane, rows, p.scale_log2, p.phi2, p.lo2);
            else
                mma_consume_tile<D>(ac, qa0, qa2, smem_u32(sk), smem_u32(sk + BOXES * kBoxBytes),
                                    sk + BOXES * kBoxBytes, warp, lane, rows, p.scale_log2);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        if (UMAX && unified) fixed_ref_finish(ac, seen, make_float2(p.phi2, p.phi2));
        pdl_launch_dependents();
        combine_tok_warps_and_store<D, CW>(smem, warp, lane, p.G, b * p.Hq + hq0, split, ac, failed, p.st);
        return;
    } else {
    // ------------------------ CUDA-core consumers --------------------------
    const int c = lane % Gm::LPR;   // 16-byte column of a row
    const int rg = lane / Gm::LPR;  // row group within a warp-wide load
    // my token slot after the transposing reduction
    const int my_i = (lane >> Gm::SH) & (Gm::NIT - 1);
    const int my_row = warp * Gm::TPW + Gm::RPI * my_i + rg;
    const bool my_dup = (lane & ((1 << Gm::SH) - 1)) != 0;

    float2 qv[GP][4];
#pragma unroll
    for (int g = 0; g < GP; ++g) {
        if (g < p.G) {
            const uint4 w = *reinterpret_cast<const uint4*>(p.q + (size_t)(b * p.Hq + hq0 + g) * D + c * 8);
            qv[g][0] = bf16x2_to_float2(w.x);
            qv[g][1] = bf16x2_to_float2(w.y);
            qv[g][2] = bf16x2_to_float2(w.z);
            qv[g][3] = bf16x2_to_float2(w.w);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) qv[g][e] = make_float2(0.f, 0.f);
        }
    }

    float m_run[GP], l_lane[GP], seen[GP];
    float2 o[GP][4];
#pragma unroll
    for (int g = 0; g < GP; ++g) {
        m_run[g] = -INFINITY;
        l_lane[g] = 0.f;
        seen[g] = -INFINITY;
#pragma unroll
        for (int e = 0; e < 4; ++e) o[g][e] = make_float2(0.f, 0.f);
    }
    bool unified = UMAX;  // on the fixed reference phi (see kUnifiedRange)

    for (int t = 0; t < ntiles; ++t) {
        const int s = t % STAGES;
        const uint32_t ph = (uint32_t)(t / STAGES) & 1u;
        if (!warp_wait(&full[s], ph, p.wait_limit_ns)) {
            atomicOr(&g_status_decode, kStatusTimeout);
            failed = true;
            break;
        }
        const int rows = stage_rows[s];
        const unsigned char* sk = smem + s * STAGE;
        const unsigned char* sv = sk + BOXES * kBoxBytes;

        // ---- scores: partial dots over my 8 dims, then butterfly -----------
        float part[GP][Gm::NIT];
#pragma unroll
        for (int i = 0; i < Gm::NIT; ++i) {
            const int row = warp * Gm::TPW + Gm::RPI * i + rg;
            const uint4 w = lds128(sk + swz(row, c));
            const float2 k0 = bf16x2_to_float2(w.x), k1 = bf16x2_to_float2(w.y);
            const float2 k2 = bf16x2_to_float2(w.z), k3 = bf16x2_to_float2(w.w);
#pragma unroll
            for (int g = 0; g < GP; ++g) {
                float2 acc = f2mul(qv[g][0], k0);
                acc = f2fma(qv[g][1], k1, acc);
                acc = f2fma(qv[g][2], k2, acc);
                acc = f2fma(qv[g][3], k3, acc);
                part[g][i] = acc.x + acc.y;
            }
        }
        float sc[GP];
        const bool my_valid = my_row < rows;
#pragma unroll
        for (int g = 0; g < GP; ++g) {
            const float sum = transpose_reduce<Gm::NIT, Gm::LPR>(part[g], lane);
            sc[g] = my_valid ? sum * p.scale_log2 : -INFINITY;
        }

        // ---- online softmax update -----------------------------------------
        float pr[GP];
        bool on_reference = false;
        if constexpr (UMAX) {
            if (unified) {
                bool ok = true;
#pragma unroll
                for (int g = 0; g < GP; ++g) ok &= sc[g] == -INFINITY || (sc[g] >= p.lo2 && sc[g] <= p.phi2);
                if (__all_sync(0xffffffffu, ok)) {
                    on_reference = true;  // weights 2^(s - phi), no max, no rescale
#pragma unroll
                    for (int g = 0; g < GP; ++g) {
                        pr[g] = exp2_approx(sc[g] - p.phi2);
                        seen[g] = fmaxf(seen[g], sc[g]);
                        l_lane[g] += my_dup ? 0.f : pr[g];
                    }
                } else {
                    // fallback: rebase O and l from phi to the largest attended score
                    unified = false;
#pragma unroll
                    for (int g = 0; g < GP; ++g) {
                        float m = seen[g];
#pragma unroll
                        for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
                        const float a = m == -INFINITY ? 1.f : exp2_approx(p.phi2 - m);
                        m_run[g] = m;
                        l_lane[g] *= a;
                        const float2 a2 = make_float2(a, a);
#pragma unroll
                        for (int e = 0; e < 4; ++e) o[g][e] = f2mul(o[g][e], a2);
                    }
                }
            }
        }
        if (!on_reference) {
#pragma unroll
        for (int g = 0; g < GP; ++g) {
            float mx = sc[g];
#pragma unroll
            for (int off = 16; off >= (1 << Gm::SH); off >>= 1)
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float m_new = fmaxf(m_run[g], mx);
            if (m_new == -INFINITY) {  // nothing valid yet (warp-uniform)
                pr[g] = 0.f;
                continue;
            }
            const float alpha = exp2_approx(m_run[g] - m_new);
            m_run[g] = m_new;
            pr[g] = exp2_approx(sc[g] - m_new);
            l_lane[g] = l_lane[g] * alpha + (my_dup ? 0.f : pr[g]);
            const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
            for (int e = 0; e < 4; ++e) o[g][e] = f2mul(o[g][e], a2);
        }
        }

        // ---- o += p * v over my rows --------------------------------------
#pragma unroll
        for (int i = 0; i < Gm::NIT; ++i) {
            const int row = warp * Gm::TPW + Gm::RPI * i + rg;
            const int src = rg * Gm::LPR + (i << Gm::SH);
            float pi[GP];
#pragma unroll
            for (int g = 0; g < GP; ++g) pi[g] = __shfl_sync(0xffffffffu, pr[g], src);
            if (row < rows) {
                const uint4 w = lds128(sv + swz(row, c));
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
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (UMAX && unified) {
        // still on the reference: the partial is relative to phi (none when
        // nothing was attended)
#pragma unroll
        for (int g = 0; g < GP; ++g) {
            float m = seen[g];
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
            m_run[g] = m == -INFINITY ? -INFINITY : p.phi2;
        }
    }
    pdl_launch_dependents();
    combine_warps_and_store<D, GP, CW>(smem, warp, lane, p.G, b * p.Hq + hq0, split, m_run, l_lane, o, failed,
                                       p.st);
    }
}

// ---------------------------------------------------------------------------
// Merge: one CTA of D threads per (sequence, query head).  Each thread (one
// output channel) starts the loads of its channel's first MB chunk outputs
// before anything else; meanwhile the chunks' (m, l) pairs are read one per
// thread, reduced to M by the whole CTA and turned into weights in shared
// memory.  The channel is then summed over the chunks in chunk order, MB
// loads in flight at a time, so a long list of chunks costs a few memory
// latencies, not one per chunk.  Sums run in chunk order: the result does
// not depend on D or MB.
template <int D>
__global__ void __launch_bounds__(D)
merge_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml,
             const int32_t* __restrict__ seq_lens, int Hq, int L_max, int splits, int chunk_fixed,
             void* __restrict__ out, int out_bf16, float* __restrict__ lse) {
    constexpr int NWARP = D / 32;
    constexpr int MB = 32;  // chunk outputs in flight per thread
    __shared__ float w_s[D];
    __shared__ float red[NWARP];
    pdl_wait_primary();
    pdl_launch_dependents();  // the next call's partial pass waits for this grid before reading
    const int row = blockIdx.x;
    const int b = row / Hq;
    const int dim = threadIdx.x, lane = dim & 31, warp = dim >> 5;
    const int L = clamped_len(seq_lens, b, L_max, nullptr);
    const int chunk = chunk_len(L, splits, chunk_fixed);
    const int n = L > 0 ? min(splits, (L + chunk - 1) / chunk) : 0;
    const float2* ml = reinterpret_cast<const float2*>(part_ml) + (size_t)row * splits;
    const float* po = part_o + (size_t)row * splits * D + dim;
    float v[MB];
#pragma unroll
    for (int u = 0; u < MB; ++u) v[u] = u < n ? po[(size_t)u * D] : 0.f;
    float M = -INFINITY;
    for (int i = dim; i < n; i += D) M = fmaxf(M, ml[i].x);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    if (lane == 0) red[warp] = M;
    __syncthreads();
    M = red[0];
#pragma unroll
    for (int w = 1; w < NWARP; ++w) M = fmaxf(M, red[w]);
    float wsum = 0.f, acc = 0.f;
    if (M != -INFINITY) {
        for (int base = 0; base < n; base += D) {
            const int i = base + dim;
            float w = 0.f;
            if (i < n) {
                const float2 mli = ml[i];
                if (mli.x != -INFINITY) w = exp2_approx(mli.x - M) * mli.y;
            }
            __syncthreads();  // the previous weights are consumed
            w_s[dim] = w;
            __syncthreads();
            const int cnt = min(D, n - base);
            for (int j = 0; j < cnt; j += MB) {
                if (base + j > 0) {  // the first MB outputs were loaded up front
#pragma unroll
                    for (int u = 0; u < MB; ++u) v[u] = j + u < cnt ? po[(size_t)(base + j + u) * D] : 0.f;
                }
#pragma unroll
                for (int u = 0; u < MB; ++u) {
                    const float wu = j + u < cnt ? w_s[j + u] : 0.f;
                    if (wu != 0.f) {
                        wsum += wu;
                        acc += wu * v[u];
                    }
                }
            }
        }
    }
    const float val = wsum > 0.f ? acc / wsum : 0.f;
    const size_t oi = (size_t)row * D + dim;
    if (out_bf16) static_cast<uint16_t*>(out)[oi] = f32_to_bf16_bits(val);
    else static_cast<float*>(out)[oi] = val;
    if (dim == 0 && lse) lse[row] = wsum > 0.f ? (M + __log2f(wsum)) * kLn2 : -INFINITY;
}

template <int D, int GP, bool PAGED, bool UMAX = false>
struct PartialLauncher {
    // groups of 2..8 run on the tensor cores; single queries on CUDA cores
    static constexpr bool MMA = GP >= 2;
    static constexpr int CW = 4;
    static constexpr int STAGES = D == 128 ? 3 : 4;
    static constexpr int STAGE = 2 * (D / 64) * kBoxBytes;
    static constexpr int SMEM = 1024 + STAGES * STAGE + STAGES * 16 + STAGES * 4 + 64;
    static constexpr int RED = CW * 8 * D * 4 + 2 * CW * 8 * 4;
    static_assert(STAGES * STAGE >= RED, "reduction scratch must fit in the ring");
    static constexpr auto kernel = partial_kernel<D, MMA ? 8 : GP, CW, STAGES, PAGED, MMA, UMAX>;

    // Per device: raise the dynamic shared-memory limit once, and remember
    // the occupancy the planner sizes its grids with.
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
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, (CW + 1) * 32, SMEM) != cudaSuccess || n <= 0)
            return 1;
        if (dev < kMaxDevices) cache[dev] = n;
        return n;
    }
    static cudaError_t launch(const CUtensorMap& tk, const CUtensorMap& tv, const PartialParams& pp, dim3 grid,
                              cudaStream_t st) {
        cudaError_t e = prepare();
        if (e != cudaSuccess) return e;
        return launch_pdl(kernel, grid, dim3((CW + 1) * 32), SMEM, st, tk, tv, pp);
    }
};

template <int D, bool PAGED>
int ctas_per_sm_dispatch(int G) {
    if (G <= 1) return PartialLauncher<D, 1, PAGED>::ctas_per_sm();
    return PartialLauncher<D, 8, PAGED>::ctas_per_sm();
}

template <int D, bool PAGED, bool UMAX>
cudaError_t launch_dispatch_v(int G, const CUtensorMap& tk, const CUtensorMap& tv, const PartialParams& pp,
                              dim3 grid, cudaStream_t st) {
    if (G <= 1) return PartialLauncher<D, 1, PAGED, UMAX>::launch(tk, tv, pp, grid, st);
    return PartialLauncher<D, 8, PAGED, UMAX>::launch(tk, tv, pp, grid, st);
}

template <int D, bool PAGED>
cudaError_t launch_dispatch(int G, bool unified, const CUtensorMap& tk, const CUtensorMap& tv,
                            const PartialParams& pp, dim3 grid, cudaStream_t st) {
    return unified ? launch_dispatch_v<D, PAGED, true>(G, tk, tv, pp, grid, st)
                   : launch_dispatch_v<D, PAGED, false>(G, tk, tv, pp, grid, st);
}

}  // namespace

size_t decode_workspace_bytes(int B, int Hq, int D, int splits) {
    if (splits <= 1) return 0;
    const size_t rows = (size_t)B * Hq * splits;
    return rows * D * sizeof(float) + rows * 2 * sizeof(float) + 256;
}

int decode_ctas_per_sm(int D, int G, bool paged) {
    if (D == 128) return paged ? ctas_per_sm_dispatch<128, true>(G) : ctas_per_sm_dispatch<128, false>(G);
    return paged ? ctas_per_sm_dispatch<64, true>(G) : ctas_per_sm_dispatch<64, false>(G);
}

cudaError_t launch_merge(const float* part_o, const float* part_ml, const int32_t* seq_lens,
                         int B, int Hq, int L_max, int D, int splits, int chunk_fixed,
                         void* out, int out_bf16, float* lse, cudaStream_t stream) {
    const dim3 grid((unsigned)(B * Hq)), block((unsigned)D);
    if (D == 128)
        return launch_pdl(merge_kernel<128>, grid, block, 0, stream, part_o, part_ml, seq_lens, Hq, L_max, splits,
                          chunk_fixed, out, out_bf16, lse);
    return launch_pdl(merge_kernel<64>, grid, block, 0, stream, part_o, part_ml, seq_lens, Hq, L_max, splits,
                      chunk_fixed, out, out_bf16, lse);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
    if (a.B == 0) return cudaSuccess;
    const bool paged = a.page_table != nullptr;
    const uint64_t rows = paged ? (uint64_t)a.num_pages * a.Hkv * kTile : (uint64_t)a.B * a.Hkv * a.L_max;
    CUtensorMap tk, tv;
    if (rows == 0) {
        // nothing can be read (an empty pool or cache): any well-formed map will do
        if (!make_row_map(&tk, a.q, 1, (uint32_t)a.D * 2) || !make_row_map(&tv, a.q, 1, (uint32_t)a.D * 2))
            return cudaErrorInvalidValue;
    } else if (!make_row_map(&tk, a.k, rows, (uint32_t)a.D * 2) || !make_row_map(&tv, a.v, rows, (uint32_t)a.D * 2)) {
        return cudaErrorInvalidValue;
    }
    PartialParams pp;
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
    pp.phi2 = a.phi * kLog2e;
    pp.lo2 = (a.phi - kUnifiedRange) * kLog2e;
    const unsigned long long lim = g_inject_wait_limit_ns.load(std::memory_order_relaxed);
    pp.wait_limit_ns = lim ? lim : kWaitLimitNs;
    pp.withhold_tile = g_inject_withhold_tile.load(std::memory_order_relaxed);
    pp.st.part_o = a.part_o;
    pp.st.part_ml = a.part_ml;
    pp.st.out = a.out;
    pp.st.out_bf16 = a.out_bf16;
    pp.st.lse = a.lse;
    pp.st.direct = a.splits == 1 ? 1 : 0;
    pp.st.splits = a.splits;
    const dim3 grid((unsigned)a.splits, (unsigned)a.Hkv, (unsigned)a.B);
    cudaError_t e;
    const bool u = a.unified != 0;
    if (a.D == 128) e = paged ? launch_dispatch<128, true>(pp.G, u, tk, tv, pp, grid, stream)
                              : launch_dispatch<128, false>(pp.G, u, tk, tv, pp, grid, stream);
    else e = paged ? launch_dispatch<64, true>(pp.G, u, tk, tv, pp, grid, stream)
                   : launch_dispatch<64, false>(pp.G, u, tk, tv, pp, grid, stream);
    if (e != cudaSuccess || a.splits == 1) return e;
    return launch_merge(a.part_o, a.part_ml, a.seq_lens, a.B, a.Hq, a.L_max, a.D, a.splits, a.chunk_fixed,
                        a.out, a.out_bf16, a.lse, stream);
}

void inject_wait_timeout(unsigned long long wait_limit_ns, int withhold_tile) {
    g_inject_wait_limit_ns.store(wait_limit_ns, std::memory_order_relaxed);
    g_inject_withhold_tile.store(withhold_tile < 0 ? -1 : withhold_tile, std::memory_order_relaxed);
}

cudaError_t decode_status_read(unsigned* bits, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(bits, g_status_decode, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_status_decode, &zero, sizeof(unsigned));
}

}  // namespace fd
