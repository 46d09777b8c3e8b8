// fd_device.cuh -- device-side building blocks shared by the libfd kernels:
// mbarrier pipeline primitives, bulk (TMA) global->shared copies, bounded
// waits, bf16 unpacking and the packed fp32x2 arithmetic of sm_100-family GPUs.
// Everything here is inline PTX or CUDA intrinsics for sm_103a.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace fd {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Device status bits (see fd_device_status in fd.h).
constexpr unsigned kStatusBadPage = 1u;
constexpr unsigned kStatusTimeout = 2u;
constexpr unsigned kStatusBadSeqLen = 4u;

// Sequence length as the kernels use it: seq_lens[b] clamped to [0, L_max]
// (an out-of-range entry is recorded in `status`).
__device__ __forceinline__ int clamped_len(const int32_t* seq_lens, int b, int L_max, unsigned* status) {
    if (!seq_lens) return L_max;
    const int L = seq_lens[b];
    if (L < 0 || L > L_max) {
        if (status && threadIdx.x == 0) atomicOr(status, kStatusBadSeqLen);
        return L < 0 ? 0 : L_max;
    }
    return L;
}

// A pipeline wait gives up after this long (nanoseconds of %globaltimer) or
// this many polls, whichever comes first; the kernel then records
// kStatusTimeout and finishes without touching the stage.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
constexpr unsigned kWaitLimitPolls = 1u << 26;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// bf16x2 word -> two fp32 (exact: bf16 is the top half of binary32).
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Makes initialised barriers visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete.  Returns false if
// the wait hit its limit (the caller records kStatusTimeout and stops):
// limit_ns of %globaltimer (checked every 16 polls) or kWaitLimitPolls polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          unsigned long long limit_ns = kWaitLimitNs) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    for (unsigned it = 1; it < kWaitLimitPolls; ++it) {
        if (mbar_try_wait(a, parity)) return true;
        if ((it & 15u) == 0u && global_timer_ns() - t0 > limit_ns) return false;
    }
    return false;
}

// mbar_wait for all 32 lanes of a warp, with one outcome for the whole warp
// (so a time-out can never split the warp before its shuffles).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity,
                                          unsigned long long limit_ns = kWaitLimitNs) {
    const bool ok = mbar_wait(bar, parity, limit_ns);
    return __all_sync(0xffffffffu, ok);
}

// L2 policy for data that is streamed exactly once.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Bulk asynchronous copy global -> shared (TMA, non-tensor form); completion
// is signalled on `bar` as transaction bytes.  dst, src 16-byte aligned;
// bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Tiled TMA load of one 64-row x 128-byte box (coordinates: x in 2-byte
// units along the row, y = row) into `dst` (1024-byte aligned, 128-byte
// swizzle as encoded in the tensor map).  Completion counts 8192 bytes on `bar`.
__device__ __forceinline__ void tma_load_box(void* dst, const void* tmap, int x, int y, uint64_t* bar,
                                             uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar)),
        "l"(policy)
        : "memory");
}

// Tiled TMA load of one box of a rank-1 tensor map starting at element x
// (x * element size a multiple of 16 bytes); dst 128-byte aligned.
__device__ __forceinline__ void tma_load_1d(void* dst, const void* tmap, int x, uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.1d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2}], [%3], %4;"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

constexpr int kBoxBytes = 64 * 128;  // one TMA box: 64 rows x 128 bytes

// Byte offset of 16-byte chunk `chunk` of row `row` in a tile stored as
// consecutive 64x128-byte boxes with the 128-byte swizzle (chunk c of a row
// lives in box c / 8 at position (c % 8) ^ (row % 8)).
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return (uint32_t)((chunk >> 3) * kBoxBytes + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

// The same for a box of 64-byte rows with the 64-byte swizzle (chunk c of
// row r at position c ^ ((r / 2) % 4)).
__device__ __forceinline__ uint32_t swz64(int row, int chunk) {
    return (uint32_t)(row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4));
}

// TMA load of one box of 64 rows x 64 bytes (64-byte swizzle): 4096 bytes.
__device__ __forceinline__ void tma_load_box64(void* dst, const void* tmap, int y, uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(0), "r"(y), "r"(smem_u32(bar)),
        "l"(policy)
        : "memory");
}

// ldmatrix: four 8x8 b16 matrices; lanes 8j..8j+7 give the row addresses of matrix j.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D += A * B for one m16n8k16 tile, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Same with fp16 inputs.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 matrix of 16-bit values held as in an MMA fragment
// (lane 4*gid + t holds row gid, columns 2t and 2t + 1; the lower column in
// the lower half): the result holds the transpose in the same layout.  This
// turns the P values of an S = K Q^T accumulator (rows = tokens) into the B
// fragment of P^T (k = tokens, n = query heads).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// Two fp32 -> packed bf16x2 (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two fp32 -> packed fp16x2 (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Probability pair p -> bf16 hi part and bf16 remainder (p ~= hi + lo with
// relative error ~2^-16), so the P.V product keeps fp32-level accuracy.
__device__ __forceinline__ void split_bf16(float p0, float p1, uint32_t& hi, uint32_t& lo) {
    hi = pack_bf16(p0, p1);
    const float2 h = bf16x2_to_float2(hi);
    lo = pack_bf16(p0 - h.x, p1 - h.y);
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue, and (in that kernel) wait for this grid's results.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Named barrier over a subset of warps (id 1..15; the count is in threads).
__device__ __forceinline__ void named_barrier(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// 16-byte shared-memory load.
__device__ __forceinline__ uint4 lds128(const void* p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_u32(p)));
    return v;
}


__device__ __forceinline__ float exp2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float2 f2mul(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 f2fma(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

__device__ __forceinline__ unsigned short f32_to_bf16_bits(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// Butterfly over the LPR lanes of a row group that both sums the per-lane
// partial dot products and transposes them: on entry lane l holds N partial
// sums (one per row it touched), on exit it holds the full sum of the row
// with index (l >> SH) & (N-1).
template <int N, int LPR>
__device__ __forceinline__ float transpose_reduce(float (&v)[N], int lane) {
#pragma unroll
    for (int n = N, o = LPR / 2; n > 1; n >>= 1, o >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int k = 0; k < n / 2; ++k) {
            const float send = upper ? v[k] : v[k + n / 2];
            const float keep = upper ? v[k + n / 2] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    float r = v[0];
#pragma unroll
    for (int o = LPR / N / 2; o >= 1; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    return r;
}


// Attend state of one tensor-core consumer warp in the S = K Q^T layout: the
// warp owns 16 token rows of every 64-token tile; lane (gid, tig) holds
// accumulator rows gid, gid + 8 (tokens) and columns 2 tig, 2 tig + 1 (query
// heads of the group, padded to 8).  O^T is D rows x 8 columns; m and l are
// the running max (log2 units) and the lane's share of the exp-sum of its two
// columns.
template <int D>
struct TokAcc {
    float o[D / 16][4];  // O^T: [column 2*tig + (i&1)][dim 16*mt + gid + 8*(i>>1)]
    float2 m, l;
};

template <int D>
__device__ __forceinline__ void tok_acc_init(TokAcc<D>& ac) {
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) ac.o[mt][i] = 0.f;
    ac.m = make_float2(-INFINITY, -INFINITY);
    ac.l = make_float2(0.f, 0.f);
}

// Online softmax over one tile and O^T += V^T P^T for scores in the S = K Q^T
// layout (sc[i]: row warp*16 + gid + 8*(i >> 1), column 2*tig + (i & 1), log2
// units; -inf = not attended).  V rows at or past `rows` are cleared first
// (they may hold anything; P is 0 there, but 0 * NaN is NaN).  P goes to the
// tensor cores as bf16 hi + lo (~2^-16 relative accuracy); movmatrix turns
// each 8x8 block of the lane's P values into the B fragment of P^T.  The V
// tile is stored as 64-row x 128-byte swizzled boxes.
template <int D>
__device__ __forceinline__ void mma_softmax_pv(TokAcc<D>& ac, const float (&sc)[4], uint32_t vs, unsigned char* vgen,
                                               int warp, int lane, int rows) {
    const int mi = lane >> 3;
    const int ld_row = warp * 16 + 8 * (mi >> 1) + (lane & 7);
    if (warp * 16 + 16 > rows) {
        for (int i = lane; i < 16 * (D / 8); i += 32) {
            const int r = warp * 16 + i / (D / 8);
            if (r >= rows) *reinterpret_cast<uint4*>(vgen + swz(r, i % (D / 8))) = make_uint4(0u, 0u, 0u, 0u);
        }
        // order these generic stores before the tile copy that later refills the stage
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
    }
    // per column: max over the 16 rows (the lanes of equal tig)
    float mx0 = fmaxf(sc[0], sc[2]), mx1 = fmaxf(sc[1], sc[3]);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float m0 = fmaxf(ac.m.x, mx0), m1 = fmaxf(ac.m.y, mx1);
    const bool none0 = m0 == -INFINITY, none1 = m1 == -INFINITY;
    const float a0 = none0 ? 1.f : exp2_approx(ac.m.x - m0);
    const float a1 = none1 ? 1.f : exp2_approx(ac.m.y - m1);
    float pr[4];
    pr[0] = none0 ? 0.f : exp2_approx(sc[0] - m0);
    pr[1] = none1 ? 0.f : exp2_approx(sc[1] - m1);
    pr[2] = none0 ? 0.f : exp2_approx(sc[2] - m0);
    pr[3] = none1 ? 0.f : exp2_approx(sc[3] - m1);
    ac.m = make_float2(m0, m1);
    ac.l.x = ac.l.x * a0 + (pr[0] + pr[2]);
    ac.l.y = ac.l.y * a1 + (pr[1] + pr[3]);
    uint32_t h0, l0, h1, l1;
    split_bf16(pr[0], pr[1], h0, l0);  // row gid
    split_bf16(pr[2], pr[3], h1, l1);  // row gid + 8
    h0 = movmatrix_trans(h0);
    l0 = movmatrix_trans(l0);
    h1 = movmatrix_trans(h1);
    l1 = movmatrix_trans(l1);
    // rescale only when some column's max moved (the lane holds its own columns' factors)
    if (!__all_sync(0xffffffffu, a0 == 1.f && a1 == 1.f)) {
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            ac.o[mt][0] *= a0;
            ac.o[mt][1] *= a1;
            ac.o[mt][2] *= a0;
            ac.o[mt][3] *= a1;
        }
    }
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
        uint32_t v0, v1, v2, v3;
        ldsm_x4_t(vs + swz(ld_row, 2 * mt + (mi & 1)), v0, v1, v2, v3);
        mma_bf16(ac.o[mt], v0, v1, v2, v3, h0, h1);
        mma_bf16(ac.o[mt], v0, v1, v2, v3, l0, l1);
    }
}

// Column-wise (per query) maximum over the 8 lanes of equal tig of a value
// held per lane for its two accumulator columns.
__device__ __forceinline__ float2 column_max(float2 v) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        v.x = fmaxf(v.x, __shfl_xor_sync(0xffffffffu, v.x, off));
        v.y = fmaxf(v.y, __shfl_xor_sync(0xffffffffu, v.y, off));
    }
    return v;
}

// One tile of a TokAcc consumer on a fixed reference max (FlashDecoding++
// summary, sections 1, 3, 5: one max value known before the scores, no
// reduction to the tile's max, a fallback when the scores leave the range it
// was chosen for).  phi2 / lo2 (log2 units) hold the reference and its lower
// end for the lane's two columns (queries 2 tig, 2 tig + 1).  While every
// valid score of the tile lies in [lo2, phi2] (one warp vote) the weights are
// 2^(s - phi2), normal binary32 numbers in [2^(lo2 - phi2), 1]: no max
// reduction, no rescale; `seen` keeps the lane's max of the attended scores.
// At the first tile outside the range the warp rebases O and l from phi2 to
// the largest score it attended (the state the running-max computation holds
// there) and continues with mma_softmax_pv.
template <int D>
__device__ __forceinline__ void fixed_ref_softmax_pv(TokAcc<D>& ac, bool& on_ref, float2& seen, const float (&sc)[4],
                                                     uint32_t vs, unsigned char* vgen, int warp, int lane, int rows,
                                                     float2 phi2, float2 lo2) {
    if (on_ref) {
        bool ok = true;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float ph = (i & 1) ? phi2.y : phi2.x, lo = (i & 1) ? lo2.y : lo2.x;
            ok &= sc[i] == -INFINITY || (sc[i] >= lo && sc[i] <= ph);
        }
        if (__all_sync(0xffffffffu, ok)) {
            const int mi = lane >> 3;
            const int ld_row = warp * 16 + 8 * (mi >> 1) + (lane & 7);
            if (warp * 16 + 16 > rows) {
                for (int i = lane; i < 16 * (D / 8); i += 32) {
                    const int r = warp * 16 + i / (D / 8);
                    if (r >= rows) *reinterpret_cast<uint4*>(vgen + swz(r, i % (D / 8))) = make_uint4(0u, 0u, 0u, 0u);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
            }
            float pr[4];
            pr[0] = exp2_approx(sc[0] - phi2.x);  // 2^-inf = +0
            pr[1] = exp2_approx(sc[1] - phi2.y);
            pr[2] = exp2_approx(sc[2] - phi2.x);
            pr[3] = exp2_approx(sc[3] - phi2.y);
            seen.x = fmaxf(seen.x, fmaxf(sc[0], sc[2]));
            seen.y = fmaxf(seen.y, fmaxf(sc[1], sc[3]));
            ac.l.x += pr[0] + pr[2];
            ac.l.y += pr[1] + pr[3];
            uint32_t h0, l0, h1, l1;
            split_bf16(pr[0], pr[1], h0, l0);
            split_bf16(pr[2], pr[3], h1, l1);
            h0 = movmatrix_trans(h0);
            l0 = movmatrix_trans(l0);
            h1 = movmatrix_trans(h1);
            l1 = movmatrix_trans(l1);
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                uint32_t v0, v1, v2, v3;
                ldsm_x4_t(vs + swz(ld_row, 2 * mt + (mi & 1)), v0, v1, v2, v3);
                mma_bf16(ac.o[mt], v0, v1, v2, v3, h0, h1);
                mma_bf16(ac.o[mt], v0, v1, v2, v3, l0, l1);
            }
            return;
        }
        // fallback: O and l are relative to phi2; rebase them to the largest
        // attended score (every one of them lies in [lo2, phi2])
        on_ref = false;
        const float2 m = column_max(seen);
        const float a0 = m.x == -INFINITY ? 1.f : exp2_approx(phi2.x - m.x);
        const float a1 = m.y == -INFINITY ? 1.f : exp2_approx(phi2.y - m.y);
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            ac.o[mt][0] *= a0;
            ac.o[mt][1] *= a1;
            ac.o[mt][2] *= a0;
            ac.o[mt][3] *= a1;
        }
        ac.l.x *= a0;
        ac.l.y *= a1;
        ac.m = m;
    }
    mma_softmax_pv<D>(ac, sc, vs, vgen, warp, lane, rows);
}

// End of a consumer that may still be on its fixed reference: a column's
// partial is then relative to phi2 (none when it attended nothing).
template <int D>
__device__ __forceinline__ void fixed_ref_finish(TokAcc<D>& ac, float2 seen, float2 phi2) {
    const float2 m = column_max(seen);
    ac.m = make_float2(m.x == -INFINITY ? -INFINITY : phi2.x, m.y == -INFINITY ? -INFINITY : phi2.y);
}

// Where a CTA's combined result goes: the final output (one chunk per
// sequence) or its chunk's slot of the merge workspace.
struct StoreTarget {
    void* out;
    int out_bf16;
    float* lse;
    float* part_o;   // [rows, splits, D]: O_i / l_i
    float* part_ml;  // [rows, splits, 2]: (m_i in log2 units, l_i)
    int direct;
    int splits;
};

// Final step of both combines: red_o/red_m/red_l hold every consumer warp's
// (O, m, l) per query; merge the warps and write the CTA's result.
template <int D, int GP, int CW>
__device__ __forceinline__ void store_combined(unsigned char* smem, int tid, int G, int row0, int split,
                                               const StoreTarget& st) {
    const float* red_o = reinterpret_cast<const float*>(smem);
    const float* red_m = red_o + CW * GP * D;
    const float* red_l = red_m + CW * GP;
    for (int idx = tid; idx < G * D; idx += CW * 32) {
        const int g = idx / D, dim = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < CW; ++w) M = fmaxf(M, red_m[w * GP + g]);
        float lsum = 0.f, acc = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < CW; ++w) {
                const float mw = red_m[w * GP + g];
                const float sc = mw == -INFINITY ? 0.f : exp2_approx(mw - M);
                lsum += sc * red_l[w * GP + g];
                acc += sc * red_o[(w * GP + g) * D + dim];
            }
        }
        const int row = row0 + g;
        const float val = lsum > 0.f ? acc / lsum : 0.f;
        if (st.direct) {
            const size_t oi = (size_t)row * D + dim;
            if (st.out_bf16) static_cast<uint16_t*>(st.out)[oi] = f32_to_bf16_bits(val);
            else static_cast<float*>(st.out)[oi] = val;
            if (dim == 0 && st.lse) st.lse[row] = lsum > 0.f ? (M + __log2f(lsum)) * kLn2 : -INFINITY;
        } else {
            const size_t pi = (size_t)row * st.splits + split;
            st.part_o[pi * D + dim] = val;
            if (dim == 0) {
                st.part_ml[2 * pi + 0] = lsum > 0.f ? M : -INFINITY;
                st.part_ml[2 * pi + 1] = lsum;
            }
        }
    }
}


// End of a partial pass: every consumer warp holds, per query g of the
// group, a running max m (log2 units, warp-uniform), a per-lane share of the
// exp-sum l and, in the lanes of each row group, the output accumulator for
// 8 columns.  Sum l over the warp and o over row groups, combine the CW warps
// through shared memory (the stage ring is reused, after a barrier over the
// consumer warps) and store.  row0 = b * Hq + first query head of the group.
template <int D, int GP, int CW>
__device__ __forceinline__ void combine_warps_and_store(unsigned char* smem, int warp, int lane, int G, int row0,
                                                        int split, const float (&m_run)[GP], float (&l_lane)[GP],
                                                        float2 (&o)[GP][4], bool failed, const StoreTarget& st) {
    constexpr int LPR = D / 8;
    const int c = lane % LPR;
#pragma unroll
    for (int g = 0; g < GP; ++g) {
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) l_lane[g] += __shfl_xor_sync(0xffffffffu, l_lane[g], off);
#pragma unroll
        for (int off = 16; off >= LPR; off >>= 1) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                o[g][e].x += __shfl_xor_sync(0xffffffffu, o[g][e].x, off);
                o[g][e].y += __shfl_xor_sync(0xffffffffu, o[g][e].y, off);
            }
        }
    }
    named_barrier(1, CW * 32);  // every consumer is done with the stage rings
    float* red_o = reinterpret_cast<float*>(smem);  // [CW][GP][D]
    float* red_m = red_o + CW * GP * D;             // [CW][GP]
    float* red_l = red_m + CW * GP;                 // [CW][GP]
    if (lane < LPR) {
#pragma unroll
        for (int g = 0; g < GP; ++g) {
            float4* dst = reinterpret_cast<float4*>(red_o + (warp * GP + g) * D + c * 8);
            dst[0] = make_float4(o[g][0].x, o[g][0].y, o[g][1].x, o[g][1].y);
            dst[1] = make_float4(o[g][2].x, o[g][2].y, o[g][3].x, o[g][3].y);
        }
    }
    if (lane == 0) {
#pragma unroll
        for (int g = 0; g < GP; ++g) {
            red_m[warp * GP + g] = failed ? -INFINITY : m_run[g];
            red_l[warp * GP + g] = failed ? 0.f : l_lane[g];
        }
    }
    named_barrier(1, CW * 32);
    store_combined<D, GP, CW>(smem, warp * 32 + lane, G, row0, split, st);
}

// The same for the tensor-core consumers: a warp's output lives in O^T
// accumulator fragments (o[mt][i] = O[query 2*tig + (i & 1)][dim 16*mt +
// gid + 8*(i >> 1)], gid = lane / 4, tig = lane % 4), its running max m (log2
// units) and exp-sum share l belong to query gid (each quad shares m; l is a
// per-lane share).
template <int D, int GP, int CW>
__device__ __forceinline__ void combine_mma_warps_and_store(unsigned char* smem, int warp, int lane, int G, int row0,
                                                            int split, float m_run, float l_run,
                                                            float (&o)[D / 16][4], bool failed,
                                                            const StoreTarget& st) {
    static_assert(GP == 8, "tensor-core consumers hold 8 query columns");
    const int gid = lane >> 2, tig = lane & 3;
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    named_barrier(1, CW * 32);
    float* red_o = reinterpret_cast<float*>(smem);  // [CW][GP][D]
    float* red_m = red_o + CW * GP * D;             // [CW][GP]
    float* red_l = red_m + CW * GP;                 // [CW][GP]
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int q = 2 * tig + (i & 1);
            const int dim = 16 * mt + gid + 8 * (i >> 1);
            red_o[(warp * GP + q) * D + dim] = o[mt][i];
        }
    }
    if (tig == 0) {
        red_m[warp * GP + gid] = failed ? -INFINITY : m_run;
        red_l[warp * GP + gid] = failed ? 0.f : l_run;
    }
    named_barrier(1, CW * 32);
    store_combined<D, GP, CW>(smem, warp * 32 + lane, G, row0, split, st);
}

// The end of a TokAcc consumer: exp-sums over the warp's 16 rows, (m, l) of
// query gid moved to the lane layout combine_mma_warps_and_store expects
// (query gid's values from lane gid / 2, column gid & 1; l only in the
// quad's first lane, the combine sums l over the quad), then the combine.
template <int D, int CW>
__device__ __forceinline__ void combine_tok_warps_and_store(unsigned char* smem, int warp, int lane, int G, int row0,
                                                            int split, TokAcc<D>& ac, bool failed,
                                                            const StoreTarget& st) {
    const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        ac.l.x += __shfl_xor_sync(0xffffffffu, ac.l.x, off);
        ac.l.y += __shfl_xor_sync(0xffffffffu, ac.l.y, off);
    }
    const float me = __shfl_sync(0xffffffffu, ac.m.x, gid >> 1), mo = __shfl_sync(0xffffffffu, ac.m.y, gid >> 1);
    const float le = __shfl_sync(0xffffffffu, ac.l.x, gid >> 1), lo = __shfl_sync(0xffffffffu, ac.l.y, gid >> 1);
    const float m_q = (gid & 1) ? mo : me;
    const float l_q = tig == 0 ? ((gid & 1) ? lo : le) : 0.f;
    combine_mma_warps_and_store<D, 8, CW>(smem, warp, lane, G, row0, split, m_q, l_q, ac.o, failed, st);
}

}  // namespace fd
