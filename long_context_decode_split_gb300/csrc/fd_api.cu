// fd_api.cu -- the extern "C" entry points declared in include/fd.h: host-side
// argument checks, the split planner and the dispatch to the kernels.  No
// entry point allocates memory or synchronises (except fd_device_status).
#include <cmath>
#include <cstdint>
#include <cstring>

#include <cuda_runtime.h>

#include "fd.h"
#include "fd_internal.h"

namespace {

using fd::kTile;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int current_sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return -1;
    if (dev >= 0 && dev < 64) cache[dev] = n;
    return n;
}

int check_shape(int B, int Hq, int Hkv, int L_max, int d) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || L_max < 0) return FD_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return FD_ERR_INVALID_ARG;
    if (B > 65535 || Hkv > 65535 || L_max > (1 << 30)) return FD_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FD_ERR_UNSUPPORTED;
    if (Hq / Hkv > 8) return FD_ERR_UNSUPPORTED;
    return FD_OK;
}

// Chunk plan shared by the planner queries, the workspace sizes and the
// launches.  `chunk_fixed` = 0 means per-sequence chunks of
// ceil(L_b / splits) rounded up to 64 tokens.
struct Plan {
    int splits;
    int chunk_fixed;
};

// The "Flash Decoding" tutorial (section 6, misconception 2) asks for a chunk
// count that keeps every compute unit busy, chunks of at least a few hundred
// tokens, and no more chunks than that: each costs merge work.  Here that is
// a cost model over whole 64-token tiles, in units of one tile's bytes at
// the GPU's full HBM bandwidth.  A wave of n CTAs with c tiles each takes
//   c * max(n, r),
// r being the number of CTAs whose copy pipelines together saturate HBM
// (a lone CTA streams at about 1/r of the GPU's bandwidth); CTAs beyond
// the resident slots form further waves; each chunk adds a small fixed cost
// and so does each wave (wave_tiles > 0: that many tiles of a CTA's time,
// for the passes whose CTAs are bound by their SM's issue, not by HBM).
// So: few, long chunks while HBM stays saturated, and no small trailing
// wave.  Ragged batches (lengths unknown on the host) take
// chunks such that sequences of length L_max span about four waves, so the
// hardware block scheduler can even out the load.
Plan plan_uncached(int B, int Hkv, int L_max, int requested, bool ragged, int ctas_per_sm, int sms, double r,
                   bool fill_slots, double wave_tiles);

// The cost model walks every chunk count (thousands for a 1M-token cache):
// its answers are remembered per thread for the last few argument sets.
Plan plan(int B, int Hkv, int L_max, int requested, bool ragged, int ctas_per_sm, int sms, double r,
          bool fill_slots = false, double wave_tiles = 0.0) {
    struct Entry {
        int B, Hkv, L_max, requested, ragged, ctas_per_sm, sms, fill_slots;
        double r, wave_tiles;
        Plan pl;
        bool used;
    };
    constexpr int kEntries = 8;
    thread_local Entry cache[kEntries] = {};
    thread_local int next = 0;
    for (const Entry& e : cache)
        if (e.used && e.B == B && e.Hkv == Hkv && e.L_max == L_max && e.requested == requested &&
            e.ragged == (int)ragged && e.ctas_per_sm == ctas_per_sm && e.sms == sms &&
            e.fill_slots == (int)fill_slots && e.r == r && e.wave_tiles == wave_tiles)
            return e.pl;
    const Plan pl = plan_uncached(B, Hkv, L_max, requested, ragged, ctas_per_sm, sms, r, fill_slots, wave_tiles);
    cache[next] = Entry{B, Hkv, L_max, requested, (int)ragged, ctas_per_sm, sms, (int)fill_slots, r, wave_tiles, pl,
                        true};
    next = (next + 1) % kEntries;
    return pl;
}

Plan plan_uncached(int B, int Hkv, int L_max, int requested, bool ragged, int ctas_per_sm, int sms, double r,
                   bool fill_slots, double wave_tiles) {
    Plan pl{1, 0};
    if (requested > 0) {
        pl.splits = requested;
        return pl;
    }
    const int tiles = (L_max + kTile - 1) / kTile;
    if (tiles <= 4 || sms <= 0) return pl;
    const long units = (long)B * Hkv;
    const long slots = (long)sms * (ctas_per_sm > 0 ? ctas_per_sm : 1);
    const int min_chunk_tiles = 4;  // 256 tokens
    int best_chunk = tiles;
    if (!ragged) {
        const double wave_cost = wave_tiles > 0.0 ? wave_tiles * (double)slots : 400.0, split_cost = 20.0;
        double best = 1e300;
        const int max_s = tiles / min_chunk_tiles;
        for (int S = 1; S <= max_s; ++S) {
            const int ct = (tiles + S - 1) / S;
            const int s_eff = (tiles + ct - 1) / ct;
            if (s_eff != S) continue;  // same chunk as a smaller S
            const long ctas = units * s_eff;
            const long full = ctas / slots, rest = ctas % slots;
            double cost = (double)full * ct * (slots > r ? (double)slots : r);
            if (rest) cost += (double)ct * (rest > r ? (double)rest : r);
            cost += wave_cost * (double)(full + (rest ? 1 : 0)) + split_cost * s_eff * units / (double)slots;
            if (cost < best - 1e-9) {
                best = cost;
                best_chunk = ct;
            }
        }
        // (bf16 pass) A single wave that leaves resident slots empty (some
        // SMs run two CTAs, others one) streams below the bandwidth the full
        // machine reaches; twice the chunks fill every slot once and most of
        // them a second time.  A context-length ladder (B = 1, 8, 32;
        // L = 4K..1M) measured this 5-6% faster at B = 32 and ~1% at B = 8,
        // and slower only where the halved chunks fall below 64 tiles, which
        // stay as they are.
        const int S1 = (tiles + best_chunk - 1) / best_chunk;
        const long n1 = units * S1;
        const int ct2 = (best_chunk + 1) / 2;
        const int S2 = (tiles + ct2 - 1) / ct2;
        const long n2 = units * S2;
        if (fill_slots && n1 >= sms && n1 < slots && ct2 >= 64 && n2 >= slots && n2 % slots >= slots / 2)
            best_chunk = ct2;
    } else {
        // aim at ~4 waves for sequences of length L_max, chunks of 8..256 tiles
        // (on a batch of lengths U[L_max/8, L_max] fewer, longer chunks win
        // until about four waves; shorter sequences then fill the gaps)
        long ct = (units * tiles + 4 * slots - 1) / (4 * slots);
        if (ct < 8) ct = 8;
        if (ct > 256) ct = 256;
        if (ct > tiles) ct = tiles;
        best_chunk = (int)ct;
    }
    pl.chunk_fixed = best_chunk * kTile;
    pl.splits = (L_max + pl.chunk_fixed - 1) / pl.chunk_fixed;
    if (pl.splits <= 1) pl = Plan{1, 0};
    return pl;
}

// CTAs that saturate HBM.  On GB300 a CTA of the d=128 pass (3 stages of
// 32 KiB in flight) streams ~64 GB/s alone, so ~110 would do in theory; one
// CTA per SM is the measured safe point (a chunk-count sweep of the 32K and
// 1M-token workloads has its optimum there).  The d=64 pass keeps 2/3 of the
// bytes in flight, so it needs 1.5x as many.
double saturating_ctas(int d, int sms) { return (d == 128 ? 1.0 : 1.5) * (sms > 0 ? sms : 1); }

Plan decode_plan(int B, int Hq, int Hkv, int L_max, int d, int requested, bool ragged) {
    const int sms = current_sm_count();
    const int occ = requested > 0 ? 1 : fd::decode_ctas_per_sm(d, Hq / Hkv, ragged);
    return plan(B, Hkv, L_max, requested, ragged, occ, sms, saturating_ctas(d, sms), true);
}

// The fp8 cache moves d + 4 bytes per row and operand where the bf16 cache
// moves 2d: a tile carries the bytes of a bf16 tile of half the head size.
Plan fp8_plan(int B, int Hq, int Hkv, int L_max, int d, int requested, bool ragged) {
    const int sms = current_sm_count();
    const int occ = requested > 0 ? 1 : fd::fp8_ctas_per_sm(d, ragged);
    return plan(B, Hkv, L_max, requested, ragged, occ, sms, saturating_ctas(d / 2, sms));
}

// The fp4 cache moves d/2 + d/32 bytes per row and operand, but its pass is
// bound by the widening of the codes on the CUDA cores, not by HBM: like the
// top-delta pass it needs every resident CTA slot busy.  (Counting only the
// CTAs that would saturate HBM left 48 of 304 slots empty on the 1M-token and
// FFD caches: 293 -> 250 us and 149 -> 130 us when the chunks fill them.)
// Each further wave costs about 4.5 tiles of a CTA's time (pipeline fill,
// the last tile, the combine): a chunk-count sweep at 3 CTAs/SM measured one
// full wave 7% faster than four on the FFD cache (124.3 vs 133.3 us) and 11%
// faster than two on MHA-32K (40.0 vs 45.0 us).
Plan fp4_plan(int B, int Hq, int Hkv, int L_max, int d, int requested, bool ragged) {
    const int sms = current_sm_count();
    const int occ = requested > 0 ? 1 : fd::fp4_ctas_per_sm(d, ragged);
    return plan(B, Hkv, L_max, requested, ragged, occ, sms, (double)occ * (sms > 0 ? sms : 1), false, 4.5);
}

Plan topdelta_plan(int B, int Hq, int Hkv, int L_max, int d, int requested) {
    const int sms = current_sm_count();
    const int occ = requested > 0 ? 1 : fd::topdelta_ctas_per_sm(d, Hq / Hkv);
    // the fused sparse pass is bound by its instruction issue, not by HBM: it
    // needs every resident CTA slot busy to reach full speed.  A further wave
    // costs it about 20 tiles of a CTA's time (the anchor pass, two pipelines
    // to fill, the last tiles): on the FFD cache one wave of 9 chunks ran
    // 272.7 us against 281.3 us for two waves of 19.
    return plan(B, Hkv, L_max, requested, false, occ, sms, (double)occ * (sms > 0 ? sms : 1), false, 20.0);
}

int to_status(cudaError_t e) { return e == cudaSuccess ? FD_OK : FD_ERR_CUDA; }

enum class Cache { BF16, FP8, FP4 };

Plan cache_plan(Cache cache, int B, int Hq, int Hkv, int L_max, int d, int requested, bool ragged) {
    switch (cache) {
        case Cache::FP8: return fp8_plan(B, Hq, Hkv, L_max, d, requested, ragged);
        case Cache::FP4: return fp4_plan(B, Hq, Hkv, L_max, d, requested, ragged);
        default: return decode_plan(B, Hq, Hkv, L_max, d, requested, ragged);
    }
}

// Chunks per sequence (negative status on bad arguments) and workspace bytes
// (0 on bad arguments) of a dense or paged call over the given cache.
int num_splits_for(Cache cache, int B, int Hq, int Hkv, int L_max, int d, int num_splits, int ragged) {
    const int st = check_shape(B, Hq, Hkv, L_max, d);
    if (st != FD_OK) return -st;
    if (num_splits < 0) return -FD_ERR_INVALID_ARG;
    return cache_plan(cache, B, Hq, Hkv, L_max, d, num_splits, ragged != 0).splits;
}

size_t workspace_for(Cache cache, int B, int Hq, int Hkv, int L_max, int d, int num_splits, int ragged) {
    if (check_shape(B, Hq, Hkv, L_max, d) != FD_OK || num_splits < 0) return 0;
    const Plan pl = cache_plan(cache, B, Hq, Hkv, L_max, d, num_splits, ragged != 0);
    return fd::decode_workspace_bytes(B, Hq, d, pl.splits);
}

// Validates the arguments every decode entry point shares, plans the chunks
// and enqueues the partial pass (+ merge) for the given cache.
int decode_common(fd::DecodeArgs& a, int num_splits, bool ragged, int out_dtype, void* workspace,
                  size_t workspace_bytes, void* stream, Cache cache) {
    const bool quantized = cache != Cache::BF16;  // scale arrays required
    if (out_dtype != FD_OUT_F32 && out_dtype != FD_OUT_BF16) return FD_ERR_INVALID_ARG;
    if (num_splits < 0 || !std::isfinite(a.scale)) return FD_ERR_INVALID_ARG;
    if (a.B > 0 && (!a.q || !a.k || !a.v || !a.out)) return FD_ERR_INVALID_ARG;
    if (!aligned16(a.q) || !aligned16(a.k) || !aligned16(a.v) || !aligned16(a.out)) return FD_ERR_INVALID_ARG;
    if (quantized && ((a.B > 0 && (!a.k_scales || !a.v_scales)) || !aligned16(a.k_scales) || !aligned16(a.v_scales)))
        return FD_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(a.lse) & 3u) || (reinterpret_cast<uintptr_t>(a.seq_lens) & 3u))
        return FD_ERR_INVALID_ARG;
    // tile copies address cache rows with 32-bit coordinates
    const long long cache_rows = a.page_table ? (long long)a.num_pages * a.Hkv * kTile
                                              : (long long)a.B * a.Hkv * a.L_max;
    if (cache_rows > 0x7fffffffLL) return FD_ERR_UNSUPPORTED;
    const Plan pl = cache_plan(cache, a.B, a.Hq, a.Hkv, a.L_max, a.D, num_splits, ragged);
    const size_t need = fd::decode_workspace_bytes(a.B, a.Hq, a.D, pl.splits);
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return FD_ERR_WORKSPACE_TOO_SMALL;
        if (!aligned16(workspace)) return FD_ERR_INVALID_ARG;
    }
    a.splits = pl.splits;
    a.chunk_fixed = pl.chunk_fixed;
    a.out_bf16 = out_dtype == FD_OUT_BF16;
    float* ws = static_cast<float*>(workspace);
    a.part_o = ws;
    a.part_ml = ws ? ws + (size_t)a.B * a.Hq * pl.splits * a.D : nullptr;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    return to_status(cache == Cache::FP8   ? fd::launch_decode_fp8(a, st)
                     : cache == Cache::FP4 ? fd::launch_decode_fp4(a, st)
                                           : fd::launch_decode(a, st));
}

// Contiguous cache [B, Hkv, L_max, ...]: K and V (codes for fp8/fp4) and, for
// the quantized caches, their scale arrays.
// The unified-max variant takes a finite fixed max value phi.
constexpr float kMaxAbsPhi = 1e30f;

int dense_entry(Cache cache, const void* q, const void* k, const void* v, const void* k_scales,
                const void* v_scales, const int32_t* seq_lens, int B, int Hq, int Hkv, int L_max, int d,
                float scale, int num_splits, void* out, int out_dtype, float* lse, void* workspace,
                size_t workspace_bytes, void* stream, bool unified = false, float phi = 0.f) {
    const int st = check_shape(B, Hq, Hkv, L_max, d);
    if (st != FD_OK) return st;
    if (unified && !(std::fabs(phi) <= kMaxAbsPhi)) return FD_ERR_INVALID_ARG;
    fd::DecodeArgs a = {};
    a.unified = unified ? 1 : 0;
    a.phi = phi;
    a.q = q;
    a.k = k;
    a.v = v;
    a.k_scales = k_scales;
    a.v_scales = v_scales;
    a.seq_lens = seq_lens;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.L_max = L_max;
    a.D = d;
    a.scale = scale;
    a.out = out;
    a.lse = lse;
    return decode_common(a, num_splits, seq_lens != nullptr, out_dtype, workspace, workspace_bytes, stream, cache);
}

// Paged cache: pools [num_pages, Hkv, 64, ...] and a page table [B, max_pages].
int paged_entry(Cache cache, const void* q, const void* k_pages, const void* v_pages, const void* k_scales,
                const void* v_scales, const int32_t* page_table, int max_pages, int num_pages,
                const int32_t* seq_lens, int page_size, int B, int Hq, int Hkv, int d, float scale, int num_splits,
                void* out, int out_dtype, float* lse, void* workspace, size_t workspace_bytes, void* stream,
                bool unified = false, float phi = 0.f) {
    if (page_size != kTile) return page_size > 0 ? FD_ERR_UNSUPPORTED : FD_ERR_INVALID_ARG;
    if (unified && !(std::fabs(phi) <= kMaxAbsPhi)) return FD_ERR_INVALID_ARG;
    if (max_pages <= 0 || num_pages < 0 || max_pages > (1 << 24)) return FD_ERR_INVALID_ARG;
    const int L_max = max_pages * page_size;
    const int st = check_shape(B, Hq, Hkv, L_max, d);
    if (st != FD_OK) return st;
    if (B > 0 && (!page_table || !seq_lens)) return FD_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(page_table) & 3u) return FD_ERR_INVALID_ARG;
    fd::DecodeArgs a = {};
    a.unified = unified ? 1 : 0;
    a.phi = phi;
    a.q = q;
    a.k = k_pages;
    a.v = v_pages;
    a.k_scales = k_scales;
    a.v_scales = v_scales;
    a.seq_lens = seq_lens;
    a.page_table = page_table;
    a.max_pages = max_pages;
    a.num_pages = num_pages;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.L_max = L_max;
    a.D = d;
    a.scale = scale;
    a.out = out;
    a.lse = lse;
    return decode_common(a, num_splits, true, out_dtype, workspace, workspace_bytes, stream, cache);
}

}  // namespace

extern "C" {

int fd_abi_version(void) { return FD_ABI_VERSION; }

const char* fd_status_string(int status) {
    switch (status) {
        case FD_OK: return "FD_OK";
        case FD_ERR_INVALID_ARG: return "FD_ERR_INVALID_ARG: invalid argument";
        case FD_ERR_UNSUPPORTED: return "FD_ERR_UNSUPPORTED: shape not supported (d, group size or page size)";
        case FD_ERR_WORKSPACE_TOO_SMALL: return "FD_ERR_WORKSPACE_TOO_SMALL: workspace smaller than required";
        case FD_ERR_BAD_PAGE_TABLE: return "FD_ERR_BAD_PAGE_TABLE: a page id was outside the page pool";
        case FD_ERR_CUDA: return "FD_ERR_CUDA: a CUDA call failed";
        case FD_ERR_DEVICE_TIMEOUT: return "FD_ERR_DEVICE_TIMEOUT: a kernel pipeline wait hit its time limit";
        default: return "unknown fd_status";
    }
}

int fd_num_splits(int B, int Hq, int Hkv, int L_max, int d, int num_splits, int ragged) {
    return num_splits_for(Cache::BF16, B, Hq, Hkv, L_max, d, num_splits, ragged);
}

size_t fd_decode_workspace_size(int B, int Hq, int Hkv, int L_max, int d, int num_splits, int ragged) {
    return workspace_for(Cache::BF16, B, Hq, Hkv, L_max, d, num_splits, ragged);
}

int fd_decode_dense(const void* q, const void* k, const void* v, const int32_t* seq_lens,
                    int B, int Hq, int Hkv, int L_max, int d, float scale, int num_splits,
                    void* out, int out_dtype, float* lse,
                    void* workspace, size_t workspace_bytes, void* stream) {
    return dense_entry(Cache::BF16, q, k, v, nullptr, nullptr, seq_lens, B, Hq, Hkv, L_max, d, scale, num_splits,
                       out, out_dtype, lse, workspace, workspace_bytes, stream);
}

int fd_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                    const int32_t* page_table, int max_pages, int num_pages,
                    const int32_t* seq_lens, int page_size,
                    int B, int Hq, int Hkv, int d, float scale, int num_splits,
                    void* out, int out_dtype, float* lse,
                    void* workspace, size_t workspace_bytes, void* stream) {
    return paged_entry(Cache::BF16, q, k_pages, v_pages, nullptr, nullptr, page_table, max_pages, num_pages,
                       seq_lens, page_size, B, Hq, Hkv, d, scale, num_splits, out, out_dtype, lse, workspace,
                       workspace_bytes, stream);
}

int fd_decode_dense_unified(const void* q, const void* k, const void* v, const int32_t* seq_lens,
                            int B, int Hq, int Hkv, int L_max, int d, float scale, float phi, int num_splits,
                            void* out, int out_dtype, float* lse,
                            void* workspace, size_t workspace_bytes, void* stream) {
    return dense_entry(Cache::BF16, q, k, v, nullptr, nullptr, seq_lens, B, Hq, Hkv, L_max, d, scale, num_splits,
                       out, out_dtype, lse, workspace, workspace_bytes, stream, true, phi);
}

int fd_decode_paged_unified(const void* q, const void* k_pages, const void* v_pages,
                            const int32_t* page_table, int max_pages, int num_pages,
                            const int32_t* seq_lens, int page_size,
                            int B, int Hq, int Hkv, int d, float scale, float phi, int num_splits,
                            void* out, int out_dtype, float* lse,
                            void* workspace, size_t workspace_bytes, void* stream) {
    return paged_entry(Cache::BF16, q, k_pages, v_pages, nullptr, nullptr, page_table, max_pages, num_pages,
                       seq_lens, page_size, B, Hq, Hkv, d, scale, num_splits, out, out_dtype, lse, workspace,
                       workspace_bytes, stream, true, phi);
}

int fd_quantize_kv_fp8(const void* x, const int32_t* seq_lens, int B, int H, int L_max, int d,
                       uint8_t* codes, float* scales, void* stream) {
    const int st = check_shape(B, H, H, L_max, d);
    if (st != FD_OK) return st;
    if (B > 0 && L_max > 0 && (!x || !codes || !scales)) return FD_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(codes) || !aligned16(scales)) return FD_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(seq_lens) & 3u) return FD_ERR_INVALID_ARG;
    fd::Fp8QuantArgs a = {x, seq_lens, B, H, L_max, d, codes, scales};
    return to_status(fd::launch_quantize_fp8(a, static_cast<cudaStream_t>(stream)));
}

int fd_num_splits_fp8(int B, int Hq, int Hkv, int L_max, int d, int num_splits, int ragged) {
    return num_splits_for(Cache::FP8, B, Hq, Hkv, L_max, d, num_splits, ragged);
}

size_t fd_decode_fp8_workspace_size(int B, int Hq, int Hkv, int L_max, int d, int num_splits, int ragged) {
    return workspace_for(Cache::FP8, B, Hq, Hkv, L_max, d, num_splits, ragged);
}

int fd_decode_dense_fp8(const void* q, const uint8_t* k_codes, const float* k_scales, const uint8_t* v_codes,
                        const float* v_scales, const int32_t* seq_lens, int B, int Hq, int Hkv, int L_max, int d,
                        float scale, int num_splits, void* out, int out_dtype, float* lse,
                        void* workspace, size_t workspace_bytes, void* stream) {
    return dense_entry(Cache::FP8, q, k_codes, v_codes, k_scales, v_scales, seq_lens, B, Hq, Hkv, L_max, d, scale,
                       num_splits, out, out_dtype, lse, workspace, workspace_bytes, stream);
}

int fd_decode_paged_fp8(const void* q, const uint8_t* k_pages, const float* k_page_scales, const uint8_t* v_pages,
                        const float* v_page_scales, const int32_t* page_table, int max_pages, int num_pages,
                        const int32_t* seq_lens, int page_size, int B, int Hq, int Hkv, int d, float scale,
                        int num_splits, void* out, int out_dtype, float* lse,
                        void* workspace, size_t workspace_bytes, void* stream) {
    return paged_entry(Cache::FP8, q, k_pages, v_pages, k_page_scales, v_page_scales, page_table, max_pages,
                       num_pages, seq_lens, page_size, B, Hq, Hkv, d, scale, num_splits, out, out_dtype, lse,
                       workspace, workspace_bytes, stream);
}

int fd_quantize_kv_fp4(const void* x, const int32_t* seq_lens, int B, int H, int L_max, int d,
                       uint8_t* codes, uint8_t* scales, void* stream) {
    const int st = check_shape(B, H, H, L_max, d);
    if (st != FD_OK) return st;
    if (B > 0 && L_max > 0 && (!x || !codes || !scales)) return FD_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(codes) || !aligned16(scales)) return FD_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(seq_lens) & 3u) return FD_ERR_INVALID_ARG;
    fd::Fp4QuantArgs a = {x, seq_lens, B, H, L_max, d, codes, scales, 0};
    return to_status(fd::launch_quantize_fp4(a, static_cast<cudaStream_t>(stream)));
}

int fd_quantize_v_fp4(const void* x, const int32_t* seq_lens, int B, int H, int L_max, int d,
                      uint8_t* codes, uint8_t* scales, void* stream) {
    const int st = check_shape(B, H, H, L_max, d);
    if (st != FD_OK) return st;
    if (B > 0 && L_max > 0 && (!x || !codes || !scales)) return FD_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(codes) || !aligned16(scales)) return FD_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(seq_lens) & 3u) return FD_ERR_INVALID_ARG;
    fd::Fp4QuantArgs a = {x, seq_lens, B, H, L_max, d, codes, scales, 1};
    return to_status(fd::launch_quantize_fp4(a, static_cast<cudaStream_t>(stream)));
}

int fd_num_splits_fp4(int B, int Hq, int Hkv, int L_max, int d, int num_splits, int ragged) {
    return num_splits_for(Cache::FP4, B, Hq, Hkv, L_max, d, num_splits, ragged);
}

size_t fd_decode_fp4_workspace_size(int B, int Hq, int Hkv, int L_max, int d, int num_splits, int ragged) {
    return workspace_for(Cache::FP4, B, Hq, Hkv, L_max, d, num_splits, ragged);
}

int fd_decode_dense_fp4(const void* q, const uint8_t* k_codes, const uint8_t* k_scales, const uint8_t* v_codes,
                        const uint8_t* v_scales, const int32_t* seq_lens, int B, int Hq, int Hkv, int L_max, int d,
                        float scale, int num_splits, void* out, int out_dtype, float* lse,
                        void* workspace, size_t workspace_bytes, void* stream) {
    return dense_entry(Cache::FP4, q, k_codes, v_codes, k_scales, v_scales, seq_lens, B, Hq, Hkv, L_max, d, scale,
                       num_splits, out, out_dtype, lse, workspace, workspace_bytes, stream);
}

int fd_decode_paged_fp4(const void* q, const uint8_t* k_pages, const uint8_t* k_page_scales, const uint8_t* v_pages,
                        const uint8_t* v_page_scales, const int32_t* page_table, int max_pages, int num_pages,
                        const int32_t* seq_lens, int page_size, int B, int Hq, int Hkv, int d, float scale,
                        int num_splits, void* out, int out_dtype, float* lse,
                        void* workspace, size_t workspace_bytes, void* stream) {
    return paged_entry(Cache::FP4, q, k_pages, v_pages, k_page_scales, v_page_scales, page_table, max_pages,
                       num_pages, seq_lens, page_size, B, Hq, Hkv, d, scale, num_splits, out, out_dtype, lse,
                       workspace, workspace_bytes, stream);
}

int fd_quantize_keys(const void* k, const int32_t* seq_lens, int B, int Hkv, int L_max, int d,
                     uint8_t* codes, void* mn_scale, int8_t* res, void* res_scale, void* stream) {
    const int st = check_shape(B, Hkv, Hkv, L_max, d);
    if (st != FD_OK) return st;
    if (B > 0 && L_max > 0 && (!k || !codes || !mn_scale || !res || !res_scale)) return FD_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(codes) || !aligned16(mn_scale) || !aligned16(res) || !aligned16(res_scale))
        return FD_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(seq_lens) & 3u) return FD_ERR_INVALID_ARG;
    fd::QuantArgs a = {k, seq_lens, B, Hkv, L_max, d, codes, mn_scale, res, res_scale};
    return to_status(fd::launch_quantize(a, static_cast<cudaStream_t>(stream)));
}

size_t fd_topdelta_workspace_size(int B, int Hq, int Hkv, int L_max, int d, int num_splits) {
    if (check_shape(B, Hq, Hkv, L_max, d) != FD_OK || num_splits < 0) return 0;
    const Plan pl = topdelta_plan(B, Hq, Hkv, L_max, d, num_splits);
    return fd::decode_workspace_bytes(B, Hq, d, pl.splits);
}

}  // extern "C"

namespace {

int topdelta_entry(const void* q, const uint8_t* codes, const void* mn_scale, const int8_t* res,
                   const void* res_scale, const void* v, const int32_t* seq_lens,
                   int B, int Hq, int Hkv, int L_max, int d, float scale, float delta,
                   int n_sink, int window, int num_splits,
                   void* out, int out_dtype, float* lse, uint32_t* sel_mask, int32_t* sel_count,
                   void* workspace, size_t workspace_bytes, void* stream, bool group_union) {
    const int st = check_shape(B, Hq, Hkv, L_max, d);
    if (st != FD_OK) return st;
    if (out_dtype != FD_OUT_F32 && out_dtype != FD_OUT_BF16) return FD_ERR_INVALID_ARG;
    if (num_splits < 0 || !std::isfinite(scale) || std::isnan(delta) || delta < 0.f) return FD_ERR_INVALID_ARG;
    if (n_sink < 0 || window < 0) return FD_ERR_INVALID_ARG;
    if (L_max % 4 != 0) return FD_ERR_UNSUPPORTED;  // keeps every tile copy 16-byte aligned
    if ((long long)B * Hkv * L_max > 0x7fffffffLL) return FD_ERR_UNSUPPORTED;  // 32-bit row coordinates
    if (B > 0 && (!q || !codes || !mn_scale || !res || !res_scale || !v || !out)) return FD_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(codes) || !aligned16(mn_scale) || !aligned16(res) || !aligned16(res_scale) ||
        !aligned16(v) || !aligned16(out))
        return FD_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
        (reinterpret_cast<uintptr_t>(sel_mask) & 3u) || (reinterpret_cast<uintptr_t>(sel_count) & 3u))
        return FD_ERR_INVALID_ARG;
    const Plan pl = topdelta_plan(B, Hq, Hkv, L_max, d, num_splits);
    const size_t need = fd::decode_workspace_bytes(B, Hq, d, pl.splits);
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return FD_ERR_WORKSPACE_TOO_SMALL;
        if (!aligned16(workspace)) return FD_ERR_INVALID_ARG;
    }
    fd::TopDeltaArgs a = {};
    a.q = q;
    a.codes = codes;
    a.mn_scale = mn_scale;
    a.res = res;
    a.res_scale = res_scale;
    a.v = v;
    a.seq_lens = seq_lens;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.L_max = L_max;
    a.D = d;
    a.scale = scale;
    a.delta = delta;
    a.n_sink = n_sink;
    a.window = window;
    a.splits = pl.splits;
    a.chunk_fixed = pl.chunk_fixed;
    a.group_union = group_union ? 1 : 0;
    a.out = out;
    a.out_bf16 = out_dtype == FD_OUT_BF16;
    a.lse = lse;
    a.sel_mask = sel_mask;
    a.sel_count = sel_count;
    float* ws = static_cast<float*>(workspace);
    a.part_o = ws;
    a.part_ml = ws ? ws + (size_t)B * Hq * pl.splits * d : nullptr;
    return to_status(fd::launch_topdelta(a, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

int fd_decode_topdelta(const void* q, const uint8_t* codes, const void* mn_scale, const int8_t* res,
                       const void* res_scale, const void* v, const int32_t* seq_lens,
                       int B, int Hq, int Hkv, int L_max, int d, float scale, float delta,
                       int n_sink, int window, int num_splits,
                       void* out, int out_dtype, float* lse, uint32_t* sel_mask, int32_t* sel_count,
                       void* workspace, size_t workspace_bytes, void* stream) {
    return topdelta_entry(q, codes, mn_scale, res, res_scale, v, seq_lens, B, Hq, Hkv, L_max, d, scale, delta,
                          n_sink, window, num_splits, out, out_dtype, lse, sel_mask, sel_count, workspace,
                          workspace_bytes, stream, false);
}

int fd_decode_topdelta_group_union(const void* q, const uint8_t* codes, const void* mn_scale, const int8_t* res,
                                   const void* res_scale, const void* v, const int32_t* seq_lens,
                                   int B, int Hq, int Hkv, int L_max, int d, float scale, float delta,
                                   int n_sink, int window, int num_splits,
                                   void* out, int out_dtype, float* lse, uint32_t* sel_mask, int32_t* sel_count,
                                   void* workspace, size_t workspace_bytes, void* stream) {
    return topdelta_entry(q, codes, mn_scale, res, res_scale, v, seq_lens, B, Hq, Hkv, L_max, d, scale, delta,
                          n_sink, window, num_splits, out, out_dtype, lse, sel_mask, sel_count, workspace,
                          workspace_bytes, stream, true);
}

int fd_debug_inject_wait_timeout(unsigned long long wait_limit_ns, int withhold_tile) {
    fd::inject_wait_timeout(wait_limit_ns, withhold_tile);
    return FD_OK;
}

int fd_device_status(int clear, void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FD_ERR_CUDA;
    unsigned a = 0, b = 0, c = 0, e = 0;
    if (fd::decode_status_read(&a, clear != 0) != cudaSuccess) return FD_ERR_CUDA;
    if (fd::topdelta_status_read(&b, clear != 0) != cudaSuccess) return FD_ERR_CUDA;
    if (fd::fp8_status_read(&c, clear != 0) != cudaSuccess) return FD_ERR_CUDA;
    if (fd::fp4_status_read(&e, clear != 0) != cudaSuccess) return FD_ERR_CUDA;
    const unsigned bits = a | b | c | e;
    if (bits & 2u) return FD_ERR_DEVICE_TIMEOUT;
    if (bits & 1u) return FD_ERR_BAD_PAGE_TABLE;
    if (bits & 4u) return FD_ERR_INVALID_ARG;
    return FD_OK;
}

}  // extern "C"
