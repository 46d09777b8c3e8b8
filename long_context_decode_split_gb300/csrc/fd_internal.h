// fd_internal.h -- host-side interface between the C-ABI layer (fd_api.cu)
// and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

namespace fd {

constexpr int kTile = 64;  // tokens per pipeline stage; also the page size

#ifdef __CUDACC__
#define FD_HD __host__ __device__
#else
#define FD_HD
#endif

// Chunk length in tokens for a sequence of length L: `chunk_fixed` when the
// plan fixed one, else ceil(L / splits) rounded up to whole 64-token tiles.
FD_HD inline int chunk_len(int L, int splits, int chunk_fixed) {
    if (chunk_fixed > 0) return chunk_fixed;
    int c = (L + splits - 1) / splits;
    c = (c + kTile - 1) / kTile * kTile;
    return c > 0 ? c : kTile;
}

// Inputs and outputs of one split-KV decode launch (dense or paged).
struct DecodeArgs {
    const void* q;            // [B, Hq, D] bf16
    const void* k;            // contiguous [B, Hkv, L_max, D] or pool [P, Hkv, 64, D]
    const void* v;
    const void* k_scales;     // fp8 cache: [rows] binary32 row scales; fp4 cache: [rows, D/32] u8 block
    const void* v_scales;     // exponents (of K and of V)
    const int32_t* seq_lens;  // [B] or null (= L_max)
    const int32_t* page_table;// [B, max_pages] when paged, else null
    int max_pages, num_pages;
    int B, Hq, Hkv, L_max, D;
    float scale;
    int splits;               // chunks per sequence = grid.x
    int chunk_fixed;          // > 0: every sequence uses this chunk (tokens)
    void* out;                // [B, Hq, D]
    int out_bf16;
    float* lse;               // [B, Hq] or null
    float* part_o;            // workspace: [B, Hq, splits, D]
    float* part_ml;           // workspace: [B, Hq, splits, 2]
    int unified;              // bf16 cache only: unified-max variant with fixed max value `phi`
    float phi;                // (natural-log units of the scaled score)
};

// Workspace bytes for `splits` chunks (0 when splits == 1).
size_t decode_workspace_bytes(int B, int Hq, int D, int splits);

// Occupancy (resident CTAs per SM) of the partial-pass kernel for this shape.
int decode_ctas_per_sm(int D, int G, bool paged);

// Enqueue the partial pass (+ merge when splits > 1).  Returns a cudaError_t.
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

// Device status words, one per translation unit that owns kernels.
cudaError_t decode_status_read(unsigned* bits, bool clear);

// Fault injection for the bf16 dense/paged pass (fd_debug_inject_wait_timeout).
void inject_wait_timeout(unsigned long long wait_limit_ns, int withhold_tile);

struct QuantArgs {
    const void* k;            // [B, Hkv, L_max, D] bf16
    const int32_t* seq_lens;
    int B, Hkv, L_max, D;
    uint8_t* codes;
    void* mn_scale;
    int8_t* res;
    void* res_scale;
};
cudaError_t launch_quantize(const QuantArgs& a, cudaStream_t stream);

struct TopDeltaArgs {
    const void* q;
    const uint8_t* codes;
    const void* mn_scale;
    const int8_t* res;
    const void* res_scale;
    const void* v;
    const int32_t* seq_lens;
    int B, Hq, Hkv, L_max, D;
    float scale, delta;
    int n_sink, window;
    int splits, chunk_fixed;
    int group_union;
    void* out;
    int out_bf16;
    float* lse;
    uint32_t* sel_mask;
    int32_t* sel_count;
    float* part_o;
    float* part_ml;
};
int topdelta_ctas_per_sm(int D, int G);
cudaError_t launch_topdelta(const TopDeltaArgs& a, cudaStream_t stream);
cudaError_t topdelta_status_read(unsigned* bits, bool clear);

// fp8 (e4m3) KV cache: encoder and decode (DecodeArgs with k/v = codes,
// k_scales/v_scales = row scales; same workspace layout as the bf16 path).
struct Fp8QuantArgs {
    const void* x;            // [B, H, L_max, D] bf16
    const int32_t* seq_lens;
    int B, H, L_max, D;
    uint8_t* codes;           // [B, H, L_max, D]
    float* scales;            // [B, H, L_max]
};
cudaError_t launch_quantize_fp8(const Fp8QuantArgs& a, cudaStream_t stream);
int fp8_ctas_per_sm(int D, bool paged);
cudaError_t launch_decode_fp8(const DecodeArgs& a, cudaStream_t stream);
cudaError_t fp8_status_read(unsigned* bits, bool clear);

// fp4 (e2m1, power-of-two block scales) KV cache: encoder and decode.
struct Fp4QuantArgs {
    const void* x;            // [B, H, L_max, D] bf16
    const int32_t* seq_lens;
    int B, H, L_max, D;
    uint8_t* codes;           // [B, H, L_max, D/2] (channel pairs), or [B, H, (L_max+1)/2, D] (token pairs)
    uint8_t* scales;          // [B, H, L_max, D/32]
    int token_pairs;          // the value-cache layout: one byte = one channel of tokens 2p, 2p + 1
};
cudaError_t launch_quantize_fp4(const Fp4QuantArgs& a, cudaStream_t stream);
int fp4_ctas_per_sm(int D, bool paged);
cudaError_t launch_decode_fp4(const DecodeArgs& a, cudaStream_t stream);
cudaError_t fp4_status_read(unsigned* bits, bool clear);

// Launch with programmatic stream serialization: the grid may be scheduled
// while the previous kernel in the stream is still running, so the kernel
// must execute griddepcontrol.wait before it touches global memory (every
// kernel launched this way does so first).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Merge of per-chunk partials (shared by the dense and top-delta paths).
cudaError_t launch_merge(const float* part_o, const float* part_ml, const int32_t* seq_lens,
                         int B, int Hq, int L_max, int D, int splits, int chunk_fixed,
                         void* out, int out_bf16, float* lse, cudaStream_t stream);

}  // namespace fd
