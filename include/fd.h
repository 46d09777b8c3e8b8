/*
 * fd.h -- C ABI of libfd: split-KV decode attention for long KV caches on
 * NVIDIA GB300 (sm_103a), with an opt-in sparse top-delta path.
 *
 * Sources of the operations declared here:
 *   [FD]  "Flash Decoding" tutorial (aiqz.cc/article/flash-decoding.html):
 *         section 1 (standard attention and its four steps), section 2 (the
 *         sequence split into chunks, per-chunk m_i, l_i, O_i, and the merge
 *         O = sum_i e^{m_i-m} l_i O_i / sum_j e^{m_j-m} l_j, m = max_i m_i),
 *         section 3 (KV cache cut into fixed-size pages), section 6 and the
 *         misconceptions section (how many chunks to use).
 *   [FFD] "Faster Than Flash: Exploiting Attention Sparsity for Efficient
 *         Long-Context Decoding" summary (PaperDaily): section 3 (top-delta
 *         rule s_ij >= m_i - delta), section 4 (pseudo-max from attention
 *         sinks and the local window), section 5 (2-bit body for the full
 *         scan, 8-bit residual loaded for candidates only), section 6 and
 *         Fig. 2 (one fused kernel: scan, select, correct, attend, aggregate).
 *   [FD++] FlashDecoding++ summary (nxbn.cn blog): asynchronous partial
 *         softmax with a unified (fixed) max value, and the fallback to the
 *         safe computation when the inputs leave its range.
 *   [KV8] Benchmarking blog on a hosted 1M-context model (xxmr.cn/news/240041),
 *         section 1: a narrow floating-point KV cache as the lever on the
 *         bytes a decode step reads.  The page gives no format; the fp8
 *         encoding below is this library's definition.
 *
 * Conventions shared by every entry point
 *   - Every data pointer is a DEVICE pointer owned by the caller, 16-byte
 *     aligned, to a C-contiguous (row-major) array.  bf16 and fp16 values are
 *     passed as their 16-bit patterns.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     only enqueue work on it: they never synchronise and never allocate
 *     memory.  Scratch memory is the caller's `workspace`.
 *   - Return value: an fd_status.  Arguments are checked on the host before
 *     anything is enqueued; a call that returns anything but FD_OK has
 *     enqueued nothing, except FD_ERR_CUDA, which reports a launch failure.
 *   - Faults found by the kernels themselves (a page id outside the pool, a
 *     pipeline wait that exceeded its time limit) do not stop the stream;
 *     they set a per-process device status word read by fd_device_status().
 *   - Softmax runs in natural-log units of the scaled score s = scale*<q,k>.
 *     lse[b,hq] = log sum_j exp(s_j) over the attended keys.  A sequence of
 *     length 0 yields out = 0 and lse = -inf.
 *   - Head grouping: query head hq reads KV head hq / (Hq / Hkv).
 *   - Supported shapes: d in {64, 128}; 1 <= Hq/Hkv <= 8; page_size == 64;
 *     at most 2^31 - 1 cache rows (B * Hkv * L_max, or num_pages * Hkv * 64)
 *     for the dense and paged decode (FD_ERR_UNSUPPORTED otherwise).
 *   - Results are deterministic for fixed inputs, shapes and num_splits.
 */
#ifndef FD_H
#define FD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FD_ABI_VERSION 2  /* 2: the fp4 value cache is stored in token pairs (fd_quantize_v_fp4) */

#if defined(__GNUC__)
#define FD_API __attribute__((visibility("default")))
#else
#define FD_API
#endif

typedef enum fd_status {
    FD_OK = 0,
    FD_ERR_INVALID_ARG = 1,          /* null/misaligned pointer, bad size or relation */
    FD_ERR_UNSUPPORTED = 2,          /* valid but not implemented: d, group size, page size */
    FD_ERR_WORKSPACE_TOO_SMALL = 3,  /* workspace_bytes below the *_workspace_size() value */
    FD_ERR_BAD_PAGE_TABLE = 4,       /* (device status) a page id outside [0, num_pages) */
    FD_ERR_CUDA = 5,                 /* a CUDA launch or query failed */
    FD_ERR_DEVICE_TIMEOUT = 6        /* (device status) a pipeline wait hit its time limit */
} fd_status;

typedef enum fd_out_dtype {
    FD_OUT_F32 = 0,                  /* out is float32 */
    FD_OUT_BF16 = 1                  /* out is bf16, rounded to nearest even */
} fd_out_dtype;

/* Version of this ABI (FD_ABI_VERSION of the built library). */
FD_API int fd_abi_version(void);

/* Static, human-readable name of a status code (never NULL). */
FD_API const char* fd_status_string(int status);

/* Number of chunks per sequence ("num_splits", [FD] section 2) that the
 * decode entry points will use on the CURRENT device for these sizes.
 * num_splits > 0 is honoured as the chunk count: chunk = ceil(L_b/num_splits)
 * rounded up to a multiple of 64 tokens (so trailing chunks may be empty).
 * num_splits == 0 lets the planner choose from the device's SM count
 * ([FD] section 6: fill every SM, chunks of at least a few hundred tokens).
 * `ragged` != 0 says sequence lengths may differ (paged batches).
 * Returns the chunk count (>= 1), or -FD_ERR_* on bad arguments. */
FD_API int fd_num_splits(int B, int Hq, int Hkv, int L_max, int d, int num_splits, int ragged);

/* Bytes of workspace the dense and paged decode need for these sizes on the
 * current device (same arguments as fd_num_splits).  0 when no
 * workspace is needed (one chunk).  Returns 0 on bad arguments too. */
FD_API size_t fd_decode_workspace_size(int B, int Hq, int Hkv, int L_max, int d,
                                int num_splits, int ragged);

/* Dense split-KV decode ([FD] sections 1-2): one new query token per
 * sequence attends to that sequence's whole contiguous KV cache.
 *   q         [B, Hq, d]          bf16
 *   k, v      [B, Hkv, L_max, d]  bf16
 *   seq_lens  [B] int32 in [0, L_max], or NULL: every sequence has L_max
 *   scale     softmax scale (usually 1/sqrt(d))
 *   num_splits 0 = planner, > 0 = chunk count (see fd_num_splits)
 *   out       [B, Hq, d] in out_dtype;  lse [B, Hq] float32, or NULL
 *   workspace fd_decode_workspace_size(B, Hq, Hkv, L_max, d, num_splits,
 *             seq_lens != NULL) bytes; may be NULL when that size is 0.
 * Tokens t >= seq_lens[b] are never read. */
FD_API int fd_decode_dense(const void* q, const void* k, const void* v,
                    const int32_t* seq_lens,
                    int B, int Hq, int Hkv, int L_max, int d,
                    float scale, int num_splits,
                    void* out, int out_dtype, float* lse,
                    void* workspace, size_t workspace_bytes, void* stream);

/* Paged split-KV decode ([FD] section 3 with sections 1-2): the cache is a
 * pool of fixed-size pages.
 *   k_pages, v_pages [num_pages, Hkv, page_size, d] bf16
 *   page_table [B, max_pages] int32: token t of sequence b is row
 *              t % page_size of page page_table[b * max_pages + t / page_size]
 *   seq_lens   [B] int32 in [0, max_pages * page_size] (required)
 *   page_size  must be 64
 * Other arguments as fd_decode_dense, with L_max = max_pages * page_size for
 * the workspace size (ragged = 1).  Only the first ceil(seq_lens[b]/64)
 * entries of a table row are read; an entry outside [0, num_pages) is not
 * dereferenced: its tokens are skipped and the device status records
 * FD_ERR_BAD_PAGE_TABLE. */
FD_API int fd_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                    const int32_t* page_table, int max_pages, int num_pages,
                    const int32_t* seq_lens, int page_size,
                    int B, int Hq, int Hkv, int d,
                    float scale, int num_splits,
                    void* out, int out_dtype, float* lse,
                    void* workspace, size_t workspace_bytes, void* stream);

/* Unified-max variants of fd_decode_dense and fd_decode_paged ([FD++]
 * sections 1 and 3, asynchronous
 * partial softmax with one fixed max value instead of a per-chunk maximum,
 * and section 5, the fallback to the safe computation when the softmax inputs
 * leave the range that value was chosen for).
 *   phi  the fixed max value, in natural-log units of the scaled score
 *        s = scale * <q, k>; finite (|phi| <= 1e30, else FD_ERR_INVALID_ARG).
 *        A good choice is the upper end of the scores the model produces
 *        (that summary quotes [-16.8, 6.5] for Llama2-7B).
 * Every chunk weights its keys by e^(s - phi) directly, with no maximum
 * reduction and no rescaling, while all of its scores lie in
 * [phi - 60, phi]; then every weight is a normal binary32 number in
 * [e^-60, 1] and no sum can overflow.  A chunk that meets a score outside
 * that range (above phi, or more than 60 below it) rebases what it has
 * accumulated to the largest score it attended and continues with the
 * running maximum of fd_decode_dense.  The result is the attention that
 * fd_decode_dense computes, up to fp32 rounding, for any phi.  All other
 * arguments, layouts, the workspace (fd_decode_workspace_size with the same
 * sizes) and errors are those of fd_decode_dense / fd_decode_paged. */
FD_API int fd_decode_dense_unified(const void* q, const void* k, const void* v,
                                   const int32_t* seq_lens,
                                   int B, int Hq, int Hkv, int L_max, int d,
                                   float scale, float phi, int num_splits,
                                   void* out, int out_dtype, float* lse,
                                   void* workspace, size_t workspace_bytes, void* stream);
FD_API int fd_decode_paged_unified(const void* q, const void* k_pages, const void* v_pages,
                                   const int32_t* page_table, int max_pages, int num_pages,
                                   const int32_t* seq_lens, int page_size,
                                   int B, int Hq, int Hkv, int d,
                                   float scale, float phi, int num_splits,
                                   void* out, int out_dtype, float* lse,
                                   void* workspace, size_t workspace_bytes, void* stream);

/* Key encoder for the sparse path ([FFD] section 5): per token and per
 * group of 32 channels, a 2-bit asymmetric body and an int8 symmetric
 * residual.  With x the group's bf16 values, in IEEE binary32 arithmetic:
 *   mn16 = fp16(min x), s16 = fp16((max x - min x) / 3)  (a zero min or
 *          max counts as +0)
 *   code = clamp(rint((x - mn16) / s16), 0, 3)      (0 when s16 == 0)
 *   deq2 = mn16 + code * s16,  r = x - deq2
 *   rs16 = fp16(max |r| / 127)
 *   rq   = clamp(rint(r / rs16), -127, 127)         (0 when rs16 == 0)
 * fp16() and rint() round to nearest, ties to even.  Keys must lie within
 * the fp16 range.  Layouts (row = (b * Hkv + h) * L_max + t):
 *   k          [B, Hkv, L_max, d] bf16 (input)
 *   codes      [row, d/4]     uint8: channel c in byte c/4, bits 2*(c%4)+{0,1}
 *   mn_scale   [row, d/32, 2] fp16 (mn16, s16)
 *   res        [row, d]       int8
 *   res_scale  [row, d/32]    fp16 (rs16)
 * Rows with t >= seq_lens[b] (seq_lens may be NULL) are not written.
 * d must be 64 or 128. */
FD_API int fd_quantize_keys(const void* k, const int32_t* seq_lens,
                     int B, int Hkv, int L_max, int d,
                     uint8_t* codes, void* mn_scale, int8_t* res, void* res_scale,
                     void* stream);

/* Bytes of workspace fd_decode_topdelta needs (0 when none). */
FD_API size_t fd_topdelta_workspace_size(int B, int Hq, int Hkv, int L_max, int d,
                                  int num_splits);

/* Top-delta sparse decode ([FFD] sections 3-6, Fig. 2), one fused pass per
 * chunk of the cache.  For each (b, query head):
 *   1. s~_j  = scale * <q, deq2_j>   for every cached token (2-bit body only)
 *   2. m^    = max of s~ over the anchors {0..n_sink-1} U {L-window..L-1}
 *   3. Sel   = { j : s~_j >= m^ - delta }       (delta = +inf keeps all)
 *   4. s_j   = scale * <q, deq2_j + deq8_j>     for j in Sel (int8 residual)
 *   5. out   = sum_{Sel} e^{s_j} v_j / sum_{Sel} e^{s_j}; lse over Sel.
 * Inputs are fd_quantize_keys' outputs for the same cache, plus
 *   q [B, Hq, d] bf16, v [B, Hkv, L_max, d] bf16, seq_lens [B] or NULL,
 *   delta >= 0 (may be +inf), n_sink >= 0, window >= 0.
 * Optional outputs for inspection (NULL to skip): sel_mask
 * [B, Hq, ceil(L_max/32)] uint32 (bit j%32 of word j/32 set when j is in
 * Sel) and sel_count [B, Hq] int32.  The residual and V of a token are read
 * only when some query head of its KV group selects a token in the same
 * 64-token tile.  L_max must be a multiple of 4 and B * Hkv * L_max at most
 * 2^31 - 1 (FD_ERR_UNSUPPORTED otherwise).  workspace:
 * fd_topdelta_workspace_size() bytes. */
FD_API int fd_decode_topdelta(const void* q, const uint8_t* codes, const void* mn_scale,
                       const int8_t* res, const void* res_scale, const void* v,
                       const int32_t* seq_lens,
                       int B, int Hq, int Hkv, int L_max, int d,
                       float scale, float delta, int n_sink, int window,
                       int num_splits,
                       void* out, int out_dtype, float* lse,
                       uint32_t* sel_mask, int32_t* sel_count,
                       void* workspace, size_t workspace_bytes, void* stream);

/* fd_decode_topdelta with one candidate set per KV group: steps 1-3 are
 * taken per query head as above, then every query head of a group (the
 * Hq / Hkv heads that read one KV head) attends, in steps 4-5, to the union
 * of the group's sets, Sel_group = U_g Sel_g, each with its own exact scores.
 * The pages define the rule per query ([FFD] section 3) and give no group
 * variant; this one reads no more bytes than the per-head rule (the tiles
 * whose residual and V are loaded are the same) and every head keeps at
 * least its own candidates.  sel_mask / sel_count report the attended set
 * (the same for every head of a group).  Arguments, layouts, workspace
 * (fd_topdelta_workspace_size) and errors are those of fd_decode_topdelta. */
FD_API int fd_decode_topdelta_group_union(const void* q, const uint8_t* codes, const void* mn_scale,
                                          const int8_t* res, const void* res_scale, const void* v,
                                          const int32_t* seq_lens,
                                          int B, int Hq, int Hkv, int L_max, int d,
                                          float scale, float delta, int n_sink, int window,
                                          int num_splits,
                                          void* out, int out_dtype, float* lse,
                                          uint32_t* sel_mask, int32_t* sel_count,
                                          void* workspace, size_t workspace_bytes, void* stream);

/* fp8 KV cache encoder ([KV8]).  For each cache row x (one token of one
 * head, d bf16 values), in IEEE binary32 arithmetic:
 *   s      = max_c |x_c| / 448
 *   code_c = e4m3(x_c / s)        (0 for every c when s == 0)
 * e4m3(): the OCP 8-bit float with 4 exponent bits (bias 7) and 3 mantissa
 * bits, no infinities, largest finite 448; round to nearest, ties to even,
 * magnitudes above 448 saturate to +-448.  The decoded value is
 * e4m3(code) * s, within 2^-4 |x| + 2^-10 s of x.  Layouts
 * (row = (b * H + h) * L_max + t):
 *   x       [B, H, L_max, d] bf16 (input)
 *   codes   [row, d] uint8 (output)
 *   scales  [row]    float32 (output)
 * Rows with t >= seq_lens[b] (seq_lens may be NULL) are not written.  Use
 * it for K and for V of the same cache (H = Hkv).  d must be 64 or 128. */
FD_API int fd_quantize_kv_fp8(const void* x, const int32_t* seq_lens,
                              int B, int H, int L_max, int d,
                              uint8_t* codes, float* scales, void* stream);

/* fd_num_splits / fd_decode_workspace_size for the fp8 decode entry points
 * (the planner counts the fp8 cache's bytes per tile). */
FD_API int fd_num_splits_fp8(int B, int Hq, int Hkv, int L_max, int d, int num_splits, int ragged);
FD_API size_t fd_decode_fp8_workspace_size(int B, int Hq, int Hkv, int L_max, int d,
                                           int num_splits, int ragged);

/* Split-KV decode ([FD] sections 1-2) over an fp8 cache written by
 * fd_quantize_kv_fp8: the result is the attention of q over the decoded rows
 * K~ = e4m3(k_codes) * k_scales, V~ = e4m3(v_codes) * v_scales (computed
 * with fp16 tensor-core products and fp32 accumulation).
 *   k_codes, v_codes    [B, Hkv, L_max, d] uint8
 *   k_scales, v_scales  [B, Hkv, L_max]    float32
 * All other arguments, outputs and the workspace contract are those of
 * fd_decode_dense, with fd_decode_fp8_workspace_size() for the workspace. */
FD_API int fd_decode_dense_fp8(const void* q, const uint8_t* k_codes, const float* k_scales,
                               const uint8_t* v_codes, const float* v_scales,
                               const int32_t* seq_lens,
                               int B, int Hq, int Hkv, int L_max, int d,
                               float scale, int num_splits,
                               void* out, int out_dtype, float* lse,
                               void* workspace, size_t workspace_bytes, void* stream);

/* The same over a paged fp8 cache ([FD] section 3): pages of 64 tokens,
 *   k_pages, v_pages              [num_pages, Hkv, 64, d] uint8 codes
 *   k_page_scales, v_page_scales  [num_pages, Hkv, 64] float32
 * page_table, seq_lens and the remaining arguments as fd_decode_paged
 * (workspace: fd_decode_fp8_workspace_size(..., L_max = max_pages * 64,
 * ragged = 1)). */
FD_API int fd_decode_paged_fp8(const void* q, const uint8_t* k_pages, const float* k_page_scales,
                               const uint8_t* v_pages, const float* v_page_scales,
                               const int32_t* page_table, int max_pages, int num_pages,
                               const int32_t* seq_lens, int page_size,
                               int B, int Hq, int Hkv, int d,
                               float scale, int num_splits,
                               void* out, int out_dtype, float* lse,
                               void* workspace, size_t workspace_bytes, void* stream);

/* fp4 KV cache encoder ([KV8] names an "FP4" cache; this format is this
 * library's definition).  For each cache row x (one token of one head) and
 * each 32-channel block b of it, in exact arithmetic:
 *   e_b   = the smallest integer in [-126, 127] with 6 * 2^e_b >= max |x|
 *           over the block (-126 for an all-zero block)
 *   code  = e2m1(x * 2^-e_b)
 * e2m1(): 1 sign, 2 exponent bits (bias 1), 1 mantissa bit, magnitudes
 * 0, 0.5, 1, 1.5, 2, 3, 4, 6, round to nearest with ties to the even code.
 * The decoded value is e2m1(code) * 2^e_b.  Layouts (row = (b*H + h)*L_max + t):
 *   x       [B, H, L_max, d] bf16 (input)
 *   codes   [row, d/2]  uint8: channel c in byte c/2, the low nibble for even c
 *   scales  [row, d/32] uint8: e_b + 127
 * Rows with t >= seq_lens[b] (seq_lens may be NULL) are not written; the
 * sign of a code rounded to zero follows x.  d must be 64 or 128.  This is
 * the KEY cache layout; the value cache uses fd_quantize_v_fp4. */
FD_API int fd_quantize_kv_fp4(const void* x, const int32_t* seq_lens,
                              int B, int H, int L_max, int d,
                              uint8_t* codes, uint8_t* scales, void* stream);

/* The same fp4 encoding for the VALUE cache, stored in token pairs (the layout
 * the P.V product of the decode reads without transposes).  Codes and scales
 * of every row are those fd_quantize_kv_fp4 computes; only the code layout
 * differs (pair p = tokens 2p, 2p + 1 of one head; Lp = (L_max + 1) / 2):
 *   codes   [B, H, Lp, d] uint8: byte (p, c) = code(2p+1, c) << 4 | code(2p, c)
 *   scales  [B, H, L_max, d/32] uint8: e_b + 127 (as fd_quantize_kv_fp4)
 * A pair whose first token is at or past seq_lens[b] is not written; a second
 * token past it writes code 0 and no scale byte.  To append a token to a
 * cache, encode its pair again from the two bf16 rows (a token at an even
 * position: with its partner still absent).  d must be 64 or 128. */
FD_API int fd_quantize_v_fp4(const void* x, const int32_t* seq_lens,
                             int B, int H, int L_max, int d,
                             uint8_t* codes, uint8_t* scales, void* stream);

/* fd_num_splits / fd_decode_workspace_size for the fp4 decode entry points. */
FD_API int fd_num_splits_fp4(int B, int Hq, int Hkv, int L_max, int d, int num_splits, int ragged);
FD_API size_t fd_decode_fp4_workspace_size(int B, int Hq, int Hkv, int L_max, int d,
                                           int num_splits, int ragged);

/* Split-KV decode ([FD] sections 1-2) over an fp4 cache: keys written by
 * fd_quantize_kv_fp4, values by fd_quantize_v_fp4; the attention of q over
 * the decoded rows (computed with fp16 tensor-core products and fp32
 * accumulation).
 *   k_codes             [B, Hkv, L_max, d/2]         uint8
 *   v_codes             [B, Hkv, (L_max + 1)/2, d]   uint8 (token pairs)
 *   k_scales, v_scales  [B, Hkv, L_max, d/32]        uint8
 * All other arguments, outputs and the workspace contract are those of
 * fd_decode_dense, with fd_decode_fp4_workspace_size() for the workspace. */
FD_API int fd_decode_dense_fp4(const void* q, const uint8_t* k_codes, const uint8_t* k_scales,
                               const uint8_t* v_codes, const uint8_t* v_scales,
                               const int32_t* seq_lens,
                               int B, int Hq, int Hkv, int L_max, int d,
                               float scale, int num_splits,
                               void* out, int out_dtype, float* lse,
                               void* workspace, size_t workspace_bytes, void* stream);

/* The same over a paged fp4 cache ([FD] section 3): pages of 64 tokens,
 *   k_pages                       [num_pages, Hkv, 64, d/2]  uint8 codes
 *   v_pages                       [num_pages, Hkv, 32, d]    uint8 codes (token pairs)
 *   k_page_scales, v_page_scales  [num_pages, Hkv, 64, d/32] uint8
 * page_table, seq_lens and the remaining arguments as fd_decode_paged
 * (workspace: fd_decode_fp4_workspace_size(..., L_max = max_pages * 64,
 * ragged = 1)). */
FD_API int fd_decode_paged_fp4(const void* q, const uint8_t* k_pages, const uint8_t* k_page_scales,
                               const uint8_t* v_pages, const uint8_t* v_page_scales,
                               const int32_t* page_table, int max_pages, int num_pages,
                               const int32_t* seq_lens, int page_size,
                               int B, int Hq, int Hkv, int d,
                               float scale, int num_splits,
                               void* out, int out_dtype, float* lse,
                               void* workspace, size_t workspace_bytes, void* stream);

/* Size of the fixed device scratch array used by fd_decode_dense_noalloc. */
#define FD_NOALLOC_SCRATCH_BYTES (4u << 20)

/* fd_decode_dense without a workspace argument, for callers that cannot
 * allocate device memory: for example a plug-in inside a host engine that
 * has reserved all device memory and exposes no allocator, or a decode loop
 * that must not call cudaMalloc/cudaFree because they can synchronise the
 * device.  The source pages have no counterpart of this entry point.
 *   - Arguments, layouts and results are those of fd_decode_dense.
 *   - Scratch comes from one static device array of FD_NOALLOC_SCRATCH_BYTES
 *     (4 MiB) inside the library, held by every GPU that loads the library
 *     until the process exits.  When the plan for these sizes needs more
 *     (fd_decode_workspace_size(B, Hq, Hkv, L_max, d, num_splits,
 *     seq_lens != NULL) > FD_NOALLOC_SCRATCH_BYTES) the call returns
 *     FD_ERR_WORKSPACE_TOO_SMALL and enqueues nothing.
 *   - The call allocates nothing.  Its first call on a device (with that
 *     device current) looks up the array's device address; make that first
 *     call before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents
 *     (nothing in it needs to start at zero: a call reads only what it wrote
 *     earlier in the same call).  Calls that overlap on the GPU, e.g. on two
 *     streams at once, race on it. */
FD_API int fd_decode_dense_noalloc(const void* q, const void* k, const void* v,
                                   const int32_t* seq_lens,
                                   int B, int Hq, int Hkv, int L_max, int d,
                                   float scale, int num_splits,
                                   void* out, int out_dtype, float* lse, void* stream);

/* Fault injection for tests of the time-out path; not for production use.
 * Applies to the bf16 dense and paged decode (fd_decode_dense,
 * fd_decode_paged, their unified-max variants and fd_decode_dense_noalloc)
 * launched afterwards from this process:
 *   wait_limit_ns  > 0: the time limit of every pipeline wait (default 2 s;
 *                  0 restores it)
 *   withhold_tile  >= 0: the producer of every chunk issues no copy and no
 *                  arrival for that tile index of the chunk (-1: off), so the
 *                  consumers' wait for it runs out.
 * A kernel whose wait runs out records FD_ERR_DEVICE_TIMEOUT in the device
 * status word, stops using its pipeline, lets every copy it started land
 * and exits; the call's out and lse are then undefined.  The GPU stays
 * usable.  Always returns FD_OK. */
FD_API int fd_debug_inject_wait_timeout(unsigned long long wait_limit_ns, int withhold_tile);

/* Synchronises `stream`, then reports the device status word of the current
 * device: FD_ERR_DEVICE_TIMEOUT, FD_ERR_BAD_PAGE_TABLE, FD_ERR_INVALID_ARG (a
 * seq_lens entry outside [0, L_max]; the kernels clamped it) or FD_OK, in
 * that order of precedence (FD_ERR_CUDA if the synchronisation itself
 * failed).  clear != 0 resets the word afterwards. */
FD_API int fd_device_status(int clear, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FD_H */
