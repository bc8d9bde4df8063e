/*
 * decattn.h - C ABI of the B300 (sm_103a) decode-attention library.
 *
 * One GPU, one process. Every entry point enqueues work on the caller's CUDA
 * stream and returns at once; none synchronises, none allocates device
 * memory, none falls back to the CPU or to another library. All tensor
 * pointers are DEVICE pointers to dense row-major arrays in the layouts
 * stated below, owned by the caller, and must stay valid until the enqueued
 * work completes. bf16 tensors are passed as 16-bit storage (decattn_bf16).
 *
 * Sources (the web pages this library follows):
 *   [SKILL]  "Mla Analysis" skill page: "Tensor Shapes (DeepSeek-V3 defaults)"
 *            (layouts Q [B,H,S,D], K/V [B,T,H,D], Z [B,T,K], QPE [B,H,S,P],
 *            KPE [B,T,P]), "Absorption Trick (FlashMLA)" (scores Qz Z^T,
 *            values (softmax Z) Wv, decompression in a separate kernel).
 *   [FIGHT]  "Why MLA and MTP Fight Each Other" post, summary table
 *            (MHA / GQA / MQA / MLA) and the MTP discussion (several new
 *            tokens per step).
 *   [QA]     "MHA vs GQA" Q&A, section 1 (query heads sharing a KV head).
 *   [LESSON] "MQA, GQA & MLA" lesson, Concept (contiguous groups; MLA caches
 *            a latent plus a decoupled RoPE part).
 *
 * Conventions shared by all calls
 *   b   sequences, s new tokens per sequence (1..1024), seqlens[i] = keys of
 *       sequence i INCLUDING its s new tokens (a device int32[b]); token r of
 *       the s new ones attends to keys 0 .. seqlens[i]-s+r (causal among the
 *       new tokens, aligned to the end); seqlens[i] = 0 gives a zero output
 *       row and LSE = -inf; 0 < seqlens[i] < s is undefined (the kernels
 *       treat the missing keys as absent).
 *   max_seqlen  host-side upper bound of seqlens (sizes the launch grid).
 *   scale       softmax scale applied to the whole score.
 *   lse         optional float[b, heads, s] natural-log log-sum-exp of the
 *               scaled scores (NULL to skip).
 *   workspace   caller-allocated scratch of at least *_workspace_size() bytes
 *               (16-byte aligned); its content on entry does not matter.
 *   Return: DECATTN_OK or an error status; on an argument error nothing is
 *   launched. Device-side faults detected by the kernels (a bounded wait that
 *   ran out, a page index outside the pool) are recorded in a device error
 *   word and reported by decattn_check_errors().
 *   Launch: every kernel is launched as a programmatic dependent of the
 *   kernel before it on the stream (CUDA programmatic dependent launch): its
 *   CTAs may start while that kernel finishes, and wait for its completion
 *   and memory before reading any argument tensor. The one exception is the
 *   weight of mla_absorb_q / mla_out_proj (w_uk / w_uv), whose first tiles
 *   are requested before that wait: the weight must not be written by the
 *   kernel launched immediately before on the same stream (writes by earlier
 *   kernels, copies or other streams ordered by events are fine).
 */
#ifndef DECATTN_H
#define DECATTN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t decattn_bf16; /* bfloat16 bit pattern */

enum decattn_status {
  DECATTN_OK = 0,
  DECATTN_ERR_INVALID_ARG = 1, /* null pointer, Hq % Hkv != 0, s outside 1..1024, page_size != 64, ... */
  DECATTN_ERR_UNSUPPORTED = 2, /* head dim / (k, p) without a compiled instance */
  DECATTN_ERR_WORKSPACE = 3,   /* workspace missing or too small */
  DECATTN_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
  DECATTN_ERR_TIMEOUT = 5      /* a device-side bounded wait ran out (from decattn_check_errors) */
};

/* Cache description shared by both attention forms.
 *   paged = 0: contiguous cache, sequence i owns rows [i*capacity, (i+1)*capacity)
 *              of the cache tensor ([b, capacity, ...]).
 *   paged = 1: page pool [num_pages, page_size, ...]; token j of sequence i
 *              lives in page block_table[i*max_pages + j/page_size], row
 *              j % page_size. block_table is a DEVICE int32[b, max_pages];
 *              entries past a sequence's last page are never read. */
typedef struct decattn_kv {
  int paged;
  int capacity;                /* contiguous only: token slots per sequence */
  const int32_t* block_table;  /* paged only */
  int max_pages;               /* paged only: columns of block_table */
  int page_size;               /* paged only: must be 64 */
  int num_pages;               /* paged only: pages in the pool */
} decattn_kv;

/* Text for a status code (static storage). */
const char* decattn_status_string(int status);

/* ------------------------------------------------------------------------
 * Grouped-head decode attention: MHA (Hkv = Hq), GQA, MQA (Hkv = 1).
 * [QA] section 1; [FIGHT] summary table; [LESSON] contiguous groups: query
 * head j reads KV head j / (Hq / Hkv).
 *   q    [b, Hq, s, d] bf16 ([SKILL] Q layout)
 *   k, v contiguous [b, capacity, Hkv, d] bf16 ([SKILL] K, V layout) or
 *        paged [num_pages, 64, Hkv, d]
 *   out  [b, Hq, s, d] bf16 (round-to-nearest-even)
 *   d in {64, 128, 256}. Split-KV: the context is cut into chunks processed
 *   in parallel and merged by log-sum-exp in a second kernel.
 */
size_t gqa_decode_workspace_size(int b, int s, int hq, int hkv, int d, int max_seqlen);
int gqa_decode(const decattn_bf16* q, const decattn_bf16* k, const decattn_bf16* v, decattn_kv kv,
               const int32_t* seqlens, int max_seqlen, int b, int s, int hq, int hkv, int d, float scale,
               decattn_bf16* out, float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Grouped-head decode with value rows narrower than key rows: the same
 * computation, arguments, layouts, errors and workspace rules as gqa_decode,
 * with the width split in two.
 *   q    [b, Hq, s, dk]; k contiguous [b, capacity, Hkv, dk] or paged
 *        [num_pages, 64, Hkv, dk]; v likewise with dv; out [b, Hq, s, dv].
 *   Compiled (dk, dv): (64, 64), (128, 128), (256, 256) and (192, 128), the
 *   last for the expanded MLA form ([SKILL] Cost Models - FlashAttention:
 *   keys carry d + p = 192 values, values d = 128), run with Hkv = Hq = h.
 *   Other pairs return DECATTN_ERR_UNSUPPORTED.
 */
size_t gqa_decode_dv_workspace_size(int b, int s, int hq, int hkv, int dk, int dv, int max_seqlen);
int gqa_decode_dv(const decattn_bf16* q, const decattn_bf16* k, const decattn_bf16* v, decattn_kv kv,
                  const int32_t* seqlens, int max_seqlen, int b, int s, int hq, int hkv, int dk, int dv, float scale,
                  decattn_bf16* out, float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Grouped-head decode over an FP8 KV cache ([LESSON] Concept, the
 * deployment paragraph: the cache may be quantised; the pages otherwise
 * assume BF16). k and v hold OCP FP8 E4M3 bytes (1 sign, 4 exponent bits
 * with bias 7, 3 mantissa bits; subnormals; S.1111.111 is NaN; no
 * infinities), in the layouts of gqa_decode with one byte per value, and
 * stand for k_scale * K8 and v_scale * V8 (per-tensor scales, finite and
 * > 0). Queries, outputs, workspace, errors and everything else as
 * gqa_decode; d in {64, 128, 256}. Cache values are widened exactly: for
 * d >= 128 in registers to float16 (the MMAs then take the query and the
 * softmax weights as float16: exact for query values of magnitude 2^-14 ..
 * 65504), for d = 64 to bf16 in shared memory. The key scale multiplies the
 * softmax scale and the value scale the output. Cache rows past each
 * sequence's end are never used (NaN bytes there are harmless).
 */
size_t gqa_decode_fp8_workspace_size(int b, int s, int hq, int hkv, int d, int max_seqlen);
int gqa_decode_fp8(const decattn_bf16* q, const uint8_t* k, const uint8_t* v, decattn_kv kv, const int32_t* seqlens,
                   int max_seqlen, int b, int s, int hq, int hkv, int d, float scale, float k_scale, float v_scale,
                   decattn_bf16* out, float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Expanded MLA, cache decompression ([SKILL] Absorption Trick: the keys and
 * values the latent cache stands for; Cost Models - FlashAttention; Regime
 * Selection). For every cache row m < rows and head j < h:
 *   k_out[m, j, 0:d]   = z[m, :] @ w_uk[j]^T      (w_uk [h, d, k])
 *   k_out[m, j, d:d+p] = k_pe[m, :]               (shared RoPE part)
 *   v_out[m, j, :]     = z[m, :] @ w_uv[j]        (w_uv [h, k, d])
 *   z [rows, k], k_pe [rows, p] (the latent cache, contiguous [b*capacity]
 *   rows or a paged pool of num_pages*64 rows: the result keeps the row
 *   order, so the same block table addresses it), k_out [rows, h, d+p],
 *   v_out [rows, h, d]; all bf16, fp32 accumulation, bf16 output (round to
 *   nearest even). Compiled for d = 128, p = 64, k a multiple of 64 up to
 *   512 (else DECATTN_ERR_UNSUPPORTED). Pointers 16-byte aligned. Tensor-core
 *   (tcgen05) GEMM. gqa_decode_dv with Hkv = Hq = h, dk = d + p, dv = d then
 *   runs the expanded attention.
 */
int mla_decompress_kv(const decattn_bf16* z, const decattn_bf16* k_pe, const decattn_bf16* w_uk,
                      const decattn_bf16* w_uv, int rows, int h, int d, int k, int p, decattn_bf16* k_out,
                      decattn_bf16* v_out, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Log-sum-exp merge of two attention results over disjoint key sets of the
 * same query rows ([SKILL] MLAvar6+ Design: older keys in latent form,
 * recent keys decompressed, joined into one softmax):
 *   lse = log(exp(lse_a) + exp(lse_b))
 *   out = exp(lse_a - lse) * out_a + exp(lse_b - lse) * out_b
 *   out_a, out_b, out [rows, d] bf16 (out may alias out_a or out_b);
 *   lse_a, lse_b [rows] float (natural log; -inf = that side saw no key);
 *   lse [rows] float or NULL. Rows where both sides are -inf get out = 0,
 *   lse = -inf; an empty side's out values are never used. d a multiple of 8,
 *   bf16 pointers 16-byte aligned.
 */
int attn_merge_lse(const decattn_bf16* out_a, const float* lse_a, const decattn_bf16* out_b, const float* lse_b,
                   int rows, int d, decattn_bf16* out, float* lse, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Absorbed MLA, step 1: query absorption ([SKILL] Absorption Trick, score
 * line: Q K^T = (Q Wk^T) Z^T = Qz Z^T).
 *   qz[b, j, r, :] = scale * q_nope[b, j, r, :] @ w_uk[j]
 *   q_nope [b, h, s, d], w_uk [h, d, k], qz [b, h, s, k], all bf16; fp32
 *   accumulation, bf16 output. seqlens may be NULL; where given, rows of
 *   sequences with seqlens[i] == 0 are written as zeros. scale is an output
 *   multiplier (normally 1). d, k multiples of 8, s * b <= 65535 * 64.
 */
int mla_absorb_q(const decattn_bf16* q_nope, const decattn_bf16* w_uk, decattn_bf16* qz, const int32_t* seqlens,
                 int b, int s, int h, int d, int k, float scale, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Absorbed MLA, step 2: latent attention over the latent cache ([SKILL]
 * Absorption Trick; Tensor Shapes: Z [B,T,K], KPE [B,T,P] shared by all
 * heads; [LESSON] decoupled RoPE part). For each sequence all h*s query rows
 * (row = head*s + token) share every latent tile:
 *   score_m = scale * (<qz_row, z_m> + <q_pe_row, k_pe_m>)
 *   o_lat_row = sum_m softmax(score)_m z_m
 *   qz   [b, h, s, k] bf16 (output of mla_absorb_q)
 *   q_pe [b, h, s, p] bf16
 *   z    contiguous [b, capacity, k] or paged [num_pages, 64, k] bf16
 *   k_pe contiguous [b, capacity, p] or paged [num_pages, 64, p] bf16
 *   o_lat [b, h, s, k] bf16; lse [b, h, s] float or NULL.
 *   Compiled instances (k, p): (512, 64) and (64, 16). Pointers 16-byte
 *   aligned. Tensor-core (tcgen05) kernel with TMA tile loads, split over
 *   the context (a chunk count planned from b, s, h and max_seqlen) and
 *   merged by a second kernel.
 */
size_t mla_decode_workspace_size(int b, int s, int h, int k, int max_seqlen);
int mla_decode(const decattn_bf16* qz, const decattn_bf16* q_pe, const decattn_bf16* z, const decattn_bf16* k_pe,
               decattn_kv kv, const int32_t* seqlens, int max_seqlen, int b, int s, int h, int k, int p,
               float scale, decattn_bf16* o_lat, float* lse, void* workspace, size_t workspace_bytes,
               cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Absorbed MLA, step 3: output decompression, done as a separate kernel
 * ([SKILL] Absorption Trick, value line: (softmax(A) Z) Wv).
 *   out[b, j, r, :] = scale * o_lat[b, j, r, :] @ w_uv[j]
 *   o_lat [b, h, s, k], w_uv [h, k, d], out [b, h, s, d], all bf16.
 *   seqlens and scale as in mla_absorb_q.
 */
int mla_out_proj(const decattn_bf16* o_lat, const decattn_bf16* w_uv, decattn_bf16* out, const int32_t* seqlens,
                 int b, int s, int h, int k, int d, float scale, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Grouped-head decode that allocates nothing and takes no workspace.
 * The pages have no counterpart: this is a convenience for callers that
 * cannot allocate device memory - an engine whose allocator already holds
 * nearly all of HBM, a plug-in host that exposes no device allocator, a
 * loop that cannot afford cudaMalloc's implicit synchronisation.
 * Same arguments, layouts, results and errors as gqa_decode, minus the
 * workspace: the split partials live in one fixed array of
 * DECATTN_NO_ALLOC_SCRATCH_BYTES in the library's device image, which every
 * GPU that loads the library holds until the process exits.
 *   - Returns DECATTN_ERR_WORKSPACE, launching nothing, when the split plan
 *     needs more than DECATTN_NO_ALLOC_SCRATCH_BYTES
 *     (gqa_decode_workspace_size(...) > the limit).
 *   - The first call on a device (with that device current) looks up the
 *     array's device address (cudaGetSymbolAddress); make that first call
 *     before any stream capture on the device.
 *   - All calls on a device share the one array and it keeps the last
 *     call's contents (no call relies on them). Calls that overlap on the
 *     GPU (other streams, other host threads) race on it: serialise them.
 *   - Calls no cudaMalloc, cudaFree or allocating library routine.
 */
#define DECATTN_NO_ALLOC_SCRATCH_BYTES ((size_t)16 << 20) /* 16 MiB */
int gqa_decode_no_alloc(const decattn_bf16* q, const decattn_bf16* k, const decattn_bf16* v, decattn_kv kv,
                        const int32_t* seqlens, int max_seqlen, int b, int s, int hq, int hkv, int d, float scale,
                        decattn_bf16* out, float* lse, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Diagnostics.
 * decattn_check_errors: synchronises `stream`, reads and clears the device
 * error word of the current device; returns DECATTN_ERR_TIMEOUT if a bounded
 * wait ran out, DECATTN_ERR_INVALID_ARG if a page index was outside the pool,
 * DECATTN_ERR_CUDA on a CUDA error, else DECATTN_OK. There is ONE error word
 * per device, shared by every stream and host thread: it collects the faults
 * of all calls on that device since it was last cleared, whichever stream they
 * ran on, and the first decattn_check_errors to read it (on any stream) reports
 * and clears them. Only work ordered before the synchronised stream's point is
 * sure to have landed in it; to attribute a fault to one call, run that call
 * alone (or synchronise the other streams first) before checking.
 * decattn_set_wait_limit_ns: limit of every device-side wait (0 = default,
 * 2 s). decattn_set_forced_splits: 0 = let the planner choose the number of
 * context chunks; n > 0 forces n (for split-invariance tests); it also
 * changes the workspace sizes returned afterwards.
 * decattn_last_num_splits: number of chunks the last attention call used (0:
 * the tensor-core grouped-head kernel's balanced split, whose pieces are
 * planned on the device from the actual lengths).
 * decattn_set_grouped_kernel: which grouped-head kernel gqa_decode and
 * gqa_decode_dv run (diagnostics and tests; 0 = automatic, the default).
 * 1 = the split-KV kernels (16-row tiles, context split over CTAs, combine);
 * 2 = the tensor-core kernel (tcgen05, 128 query rows per CTA; the context cut
 * into chunks planned from max_seqlen, or, when the work items are fewer than
 * the SMs, into pieces balanced over one wave from the actual lengths, merged
 * by a combine kernel) where the widths allow ((dk, dv) in
 * {(128, 128), (192, 128), (256, 256)}). Automatic takes the tensor-core
 * kernel for (dk, dv) = (192, 128) at any row count, for (256, 256) from 24
 * and for (128, 128) from 32 query rows per KV head, over a bf16 or (d = 128
 * or 256) an FP8 cache. Results agree within rounding.
 * decattn_test_force_timeout: when nonzero, the next mla_decode and gqa_decode
 * kernels wait once on a barrier that nothing signals, with a 1 ms limit, so that
 * the timeout path runs; the kernels then wind down (no new copies, their own
 * copies in flight waited for, Tensor Memory freed) and report
 * DECATTN_ERR_TIMEOUT through decattn_check_errors. Their outputs are not
 * valid then. Test use only.
 */
int decattn_check_errors(cudaStream_t stream);
void decattn_set_wait_limit_ns(unsigned long long ns);
void decattn_set_forced_splits(int nsplit);
int decattn_last_num_splits(void);
void decattn_test_force_timeout(int on);
void decattn_set_grouped_kernel(int mode);

#ifdef __cplusplus
}
#endif

#endif /* DECATTN_H */
