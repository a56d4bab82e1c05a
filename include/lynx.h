/*
 * lynx.h -- C ABI of the GB300 (sm_103a) Lynx progressive KV quantizer.
 *
 * The method: "Lynx: the KV cache does not have to arrive whole" (aigenapps
 * reading of Han et al.). Section 3 "The quantizer" defines the per-page
 * encoder (page-level normalisation; chunk-wise outlier isolation with C = 32;
 * an alpha-law log map onto 127 levels with sign-aware mapping; the +7
 * round-half-down bias and the 4-bit anchor / 4-bit residual cut). Section 4
 * "Speculation at the communication boundary" defines the two decoders: the
 * anchor stream alone is the draft cache, and the residual refines the cache
 * to the full reconstruction. The fused decode attention follows the
 * "KV-cache quantization" explainer (aicassindra), "Middle row" and
 * "Bottom-right": the compact cache is read as is and expanded only in
 * registers inside Q.K^T, softmax and the weighted sum over V.
 *
 * Conventions shared by every call
 *  - Every pointer argument marked "device" is CUDA device memory owned by the
 *    caller; the library allocates nothing and keeps no pointer after a call.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). Every
 *    compute call is asynchronous on that stream; its status reports host-side
 *    argument checks and launch errors only.
 *  - Device pointers must be 16-byte aligned (LYNX_ERR_ALIGN otherwise).
 *  - head_dim must be 128 and tokens a multiple of 256 (LYNX_ERR_SHAPE).
 *  - No call traps, asserts or spins on the device. Errors found on the
 *    device (a page-table entry outside the page pool, a context length
 *    outside [0, max_pages*256]) set bits in *dev_err (when given) and the
 *    affected work is skipped or clamped.
 *
 * Numeric contract of the encoder (both this library and any conforming
 * encoder produce identical bytes): fp32 arithmetic, each operation rounded to
 * nearest, no fused multiply-add:
 *   stage 1  mn = min x, rng = max x - mn (a zero extreme taken as +0),
 *            inv_r = rng > 0 ? 1/rng : 0, u = (x - mn) * inv_r   (valid tokens only)
 *   stage 2  per 32-token chunk: sum = stride-halving pairwise tree over the 32
 *            slots (+16, +8, +4, +2, +1; absent slots hold +0); mean = sum/n_c;
 *            mu = fp16 nearest(mean); v = u - mu; s = fp16 rounded toward
 *            +inf(max |v|); inv_s = s > 0 ? 1/s : 0; w = v * inv_s
 *   stage 3  q = #{k in 1..63 : |w| >= T_k},
 *            T_k = fp32 nearest(((1+alpha)^((k-1/2)/63) - 1)/alpha), alpha = 255;
 *            c = q for w >= 0, c = -max(q, 1) for w < 0      (c in -63..63)
 *   stage 4  b = c + 7; A = floor(b/16) in -4..4; r = b - 16A in 0..15.
 * Statistics fp32 cannot carry (the pages are silent; the reading taken): a
 *   NaN among a channel's valid values stores the channel's page minimum and
 *   range as the quiet NaN 0x7FC00000 (any NaN range is stored as that
 *   pattern); when the range or its reciprocal is not finite (a NaN or
 *   infinite input, a range beyond fp32, a subnormal range whose reciprocal
 *   overflows) every u of the channel is 0, so its chunk means and scales are
 *   0 and its codes 0 (anchor 0, residual 7).
 * Decoders: Lv[k] = fp16 nearest(((1+alpha)^(k/63) - 1)/alpha), k = 0..64;
 *   anchor-only code 16A, full code 16A + r - 7 (magnitudes above 64, which
 *   the encoder never writes, saturate at Lv[64]);
 *   x = mn + rng * (mu + s * sgn(code) * Lv[|code|]).
 */
#ifndef LYNX_H
#define LYNX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LYNX_OK = 0,
    LYNX_ERR_NULL = 1,        /* a required pointer is NULL */
    LYNX_ERR_SHAPE = 2,       /* a size is negative, inconsistent or not supported by the layout */
    LYNX_ERR_ALIGN = 3,       /* a device pointer is not 16-byte aligned */
    LYNX_ERR_UNSUPPORTED = 4, /* a legal but unsupported configuration (e.g. group size > 32) */
    LYNX_ERR_WORKSPACE = 5,   /* workspace smaller than lynx_decode_attn_workspace() */
    LYNX_ERR_CUDA = 6         /* a CUDA launch or query failed */
} lynx_status;

typedef enum { LYNX_OUT_BF16 = 0, LYNX_OUT_F32 = 1 } lynx_out_dtype;
typedef enum { LYNX_MODE_ANCHOR = 0, LYNX_MODE_FULL = 1 } lynx_mode;

/* Device-error bits written (OR-ed) into *dev_err by lynx_decode_attn and lynx_quantize_append. */
#define LYNX_DEVERR_PAGE 1u   /* a page-table entry outside [0, tokens/256) */
#define LYNX_DEVERR_CTX 2u    /* a context length outside [0, max_pages*256] */
#define LYNX_DEVERR_TIMEOUT 4u /* a wait (a bulk copy, a tensor-core completion, a barrier between the
                                  kernel's warps) ran past its limit, or the kernel could not start
                                  (its shared-memory window was not where it needs it); the outputs
                                  the wait guarded are not valid */

/*
 * One quantized tensor (K or V): a view of caller-owned device memory.
 * The page pool of a paged cache is the `tokens` axis: physical page p is
 * rows [256p, 256p + 256). A sub-range of layers is passed as a view with
 * offset pointers and a smaller `layers`.
 *   anchor      [layers][kv_heads][tokens][head_dim/2] u8: two 4-bit anchors
 *               per byte, channel 2i in the low nibble, two's complement
 *   residual    same shape: two 4-bit residuals per byte; may be NULL where
 *               only the anchor stream exists (anchor-only calls)
 *   page_meta   [layers][kv_heads][tokens/256][2][head_dim] fp32: page minimum,
 *               page range, per channel
 *   chunk_meta  [layers][kv_heads][tokens/256][8][2][head_dim] fp16 bits: chunk
 *               mean, chunk scale, per channel
 */
typedef struct {
    int32_t layers, kv_heads, tokens, head_dim;
    uint8_t *anchor;
    uint8_t *residual;
    float *page_meta;
    uint16_t *chunk_meta;
} lynx_qkv;

/*
 * Encode a bf16 tensor page by page (section 3, all four stages, and the 4+4
 * cut). One call per tensor: K and V take one call each.
 *   x_bf16      device, [layers][kv_heads][tokens][128] bf16 (layout of `out`)
 *   page_valid  device, [tokens/256] int32 valid-token counts in 0..256 for
 *               each page (the ragged last page), shared by every layer and
 *               head; NULL = every page full. Statistics use valid tokens only;
 *               invalid tokens store code 0 (anchor 0, residual 7). Counts
 *               outside 0..256 are clamped.
 *   out         planes and metadata written; residual must be non-NULL.
 * The call has no device-error word: a page copy that never lands (every wait
 * in the kernel is bounded) ends the kernel early without a report, leaving
 * later pages unwritten; lynx_quantize_append reports the same event.
 * Returns LYNX_ERR_UNSUPPORTED when layers * kv_heads * tokens / 256 exceeds
 * 2^31 / 256 pages (the kernel addresses rows with 32-bit tile coordinates)
 * or the driver provides no tensor-map encoder.
 */
lynx_status lynx_quantize_pages(const void *x_bf16, const int32_t *page_valid, const lynx_qkv *out,
                                void *stream);

/*
 * Quantize-on-append for the decode tail. The explainer's "Top row" compresses
 * each token's K and V as they are produced (quantize-on-write); the Lynx
 * encoder works on whole 256-token pages (section 3), so a page that is still
 * growing is re-encoded whole from its bf16 staging copy each time tokens are
 * added. This call does that for n tails at once: tail i is encoded into
 * physical page phys_page[i] of every layer and KV head of `out`, with
 * valid[i] valid tokens (statistics over those tokens only; the others store
 * code 0), exactly as lynx_quantize_pages encodes a page with that count.
 *   tail_bf16  device, [n][layers][kv_heads][256][128] bf16
 *   phys_page  device, [n] int32 destination pages in [0, tokens/256); an
 *              entry outside is skipped and sets LYNX_DEVERR_PAGE in *dev_err
 *   valid      device, [n] int32 valid-token counts (clamped to 0..256)
 *   out        the pool: planes and metadata of every layer and KV head
 *              (residual non-NULL); only the destination pages are written
 *   dev_err    device or NULL, one uint32 (LYNX_DEVERR_PAGE, and LYNX_DEVERR_TIMEOUT
 *              when a tail's copy into the kernel never landed)
 * Tails naming the same physical page race on it: pass distinct pages.
 * Returns LYNX_ERR_UNSUPPORTED under the same limits as lynx_quantize_pages
 * (for the n tails' pages and for the pool's).
 */
lynx_status lynx_quantize_append(const void *tail_bf16, const int32_t *phys_page, const int32_t *valid,
                                 int32_t n, const lynx_qkv *out, uint32_t *dev_err, void *stream);

/*
 * Anchor-only reconstruction, the draft cache of section 4 (decoding begins
 * as soon as the anchor planes are in, its tokens marked as drafts): every
 * element decoded from its anchor with the residual taken at its centre
 * (code 16A).
 *   in   planes and metadata (residual may be NULL)
 *   out  device, [layers][kv_heads][tokens][128] in `dt` (bf16 nearest or fp32)
 */
lynx_status lynx_dequant_anchor(const lynx_qkv *in, void *out, lynx_out_dtype dt, void *stream);

/*
 * Residual refinement in place (section 4: once the residual planes are in,
 * the cache is brought to the full quantization): overwrites the dense cache that lynx_dequant_anchor wrote with the
 * full reconstruction from anchor and residual planes (code 16A + r - 7). The
 * planes are not modified. `inout` has the layout and dtype of the
 * lynx_dequant_anchor output; in->residual must be non-NULL.
 */
lynx_status lynx_refine_residual(const lynx_qkv *in, void *inout, lynx_out_dtype dt, void *stream);

/*
 * Workspace bytes lynx_decode_attn needs for this batch shape on the current
 * device (split-K partials). Returns 0 for invalid sizes.
 */
size_t lynx_decode_attn_workspace(int32_t batch, int32_t q_heads, int32_t max_pages);

/*
 * One decode step of attention over one layer of the quantized paged cache,
 * dequantizing in registers (explainer, "Bottom-right"):
 *   out[b][h] = sum_t softmax_t(sm_scale * q[b][h] . K[t]) V[t],  t < ctx_lens[b],
 * where K, V are the anchor-only (LYNX_MODE_ANCHOR) or full (LYNX_MODE_FULL)
 * reconstructions, token t of request b lives in physical page
 * page_table[b][t/256], row t%256, and query head h reads KV head
 * h / (q_heads / kv_heads). The pages of each (request, KV head) are split
 * across CTAs (split-K) and the partial (max, sum, output) triples are merged
 * with a log-sum-exp combine.
 *   q_bf16      device, [batch][q_heads][128] bf16
 *   k, v        quantized K and V of the whole pool; `layer` selects the layer;
 *               residual planes required in FULL mode
 *   page_table  device, [batch][max_pages] int32
 *   ctx_lens    device, [batch] int32; 0 gives an output of zeros
 *   out         device, [batch][q_heads][128] fp32
 *   scores      device or NULL, [batch][q_heads][max_pages*256] fp32: the scaled
 *               logits sm_scale * q.K for t < ctx, -inf for the rest
 *   workspace   device, ws_bytes >= lynx_decode_attn_workspace(batch, q_heads, max_pages)
 *   dev_err     device or NULL, one uint32 (LYNX_DEVERR_* bits OR-ed in)
 * q_heads must be a multiple of kv_heads with a group size of at most 32.
 * Groups of up to 16 query heads run on a tensor-core kernel whose level
 * table sits at a fixed shared-memory address; on a device whose dynamic
 * shared-memory window does not start 1 KiB into the CTA's shared memory
 * (measured once per device) the call returns LYNX_ERR_UNSUPPORTED.
 */
lynx_status lynx_decode_attn(const void *q_bf16, const lynx_qkv *k, const lynx_qkv *v, int32_t layer,
                             const int32_t *page_table, const int32_t *ctx_lens, int32_t batch,
                             int32_t q_heads, int32_t max_pages, float sm_scale, lynx_mode mode,
                             float *out, float *scores, void *workspace, size_t ws_bytes,
                             uint32_t *dev_err, void *stream);

/*
 * Decode attention without a caller-provided workspace. (The Lynx reading has
 * no counterpart for this call: it serves callers that cannot allocate device
 * memory, such as a serving engine whose pool has already claimed all free
 * memory for the KV cache, a plugin that is handed only its input and output
 * buffers, or a latency-critical path where cudaMalloc, which may synchronise
 * the device, is not allowed.)
 * Same arguments and results as lynx_decode_attn, minus the workspace: the
 * split-K partials go to a fixed array of LYNX_NOALLOC_SCRATCH_BYTES inside
 * the library, which every GPU that loads the library holds until the process
 * exits. The call allocates nothing.
 *  - Argument checks are those of lynx_decode_attn, in the same order. Then,
 *    without launching, it returns LYNX_ERR_WORKSPACE when the split-K plan of
 *    this shape (batch, q_heads, kv_heads, max_pages on this device) needs more
 *    than LYNX_NOALLOC_SCRATCH_BYTES; lynx_decode_attn_workspace(batch,
 *    q_heads, max_pages), the largest need over every kv_heads, is an upper
 *    bound of it.
 *  - The first call on each device looks up the array's device address once
 *    (a host-side query); make that first call before any stream capture.
 *  - Every call on a device shares the one array, and it keeps whatever the
 *    previous call left there (nothing in it needs to start at zero: each
 *    partial is written before it is read). Calls that overlap on the GPU,
 *    e.g. on two streams at once, race on it; serialise them.
 */
#define LYNX_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
lynx_status lynx_decode_attn_noalloc(const void *q_bf16, const lynx_qkv *k, const lynx_qkv *v, int32_t layer,
                                     const int32_t *page_table, const int32_t *ctx_lens, int32_t batch,
                                     int32_t q_heads, int32_t max_pages, float sm_scale, lynx_mode mode,
                                     float *out, float *scores, uint32_t *dev_err, void *stream);

/*
 * Workspace bytes lynx_verify_attn needs for this shape on the current device
 * (split-K partials of every draft position). Returns 0 for invalid sizes.
 */
size_t lynx_verify_attn_workspace(int32_t batch, int32_t draft, int32_t q_heads, int32_t max_pages);

/*
 * Multi-token verify attention over one layer of the quantized paged cache.
 * Section 4 of the Lynx reading drafts tokens on the anchor-only cache and,
 * once the residuals have refined it, verifies the drafted positions against
 * the full cache; this is the attention of that verify pass: `draft` query
 * positions per request (at most 64), the last `draft` tokens of each context
 * being the drafted ones, causal within the block:
 *   out[b][i][h] = sum_{t < n_bi} softmax_t(sm_scale * q[b][i][h] . K[t]) V[t],
 *   n_bi = ctx_lens[b] - draft + i + 1  (rows with n_bi <= 0 give zeros),
 * with K, V, the page table and GQA mapping as in lynx_decode_attn (FULL:
 * the refined reconstruction; ANCHOR: the draft one). The cache is decoded on
 * chip into fp16 hi/lo tiles and multiplied on the tensor cores with three
 * products per pair, keeping fp32-level accuracy; reconstructed values must
 * lie inside the fp16 range (|x| < 65504).
 *   q_bf16      device, [batch][draft][q_heads][128] bf16
 *   out         device, [batch][draft][q_heads][128] fp32
 *   workspace   device, ws_bytes >= lynx_verify_attn_workspace(batch, draft, q_heads, max_pages)
 *   dev_err     device or NULL, one uint32 (LYNX_DEVERR_* bits OR-ed in)
 */
lynx_status lynx_verify_attn(const void *q_bf16, const lynx_qkv *k, const lynx_qkv *v, int32_t layer,
                             const int32_t *page_table, const int32_t *ctx_lens, int32_t batch, int32_t draft,
                             int32_t q_heads, int32_t max_pages, float sm_scale, lynx_mode mode, float *out,
                             void *workspace, size_t ws_bytes, uint32_t *dev_err, void *stream);

/* Human-readable name of a status. Never NULL. */
const char *lynx_status_string(lynx_status s);

/*
 * Variants and ablations of the quantizer, for quality studies. Section 7 of
 * the Lynx reading ("What the paper does not establish") lists what was never
 * measured: other splits (INT6 and INT2 splits are future work), the chunk
 * size (only C = 32; smaller chunks are claimed to reduce error), and which
 * stage of the bundle earns its gain over uniform INT4. A lynx_variant selects:
 *   chunk          C: 16, 32 or 64 tokens per chunk
 *   anchor_bits    a in 1..6, residual_bits r in 1..4, a + r <= 8: codes have
 *                  2^(a+r-1) - 1 levels (4 + 4: the page's 127), the bias is
 *                  2^(r-1) - 1 (+7 at r = 4), anchor-only decoding takes 2^r A
 *   alpha          > 0: the alpha-law map; 0: its limit, the linear grid
 *   flags          LYNX_VAR_* below, each switching one stage off:
 *                  NO_PAGE_NORM (u = x), NO_CHUNK_ISOLATION (mean = scale = 1/2,
 *                  i.e. w = 2u - 1), NO_BIAS (a plain floor cut), NO_SIGN_AWARE
 *                  (c = -q for w < 0)
 *   uniform_bits   > 0 (1..8): instead of the method, the uniform comparator: per
 *                  (page, channel) min and range, code = floor((x - mn) *
 *                  ((2^b - 1) / rng) + 1/2) in fp32, decoded mn + code rng / (2^b - 1);
 *                  with flags = LYNX_VAR_UNIFORM_PER_TOKEN the grid is per token
 *                  (min and range over its 128 channels; page_meta is then zeros)
 * The default configuration {32, 4, 4, 255, 0, 0} encodes exactly as
 * lynx_quantize_pages.
 */
#define LYNX_VAR_NO_PAGE_NORM 1u
#define LYNX_VAR_NO_CHUNK_ISOLATION 2u
#define LYNX_VAR_NO_BIAS 4u
#define LYNX_VAR_NO_SIGN_AWARE 8u
#define LYNX_VAR_UNIFORM_PER_TOKEN 16u
typedef struct {
    int32_t chunk;
    int32_t anchor_bits;
    int32_t residual_bits;
    float alpha;
    uint32_t flags;
    int32_t uniform_bits;
} lynx_variant;

/*
 * Encode n tensors of `tokens` x 128 bf16 values (tokens % 256 == 0) page by
 * page with variant *v, in one pass. Every output is optional (NULL skips it);
 * all are device memory, 16-byte aligned, caller-owned:
 *   x_bf16      [n][tokens][128] bf16
 *   codes       [n][tokens][128] int16: the signed code c (uniform: the grid code)
 *   anchor      [n][tokens][128] int8: A = floor((c + bias) / 2^r) (method only)
 *   residual    [n][tokens][128] uint8: c + bias - 2^r A (method only)
 *   page_meta   [n][tokens/256][2][128] fp32 (min, range)
 *   chunk_meta  [n][tokens/256][256/C][2][128] fp16 bits (mean, scale; method only)
 *   err         [n][tokens/256][3] fp64 per page: sum x^2, sum (x_anchor - x)^2,
 *               sum (x_full - x)^2 (uniform: the last two are equal); the
 *               reconstructions are evaluated in fp32
 *   x_anchor    [n][tokens][128] fp32: the anchor-only reconstruction
 *   x_full      [n][tokens][128] fp32: the full reconstruction (uniform: both
 *               hold the comparator's reconstruction)
 * Returns LYNX_ERR_SHAPE / LYNX_ERR_UNSUPPORTED for sizes or knobs outside
 * the ranges above, LYNX_ERR_ALIGN for misaligned pointers.
 */
lynx_status lynx_quantize_variant(const void *x_bf16, int32_t n, int32_t tokens, const lynx_variant *v,
                                  int16_t *codes, int8_t *anchor, uint8_t *residual, float *page_meta,
                                  uint16_t *chunk_meta, double *err, float *x_anchor, float *x_full,
                                  void *stream);

/*
 * Decode attention over a DENSE fp32 cache, for quality studies: the Lynx
 * reading's evaluation (section 5) measures the error of the attention
 * output, so a reconstruction (x_anchor / x_full above) is scored by running
 * this on it and on the original values. Not part of the method's path.
 *   q_bf16  [batch][q_heads][128] bf16, one query per request
 *   k, v    [kv_heads][tokens][128] fp32, shared by every request, 16-byte aligned
 *   out     [batch][q_heads][128] fp32
 * out[b][h] = sum_t softmax_t(sm_scale q[b][h] . k[g][t]) v[g][t] with
 * g = h / (q_heads / kv_heads), fp32 arithmetic. Device memory, caller-owned,
 * asynchronous on `stream`. Returns LYNX_ERR_SHAPE unless q_heads is a
 * multiple of kv_heads and 1 <= tokens <= 49152 (batch or q_heads 0: no-op).
 */
lynx_status lynx_dense_attn(const void *q_bf16, const float *k, const float *v, int32_t batch, int32_t q_heads,
                            int32_t kv_heads, int32_t tokens, float sm_scale, float *out, void *stream);

/*
 * Diagnostics (no counterpart in the method: they expose the library's own
 * tables and its stage-3 code path so that tests can compare them with an
 * independent implementation).
 *   lynx_host_tables  host call, no GPU needed: thr[64] (thr[0] = 0) and
 *                     lv[65] fp16 bits, exactly as the kernels use them
 *   lynx_level_codes  device: codes[i] = stage-3 code (-63..63) of w[i], for
 *                     finite |w| < 2 (stage 2 only produces |w| <= 1 + 2^-23;
 *                     larger magnitudes are outside the encoder's domain and
 *                     their codes are unspecified)
 */
void lynx_host_tables(float *thr, uint16_t *lv);
lynx_status lynx_level_codes(const float *w, int64_t n, int8_t *codes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* LYNX_H */
