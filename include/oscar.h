/*
 * oscar.h — C ABI of liboscar.so, the GB300 (sm_103a) implementation of the
 * OSCAR INT2 KV-cache decode path.
 *
 * The method (cited by page title and section):
 *   [news]  OSCAR news article (m.kljzs.com mirror), paragraph on the online
 *           path: sink and recent tokens stay BF16, the long middle history is
 *           rotated INT2; the oldest recent token is rotated, clipped,
 *           quantized and packed (4 codes per byte) into the INT2 history; at
 *           decode an INT2 kernel (unpack, scale/zero restore, float
 *           accumulation) and a BF16 kernel (sink/recent) produce partial
 *           results that an online-softmax merge combines.
 *   [tai]   "Together AI 開源 OSCAR" (news.chathome.org), "OSCAR 的不同之處":
 *           R_K = U_Q·H·P_br, R_V = U_S·H·P_br; "服務系統": first 64 tokens and
 *           last 256 tokens in BF16, paged-attention compatible.
 *   [notes] "OSCAR — 离线转个方向，把 KV Cache 压到 2-bit" (estelledc notes),
 *           "核心要点" item 3: layout [BF16 sink] || [INT2 history] || [BF16
 *           recent]; "案例 2": c_K ~ 0.96, c_V ~ 0.92.
 *
 * Conventions (row vectors): x_rot = x · R.  Keys/values in the INT2 history
 * are stored rotated; a query is rotated by its kv head's R_K before it meets
 * them (q_rot · k_rot = q · k), and the history part of the output is rotated
 * back by R_V^T.  INT2 is asymmetric per group of `group` consecutive rotated
 * channels: lo = c·min, hi = c·max, zero = bf16(lo), scale = bf16((hi-lo)/3),
 * code = clamp(rint((x - zero)/scale), 0, 3), code 0 if scale == 0; code i of
 * a row sits at bits 2·(i mod 4) of byte i/4.  Dequantized value:
 * zero + code·scale.
 *
 * Regions of a request with seq_len T (current token included) and history
 * end h (sink <= h <= T): positions [0, sink) and [h, T) are read from the
 * BF16 pool, positions [sink, h) from the INT2 pool.  h is passed per call so
 * that a demotion of position h may run concurrently with attention that
 * still reads it from BF16.
 *
 * Memory: every pointer is a device pointer owned by the caller, except the
 * layout/pool/partials descriptors themselves, which are host structs read
 * during the call only.  The library allocates no memory on any call below.
 * Every call is asynchronous on the CUDA stream passed as `stream`
 * (a cudaStream_t; NULL = legacy default stream) and returns after enqueueing.
 *
 * Errors: host-side argument checks return OSCAR_ERR_INVALID_ARG or
 * OSCAR_ERR_UNSUPPORTED before anything is enqueued; a failed launch returns
 * OSCAR_ERR_CUDA.  oscar_last_error_string() gives a one-line reason (thread
 * local).  Device-side checks (page ids outside [0, n_pages), seq_len or
 * hist_end out of range, a pipeline wait that gave up) never trap: the
 * offending page/request is skipped, a bit is set in a device status word,
 * and oscar_get_device_status() reads and clears it.
 */
#ifndef OSCAR_H
#define OSCAR_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define OSCAR_API __attribute__((visibility("default")))
#else
#define OSCAR_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    OSCAR_OK = 0,
    OSCAR_ERR_INVALID_ARG = 1,
    OSCAR_ERR_UNSUPPORTED = 2,
    OSCAR_ERR_CUDA = 3,
    OSCAR_ERR_DEVICE_FLAG = 4
} oscar_status_t;

/* Device status bits reported by oscar_get_device_status(). */
#define OSCAR_DEV_BAD_INT2_PAGE 0x1   /* INT2 page id outside [0, n_pages) */
#define OSCAR_DEV_BAD_BF16_PAGE 0x2   /* BF16 page id outside [0, n_pages) */
#define OSCAR_DEV_BAD_LENGTH    0x4   /* seq_len/hist_end/position out of range (clamped) */
#define OSCAR_DEV_WAIT_TIMEOUT  0x8   /* a bounded pipeline wait gave up */

/*
 * Model/cache shape shared by every call.
 *   head_dim   D, must be 128.
 *   n_kv_heads Hkv, 1..64.
 *   gqa        G = query heads per kv head, one of 1, 2, 4, 8 (Hq = G·Hkv).
 *   page_size  tokens per page: 16, 32 or 64, and sink % page_size == 0.
 *   group      INT2 quantization group along the rotated channels: 32, 64, 128.
 *   sink       BF16 sink tokens ([tai] "服務系統": 64).
 *   recent     BF16 recent tokens ([tai] "服務系統": 256); informative only,
 *              the per-request hist_end decides the regions.
 */
typedef struct {
    int32_t head_dim;
    int32_t n_kv_heads;
    int32_t gqa;
    int32_t page_size;
    int32_t group;
    int32_t sink;
    int32_t recent;
    /*
     * Codebook of the 2-bit codes on a group's normalised axis u = (x - zero) / scale, where
     * zero and scale are the uniform quantizer's (zero = bf16(c·min), scale = bf16((c·max -
     * c·min) / 3)).  All four zero: the uniform levels 0, 1, 2, 3 (code = clamp(rint(u), 0, 3)).
     * Otherwise four finite, strictly increasing levels lv (a non-uniform codebook such as a
     * Lloyd-Max one, OSCAR news article, closing paragraph): code = the number of fp32 midpoints
     * (lv[k] + lv[k+1]) * 0.5 at or below u (code 0 for NaN or scale 0), restored as
     * zero + lv[code] · scale.  levels_k for keys, levels_v for values.  A non-uniform codebook is
     * served by oscar_quantize_rotated (with levels_k), oscar_demote, oscar_decode_attention and
     * oscar_decode_attention_noalloc (their INT2 part on the CUDA cores); the tensor-core-only
     * paths (oscar_decode_attention_fused, oscar_demote_range) return OSCAR_ERR_UNSUPPORTED.
     */
    float levels_k[4];
    float levels_v[4];
} oscar_layout_t;

/*
 * Paged INT2 pool of one layer (device memory, caller-owned):
 *   codes_k, codes_v : uint8 [n_pages][page_size][n_kv_heads][head_dim/4]
 *   scale_k, zero_k, scale_v, zero_v : bf16 bits [n_pages][page_size][n_kv_heads][head_dim/group]
 * All six base addresses must be 16-byte aligned.
 */
typedef struct {
    uint8_t *codes_k;
    uint8_t *codes_v;
    uint16_t *scale_k;
    uint16_t *zero_k;
    uint16_t *scale_v;
    uint16_t *zero_v;
    int32_t n_pages;
} oscar_int2_pool_t;

/* Paged BF16 pool of one layer: k, v bf16 bits [n_pages][page_size][n_kv_heads][head_dim], 16-byte aligned. */
typedef struct {
    uint16_t *k;
    uint16_t *v;
    int32_t n_pages;
} oscar_bf16_pool_t;

/*
 * Flash-decoding partials (device scratch, caller-owned), base-2 domain:
 *   m   fp32 [batch][Hq][n_splits + 1]   running max of sm_scale·logit·log2(e)
 *   l   fp32 [batch][Hq][n_splits + 1]   sum of 2^(t - m)
 *   acc fp32 [batch][Hq][n_splits + 1][head_dim]  sum of 2^(t - m)·value
 * Slots 0..n_splits-1 are history splits in ascending token order (values in
 * the ROTATED basis); slot n_splits is the BF16 partial (unrotated).  An empty
 * slot has m = -inf, l = 0, acc = 0.  n_splits in 1..1024.
 */
typedef struct {
    float *m;
    float *l;
    float *acc;
    int32_t n_splits;
} oscar_partials_t;

/* Number of floats in m, l and acc for a batch (sizes for the caller's allocation). */
OSCAR_API size_t oscar_partials_ml_floats(const oscar_layout_t *layout, int32_t batch, int32_t n_splits);
OSCAR_API size_t oscar_partials_acc_floats(const oscar_layout_t *layout, int32_t batch, int32_t n_splits);

/*
 * A split count that fills the GPU for `batch` requests whose longest history
 * spans max_hist_tokens tokens: each split is computed by a cluster of up to 8
 * CTAs that combine their results before writing the split's partial, one or
 * two more clusters per request compute the BF16 window (two for batch 1 with
 * 8 kv heads, four heads each).  With A the number of such clusters the current
 * device keeps resident at once (from sm_count when no device is visible) and
 * W the window clusters per request, the count is A / batch - W (one wave)
 * when batch·(1 + W) <= A, else 4·A / batch - W (about four waves, so that
 * requests of different lengths finish evenly).  Layouts that the tensor-core
 * kernel does not take (other kv-head counts, a non-uniform codebook) run one
 * 4-warp CTA per (split, kv head): about 16·sm_count / (batch·n_kv_heads) splits.
 * At least one 16-token history tile per split, clamped to [1, 1024].
 */
OSCAR_API int32_t oscar_suggest_splits(const oscar_layout_t *layout, int32_t batch, int32_t max_hist_tokens,
                             int32_t sm_count);

/*
 * Demotion ([news] online path: "rotate / clip / quantize / pack"; [notes]
 * "核心要点" item 3).  For each i < n, request b = req_idx[i] and position
 * p = positions[i]: for every kv head h, the BF16 key row at
 * (bf16_page_table[b·max_pages_per_req + p/ps], p % ps, h) is rotated by
 * R_K[h] (fp32 accumulation, one fused multiply-add per term in ascending
 * input-channel order), clipped with c_K, quantized and packed into the INT2
 * pool at (int2_page_table[b·max_pages_per_req + p/ps], p % ps, h); the value
 * row likewise with R_V[h] and c_V.
 *   R_K, R_V       fp32 [n_kv_heads][head_dim][head_dim], row-major R[i][j].
 *                  R_V may be NULL when the value rotation is folded into the
 *                  model's projections ([notes] "核心要点" item 3: the value
 *                  rotation can be absorbed into the projection weights): the
 *                  values then arrive already rotated and are quantized as
 *                  stored (y = x; merge them with oscar_merge(R_V = NULL)).
 *   batch          rows of both page tables ([batch][max_pages_per_req]).
 *   req_idx, positions  int32 [n] device arrays; an entry with req_idx outside
 *                  [0, batch) or a position outside the page table is skipped
 *                  and flagged (OSCAR_DEV_BAD_LENGTH).
 *   rotated_out    NULL or fp32 [n][2][n_kv_heads][head_dim]: the rotated
 *                  rows (index 0 = K, 1 = V) before quantization.
 * n may be large (bulk demotion of a whole prompt); n = 0 is a no-op.
 * Rows that two entries of (req_idx, positions) map to the same INT2 slot
 * race; callers demote each position once.
 */
OSCAR_API oscar_status_t oscar_demote(const oscar_layout_t *layout,
                            const oscar_bf16_pool_t *src, const int32_t *bf16_page_table,
                            const oscar_int2_pool_t *dst, const int32_t *int2_page_table,
                            int32_t max_pages_per_req, int32_t batch,
                            const int32_t *req_idx, const int32_t *positions, int32_t n,
                            const float *R_K, const float *R_V, float c_K, float c_V,
                            float *rotated_out, void *stream);

/*
 * Bulk demotion of position ranges on the tensor cores (the step that fills the
 * INT2 history after prefill: [news] online path "rotate / clip / quantize /
 * pack"; [notes] "核心要点" item 3).  For each request b, every position p in
 * [pos_begin[b], pos_end[b]) is demoted as oscar_demote would, every kv head, K
 * and V, with one difference: the rotation x · R runs on the tensor cores as
 * x · R_hi + x · R_lo with R_hi = bf16(R), R_lo = bf16(R − R_hi) and fp32
 * accumulation, so each rotated element lies within 2^-14 · ||x||_2 of the exact
 * product (oscar_demote's fp32 chain lies closer); codes, scale and zero are the
 * quantizer's output on these rotated rows, bit for bit.
 *   pos_begin, pos_end  int32 [batch] device arrays; a range with
 *                  pos_begin < 0, pos_end < pos_begin or pos_end beyond the page
 *                  table is skipped and flagged (OSCAR_DEV_BAD_LENGTH); an empty
 *                  range demotes nothing.
 *   rotated_out    NULL or fp32 [int2 pool n_pages][page_size][2][n_kv_heads]
 *                  [head_dim], indexed like the destination INT2 slot (index 0 =
 *                  K, 1 = V): the rotated rows before quantization; slots not
 *                  demoted are not written.
 * Other arguments as for oscar_demote (R_V may be NULL: values stored as they
 * are, exactly); both pools' arrays and rotated_out must
 * be 16-byte aligned.  Positions that two requests map to the same INT2 slot
 * race.
 */
OSCAR_API oscar_status_t oscar_demote_range(const oscar_layout_t *layout,
                                  const oscar_bf16_pool_t *src, const int32_t *bf16_page_table,
                                  const oscar_int2_pool_t *dst, const int32_t *int2_page_table,
                                  int32_t max_pages_per_req, int32_t batch,
                                  const int32_t *pos_begin, const int32_t *pos_end,
                                  const float *R_K, const float *R_V, float c_K, float c_V,
                                  float *rotated_out, void *stream);

/*
 * The codec alone: quantize n fp32 rows x_rot [n][head_dim] that are already
 * rotated, with clip ratio `clip`, into codes [n][head_dim/4] and bf16
 * scale/zero [n][head_dim/group].  Bit-exact contract: given the same fp32
 * input rows, codes, scale and zero equal the definition above bit for bit.
 */
OSCAR_API oscar_status_t oscar_quantize_rotated(const oscar_layout_t *layout, const float *x_rot, int32_t n,
                                      float clip, uint8_t *codes, uint16_t *scale, uint16_t *zero,
                                      void *stream);

/*
 * Query rotation q_rot = q · R_K[h / gqa] for every query head h of every
 * request ("q pre-rotated by R_K" so that q_rot · k_rot = q · k, [tai]
 * "OSCAR 的不同之處").  q: bf16 [batch][Hq][head_dim]; q_rot: fp32, same shape;
 * fp32 fused multiply-add chain in ascending input-channel order.
 */
OSCAR_API oscar_status_t oscar_rotate_q(const oscar_layout_t *layout, const uint16_t *q, const float *R_K,
                              int32_t batch, float *q_rot, void *stream);

/*
 * Decode attention partials for one layer ([news] INT2 kernel + BF16 kernel).
 *   q        bf16 [batch][Hq][head_dim], unrotated (meets the BF16 rows)
 *   q_rot    fp32 [batch][Hq][head_dim] = q · R_K (meets the INT2 history)
 *   bf16_pool / bf16_page_table   sink and recent rows
 *   int2_pool / int2_page_table   history rows
 *   page tables: int32 [batch][max_pages_per_req], logical page -> physical page
 *   seq_len  int32 [batch] T (current token included), 1 <= T <= max_pages_per_req·page_size
 *   hist_end int32 [batch] h, sink <= h <= T (values outside are clamped and flagged)
 *   sm_scale softmax scale (1/sqrt(head_dim) for standard attention)
 * Writes every slot of `partials` for every (request, query head): the
 * history [sink, h) is cut into partials->n_splits contiguous splits of whole
 * 16-token tiles (tile i = positions 16i..16i+15): with first = sink/16 and
 * n = ceil(h/16) - first, split s covers tiles [first + floor(s·n/S),
 * first + floor((s+1)·n/S)) clipped to [sink, h); the BF16 partial covers
 * [0, sink) ∪ [h, T).  When the tensor-core kernels support the layout (1, 2,
 * 4 or 8 kv heads) both parts are computed by one launch, whose first cluster
 * per request (first two for batch 1 with 8 kv heads, four kv heads each) takes
 * the BF16 window.
 */
OSCAR_API oscar_status_t oscar_decode_attention(const oscar_layout_t *layout,
                                      const uint16_t *q, const float *q_rot,
                                      const oscar_bf16_pool_t *bf16_pool, const int32_t *bf16_page_table,
                                      const oscar_int2_pool_t *int2_pool, const int32_t *int2_page_table,
                                      int32_t max_pages_per_req,
                                      const int32_t *seq_len, const int32_t *hist_end, int32_t batch,
                                      float sm_scale, const oscar_partials_t *partials, void *stream);

/*
 * oscar_decode_attention with the query rotation folded in: takes the unrotated q
 * and R_K (fp32 [n_kv_heads][head_dim][head_dim], as for oscar_rotate_q) instead
 * of q_rot.  Each cluster of history CTAs rotates the queries of its request, one
 * kv head per CTA, from R_K staged in shared memory, and shares the rows across
 * the cluster; the arithmetic is oscar_rotate_q's (one fused multiply-add per
 * term, ascending input channel), so the partials are bit for bit those of
 * oscar_rotate_q followed by oscar_decode_attention.  Requires a layout the
 * tensor-core kernels take (n_kv_heads 1, 2, 4 or 8); otherwise returns
 * OSCAR_ERR_UNSUPPORTED and the caller uses the two calls.  No method page
 * describes this fusion; it removes one launch per layer.
 *
 * Optional per-step demotion ([news] online path: the token leaving the recent
 * window is demoted): with demote_pos non-NULL (int32 [batch], -1 = none),
 * position demote_pos[b] of request b is demoted for every kv head, K with R_K and
 * c_K, V with R_V and c_V, exactly as oscar_demote would (same arithmetic, same
 * bytes), by the CTAs that compute the BF16 window.  The position must be at or
 * after hist_end[b] and before seq_len[b] (this launch still reads it from BF16);
 * otherwise it is skipped and OSCAR_DEV_BAD_LENGTH is set.  demote_pos NULL: c_K,
 * c_V are ignored.
 *
 * R_V NULL (the value rotation folded into the projections): the demotion
 * stores values as they are and the merge does not rotate back.
 *
 * Optional merge: with out or out_f32 non-NULL the call also runs oscar_merge (same
 * bits; lse optional) as a second launch.  Without merge_counters that launch waits
 * for the whole decode grid (programmatic dependent launch when launch overlap is
 * on).  With merge_counters (int32 [2·batch], all zero; the call leaves them zero)
 * each cluster of request b adds 1 to merge_counters[b] once its partial slot is
 * written, and the merge of request b starts as soon as the count is complete
 * (acquire load, bounded wait: OSCAR_DEV_WAIT_TIMEOUT), without waiting for the
 * rest of the grid; merge_counters[batch + b] counts the merge CTAs that have
 * passed, and the last one resets both.  Calls that may run concurrently must not
 * share merge_counters.
 *
 * Optional dynamic scheduling: with tile_counters (int32 [2·batch], all zero; the
 * call leaves them zero) the history is not cut into fixed splits: the CTAs of
 * request b take units of 64 tokens of [sink, hist_end[b]) in turn from the shared
 * count tile_counters[b] (tile_counters[batch + b] counts the CTAs that are done;
 * the last one resets both), so that CTAs that run faster take more.  Each history
 * slot then holds the partial of whichever units its CTAs took: only the merged
 * result is defined (the same up to fp32 rounding order).  The per-step demotion,
 * if any, then runs in the first history CTAs of the request (one kv head each),
 * whose delay the shared units absorb; its bytes are the same.  Calls that may run
 * concurrently must not share tile_counters.
 */
OSCAR_API oscar_status_t oscar_decode_attention_fused(const oscar_layout_t *layout, const uint16_t *q,
                                                      const float *R_K, const oscar_bf16_pool_t *bf16_pool,
                                                      const int32_t *bf16_page_table,
                                                      const oscar_int2_pool_t *int2_pool,
                                                      const int32_t *int2_page_table, int32_t max_pages_per_req,
                                                      const int32_t *seq_len, const int32_t *hist_end,
                                                      int32_t batch, float sm_scale,
                                                      const oscar_partials_t *partials,
                                                      const int32_t *demote_pos, const float *R_V, float c_K,
                                                      float c_V, uint16_t *out, float *out_f32, float *lse,
                                                      int32_t *merge_counters, int32_t *tile_counters,
                                                      void *stream);

/*
 * Decode attention partials of a batch whose requests share the INT2 history pages
 * of a prefix [sink, prefix_end) (a radix prefix cache: "Together AI 開源 OSCAR",
 * section 服務系統, paged and prefix-cache compatible; OSCAR news article, the
 * paragraphs on prefix-cache hits).  The shared prefix is read once per kv head for
 * every request, on the 5th-generation tensor cores (all requests' query rows of a
 * kv head meet the same keys: one 128-row operand per 128 / gqa requests), and cut
 * into prefix_splits token splits written to partial slots 0 .. prefix_splits - 1;
 * each request's own history [prefix_end, hist_end) goes to slots prefix_splits ..
 * S - 1 and its BF16 window [0, sink) ∪ [hist_end, seq_len) to slot S
 * (S = partials->n_splits).  Merge with oscar_merge as usual.
 *   q, q_rot, pools, page tables, max_pages_per_req, seq_len, hist_end, sm_scale:
 *       as oscar_decode_attention
 *   prefix_end     multiple of 16, sink < prefix_end <= max_pages_per_req·page_size
 *                  (a multiple of 64 keeps the suffix's 64-token units page-aligned);
 *                  every request's hist_end must be >= prefix_end and its INT2 page
 *                  table row must hold the same pages for [0, prefix_end) (the prefix
 *                  is read through request 0's row); neither is checked
 *   prefix_splits  1 <= prefix_splits < S
 *   tile_counters  NULL, or int32 [2·batch] zero: the suffix histories taken in dynamic
 *                  64-token units (as oscar_decode_attention_fused)
 * Needs the tensor-core layout (1, 2, 4 or 8 kv heads, uniform codebook) and group
 * 128 (else OSCAR_ERR_UNSUPPORTED).
 */
OSCAR_API oscar_status_t oscar_decode_attention_shared_prefix(
    const oscar_layout_t *layout, const uint16_t *q, const float *q_rot, const oscar_bf16_pool_t *bf16_pool,
    const int32_t *bf16_page_table, const oscar_int2_pool_t *int2_pool, const int32_t *int2_page_table,
    int32_t max_pages_per_req, const int32_t *seq_len, const int32_t *hist_end, int32_t batch, float sm_scale,
    int32_t prefix_end, int32_t prefix_splits, const oscar_partials_t *partials, int32_t *tile_counters,
    void *stream);

/*
 * The two halves of oscar_decode_attention, for callers that run them on two
 * streams so that they overlap (they write disjoint slots of `partials`):
 * _history writes the history slots 0..S-1 from the INT2 pool and q_rot;
 * _window writes the BF16 slot S (sink + recent) from the BF16 pool and q.
 * Arguments as for oscar_decode_attention.  Each half writes the same bits as
 * the combined call.
 */
OSCAR_API oscar_status_t oscar_decode_attention_history(const oscar_layout_t *layout, const float *q_rot,
                                                        const oscar_int2_pool_t *int2_pool,
                                                        const int32_t *int2_page_table, int32_t max_pages_per_req,
                                                        const int32_t *seq_len, const int32_t *hist_end,
                                                        int32_t batch, float sm_scale,
                                                        const oscar_partials_t *partials, void *stream);
OSCAR_API oscar_status_t oscar_decode_attention_window(const oscar_layout_t *layout, const uint16_t *q,
                                                       const oscar_bf16_pool_t *bf16_pool,
                                                       const int32_t *bf16_page_table, int32_t max_pages_per_req,
                                                       const int32_t *seq_len, const int32_t *hist_end,
                                                       int32_t batch, float sm_scale,
                                                       const oscar_partials_t *partials, void *stream);

/*
 * Online-softmax merge ([news] "online softmax merge"): per (request, query
 * head), combine history slots 0..S-1 in ascending order, rotate that
 * accumulator back by R_V[h / gqa]^T, add the BF16 slot S, divide by the
 * total weight.  The fixed fp32 order (equal partials give equal bits):
 *   M = max m_i over non-empty slots (l_i > 0), w_i = 2^(m_i - M);
 *   L = fma(l_i, w_i, L); A_d = fma(acc_i,d, w_i, A_d) for i = 0..S-1;
 *   A'_j = fma-chain over i of A_i·R_V[j][i]; then slot S with w_S; o = A'/L,
 * with 2^x computed by Cody–Waite reduction and a degree-7 Taylor polynomial
 * (not the hardware approximation).
 *   R_V  fp32 [n_kv_heads][head_dim][head_dim], or NULL: no slot is rotated
 *        back (an all-BF16 cache, or values stored in the rotated basis
 *        because R_V is folded into the projections; o is then in that basis).
 *   out      NULL or bf16 [batch][Hq][head_dim]: o rounded to nearest even.
 *   out_f32  NULL or fp32 [batch][Hq][head_dim]: o before that rounding.
 *            At least one of out / out_f32 must be given.
 *   lse      NULL or fp32 [batch][Hq]: natural log-sum-exp of sm_scale·logits.
 */
OSCAR_API oscar_status_t oscar_merge(const oscar_layout_t *layout, const oscar_partials_t *partials,
                           const float *R_V, int32_t batch, uint16_t *out, float *out_f32, float *lse,
                           void *stream);

/*
 * Comparison kernel: decode attention over an all-BF16 paged cache (no INT2
 * history, no rotation), same split-K structure.  Positions [0, T) are cut
 * into partials->n_splits splits of whole 16-token tiles by the rule of
 * oscar_decode_attention (with first = 0) into slots 0..S-1; slot S is
 * written empty.  Merge with oscar_merge(..., R_V = NULL, ...).
 */
OSCAR_API oscar_status_t oscar_bf16_decode_attention(const oscar_layout_t *layout, const uint16_t *q,
                                           const oscar_bf16_pool_t *pool, const int32_t *page_table,
                                           int32_t max_pages_per_req, const int32_t *seq_len,
                                           int32_t batch, float sm_scale,
                                           const oscar_partials_t *partials, void *stream);

/*
 * Decode attention and merge in one call with no caller scratch (this entry
 * point has no counterpart on the pages; it exists for callers that cannot
 * allocate device memory, e.g. code inside a host framework that owns every
 * device allocation and offers no workspace, or a loop that must never call
 * an allocator).  Same inputs and outputs as oscar_decode_attention followed
 * by oscar_merge, with n_splits history splits; the partials live in a
 * library-owned device array of OSCAR_NOALLOC_SCRATCH_BYTES per device, part
 * of the library's device code and held until the process exits.  This call
 * makes no cudaMalloc/cudaFree.  CUDA may load the library's device code, and
 * with it reserve the array, only when a device first uses it (lazy module
 * loading): make one call on each device at initialisation, outside any loop
 * and before any stream capture; later calls reserve nothing.  Each call looks
 * the array's device address up again (a host-side query), so a device reset
 * between calls leaves no stale address.  Limit:
 * 2*ceil64(batch*Hq*(n_splits+1)) + batch*Hq*(n_splits+1)*head_dim floats
 * must fit, else OSCAR_ERR_INVALID_ARG.  All calls share the array: calls
 * whose GPU work overlaps race and must be serialised by the caller.  Every
 * slot is written before it is read, so no state carries over between calls.
 */
#define OSCAR_NOALLOC_SCRATCH_BYTES (4u << 20)
OSCAR_API oscar_status_t oscar_decode_attention_noalloc(
    const oscar_layout_t *layout, const uint16_t *q, const float *q_rot, const oscar_bf16_pool_t *bf16_pool,
    const int32_t *bf16_page_table, const oscar_int2_pool_t *int2_pool, const int32_t *int2_page_table,
    int32_t max_pages_per_req, const int32_t *seq_len, const int32_t *hist_end, int32_t batch, float sm_scale,
    int32_t n_splits, const float *R_V, uint16_t *out, float *out_f32, float *lse, void *stream);

/*
 * Launch overlap between consecutive decode kernels (programmatic dependent
 * launch), process-wide, off by default; applies to calls made after it returns.
 * No method page describes it: it is a launch policy of this library.
 *
 * When on, oscar_rotate_q, oscar_decode_attention_history (tensor-core path),
 * oscar_decode_attention, oscar_decode_attention_fused and oscar_merge launch
 * their kernels so that each may
 * start while the kernel before it in the same stream is still running.  Before
 * it waits for that kernel, a kernel only reads what a decode step treats as
 * fixed: R_K / R_V, the INT2 and BF16 pools, the page tables, seq_len and
 * hist_end.  Everything else (q, q_rot, the partials, the outputs) is read or
 * written after the wait.  The caller therefore guarantees that the kernel
 * preceding one of these calls in the stream does not write R_K, R_V, a pool,
 * a page table, seq_len or hist_end; oscar_demote, for example, must be followed
 * by an event or another kernel before the decode kernels that read its pages,
 * or overlap must be off.  With overlap off every launch waits for the previous
 * kernel to complete, as CUDA streams do by default.
 *
 * Returns OSCAR_OK; oscar_get_launch_overlap() reads the current setting (0/1).
 */
OSCAR_API oscar_status_t oscar_set_launch_overlap(int32_t enabled);
OSCAR_API int32_t oscar_get_launch_overlap(void);

/* Read and clear the device status word of the current device (synchronizes `stream`). */
OSCAR_API oscar_status_t oscar_get_device_status(int32_t *status_bits, void *stream);

/* One-line reason for the last non-OK status returned on this thread. */
OSCAR_API const char *oscar_last_error_string(void);

/* Library version, e.g. "0.1.0". */
OSCAR_API const char *oscar_version(void);

#ifdef __cplusplus
}
#endif

#endif /* OSCAR_H */
