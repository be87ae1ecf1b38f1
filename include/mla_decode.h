/*
 * mla_decode.h -- C ABI of the GB300 (sm_103a) MLA paged-decode library.
 *
 * One decode step of a Multi-head Latent Attention layer, in three calls:
 *
 *   mla_decode_attend  : bf16 absorbed queries over a paged fp8 latent KV
 *                        cache -> split-KV partials (o, lse)
 *   mla_merge_splits   : LSE merge of the partials -> latent
 *   mla_value_gate     : absorbed W_UV projection fused with the sigmoid gate
 *                        -> o_proj's input
 *
 * Sources (vLLM API pages):
 *   - vllm.models.kimi_k3.amd.specialized_decode.runtime.mla: attend,
 *     m1c_inputs, post (the decode split, the cache as one 576-byte row per
 *     token, the padded query, the partials and their merge);
 *   - vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.mla.value:
 *     MlaValue, MlaGate, value_bmm (W_UV and the gate).
 *
 * Conventions shared by every call
 *   - Every pointer is a device pointer owned by the caller, unless stated.
 *     The library never allocates, frees or synchronises.  Each call checks
 *     its arguments on the host, enqueues its kernel(s) on `stream` (a
 *     cudaStream_t; NULL = the legacy default stream) and returns.
 *   - Argument errors return MLA_ERR_INVALID / MLA_ERR_UNSUPPORTED before
 *     anything is launched.  A failed launch returns MLA_ERR_CUDA;
 *     mla_last_error() then holds the CUDA message (per host thread).
 *   - Data errors that only the device can see (a page index outside the
 *     pool, a non-monotone indptr, a bounded wait that ran out) never fault:
 *     the kernel clamps the access, records a flag in a per-device status
 *     word and carries on.  mla_device_status() reads and clears the word.
 *   - Layouts are dense, row-major, 16-byte aligned.  Element types:
 *     bf16 = IEEE bfloat16 bits (uint16), fp8 = OCP E4M3 ("e4m3fn") bytes.
 */
#ifndef MLA_DECODE_H
#define MLA_DECODE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_D_QK 576     /* query / KV row: 512 latent + 64 rope dims      */
#define MLA_D_LATENT 512 /* latent (value) width                            */
#define MLA_D_ROPE 64
#define MLA_D_V 128      /* W_UV output width per head                      */
#define MLA_MAX_HEADS 128
#define MLA_MAX_QLEN 16
#define MLA_MAX_SPLITS 256

typedef int mla_status;
#define MLA_OK 0
#define MLA_ERR_INVALID (-1)     /* bad argument (null, size, stride, alignment) */
#define MLA_ERR_UNSUPPORTED (-2) /* valid but outside what the kernels support   */
#define MLA_ERR_CUDA (-3)        /* a CUDA runtime call or launch failed         */

/* Bits of the per-device status word (mla_device_status). */
#define MLA_DEV_BAD_PAGE 1u      /* a page index was outside [0, pool_rows)      */
#define MLA_DEV_BAD_INDPTR 2u    /* indptr not monotone or beyond num_pages      */
#define MLA_DEV_TIMEOUT 4u       /* a bounded device wait ran out                */
#define MLA_DEV_BAD_PLAN 8u      /* a work plan did not fit this launch          */

/*
 * mla_decode_attend -- split-KV attention of one decode step.
 *
 * Defined by: vllm.models.kimi_k3.amd.specialized_decode.runtime.mla,
 * m1c_inputs (inputs q [S, 12, 576] bf16, kv = one 576-byte row per token,
 * pages = paged_kv_indices, indptr = paged_kv_indptr, scale, kv_scale; outputs the
 * partials o [splits, S, 12, 512] bf16 and LSE [splits, S, 12] f32) and
 * attend (multi-query attention over the latent cache; a query whose row
 * stride spans padded heads).
 *
 * For request r (rows t = r*qlen .. r*qlen+qlen-1), head h < heads, and
 * the tokens j of split k's range of r:
 *   K_j = e4m3fn(kv[pages[indptr[r] + j]]) * kv_scale        (576 wide)
 *   s_j = scale * <q[t, h, :], K_j>
 *   lse[k, t, h] = ln sum_j exp(s_j)
 *   o[k, t, h, :] = sum_j exp(s_j - lse[k, t, h]) * K_j[:512]
 * No mask within a request: every row of r attends over all of r's tokens
 * (mla_decode_attend_ex with MLA_ATTEND_CAUSAL adds the causal reading).
 *
 * Split plan: request r (length L_r = indptr[r+1] - indptr[r]) is cut into
 *   n_r = min(num_splits, max(1, ceil(L_r / split_tokens)))
 * contiguous ranges; with b = L_r / n_r and m = L_r % n_r, split k covers
 * [k*b + min(k, m), (k+1)*b + min(k+1, m)).  Splits k >= n_r get
 * lse = -inf and an unspecified o.  A request with L_r = 0 has one split
 * with lse = -inf.
 *
 *   q            bf16, row t head h at q + t*q_row_stride + h*576 (elements).
 *                q_row_stride >= heads*576 and a multiple of 8; padded heads
 *                (h >= heads) are never read.
 *   kv           fp8 codes [pool_rows, 576], contiguous.
 *   pages        int32 [num_pages]; indptr int32 [num_requests + 1] with
 *                indptr[0] = 0, non-decreasing, indptr[R] <= num_pages.
 *   qlen         query rows per request (1..16); S = num_requests * qlen.
 *   heads        real heads (1..128).
 *   num_splits   capacity of o / lse's first dimension (1..256).
 *   split_tokens target tokens per split (>= 1); see mla_choose_splits.
 *   o            bf16 [num_splits, S, heads, 512] (written);
 *   lse          f32  [num_splits, S, heads]       (written).
 */
mla_status mla_decode_attend(const void *q, int64_t q_row_stride, const void *kv,
                             int64_t pool_rows, const int32_t *pages, int64_t num_pages,
                             const int32_t *indptr, int num_requests, int qlen, int heads,
                             float scale, float kv_scale, int num_splits, int split_tokens,
                             void *o, float *lse, void *stream);

/* Flags of mla_decode_attend_ex. */
#define MLA_ATTEND_CAUSAL 1u   /* causal mask within a request (qlen > 1)    */
#define MLA_ATTEND_Q_FP8 2u    /* q holds fp8 e4m3 codes (DCP8's q8)         */

/*
 * mla_decode_attend_ex -- mla_decode_attend with option flags.
 *
 * The pages give no mask within a request; MLA_ATTEND_CAUSAL applies the
 * speculative-decode reading (a request's qlen query rows are its last qlen
 * token positions): row tq (0 <= tq < qlen) of request r sees only the
 * first L_r - qlen + tq + 1 of r's tokens.  Each split's partial for a row
 * covers the tokens of the split's range that the row sees; where it sees
 * none, lse = -inf and o is 0 (so a row that sees no token at all merges
 * to latent 0, LSE -inf).  flags = 0 is exactly mla_decode_attend.
 *
 * MLA_ATTEND_Q_FP8: q holds e4m3 codes, one byte per element (the pages'
 * decode-context-parallel input q8, whose _q_scale multiplies every score:
 * here pass scale * q_scale as scale, or give q_scale to
 * mla_decode_attend_planned); q_row_stride counts bytes and must be a
 * multiple of 16.  The score is scale * <e4m3(q), K>.
 *
 * Arguments as mla_decode_attend.  Unknown flag bits: MLA_ERR_INVALID.
 */
mla_status mla_decode_attend_ex(const void *q, int64_t q_row_stride, const void *kv,
                                int64_t pool_rows, const int32_t *pages, int64_t num_pages,
                                const int32_t *indptr, int num_requests, int qlen, int heads,
                                float scale, float kv_scale, int num_splits, int split_tokens,
                                void *o, float *lse, unsigned int flags, void *stream);

/*
 * mla_decode_attend_paged -- mla_decode_attend_ex over a block-table cache.
 *
 * The pages address the cache one 576-byte row per page index (m1c_inputs:
 * page size 1).  vLLM's paged layout groups page_size rows per block: here
 * pages holds block indices, indptr[r+1] - indptr[r] counts request r's
 * blocks, the last block holds last_page_len[r] rows, and token j of
 * request r is the flat row
 *   pages[indptr[r] + j / page_size] * page_size + j % page_size,
 * so L_r = (blocks - 1) * page_size + last_page_len[r] (0 with no blocks).
 * Everything else (split plan in tokens, outputs, flags) as
 * mla_decode_attend_ex; page_size 1 ignores last_page_len (may be NULL).
 *
 *   page_size      power of two, 1..256; pool_rows a multiple of it.
 *   last_page_len  int32 [num_requests], device, each in 1..page_size for a
 *                  request with blocks (else MLA_DEV_BAD_INDPTR, request empty).
 * A block index whose rows fall outside the pool sets MLA_DEV_BAD_PAGE.
 */
mla_status mla_decode_attend_paged(const void *q, int64_t q_row_stride, const void *kv,
                                   int64_t pool_rows, const int32_t *pages, int64_t num_pages,
                                   const int32_t *indptr, const int32_t *last_page_len, int page_size,
                                   int num_requests, int qlen, int heads, float scale, float kv_scale,
                                   int num_splits, int split_tokens, void *o, float *lse,
                                   unsigned int flags, void *stream);

/*
 * mla_plan_units -- a balanced work plan for the persistent attend kernel.
 *
 * The pages have no counterpart: they fix the partials (one per split of a
 * request, merged by LSE afterwards) but not where a request is cut.  The
 * attend kernel runs one CTA per SM; by default each takes whole units
 * (request, split, query-row group) round robin under the split rule of
 * mla_decode_attend, which leaves some CTAs with far more 128-token tiles
 * than others when contexts differ in length.  This host routine, given the
 * requests' token counts, cuts the requests into splits itself: it fills
 * the CTAs in request order, each up to one budget of tiles (plus a fixed
 * share per split), cutting a request at a tile boundary where a CTA fills
 * up, with the smallest budget that fits the grid and at most num_splits
 * splits per request.  With g query-row groups (rows = qlen * heads cut
 * into groups of at most 48) it fills G / g virtual CTAs and gives virtual
 * CTA v's list to CTAs v * g + j, row group j.
 *
 * Layout (int32): plan = [G, offsets[0 .. G], items..., first[0 .. G-1]],
 * CTA b takes items offsets[b] .. offsets[b + 1] - 1, each
 * MLA_PLAN_ITEM_WORDS int32
 *   { r, k | n_r << 9 | group << 18, start, count }:
 * split k (0-based) of the n_r splits of request r covers its tokens
 * [start, start + count) for query-row group `group`; the splits of a
 * request are consecutive ranges that cover all its tokens (an empty
 * request has one split of count 0).  first[b] repeats CTA b's first item
 * (zeros for a CTA without items): the kernel starts a CTA from this copy,
 * which it finds from the plan's length alone, so the offsets and the first
 * item cost one round trip of loads instead of two.  A plan whose copies
 * differ from the items is not one this routine writes.
 *
 *   host_lengths  int32 [num_requests], host: tokens per request (<= 0: empty).
 *   num_splits    most splits of one request (the partial buffers' split
 *                 dimension of the attend call that uses the plan).
 *   sm_count      G (at most 65536); <= 0 takes the current device's SM
 *                 count (the grid the attend kernel launches), and
 *                 MLA_ERR_CUDA when there is no usable device.
 *   plan          int32 [plan_capacity], host, caller-owned; NULL asks for
 *                 the size only.
 *   splits_used   optional out: the most splits any request got (<= num_splits).
 * Returns the plan's length in int32, or a negative mla_status
 * (MLA_ERR_INVALID: bad argument, plan_capacity too small or no host
 * memory for the plan's working lists;
 * MLA_ERR_UNSUPPORTED: fewer SMs than query-row groups).
 */
#define MLA_PLAN_ITEM_WORDS 4
int64_t mla_plan_units(int num_requests, int qlen, int heads, const int32_t *host_lengths,
                       int num_splits, int sm_count, int32_t *plan, int64_t plan_capacity,
                       int *splits_used);

/*
 * mla_plan_units_ex -- mla_plan_units with a floor on the splits per request:
 * no split of a request takes more than floor(tiles / min_splits) of its
 * 128-token tiles (at least one, and at least ceil(tiles / num_splits)), so
 * each request gets at least min_splits splits where its tile count and
 * num_splits allow; the fill is otherwise the same.  For a workload stated
 * as "each request split into m..n partials" (min_splits = m, num_splits =
 * n); min_splits = 1 is mla_plan_units.  1 <= min_splits <= num_splits, else
 * MLA_ERR_INVALID.
 */
int64_t mla_plan_units_ex(int num_requests, int qlen, int heads, const int32_t *host_lengths,
                          int min_splits, int num_splits, int sm_count, int32_t *plan,
                          int64_t plan_capacity, int *splits_used);

/*
 * mla_decode_attend_planned -- mla_decode_attend_paged with a work plan.
 *
 * plan (int32 [plan_len], device, 4-byte aligned) as mla_plan_units wrote
 * it, copied to the device; NULL is the round robin of
 * mla_decode_attend_paged.  The plan's splits replace the split rule
 * (split_tokens is then unused): each split's partial o / lse is the
 * attention over its token range, unused splits k >= n_r get lse = -inf,
 * and the merged result is the same attention up to rounding.  A plan for
 * another grid, offsets outside the buffer, or an item outside the launch
 * (r >= num_requests, k >= n_r, n_r > num_splits, group >= the row groups,
 * a range past the request's tokens, a zero-token item for a request that
 * has tokens) sets MLA_DEV_BAD_PLAN and ends that CTA's list, leaving its
 * remaining splits unwritten.  A plan with plan_len < 3 or > 2^31 - 1, or
 * not 4-byte aligned: MLA_ERR_INVALID.
 *
 * q_scale multiplies every score (the pages' _q_scale of an fp8 query,
 * MLA_ATTEND_Q_FP8; 1 for a bf16 query): the score is
 * scale * q_scale * <q, K>.  It must be finite.
 */
mla_status mla_decode_attend_planned(const void *q, int64_t q_row_stride, const void *kv,
                                     int64_t pool_rows, const int32_t *pages, int64_t num_pages,
                                     const int32_t *indptr, const int32_t *last_page_len,
                                     int page_size, int num_requests, int qlen, int heads,
                                     float scale, float kv_scale, float q_scale, int num_splits,
                                     int split_tokens, void *o, float *lse, unsigned int flags,
                                     const int32_t *plan, int64_t plan_len, void *stream);

/*
 * mla_merge_splits -- LSE merge of split partials into the latent.
 *
 * Defined by: vllm.models.kimi_k3.amd.specialized_decode.runtime.mla,
 * m1c_inputs (the split partials are merged by their LSE) and post (the same LSE combine
 * across decode-context-parallel ranks).  For every row t < rows, head h:
 *   LSE = ln sum_k exp(lse[k, t, h])   over splits with lse > -inf
 *   latent[t, h, :] = sum_k exp(lse[k, t, h] - LSE) * o[k, t, h, :]
 * Splits with lse = -inf are skipped (their o is never read).  A row whose
 * splits are all empty gets latent 0 and LSE -inf.
 *
 *   o        bf16 [num_splits, rows, heads, 512]; lse f32 [num_splits, rows, heads]
 *   latent   bf16 [rows, heads, 512] (written)
 *   lse_out  f32  [rows, heads] (written; may be NULL)
 *
 * A kernel enqueued after this call with programmatic dependent launch may
 * start while the merge runs; it must wait for the grid dependency
 * (griddepcontrol.wait / cudaGridDependencySynchronize) before it reads
 * latent or lse_out, as mla_value_gate does.
 */
mla_status mla_merge_splits(const void *o, const float *lse, int num_splits, int rows,
                            int heads, void *latent, float *lse_out, void *stream);

/*
 * mla_value_gate -- absorbed W_UV projection fused with the sigmoid gate.
 *
 * Defined by: vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.mla.value,
 * MlaValue (W_UV on the [B, H, 512] bf16 latent with bf16 MMA and fp32
 * accumulation; W_UV with a contiguous latent axis; rows are tokens, qlen
 * per request) and MlaGate (the bf16 value times the fp32 sigmoid of the
 * gate, rounded to bf16; rows of empty requests zero).  For row t, head h,
 * output v < 128, with r = t / qlen:
 *   val = bf16( sum_c latent[t, h, c] * w_uv[h, v, c] )      (fp32 sum)
 *   out[t, h*128 + v] = lengths[r] > 0 ? bf16( f32(val) * sigmoid(f32(gate[t, h*128 + v])) ) : 0
 * The zeroing is a select, so NaN gates of empty rows never reach out.
 *
 *   latent   bf16 [S, heads, 512];  w_uv bf16 [heads, 128, 512]
 *   gate     bf16 [S, heads*128] (raw logits);  lengths int32 [num_requests]
 *   out      bf16 [S, heads*128] (written);  S = num_requests * qlen
 *
 * The sum runs on the tensor cores (fp32 accumulation, in the hardware's
 * order); the sigmoid uses the hardware exponential and reciprocal
 * approximations (relative error below 1e-6, far under the bf16 rounding).
 * The kernel starts reading w_uv before the kernel enqueued just before it
 * on the stream has finished (programmatic dependent launch; latent, gate
 * and lengths are read after that kernel completes): w_uv must not be
 * written by that kernel.
 */
mla_status mla_value_gate(const void *latent, const void *w_uv, const void *gate,
                          const int32_t *lengths, int num_requests, int qlen, int heads,
                          void *out, void *stream);

/*
 * mla_merge_value_gate -- mla_merge_splits followed by mla_value_gate in one
 * call.  Small batches (at most twice as many 16-row tiles x heads as SMs)
 * run as a single launch that merges 16 rows of a head, writes them, and
 * projects and gates them straight from shared memory (the same tensor-core
 * MMAs as mla_value_gate); larger ones run the two kernels.  Both routes
 * give the same latent, LSE and out bytes as the two calls (the latent is
 * rounded to bf16 before the projection).
 *
 * Defined by: vllm.models.kimi_k3.amd.specialized_decode.runtime.mla,
 * m1c_inputs / post (the LSE merge of the splits, then W_UV and the gate)
 * and vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.mla.value,
 * MlaValue / MlaGate (projection, rounding and gating as in mla_value_gate).
 *
 *   o, lse, num_splits   as mla_merge_splits (rows = num_requests * qlen)
 *   w_uv, gate, lengths  as mla_value_gate;  out bf16 [S, heads*128] (written)
 *   latent               bf16 [S, heads, 512] (written: the merged latent)
 *   lse_out              f32 [S, heads] (written; may be NULL)
 *
 * Both routes start reading w_uv before the kernel enqueued just before
 * them on the stream has finished (programmatic dependent launch; every
 * other input is read after that kernel completes): w_uv must not be
 * written by that kernel.
 */
mla_status mla_merge_value_gate(const void *o, const float *lse, int num_splits, const void *w_uv,
                                const void *gate, const int32_t *lengths, int num_requests, int qlen,
                                int heads, void *out, void *latent, float *lse_out, void *stream);

/*
 * mla_kv_append -- write new tokens into the fp8 latent cache.
 *
 * Defined by: vllm.models.kimi_k3.amd.specialized_decode.runtime.mla, pre
 * (do_kv_cache_update: each new token's kv_c (512 latent values) and k_pe
 * (64 rope values) are stored, scaled by 1/_k_scale and converted to fp8,
 * at the token's slot: the row of the cache that mla_decode_attend reads).
 * For token i with slots[i] >= 0 and every d < 576:
 *   kv[slots[i], d] = e4m3(x / k_scale),  x = kv_c[i, d] (d < 512) or k_pe[i, d - 512]
 * with the quotient in float32 (IEEE division) and e4m3 round-to-nearest-
 * even, saturating (magnitudes above 448 and infinities give +-448, NaN
 * stays NaN).  A negative slot skips its token (padding).  Two tokens with
 * the same slot: which one lands is unspecified.
 *
 *   kv_c         bf16, token i at kv_c + i*kv_c_row_stride (elements, >= 512,
 *                multiple of 8).
 *   k_pe         bf16, token i at k_pe + i*k_pe_row_stride (>= 64, multiple of 8).
 *   slots        int64 [num_tokens], device memory.
 *   kv           fp8 codes [pool_rows, 576] (written at the slots only).
 * Slots >= pool_rows are skipped and set MLA_DEV_BAD_PAGE.  k_scale must be
 * finite and > 0.  kv_c, k_pe, kv 16-byte aligned; slots 8-byte aligned.
 */
mla_status mla_kv_append(const void *kv_c, int64_t kv_c_row_stride, const void *k_pe, int64_t k_pe_row_stride,
                         const int64_t *slots, int64_t num_tokens, float k_scale, void *kv, int64_t pool_rows,
                         void *stream);

/*
 * mla_choose_splits -- a split plan for mla_decode_attend from host-known
 * sizes (no device read).  Returns num_splits (>= 1) and writes
 * *split_tokens.  The plan minimises a model of the attend time: work units
 * are dealt round-robin to one persistent CTA per SM, so the busiest CTA
 * sets the time; every unit costs a fixed start-up plus its KV bytes, and
 * the partials cost a write and a read.  With host_lengths (int32 [R], host
 * memory, may be NULL) the unit sizes are exact; otherwise they are
 * estimated from max_len and total_len (total_len <= 0: R * max_len).
 * sm_count <= 0 means the current device's SM count (MLA_ERR_CUDA when
 * there is no usable device).  qlen outside 1..16, heads outside 1..128 or
 * sm_count above 65536: returns MLA_ERR_INVALID.
 */
int mla_choose_splits(int num_requests, int qlen, int heads, int max_len, int64_t total_len,
                      const int32_t *host_lengths, int sm_count, int *split_tokens);

/*
 * mla_debug_gather -- copies every request's KV rows, in request order, to
 * out (fp8 codes [indptr[R], 576]) through the attend kernel's own row
 * addressing and bulk-copy code, so that page indexing can be checked
 * byte for byte.  Same pointer rules as mla_decode_attend.
 */
mla_status mla_debug_gather(const void *kv, int64_t pool_rows, const int32_t *pages,
                            int64_t num_pages, const int32_t *indptr, int num_requests,
                            int64_t total_rows, void *out, void *stream);

/*
 * mla_debug_attend_mma -- a second, independently written attend kernel,
 * kept as a cross-check for the tests (no counterpart on the pages: it
 * computes what mla_decode_attend computes, with warp-level mma.sync f16
 * MMAs on e4m3 -> f16 converted rows instead of tcgen05 tensor memory).
 * Arguments, outputs and split rule as mla_decode_attend (page size 1,
 * bf16 query, no mask, no work plan).  Not used by any other call.
 */
mla_status mla_debug_attend_mma(const void *q, int64_t q_row_stride, const void *kv, int64_t pool_rows,
                                const int32_t *pages, int64_t num_pages, const int32_t *indptr,
                                int num_requests, int qlen, int heads, float scale, float kv_scale,
                                int num_splits, int split_tokens, void *o, float *lse, void *stream);

/*
 * mla_debug_wait_timeout -- test hook for the device-side failure path (no
 * counterpart on the pages: it belongs to this library's error handling).
 * Enqueues one 32-thread CTA whose first thread waits, through the same
 * bounded mbarrier wait every kernel here uses, on a barrier that nothing
 * arrives at.  After the wait budget (4e9 SM cycles, about 2 s at 2 GHz) it
 * sets MLA_DEV_TIMEOUT and returns: the context stays usable and nothing is
 * left in flight.  Returns MLA_ERR_CUDA without a device or if the launch
 * fails.
 */
mla_status mla_debug_wait_timeout(void *stream);

/*
 * mla_device_status -- synchronises `stream`, returns the current device's
 * status word (MLA_DEV_* bits set by kernels since the last read) in
 * *flags and clears it.  Returns MLA_ERR_CUDA if the synchronisation fails.
 */
mla_status mla_device_status(void *stream, unsigned int *flags);

/*
 * mla_decode_step_static -- one whole decode step that allocates nothing.
 *
 * The pages have no counterpart: this entry point exists for callers that
 * cannot allocate device memory while they run -- a serving loop whose
 * memory is planned up front and may not grow, a plain C host with no
 * device allocator, code that must not stall on cudaMalloc's implicit
 * synchronisation.  Such callers can hold the step's inputs and outputs,
 * but not the split partials that pass from attend to the merge.  Here
 * those partials live in one buffer inside the library, a static device
 * array of MLA_STATIC_SCRATCH_BYTES (32 MiB) that every GPU loading the
 * library keeps until the process exits.
 *
 * It runs mla_decode_attend_planned (page size 1, bf16 query, no flags)
 * into that buffer and then mla_merge_value_gate from it, so its results
 * are those of the two calls with caller-owned partials.  Arguments as
 * those two calls (plan may be NULL: round robin under the split rule;
 * latent is required, lse_out may be NULL).
 *
 *   - Size limit: the partials need num_splits * S * heads * 1028 bytes
 *     (plus up to 255 bytes of alignment); above MLA_STATIC_SCRATCH_BYTES
 *     the call returns MLA_ERR_UNSUPPORTED before launching anything, and
 *     mla_last_error() gives the size needed.
 *   - Allocation: none (no cudaMalloc, cudaFree or allocating library
 *     routine).  The first call on a device looks up the buffer's device
 *     address (cudaGetSymbolAddress, which also loads the library's module
 *     there); make that first call before any stream capture.
 *   - Sharing: every call uses the same buffer and leaves its partials in
 *     it.  Nothing in it has to start at zero (attend writes every LSE of
 *     the launch, -inf for unused splits, and the merge reads a partial row
 *     only where its LSE is finite), but two calls whose kernels overlap on
 *     the GPU (different streams without ordering, or several host threads)
 *     race on it: order them on one stream.
 */
#define MLA_STATIC_SCRATCH_BYTES 33554432 /* 32 MiB */
mla_status mla_decode_step_static(const void *q, int64_t q_row_stride, const void *kv, int64_t pool_rows,
                                  const int32_t *pages, int64_t num_pages, const int32_t *indptr,
                                  int num_requests, int qlen, int heads, float scale, float kv_scale,
                                  int num_splits, int split_tokens, const int32_t *plan, int64_t plan_len,
                                  const void *w_uv, const void *gate, const int32_t *lengths, void *out,
                                  void *latent, float *lse_out, void *stream);

/* Static description of a status code. */
const char *mla_status_string(mla_status status);

/* Detail of the last error on this host thread ("" if none). */
const char *mla_last_error(void);

/* Library version string. */
const char *mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H */
