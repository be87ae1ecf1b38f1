// Host side of the C ABI declared in include/mla_decode.h: argument
// validation (before any launch), kernel dispatch, the split-plan
// heuristic, error strings and the device status word.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <new>
#include <string>
#include <algorithm>
#include <atomic>
#include <utility>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/mla_decode.h"

namespace mla {
cudaError_t attend_mma_launch(const void *q, int64_t q_row_stride, const void *kv, int64_t pool_rows,
                              const int32_t *pages, int64_t num_pages, const int32_t *indptr, int R,
                              int qlen, int heads, float scale, float kv_scale, int num_splits,
                              int split_tokens, void *o, float *lse, int grid, cudaStream_t st);
cudaError_t attend_mma_status(unsigned int *flags, bool clear);
cudaError_t attend_tc_launch(const void *q, int64_t q_row_stride, const void *kv, int64_t pool_rows,
                             const int32_t *pages, int64_t num_pages, const int32_t *indptr, int R, int qlen,
                             int heads, float scale, float kv_scale, int num_splits, int split_tokens, void *o,
                             float *lse, bool causal, int log2p, const int32_t *last_page_len, bool q8,
                             const int32_t *plan, int64_t plan_len, int grid, cudaStream_t st);
void attend_tc_shape(int rows, int *groups, int *nq);
cudaError_t attend_tc_status(unsigned int *flags, bool clear);
cudaError_t merge_launch(const void *o, const float *lse, int num_splits, int rows, int heads,
                         void *latent, float *lse_out, cudaStream_t st);
cudaError_t merge_status(unsigned int *flags, bool clear);
cudaError_t value_gate_launch(const void *latent, const void *w_uv, const void *gate,
                              const int32_t *lengths, int R, int qlen, int H, void *out, int sms, cudaStream_t st);
cudaError_t value_gate_status(unsigned int *flags, bool clear);
cudaError_t merge_value_launch(const void *o, const float *lse, int num_splits, const void *w_uv, const void *gate,
                               const int32_t *lengths, int R, int qlen, int H, void *out, void *latent,
                               float *lse_out, cudaStream_t st);
cudaError_t gather_launch(const void *kv, int64_t pool_rows, const int32_t *pages, const int32_t *indptr,
                          int R, int64_t total_rows, void *out, cudaStream_t st);
cudaError_t gather_status(unsigned int *flags, bool clear);
cudaError_t stuck_wait_launch(cudaStream_t st);
cudaError_t kv_append_launch(const void *kv_c, int64_t kv_c_stride, const void *k_pe, int64_t k_pe_stride,
                             const int64_t *slots, int64_t T, float k_scale, void *kv, int64_t pool_rows, int sms,
                             cudaStream_t st);
cudaError_t kv_append_status(unsigned int *flags, bool clear);
}  // namespace mla

namespace {

thread_local std::string g_last_error;

mla_status fail(mla_status s, const char *msg) {
    g_last_error = msg;
    return s;
}

mla_status cuda_fail(cudaError_t e, const char *where) {
    g_last_error = std::string(where) + ": " + cudaGetErrorString(e);
    return MLA_ERR_CUDA;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// The current device's SM count, or 0 when there is no usable device (the
// callers then fail with MLA_ERR_CUDA rather than size a grid for a guess).
int device_sms() {
    static std::atomic<int> cached[64] = {};   // per device ordinal; 0: not read yet
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (dev >= 0 && dev < 64 && (n = cached[dev].load(std::memory_order_relaxed)) > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 0;
    }
    if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

}  // namespace

namespace mla {
// Error text for calls defined in other translation units (mla_last_error()).
void set_last_error(const char *msg) { g_last_error = msg; }
}  // namespace mla

extern "C" {

mla_status mla_decode_attend(const void *q, int64_t q_row_stride, const void *kv, int64_t pool_rows,
                             const int32_t *pages, int64_t num_pages, const int32_t *indptr,
                             int num_requests, int qlen, int heads, float scale, float kv_scale,
                             int num_splits, int split_tokens, void *o, float *lse, void *stream) {
    return mla_decode_attend_ex(q, q_row_stride, kv, pool_rows, pages, num_pages, indptr, num_requests, qlen,
                                heads, scale, kv_scale, num_splits, split_tokens, o, lse, 0u, stream);
}

mla_status mla_decode_attend_ex(const void *q, int64_t q_row_stride, const void *kv, int64_t pool_rows,
                                const int32_t *pages, int64_t num_pages, const int32_t *indptr,
                                int num_requests, int qlen, int heads, float scale, float kv_scale,
                                int num_splits, int split_tokens, void *o, float *lse, unsigned int flags,
                                void *stream) {
    return mla_decode_attend_paged(q, q_row_stride, kv, pool_rows, pages, num_pages, indptr, nullptr, 1,
                                   num_requests, qlen, heads, scale, kv_scale, num_splits, split_tokens, o, lse,
                                   flags, stream);
}

mla_status mla_decode_attend_paged(const void *q, int64_t q_row_stride, const void *kv, int64_t pool_rows,
                                   const int32_t *pages, int64_t num_pages, const int32_t *indptr,
                                   const int32_t *last_page_len, int page_size, int num_requests, int qlen,
                                   int heads, float scale, float kv_scale, int num_splits, int split_tokens,
                                   void *o, float *lse, unsigned int flags, void *stream) {
    return mla_decode_attend_planned(q, q_row_stride, kv, pool_rows, pages, num_pages, indptr, last_page_len,
                                     page_size, num_requests, qlen, heads, scale, kv_scale, 1.0f, num_splits,
                                     split_tokens, o, lse, flags, nullptr, 0, stream);
}

mla_status mla_decode_attend_planned(const void *q, int64_t q_row_stride, const void *kv, int64_t pool_rows,
                                     const int32_t *pages, int64_t num_pages, const int32_t *indptr,
                                     const int32_t *last_page_len, int page_size, int num_requests, int qlen,
                                     int heads, float scale, float kv_scale, float q_scale, int num_splits,
                                     int split_tokens, void *o, float *lse, unsigned int flags,
                                     const int32_t *plan, int64_t plan_len, void *stream) {
    if (flags & ~(MLA_ATTEND_CAUSAL | MLA_ATTEND_Q_FP8)) return fail(MLA_ERR_INVALID, "unknown flag bits");
    if (plan && (plan_len < 3 || plan_len > INT32_MAX || !aligned(plan, 4)))
        return fail(MLA_ERR_INVALID, "plan too short, too long or misaligned");
    const bool q8 = (flags & MLA_ATTEND_Q_FP8) != 0;
    int log2p = 0;
    while ((1 << log2p) < page_size && log2p < 9) ++log2p;
    if (page_size < 1 || page_size > 256 || (1 << log2p) != page_size)
        return fail(MLA_ERR_INVALID, "page_size must be a power of two in 1..256");
    if (page_size > 1 && (pool_rows % page_size != 0))
        return fail(MLA_ERR_INVALID, "pool_rows must be a multiple of page_size");
    const bool causal = (flags & MLA_ATTEND_CAUSAL) != 0;
    if (num_requests < 0) return fail(MLA_ERR_INVALID, "num_requests < 0");
    if (qlen < 1 || qlen > MLA_MAX_QLEN) return fail(MLA_ERR_INVALID, "qlen outside 1..16");
    if (heads < 1 || heads > MLA_MAX_HEADS) return fail(MLA_ERR_INVALID, "heads outside 1..128");
    if (num_splits < 1 || num_splits > MLA_MAX_SPLITS) return fail(MLA_ERR_INVALID, "num_splits outside 1..256");
    if (split_tokens < 1) return fail(MLA_ERR_INVALID, "split_tokens < 1");
    if (q_row_stride < (int64_t)heads * MLA_D_QK || q_row_stride % (q8 ? 16 : 8) != 0)
        return fail(MLA_ERR_INVALID, q8 ? "q_row_stride must be >= heads*576 and a multiple of 16 (fp8 q)"
                                        : "q_row_stride must be >= heads*576 and a multiple of 8");
    if (pool_rows < 0 || num_pages < 0) return fail(MLA_ERR_INVALID, "negative pool_rows / num_pages");
    if (!std::isfinite(scale) || !std::isfinite(kv_scale) || !std::isfinite(q_scale))
        return fail(MLA_ERR_INVALID, "non-finite scale");
    if (num_requests == 0) return MLA_OK;
    if (!q || !kv || !indptr || !o || !lse || (num_pages > 0 && !pages))
        return fail(MLA_ERR_INVALID, "null pointer");
    if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
        !aligned(indptr, 4) || !aligned(pages, 4))
        return fail(MLA_ERR_INVALID, "misaligned pointer (q, kv, o need 16 bytes)");
    if (pool_rows == 0) return fail(MLA_ERR_INVALID, "empty KV pool");
    if (pool_rows > INT32_MAX) return fail(MLA_ERR_UNSUPPORTED, "pool_rows above 2^31 - 1");
    if (page_size > 1 && (!last_page_len || !aligned(last_page_len, 4)))
        return fail(MLA_ERR_INVALID, "page_size > 1 needs last_page_len (int32, 4-byte aligned)");
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int sms = device_sms();
    if (sms <= 0) return fail(MLA_ERR_CUDA, "no CUDA device");
    // The fp8 query's scale multiplies every score: folded into the softmax scale.
    cudaError_t e = mla::attend_tc_launch(q, q_row_stride, kv, pool_rows, pages, num_pages, indptr, num_requests,
                                          qlen, heads, scale * q_scale, kv_scale, num_splits, split_tokens, o, lse,
                                          causal, log2p, last_page_len, q8, plan, plan_len, sms, st);
    if (e != cudaSuccess) return cuda_fail(e, "attend launch");
    return MLA_OK;
}

mla_status mla_debug_attend_mma(const void *q, int64_t q_row_stride, const void *kv, int64_t pool_rows,
                                const int32_t *pages, int64_t num_pages, const int32_t *indptr, int num_requests,
                                int qlen, int heads, float scale, float kv_scale, int num_splits, int split_tokens,
                                void *o, float *lse, void *stream) {
    // The argument rules of mla_decode_attend (page size 1, bf16 query,
    // no options), then the warp-MMA kernel.
    if (num_requests < 0) return fail(MLA_ERR_INVALID, "num_requests < 0");
    if (qlen < 1 || qlen > MLA_MAX_QLEN) return fail(MLA_ERR_INVALID, "qlen outside 1..16");
    if (heads < 1 || heads > MLA_MAX_HEADS) return fail(MLA_ERR_INVALID, "heads outside 1..128");
    if (num_splits < 1 || num_splits > MLA_MAX_SPLITS) return fail(MLA_ERR_INVALID, "num_splits outside 1..256");
    if (split_tokens < 1) return fail(MLA_ERR_INVALID, "split_tokens < 1");
    if (q_row_stride < (int64_t)heads * MLA_D_QK || q_row_stride % 8 != 0)
        return fail(MLA_ERR_INVALID, "q_row_stride must be >= heads*576 and a multiple of 8");
    if (pool_rows < 0 || num_pages < 0) return fail(MLA_ERR_INVALID, "negative pool_rows / num_pages");
    if (!std::isfinite(scale) || !std::isfinite(kv_scale)) return fail(MLA_ERR_INVALID, "non-finite scale");
    if (num_requests == 0) return MLA_OK;
    if (!q || !kv || !indptr || !o || !lse || (num_pages > 0 && !pages)) return fail(MLA_ERR_INVALID, "null pointer");
    if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(o, 16) || !aligned(lse, 4) || !aligned(indptr, 4) ||
        !aligned(pages, 4))
        return fail(MLA_ERR_INVALID, "misaligned pointer (q, kv, o need 16 bytes)");
    if (pool_rows == 0) return fail(MLA_ERR_INVALID, "empty KV pool");
    if (pool_rows > INT32_MAX) return fail(MLA_ERR_UNSUPPORTED, "pool_rows above 2^31 - 1");
    const int sms = device_sms();
    if (sms <= 0) return fail(MLA_ERR_CUDA, "no CUDA device");
    cudaError_t e = mla::attend_mma_launch(q, q_row_stride, kv, pool_rows, pages, num_pages, indptr, num_requests,
                                           qlen, heads, scale, kv_scale, num_splits, split_tokens, o, lse, sms,
                                           static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "warp-MMA attend launch");
    return MLA_OK;
}

mla_status mla_merge_splits(const void *o, const float *lse, int num_splits, int rows, int heads,
                            void *latent, float *lse_out, void *stream) {
    if (num_splits < 1 || num_splits > MLA_MAX_SPLITS) return fail(MLA_ERR_INVALID, "num_splits outside 1..256");
    if (rows < 0) return fail(MLA_ERR_INVALID, "rows < 0");
    if (heads < 1 || heads > MLA_MAX_HEADS) return fail(MLA_ERR_INVALID, "heads outside 1..128");
    if (rows == 0) return MLA_OK;
    if (!o || !lse || !latent) return fail(MLA_ERR_INVALID, "null pointer");
    if (!aligned(o, 16) || !aligned(latent, 16) || !aligned(lse, 4) || !aligned(lse_out, 4))
        return fail(MLA_ERR_INVALID, "misaligned pointer (o, latent need 16 bytes)");
    cudaError_t e = mla::merge_launch(o, lse, num_splits, rows, heads, latent, lse_out,
                                      static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "merge launch");
    return MLA_OK;
}

mla_status mla_value_gate(const void *latent, const void *w_uv, const void *gate, const int32_t *lengths,
                          int num_requests, int qlen, int heads, void *out, void *stream) {
    if (num_requests < 0) return fail(MLA_ERR_INVALID, "num_requests < 0");
    if (qlen < 1 || qlen > MLA_MAX_QLEN) return fail(MLA_ERR_INVALID, "qlen outside 1..16");
    if (heads < 1 || heads > MLA_MAX_HEADS) return fail(MLA_ERR_INVALID, "heads outside 1..128");
    if (num_requests == 0) return MLA_OK;
    if (!latent || !w_uv || !gate || !lengths || !out) return fail(MLA_ERR_INVALID, "null pointer");
    if (!aligned(latent, 16) || !aligned(w_uv, 16) || !aligned(gate, 4) || !aligned(out, 4) ||
        !aligned(lengths, 4))
        return fail(MLA_ERR_INVALID, "misaligned pointer (latent, w_uv need 16 bytes)");
    if ((int64_t)num_requests * qlen > INT32_MAX) return fail(MLA_ERR_UNSUPPORTED, "too many rows");
    const int sms = device_sms();
    if (sms <= 0) return fail(MLA_ERR_CUDA, "no CUDA device");
    cudaError_t e = mla::value_gate_launch(latent, w_uv, gate, lengths, num_requests, qlen, heads, out, sms,
                                           static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "value_gate launch");
    return MLA_OK;
}

mla_status mla_merge_value_gate(const void *o, const float *lse, int num_splits, const void *w_uv,
                                const void *gate, const int32_t *lengths, int num_requests, int qlen, int heads,
                                void *out, void *latent, float *lse_out, void *stream) {
    if (num_splits < 1 || num_splits > MLA_MAX_SPLITS) return fail(MLA_ERR_INVALID, "num_splits outside 1..256");
    if (num_requests < 0) return fail(MLA_ERR_INVALID, "num_requests < 0");
    if (qlen < 1 || qlen > MLA_MAX_QLEN) return fail(MLA_ERR_INVALID, "qlen outside 1..16");
    if (heads < 1 || heads > MLA_MAX_HEADS) return fail(MLA_ERR_INVALID, "heads outside 1..128");
    if (num_requests == 0) return MLA_OK;
    if (!o || !lse || !w_uv || !gate || !lengths || !out || !latent) return fail(MLA_ERR_INVALID, "null pointer");
    if (!aligned(o, 16) || !aligned(w_uv, 16) || !aligned(latent, 16) || !aligned(lse, 4) || !aligned(gate, 4) ||
        !aligned(out, 4) || !aligned(lengths, 4) || !aligned(lse_out, 4))
        return fail(MLA_ERR_INVALID, "misaligned pointer (o, w_uv, latent need 16 bytes)");
    if ((int64_t)num_requests * qlen > INT32_MAX) return fail(MLA_ERR_UNSUPPORTED, "too many rows");
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int sms = device_sms();
    if (sms <= 0) return fail(MLA_ERR_CUDA, "no CUDA device");
    const int64_t S = (int64_t)num_requests * qlen;
    cudaError_t e;
    // One launch while its 16-row CTAs (one per SM at a time) number at most
    // two waves; past that, loading the head's 128 KB W_UV slice per 16 rows
    // costs more than the separate merge and the 64- or 96-row value kernel save.
    // Graph-replayed steps on one GB300: 64 x 12 rows (48 CTAs) and 32 x 96
    // (192) are faster fused, 512 x 12 (384) and 2,048 x 12 (1,536) split.
    if (((S + 15) / 16) * heads <= 2 * (int64_t)sms) {
        e = mla::merge_value_launch(o, lse, num_splits, w_uv, gate, lengths, num_requests, qlen, heads, out, latent,
                                    lse_out, st);
    } else {
        e = mla::merge_launch(o, lse, num_splits, (int)S, heads, latent, lse_out, st);
        if (e == cudaSuccess)
            e = mla::value_gate_launch(latent, w_uv, gate, lengths, num_requests, qlen, heads, out, sms, st);
    }
    if (e != cudaSuccess) return cuda_fail(e, "merge_value_gate launch");
    return MLA_OK;
}

namespace {
// Most CTAs a host split or work plan is made for.
constexpr int kPlanMaxCtas = 65536;
}  // namespace

int mla_choose_splits(int num_requests, int qlen, int heads, int max_len, int64_t total_len,
                      const int32_t *host_lengths, int sm_count, int *split_tokens) {
    if (qlen < 1 || qlen > MLA_MAX_QLEN || heads < 1 || heads > MLA_MAX_HEADS || sm_count > kPlanMaxCtas)
        return fail(MLA_ERR_INVALID, "choose_splits: qlen, heads or sm_count out of range");
    if (sm_count <= 0 && (sm_count = device_sms()) <= 0)
        return fail(MLA_ERR_CUDA, "choose_splits: no CUDA device to take the SM count from (pass sm_count)");
    if (host_lengths) {
        max_len = 0;
        total_len = 0;
        for (int r = 0; r < num_requests; ++r) {
            const int L = host_lengths[r] > 0 ? host_lengths[r] : 0;
            max_len = L > max_len ? L : max_len;
            total_len += L;
        }
    }
    if (num_requests <= 0 || max_len <= 0) {
        if (split_tokens) *split_tokens = max_len > 0 ? max_len : 1;
        return 1;
    }
    if (total_len <= 0) total_len = (int64_t)num_requests * max_len;
    const int rows = qlen * heads;
    int groups = 1, nq = 16;
    mla::attend_tc_shape(rows, &groups, &nq);
    const double bw_sm = 6.5e12 / sm_count;   // bytes/s per SM at the HBM roofline
    const double t_tok = MLA_D_QK / bw_sm;     // seconds per KV row on one SM
    const double t_unit = 1.5e-6;              // per-unit start-up (query load, epilogue)
    const double t_part_unit = rows * (MLA_D_LATENT * 2.0 + 4.0) * 2.0 / (bw_sm * sm_count);
    const double avg_fill = (double)total_len / ((double)num_requests * max_len);
    std::vector<double> load;
    int best_ns = 1, best_st = max_len;
    double best_t = 1e30;
    for (int ns = 1; ns <= MLA_MAX_SPLITS; ++ns) {
        const int st = (max_len + ns - 1) / ns;
        if (ns > 1 && st < 64) break;
        double t, units;
        if (host_lengths) {
            // exact: walk the units in the kernel's order and deal them out
            load.assign(sm_count, 0.0);
            long long u = 0;
            for (int r = 0; r < num_requests; ++r) {
                const int L = host_lengths[r] > 0 ? host_lengths[r] : 0;
                int n = (L + st - 1) / st;
                n = n < 1 ? 1 : (n > ns ? ns : n);
                const int b = L / n, m = L % n;
                for (int k = 0; k < n; ++k)
                    for (int g = 0; g < groups; ++g, ++u)
                        load[u % sm_count] += (b + (k < m ? 1 : 0)) * t_tok + t_unit;
            }
            units = (double)u / groups;
            double mx = 0;
            for (double x : load) mx = x > mx ? x : mx;
            t = mx;
        } else {
            units = std::ceil((double)total_len / st + 0.5 * num_requests * (1.0 - avg_fill));
            t = std::ceil(units * groups / sm_count) * (st * t_tok + t_unit);
        }
        t += units * t_part_unit;
        if (t < best_t * 0.999) {
            best_t = t;
            best_ns = ns;
            best_st = st;
        }
    }
    if (split_tokens) *split_tokens = best_st;
    return best_ns;
}

namespace {

// Cost model of the work plan, in tenths of a 128-token tile: a tile and an
// empty request; plan_piece_cost gives the fixed cost of a split.
constexpr int64_t kPlanTile = 10, kPlanEmpty = 2;

// The fixed cost of a split (a unit change in the kernel: the next unit's
// query converted, the finished unit's o and LSE written, the first tile's
// rebase) for nq query rows per CTA.  Measured on GB300 with clock stamps
// at 48 rows, ~18,500 cycles against a ~4,600-cycle tile; costed here at 4
// tiles for 48 rows, 3 for 32 and half a tile for 16, the settings that
// measured fastest in attend A/Bs of the plan (at 48 rows 4 tiles beat 3 and
// 5, and earlier 3 beat 0.5, 2 and 5; at 32 rows 3 beat 0.5 and 1.5; at 16
// rows 0.5 beat 1.5, 2.5 and 3).
int64_t plan_piece_cost(int nq) { return nq >= 48 ? 40 : nq >= 32 ? 30 : 5; }

struct PlanPiece {
    int r, k, start, count;
};

// Greedy contiguous fill of the requests' tiles, in request order, into
// virtual CTAs of at most `budget` each; a request is cut at tile
// boundaries where a CTA fills up.  Returns the CTAs used (V + 1 when more
// than V would be needed or a request would need more than max_splits
// pieces); pieces are appended per CTA when `out` is given.
// The most tiles one piece of a request of ntiles tiles may take: so that it
// gets at least min_splits pieces (one per tile when it has fewer tiles),
// but never so few tiles that it would need more than max_splits pieces.
int plan_piece_cap(int ntiles, int min_splits, int max_splits) {
    const int lo = (ntiles + max_splits - 1) / max_splits;
    return std::max(ntiles >= min_splits ? ntiles / min_splits : 1, std::max(lo, 1));
}

int plan_fill(const int32_t *lengths, int R, int64_t budget, int V, int max_splits, int min_splits, int64_t piece,
              std::vector<std::vector<PlanPiece>> *out) {
    int v = 0;
    int64_t load = 0;
    if (out) out->assign(V, {});
    for (int r = 0; r < R; ++r) {
        const int L = lengths[r] > 0 ? lengths[r] : 0;
        if (L == 0) {
            if (load > 0 && load + kPlanEmpty > budget) {
                if (++v >= V) return V + 1;
                load = 0;
            }
            load += kPlanEmpty;
            if (out) (*out)[v].push_back({r, 0, 0, 0});
            continue;
        }
        const int ntiles = (L + 127) / 128;
        const int cap = plan_piece_cap(ntiles, min_splits, max_splits);
        int done = 0, k = 0;
        while (done < ntiles) {
            const int64_t room = budget - load;
            if (load > 0 && room < piece + kPlanTile) {
                if (++v >= V) return V + 1;
                load = 0;
                continue;
            }
            int64_t take = (room - piece) / kPlanTile;
            if (take < 1) take = 1;
            if (take > ntiles - done) take = ntiles - done;
            if (take > cap) take = cap;
            if (++k > max_splits) return V + 1;
            if (out) {
                const int start = done * 128;
                const int count = (int)std::min<int64_t>((int64_t)take * 128, (int64_t)L - start);
                (*out)[v].push_back({r, k - 1, start, count});
            }
            load += take * kPlanTile + piece;
            done += (int)take;
        }
    }
    return v + 1;
}

}  // namespace

namespace {
int64_t plan_build(int num_requests, int qlen, int heads, const int32_t *host_lengths, int num_splits,
                   int min_splits, int sm_count, int32_t *plan, int64_t plan_capacity, int *splits_used);
}  // namespace

int64_t mla_plan_units(int num_requests, int qlen, int heads, const int32_t *host_lengths, int num_splits,
                       int sm_count, int32_t *plan, int64_t plan_capacity, int *splits_used) {
    return mla_plan_units_ex(num_requests, qlen, heads, host_lengths, 1, num_splits, sm_count, plan, plan_capacity,
                             splits_used);
}

int64_t mla_plan_units_ex(int num_requests, int qlen, int heads, const int32_t *host_lengths, int min_splits,
                          int num_splits, int sm_count, int32_t *plan, int64_t plan_capacity, int *splits_used) {
    if (num_requests < 0 || qlen < 1 || qlen > MLA_MAX_QLEN || heads < 1 || heads > MLA_MAX_HEADS ||
        num_splits < 1 || num_splits > MLA_MAX_SPLITS || (num_requests > 0 && !host_lengths))
        return fail(MLA_ERR_INVALID, "bad plan arguments");
    if (min_splits < 1 || min_splits > num_splits) return fail(MLA_ERR_INVALID, "min_splits outside 1..num_splits");
    if (sm_count <= 0 && (sm_count = device_sms()) <= 0)
        return fail(MLA_ERR_CUDA, "plan_units: no CUDA device to take the SM count from (pass sm_count)");
    if (sm_count > kPlanMaxCtas) return fail(MLA_ERR_INVALID, "sm_count above 65536");
    try {
        return plan_build(num_requests, qlen, heads, host_lengths, num_splits, min_splits, sm_count, plan,
                          plan_capacity, splits_used);
    } catch (const std::bad_alloc &) {
        return fail(MLA_ERR_INVALID, "host memory for the plan");
    }
}

namespace {

int64_t plan_build(int num_requests, int qlen, int heads, const int32_t *host_lengths, int num_splits,
                   int min_splits, int sm_count, int32_t *plan, int64_t plan_capacity, int *splits_used) {
    int groups, nq;
    mla::attend_tc_shape(qlen * heads, &groups, &nq);
    // Each row group of a request runs on its own CTA; the plan fills
    // V = G / groups virtual CTAs and gives virtual CTA v's items to CTAs
    // v * groups + g (row group g), so a request's groups read the same KV
    // tiles at about the same time.
    const int V = sm_count / groups;
    if (V < 1) return fail(MLA_ERR_UNSUPPORTED, "fewer SMs than query-row groups");
    const int64_t piece = plan_piece_cost(nq);
    // Smallest budget whose fill fits V CTAs within num_splits pieces per
    // request (the fill with an unbounded budget always fits: one CTA, the
    // fewest pieces min_splits allows per request).
    int64_t total = 0;
    for (int r = 0; r < num_requests; ++r) {
        const int t = host_lengths[r] > 0 ? (host_lengths[r] + 127) / 128 : 0;
        const int cap = plan_piece_cap(t, min_splits, num_splits);
        total += t > 0 ? (int64_t)t * kPlanTile + (int64_t)((t + cap - 1) / cap) * piece : kPlanEmpty;
    }
    int64_t lo = 0, hi = total + piece + kPlanTile;
    while (hi - lo > 1) {
        const int64_t mid = lo + (hi - lo) / 2;
        if (plan_fill(host_lengths, num_requests, mid, V, num_splits, min_splits, piece, nullptr) <= V) hi = mid;
        else lo = mid;
    }
    std::vector<std::vector<PlanPiece>> vc;
    plan_fill(host_lengths, num_requests, hi, V, num_splits, min_splits, piece, &vc);
    // pieces per request (n_r) and the plan's size
    std::vector<int> n_r(num_requests > 0 ? num_requests : 1, 1);
    int64_t items = 0;
    int used = 1;
    for (const auto &list : vc)
        for (const PlanPiece &pc : list) {
            n_r[pc.r] = std::max(n_r[pc.r], pc.k + 1);
            used = std::max(used, pc.k + 1);
            items += groups;
        }
    if (splits_used) *splits_used = used;
    // header, items, then each CTA's first item again (zeros for a CTA with none)
    const int64_t need = 2 + (int64_t)sm_count + (int64_t)MLA_PLAN_ITEM_WORDS * (items + sm_count);
    if (!plan) return need;
    if (plan_capacity < need) return fail(MLA_ERR_INVALID, "plan buffer too small");
    plan[0] = sm_count;
    int32_t *it = plan + 2 + sm_count;
    int64_t pos = 0;
    for (int b = 0; b < sm_count; ++b) {
        plan[1 + b] = (int32_t)pos;
        const int v = b / groups, g = b % groups;
        if (v >= V) continue;
        for (const PlanPiece &pc : vc[v]) {
            it[0] = pc.r;
            it[1] = pc.k | (n_r[pc.r] << 9) | (g << 18);
            it[2] = pc.start;
            it[3] = pc.count;
            it += MLA_PLAN_ITEM_WORDS;
            ++pos;
        }
    }
    plan[1 + sm_count] = (int32_t)pos;
    // The first items again, at a place the kernel finds from the plan's
    // length alone: a CTA loads its offsets and its first item at once.
    int32_t *first = plan + 2 + sm_count + (int64_t)MLA_PLAN_ITEM_WORDS * items;
    for (int b = 0; b < sm_count; ++b) {
        const int32_t a = plan[1 + b], e = plan[2 + b];
        for (int w = 0; w < MLA_PLAN_ITEM_WORDS; ++w)
            first[(int64_t)MLA_PLAN_ITEM_WORDS * b + w] =
                a < e ? plan[2 + sm_count + (int64_t)MLA_PLAN_ITEM_WORDS * a + w] : 0;
    }
    return need;
}

}  // namespace

mla_status mla_kv_append(const void *kv_c, int64_t kv_c_row_stride, const void *k_pe, int64_t k_pe_row_stride,
                         const int64_t *slots, int64_t num_tokens, float k_scale, void *kv, int64_t pool_rows,
                         void *stream) {
    if (num_tokens < 0 || pool_rows < 0) return fail(MLA_ERR_INVALID, "negative size");
    if (kv_c_row_stride < MLA_D_LATENT || kv_c_row_stride % 8 != 0)
        return fail(MLA_ERR_INVALID, "kv_c_row_stride must be >= 512 and a multiple of 8");
    if (k_pe_row_stride < MLA_D_ROPE || k_pe_row_stride % 8 != 0)
        return fail(MLA_ERR_INVALID, "k_pe_row_stride must be >= 64 and a multiple of 8");
    if (!std::isfinite(k_scale) || !(k_scale > 0.f)) return fail(MLA_ERR_INVALID, "k_scale must be finite and > 0");
    if (num_tokens == 0) return MLA_OK;
    if (!kv_c || !k_pe || !slots || !kv) return fail(MLA_ERR_INVALID, "null pointer");
    if (!aligned(kv_c, 16) || !aligned(k_pe, 16) || !aligned(kv, 16) || !aligned(slots, 8))
        return fail(MLA_ERR_INVALID, "misaligned pointer (kv_c, k_pe, kv need 16 bytes, slots 8)");
    if (pool_rows == 0) return fail(MLA_ERR_INVALID, "empty KV pool");
    const int sms = device_sms();
    if (sms <= 0) return fail(MLA_ERR_CUDA, "no CUDA device");
    cudaError_t e = mla::kv_append_launch(kv_c, kv_c_row_stride, k_pe, k_pe_row_stride, slots, num_tokens, k_scale,
                                          kv, pool_rows, sms, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
    return MLA_OK;
}

mla_status mla_debug_wait_timeout(void *stream) {
    if (device_sms() <= 0) return fail(MLA_ERR_CUDA, "no CUDA device");
    cudaError_t e = mla::stuck_wait_launch(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "wait-timeout launch");
    return MLA_OK;
}

mla_status mla_debug_gather(const void *kv, int64_t pool_rows, const int32_t *pages, int64_t num_pages,
                            const int32_t *indptr, int num_requests, int64_t total_rows, void *out,
                            void *stream) {
    if (num_requests < 0 || total_rows < 0 || pool_rows < 0 || num_pages < 0)
        return fail(MLA_ERR_INVALID, "negative size");
    if (total_rows > num_pages) return fail(MLA_ERR_INVALID, "total_rows > num_pages");
    if (total_rows == 0) return MLA_OK;
    if (!kv || !pages || !indptr || !out) return fail(MLA_ERR_INVALID, "null pointer");
    if (pool_rows == 0) return fail(MLA_ERR_INVALID, "empty KV pool");
    if (!aligned(kv, 16) || !aligned(out, 16) || !aligned(pages, 4) || !aligned(indptr, 4))
        return fail(MLA_ERR_INVALID, "misaligned pointer (kv, out need 16 bytes)");
    cudaError_t e = mla::gather_launch(kv, pool_rows, pages, indptr, num_requests, total_rows, out,
                                       static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "gather launch");
    return MLA_OK;
}

mla_status mla_device_status(void *stream, unsigned int *flags) {
    if (!flags) return fail(MLA_ERR_INVALID, "null flags");
    *flags = 0;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    cudaError_t (*readers[])(unsigned int *, bool) = {mla::attend_mma_status, mla::attend_tc_status, mla::merge_status,
                                                      mla::value_gate_status, mla::gather_status,
                                                      mla::kv_append_status};
    for (auto rd : readers) {
        unsigned int f = 0;
        e = rd(&f, true);
        if (e != cudaSuccess) return cuda_fail(e, "status read");
        *flags |= f;
    }
    return MLA_OK;
}

const char *mla_status_string(mla_status s) {
    switch (s) {
        case MLA_OK: return "ok";
        case MLA_ERR_INVALID: return "invalid argument";
        case MLA_ERR_UNSUPPORTED: return "unsupported argument";
        case MLA_ERR_CUDA: return "CUDA error";
        default: return "unknown status";
    }
}

const char *mla_last_error(void) { return g_last_error.c_str(); }

const char *mla_version(void) { return "mla_decode_paged_gb300 0.1 (sm_103a)"; }

}  // extern "C"
