// mla_decode_step_static: the whole decode step (attend, LSE merge, W_UV and
// gate) with its split partials kept in a fixed buffer that the library
// owns, so that the call allocates nothing.
//
// Who needs it: a caller that cannot call cudaMalloc while it runs -- a
// serving loop whose memory is planned up front and that may not ask the
// CUDA allocator for more (its pool is exhausted or the call would block
// on other streams), a host runtime with no device allocator of its own
// (plain C, an embedded engine), or code running in a context where an
// allocation would break its guarantees.  Such a caller can provide the
// step's inputs and outputs, but not the scratch between attend and merge.
//
// The scratch is a file-scope __device__ array of MLA_STATIC_SCRATCH_BYTES.
// Its host-side name is only a stand-in for the symbol, never a device
// address: the address comes from cudaGetSymbolAddress, looked up once per
// device (with that device current) and cached.  The partials then go
// through the same two calls as any other step (mla_decode_attend_planned,
// mla_merge_value_gate); nothing else differs.
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <string>

#include <cuda_runtime.h>

#include "../../include/mla_decode.h"

namespace mla {
void set_last_error(const char *msg);   // api.cu: the text mla_last_error() returns
}

namespace {

// Split partials of one step: o [num_splits, S, heads, 512] bf16 at offset
// 0, then lse [num_splits, S, heads] f32 at the next 256-byte boundary.
// Every GPU that loads this library keeps the array until the process exits.
static __device__ __align__(256) unsigned char g_step_scratch[MLA_STATIC_SCRATCH_BYTES];

// Device address of g_step_scratch on the current device (looked up once
// per device ordinal < 64; later ordinals look it up on every call).
cudaError_t scratch_address(void **addr) {
    static std::atomic<void *> cache[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) {
        void *p = cache[dev].load(std::memory_order_acquire);
        if (p) {
            *addr = p;
            return cudaSuccess;
        }
    }
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_step_scratch);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) cache[dev].store(p, std::memory_order_release);
    *addr = p;
    return cudaSuccess;
}

}  // namespace

extern "C" {

mla_status mla_decode_step_static(const void *q, int64_t q_row_stride, const void *kv, int64_t pool_rows,
                                  const int32_t *pages, int64_t num_pages, const int32_t *indptr,
                                  int num_requests, int qlen, int heads, float scale, float kv_scale,
                                  int num_splits, int split_tokens, const int32_t *plan, int64_t plan_len,
                                  const void *w_uv, const void *gate, const int32_t *lengths, void *out,
                                  void *latent, float *lse_out, void *stream) {
    // Ranges first: the scratch size below is computed from them.
    if (num_requests < 0 || qlen < 1 || qlen > MLA_MAX_QLEN || heads < 1 || heads > MLA_MAX_HEADS ||
        num_splits < 1 || num_splits > MLA_MAX_SPLITS) {
        mla::set_last_error("mla_decode_step_static: num_requests < 0, or qlen, heads or num_splits outside "
                            "1..16, 1..128, 1..256");
        return MLA_ERR_INVALID;
    }
    const int64_t entries = (int64_t)num_splits * num_requests * qlen * heads;
    const int64_t o_bytes = entries * MLA_D_LATENT * 2;
    const int64_t lse_off = (o_bytes + 255) / 256 * 256;
    const int64_t need = lse_off + entries * 4;
    if (need > (int64_t)MLA_STATIC_SCRATCH_BYTES) {
        // Refused before anything is launched; mla_last_error() carries the sizes.
        char msg[200];
        std::snprintf(msg, sizeof msg,
                      "mla_decode_step_static: the split partials need %lld bytes, above the %lld-byte static "
                      "buffer (use fewer splits, or mla_decode_attend with caller buffers)",
                      (long long)need, (long long)MLA_STATIC_SCRATCH_BYTES);
        mla::set_last_error(msg);
        return MLA_ERR_UNSUPPORTED;
    }
    if (num_requests == 0) return MLA_OK;
    void *base = nullptr;
    cudaError_t e = scratch_address(&base);
    if (e != cudaSuccess) {
        mla::set_last_error((std::string("mla_decode_step_static: cudaGetSymbolAddress: ") +
                             cudaGetErrorString(e)).c_str());
        return MLA_ERR_CUDA;
    }
    unsigned char *scratch = static_cast<unsigned char *>(base);
    void *o = scratch;
    float *lse = reinterpret_cast<float *>(scratch + lse_off);
    mla_status s = mla_decode_attend_planned(q, q_row_stride, kv, pool_rows, pages, num_pages, indptr, nullptr, 1,
                                             num_requests, qlen, heads, scale, kv_scale, 1.0f, num_splits,
                                             split_tokens, o, lse, 0u, plan, plan_len, stream);
    if (s != MLA_OK) return s;
    return mla_merge_value_gate(o, lse, num_splits, w_uv, gate, lengths, num_requests, qlen, heads, out, latent,
                                lse_out, stream);
}

}  // extern "C"
