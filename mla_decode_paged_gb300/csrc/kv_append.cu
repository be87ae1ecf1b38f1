// KV-cache append: new tokens' kv_c (512) and k_pe (64), divided by
// k_scale and converted to fp8 e4m3, written to their slots of the flat
// token rows.
//
// What it computes: vLLM API page
// vllm.models.kimi_k3.amd.specialized_decode.runtime.mla, pre
// (do_kv_cache_update: the cache rows the decode step reads are written
// with _k_scale).  The conversion saturates (CUDA's satfinite: magnitudes
// above 448 and infinities become +-448, NaN stays NaN), the quotient is
// formed in float32 with IEEE division.
//
// Design: a scatter bound by its instruction issue (the division above is
// most of it) more than by DRAM.  One thread per 16 elements of a row (36
// per token: 32 from kv_c, 4 from k_pe): two 16-byte loads of 8 bf16, eight
// two-element conversions, one 16-byte store into the slot's row; a token's
// index and slot are found once per 16 elements (measured 17 % faster than
// one thread per 8 elements, and no slower for a few thousand tokens).
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace mla {
namespace {

constexpr int kUnits = MLA_D_QK / 16;        // 36 sixteen-element units per row
constexpr int kLatUnits = MLA_D_LATENT / 16;  // 32 of them from kv_c
constexpr int kThreads = 256;

// Eight bf16 (one 16-byte vector) -> eight e4m3 codes (8 bytes).
__device__ __forceinline__ uint2 to_e4m3x8(uint4 v, float k_scale) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t out[2];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 x = make_float2(__fdiv_rn(bf16_lo(w[e]), k_scale), __fdiv_rn(bf16_hi(w[e]), k_scale));
        const uint32_t c = __nv_cvt_float2_to_fp8x2(x, __NV_SATFINITE, __NV_E4M3);
        if (e & 1) out[e >> 1] |= c << 16;
        else out[e >> 1] = c;
    }
    return make_uint2(out[0], out[1]);
}

__global__ void __launch_bounds__(kThreads) kv_append_kernel(
    const __nv_bfloat16 *__restrict__ kv_c, int64_t kv_c_stride, const __nv_bfloat16 *__restrict__ k_pe,
    int64_t k_pe_stride, const int64_t *__restrict__ slots, int64_t T, float k_scale, uint8_t *__restrict__ kv,
    int64_t pool_rows) {
    const int64_t n = T * kUnits;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n; i += (int64_t)gridDim.x * kThreads) {
        const int64_t tok = i / kUnits;
        const int u = (int)(i - tok * kUnits);
        const int64_t slot = __ldg(slots + tok);
        if (slot < 0) continue;                 // padding token
        if (slot >= pool_rows) {
            if (u == 0) flag(MLA_DEV_BAD_PAGE);
            continue;
        }
        const uint4 *src = reinterpret_cast<const uint4 *>(u < kLatUnits ? kv_c + tok * kv_c_stride + u * 16
                                                                         : k_pe + tok * k_pe_stride + (u - kLatUnits) * 16);
        const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
        const uint2 a = to_e4m3x8(v0, k_scale), b = to_e4m3x8(v1, k_scale);
        *reinterpret_cast<uint4 *>(kv + slot * MLA_D_QK + u * 16) = make_uint4(a.x, a.y, b.x, b.y);
    }
}

}  // namespace

cudaError_t kv_append_launch(const void *kv_c, int64_t kv_c_stride, const void *k_pe, int64_t k_pe_stride,
                             const int64_t *slots, int64_t T, float k_scale, void *kv, int64_t pool_rows, int sms,
                             cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const int64_t blocks_needed = (T * kUnits + kThreads - 1) / kThreads;
    const int grid = (int)(blocks_needed < (int64_t)sms * 8 ? blocks_needed : (int64_t)sms * 8);
    kv_append_kernel<<<grid, kThreads, 0, st>>>(static_cast<const __nv_bfloat16 *>(kv_c), kv_c_stride,
                                                static_cast<const __nv_bfloat16 *>(k_pe), k_pe_stride, slots, T,
                                                k_scale, static_cast<uint8_t *>(kv), pool_rows);
    return cudaGetLastError();
}

cudaError_t kv_append_status(unsigned int *flags, bool clear) { return read_status(flags, clear); }

}  // namespace mla
