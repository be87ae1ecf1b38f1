// LSE merge of split-KV partials into the latent.
//
// What it computes: vLLM API page
// vllm.models.kimi_k3.amd.specialized_decode.runtime.mla -- m1c_inputs
// (partials o [splits, S, H, 512] bf16, LSE [splits, S, H] f32, "M1b
// merges the splits") and post (the same LSE combine across ranks):
//   LSE = ln sum_k exp(lse_k);  latent = sum_k exp(lse_k - LSE) o_k,
// skipping splits whose lse is -inf (their o is never read).
//
// Bandwidth-bound: one warp per (row, head); each lane owns 16 of the 512
// latent columns as two 16-byte vectors, so a split's 1 KB row is read
// with fully coalesced 512-byte warp accesses.  The split weights are held
// one per lane (32 splits per pass) and broadcast with shuffles.
#include <cuda_runtime.h>

#include "common.cuh"

namespace mla {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ void fma8(float (&acc)[8], float w, uint4 v) {
    acc[0] += w * bf16_lo(v.x); acc[1] += w * bf16_hi(v.x);
    acc[2] += w * bf16_lo(v.y); acc[3] += w * bf16_hi(v.y);
    acc[4] += w * bf16_lo(v.z); acc[5] += w * bf16_hi(v.z);
    acc[6] += w * bf16_lo(v.w); acc[7] += w * bf16_hi(v.w);
}

__global__ void __launch_bounds__(kWarps * 32) merge_kernel(const __nv_bfloat16 *__restrict__ o,
                                                            const float *__restrict__ lse,
                                                            int num_splits, long long nrow,
                                                            __nv_bfloat16 *__restrict__ latent,
                                                            float *__restrict__ lse_out) {
    // A kernel launched after this one with programmatic dependent launch
    // (the W_UV + gate kernel) may start now; it waits for this grid's
    // completion before it reads what this kernel writes.
    asm volatile("griddepcontrol.launch_dependents;");
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (row >= nrow) return;

    float mx = -INFINITY;
    for (int k = lane; k < num_splits; k += 32) mx = fmaxf(mx, __ldg(lse + (long long)k * nrow + row));
#pragma unroll
    for (int d = 16; d; d >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));

    float a0[8], a1[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) a0[e] = a1[e] = 0.f;
    float tot = 0.f;
    if (mx > -INFINITY) {
        for (int kb = 0; kb < num_splits; kb += 32) {
            const int k = kb + lane;
            float w = 0.f;
            bool valid = false;
            if (k < num_splits) {
                const float l = __ldg(lse + (long long)k * nrow + row);
                valid = l > -INFINITY;
                w = valid ? expf(l - mx) : 0.f;
            }
            tot += w;
            // Valid splits of this pass, four at a time: their loads are
            // independent, so they are all in flight together.
            unsigned m = __ballot_sync(0xffffffffu, valid);
            while (m) {
                int src[4];
                float ws[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    src[j] = m ? __ffs(m) - 1 : -1;
                    if (m) m &= m - 1;
                }
                uint4 v0[4], v1[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    ws[j] = __shfl_sync(0xffffffffu, w, src[j] < 0 ? 0 : src[j]);
                    if (src[j] >= 0) {
                        const uint4 *p = reinterpret_cast<const uint4 *>(
                            o + ((long long)(kb + src[j]) * nrow + row) * MLA_D_LATENT);
                        v0[j] = __ldg(p + lane);
                        v1[j] = __ldg(p + 32 + lane);
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (src[j] >= 0) {
                        fma8(a0, ws[j], v0[j]);
                        fma8(a1, ws[j], v1[j]);
                    }
                }
            }
        }
#pragma unroll
        for (int d = 16; d; d >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, d);
    }
    const float inv = tot > 0.f ? 1.f / tot : 0.f;
    uint4 r0, r1;
    r0.x = pack_bf16x2(a0[0] * inv, a0[1] * inv); r0.y = pack_bf16x2(a0[2] * inv, a0[3] * inv);
    r0.z = pack_bf16x2(a0[4] * inv, a0[5] * inv); r0.w = pack_bf16x2(a0[6] * inv, a0[7] * inv);
    r1.x = pack_bf16x2(a1[0] * inv, a1[1] * inv); r1.y = pack_bf16x2(a1[2] * inv, a1[3] * inv);
    r1.z = pack_bf16x2(a1[4] * inv, a1[5] * inv); r1.w = pack_bf16x2(a1[6] * inv, a1[7] * inv);
    uint4 *dst = reinterpret_cast<uint4 *>(latent + row * MLA_D_LATENT);
    dst[lane] = r0;
    dst[32 + lane] = r1;
    if (lse_out && lane == 0) lse_out[row] = tot > 0.f ? mx + logf(tot) : -INFINITY;
}

}  // namespace

cudaError_t merge_launch(const void *o, const float *lse, int num_splits, int rows, int heads,
                         void *latent, float *lse_out, cudaStream_t st) {
    const long long nrow = (long long)rows * heads;
    if (nrow == 0) return cudaSuccess;
    const long long blocks = (nrow + kWarps - 1) / kWarps;
    merge_kernel<<<(unsigned)blocks, kWarps * 32, 0, st>>>(static_cast<const __nv_bfloat16 *>(o), lse,
                                                         num_splits, nrow,
                                                         static_cast<__nv_bfloat16 *>(latent), lse_out);
    return cudaGetLastError();
}

cudaError_t merge_status(unsigned int *flags, bool clear) { return read_status(flags, clear); }

}  // namespace mla
