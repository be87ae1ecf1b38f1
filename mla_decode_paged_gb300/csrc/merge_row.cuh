// One (row, head) of the LSE merge of split-KV partials, by one warp.
//
// What it computes: vLLM API page
// vllm.models.kimi_k3.amd.specialized_decode.runtime.mla -- m1c_inputs
// (the split partials are merged by their LSE) and post (the same LSE
// combine across ranks):
//   LSE = ln sum_k exp(lse_k);  latent = sum_k exp(lse_k - LSE) o_k,
// skipping splits whose lse is -inf (their o is never read).
//
// Shared by the merge kernel and the fused merge + W_UV kernel, so both
// produce the same bits.  Each lane owns 16 of the 512 latent columns as two
// 16-byte vectors (columns 8 lane .. 8 lane + 7 and 256 + 8 lane ..); the
// split weights are held one per lane (32 splits per pass) and broadcast
// with shuffles; a pass's valid splits are loaded four at a time.
#pragma once

#include "common.cuh"

namespace mla {

__device__ __forceinline__ void merge_fma8(float (&acc)[8], float w, uint4 v) {
    acc[0] += w * bf16_lo(v.x); acc[1] += w * bf16_hi(v.x);
    acc[2] += w * bf16_lo(v.y); acc[3] += w * bf16_hi(v.y);
    acc[4] += w * bf16_lo(v.z); acc[5] += w * bf16_hi(v.z);
    acc[6] += w * bf16_lo(v.w); acc[7] += w * bf16_hi(v.w);
}

// o [num_splits, nrow, 512] bf16, lse [num_splits, nrow] f32 (nrow = rows x
// heads); `row` indexes the nrow axis.  On return (every lane): r0 / r1 the
// lane's two 16-byte vectors of the bf16 latent, and lse_row the merged LSE
// (-inf for a row whose splits are all empty, whose latent is then 0).
__device__ __forceinline__ void merge_row(const __nv_bfloat16 *__restrict__ o, const float *__restrict__ lse,
                                          int num_splits, long long nrow, long long row, int lane, uint4 &r0,
                                          uint4 &r1, float &lse_row) {
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
                        merge_fma8(a0, ws[j], v0[j]);
                        merge_fma8(a1, ws[j], v1[j]);
                    }
                }
            }
        }
#pragma unroll
        for (int d = 16; d; d >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, d);
    }
    const float inv = tot > 0.f ? 1.f / tot : 0.f;
    r0.x = pack_bf16x2(a0[0] * inv, a0[1] * inv); r0.y = pack_bf16x2(a0[2] * inv, a0[3] * inv);
    r0.z = pack_bf16x2(a0[4] * inv, a0[5] * inv); r0.w = pack_bf16x2(a0[6] * inv, a0[7] * inv);
    r1.x = pack_bf16x2(a1[0] * inv, a1[1] * inv); r1.y = pack_bf16x2(a1[2] * inv, a1[3] * inv);
    r1.z = pack_bf16x2(a1[4] * inv, a1[5] * inv); r1.w = pack_bf16x2(a1[6] * inv, a1[7] * inv);
    lse_row = tot > 0.f ? mx + logf(tot) : -INFINITY;
}

}  // namespace mla
