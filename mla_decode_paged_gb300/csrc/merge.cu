// LSE merge of split-KV partials into the latent.
//
// What it computes: vLLM API page
// vllm.models.kimi_k3.amd.specialized_decode.runtime.mla -- m1c_inputs
// (partials o [splits, S, H, 512] bf16 and LSE [splits, S, H] f32, merged
// by their LSE in the step after attention) and post (the same LSE combine
// across ranks):
//   LSE = ln sum_k exp(lse_k);  latent = sum_k exp(lse_k - LSE) o_k,
// skipping splits whose lse is -inf (their o is never read).
//
// Bandwidth-bound: one warp per (row, head), the row arithmetic in
// merge_row.cuh (shared with the fused merge + W_UV kernel).
#include <cuda_runtime.h>

#include "common.cuh"
#include "merge_row.cuh"

namespace mla {
namespace {

constexpr int kWarps = 8;

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
    uint4 r0, r1;
    float lse_row;
    merge_row(o, lse, num_splits, nrow, row, lane, r0, r1, lse_row);
    uint4 *dst = reinterpret_cast<uint4 *>(latent + row * MLA_D_LATENT);
    dst[lane] = r0;
    dst[32 + lane] = r1;
    if (lse_out && lane == 0) lse_out[row] = lse_row;
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
