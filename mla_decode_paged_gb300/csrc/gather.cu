// Debug gather of the paged KV rows, through the same row addressing
// (kv_row: page lookup with bounds check) and the same 576-byte bulk copy
// into shared memory that the attend kernels use, so that page indexing can
// be checked byte for byte against a host gather.  Paged rows: vLLM API
// page vllm.models.kimi_k3.amd.specialized_decode.runtime.mla, m1c_inputs
// (kv viewed as one 576-byte row per token, pages = paged_kv_indices,
// indptr).
#include <cuda_runtime.h>

#include "common.cuh"

namespace mla {
namespace {

constexpr int kRowsPerCta = 32;

__global__ void __launch_bounds__(32) gather_kernel(const uint8_t *__restrict__ kv, int64_t pool_rows,
                                                    const int32_t *__restrict__ pages,
                                                    const int32_t *__restrict__ indptr, int R,
                                                    int64_t total_rows, uint8_t *__restrict__ out) {
    __shared__ __align__(128) uint8_t rows[kRowsPerCta][MLA_D_QK];
    __shared__ __align__(8) uint64_t bar;
    const int lane = threadIdx.x;
    const int64_t r0 = (int64_t)blockIdx.x * kRowsPerCta;
    const int64_t rem = total_rows - r0;
    const int n = rem < kRowsPerCta ? (int)rem : kRowsPerCta;
    if (blockIdx.x == 0 && lane == 0 && __ldg(indptr + R) != total_rows) flag(MLA_DEV_BAD_INDPTR);
    if (lane == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(&bar, (uint32_t)n * MLA_D_QK);
    __syncwarp();
    if (lane < n) bulk_g2s(rows[lane], kv_row(kv, pages, r0 + lane, pool_rows), MLA_D_QK, &bar);
    if (!mbar_wait(&bar, 0)) return;
    for (int c = lane; c < n * (MLA_D_QK / 16); c += 32) {
        const int row = c / (MLA_D_QK / 16), ch = c % (MLA_D_QK / 16);
        reinterpret_cast<uint4 *>(out + (r0 + row) * MLA_D_QK)[ch] = reinterpret_cast<const uint4 *>(rows[row])[ch];
    }
}

// One thread waits, through the kernels' own bounded wait (mbar_wait), on
// an mbarrier that nothing arrives at and no copy completes: after the wait
// budget it flags MLA_DEV_TIMEOUT and the kernel returns.  Nothing is in
// flight when it exits.
__global__ void __launch_bounds__(32) stuck_wait_kernel() {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
        mbar_wait(&bar, 0);
    }
}

}  // namespace

cudaError_t stuck_wait_launch(cudaStream_t st) {
    stuck_wait_kernel<<<1, 32, 0, st>>>();
    return cudaGetLastError();
}

cudaError_t gather_launch(const void *kv, int64_t pool_rows, const int32_t *pages, const int32_t *indptr,
                          int R, int64_t total_rows, void *out, cudaStream_t st) {
    if (total_rows == 0) return cudaSuccess;
    const int64_t blocks = (total_rows + kRowsPerCta - 1) / kRowsPerCta;
    gather_kernel<<<(unsigned)blocks, 32, 0, st>>>(static_cast<const uint8_t *>(kv), pool_rows, pages, indptr,
                                                   R, total_rows, static_cast<uint8_t *>(out));
    return cudaGetLastError();
}

cudaError_t gather_status(unsigned int *flags, bool clear) { return read_status(flags, clear); }

}  // namespace mla
