// Absorbed W_UV projection fused with the sigmoid gate -- tcgen05 kernel.
//
// What it computes: vLLM API page
// vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.mla.value --
// MlaValue (the [B, H, 512] bf16 latent times W_UV [H, 128, 512], latent
// axis contiguous, bf16 MMA with fp32 accumulation; rows are tokens, qlen
// per request) and MlaGate (the value rounded to bf16, times the fp32
// sigmoid of the raw gate, rounded to bf16; rows of empty requests are 0,
// chosen by a select so a NaN gate never leaks).
//
// Design: one CTA per (64 query rows, head), 512 threads.  The head's whole
// W_UV slice [128 x 512] and the 64 latent rows [64 x 512] arrive by TMA in
// one round trip, K-major with 128B swizzle (eight 64-element column blocks
// each); they are the A (M = 128 output columns) and B (N = 64 rows)
// operands of 32 bf16 tcgen05 MMAs (K = 16) issued by one thread into a
// 64-column f32 TMEM accumulator D[v][row].  The epilogue reads D (four
// warps, thread = output column v = TMEM lane), rounds the value to bf16
// into a shared [64][128] tile, then all 16 warps write each row's 128
// outputs with coalesced 4-byte stores (the gate words, loaded the same way, are in flight during the
// copies and MMAs).  The W_UV slice is read before the wait on
// the previous kernel (programmatic dependent launch); the latent, gate and
// lengths after it.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "tc.cuh"

namespace mla {
namespace {

constexpr int kRows = 64;                                  // query rows per CTA (MMA N)
constexpr int kThreads = 512;                              // warps 0-3 read TMEM; all write
constexpr int kColBlocks = MLA_D_LATENT / 64;              // 128-byte column blocks of the K axis
constexpr int kABlock = MLA_D_V * 128;                     // one column block of W_UV[h]: 16 KB
constexpr int kBBlock = kRows * 128;                       // one column block of the latent rows: 8 KB
constexpr int kAOff = 0, kBOff = kColBlocks * kABlock;     // 128 KB, then 64 KB
constexpr int kSmem = kBOff + kColBlocks * kBBlock + 1024; // + alignment slack
constexpr uint32_t kTmemCols = 64;

// kind::f16 instruction descriptor: bf16 A and B (K-major), f32 D, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kRows >> 3) << 17) |
                            ((uint32_t)(128 >> 4) << 24);

__device__ __forceinline__ void mma_bf16_tc(uint32_t d_tmem, uint64_t a, uint64_t b, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(kIdesc), "r"((uint32_t)accumulate));
}

__device__ __forceinline__ void tma_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_3d(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
        "%4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// 1 / (1 + e^-x) in fp32 from the hardware exponential and reciprocal
// approximations (relative errors near 2^-21 and 2^-23, far below the bf16
// rounding of the product); e^-x = inf gives 0.
__device__ __forceinline__ float sigmoid_f32(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + __expf(-x)));
    return r;
}

__global__ void __launch_bounds__(kThreads, 1)
    value_gate_kernel(const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap ml,
                      const __nv_bfloat16 *__restrict__ gate, const int32_t *__restrict__ lengths, int S, int qlen,
                      int H, __nv_bfloat16 *__restrict__ out) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t full_w, full_l, done;
    __shared__ uint32_t tmem;
    __shared__ int active[kRows];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = blockIdx.x * kRows, h = blockIdx.y;
    const int nrows = min(kRows, S - t0);

    if (tid == 0) {
        mbar_init(&full_w, 1);
        mbar_init(&full_l, 1);
        mbar_init(&done, 1);
        mbar_fence_init();
    }
    if (warp == 0) tc::tmem_alloc(&tmem, kTmemCols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (tid == 0) {
        // W_UV is not written by the kernel before this one: fetch it first.
        mbar_arrive_expect_tx(&full_w, kColBlocks * kABlock);
        for (int kb = 0; kb < kColBlocks; ++kb) tma_2d(sm + kAOff + kb * kABlock, &mw, 64 * kb, MLA_D_V * h, &full_w);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (tid == 0) {
        // Rows past S read as zeros (their outputs are not written).
        mbar_arrive_expect_tx(&full_l, kColBlocks * kBBlock);
        for (int kb = 0; kb < kColBlocks; ++kb) tma_3d(sm + kBOff + kb * kBBlock, &ml, 64 * kb, h, t0, &full_l);
    }
    if (tid < kRows) active[tid] = tid < nrows && __ldg(lengths + (t0 + tid) / qlen) > 0;
    // This thread's gate words (bf16 pairs w = tid + 128 k: row w / 64, pair
    // w % 64), loaded while the copies and the MMAs are in flight.
    constexpr int kPairs = kRows * (MLA_D_V / 2) / kThreads;
    uint32_t gw[kPairs];
#pragma unroll
    for (int k = 0; k < kPairs; ++k) {
        const int w = tid + kThreads * k, r = w / (MLA_D_V / 2), p = w - r * (MLA_D_V / 2);
        gw[k] = r < nrows ? __ldg(reinterpret_cast<const uint32_t *>(gate + ((long long)(t0 + r) * H + h) * MLA_D_V +
                                                                      2 * p))
                          : 0u;
    }

    const uint32_t base = smem_u32(sm), tm = tmem;
    bool ok = true, issued = false;
    if (tid == 0) {
        ok = mbar_wait(&full_w, 0) && mbar_wait(&full_l, 0);
        if (ok) {
            issued = true;
            tc::fence_after();
#pragma unroll
            for (int j = 0; j < MLA_D_LATENT / 16; ++j) {
                const int kb = j >> 2, off = (j & 3) * 32;
                mma_bf16_tc(tm, tc::sdesc(base + kAOff + kb * kABlock + off, 16, 1024, tc::kSw128),
                            tc::sdesc(base + kBOff + kb * kBBlock + off, 16, 1024, tc::kSw128), j > 0);
            }
            tc::commit(&done);
        }
    }
    ok = __syncthreads_and(ok);
    if (ok) ok = mbar_wait(&done, 0);
    ok = __syncthreads_and(ok);
    if (!ok) {
        // Flagged.  Before the CTA exits let the copies and MMAs in flight
        // finish (one more bounded wait each), then release TMEM.
        if (tid == 0) {
            mbar_wait(&full_w, 0);
            mbar_wait(&full_l, 0);
            if (issued) mbar_wait(&done, 0);
        }
        tc::fence_before();
        __syncthreads();
        if (warp == 0) tc::tmem_free(tm, kTmemCols);
        return;
    }
    tc::fence_after();

    // D[v][row] -> bf16(value) in a [64][128] tile (the W_UV slice is no
    // longer read: its first 16 KB hold the tile); warps 0-3 cover the 128
    // TMEM lanes.
    __nv_bfloat16 *tile = reinterpret_cast<__nv_bfloat16 *>(sm + kAOff);
    if (warp < 4) {
        const int v = 32 * warp + lane;
#pragma unroll
        for (int c = 0; c < kRows; c += 16) {
            float d[16];
            tc::ld16(tm + ((uint32_t)(32 * warp) << 16) + c, d);
            tc::wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) tile[(c + i) * MLA_D_V + v] = __float2bfloat16_rn(d[i]);
        }
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_free(tm, kTmemCols);

    // Row by row, 64 bf16 pairs per row: out = bf16(value * sigmoid(gate)),
    // 0 for rows of empty requests (selected, so a NaN gate never leaks).
    const uint32_t *tile2 = reinterpret_cast<const uint32_t *>(tile);
#pragma unroll
    for (int k = 0; k < kPairs; ++k) {
        const int w = tid + kThreads * k, r = w / (MLA_D_V / 2), p = w - r * (MLA_D_V / 2);
        if (r >= nrows) break;
        uint32_t res = 0u;
        if (active[r]) {
            const uint32_t val = tile2[w], g = gw[k];
            res = pack_bf16x2(bf16_lo(val) * sigmoid_f32(bf16_lo(g)), bf16_hi(val) * sigmoid_f32(bf16_hi(g)));
        }
        *reinterpret_cast<uint32_t *>(out + ((long long)(t0 + r) * H + h) * MLA_D_V + 2 * p) = res;
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &p, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

}  // namespace

// latent [S, H, 512] and w_uv [H, 128, 512] bf16 (16-byte aligned); gate
// [S, H*128] bf16 and out (4-byte aligned).
cudaError_t value_gate_launch(const void *latent, const void *w_uv, const void *gate,
                              const int32_t *lengths, int R, int qlen, int H, void *out, cudaStream_t st) {
    const int S = R * qlen;
    if (S == 0) return cudaSuccess;
    // W_UV as [H*128 rows, 512] and the latent as [S][H][512], 64-element
    // (128-byte) boxes with 128B swizzle: the UMMA K-major layout.  Encoded
    // once per (device, buffer, shape) and reused while a thread keeps
    // launching on the same buffers.
    struct MapCache {
        int dev;
        const void *ptr;
        int S, H;
        CUtensorMap map;
    };
    static thread_local MapCache cw = {-1, nullptr, 0, 0, {}}, cl = {-1, nullptr, 0, 0, {}};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (cw.dev != dev || cw.ptr != w_uv || cw.H != H || cl.dev != dev || cl.ptr != latent || cl.S != S || cl.H != H) {
        PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
        if (!enc) return cudaErrorNotSupported;
        if (cw.dev != dev || cw.ptr != w_uv || cw.H != H) {
            cw.dev = -1;
            cuuint64_t dim[2] = {(cuuint64_t)MLA_D_LATENT, (cuuint64_t)H * MLA_D_V};
            cuuint64_t stride[1] = {(cuuint64_t)MLA_D_LATENT * 2};
            cuuint32_t box[2] = {64, (cuuint32_t)MLA_D_V}, es[2] = {1, 1};
            if (enc(&cw.map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(w_uv), dim, stride, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return cudaErrorInvalidValue;
            cw.dev = dev;
            cw.ptr = w_uv;
            cw.H = H;
        }
        if (cl.dev != dev || cl.ptr != latent || cl.S != S || cl.H != H) {
            cl.dev = -1;
            cuuint64_t dim[3] = {(cuuint64_t)MLA_D_LATENT, (cuuint64_t)H, (cuuint64_t)S};
            cuuint64_t stride[2] = {(cuuint64_t)MLA_D_LATENT * 2, (cuuint64_t)H * MLA_D_LATENT * 2};
            cuuint32_t box[3] = {64, 1, (cuuint32_t)kRows}, es[3] = {1, 1, 1};
            if (enc(&cl.map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(latent), dim, stride, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return cudaErrorInvalidValue;
            cl.dev = dev;
            cl.ptr = latent;
            cl.S = S;
            cl.H = H;
        }
    }
    const CUtensorMap &mw = cw.map, &ml = cl.map;
    cudaError_t e = smem_attr_once<value_gate_kernel>(kSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((S + kRows - 1) / kRows, H, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, value_gate_kernel, mw, ml, static_cast<const __nv_bfloat16 *>(gate), lengths,
                              S, qlen, H, static_cast<__nv_bfloat16 *>(out));
}

cudaError_t value_gate_status(unsigned int *flags, bool clear) { return read_status(flags, clear); }

}  // namespace mla
