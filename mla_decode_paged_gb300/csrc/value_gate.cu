// Absorbed W_UV projection fused with the sigmoid gate.
//
// What it computes: vLLM API page
// vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.mla.value --
// MlaValue (the [B, H, 512] bf16 latent times W_UV [H, 128, 512], latent
// axis contiguous, bf16 MMA with fp32 accumulation; rows are tokens, qlen
// per request) and MlaGate (the value rounded to bf16, times the fp32
// sigmoid of the raw gate, rounded to bf16; rows of empty requests are 0,
// chosen by a select so a NaN gate never leaks).
//
// Design: one CTA per (64 rows, head, 32 output columns); 4 warps, each
// 16 rows x 32 columns (4 m16n8k16 tiles).  The whole 512-wide latent axis
// of the CTA's 64 latent rows and 32 W_UV rows arrives in one round trip:
// one warp issues a 1 KB cp.async.bulk per row into padded smem rows
// (stride 1040 B, so ldmatrix is conflict-free) on one mbarrier.  W_UV rows
// are the B operand's n index and their latent axis the k index, which is
// the "col" B layout ldmatrix delivers without a transpose.
#include <cuda_runtime.h>

#include "common.cuh"

namespace mla {
namespace {

constexpr int kRows = 64, kCols = 32, kStride = MLA_D_LATENT + 8;  // bf16 elements per smem row
constexpr int kThreads = 128;

struct Smem {
    __nv_bfloat16 a[kRows][kStride];
    __nv_bfloat16 b[kCols][kStride];
    uint64_t bar;
};

__device__ __forceinline__ float sigmoid_f32(float x) { return 1.f / (1.f + expf(-x)); }

__global__ void __launch_bounds__(kThreads) value_gate_kernel(
    const __nv_bfloat16 *__restrict__ latent, const __nv_bfloat16 *__restrict__ w_uv,
    const __nv_bfloat16 *__restrict__ gate, const int32_t *__restrict__ lengths, int S, int qlen,
    int H, __nv_bfloat16 *__restrict__ out) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, qd = lane & 3;
    const int t0 = blockIdx.x * kRows, h = blockIdx.y, v0 = blockIdx.z * kCols;
    const int nrows = min(kRows, S - t0);

    if (tid == 0) {
        mbar_init(&sm.bar, 1);
        mbar_fence_init();
    }
    __syncthreads();
    if (warp == 0) {
        if (lane == 0) mbar_arrive_expect_tx(&sm.bar, (uint32_t)(nrows + kCols) * MLA_D_LATENT * 2);
        __syncwarp();
        for (int i = lane; i < nrows + kCols; i += 32) {
            if (i < nrows)
                bulk_g2s(sm.a[i], latent + ((long long)(t0 + i) * H + h) * MLA_D_LATENT, MLA_D_LATENT * 2, &sm.bar);
            else
                bulk_g2s(sm.b[i - nrows], w_uv + ((long long)h * MLA_D_V + v0 + i - nrows) * MLA_D_LATENT,
                         MLA_D_LATENT * 2, &sm.bar);
        }
    }
    // Gate words and the row activity do not depend on the MMA: load them
    // while the bulk copies are in flight.
    uint32_t gw[2][4];
    bool active[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int t = t0 + 16 * warp + 8 * hh + g;
        active[hh] = t < S && __ldg(lengths + t / qlen) > 0;
        const long long rowoff = (long long)t * H * MLA_D_V + (long long)h * MLA_D_V + v0;
#pragma unroll
        for (int n = 0; n < 4; ++n)
            gw[hh][n] = active[hh] ? __ldg(reinterpret_cast<const uint32_t *>(gate + rowoff + 8 * n + 2 * qd)) : 0u;
    }
    if (!mbar_wait(&sm.bar, 0)) {
        // Flagged; before the CTA may exit (and its shared memory be reused)
        // give the bulk copies one more bounded wait to land.
        mbar_wait(&sm.bar, 0);
        return;
    }

    float acc[4][4];
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;
    if (16 * warp < nrows) {
#pragma unroll 8
        for (int ks = 0; ks < MLA_D_LATENT / 16; ++ks) {
            uint32_t a[4];
            ldmatrix_x4(a, &sm.a[16 * warp + (lane & 15)][16 * ks + (lane >> 4) * 8]);
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                uint32_t b[4];
                ldmatrix_x4(b, &sm.b[16 * np + (lane & 7) + ((lane >> 4) << 3)][16 * ks + ((lane >> 3) & 1) * 8]);
                mma_bf16(acc[2 * np], a, b[0], b[1]);
                mma_bf16(acc[2 * np + 1], a, b[2], b[3]);
            }
        }
    }

    // Epilogue: bf16(value) * sigmoid(gate) -> bf16; empty requests -> 0.
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int t = t0 + 16 * warp + 8 * hh + g;
        if (t >= S) continue;
        const long long rowoff = (long long)t * H * MLA_D_V + (long long)h * MLA_D_V + v0;
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            uint32_t res = 0u;
            if (active[hh]) {
                const float v_lo = __bfloat162float(__float2bfloat16_rn(acc[n][2 * hh]));
                const float v_hi = __bfloat162float(__float2bfloat16_rn(acc[n][2 * hh + 1]));
                res = pack_bf16x2(v_lo * sigmoid_f32(bf16_lo(gw[hh][n])), v_hi * sigmoid_f32(bf16_hi(gw[hh][n])));
            }
            *reinterpret_cast<uint32_t *>(out + rowoff + 8 * n + 2 * qd) = res;
        }
    }
}

}  // namespace

cudaError_t value_gate_launch(const void *latent, const void *w_uv, const void *gate,
                              const int32_t *lengths, int R, int qlen, int H, void *out, cudaStream_t st) {
    const int S = R * qlen;
    if (S == 0) return cudaSuccess;
    const size_t smem = sizeof(Smem);
    cudaError_t e = smem_attr_once<value_gate_kernel>((int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((S + kRows - 1) / kRows, H, MLA_D_V / kCols);
    value_gate_kernel<<<grid, kThreads, smem, st>>>(
        static_cast<const __nv_bfloat16 *>(latent), static_cast<const __nv_bfloat16 *>(w_uv),
        static_cast<const __nv_bfloat16 *>(gate), lengths, S, qlen, H, static_cast<__nv_bfloat16 *>(out));
    return cudaGetLastError();
}

cudaError_t value_gate_status(unsigned int *flags, bool clear) { return read_status(flags, clear); }

}  // namespace mla
