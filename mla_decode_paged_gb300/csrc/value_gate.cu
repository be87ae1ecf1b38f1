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
// Design: one CTA per (64 rows, head, 64-column half); 4 warps, each 16
// rows x 64 columns (8 m16n8k16 tiles).  The 512-wide latent axis streams
// through smem in 64-wide chunks with double-buffered 16-byte cp.async;
// ldmatrix feeds both operands (W_UV rows are the B operand's n index, its
// latent axis the k index, which is exactly the "col" B layout).
#include <cuda_runtime.h>

#include "common.cuh"

namespace mla {
namespace {

constexpr int kRows = 64, kCols = 64, kChunk = 64, kStride = kChunk + 8;  // bf16 elements
constexpr int kThreads = 128;

struct Smem {
    __nv_bfloat16 a[2][kRows][kStride];
    __nv_bfloat16 b[2][kCols][kStride];
};

__device__ __forceinline__ void cp_async16_zfill(void *dst, const void *src, bool valid) {
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(n)
                 : "memory");
}

__device__ __forceinline__ float sigmoid_f32(float x) { return 1.f / (1.f + expf(-x)); }

__global__ void __launch_bounds__(kThreads) value_gate_kernel(
    const __nv_bfloat16 *__restrict__ latent, const __nv_bfloat16 *__restrict__ w_uv,
    const __nv_bfloat16 *__restrict__ gate, const int32_t *__restrict__ lengths, int S, int qlen,
    int H, __nv_bfloat16 *__restrict__ out) {
    __shared__ __align__(128) Smem sm;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, qd = lane & 3;
    const int t0 = blockIdx.x * kRows, h = blockIdx.y, v0 = blockIdx.z * kCols;

    auto load = [&](int buf, int c0) {
        for (int c = tid; c < kRows * (kChunk / 8); c += kThreads) {
            const int row = c >> 3, ch = c & 7;
            const int t = t0 + row;
            const bool ok = t < S;
            const __nv_bfloat16 *src = latent + ((long long)(ok ? t : 0) * H + h) * MLA_D_LATENT + c0 + ch * 8;
            cp_async16_zfill(&sm.a[buf][row][ch * 8], src, ok);
        }
        for (int c = tid; c < kCols * (kChunk / 8); c += kThreads) {
            const int row = c >> 3, ch = c & 7;
            const __nv_bfloat16 *src = w_uv + ((long long)h * MLA_D_V + v0 + row) * MLA_D_LATENT + c0 + ch * 8;
            cp_async16(&sm.b[buf][row][ch * 8], src);
        }
        cp_async_commit();
    };

    float acc[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[n][e] = 0.f;

    constexpr int kNChunks = MLA_D_LATENT / kChunk;
    load(0, 0);
    for (int c = 0; c < kNChunks; ++c) {
        if (c + 1 < kNChunks) {
            load((c + 1) & 1, (c + 1) * kChunk);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const int buf = c & 1;
#pragma unroll
        for (int ks = 0; ks < kChunk / 16; ++ks) {
            uint32_t a[4];
            ldmatrix_x4(a, &sm.a[buf][16 * warp + (lane & 15)][16 * ks + (lane >> 4) * 8]);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t b[4];
                ldmatrix_x4(b, &sm.b[buf][16 * np + (lane & 7) + ((lane >> 4) << 3)][16 * ks + ((lane >> 3) & 1) * 8]);
                mma_bf16(acc[2 * np], a, b[0], b[1]);
                mma_bf16(acc[2 * np + 1], a, b[2], b[3]);
            }
        }
        __syncthreads();
    }

    // Epilogue: bf16(value) * sigmoid(gate) -> bf16; empty requests -> 0.
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int t = t0 + 16 * warp + 8 * hh + g;
        if (t >= S) continue;
        const bool active = __ldg(lengths + t / qlen) > 0;
        const long long rowoff = (long long)t * H * MLA_D_V + (long long)h * MLA_D_V + v0;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            const int col = 8 * n + 2 * qd;
            uint32_t res = 0u;
            if (active) {
                const uint32_t gw = __ldg(reinterpret_cast<const uint32_t *>(gate + rowoff + col));
                const float v_lo = __bfloat162float(__float2bfloat16_rn(acc[n][2 * hh]));
                const float v_hi = __bfloat162float(__float2bfloat16_rn(acc[n][2 * hh + 1]));
                res = pack_bf16x2(v_lo * sigmoid_f32(bf16_lo(gw)), v_hi * sigmoid_f32(bf16_hi(gw)));
            }
            *reinterpret_cast<uint32_t *>(out + rowoff + col) = res;
        }
    }
}

}  // namespace

cudaError_t value_gate_launch(const void *latent, const void *w_uv, const void *gate,
                              const int32_t *lengths, int R, int qlen, int H, void *out, cudaStream_t st) {
    const int S = R * qlen;
    if (S == 0) return cudaSuccess;
    dim3 grid((S + kRows - 1) / kRows, H, MLA_D_V / kCols);
    value_gate_kernel<<<grid, kThreads, 0, st>>>(
        static_cast<const __nv_bfloat16 *>(latent), static_cast<const __nv_bfloat16 *>(w_uv),
        static_cast<const __nv_bfloat16 *>(gate), lengths, S, qlen, H, static_cast<__nv_bfloat16 *>(out));
    return cudaGetLastError();
}

cudaError_t value_gate_status(unsigned int *flags, bool clear) { return read_status(flags, clear); }

}  // namespace mla
