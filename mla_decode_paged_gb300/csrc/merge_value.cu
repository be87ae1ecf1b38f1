// Split merge fused with the absorbed W_UV projection and the sigmoid gate.
//
// What it computes: vLLM API page
// vllm.models.kimi_k3.amd.specialized_decode.runtime.mla -- m1c_inputs
// (the split partials are merged by their LSE) and post (LSE combine, then
// W_UV and the gate);
// page vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.mla.value --
// MlaValue / MlaGate (bf16 latent x W_UV with fp32 accumulation; value
// rounded to bf16 times the fp32 sigmoid of the raw gate, rounded to bf16;
// rows of empty requests selected to 0).  Same arithmetic as
// mla_merge_splits followed by mla_value_gate (the merged latent is rounded
// to bf16 before the projection), in one launch.
//
// Design: one CTA (16 warps) per (16 rows, head, COLS output columns).
// One warp bulk-copies the CTA's W_UV rows into padded smem while each warp
// LSE-merges one latent row straight into smem (lanes own 16 columns; the
// first eight splits' LSE and rows loaded in one round, further splits four
// at a time); then warp MMA
// (bf16, m16n8k16, one 8-column tile per warp) over the 512-wide latent and
// the gate epilogue.  COLS (32, 64 or 128) is the narrowest column block
// whose grid still fits one wave of one CTA per SM, so a small batch
// spreads over the SMs without a second wave (the host routes large
// batches to the separate merge and value kernels, which read each partial
// row once).
// Launched with programmatic dependent launch: only the W_UV copies start
// while the grid before it on the stream may still be running (W_UV is a
// weight: nothing in the step writes it); griddepcontrol.wait orders every
// other read (partials, gate, lengths) and every global write after that
// grid's completion, so a kernel just before this one may produce any of
// them.
#include <cuda_runtime.h>

#include "common.cuh"

namespace mla {
namespace {

constexpr int kRows = 16, kStride = MLA_D_LATENT + 8;  // bf16 elements per padded smem row
constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;

template <int COLS>
struct Smem {
    __nv_bfloat16 lat[kRows][kStride];
    __nv_bfloat16 w[COLS][kStride];
    uint64_t bar;
};

__device__ __forceinline__ void fma8(float (&acc)[8], float w, uint4 v) {
    acc[0] += w * bf16_lo(v.x); acc[1] += w * bf16_hi(v.x);
    acc[2] += w * bf16_lo(v.y); acc[3] += w * bf16_hi(v.y);
    acc[4] += w * bf16_lo(v.z); acc[5] += w * bf16_hi(v.z);
    acc[6] += w * bf16_lo(v.w); acc[7] += w * bf16_hi(v.w);
}

__device__ __forceinline__ float sigmoid_f32(float x) { return 1.f / (1.f + expf(-x)); }

// Merged latent row `row` of head h into smem (and optionally global).
// The first kFirst splits' LSE and partial rows are loaded in one round
// (rows of unused splits, lse = -inf, are read but never used: their
// contents are unspecified); any further splits follow four at a time.
constexpr int kFirst = 8;

__device__ void merge_row(const __nv_bfloat16 *__restrict__ o, const float *__restrict__ lse, int num_splits,
                          long long nrow, long long rowidx, __nv_bfloat16 *dst_smem, __nv_bfloat16 *latent,
                          float *lse_out, int lane) {
    float lk[kFirst];
    uint4 f0[kFirst], f1[kFirst];
#pragma unroll
    for (int j = 0; j < kFirst; ++j) {
        lk[j] = -INFINITY;
        if (j < num_splits) {
            lk[j] = __ldg(lse + (long long)j * nrow + rowidx);
            const uint4 *p = reinterpret_cast<const uint4 *>(o + ((long long)j * nrow + rowidx) * MLA_D_LATENT);
            f0[j] = __ldg(p + lane);
            f1[j] = __ldg(p + 32 + lane);
        }
    }
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < kFirst; ++j) mx = fmaxf(mx, lk[j]);
    for (int k = kFirst + lane; k < num_splits; k += 32) mx = fmaxf(mx, __ldg(lse + (long long)k * nrow + rowidx));
#pragma unroll
    for (int d = 16; d; d >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));
    float a0[8], a1[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) a0[e] = a1[e] = 0.f;
    // Each lane sums the weights of splits lane, lane + 32, ... and the warp
    // adds the lanes up (the same order as the separate merge kernel, so
    // both give the same LSE bits).
    float tot = 0.f;
    if (mx > -INFINITY) {
#pragma unroll
        for (int j = 0; j < kFirst; ++j)
            if (lk[j] > -INFINITY) {
                const float w = expf(lk[j] - mx);
                if (j == lane) tot += w;
                fma8(a0, w, f0[j]);
                fma8(a1, w, f1[j]);
            }
        for (int kb = 0; kb < num_splits; kb += 32) {
            const int k = kb + lane;
            float w = 0.f;
            bool valid = false;
            if (k >= kFirst && k < num_splits) {
                const float l = __ldg(lse + (long long)k * nrow + rowidx);
                valid = l > -INFINITY;
                w = valid ? expf(l - mx) : 0.f;
            }
            tot += w;
            unsigned m = __ballot_sync(0xffffffffu, valid);
            while (m) {
                int src[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    src[j] = m ? __ffs(m) - 1 : -1;
                    if (m) m &= m - 1;
                }
                uint4 v0[4], v1[4];
                float ws[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    ws[j] = __shfl_sync(0xffffffffu, w, src[j] < 0 ? 0 : src[j]);
                    if (src[j] >= 0) {
                        const uint4 *p = reinterpret_cast<const uint4 *>(o + ((long long)(kb + src[j]) * nrow + rowidx) * MLA_D_LATENT);
                        v0[j] = __ldg(p + lane);
                        v1[j] = __ldg(p + 32 + lane);
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (src[j] >= 0) {
                        fma8(a0, ws[j], v0[j]);
                        fma8(a1, ws[j], v1[j]);
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
    reinterpret_cast<uint4 *>(dst_smem)[lane] = r0;
    reinterpret_cast<uint4 *>(dst_smem)[32 + lane] = r1;
    if (latent) {
        uint4 *g = reinterpret_cast<uint4 *>(latent + rowidx * MLA_D_LATENT);
        g[lane] = r0;
        g[32 + lane] = r1;
    }
    if (lse_out && lane == 0) lse_out[rowidx] = tot > 0.f ? mx + logf(tot) : -INFINITY;
}

template <int COLS>
__global__ void __launch_bounds__(kThreads, 1) merge_value_kernel(
    const __nv_bfloat16 *__restrict__ o, const float *__restrict__ lse, int num_splits,
    const __nv_bfloat16 *__restrict__ w_uv, const __nv_bfloat16 *__restrict__ gate,
    const int32_t *__restrict__ lengths, int S, int qlen, int H, __nv_bfloat16 *__restrict__ out,
    __nv_bfloat16 *__restrict__ latent, float *__restrict__ lse_out) {
    constexpr int MW = COLS / 8;    // warps with an 8-column MMA tile
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Smem<COLS> &sm = *reinterpret_cast<Smem<COLS> *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, qd = lane & 3;
    const int t0 = blockIdx.x * kRows, h = blockIdx.y, v0 = blockIdx.z * COLS;
    const bool writer = blockIdx.z == 0;   // one column block writes the merged latent / LSE

    if (tid == 0) {
        mbar_init(&sm.bar, 1);
        mbar_fence_init();
    }
    __syncthreads();
    if (warp == 0) {
        if (lane == 0) mbar_arrive_expect_tx(&sm.bar, (uint32_t)COLS * MLA_D_LATENT * 2);
        __syncwarp();
        for (int i = lane; i < COLS; i += 32)
            bulk_g2s(sm.w[i], w_uv + ((long long)h * MLA_D_V + v0 + i) * MLA_D_LATENT, MLA_D_LATENT * 2, &sm.bar);
    }
    // Everything below may come from the previous grid on the stream.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // Gate words and row activity for the epilogue, in flight during the merge.
    uint32_t gw[2] = {0u, 0u};
    bool active[2] = {false, false};
    if (warp < MW) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int t = t0 + 8 * hh + g;
            active[hh] = t < S && __ldg(lengths + t / qlen) > 0;
            const long long rowoff = (long long)t * H * MLA_D_V + (long long)h * MLA_D_V + v0;
            if (active[hh]) gw[hh] = __ldg(reinterpret_cast<const uint32_t *>(gate + rowoff + 8 * warp + 2 * qd));
        }
    }
    // One latent row per warp into smem.
    {
        const long long nrow = (long long)S * H;
        const int t = t0 + warp;
        if (t < S) {
            merge_row(o, lse, num_splits, nrow, (long long)t * H + h, sm.lat[warp], writer ? latent : nullptr,
                      writer ? lse_out : nullptr, lane);
        } else {
            reinterpret_cast<uint4 *>(sm.lat[warp])[lane] = make_uint4(0, 0, 0, 0);
            reinterpret_cast<uint4 *>(sm.lat[warp])[32 + lane] = make_uint4(0, 0, 0, 0);
        }
    }
    __syncthreads();
    if (warp >= MW) return;
    if (!mbar_wait(&sm.bar, 0)) {
        // Flagged; before the CTA may exit (and its shared memory be reused)
        // give the W_UV copies one more bounded wait to land.
        mbar_wait(&sm.bar, 0);
        return;
    }

    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int ks = 0; ks < MLA_D_LATENT / 16; ++ks) {
        uint32_t a[4], b0, b1;
        ldmatrix_x4(a, &sm.lat[lane & 15][16 * ks + (lane >> 4) * 8]);
        ldmatrix_x2(b0, b1, &sm.w[8 * warp + (lane & 7)][16 * ks + ((lane >> 3) & 1) * 8]);
        mma_bf16(acc, a, b0, b1);
    }
    // Epilogue: bf16(value) * sigmoid(gate) -> bf16; empty requests -> 0.
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int t = t0 + 8 * hh + g;
        if (t >= S) continue;
        const long long rowoff = (long long)t * H * MLA_D_V + (long long)h * MLA_D_V + v0;
        uint32_t res = 0u;
        if (active[hh]) {
            const float v_lo = __bfloat162float(__float2bfloat16_rn(acc[2 * hh]));
            const float v_hi = __bfloat162float(__float2bfloat16_rn(acc[2 * hh + 1]));
            res = pack_bf16x2(v_lo * sigmoid_f32(bf16_lo(gw[hh])), v_hi * sigmoid_f32(bf16_hi(gw[hh])));
        }
        *reinterpret_cast<uint32_t *>(out + rowoff + 8 * warp + 2 * qd) = res;
    }
}

template <int COLS>
cudaError_t launch(const void *o, const float *lse, int num_splits, const void *w_uv, const void *gate,
                   const int32_t *lengths, int S, int qlen, int H, void *out, void *latent, float *lse_out,
                   cudaStream_t st) {
    const size_t smem = sizeof(Smem<COLS>);
    cudaError_t e = smem_attr_once<merge_value_kernel<COLS>>((int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((S + kRows - 1) / kRows, H, MLA_D_V / COLS);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, merge_value_kernel<COLS>, static_cast<const __nv_bfloat16 *>(o), lse, num_splits,
                              static_cast<const __nv_bfloat16 *>(w_uv), static_cast<const __nv_bfloat16 *>(gate),
                              lengths, S, qlen, H, static_cast<__nv_bfloat16 *>(out),
                              static_cast<__nv_bfloat16 *>(latent), lse_out);
}

}  // namespace

cudaError_t merge_value_launch(const void *o, const float *lse, int num_splits, const void *w_uv, const void *gate,
                               const int32_t *lengths, int R, int qlen, int H, void *out, void *latent,
                               float *lse_out, int sms, cudaStream_t st) {
    const int S = R * qlen;
    if (S == 0) return cudaSuccess;
    // One CTA per SM (16 warps, ~94 registers each): the most column blocks
    // whose grid still fits one wave.
    const long long tiles = (long long)((S + kRows - 1) / kRows) * H;
    if (tiles * (MLA_D_V / 32) <= sms)
        return launch<32>(o, lse, num_splits, w_uv, gate, lengths, S, qlen, H, out, latent, lse_out, st);
    if (tiles * (MLA_D_V / 64) <= sms)
        return launch<64>(o, lse, num_splits, w_uv, gate, lengths, S, qlen, H, out, latent, lse_out, st);
    return launch<128>(o, lse, num_splits, w_uv, gate, lengths, S, qlen, H, out, latent, lse_out, st);
}

cudaError_t merge_value_status(unsigned int *flags, bool clear) { return read_status(flags, clear); }

}  // namespace mla
