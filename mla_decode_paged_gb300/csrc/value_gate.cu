// Absorbed W_UV projection fused with the sigmoid gate -- tcgen05 kernel,
// optionally preceded in the same launch by the LSE merge of the splits.
//
// What it computes: vLLM API page
// vllm.models.kimi_k3.amd.specialized_decode.runtime.mla -- m1c_inputs /
// post (the split partials merged by their LSE, then W_UV and the gate) and
// page
// vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.mla.value --
// MlaValue (the [B, H, 512] bf16 latent times W_UV [H, 128, 512], latent
// axis contiguous, bf16 MMA with fp32 accumulation; rows are tokens, qlen
// per request) and MlaGate (the value rounded to bf16, times the fp32
// sigmoid of the raw gate, rounded to bf16; rows of empty requests are 0,
// chosen by a select so a NaN gate never leaks).
//
// Design: one CTA per (NR query rows, head), 512 threads.  The head's whole
// W_UV slice [128 x 512] arrives by TMA, K-major with 128B swizzle (eight
// 64-element column blocks); it is the A operand (M = 128 output columns) of
// 32 bf16 tcgen05 MMAs (K = 16) issued by one thread into an f32 TMEM
// accumulator D[v][row].  The B operand (N = NR rows) is either
//   * the latent rows, loaded by TMA in the same layout (NR = 64, or 96 for
//     batches that 64-row tiles would spread over more than two waves; the
//     value kernel, after the separate merge), or
//   * the merged rows themselves (NR = 16; the fused route for small
//     batches): each of the 16 warps LSE-merges one row with the merge
//     kernel's row function, writes it (and its LSE) to global memory and
//     into the swizzled B tile, so the latent and the LSE are the same bytes
//     as the merge kernel's.
// The epilogue reads D (four warps, thread = output column v = TMEM lane),
// rounds the value to bf16 into a shared [NR][128] tile, then all 16 warps
// write each row's 128 outputs with coalesced 4-byte stores (the gate words,
// loaded the same way, are in flight during the copies, the merge and the
// MMAs).  The W_UV slice is read before the wait on the previous kernel
// (programmatic dependent launch): no kernel of the step writes it; the
// latent or partials, the gate and the lengths after it.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "merge_row.cuh"
#include "tc.cuh"

namespace mla {
namespace {

constexpr int kThreads = 512;                              // warps 0-3 read TMEM; all write
constexpr int kWarps = kThreads / 32;
constexpr int kColBlocks = MLA_D_LATENT / 64;              // 128-byte column blocks of the K axis
constexpr int kABlock = MLA_D_V * 128;                     // one column block of W_UV[h]: 16 KB
constexpr int kAOff = 0, kBOff = kColBlocks * kABlock;     // 128 KB of W_UV, then the B operand

template <int NR>
struct Tile {
    static_assert(NR % 16 == 0 && NR <= 256, "M = 128 MMAs take N = 16 .. 256 in steps of 16");
    static constexpr int kBBlock = NR * 128;                         // one column block of the rows
    static constexpr int kSmem = kBOff + kColBlocks * kBBlock + 1024; // + alignment slack
    static constexpr uint32_t kTmemCols = NR <= 32 ? 32 : NR <= 64 ? 64 : NR <= 128 ? 128 : 256;   // 2^k >= 32
    static constexpr int kPairs = NR * (MLA_D_V / 2) / kThreads;     // gate / output words per thread
    // kind::f16 instruction descriptor: bf16 A and B (K-major), f32 D, M = 128, N = NR.
    static constexpr uint32_t kIdesc =
        (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(NR >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
};

struct Args {
    const __nv_bfloat16 *o;   // fused: partials [num_splits, S*H, 512]
    const float *lse;         // fused: [num_splits, S*H]
    int num_splits;
    const __nv_bfloat16 *gate;
    const int32_t *lengths;
    int S, qlen, H;
    __nv_bfloat16 *out;
    __nv_bfloat16 *latent;    // fused: written
    float *lse_out;           // fused: written when non-null
};

__device__ __forceinline__ void mma_bf16_tc(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                            bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"((uint32_t)accumulate));
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

// MERGE = false: ml maps the latent [S][H][512]; MERGE = true: ml is unused
// and the rows are merged from the partials (NR = 16, one row per warp).
template <int NR, bool MERGE>
__global__ void __launch_bounds__(kThreads, 1)
    value_gate_kernel(const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap ml, const Args a) {
    using T = Tile<NR>;
    static_assert(!MERGE || NR == kWarps, "the fused kernel merges one row per warp");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t full_w, full_l, done;
    __shared__ uint32_t tmem;
    __shared__ int active[NR];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = blockIdx.x * NR, h = blockIdx.y;
    const int nrows = min(NR, a.S - t0);

    if (tid == 0) {
        mbar_init(&full_w, 1);
        mbar_init(&full_l, 1);
        mbar_init(&done, 1);
        mbar_fence_init();
    }
    if (warp == 0) tc::tmem_alloc(&tmem, T::kTmemCols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (tid == 0) {
        // W_UV is not written by the kernel before this one: fetch it first.
        mbar_arrive_expect_tx(&full_w, kColBlocks * kABlock);
        for (int kb = 0; kb < kColBlocks; ++kb) tma_2d(sm + kAOff + kb * kABlock, &mw, 64 * kb, MLA_D_V * h, &full_w);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (!MERGE && tid == 0) {
        // Rows past S read as zeros (their outputs are not written).
        mbar_arrive_expect_tx(&full_l, kColBlocks * T::kBBlock);
        for (int kb = 0; kb < kColBlocks; ++kb)
            tma_3d(sm + kBOff + kb * T::kBBlock, &ml, 64 * kb, h, t0, &full_l);
    }
    if (tid < NR) active[tid] = tid < nrows && __ldg(a.lengths + (t0 + tid) / a.qlen) > 0;
    // This thread's gate words (bf16 pairs w = tid + 512 k: row w / 64, pair
    // w % 64), loaded while the copies, the merge and the MMAs are in flight.
    uint32_t gw[T::kPairs];
#pragma unroll
    for (int k = 0; k < T::kPairs; ++k) {
        const int w = tid + kThreads * k, r = w / (MLA_D_V / 2), p = w - r * (MLA_D_V / 2);
        gw[k] = r < nrows ? __ldg(reinterpret_cast<const uint32_t *>(
                                a.gate + ((long long)(t0 + r) * a.H + h) * MLA_D_V + 2 * p))
                          : 0u;
    }
    if constexpr (MERGE) {
        // Row r = warp.  Lane l holds latent columns 8l .. 8l+7 (column block
        // l / 8, 16-byte chunk l % 8) and 256 + 8l .. (block 4 + l / 8); in
        // the 128B-swizzled K-major tile chunk c of row r sits at c ^ (r % 8).
        const int r = warp;
        uint4 r0 = make_uint4(0, 0, 0, 0), r1 = r0;
        if (r < nrows) {
            const long long nrow = (long long)a.S * a.H, row = (long long)(t0 + r) * a.H + h;
            float lse_row;
            merge_row(a.o, a.lse, a.num_splits, nrow, row, lane, r0, r1, lse_row);
            uint4 *g = reinterpret_cast<uint4 *>(a.latent + row * MLA_D_LATENT);
            g[lane] = r0;
            g[32 + lane] = r1;
            if (a.lse_out && lane == 0) a.lse_out[row] = lse_row;
        }
        uint8_t *dst = sm + kBOff + (lane >> 3) * T::kBBlock + r * 128 + (((lane & 7) ^ (r & 7)) << 4);
        *reinterpret_cast<uint4 *>(dst) = r0;
        *reinterpret_cast<uint4 *>(dst + 4 * T::kBBlock) = r1;
        tc::fence_async_smem();   // the MMAs read these rows through the async proxy
        __syncthreads();
    }

    const uint32_t base = smem_u32(sm), tm = tmem;
    bool ok = true, issued = false;
    if (tid == 0) {
        ok = mbar_wait(&full_w, 0) && (MERGE || mbar_wait(&full_l, 0));
        if (ok) {
            issued = true;
            tc::fence_after();
#pragma unroll
            for (int j = 0; j < MLA_D_LATENT / 16; ++j) {
                const int kb = j >> 2, off = (j & 3) * 32;
                mma_bf16_tc(tm, tc::sdesc(base + kAOff + kb * kABlock + off, 16, 1024, tc::kSw128),
                            tc::sdesc(base + kBOff + kb * T::kBBlock + off, 16, 1024, tc::kSw128), T::kIdesc,
                            j > 0);
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
            if (!MERGE) mbar_wait(&full_l, 0);
            if (issued) mbar_wait(&done, 0);
        }
        tc::fence_before();
        __syncthreads();
        if (warp == 0) tc::tmem_free(tm, T::kTmemCols);
        return;
    }
    tc::fence_after();

    // D[v][row] -> bf16(value) in a [NR][128] tile (the W_UV slice is no
    // longer read: its first bytes hold the tile); warps 0-3 cover the 128
    // TMEM lanes.
    __nv_bfloat16 *tile = reinterpret_cast<__nv_bfloat16 *>(sm + kAOff);
    if (warp < 4) {
        const int v = 32 * warp + lane;
#pragma unroll
        for (int c = 0; c < NR; c += 16) {
            float d[16];
            tc::ld16(tm + ((uint32_t)(32 * warp) << 16) + c, d);
            tc::wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) tile[(c + i) * MLA_D_V + v] = __float2bfloat16_rn(d[i]);
        }
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_free(tm, T::kTmemCols);

    // Row by row, 64 bf16 pairs per row: out = bf16(value * sigmoid(gate)),
    // 0 for rows of empty requests (selected, so a NaN gate never leaks).
    const uint32_t *tile2 = reinterpret_cast<const uint32_t *>(tile);
#pragma unroll
    for (int k = 0; k < T::kPairs; ++k) {
        const int w = tid + kThreads * k, r = w / (MLA_D_V / 2), p = w - r * (MLA_D_V / 2);
        if (r >= nrows) break;
        uint32_t res = 0u;
        if (active[r]) {
            const uint32_t val = tile2[w], g = gw[k];
            res = pack_bf16x2(bf16_lo(val) * sigmoid_f32(bf16_lo(g)), bf16_hi(val) * sigmoid_f32(bf16_hi(g)));
        }
        *reinterpret_cast<uint32_t *>(a.out + ((long long)(t0 + r) * a.H + h) * MLA_D_V + 2 * p) = res;
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

// Tensor maps, encoded once per (device, buffer, shape) and reused while a
// thread keeps launching on the same buffers: W_UV as [H*128 rows, 512] and
// the latent as [S][H][512], 64-element (128-byte) boxes with 128B swizzle
// (the UMMA K-major layout), no L2 promotion.
struct MapCache {
    int dev = -1;
    const void *ptr = nullptr;
    int S = 0, H = 0;
    CUtensorMap map = {};
    bool hit(int d, const void *p, int s, int hh) const { return dev == d && ptr == p && S == s && H == hh; }
};

cudaError_t encode_map(MapCache &c, int dev, const void *ptr, int S, int H, int rank, const cuuint64_t *dim,
                       const cuuint64_t *stride, const cuuint32_t *box) {
    if (c.hit(dev, ptr, S, H)) return cudaSuccess;
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    c.dev = -1;
    const cuuint32_t es[3] = {1, 1, 1};
    if (enc(&c.map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(ptr), dim, stride, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    c.dev = dev;
    c.ptr = ptr;
    c.S = S;
    c.H = H;
    return cudaSuccess;
}

cudaError_t wuv_map(const void *w_uv, int H, const CUtensorMap **m) {
    static thread_local MapCache c;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    const cuuint64_t dim[2] = {(cuuint64_t)MLA_D_LATENT, (cuuint64_t)H * MLA_D_V};
    const cuuint64_t stride[1] = {(cuuint64_t)MLA_D_LATENT * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)MLA_D_V};
    cudaError_t e = encode_map(c, dev, w_uv, 0, H, 2, dim, stride, box);
    *m = &c.map;
    return e;
}

// One cache per tile height (the box has `rows` rows).
template <int ROWS>
cudaError_t latent_map(const void *latent, int S, int H, const CUtensorMap **m) {
    constexpr int rows = ROWS;
    static thread_local MapCache c;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    const cuuint64_t dim[3] = {(cuuint64_t)MLA_D_LATENT, (cuuint64_t)H, (cuuint64_t)S};
    const cuuint64_t stride[2] = {(cuuint64_t)MLA_D_LATENT * 2, (cuuint64_t)H * MLA_D_LATENT * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)rows};
    cudaError_t e = encode_map(c, dev, latent, S, H, 3, dim, stride, box);
    *m = &c.map;
    return e;
}

template <int NR, bool MERGE>
cudaError_t launch(const CUtensorMap &mw, const CUtensorMap &ml, const Args &a, cudaStream_t st) {
    cudaError_t e = smem_attr_once<value_gate_kernel<NR, MERGE>>(Tile<NR>::kSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((a.S + NR - 1) / NR, a.H, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Tile<NR>::kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, value_gate_kernel<NR, MERGE>, mw, ml, a);
}

template <int ROWS>
cudaError_t value_gate_rows(const void *latent, const void *w_uv, const void *gate, const int32_t *lengths, int S,
                            int qlen, int H, void *out, cudaStream_t st) {
    const CUtensorMap *mw = nullptr, *ml = nullptr;
    cudaError_t e = wuv_map(w_uv, H, &mw);
    if (e == cudaSuccess) e = latent_map<ROWS>(latent, S, H, &ml);
    if (e != cudaSuccess) return e;
    Args a = {};
    a.gate = static_cast<const __nv_bfloat16 *>(gate);
    a.lengths = lengths;
    a.S = S;
    a.qlen = qlen;
    a.H = H;
    a.out = static_cast<__nv_bfloat16 *>(out);
    return launch<ROWS, false>(*mw, *ml, a, st);
}

}  // namespace

// latent [S, H, 512] and w_uv [H, 128, 512] bf16 (16-byte aligned); gate
// [S, H*128] bf16 and out (4-byte aligned).  64 rows per CTA, or 96 when
// 64-row tiles would take more than two waves of CTAs (one per SM: each
// loads its head's 128 KB W_UV slice, so fewer, taller tiles finish sooner
// there -- 2,048 x 12 rows: merge + value/gate 31.4 -> 27.8 us).
cudaError_t value_gate_launch(const void *latent, const void *w_uv, const void *gate,
                              const int32_t *lengths, int R, int qlen, int H, void *out, int sms, cudaStream_t st) {
    const int S = R * qlen;
    if (S == 0) return cudaSuccess;
    if ((int64_t)((S + 63) / 64) * H > 2 * (int64_t)sms)
        return value_gate_rows<96>(latent, w_uv, gate, lengths, S, qlen, H, out, st);
    return value_gate_rows<64>(latent, w_uv, gate, lengths, S, qlen, H, out, st);
}

// The fused route: partials o [num_splits, S*H, 512] bf16 and latent
// (16-byte aligned), lse [num_splits, S*H] f32; 16 rows per CTA, each row
// merged once.
cudaError_t merge_value_launch(const void *o, const float *lse, int num_splits, const void *w_uv, const void *gate,
                               const int32_t *lengths, int R, int qlen, int H, void *out, void *latent,
                               float *lse_out, cudaStream_t st) {
    const int S = R * qlen;
    if (S == 0) return cudaSuccess;
    const CUtensorMap *mw = nullptr;
    cudaError_t e = wuv_map(w_uv, H, &mw);
    if (e != cudaSuccess) return e;
    Args a = {};
    a.o = static_cast<const __nv_bfloat16 *>(o);
    a.lse = lse;
    a.num_splits = num_splits;
    a.gate = static_cast<const __nv_bfloat16 *>(gate);
    a.lengths = lengths;
    a.S = S;
    a.qlen = qlen;
    a.H = H;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.latent = static_cast<__nv_bfloat16 *>(latent);
    a.lse_out = lse_out;
    return launch<kWarps, true>(*mw, *mw, a, st);
}

cudaError_t value_gate_status(unsigned int *flags, bool clear) { return read_status(flags, clear); }

}  // namespace mla
