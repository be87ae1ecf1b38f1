// Device helpers shared by the MLA decode kernels: mbarriers with bounded
// waits, bulk async copies, fp8/f16/bf16 conversions, warp MMA, and the
// per-device status word.  Inline PTX for sm_103a.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../include/mla_decode.h"

namespace mla {

// Per-device status word (MLA_DEV_* bits), one per translation unit (no
// relocatable device code needed).  Kernels only OR bits into it;
// read_status() below (called by mla_device_status) reads and clears it.
static __device__ unsigned int g_status;

__device__ __forceinline__ void flag(unsigned int bits) { atomicOr(&g_status, bits); }

// Sets a kernel's dynamic shared-memory limit once per device ordinal
// (< 64): the runtime call otherwise costs host time on every launch.
template <auto *KERNEL>
inline cudaError_t smem_attr_once(int bytes) {
    static std::atomic<unsigned long long> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(KERNEL, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
}

static inline cudaError_t read_status(unsigned int *flags, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_status, sizeof(unsigned int));
    if (e == cudaSuccess && clear) {
        unsigned int z = 0;
        e = cudaMemcpyToSymbol(g_status, &z, sizeof(unsigned int));
    }
    return e;
}

// Upper bound on any single wait, in SM clock cycles (~2 s at 2 GHz).  A
// correct launch never comes near it; when it runs out the waiter records
// MLA_DEV_TIMEOUT and gives up instead of hanging the GPU.
constexpr long long kWaitCycles = 4000000000LL;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking probe: true if the phase of `parity` has completed.
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase of `parity` to complete.  Returns false (after
// flagging MLA_DEV_TIMEOUT) if it has not completed within kWaitCycles.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kWaitCycles) {
            flag(MLA_DEV_TIMEOUT);
            return false;
        }
    }
    return true;
}

// ------------------------------------------------------------ bulk copies

// Global -> shared bulk copy of `bytes` (multiple of 16, both addresses
// 16-byte aligned) completing on `bar` with complete_tx.
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ------------------------------------------------------------ conversions

// Two OCP E4M3 codes (low byte -> low half) to f16x2; exact (every E4M3
// value is an f16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(two));
    return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ float2 unpack_f16x2(uint32_t v) {
    __half2 h = *reinterpret_cast<__half2 *>(&v);
    return __half22float2(h);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// ------------------------------------------------------------------ warp MMA

// D += A * B, m16n8k16, f16 inputs, f32 accumulate.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D += A * B, m16n8k16, bf16 inputs, f32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void *smem_row) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(smem_row)));
}

__device__ __forceinline__ void ldmatrix_x2(uint32_t &r0, uint32_t &r1, const void *smem_row) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
                 : "=r"(r0), "=r"(r1)
                 : "r"(smem_u32(smem_row)));
}

// Named barrier over `count` threads (multiple of 32).
__device__ __forceinline__ void named_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---------------------------------------------------- cp.async (16 bytes)

__device__ __forceinline__ void cp_async16(void *dst_smem, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst_smem)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------- split plan

// Splits of a request of `len` tokens (the rule stated in mla_decode.h).
__device__ __forceinline__ int split_count(int len, int num_splits, int split_tokens) {
    int n = (len + split_tokens - 1) / split_tokens;
    n = n < 1 ? 1 : n;
    return n > num_splits ? num_splits : n;
}

// Token range [*start, *start + *count) of split k of n over `len` tokens.
__device__ __forceinline__ void split_range(int len, int n, int k, int *start, int *count) {
    int b = len / n, m = len % n;
    *start = k * b + (k < m ? k : m);
    *count = b + (k < m ? 1 : 0);
}

// Length (tokens) of request r from indptr, validated against num_pages:
// a decreasing or out-of-range entry flags MLA_DEV_BAD_INDPTR and yields an
// empty request (the kernels then never index pages with it).  With blocks
// of 2^log2p rows, indptr counts blocks and the last block holds
// last_page_len[r] (1..2^log2p) rows; a value outside that range is flagged
// the same way.
__device__ __forceinline__ int request_len(const int32_t *indptr, int r, int64_t num_pages, int *base,
                                           int log2p = 0, const int32_t *last_page_len = nullptr) {
    int a = __ldg(indptr + r), b = __ldg(indptr + r + 1);
    if (a < 0 || b < a || (int64_t)b > num_pages) {
        flag(MLA_DEV_BAD_INDPTR);
        *base = 0;
        return 0;
    }
    *base = a;
    if (log2p == 0 || b == a) return b - a;
    const int last = __ldg(last_page_len + r);
    if (last < 1 || last > (1 << log2p)) {
        flag(MLA_DEV_BAD_INDPTR);
        return 0;
    }
    return ((b - a - 1) << log2p) + last;
}

// Address of the KV row that token slot i (an index into pages) names.  A
// page outside [0, pool_rows) flags MLA_DEV_BAD_PAGE and reads row 0
// instead, so the copy never leaves the pool.  Both the attend kernels and
// mla_debug_gather address rows through this function.
__device__ __forceinline__ const uint8_t *kv_row_of_page(const uint8_t *kv, int64_t p, int64_t pool_rows) {
    if (p < 0 || p >= pool_rows) {
        flag(MLA_DEV_BAD_PAGE);
        p = 0;
    }
    return kv + p * (int64_t)MLA_D_QK;
}

__device__ __forceinline__ const uint8_t *kv_row(const uint8_t *kv, const int32_t *pages,
                                                 int64_t i, int64_t pool_rows) {
    return kv_row_of_page(kv, __ldg(pages + i), pool_rows);
}

// Walks the work units (request r, split k), enumerated request-major:
// unit u belongs to the first request whose running split count exceeds u.
// Warp-cooperative: lane l holds request r_base + l of a 32-request window
// and an inclusive prefix sum of the split counts.  Queries must come in
// non-decreasing u order.  Every lane of the warp must call find() together.
// PAGED: indptr counts blocks of 2^log2p rows (see request_len).
template <bool PAGED = false>
struct UnitCursor {
    const int32_t *indptr;
    const int32_t *last_page_len;   // block tables only
    int64_t num_pages;
    int R, num_splits, split_tokens, log2p;
    int r_base;
    long long cum_base;
    int n, incl, len, base;

    // `window`: load the first 32 requests' split counts (not needed when a
    // work plan names the units).
    __device__ void init(const int32_t *ip, int r_count, int64_t pages_len, int ns, int st, int lane,
                         int lp = 0, const int32_t *last = nullptr, bool window = true) {
        indptr = ip;
        last_page_len = PAGED ? last : nullptr;
        log2p = PAGED ? lp : 0;
        R = r_count;
        num_pages = pages_len;
        num_splits = ns;
        split_tokens = st;
        r_base = 0;
        cum_base = 0;
        if (window) load(lane);
    }

    __device__ void load(int lane) {
        const int r = r_base + lane;
        if (r < R) {
            len = PAGED ? request_len(indptr, r, num_pages, &base, log2p, last_page_len)
                        : request_len(indptr, r, num_pages, &base);
            n = split_count(len, num_splits, split_tokens);
        } else {
            len = 0;
            base = 0;
            n = 0;
        }
        incl = n;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += v;
        }
    }

    // Unit u -> (r, k, n_r, len, base); false when u is past the last unit.
    __device__ bool find(long long u, int lane, int *r, int *k, int *n_r, int *len_r, int *base_r) {
        while (true) {
            if (r_base >= R) return false;
            const int total = __shfl_sync(0xffffffffu, incl, 31);
            if (u < cum_base + total) {
                const unsigned m = __ballot_sync(0xffffffffu, cum_base + incl > u);
                const int src = __ffs(m) - 1;
                const int nn = __shfl_sync(0xffffffffu, n, src);
                const int in = __shfl_sync(0xffffffffu, incl, src);
                *r = r_base + src;
                *n_r = nn;
                *k = (int)(u - (cum_base + in - nn));
                *len_r = __shfl_sync(0xffffffffu, len, src);
                *base_r = __shfl_sync(0xffffffffu, base, src);
                return true;
            }
            cum_base += total;
            r_base += 32;
            load(lane);
        }
    }
};

constexpr int kTileFirst = 1, kTileLast = 2;

// One tile of one work unit, as the producer hands it to the consumers.
struct Tile {
    int r, k, n_r, base, tok0, ntok, flags;
    bool valid;
};

// Iterates this CTA's tiles in order, each unit (request, split, row group;
// numbered request-major, u = unit * groups + group) cut into TILE-token
// tiles.  Units u = blockIdx.x, +gridDim.x, ... by default.  With a work
// plan (int32: [G, offsets[G + 1], items]) the CTA takes the items
// offsets[b] .. offsets[b + 1] - 1, each four int32
//   {r, k | n_r << 9 | group << 18, start, count}:
// split k of n_r of request r covers its tokens [start, start + count).  An
// item that does not fit the launch flags MLA_DEV_BAD_PLAN and ends the
// CTA's list.
constexpr int kPlanItemWords = MLA_PLAN_ITEM_WORDS;

template <int TILE, bool PAGED = false>
struct TileIter {
    UnitCursor<PAGED> cur;
    long long u;
    int t, ntiles, start, count, r, k, n_r, base, grp;
    bool have_unit;
    int plan_pos, plan_end;      // plan_end: -1 round robin, -2 a plan not opened yet
    int plan_items;              // items in the plan (from its length)

    int row_groups;
    __device__ void init(const int32_t *indptr, int R, int64_t num_pages, int num_splits, int split_tokens,
                         int groups, int lane, int log2p = 0, const int32_t *last_page_len = nullptr,
                         const int32_t *plan = nullptr, int64_t plan_len = 0) {
        cur.init(indptr, R, num_pages, num_splits, split_tokens, lane, log2p, last_page_len, plan == nullptr);
        row_groups = groups;
        u = (long long)blockIdx.x - gridDim.x;
        have_unit = false;
        plan_pos = 0;
        plan_end = -1;
        if (plan) {
            plan_end = -2;
            const int64_t items = (plan_len - 2 - (int64_t)gridDim.x) / kPlanItemWords - (int64_t)gridDim.x;
            plan_items = items < 0 ? -1 : (int)min(items, (int64_t)INT32_MAX);
        }
    }

    // The next plan item into (r, k, n_r, grp, start, count, base); false at
    // the end of the list or on an item that does not fit (flagged).
    // Opening the plan: the grid check, this CTA's offsets and the copy of
    // its first item (after the items) are independent loads, one round
    // trip; item[] gets the first item's words.  A plan for another grid, or
    // offsets outside the buffer: flagged, no work.  False when the list is
    // empty or flagged.
    __device__ bool open_plan(const int32_t *plan, int (&item)[4]) {
        plan_end = 0;
        if (plan_items < 0) {
            flag(MLA_DEV_BAD_PLAN);
            return false;
        }
        const int32_t *fi = plan + 2 + gridDim.x + (int64_t)kPlanItemWords * ((int64_t)plan_items + blockIdx.x);
        const int g0 = __ldg(plan), a = __ldg(plan + 1 + blockIdx.x), b = __ldg(plan + 2 + blockIdx.x);
#pragma unroll
        for (int i = 0; i < 4; ++i) item[i] = __ldg(fi + i);
        if (g0 != (int)gridDim.x || a < 0 || b < a || b > plan_items) {
            flag(MLA_DEV_BAD_PLAN);
            return false;
        }
        plan_pos = a;
        plan_end = b;
        return a < b;
    }

    // The next plan item into (r, k, n_r, grp, start, count, base); false at
    // the end of the list or on an item that does not fit (flagged).  `first`:
    // the words open_plan returned, for the list's first item.
    __device__ bool plan_next(const int32_t *plan, const int *first = nullptr) {
        int ir, w, s0, c;
        if (plan_end == -2) {
            int item[4];
            if (!open_plan(plan, item)) return false;
            ++plan_pos;
            ir = item[0]; w = item[1]; s0 = item[2]; c = item[3];
        } else {
            if (plan_pos >= plan_end) return false;
            if (first) {
                ++plan_pos;
                ir = first[0]; w = first[1]; s0 = first[2]; c = first[3];
            } else {
                const int32_t *it = plan + 2 + gridDim.x + (int64_t)kPlanItemWords * plan_pos++;
                ir = __ldg(it); w = __ldg(it + 1); s0 = __ldg(it + 2); c = __ldg(it + 3);
            }
        }
        const int ik = w & 511, inr = (w >> 9) & 511, ig = (w >> 18) & 8191;
        bool ok = w >= 0 && ir >= 0 && ir < cur.R && inr >= 1 && inr <= cur.num_splits && ik < inr &&
                  ig < row_groups && s0 >= 0 && c >= 0;
        if (ok) {
            const int len = PAGED ? request_len(cur.indptr, ir, cur.num_pages, &base, cur.log2p, cur.last_page_len)
                                  : request_len(cur.indptr, ir, cur.num_pages, &base);
            // a range inside the request; a zero-token item only as the one
            // split of an empty request (elsewhere it would write LSE -inf
            // over partials other CTAs produce)
            ok = (int64_t)s0 + c <= len && (c > 0 || (len == 0 && ik == 0 && inr == 1));
        }
        if (!ok) {
            flag(MLA_DEV_BAD_PLAN);
            plan_pos = plan_end;
            return false;
        }
        r = ir; k = ik; n_r = inr; grp = ig; start = s0; count = c;
        return true;
    }

    // `plan`: the work plan the iterator was initialised with (or null);
    // `first`: open_plan's words of the first item, on the first call.
    __device__ Tile next(int lane, const int32_t *plan = nullptr, const int *first = nullptr) {
        Tile T;
        T.valid = false;
        if (!have_unit || t >= ntiles) {
            if (plan_end != -1) {
                if (!plan_next(plan, first)) {
                    have_unit = false;
                    return T;
                }
            } else {
                u += gridDim.x;
                int len;
                if (!cur.find(u / row_groups, lane, &r, &k, &n_r, &len, &base)) {
                    have_unit = false;
                    return T;
                }
                grp = (int)(u % row_groups);
                split_range(len, n_r, k, &start, &count);
            }
            ntiles = count > 0 ? (count + TILE - 1) / TILE : 1;
            t = 0;
            have_unit = true;
        }
        T.valid = true;
        T.r = r; T.k = k; T.n_r = n_r; T.base = base;
        T.tok0 = start + t * TILE;
        T.ntok = count > 0 ? min(TILE, count - t * TILE) : 0;
        T.flags = (t == 0 ? kTileFirst : 0) | (t == ntiles - 1 ? kTileLast : 0) | (grp << 8);
        ++t;
        return T;
    }
};

}  // namespace mla
