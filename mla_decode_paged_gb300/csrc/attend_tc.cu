// Split-KV MLA decode attention over a paged fp8 latent cache -- tcgen05
// tensor-memory kernel (sm_103a).
//
// What it computes: vLLM API page
// vllm.models.kimi_k3.amd.specialized_decode.runtime.mla, m1c_inputs (bf16
// query [S, H, 576], flat fp8 token rows addressed by pages / indptr,
// scale and kv_scale, partials o [splits, S, H, 512] bf16 and LSE
// [splits, S, H] f32) and attend (multi-query attention over one latent row
// per token; padded heads skipped through the row stride).  Same work units
// and split plan as the warp-MMA kernel.
//
// Design (one persistent CTA per SM, 12 warps):
//   * warps 5..11 (producers): TMA tile::gather4 copies 4 paged KV rows per
//     instruction straight into the UMMA canonical layout: the 512 latent
//     bytes as four 128-byte column blocks with 128B swizzle, the 64 rope
//     bytes with 64B swizzle.  Rows past the tile's tokens (and bad page
//     indices) use an out-of-range row, which the TMA fills with zeros.
//   * The fp8 tile is used as stored (no dequant pass): tokens are the MMA M
//     dimension (128).  QK^T: S^T[tok, n] = K[tok, :576] . Q'[n, :576]; the
//     query is split into two e4m3 terms per row, q*2^e = hi + lo/16, stacked
//     as the B operand's 2*NQ rows, so one MMA chain yields both partial
//     scores.  P.V: O^T[lat, n] = V^T[lat, tok] . P'^T[tok, n], with the same
//     smem bytes read MN-major as V^T and P likewise split into hi + lo/16.
//     kind::f8f6f4 E4M3 x E4M3 with f32 accumulation in TMEM:
//     S' at columns [0, 2NQ), O' for latent block b at [2NQ(1+b), 2NQ(2+b)).
//   * warp 4 (MMA): one thread issues 18 QK MMAs (K = 32 each) and, once P
//     is in smem, 16 PV MMAs per tile; tcgen05.commit releases the stage.
//   * warps 0..3 (softmax, thread = TMEM lane = token): combine the hi/lo
//     scores, online softmax in the log2 domain with a lazily updated
//     reference max (rebased, and O rescaled in TMEM, only when a score
//     exceeds it by more than 2^8), write P' (hi/lo e4m3) to smem, prepare
//     the next unit's query, and at a unit's end reduce the row sums and
//     write o / lse.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "tc.cuh"

namespace mla {
namespace {

constexpr int kT = 128;              // tokens per tile = MMA M
constexpr int kStages = 2;
constexpr int kStageBytes = 73728;   // 4 x (16 x 1024) latent + 16 x 512 rope
constexpr int kRopeOff = 65536;
constexpr int kSoftWarps = 4, kMmaWarp = 4, kProdWarp0 = 5, kProdWarps = 7;
constexpr int kThreads = (kSoftWarps + 1 + kProdWarps) * 32;
constexpr int kOps = 160;            // gather4 ops per tile: 32 groups of 4 rows x (4 latent + 1 rope)
constexpr int kSoftBar = 1;          // named barrier of the softmax warpgroup
constexpr float kRebase = 8.f;       // log2 headroom before the reference max moves

template <int NQ>
struct Cfg {
    static constexpr int NP = 2 * NQ;                      // MMA N (hi and lo terms)
    static constexpr int OffQ = kStages * kStageBytes;
    static constexpr int QLatBlock = (NP / 8) * 1024;      // one 128-byte column block of Q'
    static constexpr int QRope = 4 * QLatBlock;
    static constexpr int OffP = OffQ + NP * 576;
    static constexpr int OffMisc = OffP + 16384;
    static constexpr uint32_t TmemCols = (10 * NQ <= 256) ? 256 : 512;
};

template <int NQ>
struct Misc {
    uint64_t kv_full[kStages], kv_empty[kStages];
    uint64_t s_full, p_full, q_ready, o_done, fin;
    uint32_t tmem;
    int abort_flag;
    float c[NQ];            // per query row: scale*kv_scale*log2(e) / 2^e (0 for padding rows)
    float m[NQ];            // reference max of the row, log2 domain
    float alpha[NQ];
    float invl[NQ];
    float red[kSoftWarps][NQ];
};

struct Params {
    const __nv_bfloat16 *q;
    int64_t q_row_stride;
    int64_t pool_rows;
    const int32_t *pages;
    int64_t num_pages;
    const int32_t *indptr;
    int R, qlen, heads, num_splits, split_tokens, row_groups, nq;
    float sc_log2;
    float kv_scale;
    __nv_bfloat16 *o;
    float *lse;
};

template <int NQ>
__device__ __forceinline__ Misc<NQ> &misc(uint8_t *sm) {
    return *reinterpret_cast<Misc<NQ> *>(sm + Cfg<NQ>::OffMisc);
}

__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t par, int *abort_flag) {
    if (*(volatile int *)abort_flag) return false;
    if (!mbar_wait(bar, par)) {
        *(volatile int *)abort_flag = 1;
        return false;
    }
    return true;
}

// ------------------------------------------------------------------ producers

template <int NQ>
__device__ void producer(const Params &P, const CUtensorMap *mlat, const CUtensorMap *mrope, uint8_t *sm) {
    Misc<NQ> &ms = misc<NQ>(sm);
    const int lane = threadIdx.x & 31, pw = (threadIdx.x >> 5) - kProdWarp0;
    const int op = pw + kProdWarps * lane;  // ops dealt round-robin over the producer warps
    const bool has_op = op < kOps;
    const int g4 = op / 5, part = op % 5;
    TileIter<kT> iter;
    iter.init(P.indptr, P.R, P.num_pages, P.num_splits, P.split_tokens, P.row_groups, lane);
    auto fetch = [&](const Tile &T, int (&rows)[4]) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int tok = 4 * g4 + i;
            int r = -1;
            if (T.valid && has_op && tok < T.ntok) {
                const int64_t p = __ldg(P.pages + (int64_t)T.base + T.tok0 + tok);
                if (p < 0 || p >= P.pool_rows) flag(MLA_DEV_BAD_PAGE);
                else r = (int)p;
            }
            rows[i] = r;
        }
    };
    Tile cur = iter.next(lane);
    int rows[4];
    fetch(cur, rows);
    for (int it = 0; cur.valid; ++it) {
        Tile nxt = iter.next(lane);
        int nrows[4];
        fetch(nxt, nrows);
        const int s = it % kStages;
        if (!wait_or_abort(&ms.kv_empty[s], ((it / kStages) & 1) ^ 1, &ms.abort_flag)) return;
        const bool issue = has_op && cur.ntok > 0;
        uint32_t bytes = issue ? (part < 4 ? 512u : 256u) : 0u;
#pragma unroll
        for (int d = 16; d; d >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, d);
        if (lane == 0) mbar_arrive_expect_tx(&ms.kv_full[s], bytes);
        __syncwarp();
        if (issue) {
            uint8_t *st = sm + s * kStageBytes;
            const int g8 = g4 >> 1, half = g4 & 1;
            if (part < 4)
                tc::gather4(st + part * 16384 + g8 * 1024 + half * 512, mlat, part * 128, rows[0], rows[1], rows[2],
                            rows[3], &ms.kv_full[s]);
            else
                tc::gather4(st + kRopeOff + g8 * 512 + half * 256, mrope, 512, rows[0], rows[1], rows[2], rows[3],
                            &ms.kv_full[s]);
        }
        cur = nxt;
#pragma unroll
        for (int i = 0; i < 4; ++i) rows[i] = nrows[i];
    }
}

// ------------------------------------------------------------------ MMA issuer

template <int NQ>
__device__ void mma_issuer(const Params &P, uint8_t *sm) {
    using C = Cfg<NQ>;
    Misc<NQ> &ms = misc<NQ>(sm);
    const int lane = threadIdx.x & 31;
    const uint32_t base = smem_u32(sm);
    const uint32_t tm = ms.tmem;
    constexpr uint32_t kIdQK = tc::idesc_e4m3(C::NP, false, false);
    constexpr uint32_t kIdPV = tc::idesc_e4m3(C::NP, true, true);
    TileIter<kT> iter;
    iter.init(P.indptr, P.R, P.num_pages, P.num_splits, P.split_tokens, P.row_groups, lane);
    int n_tiles = 0, n_units = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
        const Tile T = iter.next(lane);
        if (!T.valid) break;
        const int s = it % kStages;
        if (!(ok = wait_or_abort(&ms.kv_full[s], (it / kStages) & 1, &ms.abort_flag))) break;
        if (T.ntok == 0) {  // empty request: nothing to multiply
            if (lane == 0) mbar_arrive(&ms.kv_empty[s]);
            continue;
        }
        const bool first = T.flags & kTileFirst;
        if (first && !(ok = wait_or_abort(&ms.q_ready, n_units & 1, &ms.abort_flag))) break;
        tc::fence_after();
        const uint32_t st = base + s * kStageBytes;
        if (lane == 0) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int a = j >> 2, off = (j & 3) * 32;
                tc::mma_e4m3(tm, tc::sdesc(st + a * 16384 + off, 16, 1024, tc::kSw128),
                             tc::sdesc(base + C::OffQ + a * C::QLatBlock + off, 16, 1024, tc::kSw128), kIdQK, j > 0);
            }
#pragma unroll
            for (int j = 0; j < 2; ++j)
                tc::mma_e4m3(tm, tc::sdesc(st + kRopeOff + j * 32, 16, 512, tc::kSw64),
                             tc::sdesc(base + C::OffQ + C::QRope + j * 32, 16, 512, tc::kSw64), kIdQK, true);
            tc::commit(&ms.s_full);
        }
        __syncwarp();
        if (!(ok = wait_or_abort(&ms.p_full, n_tiles & 1, &ms.abort_flag))) break;
        tc::fence_after();
        if (lane == 0) {
#pragma unroll
            for (int b = 0; b < 4; ++b)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc::mma_e4m3(tm + C::NP * (1 + b), tc::sdesc(st + b * 16384 + kk * 4096, 16384, 1024, tc::kSw128),
                                 tc::sdesc(base + C::OffP + kk * 4096, 16384, 1024, tc::kSw128), kIdPV,
                                 !(first && kk == 0));
            tc::commit(&ms.kv_empty[s]);
            if (T.flags & kTileLast) tc::commit(&ms.o_done);
        }
        __syncwarp();
        ++n_tiles;
        if (first) ++n_units;
    }
    // Every MMA issued so far must be complete before TMEM is released.
    if (lane == 0) tc::commit(&ms.fin);
    __syncwarp();
    mbar_wait(&ms.fin, 0);
}

// ------------------------------------------------------------------ softmax

// The query rows of tile T's request and row group as the B operand Q':
// row n = q_n * 2^e_n rounded to e4m3 (hi), row NQ + n = 16 * (q_n * 2^e_n
// - hi) rounded to e4m3 (lo), in the K-major 128B / 64B swizzled layouts;
// c[n] = scale * kv_scale * log2(e) / 2^e_n.
template <int NQ>
__device__ void prep_query(const Params &P, uint8_t *sm, const Tile &T) {
    using C = Cfg<NQ>;
    Misc<NQ> &ms = misc<NQ>(sm);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rows_total = P.qlen * P.heads, grp = T.flags >> 8;
    constexpr int kPerWarp = NQ / kSoftWarps;
#pragma unroll 1
    for (int i0 = 0; i0 < kPerWarp; i0 += 4) {
        uint4 v[4][3];
        bool valid[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int n = warp + kSoftWarps * (i0 + i);
            const int rho = grp * NQ + n;
            valid[i] = (i0 + i < kPerWarp) && rho < rows_total;
            const __nv_bfloat16 *src = P.q;
            if (valid[i]) {
                const int tq = rho / P.heads, h = rho % P.heads;
                src = P.q + ((int64_t)T.r * P.qlen + tq) * P.q_row_stride + (int64_t)h * MLA_D_QK;
            }
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                const int ch = lane + 32 * j;
                v[i][j] = (valid[i] && ch < 72) ? __ldg(reinterpret_cast<const uint4 *>(src) + ch) : make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (i0 + i >= kPerWarp) break;
            const int n = warp + kSoftWarps * (i0 + i);
            float amax = 0.f;
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                const uint32_t w[4] = {v[i][j].x, v[i][j].y, v[i][j].z, v[i][j].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[e])), fabsf(bf16_hi(w[e]))));
            }
#pragma unroll
            for (int d = 16; d; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
            int ex = 0;
            if (amax > 0.f) frexpf(amax, &ex);      // amax < 2^ex
            ex = max(-92, min(ex, 120));            // keep 2^e and 2^-e finite
            const int e = 8 - ex;                   // scaled magnitudes < 256
            const float sc = ldexpf(1.f, e);
            if (lane == 0) ms.c[n] = valid[i] ? P.sc_log2 * ldexpf(1.f, -e) : 0.f;
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                const int ch = lane + 32 * j;
                if (ch >= 72) continue;
                const uint32_t w[4] = {v[i][j].x, v[i][j].y, v[i][j].z, v[i][j].w};
                uint32_t hi[2], lo[2];
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    const float2 x = make_float2(bf16_lo(w[e2]) * sc, bf16_hi(w[e2]) * sc);
                    const __nv_fp8x2_storage_t h8 = __nv_cvt_float2_to_fp8x2(x, __NV_SATFINITE, __NV_E4M3);
                    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(h8, __NV_E4M3);
                    const float2 hf = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
                    const float2 r = make_float2((x.x - hf.x) * 16.f, (x.y - hf.y) * 16.f);
                    const __nv_fp8x2_storage_t l8 = __nv_cvt_float2_to_fp8x2(r, __NV_SATFINITE, __NV_E4M3);
                    const int sh = (e2 & 1) * 16;
                    if (sh == 0) {
                        hi[e2 >> 1] = h8;
                        lo[e2 >> 1] = l8;
                    } else {
                        hi[e2 >> 1] |= (uint32_t)h8 << 16;
                        lo[e2 >> 1] |= (uint32_t)l8 << 16;
                    }
                }
                const int d = ch * 8;
                uint32_t off_hi, off_lo;
                if (d < 512) {
                    const uint32_t blk = C::OffQ + (d >> 7) * C::QLatBlock;
                    off_hi = blk + (n >> 3) * 1024 + tc::sw128(n, d & 127);
                    off_lo = blk + ((NQ + n) >> 3) * 1024 + tc::sw128(NQ + n, d & 127);
                } else {
                    const uint32_t blk = C::OffQ + C::QRope;
                    off_hi = blk + (n >> 3) * 512 + tc::sw64(n, d - 512);
                    off_lo = blk + ((NQ + n) >> 3) * 512 + tc::sw64(NQ + n, d - 512);
                }
                *reinterpret_cast<uint2 *>(sm + off_hi) = make_uint2(hi[0], hi[1]);
                *reinterpret_cast<uint2 *>(sm + off_lo) = make_uint2(lo[0], lo[1]);
            }
        }
    }
    tc::fence_async_smem();   // generic-proxy writes -> tensor-core reads
    named_sync(kSoftBar, kSoftWarps * 32);
}

template <int NQ>
__device__ void softmax(const Params &P, uint8_t *sm) {
    using C = Cfg<NQ>;
    Misc<NQ> &ms = misc<NQ>(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t tm = ms.tmem + ((uint32_t)(warp * 32) << 16);
    const int S = P.R * P.qlen, rows_total = P.qlen * P.heads;
    TileIter<kT> iter;
    iter.init(P.indptr, P.R, P.num_pages, P.num_splits, P.split_tokens, P.row_groups, lane);
    Tile cur = iter.next(lane);
    Tile nxt = iter.next(lane);
    if (cur.valid && cur.ntok > 0) {
        prep_query<NQ>(P, sm, cur);
        if (lane == 0) mbar_arrive(&ms.q_ready);
    }
    float l[NQ];
    int n_tiles = 0, n_units = 0;
    while (cur.valid) {
        const int grp = cur.flags >> 8;
        if (cur.ntok == 0) {
            // Empty request: LSE -inf for its rows and every split.
            for (int i = tid; i < NQ * P.num_splits; i += kSoftWarps * 32) {
                const int n = i % NQ, k = i / NQ, rho = grp * NQ + n;
                if (rho < rows_total) {
                    const int64_t t = (int64_t)cur.r * P.qlen + rho / P.heads;
                    P.lse[((int64_t)k * S + t) * P.heads + rho % P.heads] = -INFINITY;
                }
            }
            if (nxt.valid && nxt.ntok > 0) {   // nxt is the first tile of a new unit
                prep_query<NQ>(P, sm, nxt);
                if (lane == 0) mbar_arrive(&ms.q_ready);
            }
            cur = nxt;
            nxt = iter.next(lane);
            continue;
        }
        const bool first = cur.flags & kTileFirst, last = cur.flags & kTileLast;
        if (first) {
#pragma unroll
            for (int n = 0; n < NQ; ++n) l[n] = 0.f;
            if (tid < NQ) ms.m[tid] = -INFINITY;
        }
        // ---- scores of this thread's token
        if (!wait_or_abort(&ms.s_full, n_tiles & 1, &ms.abort_flag)) return;
        tc::fence_after();
        named_sync(kSoftBar, kSoftWarps * 32);   // m[] initialised, c[] of this unit visible
        float s[NQ];
#pragma unroll
        for (int c0 = 0; c0 < NQ; c0 += 16) {
            float hi[16], lo[16];
            tc::ld16(tm + c0, hi);
            tc::ld16(tm + NQ + c0, lo);
            tc::wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) s[c0 + j] = (hi[j] + lo[j] * 0.0625f) * ms.c[c0 + j];
        }
        const bool live = tid < cur.ntok;
#pragma unroll
        for (int n = 0; n < NQ; ++n) s[n] = live ? s[n] : -INFINITY;
        // ---- lazy reference max
        bool over = false;
#pragma unroll
        for (int n = 0; n < NQ; ++n) over |= s[n] > ms.m[n] + kRebase;
        if (tc::bar_any(kSoftBar, kSoftWarps * 32, over)) {
#pragma unroll
            for (int n = 0; n < NQ; ++n) {
                float v = s[n];
#pragma unroll
                for (int d = 16; d; d >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, d));
                if (lane == 0) ms.red[warp][n] = v;
            }
            named_sync(kSoftBar, kSoftWarps * 32);
            if (tid < NQ) {
                const float mo = ms.m[tid];
                float mn = fmaxf(fmaxf(ms.red[0][tid], ms.red[1][tid]), fmaxf(ms.red[2][tid], ms.red[3][tid]));
                mn = fmaxf(mn, mo);
                ms.alpha[tid] = mo == -INFINITY ? 0.f : exp2f(mo - mn);
                ms.m[tid] = mn;
            }
            named_sync(kSoftBar, kSoftWarps * 32);
#pragma unroll
            for (int n = 0; n < NQ; ++n) l[n] *= ms.alpha[n];
            if (!first) {
                // O holds earlier tiles of this unit (the PV before this QK is
                // complete): scale its hi and lo columns of every latent block.
#pragma unroll 1
                for (int b = 0; b < 4; ++b) {
#pragma unroll
                    for (int c0 = 0; c0 < C::NP; c0 += 16) {
                        float v[16];
                        const uint32_t addr = tm + C::NP * (1 + b) + c0;
                        tc::ld16(addr, v);
                        tc::wait_ld();
#pragma unroll
                        for (int j = 0; j < 16; ++j) v[j] *= ms.alpha[(c0 + j) % NQ];
                        tc::st16(addr, v);
                    }
                }
                tc::wait_st();
            }
        }
        // ---- P' = hi + lo/16 of p = 2^(s - m) (<= 2^8), row `tid` of P'^T,
        // written 16 columns at a time (hi chunk c, lo chunk NQ/16 + c)
        uint8_t *prow = sm + C::OffP + (tid >> 3) * 1024 + (tid & 7) * 128;
#pragma unroll
        for (int c0 = 0; c0 < NQ; c0 += 16) {
            uint32_t ph[4], pl[4];
#pragma unroll
            for (int n = c0; n < c0 + 16; n += 2) {
                const float p0 = exp2f(s[n] - ms.m[n]), p1 = exp2f(s[n + 1] - ms.m[n + 1]);
                l[n] += p0;
                l[n + 1] += p1;
                const __nv_fp8x2_storage_t h8 =
                    __nv_cvt_float2_to_fp8x2(make_float2(p0, p1), __NV_SATFINITE, __NV_E4M3);
                const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(h8, __NV_E4M3);
                const float2 hf = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
                const __nv_fp8x2_storage_t l8 = __nv_cvt_float2_to_fp8x2(
                    make_float2((p0 - hf.x) * 16.f, (p1 - hf.y) * 16.f), __NV_SATFINITE, __NV_E4M3);
                const int wi = (n - c0) >> 2, sh = (n & 2) * 8;
                ph[wi] = (sh ? ph[wi] : 0u) | ((uint32_t)h8 << sh);
                pl[wi] = (sh ? pl[wi] : 0u) | ((uint32_t)l8 << sh);
            }
            const int ch = c0 >> 4, cl = (NQ >> 4) + ch;
            *reinterpret_cast<uint4 *>(prow + (((ch ^ tid) & 7) << 4)) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
            *reinterpret_cast<uint4 *>(prow + (((cl ^ tid) & 7) << 4)) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
        }
        tc::fence_async_smem();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ms.p_full);
        ++n_tiles;
        // QK of the unit's last tile is complete: refill the query buffer
        // for the next unit while the tensor cores run this tile's PV.
        if (last && nxt.valid && nxt.ntok > 0) {
            named_sync(kSoftBar, kSoftWarps * 32);   // every thread is done with c[]
            prep_query<NQ>(P, sm, nxt);
            if (lane == 0) mbar_arrive(&ms.q_ready);
        }

        if (last) {
            // ---- unit epilogue: row sums, o, lse
#pragma unroll
            for (int n = 0; n < NQ; ++n) {
                float v = l[n];
#pragma unroll
                for (int d = 16; d; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
                if (lane == 0) ms.red[warp][n] = v;
            }
            if (!wait_or_abort(&ms.o_done, n_units & 1, &ms.abort_flag)) return;
            tc::fence_after();
            named_sync(kSoftBar, kSoftWarps * 32);
            if (tid < NQ) {
                const float lt = ms.red[0][tid] + ms.red[1][tid] + ms.red[2][tid] + ms.red[3][tid];
                ms.invl[tid] = P.kv_scale / lt;
                const int rho = grp * NQ + tid;
                if (rho < rows_total) {
                    const int64_t t = (int64_t)cur.r * P.qlen + rho / P.heads;
                    const int h = rho % P.heads;
                    P.lse[((int64_t)cur.k * S + t) * P.heads + h] = (ms.m[tid] + __log2f(lt)) * 0.69314718055994531f;
                    if (cur.k == cur.n_r - 1)
                        for (int k2 = cur.k + 1; k2 < P.num_splits; ++k2)
                            P.lse[((int64_t)k2 * S + t) * P.heads + h] = -INFINITY;
                }
            }
            named_sync(kSoftBar, kSoftWarps * 32);
#pragma unroll 1
            for (int b = 0; b < 4; ++b) {
#pragma unroll
                for (int c0 = 0; c0 < NQ; c0 += 16) {
                    float hi[16], lo[16];
                    tc::ld16(tm + C::NP * (1 + b) + c0, hi);
                    tc::ld16(tm + C::NP * (1 + b) + NQ + c0, lo);
                    tc::wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int n = c0 + j, rho = grp * NQ + n;
                        if (rho < rows_total) {
                            const int64_t t = (int64_t)cur.r * P.qlen + rho / P.heads;
                            const int64_t orow = ((int64_t)cur.k * S + t) * P.heads + rho % P.heads;
                            P.o[orow * MLA_D_LATENT + 128 * b + tid] =
                                __float2bfloat16_rn((hi[j] + lo[j] * 0.0625f) * ms.invl[n]);
                        }
                    }
                }
            }
            tc::fence_before();
            named_sync(kSoftBar, kSoftWarps * 32);
            ++n_units;
        }
        cur = nxt;
        nxt = iter.next(lane);
    }
}

template <int NQ>
__global__ void __launch_bounds__(kThreads, 1)
    attend_tc_kernel(const __grid_constant__ CUtensorMap mlat, const __grid_constant__ CUtensorMap mrope, const Params P) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Misc<NQ> &ms = misc<NQ>(sm);
    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ms.kv_full[s], kProdWarps);
            mbar_init(&ms.kv_empty[s], 1);
        }
        mbar_init(&ms.s_full, 1);
        mbar_init(&ms.p_full, kSoftWarps);
        mbar_init(&ms.q_ready, kSoftWarps);
        mbar_init(&ms.o_done, 1);
        mbar_init(&ms.fin, 1);
        ms.abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == kMmaWarp) tc::tmem_alloc(&ms.tmem, Cfg<NQ>::TmemCols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    // Register split (per warpgroup, 384 x 168 at launch): the softmax
    // warpgroup holds two NQ-wide rows per thread, the others little.
    // 128 x 232 + 256 x 104 = 56320 <= 64512.
    if (warp < kSoftWarps) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 232;");
        softmax<NQ>(P, sm);
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 104;");
        if (warp == kMmaWarp) mma_issuer<NQ>(P, sm);
        else producer<NQ>(P, &mlat, &mrope, sm);
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == kMmaWarp) tc::tmem_free(ms.tmem, Cfg<NQ>::TmemCols);
}

template <int NQ>
constexpr size_t smem_bytes() {
    return Cfg<NQ>::OffMisc + sizeof(Misc<NQ>) + 1024;
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

template <int NQ>
cudaError_t launch(const CUtensorMap &ml, const CUtensorMap &mr, const Params &P, int grid, cudaStream_t st) {
    const size_t smem = smem_bytes<NQ>();
    cudaError_t e = cudaFuncSetAttribute(attend_tc_kernel<NQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attend_tc_kernel<NQ><<<grid, kThreads, smem, st>>>(ml, mr, P);
    return cudaGetLastError();
}

}  // namespace

// Rows per CTA for the tensor-memory kernel: query rows are split into
// groups of at most 48 (TMEM holds 10 * rows f32 columns), each rounded up
// to a multiple of 16.
void attend_tc_shape(int rows, int *groups, int *nq) {
    int g = (rows + 47) / 48;
    int n = (rows + g - 1) / g;
    n = (n + 15) / 16 * 16;
    *groups = g;
    *nq = n;
}

cudaError_t attend_tc_launch(const void *q, int64_t q_row_stride, const void *kv, int64_t pool_rows,
                             const int32_t *pages, int64_t num_pages, const int32_t *indptr, int R, int qlen,
                             int heads, float scale, float kv_scale, int num_splits, int split_tokens, void *o,
                             float *lse, int grid, cudaStream_t st) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap ml, mr;
    cuuint64_t gdim[2] = {(cuuint64_t)MLA_D_QK, (cuuint64_t)pool_rows};
    cuuint64_t gstr[1] = {(cuuint64_t)MLA_D_QK};
    cuuint32_t box_lat[2] = {128, 1}, box_rope[2] = {64, 1}, es[2] = {1, 1};
    void *base = const_cast<void *>(kv);
    if (enc(&ml, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, gdim, gstr, box_lat, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
            CUDA_SUCCESS ||
        enc(&mr, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, gdim, gstr, box_rope, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
            CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    Params P;
    P.q = static_cast<const __nv_bfloat16 *>(q);
    P.q_row_stride = q_row_stride;
    P.pool_rows = pool_rows;
    P.pages = pages;
    P.num_pages = num_pages;
    P.indptr = indptr;
    P.R = R;
    P.qlen = qlen;
    P.heads = heads;
    P.num_splits = num_splits;
    P.split_tokens = split_tokens;
    P.sc_log2 = scale * kv_scale * 1.4426950408889634f;
    P.kv_scale = kv_scale;
    P.o = static_cast<__nv_bfloat16 *>(o);
    P.lse = lse;
    int groups, nq;
    attend_tc_shape(qlen * heads, &groups, &nq);
    P.row_groups = groups;
    P.nq = nq;
    switch (nq) {
        case 16: return launch<16>(ml, mr, P, grid, st);
        case 32: return launch<32>(ml, mr, P, grid, st);
        default: return launch<48>(ml, mr, P, grid, st);
    }
}

cudaError_t attend_tc_status(unsigned int *flags, bool clear) { return read_status(flags, clear); }

}  // namespace mla
