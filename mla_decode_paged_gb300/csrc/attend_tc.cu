// Split-KV MLA decode attention over a paged fp8 latent cache -- tcgen05
// tensor-memory kernel (sm_103a).
//
// What it computes: vLLM API page
// vllm.models.kimi_k3.amd.specialized_decode.runtime.mla, m1c_inputs (bf16
// query [S, H, 576], flat fp8 token rows addressed by pages / indptr,
// scale and kv_scale, partials o [splits, S, H, 512] bf16 and LSE
// [splits, S, H] f32) and attend (multi-query attention over one latent row
// per token; padded heads skipped through the row stride).  Same work units
// and split rule as the warp-MMA kernel, or the cuts of a host work plan.
//
// Design (one persistent CTA per SM, 16 warps, 512 threads):
//   * warps 9..15 (producers): walk the CTA's tiles (units dealt round robin,
//     or the plan's items) and copy each tile's 128 paged KV rows with TMA
//     tile::gather4 (4 rows per instruction) straight into the UMMA
//     canonical layout: the 512 latent bytes as four 128-byte column blocks
//     with 128B swizzle, the 64 rope bytes with 64B swizzle, two 72 KB
//     stages.  Rows past the tile's tokens (and bad page indices) use an
//     out-of-range row, which the TMA fills with zeros.
//   * The fp8 tile is used as stored (no dequant pass): tokens are the MMA M
//     dimension (128).  QK^T: S^T[tok, n] = K[tok, :576] . Q'[n, :576]; the
//     query is split into two e4m3 terms per row, q*2^e = hi + lo/16, stacked
//     as the B operand's 2*NQ rows, so one MMA chain yields both partial
//     scores (an fp8 query is used as one exact term).  P.V:
//     O^T[lat, n] = V^T[lat, tok] . P'^T[tok, n], with the same smem bytes
//     read MN-major as V^T and P likewise split into hi + lo (p taken
//     against a reference 4 below the running max, so lo ~ p/16 stays in
//     e4m3's normal range).
//     kind::f8f6f4 E4M3 x E4M3 with f32 accumulation in TMEM:
//     S' at columns [0, 2NQ) (all hi, then all lo), O' for latent block b at
//     [2NQ(1+b), 2NQ(2+b)) in P' order (per softmax warpgroup: the hi terms
//     of its query columns, then their lo terms).
//   * warp 8 (MMA): one thread issues 18 QK MMAs (K = 32 each) and, once P
//     is in smem, 16 PV MMAs per tile; tcgen05.commit releases the stage.
//   * warps 0..7 (softmax, two warpgroups, thread = TMEM lane = token, each
//     warpgroup half of the query columns): combine the hi/lo scores, online
//     softmax in the log2 domain with a lazily updated reference max
//     (rebased, and O rescaled in TMEM, only when a score exceeds it by more
//     than 2^8), write P' (hi/lo e4m3) to smem, prepare the next unit's
//     query, and at a unit's end reduce the row sums and write o / lse.
//     With the causal option, column n (query row tq) masks token positions
//     >= L_r - qlen + tq + 1 (a separate instantiation).
//   * Registers: the softmax warpgroups take 176 (184 causal at 48 rows), the
//     MMA and producer warpgroups 80 (72) by setmaxnreg.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <type_traits>

#include "common.cuh"
#include "tc.cuh"

namespace mla {
namespace {

constexpr int kSoftWarps = 8, kMmaWarp = 8, kProdWarp0 = 9, kProdWarps = 7;
constexpr int kSoftThreads = kSoftWarps * 32;
constexpr int kThreads = (kSoftWarps + 1 + kProdWarps) * 32;
constexpr int kSoftBar = 1;          // named barrier of the two softmax warpgroups
constexpr int kGroupBar = 2;         // 2 + g: named barrier of softmax warpgroup g alone
constexpr float kRebase = 8.f;       // log2 headroom before the reference max moves
constexpr float kRefGap = 4.f;       // a rebase puts the reference this far (log2) below the new max

// Tile shape and shared-memory layout per row count NQ: two 128-token
// stages.  (The layout also admits shorter tiles -- a 96-token tile still
// runs M = 128 QK^T MMAs that read 32 rows past it, inside the CTA's
// allocation, with those score lanes ignored -- e.g. three 96-token stages
// at 16 rows; on GB300 that measured slower, the per-tile MMA and sync
// costs being fixed.)
template <int NQ>
struct Cfg {
    static constexpr int T = 128;                          // tokens per tile
    static constexpr int STAGES = 2;
    static constexpr int Blk = (T / 8) * 1024;             // one 128-byte latent column block of a stage
    static constexpr int RopeOff = 4 * Blk;                // rope bytes, 64B swizzle
    static constexpr int StageBytes = RopeOff + (T / 8) * 512;
    static constexpr int KSteps = T / 32;                  // P.V MMAs (K = 32 tokens) per latent block
    static constexpr int Ops = (T / 4) * 5;                // gather4 ops: 4-row groups x (4 latent + 1 rope)
    static constexpr int NP = 2 * NQ;                      // MMA N (hi and lo terms)
    static constexpr int HALF = NQ / 2;                    // columns per softmax warpgroup
    static constexpr int OffQ = STAGES * StageBytes;
    static constexpr int QLatBlock = (NP / 8) * 1024;      // one 128-byte column block of Q'
    static constexpr int QRope = 4 * QLatBlock;
    static constexpr int OffP = OffQ + NP * 576;
    static constexpr int PBytes = (T / 8) * 1024;          // P'^T: one 128-byte row per token
    static constexpr int OffMisc = OffP + PBytes;
    static constexpr uint32_t TmemCols = (10 * NQ <= 256) ? 256 : 512;
    static_assert(T % 32 == 0 && T <= 128, "whole P.V K-steps, at most the MMA M");
    static_assert(Ops <= kProdWarps * 32, "one gather4 per producer lane");
    static_assert(NP <= 128, "a P' row is one 128-byte swizzle span");
};

// Descriptor of the tile in a stage (and of the tile after it), written by
// producer warp 0 before it arrives on the stage's full barrier, so the
// MMA and softmax roles read the work sequence instead of walking indptr.
struct TileMeta {
    int r, k, n_r, ntok, flags;         // flags: kTileFirst / kTileLast / kMetaDone, row group << 8
    int nxt_r, nxt_ntok, nxt_flags;     // nxt_flags = 0: no next tile
    int tok0;                           // the tile's first token position in its request
};
constexpr int kMetaDone = 4, kNxtValid = 16;

template <int NQ>
struct Misc {
    TileMeta meta[Cfg<NQ>::STAGES];
    int64_t orow[NQ];       // o row (element offset / 512) of each query column, -1 for padding
    uint64_t kv_full[Cfg<NQ>::STAGES], kv_empty[Cfg<NQ>::STAGES];
    uint64_t s_full, p_full, q_ready, o_done, fin;
    uint32_t tmem;
    int abort_flag;
    int first[4];           // this CTA's first tile: r, ntok, flags (published before any load)
    uint64_t first_ready;
    int vis[NQ];            // causal: tokens of the request each query column sees
    float c[NQ];            // per query row: scale*kv_scale*log2(e) / 2^e (0 for padding rows)
    float m[NQ];            // reference max of the row, log2 domain
    float alpha[NQ];
    float invl[NQ];
    float red[4][NQ];       // per TMEM lane quarter
};

// Launch parameters.  The field list is shared; the unmasked kernels take
// it with two unused ints after row_groups (Params), the causal ones
// without (ParamsCausal): on GB300 each variant measured 2-10 % faster with
// its own layout (ptxas allocates the two softmax variants' registers
// differently for the two sets of offsets; the causal 48-row kernel spilled
// 92 / 160 bytes with the padded one).
#define MLA_ATTEND_PARAMS(PAD)                                                                      \
    const __nv_bfloat16 *q;                                                                         \
    int64_t q_row_stride;                                                                           \
    int64_t pool_rows;                                                                              \
    const int32_t *pages;                                                                           \
    int64_t num_pages;                                                                              \
    const int32_t *indptr;                                                                          \
    int R, qlen, heads, num_splits, split_tokens, row_groups;                                       \
    PAD                                                                                             \
    int log2p;                    /* blocks of 2^log2p rows (0: one row per page) */                 \
    int q8;                       /* q holds e4m3 codes (row stride in bytes) */                    \
    const int32_t *plan;          /* work plan (null: units dealt round robin) */                   \
    int plan_len;                 /* its length in int32 (the host caps it at INT32_MAX) */         \
    const int32_t *last_page_len; /* rows used in each request's last block (log2p > 0) */          \
    float sc_log2;                                                                                  \
    float kv_scale;                                                                                 \
    __nv_bfloat16 *o;                                                                               \
    float *lse;

struct Params {
    MLA_ATTEND_PARAMS(int unused_[2];)
};
struct ParamsCausal {
    MLA_ATTEND_PARAMS()
};
#undef MLA_ATTEND_PARAMS

template <bool CAUSAL>
using ParamsOf = typename std::conditional<CAUSAL, ParamsCausal, Params>::type;

// Tokens of request r (indptr already validated by the producers for any
// request that reaches the softmax with tokens).
template <class PP>
__device__ __forceinline__ int request_tokens(const PP &P, int r) {
    const int a = __ldg(P.indptr + r), b = __ldg(P.indptr + r + 1);
    return (P.log2p == 0 || b == a) ? b - a : ((b - a - 1) << P.log2p) + __ldg(P.last_page_len + r);
}

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

// N consecutive f32 TMEM columns (N a multiple of 8) of this warp's lanes.
template <int N>
__device__ __forceinline__ void ld_cols(uint32_t taddr, float (&v)[N]) {
#pragma unroll
    for (int c = 0; c < N; c += 8) {
        uint32_t r[8];
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                     : "r"(taddr + c));
#pragma unroll
        for (int i = 0; i < 8; ++i) v[c + i] = __uint_as_float(r[i]);
    }
}

template <int N>
__device__ __forceinline__ void st_cols(uint32_t taddr, const float (&v)[N]) {
#pragma unroll
    for (int c = 0; c < N; c += 8) {
        asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr + c),
                     "r"(__float_as_uint(v[c])), "r"(__float_as_uint(v[c + 1])), "r"(__float_as_uint(v[c + 2])),
                     "r"(__float_as_uint(v[c + 3])), "r"(__float_as_uint(v[c + 4])), "r"(__float_as_uint(v[c + 5])),
                     "r"(__float_as_uint(v[c + 6])), "r"(__float_as_uint(v[c + 7]))
                     : "memory");
    }
}

__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Sums (MAX: maxima) over the warp's 32 lanes of each of a lane's C
// values, by a transposing butterfly: while C is even, a step exchanges half
// of the values with the partner lane and keeps the combination of the other
// half, so later steps move fewer values.  On return a lane holds
// colsum_count(C) results, of columns base + [0, count); lanes that differ
// only in the bits colsum_dup(C) hold the same results.
__host__ __device__ constexpr int colsum_count(int c) {
    for (int d = 16; d >= 1; d >>= 1)
        if (c % 2 == 0) c /= 2;
    return c;
}
__host__ __device__ constexpr int colsum_dup(int c) {
    int m = 0;
    for (int d = 16; d >= 1; d >>= 1) {
        if (c % 2 == 0) c /= 2;
        else m |= d;
    }
    return m;
}
template <int C, int D, bool MAX = false>
__device__ __forceinline__ void colsum(float *v, int lane, int &base) {
    if constexpr (D >= 1) {
        if constexpr (C % 2 == 0) {
            const bool up = (lane & D) != 0;
#pragma unroll
            for (int i = 0; i < C / 2; ++i) {
                const float send = up ? v[i] : v[C / 2 + i];
                const float keep = up ? v[C / 2 + i] : v[i];
                const float got = __shfl_xor_sync(0xffffffffu, send, D);
                v[i] = MAX ? fmaxf(keep, got) : keep + got;
            }
            if (up) base += C / 2;
            colsum<C / 2, D / 2, MAX>(v, lane, base);
        } else {
#pragma unroll
            for (int i = 0; i < C; ++i) {
                const float got = __shfl_xor_sync(0xffffffffu, v[i], D);
                v[i] = MAX ? fmaxf(v[i], got) : v[i] + got;
            }
            colsum<C, D / 2, MAX>(v, lane, base);
        }
    }
}

// ------------------------------------------------------------------ producers

// PAGED compiles in block-table addressing (a separate instantiation: the
// flat-row path keeps its plain page lookup).
template <int NQ, bool PAGED, class PP>
__device__ void producer(const PP &P, const CUtensorMap *mlat, const CUtensorMap *mrope, uint8_t *sm) {
    using C = Cfg<NQ>;
    Misc<NQ> &ms = misc<NQ>(sm);
    const int lane = threadIdx.x & 31, pw = (threadIdx.x >> 5) - kProdWarp0;
    const int op = pw + kProdWarps * lane;  // ops dealt round-robin over the producer warps
    const bool has_op = op < C::Ops;
    const int g4 = op / 5, part = op % 5;
    TileIter<C::T, PAGED> iter;
    if (PAGED)
        iter.init(P.indptr, P.R, P.num_pages, P.num_splits, P.split_tokens, P.row_groups, lane, P.log2p,
                  P.last_page_len, P.plan, P.plan_len);
    else
        iter.init(P.indptr, P.R, P.num_pages, P.num_splits, P.split_tokens, P.row_groups, lane, 0, nullptr,
                  P.plan, P.plan_len);
    // KV rows stream through L2 evicted first: the split partials written
    // meanwhile stay for the merge, and dirty lines left in L2 by earlier
    // work are not forced out by the stream (with several row groups the
    // other CTAs of a tile read it at about the same time and still find
    // it: measured faster for one and for two groups).
    const uint64_t pol = tc::l2_policy(true);
    auto fetch = [&](const Tile &T, int (&rows)[4]) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int tok = 4 * g4 + i;
            int r = -1;
            if (T.valid && has_op && tok < T.ntok) {
                if (PAGED) {
                    // token j of the request: row pages[base + j / 2^log2p] * 2^log2p + j % 2^log2p
                    const int j = T.tok0 + tok;
                    const int64_t p = __ldg(P.pages + (int64_t)T.base + (j >> P.log2p));
                    const int64_t row = (p << P.log2p) + (j & ((1 << P.log2p) - 1));
                    if (p < 0 || row >= P.pool_rows) flag(MLA_DEV_BAD_PAGE);
                    else r = (int)row;
                } else {
                    const int64_t p = __ldg(P.pages + (int64_t)T.base + T.tok0 + tok);
                    if (p < 0 || p >= P.pool_rows) flag(MLA_DEV_BAD_PAGE);
                    else r = (int)p;
                }
            }
            rows[i] = r;
        }
    };
    // The first unit for the softmax warps' query preparation.  With a plan
    // and 32 or 48 query rows (whose preparation the first QK^T waits for) it
    // is published as soon as the first item is read (its request and row
    // group checked against the launch here; its token range, which needs
    // the request's page offsets, by next()), one round of loads earlier.
    int fi[4] = {0, 0, 0, 0};
    bool early = false;
    if (NQ >= 32 && P.plan) {
        early = iter.open_plan(P.plan, fi);
        const int ig = (fi[1] >> 18) & 8191;
        early = early && fi[1] >= 0 && fi[0] >= 0 && fi[0] < P.R && ig < P.row_groups && fi[3] >= 0;
        if (early && pw == 0 && lane == 0) {
            ms.first[0] = fi[0];
            ms.first[1] = min(C::T, fi[3]);
            ms.first[2] = kTileFirst | (ig << 8);
            mbar_arrive(&ms.first_ready);
        }
    }
    Tile cur = iter.next(lane, P.plan, NQ >= 32 && P.plan ? fi : nullptr);
    if (!early && pw == 0 && lane == 0) {
        ms.first[0] = cur.r;
        ms.first[1] = cur.ntok;
        ms.first[2] = cur.valid ? cur.flags : kMetaDone;
        mbar_arrive(&ms.first_ready);
    }
    int rows[4];
    fetch(cur, rows);
    // The next tile's descriptor goes into this tile's stage; its rows are
    // fetched after this tile's copies are issued (so the first copies wait
    // for one round of index loads, not two).
    Tile nxt = iter.next(lane, P.plan);
    int n_issued = 0;
    const int rows_total = P.qlen * P.heads;
    for (int it = 0; cur.valid; ++it) {
        // The next unit's query rows into L2, kept there against the KV
        // stream (the softmax converts them when this unit ends): one bulk
        // prefetch per row, or line prefetches for a row that is not
        // 16-byte aligned (a row stride that is not a multiple of 8).
        if (pw == kProdWarps - 1 && nxt.valid && (nxt.flags & kTileFirst) && nxt.ntok > 0) {
            const int grp = nxt.flags >> 8;
            const int esz = P.q8 ? 1 : 2;   // bytes per query element (the row stride counts elements)
            const uint64_t keep = tc::l2_policy_last();
            for (int n = lane; n < NQ; n += 32) {
                const int rho = grp * NQ + n;
                if (rho < rows_total) {
                    const int tq = rho / P.heads, h = rho - tq * P.heads;
                    const uint8_t *row = reinterpret_cast<const uint8_t *>(P.q) +
                                         (((int64_t)nxt.r * P.qlen + tq) * P.q_row_stride + (int64_t)h * MLA_D_QK) * esz;
                    if ((reinterpret_cast<uintptr_t>(row) & 15) == 0) tc::bulk_prefetch_l2(row, MLA_D_QK * esz, keep);
                    else
                        for (int b = 0; b < MLA_D_QK * esz; b += 128) prefetch_l2(row + b);
                }
            }
        }
        const int s = it % C::STAGES;
        if (!wait_or_abort(&ms.kv_empty[s], ((it / C::STAGES) & 1) ^ 1, &ms.abort_flag)) return;
        const bool issue = has_op && cur.ntok > 0;
        uint32_t bytes = issue ? (part < 4 ? 512u : 256u) : 0u;
#pragma unroll
        for (int d = 16; d; d >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, d);
        if (lane == 0) {
            if (pw == 0) {
                TileMeta m;
                m.r = cur.r; m.k = cur.k; m.n_r = cur.n_r; m.ntok = cur.ntok; m.flags = cur.flags;
                m.nxt_r = nxt.r; m.nxt_ntok = nxt.ntok; m.nxt_flags = nxt.valid ? (nxt.flags | kNxtValid) : 0;
                m.tok0 = cur.tok0;
                ms.meta[s] = m;
            }
            mbar_arrive_expect_tx(&ms.kv_full[s], bytes);
        }
        __syncwarp();
        if (issue) {
            uint8_t *st = sm + s * C::StageBytes;
            const int g8 = g4 >> 1, half = g4 & 1;
            if (part < 4)
                tc::gather4_hint(st + part * C::Blk + g8 * 1024 + half * 512, mlat, part * 128, rows[0], rows[1],
                                 rows[2], rows[3], &ms.kv_full[s], pol);
            else
                tc::gather4_hint(st + C::RopeOff + g8 * 512 + half * 256, mrope, 512, rows[0], rows[1], rows[2],
                                 rows[3], &ms.kv_full[s], pol);
        }
        fetch(nxt, rows);
        cur = nxt;
        if (cur.valid) nxt = iter.next(lane, P.plan);
        n_issued = it + 1;
    }
    // No more work: one last "done" descriptor through the next stage.
    const int s2 = n_issued % C::STAGES;
    if (!wait_or_abort(&ms.kv_empty[s2], ((n_issued / C::STAGES) & 1) ^ 1, &ms.abort_flag)) return;
    if (lane == 0) {
        if (pw == 0) ms.meta[s2].flags = kMetaDone;
        mbar_arrive(&ms.kv_full[s2]);
    }
}

// ------------------------------------------------------------------ MMA issuer

// Per tile, in order: QK^T (18 MMAs into S), then -- once the softmax has
// written P' -- P.V (16 MMAs, latent blocks interleaved so consecutive MMAs
// feed different accumulators).  A stage is held only for its own tile.
template <int NQ, class PP>
__device__ void mma_issuer(const PP &P, uint8_t *sm) {
    using C = Cfg<NQ>;
    Misc<NQ> &ms = misc<NQ>(sm);
    const int lane = threadIdx.x & 31;
    const uint32_t base = smem_u32(sm);
    const uint32_t tm = ms.tmem;
    constexpr uint32_t kIdQK = tc::idesc_e4m3(C::NP, false, false);
    constexpr uint32_t kIdPV = tc::idesc_e4m3(C::NP, true, true);
    int n_p = 0, n_units = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
        const int s = it % C::STAGES;
        if (!(ok = wait_or_abort(&ms.kv_full[s], (it / C::STAGES) & 1, &ms.abort_flag))) break;
        const TileMeta M = ms.meta[s];
        if (M.flags & kMetaDone) break;
        if (M.ntok == 0) {
            // Empty request: nothing to multiply (the softmax warps read the
            // descriptor on their own).
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.kv_empty[s]);
            continue;
        }
        const bool first = M.flags & kTileFirst;
        if (first) {
            if (!(ok = wait_or_abort(&ms.q_ready, n_units & 1, &ms.abort_flag))) break;
            ++n_units;
        }
        tc::fence_after();
        const uint32_t st = base + s * C::StageBytes;
        if (lane == 0) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int a = j >> 2, off = (j & 3) * 32;
                tc::mma_e4m3(tm, tc::sdesc(st + a * C::Blk + off, 16, 1024, tc::kSw128),
                             tc::sdesc(base + C::OffQ + a * C::QLatBlock + off, 16, 1024, tc::kSw128), kIdQK, j > 0);
            }
#pragma unroll
            for (int j = 0; j < 2; ++j)
                tc::mma_e4m3(tm, tc::sdesc(st + C::RopeOff + j * 32, 16, 512, tc::kSw64),
                             tc::sdesc(base + C::OffQ + C::QRope + j * 32, 16, 512, tc::kSw64), kIdQK, true);
            tc::commit(&ms.s_full);
        }
        __syncwarp();
        if (!(ok = wait_or_abort(&ms.p_full, (n_p++) & 1, &ms.abort_flag))) break;
        tc::fence_after();
        if (lane == 0) {
#pragma unroll
            for (int kk = 0; kk < C::KSteps; ++kk)
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    tc::mma_e4m3(tm + C::NP * (1 + b), tc::sdesc(st + b * C::Blk + kk * 4096, C::Blk, 1024, tc::kSw128),
                                 tc::sdesc(base + C::OffP + kk * 4096, C::Blk, 1024, tc::kSw128), kIdPV,
                                 !(first && kk == 0));
            tc::commit(&ms.kv_empty[s]);
            if (M.flags & kTileLast) tc::commit(&ms.o_done);
        }
        __syncwarp();
    }
    // Every MMA issued so far must be complete before TMEM is released.
    if (lane == 0) tc::commit(&ms.fin);
    __syncwarp();
    mbar_wait(&ms.fin, 0);
}

// ------------------------------------------------------------------ softmax

// An fp8 query (e4m3 codes, the q_scale folded into the softmax scale):
// row n of Q' holds the codes as they are, row NQ + n (the lo term) zeros,
// c[n] = scale * kv_scale * log2(e).  Run by the 8 softmax warps; a warp
// copies a 576-byte row as 36 16-byte chunks into the swizzled layouts.
template <int NQ, class PP>
__device__ __noinline__ void prep_rows_q8(const PP &P, uint8_t *sm, int req, int grp) {
    using C = Cfg<NQ>;
    Misc<NQ> &ms = misc<NQ>(sm);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rows_total = P.qlen * P.heads;
    for (int n = warp; n < NQ; n += kSoftWarps) {
        const int rho = grp * NQ + n;
        const bool valid = rho < rows_total;
        const uint8_t *src = reinterpret_cast<const uint8_t *>(P.q);
        if (valid) {
            const int tq = rho / P.heads, h = rho % P.heads;
            src += ((int64_t)req * P.qlen + tq) * P.q_row_stride + (int64_t)h * MLA_D_QK;
        }
        for (int ch = lane; ch < MLA_D_QK / 16; ch += 32) {
            const uint4 v = valid ? __ldg(reinterpret_cast<const uint4 *>(src) + ch) : make_uint4(0, 0, 0, 0);
            const int d = ch * 16;
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
            *reinterpret_cast<uint4 *>(sm + off_hi) = v;
            *reinterpret_cast<uint4 *>(sm + off_lo) = make_uint4(0, 0, 0, 0);
        }
        if (lane == 0) ms.c[n] = valid ? P.sc_log2 : 0.f;
    }
}

// The query rows of tile T's request and row group as the B operand Q':
// row n = q_n * 2^e_n rounded to e4m3 (hi), row NQ + n = 16 * (q_n * 2^e_n
// - hi) rounded to e4m3 (lo), in the K-major 128B / 64B swizzled layouts;
// c[n] = scale * kv_scale * log2(e) / 2^e_n.  Run by the 8 softmax warps,
// out of line (once per unit; up to three of a warp's rows loaded at a
// time).  At a unit change its conversion work and its code, fetched
// cold, bound the cost of the change; fully unrolled and inlined at its
// three call sites it measured slower.
template <int NQ, class PP>
__device__ __noinline__ void prep_query(const PP &P, uint8_t *sm, int req, int grp) {
    using C = Cfg<NQ>;
    Misc<NQ> &ms = misc<NQ>(sm);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rows_total = P.qlen * P.heads;
    if (P.q8) {
        prep_rows_q8<NQ>(P, sm, req, grp);
    } else {
    constexpr int kPerWarp = NQ / kSoftWarps;   // 2, 4 or 6 rows per warp
    constexpr int kBatch = kPerWarp % 3 == 0 ? 3 : 2;   // rows whose loads are in flight together
#pragma unroll 1
    for (int i0 = 0; i0 < kPerWarp; i0 += kBatch) {
        uint4 v[kBatch][3];
        bool valid[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int n = warp + kSoftWarps * (i0 + i);
            const int rho = grp * NQ + n;
            valid[i] = rho < rows_total;
            const __nv_bfloat16 *src = P.q;
            if (valid[i]) {
                const int tq = rho / P.heads, h = rho % P.heads;
                src = P.q + ((int64_t)req * P.qlen + tq) * P.q_row_stride + (int64_t)h * MLA_D_QK;
            }
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                const int ch = lane + 32 * j;
                v[i][j] = (valid[i] && ch < 72) ? __ldg(reinterpret_cast<const uint4 *>(src) + ch)
                                                : make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
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
                    // lo = 16 (x - hi) in f16x2, exactly: x (a bf16 value times
                    // a power of two, |x| < 256) and hi are f16 values, x - hi
                    // is exact (hi is x rounded to e4m3), and so is the x16.
                    const float2 x = make_float2(bf16_lo(w[e2]) * sc, bf16_hi(w[e2]) * sc);
                    const __nv_fp8x2_storage_t h8 = __nv_cvt_float2_to_fp8x2(x, __NV_SATFINITE, __NV_E4M3);
                    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(h8, __NV_E4M3);
                    const __half2 r = __hmul2(__hsub2(__float22half2_rn(x), *reinterpret_cast<const __half2 *>(&hr)),
                                              __float2half2_rn(16.f));
                    const __nv_fp8x2_storage_t l8 =
                        __nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<const __half2_raw *>(&r), __NV_SATFINITE, __NV_E4M3);
                    if ((e2 & 1) == 0) {
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
    }
    tc::fence_async_smem();   // generic-proxy writes -> tensor-core reads
    named_sync(kSoftBar, kSoftThreads);
    __syncwarp();
    if (lane == 0) mbar_arrive(&ms.q_ready);
}

// p = 2^(s - m) of a thread's H2 scores, added to the row sums l and split
// into e4m3 hi + lo (hi = p rounded to 3 mantissa bits in fp32, exact in
// e4m3; lo = p - hi), packed four columns per word.  The reference m sits
// kRefGap = 4 below the largest score seen when it was last moved, so p is
// at most 16 then and below 2^kRebase until the next move: 16 times the
// max-referenced probability, which keeps lo (~p/16) in e4m3's normal range
// as far down as the max-referenced p = 2^-6.  REL (the unmasked kernel): sc
// holds s - m already.  GUARD maps s = -inf to 0 even where m is still -inf
// (causal tiles; without the mask every column sees each tile's live tokens,
// so m is finite by then).
// 2^x by the hardware approximation (PTX ex2.approx.ftz.f32: relative
// error ~2^-22, results below 2^-126 flushed to 0).  p is then rounded to
// two e4m3 terms (~8 significant bits), so the approximation is invisible
// next to that rounding.
__device__ __forceinline__ float exp2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int H2, bool GUARD, bool REL>
__device__ __forceinline__ void p_split(const float (&sc)[H2], const float (&mr)[H2], float (&l)[H2],
                                        uint32_t (&ph)[H2 / 4], uint32_t (&pl)[H2 / 4]) {
#pragma unroll
    for (int j = 0; j < H2; j += 2) {
        float hv[2], lv[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const float x = REL ? sc[j + e] : sc[j + e] - mr[j + e];   // REL: sc already holds s - m
            const float pv = (!GUARD || sc[j + e] > -INFINITY) ? exp2_approx(x) : 0.f;
            l[j + e] += pv;
            hv[e] = __uint_as_float((__float_as_uint(pv) + 0x80000u) & 0xFFF00000u);
            lv[e] = pv - hv[e];
        }
        const uint32_t h8 = __nv_cvt_float2_to_fp8x2(make_float2(hv[0], hv[1]), __NV_SATFINITE, __NV_E4M3);
        const uint32_t l8 = __nv_cvt_float2_to_fp8x2(make_float2(lv[0], lv[1]), __NV_SATFINITE, __NV_E4M3);
        const int wi = j >> 2;
        if ((j & 2) == 0) {
            ph[wi] = h8;
            pl[wi] = l8;
        } else {
            ph[wi] |= h8 << 16;
            pl[wi] |= l8 << 16;
        }
    }
}

// The end of a unit, once its row sums are in red[] and its reference maxima
// in m[]: waits for the unit's last P.V, writes each row's LSE (and -inf for
// the splits past the request's last, k = n_r - 1) and its o rows.  Kept
// out of line: it runs once per unit, and inlined it only lengthens the
// per-tile code the instruction cache has to hold.
template <int NQ, class PP>
__device__ __noinline__ bool unit_epilogue(const PP &P, uint8_t *sm, int k, int n_r, uint32_t o_parity) {
    using C = Cfg<NQ>;
    constexpr int H2 = C::HALF;
    Misc<NQ> &ms = misc<NQ>(sm);
    const int tid = threadIdx.x, warp = tid >> 5, wq = warp & 3, t = tid & 127, n0 = (warp >> 2) * H2;
    const uint32_t tm = ms.tmem + ((uint32_t)(wq * 32) << 16);
    const int S = P.R * P.qlen;
    if (!wait_or_abort(&ms.o_done, o_parity, &ms.abort_flag)) return false;
    tc::fence_after();
    named_sync(kSoftBar, kSoftThreads);
    if (tid < NQ) {
        const float lt = ms.red[0][tid] + ms.red[1][tid] + ms.red[2][tid] + ms.red[3][tid];
        ms.invl[tid] = lt > 0.f ? P.kv_scale / lt : 0.f;   // a row that saw no token: o = 0
        const int64_t orow = ms.orow[tid];
        if (orow >= 0) {
            P.lse[orow] = (ms.m[tid] + __log2f(lt)) * 0.69314718055994531f;
            if (k == n_r - 1) {
                const int64_t step = (int64_t)S * P.heads;
                for (int k2 = k + 1; k2 < P.num_splits; ++k2) P.lse[orow + (k2 - k) * step] = -INFINITY;
            }
        }
    }
    named_sync(kSoftBar, kSoftThreads);
    // o rows: each latent block as bf16 [row][128] in the P' buffer
    // (idle: this tile's P.V is done), then 16-byte row chunks out.
    float iv[H2];
#pragma unroll
    for (int j = 0; j < H2; ++j) iv[j] = ms.invl[n0 + j];
    __nv_bfloat16 *stg = reinterpret_cast<__nv_bfloat16 *>(sm + C::OffP);
    // latent blocks staged at a time (4, 2 or 1: a divisor of 4)
    constexpr int kBlkRound = 4 * NQ * 256 <= C::PBytes ? 4 : 2 * NQ * 256 <= C::PBytes ? 2 : 1;
#pragma unroll 1
    for (int b0 = 0; b0 < 4; b0 += kBlkRound) {
#pragma unroll 1
        for (int bb = 0; bb < kBlkRound; ++bb) {
            float hi[H2], lo[H2];
            ld_cols<H2>(tm + C::NP * (1 + b0 + bb) + 2 * n0, hi);   // P' column order: see softmax
            ld_cols<H2>(tm + C::NP * (1 + b0 + bb) + 2 * n0 + H2, lo);
            tc::wait_ld();
#pragma unroll
            for (int j = 0; j < H2; ++j)
                stg[(bb * NQ + n0 + j) * 128 + t] = __float2bfloat16_rn((hi[j] + lo[j]) * iv[j]);
        }
        named_sync(kSoftBar, kSoftThreads);
        for (int c = tid; c < kBlkRound * NQ * 16; c += kSoftThreads) {
            const int row = c >> 4, ch = c & 15, bb = row / NQ, n = row - bb * NQ;
            const int64_t orow = ms.orow[n];
            if (orow >= 0)
                *reinterpret_cast<uint4 *>(P.o + orow * MLA_D_LATENT + 128 * (b0 + bb) + 8 * ch) =
                    *reinterpret_cast<const uint4 *>(stg + row * 128 + 8 * ch);
        }
        named_sync(kSoftBar, kSoftThreads);
    }
    return true;
}

// Softmax warpgroups: thread (warpgroup g, TMEM lane t) owns token t of the
// tile (latent row t of O in the epilogue) and query columns
// [g*NQ/2, (g+1)*NQ/2).  Per column it keeps c (the score scale) and
// the reference m in registers (kRefGap below the running max).  The tile
// sequence comes from the
// stage descriptors.  CAUSAL compiles the causal mask in (a separate
// instantiation, so the unmasked path carries none of its work).
template <int NQ, bool CAUSAL, class PP>
__device__ void softmax(const PP &P, uint8_t *sm) {
    using C = Cfg<NQ>;
    constexpr int H2 = C::HALF;
    Misc<NQ> &ms = misc<NQ>(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wq = warp & 3, t = tid & 127, n0 = (warp >> 2) * H2;
    const uint32_t tm = ms.tmem + ((uint32_t)(wq * 32) << 16);
    const int S = P.R * P.qlen, rows_total = P.qlen * P.heads;
    float l[H2], cr[H2], mr[H2];
    int n_s = 0, n_units = 0;
    int vmin = 0;   // causal: tokens of the request every query row sees (L_r - qlen + 1)
    uint8_t *prow = sm + C::OffP + (t >> 3) * 1024 + (t & 7) * 128;
    // The first unit's query is prepared while its first tile is loading;
    // later ones at the end of the unit before them.
    if (!wait_or_abort(&ms.first_ready, 0, &ms.abort_flag)) return;
    if (!(ms.first[2] & kMetaDone) && ms.first[1] > 0) prep_query<NQ>(P, sm, ms.first[0], ms.first[2] >> 8);
    for (int it = 0;; ++it) {
        const int s = it % C::STAGES;
        if (!wait_or_abort(&ms.kv_full[s], (it / C::STAGES) & 1, &ms.abort_flag)) return;
        const TileMeta M = ms.meta[s];
        __syncwarp();
        if (M.flags & kMetaDone) return;
        if (lane == 0) mbar_arrive(&ms.kv_empty[s]);   // descriptor read
        const int grp = M.flags >> 8;
        const bool first = M.flags & kTileFirst, last = M.flags & kTileLast;
        const bool next_unit = (M.nxt_flags & kNxtValid) && M.nxt_ntok > 0 && last;
        if (M.ntok == 0) {
            // Empty request: LSE -inf for its rows and every split.
            for (int i = tid; i < NQ * P.num_splits; i += kSoftThreads) {
                const int n = i % NQ, k = i / NQ, rho = grp * NQ + n;
                if (rho < rows_total) {
                    const int64_t tt = (int64_t)M.r * P.qlen + rho / P.heads;
                    P.lse[((int64_t)k * S + tt) * P.heads + rho % P.heads] = -INFINITY;
                }
            }
            if (next_unit) prep_query<NQ>(P, sm, M.nxt_r, M.nxt_flags >> 8);
            continue;
        }
        if (first) {
            // c[] of this unit was published by prep_query's barrier.
#pragma unroll
            for (int j = 0; j < H2; ++j) {
                l[j] = 0.f;
                cr[j] = ms.c[n0 + j];
                mr[j] = CAUSAL ? -INFINITY : 0.f;
            }
            if (tid < NQ) {
                const int rho = grp * NQ + tid;
                ms.orow[tid] = rho < rows_total
                                   ? ((int64_t)M.k * S + (int64_t)M.r * P.qlen + rho / P.heads) * P.heads + rho % P.heads
                                   : -1;
                if (CAUSAL) {   // L_r from indptr (validated by the producers: ntok > 0 here)
                    const int len = request_tokens(P, M.r);
                    ms.vis[tid] = len - P.qlen + rho / P.heads + 1;
                }
            }
            // vis[] is read below by every softmax thread in this same tile
            if (CAUSAL) {
                vmin = request_tokens(P, M.r) - P.qlen + 1;
                named_sync(kSoftBar, kSoftThreads);
            }
        }
        // Only a tile that reaches past vmin needs the per-column mask.
        const bool mask_tile = CAUSAL && M.tok0 + M.ntok > vmin;
        // ---- scores (log2 domain) of this thread's token and columns
        if (!wait_or_abort(&ms.s_full, n_s & 1, &ms.abort_flag)) return;
        ++n_s;
        tc::fence_after();
        float sc[H2];
        bool over = false;
        {
            float hi[H2], lo[H2];
            ld_cols<H2>(tm + n0, hi);
            ld_cols<H2>(tm + NQ + n0, lo);
            tc::wait_ld();
            const bool live = t < M.ntok;
            if constexpr (!CAUSAL) {
                // Unmasked: scores kept relative to the reference max, s - m,
                // with m folded into the scaling FMA.  A unit's first tile
                // runs with m = 0 (so sc = s) and always votes; every column
                // sees that tile's live tokens, so m is finite after it.
                if (live) {
#pragma unroll
                    for (int j = 0; j < H2; ++j) {
                        sc[j] = fmaf(cr[j], fmaf(lo[j], 0.0625f, hi[j]), -mr[j]);
                        over |= sc[j] > kRebase;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < H2; ++j) sc[j] = -INFINITY;
                }
                over |= first;
            } else if (!mask_tile) {
#pragma unroll
                for (int j = 0; j < H2; ++j) {
                    sc[j] = live ? cr[j] * fmaf(lo[j], 0.0625f, hi[j]) : -INFINITY;
                    over |= sc[j] - mr[j] > kRebase;   // also true for every live token while m = -inf
                }
            } else {
                const int pos = M.tok0 + t;   // token position in the request
#pragma unroll
                for (int j = 0; j < H2; ++j) {
                    sc[j] = live && pos < ms.vis[n0 + j] ? cr[j] * fmaf(lo[j], 0.0625f, hi[j]) : -INFINITY;
                    over |= sc[j] - mr[j] > kRebase;
                }
            }
        }
        // ---- lazy reference max (rare after a unit's first tile).  A
        // warpgroup's columns are its own, so the vote and the rebase stay
        // within the warpgroup.
        const bool g1 = warp >= 4;
        if (g1 ? tc::bar_any(kGroupBar + 1, 128, over) : tc::bar_any(kGroupBar, 128, over)) {
            {
                // per-warp column maxima (transposing butterfly)
                float v[H2];
#pragma unroll
                for (int j = 0; j < H2; ++j) v[j] = sc[j];
                int cb = 0;
                colsum<H2, 16, true>(v, lane, cb);
                if ((lane & colsum_dup(H2)) == 0) {
#pragma unroll
                    for (int i = 0; i < colsum_count(H2); ++i) ms.red[wq][n0 + cb + i] = v[i];
                }
            }
            if (g1) named_sync(kGroupBar + 1, 128);
            else named_sync(kGroupBar, 128);
            if (t < H2) {
                const int n = n0 + t;
                const float mx = fmaxf(fmaxf(ms.red[0][n], ms.red[1][n]), fmaxf(ms.red[2][n], ms.red[3][n]));
                if constexpr (!CAUSAL) {
                    // mx is the tile's largest s (first tile) or s - m; the
                    // reference goes kRefGap below the new max (p <= 16 after
                    // a rebase, < 2^kRebase before the next).
                    if (first) {
                        ms.alpha[n] = 0.f;
                        ms.m[n] = mx - kRefGap;
                    } else {
                        const float d = fmaxf(mx - kRefGap, 0.f);
                        ms.alpha[n] = exp2f(-d);
                        ms.m[n] += d;
                    }
                } else {
                    const float mo = first ? -INFINITY : ms.m[n];
                    const float mn = fmaxf(mx - kRefGap, mo);   // stays -inf for a column with no visible token
                    ms.alpha[n] = mo == -INFINITY ? 0.f : exp2f(mo - mn);
                    ms.m[n] = mn;
                }
            }
            if (g1) named_sync(kGroupBar + 1, 128);
            else named_sync(kGroupBar, 128);
#pragma unroll
            for (int j = 0; j < H2; ++j) {
                const float mn = ms.m[n0 + j];
                if constexpr (!CAUSAL) sc[j] -= mn - mr[j];   // now s - (new m); mr = 0 on a first tile
                mr[j] = mn;
                l[j] *= ms.alpha[n0 + j];
            }
            if (!first) {
                // O holds this unit's earlier tiles (their P.V is complete:
                // this tile's QK^T was issued after it): scale this
                // warpgroup's hi and lo columns of every latent block.
                if constexpr (NQ == 32) {
                    // Eight columns at a time: this kernel's register
                    // allocation spills on this rare path otherwise.
#pragma unroll 1
                    for (int c = 0; c < H2; c += 8) {
                        float a[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) a[i] = ms.alpha[n0 + c + i];
#pragma unroll 1
                        for (int bp = 0; bp < 8; ++bp) {
                            float v[8];
                            const uint32_t addr = tm + C::NP * (1 + (bp >> 1)) + 2 * n0 + (bp & 1) * H2 + c;
                            ld_cols<8>(addr, v);
                            tc::wait_ld();
#pragma unroll
                            for (int i = 0; i < 8; ++i) v[i] *= a[i];
                            st_cols<8>(addr, v);
                        }
                    }
                } else {
#pragma unroll 1
                    for (int b = 0; b < 4; ++b) {
#pragma unroll 1
                        for (int part = 0; part < 2; ++part) {
                            float v[H2];
                            const uint32_t addr = tm + C::NP * (1 + b) + 2 * n0 + part * H2;
                            ld_cols<H2>(addr, v);
                            tc::wait_ld();
#pragma unroll
                            for (int j = 0; j < H2; ++j) v[j] *= ms.alpha[n0 + j];
                            st_cols<H2>(addr, v);
                        }
                    }
                }
                tc::wait_st();
            }
        }
        // ---- P' = hi + lo of p = 2^(s - m) (<= 2^8): hi = p rounded to 3
        // mantissa bits in fp32 (exact in e4m3), lo = p - hi; this thread's
        // bytes of row t of P'^T
        uint32_t ph[H2 / 4], pl[H2 / 4];
        if constexpr (!CAUSAL) p_split<H2, false, true>(sc, mr, l, ph, pl);
        else if (!mask_tile) p_split<H2, false, false>(sc, mr, l, ph, pl);
        else p_split<H2, true, false>(sc, mr, l, ph, pl);   // masked entries: 0 even while a column's m is -inf
        if (C::T == 128 || t < C::T) {   // lanes past a shorter tile have no P' row
            // P' columns are ordered by warpgroup, [hi of its H2 columns, lo
            // of them]: this thread's 2*H2 bytes of row t start at 2*n0 and
            // fill H2/8 whole 16-byte swizzle chunks (one store each).
            uint32_t w[H2 / 2];
#pragma unroll
            for (int i = 0; i < H2 / 4; ++i) {
                w[i] = ph[i];
                w[H2 / 4 + i] = pl[i];
            }
#pragma unroll
            for (int q = 0; q < H2 / 8; ++q) {
                const int chunk = 2 * n0 / 16 + q;
                *reinterpret_cast<uint4 *>(prow + (((chunk ^ t) & 7) << 4)) =
                    make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
            }
        }
        tc::fence_async_smem();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ms.p_full);
        if (last) {
            // Refill the query buffer for the next unit (its QK^T may start
            // once this tile's P.V has been issued).
            if (next_unit) prep_query<NQ>(P, sm, M.nxt_r, M.nxt_flags >> 8);
            // ---- unit epilogue: row sums, o, lse
            {
                int cb = 0;
                colsum<H2, 16>(l, lane, cb);
                if ((lane & colsum_dup(H2)) == 0) {
#pragma unroll
                    for (int i = 0; i < colsum_count(H2); ++i) ms.red[wq][n0 + cb + i] = l[i];
                }
                if (lane == 0 && wq == 0) {
#pragma unroll
                    for (int j = 0; j < H2; ++j) ms.m[n0 + j] = mr[j];
                }
            }
            if (!unit_epilogue<NQ>(P, sm, M.k, M.n_r, n_units & 1)) return;
            tc::fence_before();
            ++n_units;
        }
    }
}

template <int NQ, bool CAUSAL, bool PAGED>
__global__ void __launch_bounds__(kThreads, 1)
    attend_tc_kernel(const __grid_constant__ CUtensorMap mlat, const __grid_constant__ CUtensorMap mrope,
                     const ParamsOf<CAUSAL> P) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Misc<NQ> &ms = misc<NQ>(sm);
    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) {
        for (int s = 0; s < Cfg<NQ>::STAGES; ++s) {
            mbar_init(&ms.kv_full[s], kProdWarps);
            // released by the softmax warps' read of the descriptor and the MMA warp
            mbar_init(&ms.kv_empty[s], kSoftWarps + 1);
        }
        mbar_init(&ms.s_full, 1);
        mbar_init(&ms.p_full, kSoftWarps);
        mbar_init(&ms.q_ready, kSoftWarps);
        mbar_init(&ms.o_done, 1);
        mbar_init(&ms.fin, 1);
        mbar_init(&ms.first_ready, 1);
        ms.abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == kMmaWarp) tc::tmem_alloc(&ms.tmem, Cfg<NQ>::TmemCols);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    // Every CTA is resident (one per SM): a kernel launched after this one
    // with programmatic dependent launch may start on SMs as they free up;
    // it waits for this grid's completion before reading its results.
    asm volatile("griddepcontrol.launch_dependents;");
    // Register split (per warpgroup; 512 x 128 at launch): the two softmax
    // warpgroups take 176 (184 for the causal mask's extra state at 48 rows),
    // the MMA / producer warpgroups the rest: 256 x 176 + 256 x 80 =
    // 256 x 184 + 256 x 72 = 65536.
    constexpr bool kWideSoft = CAUSAL && NQ == 48;
    constexpr int kSoftRegs = kWideSoft ? 184 : 176, kRoleRegs = kWideSoft ? 72 : 80;
    static_assert(2 * 128 * (kSoftRegs + kRoleRegs) == 65536, "register split must fill the launch's registers");
    if (warp < kSoftWarps) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftRegs));
        softmax<NQ, CAUSAL>(P, sm);
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRoleRegs));
        if (warp == kMmaWarp) mma_issuer<NQ>(P, sm);
        else producer<NQ, PAGED>(P, &mlat, &mrope, sm);
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

// The causal kernels' parameter layout (same fields, no padding).
ParamsCausal causal_params(const Params &P) {
    ParamsCausal C;
    C.q = P.q;
    C.q_row_stride = P.q_row_stride;
    C.pool_rows = P.pool_rows;
    C.pages = P.pages;
    C.num_pages = P.num_pages;
    C.indptr = P.indptr;
    C.R = P.R;
    C.qlen = P.qlen;
    C.heads = P.heads;
    C.num_splits = P.num_splits;
    C.split_tokens = P.split_tokens;
    C.row_groups = P.row_groups;
    C.log2p = P.log2p;
    C.q8 = P.q8;
    C.plan = P.plan;
    C.plan_len = P.plan_len;
    C.last_page_len = P.last_page_len;
    C.sc_log2 = P.sc_log2;
    C.kv_scale = P.kv_scale;
    C.o = P.o;
    C.lse = P.lse;
    return C;
}

template <int NQ, bool CAUSAL, bool PAGED>
cudaError_t launch_as(const CUtensorMap &ml, const CUtensorMap &mr, const Params &P, int grid, cudaStream_t st) {
    const size_t smem = smem_bytes<NQ>();
    cudaError_t e = smem_attr_once<attend_tc_kernel<NQ, CAUSAL, PAGED>>((int)smem);
    if (e != cudaSuccess) return e;
    if constexpr (CAUSAL)
        attend_tc_kernel<NQ, CAUSAL, PAGED><<<grid, kThreads, smem, st>>>(ml, mr, causal_params(P));
    else
        attend_tc_kernel<NQ, CAUSAL, PAGED><<<grid, kThreads, smem, st>>>(ml, mr, P);
    return cudaGetLastError();
}

template <int NQ>
cudaError_t launch(const CUtensorMap &ml, const CUtensorMap &mr, const Params &P, bool causal, int grid,
                   cudaStream_t st) {
    if (P.log2p > 0)
        return causal ? launch_as<NQ, true, true>(ml, mr, P, grid, st) : launch_as<NQ, false, true>(ml, mr, P, grid, st);
    return causal ? launch_as<NQ, true, false>(ml, mr, P, grid, st) : launch_as<NQ, false, false>(ml, mr, P, grid, st);
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
                             float *lse, bool causal, int log2p, const int32_t *last_page_len, bool q8,
                             const int32_t *plan, int64_t plan_len, int grid, cudaStream_t st) {
    // The two tensor maps over the KV pool, encoded once per (device, pool)
    // and reused while a thread keeps launching over the same pool.
    struct MapCache {
        int dev;
        const void *kv;
        int64_t pool_rows;
        CUtensorMap ml, mr;
    };
    static thread_local MapCache cache = {-1, nullptr, 0, {}, {}};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    if (cache.dev != dev || cache.kv != kv || cache.pool_rows != pool_rows) {
        PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
        if (!enc) return cudaErrorNotSupported;
        cuuint64_t gdim[2] = {(cuuint64_t)MLA_D_QK, (cuuint64_t)pool_rows};
        cuuint64_t gstr[1] = {(cuuint64_t)MLA_D_QK};
        cuuint32_t box_lat[2] = {128, 1}, box_rope[2] = {64, 1}, es[2] = {1, 1};
        void *base = const_cast<void *>(kv);
        cache.dev = -1;
        if (enc(&cache.ml, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, gdim, gstr, box_lat, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
            enc(&cache.mr, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, gdim, gstr, box_rope, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        cache.dev = dev;
        cache.kv = kv;
        cache.pool_rows = pool_rows;
    }
    const CUtensorMap &ml = cache.ml, &mr = cache.mr;
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
    P.log2p = log2p;
    P.q8 = q8 ? 1 : 0;
    P.plan = plan;
    P.plan_len = (int)plan_len;
    P.last_page_len = last_page_len;
    P.sc_log2 = scale * kv_scale * 1.4426950408889634f;
    P.kv_scale = kv_scale;
    P.o = static_cast<__nv_bfloat16 *>(o);
    P.lse = lse;
    int groups, nq;
    attend_tc_shape(qlen * heads, &groups, &nq);
    P.row_groups = groups;
    switch (nq) {
        case 16: return launch<16>(ml, mr, P, causal, grid, st);
        case 32: return launch<32>(ml, mr, P, causal, grid, st);
        default: return launch<48>(ml, mr, P, causal, grid, st);
    }
}

cudaError_t attend_tc_status(unsigned int *flags, bool clear) { return read_status(flags, clear); }

}  // namespace mla
