// Split-KV MLA decode attention over a paged fp8 latent cache -- warp-MMA
// kernel (mma.sync m16n8k16, f16 inputs, f32 accumulation).
//
// What it computes: vLLM API page
// vllm.models.kimi_k3.amd.specialized_decode.runtime.mla, m1c_inputs (the
// bf16 query [S, H, 576], the flat fp8 token rows addressed by pages /
// indptr, scale and kv_scale, partials o [splits, S, H, 512] bf16 and LSE
// [splits, S, H] f32) and attend (multi-query attention over one latent
// row per token; padded heads are skipped through the row stride).
//
// Design (one persistent CTA per SM, 8 consumer warps + 1 producer warp):
//   * Work units are (request, split) pairs, enumerated request-major and
//     dealt round-robin to CTAs.  The producer warp walks them with a warp
//     prefix scan over indptr (no scratch memory, no host round trip).
//   * For each tile of kTile tokens the producer warps issue one 576-byte
//     cp.async.bulk per KV row (one row per lane, rows spread over 4 warps)
//     into a smem stage (row stride 592 bytes, so both fragment load
//     patterns below are bank-conflict free), completing on the stage's
//     "full" mbarrier; consumers release it on "empty".
//   * The query rows of all heads x qlen of the request (MQA: they share
//     every KV row) form the MMA M dimension; a CTA takes up to 16*MT rows
//     (larger head counts use several row groups, which re-read the same KV
//     rows from L2).
//   * QK^T: warp w owns kTile/8 tokens.  The B fragment of K is one 32-bit
//     smem load of 4 fp8 codes, converted in registers (cvt e4m3x2->f16x2,
//     exact).  The 16-wide k-step is permuted (logical 2q,2q+1,2q+8,2q+9
//     <-> bytes 4q..4q+3) and the query is stored in smem in the same
//     permuted order, so ldmatrix delivers matching A fragments.
//   * Online softmax in the log2 domain; the per-tile row max is combined
//     across warps through smem; P goes to smem as f16.
//   * P.V: warp w owns latent columns [64w, 64w+64).  B fragments come from
//     4 fp8 rows (tokens 2q, 2q+1, 2q+8, 2q+9) with byte permutes; the
//     latent columns are permuted so each thread finally stores 8
//     consecutive outputs (16 bytes).
#include <cuda_runtime.h>

#include "common.cuh"

namespace mla {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
// Several producer warps: a warp issues its bulk copies one lane at a time,
// so spreading a tile's rows over 4 warps (one row per lane) is what lets
// random 576-byte rows stream at close to the HBM copy rate.
constexpr int kProducerWarps = 4;
constexpr int kThreads = kConsumers + kProducerWarps * 32;
constexpr int kRowStride = 592;  // smem bytes per KV row (576 + 16)
constexpr int kQStride = 584;    // f16 elements per query smem row (576 + 8)
constexpr int kStages = 2;

constexpr unsigned kFirst = kTileFirst, kLast = kTileLast, kDone = 4;

struct Meta {
    int r, k, n_r, tok0, ntok, flags;
};

template <int MT, int TILE>
struct Smem {
    static constexpr int kPStride = TILE + 8;  // f16 elements per P row
    uint8_t kv[kStages][TILE * kRowStride];
    __half q[16 * MT][kQStride];
    __half p[16 * MT][kPStride];
    float red[kConsumerWarps][16 * MT];
    Meta meta[kStages];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    int abort_flag;
};

struct Params {
    const __nv_bfloat16 *q;
    int64_t q_row_stride;
    const uint8_t *kv;
    int64_t pool_rows;
    const int32_t *pages;
    int64_t num_pages;
    const int32_t *indptr;
    int R, qlen, heads, num_splits, split_tokens, row_groups;
    float sc_log2;   // scale * kv_scale * log2(e)
    float kv_scale;
    __nv_bfloat16 *o;
    float *lse;
};

// ---------------------------------------------------------------- producer

template <int MT, int TILE>
__device__ void producer(const Params &P, Smem<MT, TILE> &sm) {
    constexpr int ROWS = TILE / kProducerWarps;   // rows of a tile this warp copies
    constexpr int PER_LANE = (ROWS + 31) / 32;
    const int lane = threadIdx.x & 31;
    const int pw = (threadIdx.x >> 5) - kConsumerWarps;
    TileIter<TILE> iter;   // every producer warp walks the same tile sequence
    iter.init(P.indptr, P.R, P.num_pages, P.num_splits, P.split_tokens, P.row_groups, lane);
    // Page indices of a tile are loaded one tile ahead, so their latency
    // hides behind the wait for a free stage.
    auto fetch_pages = [&](const Tile &T, int (&pg)[PER_LANE]) {
#pragma unroll
        for (int j = 0; j < PER_LANE; ++j) {
            const int i = pw * ROWS + lane + 32 * j;
            pg[j] = (T.valid && lane + 32 * j < ROWS && i < T.ntok) ? __ldg(P.pages + (int64_t)T.base + T.tok0 + i) : 0;
        }
    };
    Tile cur = iter.next(lane);
    int pg[PER_LANE];
    fetch_pages(cur, pg);
    int it = 0;
    while (cur.valid) {
        Tile nxt = iter.next(lane);
        int npg[PER_LANE];
        fetch_pages(nxt, npg);
        const int s = it % kStages;
        const uint32_t par = ((it / kStages) & 1) ^ 1;
        if (!mbar_wait(&sm.empty[s], par)) { sm.abort_flag = 1; return; }
        const int r0 = pw * ROWS;
        const int mine = max(0, min(ROWS, cur.ntok - r0));
        if (lane == 0) {
            if (pw == 0) {
                Meta m;
                m.r = cur.r; m.k = cur.k; m.n_r = cur.n_r; m.tok0 = cur.tok0; m.ntok = cur.ntok;
                m.flags = cur.flags;
                sm.meta[s] = m;
            }
            mbar_arrive_expect_tx(&sm.full[s], (uint32_t)mine * MLA_D_QK);
        }
        __syncwarp();
#pragma unroll
        for (int j = 0; j < PER_LANE; ++j) {
            const int i = lane + 32 * j;
            if (i < mine)
                bulk_g2s(&sm.kv[s][(r0 + i) * kRowStride], kv_row_of_page(P.kv, pg[j], P.pool_rows), MLA_D_QK,
                         &sm.full[s]);
        }
        ++it;
        cur = nxt;
#pragma unroll
        for (int j = 0; j < PER_LANE; ++j) pg[j] = npg[j];
    }
    // Tell the consumers there is no more work (every producer warp arrives).
    const int s = it % kStages;
    const uint32_t par = ((it / kStages) & 1) ^ 1;
    if (!mbar_wait(&sm.empty[s], par)) { sm.abort_flag = 1; return; }
    if (lane == 0) {
        if (pw == 0) sm.meta[s].flags = kDone;
        mbar_arrive(&sm.full[s]);
    }
}

// ---------------------------------------------------------------- consumers

// Query rows of request r, row group grp, into smem as f16 in the permuted
// k order (see the file comment).  Rows past the request's qlen*heads are 0.
template <int MT, int TILE>
__device__ void load_query(const Params &P, Smem<MT, TILE> &sm, int r, int grp) {
    const int tid = threadIdx.x;
    const int rows_total = P.qlen * P.heads;
    for (int c = tid; c < 16 * MT * 72; c += kConsumers) {
        const int row = c / 72, ch = c % 72;
        const int rho = grp * 16 * MT + row;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (rho < rows_total) {
            const int tq = rho / P.heads, h = rho % P.heads;
            const int64_t off = ((int64_t)r * P.qlen + tq) * P.q_row_stride + (int64_t)h * MLA_D_QK + ch * 8;
            v = __ldg(reinterpret_cast<const uint4 *>(P.q + off));
        }
        // bf16 pairs -> f16 pairs
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = pack_f16x2(bf16_lo(w[e]), bf16_hi(w[e]));
        // physical elements (0,1,4,5) -> logical 4c'..4c'+3, (2,3,6,7) -> 4c'+8..4c'+11
        const int blk16 = ch >> 1, half = ch & 1;
        __half *dst = &sm.q[row][blk16 * 16 + 4 * half];
        *reinterpret_cast<uint2 *>(dst) = make_uint2(w[0], w[2]);
        *reinterpret_cast<uint2 *>(dst + 8) = make_uint2(w[1], w[3]);
    }
}

template <int MT, int TILE>
__device__ void consumers(const Params &P, Smem<MT, TILE> &sm) {
    constexpr int NT = TILE / 64;   // QK n-tiles (8 tokens) per warp
    constexpr int TPW = TILE / 8;   // tokens per warp in QK
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, qd = lane & 3;
    const int S = P.R * P.qlen;
    const int rows_total = P.qlen * P.heads;

    float m_run[MT][2], l_run[MT][2];
    float acc[MT][8][4];

    for (int it = 0;; ++it) {
        const int s = it % kStages;
        const uint32_t par = (it / kStages) & 1;
        if (!mbar_wait(&sm.full[s], par)) { sm.abort_flag = 1; return; }
        if (sm.abort_flag) return;
        const Meta meta = sm.meta[s];
        if (meta.flags & kDone) return;
        const int grp = meta.flags >> 8;
        const int ntok = meta.ntok;
        const uint8_t *kvs = sm.kv[s];

        if (meta.flags & kFirst) {
            named_sync(1, kConsumers);           // previous unit done with q
            load_query(P, sm, meta.r, grp);
#pragma unroll
            for (int i = 0; i < MT; ++i) {
                m_run[i][0] = m_run[i][1] = -INFINITY;
                l_run[i][0] = l_run[i][1] = 0.f;
#pragma unroll
                for (int n = 0; n < 8; ++n)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[i][n][e] = 0.f;
            }
            named_sync(1, kConsumers);
        }

        if (ntok > 0) {
            // ---------------- S = Q K^T for this warp's tokens
            float sacc[MT][NT][4];
#pragma unroll
            for (int i = 0; i < MT; ++i)
#pragma unroll
                for (int j = 0; j < NT; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sacc[i][j][e] = 0.f;
            const int tokw = warp * TPW;
            const uint8_t *krow[NT];
#pragma unroll
            for (int j = 0; j < NT; ++j) krow[j] = kvs + (tokw + 8 * j + g) * kRowStride + 4 * qd;
            const int lrow = lane & 15, lcol = (lane >> 4) * 8;
#pragma unroll 4
            for (int ks = 0; ks < MLA_D_QK / 16; ++ks) {
                uint32_t bfr[NT][2];
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const uint32_t w = *reinterpret_cast<const uint32_t *>(krow[j] + ks * 16);
                    bfr[j][0] = e4m3x2_to_f16x2((uint16_t)(w & 0xffff));
                    bfr[j][1] = e4m3x2_to_f16x2((uint16_t)(w >> 16));
                }
#pragma unroll
                for (int i = 0; i < MT; ++i) {
                    uint32_t a[4];
                    ldmatrix_x4(a, &sm.q[16 * i + lrow][ks * 16 + lcol]);
#pragma unroll
                    for (int j = 0; j < NT; ++j) mma_f16(sacc[i][j], a, bfr[j][0], bfr[j][1]);
                }
            }
            // ---------------- tile row max across warps
#pragma unroll
            for (int i = 0; i < MT; ++i) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float mx = -INFINITY;
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int tok = tokw + 8 * j + 2 * qd + e;
                            float v = sacc[i][j][2 * hh + e] * P.sc_log2;
                            v = tok < ntok ? v : -INFINITY;
                            sacc[i][j][2 * hh + e] = v;
                            mx = fmaxf(mx, v);
                        }
                    }
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                    if (qd == 0) sm.red[warp][16 * i + 8 * hh + g] = mx;
                }
            }
            named_sync(1, kConsumers);
            float alpha[MT][2];
#pragma unroll
            for (int i = 0; i < MT; ++i) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float mx = m_run[i][hh];
#pragma unroll
                    for (int w2 = 0; w2 < kConsumerWarps; ++w2) mx = fmaxf(mx, sm.red[w2][16 * i + 8 * hh + g]);
                    alpha[i][hh] = exp2f(m_run[i][hh] - mx);   // m_run = -inf -> 0
                    m_run[i][hh] = mx;
                    // p = 2^(s - m), rounded to f16; the row sum uses the rounded values
                    float sum = 0.f;
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        const float p0 = exp2f(sacc[i][j][2 * hh] - mx);
                        const float p1 = exp2f(sacc[i][j][2 * hh + 1] - mx);
                        const uint32_t ph = pack_f16x2(p0, p1);
                        const float2 pr = unpack_f16x2(ph);
                        sum += pr.x + pr.y;
                        *reinterpret_cast<uint32_t *>(&sm.p[16 * i + 8 * hh + g][tokw + 8 * j + 2 * qd]) = ph;
                    }
                    l_run[i][hh] = l_run[i][hh] * alpha[i][hh] + sum;
                }
            }
            named_sync(1, kConsumers);

            // ---------------- O = O*alpha + P V over this warp's latent slice
#pragma unroll
            for (int i = 0; i < MT; ++i)
#pragma unroll
                for (int n = 0; n < 8; ++n) {
                    acc[i][n][0] *= alpha[i][0];
                    acc[i][n][1] *= alpha[i][0];
                    acc[i][n][2] *= alpha[i][1];
                    acc[i][n][3] *= alpha[i][1];
                }
            const int ksteps = (ntok + 15) >> 4;
            const uint8_t *vbase = kvs + warp * 64 + 4 * g;
            for (int kk = 0; kk < ksteps; ++kk) {
                const int t0 = 16 * kk + 2 * qd;
                const int rows4[4] = {t0, t0 + 1, t0 + 8, t0 + 9};
                uint32_t bfr[8][2];
#pragma unroll
                for (int blk = 0; blk < 2; ++blk) {
                    uint32_t x[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint32_t w = *reinterpret_cast<const uint32_t *>(vbase + rows4[e] * kRowStride + 32 * blk);
                        x[e] = rows4[e] < ntok ? w : 0u;
                    }
                    // bytes j of (token 2q, token 2q+1) -> b0b1 of n-tile j; (2q+8, 2q+9) -> b2b3
                    const uint32_t lo01 = prmt(x[0], x[1], 0x5140), hi01 = prmt(x[0], x[1], 0x7362);
                    const uint32_t lo89 = prmt(x[2], x[3], 0x5140), hi89 = prmt(x[2], x[3], 0x7362);
                    bfr[4 * blk + 0][0] = e4m3x2_to_f16x2((uint16_t)(lo01 & 0xffff));
                    bfr[4 * blk + 1][0] = e4m3x2_to_f16x2((uint16_t)(lo01 >> 16));
                    bfr[4 * blk + 2][0] = e4m3x2_to_f16x2((uint16_t)(hi01 & 0xffff));
                    bfr[4 * blk + 3][0] = e4m3x2_to_f16x2((uint16_t)(hi01 >> 16));
                    bfr[4 * blk + 0][1] = e4m3x2_to_f16x2((uint16_t)(lo89 & 0xffff));
                    bfr[4 * blk + 1][1] = e4m3x2_to_f16x2((uint16_t)(lo89 >> 16));
                    bfr[4 * blk + 2][1] = e4m3x2_to_f16x2((uint16_t)(hi89 & 0xffff));
                    bfr[4 * blk + 3][1] = e4m3x2_to_f16x2((uint16_t)(hi89 >> 16));
                }
#pragma unroll
                for (int i = 0; i < MT; ++i) {
                    uint32_t a[4];
                    ldmatrix_x4(a, &sm.p[16 * i + (lane & 15)][16 * kk + (lane >> 4) * 8]);
#pragma unroll
                    for (int n = 0; n < 8; ++n) mma_f16(acc[i][n], a, bfr[n][0], bfr[n][1]);
                }
            }
        }
        // Release the stage.
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[s]);

        if (meta.flags & kLast) {
            // ---------------- finalize: row sums across warps, write o and lse
            float lsum[MT][2];
#pragma unroll
            for (int i = 0; i < MT; ++i)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float v = l_run[i][hh];
                    v += __shfl_xor_sync(0xffffffffu, v, 1);
                    v += __shfl_xor_sync(0xffffffffu, v, 2);
                    lsum[i][hh] = v;
                }
            named_sync(1, kConsumers);   // everyone done reading red / p
            if (qd == 0) {
#pragma unroll
                for (int i = 0; i < MT; ++i)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) sm.red[warp][16 * i + 8 * hh + g] = lsum[i][hh];
            }
            named_sync(1, kConsumers);
#pragma unroll
            for (int i = 0; i < MT; ++i) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int rl = 16 * i + 8 * hh + g;
                    float l = 0.f;
#pragma unroll
                    for (int w2 = 0; w2 < kConsumerWarps; ++w2) l += sm.red[w2][rl];
                    const int rho = grp * 16 * MT + rl;
                    if (rho >= rows_total) continue;
                    const int tq = rho / P.heads, h = rho % P.heads;
                    const int64_t t = (int64_t)meta.r * P.qlen + tq;
                    const int64_t orow = ((int64_t)meta.k * S + t) * P.heads + h;
                    const bool empty = ntok == 0;  // only an empty request has a 0-token last tile
                    if (!empty) {
                        const float inv = P.kv_scale / l;
#pragma unroll
                        for (int blk = 0; blk < 2; ++blk) {
                            uint4 pk;
                            float v[8];
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                v[j] = acc[i][4 * blk + j][2 * hh] * inv;
                                v[4 + j] = acc[i][4 * blk + j][2 * hh + 1] * inv;
                            }
                            pk.x = pack_bf16x2(v[0], v[1]);
                            pk.y = pack_bf16x2(v[2], v[3]);
                            pk.z = pack_bf16x2(v[4], v[5]);
                            pk.w = pack_bf16x2(v[6], v[7]);
                            *reinterpret_cast<uint4 *>(P.o + orow * MLA_D_LATENT + warp * 64 + 32 * blk + 8 * qd) = pk;
                        }
                    }
                    if (warp == 0 && qd == 0) {
                        // natural-log LSE of the scaled scores: (m + log2 l) * ln 2
                        P.lse[orow] = empty ? -INFINITY : (m_run[i][hh] + __log2f(l)) * 0.69314718055994531f;
                        for (int k2 = meta.k + 1; k2 < P.num_splits && meta.k == meta.n_r - 1; ++k2)
                            P.lse[((int64_t)k2 * S + t) * P.heads + h] = -INFINITY;
                    }
                }
            }
        }
    }
}

template <int MT, int TILE>
__global__ void __launch_bounds__(kThreads, 1) attend_mma_kernel(const Params P) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    auto &sm = *reinterpret_cast<Smem<MT, TILE> *>(smem_raw);
    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], kProducerWarps);
            mbar_init(&sm.empty[s], kConsumerWarps);
        }
        sm.abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    if (tid >= kConsumers) {
        producer<MT, TILE>(P, sm);
    } else {
        consumers<MT, TILE>(P, sm);
    }
}

template <int MT, int TILE>
cudaError_t launch(const Params &P, int sms, cudaStream_t st) {
    const size_t smem = sizeof(Smem<MT, TILE>);
    cudaError_t e = smem_attr_once<attend_mma_kernel<MT, TILE>>((int)smem);
    if (e != cudaSuccess) return e;
    attend_mma_kernel<MT, TILE><<<sms, kThreads, smem, st>>>(P);
    return cudaGetLastError();
}

}  // namespace

cudaError_t attend_mma_launch(const void *q, int64_t q_row_stride, const void *kv, int64_t pool_rows,
                              const int32_t *pages, int64_t num_pages, const int32_t *indptr, int R,
                              int qlen, int heads, float scale, float kv_scale, int num_splits,
                              int split_tokens, void *o, float *lse, int grid, cudaStream_t st) {
    Params P;
    P.q = static_cast<const __nv_bfloat16 *>(q);
    P.q_row_stride = q_row_stride;
    P.kv = static_cast<const uint8_t *>(kv);
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
    // Query rows per CTA: at most 64 (four m16 tiles); more rows use several
    // row groups, sized to waste the fewest padded rows.
    const int rows = qlen * heads;
    const int groups = (rows + 63) / 64;
    const int mt = (rows + 16 * groups - 1) / (16 * groups);
    P.row_groups = groups;
    switch (mt) {
        case 1: return launch<1, 128>(P, grid, st);
        case 2: return launch<2, 128>(P, grid, st);
        case 3: return launch<3, 64>(P, grid, st);
        default: return launch<4, 64>(P, grid, st);
    }
}

cudaError_t attend_mma_status(unsigned int *flags, bool clear) { return read_status(flags, clear); }

}  // namespace mla
