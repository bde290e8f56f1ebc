// Pieces shared by the warp-level tensor-core kernels (16-bit pools and FP8 pools):
// shared-memory row addressing, output row indexing, stores, and the two epilogues.
#pragma once

#include "kernels.h"

namespace pa {
namespace mmac {

template <int D>
struct Geo {
    static constexpr int NH = D / 64;                              // 128-byte halves of a row
    static constexpr int kStageBytes = kMmaTileKeys * D * 2;       // K (or V) bytes of one stage
    static constexpr int kChunks = D / 8;                          // 16-byte chunks per row
};

// Shared address of 16-byte chunk c of key row k (0..63) of a stage buffer.
// A stage holds 64 / page_size page boxes; a box is [NH halves][page_size][64]
// with the TMA 128-byte swizzle (chunk index XOR row % 8, row % 8 == k % 8).
template <int D>
__device__ __forceinline__ uint32_t kv_chunk_addr(uint32_t base, int k, int c, int ps_shift) {
    const int page = k >> ps_shift;
    const int t = k & ((1 << ps_shift) - 1);
    const int row = ((page * Geo<D>::NH + (c >> 3)) << ps_shift) + t;
    return base + (uint32_t)(row << 7) + (uint32_t)((((c & 7) ^ (k & 7))) << 4);
}

// The query tokens of one sequence: its first token in the packed [tokens, Hq, D] layout
// (b * Sq for a uniform batch) and its token count.
struct SeqRows {
    long long q0;
    int Sq;
};

__device__ __forceinline__ SeqRows uniform_seq(const FwdParams &p, int b) { return {(long long)b * p.Sq, p.Sq}; }

// Packed row (token x Hq + head) of unit row r (query token r / G, head kvh G + r % G).
__device__ __forceinline__ long long out_row_index(const FwdParams &p, const SeqRows &sq, int kvh, int r) {
    const int i = r / p.G;
    const int h = kvh * p.G + (r - i * p.G);
    return (sq.q0 + i) * p.Hq + h;
}

// Write two adjacent output columns of one row.
template <typename T>
__device__ __forceinline__ void store_pair(const FwdParams &p, int s, long long ridx, int col, float v0, float v1) {
    if (p.split_kv == 1) {
        T *o = reinterpret_cast<T *>(p.out) + ridx * p.D + col;
        o[0] = from_float<T>(v0);
        o[1] = from_float<T>(v1);
    } else {
        float2 *o = reinterpret_cast<float2 *>(reinterpret_cast<float *>(p.out) +
                                               ((long long)s * p.rows_total + ridx) * p.D + col);
        *o = make_float2(v0, v1);
    }
}

__device__ __forceinline__ void store_lse(const FwdParams &p, int s, long long ridx, float v) {
    if (p.split_kv == 1) {
        if (p.lse) p.lse[ridx] = v;
    } else {
        p.lse[(long long)s * p.rows_total + ridx] = v;
    }
}

// The producer warp of a unit over 16-bit pools: page ids 32 at a time (one per lane, never past
// the unit's pages), then per 64-key stage t one 4-D TMA box per page and pool (page_size tokens
// x one kv head x head_dim, 128-byte swizzled) into ring stage t % NSTAGE, armed on the stage's K
// and V full barriers once the consumers have released it (rocm-libraries PR #14349, Technical
// Details: page ids loaded once per tile).  An id outside [0, num_pages) is not dereferenced: its
// box starts before the tensor and reads as zeros, and PA_ERRBIT_PAGE_RANGE is set.
template <int D, int NSTAGE>
__device__ __forceinline__ void produce_pages16(const CUtensorMap *tmK, const CUtensorMap *tmV, const FwdParams &p,
                                                int b, int kvh, int pg0, int k_hi, int n_tiles, int ps_shift,
                                                uint32_t sbase, uint32_t bar_fk, uint32_t bar_fv, uint32_t bar_em,
                                                int lane) {
    constexpr int kStage = Geo<D>::kStageBytes;
    const int ps = 1 << ps_shift;
    if (lane == 0) {
        tma_prefetch_desc(tmK);
        tma_prefetch_desc(tmV);
    }
    const int pps = kMmaTileKeys >> ps_shift;                 // pages per stage (divides 32)
    const uint32_t box_bytes = (uint32_t)(Geo<D>::NH * ps * 128);
    const int pg_end = (k_hi + ps - 1) >> ps_shift;          // pages this unit reads
    const int32_t *bt_row = p.block_table + (long long)b * p.W;
    int batch = pg0;                                           // page held by lane 0 of id_cur
    int id_cur = (batch + lane < pg_end) ? __ldg(bt_row + batch + lane) : 0;
    int id_next = (batch + 32 + lane < pg_end) ? __ldg(bt_row + batch + 32 + lane) : 0;
    bool bad = false;
    int issued = 0;
    for (int t = 0; t < n_tiles; ++t) {
        const int st = t % NSTAGE;
        if (t >= NSTAGE && !bad) {
            const bool ok = mbar_wait(bar_em + 8 * st, ((t / NSTAGE) - 1) & 1, p.err);
            bad = __any_sync(0xffffffffu, !ok);
        }
        const int pg_first = pg0 + t * pps;
        if (pg_first >= batch + 32) {
            batch += 32;
            id_cur = id_next;
            const int nx = batch + 32 + lane;
            id_next = (nx < pg_end) ? __ldg(bt_row + nx) : 0;
        }
        const int my_pg = pg_first + lane;
        const int id = __shfl_sync(0xffffffffu, id_cur, (my_pg - batch) & 31);
        if (bad) break;
        const int nvalid = min(pps, pg_end - pg_first);
        if (lane == 0) {
            mbar_arrive_expect_tx(bar_fk + 8 * st, (uint32_t)nvalid * box_bytes);
            mbar_arrive_expect_tx(bar_fv + 8 * st, (uint32_t)nvalid * box_bytes);
        }
        __syncwarp();
        if (lane < nvalid) {
            int tok;
            if (id < 0 || (long long)id >= p.num_pages) {
                atomicOr(p.err, (unsigned int)PA_ERRBIT_PAGE_RANGE);
                tok = -ps;  // wholly out of the tensor: the box reads as zeros
            } else {
                tok = id << ps_shift;
            }
            const uint32_t off = (uint32_t)lane * box_bytes;
            const uint32_t kdst = sbase + (uint32_t)(st * 2 * kStage) + off;
            tma_load_4d(kdst, tmK, bar_fk + 8 * st, 0, tok, 0, kvh);
            tma_load_4d(kdst + kStage, tmV, bar_fv + 8 * st, 0, tok, 0, kvh);
        }
        issued = t + 1;
    }
    // Every copy must have landed before the CTA may exit: wait (bounded) for the
    // last phase of each stage that was armed.
    for (int t = max(0, issued - NSTAGE); t < issued; ++t) {
        const int st = t % NSTAGE;
        const uint32_t par = (t / NSTAGE) & 1;
        mbar_wait(bar_fk + 8 * st, par, p.err);
        mbar_wait(bar_fv + 8 * st, par, p.err);
    }
}

// Producer of a split group (MODE_SPLITS): split w of the group reads pages [pg0[w], pe[w]) in
// nt[w] 64-key tiles; the group's pages are consecutive from pg0[0] and at most 32, so one id per
// lane covers them.  Stages go out interleaved, round t holding tile t of every split that has
// one (in split order), and stage k lands in ring slot k % NSTAGE, so the four consumer warps
// work on their own splits at once.  Stage k completes on its own full barriers bar_fk / bar_fv
// + 8 k (used once); slot st frees on bar_em + 8 st, which only this warp waits on, in order.
template <int D, int NSTAGE>
__device__ __forceinline__ void produce_split_group(const CUtensorMap *tmK, const CUtensorMap *tmV,
                                                    const FwdParams &p, int b, int kvh,
                                                    const int (&pg0)[kMmaConsumerWarps],
                                                    const int (&pe)[kMmaConsumerWarps],
                                                    const int (&nt)[kMmaConsumerWarps], int ps_shift, uint32_t sbase,
                                                    uint32_t bar_fk, uint32_t bar_fv, uint32_t bar_em, int lane) {
    constexpr int kStage = Geo<D>::kStageBytes;
    constexpr int NW = kMmaConsumerWarps;
    const int ps = 1 << ps_shift;
    if (lane == 0) {
        tma_prefetch_desc(tmK);
        tma_prefetch_desc(tmV);
    }
    const int pps = kMmaTileKeys >> ps_shift;  // pages per stage
    const uint32_t box_bytes = (uint32_t)(Geo<D>::NH * ps * 128);
    // lane i: the id of page pg0[0] + i, loaded only when one of the splits reads that page
    const int my_page = pg0[0] + lane;
    bool read = false;
    int max_nt = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        read |= my_page >= pg0[w] && my_page < pe[w];
        max_nt = max(max_nt, nt[w]);
    }
    const int id_lane = read ? __ldg(p.block_table + (long long)b * p.W + my_page) : 0;
    bool bad = false;
    int k = 0;  // stages issued
    for (int t = 0; t < max_nt && !bad; ++t) {
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            if (t >= nt[w] || bad) continue;  // warp-uniform
            const int st = k % NSTAGE;
            if (k >= NSTAGE) {
                const bool ok = mbar_wait(bar_em + 8 * st, ((k / NSTAGE) - 1) & 1, p.err);
                bad = __any_sync(0xffffffffu, !ok);
                if (bad) break;
            }
            const int pg_first = pg0[w] + t * pps;
            const int nvalid = min(pps, pe[w] - pg_first);
            const int id = __shfl_sync(0xffffffffu, id_lane, (pg_first - pg0[0] + lane) & 31);
            if (lane == 0) {
                mbar_arrive_expect_tx(bar_fk + 8 * k, (uint32_t)nvalid * box_bytes);
                mbar_arrive_expect_tx(bar_fv + 8 * k, (uint32_t)nvalid * box_bytes);
            }
            __syncwarp();
            if (lane < nvalid) {
                int tok;
                if (id < 0 || (long long)id >= p.num_pages) {
                    atomicOr(p.err, (unsigned int)PA_ERRBIT_PAGE_RANGE);
                    tok = -ps;  // wholly out of the tensor: the box reads as zeros
                } else {
                    tok = id << ps_shift;
                }
                const uint32_t kdst = sbase + (uint32_t)(st * 2 * kStage) + (uint32_t)lane * box_bytes;
                tma_load_4d(kdst, tmK, bar_fk + 8 * k, 0, tok, 0, kvh);
                tma_load_4d(kdst + kStage, tmV, bar_fv + 8 * k, 0, tok, 0, kvh);
            }
            ++k;
        }
    }
    // Every copy must have landed before the CTA may exit: the last NSTAGE stages' barriers
    // (bounded waits; earlier stages were consumed before their slots were reused).
    for (int kk = max(0, k - NSTAGE); kk < k; ++kk) {
        mbar_wait(bar_fk + 8 * kk, 0, p.err);
        mbar_wait(bar_fv + 8 * kk, 0, p.err);
    }
}

// A unit with no valid key for any of its rows: output 0, lse -inf (every consumer thread, or
// with one_warp the 32 threads of one warp).
template <typename T, int D>
__device__ __forceinline__ void store_empty_unit(const FwdParams &p, const SeqRows &sq, int kvh, int s, int row0,
                                                 int row_end, bool one_warp = false) {
    const int nrows = row_end - row0;
    const int i0 = one_warp ? (int)(threadIdx.x & 31) : (int)threadIdx.x;
    const int stride = one_warp ? 32 : kMmaConsumerWarps * 32;
    for (int idx = i0; idx < nrows * (D / 2); idx += stride) {
        const int r = row0 + idx / (D / 2);
        const int col = (idx % (D / 2)) * 2;
        const long long ridx = out_row_index(p, sq, kvh, r);
        store_pair<T>(p, s, ridx, col, 0.f, 0.f);
        if (col == 0) store_lse(p, s, ridx, kNegInf);
    }
}

// Prefill epilogue: each warp owns rows ra / rb (fragment rows g, g + 8 of its m16 tile);
// l_a / l_b are already summed over the quad.  0/0 guard: a row with l == 0 stores 0, lse -inf.
template <typename T, int D>
__device__ __forceinline__ void finish_prefill_rows(const FwdParams &p, const SeqRows &sq, int kvh, int s, int ra, int rb,
                                                    int row_end, int tq, float m_a, float m_b, float l_a,
                                                    float l_b, const float (&acc)[D / 8][4]) {
    const float inv_a = l_a > 0.f ? 1.f / l_a : 0.f;
    const float inv_b = l_b > 0.f ? 1.f / l_b : 0.f;
    const bool va = ra < row_end, vb = rb < row_end;
    const long long ia = va ? out_row_index(p, sq, kvh, ra) : 0;
    const long long ib = vb ? out_row_index(p, sq, kvh, rb) : 0;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
        const int col = n * 8 + 2 * tq;
        if (va) store_pair<T>(p, s, ia, col, acc[n][0] * inv_a, acc[n][1] * inv_a);
        if (vb) store_pair<T>(p, s, ib, col, acc[n][2] * inv_b, acc[n][3] * inv_b);
    }
    if (tq == 0) {
        if (va) store_lse(p, s, ia, l_a > 0.f ? m_a * kLn2 + logf(l_a) : kNegInf);
        if (vb) store_lse(p, s, ib, l_b > 0.f ? m_b * kLn2 + logf(l_b) : kNegInf);
    }
}

// Decode epilogue: the four consumer warps hold softmax states (m, l, acc) of the same 16 rows
// over disjoint keys; merge them through shared memory `sm` (>= merge_scratch_bytes(D), 16-byte
// aligned, no longer read by anyone) and store.  Every consumer thread must call it.
__host__ __device__ constexpr size_t merge_scratch_bytes(int D) {
    return (size_t)kMmaConsumerWarps * 16 * (D + 4) * 4 + 2 * kMmaConsumerWarps * 16 * 4;
}

// Second half of the decode merge: shared memory `sm` holds, for each consumer warp w, rows
// [w][16][D + 4] of unnormalised outputs, then maxima [w][16] and sums [w][16] (log2 domain), for
// unit rows row0 .. row0 + 15.  Each row below row_end is combined over the warps (0/0 guard:
// l == 0 stores 0, lse -inf) and stored.
template <typename T, int D>
__device__ __forceinline__ void decode_merge_store(const FwdParams &p, const float *sm, const SeqRows &sq, int kvh,
                                                   int s, int row0, int row_end) {
    constexpr int ACC_STRIDE = D + 4;
    const float *s_acc = sm;
    const float *s_m = sm + kMmaConsumerWarps * 16 * ACC_STRIDE;
    const float *s_l = s_m + kMmaConsumerWarps * 16;
    const int tid = threadIdx.x;  // 0..127
    const int r = tid >> 3;       // 16 rows x 8 column groups
    const int cg = tid & 7;
    constexpr int COLS = D / 8;
    if (row0 + r < row_end) {
        float M = kNegInf;
#pragma unroll
        for (int w = 0; w < kMmaConsumerWarps; ++w) M = fmaxf(M, s_m[w * 16 + r]);
        float wsc[kMmaConsumerWarps];
        float Lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kMmaConsumerWarps; ++w) {
            wsc[w] = (M == kNegInf) ? 0.f : exp2f(s_m[w * 16 + r] - M);
            Lsum += wsc[w] * s_l[w * 16 + r];
        }
        const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
        const long long ridx = out_row_index(p, sq, kvh, row0 + r);
#pragma unroll
        for (int c = 0; c < COLS; c += 2) {
            const int col = cg * COLS + c;
            float o0 = 0.f, o1 = 0.f;
#pragma unroll
            for (int w = 0; w < kMmaConsumerWarps; ++w) {
                const float2 v = *reinterpret_cast<const float2 *>(s_acc + (w * 16 + r) * ACC_STRIDE + col);
                o0 += wsc[w] * v.x;
                o1 += wsc[w] * v.y;
            }
            store_pair<T>(p, s, ridx, col, o0 * inv, o1 * inv);
        }
        if (cg == 0) store_lse(p, s, ridx, Lsum > 0.f ? M * kLn2 + logf(Lsum) : kNegInf);
    }
}

template <typename T, int D>
__device__ __forceinline__ void decode_merge(const FwdParams &p, float *sm, const SeqRows &sq, int kvh, int s, int row_end,
                                             int warp, int lane, float m_a, float m_b, float l_a, float l_b,
                                             const float (&acc)[D / 8][4], bool bad) {
    constexpr int ACC_STRIDE = D + 4;
    const int g = lane >> 2;
    const int tq = lane & 3;
    float *s_acc = sm;                                            // [4][16][ACC_STRIDE]
    float *s_m = sm + kMmaConsumerWarps * 16 * ACC_STRIDE;        // [4][16]
    float *s_l = s_m + kMmaConsumerWarps * 16;                    // [4][16]
    named_bar_sync(1, kMmaConsumerWarps * 32);  // every warp is done reading the buffers below
    {
        float *wa = s_acc + (warp * 16) * ACC_STRIDE;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
            const int col = n * 8 + 2 * tq;
            *reinterpret_cast<float2 *>(wa + g * ACC_STRIDE + col) = make_float2(acc[n][0], acc[n][1]);
            *reinterpret_cast<float2 *>(wa + (g + 8) * ACC_STRIDE + col) = make_float2(acc[n][2], acc[n][3]);
        }
        if (tq == 0) {
            s_m[warp * 16 + g] = m_a;
            s_m[warp * 16 + g + 8] = m_b;
            s_l[warp * 16 + g] = l_a;
            s_l[warp * 16 + g + 8] = l_b;
        }
    }
    named_bar_sync(1, kMmaConsumerWarps * 32);
    if (!bad) decode_merge_store<T, D>(p, sm, sq, kvh, s, 0, row_end);
}

}  // namespace mmac
}  // namespace pa
