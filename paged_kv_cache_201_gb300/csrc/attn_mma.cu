// Tensor-core paged attention for sm_103a (bf16 / f16, head_dim 64 or 128).
//
// One CTA = one (sequence b, kv head, split s[, query-row tile]) unit:
//   * warp 4 (producer) walks the unit's pages.  It loads the block-table ids
//     of 32 pages at a time (one id per lane, guarded by the sequence's page
//     count, never past it) and turns each id into a TMA coordinate; the TMA
//     unit forms the 64-bit address, so pools past 2^31 bytes need no special
//     path.  Each page of each pool is one 4-D TMA box (page_size tokens x one
//     kv head x head_dim) landing 128-byte-swizzled in a NSTAGE-deep ring of
//     64-key stages (rocm-libraries PR #14349, Technical Details: page ids
//     loaded once per tile, no per-copy reload).
//   * warps 0-3 (consumers) compute S = Q K^T and O += P V with
//     mma.m16n8k16 (fp32 accumulate).  Decode mode: the 16 rows are the GQA
//     group (x query tokens) and the 4 warps split each stage's 64 keys, then
//     merge their softmax states once at the end.  Prefill mode: each warp owns
//     16 query rows and reads all 64 keys of the stage.  Split-group mode
//     (decode with short splits): the CTA takes 4 consecutive splits, each warp
//     owns one of them (the same 16 rows, all 64 keys of each of its stages) and
//     stores its own partial, so short splits need neither a key split nor a
//     merge, and a quarter as many CTAs.
//   * online softmax in the log2 domain with the rocMLIR PR #2371 guards: a
//     running max of -inf is replaced by 0 before exp2 (so -inf - (-inf)
//     never appears), and a row whose sum is 0 stores 0 / lse -inf.
// The unit body is one device function; the uniform kernel gives it the units
// of a batch with one query count, and the variable-length kernel (below) the
// decode units and 64-row tiles of a batch whose sequences differ in it.
#include "mma_common.cuh"

namespace pa {

using namespace mmac;

// One unit: sequence b, whose query tokens are `sq` (rows = sq.Sq x G query rows), kv head kvh,
// split s (in split-group mode the group: splits 4 s .. 4 s + 3) and, in prefill mode, 64-row
// query tile rt.  Every thread of the CTA calls it.
template <typename T, int D, int MODE, int NSTAGE>
__device__ __forceinline__ void mma_unit(const CUtensorMap *tmK, const CUtensorMap *tmV, const FwdParams &p, int b,
                                         const SeqRows &sq, int rows, int kvh, int s, int rt, int ps_shift,
                                         uint8_t *smem_raw, uint64_t *bars) {
    using Op = MmaOp<T>;
    constexpr int kStage = Geo<D>::kStageBytes;
    constexpr int kChunks = Geo<D>::kChunks;
    constexpr int NW = kMmaConsumerWarps;
    constexpr bool GROUP = MODE == MODE_SPLITS;
    constexpr int KB = (MODE == MODE_PREFILL) ? 32 : 16;  // keys per softmax block
    constexpr int SUBS = (MODE == MODE_DECODE) ? 1 : kMmaTileKeys / KB;  // blocks a warp handles per stage
    constexpr int NTB = KB / 8;                           // score n-tiles per block
    constexpr int CTA_ROWS = (MODE == MODE_PREFILL) ? kPrefillRows : kDecodeRows;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int ps = 1 << ps_shift;

    int L = max(p.seq_lens[b], 0);
    if (L > p.W * ps) {  // never read past the sequence's block-table row
        if (threadIdx.x == 0) atomicOr(p.err, (unsigned int)PA_ERRBIT_SEQ_CLIPPED);
        L = p.W * ps;
    }
    const int row0 = rt * CTA_ROWS;
    const int row_end = min(row0 + CTA_ROWS, rows);
    // causal reach grows with the query index, so the CTA's last row reaches furthest
    const int reach = row_key_limit(p, b, L, (row_end - 1) / p.G, sq.Sq);
    int pg0, pg1;
    int k_lo, k_hi_split, k_hi, n_tiles;
    // split-group mode: every thread knows the four splits' pages and tiles, and warp w takes
    // split 4 s + w (a split past the last has no pages)
    int gpg0[NW], gpe[NW], gnt[NW];
    int my_s = s;
    if constexpr (GROUP) {
        const int nblk = (L + ps - 1) >> ps_shift;
        int any = 0;
        n_tiles = 0;
        k_lo = k_hi_split = k_hi = 0;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const int sw = s * NW + w;
            int a = nblk, e = nblk;
            if (sw < p.split_kv) split_pages(L, ps, p.split_kv, sw, a, e);
            const int kl = a * ps, khs = min(e * ps, L), kh = min(khs, reach);
            gpg0[w] = a;
            gnt[w] = kh > kl ? (kh - kl + kMmaTileKeys - 1) / kMmaTileKeys : 0;
            gpe[w] = gnt[w] > 0 ? (kh + ps - 1) >> ps_shift : a;
            any += gnt[w];
            if (w == warp) {
                my_s = sw;
                k_lo = kl;
                k_hi_split = khs;
                k_hi = kh;
                n_tiles = gnt[w];
            }
        }
        if (any == 0) {
            // no valid key for any row of the group's splits: output 0, lse -inf
            if (warp < NW && my_s < p.split_kv) store_empty_unit<T, D>(p, sq, kvh, my_s, row0, row_end, true);
            return;
        }
    } else {
        split_pages(L, ps, p.split_kv, s, pg0, pg1);
        k_lo = pg0 * ps;
        k_hi_split = min(pg1 * ps, L);
        k_hi = min(k_hi_split, reach);
        n_tiles = k_hi > k_lo ? (k_hi - k_lo + kMmaTileKeys - 1) / kMmaTileKeys : 0;
        if (n_tiles == 0) {
            // no valid key for any row of this unit: output 0, lse -inf
            if (warp < NW) store_empty_unit<T, D>(p, sq, kvh, s, row0, row_end);
            return;
        }
    }

    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    // full barriers: one per ring slot, or in split-group mode one per stage (kGroupMaxStages)
    constexpr int NFULL = GROUP ? kGroupMaxStages : NSTAGE;
    const uint32_t bar_fk = smem_u32(&bars[0]);
    const uint32_t bar_fv = smem_u32(&bars[NFULL]);
    const uint32_t bar_em = smem_u32(&bars[2 * NFULL]);

    if (threadIdx.x == 0) {
        for (int i = 0; i < NFULL; ++i) {
            mbar_init(bar_fk + 8 * i, 1);
            mbar_init(bar_fv + 8 * i, 1);
        }
        for (int st = 0; st < NSTAGE; ++st) mbar_init(bar_em + 8 * st, GROUP ? 1 : NW);  // a group's stage: one warp
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == NW) {
        if constexpr (GROUP)
            produce_split_group<D, NSTAGE>(tmK, tmV, p, b, kvh, gpg0, gpe, gnt, ps_shift, sbase, bar_fk, bar_fv, bar_em,
                                           lane);
        else
            produce_pages16<D, NSTAGE>(tmK, tmV, p, b, kvh, pg0, k_hi, n_tiles, ps_shift, sbase, bar_fk, bar_fv,
                                       bar_em, lane);
        return;
    }
    if constexpr (GROUP) {
        if (my_s >= p.split_kv) return;  // no fourth (or third ...) split in the last group
        if (n_tiles == 0) {              // this warp's split has no valid key: output 0, lse -inf
            store_empty_unit<T, D>(p, sq, kvh, my_s, row0, row_end, true);
            return;
        }
    }

    // ==================================================================== consumers
    const int g = lane >> 2;
    const int tq = lane & 3;
    const int rbase = (MODE == MODE_PREFILL) ? row0 + warp * 16 : 0;
    const int ra = rbase + g, rb = rbase + g + 8;
    const int kw0 = (MODE == MODE_DECODE) ? warp * 16 : 0;  // first key (in the stage) of this warp
    // split-group mode: this warp's tile t is stage (tiles of earlier rounds, all splits) + (tile t
    // of earlier splits), the producer's interleaved order
    auto stage_of = [&](int t) {
        int k = 0;
        if constexpr (GROUP) {
#pragma unroll
            for (int w = 0; w < NW; ++w) k += min(t, gnt[w]) + ((w < warp && gnt[w] > t) ? 1 : 0);
        } else {
            k = t;
        }
        return k;
    };

    // Q fragments (A operand, row-major 16 x D): rows ra / rb, zero beyond the unit's rows
    uint32_t qf[D / 16][4];
    {
        const T *q = reinterpret_cast<const T *>(p.q);
        const bool va = ra < rows, vb = rb < rows;
        const T *qa = q + (va ? q_row_offset(p, out_row_index(p, sq, kvh, ra)) : 0);
        const T *qb = q + (vb ? q_row_offset(p, out_row_index(p, sq, kvh, rb)) : 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const int c0 = kk * 16 + 2 * tq;
            qf[kk][0] = va ? __ldg(reinterpret_cast<const uint32_t *>(qa + c0)) : 0u;
            qf[kk][1] = vb ? __ldg(reinterpret_cast<const uint32_t *>(qb + c0)) : 0u;
            qf[kk][2] = va ? __ldg(reinterpret_cast<const uint32_t *>(qa + c0 + 8)) : 0u;
            qf[kk][3] = vb ? __ldg(reinterpret_cast<const uint32_t *>(qb + c0 + 8)) : 0u;
        }
    }
    // exclusive key bounds of the two rows (pad rows see nothing)
    const int lim_a = ra < rows ? min(k_hi_split, row_key_limit(p, b, L, ra / p.G, sq.Sq)) : k_lo;
    const int lim_b = rb < rows ? min(k_hi_split, row_key_limit(p, b, L, rb / p.G, sq.Sq)) : k_lo;

    float m_a = kNegInf, m_b = kNegInf, l_a = 0.f, l_b = 0.f;
    float acc[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;

    // Keys at or past the furthest limit of this warp's rows are masked for all of them.
    const int warp_lim = __reduce_max_sync(0xffffffffu, (unsigned)max(lim_a, lim_b));

    bool bad = false;
    for (int t = 0; t < n_tiles; ++t) {
        const int kst = stage_of(t);
        const int st = kst % NSTAGE;
        const uint32_t par = GROUP ? 0u : (uint32_t)(kst / NSTAGE) & 1;  // group: the stage's own barriers
        const uint32_t bk = GROUP ? (uint32_t)kst : (uint32_t)st;            // full-barrier index
        const uint32_t kbuf = sbase + (uint32_t)(st * 2 * kStage);
        const uint32_t vbuf = kbuf + kStage;
        const int tile_k0 = k_lo + t * kMmaTileKeys;

        if (!bad) {
            const bool ok = mbar_wait(bar_fk + 8 * bk, par, p.err);
            bad = __any_sync(0xffffffffu, !ok);
        }
#pragma unroll
        for (int sb = 0; sb < SUBS; ++sb) {
            const int kb0 = kw0 + sb * KB;                              // first key (in the stage) of the block
            const bool active = tile_k0 + kb0 < min(k_hi, warp_lim);    // warp-uniform
            // P split into a bf16/f16 high part and the rounding remainder: P V = Ph V + Pl V keeps
            // the weights to ~2^-17 relative instead of the 2^-9 of a single 16-bit P.
            uint32_t ph[NTB][2], pl[NTB][2];
            if (!bad && active) {
                float sc[NTB][4];
#pragma unroll
                for (int n = 0; n < NTB; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
                // ---- S = Q K^T over the block's KB keys
                const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
                for (int np = 0; np < NTB / 2; ++np) {
                    const int key = kb0 + np * 16 + rr + ((mi >> 1) << 3);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        uint32_t b0, b1, b2, b3;
                        ldmatrix_x4(kv_chunk_addr<D>(kbuf, key, 2 * kk + (mi & 1), ps_shift), b0, b1, b2, b3);
                        Op::run(sc[2 * np], qf[kk], b0, b1);
                        Op::run(sc[2 * np + 1], qf[kk], b2, b3);
                    }
                }
                // ---- mask + scale (log2 domain)
                float mx_a = kNegInf, mx_b = kNegInf;
#pragma unroll
                for (int n = 0; n < NTB; ++n) {
                    const int j = tile_k0 + kb0 + n * 8 + 2 * tq;
                    sc[n][0] = (j < lim_a) ? sc[n][0] * p.scale_log2 : kNegInf;
                    sc[n][1] = (j + 1 < lim_a) ? sc[n][1] * p.scale_log2 : kNegInf;
                    sc[n][2] = (j < lim_b) ? sc[n][2] * p.scale_log2 : kNegInf;
                    sc[n][3] = (j + 1 < lim_b) ? sc[n][3] * p.scale_log2 : kNegInf;
                    mx_a = fmaxf(mx_a, fmaxf(sc[n][0], sc[n][1]));
                    mx_b = fmaxf(mx_b, fmaxf(sc[n][2], sc[n][3]));
                }
                mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
                mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
                mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
                mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
                const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
                // -inf - (-inf) guard: an all-masked row keeps max -inf and uses 0 as its offset
                const float mu_a = (mn_a == kNegInf) ? 0.f : mn_a;
                const float mu_b = (mn_b == kNegInf) ? 0.f : mn_b;
                const float al_a = exp2f(m_a - mu_a), al_b = exp2f(m_b - mu_b);
                m_a = mn_a;
                m_b = mn_b;
                float rs_a = 0.f, rs_b = 0.f;
#pragma unroll
                for (int n = 0; n < NTB; ++n) {
                    const float p0 = exp2f(sc[n][0] - mu_a), p1 = exp2f(sc[n][1] - mu_a);
                    const float p2 = exp2f(sc[n][2] - mu_b), p3 = exp2f(sc[n][3] - mu_b);
                    ph[n][0] = Op::pack(p0, p1);
                    ph[n][1] = Op::pack(p2, p3);
                    const float2 ha = Op::unpack(ph[n][0]), hb = Op::unpack(ph[n][1]);
                    pl[n][0] = Op::pack(p0 - ha.x, p1 - ha.y);
                    pl[n][1] = Op::pack(p2 - hb.x, p3 - hb.y);
                    rs_a += p0 + p1;
                    rs_b += p2 + p3;
                }
                l_a = l_a * al_a + rs_a;
                l_b = l_b * al_b + rs_b;
#pragma unroll
                for (int n = 0; n < D / 8; ++n) {
                    acc[n][0] *= al_a;
                    acc[n][1] *= al_a;
                    acc[n][2] *= al_b;
                    acc[n][3] *= al_b;
                }
            }

            if (sb == 0) {
                if (!bad) {
                    const bool ok = mbar_wait(bar_fv + 8 * bk, par, p.err);
                    bad = __any_sync(0xffffffffu, !ok);
                }
                if (tile_k0 + kMmaTileKeys > k_hi) {
                    // Last stage: keys at or past k_hi (past the sequence, or pages never loaded)
                    // may hold any bits.  Their weight is 0, but 0 * NaN is NaN, so zero those V rows
                    // (the warp's own 16 keys; a split-group warp owns all 64 of the stage).
                    const int kz0 = (MODE == MODE_DECODE) ? kw0 : (GROUP ? 0 : warp * 16);
                    for (int idx = lane; idx < (GROUP ? 64 : 16) * kChunks; idx += 32) {
                        const int key = kz0 + idx / kChunks;
                        if (tile_k0 + key >= k_hi) {
                            const uint32_t a = kv_chunk_addr<D>(vbuf, key, idx % kChunks, ps_shift);
                            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
                        }
                    }
                    fence_proxy_async_smem();
                    if (MODE != MODE_PREFILL)
                        __syncwarp();
                    else
                        named_bar_sync(1, kMmaConsumerWarps * 32);
                }
            }
            if (!bad && active) {
                // ---- O += (Ph + Pl) V  (P from the score fragments, V via transposed ldmatrix)
                const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
                for (int ks = 0; ks < KB / 16; ++ks) {
                    const uint32_t ah[4] = {ph[2 * ks][0], ph[2 * ks][1], ph[2 * ks + 1][0], ph[2 * ks + 1][1]};
                    const uint32_t al[4] = {pl[2 * ks][0], pl[2 * ks][1], pl[2 * ks + 1][0], pl[2 * ks + 1][1]};
                    const int key = kb0 + ks * 16 + rr + ((mi & 1) << 3);
#pragma unroll
                    for (int j = 0; j < D / 16; ++j) {
                        uint32_t b0, b1, b2, b3;
                        ldmatrix_x4_trans(kv_chunk_addr<D>(vbuf, key, 2 * j + (mi >> 1), ps_shift), b0, b1, b2,
                                          b3);
                        Op::run(acc[2 * j], ah, b0, b1);
                        Op::run(acc[2 * j + 1], ah, b2, b3);
                        Op::run(acc[2 * j], al, b0, b1);
                        Op::run(acc[2 * j + 1], al, b2, b3);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_em + 8 * st);
    }

    // quad sums of the row sums (alpha is uniform across a quad)
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);

    if (MODE != MODE_DECODE) {
        // each warp owns its rows (prefill) or its split (split group): finalise and store
        if (!bad) finish_prefill_rows<T, D>(p, sq, kvh, my_s, ra, rb, row_end, tq, m_a, m_b, l_a, l_b, acc);
        return;
    }
    // decode: merge the four warps' (m, l, acc) through shared memory (reuses the ring)
    decode_merge<T, D>(p, reinterpret_cast<float *>(smem_raw + (sbase - raw)), sq, kvh, s, row_end, warp, lane, m_a,
                       m_b, l_a, l_b, acc, bad);
}


template <typename T, int D, int MODE, int NSTAGE>
__global__ void __launch_bounds__(kMmaThreads, (NSTAGE <= 3 ? 2 : 1))
    paged_attn_mma_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                          const FwdParams p, int ps_shift) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[MODE == MODE_SPLITS ? 2 * kGroupMaxStages + NSTAGE : 3 * NSTAGE];
    int unit = blockIdx.x;
    int rt = 0;
    if (MODE == MODE_PREFILL) {
        rt = unit % p.row_tiles;
        unit /= p.row_tiles;
    }
    const int kvh = unit % p.Hkv;
    unit /= p.Hkv;
    // split-group mode: s indexes groups of kMmaConsumerWarps splits
    const int ns = MODE == MODE_SPLITS ? (p.split_kv + kMmaConsumerWarps - 1) / kMmaConsumerWarps : p.split_kv;
    const int s = unit % ns;
    const int b = unit / ns;
    mma_unit<T, D, MODE, NSTAGE>(&tmK, &tmV, p, b, uniform_seq(p, b), p.rows, kvh, s, rt, ps_shift, smem_raw, bars);
}

// ---------------------------------------------------------------- variable-length batches
// Sequence b's query tokens are packed rows [q_start[b], q_start[b + 1]) of q and out.  The grid
// enumerates blocks of the packed rows: sequence b owns blocks [first_block(b), first_block(b + 1))
// with first_block(b) = floor(q_start[b] G / 64) + b, at least as many as its 64-row tiles (and
// one decode unit when it has at most 16 rows); blocks beyond what it needs exit at once.
__device__ __forceinline__ long long varlen_first_block(const FwdParams &p, int b) {
    return (long long)__ldg(p.q_start + b) * p.G / kPrefillRows + b;
}

// The sequence owning block t: the largest b in [0, B) with first_block(b) <= t, by a 32-way
// search of one warp (first_block is strictly increasing for a valid q_start).
__device__ __forceinline__ int varlen_sequence(const FwdParams &p, long long t, int lane) {
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {
        const int stride = (hi - lo + 32) / 32;
        const int idx = min(lo + lane * stride, hi);
        const unsigned ok = __ballot_sync(0xffffffffu, varlen_first_block(p, idx) <= t);
        const int last = ok ? 31 - __clz((int)ok) : 0;
        lo = min(lo + last * stride, hi);
        hi = stride == 1 ? lo : min(lo + stride - 1, hi);
    }
    return lo;
}

// Mixed decode and prefill sequences in one grid: each CTA finds its sequence, then runs a
// 16-row decode unit (sequences with at most 16 query rows) or a 64-row prefill tile.  Units are
// visited in the order u -> u * p.row_tiles mod gridDim.x (p.row_tiles coprime to the grid), which
// spreads each sequence's units over the whole launch: the prefill tiles (tensor-bound) then run
// beside the decode units (HBM-bound) instead of in a phase of their own.  With a row cap
// (p.varlen_rows_cap: the tcgen05 kernel takes the sequences of that many rows or more) every
// sequence left fits one block, block t is sequence t, and the order is plain (row_tiles = 1).
template <typename T, int D, int NSTAGE>
__global__ void __launch_bounds__(kMmaThreads, (NSTAGE <= 3 ? 2 : 1))
    paged_attn_mma_varlen_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                                 const FwdParams p, int ps_shift) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[3 * NSTAGE];
    int unit = (int)(((unsigned long long)blockIdx.x * (unsigned)p.row_tiles) % gridDim.x);
    const int kvh = unit % p.Hkv;
    unit /= p.Hkv;
    const int s = unit % p.split_kv;
    const long long t = unit / p.split_kv;
    // with a row cap, every sequence this kernel takes fits one block: block t is sequence t
    const bool capped = p.varlen_rows_cap > 0;
    const int b = capped ? (int)t : varlen_sequence(p, t, threadIdx.x & 31);
    const int q0 = __ldg(p.q_start + b), q1 = __ldg(p.q_start + b + 1);
    if (q0 < 0 || q1 < q0 || (long long)q1 * p.Hq > p.rows_total) {
        if (threadIdx.x == 0) atomicOr(p.err, (unsigned int)PA_ERRBIT_QSTART);
        return;
    }
    const SeqRows sq{q0, q1 - q0};
    const int rows = sq.Sq * p.G;
    const long long j = capped ? 0 : t - varlen_first_block(p, b);  // block within the sequence
    if (rows == 0 || j < 0) return;
    if (p.varlen_rows_cap > 0 && rows >= p.varlen_rows_cap) return;  // the tcgen05 kernel's
    if (rows <= kDecodeRows) {
        if (j == 0) mma_unit<T, D, MODE_DECODE, NSTAGE>(&tmK, &tmV, p, b, sq, rows, kvh, s, 0, ps_shift, smem_raw, bars);
    } else if (j < (rows + kPrefillRows - 1) / kPrefillRows) {
        mma_unit<T, D, MODE_PREFILL, NSTAGE>(&tmK, &tmV, p, b, sq, rows, kvh, s, (int)j, ps_shift, smem_raw, bars);
    }
}

// ------------------------------------------------------------------------ host side

size_t mma_smem_bytes(int head_dim, int stages) {
    return (size_t)stages * 2 * kMmaTileKeys * head_dim * 2 + 1024;
}

template <typename T, int D, int MODE, int NSTAGE>
static cudaError_t launch_mma_t(const FwdParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                cudaStream_t stream) {
    auto kern = paged_attn_mma_kernel<T, D, MODE, NSTAGE>;
    const size_t smem = mma_smem_bytes(D, NSTAGE);
    static_assert(merge_scratch_bytes(D) <= (size_t)NSTAGE * 2 * kMmaTileKeys * D * 2,
                  "decode merge scratch must fit in the ring");
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int ps_shift = 0;
    while ((1 << ps_shift) < p.ps) ++ps_shift;
    const long long ns = MODE == MODE_SPLITS ? (p.split_kv + kMmaConsumerWarps - 1) / kMmaConsumerWarps : p.split_kv;
    const long long units = (long long)p.B * ns * p.Hkv * (MODE == MODE_PREFILL ? p.row_tiles : 1);
    if (units <= 0) return cudaSuccess;
    if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)units, kMmaThreads, smem, stream>>>(tmk, tmv, p, ps_shift);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_mma_dt(const FwdParams &p, int mode, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                 cudaStream_t stream) {
    if (p.D == 128) {
        if (mode == MODE_SPLITS) return launch_mma_t<T, 128, MODE_SPLITS, 3>(p, tmk, tmv, stream);
        return mode == MODE_DECODE ? launch_mma_t<T, 128, MODE_DECODE, 3>(p, tmk, tmv, stream)
                                   : launch_mma_t<T, 128, MODE_PREFILL, 3>(p, tmk, tmv, stream);
    }
    if (mode == MODE_SPLITS) return launch_mma_t<T, 64, MODE_SPLITS, 4>(p, tmk, tmv, stream);
    return mode == MODE_DECODE ? launch_mma_t<T, 64, MODE_DECODE, 4>(p, tmk, tmv, stream)
                               : launch_mma_t<T, 64, MODE_PREFILL, 4>(p, tmk, tmv, stream);
}

template <typename T, int D, int NSTAGE>
static cudaError_t launch_varlen_t(const FwdParams &p, long long blocks, const CUtensorMap &tmk,
                                   const CUtensorMap &tmv, cudaStream_t stream) {
    auto kern = paged_attn_mma_varlen_kernel<T, D, NSTAGE>;
    const size_t smem = mma_smem_bytes(D, NSTAGE);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int ps_shift = 0;
    while ((1 << ps_shift) < p.ps) ++ps_shift;
    const long long units = blocks * p.split_kv * p.Hkv;
    if (units <= 0) return cudaSuccess;
    if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    // visiting stride: the first value >= 0.618 units that is coprime to units (1 for tiny grids),
    // which mixes prefill tiles into the decode units; with a row cap (the tcgen05 kernel has the
    // prefill sequences) 1, so neighbouring CTAs read the kv heads of the same pages
    FwdParams q = p;
    long long stride = (units > 2 && p.varlen_rows_cap == 0) ? (units * 618) / 1000 : 1;
    auto gcd = [](long long a, long long b) { while (b) { const long long r = a % b; a = b; b = r; } return a; };
    while (stride > 1 && gcd(stride, units) != 1) ++stride;
    q.row_tiles = (int)(stride < 1 ? 1 : stride);
    kern<<<(unsigned)units, kMmaThreads, smem, stream>>>(tmk, tmv, q, ps_shift);
    return cudaGetLastError();
}

cudaError_t launch_mma_varlen(const FwdParams &p, long long total_q, int dtype, const CUtensorMap &tmk,
                              const CUtensorMap &tmv, cudaStream_t stream) {
    // blocks of the packed rows: floor(T G / 64) + B (see varlen_first_block); with a row cap of at
    // most 64 rows, one per sequence
    const long long blocks =
        (p.varlen_rows_cap > 0 && p.varlen_rows_cap <= kPrefillRows) ? p.B : total_q * p.G / kPrefillRows + p.B;
    if (dtype == PA_BF16) {
        return p.D == 128 ? launch_varlen_t<__nv_bfloat16, 128, 3>(p, blocks, tmk, tmv, stream)
                          : launch_varlen_t<__nv_bfloat16, 64, 4>(p, blocks, tmk, tmv, stream);
    }
    return p.D == 128 ? launch_varlen_t<__half, 128, 3>(p, blocks, tmk, tmv, stream)
                      : launch_varlen_t<__half, 64, 4>(p, blocks, tmk, tmv, stream);
}

cudaError_t launch_mma(const FwdParams &p, int mode, int dtype, const CUtensorMap &tmk, const CUtensorMap &tmv,
                       cudaStream_t stream) {
    if (dtype == PA_BF16) return launch_mma_dt<__nv_bfloat16>(p, mode, tmk, tmv, stream);
    return launch_mma_dt<__half>(p, mode, tmk, tmv, stream);
}

}  // namespace pa
