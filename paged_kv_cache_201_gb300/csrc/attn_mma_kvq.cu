// Tensor-core paged attention over FP8 E4M3 K/V pools with one float scale per (page, kv head),
// for bf16 / f16 queries, head_dim 64 or 128 (sm_103a).
//
// The pages' sweeps include i8 attention (rocMLIR PR #2371, Motivation; rocMLIR PR #2222, the
// reviewed files); a quantized pool here holds E4M3 elements whose value is element x scale of
// the element's (page, kv head).
//
// Units, producer warp and online softmax follow the 16-bit kernel (attn_mma.cu).  What differs:
//   * the producer copies each page's raw E4M3 rows (page_size tokens x head_dim bytes of one kv
//     head: one 3-D TMA box, half the bytes of a 16-bit page) into a ring of 64-key stages, and
//     with the page ids it loads the pages' K and V scales, which it leaves in shared memory
//     beside the stage before arming the stage's barriers.
//   * Q K^T runs in f16 straight from the ring: a lane converts the E4M3 bytes of its key into the
//     MMA operand registers (one conversion per element pair, exact: every E4M3 value is an f16
//     number).  The head dimension is visited in a permuted order, the same for Q and K, so that
//     a lane's operand bytes are 16 contiguous bytes of one row (one conflict-free shared load);
//     a dot product does not depend on the order of its terms.  bf16 queries enter as f16 after
//     multiplying each query row by a power of two that puts its largest element in [2^14, 2^15);
//     the score is scaled back by the inverse power exactly.
//   * V rows are widened to f16 in shared memory (exact) for the transposing ldmatrix; warp w
//     widens keys [16w, 16w + 16) of the stage.  Decode mode reads only its own 16 keys; prefill
//     mode (each warp owning 16 query rows over all 64 keys) meets the other warps at a named
//     barrier first.
//   * the scale of key j's page multiplies its score (scale x k_scale x q.k), and each 16-key step
//     of P V is accumulated separately and added to O times that step's page v_scale (a 16-key
//     step never crosses a page).  P itself is the unscaled softmax weight in [0, 1], split into
//     an f16 high part and its rounding remainder.
#include <type_traits>

#include "mma_common.cuh"

namespace pa {

using namespace mmac;

namespace {

constexpr int kMaxPagesPerStage = kMmaTileKeys / 16;  // page_size >= 16

template <int D>
struct Geo8 {
    static constexpr int kStage8 = kMmaTileKeys * D;     // bytes of one K (or V) stage, E4M3
    static constexpr int kWide = kMmaTileKeys * D * 2;   // the same 64 keys widened to 16 bits
};

// Widened rows: [4 warps][D/64 halves][16 keys][64 elements].  A row is 128 bytes; its 16-byte
// chunk c sits at position (c % 8) XOR (key % 8) XOR half, so that the 8 row addresses of an
// ldmatrix phase, and the 8 chunks a store phase of the widening writes, fall in 8 banks.
template <int D>
__device__ __forceinline__ uint32_t wide_addr(uint32_t base, int k, int c) {
    const int half = c >> 3;
    return base + (uint32_t)((k >> 4) * (16 * D * 2)) + (uint32_t)(((half << 4) + (k & 15)) << 7) +
           (uint32_t)((((c & 7) ^ (k & 7) ^ half)) << 4);
}

// Four E4M3 bytes (element 0 in the low byte) -> two f16 pairs, exactly.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t four, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 a, b;\n\t"
        "mov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(four));
}

// An f16 pair holding E4M3 values -> the same values as a bf16 pair (exact: 4 significant bits).
__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t h) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h));
    const __nv_bfloat162 v = __floats2bfloat162_rn(f.x, f.y);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// Widen keys [kw0, kw0 + 16) of one E4M3 stage (rows of D bytes, as the TMA left them) into
// 16-bit rows at `wide` (bf16 when TO_BF16, else f16).  Keys at or past key_end (relative to the
// stage) become zero rows: they hold whatever the ring held before, and a zero V row keeps
// 0 x NaN out of the output.
// Shared address of 16-byte chunk c of key row k in an E4M3 ring stage: rows of D bytes; for
// D = 128 the TMA wrote them with the 128-byte swizzle (chunk c at position c XOR (k % 8)).
template <int D>
__device__ __forceinline__ uint32_t ring_chunk_addr(uint32_t stage, int k, int c) {
    const int pc = (D == 128) ? (c ^ (k & 7)) : c;
    return stage + (uint32_t)(k * D + (pc << 4));
}

__device__ __forceinline__ void lds_v4(uint32_t addr, uint32_t (&w)[4]) {
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                 : "r"(addr)
                 : "memory");
}

template <int D, bool TO_BF16>
__device__ __forceinline__ void widen_keys(uint32_t ring, uint32_t wide, int kw0, int key_end, int lane) {
    constexpr int C8 = D / 16;  // 16-byte E4M3 chunks per row
#pragma unroll
    for (int it = 0; it < 16 * C8 / 32; ++it) {
        const int idx = it * 32 + lane;
        const int key = kw0 + idx / C8;
        const int c8 = idx % C8;
        uint32_t w[8];
        if (key < key_end) {
            uint32_t x[4];
            lds_v4(ring_chunk_addr<D>(ring, key, c8), x);
            e4m3x4_to_f16x4(x[0], w[0], w[1]);
            e4m3x4_to_f16x4(x[1], w[2], w[3]);
            e4m3x4_to_f16x4(x[2], w[4], w[5]);
            e4m3x4_to_f16x4(x[3], w[6], w[7]);
            if (TO_BF16) {
#pragma unroll
                for (int i = 0; i < 8; ++i) w[i] = f16x2_to_bf16x2(w[i]);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) w[i] = 0u;
        }
        // elements 16 c8 .. 16 c8 + 7 form 16-bit chunk 2 c8, the next eight chunk 2 c8 + 1
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(wide_addr<D>(wide, key, 2 * c8)), "r"(w[0]),
                     "r"(w[1]), "r"(w[2]), "r"(w[3])
                     : "memory");
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(wide_addr<D>(wide, key, 2 * c8 + 1)),
                     "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                     : "memory");
    }
}

// Power of two that brings a row whose largest magnitude is amax into f16 with amax x scale in
// [2^14, 2^15) (clamped to 2^[-113, 100], so both it and its inverse are normal floats); the inverse
// goes to inv.  Elements below 2^-28 amax become f16 subnormals: their terms of a dot product are
// below 2^-28 of its largest term.
__device__ __forceinline__ float f16_row_scale(float amax, float &inv) {
    const int e = (int)((__float_as_uint(amax) >> 23) & 0xffu) - 127;  // amax in [2^e, 2^(e+1))
    const int s = max(-113, min(14 - e, 100));
    inv = __uint_as_float((uint32_t)(127 - s) << 23);
    return __uint_as_float((uint32_t)(127 + s) << 23);
}

// bf16 pair x (power of two) -> f16 pair, round to nearest even (exact for normal f16 results:
// a bf16 number has 8 significant bits).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_scaled(uint32_t w, float sc) {
    const __half2 h = __floats2half2_rn(__uint_as_float(w << 16) * sc, __uint_as_float(w & 0xffff0000u) * sc);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// K operand of one n-tile (8 keys) for every MMA step: this lane's key row `k`, bytes
// [tq D/4, (tq + 1) D/4) of it, as f16 pairs.  Step kk takes bytes tq D/4 + 4 kk + {0, 1} (b0)
// and + {2, 3} (b1); the query fragments use the same head-dim order.  For D = 128 the lane's two
// chunks are 2 tq and 2 tq + 1: with the swizzle, the two keys of a load phase then read
// chunks of opposite parity, so the 8 lanes of a phase hit 8 different banks.
template <int D>
__device__ __forceinline__ void load_k_frags(uint32_t stage, int k, int tq, uint32_t (&bk)[D / 16][2]) {
#pragma unroll
    for (int h = 0; h < D / 64; ++h) {
        uint32_t w[4];
        lds_v4(ring_chunk_addr<D>(stage, k, (D / 64) * tq + h), w);
#pragma unroll
        for (int i = 0; i < 4; ++i) e4m3x4_to_f16x4(w[i], bk[4 * h + i][0], bk[4 * h + i][1]);
    }
}

}  // namespace

template <typename T, int D, int MODE, int NSTAGE>
__global__ void __launch_bounds__(kMmaThreads, 2)
    paged_attn_mma_kvq_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                              const FwdParams p, int ps_shift) {
    using Op = MmaOp<__half>;  // Q K^T and P V both in f16
    constexpr bool kQBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr int kStage8 = Geo8<D>::kStage8;
    constexpr int KB = (MODE == MODE_DECODE) ? 16 : 32;   // keys per softmax block
    constexpr int SUBS = (MODE == MODE_DECODE) ? 1 : 2;   // blocks a warp handles per stage
    constexpr int NTB = KB / 8;                           // score n-tiles per block
    constexpr int CTA_ROWS = (MODE == MODE_DECODE) ? kDecodeRows : kPrefillRows;
    constexpr int kSlots = 2 * NSTAGE;                    // scale slots (see the producer)

    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[3 * NSTAGE];
    __shared__ float s_ks[kSlots][kMaxPagesPerStage];
    __shared__ float s_vs[kSlots][kMaxPagesPerStage];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int ps = 1 << ps_shift;

    // ---- unit coordinates
    int unit = blockIdx.x;
    int rt = 0;
    if (MODE == MODE_PREFILL) {
        rt = unit % p.row_tiles;
        unit /= p.row_tiles;
    }
    const int kvh = unit % p.Hkv;
    unit /= p.Hkv;
    const int s = unit % p.split_kv;
    const int b = unit / p.split_kv;

    int L = max(p.seq_lens[b], 0);
    if (L > p.W * ps) {  // never read past the sequence's block-table row
        if (threadIdx.x == 0) atomicOr(p.err, (unsigned int)PA_ERRBIT_SEQ_CLIPPED);
        L = p.W * ps;
    }
    int pg0, pg1;
    split_pages(L, ps, p.split_kv, s, pg0, pg1);
    const int k_lo = pg0 * ps;
    const int k_hi_split = min(pg1 * ps, L);
    const int row0 = rt * CTA_ROWS;
    const int row_end = min(row0 + CTA_ROWS, p.rows);
    const int k_hi = min(k_hi_split, row_key_limit(p, b, L, (row_end - 1) / p.G));
    const int n_tiles = k_hi > k_lo ? (k_hi - k_lo + kMmaTileKeys - 1) / kMmaTileKeys : 0;

    if (n_tiles == 0) {
        if (warp < kMmaConsumerWarps) store_empty_unit<T, D>(p, b, kvh, s, row0, row_end);
        return;
    }

    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    const uint32_t wideV = sbase + (uint32_t)(NSTAGE * 2 * kStage8);
    const uint32_t bar_fk = smem_u32(&bars[0]);
    const uint32_t bar_fv = smem_u32(&bars[NSTAGE]);
    const uint32_t bar_em = smem_u32(&bars[2 * NSTAGE]);

    if (threadIdx.x == 0) {
        for (int st = 0; st < NSTAGE; ++st) {
            mbar_init(bar_fk + 8 * st, 1);
            mbar_init(bar_fv + 8 * st, 1);
            mbar_init(bar_em + 8 * st, kMmaConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kMmaConsumerWarps) {
        // ================================================================ producer
        if (lane == 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
        }
        const int pps = kMmaTileKeys >> ps_shift;       // pages per stage (1, 2 or 4)
        const uint32_t box_bytes = (uint32_t)(ps * D);  // one page of one kv head, E4M3
        const int pg_end = (k_hi + ps - 1) >> ps_shift;
        const int32_t *bt_row = p.block_table + (long long)b * p.W;
        // Page ids come 32 at a time, one per lane; each lane also holds its page's two scales.
        // An id outside [0, num_pages) gets scale 0 (its rows read as zeros).
        auto scale_of = [&](const float *sc, int id) -> float {
            return (id >= 0 && (long long)id < p.num_pages) ? __ldg(sc + (long long)id * p.Hkv + kvh) : 0.f;
        };
        int batch = pg0;
        int id_cur = (batch + lane < pg_end) ? __ldg(bt_row + batch + lane) : 0;
        int id_next = (batch + 32 + lane < pg_end) ? __ldg(bt_row + batch + 32 + lane) : 0;
        float ks_cur = 0.f, vs_cur = 0.f, ks_next = 0.f, vs_next = 0.f;
        if (batch + lane < pg_end) {
            ks_cur = scale_of(p.k_scale, id_cur);
            vs_cur = scale_of(p.v_scale, id_cur);
        }
        bool pend = true;  // scales of id_next not loaded yet
        bool bad = false;
        int issued = 0;
        for (int t = 0; t < n_tiles; ++t) {
            const int st = t % NSTAGE;
            const int slot = t % kSlots;
            if (t >= NSTAGE && !bad) {
                const bool ok = mbar_wait(bar_em + 8 * st, ((t / NSTAGE) - 1) & 1, p.err);
                bad = __any_sync(0xffffffffu, !ok);
            }
            const int pg_first = pg0 + t * pps;
            if (pg_first >= batch + 32) {
                if (pend && batch + 32 + lane < pg_end) {
                    ks_next = scale_of(p.k_scale, id_next);
                    vs_next = scale_of(p.v_scale, id_next);
                }
                batch += 32;
                id_cur = id_next;
                ks_cur = ks_next;
                vs_cur = vs_next;
                const int nx = batch + 32 + lane;
                id_next = (nx < pg_end) ? __ldg(bt_row + nx) : 0;
                ks_next = vs_next = 0.f;
                pend = true;
            }
            const int src = (pg_first + lane - batch) & 31;
            const int id = __shfl_sync(0xffffffffu, id_cur, src);
            const float ks = __shfl_sync(0xffffffffu, ks_cur, src);
            const float vs = __shfl_sync(0xffffffffu, vs_cur, src);
            if (bad) break;
            const int nvalid = min(pps, pg_end - pg_first);
            // Slot t % (2 NSTAGE) was last read for stage t - 2 NSTAGE; every consumer warp has
            // finished that stage once it released stage t - NSTAGE, which the wait above saw.
            if (lane < pps) {
                s_ks[slot][lane] = ks;
                s_vs[slot][lane] = vs;
            }
            __syncwarp();
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
                const uint32_t kdst = sbase + (uint32_t)(st * 2 * kStage8) + (uint32_t)lane * box_bytes;
                tma_load_3d(kdst, &tmK, bar_fk + 8 * st, 0, tok, kvh);
                tma_load_3d(kdst + kStage8, &tmV, bar_fv + 8 * st, 0, tok, kvh);
            }
            issued = t + 1;
            if (pend) {  // after this stage's copies are on their way
                if (batch + 32 + lane < pg_end) {
                    ks_next = scale_of(p.k_scale, id_next);
                    vs_next = scale_of(p.v_scale, id_next);
                }
                pend = false;
            }
        }
        for (int t = max(0, issued - NSTAGE); t < issued; ++t) {
            const int st = t % NSTAGE;
            const uint32_t par = (t / NSTAGE) & 1;
            mbar_wait(bar_fk + 8 * st, par, p.err);
            mbar_wait(bar_fv + 8 * st, par, p.err);
        }
        return;
    }

    // ==================================================================== consumers
    const int g = lane >> 2;
    const int tq = lane & 3;
    const int rbase = (MODE == MODE_DECODE) ? 0 : row0 + warp * 16;
    const int ra = rbase + g, rb = rbase + g + 8;
    const int kw0 = warp * 16;  // the stage keys whose V rows this warp widens (decode mode: its keys)

    // Q fragments in f16 over the permuted head-dim order: lane tq holds elements
    // [tq D/4, (tq + 1) D/4) of rows ra and rb, and step kk takes elements tq D/4 + 4 kk + {0, 1}
    // (a0 / a1) and + {2, 3} (a2 / a3).  q_inv_* undoes the power-of-two scaling of bf16 rows.
    uint32_t qf[D / 16][4];
    float q_inv_a = 1.f, q_inv_b = 1.f;
    {
        constexpr int NW = D / 8;  // element pairs a lane holds per row
        uint32_t wa[NW], wb[NW];
        const T *q = reinterpret_cast<const T *>(p.q);
        const bool va = ra < p.rows, vb = rb < p.rows;
        const uint4 *qa = reinterpret_cast<const uint4 *>(q + (va ? out_row_index(p, b, kvh, ra) * D : 0) + tq * (D / 4));
        const uint4 *qb = reinterpret_cast<const uint4 *>(q + (vb ? out_row_index(p, b, kvh, rb) * D : 0) + tq * (D / 4));
#pragma unroll
        for (int i = 0; i < NW / 4; ++i) {
            const uint4 xa = va ? __ldg(qa + i) : make_uint4(0u, 0u, 0u, 0u);
            const uint4 xb = vb ? __ldg(qb + i) : make_uint4(0u, 0u, 0u, 0u);
            wa[4 * i] = xa.x, wa[4 * i + 1] = xa.y, wa[4 * i + 2] = xa.z, wa[4 * i + 3] = xa.w;
            wb[4 * i] = xb.x, wb[4 * i + 1] = xb.y, wb[4 * i + 2] = xb.z, wb[4 * i + 3] = xb.w;
        }
        if (kQBf16) {
            float am_a = 0.f, am_b = 0.f;
#pragma unroll
            for (int i = 0; i < NW; ++i) {
                am_a = fmaxf(am_a, fmaxf(fabsf(__uint_as_float(wa[i] << 16)), fabsf(__uint_as_float(wa[i] & 0xffff0000u))));
                am_b = fmaxf(am_b, fmaxf(fabsf(__uint_as_float(wb[i] << 16)), fabsf(__uint_as_float(wb[i] & 0xffff0000u))));
            }
            am_a = fmaxf(am_a, __shfl_xor_sync(0xffffffffu, am_a, 1));
            am_a = fmaxf(am_a, __shfl_xor_sync(0xffffffffu, am_a, 2));
            am_b = fmaxf(am_b, __shfl_xor_sync(0xffffffffu, am_b, 1));
            am_b = fmaxf(am_b, __shfl_xor_sync(0xffffffffu, am_b, 2));
            const float sc_a = f16_row_scale(am_a, q_inv_a), sc_b = f16_row_scale(am_b, q_inv_b);
#pragma unroll
            for (int i = 0; i < NW; ++i) {
                wa[i] = bf16x2_to_f16x2_scaled(wa[i], sc_a);
                wb[i] = bf16x2_to_f16x2_scaled(wb[i], sc_b);
            }
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            qf[kk][0] = wa[2 * kk];
            qf[kk][1] = wb[2 * kk];
            qf[kk][2] = wa[2 * kk + 1];
            qf[kk][3] = wb[2 * kk + 1];
        }
    }
    const int lim_a = ra < p.rows ? min(k_hi_split, row_key_limit(p, b, L, ra / p.G)) : k_lo;
    const int lim_b = rb < p.rows ? min(k_hi_split, row_key_limit(p, b, L, rb / p.G)) : k_lo;
    // scale x log2(e) x the rows' inverse query scaling; times k_scale of the key's page below
    const float srow_a = p.scale_log2 * q_inv_a, srow_b = p.scale_log2 * q_inv_b;

    float m_a = kNegInf, m_b = kNegInf, l_a = 0.f, l_b = 0.f;
    float acc[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    const int warp_lim = __reduce_max_sync(0xffffffffu, (unsigned)max(lim_a, lim_b));
    const int mi = lane >> 3, rr = lane & 7;

    bool bad = false;
    for (int t = 0; t < n_tiles; ++t) {
        const int st = t % NSTAGE;
        const uint32_t par = (t / NSTAGE) & 1;
        const int slot = t % kSlots;
        const uint32_t kring = sbase + (uint32_t)(st * 2 * kStage8);
        const uint32_t vring = kring + (uint32_t)kStage8;
        const int tile_k0 = k_lo + t * kMmaTileKeys;

        if (!bad) {
            const bool ok = mbar_wait(bar_fk + 8 * st, par, p.err);
            bad = __any_sync(0xffffffffu, !ok);
        }
        if (MODE == MODE_PREFILL) {
            named_bar_sync(1, kMmaConsumerWarps * 32);  // every warp is done with the previous V rows
            if (!bad) {
                const bool ok = mbar_wait(bar_fv + 8 * st, par, p.err);
                bad = __any_sync(0xffffffffu, !ok);
            }
            if (!bad) widen_keys<D, false>(vring, wideV, kw0, k_hi - tile_k0, lane);
            named_bar_sync(1, kMmaConsumerWarps * 32);  // the stage's V rows are complete
        }

#pragma unroll
        for (int sb = 0; sb < SUBS; ++sb) {
            const int kb0 = ((MODE == MODE_DECODE) ? kw0 : 0) + sb * KB;  // first key (in the stage) of the block
            const bool active = tile_k0 + kb0 < min(k_hi, warp_lim);   // warp-uniform
            uint32_t ph[NTB][2], pl[NTB][2];
            if (!bad && active) {
                // ---- S = Q K^T over the block's KB keys, K converted from the ring
                float sc[NTB][4];
#pragma unroll
                for (int n = 0; n < NTB; ++n) {
                    sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
                    uint32_t bk[D / 16][2];
                    load_k_frags<D>(kring, kb0 + n * 8 + g, tq, bk);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) Op::run(sc[n], qf[kk], bk[kk][0], bk[kk][1]);
                }
                // ---- mask; scale x k_scale of the key's page (log2 domain)
                float mx_a = kNegInf, mx_b = kNegInf;
#pragma unroll
                for (int n = 0; n < NTB; ++n) {
                    const float ksc = s_ks[slot][(kb0 + n * 8) >> ps_shift];  // 8 keys share a page
                    const float fa = srow_a * ksc, fb = srow_b * ksc;
                    const int j = tile_k0 + kb0 + n * 8 + 2 * tq;
                    sc[n][0] = (j < lim_a) ? sc[n][0] * fa : kNegInf;
                    sc[n][1] = (j + 1 < lim_a) ? sc[n][1] * fa : kNegInf;
                    sc[n][2] = (j < lim_b) ? sc[n][2] * fb : kNegInf;
                    sc[n][3] = (j + 1 < lim_b) ? sc[n][3] * fb : kNegInf;
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
                // P split into an f16 high part and its rounding remainder: ~2^-22 relative
                float rs_a = 0.f, rs_b = 0.f;
#pragma unroll
                for (int n = 0; n < NTB; ++n) {
                    const float p0 = exp2f(sc[n][0] - mu_a), p1 = exp2f(sc[n][1] - mu_a);
                    const float p2 = exp2f(sc[n][2] - mu_b), p3 = exp2f(sc[n][3] - mu_b);
                    rs_a += p0 + p1;
                    rs_b += p2 + p3;
                    ph[n][0] = Op::pack(p0, p1);
                    ph[n][1] = Op::pack(p2, p3);
                    const float2 ha = Op::unpack(ph[n][0]), hb = Op::unpack(ph[n][1]);
                    pl[n][0] = Op::pack(p0 - ha.x, p1 - ha.y);
                    pl[n][1] = Op::pack(p2 - hb.x, p3 - hb.y);
                }
                l_a = l_a * al_a + rs_a;
                l_b = l_b * al_b + rs_b;
                if (__any_sync(0xffffffffu, al_a != 1.f || al_b != 1.f)) {  // the running max moved
#pragma unroll
                    for (int n = 0; n < D / 8; ++n) {
                        acc[n][0] *= al_a;
                        acc[n][1] *= al_a;
                        acc[n][2] *= al_b;
                        acc[n][3] *= al_b;
                    }
                }
            }

            if (MODE == MODE_DECODE) {
                if (!bad) {
                    const bool ok = mbar_wait(bar_fv + 8 * st, par, p.err);
                    bad = __any_sync(0xffffffffu, !ok);
                }
                if (!bad && active) widen_keys<D, false>(vring, wideV, kw0, k_hi - tile_k0, lane);
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_em + 8 * st);  // K read above, V widened: free the stage
            }

            if (!bad && active) {
                // ---- O += v_scale x (Ph + Pl) V, one 16-key step (one page) at a time
#pragma unroll
                for (int kst = 0; kst < KB / 16; ++kst) {
                    const float vsc = s_vs[slot][(kb0 + kst * 16) >> ps_shift];
                    const uint32_t ah[4] = {ph[2 * kst][0], ph[2 * kst][1], ph[2 * kst + 1][0], ph[2 * kst + 1][1]};
                    const uint32_t al[4] = {pl[2 * kst][0], pl[2 * kst][1], pl[2 * kst + 1][0], pl[2 * kst + 1][1]};
                    const int key = kb0 + kst * 16 + rr + ((mi & 1) << 3);
#pragma unroll
                    for (int j = 0; j < D / 16; ++j) {
                        uint32_t b0, b1, b2, b3;
                        ldmatrix_x4_trans(wide_addr<D>(wideV, key, 2 * j + (mi >> 1)), b0, b1, b2, b3);
                        float t0[4] = {0.f, 0.f, 0.f, 0.f}, t1[4] = {0.f, 0.f, 0.f, 0.f};
                        Op::run(t0, ah, b0, b1);
                        Op::run(t1, ah, b2, b3);
                        Op::run(t0, al, b0, b1);
                        Op::run(t1, al, b2, b3);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            acc[2 * j][e] = fmaf(vsc, t0[e], acc[2 * j][e]);
                            acc[2 * j + 1][e] = fmaf(vsc, t1[e], acc[2 * j + 1][e]);
                        }
                    }
                }
            }
        }
        if (MODE == MODE_PREFILL) {
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_em + 8 * st);  // K of the whole stage read, V widened
        }
    }

    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);

    if (MODE == MODE_PREFILL) {
        if (!bad) finish_prefill_rows<T, D>(p, b, kvh, s, ra, rb, row_end, tq, m_a, m_b, l_a, l_b, acc);
        return;
    }
    // decode: merge the four warps' states through shared memory (reuses the ring and the rows)
    decode_merge<T, D>(p, reinterpret_cast<float *>(smem_raw + (sbase - raw)), b, kvh, s, row_end, warp, lane, m_a,
                       m_b, l_a, l_b, acc, bad);
}

// ------------------------------------------------------------------------ host side
static constexpr int kvq_stages(int head_dim) { return head_dim == 128 ? 4 : 6; }

static size_t kvq_smem_bytes(int head_dim) {
    const int n = kvq_stages(head_dim);
    return (size_t)n * 2 * kMmaTileKeys * head_dim + (size_t)kMmaTileKeys * head_dim * 2 + 1024;
}

template <typename T, int D, int MODE>
static cudaError_t launch_kvq_t(const FwdParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                cudaStream_t stream) {
    constexpr int NSTAGE = kvq_stages(D);
    static_assert(merge_scratch_bytes(D) <= (size_t)NSTAGE * 2 * Geo8<D>::kStage8 + Geo8<D>::kWide,
                  "decode merge scratch must fit in the ring and the widened rows");
    auto kern = paged_attn_mma_kvq_kernel<T, D, MODE, NSTAGE>;
    const size_t smem = kvq_smem_bytes(D);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int ps_shift = 0;
    while ((1 << ps_shift) < p.ps) ++ps_shift;
    const long long units = (long long)p.B * p.split_kv * p.Hkv * (MODE == MODE_PREFILL ? p.row_tiles : 1);
    if (units <= 0) return cudaSuccess;
    if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)units, kMmaThreads, smem, stream>>>(tmk, tmv, p, ps_shift);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_kvq_dt(const FwdParams &p, int mode, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                 cudaStream_t stream) {
    if (p.D == 128) {
        return mode == MODE_DECODE ? launch_kvq_t<T, 128, MODE_DECODE>(p, tmk, tmv, stream)
                                   : launch_kvq_t<T, 128, MODE_PREFILL>(p, tmk, tmv, stream);
    }
    return mode == MODE_DECODE ? launch_kvq_t<T, 64, MODE_DECODE>(p, tmk, tmv, stream)
                               : launch_kvq_t<T, 64, MODE_PREFILL>(p, tmk, tmv, stream);
}

cudaError_t launch_mma_kvq(const FwdParams &p, int mode, int dtype, const CUtensorMap &tmk, const CUtensorMap &tmv,
                           cudaStream_t stream) {
    if (dtype == PA_BF16) return launch_kvq_dt<__nv_bfloat16>(p, mode, tmk, tmv, stream);
    return launch_kvq_dt<__half>(p, mode, tmk, tmv, stream);
}

}  // namespace pa
