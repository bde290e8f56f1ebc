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
//   * consumer warp w widens keys [16w, 16w + 16) of each stage to 16-bit rows (K to the query's
//     type, V to bf16).  Both are exact: every E4M3 value is an f16 and a bf16 number.  The warp
//     then releases the ring stage at once, so the next pages stream in while it computes.
//     Decode mode reads only its own 16 keys; prefill mode (each warp owning 16 query rows over
//     all 64 keys) meets the other warps at a named barrier first.
//   * the scale of key j's page enters its score (scale x k_scale x q.k) and the weight of its
//     V row (p_j x v_scale); the softmax sum takes the unscaled p_j.  The tensor-core operands
//     are the stored values, so the only rounding added is that of these float products.
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
            uint32_t x0, x1, x2, x3;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                         : "r"(ring + (uint32_t)(key * D + c8 * 16))
                         : "memory");
            e4m3x4_to_f16x4(x0, w[0], w[1]);
            e4m3x4_to_f16x4(x1, w[2], w[3]);
            e4m3x4_to_f16x4(x2, w[4], w[5]);
            e4m3x4_to_f16x4(x3, w[6], w[7]);
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

}  // namespace

template <typename T, int D, int MODE, int NSTAGE>
__global__ void __launch_bounds__(kMmaThreads, 2)
    paged_attn_mma_kvq_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                              const FwdParams p, int ps_shift) {
    using Op = MmaOp<T>;                  // Q K^T in the query's type
    using OpV = MmaOp<__nv_bfloat16>;     // P V in bf16 (P x v_scale keeps bf16's exponent range)
    constexpr bool kKBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr int kStage8 = Geo8<D>::kStage8;
    constexpr int kWide = Geo8<D>::kWide;
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
    const uint32_t wideK = sbase + (uint32_t)(NSTAGE * 2 * kStage8);
    const uint32_t wideV = wideK + (uint32_t)kWide;
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
    const int kw0 = warp * 16;  // the stage keys this warp widens (and, in decode mode, reads)

    uint32_t qf[D / 16][4];
    {
        const T *q = reinterpret_cast<const T *>(p.q);
        const bool va = ra < p.rows, vb = rb < p.rows;
        const T *qa = q + (va ? out_row_index(p, b, kvh, ra) * D : 0);
        const T *qb = q + (vb ? out_row_index(p, b, kvh, rb) * D : 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const int c0 = kk * 16 + 2 * tq;
            qf[kk][0] = va ? __ldg(reinterpret_cast<const uint32_t *>(qa + c0)) : 0u;
            qf[kk][1] = vb ? __ldg(reinterpret_cast<const uint32_t *>(qb + c0)) : 0u;
            qf[kk][2] = va ? __ldg(reinterpret_cast<const uint32_t *>(qa + c0 + 8)) : 0u;
            qf[kk][3] = vb ? __ldg(reinterpret_cast<const uint32_t *>(qb + c0 + 8)) : 0u;
        }
    }
    const int lim_a = ra < p.rows ? min(k_hi_split, row_key_limit(p, b, L, ra / p.G)) : k_lo;
    const int lim_b = rb < p.rows ? min(k_hi_split, row_key_limit(p, b, L, rb / p.G)) : k_lo;

    float m_a = kNegInf, m_b = kNegInf, l_a = 0.f, l_b = 0.f;
    float acc[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    const int warp_lim = __reduce_max_sync(0xffffffffu, (unsigned)max(lim_a, lim_b));

    bool bad = false;
    for (int t = 0; t < n_tiles; ++t) {
        const int st = t % NSTAGE;
        const uint32_t par = (t / NSTAGE) & 1;
        const int slot = t % kSlots;
        const uint32_t kring = sbase + (uint32_t)(st * 2 * kStage8);
        const uint32_t vring = kring + (uint32_t)kStage8;
        const int tile_k0 = k_lo + t * kMmaTileKeys;
        // decode mode reads only this warp's keys, prefill mode every warp's
        const bool widen = (MODE == MODE_PREFILL) || (tile_k0 + kw0 < min(k_hi, warp_lim));

        if (MODE == MODE_PREFILL) named_bar_sync(1, kMmaConsumerWarps * 32);  // previous rows read by all
        if (!bad) {
            const bool ok = mbar_wait(bar_fk + 8 * st, par, p.err);
            bad = __any_sync(0xffffffffu, !ok);
        }
        if (!bad && widen) widen_keys<D, kKBf16>(kring, wideK, kw0, k_hi - tile_k0, lane);
        if (!bad) {
            const bool ok = mbar_wait(bar_fv + 8 * st, par, p.err);
            bad = __any_sync(0xffffffffu, !ok);
        }
        if (!bad && widen) widen_keys<D, true>(vring, wideV, kw0, k_hi - tile_k0, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_em + 8 * st);  // the ring stage is widened: free it
        if (MODE == MODE_PREFILL)
            named_bar_sync(1, kMmaConsumerWarps * 32);
        else
            __syncwarp();

#pragma unroll
        for (int sb = 0; sb < SUBS; ++sb) {
            const int kb0 = ((MODE == MODE_DECODE) ? kw0 : 0) + sb * KB;  // first key (in the stage) of the block
            const bool active = tile_k0 + kb0 < min(k_hi, warp_lim);   // warp-uniform
            if (bad || !active) continue;
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
                    ldmatrix_x4(wide_addr<D>(wideK, key, 2 * kk + (mi & 1)), b0, b1, b2, b3);
                    Op::run(sc[2 * np], qf[kk], b0, b1);
                    Op::run(sc[2 * np + 1], qf[kk], b2, b3);
                }
            }
            // ---- mask, scale x k_scale of the key's page (log2 domain)
            float vsn[NTB];
            float mx_a = kNegInf, mx_b = kNegInf;
#pragma unroll
            for (int n = 0; n < NTB; ++n) {
                const int pis = (kb0 + n * 8) >> ps_shift;  // page within the stage (8 keys share one)
                const float kq = p.scale_log2 * s_ks[slot][pis];
                vsn[n] = s_vs[slot][pis];
                const int j = tile_k0 + kb0 + n * 8 + 2 * tq;
                sc[n][0] = (j < lim_a) ? sc[n][0] * kq : kNegInf;
                sc[n][1] = (j + 1 < lim_a) ? sc[n][1] * kq : kNegInf;
                sc[n][2] = (j < lim_b) ? sc[n][2] * kq : kNegInf;
                sc[n][3] = (j + 1 < lim_b) ? sc[n][3] * kq : kNegInf;
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
            // P x v_scale split into a bf16 high part and the rounding remainder (see attn_mma.cu)
            uint32_t ph[NTB][2], pl[NTB][2];
            float rs_a = 0.f, rs_b = 0.f;
#pragma unroll
            for (int n = 0; n < NTB; ++n) {
                const float p0 = exp2f(sc[n][0] - mu_a), p1 = exp2f(sc[n][1] - mu_a);
                const float p2 = exp2f(sc[n][2] - mu_b), p3 = exp2f(sc[n][3] - mu_b);
                rs_a += p0 + p1;
                rs_b += p2 + p3;
                const float w0 = p0 * vsn[n], w1 = p1 * vsn[n], w2 = p2 * vsn[n], w3 = p3 * vsn[n];
                ph[n][0] = OpV::pack(w0, w1);
                ph[n][1] = OpV::pack(w2, w3);
                const float2 ha = OpV::unpack(ph[n][0]), hb = OpV::unpack(ph[n][1]);
                pl[n][0] = OpV::pack(w0 - ha.x, w1 - ha.y);
                pl[n][1] = OpV::pack(w2 - hb.x, w3 - hb.y);
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
            // ---- O += (Ph + Pl) V
#pragma unroll
            for (int ks = 0; ks < KB / 16; ++ks) {
                const uint32_t ah[4] = {ph[2 * ks][0], ph[2 * ks][1], ph[2 * ks + 1][0], ph[2 * ks + 1][1]};
                const uint32_t al[4] = {pl[2 * ks][0], pl[2 * ks][1], pl[2 * ks + 1][0], pl[2 * ks + 1][1]};
                const int key = kb0 + ks * 16 + rr + ((mi & 1) << 3);
#pragma unroll
                for (int j = 0; j < D / 16; ++j) {
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4_trans(wide_addr<D>(wideV, key, 2 * j + (mi >> 1)), b0, b1, b2, b3);
                    OpV::run(acc[2 * j], ah, b0, b1);
                    OpV::run(acc[2 * j + 1], ah, b2, b3);
                    OpV::run(acc[2 * j], al, b0, b1);
                    OpV::run(acc[2 * j + 1], al, b2, b3);
                }
            }
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
    return (size_t)n * 2 * kMmaTileKeys * head_dim + 2 * (size_t)kMmaTileKeys * head_dim * 2 + 1024;
}

template <typename T, int D, int MODE>
static cudaError_t launch_kvq_t(const FwdParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                cudaStream_t stream) {
    constexpr int NSTAGE = kvq_stages(D);
    static_assert(merge_scratch_bytes(D) <= (size_t)NSTAGE * 2 * Geo8<D>::kStage8 + 2 * Geo8<D>::kWide,
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
