// Tensor-core paged attention over 8-bit K/V pools (FP8 E4M3 or int8 elements) with one float
// scale per (page, kv head), for bf16 / f16 queries, head_dim 64 or 128 (sm_103a).
//
// The pages' sweeps include i8 attention (rocMLIR PR #2371, Motivation; rocMLIR PR #2222, the
// reviewed files); a quantized pool here holds E4M3 or two's-complement int8 elements whose value
// is element x scale of the element's (page, kv head).  Both formats convert exactly to f16 (every
// E4M3 value and every integer in [-128, 127] is an f16 number), so one kernel body serves both;
// the element format is a template parameter (FMT) that picks the conversion.
//
// Units (one CTA per (sequence, kv head, split[, 64-row query tile])), the producer warp and the
// online softmax with its guards follow the 16-bit kernel (attn_mma.cu).  What differs:
//   * the producer copies each page's raw 8-bit rows (page_size tokens x head_dim bytes of one kv
//     head: one 3-D TMA box, half the bytes of a 16-bit page) into a ring of 64-key stages, and
//     with the page ids it loads the pages' K and V scales, which it leaves in shared memory
//     beside the stage before arming the stage's barriers.
//   * K enters the tensor cores in f16 straight from the ring: a lane converts the 8-bit bytes of
//     its key into MMA operand registers (exact).  The head dimension is visited in a permuted
//     order, the same for Q and K, so that a lane's operand bytes are 16 contiguous bytes of one
//     row (one conflict-free shared load); a dot product does not depend on the order of its terms.  bf16 queries enter as f16
//     after multiplying each query row by a power of two that puts its largest element in
//     [2^14, 2^15); the score is scaled back by the inverse power exactly.
//   * decode converts V from the ring the same way and transposes it in registers (movmatrix);
//     prefill widens V rows to f16 in shared memory (exact) for the transposing ldmatrix.
//   * the scale of key j's page multiplies its score (scale x k_scale x q.k); each 16-key step of
//     P V (one page: page_size >= 16) is accumulated on its own and added to O times the page's
//     v_scale.  P is the unscaled softmax weight in [0, 1], split into an f16 high part and its
//     rounding remainder.
//   * decode (at most 16 query rows per unit) computes the transposed products S^T = K Q^T and
//     O^T = V^T P^T: keys and head dimension fill the MMA's 16-row side, the GQA group its 8-wide
//     side, so a group of 4 or 8 heads does not pay for 16 rows; P^T is turned into the second
//     operand's layout with movmatrix.  Prefill keeps S = Q K^T over 64-row query tiles.
#include <type_traits>

#include "mma_common.cuh"

namespace pa {

using namespace mmac;

namespace {

constexpr int kMaxPagesPerStage = kMmaTileKeys / 16;  // prefill stages: page_size >= 16

template <int D>
struct Geo8 {
    static constexpr int kStage8 = kMmaTileKeys * D;     // bytes of one K (or V) stage, 8-bit elements
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

// Four int8 bytes (element 0 in the low byte) -> two f16 pairs, exactly.  Byte XOR 0x80 is v + 128
// in [0, 255]; placed as the low mantissa byte of an f16 with biased exponent 25 (0x64 in the high
// byte: the binade [1024, 2048), whose spacing is 1) it reads 1024 + v + 128, and subtracting 1152
// (0x6480) leaves v.
__device__ __forceinline__ void s8x4_to_f16x4(uint32_t four, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = four ^ 0x80808080u;
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);  // bytes u0, 0x64, u1, 0x64
    const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);  // bytes u2, 0x64, u3, 0x64
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
}

constexpr int kFmtE4M3 = 0, kFmtInt8 = 1;  // element formats of a quantized pool

template <int FMT>
__device__ __forceinline__ void q8x4_to_f16x4(uint32_t four, uint32_t &lo, uint32_t &hi) {
    if constexpr (FMT == kFmtInt8)
        s8x4_to_f16x4(four, lo, hi);
    else
        e4m3x4_to_f16x4(four, lo, hi);
}

// Widen keys [kw0, kw0 + 16) of one 8-bit stage (rows of D bytes, as the TMA left them) into
// f16 rows at `wide`.  Keys at or past key_end (relative to the
// stage) become zero rows: they hold whatever the ring held before, and a zero V row keeps
// 0 x NaN out of the output.
// Shared address of 16-byte chunk c of key row k in an 8-bit ring stage: rows of D bytes; for
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

template <int FMT, int D>
__device__ __forceinline__ void widen_keys(uint32_t ring, uint32_t wide, int kw0, int key_end, int lane) {
    constexpr int C8 = D / 16;  // 16-byte chunks of 8-bit elements per row
#pragma unroll
    for (int it = 0; it < 16 * C8 / 32; ++it) {
        const int idx = it * 32 + lane;
        const int key = kw0 + idx / C8;
        const int c8 = idx % C8;
        uint32_t w[8];
        if (key < key_end) {
            uint32_t x[4];
            lds_v4(ring_chunk_addr<D>(ring, key, c8), x);
            q8x4_to_f16x4<FMT>(x[0], w[0], w[1]);
            q8x4_to_f16x4<FMT>(x[1], w[2], w[3]);
            q8x4_to_f16x4<FMT>(x[2], w[4], w[5]);
            q8x4_to_f16x4<FMT>(x[3], w[6], w[7]);
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
template <int FMT, int D>
__device__ __forceinline__ void load_k_frags(uint32_t stage, int k, int tq, uint32_t (&bk)[D / 16][2]) {
#pragma unroll
    for (int h = 0; h < D / 64; ++h) {
        uint32_t w[4];
        lds_v4(ring_chunk_addr<D>(stage, k, (D / 64) * tq + h), w);
#pragma unroll
        for (int i = 0; i < 4; ++i) q8x4_to_f16x4<FMT>(w[i], bk[4 * h + i][0], bk[4 * h + i][1]);
    }
}


// One query row as f16 operand pairs in the permuted head-dim order: this lane's elements
// [tq D/4, (tq + 1) D/4), pair i = elements tq D/4 + 2 i and + 1.  bf16 rows are multiplied by the
// f16_row_scale power of two of the whole row (the 4 lanes of a quad hold one row) and inv gets
// its inverse; f16 rows are taken as they are (inv = 1).  A row that is not valid reads as zeros.
template <typename T, int D>
__device__ __forceinline__ void load_q_row(const T *row, bool valid, int tq, uint32_t (&w)[D / 8], float &inv) {
    const uint4 *src = reinterpret_cast<const uint4 *>(row + tq * (D / 4));
#pragma unroll
    for (int i = 0; i < D / 32; ++i) {
        const uint4 x = valid ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u);
        w[4 * i] = x.x;
        w[4 * i + 1] = x.y;
        w[4 * i + 2] = x.z;
        w[4 * i + 3] = x.w;
    }
    inv = 1.f;
    if (std::is_same<T, __nv_bfloat16>::value) {
        float am = 0.f;
#pragma unroll
        for (int i = 0; i < D / 8; ++i)
            am = fmaxf(am, fmaxf(fabsf(__uint_as_float(w[i] << 16)), fabsf(__uint_as_float(w[i] & 0xffff0000u))));
        am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
        am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
        const float sc = f16_row_scale(am, inv);
#pragma unroll
        for (int i = 0; i < D / 8; ++i) w[i] = bf16x2_to_f16x2_scaled(w[i], sc);
    }
}

// Transpose of an 8 x 8 matrix of 16-bit elements held one row pair per lane (lane 4 r + c holds
// elements (r, 2c) and (r, 2c + 1)); returns the same lane's pair of the transpose.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// The producer warp of one unit.  Page ids come 32 at a time, one per lane, never past the unit's
// pages; each lane also holds its page's K and V scales (an id outside [0, num_pages) gets scale 0
// and its rows read as zeros).  Per SK-key stage t it writes the stage's page scales into slot
// t % (2 NSTAGE), arms the stage's barriers and issues one 3-D TMA box per page and pool into
// ring stage t % NSTAGE.
template <int D, int NSTAGE, int SK>
__device__ __forceinline__ void kvq_produce(const CUtensorMap *tmK, const CUtensorMap *tmV, const FwdParams &p,
                                            int b, int kvh, int pg0, int k_hi, int n_tiles, int ps_shift,
                                            uint32_t sbase, uint32_t bar_fk, uint32_t bar_fv, uint32_t bar_em,
                                            float (*s_ks)[SK / 16], float (*s_vs)[SK / 16], int lane) {
    constexpr int kStage8 = SK * D;  // bytes of one K (or V) stage of SK keys
    constexpr int kSlots = 2 * NSTAGE;
    if (lane == 0) {
        tma_prefetch_desc(tmK);
        tma_prefetch_desc(tmV);
    }
    const int ps = 1 << ps_shift;
    const int pps = SK >> ps_shift;                 // pages per stage (page_size >= 16: at most SK / 16)
    const uint32_t box_bytes = (uint32_t)(ps * D);  // one page of one kv head, 8-bit elements
    const int pg_end = (k_hi + ps - 1) >> ps_shift;
    const int32_t *bt_row = p.block_table + (long long)b * p.W;
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
            tma_load_3d(kdst, tmK, bar_fk + 8 * st, 0, tok, kvh);
            tma_load_3d(kdst + kStage8, tmV, bar_fv + 8 * st, 0, tok, kvh);
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
    // every copy must have landed before the CTA may exit
    for (int t = max(0, issued - NSTAGE); t < issued; ++t) {
        const int st = t % NSTAGE;
        const uint32_t par = (t / NSTAGE) & 1;
        mbar_wait(bar_fk + 8 * st, par, p.err);
        mbar_wait(bar_fv + 8 * st, par, p.err);
    }
}

// Unit bounds shared by both kernels: sequence length clipped to the block-table row, the
// split's key range [k_lo, k_hi_split) and its 64-key stage count up to key k_hi.
struct KvqUnit {
    int L, pg0, k_lo, k_hi_split;
};

__device__ __forceinline__ KvqUnit kvq_unit(const FwdParams &p, int b, int s, int ps_shift) {
    KvqUnit u;
    const int ps = 1 << ps_shift;
    u.L = max(p.seq_lens[b], 0);
    if (u.L > p.W * ps) {  // never read past the sequence's block-table row
        if (threadIdx.x == 0) atomicOr(p.err, (unsigned int)PA_ERRBIT_SEQ_CLIPPED);
        u.L = p.W * ps;
    }
    int pg1;
    split_pages(u.L, ps, p.split_kv, s, u.pg0, pg1);
    u.k_lo = u.pg0 * ps;
    u.k_hi_split = min(pg1 * ps, u.L);
    return u;
}

}  // namespace

// ============================================================================ decode
// At most 16 query rows per (sequence, kv head): the kernel computes S^T = K Q^T and O^T = V^T P^T,
// so that keys and head dimension fill the MMA's 16-row side and the few query rows (GQA group x
// query tokens, padded to NR x 8) its 8-column side.  Warp w reads keys [16 w, 16 w + 16) of every
// stage (one page: page_size >= 16); the four warps' softmax states are merged at the end.
template <typename T, int FMT, int D, int NR, int NSTAGE, int KPW, int MINB>
__global__ void __launch_bounds__(kMmaThreads, MINB)
    paged_attn_kvq_decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                                 const FwdParams p, int ps_shift) {
    using Op = MmaOp<__half>;
    constexpr int SK = kMmaConsumerWarps * KPW;  // keys per stage
    constexpr int NB = KPW / 16;                 // 16-key blocks per warp and stage (one page each)
    constexpr int kStage8 = SK * D;              // bytes of one K (or V) stage
    constexpr int kSlots = 2 * NSTAGE;
    constexpr int MT = D / 16;                   // 16-wide head-dim tiles of O^T
    // Release each stage as soon as it is in registers: int8 2.3 % faster on the Llama-3-8B-shaped
    // decode; E4M3 the same or 1 % slower (so not there), and two row tiles would spill.
    constexpr bool kEarly = NR == 1 && FMT == kFmtInt8;

    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[3 * NSTAGE];
    __shared__ float s_ks[kSlots][SK / 16];
    __shared__ float s_vs[kSlots][SK / 16];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int unit = blockIdx.x;
    const int kvh = unit % p.Hkv;
    unit /= p.Hkv;
    const int s = unit % p.split_kv;
    const int b = unit / p.split_kv;
    const KvqUnit u = kvq_unit(p, b, s, ps_shift);
    const SeqRows sq = uniform_seq(p, b);
    const int rows = p.rows;  // <= 8 NR
    const int k_hi = min(u.k_hi_split, row_key_limit(p, b, u.L, (rows - 1) / p.G));
    const int n_tiles = k_hi > u.k_lo ? (k_hi - u.k_lo + SK - 1) / SK : 0;
    if (n_tiles == 0) {
        if (warp < kMmaConsumerWarps) store_empty_unit<T, D>(p, sq, kvh, s, 0, rows);
        return;
    }

    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
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
        kvq_produce<D, NSTAGE, SK>(&tmK, &tmV, p, b, kvh, u.pg0, k_hi, n_tiles, ps_shift, sbase, bar_fk, bar_fv,
                                   bar_em, s_ks, s_vs, lane);
        return;
    }

    // ==================================================================== consumers
    const int g = lane >> 2;
    const int tq = lane & 3;
    const int kw0 = warp * KPW;  // this warp's keys in every stage: NB blocks of 16
    // Q^T operands: row-tile nr, this lane's row 8 nr + g.  The score and output fragments hold
    // rows 8 nr + 2 tq + e (e = 0, 1): their inverse query scalings come from lanes 4 (2 tq + e).
    uint32_t qb[NR][D / 16][2];
    float srow[NR][2];
    int lim[NR][2];
    int lmax = u.k_lo;
#pragma unroll
    for (int nr = 0; nr < NR; ++nr) {
        const int r = nr * 8 + g;
        const bool valid = r < rows;
        const T *qrow = reinterpret_cast<const T *>(p.q) + (valid ? q_row_offset(p, out_row_index(p, sq, kvh, r)) : 0);
        uint32_t w[D / 8];
        float inv;
        load_q_row<T, D>(qrow, valid, tq, w, inv);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            qb[nr][kk][0] = w[2 * kk];
            qb[nr][kk][1] = w[2 * kk + 1];
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int rc = nr * 8 + 2 * tq + e;
            srow[nr][e] = p.scale_log2 * __shfl_sync(0xffffffffu, inv, 4 * (2 * tq + e));
            lim[nr][e] = rc < rows ? min(u.k_hi_split, row_key_limit(p, b, u.L, rc / p.G)) : u.k_lo;
            lmax = max(lmax, lim[nr][e]);
        }
    }
    // keys at or past the furthest limit of the unit's rows are masked for all of them
    const int key_lim = min(k_hi, (int)__reduce_max_sync(0xffffffffu, (unsigned)lmax));

    float m[NR][2], l[NR][2];
    float acc[NR][MT][4];
#pragma unroll
    for (int nr = 0; nr < NR; ++nr) {
        m[nr][0] = m[nr][1] = kNegInf;
        l[nr][0] = l[nr][1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) acc[nr][mt][0] = acc[nr][mt][1] = acc[nr][mt][2] = acc[nr][mt][3] = 0.f;
    }

    bool bad = false;
    for (int t = 0; t < n_tiles; ++t) {
        const int st = t % NSTAGE;
        const uint32_t par = (t / NSTAGE) & 1;
        const int slot = t % kSlots;
        const uint32_t kring = sbase + (uint32_t)(st * 2 * kStage8);
        const uint32_t vring = kring + (uint32_t)kStage8;
        const int tile_k0 = u.k_lo + t * SK;
        const bool active = tile_k0 + kw0 < key_lim;  // warp-uniform

        if (!bad) {
            const bool ok = mbar_wait(bar_fk + 8 * st, par, p.err) && (!kEarly || mbar_wait(bar_fv + 8 * st, par, p.err));
            bad = __any_sync(0xffffffffu, !ok);
        }
        // This lane's bytes of keys g and g + 8 of each block (D/4 of each row; [block][key half]
        // [16-byte chunk][word] for K).  kEarly: K and V go to registers first and the stage is
        // released at once, so the ring slot refills while the warp computes; else K is read in the
        // product and V after the softmax (two query-row tiles leave no registers for it).
        uint32_t kw[NB][2][D / 64][4], vw[NB][2][D / 16];
        auto read_v = [&]() {
#pragma unroll
            for (int hb = 0; hb < NB; ++hb)
#pragma unroll
                for (int kh = 0; kh < 2; ++kh)
#pragma unroll
                    for (int h = 0; h < D / 64; ++h) {
                        uint32_t w[4];
                        lds_v4(ring_chunk_addr<D>(vring, kw0 + 16 * hb + g + 8 * kh, (D / 64) * tq + h), w);
#pragma unroll
                        for (int i = 0; i < 4; ++i) vw[hb][kh][4 * h + i] = w[i];
                    }
        };
        auto read_k = [&](int hb, int h) {
#pragma unroll
            for (int kh = 0; kh < 2; ++kh)
                lds_v4(ring_chunk_addr<D>(kring, kw0 + 16 * hb + g + 8 * kh, (D / 64) * tq + h), kw[hb][kh][h]);
        };
        if constexpr (kEarly) {
            if (!bad && active) {
#pragma unroll
                for (int hb = 0; hb < NB; ++hb)
#pragma unroll
                    for (int h = 0; h < D / 64; ++h) read_k(hb, h);
                read_v();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_em + 8 * st);  // K and V of the stage are read: free it
        }
        uint32_t pb[NB][NR][2][2];  // P^T operands: [block][row tile][high / low part][keys 0-7 / 8-15]
        if (!bad && active) {
            // ---- S^T = K Q^T: keys g and g + 8 of each of the warp's blocks, two partial sums each
            float sc[NB][NR][2][4];
#pragma unroll
            for (int hb = 0; hb < NB; ++hb)
#pragma unroll
                for (int nr = 0; nr < NR; ++nr)
#pragma unroll
                    for (int c = 0; c < 2; ++c) sc[hb][nr][c][0] = sc[hb][nr][c][1] = sc[hb][nr][c][2] = sc[hb][nr][c][3] = 0.f;
#pragma unroll
            for (int hb = 0; hb < NB; ++hb) {
#pragma unroll
                for (int h = 0; h < D / 64; ++h) {
                    if constexpr (!kEarly) read_k(hb, h);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int kk = 4 * h + i;
                        uint32_t a[4];
                        q8x4_to_f16x4<FMT>(kw[hb][0][h][i], a[0], a[2]);
                        q8x4_to_f16x4<FMT>(kw[hb][1][h][i], a[1], a[3]);
#pragma unroll
                        for (int nr = 0; nr < NR; ++nr) Op::run(sc[hb][nr][i & 1], a, qb[nr][kk][0], qb[nr][kk][1]);
                    }
                }
            }
            // ---- mask; scale x k_scale of each block's page (log2 domain); one online-softmax step
            // per row over the warp's KPW keys
            float ksc[NB];
#pragma unroll
            for (int hb = 0; hb < NB; ++hb) ksc[hb] = s_ks[slot][(kw0 + 16 * hb) >> ps_shift];
            float al[NR][2], pv[NB][NR][2][2];
            bool moved = false;
#pragma unroll
            for (int nr = 0; nr < NR; ++nr) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float x[NB][2];
                    float mx = kNegInf;
#pragma unroll
                    for (int hb = 0; hb < NB; ++hb) {
                        const float f = srow[nr][e] * ksc[hb];
                        const int j0 = tile_k0 + kw0 + 16 * hb + g;  // key of elements 0-1; j0 + 8 for 2-3
                        const float x0 = sc[hb][nr][0][e] + sc[hb][nr][1][e];
                        const float x1 = sc[hb][nr][0][2 + e] + sc[hb][nr][1][2 + e];
                        x[hb][0] = (j0 < lim[nr][e]) ? x0 * f : kNegInf;
                        x[hb][1] = (j0 + 8 < lim[nr][e]) ? x1 * f : kNegInf;
                        mx = fmaxf(mx, fmaxf(x[hb][0], x[hb][1]));
                    }
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                    const float mn = fmaxf(m[nr][e], mx);
                    // -inf - (-inf) guard: an all-masked row keeps max -inf and uses 0 as its offset
                    const float mu = (mn == kNegInf) ? 0.f : mn;
                    al[nr][e] = fast_exp2(m[nr][e] - mu);
                    m[nr][e] = mn;
                    float rs = 0.f;
#pragma unroll
                    for (int hb = 0; hb < NB; ++hb) {
                        pv[hb][nr][e][0] = fast_exp2(x[hb][0] - mu);
                        pv[hb][nr][e][1] = fast_exp2(x[hb][1] - mu);
                        rs += pv[hb][nr][e][0] + pv[hb][nr][e][1];
                    }
                    l[nr][e] = l[nr][e] * al[nr][e] + rs;
                    moved |= al[nr][e] != 1.f;
                }
            }
            // P^T tiles (rows: keys g / g + 8; columns: rows 2 tq, 2 tq + 1), high f16 part and
            // remainder, transposed into the B operand layout (keys along k)
#pragma unroll
            for (int hb = 0; hb < NB; ++hb)
#pragma unroll
                for (int nr = 0; nr < NR; ++nr) {
                    const uint32_t h0 = Op::pack(pv[hb][nr][0][0], pv[hb][nr][1][0]);
                    const uint32_t h1 = Op::pack(pv[hb][nr][0][1], pv[hb][nr][1][1]);
                    const float2 u0 = Op::unpack(h0), u1 = Op::unpack(h1);
                    const uint32_t r0 = Op::pack(pv[hb][nr][0][0] - u0.x, pv[hb][nr][1][0] - u0.y);
                    const uint32_t r1 = Op::pack(pv[hb][nr][0][1] - u1.x, pv[hb][nr][1][1] - u1.y);
                    pb[hb][nr][0][0] = movmatrix_trans(h0);
                    pb[hb][nr][0][1] = movmatrix_trans(h1);
                    pb[hb][nr][1][0] = movmatrix_trans(r0);
                    pb[hb][nr][1][1] = movmatrix_trans(r1);
                }
            if (__any_sync(0xffffffffu, moved)) {  // a running max moved: rescale O
#pragma unroll
                for (int nr = 0; nr < NR; ++nr)
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        acc[nr][mt][0] *= al[nr][0];
                        acc[nr][mt][1] *= al[nr][1];
                        acc[nr][mt][2] *= al[nr][0];
                        acc[nr][mt][3] *= al[nr][1];
                    }
            }
        }
        if constexpr (!kEarly) {
            if (!bad) {
                const bool ok = mbar_wait(bar_fv + 8 * st, par, p.err);
                bad = __any_sync(0xffffffffu, !ok);
            }
            if (!bad && active) read_v();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_em + 8 * st);  // K and V of the stage are read: free it
        }
        if (!bad && active) {
#pragma unroll
            for (int hb = 0; hb < NB; ++hb) {
                // Keys at or past k_hi hold whatever the ring held before: zero V rows keep 0 x NaN out.
#pragma unroll
                for (int kh = 0; kh < 2; ++kh)
                    if (tile_k0 + kw0 + 16 * hb + g + 8 * kh >= k_hi)
#pragma unroll
                        for (int i = 0; i < D / 16; ++i) vw[hb][kh][i] = 0u;
                // ---- O^T += v_scale x V^T (Ph + Pl)^T over the block's 16 keys.  Head-dim tile mt takes
                // this lane's bytes 4 mt + {0..3} of keys g and g + 8: four 8 x 8 blocks (keys x 2-byte
                // d slots) which movmatrix turns into the A operand (d x keys), so output row m of the
                // tile is head-dim index out_d(mt, m) (see the merge below).
                const float vsc = s_vs[slot][(kw0 + 16 * hb) >> ps_shift];
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    uint32_t x00, x01, x10, x11;  // [key half][d slot half]
                    q8x4_to_f16x4<FMT>(vw[hb][0][mt], x00, x01);
                    q8x4_to_f16x4<FMT>(vw[hb][1][mt], x10, x11);
                    const uint32_t a[4] = {movmatrix_trans(x00), movmatrix_trans(x01), movmatrix_trans(x10),
                                           movmatrix_trans(x11)};
#pragma unroll
                    for (int nr = 0; nr < NR; ++nr) {
                        float tt[4] = {0.f, 0.f, 0.f, 0.f};
                        Op::run(tt, a, pb[hb][nr][0][0], pb[hb][nr][0][1]);
                        Op::run(tt, a, pb[hb][nr][1][0], pb[hb][nr][1][1]);
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[nr][mt][e] = fmaf(vsc, tt[e], acc[nr][mt][e]);
                    }
                }
            }
        }
    }

    // row sums over the 8 key lanes of each row
#pragma unroll
    for (int nr = 0; nr < NR; ++nr)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            l[nr][e] += __shfl_xor_sync(0xffffffffu, l[nr][e], 4);
            l[nr][e] += __shfl_xor_sync(0xffffffffu, l[nr][e], 8);
            l[nr][e] += __shfl_xor_sync(0xffffffffu, l[nr][e], 16);
        }
    // ---- merge the four warps' states through shared memory (reuses the ring and the rows)
    constexpr int ACC_STRIDE = D + 4;
    float *sm = reinterpret_cast<float *>(smem_raw + (sbase - raw));
    named_bar_sync(1, kMmaConsumerWarps * 32);  // every warp is done reading the ring and the rows
    {
        float *wa = sm + warp * 16 * ACC_STRIDE;
        float *s_m = sm + kMmaConsumerWarps * 16 * ACC_STRIDE;
        float *s_l = s_m + kMmaConsumerWarps * 16;
#pragma unroll
        for (int nr = 0; nr < NR; ++nr) {
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    // tile row g holds head-dim index out_d(mt, g) = (g / 2) D/4 + 4 mt + (g % 2),
                    // tile row g + 8 the index two above it
                    const int r = nr * 8 + 2 * tq + e;
                    const int d0 = (g >> 1) * (D / 4) + 4 * mt + (g & 1);
                    wa[r * ACC_STRIDE + d0] = acc[nr][mt][e];
                    wa[r * ACC_STRIDE + d0 + 2] = acc[nr][mt][2 + e];
                }
            if (g == 0) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    s_m[warp * 16 + nr * 8 + 2 * tq + e] = m[nr][e];
                    s_l[warp * 16 + nr * 8 + 2 * tq + e] = l[nr][e];
                }
            }
        }
    }
    named_bar_sync(1, kMmaConsumerWarps * 32);
    if (!bad) decode_merge_store<T, D>(p, sm, sq, kvh, s, 0, rows);
}

// ============================================================================ prefill
// More than 16 query rows: 64-row tiles, each consumer warp owning 16 rows over all 64 keys of a
// stage (S = Q K^T, O = P V); V rows are widened once per stage by the four warps together.
template <typename T, int FMT, int D, int NSTAGE>
__global__ void __launch_bounds__(kMmaThreads, 2)
    paged_attn_kvq_prefill_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                                  const FwdParams p, int ps_shift) {
    using Op = MmaOp<__half>;
    constexpr int kStage8 = Geo8<D>::kStage8;
    constexpr int KB = 32;      // keys per softmax block
    constexpr int SUBS = 2;     // blocks per stage
    constexpr int NTB = KB / 8; // score n-tiles per block
    constexpr int kSlots = 2 * NSTAGE;

    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[3 * NSTAGE];
    __shared__ float s_ks[kSlots][kMaxPagesPerStage];
    __shared__ float s_vs[kSlots][kMaxPagesPerStage];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int unit = blockIdx.x;
    const int rt = unit % p.row_tiles;
    unit /= p.row_tiles;
    const int kvh = unit % p.Hkv;
    unit /= p.Hkv;
    const int s = unit % p.split_kv;
    const int b = unit / p.split_kv;
    const KvqUnit u = kvq_unit(p, b, s, ps_shift);
    const SeqRows sq = uniform_seq(p, b);
    const int row0 = rt * kPrefillRows;
    const int row_end = min(row0 + kPrefillRows, p.rows);
    // causal reach grows with the query index, so the tile's last row reaches furthest
    const int k_hi = min(u.k_hi_split, row_key_limit(p, b, u.L, (row_end - 1) / p.G));
    const int n_tiles = k_hi > u.k_lo ? (k_hi - u.k_lo + kMmaTileKeys - 1) / kMmaTileKeys : 0;
    if (n_tiles == 0) {
        if (warp < kMmaConsumerWarps) store_empty_unit<T, D>(p, sq, kvh, s, row0, row_end);
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
        kvq_produce<D, NSTAGE, kMmaTileKeys>(&tmK, &tmV, p, b, kvh, u.pg0, k_hi, n_tiles, ps_shift, sbase, bar_fk,
                                             bar_fv, bar_em, s_ks, s_vs, lane);
        return;
    }

    // ==================================================================== consumers
    const int g = lane >> 2;
    const int tq = lane & 3;
    const int ra = row0 + warp * 16 + g, rb = ra + 8;
    const int kw0 = warp * 16;  // the stage keys whose V rows this warp widens
    // Q fragments (A operand) in f16 over the permuted head-dim order: step kk takes elements
    // tq D/4 + 4 kk + {0, 1} (a0 / a1) and + {2, 3} (a2 / a3) of rows ra / rb.
    uint32_t qf[D / 16][4];
    float q_inv_a, q_inv_b;
    {
        uint32_t wa[D / 8], wb[D / 8];
        const T *q = reinterpret_cast<const T *>(p.q);
        const bool va = ra < p.rows, vb = rb < p.rows;
        load_q_row<T, D>(q + (va ? q_row_offset(p, out_row_index(p, sq, kvh, ra)) : 0), va, tq, wa, q_inv_a);
        load_q_row<T, D>(q + (vb ? q_row_offset(p, out_row_index(p, sq, kvh, rb)) : 0), vb, tq, wb, q_inv_b);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            qf[kk][0] = wa[2 * kk];
            qf[kk][1] = wb[2 * kk];
            qf[kk][2] = wa[2 * kk + 1];
            qf[kk][3] = wb[2 * kk + 1];
        }
    }
    const int lim_a = ra < p.rows ? min(u.k_hi_split, row_key_limit(p, b, u.L, ra / p.G)) : u.k_lo;
    const int lim_b = rb < p.rows ? min(u.k_hi_split, row_key_limit(p, b, u.L, rb / p.G)) : u.k_lo;
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
        const int tile_k0 = u.k_lo + t * kMmaTileKeys;

        if (!bad) {
            const bool ok = mbar_wait(bar_fk + 8 * st, par, p.err);
            bad = __any_sync(0xffffffffu, !ok);
        }
        named_bar_sync(1, kMmaConsumerWarps * 32);  // every warp is done with the previous V rows
        if (!bad) {
            const bool ok = mbar_wait(bar_fv + 8 * st, par, p.err);
            bad = __any_sync(0xffffffffu, !ok);
        }
        if (!bad) widen_keys<FMT, D>(vring, wideV, kw0, k_hi - tile_k0, lane);
        named_bar_sync(1, kMmaConsumerWarps * 32);  // the stage's V rows are complete

#pragma unroll
        for (int sb = 0; sb < SUBS; ++sb) {
            const int kb0 = sb * KB;                                   // first key (in the stage) of the block
            const bool active = tile_k0 + kb0 < min(k_hi, warp_lim);   // warp-uniform
            if (bad || !active) continue;
            // ---- S = Q K^T over the block's KB keys, K converted from the ring
            float sc[NTB][4];
#pragma unroll
            for (int n = 0; n < NTB; ++n) {
                sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
                uint32_t bk[D / 16][2];
                load_k_frags<FMT, D>(kring, kb0 + n * 8 + g, tq, bk);
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
            // P split into an f16 high part and its rounding remainder
            uint32_t ph[NTB][2], pl[NTB][2];
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
            if (__any_sync(0xffffffffu, al_a != 1.f || al_b != 1.f)) {  // a running max moved
#pragma unroll
                for (int n = 0; n < D / 8; ++n) {
                    acc[n][0] *= al_a;
                    acc[n][1] *= al_a;
                    acc[n][2] *= al_b;
                    acc[n][3] *= al_b;
                }
            }
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
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_em + 8 * st);  // K of the whole stage read, V widened
    }

    // quad sums of the row sums (alpha is uniform across a quad)
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
    if (!bad) finish_prefill_rows<T, D>(p, sq, kvh, s, ra, rb, row_end, tq, m_a, m_b, l_a, l_b, acc);
}

// ------------------------------------------------------------------------ host side
static constexpr int kvq_prefill_stages(int D) { return D == 128 ? 4 : 6; }

// ring (+ the widened V rows of the prefill kernel) + alignment slack
static constexpr size_t kvq_smem_bytes(int D, int nstage, bool wide_v) {
    return (size_t)nstage * 2 * kMmaTileKeys * D + (wide_v ? (size_t)kMmaTileKeys * D * 2 : 0) + 1024;
}

static int ps_shift_of(int ps) {
    int sh = 0;
    while ((1 << sh) < ps) ++sh;
    return sh;
}

// Decode shape: KPW keys per consumer warp and stage (stages of 4 KPW keys), NSTAGE-deep ring,
// MINB CTAs per SM.
template <typename T, int FMT, int D, int NR, int KPW, int NSTAGE, int MINB>
static cudaError_t launch_kvq_decode(const FwdParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                     cudaStream_t stream) {
    constexpr size_t smem = (size_t)NSTAGE * 2 * kMmaConsumerWarps * KPW * D + 1024;
    static_assert(merge_scratch_bytes(D) + 1024 <= smem, "decode merge scratch must fit in the ring");
    auto kern = paged_attn_kvq_decode_kernel<T, FMT, D, NR, NSTAGE, KPW, MINB>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const long long units = (long long)p.B * p.split_kv * p.Hkv;
    if (units <= 0) return cudaSuccess;
    if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)units, kMmaThreads, smem, stream>>>(tmk, tmv, p, ps_shift_of(p.ps));
    return cudaGetLastError();
}

template <typename T, int FMT, int D>
static cudaError_t launch_kvq_prefill(const FwdParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                      cudaStream_t stream) {
    constexpr int NSTAGE = kvq_prefill_stages(D);
    constexpr size_t smem = kvq_smem_bytes(D, NSTAGE, true);
    auto kern = paged_attn_kvq_prefill_kernel<T, FMT, D, NSTAGE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const long long units = (long long)p.B * p.split_kv * p.Hkv * p.row_tiles;
    if (units <= 0) return cudaSuccess;
    if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)units, kMmaThreads, smem, stream>>>(tmk, tmv, p, ps_shift_of(p.ps));
    return cudaGetLastError();
}

template <typename T, int FMT, int D>
static cudaError_t launch_kvq_d(const FwdParams &p, int mode, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                cudaStream_t stream) {
    if (mode == MODE_PREFILL) return launch_kvq_prefill<T, FMT, D>(p, tmk, tmv, stream);
    // 16 keys per warp and stage, 4 (D = 128) or 8 (D = 64) 64-key stages: 65 KiB, so 3 CTAs per SM
    // for <= 8 rows.  Measured on the FP8 Llama-3-8B decode: 32 keys per warp (two blocks sharing one
    // softmax step) with 2 or 3 stages, and 6 stages at 2 CTAs per SM, were no faster.
    if (p.rows <= 8) return launch_kvq_decode<T, FMT, D, 1, 16, (D == 128 ? 4 : 8), 3>(p, tmk, tmv, stream);
    return launch_kvq_decode<T, FMT, D, 2, 16, (D == 128 ? 4 : 8), 2>(p, tmk, tmv, stream);
}

template <int FMT>
static cudaError_t launch_kvq_fmt(const FwdParams &p, int mode, int dtype, const CUtensorMap &tmk,
                                  const CUtensorMap &tmv, cudaStream_t stream) {
    if (dtype == PA_BF16) {
        return p.D == 128 ? launch_kvq_d<__nv_bfloat16, FMT, 128>(p, mode, tmk, tmv, stream)
                          : launch_kvq_d<__nv_bfloat16, FMT, 64>(p, mode, tmk, tmv, stream);
    }
    return p.D == 128 ? launch_kvq_d<__half, FMT, 128>(p, mode, tmk, tmv, stream)
                      : launch_kvq_d<__half, FMT, 64>(p, mode, tmk, tmv, stream);
}

cudaError_t launch_mma_kvq(const FwdParams &p, int mode, int dtype, int kv_dtype, const CUtensorMap &tmk,
                           const CUtensorMap &tmv, cudaStream_t stream) {
    if (kv_dtype == PA_INT8) return launch_kvq_fmt<kFmtInt8>(p, mode, dtype, tmk, tmv, stream);
    return launch_kvq_fmt<kFmtE4M3>(p, mode, dtype, tmk, tmv, stream);
}

}  // namespace pa
