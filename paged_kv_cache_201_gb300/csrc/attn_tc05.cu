// Paged attention on the 5th-generation tensor cores (tcgen05 + tensor memory), sm_103a.
//
// For query runs long enough to fill a 128-row tile (prefill, head_dim 128, bf16/f16).
// A work unit = (sequence b, kv head, split s, tile of 128/G query tokens x the G query heads of
// the kv head's group), so all 128 rows share every K/V tile.  The kernel is persistent: one CTA
// per SM takes units until none is left.  With split_kv = 1 the grid has one CTA per unit, of which
// one fits an SM; a running CTA takes the next unit by cancelling the launch of a CTA that has not
// started (cluster launch control), so units go, in CTA order, to whichever SM frees up first, and
// that order puts the most key tiles first: the sequences by key count, longest first, each from
// its last row tile down.  Lane 0 of warp 0 takes the units and posts each to an 8-entry
// shared-memory ring that every other role reads.  Otherwise (split_kv > 1, whose units include
// long runs of empty ones, and variable-length batches) CTA c takes units c, c + gridDim.x, ...,
// each role walking them by itself.  Four warpgroups:
//   warps 0,2   TMA producers (0: Q and K, 2: V): each unit's Q tile (double-buffered), then per 128-key
//               tile the block-table ids (32 pages per batch, never past the sequence's page count)
//               and one box per page, half-row and pool into 2-slot K and V rings.  From the ring they
//               take the next unit only once every load of the current one is out (a post waits for
//               the readers of an older entry, which may need those loads); the static walk takes it
//               one unit ahead.
//   warp 1      allocates all 512 TMEM columns and issues tcgen05.mma from one thread:
//               S_g = Q K_g^T into one of two S buffers (128 fp32 columns each), then
//               O += Ph_{g-1} V_{g-1} + Pl_{g-1} V_{g-1} with P read from TMEM into one of two O
//               buffers (one per unit, alternating).
//   warp 3      V gate: clears the V rows of a unit's last tile that lie past its last valid key
//               (they may hold any bits, and a zero weight times NaN is NaN), then releases the slot
//               to the P V product (one barrier with the softmax's P).
//   warps 4-11  softmax, two threads per TMEM lane (query row), 64 columns each: mask (sequence
//               length, split end, causal reach with q_offset), running max in the log2 domain,
//               P = exp2(s - m) written back over S as a 16-bit high part (bf16: p truncated to
//               its top 16 bits) and its remainder (at split 1 every high part first, on its
//               own barrier).  O is rescaled
//               in TMEM only when the running max grows by more than 2^8 (otherwise the stale max
//               is kept), and the -inf - (-inf) guard of rocMLIR PR #2371 applies.  At a unit's
//               end they hand its row maximum and sum over.
//   warps 12-15 epilogue: one thread per query row reads the unit's O out of TMEM, divides by the
//               row sum (0/0 guard), stages the rows in shared memory and stores them with TMA (the
//               log-sum-exp with plain stores), while the softmax warps already work on the next
//               unit.
// The register file is split with setmaxnreg: 64 per thread for warps 0-3, 176 for the softmax
// warpgroups, 96 for the epilogue (128 x (64 + 2 x 176 + 96) = the 65536 of a 512 x 128 launch).
// Instantiations: PART (split_kv > 1's fp32 partials, or the final rows) x VARLEN (a batch of
// sequences with their own query counts, whose units are blocks of the packed rows).  The row
// maximum is taken over unscaled scores, so the host launches this kernel only for scale > 0.
#include <atomic>
#include <type_traits>

#include "kernels.h"
#include "tc05.cuh"

namespace pa {

namespace {

constexpr int kT5Threads = 512;               // 16 warps, four warpgroups
constexpr uint32_t kRegLoad = 64, kRegSoftmax = 176, kRegEpilogue = 96;  // per thread, see above
constexpr int kT5LaunchRegs = 128;            // registers per thread the launch must hold
static_assert(128 * (kRegLoad + 2 * kRegSoftmax + kRegEpilogue) <= kT5Threads * kT5LaunchRegs,
              "the register split must fit the launch");
constexpr int kT5Half = 128 * 128;            // bytes of one 64-column half of a 128-row tile
constexpr int kT5Tile = 2 * kT5Half;          // a 128 x 128 bf16 tile (Q, K or V)
constexpr int kT5Stage = 32 * 128;            // one epilogue warp's output staging: 32 rows x 128 bytes
constexpr uint32_t kT5TmemCols = 512;
constexpr uint32_t kColO = 256;               // O buffers at columns 256 and 384
constexpr float kRescaleLog2 = 8.f;           // rescale O only when the max grows by > 2^8
constexpr int kT5StageLens = 1024;            // batches up to this size keep seq_lens / q_offset in smem
constexpr int kT5SortMax = 256;               // batches up to this size are ordered by key count
constexpr int kT5Ring = 8;                    // entries of the unit ring (a power of two)
// ring readers' arrivals per entry: lane 0 of warps 2 and 3, the MMA thread, 8 softmax and 4 epilogue warps
constexpr uint32_t kT5RingReaders = 15;

// barrier slots (pairs are indexed by buffer / ring slot); each commit costs the MMA thread issue
// time, so one completion serves every waiter that needs it:
//   QF/QE  Q buffer full (TMA) / empty (after the unit's last Q K^T)
//   KF/KE  K ring slot full (TMA) / Q K^T of its tile done: the slot is free, and the S buffer of
//          the same index holds the scores (the softmax waits on it too)
//   VF/VE  V ring slot full (TMA) / P V of its tile done: the slot is free, and O holds that
//          tile's product (the softmax waits on it before rescaling O).  Every such wait is at
//          most one phase behind: the barrier's next phase needs the waiter's own later work.
//   PF     P written back over the S buffer (256 softmax threads arrive; at split 1 its high parts
//          only) and the V slot of the same index cleared past the unit's last key, where needed
//          (32 V-gate threads arrive)
//   PL     at split 1 (bf16), P's remainders written (256 softmax threads arrive)
//   OF     once per use of an O buffer, after the unit's last P V
//   OFREE  O buffer read out by the epilogue threads (128 arrive)
//   LF/LE  a unit's row maxima and sums handed to the epilogue (256 softmax threads arrive) / read
//          by it (128 epilogue threads arrive); indexed like the O buffers
//   RF/RE  unit ring entry written (warp 0) / read by every reader (kT5RingReaders arrive)
//   CLC    the response to a launch-cancel request has landed (16 bytes)
enum {
    B_QF = 0, B_QE = 2, B_KF = 4, B_KE = 6, B_VF = 8, B_VE = 10, B_PF = 12, B_OF = 14, B_OFREE = 16, B_LF = 18,
    B_LE = 20, B_PL = 22, B_RF = 24, B_RE = B_RF + kT5Ring, B_CLC = B_RE + kT5Ring, B_COUNT = B_CLC + 1
};

// Cluster launch control (sm_100 family): ask to cancel the launch of a CTA that has not started;
// the 16-byte response lands at `resp` and completes 16 bytes of transactions on `bar`.
__device__ __forceinline__ void clc_try_cancel(uint32_t resp, uint32_t bar) {
    asm volatile("clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 [%0], [%1];" ::"r"(
                     resp),
                 "r"(bar)
                 : "memory");
}
// Whether the request whose response is at `resp` cancelled a CTA, and if so its blockIdx.x.
__device__ __forceinline__ bool clc_query(uint32_t resp, int &cta) {
    uint32_t ok, x = 0;
    asm volatile(
        "{\n\t.reg .b128 h;\n\t.reg .pred p;\n\t"
        "ld.shared.b128 h, [%2];\n\t"
        "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, h;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t"
        "@p clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, h;\n\t}"
        : "=r"(ok), "+r"(x)
        : "r"(resp)
        : "memory");
    cta = (int)x;
    return ok != 0;
}

// Named barrier over `count` threads that also ANDs a predicate across them.
__device__ __forceinline__ bool named_bar_and(int id, int count, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// Output row of query token tok (of the sequence whose first packed token is q0) and head kvh G + g.
__device__ __forceinline__ long long t5_row_index(const FwdParams &p, int q0, int kvh, int tok, int g) {
    return ((long long)q0 + tok) * p.Hq + (long long)kvh * p.G + g;
}

// The log-sum-exp of one row: the final one (split_kv = 1, if wanted) or split s's.
template <bool PART>
__device__ __forceinline__ void t5_store_lse(const FwdParams &p, int s, long long ridx, float lse) {
    if constexpr (!PART) {
        if (p.lse) p.lse[ridx] = lse;
    } else {
        p.lse[(long long)s * p.rows_total + ridx] = lse;
    }
}

}  // namespace

// P V with P split into a 16-bit high part and its rounding remainder (two products) for bf16; f16
// rounds P to 2^-11 relative (p in [0, 1]), well inside the tolerance, so one product is enough.
template <typename T>
__host__ __device__ constexpr bool t5_split_p() { return !std::is_same<T, __half>::value; }

// P for 32 keys of one row: p = exp2(s * c2 + nmu), where the caller has set the scores of masked
// keys to -inf (c2 > 0, so their p is exactly 0: one code path for every tile keeps the loop small
// in the instruction cache); l accumulates the p; the 32 columns at `taddr` receive [16 columns of
// high parts | 16 columns of remainders] (bf16/f16 pairs; the remainders only when t5_split_p<T>()).
// Packed pairs of fp32 (the f32x2 arithmetic of sm_100-family cores: one instruction per pair,
// each lane rounded as its scalar counterpart).
__device__ __forceinline__ uint64_t f2_pack(float x, float y) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
    return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

template <typename T>
__device__ __forceinline__ void t5_exp_chunk(const uint32_t (&u)[32], float c2, float nmu, float &l, uint32_t taddr) {
    uint32_t hi[16], lo[16];
    const uint64_t c2x2 = f2_pack(c2, c2), nmux2 = f2_pack(nmu, nmu);
    uint64_t l2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};  // two pair sums: short dependency chains
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint64_t sc = f2_pack(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1]));
        const float2 x = f2_unpack(f2_fma(sc, c2x2, nmux2));
        const float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
        const uint64_t pp = f2_pack(p0, p1);
        l2[i & 1] = f2_add(l2[i & 1], pp);
        if (t5_split_p<T>()) {
            // bf16: the high parts truncated (the top 16 bits of each p); p - hi is then exact in
            // fp32 and below 2^-7 p, and its bf16 rounding leaves P within 2^-16 of p
            hi[i] = __byte_perm(__float_as_uint(p0), __float_as_uint(p1), 0x7632);
            const uint64_t h2 = f2_pack(__uint_as_float(__float_as_uint(p0) & 0xffff0000u),
                                        __uint_as_float(__float_as_uint(p1) & 0xffff0000u));
            const float2 d = f2_unpack(f2_sub(pp, h2));
            lo[i] = MmaOp<T>::pack(d.x, d.y);
        } else {
            hi[i] = MmaOp<T>::pack(p0, p1);
        }
    }
    const float2 ls = f2_unpack(f2_add(l2[0], l2[1]));
    l += ls.x + ls.y;
    tc05::st_16cols(taddr, hi);
    if (t5_split_p<T>()) tc05::st_16cols(taddr + 16u, lo);
}

// The same in two passes (the split-1 schedule releases P's high parts before the remainders).
// Pass 1 over 32 keys of one row: p = exp2(s * c2 + nmu), where the caller has set the scores of
// masked keys to -inf (c2 > 0, so their p is exactly 0); l accumulates the p, u is overwritten with
// the p (fp32 bits), and their 16-bit high parts go to the first 16 of the 32 columns at `taddr`.
template <typename T>
__device__ __forceinline__ void t5_exp_hi(uint32_t (&u)[32], float c2, float nmu, float &l, uint32_t taddr) {
    uint32_t hi[16];
    const uint64_t c2x2 = f2_pack(c2, c2), nmux2 = f2_pack(nmu, nmu);
    uint64_t l2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};  // two pair sums: short dependency chains
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint64_t sc = f2_pack(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1]));
        const float2 x = f2_unpack(f2_fma(sc, c2x2, nmux2));
        const float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
        l2[i & 1] = f2_add(l2[i & 1], f2_pack(p0, p1));
        // bf16: the high parts truncated (the top 16 bits of each p), so that pass 2 finds them with a
        // mask; the remainder p - hi is then exact in fp32 and below 2^-7 p
        hi[i] = t5_split_p<T>() ? __byte_perm(__float_as_uint(p0), __float_as_uint(p1), 0x7632) : MmaOp<T>::pack(p0, p1);
        u[2 * i] = __float_as_uint(p0);
        u[2 * i + 1] = __float_as_uint(p1);
    }
    const float2 ls = f2_unpack(f2_add(l2[0], l2[1]));
    l += ls.x + ls.y;
    tc05::st_16cols(taddr, hi);
}

// Pass 2 (bf16): the remainders p - hi of the same 32 keys (hi = p with its low 16 bits cleared,
// as pass 1 stored it), rounded to bf16, into the last 16 columns.
template <typename T>
__device__ __forceinline__ void t5_exp_lo(const uint32_t (&u)[32], uint32_t taddr) {
    uint32_t lo[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint64_t h2 =
            f2_pack(__uint_as_float(u[2 * i] & 0xffff0000u), __uint_as_float(u[2 * i + 1] & 0xffff0000u));
        const float2 d = f2_unpack(f2_sub(f2_pack(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1])), h2));
        lo[i] = MmaOp<T>::pack(d.x, d.y);
    }
    tc05::st_16cols(taddr + 16u, lo);
}

// Everything a role needs to know about one work unit; every role derives it the same way.
// q0: the sequence's first packed query token, Sq its query count; skip: a unit of the
// variable-length launch that is not this kernel's (no loads, no product, no output).
struct T5Unit {
    int b, kvh, s, L, k_lo, k_hi_split, k_hi, pg0, tok0, tok_end, n_tiles, q0, Sq;
    bool skip;
};

// seq_lens / q_offset as staged by the CTA (shared memory when the batch fits, else global).
struct T5Lens {
    const int32_t *seq_lens;
    const int32_t *q_offset;  // null: seq_lens[b] - Sq
};

__device__ __forceinline__ int t5_key_limit(const FwdParams &p, const T5Lens &ln, int b, int L, int Sq, int i) {
    if (!p.causal) return L;
    const long long qoff = ln.q_offset ? (long long)ln.q_offset[b] : (long long)L - Sq;
    long long reach = qoff + i + 1;
    reach = reach < 0 ? 0 : reach;
    return (int)(reach < L ? reach : L);
}

// A unit's digits: sequence b (in a variable-length batch, block b of the packed rows), split s,
// kv head kvh, row tile rt.  The static walk's unit order is
// unit = ((b * split_kv + s) * Hkv + kvh) * row_tiles + rt, and every role walks its CTA's units c,
// c + gridDim.x, ... by adding gridDim.x's own digits with one carry per digit (no division per
// unit: the per-unit code stays small, so it does not push the softmax's loop out of the
// instruction cache).
struct T5Pos {
    int rt, kvh, s, b;
};

__device__ __forceinline__ T5Pos t5_pos(const FwdParams &p, int unit) {
    T5Pos u;
    u.rt = unit % p.row_tiles;
    unit /= p.row_tiles;
    u.kvh = unit % p.Hkv;
    unit /= p.Hkv;
    u.s = unit % p.split_kv;
    u.b = unit / p.split_kv;
    return u;
}

// u += d, for d's digits each below its radix; u.b at or past the b digit's count past the last unit.
__device__ __forceinline__ void t5_advance(const FwdParams &p, T5Pos &u, const T5Pos &d) {
    u.rt += d.rt;
    int c = u.rt >= p.row_tiles;
    if (c) u.rt -= p.row_tiles;
    u.kvh += d.kvh + c;
    c = u.kvh >= p.Hkv;
    if (c) u.kvh -= p.Hkv;
    u.s += d.s + c;
    c = u.s >= p.split_kv;
    if (c) u.s -= p.split_kv;
    u.b += d.b + c;
}

// The cancelled-CTA schedule (split_kv = 1): the unit of CTA r.  Sequences by key count, longest
// first (perm; null: the last sequence first), each from its last row tile down with the kv heads
// of a row tile side by side, so a sequence's units come in falling order of key tiles: the
// longest start first and the short ones fill in at the end.
__device__ __forceinline__ T5Pos t5_dyn_pos(const FwdParams &p, int r, const int16_t *perm) {
    T5Pos u;
    u.kvh = r % p.Hkv;
    r /= p.Hkv;
    const int ri = r % p.row_tiles;
    const int bi = r / p.row_tiles;
    u.rt = p.row_tiles - 1 - ri;
    u.s = 0;
    u.b = perm ? (int)perm[bi] : p.B - 1 - bi;
    return u;
}

// Variable-length batches (at most kT5StageLens sequences): q_start staged in shared memory by
// the CTA (a fixed address, so reading it costs the softmax warps no pointer register).
__shared__ int32_t t5_qstart[kT5StageLens + 1];
static_assert(kTc05VarlenMaxBatch <= kT5StageLens, "the host's variable-length batch limit must fit the stage");
// The sequences by key count, longest first (batches of at most kT5SortMax sequences).
__shared__ int16_t t5_perm[kT5SortMax];
static_assert(kT5SortMax <= kT5StageLens, "the order is taken over staged sequence lengths");

// The packed rows are cut into blocks, sequence b's first being floor(q_start[b] G / 128) + b
// (strictly increasing, and at least as many blocks as the sequence has 128-row tiles before the
// next one starts).  Block blk belongs to the largest such b.
__device__ __forceinline__ long long t5_first_block(int b, int g_shift) {
    return (((long long)t5_qstart[b]) << g_shift >> 7) + b;
}

template <bool VARLEN>
__device__ __forceinline__ T5Unit t5_unit(const FwdParams &p, const T5Lens &ln, const T5Pos &q, int tpt,
                                          int ps_shift, int g_shift) {
    T5Unit U;
    const int ps = 1 << ps_shift;
    int rt;
    U.kvh = q.kvh;
    U.s = q.s;
    U.skip = false;
    if constexpr (VARLEN) {
        // the b digit is the block: find its sequence (binary search on the first blocks)
        int lo = 0, hi = p.B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (t5_first_block(mid, g_shift) <= q.b) lo = mid;
            else hi = mid - 1;
        }
        U.b = lo;
        U.q0 = t5_qstart[lo];
        const int q1 = t5_qstart[lo + 1];
        U.Sq = q1 - U.q0;
        rt = (int)(q.b - t5_first_block(lo, g_shift));
        // an invalid q_start entry (the one-grid kernel flags it), a sequence of fewer than 64
        // query rows (the one-grid kernel takes it) or a block past the sequence's tiles
        U.skip = U.q0 < 0 || U.Sq < 0 || (long long)q1 * p.Hq > p.rows_total || (U.Sq << g_shift) < 64 || rt < 0 ||
                 rt >= ((U.Sq + tpt - 1) >> (7 - g_shift));
        if (U.skip) {
            U.n_tiles = 0;
            return U;
        }
    } else {
        rt = q.rt;
        U.b = q.b;
        U.Sq = p.Sq;
        U.q0 = q.b * p.Sq;
    }
    U.L = min(max(ln.seq_lens[U.b], 0), p.W * ps);
    // the split plan of split_pages, with the page count by shift
    const int nblk = (U.L + ps - 1) >> ps_shift;
    const int per = (nblk + p.split_kv - 1) / p.split_kv;
    const long long a = (long long)U.s * per, e = (long long)(U.s + 1) * per;
    U.pg0 = (int)(a < nblk ? a : nblk);
    const int pg1 = (int)(e < nblk ? e : nblk);
    U.k_lo = U.pg0 * ps;
    U.k_hi_split = min(pg1 * ps, U.L);
    U.tok0 = rt * tpt;
    U.tok_end = min(U.tok0 + tpt, U.Sq);
    U.k_hi = min(U.k_hi_split, t5_key_limit(p, ln, U.b, U.L, U.Sq, U.tok_end - 1));
    U.n_tiles = U.k_hi > U.k_lo ? (U.k_hi - U.k_lo + 127) / 128 : 0;
    return U;
}

// Persistent: a CTA takes units until none is left (the schedule at the top of the file; DYN: by
// cancelling CTAs, the grid then holding one CTA per unit).  Barrier phases and the K / V rings run
// on the CTA's global tile counter g; Q and O are double-buffered by the CTA's count of non-empty
// units n, so a unit's read-out and the next unit's loads overlap its neighbours' work.  PART: the
// output is split_kv > 1's fp32 partials (else the final rows in T); one store path per kernel keeps
// the code the SM must hold small.  G = 2^g_shift (it divides 128).  VARLEN: a variable-length
// batch (q_start), whose sequences of at least 64 query rows this kernel takes; the unit order's
// b digit is then the block of the packed rows (nb of them), and row_tiles is 1.  units: the unit
// count, nb * split_kv * Hkv * row_tiles.
template <typename T, bool PART, bool VARLEN>
__global__ void __launch_bounds__(kT5Threads, 1)
    paged_attn_tc05_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                           const FwdParams p, int tpt, int ps_shift, int g_shift, uint32_t idesc_qk,
                           uint32_t idesc_pv, int nb, int units) {
    constexpr bool DYN = !PART && !VARLEN;
    // In the split-1 schedule the softmax writes P in two passes (every high part, released on PF,
    // then every remainder, released on PL) and P V takes the high parts' products first: 3 %
    // faster there.  Next to the partial-output epilogue that larger code measured 5 % slower, so
    // the other schedules keep one pass per 32-key chunk (one copy run twice) and one release.
    constexpr bool kEarlyHi = DYN;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[B_COUNT];
    __shared__ int4 s_ring[kT5Ring];      // the unit ring: {rt, kvh, s, b}, b = -1 after the last unit
    __shared__ __align__(16) uint4 s_clc;  // the launch-cancel response
    __shared__ uint32_t s_tmem;
    __shared__ float s_xmax[2][2][128];   // [tile parity][column half][row]: partial row maxima
    __shared__ float s_lsum[2][2][128];   // [O buffer][column half][row]: a unit's partial row sums
    __shared__ float s_lmax[2][128];      // [O buffer][row]: a unit's running row maximum (log2 domain)
    __shared__ int32_t s_seqlen[kT5StageLens], s_qoff[kT5StageLens];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ps = 1 << ps_shift;

    // Every role walks every unit of this CTA and derives its bounds from seq_lens / q_offset: stage
    // them in shared memory once, so no unit waits on a global load for them.
    T5Lens ln{p.seq_lens, p.q_offset};
    if (p.B <= kT5StageLens) {
        for (int i = threadIdx.x; i < p.B; i += kT5Threads) {
            s_seqlen[i] = p.seq_lens[i];
            if (p.q_offset) s_qoff[i] = p.q_offset[i];
        }
        ln.seq_lens = s_seqlen;
        ln.q_offset = p.q_offset ? s_qoff : nullptr;
    }
    if constexpr (VARLEN)  // the host launches this kernel only for B <= kT5StageLens
        for (int i = threadIdx.x; i <= p.B; i += kT5Threads) t5_qstart[i] = p.q_start[i];

    // shared memory: Q x2 | K x2 | V x2 (128 x 128 tiles, two 64-column swizzled halves each)
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    auto sQ = [&](int qb) { return sbase + (uint32_t)kT5Tile * (uint32_t)qb; };
    auto sK = [&](int ks) { return sbase + (uint32_t)kT5Tile * (2u + (uint32_t)ks); };
    auto sV = [&](int vs) { return sbase + (uint32_t)kT5Tile * (4u + (uint32_t)vs); };
    auto bar = [&](int i) { return smem_u32(&bars[i]); };

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_QF + i), 1);
            mbar_init(bar(B_QE + i), 1);
            mbar_init(bar(B_KF + i), 1);
            mbar_init(bar(B_KE + i), 1);
            mbar_init(bar(B_VF + i), 1);
            mbar_init(bar(B_VE + i), 1);
            mbar_init(bar(B_PF + i), 256 + 32);
            mbar_init(bar(B_PL + i), 256);
            mbar_init(bar(B_OF + i), 1);
            mbar_init(bar(B_OFREE + i), 128);
            mbar_init(bar(B_LF + i), 256);
            mbar_init(bar(B_LE + i), 128);
        }
        for (int i = 0; i < kT5Ring; ++i) {
            mbar_init(bar(B_RF + i), 1);
            mbar_init(bar(B_RE + i), kT5RingReaders);
        }
        mbar_init(bar(B_CLC), 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        tc05::tmem_alloc(smem_u32(&s_tmem), kT5TmemCols);
        tc05::tmem_relinquish();
    }
    tc05::fence_before_sync();
    __syncthreads();
    tc05::fence_after_sync();
    const uint32_t tmem = s_tmem;
    const int wg = warp >> 2;

    // DYN: the sequences by key count (the clipped length), longest first, ties by index.
    const int16_t *perm = nullptr;
    if constexpr (DYN) {
        if (p.B <= kT5SortMax) {  // seq_lens staged
            const int cap = p.W * ps;
            for (int b = threadIdx.x; b < p.B; b += kT5Threads) {
                const int lb = min(max(ln.seq_lens[b], 0), cap);
                int rank = 0;
                for (int c = 0; c < p.B; ++c) {
                    const int lc = min(max(ln.seq_lens[c], 0), cap);
                    rank += (lc > lb) || (lc == lb && c < b);
                }
                t5_perm[rank] = (int16_t)b;
            }
            __syncthreads();
            perm = t5_perm;
        }
    }

    // Ring entry k (the CTA's k-th unit): 1 a unit (in q), 0 the end, -1 a time-out.  whole_warp:
    // every lane of the calling warp reads it (and agrees on a time-out); else one thread.
    auto ring_read = [&](int k, T5Pos &q, bool whole_warp) -> int {
        const int slot = k & (kT5Ring - 1);
        bool ok = mbar_wait(bar(B_RF + slot), (uint32_t)(k / kT5Ring) & 1u, p.err);
        if (whole_warp) ok = __all_sync(0xffffffffu, ok);
        if (!ok) return -1;
        const int4 e = s_ring[slot];
        if (whole_warp) __syncwarp();
        if (!whole_warp || lane == 0) mbar_arrive(bar(B_RE + slot));
        q = T5Pos{e.x, e.y, e.z, e.w};
        return e.w >= 0 ? 1 : 0;
    };
    // Static walk: gridDim.x's digits (gridDim.x <= the unit count, so b < nb here); each role's
    // cursor starts at the CTA's first unit.
    T5Pos step{};
    if constexpr (!DYN) step = t5_pos(p, gridDim.x);
    auto start = [&]() { return DYN ? T5Pos{} : t5_pos(p, blockIdx.x); };
    // A role's next unit: 1 a unit (in q), 0 none left, -1 a time-out.  DYN: ring entry k (whole_warp
    // as for ring_read); else the static walk from cursor c.
    auto walk = [&](int &k, T5Pos &c, T5Pos &q, bool whole_warp) -> int {
        if constexpr (DYN) {
            return ring_read(k++, q, whole_warp);
        } else {
            if (c.b >= nb) return 0;
            q = c;
            t5_advance(p, c, step);
            return 1;
        }
    };

    if (wg == 0) {
        tc05::setmaxnreg_dec<kRegLoad>();
        if (warp == 0 || warp == 2) {
            // ================================================================ TMA producers
            // warp 0 loads Q and K, warp 2 loads V: the two rings free at different times (K after
            // Q K^T, V after P V), so one must not wait behind the other.
            const bool kq = warp == 0;
            if (lane == 0) {
                if (kq) {
                    tma_prefetch_desc(&tmQ);
                    tma_prefetch_desc(&tmK);
                } else {
                    tma_prefetch_desc(&tmV);
                }
            }
            const int ppt = 128 >> ps_shift;                     // pages per tile (divides 32)
            const uint32_t box = (uint32_t)ps * 128u;            // bytes of one page half-row box
            bool bad = false;
            int n = 0, g0 = 0;                                   // non-empty units so far, global tile base
            // the first block-table batch of a unit
            auto first_ids = [&](const T5Unit &V) {
                const int pe = (V.k_hi + ps - 1) >> ps_shift;
                return (V.pg0 + lane < pe) ? __ldg(p.block_table + (long long)V.b * p.W + V.pg0 + lane) : 0;
            };
            // ---- DYN: warp 0 takes units (its own CTA's, then cancelled CTAs') and posts each, or the
            // end, to the ring; warp 2 reads them from it.  Both take the next unit only once every load
            // of the current one is out: a post waits for the ring's readers, and a reader of an older
            // entry may need those loads.
            int kr = 0;                                          // ring entries written (warp 0) / read (warp 2)
            bool own = true, clc_pending = false;                // warp 0, lane 0
            uint32_t clc_parity = 0;
            auto clc_request = [&]() {
                fence_proxy_async_smem();  // the previous response has been read (generic) before the async write
                mbar_arrive_expect_tx(bar(B_CLC), 16u);
                clc_try_cancel(smem_u32(&s_clc), bar(B_CLC));
                clc_pending = true;
            };
            // lane 0 of warp 0: the next CTA whose unit this CTA takes; -1: none left; -2: a time-out
            auto next_cta = [&]() -> int {
                if (own) {  // the CTA's own unit; ask for the next one at once
                    own = false;
                    clc_request();
                    return (int)blockIdx.x;
                }
                if (!clc_pending) return -1;
                if (!mbar_wait(bar(B_CLC), clc_parity, p.err)) return -2;
                clc_parity ^= 1u;
                clc_pending = false;
                int r;
                if (!clc_query(smem_u32(&s_clc), r)) return -1;  // no CTA left to cancel: no request after this
                clc_request();
                return r;
            };
            // ---- static: the walk of units c, c + gridDim.x, ..., the next unit with key tiles and its
            // first block-table batch taken one unit ahead
            T5Pos spos{};
            T5Unit sU{};
            int s_ids = 0;
            // the first unit with key tiles at or after position q (q.b >= nb: none), into V
            auto next_unit = [&](T5Pos q, T5Unit &V) {
                for (; q.b < nb; t5_advance(p, q, step)) {
                    V = t5_unit<VARLEN>(p, ln, q, tpt, ps_shift, g_shift);
                    if (V.n_tiles > 0) break;
                }
                return q;
            };
            if constexpr (!DYN) {
                spos = next_unit(t5_pos(p, blockIdx.x), sU);
                s_ids = spos.b < nb ? first_ids(sU) : 0;
            }
            // the CTA's next unit with key tiles and its first ids (false: none left, or a wait gave up)
            auto next_work = [&](T5Unit &V, int &ids) -> bool {
                if (bad) return false;
                if constexpr (DYN) {
                    for (;;) {
                        T5Pos q{0, 0, 0, -1};
                        if (kq) {
                            int r = 0;
                            if (lane == 0) r = next_cta();
                            r = __shfl_sync(0xffffffffu, r, 0);
                            if (r == -2) {
                                bad = true;
                                return false;
                            }
                            if (r >= 0) q = t5_dyn_pos(p, r, perm);
                            const int slot = kr & (kT5Ring - 1);
                            if (kr >= kT5Ring) {  // every reader is done with entry kr - kT5Ring
                                const bool ok =
                                    mbar_wait(bar(B_RE + slot), (uint32_t)(kr / kT5Ring - 1) & 1u, p.err);
                                bad = __any_sync(0xffffffffu, !ok);
                                if (bad) return false;
                            }
                            if (lane == 0) {
                                s_ring[slot] = make_int4(q.rt, q.kvh, q.s, q.b);
                                mbar_arrive(bar(B_RF + slot));  // release: the entry is visible to its readers
                            }
                            ++kr;
                        } else {
                            const int got = ring_read(kr++, q, true);
                            if (got < 0) bad = true;
                            if (got != 1) return false;
                        }
                        if (q.b < 0) return false;
                        V = t5_unit<VARLEN>(p, ln, q, tpt, ps_shift, g_shift);
                        if (V.n_tiles > 0) {
                            ids = first_ids(V);
                            return true;
                        }
                    }
                } else {
                    if (spos.b >= nb) return false;
                    V = sU;
                    ids = s_ids;
                    t5_advance(p, spos, step);
                    spos = next_unit(spos, sU);
                    s_ids = spos.b < nb ? first_ids(sU) : 0;
                    return true;
                }
            };
            T5Unit U{};
            int ids_now = 0;
            bool have = next_work(U, ids_now);
            while (have && !bad) {
                const int qb = n & 1;
                if (kq && n >= 2) {  // Q buffer free once every Q K^T of unit n-2 is done
                    const bool ok = mbar_wait(bar(B_QE + qb), ((n >> 1) - 1) & 1, p.err);
                    bad = __any_sync(0xffffffffu, !ok);
                    if (bad) break;
                }
                if (kq && lane == 0) {
                    mbar_arrive_expect_tx(bar(B_QF + qb), (uint32_t)kT5Tile);
                    const int qtok = U.q0 + U.tok0;
                    tma_load_4d(sQ(qb), &tmQ, bar(B_QF + qb), 0, 0, U.kvh * p.G, qtok);
                    tma_load_4d(sQ(qb) + kT5Half, &tmQ, bar(B_QF + qb), 0, 1, U.kvh * p.G, qtok);
                }
                const int pg_end = (U.k_hi + ps - 1) >> ps_shift;
                const int32_t *bt_row = p.block_table + (long long)U.b * p.W;
                int batch = U.pg0;
                int id_cur = ids_now;
                int id_next = (batch + 32 + lane < pg_end) ? __ldg(bt_row + batch + 32 + lane) : 0;
                for (int t = 0; t < U.n_tiles; ++t) {
                    const int g = g0 + t, slot = g & 1;
                    const int pg_first = U.pg0 + t * ppt;
                    if (pg_first >= batch + 32) {
                        batch += 32;
                        id_cur = id_next;
                        const int nx = batch + 32 + lane;
                        id_next = (nx < pg_end) ? __ldg(bt_row + nx) : 0;
                    }
                    const int id = __shfl_sync(0xffffffffu, id_cur, (pg_first + lane - batch) & 31);
                    const int nvalid = min(ppt, pg_end - pg_first);
                    int tok = 0;
                    if (lane < nvalid) {
                        if (id < 0 || (long long)id >= p.num_pages) {
                            atomicOr(p.err, (unsigned int)PA_ERRBIT_PAGE_RANGE);
                            tok = -ps;  // wholly outside the tensor: reads as zeros
                        } else {
                            tok = id << ps_shift;
                        }
                    }
                    // K slot free once Q K^T of tile g-2 is done; V slot once P V of tile g-2 is done
                    const int b_empty = kq ? B_KE : B_VE, b_full = kq ? B_KF : B_VF;
                    if (g >= 2) {
                        const bool ok = mbar_wait(bar(b_empty + slot), ((g >> 1) - 1) & 1, p.err);
                        bad = __any_sync(0xffffffffu, !ok);
                        if (bad) break;
                    }
                    if (lane == 0) mbar_arrive_expect_tx(bar(b_full + slot), (uint32_t)nvalid * 2u * box);
                    __syncwarp();
                    if (lane < nvalid) {
                        const uint32_t dst = (kq ? sK(slot) : sV(slot)) + (uint32_t)lane * box;
    #pragma unroll
                        for (int h = 0; h < 2; ++h)
                            tma_load_4d(dst + (uint32_t)h * kT5Half, kq ? &tmK : &tmV, bar(b_full + slot), 0, tok, h,
                                        U.kvh);
                    }
                }
                g0 += U.n_tiles;
                ++n;
                have = next_work(U, ids_now);  // every load of this unit is out
            }
            // No copy may outlive the CTA: wait (bounded) for the last phase armed on every slot.  After a
            // time-out some of these were never armed; their waits then give up too.
            if (!bad) {
                for (int g = max(0, g0 - 2); g < g0; ++g)
                    mbar_wait(bar((kq ? B_KF : B_VF) + (g & 1)), (g >> 1) & 1, p.err);
                if (kq)
                    for (int k = max(0, n - 2); k < n; ++k) mbar_wait(bar(B_QF + (k & 1)), (k >> 1) & 1, p.err);
            }
            // nor a launch-cancel response (one is outstanding only after a time-out)
            if (DYN && kq && lane == 0 && clc_pending) mbar_wait(bar(B_CLC), clc_parity, p.err);
        } else if (warp == 1) {
            // ================================================================ MMA issuer
            if (lane == 0) {
                bool bad = false;
                // Operand descriptors: the low halves of the buffers' first 16-column slices (the
                // slices of one operand sit at constant offsets from it), one high half for all.
                const uint32_t dhi = tc05::smem_desc_sw128_hi(1024);
                const uint32_t dq0 = tc05::smem_desc_sw128_lo(sQ(0), 16), dq1 = tc05::smem_desc_sw128_lo(sQ(1), 16);
                const uint32_t dk0 = tc05::smem_desc_sw128_lo(sK(0), 16), dk1 = tc05::smem_desc_sw128_lo(sK(1), 16);
                const uint32_t dv0 = tc05::smem_desc_sw128_lo(sV(0), (uint32_t)kT5Half);
                const uint32_t dv1 = tc05::smem_desc_sw128_lo(sV(1), (uint32_t)kT5Half);
                // P V of tile g is issued after Q K^T of tile g+1 (which may belong to the next unit)
                bool pend = false;
                int pg = 0, pn = 0;
                bool pfirst = false, plast = false;
                auto issue_pv = [&](int g, int un, bool first, bool last) -> bool {
                    const int slot = g & 1, ob = un & 1;
                    if (!mbar_wait(bar(B_PF + slot), (g >> 1) & 1, p.err)) return false;  // P, V cleared
                    if (first && un >= 2 && !mbar_wait(bar(B_OFREE + ob), ((un >> 1) - 1) & 1, p.err)) return false;
                    tc05::fence_after_sync();
                    const uint32_t pcol = tmem + (slot ? 128u : 0u);
                    const uint32_t ocol = tmem + kColO + 128u * (uint32_t)ob;
                    const uint32_t dv = slot ? dv1 : dv0;
                    // keys 16kk..16kk+15 are chunk kk/2 of 32 keys: highs at +0, remainders at +16
                    auto pv_one = [&](int kk, uint32_t part, uint32_t acc) {
                        const uint32_t vlo = dv + (uint32_t)kk * (2048u >> 4);  // V rows 16kk..16kk+15
                        const uint32_t pa = pcol + 32u * (uint32_t)(kk >> 1) + 8u * (uint32_t)(kk & 1) + part;
                        tc05::mma_ts_lh(ocol, pa, vlo, dhi, idesc_pv, acc);
                    };
                    if constexpr (kEarlyHi && t5_split_p<T>()) {
                        // the high parts' products, then (once written) the remainders'
    #pragma unroll
                        for (int kk = 0; kk < 8; ++kk) pv_one(kk, 0u, (!first || kk > 0) ? 1u : 0u);
                        if (!mbar_wait(bar(B_PL + slot), (g >> 1) & 1, p.err)) return false;  // P's remainders
                        tc05::fence_after_sync();
    #pragma unroll
                        for (int kk = 0; kk < 8; ++kk) pv_one(kk, 16u, 1u);
                    } else {
                        // both products of each V slice back to back
    #pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            pv_one(kk, 0u, (!first || kk > 0) ? 1u : 0u);
                            if (t5_split_p<T>()) pv_one(kk, 16u, 1u);
                        }
                    }
                    tc05::commit(bar(B_VE + slot));  // V slot free, O holds this product
                    if (last) tc05::commit(bar(B_OF + ob));
                    return true;
                };
                int n = 0, g0 = 0, kr = 0;
                T5Pos cur = start();
                while (!bad) {
                    T5Pos pos;
                    const int got = walk(kr, cur, pos, false);
                    if (got != 1) {
                        bad = got < 0;
                        break;
                    }
                    const T5Unit U = t5_unit<VARLEN>(p, ln, pos, tpt, ps_shift, g_shift);
                    if (U.n_tiles == 0) {
                        // From the ring, issue the held-back P V now: the producer posts units with
                        // no key tile without loads, so a run of them (a sequence of length 0 or
                        // masked whole) may take it a ring's length ahead of the epilogue, which
                        // waits for that product before it reads further entries.
                        if (DYN && pend) {
                            if (!issue_pv(pg, pn, pfirst, plast)) { bad = true; break; }
                            pend = false;
                        }
                        continue;
                    }
                    const int qb = n & 1;
                    if (!mbar_wait(bar(B_QF + qb), (n >> 1) & 1, p.err)) { bad = true; break; }
                    for (int t = 0; t < U.n_tiles; ++t) {
                        const int g = g0 + t, slot = g & 1;
                        if (!mbar_wait(bar(B_KF + slot), (g >> 1) & 1, p.err)) { bad = true; break; }
                        tc05::fence_after_sync();
                        const uint32_t d = tmem + (slot ? 128u : 0u);
                        const uint32_t dq = qb ? dq1 : dq0, dk = slot ? dk1 : dk0;
    #pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            // columns 16kk..16kk+15: 64-column half kk/4, 32-byte slice kk%4 of its rows
                            const uint32_t off = ((uint32_t)(kk >> 2) * kT5Half + (uint32_t)(kk & 3) * 32u) >> 4;
                            tc05::mma_ss_lh(d, dq + off, dhi, dk + off, dhi, idesc_qk, kk > 0 ? 1u : 0u);
                        }
                        tc05::commit(bar(B_KE + slot));  // K slot free, S holds the scores
                        if (t == U.n_tiles - 1) tc05::commit(bar(B_QE + qb));
                        if (pend && !issue_pv(pg, pn, pfirst, plast)) { bad = true; break; }
                        pend = true;
                        pg = g;
                        pn = n;
                        pfirst = t == 0;
                        plast = t == U.n_tiles - 1;
                    }
                    g0 += U.n_tiles;
                    ++n;
                }
                if (!bad && pend) issue_pv(pg, pn, pfirst, plast);
            }
            __syncwarp();
        } else if (warp == 3) {
            // ================================================================ V gate
            // Keys at or past the unit's k_hi (past the sequence, past the split, past every row's causal
            // reach, or never loaded) sit in the V rows of the unit's last tile with any bits: their
            // weight is 0, but 0 * NaN is NaN, so those rows are cleared before P V reads the slot.
            // Every tile passes through here (the P V product waits for the V gate's arrival on PF,
            // not for VF), so the phases stay in step with the ring.  The gate cannot arrive for tile
            // g + 2 before PF's phase for tile g completes: V of g + 2 lands only after P V of g.
            bool bad = false;
            int g0 = 0, kr = 0;
            T5Pos cur = start(), pos;
            while (walk(kr, cur, pos, true) == 1) {
                const T5Unit U = t5_unit<VARLEN>(p, ln, pos, tpt, ps_shift, g_shift);
                for (int t = 0; t < U.n_tiles; ++t) {
                    const int g = g0 + t, st = g & 1;
                    if (!bad) {
                        const bool ok = mbar_wait(bar(B_VF + st), (g >> 1) & 1, p.err);
                        bad = __any_sync(0xffffffffu, !ok);
                    }
                    const int z0 = U.k_hi - (U.k_lo + t * 128);  // first row to clear (< 128 on the last tile only)
                    if (!bad && z0 < 128) {
                        // (128 - z0) rows x 2 halves x 8 16-byte chunks; a quarter warp covers one 128-byte row half
                        for (int i = lane; i < (128 - z0) * 16; i += 32) {
                            const uint32_t a = sV(st) + (uint32_t)((i >> 3) & 1) * kT5Half +
                                               (uint32_t)(z0 + (i >> 4)) * 128u + 16u * (uint32_t)(i & 7);
                            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
                        }
                        fence_proxy_async_smem();
                    }
                    mbar_arrive(bar(B_PF + st));
                }
                g0 += U.n_tiles;
            }
        }
    } else if (wg == 1 || wg == 2) {
        tc05::setmaxnreg_inc<kRegSoftmax>();
        // ================================================================ softmax (warps 4-11)
        // Two warpgroups share every row: group hh (warps 4-7: hh = 0, warps 8-11: hh = 1) owns
        // score columns / keys [64 hh, 64 hh + 64).  They exchange the row maximum once per tile;
        // both keep the same running maximum, so the rescale decisions agree.  Every named barrier
        // is reached on every path (a warp that gave up on a wait still walks the loops, and the eight
        // warps agree on each unit before they walk it), so none can hang.
        const int hh = wg - 1;
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;                       // TMEM lane = query row of the tile
        const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
        bool bad = false;
        int n = 0, g0 = 0, kr = 0;
        T5Pos cur = start();
        for (;;) {
            T5Pos pos;
            const int got = walk(kr, cur, pos, true);
            if (DYN ? !named_bar_and(3, 256, got == 1) : got != 1) break;
            const T5Unit U = t5_unit<VARLEN>(p, ln, pos, tpt, ps_shift, g_shift);
            if (U.n_tiles == 0) continue;  // the epilogue warps write its rows
            const int tk = U.tok0 + (r >> g_shift);
            const bool row_valid = tk < U.tok_end;
            const int ob = n & 1;
            const uint32_t ocol = kColO + 128u * (uint32_t)ob;
            const int lim = row_valid ? min(U.k_hi_split, t5_key_limit(p, ln, U.b, U.L, U.Sq, tk)) : U.k_lo;
            float m_used = kNegInf, l = 0.f;
            for (int t = 0; t < U.n_tiles; ++t) {
                const int g = g0 + t, st = g & 1;
                if (!bad) {
                    const bool ok = mbar_wait(bar(B_KE + st), (g >> 1) & 1, p.err);  // S = Q K^T of tile g
                    bad = __any_sync(0xffffffffu, !ok);
                }
                tc05::fence_after_sync();
                const uint32_t sbuf = tmem + lane_addr + (st ? 128u : 0u);
                const int tile_k0 = U.k_lo + t * 128;
                const int nvalid_row = lim - tile_k0;       // keys [0, nvalid_row) of the tile are valid here
                // my 64 score columns: two 32-column loads, one wait; kept in registers for both passes
                uint32_t ua[32], ub[32];
                float mx = kNegInf;
                if (!bad) {
                    tc05::ld_32cols(sbuf + 64u * hh, ua);
                    tc05::ld_32cols(sbuf + 64u * hh + 32u, ub);
                    tc05::wait_ld();
                    // pass 1: maximum of this row's valid raw scores (scale > 0, which the host
                    // checks, commutes with max)
                    // four independent running maxima (max is exact, so the grouping does not matter)
                    const int nv = nvalid_row - 64 * hh;
                    if (nv < 64) {  // keys past this row's limit become -inf: weight exactly 0 below
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            if (j >= nv) ua[j] = 0xff800000u;
                            if (j + 32 >= nv) ub[j] = 0xff800000u;
                        }
                    }
                    float m4[4] = {kNegInf, kNegInf, kNegInf, kNegInf};
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        m4[j & 3] = fmaxf(m4[j & 3], fmaxf(__uint_as_float(ua[j]), __uint_as_float(ub[j])));
                    mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                }
                s_xmax[st][hh][r] = mx;
                named_bar_sync(2, 256);
                mx = fmaxf(mx, s_xmax[st][hh ^ 1][r]);
                const float m_new = fmaxf(m_used, mx * p.scale_log2);
                const bool need = m_new > m_used + kRescaleLog2;  // also true when m_used is -inf and m_new is not
                if (__any_sync(0xffffffffu, need) && !bad) {
                    const float alpha = need ? exp2f(m_used - m_new) : 1.f;
                    if (need) {
                        l *= alpha;
                        m_used = m_new;
                    }
                    if (t > 0) {
                        // O holds P V of this unit's earlier tiles: wait for the last one (tile g-1; its
                        // slot's next phase needs P of tile g+1, so the parity wait is exact), then
                        // rescale my half of the row
                        const bool ok = mbar_wait(bar(B_VE + ((g - 1) & 1)), ((g - 1) >> 1) & 1, p.err);
                        bad = __any_sync(0xffffffffu, !ok);
                        if (!bad) {
                            tc05::fence_after_sync();
#pragma unroll 1
                            for (int c = 2 * hh; c < 2 * hh + 2; ++c) {
                                uint32_t o[32];
                                tc05::ld_32cols(tmem + lane_addr + ocol + 32u * c, o);
                                tc05::wait_ld();
#pragma unroll
                                for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                                tc05::st_32cols(tmem + lane_addr + ocol + 32u * c, o);
                            }
                        }
                    }
                }
                // pass 2: P = exp2(scale_log2 * s - m) for 32 keys at a time, stored over the same 32
                // columns as [16 columns of high parts | 16 columns of remainders] (bf16/f16 pairs); at
                // split 1 every high part first (PF), then every remainder (PL).
                if (!bad) {
                    const float nmu = (m_used == kNegInf) ? 0.f : -m_used;  // -inf - (-inf) guard
                    const float c2 = p.scale_log2;
                    if constexpr (kEarlyHi && t5_split_p<T>()) {
                        t5_exp_hi<T>(ua, c2, nmu, l, sbuf + 64u * hh);  // ua, ub <- p
                        t5_exp_hi<T>(ub, c2, nmu, l, sbuf + 64u * hh + 32u);
                    } else {
                        // one copy of the chunk's code, run twice (small in the instruction cache next to
                        // the partial-output epilogue)
#pragma unroll 1
                        for (int c = 0; c < 2; ++c) {  // the second 32 scores moved into ua
                            t5_exp_chunk<T>(ua, c2, nmu, l, sbuf + 64u * hh + 32u * (uint32_t)c);
                            if (c == 0) {
#pragma unroll
                                for (int j = 0; j < 32; ++j) ua[j] = ub[j];
                            }
                        }
                    }
                    tc05::wait_st();
                }
                tc05::fence_before_sync();
                mbar_arrive(bar(B_PF + st));
                if constexpr (kEarlyHi && t5_split_p<T>()) {
                    if (!bad) {
                        t5_exp_lo<T>(ua, sbuf + 64u * hh);
                        t5_exp_lo<T>(ub, sbuf + 64u * hh + 32u);
                        tc05::wait_st();
                    }
                    tc05::fence_before_sync();
                    mbar_arrive(bar(B_PL + st));
                }
            }
            // hand the row's maximum and partial sum to the epilogue (the slot of unit n-2 read first)
            if (!bad && n >= 2) {
                const bool ok = mbar_wait(bar(B_LE + ob), ((n >> 1) - 1) & 1, p.err);
                bad = __any_sync(0xffffffffu, !ok);
            }
            s_lsum[ob][hh][r] = l;
            if (hh == 0) s_lmax[ob][r] = m_used;
            mbar_arrive(bar(B_LF + ob));
            g0 += U.n_tiles;
            ++n;
        }
    } else {
        tc05::setmaxnreg_dec<kRegEpilogue>();
        // ================================================================ epilogue (warps 12-15)
        // One thread per query row: wait for the unit's last P V and its row statistics, read the
        // 128 output columns out of TMEM, scale by 1 / l (0 when l = 0: a row with no valid key),
        // and free the O buffer for unit n + 2.  The rows leave through shared memory: each warp
        // stages its 32 rows x 128 bytes of columns (128-byte swizzle: conflict-free) and one
        // lane stores the box with TMA, so no warp issues a store per row; tokens past Sq fall
        // outside the tensor and are clipped.  In a variable-length batch the next sequence's rows
        // follow, so a warp whose rows run past its sequence's last token stores its valid rows
        // itself (one per lane).  The log-sum-exp goes out with plain stores.
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane, r0 = q4 * 32;
        const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
        const uint32_t stage = sbase + (uint32_t)kT5Tile * 6u + (uint32_t)q4 * (uint32_t)kT5Stage;
        const uint32_t srow = stage + (uint32_t)lane * 128u, sw = (uint32_t)(lane & 7);
        constexpr int nch = PART ? 4 : 2;  // 128-byte column chunks of a row: 32 fp32 or 64 16-bit values
        auto put16 = [&](int j, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {  // 16-byte chunk j of my row
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(srow + 16u * ((uint32_t)j ^ sw)), "r"(a),
                         "r"(b), "r"(c), "r"(d)
                         : "memory");
        };
        // 16-byte chunk j of column chunk ch of my row, straight to global memory
        auto gput16 = [&](const T5Unit &U, long long ridx, int ch, int j, uint32_t a, uint32_t b, uint32_t c,
                          uint32_t d) {
            uint4 *dst;
            if constexpr (PART)
                dst = reinterpret_cast<uint4 *>(reinterpret_cast<float *>(p.out) +
                                                ((long long)U.s * p.rows_total + ridx) * 128 + 32 * ch) + j;
            else
                dst = reinterpret_cast<uint4 *>(reinterpret_cast<T *>(p.out) + ridx * 128 + 64 * ch) + j;
            *dst = make_uint4(a, b, c, d);
        };
        auto stage_free = [&]() {  // the previous box has been read out of the staging rows
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
        };
        auto store_box = [&](const T5Unit &U, int ch, bool direct) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && !direct) {
                if constexpr (VARLEN)  // map (D, Hq, T, S): packed tokens
                    tma_store_4d(&tmO, stage, PART ? 32 * ch : 64 * ch, U.kvh * p.G + (r0 & (p.G - 1)),
                                 U.q0 + U.tok0 + (r0 >> g_shift), PART ? U.s : 0);
                else  // map (D, Hq, Sq, B x S)
                    tma_store_4d(&tmO, stage, PART ? 32 * ch : 64 * ch, U.kvh * p.G + (r0 & (p.G - 1)),
                                 U.tok0 + (r0 >> g_shift), PART ? U.s * p.B + U.b : U.b);
                bulk_commit_group();
            }
        };
        bool bad = false;
        int n = 0, kr = 0;
        T5Pos cur = start(), pos;
        while (walk(kr, cur, pos, true) == 1) {
            const T5Unit U = t5_unit<VARLEN>(p, ln, pos, tpt, ps_shift, g_shift);
            if (U.skip) continue;  // another kernel's unit (variable-length batches)
            if (threadIdx.x == 384 && U.s == 0 && U.tok0 == 0 && p.seq_lens[U.b] > p.W * ps)
                atomicOr(p.err, (unsigned int)PA_ERRBIT_SEQ_CLIPPED);
            const int tk = U.tok0 + (r >> g_shift);
            const bool row_valid = tk < U.tok_end;
            const long long ridx = row_valid ? t5_row_index(p, U.q0, U.kvh, tk, r & (p.G - 1)) : 0;
            // variable-length batches: this warp's rows run past the sequence (warp-uniform)
            const bool direct = VARLEN && U.tok0 + ((r0 + 31) >> g_shift) >= U.tok_end;
            auto emit16 = [&](int ch, int j, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
                if (!direct) put16(j, a, b, c, d);
                else if (row_valid) gput16(U, ridx, ch, j, a, b, c, d);
            };
            if (U.n_tiles == 0) {  // no valid key for any row of the unit: lse -inf, output 0
                // split partials (uniform batches): the rows stay unwritten, since a row with lse
                // -inf has weight 0 and the combine never reads it (17 % of the causal prefill's
                // units at split 8)
                if constexpr (!PART || VARLEN) {
#pragma unroll 1
                    for (int ch = 0; ch < nch; ++ch) {
                        stage_free();
#pragma unroll
                        for (int j = 0; j < 8; ++j) emit16(ch, j, 0u, 0u, 0u, 0u);
                        store_box(U, ch, direct);
                    }
                }
                if (row_valid) t5_store_lse<PART>(p, U.s, ridx, kNegInf);
                continue;
            }
            const int ob = n & 1;
            if (!bad) {
                bool ok = mbar_wait(bar(B_LF + ob), (n >> 1) & 1, p.err);
                ok = ok && mbar_wait(bar(B_OF + ob), (n >> 1) & 1, p.err);
                bad = __any_sync(0xffffffffu, !ok);
            }
            const float l_tot = s_lsum[ob][0][r] + s_lsum[ob][1][r];
            const float m = s_lmax[ob][r];
            mbar_arrive(bar(B_LE + ob));
            if (!bad) {
                tc05::fence_after_sync();
                const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
                const uint32_t ocol = tmem + lane_addr + kColO + 128u * (uint32_t)ob;
#pragma unroll 1
                for (int ch = 0; ch < nch; ++ch) {
                    if constexpr (PART) {
                        uint32_t u[32];
                        tc05::ld_32cols(ocol + 32u * (uint32_t)ch, u);
                        stage_free();
                        tc05::wait_ld();
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            emit16(ch, j, __float_as_uint(__uint_as_float(u[4 * j]) * inv),
                                  __float_as_uint(__uint_as_float(u[4 * j + 1]) * inv),
                                  __float_as_uint(__uint_as_float(u[4 * j + 2]) * inv),
                                  __float_as_uint(__uint_as_float(u[4 * j + 3]) * inv));
                    } else {
                        stage_free();
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            uint32_t u[32];
                            tc05::ld_32cols(ocol + 64u * (uint32_t)ch + 32u * (uint32_t)hf, u);
                            tc05::wait_ld();
                            auto pk = [&](int i) {
                                return MmaOp<T>::pack(__uint_as_float(u[i]) * inv, __uint_as_float(u[i + 1]) * inv);
                            };
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                emit16(ch, 4 * hf + j, pk(8 * j), pk(8 * j + 2), pk(8 * j + 4), pk(8 * j + 6));
                        }
                    }
                    store_box(U, ch, direct);
                }
                if (row_valid) t5_store_lse<PART>(p, U.s, ridx, l_tot > 0.f ? m * kLn2 + logf(l_tot) : kNegInf);
            }
            tc05::fence_before_sync();
            mbar_arrive(bar(B_OFREE + ob));  // O buffer may take unit n + 2's products
            ++n;
        }
        if (lane == 0) bulk_wait_all();  // no store may outlive the CTA's shared memory
        __syncwarp();
    }

    tc05::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc05::fence_after_sync();
        tc05::tmem_dealloc(tmem, kT5TmemCols);
    }
}

// ------------------------------------------------------------------------ host side
size_t tc05_smem_bytes() { return (size_t)(kT5Tile * 6 + 4 * kT5Stage + 1024); }

static int num_sms_of_current_device() {
    static std::atomic<int> cached[128];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 0;
    int v = cached[dev].load(std::memory_order_relaxed);
    if (!v) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

// split_kv = 1: one CTA per unit, of which one runs per SM and takes the rest by cancelling their
// launches.  Otherwise one persistent CTA per SM; max_ctas > 0 caps the grid when the kernel shares
// the GPU with another kernel running at the same time.  Any grid up to the unit count computes the
// same results, since a unit's work does not depend on the CTA that takes it.
template <typename T, bool PART, bool VARLEN>
static cudaError_t launch_tc05_t(const FwdParams &p, long long total_q, const CUtensorMap &tmq,
                                 const CUtensorMap &tmk, const CUtensorMap &tmv, const CUtensorMap &tmo,
                                 int max_ctas, cudaStream_t stream) {
    auto kern = paged_attn_tc05_kernel<T, PART, VARLEN>;
    const size_t smem = tc05_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // The softmax warpgroups' setmaxnreg increase is served from what the launch holds: a build
    // that gave the kernel fewer registers per thread would leave them waiting, so refuse it.
    static std::atomic<int> launch_regs{0};
    int regs = launch_regs.load(std::memory_order_relaxed);
    if (!regs) {
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        regs = fa.numRegs;
        launch_regs.store(regs, std::memory_order_relaxed);
    }
    if (regs < kT5LaunchRegs) return cudaErrorInvalidConfiguration;
    int ps_shift = 0, g_shift = 0;
    while ((1 << ps_shift) < p.ps) ++ps_shift;
    while ((1 << g_shift) < p.G) ++g_shift;
    if ((1 << g_shift) != p.G || g_shift > 7) return cudaErrorInvalidValue;  // G must divide 128
    const int tpt = 128 >> g_shift;
    FwdParams q = p;
    long long nb;  // values of the unit order's b digit
    if (VARLEN && p.B > kT5StageLens) return cudaErrorInvalidValue;  // q_start must fit its stage
    if (VARLEN) {
        q.row_tiles = 1;
        nb = (total_q << g_shift >> 7) + p.B;  // blocks of the packed rows (t5_first_block)
    } else {
        q.row_tiles = (p.Sq + tpt - 1) / tpt;
        nb = p.B;
    }
    const long long units = nb * p.split_kv * p.Hkv * q.row_tiles;
    if (units <= 0) return cudaSuccess;
    if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    int sms = num_sms_of_current_device();
    if (sms <= 0) return cudaErrorInvalidDevice;
    if (max_ctas > 0 && max_ctas < sms) sms = max_ctas;
    constexpr bool dyn = !PART && !VARLEN;  // the kernel's DYN
    const int grid = dyn ? (int)units : (int)(units < sms ? units : sms);
    const bool bf = std::is_same<T, __nv_bfloat16>::value;
    const uint32_t iqk = tc05::idesc_f16(bf, false, 128, 128);
    const uint32_t ipv = tc05::idesc_f16(bf, true, 128, 128);
    kern<<<grid, kT5Threads, smem, stream>>>(tmq, tmk, tmv, tmo, q, tpt, ps_shift, g_shift, iqk, ipv, (int)nb,
                                             (int)units);
    return cudaGetLastError();
}

template <bool VARLEN>
static cudaError_t launch_tc05_any(const FwdParams &p, long long total_q, int dtype, const CUtensorMap &tmq,
                                   const CUtensorMap &tmk, const CUtensorMap &tmv, const CUtensorMap &tmo,
                                   int max_ctas, cudaStream_t stream) {
    const bool part = p.split_kv > 1;
    if (dtype == PA_BF16)
        return part ? launch_tc05_t<__nv_bfloat16, true, VARLEN>(p, total_q, tmq, tmk, tmv, tmo, max_ctas, stream)
                    : launch_tc05_t<__nv_bfloat16, false, VARLEN>(p, total_q, tmq, tmk, tmv, tmo, max_ctas, stream);
    return part ? launch_tc05_t<__half, true, VARLEN>(p, total_q, tmq, tmk, tmv, tmo, max_ctas, stream)
                : launch_tc05_t<__half, false, VARLEN>(p, total_q, tmq, tmk, tmv, tmo, max_ctas, stream);
}

cudaError_t launch_tc05(const FwdParams &p, int dtype, const CUtensorMap &tmq, const CUtensorMap &tmk,
                        const CUtensorMap &tmv, const CUtensorMap &tmo, cudaStream_t stream) {
    return launch_tc05_any<false>(p, 0, dtype, tmq, tmk, tmv, tmo, 0, stream);
}

cudaError_t launch_tc05_varlen(const FwdParams &p, long long total_q, int dtype, const CUtensorMap &tmq,
                               const CUtensorMap &tmk, const CUtensorMap &tmv, const CUtensorMap &tmo,
                               int max_ctas, cudaStream_t stream) {
    return launch_tc05_any<true>(p, total_q, dtype, tmq, tmk, tmv, tmo, max_ctas, stream);
}

}  // namespace pa
