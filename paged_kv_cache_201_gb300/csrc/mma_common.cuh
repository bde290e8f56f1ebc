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

// A unit with no valid key for any of its rows: output 0, lse -inf (consumer warps only).
template <typename T, int D>
__device__ __forceinline__ void store_empty_unit(const FwdParams &p, const SeqRows &sq, int kvh, int s, int row0,
                                                 int row_end) {
    const int nrows = row_end - row0;
    for (int idx = threadIdx.x; idx < nrows * (D / 2); idx += kMmaConsumerWarps * 32) {
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
// [w][16][D + 4] of unnormalised outputs, then maxima [w][16] and sums [w][16] (log2 domain).
// Each row is combined over the warps (0/0 guard: l == 0 stores 0, lse -inf) and stored.
template <typename T, int D>
__device__ __forceinline__ void decode_merge_store(const FwdParams &p, const float *sm, const SeqRows &sq, int kvh,
                                                   int s, int row_end) {
    constexpr int ACC_STRIDE = D + 4;
    const float *s_acc = sm;
    const float *s_m = sm + kMmaConsumerWarps * 16 * ACC_STRIDE;
    const float *s_l = s_m + kMmaConsumerWarps * 16;
    const int tid = threadIdx.x;  // 0..127
    const int r = tid >> 3;       // 16 rows x 8 column groups
    const int cg = tid & 7;
    constexpr int COLS = D / 8;
    if (r < row_end) {
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
        const long long ridx = out_row_index(p, sq, kvh, r);
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
    if (!bad) decode_merge_store<T, D>(p, sm, sq, kvh, s, row_end);
}

}  // namespace mmac
}  // namespace pa
