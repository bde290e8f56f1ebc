// Split-KV combine, split-plan export and logical gather kernels.
#include "kernels.h"

namespace pa {


// ---------------------------------------------------------------------------- combine
// rocMLIR PR #2371 (Technical Details, f32 combine for narrow floats): per row,
// M = max_s lse_s, w_s = exp(lse_s - M), out = sum w_s O_s / sum w_s, lse =
// M + log(sum w_s), all in fp32; M = -inf (every split empty) gives out 0 and
// lse -inf.  One warp per row; each lane owns D/32 consecutive columns.  Rows are taken from the
// last one back: the forward kernels write the partials in row order, so the rows at the end were
// written last and are the ones still in L2 when this kernel starts.
template <typename TO, int D>
__global__ void __launch_bounds__(256) paged_attn_combine_kernel(const float *__restrict__ part_out,
                                                                 const float *__restrict__ part_lse, int S,
                                                                 long long rows, TO *__restrict__ out,
                                                                 float *__restrict__ lse) {
    constexpr int DPL = D / 32;
    const long long idx = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (idx >= rows) return;
    const long long row = rows - 1 - idx;
    float M = kNegInf;
    for (int s0 = 0; s0 < S; s0 += 32) {
        const float v = (s0 + lane < S) ? __ldg(part_lse + (long long)(s0 + lane) * rows + row) : kNegInf;
        M = fmaxf(M, v);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float acc[DPL];
#pragma unroll
    for (int c = 0; c < DPL; ++c) acc[c] = 0.f;
    float wsum = 0.f;
    if (M != kNegInf) {
        for (int s = 0; s < S; ++s) {
            const float w = expf(__ldg(part_lse + (long long)s * rows + row) - M);  // exp(-inf) = 0
            wsum += w;
            if (w != 0.f) {
                const float *src = part_out + ((long long)s * rows + row) * D + lane * DPL;
                if constexpr (DPL % 4 == 0) {
#pragma unroll
                    for (int c4 = 0; c4 < DPL; c4 += 4) {
                        const float4 v = __ldg(reinterpret_cast<const float4 *>(src + c4));
                        acc[c4] = fmaf(w, v.x, acc[c4]);
                        acc[c4 + 1] = fmaf(w, v.y, acc[c4 + 1]);
                        acc[c4 + 2] = fmaf(w, v.z, acc[c4 + 2]);
                        acc[c4 + 3] = fmaf(w, v.w, acc[c4 + 3]);
                    }
                } else {
                    const float2 v = __ldg(reinterpret_cast<const float2 *>(src));
                    acc[0] = fmaf(w, v.x, acc[0]);
                    acc[1] = fmaf(w, v.y, acc[1]);
                }
            }
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    TO *dst = out + row * D + lane * DPL;
#pragma unroll
    for (int c = 0; c < DPL; ++c) dst[c] = from_float<TO>(acc[c] * inv);
    if (lse && lane == 0) lse[row] = wsum > 0.f ? M + logf(wsum) : kNegInf;
}

// The same combine for launches with few rows, where a warp's chain of dependent loads (lse, then
// the partial row, split after split) sets the time rather than DRAM: lane s reads lse_s (S <= 32),
// the weights reach every lane by shuffle, and the partial rows of SB splits are loaded at once.
// Sums run over the splits in the same order and with the same operations as above, so the two
// kernels give the same bits.
template <typename TO, int D, int SB>
__global__ void __launch_bounds__(256) paged_attn_combine_wide_kernel(const float *__restrict__ part_out,
                                                                      const float *__restrict__ part_lse, int S,
                                                                      long long rows, TO *__restrict__ out,
                                                                      float *__restrict__ lse) {
    constexpr int DPL = D / 32;
    const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const float l = lane < S ? __ldg(part_lse + (long long)lane * rows + row) : kNegInf;
    float M = l;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float acc[DPL];
#pragma unroll
    for (int c = 0; c < DPL; ++c) acc[c] = 0.f;
    float wsum = 0.f;
    if (M != kNegInf) {
        const float wl = expf(l - M);  // exp(-inf) = 0 for lanes past S and empty splits
        for (int s0 = 0; s0 < S; s0 += SB) {
            float w[SB], v[SB][DPL];
#pragma unroll
            for (int j = 0; j < SB; ++j) {
                w[j] = __shfl_sync(0xffffffffu, wl, (s0 + j) & 31);
                if (s0 + j >= S) w[j] = 0.f;
                const int sj = min(s0 + j, S - 1);  // an address inside the partials even when unread
                const float *src = part_out + ((long long)sj * rows + row) * D + lane * DPL;
                if constexpr (DPL % 4 == 0) {
#pragma unroll
                    for (int c4 = 0; c4 < DPL; c4 += 4) {
                        const float4 x = w[j] != 0.f ? __ldg(reinterpret_cast<const float4 *>(src + c4))
                                                     : make_float4(0.f, 0.f, 0.f, 0.f);
                        v[j][c4] = x.x;
                        v[j][c4 + 1] = x.y;
                        v[j][c4 + 2] = x.z;
                        v[j][c4 + 3] = x.w;
                    }
                } else {
                    const float2 x = w[j] != 0.f ? __ldg(reinterpret_cast<const float2 *>(src)) : make_float2(0.f, 0.f);
                    v[j][0] = x.x;
                    v[j][1] = x.y;
                }
            }
#pragma unroll
            for (int j = 0; j < SB; ++j) {
                wsum += w[j];
                if (w[j] != 0.f) {
#pragma unroll
                    for (int c = 0; c < DPL; ++c) acc[c] = fmaf(w[j], v[j][c], acc[c]);
                }
            }
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    TO *dst = out + row * D + lane * DPL;
#pragma unroll
    for (int c = 0; c < DPL; ++c) dst[c] = from_float<TO>(acc[c] * inv);
    if (lse && lane == 0) lse[row] = wsum > 0.f ? M + logf(wsum) : kNegInf;
}

template <typename TO>
static cudaError_t launch_combine_t(const float *po, const float *pl, int S, long long rows, int D, void *out,
                                    float *lse, cudaStream_t stream) {
    constexpr int kRowsPerBlock = 8;
    const long long blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    // Up to 16384 rows (a warp each: about one wave of resident warps) the launch is latency-bound.
    if (S <= 32 && rows <= 16384) {
        if (D == 256)
            paged_attn_combine_wide_kernel<TO, 256, 8>
                <<<(unsigned)blocks, kRowsPerBlock * 32, 0, stream>>>(po, pl, S, rows, static_cast<TO *>(out), lse);
        else if (D == 128)
            paged_attn_combine_wide_kernel<TO, 128, 8>
                <<<(unsigned)blocks, kRowsPerBlock * 32, 0, stream>>>(po, pl, S, rows, static_cast<TO *>(out), lse);
        else
            paged_attn_combine_wide_kernel<TO, 64, 8>
                <<<(unsigned)blocks, kRowsPerBlock * 32, 0, stream>>>(po, pl, S, rows, static_cast<TO *>(out), lse);
        return cudaGetLastError();
    }
    if (D == 256)
        paged_attn_combine_kernel<TO, 256>
            <<<(unsigned)blocks, kRowsPerBlock * 32, 0, stream>>>(po, pl, S, rows, static_cast<TO *>(out), lse);
    else if (D == 128)
        paged_attn_combine_kernel<TO, 128>
            <<<(unsigned)blocks, kRowsPerBlock * 32, 0, stream>>>(po, pl, S, rows, static_cast<TO *>(out), lse);
    else
        paged_attn_combine_kernel<TO, 64>
            <<<(unsigned)blocks, kRowsPerBlock * 32, 0, stream>>>(po, pl, S, rows, static_cast<TO *>(out), lse);
    return cudaGetLastError();
}

cudaError_t launch_combine(const float *part_out, const float *part_lse, int S, long long rows, int D,
                           int out_dtype, void *out, float *lse, cudaStream_t stream) {
    if (out_dtype == PA_F32) return launch_combine_t<float>(part_out, part_lse, S, rows, D, out, lse, stream);
    if (out_dtype == PA_BF16)
        return launch_combine_t<__nv_bfloat16>(part_out, part_lse, S, rows, D, out, lse, stream);
    return launch_combine_t<__half>(part_out, part_lse, S, rows, D, out, lse, stream);
}

// ---------------------------------------------------------------------------- plan
__global__ void paged_attn_plan_kernel(const int32_t *__restrict__ seq_lens, int B, int ps, int S,
                                       int32_t *__restrict__ plan) {
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long long)B * S) return;
    const int b = (int)(idx / S), s = (int)(idx % S);
    int p0, p1;
    split_pages(max(seq_lens[b], 0), ps, S, s, p0, p1);
    plan[idx * 2 + 0] = p0;
    plan[idx * 2 + 1] = p1;
}

cudaError_t launch_plan(const int32_t *seq_lens, int B, int ps, int S, int32_t *plan, cudaStream_t stream) {
    const long long n = (long long)B * S;
    if (n == 0) return cudaSuccess;
    const long long blocks = (n + 255) / 256;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    paged_attn_plan_kernel<<<(unsigned)blocks, 256, 0, stream>>>(seq_lens, B, ps, S, plan);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------- gather
// Logical view of a paged pool (rocMLIR PR #2222, Key Changes 1): token j of
// sequence b is row j % page_size of page block_table[b][j / page_size]; the
// kv-head term D * kvh is added inside the row.  Copies 16-byte chunks bit for
// bit; tokens past seq_lens[b] are zero.
__global__ void paged_attn_gather_kernel(const uint8_t *__restrict__ cache, const int32_t *__restrict__ block_table,
                                         const int32_t *__restrict__ seq_lens, int B, int W, int ps,
                                         long long row_bytes /* Hkv * D * esize */, long long num_pages,
                                         int out_tokens, uint8_t *__restrict__ out, unsigned int *err) {
    const long long chunks_per_tok = row_bytes / 16;
    const long long total = (long long)B * out_tokens * chunks_per_tok;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long c = idx % chunks_per_tok;
        const long long tj = idx / chunks_per_tok;
        const int j = (int)(tj % out_tokens);
        const int b = (int)(tj / out_tokens);
        const int L = min(max(seq_lens[b], 0), W * ps);
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (j < L) {
            const int id = block_table[(long long)b * W + j / ps];
            if (id >= 0 && (long long)id < num_pages) {
                const long long off = ((long long)id * ps + (j % ps)) * row_bytes + c * 16;
                v = __ldg(reinterpret_cast<const uint4 *>(cache + off));
            } else if (c == 0) {
                atomicOr(err, (unsigned int)PA_ERRBIT_PAGE_RANGE);
            }
        }
        *reinterpret_cast<uint4 *>(out + (tj * chunks_per_tok + c) * 16) = v;
    }
}

cudaError_t launch_gather(const void *cache, const int32_t *block_table, const int32_t *seq_lens, int B, int W,
                          int ps, int Hkv, int D, int esize, long long num_pages, int out_tokens, void *out,
                          unsigned int *err, cudaStream_t stream) {
    const long long row_bytes = (long long)Hkv * D * esize;
    const long long total = (long long)B * out_tokens * (row_bytes / 16);
    if (total == 0) return cudaSuccess;
    long long blocks = (total + 255) / 256;
    if (blocks > 65536) blocks = 65536;
    paged_attn_gather_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
        static_cast<const uint8_t *>(cache), block_table, seq_lens, B, W, ps, row_bytes, num_pages, out_tokens,
        static_cast<uint8_t *>(out), err);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------- bounded wait check
// One warp waits, with the kernels' bounded wait, on an mbarrier that nothing arrives at: after
// limit_ns the wait gives up and records PA_ERRBIT_TIMEOUT in the error word, as a stalled
// pipeline would.  Lets a test see the time-out path end and leave the context usable.
__global__ void paged_attn_wait_probe_kernel(unsigned int *err, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_barrier_init();
    }
    __syncwarp();
    mbar_wait(b, 0, err, limit_ns);  // phase 0 never completes
}

cudaError_t launch_wait_probe(unsigned int *err, unsigned long long limit_ns, cudaStream_t stream) {
    paged_attn_wait_probe_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace pa
