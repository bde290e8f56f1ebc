// CUDA-core paged decode for a single query row per (sequence, kv head): no GQA sharing and one
// query token (bf16 / f16, head_dim 64 or 128), sm_103a.
//
// With one row there is no dense contraction to give the tensor cores, so Q.K and P.V run as fp32
// FMAs.  The kernel is built for the HBM stream: the producer warp and the K/V ring are those of
// the tensor-core decode kernel (page ids loaded once per 32 pages, one 4-D TMA box per page and
// pool, 128-byte swizzled, 64-key stages), and consumer warp w takes keys [16 w, 16 w + 16) of
// every stage:
//   * Q.K: two lanes per key, each with half the head dimension of q in registers (fp32) and the
//     matching 16-byte chunks of its key's row from shared memory; the second lane of a pair
//     visits its chunks in a rotated order, so the 8 lanes of a load phase hit 8 banks.  One
//     shuffle adds the halves.
//   * online softmax over the warp's 16 keys in the log2 domain with the rocMLIR PR #2371 guards
//     (a running max of -inf is replaced by 0 before exp2; a row whose sum is 0 stores 0 / lse -inf);
//   * P.V: lane l owns head-dim columns [l D/32, (l + 1) D/32) and reads them from each of the 16
//     V rows (conflict-free 8- or 4-byte loads), weighting by the key's p (a shuffle).
// The four warps' states are merged through shared memory at the end.
#include "mma_common.cuh"

namespace pa {

using namespace mmac;

namespace {

// Unpack a 16-bit pair (element 0 in the low half) to two floats.
template <typename T>
__device__ __forceinline__ float2 unpack2(uint32_t w);
template <>
__device__ __forceinline__ float2 unpack2<__nv_bfloat16>(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
template <>
__device__ __forceinline__ float2 unpack2<__half>(uint32_t w) {
    return __half22float2(*reinterpret_cast<const __half2 *>(&w));
}

}  // namespace

template <typename T, int D, int NSTAGE>
__global__ void __launch_bounds__(kMmaThreads, 2)
    paged_attn_simt_decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                                  const FwdParams p, int ps_shift) {
    constexpr int kStage = Geo<D>::kStageBytes;
    constexpr int kChunks = Geo<D>::kChunks;  // 16-byte chunks per row
    constexpr int HC = kChunks / 2;           // chunks of half a row
    constexpr int CPL = D / 32;               // output columns per lane

    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[3 * NSTAGE];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int ps = 1 << ps_shift;
    int unit = blockIdx.x;
    const int kvh = unit % p.Hkv;
    unit /= p.Hkv;
    const int s = unit % p.split_kv;
    const int b = unit / p.split_kv;
    const SeqRows sq = uniform_seq(p, b);

    int L = max(p.seq_lens[b], 0);
    if (L > p.W * ps) {  // never read past the sequence's block-table row
        if (threadIdx.x == 0) atomicOr(p.err, (unsigned int)PA_ERRBIT_SEQ_CLIPPED);
        L = p.W * ps;
    }
    int pg0, pg1;
    split_pages(L, ps, p.split_kv, s, pg0, pg1);
    const int k_lo = pg0 * ps;
    const int k_hi = min(min(pg1 * ps, L), row_key_limit(p, b, L, 0));
    const int n_tiles = k_hi > k_lo ? (k_hi - k_lo + kMmaTileKeys - 1) / kMmaTileKeys : 0;
    if (n_tiles == 0) {
        if (warp < kMmaConsumerWarps) store_empty_unit<T, D>(p, sq, kvh, s, 0, 1);
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
        produce_pages16<D, NSTAGE>(&tmK, &tmV, p, b, kvh, pg0, k_hi, n_tiles, ps_shift, sbase, bar_fk, bar_fv, bar_em,
                                   lane);
        return;
    }

    // ==================================================================== consumers
    const int kw0 = warp * 16;        // this warp's keys in every stage
    const int kq = lane >> 1;         // this lane's key within them
    const int hh = lane & 1;          // which half of the head dimension it scores
    const int rot = hh ? HC / 2 : 0;  // chunk rotation of the second lane of a pair
    // q, half hh, as fp32 in the lane's visiting order: qh[8 i ..] is chunk (i + rot) % HC of the half
    float qh[D / 2];
    {
        const T *q = reinterpret_cast<const T *>(p.q) + q_row_offset(p, out_row_index(p, sq, kvh, 0)) + hh * (D / 2);
#pragma unroll
        for (int i = 0; i < HC; ++i) {
            const uint4 x = __ldg(reinterpret_cast<const uint4 *>(q) + (i + rot) % HC);
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 f = unpack2<T>(w[k]);
                qh[8 * i + 2 * k] = f.x;
                qh[8 * i + 2 * k + 1] = f.y;
            }
        }
    }
    float m = kNegInf, l = 0.f;
    float acc[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[c] = 0.f;

    bool bad = false;
    for (int t = 0; t < n_tiles; ++t) {
        const int st = t % NSTAGE;
        const uint32_t par = (t / NSTAGE) & 1;
        const uint32_t kbuf = sbase + (uint32_t)(st * 2 * kStage);
        const uint32_t vbuf = kbuf + kStage;
        const int tile_k0 = k_lo + t * kMmaTileKeys;
        const bool active = tile_k0 + kw0 < k_hi;  // warp-uniform

        if (!bad) {
            const bool ok = mbar_wait(bar_fk + 8 * st, par, p.err);
            bad = __any_sync(0xffffffffu, !ok);
        }
        float pj = 0.f;
        float al = 1.f;
        if (!bad && active) {
            // ---- score of key kw0 + kq: this lane's half, then the pair's sum
            float sc = 0.f;
#pragma unroll
            for (int i = 0; i < HC; ++i) {
                const int cc = (i + rot) % HC;
                uint32_t w[4];
                asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                             : "r"(kv_chunk_addr<D>(kbuf, kw0 + kq, hh * HC + cc, ps_shift))
                             : "memory");
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 f = unpack2<T>(w[k]);
                    sc = fmaf(qh[8 * i + 2 * k], f.x, sc);
                    sc = fmaf(qh[8 * i + 2 * k + 1], f.y, sc);
                }
            }
            sc += __shfl_xor_sync(0xffffffffu, sc, 1);
            const int j = tile_k0 + kw0 + kq;
            sc = (j < k_hi) ? sc * p.scale_log2 : kNegInf;
            // ---- online softmax over the warp's 16 keys (each held by a lane pair)
            float mx = sc;
#pragma unroll
            for (int o = 2; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float mn = fmaxf(m, mx);
            const float mu = (mn == kNegInf) ? 0.f : mn;  // -inf - (-inf) guard
            al = exp2f(m - mu);
            pj = exp2f(sc - mu);
            float ps_ = hh ? 0.f : pj;  // one lane of each pair counts the key
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) ps_ += __shfl_xor_sync(0xffffffffu, ps_, o);
            l = l * al + ps_;
            m = mn;
        }
        if (!bad) {
            const bool ok = mbar_wait(bar_fv + 8 * st, par, p.err);
            bad = __any_sync(0xffffffffu, !ok);
        }
        if (!bad && active) {
            if (tile_k0 + kMmaTileKeys > k_hi) {
                // Last stage: V rows at or past k_hi (past the sequence, or pages never loaded) may
                // hold any bits; their weight is 0, but 0 x NaN is NaN, so zero this warp's such rows.
                for (int idx = lane; idx < 16 * kChunks; idx += 32) {
                    const int key = kw0 + idx / kChunks;
                    if (tile_k0 + key >= k_hi) {
                        const uint32_t a = kv_chunk_addr<D>(vbuf, key, idx % kChunks, ps_shift);
                        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            // ---- O = al O + sum_j p_j V_j over this lane's columns
#pragma unroll
            for (int c = 0; c < CPL; ++c) acc[c] *= al;
            const int col0 = lane * CPL;
#pragma unroll 4
            for (int jj = 0; jj < 16; ++jj) {
                const float w = __shfl_sync(0xffffffffu, pj, 2 * jj);
                const uint32_t a = kv_chunk_addr<D>(vbuf, kw0 + jj, col0 / 8, ps_shift) + (uint32_t)((col0 % 8) * 2);
                if constexpr (CPL == 4) {
                    uint32_t v0, v1;
                    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v0), "=r"(v1) : "r"(a) : "memory");
                    const float2 f0 = unpack2<T>(v0), f1 = unpack2<T>(v1);
                    acc[0] = fmaf(w, f0.x, acc[0]);
                    acc[1] = fmaf(w, f0.y, acc[1]);
                    acc[2] = fmaf(w, f1.x, acc[2]);
                    acc[3] = fmaf(w, f1.y, acc[3]);
                } else {
                    uint32_t v0;
                    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v0) : "r"(a) : "memory");
                    const float2 f0 = unpack2<T>(v0);
                    acc[0] = fmaf(w, f0.x, acc[0]);
                    acc[1] = fmaf(w, f0.y, acc[1]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_em + 8 * st);
    }

    // ---- merge the four warps' states (m, l uniform per warp) through shared memory (reuses the ring)
    float *sm = reinterpret_cast<float *>(smem_raw + (sbase - raw));
    float *s_acc = sm;                             // [4][D]
    float *s_m = sm + kMmaConsumerWarps * D;       // [4]
    float *s_l = s_m + kMmaConsumerWarps;          // [4]
    named_bar_sync(1, kMmaConsumerWarps * 32);     // every warp is done reading the ring
#pragma unroll
    for (int c = 0; c < CPL; ++c) s_acc[warp * D + lane * CPL + c] = acc[c];
    if (lane == 0) {
        s_m[warp] = m;
        s_l[warp] = l;
    }
    named_bar_sync(1, kMmaConsumerWarps * 32);
    if (bad) return;
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < kMmaConsumerWarps; ++w) M = fmaxf(M, s_m[w]);
    float wsc[kMmaConsumerWarps], Lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kMmaConsumerWarps; ++w) {
        wsc[w] = (M == kNegInf) ? 0.f : exp2f(s_m[w] - M);
        Lsum += wsc[w] * s_l[w];
    }
    const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;  // 0/0 guard
    const long long ridx = out_row_index(p, sq, kvh, 0);
    for (int col = 2 * threadIdx.x; col < D; col += 2 * kMmaConsumerWarps * 32) {
        float o0 = 0.f, o1 = 0.f;
#pragma unroll
        for (int w = 0; w < kMmaConsumerWarps; ++w) {
            o0 += wsc[w] * s_acc[w * D + col];
            o1 += wsc[w] * s_acc[w * D + col + 1];
        }
        store_pair<T>(p, s, ridx, col, o0 * inv, o1 * inv);
    }
    if (threadIdx.x == 0) store_lse(p, s, ridx, Lsum > 0.f ? M * kLn2 + logf(Lsum) : kNegInf);
}

// ------------------------------------------------------------------------ host side
template <typename T, int D, int NSTAGE>
static cudaError_t launch_simt_decode_t(const FwdParams &p, const CUtensorMap &tmk, const CUtensorMap &tmv,
                                        cudaStream_t stream) {
    constexpr size_t smem = (size_t)NSTAGE * 2 * Geo<D>::kStageBytes + 1024;
    static_assert((size_t)(kMmaConsumerWarps * (D + 2)) * 4 + 1024 <= smem, "merge scratch must fit in the ring");
    auto kern = paged_attn_simt_decode_kernel<T, D, NSTAGE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int ps_shift = 0;
    while ((1 << ps_shift) < p.ps) ++ps_shift;
    const long long units = (long long)p.B * p.split_kv * p.Hkv;
    if (units <= 0) return cudaSuccess;
    if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)units, kMmaThreads, smem, stream>>>(tmk, tmv, p, ps_shift);
    return cudaGetLastError();
}

cudaError_t launch_simt_decode(const FwdParams &p, int dtype, const CUtensorMap &tmk, const CUtensorMap &tmv,
                               cudaStream_t stream) {
    if (p.rows != 1 || (p.D != 64 && p.D != 128)) return cudaErrorInvalidValue;
    if (dtype == PA_BF16) {
        return p.D == 128 ? launch_simt_decode_t<__nv_bfloat16, 128, 3>(p, tmk, tmv, stream)
                          : launch_simt_decode_t<__nv_bfloat16, 64, 4>(p, tmk, tmv, stream);
    }
    return p.D == 128 ? launch_simt_decode_t<__half, 128, 3>(p, tmk, tmv, stream)
                      : launch_simt_decode_t<__half, 64, 4>(p, tmk, tmv, stream);
}

}  // namespace pa
