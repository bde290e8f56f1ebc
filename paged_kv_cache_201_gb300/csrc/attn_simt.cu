// CUDA-core paged attention: any element type (f32 / f16 / bf16), any head grouping.
//
// Serves the shapes where a tensor-core tile would be mostly padding or where
// the element type has no matching tensor-core path at full precision: f32
// pools (tf32 would not hold the f32 tolerance) and single-head (G = 1) decode.
//
// One CTA = (sequence b, kv head, split s, chunk of 8 query rows).  Keys are
// staged 32 at a time into shared memory as fp32 (16-byte loads from each
// page's row, the page's 64-bit base formed once per key), then each warp
// handles two query rows: lane j scores key j, the warp takes the row max and
// sum with shuffles, and each lane accumulates D/32 output columns.  Keys past
// the unit's bound are staged as zeros and masked to -inf, so nothing past the
// sequence is read.
#include "kernels.h"

namespace pa {

namespace {

constexpr int kSimtWarps = 4;
constexpr int kSimtRowsPerWarp = 2;
constexpr int kSimtRows = kSimtWarps * kSimtRowsPerWarp;
constexpr int kSimtKeys = 32;


template <typename T>
__device__ __forceinline__ void load16_to_float(const T *src, float *dst);

template <>
__device__ __forceinline__ void load16_to_float<float>(const float *src, float *dst) {
    const float4 v = __ldg(reinterpret_cast<const float4 *>(src));
    dst[0] = v.x;
    dst[1] = v.y;
    dst[2] = v.z;
    dst[3] = v.w;
}

template <>
__device__ __forceinline__ void load16_to_float<__nv_bfloat16>(const __nv_bfloat16 *src, float *dst) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 f = MmaOp<__nv_bfloat16>::unpack(w[k]);
        dst[2 * k] = f.x;
        dst[2 * k + 1] = f.y;
    }
}

template <>
__device__ __forceinline__ void load16_to_float<__half>(const __half *src, float *dst) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 f = MmaOp<__half>::unpack(w[k]);
        dst[2 * k] = f.x;
        dst[2 * k + 1] = f.y;
    }
}

}  // namespace

template <typename T, int D>
__global__ void __launch_bounds__(kSimtWarps * 32) paged_attn_simt_kernel(const FwdParams p) {
    constexpr int EPV = 16 / sizeof(T);      // elements per 16-byte load
    constexpr int CPR = D / EPV;             // 16-byte chunks per key row
    constexpr int KS = D + 1;                // padded smem row (conflict-free column walks)
    constexpr int DPL = D / 32;              // output columns per lane
    // K, V and Q staging: static for D <= 128; D = 256 (74 KiB) takes dynamic shared memory
    constexpr bool kDyn = D > 128;
    constexpr int kFloats = 2 * kSimtKeys * KS + kSimtRows * D;
    __shared__ float s_static[kDyn ? 1 : kFloats];
    extern __shared__ float s_dynamic[];
    float *const s_k = kDyn ? s_dynamic : s_static;
    float *const s_v = s_k + kSimtKeys * KS;
    float *const s_q = s_v + kSimtKeys * KS;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int unit = blockIdx.x;
    const int rc = unit % p.row_tiles;
    unit /= p.row_tiles;
    const int kvh = unit % p.Hkv;
    unit /= p.Hkv;
    const int s = unit % p.split_kv;
    const int b = unit / p.split_kv;

    int L = max(p.seq_lens[b], 0);
    if (L > p.W * p.ps) {
        if (threadIdx.x == 0) atomicOr(p.err, (unsigned int)PA_ERRBIT_SEQ_CLIPPED);
        L = p.W * p.ps;
    }
    int pg0, pg1;
    split_pages(L, p.ps, p.split_kv, s, pg0, pg1);
    const int k_lo = pg0 * p.ps;
    const int k_hi_split = min(pg1 * p.ps, L);
    const int row0 = rc * kSimtRows;
    const int row_end = min(row0 + kSimtRows, p.rows);
    const int k_hi = min(k_hi_split, row_key_limit(p, b, L, (row_end - 1) / p.G));

    // query rows of this CTA -> smem (fp32)
    const T *q = reinterpret_cast<const T *>(p.q);
    for (int idx = threadIdx.x; idx < kSimtRows * D; idx += blockDim.x) {
        const int r = row0 + idx / D, c = idx % D;
        float v = 0.f;
        if (r < row_end) {
            const int i = r / p.G, h = kvh * p.G + (r - i * p.G);
            v = to_float(q[q_row_offset(p, ((long long)b * p.Sq + i) * p.Hq + h) + c]);
        }
        s_q[idx] = v;
    }

    int lim[kSimtRowsPerWarp];
    float m[kSimtRowsPerWarp], l[kSimtRowsPerWarp], acc[kSimtRowsPerWarp][DPL];
#pragma unroll
    for (int rr = 0; rr < kSimtRowsPerWarp; ++rr) {
        const int r = row0 + warp * kSimtRowsPerWarp + rr;
        lim[rr] = r < row_end ? min(k_hi_split, row_key_limit(p, b, L, r / p.G)) : k_lo;
        m[rr] = kNegInf;
        l[rr] = 0.f;
#pragma unroll
        for (int c = 0; c < DPL; ++c) acc[rr][c] = 0.f;
    }

    const T *kc = reinterpret_cast<const T *>(p.k_cache);
    const T *vc = reinterpret_cast<const T *>(p.v_cache);
    const int32_t *bt_row = p.block_table + (long long)b * p.W;
    const long long tok_stride = (long long)p.Hkv * D;  // elements between tokens of a page

    for (int k0 = k_lo; k0 < k_hi; k0 += kSimtKeys) {
        __syncthreads();  // previous tile fully consumed (and s_q written on the first pass)
        for (int idx = threadIdx.x; idx < kSimtKeys * CPR; idx += blockDim.x) {
            const int kk = idx / CPR, ch = idx % CPR;
            const int j = k0 + kk;
            float kv[EPV], vv[EPV];
            bool ok = false;
            if (j < k_hi) {
                const int id = __ldg(bt_row + j / p.ps);
                if (id >= 0 && (long long)id < p.num_pages) {
                    const long long base = ((long long)id * p.ps + (j % p.ps)) * tok_stride + (long long)kvh * D;
                    load16_to_float<T>(kc + base + ch * EPV, kv);
                    load16_to_float<T>(vc + base + ch * EPV, vv);
                    ok = true;
                } else if (ch == 0) {
                    atomicOr(p.err, (unsigned int)PA_ERRBIT_PAGE_RANGE);
                }
            }
#pragma unroll
            for (int e = 0; e < EPV; ++e) {
                s_k[kk * KS + ch * EPV + e] = ok ? kv[e] : 0.f;
                s_v[kk * KS + ch * EPV + e] = ok ? vv[e] : 0.f;
            }
        }
        __syncthreads();
#pragma unroll
        for (int rr = 0; rr < kSimtRowsPerWarp; ++rr) {
            const float *qr = s_q + (warp * kSimtRowsPerWarp + rr) * D;
            const int j = k0 + lane;
            float sc = 0.f;
#pragma unroll 8
            for (int c = 0; c < D; ++c) sc = fmaf(qr[c], s_k[lane * KS + c], sc);
            sc = (j < lim[rr]) ? sc * p.scale_log2 : kNegInf;
            float mx = sc;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float mn = fmaxf(m[rr], mx);
            const float mu = (mn == kNegInf) ? 0.f : mn;  // -inf - (-inf) guard
            const float al = exp2f(m[rr] - mu);
            const float pj = exp2f(sc - mu);
            float ps_ = pj;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ps_ += __shfl_xor_sync(0xffffffffu, ps_, o);
            l[rr] = l[rr] * al + ps_;
            m[rr] = mn;
#pragma unroll
            for (int c = 0; c < DPL; ++c) acc[rr][c] *= al;
#pragma unroll 4
            for (int kk = 0; kk < kSimtKeys; ++kk) {
                const float w = __shfl_sync(0xffffffffu, pj, kk);
#pragma unroll
                for (int c = 0; c < DPL; ++c) acc[rr][c] = fmaf(w, s_v[kk * KS + c * 32 + lane], acc[rr][c]);
            }
        }
    }

    // finalise (0/0 guard) and store
#pragma unroll
    for (int rr = 0; rr < kSimtRowsPerWarp; ++rr) {
        const int r = row0 + warp * kSimtRowsPerWarp + rr;
        if (r >= row_end) continue;
        const int i = r / p.G, h = kvh * p.G + (r - i * p.G);
        const long long ridx = ((long long)b * p.Sq + i) * p.Hq + h;
        const float inv = l[rr] > 0.f ? 1.f / l[rr] : 0.f;
        const float lse = l[rr] > 0.f ? m[rr] * kLn2 + logf(l[rr]) : kNegInf;
        if (p.split_kv == 1) {
            T *o = reinterpret_cast<T *>(p.out) + ridx * D;
#pragma unroll
            for (int c = 0; c < DPL; ++c) o[c * 32 + lane] = from_float<T>(acc[rr][c] * inv);
            if (lane == 0 && p.lse) p.lse[ridx] = lse;
        } else {
            const long long rows_total = (long long)p.B * p.Sq * p.Hq;
            float *o = reinterpret_cast<float *>(p.out) + ((long long)s * rows_total + ridx) * D;
#pragma unroll
            for (int c = 0; c < DPL; ++c) o[c * 32 + lane] = acc[rr][c] * inv;
            if (lane == 0) p.lse[(long long)s * rows_total + ridx] = lse;
        }
    }
}

template <typename T>
static cudaError_t launch_simt_t(const FwdParams &p, cudaStream_t stream) {
    FwdParams q = p;
    q.row_tiles = (p.rows + kSimtRows - 1) / kSimtRows;
    const long long units = (long long)p.B * p.split_kv * p.Hkv * q.row_tiles;
    if (units <= 0) return cudaSuccess;
    if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (p.D == 256) {
        constexpr size_t smem = (size_t)(2 * kSimtKeys * 257 + kSimtRows * 256) * 4;
        auto kern = paged_attn_simt_kernel<T, 256>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<(unsigned)units, kSimtWarps * 32, smem, stream>>>(q);
    } else if (p.D == 128) {
        paged_attn_simt_kernel<T, 128><<<(unsigned)units, kSimtWarps * 32, 0, stream>>>(q);
    } else {
        paged_attn_simt_kernel<T, 64><<<(unsigned)units, kSimtWarps * 32, 0, stream>>>(q);
    }
    return cudaGetLastError();
}

cudaError_t launch_simt(const FwdParams &p, int dtype, cudaStream_t stream) {
    if (dtype == PA_F32) return launch_simt_t<float>(p, stream);
    if (dtype == PA_BF16) return launch_simt_t<__nv_bfloat16>(p, stream);
    return launch_simt_t<__half>(p, stream);
}

}  // namespace pa
