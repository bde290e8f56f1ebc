// Device-side building blocks shared by the paged-attention kernels (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "paged_attn.h"

namespace pa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_huge_valf();
// A pipeline wait that has not completed after this long is abandoned (error bit
// PA_ERRBIT_TIMEOUT) so that a broken pipeline never hangs the GPU.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// Everything a forward kernel needs.  Pointers are device pointers.
struct FwdParams {
    const void *q;
    const int32_t *block_table;
    const int32_t *seq_lens;
    const int32_t *q_offset;   // nullable: seq_lens[b] - Sq
    void *out;                 // S == 1: [B,Sq,Hq,D] dtype; S > 1: float [S,B,Sq,Hq,D]
    float *lse;                // S == 1: [B,Sq,Hq] or null; S > 1: [S,B,Sq,Hq]
    const void *k_cache;       // raw pools (used by the CUDA-core kernel)
    const void *v_cache;
    const float *k_scale;      // FP8 pools: [num_pages, Hkv] per-(page, kv head) scales; else null
    const float *v_scale;
    const int32_t *q_start;    // variable-length batches: [B + 1] first packed query token per sequence; else null
    long long rows_total;      // query rows (tokens x heads) of the whole batch: the stride of one split's partials
    long long q_stride;        // elements between consecutive query tokens of q (Hq * D when dense)
    unsigned int *err;         // device error word
    long long num_pages;
    int B, Sq, Hq, Hkv, D, ps, W;
    int G;                     // Hq / Hkv
    int rows;                  // Sq * G query rows per (sequence, kv head)
    int causal, split_kv;
    float scale_log2;          // scale * log2(e)
    int row_tiles;             // query-row tiles per (sequence, kv head, split)
    int varlen_rows_cap;       // variable-length one-grid kernel: skip sequences with at least this many
                               // query rows (another kernel takes them); 0: take every sequence
};

// ------------------------------------------------------------------ small helpers
// Element offset in q of query row ridx = token * Hq + head (tokens q_stride elements apart).
__device__ __forceinline__ long long q_row_offset(const FwdParams &p, long long ridx) {
    const long long tok = ridx / p.Hq;
    return tok * p.q_stride + (ridx - tok * p.Hq) * (long long)p.D;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Split plan of rocMLIR PR #2371 in pages: run s of sequence b covers pages
// [min(s*per, nblk), min((s+1)*per, nblk)), per = ceil(nblk / S).
__device__ __forceinline__ void split_pages(int L, int ps, int S, int s, int &p0, int &p1) {
    const int nblk = L > 0 ? (L + ps - 1) / ps : 0;
    const int per = (nblk + S - 1) / S;
    long long a = (long long)s * per, e = (long long)(s + 1) * per;
    p0 = (int)(a < nblk ? a : nblk);
    p1 = (int)(e < nblk ? e : nblk);
}

// Exclusive key bound for query row i of sequence b, which has Sq query tokens (causal reach
// incl. q_offset; without one the queries are the sequence's last Sq tokens).
__device__ __forceinline__ int row_key_limit(const FwdParams &p, int b, int L, int i, int Sq) {
    if (!p.causal) return L;
    const long long qoff = p.q_offset ? (long long)p.q_offset[b] : (long long)L - Sq;
    long long reach = qoff + i + 1;
    reach = reach < 0 ? 0 : reach;
    return (int)(reach < L ? reach : L);
}

__device__ __forceinline__ int row_key_limit(const FwdParams &p, int b, int L, int i) {
    return row_key_limit(p, b, L, i, p.Sq);
}

// 2^x by the hardware approximation (ex2.approx, subnormal results flushed to 0; 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity; gives up after limit_ns (kWaitLimitNs in every
// kernel) and records PA_ERRBIT_TIMEOUT.  Returns false on time-out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned int *err,
                                          unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
#pragma unroll 1  // one copy per call site: warp-specialised kernels inline many of these
        for (int k = 0; k < 64; ++k)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) {
            atomicOr(err, (unsigned int)PA_ERRBIT_TIMEOUT);
            return false;
        }
    }
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 4-D tiled load global -> shared, completion counted on `bar` (bytes).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *m, uint32_t bar, int c0, int c1,
                                            int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

// 3-D tiled load global -> shared, completion counted on `bar` (bytes).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *m, uint32_t bar, int c0, int c1,
                                            int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

// 4-D tiled store shared -> global in the bulk-group completion scheme; the box is clipped to the
// tensor's bounds (coordinates must not be negative).
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *m, uint32_t src, int c0, int c1, int c2, int c3) {
    asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(m)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Every committed bulk store has finished reading its shared-memory source.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Every committed bulk store has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier over `count` threads (id 1.. are free; 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ------------------------------------------------------------------ warp MMA (m16n8k16)
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                            uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                                  uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

template <typename T>
struct MmaOp;

template <>
struct MmaOp<__nv_bfloat16> {
    __device__ __forceinline__ static void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
        asm(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    // two floats -> packed pair (low half = first), round to nearest even
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&v);
    }
    __device__ __forceinline__ static float2 unpack(uint32_t v) {
        __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162 *>(&v);
        return __bfloat1622float2(h);
    }
};

template <>
struct MmaOp<__half> {
    __device__ __forceinline__ static void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
        asm(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&v);
    }
    __device__ __forceinline__ static float2 unpack(uint32_t v) {
        __half2 h = *reinterpret_cast<__half2 *>(&v);
        return __half22float2(h);
    }
};

// ------------------------------------------------------------------ element conversion
__device__ __forceinline__ float to_float(float x) { return x; }
__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_float(__half x) { return __half2float(x); }

template <typename T>
__device__ __forceinline__ T from_float(float x);
template <>
__device__ __forceinline__ float from_float<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <>
__device__ __forceinline__ __half from_float<__half>(float x) { return __float2half_rn(x); }

}  // namespace pa
