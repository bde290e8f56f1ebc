// Host-side launchers of the paged-attention kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace pa {

// Tensor-core kernel modes.
enum { MODE_DECODE = 0, MODE_PREFILL = 1, MODE_SPLITS = 2 };

constexpr int kMmaTileKeys = 64;      // keys per pipeline stage
constexpr int kMmaConsumerWarps = 4;  // warps doing QK / softmax / PV
constexpr int kMmaThreads = (kMmaConsumerWarps + 1) * 32;
constexpr int kDecodeRows = 16;       // query rows of one decode CTA (one m16 tile)
constexpr int kPrefillRows = 64;      // query rows of one prefill CTA (4 warps x 16)
// MODE_SPLITS: decode whose splits are short.  A CTA takes kMmaConsumerWarps consecutive splits
// of one (sequence, kv head) and each consumer warp owns one of them; every split is at most
// kGroupSplitPages pages, so a group's page ids fit one warp-wide load.
constexpr int kGroupSplitPages = 32 / kMmaConsumerWarps;
// Stages of one group at most: four splits of kGroupSplitPages pages of up to 64 tokens, 64-key
// stages.  Each has its own full barriers (waited once, at phase 0): the warps consume the ring's
// slots out of step with one another, so a per-slot parity could be two phases behind.
constexpr int kGroupMaxStages = kMmaConsumerWarps * kGroupSplitPages;

// Dynamic shared memory of the tensor-core kernel for a pipeline depth.
size_t mma_smem_bytes(int head_dim, int stages);

cudaError_t launch_mma(const FwdParams &p, int mode, int dtype, const CUtensorMap &tmk, const CUtensorMap &tmv,
                       cudaStream_t stream);
// Variable-length batch (p.q_start set, p.B sequences, total_q packed query tokens).
cudaError_t launch_mma_varlen(const FwdParams &p, long long total_q, int dtype, const CUtensorMap &tmk,
                              const CUtensorMap &tmv, cudaStream_t stream);
// 8-bit pools (kv_dtype PA_FP8_E4M3 or PA_INT8) with per-(page, kv head) scales in p.k_scale /
// p.v_scale; bf16/f16 queries.
cudaError_t launch_mma_kvq(const FwdParams &p, int mode, int dtype, int kv_dtype, const CUtensorMap &tmk,
                           const CUtensorMap &tmv, cudaStream_t stream);
// tcgen05 prefill: bf16/f16, head_dim 128, (Hq/Hkv) dividing 128.
size_t tc05_smem_bytes();
cudaError_t launch_tc05(const FwdParams &p, int dtype, const CUtensorMap &tmq, const CUtensorMap &tmk,
                        const CUtensorMap &tmv, const CUtensorMap &tmo, cudaStream_t stream);
// Variable-length batch (p.q_start, total_q packed tokens, at most kTc05VarlenMaxBatch sequences):
// the sequences of at least 64 query rows, on at most max_ctas SMs (0: every SM).
constexpr int kTc05VarlenMaxBatch = 1024;
cudaError_t launch_tc05_varlen(const FwdParams &p, long long total_q, int dtype, const CUtensorMap &tmq,
                               const CUtensorMap &tmk, const CUtensorMap &tmv, const CUtensorMap &tmo,
                               int max_ctas, cudaStream_t stream);
cudaError_t launch_simt(const FwdParams &p, int dtype, cudaStream_t stream);
// One query row per (sequence, kv head), bf16/f16, head_dim 64/128: CUDA cores over the TMA ring.
cudaError_t launch_simt_decode(const FwdParams &p, int dtype, const CUtensorMap &tmk, const CUtensorMap &tmv,
                               cudaStream_t stream);
// head_dim 256, bf16/f16: transposed products, 8-row units.
cudaError_t launch_mma_t(const FwdParams &p, int dtype, const CUtensorMap &tmk, const CUtensorMap &tmv,
                         cudaStream_t stream);
cudaError_t launch_combine(const float *part_out, const float *part_lse, int S, long long rows, int D,
                           int out_dtype, void *out, float *lse, cudaStream_t stream);
cudaError_t launch_plan(const int32_t *seq_lens, int B, int ps, int S, int32_t *plan, cudaStream_t stream);
cudaError_t launch_wait_probe(unsigned int *err, unsigned long long limit_ns, cudaStream_t stream);
cudaError_t launch_gather(const void *cache, const int32_t *block_table, const int32_t *seq_lens, int B, int W,
                          int ps, int Hkv, int D, int esize, long long num_pages, int out_tokens, void *out,
                          unsigned int *err, cudaStream_t stream);

}  // namespace pa
