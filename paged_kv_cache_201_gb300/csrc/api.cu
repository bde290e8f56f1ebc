// C ABI of the paged-attention library: argument validation, kernel choice,
// TMA descriptor set-up and launches.  Everything here runs on the host; the
// arithmetic of the operation lives in the kernels.
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "kernels.h"

namespace {

// Device error word: kernels OR PA_ERRBIT_* bits into it; paged_attn_last_error_word reads and clears it.
__device__ unsigned int g_pa_error_word;

constexpr int kMaxDevices = 128;
unsigned int *g_err_ptr[kMaxDevices];
std::mutex g_err_mu;

int error_word_ptr(unsigned int **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ECUDA;
    std::lock_guard<std::mutex> lk(g_err_mu);
    if (!g_err_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_pa_error_word) != cudaSuccess) return PA_ECUDA;
        g_err_ptr[dev] = static_cast<unsigned int *>(ptr);
    }
    *out = g_err_ptr[dev];
    return PA_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

thread_local cudaError_t t_last_cuda_error = cudaSuccess;

// PA_OK, or PA_ECUDA after remembering e for paged_attn_cuda_error_string.
int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return PA_OK;
    t_last_cuda_error = e;
    return PA_ECUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int esize_of(int dtype) { return dtype == PA_F32 ? 4 : 2; }

// Shape checks shared by the forward and gather entry points.
int check_dims(const pa_dims *d) {
    if (!d) return PA_EINVAL;
    if (d->dtype != PA_F32 && d->dtype != PA_F16 && d->dtype != PA_BF16) return PA_EDTYPE;
    if (d->batch < 0 || d->q_len < 0 || d->num_q_heads <= 0 || d->num_kv_heads <= 0 || d->bt_stride < 0)
        return PA_EINVAL;
    if (d->num_q_heads % d->num_kv_heads != 0) return PA_EINVAL;
    if (d->head_dim != 64 && d->head_dim != 128 && d->head_dim != 256) return PA_EUNSUPPORTED;
    if (d->page_size != 16 && d->page_size != 32 && d->page_size != 64) return PA_EUNSUPPORTED;
    if (d->num_pages < 1) return PA_EINVAL;
    if (d->num_pages * (int64_t)d->page_size >= (int64_t)1 << 31) return PA_EUNSUPPORTED;
    if ((int64_t)d->bt_stride * d->page_size >= (int64_t)1 << 31) return PA_EUNSUPPORTED;
    if ((int64_t)d->q_len * (d->num_q_heads / d->num_kv_heads) >= (int64_t)1 << 31) return PA_EUNSUPPORTED;
    // q's token stride: dense, or at least a token's heads and keeping every row 16-byte aligned
    if (d->q_stride != 0 &&
        (d->q_stride < (int64_t)d->num_q_heads * d->head_dim || (d->q_stride * esize_of(d->dtype)) % 16 != 0 ||
         d->q_stride >= (int64_t)1 << 40))
        return PA_EINVAL;
    return PA_OK;
}

// Elements between consecutive query tokens of q.
int64_t q_token_stride(const pa_dims *d) {
    return d->q_stride ? d->q_stride : (int64_t)d->num_q_heads * d->head_dim;
}

CUtensorMapDataType tma_dtype(int dtype) {
    return dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

// 4-D view of one pool for TMA: (d within a 64-element half, token, half, kv head).
// halves_per_box = D/64 copies a page's whole rows (decode kernel); 1 copies one half-row
// (tcgen05 kernel, which keeps each half of a tile contiguous).
int make_pool_map(CUtensorMap *m, const void *base, const pa_dims *d, int halves_per_box) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return PA_ECUDA;
    const cuuint64_t esz = 2;
    const cuuint64_t D = (cuuint64_t)d->head_dim, Hkv = (cuuint64_t)d->num_kv_heads;
    const cuuint64_t dims[4] = {64, (cuuint64_t)d->num_pages * (cuuint64_t)d->page_size, D / 64, Hkv};
    const cuuint64_t strides[3] = {Hkv * D * esz, 64 * esz, D * esz};
    const cuuint32_t box[4] = {64, (cuuint32_t)d->page_size, (cuuint32_t)halves_per_box, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, tma_dtype(d->dtype), 4, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ECUDA;
}

// 3-D view of one 8-bit pool (E4M3 or int8 elements) for TMA: (byte within a row, token, kv head); one box = the page_size
// rows of one page and one kv head.  128-byte rows (head_dim 128) land with the 128-byte swizzle,
// which the kernel's conflict-free operand loads rely on; 64-byte rows land as they are.
int make_pool_map_q8(CUtensorMap *m, const void *base, const pa_dims *d) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return PA_ECUDA;
    const cuuint64_t D = (cuuint64_t)d->head_dim, Hkv = (cuuint64_t)d->num_kv_heads;
    const cuuint64_t dims[3] = {D, (cuuint64_t)d->num_pages * (cuuint64_t)d->page_size, Hkv};
    const cuuint64_t strides[2] = {Hkv * D, D};
    const cuuint32_t box[3] = {(cuuint32_t)D, (cuuint32_t)d->page_size, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapSwizzle swz = d->head_dim == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ECUDA;
}

// 4-D view of q for the tcgen05 kernel: (d within a half, half, query head, token of B*Sq, or of
// the T packed tokens of a variable-length batch); one box = one half of a 128-row tile: 128/G
// consecutive tokens x the G heads of a kv head.
int make_q_map(CUtensorMap *m, const void *q, const pa_dims *d, bool varlen = false) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return PA_ECUDA;
    const cuuint64_t esz = 2;
    const cuuint64_t D = (cuuint64_t)d->head_dim, Hq = (cuuint64_t)d->num_q_heads;
    const int G = d->num_q_heads / d->num_kv_heads;
    const cuuint64_t tokens = varlen ? (cuuint64_t)d->q_len : (cuuint64_t)d->batch * (cuuint64_t)d->q_len;
    const cuuint64_t dims[4] = {64, D / 64, Hq, tokens};
    const cuuint64_t strides[3] = {64 * esz, D * esz, (cuuint64_t)q_token_stride(d) * esz};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)G, (cuuint32_t)(128 / G)};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(m, tma_dtype(d->dtype), 4, const_cast<void *>(q), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ECUDA;
}

// 4-D view of the tcgen05 kernel's output for TMA stores: (d, query head, token, sequence) for the
// final rows (split_kv = 1, q's element type) or (d, query head, token, split x B + sequence) for
// the fp32 partials; for a variable-length batch (d, query head, packed token, split).  One box =
// one epilogue warp's 32 rows (min(G, 32) heads x max(32 / G, 1) tokens) x 128 bytes of columns,
// 128-byte swizzled; tokens past Sq fall outside and are clipped (a variable-length batch's
// kernel stores rows that run past their sequence itself).
int make_tc05_out_map(CUtensorMap *m, void *out, const pa_dims *d, int split_kv, bool varlen = false) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return PA_ECUDA;
    const bool part = split_kv > 1;
    const cuuint64_t esz = part ? 4 : 2;
    const cuuint64_t D = (cuuint64_t)d->head_dim, Hq = (cuuint64_t)d->num_q_heads, Sq = (cuuint64_t)d->q_len;
    const int G = d->num_q_heads / d->num_kv_heads;
    const cuuint64_t nsp = (cuuint64_t)(part ? split_kv : 1);
    const cuuint64_t dims[4] = {D, Hq, Sq, varlen ? nsp : (cuuint64_t)d->batch * nsp};
    const cuuint64_t strides[3] = {D * esz, Hq * D * esz, Sq * Hq * D * esz};
    const cuuint32_t bh = (cuuint32_t)(G < 32 ? G : 32), bt = (cuuint32_t)(G < 32 ? 32 / G : 1);
    const cuuint32_t box[4] = {(cuuint32_t)(128 / esz), bh, bt, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapDataType ty = part ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : tma_dtype(d->dtype);
    CUresult r = enc(m, ty, 4, out, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ECUDA;
}

// The split-group decode kernel needs every split within kGroupSplitPages pages; W (bt_stride)
// pages bound every sequence's page count.
bool split_group_fits(const pa_dims *d, int split_kv) {
    return split_kv >= 1 && ((int64_t)d->bt_stride + split_kv - 1) / split_kv <= pa::kGroupSplitPages;
}

// Multiprocessor count of the current device (cached per device; 152 if it cannot be read).
int device_sm_count() {
    static std::atomic<int> cached[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 152;
    int v = cached[dev].load(std::memory_order_relaxed);
    if (!v) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) return 152;
        cached[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

bool tc05_supports(const pa_dims *d) {
    const int G = d->num_q_heads / d->num_kv_heads;
    return d->dtype != PA_F32 && d->head_dim == 128 && G <= 128 && (128 % G) == 0 &&
           (int64_t)d->batch * d->q_len < ((int64_t)1 << 31);
}

int choose_variant(const pa_dims *d) {
    if (d->dtype == PA_F32) return PA_VARIANT_SIMT;
    const int64_t rows = (int64_t)d->q_len * (d->num_q_heads / d->num_kv_heads);
    if (rows <= 1) return PA_VARIANT_SIMT;  // single-head decode: a 16-row tile would be 1/16 used
    if (d->head_dim == 256) return PA_VARIANT_MMA_T;
    if (rows <= pa::kDecodeRows) return PA_VARIANT_MMA_DECODE;
    // 128-row tcgen05 tiles once at least half a tile of rows is real work
    if (rows >= 64 && tc05_supports(d)) return PA_VARIANT_TC05_PREFILL;
    return PA_VARIANT_MMA_PREFILL;
}

// Pointer and alignment checks shared by the forward entry points.
int check_fwd_pointers(const void *q, const void *k_cache, const void *v_cache, const int32_t *block_table,
                       const int32_t *seq_lens, const int32_t *q_offset, int split_kv, const void *out,
                       const float *lse) {
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out) return PA_EINVAL;
    if (split_kv > 1 && !lse) return PA_EINVAL;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return PA_EINVAL;
    if ((reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
        (reinterpret_cast<uintptr_t>(seq_lens) & 3u) || (reinterpret_cast<uintptr_t>(q_offset) & 3u))
        return PA_EINVAL;
    return PA_OK;
}

pa::FwdParams fill_params(const void *q, const void *k_cache, const void *v_cache, const int32_t *block_table,
                          const int32_t *seq_lens, int causal, const int32_t *q_offset, int split_kv, float scale,
                          void *out, float *lse, const pa_dims *dims, unsigned int *err) {
    pa::FwdParams p{};
    p.q = q;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.q_offset = q_offset;
    p.out = out;
    p.lse = lse;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.err = err;
    p.num_pages = dims->num_pages;
    p.B = dims->batch;
    p.Sq = dims->q_len;
    p.Hq = dims->num_q_heads;
    p.Hkv = dims->num_kv_heads;
    p.D = dims->head_dim;
    p.ps = dims->page_size;
    p.W = dims->bt_stride;
    p.G = dims->num_q_heads / dims->num_kv_heads;
    p.rows = dims->q_len * p.G;
    p.causal = causal ? 1 : 0;
    p.split_kv = split_kv;
    p.scale_log2 = scale * pa::kLog2e;
    p.row_tiles = 1;
    p.rows_total = (long long)dims->batch * dims->q_len * dims->num_q_heads;
    p.q_stride = q_token_stride(dims);
    return p;
}

// Split forward into a workspace, then the fp32 combine (rocMLIR PR #2371): the body of the
// single-call entry points.  fwd(S, part_out, part_lse) runs the forward with S partitions.
template <typename Fwd>
int splitkv_call(const pa_dims *dims, int split_kv, void *out, float *lse, void *workspace, int64_t workspace_bytes,
                 int num_sms, int64_t device_bytes, void *stream, Fwd fwd) {
    if (split_kv < 0 || split_kv > 65535) return PA_EINVAL;
    if (split_kv == 0) {
        split_kv = paged_attn_auto_split(dims, num_sms, device_bytes);
        if (split_kv < 0) return split_kv;
    }
    if (split_kv == 1) return fwd(1, out, lse);
    const int64_t need = paged_attn_workspace_bytes(dims, split_kv, num_sms, device_bytes);
    if (need < 0) return (int)need;
    const int64_t rows = (int64_t)dims->batch * dims->q_len * dims->num_q_heads;
    if (rows == 0) return PA_OK;
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return PA_EINVAL;
    if (!out || !aligned16(out) || (reinterpret_cast<uintptr_t>(lse) & 3u)) return PA_EINVAL;
    float *part_out = static_cast<float *>(workspace);
    float *part_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                                ((int64_t)split_kv * rows * dims->head_dim * 4 + 255) / 256 * 256);
    int rc = fwd(split_kv, part_out, part_lse);
    if (rc != PA_OK) return rc;
    return paged_attn_combine(part_out, part_lse, split_kv, rows, dims->head_dim, dims->dtype, out, lse, stream);
}

}  // namespace

extern "C" {

int paged_attn_fwd_variant(const void *q, const void *k_cache, const void *v_cache, const int32_t *block_table,
                           const int32_t *seq_lens, int causal, const int32_t *q_offset, int split_kv,
                           float scale, void *out, float *lse, const pa_dims *dims, int variant, void *stream) {
    int rc = check_dims(dims);
    if (rc != PA_OK) return rc;
    if (split_kv < 1 || split_kv > 65535) return PA_EINVAL;
    if (!isfinite(scale)) return PA_EINVAL;
    const int64_t nrows = (int64_t)dims->batch * dims->q_len * dims->num_q_heads;
    if (nrows == 0) return PA_OK;
    rc = check_fwd_pointers(q, k_cache, v_cache, block_table, seq_lens, q_offset, split_kv, out, lse);
    if (rc != PA_OK) return rc;
    const bool planned = variant == PA_VARIANT_AUTO;
    if (planned) {
        variant = choose_variant(dims);
        // the tcgen05 kernel takes its row maximum over unscaled scores, which needs scale > 0
        if (variant == PA_VARIANT_TC05_PREFILL && !(scale > 0.f)) variant = PA_VARIANT_MMA_PREFILL;
    }
    const int G = dims->num_q_heads / dims->num_kv_heads;
    const int rows = dims->q_len * G;
    switch (variant) {
        case PA_VARIANT_SIMT:
            break;
        case PA_VARIANT_MMA_DECODE:
            if (dims->dtype == PA_F32 || rows > pa::kDecodeRows || dims->head_dim == 256) return PA_EUNSUPPORTED;
            break;
        case PA_VARIANT_MMA_PREFILL:
            if (dims->dtype == PA_F32 || dims->head_dim == 256) return PA_EUNSUPPORTED;
            break;
        case PA_VARIANT_MMA_T:
            if (dims->dtype == PA_F32 || dims->head_dim != 256) return PA_EUNSUPPORTED;
            break;
        case PA_VARIANT_MMA_SPLIT_GROUP:
            if (dims->dtype == PA_F32 || rows > pa::kDecodeRows || dims->head_dim == 256 ||
                !split_group_fits(dims, split_kv))
                return PA_EUNSUPPORTED;
            break;
        case PA_VARIANT_TC05_PREFILL:
            if (!tc05_supports(dims) || !(scale > 0.f)) return PA_EUNSUPPORTED;
            break;
        default:
            return PA_EINVAL;
    }
    if (dims->batch == 0 || dims->q_len == 0) return PA_OK;

    unsigned int *err = nullptr;
    rc = error_word_ptr(&err);
    if (rc != PA_OK) return rc;

    pa::FwdParams p = fill_params(q, k_cache, v_cache, block_table, seq_lens, causal, q_offset, split_kv, scale,
                                  out, lse, dims, err);

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (variant == PA_VARIANT_SIMT && rows == 1 && dims->dtype != PA_F32 && dims->head_dim != 256) {
        // single-row decode: the CUDA-core kernel over the TMA ring
        CUtensorMap tmk, tmv;
        if ((rc = make_pool_map(&tmk, k_cache, dims, dims->head_dim / 64)) != PA_OK) return rc;
        if ((rc = make_pool_map(&tmv, v_cache, dims, dims->head_dim / 64)) != PA_OK) return rc;
        e = pa::launch_simt_decode(p, dims->dtype, tmk, tmv, st);
    } else if (variant == PA_VARIANT_SIMT) {
        e = pa::launch_simt(p, dims->dtype, st);
    } else if (variant == PA_VARIANT_MMA_T) {
        CUtensorMap tmk, tmv;
        if ((rc = make_pool_map(&tmk, k_cache, dims, dims->head_dim / 64)) != PA_OK) return rc;
        if ((rc = make_pool_map(&tmv, v_cache, dims, dims->head_dim / 64)) != PA_OK) return rc;
        e = pa::launch_mma_t(p, dims->dtype, tmk, tmv, st);
    } else if (variant == PA_VARIANT_TC05_PREFILL) {
        CUtensorMap tmq, tmk, tmv, tmo;
        if ((rc = make_q_map(&tmq, q, dims)) != PA_OK) return rc;
        if ((rc = make_pool_map(&tmk, k_cache, dims, 1)) != PA_OK) return rc;
        if ((rc = make_pool_map(&tmv, v_cache, dims, 1)) != PA_OK) return rc;
        if ((rc = make_tc05_out_map(&tmo, out, dims, split_kv)) != PA_OK) return rc;
        e = pa::launch_tc05(p, dims->dtype, tmq, tmk, tmv, tmo, st);
    } else {
        CUtensorMap tmk, tmv;
        if ((rc = make_pool_map(&tmk, k_cache, dims, dims->head_dim / 64)) != PA_OK) return rc;
        if ((rc = make_pool_map(&tmv, v_cache, dims, dims->head_dim / 64)) != PA_OK) return rc;
        int mode = variant == PA_VARIANT_MMA_PREFILL ? pa::MODE_PREFILL : pa::MODE_DECODE;
        if (mode == pa::MODE_PREFILL) p.row_tiles = (rows + pa::kPrefillRows - 1) / pa::kPrefillRows;
        // Short splits in more CTAs than two per SM hold at once: a CTA per four splits, one warp
        // per split.  With fewer units the one-CTA-per-split launch is already a single wave, and
        // its four warps sharing each split's keys finish sooner.
        if (variant == PA_VARIANT_MMA_SPLIT_GROUP ||
            (planned && mode == pa::MODE_DECODE && split_kv >= 2 && split_group_fits(dims, split_kv) &&
             (int64_t)dims->batch * split_kv * dims->num_kv_heads > 2LL * device_sm_count()))
            mode = pa::MODE_SPLITS;
        e = pa::launch_mma(p, mode, dims->dtype, tmk, tmv, st);
    }
    return cuda_status(e);
}

int paged_attn_fwd(const void *q, const void *k_cache, const void *v_cache, const int32_t *block_table,
                   const int32_t *seq_lens, int causal, const int32_t *q_offset, int split_kv, float scale,
                   void *out, float *lse, const pa_dims *dims, void *stream) {
    return paged_attn_fwd_variant(q, k_cache, v_cache, block_table, seq_lens, causal, q_offset, split_kv, scale, out,
                                  lse, dims, PA_VARIANT_AUTO, stream);
}

int paged_attn_auto_split(const pa_dims *dims, int num_sms, int64_t device_bytes) {
    int rc = check_dims(dims);
    if (rc != PA_OK) return rc;
    if (num_sms < 1) return PA_EINVAL;
    const int G = dims->num_q_heads / dims->num_kv_heads;
    const int64_t rows = (int64_t)dims->q_len * G;
    // query-row tiles per (sequence, kv head) of the kernel the planner would pick
    const int64_t tile_rows = dims->head_dim == 256 ? 8 : (rows <= pa::kDecodeRows ? pa::kDecodeRows : 128);
    const int64_t row_tiles = (rows + tile_rows - 1) / tile_rows;
    const int64_t units1 = (int64_t)dims->batch * dims->num_kv_heads * (row_tiles > 0 ? row_tiles : 1);
    const int64_t want = 2LL * num_sms;  // two waves of units
    int64_t S = units1 > 0 ? (want + units1 - 1) / units1 : 1;
    if (S > dims->bt_stride) S = dims->bt_stride;
    if (S > 256) S = 256;
    if (S < 1) S = 1;
    // workspace budget: device memory / 8 clamped to [1 GiB, 8 GiB] (1.5 GiB when unknown)
    int64_t budget = device_bytes > 0 ? device_bytes / 8 : (int64_t)3 << 29;
    if (budget < ((int64_t)1 << 30)) budget = (int64_t)1 << 30;
    if (budget > ((int64_t)8 << 30)) budget = (int64_t)8 << 30;
    const int64_t per_split = (int64_t)dims->batch * dims->q_len * dims->num_q_heads * (dims->head_dim + 1) * 4;
    while (S > 1 && S * per_split > budget) --S;
    return (int)S;
}

int64_t paged_attn_workspace_bytes(const pa_dims *dims, int split_kv, int num_sms, int64_t device_bytes) {
    int rc = check_dims(dims);
    if (rc != PA_OK) return rc;
    if (split_kv < 0 || split_kv > 65535) return PA_EINVAL;
    if (split_kv == 0) {
        split_kv = paged_attn_auto_split(dims, num_sms, device_bytes);
        if (split_kv < 0) return split_kv;
    }
    if (split_kv == 1) return 0;
    const int64_t rows = (int64_t)dims->batch * dims->q_len * dims->num_q_heads;
    const int64_t out_b = ((int64_t)split_kv * rows * dims->head_dim * 4 + 255) / 256 * 256;
    const int64_t lse_b = ((int64_t)split_kv * rows * 4 + 255) / 256 * 256;
    return out_b + lse_b;
}

int paged_attn_fwd_splitkv(const void *q, const void *k_cache, const void *v_cache, const int32_t *block_table,
                           const int32_t *seq_lens, int causal, const int32_t *q_offset, int split_kv, float scale,
                           void *out, float *lse, const pa_dims *dims, void *workspace, int64_t workspace_bytes,
                           int num_sms, int64_t device_bytes, void *stream) {
    int rc = check_dims(dims);
    if (rc != PA_OK) return rc;
    return splitkv_call(dims, split_kv, out, lse, workspace, workspace_bytes, num_sms, device_bytes, stream,
                        [&](int S, void *o, float *l) {
                            return paged_attn_fwd(q, k_cache, v_cache, block_table, seq_lens, causal, q_offset, S,
                                                  scale, o, l, dims, stream);
                        });
}

int paged_attn_fwd_kvq(const void *q, const void *k_cache, const void *v_cache, const float *k_scale,
                       const float *v_scale, int kv_dtype, const int32_t *block_table, const int32_t *seq_lens,
                       int causal, const int32_t *q_offset, int split_kv, float scale, void *out, float *lse,
                       const pa_dims *dims, void *stream) {
    int rc = check_dims(dims);
    if (rc != PA_OK) return rc;
    if (dims->dtype == PA_F32 || (kv_dtype != PA_FP8_E4M3 && kv_dtype != PA_INT8)) return PA_EDTYPE;
    if (dims->head_dim == 256) return PA_EUNSUPPORTED;
    if (split_kv < 1 || split_kv > 65535) return PA_EINVAL;
    if (!isfinite(scale)) return PA_EINVAL;
    const int64_t nrows = (int64_t)dims->batch * dims->q_len * dims->num_q_heads;
    if (nrows == 0) return PA_OK;
    rc = check_fwd_pointers(q, k_cache, v_cache, block_table, seq_lens, q_offset, split_kv, out, lse);
    if (rc != PA_OK) return rc;
    if (!k_scale || !v_scale || (reinterpret_cast<uintptr_t>(k_scale) & 3u) ||
        (reinterpret_cast<uintptr_t>(v_scale) & 3u))
        return PA_EINVAL;

    unsigned int *err = nullptr;
    rc = error_word_ptr(&err);
    if (rc != PA_OK) return rc;
    pa::FwdParams p = fill_params(q, k_cache, v_cache, block_table, seq_lens, causal, q_offset, split_kv, scale,
                                  out, lse, dims, err);
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    CUtensorMap tmk, tmv;
    if ((rc = make_pool_map_q8(&tmk, k_cache, dims)) != PA_OK) return rc;
    if ((rc = make_pool_map_q8(&tmv, v_cache, dims)) != PA_OK) return rc;
    const int mode = p.rows <= pa::kDecodeRows ? pa::MODE_DECODE : pa::MODE_PREFILL;
    if (mode == pa::MODE_PREFILL) p.row_tiles = (p.rows + pa::kPrefillRows - 1) / pa::kPrefillRows;
    return cuda_status(pa::launch_mma_kvq(p, mode, dims->dtype, kv_dtype, tmk, tmv, static_cast<cudaStream_t>(stream)));
}

int paged_attn_fwd_kvq_splitkv(const void *q, const void *k_cache, const void *v_cache, const float *k_scale,
                               const float *v_scale, int kv_dtype, const int32_t *block_table,
                               const int32_t *seq_lens, int causal, const int32_t *q_offset, int split_kv,
                               float scale, void *out, float *lse, const pa_dims *dims, void *workspace,
                               int64_t workspace_bytes, int num_sms, int64_t device_bytes, void *stream) {
    int rc = check_dims(dims);
    if (rc != PA_OK) return rc;
    if (dims->dtype == PA_F32 || (kv_dtype != PA_FP8_E4M3 && kv_dtype != PA_INT8)) return PA_EDTYPE;
    return splitkv_call(dims, split_kv, out, lse, workspace, workspace_bytes, num_sms, device_bytes, stream,
                        [&](int S, void *o, float *l) {
                            return paged_attn_fwd_kvq(q, k_cache, v_cache, k_scale, v_scale, kv_dtype, block_table,
                                                      seq_lens, causal, q_offset, S, scale, o, l, dims, stream);
                        });
}

namespace {

// The tcgen05 kernel's stream for paged_attn_fwd_varlen_overlap: one per device, created on first
// use at the highest priority, so that when both kernels are ready its CTAs are placed first.
int overlap_stream(cudaStream_t *out) {
    static std::mutex mu;
    static cudaStream_t streams[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ECUDA;
    std::lock_guard<std::mutex> lk(mu);
    if (!streams[dev]) {
        int least = 0, greatest = 0;
        if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) return PA_ECUDA;
        if (cudaStreamCreateWithPriority(&streams[dev], cudaStreamNonBlocking, greatest) != cudaSuccess)
            return PA_ECUDA;
    }
    *out = streams[dev];
    return PA_OK;
}

// SMs for the tcgen05 kernel when it runs beside the short-sequence kernel: about as many as make
// its estimated time equal the short sequences' K/V read time.  The rates are the kernels' measured
// ones on GB300 (useful flops per SM of causal prefill tiles; the decode kernel's read rate).  The
// estimate is raised by 1.3 because the two errors cost differently: on the mixed benchmark batch,
// half the balancing share made the call 1.9 times slower, twice the share only 1.02 times, and
// 1.2-1.5 times the share was fastest.  0 when the batch has no work of one kind (nothing to
// overlap).
int overlap_sms(const pa_dims *d, const pa_varlen_hint *h, int sms) {
    if (!h || h->long_pairs <= 0 || h->short_kv_tokens <= 0 || sms < 16) return 0;
    const double flops = 4.0 * d->head_dim * d->num_q_heads * (double)h->long_pairs;
    const double flops_per_sm = d->dtype == PA_BF16 ? 4.4e12 : 5.8e12;
    const double esz = d->dtype == PA_F32 ? 4.0 : 2.0;
    const double bytes = 2.0 * (double)h->short_kv_tokens * d->num_kv_heads * d->head_dim * esz;
    const double t_short = bytes / 6.9e12;
    double n = ceil(1.3 * flops / (flops_per_sm * t_short));
    if (n < 8) n = 8;
    if (n > sms * 3 / 4) n = sms * 3 / 4;  // keep enough SMs streaming the short sequences' pages
    return (int)n;
}

int varlen_call(const void *q, const void *k_cache, const void *v_cache, const int32_t *block_table,
                const int32_t *seq_lens, const int32_t *q_start, int causal, const int32_t *q_offset, int split_kv,
                float scale, void *out, float *lse, const pa_dims *dims, const pa_varlen_hint *hint,
                void *stream) {
    int rc = check_dims(dims);
    if (rc != PA_OK) return rc;
    if (dims->dtype == PA_F32) return PA_EDTYPE;
    if (dims->head_dim == 256) return PA_EUNSUPPORTED;
    if (split_kv < 1 || split_kv > 65535) return PA_EINVAL;
    if (!isfinite(scale)) return PA_EINVAL;
    if (dims->batch == 0 || dims->q_len == 0) return PA_OK;  // no query token
    rc = check_fwd_pointers(q, k_cache, v_cache, block_table, seq_lens, q_offset, split_kv, out, lse);
    if (rc != PA_OK) return rc;
    if (!q_start || (reinterpret_cast<uintptr_t>(q_start) & 3u)) return PA_EINVAL;
    unsigned int *err = nullptr;
    rc = error_word_ptr(&err);
    if (rc != PA_OK) return rc;
    pa::FwdParams p = fill_params(q, k_cache, v_cache, block_table, seq_lens, causal, q_offset, split_kv, scale,
                                  out, lse, dims, err);
    // q_len is the total packed token count T; per-sequence counts come from q_start
    p.q_start = q_start;
    p.Sq = 0;
    p.rows = 0;
    p.rows_total = (long long)dims->q_len * dims->num_q_heads;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    CUtensorMap tmk, tmv;
    if ((rc = make_pool_map(&tmk, k_cache, dims, dims->head_dim / 64)) != PA_OK) return rc;
    if ((rc = make_pool_map(&tmv, v_cache, dims, dims->head_dim / 64)) != PA_OK) return rc;
    // Sequences of at least 64 query rows go to the tcgen05 kernel when it takes the shape (it
    // finds them on the device, from q_start); the one-grid kernel takes the rest, or everything.
    if (!(tc05_supports(dims) && scale > 0.f && dims->batch <= pa::kTc05VarlenMaxBatch))
        return cuda_status(pa::launch_mma_varlen(p, dims->q_len, dims->dtype, tmk, tmv, st));
    CUtensorMap tmq, tmk5, tmv5, tmo;
    if ((rc = make_q_map(&tmq, q, dims, true)) != PA_OK) return rc;
    if ((rc = make_pool_map(&tmk5, k_cache, dims, 1)) != PA_OK) return rc;
    if ((rc = make_pool_map(&tmv5, v_cache, dims, 1)) != PA_OK) return rc;
    if ((rc = make_tc05_out_map(&tmo, out, dims, split_kv, true)) != PA_OK) return rc;
    pa::FwdParams ps = p;
    ps.varlen_rows_cap = 64;  // the one-grid kernel leaves those sequences to the tcgen05 kernel
    const int n_long = overlap_sms(dims, hint, device_sm_count());
    if (n_long == 0) {  // one after the other on the caller's stream
        rc = cuda_status(pa::launch_tc05_varlen(p, dims->q_len, dims->dtype, tmq, tmk5, tmv5, tmo, 0, st));
        if (rc != PA_OK) return rc;
        return cuda_status(pa::launch_mma_varlen(ps, dims->q_len, dims->dtype, tmk, tmv, st));
    }
    // Side by side: fork the tcgen05 kernel onto the high-priority stream after the caller's earlier
    // work, launch the short-sequence kernel on the caller's stream, and join.
    cudaStream_t hi = nullptr;
    if ((rc = overlap_stream(&hi)) != PA_OK) return rc;
    cudaEvent_t fork = nullptr, join = nullptr;
    if (cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) != cudaSuccess) return PA_ECUDA;
    if (cudaEventCreateWithFlags(&join, cudaEventDisableTiming) != cudaSuccess) {
        cudaEventDestroy(fork);
        return PA_ECUDA;
    }
    cudaError_t e = cudaEventRecord(fork, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hi, fork, 0);
    cudaError_t e_long = cudaSuccess, e_short = cudaSuccess;
    if (e == cudaSuccess) {
        e_long = pa::launch_tc05_varlen(p, dims->q_len, dims->dtype, tmq, tmk5, tmv5, tmo, n_long, hi);
        e = cudaEventRecord(join, hi);  // recorded even if the launch failed, so the join below holds
        e_short = pa::launch_mma_varlen(ps, dims->q_len, dims->dtype, tmk, tmv, st);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(st, join, 0);
    }
    cudaEventDestroy(fork);
    cudaEventDestroy(join);
    if (e == cudaSuccess) e = e_long != cudaSuccess ? e_long : e_short;
    return cuda_status(e);
}

}  // namespace

int paged_attn_fwd_varlen(const void *q, const void *k_cache, const void *v_cache, const int32_t *block_table,
                          const int32_t *seq_lens, const int32_t *q_start, int causal, const int32_t *q_offset,
                          int split_kv, float scale, void *out, float *lse, const pa_dims *dims, void *stream) {
    return varlen_call(q, k_cache, v_cache, block_table, seq_lens, q_start, causal, q_offset, split_kv, scale, out,
                       lse, dims, nullptr, stream);
}

int paged_attn_fwd_varlen_overlap(const void *q, const void *k_cache, const void *v_cache,
                                  const int32_t *block_table, const int32_t *seq_lens, const int32_t *q_start,
                                  int causal, const int32_t *q_offset, int split_kv, float scale, void *out,
                                  float *lse, const pa_dims *dims, const pa_varlen_hint *hint, void *stream) {
    return varlen_call(q, k_cache, v_cache, block_table, seq_lens, q_start, causal, q_offset, split_kv, scale, out,
                       lse, dims, hint, stream);
}

int paged_attn_varlen_overlap_share(const pa_dims *dims, const pa_varlen_hint *hint, int num_sms) {
    int rc = check_dims(dims);
    if (rc != PA_OK) return rc;
    if (num_sms < 1) return PA_EINVAL;
    return overlap_sms(dims, hint, num_sms);
}

int paged_attn_varlen_hint(const int32_t *q_start, const int32_t *seq_lens, const int32_t *q_offset, int causal,
                           const pa_dims *dims, pa_varlen_hint *hint) {
    if (!q_start || !seq_lens || !hint) return PA_EINVAL;
    int rc = check_dims(dims);
    if (rc != PA_OK) return rc;
    const int64_t T = dims->q_len, G = dims->num_q_heads / dims->num_kv_heads;
    int64_t long_pairs = 0, short_kv = 0;
    for (int64_t b = 0; b < dims->batch; ++b) {
        const int64_t a = q_start[b], e = q_start[b + 1];
        if (a < 0 || e > T || e <= a) continue;  // no tokens (or a malformed entry)
        const int64_t n = e - a, L = seq_lens[b] > 0 ? seq_lens[b] : 0;
        if (n * G < 64) {
            short_kv += L;
            continue;
        }
        if (!causal) {
            long_pairs += n * L;
            continue;
        }
        const int64_t qoff = q_offset ? (int64_t)q_offset[b] : L - n;
        for (int64_t i = 0; i < n; ++i) {  // token i sees keys [0, min(L, qoff + i + 1))
            const int64_t reach = qoff + i + 1;
            long_pairs += reach <= 0 ? 0 : (reach < L ? reach : L);
        }
    }
    hint->long_pairs = long_pairs;
    hint->short_kv_tokens = short_kv;
    return PA_OK;
}

int paged_attn_combine(const float *part_out, const float *part_lse, int split_kv, int64_t rows, int head_dim,
                       int out_dtype, void *out, float *lse, void *stream) {
    if (out_dtype != PA_F32 && out_dtype != PA_F16 && out_dtype != PA_BF16) return PA_EDTYPE;
    if (split_kv < 1 || split_kv > 65535 || rows < 0) return PA_EINVAL;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return PA_EUNSUPPORTED;
    if (rows == 0) return PA_OK;
    if (!part_out || !part_lse || !out) return PA_EINVAL;
    if (!aligned16(part_out) || !aligned16(out) || (reinterpret_cast<uintptr_t>(part_lse) & 3u) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u))
        return PA_EINVAL;
    cudaError_t e = pa::launch_combine(part_out, part_lse, split_kv, (long long)rows, head_dim, out_dtype, out, lse,
                                       static_cast<cudaStream_t>(stream));
    return cuda_status(e);
}

int paged_attn_plan(const int32_t *seq_lens, int batch, int page_size, int split_kv, int32_t *plan, void *stream) {
    if (batch < 0 || page_size <= 0 || split_kv < 1 || split_kv > 65535) return PA_EINVAL;
    if (batch == 0) return PA_OK;
    if (!seq_lens || !plan) return PA_EINVAL;
    cudaError_t e = pa::launch_plan(seq_lens, batch, page_size, split_kv, plan, static_cast<cudaStream_t>(stream));
    return cuda_status(e);
}

int paged_attn_debug_gather(const void *cache, const int32_t *block_table, const int32_t *seq_lens,
                            const pa_dims *dims, int out_tokens, void *out, void *stream) {
    int rc = check_dims(dims);
    if (rc != PA_OK) return rc;
    if (out_tokens < 0) return PA_EINVAL;
    if (dims->batch == 0 || out_tokens == 0) return PA_OK;
    if (!cache || !block_table || !seq_lens || !out) return PA_EINVAL;
    if (!aligned16(cache) || !aligned16(out)) return PA_EINVAL;
    unsigned int *err = nullptr;
    if ((rc = error_word_ptr(&err)) != PA_OK) return rc;
    cudaError_t e = pa::launch_gather(cache, block_table, seq_lens, dims->batch, dims->bt_stride, dims->page_size,
                                      dims->num_kv_heads, dims->head_dim, esize_of(dims->dtype), dims->num_pages,
                                      out_tokens, out, err, static_cast<cudaStream_t>(stream));
    return cuda_status(e);
}

int paged_attn_debug_wait_timeout(uint32_t limit_us, void *stream) {
    if (limit_us < 1 || limit_us > 2000000) return PA_EINVAL;
    unsigned int *err = nullptr;
    int rc = error_word_ptr(&err);
    if (rc != PA_OK) return rc;
    return cuda_status(pa::launch_wait_probe(err, 1000ull * limit_us, static_cast<cudaStream_t>(stream)));
}

int paged_attn_last_error_word(uint32_t *flags) {
    if (!flags) return PA_EINVAL;
    if (cudaDeviceSynchronize() != cudaSuccess) return PA_ECUDA;
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_pa_error_word, sizeof v) != cudaSuccess) return PA_ECUDA;
    if (cudaMemcpyToSymbol(g_pa_error_word, &zero, sizeof zero) != cudaSuccess) return PA_ECUDA;
    *flags = v;
    // The most serious condition first: a wait that gave up leaves outputs unwritten, an
    // out-of-range page id only zeroes that page's tokens.
    if (v & PA_ERRBIT_TIMEOUT) return PA_ETIMEOUT;
    if (v & PA_ERRBIT_PAGE_RANGE) return PA_EBOUNDS;
    if (v & PA_ERRBIT_QSTART) return PA_EINVAL;
    return PA_OK;
}

const char *paged_attn_strerror(int code) {
    switch (code) {
        case PA_OK: return "ok";
        case PA_EINVAL: return "invalid argument";
        case PA_EDTYPE: return "unsupported element type";
        case PA_EUNSUPPORTED: return "unsupported shape or variant";
        case PA_ECUDA: return "CUDA call failed";
        case PA_EBOUNDS: return "out-of-range page id";
        case PA_ETIMEOUT: return "a pipeline wait timed out (results invalid)";
        default: return "unknown status";
    }
}

int paged_attn_version(void) { return 100; }

const char *paged_attn_cuda_error_string(void) { return cudaGetErrorString(t_last_cuda_error); }

}  // extern "C"
