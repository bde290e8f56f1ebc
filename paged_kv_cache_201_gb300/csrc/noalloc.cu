// Single-call split-KV forward whose scratch lives in the library itself.
//
// Some callers cannot allocate device memory when they run attention: a plugin inside a
// host framework that owns and budgets every device byte, or a latency-critical serving
// loop that must never hit cudaMalloc (which can synchronise the whole device).  For them,
// paged_attn_fwd_splitkv_noalloc keeps the split partials in a fixed array that is part of
// this file's device module.  A device holds the array from the moment the CUDA runtime loads
// that module on it until the process exits: with lazy module loading (CUDA's default) that is
// the first call of this entry point on the device, with CUDA_MODULE_LOADING=EAGER it is when
// the library's modules are loaded into the device's context.
#include <mutex>

#include "kernels.h"

namespace {

// The split partials (fp32 outputs, then fp32 lse) of every call.  Host code must not use this
// name as a device address: it is only a handle for cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_pa_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxScratchDevices = 128;
void *g_scratch_ptr[kMaxScratchDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device, looked up once per device and kept
// for the life of the process: it belongs to the device's primary context, and is stale after
// cudaDeviceReset or in any other context on the device.
int scratch_ptr(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) return PA_ECUDA;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_pa_noalloc_scratch) != cudaSuccess || !ptr) return PA_ECUDA;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return PA_OK;
}

}  // namespace

extern "C" int paged_attn_fwd_splitkv_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                              const int32_t *block_table, const int32_t *seq_lens, int causal,
                                              const int32_t *q_offset, int split_kv, float scale, void *out,
                                              float *lse, const pa_dims *dims, int num_sms, int64_t device_bytes,
                                              void *stream) {
    if (split_kv == 0) {
        // The automatic split, lowered until its partials fit the fixed array (S = 1 needs none).
        split_kv = paged_attn_auto_split(dims, num_sms, device_bytes);
        if (split_kv < 0) return split_kv;
        while (split_kv > 1 &&
               paged_attn_workspace_bytes(dims, split_kv, num_sms, device_bytes) > (int64_t)PA_NOALLOC_SCRATCH_BYTES)
            --split_kv;
    }
    const int64_t need = paged_attn_workspace_bytes(dims, split_kv, num_sms, device_bytes);
    if (need < 0) return (int)need;
    if (need > (int64_t)PA_NOALLOC_SCRATCH_BYTES) return PA_EINVAL;  // partials would not fit the fixed array
    void *scratch = nullptr;
    if (need > 0) {
        const int rc = scratch_ptr(&scratch);
        if (rc != PA_OK) return rc;
    }
    // Every partial element and lse is written by the forward before the combine reads it, so
    // nothing from an earlier call needs clearing.
    return paged_attn_fwd_splitkv(q, k_cache, v_cache, block_table, seq_lens, causal, q_offset, split_kv, scale, out,
                                  lse, dims, scratch, need > 0 ? (int64_t)PA_NOALLOC_SCRATCH_BYTES : 0, num_sms,
                                  device_bytes, stream);
}
