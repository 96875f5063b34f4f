// Prefill for callers that cannot allocate device memory.
//
// kda_chunk_prefill() needs a caller-provided device workspace. Some callers have no
// way to provide one: a plugin that lives inside an engine which owns every byte of
// device memory and hands it only the tensors of the call, or code on a latency-critical
// path where cudaMalloc (which can synchronise the whole device) is not allowed. For
// them this file keeps a fixed scratch area in the library itself, a file-scope device
// array of KDA_NOALLOC_SCRATCH_BYTES, and runs the same prefill kernels on it.
//
// The array exists once per GPU that loads the library and stays until the process
// exits. Its host-side name is only a stand-in for the symbol, never a device address:
// the device address is looked up with cudaGetSymbolAddress, once per device, with that
// device current, on the first call made on it. Nothing in the scratch has to start at
// zero (the kernels write every byte they later read), and it keeps whatever the last
// call left there. All calls share it, so calls whose GPU work overlaps (on different
// streams, or from different threads without ordering) race on it.

#include <cuda_runtime.h>

#include <mutex>

#include "kda.h"

namespace kda {
int prefill_check(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *z, const float *A,
                  const float *b, const float *initial_state, const int32_t *cu_seqlens,
                  const int32_t *cu_seqlens_host, int32_t batch, int64_t seq_len, int32_t num_seqs,
                  int32_t num_heads, int32_t d_k, int32_t d_v, const void *o, int32_t o_dtype,
                  const float *final_state, int64_t *total_out);
}

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_address[kMaxDevices] = {nullptr};

// Device address of the scratch on the current device (set up on first use).
int scratch_on_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_address[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return KDA_ERR_CUDA;
        g_scratch_address[dev] = p;
    }
    *out = g_scratch_address[dev];
    return KDA_OK;
}

}  // namespace

extern "C" int kda_chunk_prefill_noalloc(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *z,
                                         const float *A, const float *b, const float *initial_state,
                                         const int32_t *cu_seqlens, const int32_t *cu_seqlens_host, int32_t batch,
                                         int64_t seq_len, int32_t num_seqs, int32_t num_heads, int32_t d_k,
                                         int32_t d_v, void *o, int32_t o_dtype, float *final_state, void *stream) {
    // the arguments are checked exactly as kda_chunk_prefill() checks them, so the same
    // error codes come back; only then is a batch whose tables and chunk records do not
    // fit the fixed scratch refused, before anything is looked up or launched
    int64_t total = 0;
    const int bad = kda::prefill_check(q, k, v, z, A, b, initial_state, cu_seqlens, cu_seqlens_host, batch, seq_len,
                                       num_seqs, num_heads, d_k, d_v, o, o_dtype, final_state, &total);
    if (bad != KDA_OK || num_seqs == 0) return bad;
    if (kda_chunk_prefill_workspace_size(total, num_seqs, num_heads) > (size_t)KDA_NOALLOC_SCRATCH_BYTES)
        return KDA_ERR_WORKSPACE;
    void *scratch = nullptr;
    const int rc = scratch_on_current_device(&scratch);
    if (rc != KDA_OK) return rc;
    return kda_chunk_prefill(q, k, v, z, A, b, initial_state, cu_seqlens, cu_seqlens_host, batch, seq_len, num_seqs,
                             num_heads, d_k, d_v, o, o_dtype, final_state, scratch, (size_t)KDA_NOALLOC_SCRATCH_BYTES,
                             stream);
}
