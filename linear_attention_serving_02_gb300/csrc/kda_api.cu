// Host side of the C ABI declared in include/kda.h: argument validation, workspace
// carving, choice of launch shapes, and the launches themselves. No allocation, no
// synchronisation (except kda_workspace_status), no exceptions.

#include <cuda_runtime.h>

#include "kda.h"
#include "kda_common.cuh"

namespace kda {
cudaError_t launch_plan(const int32_t *cu, int32_t N, int64_t seq_len, int64_t total, int32_t *status,
                        int32_t *seq_cu, int32_t *chunk_off, cudaStream_t st);
cudaError_t launch_intra(const __nv_bfloat16 *q, const __nv_bfloat16 *k, const __nv_bfloat16 *v, const float *z,
                         const float *A, const float *b, const int32_t *status, const int32_t *seq_cu,
                         const int32_t *chunk_off, int32_t N, int32_t H, int64_t nslots, uint8_t *records,
                         cudaStream_t st);
cudaError_t launch_walk(int32_t *status, const int32_t *seq_cu, const int32_t *chunk_off, int32_t N, int32_t H,
                        const uint8_t *records, const float *S0, float *Sout, void *o, int o_f32, cudaStream_t st);
cudaError_t launch_decode(const __nv_bfloat16 *q, const __nv_bfloat16 *k, const __nv_bfloat16 *v, const float *z,
                          const float *A, const float *b, float *state, float *o, int32_t N, int32_t H,
                          int num_sms, cudaStream_t st);
size_t intra_smem_bytes();
}  // namespace kda

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Device facts used to size launches, read once per device.
struct DeviceInfo {
    int sms = 0;
    int major = 0, minor = 0;
    size_t smem_optin = 0;
};

int device_info(DeviceInfo &info) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    static DeviceInfo cache[64];
    static bool have[64] = {false};
    if (dev < 0 || dev >= 64) return KDA_ERR_DEVICE;
    if (!have[dev]) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return KDA_ERR_CUDA;
        cache[dev].sms = prop.multiProcessorCount;
        cache[dev].major = prop.major;
        cache[dev].minor = prop.minor;
        cache[dev].smem_optin = prop.sharedMemPerBlockOptin;
        have[dev] = true;
    }
    info = cache[dev];
    return KDA_OK;
}

}  // namespace

extern "C" {

const char *kda_status_string(int status) {
    switch (status) {
        case KDA_OK: return "ok";
        case KDA_ERR_NULL: return "a required pointer is NULL";
        case KDA_ERR_SHAPE: return "inconsistent or negative sizes";
        case KDA_ERR_UNSUPPORTED: return "unsupported head size or output dtype (d_k = d_v = 128 only)";
        case KDA_ERR_SEQLENS: return "cu_seqlens must rise from 0 to the token count";
        case KDA_ERR_ALIGN: return "pointer not 16-byte aligned (workspace: 256-byte)";
        case KDA_ERR_WORKSPACE: return "workspace too small";
        case KDA_ERR_CUDA: return "CUDA error";
        case KDA_ERR_DEVICE: return "device unsupported";
        default: return "unknown status";
    }
}

int kda_version(void) { return 100; }

size_t kda_chunk_prefill_workspace_size(int64_t total_tokens, int32_t num_seqs, int32_t num_heads) {
    if (total_tokens < 0 || num_seqs < 0 || num_heads < 0) return 0;
    const int64_t slots = kda::chunk_bound(total_tokens, num_seqs);
    return kda::kWsHeader + 2 * kda::ws_table_bytes(num_seqs) + (size_t)slots * num_heads * kda::kRecBytes;
}

int kda_chunk_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *z, const float *A,
                      const float *b, const float *initial_state, const int32_t *cu_seqlens,
                      const int32_t *cu_seqlens_host, int32_t batch, int64_t seq_len, int32_t num_seqs,
                      int32_t num_heads, int32_t d_k, int32_t d_v, void *o, int32_t o_dtype, float *final_state,
                      void *workspace, size_t workspace_bytes, void *stream) {
    if (d_k != kda::kD || d_v != kda::kD) return KDA_ERR_UNSUPPORTED;
    if (o_dtype != KDA_OUT_BF16 && o_dtype != KDA_OUT_F32) return KDA_ERR_UNSUPPORTED;
    if (batch < 0 || seq_len < 0 || num_seqs < 0 || num_heads <= 0) return KDA_ERR_SHAPE;
    const int64_t total = (int64_t)batch * seq_len;
    if (total >= (int64_t)1 << 31) return KDA_ERR_SHAPE;  // token offsets are int32
    if (cu_seqlens) {
        if (batch != 1) return KDA_ERR_SHAPE;
    } else if (num_seqs != batch) {
        return KDA_ERR_SHAPE;
    }
    if (num_seqs == 0) return total == 0 ? KDA_OK : KDA_ERR_SHAPE;
    if (!final_state || !workspace || !A) return KDA_ERR_NULL;
    if (total > 0 && (!q || !k || !v || !z || !b || !o)) return KDA_ERR_NULL;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(z, 16) || !aligned(o, 16) ||
        !aligned(final_state, 16) || !aligned(initial_state, 16) || !aligned(A, 4) || !aligned(b, 4))
        return KDA_ERR_ALIGN;
    if (!aligned(workspace, 256)) return KDA_ERR_ALIGN;
    if (workspace_bytes < kda_chunk_prefill_workspace_size(total, num_seqs, num_heads)) return KDA_ERR_WORKSPACE;
    if (cu_seqlens_host) {
        if (cu_seqlens_host[0] != 0 || (int64_t)cu_seqlens_host[num_seqs] != total) return KDA_ERR_SEQLENS;
        for (int32_t n = 0; n < num_seqs; ++n)
            if (cu_seqlens_host[n + 1] < cu_seqlens_host[n]) return KDA_ERR_SEQLENS;
    }
    DeviceInfo dev;
    int rc = device_info(dev);
    if (rc != KDA_OK) return rc;
    if (dev.major * 10 + dev.minor < 100 || dev.smem_optin < kda::intra_smem_bytes()) return KDA_ERR_DEVICE;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int32_t *status = reinterpret_cast<int32_t *>(ws);
    int32_t *seq_cu = reinterpret_cast<int32_t *>(ws + kda::kWsHeader);
    int32_t *chunk_off = reinterpret_cast<int32_t *>(ws + kda::kWsHeader + kda::ws_table_bytes(num_seqs));
    uint8_t *records = ws + kda::kWsHeader + 2 * kda::ws_table_bytes(num_seqs);
    const int64_t nslots = kda::chunk_bound(total, num_seqs);
    const int o_f32 = (o_dtype == KDA_OUT_F32) ? 1 : 0;

    if (kda::launch_plan(cu_seqlens, num_seqs, seq_len, total, status, seq_cu, chunk_off, st) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (kda::launch_intra(reinterpret_cast<const __nv_bfloat16 *>(q), reinterpret_cast<const __nv_bfloat16 *>(k),
                          reinterpret_cast<const __nv_bfloat16 *>(v), z, A, b, status, seq_cu, chunk_off, num_seqs,
                          num_heads, nslots, records, st) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (kda::launch_walk(status, seq_cu, chunk_off, num_seqs, num_heads, records, initial_state, final_state, o, o_f32,
                         st) != cudaSuccess)
        return KDA_ERR_CUDA;
    return KDA_OK;
}

int kda_workspace_status(const void *workspace, void *stream) {
    if (!workspace) return KDA_ERR_NULL;
    int32_t st_host = 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&st_host, workspace, sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return KDA_ERR_CUDA;
    return st_host;
}

int kda_recurrent_decode(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *z, const float *A,
                         const float *b, float *state, float *o, int32_t num_seqs, int32_t num_heads, int32_t d_k,
                         int32_t d_v, void *stream) {
    if (d_k != kda::kD || d_v != kda::kD) return KDA_ERR_UNSUPPORTED;
    if (num_seqs < 0 || num_heads <= 0) return KDA_ERR_SHAPE;
    if (num_seqs == 0) return KDA_OK;
    if (!q || !k || !v || !z || !A || !b || !state || !o) return KDA_ERR_NULL;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(z, 16) || !aligned(state, 16) ||
        !aligned(o, 16) || !aligned(A, 4) || !aligned(b, 4))
        return KDA_ERR_ALIGN;
    DeviceInfo dev;
    int rc = device_info(dev);
    if (rc != KDA_OK) return rc;
    if (kda::launch_decode(reinterpret_cast<const __nv_bfloat16 *>(q), reinterpret_cast<const __nv_bfloat16 *>(k),
                           reinterpret_cast<const __nv_bfloat16 *>(v), z, A, b, state, o, num_seqs, num_heads,
                           dev.sms, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return KDA_ERR_CUDA;
    return KDA_OK;
}

}  // extern "C"
