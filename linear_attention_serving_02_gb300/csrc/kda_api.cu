// Host side of the C ABI declared in include/kda.h: argument validation, workspace
// carving, choice of launch shapes, and the launches themselves. No allocation, no
// synchronisation (except kda_workspace_status), no exceptions.

#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>

#include "kda.h"
#include "kda_common.cuh"

namespace kda {
struct WalkUnit;
cudaError_t launch_plan(const int32_t *cu, int32_t N, int64_t seq_len, int64_t total, int32_t *status,
                        int32_t *seq_cu, int32_t *chunk_off, int32_t H, const float *S0, float *Sout, WalkUnit *units,
                        int32_t *n_units, const SegPlan &sp, cudaStream_t st);
cudaError_t launch_intra(const __nv_bfloat16 *q, const __nv_bfloat16 *k, const __nv_bfloat16 *v, const float *z,
                         const float *A, const float *b, int32_t *status, const int32_t *seq_cu,
                         const int32_t *chunk_off, int32_t N, int32_t H, int64_t dense_len, int64_t items,
                         int32_t item_lo, int32_t item_hi, uint8_t *records, int num_sms, cudaStream_t st);
cudaError_t launch_walk(int32_t *status, const WalkUnit *units, const int32_t *n_units, int64_t max_units,
                        int32_t H, const uint8_t *records, void *o, int o_f32, int form, int head_major,
                        cudaStream_t st);
cudaError_t launch_combine(const int32_t *status, const int32_t *chains, int32_t N, int32_t H, float *Sin,
                           const float *Mseg, const float *Rseg, cudaStream_t st);
cudaError_t launch_decode(const __nv_bfloat16 *q, const __nv_bfloat16 *k, const __nv_bfloat16 *v, const float *z,
                          const float *A, const float *b, float *state, float *o, int32_t N, int32_t H,
                          int num_sms, cudaStream_t st);
cudaError_t launch_verify(const __nv_bfloat16 *q, const __nv_bfloat16 *k, const __nv_bfloat16 *v, const float *z,
                          const float *A, const float *b, const float *state, float *state_out, float *o,
                          float *gk_log, float *beta_log, int32_t N, int32_t H, int32_t m, int num_sms,
                          cudaStream_t st);
cudaError_t launch_fold(const __nv_bfloat16 *k, const __nv_bfloat16 *v, const float *gk_log, const float *beta_log,
                        const int32_t *accepted, float *state, int32_t N, int32_t H, int32_t m, int num_sms,
                        cudaStream_t st);
cudaError_t launch_fused_decode(const __nv_bfloat16 *xq, const __nv_bfloat16 *xk, const __nv_bfloat16 *xv,
                                __nv_bfloat16 *conv_state, const float *conv_w, const float *z, const float *A,
                                const float *b, const float *g, const float *norm_w, float eps_l2, float eps_rms,
                                float *state, float *y, int32_t N, int32_t H, int num_sms, cudaStream_t st);
size_t intra_smem_bytes();
cudaError_t set_walk_fault(int32_t skip_commit_chunk, uint64_t wait_limit_ns);
}  // namespace kda

namespace {

// Byte offsets of everything kda_chunk_prefill keeps in its workspace, a pure function of
// (total tokens, sequences, heads) shared by the size query and the call.
struct WsLayout {
    size_t seq_cu, chunk_off, records, units, unitsA, unitsC, chains, sin, mseg, rseg, total;
    int64_t nslots, seg_bound;
    int P;
};
WsLayout ws_layout(int64_t total_tokens, int64_t N, int64_t H) {
    using kda::align_up;
    WsLayout w;
    w.nslots = kda::chunk_bound(total_tokens, N);
    w.P = kda::walk_segment_chunks(total_tokens, N, H);
    w.seg_bound = w.P ? kda::segment_bound(total_tokens, N, w.P) : 0;
    const size_t unit_bytes = sizeof(kda::WalkUnit);
    size_t off = kda::kWsHeader;
    w.seq_cu = off;
    off += kda::ws_table_bytes(N);
    w.chunk_off = off;
    off += kda::ws_table_bytes(N);
    w.records = off;
    off += (size_t)w.nslots * H * kda::kRecBytes;
    w.units = off;
    off += align_up((size_t)N * unit_bytes, 256);
    w.unitsA = off;
    off += align_up((size_t)3 * w.seg_bound * unit_bytes, 256);  // 2 S - 3 per sequence, 1 if empty
    w.unitsC = off;
    off += align_up((size_t)w.seg_bound * unit_bytes, 256);
    w.chains = off;
    off += align_up((size_t)(w.P ? 2 * N : 0) * 4, 256);
    const size_t states = (size_t)w.seg_bound * H * kda::kStateFloats * 4;
    w.sin = off;
    off += states;
    w.mseg = off;
    off += states;
    w.rseg = off;
    off += states;
    w.total = off;
    return w;
}


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

namespace kda {
// Argument checks of the prefill entry points, in the order their error codes are
// documented: head size and output type, sizes (seq_len bounded before the token count
// is formed), pointers, alignment, the launch limits, then the host copy of cu_seqlens.
// Everything but the workspace. KDA_OK with num_seqs == 0 means there is nothing to do.
int prefill_check(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *z, const float *A,
                  const float *b, const float *initial_state, const int32_t *cu_seqlens,
                  const int32_t *cu_seqlens_host, int32_t batch, int64_t seq_len, int32_t num_seqs,
                  int32_t num_heads, int32_t d_k, int32_t d_v, const void *o, int32_t o_dtype,
                  const float *final_state, int64_t *total_out) {
    if (d_k != kD || d_v != kD) return KDA_ERR_UNSUPPORTED;
    if (o_dtype != KDA_OUT_BF16 && o_dtype != KDA_OUT_F32) return KDA_ERR_UNSUPPORTED;
    if (batch < 0 || seq_len < 0 || num_seqs < 0 || num_heads <= 0 || num_heads > 65535) return KDA_ERR_SHAPE;
    if (seq_len >= (int64_t)1 << 31) return KDA_ERR_SHAPE;  // no batch of it fits the int32 offsets either
    const int64_t total = (int64_t)batch * seq_len;  // < 2^62: no overflow
    if (total >= (int64_t)1 << 31) return KDA_ERR_SHAPE;  // token offsets are int32
    if (cu_seqlens) {
        if (batch != 1) return KDA_ERR_SHAPE;
    } else if (num_seqs != batch) {
        return KDA_ERR_SHAPE;
    }
    *total_out = total;
    if (num_seqs == 0) return total == 0 ? KDA_OK : KDA_ERR_SHAPE;
    if (!final_state || !A) return KDA_ERR_NULL;
    if (total > 0 && (!q || !k || !v || !z || !b || !o)) return KDA_ERR_NULL;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(z, 16) || !aligned(o, 16) ||
        !aligned(final_state, 16) || !aligned(initial_state, 16) || !aligned(A, 4) || !aligned(b, 4))
        return KDA_ERR_ALIGN;
    // (chunk slot, head) items are counted in int32 by the intra-chunk kernel
    if (chunk_bound(total, num_seqs) * num_heads > INT32_MAX) return KDA_ERR_SHAPE;
    if (cu_seqlens_host) {
        if (cu_seqlens_host[0] != 0 || (int64_t)cu_seqlens_host[num_seqs] != total) return KDA_ERR_SEQLENS;
        for (int32_t n = 0; n < num_seqs; ++n)
            if (cu_seqlens_host[n + 1] < cu_seqlens_host[n]) return KDA_ERR_SEQLENS;
    }
    return KDA_OK;
}
}  // namespace kda

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

namespace {
// Intra-chunk items deferred to a second intra launch that runs beside phase A of the
// chained segmented walk (dense batches; 0 otherwise). The first launch takes the first
// k * sms - 1 items (k = items / sms), so that its CTAs all take k items except the last
// CTA, which gets one fewer: that one usually starts late, on the SM that the plan kernel
// holds. The remaining items belong to the last segment of the last sequence, which only
// phase C reads, and they run on the SMs that phase A's walks leave free; otherwise none
// is deferred.
int64_t deferred_intra_items(int32_t N, int32_t H, int64_t seq_len, int P, int sms) {
    if (N <= 0 || seq_len <= 0 || P <= 0) return 0;
    const int64_t cps = (seq_len + kda::kC - 1) / kda::kC;
    const int64_t items = (int64_t)N * cps * H;
    const int64_t k = items / sms;
    if (k < 2 || items > INT32_MAX) return 0;
    const int64_t defer = items - (k * sms - 1);
    const int64_t S = (cps + P - 1) / P;
    if (S < 2) return 0;
    const int64_t units_a = (int64_t)N * H * (2 * S - 3);  // phase A's walks, all in one wave
    const int64_t last = S >= 3 ? kda::BalancedCut((int32_t)cps, P, (int32_t)S).last_len() : cps - (S - 1) * P;
    if (defer > sms - units_a || defer > last * H) return 0;
    return defer;
}
}  // namespace

int kda_debug_walk_fault(int32_t skip_commit_chunk, uint64_t wait_limit_ns) {
    if (wait_limit_ns == 0) return KDA_ERR_SHAPE;
    return kda::set_walk_fault(skip_commit_chunk, wait_limit_ns) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

// end factor forced by kda_debug_segment_ends (0: the cost model's)
static std::atomic<int32_t> g_debug_segment_ends{0};

int kda_debug_segment_ends(int32_t end_factor) {
    if (end_factor < 0 || end_factor > 64) return KDA_ERR_SHAPE;
    g_debug_segment_ends.store(end_factor);
    return KDA_OK;
}

size_t kda_chunk_prefill_workspace_size(int64_t total_tokens, int32_t num_seqs, int32_t num_heads) {
    if (total_tokens < 0 || num_seqs < 0 || num_heads < 0) return 0;
    return ws_layout(total_tokens, num_seqs, num_heads).total;
}

int32_t kda_chunk_prefill_launch_count(int64_t total_tokens, int32_t num_seqs, int32_t num_heads) {
    if (total_tokens < 0 || num_seqs < 0 || num_heads < 0) return -1;
    if (num_seqs == 0) return 0;
    if (!kda::walk_segment_chunks(total_tokens, num_seqs, num_heads)) return 3;
    return 5;  // plan, intra, phase A, then the deferred intra items or the combine kernel, phase C
}

int32_t kda_chunk_prefill_walk_form(int64_t total_tokens, int32_t num_seqs, int32_t num_heads) {
    if (total_tokens < 0 || num_seqs < 0 || num_heads < 0) return -1;
    if (num_seqs == 0 || !kda::walk_segment_chunks(total_tokens, num_seqs, num_heads)) return 0;
    return kda::walk_chain_mode(total_tokens, num_seqs, num_heads) ? 1 : 2;
}

int kda_chunk_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *z, const float *A,
                      const float *b, const float *initial_state, const int32_t *cu_seqlens,
                      const int32_t *cu_seqlens_host, int32_t batch, int64_t seq_len, int32_t num_seqs,
                      int32_t num_heads, int32_t d_k, int32_t d_v, void *o, int32_t o_dtype, float *final_state,
                      void *workspace, size_t workspace_bytes, void *stream) {
    int64_t total = 0;
    int rc = kda::prefill_check(q, k, v, z, A, b, initial_state, cu_seqlens, cu_seqlens_host, batch, seq_len,
                                num_seqs, num_heads, d_k, d_v, o, o_dtype, final_state, &total);
    if (rc != KDA_OK || num_seqs == 0) return rc;
    if (!workspace) return KDA_ERR_NULL;
    if (!aligned(workspace, 256)) return KDA_ERR_ALIGN;
    if (workspace_bytes < kda_chunk_prefill_workspace_size(total, num_seqs, num_heads)) return KDA_ERR_WORKSPACE;
    DeviceInfo dev;
    rc = device_info(dev);
    if (rc != KDA_OK) return rc;
    if (dev.major * 10 + dev.minor < 100 || dev.smem_optin < kda::intra_smem_bytes()) return KDA_ERR_DEVICE;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const WsLayout w = ws_layout(total, num_seqs, num_heads);
    int32_t *status = reinterpret_cast<int32_t *>(ws);
    int32_t *counts = reinterpret_cast<int32_t *>(ws + 16);  // units of the plain walk, phase A, phase C
    int32_t *seq_cu = reinterpret_cast<int32_t *>(ws + w.seq_cu);
    int32_t *chunk_off = reinterpret_cast<int32_t *>(ws + w.chunk_off);
    uint8_t *records = ws + w.records;
    kda::WalkUnit *units = reinterpret_cast<kda::WalkUnit *>(ws + w.units);
    const int o_f32 = (o_dtype == KDA_OUT_F32) ? 1 : 0;

    // the segmented walk's tables (when w.P > 0) are written by the plan kernel too
    kda::SegPlan sp{};
    sp.P = w.P;
    if (w.P > 0) {
        sp.Sin = reinterpret_cast<float *>(ws + w.sin);
        sp.Mseg = reinterpret_cast<float *>(ws + w.mseg);
        sp.Rseg = reinterpret_cast<float *>(ws + w.rseg);
        sp.unitsA = reinterpret_cast<kda::WalkUnit *>(ws + w.unitsA);
        sp.unitsC = reinterpret_cast<kda::WalkUnit *>(ws + w.unitsC);
        sp.nA = counts + 1;
        sp.nC = counts + 2;
        sp.chains = reinterpret_cast<int32_t *>(ws + w.chains);
        sp.chain_mode = kda::walk_chain_mode(total, num_seqs, num_heads) ? 1 : 0;
        // long end segments in the combine form only (the chained form keeps P throughout)
        const int32_t forced = g_debug_segment_ends.load();
        sp.E = sp.chain_mode ? 1 : (forced > 0 ? forced : kda::walk_segments(total, num_seqs, num_heads).E);
    }
    if (kda::launch_plan(cu_seqlens, num_seqs, seq_len, total, status, seq_cu, chunk_off, num_heads, initial_state,
                         final_state, units, counts, sp, st) != cudaSuccess)
        return KDA_ERR_CUDA;
    // the chained form defers the intra items past a whole number of rounds (dense batches)
    // to a second intra launch beside phase A
    const int64_t defer =
        (w.P > 0 && sp.chain_mode && !cu_seqlens) ? deferred_intra_items(num_seqs, num_heads, seq_len, w.P, dev.sms) : 0;
    const int64_t items1 = cu_seqlens ? w.nslots * num_heads
                                      : (int64_t)num_seqs * ((seq_len + kda::kC - 1) / kda::kC) * num_heads - defer;
    auto intra = [&](int64_t items, int32_t lo, int32_t hi) {
        return kda::launch_intra(reinterpret_cast<const __nv_bfloat16 *>(q), reinterpret_cast<const __nv_bfloat16 *>(k),
                                 reinterpret_cast<const __nv_bfloat16 *>(v), z, A, b, status, seq_cu, chunk_off,
                                 num_seqs, num_heads, cu_seqlens ? 0 : seq_len, items, lo, hi, records, dev.sms, st);
    };
    if (intra(items1, 0, (int32_t)std::min<int64_t>(items1, INT32_MAX)) != cudaSuccess) return KDA_ERR_CUDA;
    if (w.P == 0) {
        // heads as the fastest grid index (the plan lists the longest sequences first)
        if (kda::launch_walk(status, units, counts, num_seqs, num_heads, records, o, o_f32, 0, num_seqs <= 65535 ? 1 : 0,
                             st) != cudaSuccess)
            return KDA_ERR_CUDA;
        return KDA_OK;
    }
    // segmented walk: phase A (segment maps), phase B (chain them: the combine kernel, or in
    // the chained form each output walk itself), phase C (outputs). With long end segments
    // (listed first) heads are the fastest grid index, so every head's long walks start in
    // the first wave.
    const int hm = (sp.E > 1 && 3 * w.seg_bound <= 65535) ? 1 : 0;
    if (kda::launch_walk(status, sp.unitsA, sp.nA, 3 * w.seg_bound, num_heads, records, o, o_f32, 2, hm, st) !=
        cudaSuccess)
        return KDA_ERR_CUDA;
    // chained form: the deferred intra items (none for a cu_seqlens batch), beside phase A
    if (sp.chain_mode && intra(defer, (int32_t)std::min<int64_t>(items1, INT32_MAX), INT32_MAX) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (!sp.chain_mode &&
        kda::launch_combine(status, sp.chains, num_seqs, num_heads, sp.Sin, sp.Mseg, sp.Rseg, st) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (kda::launch_walk(status, sp.unitsC, sp.nC, w.seg_bound, num_heads, records, o, o_f32, sp.chain_mode ? 1 : 0, hm,
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

// (sequence, head) pairs are grid x of the decode-family launches; heads are grid y of
// the walk and the combine
static bool pairs_fit(int32_t num_seqs, int32_t num_heads) {
    return (int64_t)num_seqs * num_heads <= INT32_MAX && num_heads <= 65535;
}

int kda_recurrent_decode(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *z, const float *A,
                         const float *b, float *state, float *o, int32_t num_seqs, int32_t num_heads, int32_t d_k,
                         int32_t d_v, void *stream) {
    if (d_k != kda::kD || d_v != kda::kD) return KDA_ERR_UNSUPPORTED;
    if (num_seqs < 0 || num_heads <= 0 || !pairs_fit(num_seqs, num_heads)) return KDA_ERR_SHAPE;
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

int kda_recurrent_verify(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *z, const float *A,
                         const float *b, const float *state, float *state_out, float *o, float *gk_log,
                         float *beta_log, int32_t num_seqs, int32_t num_heads, int32_t num_tokens, int32_t d_k,
                         int32_t d_v, void *stream) {
    if (d_k != kda::kD || d_v != kda::kD) return KDA_ERR_UNSUPPORTED;
    if (num_seqs < 0 || num_heads <= 0 || num_tokens < 0 || !pairs_fit(num_seqs, num_heads)) return KDA_ERR_SHAPE;
    if (num_tokens > KDA_MAX_REPLAY_TOKENS) return KDA_ERR_UNSUPPORTED;
    if (num_seqs == 0 || num_tokens == 0) return KDA_OK;
    if (!q || !k || !v || !z || !A || !b || !state || !o) return KDA_ERR_NULL;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(z, 16) || !aligned(state, 16) ||
        !aligned(state_out, 16) || !aligned(o, 16) || !aligned(gk_log, 16) || !aligned(A, 4) || !aligned(b, 4) ||
        !aligned(beta_log, 4))
        return KDA_ERR_ALIGN;
    DeviceInfo dev;
    int rc = device_info(dev);
    if (rc != KDA_OK) return rc;
    if (kda::launch_verify(reinterpret_cast<const __nv_bfloat16 *>(q), reinterpret_cast<const __nv_bfloat16 *>(k),
                           reinterpret_cast<const __nv_bfloat16 *>(v), z, A, b, state, state_out, o, gk_log, beta_log,
                           num_seqs, num_heads, num_tokens, dev.sms, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return KDA_ERR_CUDA;
    return KDA_OK;
}

int kda_replay_fold(const uint16_t *k, const uint16_t *v, const float *gk_log, const float *beta_log,
                    const int32_t *num_accepted, float *state, int32_t num_seqs, int32_t num_heads,
                    int32_t num_tokens, int32_t d_k, int32_t d_v, void *stream) {
    if (d_k != kda::kD || d_v != kda::kD) return KDA_ERR_UNSUPPORTED;
    if (num_seqs < 0 || num_heads <= 0 || num_tokens < 0 || !pairs_fit(num_seqs, num_heads)) return KDA_ERR_SHAPE;
    if (num_tokens > KDA_MAX_REPLAY_TOKENS) return KDA_ERR_UNSUPPORTED;
    if (num_seqs == 0 || num_tokens == 0) return KDA_OK;
    if (!k || !v || !gk_log || !beta_log || !num_accepted || !state) return KDA_ERR_NULL;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(gk_log, 16) || !aligned(state, 16) || !aligned(beta_log, 4) ||
        !aligned(num_accepted, 4))
        return KDA_ERR_ALIGN;
    DeviceInfo dev;
    int rc = device_info(dev);
    if (rc != KDA_OK) return rc;
    if (kda::launch_fold(reinterpret_cast<const __nv_bfloat16 *>(k), reinterpret_cast<const __nv_bfloat16 *>(v),
                         gk_log, beta_log, num_accepted, state, num_seqs, num_heads, num_tokens, dev.sms,
                         static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return KDA_ERR_CUDA;
    return KDA_OK;
}

int kda_fused_decode(const uint16_t *x_q, const uint16_t *x_k, const uint16_t *x_v, uint16_t *conv_state,
                     const float *conv_w, const float *z, const float *A, const float *b, const float *g,
                     const float *norm_w, float eps_l2, float eps_rms, float *state, float *y, int32_t num_seqs,
                     int32_t num_heads, int32_t d_k, int32_t d_v, void *stream) {
    if (d_k != kda::kD || d_v != kda::kD) return KDA_ERR_UNSUPPORTED;
    if (!(eps_l2 >= 0.0f) || !(eps_rms >= 0.0f)) return KDA_ERR_UNSUPPORTED;  // NaN fails both
    if (num_seqs < 0 || num_heads <= 0 || !pairs_fit(num_seqs, num_heads)) return KDA_ERR_SHAPE;
    if (num_seqs == 0) return KDA_OK;
    if (!x_q || !x_k || !x_v || !conv_state || !conv_w || !z || !A || !b || !g || !norm_w || !state || !y)
        return KDA_ERR_NULL;
    if (!aligned(x_q, 16) || !aligned(x_k, 16) || !aligned(x_v, 16) || !aligned(conv_state, 16) ||
        !aligned(conv_w, 16) || !aligned(z, 16) || !aligned(g, 16) || !aligned(norm_w, 16) || !aligned(state, 16) ||
        !aligned(y, 16) || !aligned(A, 4) || !aligned(b, 4))
        return KDA_ERR_ALIGN;
    DeviceInfo dev;
    int rc = device_info(dev);
    if (rc != KDA_OK) return rc;
    if (kda::launch_fused_decode(
            reinterpret_cast<const __nv_bfloat16 *>(x_q), reinterpret_cast<const __nv_bfloat16 *>(x_k),
            reinterpret_cast<const __nv_bfloat16 *>(x_v), reinterpret_cast<__nv_bfloat16 *>(conv_state), conv_w, z,
            A, b, g, norm_w, eps_l2, eps_rms, state, y, num_seqs, num_heads, dev.sms,
            static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return KDA_ERR_CUDA;
    return KDA_OK;
}

}  // extern "C"
