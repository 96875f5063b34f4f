// The per-token decode step that every decode-family kernel shares: the thread layout
// over a CTA's slice of value columns, and the per-element arithmetic of the update
// S' = Diag(a) S, p = S'^T k, S = S' + beta k (v - p)^T, o = S^T q ('Kimi K3 attention
// deep dive', §2.2). Every operation is an explicitly rounded intrinsic, so the kernels
// that include this file produce the same bits for the same inputs and layout.
#pragma once

#include "kda.h"
#include "kda_common.cuh"

namespace kda {

constexpr int kDecodeThreads = 256;

template <int CWD>
struct DecodeGeom {
    static constexpr int LPR = CWD / 4;              // threads per row (one float4 each)
    static constexpr int RG = kDecodeThreads / LPR;  // row groups
    static constexpr int RPT = kD / RG;              // rows per thread
    static_assert(RG * LPR == kDecodeThreads && RPT * RG == kD, "decode layout");
};

// ---- the per-element arithmetic every kernel here shares ----

// S' = a S on one row of this thread, and its term of the projection p += k_r S'_r
__device__ __forceinline__ void decay_project(float4 &s, float a, float kr, float4 &p) {
    s.x = __fmul_rn(s.x, a); s.y = __fmul_rn(s.y, a); s.z = __fmul_rn(s.z, a); s.w = __fmul_rn(s.w, a);
    p.x = __fmaf_rn(kr, s.x, p.x); p.y = __fmaf_rn(kr, s.y, p.y);
    p.z = __fmaf_rn(kr, s.z, p.z); p.w = __fmaf_rn(kr, s.w, p.w);
}
// e = beta (v - p)
__device__ __forceinline__ float4 delta_error(float beta, float4 v, float4 p) {
    return make_float4(__fmul_rn(beta, __fsub_rn(v.x, p.x)), __fmul_rn(beta, __fsub_rn(v.y, p.y)),
                       __fmul_rn(beta, __fsub_rn(v.z, p.z)), __fmul_rn(beta, __fsub_rn(v.w, p.w)));
}
// S = S' + k_r e on one row
__device__ __forceinline__ void rank1(float4 &s, float kr, float4 e) {
    s.x = __fmaf_rn(kr, e.x, s.x); s.y = __fmaf_rn(kr, e.y, s.y);
    s.z = __fmaf_rn(kr, e.z, s.z); s.w = __fmaf_rn(kr, e.w, s.w);
}
// o += q_r S_r
__device__ __forceinline__ void readout(const float4 &s, float qr, float4 &o) {
    o.x = __fmaf_rn(qr, s.x, o.x); o.y = __fmaf_rn(qr, s.y, o.y);
    o.z = __fmaf_rn(qr, s.z, o.z); o.w = __fmaf_rn(qr, s.w, o.w);
}
// sum of the RG row-group partials of this thread's four columns, in row-group order
template <int CWD>
__device__ __forceinline__ float4 sum_partials(const float (*red)[CWD], int cq) {
    constexpr int RG = DecodeGeom<CWD>::RG;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int r = 0; r < RG; ++r) {
        const float4 x = *reinterpret_cast<const float4 *>(&red[r][4 * cq]);
        acc.x = __fadd_rn(acc.x, x.x); acc.y = __fadd_rn(acc.y, x.y);
        acc.z = __fadd_rn(acc.z, x.z); acc.w = __fadd_rn(acc.w, x.w);
    }
    return acc;
}
// the gate of one key channel, as every kernel here computes it
__device__ __forceinline__ float decode_log_decay(const float *A, int h, float z) {
    return gate_log_decay(expf(A[h]), z);
}

// Column slice per CTA: whole rows (CWD = 128) when there are enough (sequence, head)
// pairs to fill the GPU, otherwise quarter rows (CWD = 32) so that small batches still
// spread over the SMs.
inline bool whole_rows(int64_t pairs, int num_sms) { return pairs >= 4ll * num_sms; }

}  // namespace kda
