// The per-token decode step that every decode-family kernel shares: the thread layout
// over a CTA's slice of value columns, and the per-element arithmetic of the update
// S' = Diag(a) S, p = S'^T k, S = S' + beta k (v - p)^T, o = S^T q ('Kimi K3 attention
// deep dive', §2.2). Every operation is an explicitly rounded IEEE operation (packed two
// lanes at a time), so the kernels that include this file produce the same bits for the
// same inputs and layout.
#pragma once

#include "kda.h"
#include "kda_common.cuh"
#include "kda_f32x2.cuh"

namespace kda {

constexpr int kDecodeThreads = 256;

template <int CWD>
struct DecodeGeom {
    static constexpr int LPR = CWD / 4;              // threads per row (one float4 each)
    static constexpr int RG = kDecodeThreads / LPR;  // row groups
    static constexpr int RPT = kD / RG;              // rows per thread
    static_assert(RG * LPR == kDecodeThreads && RPT * RG == kD && RPT % 4 == 0, "decode layout");
};

// Thread group rg owns the RPT consecutive key rows rg * RPT ... rg * RPT + RPT - 1 (of
// its CTA's value columns), so a token's per-row values (a, k, q) are read from shared
// memory four rows at a time. A warp's load of one of its rows is still whole 128-byte
// lines of the state.
template <int CWD>
__device__ __forceinline__ int row_of(int rg, int i) {
    return rg * DecodeGeom<CWD>::RPT + i;
}
// rows row_of(rg, i) ... row_of(rg, i + 3) of a 16-byte aligned shared row vector
template <int CWD>
__device__ __forceinline__ float4 rows4(const float *vec, int rg, int i) {
    return *reinterpret_cast<const float4 *>(vec + row_of<CWD>(rg, i));
}
__device__ __forceinline__ float lane4(const float4 &v, int j) {
    return j == 0 ? v.x : (j == 1 ? v.y : (j == 2 ? v.z : v.w));
}

// ---- the per-element arithmetic every kernel here shares (packed forms in kda_f32x2.cuh) ----
// S' = a S on one row of this thread, and its term of the projection p += k_r S'_r
__device__ __forceinline__ void decay_project(float4 &s, float a, float kr, float4 &p) {
    const uint64_t a2 = pk2(a, a), k2 = pk2(kr, kr);
    const uint64_t s01 = mul2(pk2(s.x, s.y), a2), s23 = mul2(pk2(s.z, s.w), a2);
    set4(s, s01, s23);
    set4(p, fma2(k2, s01, pk2(p.x, p.y)), fma2(k2, s23, pk2(p.z, p.w)));
}
// e = beta (v - p)
__device__ __forceinline__ float4 delta_error(float beta, float4 v, float4 p) {
    const uint64_t b2 = pk2(beta, beta);
    float4 e;
    set4(e, mul2(b2, sub2(pk2(v.x, v.y), pk2(p.x, p.y))), mul2(b2, sub2(pk2(v.z, v.w), pk2(p.z, p.w))));
    return e;
}
// S = S' + k_r e on one row
__device__ __forceinline__ void rank1(float4 &s, float kr, float4 e) {
    const uint64_t k2 = pk2(kr, kr);
    set4(s, fma2(k2, pk2(e.x, e.y), pk2(s.x, s.y)), fma2(k2, pk2(e.z, e.w), pk2(s.z, s.w)));
}
// o += q_r S_r
__device__ __forceinline__ void readout(const float4 &s, float qr, float4 &o) {
    const uint64_t q2 = pk2(qr, qr);
    set4(o, fma2(q2, pk2(s.x, s.y), pk2(o.x, o.y)), fma2(q2, pk2(s.z, s.w), pk2(o.z, o.w)));
}
// sum of the RG row-group partials of this thread's four columns, in row-group order
template <int CWD>
__device__ __forceinline__ float4 sum_partials(const float (*red)[CWD], int cq) {
    constexpr int RG = DecodeGeom<CWD>::RG;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int r = 0; r < RG; ++r) {
        const float4 x = *reinterpret_cast<const float4 *>(&red[r][4 * cq]);
        set4(acc, add2(pk2(acc.x, acc.y), pk2(x.x, x.y)), add2(pk2(acc.z, acc.w), pk2(x.z, x.w)));
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
