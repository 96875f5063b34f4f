// KDA recurrent decode: one token per (sequence, head), the state updated in place.
//
// The three-step diagonal-plus-low-rank update of 'Kimi K3 attention deep dive'
// (forceinjection.github.io), §2.2, in the error form of 'Kimi K3' (llm.rainlin.net),
// section "Kimi Delta Attention":
//   S' = Diag(a) S            a = exp(-5 sigmoid(exp(A_h) z))   (row scale, key channel)
//   p  = S'^T k               prediction of the decayed state for key k
//   S  = S' + beta k (v - p)^T
//   o  = S^T q
// No d_k x d_k matrix is formed. The work is a read-modify-write of the 64 KB fp32
// state per (sequence, head): memory bound, so the kernel streams S once with 128-bit
// coalesced loads and stores (evict-first: the state is not reused before it leaves
// L2) and keeps it in registers between the two reductions over key channels.
//
// Thread layout: a CTA of 256 threads covers a slice of CWD value columns. Each thread
// owns 4 consecutive columns (one float4) of RPT key rows; the rows of the 256 threads
// interleave so that every warp-wide access is one contiguous run of a row.

#include "kda_common.cuh"

namespace kda {

constexpr int kDecodeThreads = 256;

// Three CTAs per SM (registers capped accordingly, a few spilled): each CTA has its
// 64 KB of state in flight, and the third CTA keeps loads outstanding while the others
// are in their reductions. Measured 4 % faster than two CTAs per SM, same results.
template <int CWD>
__global__ void __launch_bounds__(kDecodeThreads, 3)
    kda_decode_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                      const __nv_bfloat16 *__restrict__ v, const float *__restrict__ z, const float *__restrict__ A,
                      const float *__restrict__ bgate, float *__restrict__ state, float *__restrict__ o, int32_t H) {
    constexpr int LPR = CWD / 4;             // threads per row (one float4 each)
    constexpr int RG = kDecodeThreads / LPR; // row groups
    constexpr int RPT = kD / RG;             // rows per thread
    static_assert(RG * LPR == kDecodeThreads && RPT * RG == kD, "decode layout");

    __shared__ float s_alpha[kD], s_k[kD], s_q[kD];
    __shared__ __align__(16) float s_red[RG][CWD];
    __shared__ float s_beta;

    const int tid = threadIdx.x;
    const int64_t nh = blockIdx.x;  // n * H + h
    const int h = (int)(nh % H);
    const int cq = tid % LPR, rg = tid / LPR;
    const int col = blockIdx.y * CWD + 4 * cq;
    float *S = state + nh * (kD * kD);

    // issue the state loads first; the gate math below overlaps their latency
    float4 sv[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) sv[i] = __ldcs(reinterpret_cast<const float4 *>(S + (rg + i * RG) * kD + col));

    if (tid < kD) {
        const float eA = expf(A[h]);
        s_alpha[tid] = expf(gate_log_decay(eA, z[nh * kD + tid]));
        s_k[tid] = __bfloat162float(k[nh * kD + tid]);
        s_q[tid] = __bfloat162float(q[nh * kD + tid]);
    } else if (tid == kD) {
        s_beta = sigmoid_f(bgate[nh]);
    }
    const uint2 vraw = *reinterpret_cast<const uint2 *>(v + nh * kD + col);
    const float2 v01 = bf16x2_to_float2(vraw.x), v23 = bf16x2_to_float2(vraw.y);
    __syncthreads();

    // S' = Diag(a) S, partial p over this thread's rows
    float4 p = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int row = rg + i * RG;
        const float a = s_alpha[row], kr = s_k[row];
        sv[i].x *= a; sv[i].y *= a; sv[i].z *= a; sv[i].w *= a;
        p.x += kr * sv[i].x; p.y += kr * sv[i].y; p.z += kr * sv[i].z; p.w += kr * sv[i].w;
    }
    *reinterpret_cast<float4 *>(&s_red[rg][4 * cq]) = p;
    __syncthreads();
    float4 P = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int r = 0; r < RG; ++r) {
        const float4 x = *reinterpret_cast<const float4 *>(&s_red[r][4 * cq]);
        P.x += x.x; P.y += x.y; P.z += x.z; P.w += x.w;
    }
    __syncthreads();  // s_red is reused below

    // S = S' + beta k (v - p)^T, then o = S^T q
    const float beta = s_beta;
    const float4 e = make_float4(beta * (v01.x - P.x), beta * (v01.y - P.y), beta * (v23.x - P.z),
                                 beta * (v23.y - P.w));
    float4 oq = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int row = rg + i * RG;
        const float kr = s_k[row], qr = s_q[row];
        sv[i].x += kr * e.x; sv[i].y += kr * e.y; sv[i].z += kr * e.z; sv[i].w += kr * e.w;
        __stcs(reinterpret_cast<float4 *>(S + row * kD + col), sv[i]);
        oq.x += qr * sv[i].x; oq.y += qr * sv[i].y; oq.z += qr * sv[i].z; oq.w += qr * sv[i].w;
    }
    *reinterpret_cast<float4 *>(&s_red[rg][4 * cq]) = oq;
    __syncthreads();
    if (rg == 0) {
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
        for (int r = 0; r < RG; ++r) {
            const float4 x = *reinterpret_cast<const float4 *>(&s_red[r][4 * cq]);
            O.x += x.x; O.y += x.y; O.z += x.z; O.w += x.w;
        }
        *reinterpret_cast<float4 *>(o + nh * kD + col) = O;
    }
}

// Column slice per CTA: whole rows when there are enough (sequence, head) pairs to
// fill the GPU, otherwise quarter rows so that small batches still spread over SMs.
cudaError_t launch_decode(const __nv_bfloat16 *q, const __nv_bfloat16 *k, const __nv_bfloat16 *v, const float *z,
                          const float *A, const float *b, float *state, float *o, int32_t N, int32_t H,
                          int num_sms, cudaStream_t st) {
    const int64_t pairs = (int64_t)N * H;
    if (pairs == 0) return cudaSuccess;
    if (pairs >= 4ll * num_sms) {
        dim3 grid((unsigned)pairs, 1);
        kda_decode_kernel<128><<<grid, kDecodeThreads, 0, st>>>(q, k, v, z, A, b, state, o, H);
    } else {
        dim3 grid((unsigned)pairs, kD / 32);
        kda_decode_kernel<32><<<grid, kDecodeThreads, 0, st>>>(q, k, v, z, A, b, state, o, H);
    }
    return cudaGetLastError();
}

}  // namespace kda
