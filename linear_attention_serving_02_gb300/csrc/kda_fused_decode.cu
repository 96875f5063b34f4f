// Fused KDA decode layer step: causal conv -> recurrent update -> gated RMSNorm in one
// launch ('Kimi K3 attention deep dive', §6.3), with the projections' activations of
// the same page's §2.3:
//   q = L2Norm(Swish(ShortConv(x_q)))   k = L2Norm(Swish(ShortConv(x_k)))
//   v = Swish(ShortConv(x_v))
//   S' = Diag(a) S;  S = S' + beta k (v - S'^T k)^T;  o = S^T q   (in place, fp32)
//   y = o / sqrt(mean(o^2) + eps_rms) * w_norm * sigmoid(g)
// ShortConv is depthwise and causal with four taps: channel c of the output is
// w[c,0] x_{t-3} + w[c,1] x_{t-2} + w[c,2] x_{t-1} + w[c,3] x_t, where x_{t-3..t-1} come
// from the conv state, which then drops its oldest input and appends x_t.
//
// One (sequence, head) is one CTA of 256 threads (whole rows of the state), or, when the
// batch is too small to fill the GPU, a cluster of four CTAs that each own 32 value
// columns. Every CTA computes the conv and activations of all 128 key channels (q and k
// are needed whole by every row of the state; it is 128 x 12 multiply-adds). A cluster
// shares the output's sum of squares through distributed shared memory, and each CTA
// writes back its own quarter of the conv state once the cluster barrier shows that
// every CTA has read the old one.
//
// The step's small inputs (x, the conv state, the taps, z, g and w_norm: 10.5 KB) are
// copied into shared memory with cp.async before the state's 64 KB are requested, so they
// are not queued behind the state and hold no registers while it is in flight. That keeps
// the kernel within 80 registers, three CTAs per SM, as the plain decode.

#include <cooperative_groups.h>

#include "kda_decode_step.cuh"

namespace cg = cooperative_groups;

namespace kda {

namespace {

struct FusedArgs {
    const __nv_bfloat16 *xq, *xk, *xv;
    __nv_bfloat16 *conv_state;  // [N, 3 (q, k, v), 3 (oldest first), H, 128]
    const float *conv_w;        // [3, H, 128, 4] (oldest tap first)
    const float *z, *A, *b, *g, *norm_w;
    float eps_l2, eps_rms;
    float *state, *y;
    int32_t H;
};

// Shared-memory image of one (sequence, head)'s small inputs; every array is a whole
// number of 16-byte chunks.
struct FusedStage {
    __nv_bfloat16 x[3][kD];        // x_q, x_k, x_v of this token
    __nv_bfloat16 hist[3][3][kD];  // the three previous inputs of each stream, oldest first
    float4 w[3][kD];               // the four taps of each stream and channel
    float z[kD], g[kD], nw[kD];
};
constexpr int kRowChunks = kD * 2 / 16;                          // 16-byte chunks in a bf16 row of 128
constexpr int kStageChunks = 12 * kRowChunks + 3 * kD + 3 * 32;  // x, hist, taps, z / g / w_norm

// Issue the cp.async of chunk i of the stage (i < kStageChunks).
__device__ __forceinline__ void stage_chunk(FusedStage &st, const FusedArgs &p, int64_t n, int h, int64_t nh,
                                            int i) {
    if (i < 3 * kRowChunks) {  // x_q, x_k, x_v
        const int s = i / kRowChunks, j = i % kRowChunks;
        const __nv_bfloat16 *xs = s == 0 ? p.xq : (s == 1 ? p.xk : p.xv);
        cp_async16(&st.x[s][8 * j], xs + nh * kD + 8 * j);
        return;
    }
    i -= 3 * kRowChunks;
    if (i < 9 * kRowChunks) {  // conv state rows (stream s, age r)
        const int sr = i / kRowChunks, j = i % kRowChunks;
        cp_async16(&st.hist[sr / 3][sr % 3][8 * j], p.conv_state + ((n * 9 + sr) * p.H + h) * kD + 8 * j);
        return;
    }
    i -= 9 * kRowChunks;
    if (i < 3 * kD) {  // taps: one chunk per (stream, channel)
        const int s = i / kD, c = i % kD;
        cp_async16(&st.w[s][c], p.conv_w + (((int64_t)s * p.H + h) * kD + c) * 4);
        return;
    }
    i -= 3 * kD;
    const int a = i / 32, j = i % 32;  // z, g, w_norm: 32 chunks of four floats each
    float *dst = a == 0 ? st.z : (a == 1 ? st.g : st.nw);
    const float *src = a == 0 ? p.z + nh * kD : (a == 1 ? p.g + nh * kD : p.norm_w);
    cp_async16(dst + 4 * j, src + 4 * j);
}

// Write chunk i of the shifted conv state: age 0 <- age 1, age 1 <- age 2, age 2 <- x.
// Chunk i covers 8 channels of one (stream, age) row; bf16 bits are copied unchanged.
__device__ __forceinline__ void write_conv_chunk(const FusedStage &st, const FusedArgs &p, int64_t n, int h,
                                                 int sr, int j) {
    const int s = sr / 3, r = sr % 3;
    const __nv_bfloat16 *src = r < 2 ? &st.hist[s][r + 1][8 * j] : &st.x[s][8 * j];
    *reinterpret_cast<uint4 *>(p.conv_state + ((n * 9 + sr) * p.H + h) * kD + 8 * j) =
        *reinterpret_cast<const uint4 *>(src);
}

__device__ __forceinline__ float swish_f(float x) { return x / (1.0f + expf(-x)); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

template <int CWD>
__device__ __forceinline__ void fused_decode_body(const FusedArgs &p) {
    using G = DecodeGeom<CWD>;
    constexpr int LPR = G::LPR, RG = G::RG, RPT = G::RPT;
    constexpr int NCTA = kD / CWD;  // CTAs per (sequence, head)

    __shared__ __align__(16) FusedStage st;
    __shared__ float s_alpha[kD], s_k[kD], s_q[kD];
    __shared__ __align__(16) float s_v[kD];  // read as float4
    __shared__ __align__(16) float s_red[RG][CWD];
    __shared__ float s_sq[2][kD / 32];  // per-warp sums of q^2 and k^2
    __shared__ float s_oo[NCTA];        // per-CTA sums of o^2 (one slot per cluster rank)
    __shared__ float s_beta;

    const int tid = threadIdx.x;
    const int64_t nh = blockIdx.x;
    const int64_t n = nh / p.H;
    const int h = (int)(nh % p.H);
    const int cq = tid % LPR, rg = tid / LPR;
    const int rank = (int)blockIdx.y;  // cluster rank: the CTAs of a cluster are consecutive in y
    const int col = rank * CWD + 4 * cq;
    float *S = p.state + nh * (kD * kD);

    // ---- the small inputs first, into shared memory; then the state, into registers ----
    for (int i = tid; i < kStageChunks; i += kDecodeThreads) stage_chunk(st, p, n, h, nh, i);
    cp_async_commit();
    const float Ah = p.A[h];
    const float bv = tid == kD ? p.b[nh] : 0.f;
    float4 sv[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) sv[i] = __ldcs(reinterpret_cast<const float4 *>(S + row_of<CWD>(rg, i) * kD + col));
    cp_async_wait<0>();
    __syncthreads();

    // ---- prologue: conv, Swish, squares for the L2 norms, gate ----
    if (tid < kD) {
        const int c = tid;
        float act[3];
#pragma unroll
        for (int s = 0; s < 3; ++s) {
            const float4 w = st.w[s][c];
            float acc = __fmul_rn(w.x, __bfloat162float(st.hist[s][0][c]));
            acc = __fmaf_rn(w.y, __bfloat162float(st.hist[s][1][c]), acc);
            acc = __fmaf_rn(w.z, __bfloat162float(st.hist[s][2][c]), acc);
            acc = __fmaf_rn(w.w, __bfloat162float(st.x[s][c]), acc);
            act[s] = swish_f(acc);
        }
        s_q[c] = act[0];  // normalised below, once the sums of squares are in
        s_k[c] = act[1];
        s_v[c] = act[2];
        const float sq = warp_sum(act[0] * act[0]), sk = warp_sum(act[1] * act[1]);
        if ((tid & 31) == 0) {
            s_sq[0][tid >> 5] = sq;
            s_sq[1][tid >> 5] = sk;
        }
        s_alpha[c] = expf(gate_log_decay(expf(Ah), st.z[c]));
    } else {
        if (tid == kD) s_beta = sigmoid_f(bv);
        if constexpr (NCTA == 1) {
            // the only reader of this (sequence, head)'s conv state has staged it: shift it
            for (int i = tid - kD; i < 9 * kRowChunks; i += kDecodeThreads - kD)
                write_conv_chunk(st, p, n, h, i / kRowChunks, i % kRowChunks);
        }
    }
    __syncthreads();
    if (tid < kD) {
        const float nq = (s_sq[0][0] + s_sq[0][1]) + (s_sq[0][2] + s_sq[0][3]);
        const float nk = (s_sq[1][0] + s_sq[1][1]) + (s_sq[1][2] + s_sq[1][3]);
        s_q[tid] = s_q[tid] / sqrtf(nq + p.eps_l2);
        s_k[tid] = s_k[tid] / sqrtf(nk + p.eps_l2);
    }
    if constexpr (NCTA > 1) {
        // every CTA of the cluster has staged the old conv state (and runs) before any
        // conv-state or DSMEM write; each CTA then shifts its own quarter of the channels
        cg::this_cluster().sync();
        constexpr int QC = kRowChunks / NCTA;  // chunks of a row in one quarter
        if (tid >= kD && tid - kD < 9 * QC) {
            const int i = tid - kD;
            write_conv_chunk(st, p, n, h, i / QC, rank * QC + i % QC);
        }
    }
    __syncthreads();

    // ---- the recurrent update ----
    float4 pp = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int row = row_of<CWD>(rg, i);
        decay_project(sv[i], s_alpha[row], s_k[row], pp);
    }
    *reinterpret_cast<float4 *>(&s_red[rg][4 * cq]) = pp;
    __syncthreads();
    const float4 P = sum_partials<CWD>(s_red, cq);
    __syncthreads();
    const float4 e = delta_error(s_beta, *reinterpret_cast<const float4 *>(&s_v[col]), P);
    float4 oq = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int row = row_of<CWD>(rg, i);
        rank1(sv[i], s_k[row], e);
        __stcs(reinterpret_cast<float4 *>(S + row * kD + col), sv[i]);
        readout(sv[i], s_q[row], oq);
    }
    *reinterpret_cast<float4 *>(&s_red[rg][4 * cq]) = oq;
    __syncthreads();

    // ---- epilogue: per-head RMSNorm and the output gate (rg == 0 is part of warp 0) ----
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    float oo = 0.f;
    if (rg == 0) {
        O = sum_partials<CWD>(s_red, cq);
        oo = (O.x * O.x + O.y * O.y) + (O.z * O.z + O.w * O.w);
    }
    if (tid < 32) {
        // rg == 0 is lanes 0..LPR-1 of warp 0; the other lanes add zeros
        oo = warp_sum(oo);
        if (tid == 0) {
            if constexpr (NCTA == 1) {
                s_oo[0] = oo;
            } else {
                cg::cluster_group cluster = cg::this_cluster();
                for (int r = 0; r < NCTA; ++r) cluster.map_shared_rank(s_oo, r)[rank] = oo;
            }
        }
    }
    if constexpr (NCTA > 1) {
        cg::this_cluster().sync();  // every CTA's partial delivered
    } else {
        __syncthreads();
    }
    if (rg == 0) {
        float tot = 0.f;
#pragma unroll
        for (int r = 0; r < NCTA; ++r) tot += s_oo[r];
        const float inv = 1.0f / sqrtf(tot * (1.0f / kD) + p.eps_rms);
        const float4 w = *reinterpret_cast<const float4 *>(&st.nw[col]);
        const float4 gg = *reinterpret_cast<const float4 *>(&st.g[col]);
        float4 yv;
        yv.x = O.x * inv * w.x * sigmoid_f(gg.x);
        yv.y = O.y * inv * w.y * sigmoid_f(gg.y);
        yv.z = O.z * inv * w.z * sigmoid_f(gg.z);
        yv.w = O.w * inv * w.w * sigmoid_f(gg.w);
        *reinterpret_cast<float4 *>(p.y + nh * kD + col) = yv;
    }
}

__global__ void __launch_bounds__(kDecodeThreads, 3) kda_fused_decode_kernel(FusedArgs p) {
    fused_decode_body<128>(p);
}

__global__ void __cluster_dims__(1, 4, 1) __launch_bounds__(kDecodeThreads, 3)
    kda_fused_decode_cluster_kernel(FusedArgs p) {
    fused_decode_body<32>(p);
}

}  // namespace

cudaError_t launch_fused_decode(const __nv_bfloat16 *xq, const __nv_bfloat16 *xk, const __nv_bfloat16 *xv,
                                __nv_bfloat16 *conv_state, const float *conv_w, const float *z, const float *A,
                                const float *b, const float *g, const float *norm_w, float eps_l2, float eps_rms,
                                float *state, float *y, int32_t N, int32_t H, int num_sms, cudaStream_t st) {
    const int64_t pairs = (int64_t)N * H;
    if (pairs == 0) return cudaSuccess;
    const FusedArgs a{xq, xk, xv, conv_state, conv_w, z, A, b, g, norm_w, eps_l2, eps_rms, state, y, H};
    if (whole_rows(pairs, num_sms)) {
        kda_fused_decode_kernel<<<dim3((unsigned)pairs, 1), kDecodeThreads, 0, st>>>(a);
    } else {
        kda_fused_decode_cluster_kernel<<<dim3((unsigned)pairs, kD / 32), kDecodeThreads, 0, st>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace kda
