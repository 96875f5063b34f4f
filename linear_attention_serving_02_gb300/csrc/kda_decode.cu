// KDA recurrent decode: one token per (sequence, head), the state updated in place; and
// its speculative-decoding pair, verify (several draft tokens from a checkpoint) and
// fold (replay of the accepted prefix).
//
// The three-step diagonal-plus-low-rank update of 'Kimi K3 attention deep dive'
// (forceinjection.github.io), §2.2, in the error form of 'Kimi K3' (llm.rainlin.net),
// section "Kimi Delta Attention":
//   S' = Diag(a) S            a = exp(-5 sigmoid(exp(A_h) z))   (row scale, key channel)
//   p  = S'^T k               prediction of the decayed state for key k
//   S  = S' + beta k (v - p)^T
//   o  = S^T q
// No d_k x d_k matrix is formed. The work is a read-modify-write of the 64 KB fp32
// state per (sequence, head): memory bound, so the kernels stream S once with 128-bit
// coalesced loads and stores (evict-first: the state is not reused before it leaves
// L2) and keep it in registers between the reductions over key channels.
//
// Thread layout: a CTA of 256 threads covers a slice of CWD value columns. Each thread
// owns 4 consecutive columns (one float4) of RPT consecutive key rows; a warp-wide access
// to one of its rows is one contiguous run of that row.
//
// ReplaySSM ('Kimi K3 attention deep dive', §6.2): instead of a 64 KB state snapshot per
// draft token, the verify kernel logs each token's gate values (log a, beta) next to the
// caller's k and v, about 1 KB per token and head; once the sampler has accepted a prefix,
// the fold kernel replays just that prefix on the checkpoint. The three kernels share
// the per-element arithmetic of kda_decode_step.cuh (explicitly rounded IEEE operations,
// two lanes per instruction), the same
// column slice for the same (sequence, head) count, and the same reduction order, so a
// fold of a tokens leaves exactly the bits that a calls of the decode kernel leave, and
// verify's outputs are exactly the decode kernel's.

#include "kda.h"
#include "kda_decode_step.cuh"

namespace kda {

constexpr int kMaxReplay = KDA_MAX_REPLAY_TOKENS;  // draft tokens per verify / fold call

// Three CTAs per SM (registers capped accordingly, a few spilled): each CTA has its
// 64 KB of state in flight, and the third CTA keeps loads outstanding while the others
// are in their reductions. Measured 4 % faster than two CTAs per SM, same results.
template <int CWD>
__global__ void __launch_bounds__(kDecodeThreads, 3)
    kda_decode_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                      const __nv_bfloat16 *__restrict__ v, const float *__restrict__ z, const float *__restrict__ A,
                      const float *__restrict__ bgate, float *__restrict__ state, float *__restrict__ o, int32_t H) {
    using G = DecodeGeom<CWD>;
    constexpr int LPR = G::LPR, RG = G::RG, RPT = G::RPT;

    __shared__ float s_alpha[kD], s_k[kD], s_q[kD];
    __shared__ __align__(16) float s_red[RG][CWD];
    __shared__ float s_beta;

    const int tid = threadIdx.x;
    const int64_t nh = blockIdx.x;  // n * H + h
    const int h = (int)(nh % H);
    const int cq = tid % LPR, rg = tid / LPR;
    const int col = blockIdx.y * CWD + 4 * cq;
    float *S = state + nh * (kD * kD);

    // the token's small loads first, so that they do not queue behind the state's 64 KB;
    // the gate math then overlaps the state loads' latency
    float zc = 0.f;
    __nv_bfloat16 kc = __float2bfloat16(0.f), qc = kc;
    if (tid < kD) {
        zc = z[nh * kD + tid];
        kc = k[nh * kD + tid];
        qc = q[nh * kD + tid];
    } else if (tid == kD) {
        zc = bgate[nh];
    }
    const uint2 vraw = *reinterpret_cast<const uint2 *>(v + nh * kD + col);
    float4 sv[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) sv[i] = __ldcs(reinterpret_cast<const float4 *>(S + row_of<CWD>(rg, i) * kD + col));

    if (tid < kD) {
        s_alpha[tid] = expf(decode_log_decay(A, h, zc));
        s_k[tid] = __bfloat162float(kc);
        s_q[tid] = __bfloat162float(qc);
    } else if (tid == kD) {
        s_beta = sigmoid_f(zc);
    }
    const float2 v01 = bf16x2_to_float2(vraw.x), v23 = bf16x2_to_float2(vraw.y);
    __syncthreads();

    // S' = Diag(a) S, partial p over this thread's rows
    float4 p = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int row = row_of<CWD>(rg, i);
        decay_project(sv[i], s_alpha[row], s_k[row], p);
    }
    *reinterpret_cast<float4 *>(&s_red[rg][4 * cq]) = p;
    __syncthreads();
    const float4 P = sum_partials<CWD>(s_red, cq);
    __syncthreads();  // s_red is reused below

    // S = S' + beta k (v - p)^T, then o = S^T q
    const float4 e = delta_error(s_beta, make_float4(v01.x, v01.y, v23.x, v23.y), P);
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
    if (rg == 0) *reinterpret_cast<float4 *>(o + nh * kD + col) = sum_partials<CWD>(s_red, cq);
}

// Verify: m draft tokens of every (sequence, head) from the checkpoint state, which is
// only read. Token t of sequence n sits at row n * m + t of the [N * m, H, ...] inputs.
// Writes every token's output, and, when the pointers are given, the token's gate
// values (the ReplaySSM log) and the state after all m tokens (state_out may be the
// checkpoint itself: each CTA reads its whole slice before it writes any of it).
template <int CWD>
__global__ void __launch_bounds__(kDecodeThreads, 2)
    kda_verify_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                      const __nv_bfloat16 *__restrict__ v, const float *__restrict__ z, const float *__restrict__ A,
                      const float *__restrict__ bgate, const float *state, float *state_out, float *__restrict__ o,
                      float *__restrict__ gk_log, float *__restrict__ beta_log, int32_t H, int32_t m) {
    using G = DecodeGeom<CWD>;
    constexpr int LPR = G::LPR, RG = G::RG, RPT = G::RPT;

    // v stays bf16 in shared memory (each thread converts only its own four columns),
    // which keeps the static total under 48 KB
    __shared__ __align__(16) float s_alpha[kMaxReplay][kD];  // read four rows at a time
    __shared__ __align__(16) float s_k[kMaxReplay][kD];
    __shared__ __align__(16) float s_q[kMaxReplay][kD];
    __shared__ __align__(16) __nv_bfloat16 s_v[kMaxReplay][kD];
    __shared__ float s_beta[kMaxReplay];
    __shared__ __align__(16) float s_redp[2][RG][CWD];
    __shared__ __align__(16) float s_redo[2][RG][CWD];

    const int tid = threadIdx.x;
    const int64_t nh = blockIdx.x;
    const int64_t n = nh / H;
    const int h = (int)(nh % H);
    const int cq = tid % LPR, rg = tid / LPR;
    const int col = blockIdx.y * CWD + 4 * cq;
    const float *S = state + nh * (kD * kD);

    // every token's inputs go first, into shared memory by cp.async, so that none of them
    // queue behind the state's 64 KB or hold registers while it is in flight: z lands in
    // s_alpha, v in s_v, b in s_beta, and k and q (bf16) in the reduction buffers, which
    // the token loop only uses after they have been converted
    __nv_bfloat16(*raw)[kMaxReplay][kD] = reinterpret_cast<__nv_bfloat16(*)[kMaxReplay][kD]>(&s_redp[0][0][0]);
    static_assert(sizeof(s_redp) >= 2 * kMaxReplay * kD * sizeof(__nv_bfloat16), "k and q staging");
    constexpr int kTokenChunks = 80;  // 16-byte pieces of one token's inputs: z 32, k, q and v 16 each
    for (int i = tid; i < m * kTokenChunks; i += kDecodeThreads) {
        const int t = i / kTokenChunks, j = i % kTokenChunks;
        const int64_t row = ((n * m + t) * H + h) * kD;
        if (j < 32) {
            cp_async16(&s_alpha[t][4 * j], z + row + 4 * j);
        } else if (j < 48) {
            cp_async16(&raw[0][t][8 * (j - 32)], k + row + 8 * (j - 32));
        } else if (j < 64) {
            cp_async16(&raw[1][t][8 * (j - 48)], q + row + 8 * (j - 48));
        } else {
            cp_async16(&s_v[t][8 * (j - 64)], v + row + 8 * (j - 64));
        }
    }
    if (tid < m) cp_async4(&s_beta[tid], bgate + (n * m + tid) * H + h);
    cp_async_commit();
    const float Ah = A[h];

    float4 sv[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) sv[i] = __ldcs(reinterpret_cast<const float4 *>(S + row_of<CWD>(rg, i) * kD + col));

    // the gate of every token (and the log, while at it), k and q to fp32
    cp_async_wait<0>();
    __syncthreads();
    const float eA = expf(Ah);
    for (int idx = tid; idx < m * kD; idx += kDecodeThreads) {
        const int t = idx / kD, c = idx % kD;
        const float la = gate_log_decay(eA, s_alpha[t][c]);
        s_alpha[t][c] = expf(la);
        s_k[t][c] = __bfloat162float(raw[0][t][c]);
        s_q[t][c] = __bfloat162float(raw[1][t][c]);
        if (gk_log) gk_log[((n * m + t) * H + h) * kD + c] = la;
    }
    if (tid < m) {
        const float beta = sigmoid_f(s_beta[tid]);
        s_beta[tid] = beta;
        if (beta_log) beta_log[(n * m + tid) * H + h] = beta;
    }
    __syncthreads();

    // One barrier per token: partials alternate between two buffers, and the output of
    // token t is summed after the barrier of token t + 1.
    for (int t = 0; t < m; ++t) {
        float4 p = make_float4(0.f, 0.f, 0.f, 0.f);
        float4 a4, k4, q4;
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            if ((i & 3) == 0) a4 = rows4<CWD>(s_alpha[t], rg, i), k4 = rows4<CWD>(s_k[t], rg, i);
            decay_project(sv[i], lane4(a4, i & 3), lane4(k4, i & 3), p);
        }
        *reinterpret_cast<float4 *>(&s_redp[t & 1][rg][4 * cq]) = p;
        __syncthreads();
        if (t > 0 && rg == 0)
            *reinterpret_cast<float4 *>(o + ((n * m + t - 1) * H + h) * kD + col) =
                sum_partials<CWD>(s_redo[(t - 1) & 1], cq);
        const float4 P = sum_partials<CWD>(s_redp[t & 1], cq);
        const uint2 vraw = *reinterpret_cast<const uint2 *>(&s_v[t][col]);
        const float2 v01 = bf16x2_to_float2(vraw.x), v23 = bf16x2_to_float2(vraw.y);
        const float4 e = delta_error(s_beta[t], make_float4(v01.x, v01.y, v23.x, v23.y), P);
        float4 oq = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            if ((i & 3) == 0) k4 = rows4<CWD>(s_k[t], rg, i), q4 = rows4<CWD>(s_q[t], rg, i);
            rank1(sv[i], lane4(k4, i & 3), e);
            readout(sv[i], lane4(q4, i & 3), oq);
        }
        *reinterpret_cast<float4 *>(&s_redo[t & 1][rg][4 * cq]) = oq;
    }
    __syncthreads();
    if (m > 0 && rg == 0)
        *reinterpret_cast<float4 *>(o + ((n * m + m - 1) * H + h) * kD + col) =
            sum_partials<CWD>(s_redo[(m - 1) & 1], cq);
    if (state_out) {
        float *So = state_out + nh * (kD * kD);
#pragma unroll
        for (int i = 0; i < RPT; ++i) __stcs(reinterpret_cast<float4 *>(So + row_of<CWD>(rg, i) * kD + col), sv[i]);
    }
}

// Fold: sequence n replays the first accepted[n] (clamped to [0, m]) logged tokens on its
// checkpoint state, in place. A sequence with nothing accepted is not touched.
template <int CWD>
__global__ void __launch_bounds__(kDecodeThreads, 3)
    kda_fold_kernel(const __nv_bfloat16 *__restrict__ k, const __nv_bfloat16 *__restrict__ v,
                    const float *__restrict__ gk_log, const float *__restrict__ beta_log,
                    const int32_t *__restrict__ accepted, float *__restrict__ state, int32_t H, int32_t m) {
    using G = DecodeGeom<CWD>;
    constexpr int LPR = G::LPR, RG = G::RG, RPT = G::RPT;

    __shared__ __align__(16) float s_alpha[kMaxReplay][kD];  // staged log a, then a
    __shared__ float s_k[kMaxReplay][kD];
    __shared__ __align__(16) float s_v[kMaxReplay][kD];  // read as float4
    __shared__ __align__(16) __nv_bfloat16 s_kb[kMaxReplay][kD], s_vb[kMaxReplay][kD];
    __shared__ float s_beta[kMaxReplay];
    __shared__ __align__(16) float s_redp[2][RG][CWD];

    const int tid = threadIdx.x;
    const int64_t nh = blockIdx.x;
    const int64_t n = nh / H;
    const int h = (int)(nh % H);
    const int a = min(max(accepted[n], 0), m);
    if (a == 0) return;  // uniform over the CTA
    const int cq = tid % LPR, rg = tid / LPR;
    const int col = blockIdx.y * CWD + 4 * cq;
    float *S = state + nh * (kD * kD);

    // every accepted token's log goes first, into shared memory by cp.async, so that none
    // of it queues behind the state's 64 KB or holds registers while the state is in flight
    constexpr int kTokenChunks = 64;  // 16-byte pieces of one token's log: a 32, k 16, v 16
    for (int i = tid; i < a * kTokenChunks; i += kDecodeThreads) {
        const int t = i / kTokenChunks, j = i % kTokenChunks;
        const int64_t row = ((n * m + t) * H + h) * kD;
        if (j < 32) {
            cp_async16(&s_alpha[t][4 * j], gk_log + row + 4 * j);
        } else if (j < 48) {
            cp_async16(&s_kb[t][8 * (j - 32)], k + row + 8 * (j - 32));
        } else {
            cp_async16(&s_vb[t][8 * (j - 48)], v + row + 8 * (j - 48));
        }
    }
    if (tid < a) cp_async4(&s_beta[tid], beta_log + (n * m + tid) * H + h);
    cp_async_commit();

    float4 sv[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) sv[i] = __ldcs(reinterpret_cast<const float4 *>(S + row_of<CWD>(rg, i) * kD + col));

    cp_async_wait<0>();
    __syncthreads();
    for (int idx = tid; idx < a * kD; idx += kDecodeThreads) {
        const int t = idx / kD, c = idx % kD;
        s_alpha[t][c] = expf(s_alpha[t][c]);
        s_k[t][c] = __bfloat162float(s_kb[t][c]);
        s_v[t][c] = __bfloat162float(s_vb[t][c]);
    }
    __syncthreads();

    for (int t = 0; t < a; ++t) {
        float4 p = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            const int row = row_of<CWD>(rg, i);
            decay_project(sv[i], s_alpha[t][row], s_k[t][row], p);
        }
        *reinterpret_cast<float4 *>(&s_redp[t & 1][rg][4 * cq]) = p;
        __syncthreads();
        const float4 P = sum_partials<CWD>(s_redp[t & 1], cq);
        const float4 e = delta_error(s_beta[t], *reinterpret_cast<const float4 *>(&s_v[t][col]), P);
#pragma unroll
        for (int i = 0; i < RPT; ++i) rank1(sv[i], s_k[t][row_of<CWD>(rg, i)], e);
    }
#pragma unroll
    for (int i = 0; i < RPT; ++i) __stcs(reinterpret_cast<float4 *>(S + row_of<CWD>(rg, i) * kD + col), sv[i]);
}

// Verify and fold take the decode kernel's column slice for the same pair count
// (whole_rows), which keeps them bit-identical to it.

cudaError_t launch_decode(const __nv_bfloat16 *q, const __nv_bfloat16 *k, const __nv_bfloat16 *v, const float *z,
                          const float *A, const float *b, float *state, float *o, int32_t N, int32_t H,
                          int num_sms, cudaStream_t st) {
    const int64_t pairs = (int64_t)N * H;
    if (pairs == 0) return cudaSuccess;
    if (whole_rows(pairs, num_sms)) {
        dim3 grid((unsigned)pairs, 1);
        kda_decode_kernel<128><<<grid, kDecodeThreads, 0, st>>>(q, k, v, z, A, b, state, o, H);
    } else {
        dim3 grid((unsigned)pairs, kD / 32);
        kda_decode_kernel<32><<<grid, kDecodeThreads, 0, st>>>(q, k, v, z, A, b, state, o, H);
    }
    return cudaGetLastError();
}

cudaError_t launch_verify(const __nv_bfloat16 *q, const __nv_bfloat16 *k, const __nv_bfloat16 *v, const float *z,
                          const float *A, const float *b, const float *state, float *state_out, float *o,
                          float *gk_log, float *beta_log, int32_t N, int32_t H, int32_t m, int num_sms,
                          cudaStream_t st) {
    const int64_t pairs = (int64_t)N * H;
    if (pairs == 0 || m == 0) return cudaSuccess;
    if (whole_rows(pairs, num_sms)) {
        dim3 grid((unsigned)pairs, 1);
        kda_verify_kernel<128><<<grid, kDecodeThreads, 0, st>>>(q, k, v, z, A, b, state, state_out, o, gk_log,
                                                                beta_log, H, m);
    } else {
        dim3 grid((unsigned)pairs, kD / 32);
        kda_verify_kernel<32><<<grid, kDecodeThreads, 0, st>>>(q, k, v, z, A, b, state, state_out, o, gk_log,
                                                               beta_log, H, m);
    }
    return cudaGetLastError();
}

cudaError_t launch_fold(const __nv_bfloat16 *k, const __nv_bfloat16 *v, const float *gk_log, const float *beta_log,
                        const int32_t *accepted, float *state, int32_t N, int32_t H, int32_t m, int num_sms,
                        cudaStream_t st) {
    const int64_t pairs = (int64_t)N * H;
    if (pairs == 0 || m == 0) return cudaSuccess;
    if (whole_rows(pairs, num_sms)) {
        dim3 grid((unsigned)pairs, 1);
        kda_fold_kernel<128><<<grid, kDecodeThreads, 0, st>>>(k, v, gk_log, beta_log, accepted, state, H, m);
    } else {
        dim3 grid((unsigned)pairs, kD / 32);
        kda_fold_kernel<32><<<grid, kDecodeThreads, 0, st>>>(k, v, gk_log, beta_log, accepted, state, H, m);
    }
    return cudaGetLastError();
}

}  // namespace kda
