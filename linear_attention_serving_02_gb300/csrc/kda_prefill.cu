// KDA chunkwise prefill: kernels on one stream.
//
//   kda_plan_kernel   validate cu_seqlens, tabulate sequence starts and chunk offsets,
//                     and the walk units of a plain walk (or the segmented walk's tables)
//   kda_intra_kernel  persistent, one CTA per SM over the (chunk, head) items, all chunks
//                     independent: gate and cumulative decay, decayed K K^T / Q K^T per
//                     32-token tile row, UT transform T = (I + A_kk)^-1, W = T' Khat and
//                     U' = T' V, written as a chunk record
//   kda_walk_kernel   one CTA per walk unit (a run of chunks of one (sequence, head)):
//                     walks the chunks in order with the full state on chip, on tcgen05
//                     tensor cores (TMEM accumulators),
//                     U = U' - W S;  O = Qhat S + A_qk U;  S = Diag(gamma) S + Kend^T U
//   with few long sequences the walk is segmented (two walk launches, with
//   kda_combine_kernel between them when the segments are many; see below)
//
// The algebra is the chunkwise form of 'From Linear Attention to KDA' (blog), §7.1-7.3
// with the per-channel decay of §7.2 folded into the UT system, and tiles as in §8 for
// the decayed Gram matrices. Inside one chunk (positions i, j):
//   G_i        = sum_{m<=i} log a_m                (fp32, per key channel)
//   A_kk[i,j]  = beta_i sum_c k_i k_j exp(G_i - G_j)    j <  i
//   A_qk[i,j]  =        sum_c q_i k_j exp(G_i - G_j)    j <= i
//   T          = (I + A_kk)^-1,  T' = T Diag(beta)
//   W = T' (k * exp(G)),  U' = T' v,  U = U' - W S_0
//   O = (q * exp(G)) S_0 + A_qk U,   S_C = Diag(exp(G_C)) S_0 + (k * exp(G_C - G))^T U
//
// Every product runs on the tensor cores (mma.sync m16n8k16 in the intra kernel, tcgen05
// in the walk; bf16 inputs, fp32 accumulate) with both operands split into bf16 hi + lo
// planes (three products per tile). A plain
// bf16 operand would cost about 2^-9 of relative error per product, which the
// prediction-error cancellation in U = U' - W S amplifies beyond the accuracy the
// outputs are held to; the split keeps about 16 mantissa bits.
//
// Decay factors never overflow: for the 32-token tile row a (tokens 32a..32a+31) the
// reference point is m = 32a + 16, and exp(G_i - G_j) = exp(G_i - G_m) * exp(G_m - G_j).
// A factor exceeds 1 only across the at most 16 tokens between m and a row of the tile
// row (log decay >= -5 per token, §5.4 of the blog), so neither exceeds e^80, within
// bf16/fp32 range (the blog's §8 uses 16-token sub-chunks; the middle reference allows 32).

#include <algorithm>

#include "kda_common.cuh"
#include "kda_f32x2.cuh"
#include "kda_tc.cuh"

namespace kda {

// ---------------------------------------------------------------------------------
// plan: seq_cu[N+1] and chunk_off[N+1] (prefix sums of ceil(len / C)) in the workspace
// ---------------------------------------------------------------------------------
constexpr int kPlanSortMax = 1024;  // plain walks of up to this many sequences go longest first
// ---------------------------------------------------------------------------------
// segmented walk: tables of the two phases, written by one thread of the plan kernel
// (used only when there are few sequences). Segment g of the batch is segment sigma of
// sequence n, g = seg_base[n] + sigma; its affine map is S_out = M[g] S_in + R[g].
//   phase A  segment 0 from the initial state -> Sin[g0 + 1] (segment 1's input)
//            segment sigma (1 .. S-2) from zero     -> R[g],  with U'
//            segment sigma (1 .. S-2) from identity -> M[g],  without U' (in the chained
//            form kept as the split bf16 planes the tensor cores read)
//            (walks without outputs read only -W and Kend^T of the records)
//   phase B  (combine form) Sin[g + 1] = M[g] Sin[g] + R[g] for sigma = 1 .. S-2, by
//            kda_combine_kernel
//   phase C  segments 0 .. S-1, writing o (a sequence of one segment only here); the last
//            one writes the final state. Segment
//            sigma >= 1 starts from Sin[g0 + sigma] (combine form), or (chained form) from
//            Sin[g0 + 1], first applying X <- M[g0 + j] X + R[g0 + j] for j = 1 .. sigma - 1
//            on the tensor cores (the chained form is taken only when all of phase C runs
//            in one wave, so the longest chain is what it adds).
// ---------------------------------------------------------------------------------
__device__ void plan_segments(bool bad, const int32_t *__restrict__ seq_cu, const int32_t *__restrict__ chunk_off,
                              int32_t N, int32_t H, const float *S0, float *Sout, const SegPlan &sp) {
    const int32_t P = sp.P;
    float *Sin = sp.Sin, *Mseg = sp.Mseg, *Rseg = sp.Rseg;
    WalkUnit *unitsA = sp.unitsA, *unitsC = sp.unitsC;
    auto blank = [](const float *in, float *out, int32_t c, int32_t t, int32_t flags) {
        WalkUnit u;
        u.in = in;
        u.out = out;
        u.maps = u.offs = nullptr;
        u.c_begin = u.c_end = c;
        u.t_begin = u.t_end = t;
        u.flags = flags;
        u.chain = 0;
        return u;
    };
    if (bad) {
        // no maps to build; phase C only marks each final state invalid (NaN)
        for (int32_t n = 0; n < N; ++n) {
            unitsC[n] = blank(nullptr, Sout + (size_t)n * H * kStateFloats, 0, 0, 0);
            sp.chains[2 * n] = sp.chains[2 * n + 1] = 0;
        }
        *sp.nA = 0;
        *sp.nC = N;
        return;
    }
    const size_t seg_stride = (size_t)H * kStateFloats;  // one segment's states for all heads
    const int32_t E = sp.E;
    int32_t a = 0, cc = 0;
    // two passes over the same segments: the first lists the walks longer than P (the end
    // segments of sequences cut with long ends), the second the others, so that each phase
    // starts its longest walks first
    for (int pass = 0; pass < 2; ++pass) {
        int32_t g = 0;
        for (int32_t n = 0; n < N; ++n) {
            const int32_t c0 = chunk_off[n], c1 = chunk_off[n + 1];
            const int32_t t0 = seq_cu[n], t1 = seq_cu[n + 1];
            const int32_t len = c1 - c0;
            // long ends: segments [0, E P), then P at a time up to len - E P, then [len - E P, len)
            const bool ends = E > 1 && (int64_t)len >= (int64_t)(2 * E + 1) * P;  // then E P < len
            const int32_t S = ends ? 2 + (len - 2 * E * P + P - 1) / P : (len + P - 1) / P;
            if (pass == 0) {
                sp.chains[2 * n] = g;
                sp.chains[2 * n + 1] = S;
            }
            const float *init = S0 ? S0 + (size_t)n * seg_stride : nullptr;
            float *fin = Sout + (size_t)n * seg_stride;
            // an empty sequence: its final state is its initial state
            if (S == 0 && pass == 1) unitsA[a++] = blank(init, fin, c0, t0, 0);
            // chained form: the balanced cut (kda_common.cuh)
            const bool balanced = sp.chain_mode && !ends && S >= 3;
            const BalancedCut cut(balanced ? len : 0, P, balanced ? S : 0);
            int32_t pos = 0, grown_seen = 0;
            for (int32_t sg = 0; sg < S; ++sg) {
                int32_t cb, ce;  // the segment's chunks, relative to the sequence
                if (ends) {
                    cb = sg == 0 ? 0 : (sg == S - 1 ? len - E * P : E * P + (sg - 1) * P);
                    ce = sg == 0 ? E * P : (sg == S - 1 ? len : min(cb + P, len - E * P));
                } else if (balanced) {
                    int32_t L = BalancedCut::len_at(cut.level, sg, P);
                    if (cut.grew(sg)) {
                        if (grown_seen >= cut.grown - cut.surplus) --L;
                        ++grown_seen;
                    }
                    cb = pos;
                    ce = pos = pos + L;
                } else {
                    cb = sg * P;
                    ce = min(len, cb + P);
                }
                if ((ce - cb > P) != (pass == 0)) continue;
                WalkUnit u = blank(nullptr, nullptr, c0 + cb, t0 + cb * kC, kUnitAddUp);
                u.c_end = c0 + ce;
                u.t_end = min(t1, t0 + ce * kC);
                if (sg == 0) {
                    u.in = init;
                    if (S == 1) {  // phase C: the sequence's only walk, with outputs
                        u.out = fin;
                        u.flags = kUnitWriteO | kUnitAddUp;
                        unitsC[cc++] = u;
                        continue;
                    }
                    // phase A: the end state only (a walk without outputs is cheaper) ...
                    u.out = Sin + (size_t)(g + 1) * seg_stride;
                    u.flags = kUnitAddUp | (sp.chain_mode ? kUnitOutQuads : 0);
                    unitsA[a++] = u;
                    // ... phase C: again with outputs, alongside the other segments
                    u.out = nullptr;
                    u.flags = kUnitWriteO | kUnitAddUp;
                    unitsC[cc++] = u;
                    continue;
                }
                // phase C
                u.flags = kUnitWriteO | kUnitAddUp;
                if (sp.chain_mode) {  // from segment 1's input through the maps of segments 1 .. sg - 1
                    u.in = Sin + (size_t)(g + 1) * seg_stride;
                    u.flags |= kUnitInQuads;
                    u.chain = sg - 1;
                    if (sg > 1) {
                        u.maps = Mseg + (size_t)(g + 1) * seg_stride;
                        u.offs = Rseg + (size_t)(g + 1) * seg_stride;
                    }
                } else {  // from the combine kernel's input state
                    u.in = Sin + (size_t)(g + sg) * seg_stride;
                }
                u.out = sg == S - 1 ? fin : nullptr;
                unitsC[cc++] = u;
                // phase A: this segment's map
                if (sg <= S - 2) {
                    u.in = u.maps = u.offs = nullptr;
                    u.chain = 0;
                    u.out = Rseg + (size_t)(g + sg) * seg_stride;
                    u.flags = kUnitAddUp | (sp.chain_mode ? kUnitOutQuads : 0);
                    unitsA[a++] = u;
                    u.out = Mseg + (size_t)(g + sg) * seg_stride;
                    u.flags = kUnitIdentity | (sp.chain_mode ? kUnitOutPlanes : 0);
                    unitsA[a++] = u;
                }
            }
            g += S;
        }
    }
    *sp.nA = a;
    *sp.nC = cc;
}

// the plain walk's unit of sequence n, from the finished sequence tables
__device__ __forceinline__ WalkUnit plain_unit(int32_t n, int32_t H, const int32_t *seq_cu, const int32_t *chunk_off,
                                               const float *S0, float *Sout) {
    WalkUnit u;
    u.in = S0 ? S0 + (size_t)n * H * kStateFloats : nullptr;
    u.out = Sout + (size_t)n * H * kStateFloats;
    u.maps = u.offs = nullptr;
    u.c_begin = chunk_off[n];
    u.c_end = chunk_off[n + 1];
    u.t_begin = seq_cu[n];
    u.t_end = seq_cu[n + 1];
    u.flags = kUnitWriteO | kUnitAddUp;
    u.chain = 0;
    return u;
}

__global__ void kda_plan_kernel(const int32_t *__restrict__ cu_seqlens, int32_t N, int64_t seq_len,
                                int64_t total_tokens, int32_t *__restrict__ status, int32_t *__restrict__ seq_cu,
                                int32_t *__restrict__ chunk_off, int32_t H, const float *S0, float *Sout,
                                WalkUnit *__restrict__ units, int32_t *__restrict__ n_units, SegPlan sp,
                                int sort_n) {
    extern __shared__ uint64_t key[];  // sort_n keys (dynamic: the kernel runs beside the intra
                                       // kernel's first CTAs and must not crowd an SM)
    __shared__ int32_t carry;
    __shared__ int32_t bad;
    __shared__ int32_t scan[256];
    pdl_trigger();
    const int tid = threadIdx.x;
    if (tid == 0) {
        carry = 0;
        bad = 0;
    }
    __syncthreads();
    // validation: cu[0] == 0, cu[N] == total, non-decreasing
    if (cu_seqlens != nullptr) {
        for (int64_t n = tid; n <= N; n += blockDim.x) {
            int32_t c = cu_seqlens[n];
            if (n == 0 && c != 0) atomicOr(&bad, 1);
            if (n == N && (int64_t)c != total_tokens) atomicOr(&bad, 1);
            if (n > 0 && c < cu_seqlens[n - 1]) atomicOr(&bad, 1);
        }
    }
    __syncthreads();
    if (bad) {
        // empty walks whose only job is to mark each final state invalid (NaN)
        for (int64_t n = tid; n <= N; n += blockDim.x) {
            seq_cu[n] = 0;
            chunk_off[n] = 0;
            if (n < N) {
                WalkUnit u;
                u.in = nullptr;
                u.out = Sout + (size_t)n * H * kStateFloats;
                u.maps = u.offs = nullptr;
                u.c_begin = u.c_end = u.t_begin = u.t_end = 0;
                u.flags = 0;
                u.chain = 0;
                units[n] = u;
            }
        }
        if (tid == 0) {
            *status = -4;  // KDA_ERR_SEQLENS
            *n_units = N;
            if (sp.P > 0) plan_segments(true, seq_cu, chunk_off, N, H, S0, Sout, sp);
        }
        return;
    }
    if (tid == 0) {
        *status = 0;
        *n_units = N;
    }
    for (int64_t base = 0; base <= N; base += 256) {
        const int64_t n = base + tid;
        int32_t start = 0, len = 0;
        if (n <= N) {
            start = cu_seqlens ? cu_seqlens[n] : (int32_t)(n * seq_len);
            seq_cu[n] = start;
            if (n < N) {
                int32_t end = cu_seqlens ? cu_seqlens[n + 1] : (int32_t)((n + 1) * seq_len);
                len = (end - start + kC - 1) / kC;
            }
        }
        scan[tid] = len;
        __syncthreads();
        for (int off = 1; off < 256; off <<= 1) {  // inclusive Hillis-Steele scan
            int32_t x = tid >= off ? scan[tid - off] : 0;
            __syncthreads();
            scan[tid] += x;
            __syncthreads();
        }
        // exclusive offset of sequence n = carry + inclusive(n) - len(n)
        if (n <= N) chunk_off[n] = carry + scan[tid] - len;
        if (tid == 255) carry += scan[255];
        __syncthreads();
    }
    // the tables are complete and visible (barrier above)
    if (sp.P > 0) {  // the segmented walk's tables
        if (tid == 0) plan_segments(false, seq_cu, chunk_off, N, H, S0, Sout, sp);
        return;
    }
    // the plain walk: one unit per sequence. Up to kPlanSortMax sequences are listed longest
    // first (a bitonic sort of (chunks, sequence) keys over sort_n, the next power of two),
    // and the walk launches heads as the fastest grid index, so that every head of the
    // longest sequences starts in the first wave and the short ones fill in behind them.
    if (sort_n < N) {
        for (int32_t n = tid; n < N; n += blockDim.x) units[n] = plain_unit(n, H, seq_cu, chunk_off, S0, Sout);
        return;
    }
    for (int i = tid; i < sort_n; i += blockDim.x)  // real keys above every pad key
        key[i] = i < N ? ((uint64_t)(chunk_off[i + 1] - chunk_off[i] + 1) << 32) | (uint32_t)~i : 0ull;
    __syncthreads();
    for (int k = 2; k <= sort_n; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < sort_n; i += blockDim.x) {
                const int l = i ^ j;
                if (l > i) {
                    const uint64_t a = key[i], b = key[l];
                    if (((i & k) == 0) ? (a < b) : (a > b)) {  // descending overall
                        key[i] = b;
                        key[l] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    for (int r = tid; r < N; r += blockDim.x)
        units[r] = plain_unit((int32_t)~(uint32_t)key[r], H, seq_cu, chunk_off, S0, Sout);
}

// Phase B: Sin[g + 1] = M[g] Sin[g] + R[g] along each sequence's segments, in fp32 on the
// CUDA cores (exact accumulation, a short serial chain). One CTA of 128 threads per
// (sequence, head, 16 value columns); thread t computes rows t / 4 + 32 i (i = 0 .. 3),
// columns 4 (t % 4) .. +3 of its slice, two columns per packed FMA (each lane the IEEE
// fma of the scalar form, the terms added in k order). The step is bound by the shared
// loads of M and x, so each thread reuses every value it loads four times.
// M and R do not depend on the chain, so the next step's M (64 KB) and R slice are
// copied into shared memory (cp.async) while the current step multiplies; the chained
// slice itself stays in shared memory from one step to the next.
struct CombineSmem {
    float m[2][kD][kD + 4];  // rows padded: the 16 rows a warp reads hit distinct banks
    float r[2][kD][16];
    float x[kD][16];
};

constexpr int kCombineThreads = 128;

__global__ void __launch_bounds__(kCombineThreads)
    kda_combine_kernel(const int32_t *__restrict__ status, const int32_t *__restrict__ chains, int32_t H,
                       float *__restrict__ Sin, const float *__restrict__ Mseg, const float *__restrict__ Rseg) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    CombineSmem &s = *reinterpret_cast<CombineSmem *>(smem_raw);
    pdl_wait();
    pdl_trigger();
    if (*status != 0) return;
    const int n = blockIdx.x, h = blockIdx.y, col0 = blockIdx.z * 16;
    const int g0 = chains[2 * n], S = chains[2 * n + 1];
    if (S < 3) return;  // no step: segment 1's input state is phase A's R of segment 0
    const int tid = threadIdx.x, row = tid >> 2, cpart = (tid & 3) * 4;  // rows row + 32 i
    const size_t seg_stride = (size_t)H * kStateFloats, hoff = (size_t)h * kStateFloats;

    auto stage = [&](int sg, int buf) {
        const float *M = Mseg + (size_t)(g0 + sg) * seg_stride + hoff;
        const float *R = Rseg + (size_t)(g0 + sg) * seg_stride + hoff;
        for (int e = tid; e < kD * (kD / 4); e += kCombineThreads) {
            const int rr = e / (kD / 4), c4 = (e % (kD / 4)) * 4;
            cp_async16(&s.m[buf][rr][c4], M + rr * kD + c4);
        }
        for (int e = tid; e < kD * 4; e += kCombineThreads) {
            const int rr = e / 4, c4 = (e % 4) * 4;
            cp_async16(&s.r[buf][rr][c4], R + rr * kD + col0 + c4);
        }
        cp_async_commit();
    };

    stage(1, 0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = row + 32 * i;
        *reinterpret_cast<float4 *>(&s.x[r][cpart]) =
            *reinterpret_cast<const float4 *>(Sin + (size_t)(g0 + 1) * seg_stride + hoff + r * kD + col0 + cpart);
    }
    for (int sg = 1; sg <= S - 2; ++sg) {
        const int buf = (sg - 1) & 1;
        if (sg + 1 <= S - 2) {
            stage(sg + 1, buf ^ 1);  // buffer buf ^ 1 was last read before the previous barrier
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();  // this step's M, R and x are visible
        // acc[i][0] holds columns cpart, cpart + 1 of row + 32 i; acc[i][1] the next two
        uint64_t acc[4][2];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 r0 = *reinterpret_cast<const float4 *>(&s.r[buf][row + 32 * i][cpart]);
            acc[i][0] = pk2(r0.x, r0.y);
            acc[i][1] = pk2(r0.z, r0.w);
        }
#pragma unroll 2
        for (int k4 = 0; k4 < kD / 4; ++k4) {
            float mk[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 m = *reinterpret_cast<const float4 *>(&s.m[buf][row + 32 * i][4 * k4]);
                mk[i][0] = m.x; mk[i][1] = m.y; mk[i][2] = m.z; mk[i][3] = m.w;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 x = *reinterpret_cast<const float4 *>(&s.x[4 * k4 + q][cpart]);
                const uint64_t x01 = pk2(x.x, x.y), x23 = pk2(x.z, x.w);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint64_t m2 = pk2(mk[i][q], mk[i][q]);
                    acc[i][0] = fma2(m2, x01, acc[i][0]);
                    acc[i][1] = fma2(m2, x23, acc[i][1]);
                }
            }
        }
        __syncthreads();  // every thread is done with x and with buffer buf
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = row + 32 * i;
            const float2 a = upk2(acc[i][0]), b = upk2(acc[i][1]);
            const float4 y = make_float4(a.x, a.y, b.x, b.y);
            *reinterpret_cast<float4 *>(&s.x[r][cpart]) = y;
            *reinterpret_cast<float4 *>(Sin + (size_t)(g0 + sg + 1) * seg_stride + hoff + r * kD + col0 + cpart) = y;
        }
    }
}

// ---------------------------------------------------------------------------------
// state walk: one CTA per (sequence, head) carries the full 128 x 128 state through
// the chunks of its sequence on the tcgen05 tensor cores, accumulators in TMEM.
//
// Transposed orientation, so that the 128 value channels are the MMA's M = 128 rows
// and every accumulator row is one TMEM lane. Per chunk, two MMA groups:
//   group 1   [D_U | D_O1] = S^T [ -W ; Qhat ]^T          N = 128, K = 128
//   group 2   [D_O2 | D_S] = U^T [ A_qk ; Kend^T ]^T      N = 192, K = 64
// with U^T = U'^T + D_U, o = (D_O1 + D_O2)^T and S^T <- S^T Diag(gamma) + D_S. A walk
// that writes no outputs (a segment map) drops Qhat and A_qk: N = 64 and 128.
// Every product is split-bf16 (hi*hi + hi*lo + lo*hi). S^T and U^T, the A operands, are
// written as split planes straight into tensor memory by the threads that own their rows
// (tcgen05.st); the record tiles in shared memory are the B operands.
// A segment of a segmented walk first brings its start state through the maps of the
// segments before it: X <- M X + R, on the same tensor cores as X^T <- X^T M^T + R^T
// (X^T in the S^T planes, M's split planes as the B operand, D in D_U | D_O1), one
// 128 x 128 x 128 product per map, the next map's planes copied while the current one runs.
//
// Eight warps with fixed roles:
//   warps 0-3  U and O: thread = value channel dv (TMEM lane dv). After group 1 they
//              build U^T, then copy the next chunk's U' and [ -W ; Qhat ] into shared
//              memory while group 2 runs; after group 2 they update key rows 64-127 of
//              S and write their S^T planes, stage o in shared memory from the output
//              accumulators, and store it in 16-byte row chunks while the next chunk's
//              group 1 runs.
//   warps 4-7  state: thread = value channel dv, key rows 0-63 of S. After group 2
//              they update those rows and write their S^T planes, then copy the
//              [ A_qk ; Kend^T ] of the chunk after next into the slot group 2 has freed.
//              Thread 128 also issues the MMAs.
// The record tiles move by 16-byte cp.async, issued by the warps that wait anyway at
// that point: a bulk copy held its issuing thread for up to a thousand cycles, and on
// the MMA thread that sat on the chain. Each copying thread waits for its own copies and
// fences them for the tensor cores' proxy before the barrier that hands the tile over.
// The state rows and U' live in fp32 registers as packed pairs (rows 2j, 2j + 1; tokens
// 2j, 2j + 1), so the update, U = U' + D_U and the split into bf16 planes run on the
// two-lane FP32 instructions.
// Named barriers hand the steps over: BAR_U (U^T planes ready), BAR_OR (output
// accumulators read), and a state-warp barrier (S^T planes ready). Every role runs the
// same barrier sequence whatever happens: a wait that gives up marks the CTA failed, the
// rest of the walk skips its work but keeps the sequence, and the issuer still commits
// every MMA group so that the U and O warps' waits keep their arrivals in order.
// ---------------------------------------------------------------------------------
struct WalkSmem {
    unsigned char wq[kRecWQBytes];       // -W, Qhat hi, Qhat lo (rows 0..63, 64..127, 64..127)
    unsigned char ak[2][2 * kStackAK];   // [ A_qk ; Kend^T ] hi | lo, of chunks c (slot c & 1)
    alignas(16) float up[kC * kD];       // U' of the current chunk, rows as in the record
    alignas(16) float gam[2][kD];        // gamma of chunks c (slot c & 1), the state warps' copy
    alignas(16) float gam_uo[2][kD];     // the same, the U and O warps' copy
    alignas(16) unsigned char ut[2 * 128 * kC * 2];  // o staging: 64 tokens x 128 channels (fp32 or bf16)
    uint64_t bar_m1, bar_m2, bar_ch;
    uint32_t tmem_base;
    int fail;
};
static_assert(sizeof(WalkSmem) <= 227 * 1024, "walk shared memory");
// Before its first chunk a walk may run a chain of segment maps; their planes (hi, lo) take
// two buffers: hi at ak + 0, lo at ak + 32 KB; hi at ak + 64 KB, lo in ut.
constexpr int kPlaneSS = kD * kD * 2;  // one 128 x 128 bf16 plane
static_assert(sizeof(WalkSmem::ak) >= 3 * (size_t)kPlaneSS && sizeof(WalkSmem::ut) >= (size_t)kPlaneSS,
              "chain buffers");
static_assert(sizeof(WalkSmem::wq) + sizeof(WalkSmem::ak) >= 2 * (size_t)kPlaneSS, "plane staging");

constexpr int kWalkThreads = 256;
// TMEM columns: accumulators D_U [0,64) D_O1 [64,128) D_O2 [128,192) D_S [192,320); the
// A operands of the two MMA groups as split bf16 (two per column): S^T hi [320,384),
// S^T lo [384,448), U^T hi [448,480), U^T lo [480,512)
constexpr uint32_t kWalkTmemCols = 512;
constexpr uint32_t kColSHi = 320, kColSLo = 384, kColUHi = 448, kColULo = 480;
constexpr int kBarOR = 2, kBarU = 3;


// 16 pairs of fp32 values of this thread's lane, held as packed registers -> 16 columns
// of the hi plane and 16 of the lo plane: hi = the bf16 pair, lo = bf16 of the pair minus
// hi (one packed subtraction; the same values as split_bf16x2)
__device__ __forceinline__ void split32_tmem_pk(const uint64_t *x, uint32_t t_hi, uint32_t t_lo) {
    uint32_t h[16], l[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const float2 v = upk2(x[j]);
        h[j] = pack_bf16x2(__floats2bfloat162_rn(v.x, v.y));
        const float2 d = upk2(sub2(x[j], pk2(__uint_as_float(h[j] << 16), __uint_as_float(h[j] & 0xffff0000u))));
        l[j] = pack_bf16x2(__floats2bfloat162_rn(d.x, d.y));
    }
    tc::tmem_st16(t_hi, h);
    tc::tmem_st16(t_lo, l);
}

// Test hook (kda_debug_walk_fault): the walk's MMA issuer leaves out the group-1 commit of
// chunk g_walk_skip_commit (or, for -2 - j, the commit of map j of the map chain), and
// every wait of the walk gives up after g_walk_wait_ns, so a wait runs out with no fault;
// -1 and the default limit otherwise.
__device__ int g_walk_skip_commit = -1;
__device__ unsigned long long g_walk_wait_ns = tc::kWaitLimitNs;

// bounded wait that gives up at once when the CTA has already failed
__device__ __forceinline__ bool wait_or_fail(uint64_t *bar, uint32_t parity, volatile int &fail, uint64_t limit) {
    if (fail) return false;
    if (tc::mbar_wait(bar, parity, limit)) return true;
    fail = 1;
    return false;
}
// bounded wait that also waits after a failure: the issuer commits every group's barrier
// even when it skips the MMAs, so this returns promptly and keeps the U and O warps'
// BAR_U / BAR_OR arrivals behind the state warps' matching syncs (a named barrier counts
// arrivals, so one side may never arrive twice before the other has synced). True when
// the data behind the barrier is valid.
__device__ __forceinline__ bool wait_in_order(uint64_t *bar, uint32_t parity, volatile int &fail, uint64_t limit) {
    if (!tc::mbar_wait(bar, parity, limit)) fail = 1;
    return !fail;
}

// Three instances, each holding only its own code (a kernel with every path in it stalled
// on instruction fetch): kWalkOut walks with outputs; kWalkChain the same, first chaining
// segment maps (the chained form's phase C); kWalkMaps walks without outputs (phase A:
// segment maps, end states kept as split planes or in quads).
constexpr int kWalkOut = 0, kWalkChain = 1, kWalkMaps = 2;
template <int kForm>
__global__ void __launch_bounds__(kWalkThreads, 1)
    kda_walk_kernel(int32_t *__restrict__ status, const WalkUnit *__restrict__ units,
                    const int32_t *__restrict__ n_units, int32_t H, const uint8_t *__restrict__ records,
                    void *__restrict__ o, int o_f32, int head_major) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    WalkSmem &s = *reinterpret_cast<WalkSmem *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = head_major ? blockIdx.x : blockIdx.y;
    const int ui = head_major ? blockIdx.y : blockIdx.x;
    pdl_wait();
    pdl_trigger();
    if (ui >= *n_units) return;
    const WalkUnit unit = units[ui];
    const uint64_t wlim = g_walk_wait_ns;
    const int skip_commit = g_walk_skip_commit;
    const float *S0 = unit.in ? unit.in + (size_t)h * kStateFloats : nullptr;
    float *Sout = unit.out ? unit.out + (size_t)h * kStateFloats : nullptr;
    constexpr bool kChain = kForm == kWalkChain, kMaps = kForm == kWalkMaps;
    constexpr bool write_o = !kMaps;  // the plan gives every unit of an instance its form
    const bool add_up = (unit.flags & kUnitAddUp) != 0;
    const bool identity = (unit.flags & kUnitIdentity) != 0;
    const int dv = (warp & 3) * 32 + lane;  // value channel = TMEM lane (warps 0-7)

    if (*status != 0) {  // invalid batch table: make the failure visible in final_state
        if (warp >= 4 && Sout)
            for (int c = 0; c < kD; ++c) Sout[(int64_t)c * kD + dv] = __int_as_float(0x7fc00000);
        return;
    }
    const int c_begin = unit.c_begin, c_end = unit.c_end;
    const int64_t t_begin = unit.t_begin, t_end = unit.t_end;
    auto rec_of = [&](int c) { return records + ((int64_t)c * H + h) * (int64_t)kRecBytes; };

    if (warp == 0) {
        if (lane == 0) {
            tc::mbar_init(&s.bar_m1, 1);
            tc::mbar_init(&s.bar_m2, 1);
            tc::mbar_init(&s.bar_ch, 1);
            tc::mbar_init_fence();
            s.fail = 0;
        }
        __syncwarp();
        tc::tmem_alloc(&s.tmem_base, kWalkTmemCols);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s.tmem_base;
    const uint32_t lanes = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t D_UO = tmem, D_AK = tmem + 128;
    volatile int &fail = s.fail;

    // A walk without outputs (segment maps) needs only -W and Kend^T: it copies those
    // parts of the record and runs group 1 with N = 64, group 2 with N = 128.
    constexpr bool maps = kMaps;
    const uint32_t ds_col = maps ? 0u : 64u;  // TMEM column of D_S within D_AK
    // this thread's half of its value column of S: key rows 0 .. 63 in the state warps,
    // 64 .. 127 in the U and O warps, so that both halves are updated at the same time
    uint64_t Sh[32];  // key rows 2j, 2j + 1 of this half as one packed pair
    // tokens 32 half .. 32 half + 31 of o = D_O1 + D_O2 for this thread's value channel,
    // into the [token][channel] staging tile (fp32, or bf16 in its first half)
    auto stage_o = [&](int half) {
        uint32_t d1[32], d2[32];
        tc::fence_after_sync();
        tc::tmem_ld32_nowait(D_UO + lanes + 64 + 32 * half, d1);
        tc::tmem_ld32_nowait(D_AK + lanes + 32 * half, d2);
        tc::tmem_wait_ld();
        float *stage = reinterpret_cast<float *>(s.ut);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int i = 32 * half + j;
            const float ov = __uint_as_float(d1[j]) + __uint_as_float(d2[j]);
            if (o_f32)
                stage[i * kD + dv] = ov;
            else
                reinterpret_cast<__nv_bfloat16 *>(stage)[i * kD + dv] = __float2bfloat16_rn(ov);
        }
    };
    // chunk c's U' and [ -W ; Qhat ] (a map walk: -W alone) by this U and O thread's share
    // of 16-byte units
    auto copy_up_wq = [&](int c) {
        const unsigned char *rec = rec_of(c);
        const int wq_units = (maps ? kPlaneQK : kRecWQBytes) / 16;
        for (int u = tid; u < wq_units; u += 128) cp_async16(s.wq + 16 * u, rec + kRecW + 16 * u);
        if (add_up)
            for (int u = tid; u < kC * kD / 4; u += 128) cp_async16(s.up + 4 * u, rec + kRecUp + 16 * u);
    };
    // this thread's key rows of the start state, and their split S^T planes
    const int r0 = warp >= 4 ? 0 : 64;
    // a state in the quad layout (the chained form's own states): 16 float4 per thread
    auto load_quads = [&](const float *X) {
        const float4 *x4 = reinterpret_cast<const float4 *>(X) + (r0 / 4) * kD + dv;
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const float4 v = x4[q * kD];
            Sh[2 * q] = pk2(v.x, v.y);
            Sh[2 * q + 1] = pk2(v.z, v.w);
        }
    };
    auto load_start = [&]() {
        if (kChain && (unit.flags & kUnitInQuads)) {
            load_quads(S0);
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int r = r0 + 2 * j;
                Sh[j] = S0 ? pk2(S0[(int64_t)r * kD + dv], S0[(int64_t)(r + 1) * kD + dv])
                           : pk2((identity && r == dv) ? 1.f : 0.f, (identity && r + 1 == dv) ? 1.f : 0.f);
            }
        }
#pragma unroll
        for (int j = 0; j < 32; j += 16)
            split32_tmem_pk(&Sh[j], tmem + lanes + kColSHi + r0 / 2 + j, tmem + lanes + kColSLo + r0 / 2 + j);
        tc::tmem_wait_st();
    };

    // the chain of segment maps before the first chunk (every thread; thread 128 issues)
    const int chain = kChain ? unit.chain : 0;
    int n_ch = 0;  // chain MMA groups committed (issuer)
    if (kChain && chain > 0) {
        unsigned char *const cb = &s.ak[0][0];
        auto m_hi = [&](int b) { return cb + b * 2 * kPlaneSS; };
        auto m_lo = [&](int b) { return b ? s.ut : cb + kPlaneSS; };
        // M_j's planes into chain buffer b, in 16-byte units, by the threads outside the
        // issuer's warp (that warp is issuing the product while the copy is due)
        const bool copier = warp != 4;
        const int ct = tid < 128 ? tid : tid - 32;  // 0 .. 223 over the copying threads
        auto copy_m = [&](int j, int b) {
            const unsigned char *src =
                reinterpret_cast<const unsigned char *>(unit.maps + ((size_t)(j - 1) * H + h) * kStateFloats);
            for (int u = ct; u < 2 * kPlaneSS / 16; u += kWalkThreads - 32) {
                unsigned char *dst = u < kPlaneSS / 16 ? m_hi(b) + 16 * u : m_lo(b) + 16 * (u - kPlaneSS / 16);
                cp_async16(dst, src + 16 * u);
            }
        };
        // R_j of this thread's key rows, in flight in rq until the step's epilogue adds the
        // product (nothing reads them before, so the loads do not hold the thread up). The
        // issuer's warp loads it a step early, before it issues; the other warps first
        // thing while the product runs.
        const bool early_r = warp == 4;
        float4 rq[16];
        auto load_r = [&](int j) {
            const float4 *x4 =
                reinterpret_cast<const float4 *>(unit.offs + ((size_t)(j - 1) * H + h) * kStateFloats) +
                (r0 / 4) * kD + dv;
#pragma unroll
            for (int q = 0; q < 16; ++q) rq[q] = x4[q * kD];
        };
        if (copier) copy_m(1, 0);
        cp_async_commit();
        load_start();
        if (early_r) load_r(1);
        const uint32_t idc = tc::idesc_bf16_m128(kD);
        for (int j = 1; j <= chain; ++j) {
            const int b = (j - 1) & 1;
            cp_async_wait<0>();  // this thread's share of M_j
            fence_proxy_async();
            tc::fence_before_sync();
            __syncthreads();  // M_j in place, the S^T planes of X written
            tc::fence_after_sync();
            if (tid == 128) {
                if (!fail) {
                    const uint32_t bh = tc::smem_addr(m_hi(b)), bl = tc::smem_addr(m_lo(b));
#pragma unroll
                    for (int ks = 0; ks < kD / 16; ++ks) {
                        const uint64_t dh = tc::desc_k(bh, kD, ks), dl = tc::desc_k(bl, kD, ks);
                        tc::mma_ts(D_UO, tmem + kColSHi + 8 * ks, dh, idc, ks > 0);
                        tc::mma_ts(D_UO, tmem + kColSLo + 8 * ks, dh, idc, 1);
                        tc::mma_ts(D_UO, tmem + kColSHi + 8 * ks, dl, idc, 1);
                    }
                }
                if (skip_commit != -2 - (j - 1)) {  // (test hook: left out for one map)
                    tc::commit(&s.bar_ch);  // also after a failure, so that the count stays in step
                    ++n_ch;
                }
            }
            __syncwarp();
            // while the product runs: R_j, M_{j+1} into the other buffer (its last reader,
            // the product of step j - 1, has completed), and at the first step the first
            // chunk's U' and [ -W ; Qhat ]
            if (!early_r) load_r(j);
            if (copier && j < chain && !fail) copy_m(j + 1, b ^ 1);
            if (j == 1 && warp < 4 && c_begin < c_end) copy_up_wq(c_begin);
            cp_async_commit();
            const bool ok = wait_or_fail(&s.bar_ch, (uint32_t)b, fail, wlim);
            // X <- D + R on this thread's key rows (D column n = key row n), and the planes
            if (ok) {
                uint32_t d[2][32];
                tc::fence_after_sync();
                tc::tmem_ld32_nowait(D_UO + lanes + r0, d[0]);
                tc::tmem_ld32_nowait(D_UO + lanes + r0 + 32, d[1]);
                tc::tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const uint32_t *dq = &d[q >> 3][4 * (q & 7)];
                    Sh[2 * q] = add2(pk2(rq[q].x, rq[q].y), pk2(__uint_as_float(dq[0]), __uint_as_float(dq[1])));
                    Sh[2 * q + 1] = add2(pk2(rq[q].z, rq[q].w), pk2(__uint_as_float(dq[2]), __uint_as_float(dq[3])));
                }
            }
#pragma unroll
            for (int q = 0; q < 32; q += 16)
                split32_tmem_pk(&Sh[q], tmem + lanes + kColSHi + r0 / 2 + q, tmem + lanes + kColSLo + r0 / 2 + q);
            tc::tmem_wait_st();
            if (early_r && j < chain) load_r(j + 1);
        }
        // every map copy has landed (each was waited for at the step that used it) and the
        // last product has completed, so the chain buffers are free for the record tiles
    }

    if (warp < 4) {
        // ------------- U and O warps; they also hold key rows 64 .. 127 of S -------------
        // U' row i holds its 16-byte units (4 channels) XOR-swizzled by i % 32: a warp's
        // reads of one row hit 32 distinct banks
        auto up_at = [&](int i) { return i * kD + ((((dv >> 2) ^ (i & 31))) << 2) + (dv & 3); };
        if (chain == 0) {
            load_start();
            if (c_begin < c_end) copy_up_wq(c_begin);
        }
        cp_async_commit();
        cp_async_wait<0>();
        fence_proxy_async();  // the first [ -W ; Qhat ], for group 1
        named_sync(5, 128);   // the first U', for every U and O thread
        tc::fence_before_sync();
        named_arrive(kBarOR, 256);  // initial planes of rows 64 .. 127 written; nothing to read yet
        for (int c = c_begin; c < c_end; ++c) {
            const uint32_t ph = (uint32_t)((c - c_begin) & 1);
            const int64_t t0 = t_begin + (int64_t)(c - c_begin) * kC;
            const int L = (int)min((int64_t)kC, t_end - t0);
            const float gnext = reinterpret_cast<const float *>(rec_of(c) + kRecGam)[dv];
            // U' of this chunk into registers while group 1 runs
            uint64_t Upr[32];  // U' of tokens 2j, 2j + 1 of this value channel as one packed pair
#pragma unroll
            for (int j = 0; j < 32; ++j)
                Upr[j] = add_up ? pk2(s.up[up_at(2 * j)], s.up[up_at(2 * j + 1)]) : pk2(0.f, 0.f);
            // U^T = U'^T + D_U, written as split planes for group 2
            if (wait_in_order(&s.bar_m1, ph, fail, wlim)) {
                tc::fence_after_sync();
                uint32_t d0[32], d1[32];
                tc::tmem_ld32_nowait(D_UO + lanes, d0);
                tc::tmem_ld32_nowait(D_UO + lanes + 32, d1);
                tc::tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; j += 2) {  // two tokens per packed add
                    Upr[j / 2] = add2(Upr[j / 2], pk2(__uint_as_float(d0[j]), __uint_as_float(d0[j + 1])));
                    Upr[16 + j / 2] = add2(Upr[16 + j / 2], pk2(__uint_as_float(d1[j]), __uint_as_float(d1[j + 1])));
                }
                split32_tmem_pk(&Upr[0], tmem + lanes + kColUHi, tmem + lanes + kColULo);
                split32_tmem_pk(&Upr[16], tmem + lanes + kColUHi + 16, tmem + lanes + kColULo + 16);
                tc::tmem_wait_st();
            }
            tc::fence_before_sync();
            named_arrive(kBarU, 256);  // U^T planes complete; group 1 is done with [ -W ; Qhat ]
            s.gam_uo[ph][dv] = gnext;
            named_sync(5, 128);  // gamma of this chunk in place (this group's copy); U' read
            // the next chunk's U' and [ -W ; Qhat ] land while group 2 runs (this thread saw
            // group 1 complete, so the buffer is free)
            if (c + 1 < c_end && !fail) copy_up_wq(c + 1);
            cp_async_commit();
            const bool m2ok = wait_in_order(&s.bar_m2, ph, fail, wlim);
            // S <- Diag(gamma) S + D_S on key rows 64 .. 127, and their split planes
            {
                uint32_t dA[32], dB[32];
                if (m2ok) {
                    tc::fence_after_sync();
                    tc::tmem_ld32_nowait(D_AK + lanes + ds_col + 64, dA);
                    tc::tmem_ld32_nowait(D_AK + lanes + ds_col + 96, dB);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {  // S = gamma S + D_S, two rows per packed FMA
                        const float4 ga = *reinterpret_cast<const float4 *>(&s.gam_uo[ph][64 + j]);
                        const float4 gb = *reinterpret_cast<const float4 *>(&s.gam_uo[ph][96 + j]);
                        const int p = j / 2;
                        Sh[p] = fma2(pk2(ga.x, ga.y), Sh[p], pk2(__uint_as_float(dA[j]), __uint_as_float(dA[j + 1])));
                        Sh[p + 1] = fma2(pk2(ga.z, ga.w), Sh[p + 1],
                                         pk2(__uint_as_float(dA[j + 2]), __uint_as_float(dA[j + 3])));
                        Sh[16 + p] = fma2(pk2(gb.x, gb.y), Sh[16 + p],
                                          pk2(__uint_as_float(dB[j]), __uint_as_float(dB[j + 1])));
                        Sh[17 + p] = fma2(pk2(gb.z, gb.w), Sh[17 + p],
                                          pk2(__uint_as_float(dB[j + 2]), __uint_as_float(dB[j + 3])));
                    }
                }
                split32_tmem_pk(&Sh[0], tmem + lanes + kColSHi + 32, tmem + lanes + kColSLo + 32);
                split32_tmem_pk(&Sh[16], tmem + lanes + kColSHi + 48, tmem + lanes + kColSLo + 48);
                tc::tmem_wait_st();
            }
            // tokens 0 .. 31 of o = (D_O1 + D_O2)^T for this thread's value channel, staged
            // as [token][channel] in shared memory (the state warps stage tokens 32 .. 63)
            const bool ok = m2ok && write_o;
            if (ok) stage_o(0);
            cp_async_wait<0>();
            fence_proxy_async();  // the next [ -W ; Qhat ] in place, for group 1
            tc::fence_before_sync();
            named_sync(kBarOR, 256);  // rows 64 .. 127 of the next S^T planes written, D_S and
                                      // the output accumulators read: the next group 1 may start.
                                      // Also: the whole o tile staged, the next U' visible.
            // write the staged tile out in 16-byte row chunks while the next group 1 runs
            if (write_o) {  // uniform over the CTA: the named barrier below stays matched
                if (ok) {
                    const float *stage = reinterpret_cast<const float *>(s.ut);
                    const int chunks_per_row = o_f32 ? kD / 4 : kD / 8;  // 16-byte chunks
                    for (int e = tid; e < L * chunks_per_row; e += 128) {
                        const int i = e / chunks_per_row, ch = e % chunks_per_row;
                        const int64_t row = ((t0 + i) * H + h) * (int64_t)kD;
                        if (o_f32)
                            reinterpret_cast<uint4 *>(static_cast<float *>(o) + row)[ch] =
                                reinterpret_cast<const uint4 *>(stage + i * kD)[ch];
                        else
                            reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(o) + row)[ch] =
                                reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(stage) +
                                                                i * kD)[ch];
                    }
                }
                named_sync(5, 128);  // staged tile read out before the next output lands here
            }
        }
    } else {
        // ----------------- state warps (thread 128 issues the MMAs) -----------------
        const bool issuer = (tid == 128);
        const uint32_t kIdG1 = tc::idesc_bf16_m128(maps ? 64 : 128);
        const uint32_t kIdG1w = tc::idesc_bf16_m128(192);  // [ -W ; Qhat hi ; Qhat lo ]
        // [ A_qk ; Kend^T ] is stored MN-major (its rows n contiguous per token): B transposed
        const uint32_t kIdG2 = tc::idesc_bf16(128, maps ? 128 : 192, 1);
        const uint32_t ak_off = maps ? (uint32_t)kPlaneCC : 0u;  // group 2's B operand starts at Kend^T
        int n_m1 = 0, n_m2 = 0;  // MMA groups committed (issuer)
        // chunk c's [ A_qk ; Kend^T ] into slot (c - c_begin) & 1 by this thread's share of
        // 16-byte units (a map walk: the Kend^T rows of the hi and the lo plane). The A_qk
        // blocks above the diagonal are not in the record: both slots hold zeros there.
        auto copy_ak = [&](int c) {
            unsigned char *dst = s.ak[(c - c_begin) & 1];
            const unsigned char *src = rec_of(c) + kRecAK;
            if (maps) {
                for (int u = tid - 128; u < kPlaneKT / 16; u += 128) {
                    cp_async16(dst + kPlaneCC + 16 * u, src + kPlaneCC + 16 * u);
                    cp_async16(dst + kStackAK + kPlaneCC + 16 * u, src + kStackAK + kPlaneCC + 16 * u);
                }
            } else {
                // unrolled from one shared and one global base: this copy is issued on the
                // state warps' path between two chunks, where a loop with per-unit address
                // arithmetic measured slower
                const int t = tid - 128;
                const uint32_t sd = smem_u32(dst) + 16u * (uint32_t)t;
                const unsigned char *sg = src + 16 * t;
#pragma unroll
                for (int m = 0; m < (int)(2 * kStackAK / 2048); ++m) {
                    const int pm = m % (int)(kStackAK / 2048);  // 2048-byte step within its plane
                    if (pm >= (int)(kPlaneCC / 2048) || !aqk_zero_unit(t + 128 * pm))
                        cp_async16_s(sd + 2048u * m, sg + 2048 * m);
                }
            }
        };
        if (!maps) {
            // the zero blocks of A_qk in both slots (the map chain, if any, used these
            // buffers and has completed)
            for (int e = tid - 128; e < 4 * (int)(kPlaneCC / 16); e += 128) {
                const int u = e & (int)(kPlaneCC / 16 - 1), sp = e / (int)(kPlaneCC / 16);  // (slot, plane)
                if (aqk_zero_unit(u))
                    *reinterpret_cast<uint4 *>(&s.ak[sp >> 1][(sp & 1) * kStackAK + 16 * u]) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        // group 1 of the next chunk: [D_U | D_O1 | D_O2] = S^T [ -W ; Qhat hi ; Qhat lo ]^T
        auto issue_g1 = [&](int c) {
            tc::fence_after_sync();
            if (!fail) {
                // S^T hi times the three planes (N = 192: -W S, Qhat hi S, and Qhat lo S
                // into D_O2, which group 2 then adds A_qk U to) and S^T lo times -W and
                // Qhat hi (N = 128): 16 MMAs (W has one plane; a map walk has no Qhat)
                // (unrolled: a loop issuing from one thread cost ~90 cycles per MMA, about
                // what an N = 128 MMA takes to run)
                const uint32_t b0s = tc::smem_addr(s.wq);
                if (maps) {
#pragma unroll
                    for (int ks = 0; ks < kD / 16; ++ks) {
                        const uint64_t b0 = tc::desc_k(b0s, kD, ks);
                        tc::mma_ts(D_UO, tmem + kColSHi + 8 * ks, b0, kIdG1, ks > 0);
                        tc::mma_ts(D_UO, tmem + kColSLo + 8 * ks, b0, kIdG1, 1);
                    }
                } else {
#pragma unroll
                    for (int ks = 0; ks < kD / 16; ++ks) {
                        const uint64_t b0 = tc::desc_k(b0s, kD, ks);
                        tc::mma_ts(D_UO, tmem + kColSHi + 8 * ks, b0, kIdG1w, ks > 0);
                        tc::mma_ts(D_UO, tmem + kColSLo + 8 * ks, b0, kIdG1, 1);
                    }
                }
            }
            if (c != skip_commit) {  // (test hook: left out for one chunk)
                tc::commit(&s.bar_m1);  // also after a failure: the U and O warps wait for it in order
                ++n_m1;
            }
        };
        // group 2 of chunk c: [D_O2 | D_S] += U^T [ A_qk ; Kend^T ]^T; D_O2 holds Qhat lo S
        // from group 1, so only D_S starts from zero: the first product is issued as two
        // MMAs (A_qk rows accumulating, Kend^T rows not)
        const uint32_t kIdAq = tc::idesc_bf16(128, 64, 1), kIdKe = tc::idesc_bf16(128, 128, 1);
        auto issue_g2 = [&](int c) {
            tc::fence_after_sync();
            const int slot = (c - c_begin) & 1;
            if (!fail) {
                const uint32_t b0s = tc::smem_addr(s.ak[slot]) + ak_off, b1s = b0s + (uint32_t)kStackAK;
#pragma unroll
                for (int ks = 0; ks < kC / 16; ++ks) {
                    const uint32_t a0 = tmem + kColUHi + 8 * ks, a1 = tmem + kColULo + 8 * ks;
                    const uint64_t b0 = tc::desc_k(b0s, kC, ks), b1 = tc::desc_k(b1s, kC, ks);
                    if (ks > 0 || maps) {
                        tc::mma_ts(D_AK, a0, b0, kIdG2, ks > 0);
                    } else {
                        tc::mma_ts(D_AK, a0, b0, kIdAq, 1);
                        tc::mma_ts(D_AK + 64, a0, tc::desc_k(b0s + (uint32_t)kPlaneCC, kC, 0), kIdKe, 0);
                    }
                    tc::mma_ts(D_AK, a0, b1, kIdG2, 1);
                    tc::mma_ts(D_AK, a1, b0, kIdG2, 1);
                }
            }
            tc::commit(&s.bar_m2);  // also after a failure (see group 1)
            ++n_m2;
        };

        // the first two chunks' [ A_qk ; Kend^T ] are copied while the initial state is read:
        // one cp.async group per chunk, here and in every step, so that the group of chunk
        // c is always the second newest when its group 2 is issued
        if (c_begin < c_end) copy_ak(c_begin);
        cp_async_commit();
        if (c_begin + 1 < c_end) copy_ak(c_begin + 1);
        cp_async_commit();
        // key rows 0 .. 63 of this thread's value column (the U and O warps hold the rest)
        if (chain == 0) load_start();
        tc::fence_before_sync();
        named_sync(4, 128);  // initial S^T planes of rows 0 .. 63 complete
        named_sync(kBarOR, 256);
        if (issuer && c_begin < c_end) issue_g1(c_begin);
        __syncwarp();
        for (int c = c_begin; c < c_end; ++c) {
            const uint32_t ph = (uint32_t)((c - c_begin) & 1);
            const float gnext = reinterpret_cast<const float *>(rec_of(c) + kRecGam)[dv];
            cp_async_wait<1>();   // this thread's share of chunk c's [ A_qk ; Kend^T ]
            fence_proxy_async();  // ... for group 2
            __syncwarp();
            named_sync(kBarU, 256);  // U^T planes of this chunk written (group 1 has finished)
            if (issuer) issue_g2(c);
            __syncwarp();
            const bool ok = wait_or_fail(&s.bar_m2, ph, fail, wlim);
            s.gam[ph][dv] = gnext;
            named_sync(4, 128);  // gamma of this chunk in place
            // S <- Diag(gamma) S + D_S on key rows 0 .. 63 and their split planes, in blocks
            // of 32 key channels: the TMEM load of the second block is in flight while the
            // first is updated, split and stored
            {
                uint32_t dA[32], dB[32];
                if (ok) {
                    tc::fence_after_sync();
                    tc::tmem_ld32_nowait(D_AK + lanes + ds_col, dA);
                }
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    uint32_t(&cur)[32] = (b & 1) ? dB : dA;
                    uint32_t(&nxt)[32] = (b & 1) ? dA : dB;
                    if (ok) {
                        tc::tmem_wait_ld();
                        if (b + 1 < 2) tc::tmem_ld32_nowait(D_AK + lanes + ds_col + 32 * (b + 1), nxt);
#pragma unroll
                        for (int j = 0; j < 32; j += 4) {  // S = gamma S + D_S, two rows per packed FMA
                            const int cc = 32 * b + j, p = cc / 2;
                            const float4 g = *reinterpret_cast<const float4 *>(&s.gam[ph][cc]);
                            Sh[p] = fma2(pk2(g.x, g.y), Sh[p], pk2(__uint_as_float(cur[j]), __uint_as_float(cur[j + 1])));
                            Sh[p + 1] = fma2(pk2(g.z, g.w), Sh[p + 1],
                                             pk2(__uint_as_float(cur[j + 2]), __uint_as_float(cur[j + 3])));
                        }
                    }
                    split32_tmem_pk(&Sh[16 * b], tmem + lanes + kColSHi + 16 * b, tmem + lanes + kColSLo + 16 * b);
                }
            }
            tc::tmem_wait_st();
            if (ok && write_o) stage_o(1);  // tokens 32 .. 63 of o (the U and O warps store the tile)
            tc::fence_before_sync();
            named_sync(4, 128);       // rows 0 .. 63 of the next S^T planes complete
            named_sync(kBarOR, 256);  // the U and O warps have written rows 64 .. 127, read this
                                      // chunk's D_S and output accumulators, and copied the next
                                      // [ -W ; Qhat ]
            if (issuer && c + 1 < c_end) issue_g1(c + 1);
            __syncwarp();
            // group 2 is done with this slot (every state thread saw it complete): the chunk
            // after next lands there while the next groups run
            if (ok && c + 2 < c_end) copy_ak(c + 2);
            cp_async_commit();
        }
        if (issuer && fail) {
            // a wait gave up: let MMAs still in flight land (bounded) before shared memory
            // and TMEM are released, and report through the status word
            if (n_m1 > 0) tc::mbar_wait(&s.bar_m1, (uint32_t)((n_m1 - 1) & 1), wlim);
            if (n_m2 > 0) tc::mbar_wait(&s.bar_m2, (uint32_t)((n_m2 - 1) & 1), wlim);
            if (n_ch > 0) tc::mbar_wait(&s.bar_ch, (uint32_t)((n_ch - 1) & 1), wlim);
            atomicExch(status, -7);
        }
    }
    cp_async_wait<0>();  // no copy of this thread still in flight when the CTA ends

    tc::fence_before_sync();
    __syncthreads();
    // the final state: rows 0 .. 63 from the state warps, 64 .. 127 from the U and O warps
    // (every wait has ended: the failure flag is final)
    if (kMaps && Sout && (unit.flags & kUnitOutPlanes)) {
        // as the split planes of B[n][k] = S[n][k]: each thread's column k = dv goes into a
        // row-major staging image (the 16-byte units of row n XOR-swizzled by n % 8, so that
        // neither the column writes nor the unit reads below conflict), then out in the
        // interleaved order, 16 bytes per thread and step
        const bool failed = fail;
        unsigned char *img = s.wq;  // 64 KB over wq and ak, free now
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float2 v = upk2(Sh[j]);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int n = r0 + 2 * j + e;
                const float x = failed ? __int_as_float(0x7fc00000) : (e ? v.y : v.x);
                const __nv_bfloat16 hi = __float2bfloat16_rn(x);
                const __nv_bfloat16 lo = __float2bfloat16_rn(x - __bfloat162float(hi));
                const int off = n * 2 * kD + ((((dv >> 3) ^ (n & 7))) << 4) + (dv & 7) * 2;
                *reinterpret_cast<__nv_bfloat16 *>(img + off) = hi;
                *reinterpret_cast<__nv_bfloat16 *>(img + kPlaneSS + off) = lo;
            }
        }
        __syncthreads();
        uint4 *dst = reinterpret_cast<uint4 *>(Sout);
        for (int u = tid; u < 2 * kPlaneSS / 16; u += kWalkThreads) {
            const int pl = u / (kPlaneSS / 16), gu = u % (kPlaneSS / 16);
            const int n = ((gu >> 7) << 3) | (gu & 7), k8 = (gu >> 3) & 15;  // gu * 16 = il_off(n, 8 k8, 128)
            dst[u] = *reinterpret_cast<const uint4 *>(img + pl * kPlaneSS + n * 2 * kD + ((k8 ^ (n & 7)) << 4));
        }
    } else if (kMaps && Sout && (unit.flags & kUnitOutQuads)) {
        const bool failed = fail;
        float4 *d4 = reinterpret_cast<float4 *>(Sout) + (r0 / 4) * kD + dv;
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const float2 a = upk2(Sh[2 * q]), b = upk2(Sh[2 * q + 1]);
            const float nan = __int_as_float(0x7fc00000);
            d4[q * kD] = failed ? make_float4(nan, nan, nan, nan) : make_float4(a.x, a.y, b.x, b.y);
        }
    } else if (Sout) {
        const bool failed = fail;
        float *dst = Sout + (warp >= 4 ? 0 : (int64_t)64 * kD) + dv;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float2 v = upk2(Sh[j]);
            dst[(int64_t)(2 * j) * kD] = failed ? __int_as_float(0x7fc00000) : v.x;
            dst[(int64_t)(2 * j + 1) * kD] = failed ? __int_as_float(0x7fc00000) : v.y;
        }
    }
    if (warp == 0) tc::tmem_dealloc(tmem, kWalkTmemCols);
}

// ---------------------------------------------------------------------------------
// host-side launchers (called from kda_api.cu)
// ---------------------------------------------------------------------------------
cudaError_t set_walk_fault(int32_t skip_commit_chunk, uint64_t wait_limit_ns) {
    const unsigned long long lim = wait_limit_ns;
    cudaError_t e = cudaMemcpyToSymbol(g_walk_skip_commit, &skip_commit_chunk, sizeof(int32_t));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_walk_wait_ns, &lim, sizeof(lim));
    return e;
}

cudaError_t launch_plan(const int32_t *cu, int32_t N, int64_t seq_len, int64_t total, int32_t *status,
                        int32_t *seq_cu, int32_t *chunk_off, int32_t H, const float *S0, float *Sout, WalkUnit *units,
                        int32_t *n_units, const SegPlan &sp, cudaStream_t st) {
    int sort_n = 0;  // a plain walk of 2 .. kPlanSortMax sequences is sorted, over a power of two
    if (sp.P == 0 && N >= 2 && N <= kPlanSortMax) {
        sort_n = 2;
        while (sort_n < N) sort_n <<= 1;
    }
    kda_plan_kernel<<<1, 256, (size_t)sort_n * sizeof(uint64_t), st>>>(cu, N, seq_len, total, status, seq_cu,
                                                                        chunk_off, H, S0, Sout, units, n_units, sp,
                                                                        sort_n);
    return cudaGetLastError();
}

cudaError_t launch_combine(const int32_t *status, const int32_t *chains, int32_t N, int32_t H, float *Sin,
                           const float *Mseg, const float *Rseg, cudaStream_t st) {
    static bool configured = false;
    if (!configured) {
        const cudaError_t e = cudaFuncSetAttribute(kda_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)sizeof(CombineSmem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    dim3 grid((unsigned)N, (unsigned)H, kD / 16);
    return launch_after(kda_combine_kernel, grid, dim3(kCombineThreads), sizeof(CombineSmem), st, status, chains, H,
                        Sin, Mseg, Rseg);
}

cudaError_t launch_walk(int32_t *status, const WalkUnit *units, const int32_t *n_units, int64_t max_units,
                        int32_t H, const uint8_t *records, void *o, int o_f32, int form, int head_major,
                        cudaStream_t st) {
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kda_walk_kernel<kWalkOut>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)sizeof(WalkSmem));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kda_walk_kernel<kWalkChain>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)sizeof(WalkSmem));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kda_walk_kernel<kWalkMaps>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)sizeof(WalkSmem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    if (max_units <= 0) return cudaSuccess;
    if (head_major && max_units > 65535) return cudaErrorInvalidConfiguration;
    const dim3 grid = head_major ? dim3((unsigned)H, (unsigned)max_units) : dim3((unsigned)max_units, (unsigned)H);
    auto kernel = form == kWalkChain ? kda_walk_kernel<kWalkChain>
                                     : (form == kWalkMaps ? kda_walk_kernel<kWalkMaps> : kda_walk_kernel<kWalkOut>);
    return launch_after(kernel, grid, dim3(kWalkThreads), sizeof(WalkSmem), st, status, units, n_units, H, records, o,
                        o_f32, head_major);
}

}  // namespace kda
