// KDA chunkwise prefill: three kernels on one stream.
//
//   kda_plan_kernel   validate cu_seqlens, tabulate sequence starts and chunk offsets
//   kda_intra_kernel  one CTA per (chunk, head), all chunks in parallel: gate and
//                     cumulative decay, decayed K K^T / Q K^T per 16-token tile row,
//                     UT transform T = (I + A_kk)^-1, W = T' Khat and U' = T' V
//   kda_walk_kernel   one CTA per (sequence, head): walks the chunks in order with the
//                     full state on chip, on tcgen05 tensor cores (TMEM accumulators),
//                     U = U' - W S;  O = Qhat S + A_qk U;  S = Diag(gamma) S + Kend^T U
//
// The algebra is the chunkwise form of 'From Linear Attention to KDA' (blog), §7.1-7.3
// with the per-channel decay of §7.2 folded into the UT system, and the 16-token
// tiles of §8 for the decayed Gram matrices. Inside one chunk (positions i, j):
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
// Decay factors never overflow: for tile row a (tokens 16a..16a+15) the reference
// point is r = 16a, and exp(G_i - G_j) = exp(G_i - G_r) * exp(G_r - G_j). The first
// factor is <= 1; the second is <= 1 for j <= r and at most e^75 (15 tokens of at most
// -5 each, §5.4 of the blog) inside the diagonal tile, within bf16/fp32 range.

#include "kda_common.cuh"
#include "kda_tc.cuh"

namespace kda {

// ---------------------------------------------------------------------------------
// plan: seq_cu[N+1] and chunk_off[N+1] (prefix sums of ceil(len / C)) in the workspace
// ---------------------------------------------------------------------------------
__global__ void kda_plan_kernel(const int32_t *__restrict__ cu_seqlens, int32_t N, int64_t seq_len,
                                int64_t total_tokens, int32_t *__restrict__ status, int32_t *__restrict__ seq_cu,
                                int32_t *__restrict__ chunk_off) {
    __shared__ int32_t carry;
    __shared__ int32_t bad;
    __shared__ int32_t scan[256];
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
        for (int64_t n = tid; n <= N; n += blockDim.x) {
            seq_cu[n] = 0;
            chunk_off[n] = 0;
        }
        if (tid == 0) *status = -4;  // KDA_ERR_SEQLENS
        return;
    }
    if (tid == 0) *status = 0;
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
        __syncthreads();
        if (tid == 255) carry += scan[255];
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------------
// intra-chunk kernel
// ---------------------------------------------------------------------------------
struct IntraSmem {
    float G[kC][kD + 4];  // z of the chunk, then (in place) the cumulative log decay
    float beta[kC];
    float Akk[kC][kC + 1];
    float Aqk[kC][kC + 1];
    float T[kC][kC + 1];
    float X[3][kTile][kTile + 1];  // off-diagonal block products of the solve
    __nv_bfloat16 qs[kC][kLd128];  // the chunk's q, k, v (rows past the sequence end are zero)
    __nv_bfloat16 ks[kC][kLd128];
    __nv_bfloat16 vs[kC][kLd128];
    union {
        struct {  // operands of the decayed Gram products of one tile row
            __nv_bfloat16 aq[2][kTile][kLd128];
            __nv_bfloat16 ak[2][kTile][kLd128];
            __nv_bfloat16 bk[2][kC][kLd128];
        } g;
        struct {  // operands of W = T' Khat and U' = T' V
            __nv_bfloat16 kh[2][kC][kLd128];
            __nv_bfloat16 t[2][kC][kLd64];
        } w;
    } u;
};

constexpr int kIntraThreads = 256;

__device__ __forceinline__ int find_seq(const int32_t *chunk_off, int32_t N, int32_t slot) {
    // largest n with chunk_off[n] <= slot (empty sequences share an offset and are skipped)
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (chunk_off[mid] <= slot)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

__global__ void __launch_bounds__(kIntraThreads, 1)
    kda_intra_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                     const __nv_bfloat16 *__restrict__ v, const float *__restrict__ z, const float *__restrict__ A,
                     const float *__restrict__ bgate, const int32_t *__restrict__ status,
                     const int32_t *__restrict__ seq_cu, const int32_t *__restrict__ chunk_off, int32_t N, int32_t H,
                     uint8_t *__restrict__ records) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    IntraSmem &s = *reinterpret_cast<IntraSmem *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int slot = blockIdx.x, h = blockIdx.y;
    if (*status != 0 || N <= 0) return;
    if (slot >= chunk_off[N]) return;
    const int n = find_seq(chunk_off, N, slot);
    const int64_t t0 = (int64_t)seq_cu[n] + (int64_t)(slot - chunk_off[n]) * kC;
    const int L = (int)min((int64_t)kC, (int64_t)seq_cu[n + 1] - t0);
    const int64_t rowstride = (int64_t)H * kD;  // elements between consecutive tokens
    const int64_t hoff = (int64_t)h * kD;
    uint8_t *rec = records + ((int64_t)slot * H + h) * (int64_t)kRecBytes;

    // ---- stage z, q, k, v of the chunk in shared memory (all requests in flight at once) ----
    for (int e = tid; e < kC * (kD / 4); e += kIntraThreads) {  // z: 32 x 16 B per row
        const int i = e / (kD / 4), c = (e % (kD / 4)) * 4;
        float *dst = &s.G[i][c];
        if (i < L)
            cp_async16(dst, z + (t0 + i) * rowstride + hoff + c);
        else
            *reinterpret_cast<float4 *>(dst) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int e = tid; e < 3 * kC * (kD / 8); e += kIntraThreads) {  // q, k, v: 16 x 16 B per row
        const int which = e / (kC * (kD / 8));
        const int r = e % (kC * (kD / 8));
        const int i = r / (kD / 8), c = (r % (kD / 8)) * 8;
        const __nv_bfloat16 *src = which == 0 ? q : (which == 1 ? k : v);
        __nv_bfloat16 *dst = which == 0 ? &s.qs[i][c] : (which == 1 ? &s.ks[i][c] : &s.vs[i][c]);
        if (i < L)
            cp_async16(dst, src + (t0 + i) * rowstride + hoff + c);
        else
            *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
    cp_async_commit();
    if (tid >= kD && tid < kD + kC) {
        const int i = tid - kD;
        s.beta[i] = (i < L) ? sigmoid_f(bgate[(t0 + i) * H + h]) : 0.f;
    }
    for (int e = tid; e < kC * (kC + 1); e += kIntraThreads) {
        (&s.Akk[0][0])[e] = 0.f;
        (&s.Aqk[0][0])[e] = 0.f;
    }
    cp_async_wait<0>();
    __syncthreads();

    // ---- gate and cumulative log decay, in place over z (rows past the end add 0) ----
    if (tid < kD) {
        const float eA = expf(A[h]);
        float acc = 0.f;
#pragma unroll 8
        for (int i = 0; i < kC; ++i) {
            if (i < L) acc += gate_log_decay(eA, s.G[i][tid]);
            s.G[i][tid] = acc;
        }
    }
    __syncthreads();

    // ---- decayed Gram matrices, one 16-token tile row at a time -----------------
    for (int a = 0; a < kC / kTile; ++a) {
        const int r = a * kTile;  // reference token of this tile row
        const int nb = r + kTile; // key rows j = 0 .. r+15
        const int items = (2 * kTile + nb) * (kD / 2);
        for (int e = tid; e < items; e += kIntraThreads) {
            const int row = e / (kD / 2);
            const int c = (e % (kD / 2)) * 2;
            int tok;
            const __nv_bfloat16 *src;
            __nv_bfloat16 *dhi, *dlo;
            bool fwd;  // factor exp(G_tok - G_r) (true) or exp(G_r - G_tok) (false)
            if (row < kTile) {
                tok = r + row; src = &s.qs[tok][c]; fwd = true;
                dhi = &s.u.g.aq[0][row][c]; dlo = &s.u.g.aq[1][row][c];
            } else if (row < 2 * kTile) {
                tok = r + row - kTile; src = &s.ks[tok][c]; fwd = true;
                dhi = &s.u.g.ak[0][row - kTile][c]; dlo = &s.u.g.ak[1][row - kTile][c];
            } else {
                tok = row - 2 * kTile; src = &s.ks[tok][c]; fwd = false;
                dhi = &s.u.g.bk[0][tok][c]; dlo = &s.u.g.bk[1][tok][c];
            }
            float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(src));
            {
                const float d0 = fwd ? s.G[tok][c] - s.G[r][c] : s.G[r][c] - s.G[tok][c];
                const float d1 = fwd ? s.G[tok][c + 1] - s.G[r][c + 1] : s.G[r][c + 1] - s.G[tok][c + 1];
                x.x *= expf(d0);
                x.y *= expf(d1);
            }
            uint32_t hi, lo;
            split_bf16x2(x.x, x.y, hi, lo);
            *reinterpret_cast<uint32_t *>(dhi) = hi;
            *reinterpret_cast<uint32_t *>(dlo) = lo;
        }
        __syncthreads();
        const int ntiles = nb / 8;  // n8 tiles of key rows
        for (int p = warp; p < 2 * ntiles; p += kIntraThreads / 32) {
            const int mat = p / ntiles;  // 0: A_qk, 1: A_kk
            const int nt = p % ntiles;
            const __nv_bfloat16 *ah_base = mat ? &s.u.g.ak[0][0][0] : &s.u.g.aq[0][0][0];
            const __nv_bfloat16 *al_base = mat ? &s.u.g.ak[1][0][0] : &s.u.g.aq[1][0][0];
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < kD / 16; ++ks) {
                uint32_t ah[4], al[4], bh0, bh1, bl0, bl1;
                load_a(ah, ah_base, kLd128, 0, ks * 16, lane);
                load_a(al, al_base, kLd128, 0, ks * 16, lane);
                load_b_nk(bh0, bh1, &s.u.g.bk[0][0][0], kLd128, nt * 8, ks * 16, lane);
                load_b_nk(bl0, bl1, &s.u.g.bk[1][0][0], kLd128, nt * 8, ks * 16, lane);
                mma_split3(acc, ah, al, bh0, bh1, bl0, bl1);
            }
            const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = r + g + ((e >> 1) << 3);
                const int j = nt * 8 + 2 * t4 + (e & 1);
                if (mat == 0)
                    s.Aqk[i][j] = (j <= i) ? acc[e] : 0.f;
                else
                    s.Akk[i][j] = (j < i) ? s.beta[i] * acc[e] : 0.f;
            }
        }
        __syncthreads();
    }

    // ---- UT transform: T = (I + A_kk)^-1, unit lower triangular -----------------
    // diagonal 16x16 blocks by forward substitution, one column per thread
    if (tid < 64) {
        const int a = tid >> 4, j = tid & 15, base = a * kTile;
        for (int i = 0; i < kTile; ++i) {
            float val;
            if (i < j) {
                val = 0.f;
            } else if (i == j) {
                val = 1.f;
            } else {
                float acc = 0.f;
                for (int m = j; m < i; ++m) acc += s.Akk[base + i][base + m] * s.T[base + m][base + j];
                val = -acc;
            }
            s.T[base + i][base + j] = val;
        }
    } else {
        // zero the blocks above the diagonal
        for (int e = tid - 64; e < kC * kC; e += kIntraThreads - 64) {
            const int i = e / kC, j = e % kC;
            if ((j >> 4) > (i >> 4)) s.T[i][j] = 0.f;
        }
    }
    __syncthreads();
    // off-diagonal blocks by distance l: T_ab = -T_aa * sum_{m=b}^{a-1} A_am T_mb
    for (int l = 1; l < kC / kTile; ++l) {
        const int nblk = kC / kTile - l;
        for (int e = tid; e < nblk * kTile * kTile; e += kIntraThreads) {
            const int blk = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
            const int b = blk, a = b + l;
            float acc = 0.f;
            for (int m = b; m < a; ++m)
#pragma unroll
                for (int x = 0; x < kTile; ++x) acc += s.Akk[a * kTile + rr][m * kTile + x] * s.T[m * kTile + x][b * kTile + cc];
            s.X[blk][rr][cc] = acc;
        }
        __syncthreads();
        for (int e = tid; e < nblk * kTile * kTile; e += kIntraThreads) {
            const int blk = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
            const int b = blk, a = b + l;
            float acc = 0.f;
#pragma unroll
            for (int x = 0; x < kTile; ++x) acc += s.T[a * kTile + rr][a * kTile + x] * s.X[blk][x][cc];
            s.T[a * kTile + rr][b * kTile + cc] = -acc;
        }
        __syncthreads();
    }

    // ---- operands of W and U': T' = T Diag(beta), Khat = k * exp(G), V ------------
    for (int e = tid; e < kC * (kC / 2); e += kIntraThreads) {
        const int i = e / (kC / 2), j = (e % (kC / 2)) * 2;
        uint32_t hi, lo;
        split_bf16x2(s.T[i][j] * s.beta[j], s.T[i][j + 1] * s.beta[j + 1], hi, lo);
        *reinterpret_cast<uint32_t *>(&s.u.w.t[0][i][j]) = hi;
        *reinterpret_cast<uint32_t *>(&s.u.w.t[1][i][j]) = lo;
    }
    for (int e = tid; e < kC * (kD / 2); e += kIntraThreads) {
        const int i = e / (kD / 2), c = (e % (kD / 2)) * 2;
        const float2 kk = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&s.ks[i][c]));
        uint32_t hi, lo;
        split_bf16x2(kk.x * expf(s.G[i][c]), kk.y * expf(s.G[i][c + 1]), hi, lo);
        *reinterpret_cast<uint32_t *>(&s.u.w.kh[0][i][c]) = hi;
        *reinterpret_cast<uint32_t *>(&s.u.w.kh[1][i][c]) = lo;
    }
    __syncthreads();

    // ---- W = T' Khat (split x split), U' = T' V (split x exact bf16) ------------
    // warp w owns output columns 16w .. 16w+15 (two n8 tiles) for all 64 rows
    {
        float accW[4][2][4], accU[4][2][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    accW[a][nt][e] = 0.f;
                    accU[a][nt][e] = 0.f;
                }
        const int n0 = warp * 16;
#pragma unroll
        for (int a = 0; a < 4; ++a) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                if (ks > a) break;  // T' is lower triangular
                uint32_t th[4], tl[4], kh[4], kl[4], vb[4];
                load_a(th, &s.u.w.t[0][0][0], kLd64, a * 16, ks * 16, lane);
                load_a(tl, &s.u.w.t[1][0][0], kLd64, a * 16, ks * 16, lane);
                load_b_kn(kh, &s.u.w.kh[0][0][0], kLd128, ks * 16, n0, lane);
                load_b_kn(kl, &s.u.w.kh[1][0][0], kLd128, ks * 16, n0, lane);
                load_b_kn(vb, &s.vs[0][0], kLd128, ks * 16, n0, lane);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    mma_split3(accW[a][nt], th, tl, kh[2 * nt], kh[2 * nt + 1], kl[2 * nt], kl[2 * nt + 1]);
                    mma_bf16(accU[a][nt], tl, vb[2 * nt], vb[2 * nt + 1]);
                    mma_bf16(accU[a][nt], th, vb[2 * nt], vb[2 * nt + 1]);
                }
            }
        }
        // write -W (split, interleaved tiles) and U' (fp32, token-major) to the record
        uint8_t *Wn = rec + kRecWn;
        float *Up = reinterpret_cast<float *>(rec + kRecUp);
        const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int i = a * 16 + g + hr * 8;
                    const int c = n0 + nt * 8 + 2 * t4;
                    uint32_t hi, lo;
                    split_bf16x2(-accW[a][nt][2 * hr], -accW[a][nt][2 * hr + 1], hi, lo);
                    *reinterpret_cast<uint32_t *>(Wn + il_off(i, c, kD)) = hi;
                    *reinterpret_cast<uint32_t *>(Wn + kPlaneQK + il_off(i, c, kD)) = lo;
                    *reinterpret_cast<float2 *>(Up + (size_t)i * kD + c) =
                        make_float2(accU[a][nt][2 * hr], accU[a][nt][2 * hr + 1]);
                }
    }

    // ---- Qhat, Kend^T, A_qk, gamma (elementwise) --------------------------------
    {
        uint8_t *Qh = rec + kRecQh;
        for (int e = tid; e < kC * (kD / 2); e += kIntraThreads) {
            const int i = e / (kD / 2), c = (e % (kD / 2)) * 2;
            const float2 qq = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&s.qs[i][c]));
            uint32_t hi, lo;
            split_bf16x2(qq.x * expf(s.G[i][c]), qq.y * expf(s.G[i][c + 1]), hi, lo);
            *reinterpret_cast<uint32_t *>(Qh + il_off(i, c, kD)) = hi;
            *reinterpret_cast<uint32_t *>(Qh + kPlaneQK + il_off(i, c, kD)) = lo;
        }
        uint8_t *KeT = rec + kRecKeT;
        for (int e = tid; e < kD * (kC / 2); e += kIntraThreads) {
            const int c = e / (kC / 2), j = (e % (kC / 2)) * 2;
            const float k0 = __bfloat162float(s.ks[j][c]);
            const float k1 = __bfloat162float(s.ks[j + 1][c]);
            const float gl = s.G[kC - 1][c];
            uint32_t hi, lo;
            split_bf16x2(k0 * expf(gl - s.G[j][c]), k1 * expf(gl - s.G[j + 1][c]), hi, lo);
            *reinterpret_cast<uint32_t *>(KeT + il_off(c, j, kC)) = hi;
            *reinterpret_cast<uint32_t *>(KeT + kPlaneKT + il_off(c, j, kC)) = lo;
        }
        uint8_t *Aq = rec + kRecAqk;
        for (int e = tid; e < kC * (kC / 2); e += kIntraThreads) {
            const int i = e / (kC / 2), j = (e % (kC / 2)) * 2;
            uint32_t hi, lo;
            split_bf16x2(s.Aqk[i][j], s.Aqk[i][j + 1], hi, lo);
            *reinterpret_cast<uint32_t *>(Aq + il_off(i, j, kC)) = hi;
            *reinterpret_cast<uint32_t *>(Aq + kPlaneCC + il_off(i, j, kC)) = lo;
        }
        float *gam = reinterpret_cast<float *>(rec + kRecGam);
        if (tid < kD) gam[tid] = expf(s.G[kC - 1][tid]);
    }
}

// ---------------------------------------------------------------------------------
// state walk: one CTA per (sequence, head) carries the full 128 x 128 state through
// the chunks of its sequence, on the tensor cores (tcgen05, accumulators in TMEM).
//
// Transposed orientation, so that the 128 value channels are the MMA's M = 128 rows
// and every accumulator row is one TMEM lane:
//   D_U = S^T (-W)^T          [128 x 64]   then U^T = U'^T + D_U       (per thread)
//   D_O = S^T Qhat^T          [128 x 64]
//   D_O += U^T A_qk^T                      then o = D_O^T
//   D_S = U^T Kend             [128 x 128]  then S^T = S^T Diag(gamma) + D_S
// Each product is split-bf16 (hi*hi + hi*lo + lo*hi). S^T and U^T go to shared memory as
// split planes (the A operands); the record tiles are the B operands, fetched with bulk
// copies one chunk ahead: W and Qhat as soon as the first group of MMAs has finished
// with them, Kend, A_qk and gamma once the state update has.
//
// Thread t of warp w owns value channel dv = 32 (w % 4) + lane (TMEM lane dv) and half
// hf = w / 4 of the columns: tokens 32 hf .. 32 hf + 31 of D_U / D_O, key channels
// 64 hf .. 64 hf + 63 of the state, which it keeps in registers in fp32.
// ---------------------------------------------------------------------------------
struct WalkSmem {
    unsigned char wq[2 * kPlaneQK + 2 * kPlaneQK];             // Wn hi, lo | Qh hi, lo
    unsigned char ka[2 * kPlaneKT + 2 * kPlaneCC + kD * 4];    // KeT hi, lo | Aqk hi, lo | gamma
    unsigned char st[2 * 128 * kD * 2];                        // S^T hi, lo   (M 128 x K 128)
    unsigned char ut[2 * 128 * kC * 2];                        // U^T hi, lo   (M 128 x K 64)
    uint64_t bar_wq, bar_ka, bar_m1, bar_m2;
    uint32_t tmem_base;
    int fail;
};
static_assert(sizeof(WalkSmem) <= 227 * 1024, "walk shared memory");

constexpr int kWalkThreads = 256;
constexpr uint32_t kWalkTmemCols = 256;  // D_U [0,64) | D_O [64,128) | D_S [128,256)

// 8 consecutive fp32 values -> one 16-byte chunk of the hi plane and one of the lo plane
__device__ __forceinline__ void split8_store(const float *x, unsigned char *hi_plane, unsigned char *lo_plane,
                                             uint32_t off) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) split_bf16x2(x[2 * j], x[2 * j + 1], h[j], l[j]);
    *reinterpret_cast<uint4 *>(hi_plane + off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4 *>(lo_plane + off) = make_uint4(l[0], l[1], l[2], l[3]);
}

__global__ void __launch_bounds__(kWalkThreads, 1)
    kda_walk_kernel(int32_t *__restrict__ status, const int32_t *__restrict__ seq_cu,
                    const int32_t *__restrict__ chunk_off, int32_t H, const uint8_t *__restrict__ records,
                    const float *__restrict__ S0, float *__restrict__ Sout, void *__restrict__ o, int o_f32) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    WalkSmem &s = *reinterpret_cast<WalkSmem *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3, hf = warp >> 2;
    const int dv = 32 * q4 + lane;
    const int n = blockIdx.x, h = blockIdx.y;
    const int64_t sbase = ((int64_t)n * H + h) * kD * kD;

    if (*status != 0) {  // invalid batch table: make the failure visible in final_state
        for (int c = hf * 64; c < hf * 64 + 64; ++c) Sout[sbase + (int64_t)c * kD + dv] = __int_as_float(0x7fc00000);
        return;
    }
    const int c_begin = chunk_off[n], c_end = chunk_off[n + 1];
    const int64_t t_begin = seq_cu[n], t_end = seq_cu[n + 1];
    auto rec_of = [&](int c) { return records + ((int64_t)c * H + h) * (int64_t)kRecBytes; };

    if (tid == 0) {
        tc::mbar_init(&s.bar_wq, 1);
        tc::mbar_init(&s.bar_ka, 1);
        tc::mbar_init(&s.bar_m1, 1);
        tc::mbar_init(&s.bar_m2, 1);
        tc::mbar_init_fence();
        s.fail = 0;
    }
    if (warp == 0) tc::tmem_alloc(&s.tmem_base, kWalkTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s.tmem_base;
    const uint32_t lanes = (uint32_t)(32 * q4) << 16;
    const uint32_t D_U = tmem, D_O = tmem + 64, D_S = tmem + 128;

    auto issue_wq = [&](int c) {
        tc::mbar_arrive_expect_tx(&s.bar_wq, (uint32_t)(4 * kPlaneQK));
        tc::bulk_g2s(s.wq, rec_of(c) + kRecWn, (uint32_t)(4 * kPlaneQK), &s.bar_wq);
    };
    auto issue_ka = [&](int c) {
        const uint32_t bytes = (uint32_t)(2 * kPlaneKT + 2 * kPlaneCC + kD * 4);
        tc::mbar_arrive_expect_tx(&s.bar_ka, bytes);
        tc::bulk_g2s(s.ka, rec_of(c) + kRecKeT, bytes, &s.bar_ka);
    };
    if (tid == 0 && c_begin < c_end) {
        issue_wq(c_begin);
        issue_ka(c_begin);
    }

    // state: S[c][dv] for this thread's 64 key channels, in fp32
    float Sr[64];
#pragma unroll
    for (int j = 0; j < 64; ++j) Sr[j] = S0 ? S0[sbase + (int64_t)(hf * 64 + j) * kD + dv] : 0.f;
    auto store_state = [&]() {
#pragma unroll
        for (int j = 0; j < 64; j += 8)
            split8_store(&Sr[j], s.st, s.st + 128 * kD * 2, il_off(dv, hf * 64 + j, kD));
    };
    store_state();
    // U' of the first chunk: U'[i][dv] for this thread's 32 tokens
    float Upr[32];
    auto load_up = [&](int c) {
        const float *up = reinterpret_cast<const float *>(rec_of(c) + kRecUp);
#pragma unroll
        for (int j = 0; j < 32; ++j) Upr[j] = up[(hf * 32 + j) * kD + dv];
    };
    if (c_begin < c_end) load_up(c_begin);
    tc::fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();

    constexpr uint32_t kId64 = tc::idesc_bf16_m128(64);
    constexpr uint32_t kId128 = tc::idesc_bf16_m128(128);
    volatile int &fail = s.fail;
    // completed-phase counts, used to drain in-flight work if a wait ever gives up
    int n_wq = (c_begin < c_end) ? 1 : 0, n_ka = n_wq, w_wq = 0, w_ka = 0, n_m1 = 0, n_m2 = 0;
    for (int c = c_begin; c < c_end; ++c) {
        const uint32_t ph = (uint32_t)((c - c_begin) & 1);
        const int64_t t0 = t_begin + (int64_t)(c - c_begin) * kC;
        const int L = (int)min((int64_t)kC, t_end - t0);

        // ---- group 1: D_U = S^T (-W)^T, D_O = S^T Qhat^T ----
        if (tid == 0) {
            tc::fence_after_sync();
            if (tc::mbar_wait(&s.bar_wq, ph)) {
                ++w_wq;
                const uint32_t s0 = tc::smem_addr(s.st), s1 = s0 + 128 * kD * 2;
                const uint32_t w0 = tc::smem_addr(s.wq), w1 = w0 + kPlaneQK;
                const uint32_t q0 = w0 + 2 * kPlaneQK, q1 = q0 + kPlaneQK;
#pragma unroll 1
                for (int ks = 0; ks < kD / 16; ++ks) {
                    const uint64_t a0 = tc::desc_k(s0, kD, ks), a1 = tc::desc_k(s1, kD, ks);
                    tc::mma(D_U, a0, tc::desc_k(w0, kD, ks), kId64, ks > 0);
                    tc::mma(D_U, a0, tc::desc_k(w1, kD, ks), kId64, 1);
                    tc::mma(D_U, a1, tc::desc_k(w0, kD, ks), kId64, 1);
                    tc::mma(D_O, a0, tc::desc_k(q0, kD, ks), kId64, ks > 0);
                    tc::mma(D_O, a0, tc::desc_k(q1, kD, ks), kId64, 1);
                    tc::mma(D_O, a1, tc::desc_k(q0, kD, ks), kId64, 1);
                }
                tc::commit(&s.bar_m1);
            } else {
                fail = 1;
            }
        }
        if (tc::mbar_wait(&s.bar_m1, ph)) ++n_m1; else fail = 1;
        tc::fence_after_sync();
        {
            float d[32], u[32];
            tc::tmem_ld32(D_U + lanes + hf * 32, d);
#pragma unroll
            for (int j = 0; j < 32; ++j) u[j] = Upr[j] + d[j];
#pragma unroll
            for (int j = 0; j < 32; j += 8) split8_store(&u[j], s.ut, s.ut + 128 * kC * 2, il_off(dv, hf * 32 + j, kC));
        }
        tc::fence_proxy_async();
        tc::fence_before_sync();
        __syncthreads();
        if (fail) break;

        // ---- group 2: D_O += U^T A_qk^T, D_S = U^T Kend ----
        if (tid == 0) {
            tc::fence_after_sync();
            if (c + 1 < c_end) {
                issue_wq(c + 1);  // group 1 is done with W and Qhat
                ++n_wq;
            }
            if (tc::mbar_wait(&s.bar_ka, ph)) {
                ++w_ka;
                const uint32_t u0 = tc::smem_addr(s.ut), u1 = u0 + 128 * kC * 2;
                const uint32_t k0 = tc::smem_addr(s.ka), k1 = k0 + kPlaneKT;
                const uint32_t a0q = k0 + 2 * kPlaneKT, a1q = a0q + kPlaneCC;
#pragma unroll 1
                for (int ks = 0; ks < kC / 16; ++ks) {
                    const uint64_t a0 = tc::desc_k(u0, kC, ks), a1 = tc::desc_k(u1, kC, ks);
                    tc::mma(D_O, a0, tc::desc_k(a0q, kC, ks), kId64, 1);
                    tc::mma(D_O, a0, tc::desc_k(a1q, kC, ks), kId64, 1);
                    tc::mma(D_O, a1, tc::desc_k(a0q, kC, ks), kId64, 1);
                    tc::mma(D_S, a0, tc::desc_k(k0, kC, ks), kId128, ks > 0);
                    tc::mma(D_S, a0, tc::desc_k(k1, kC, ks), kId128, 1);
                    tc::mma(D_S, a1, tc::desc_k(k0, kC, ks), kId128, 1);
                }
                tc::commit(&s.bar_m2);
            } else {
                fail = 1;
            }
        }
        if (c + 1 < c_end) load_up(c + 1);  // next chunk's U', hidden behind group 2
        if (tc::mbar_wait(&s.bar_m2, ph)) ++n_m2; else fail = 1;
        tc::fence_after_sync();
        {
            float d[32];
            tc::tmem_ld32(D_O + lanes + hf * 32, d);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int i = hf * 32 + j;
                if (i < L) {
                    const int64_t off = ((t0 + i) * H + h) * (int64_t)kD + dv;
                    if (o_f32)
                        static_cast<float *>(o)[off] = d[j];
                    else
                        static_cast<__nv_bfloat16 *>(o)[off] = __float2bfloat16_rn(d[j]);
                }
            }
        }
        {
            const float *gam = reinterpret_cast<const float *>(s.ka + 2 * kPlaneKT + 2 * kPlaneCC);
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                float d[32];
                tc::tmem_ld32(D_S + lanes + hf * 64 + part * 32, d);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int cc = part * 32 + j;
                    Sr[cc] = gam[hf * 64 + cc] * Sr[cc] + d[j];
                }
            }
        }
        store_state();
        tc::fence_proxy_async();
        tc::fence_before_sync();
        __syncthreads();
        if (fail) break;
        if (tid == 0 && c + 1 < c_end) {
            issue_ka(c + 1);  // the state update is done with Kend, A_qk and gamma
            ++n_ka;
        }
    }

    if (fail) {
        // a wait gave up: let the copies and MMAs in flight land (bounded) before the
        // shared memory and TMEM are released, and report through the status word
        if (tid == 0) {
            if (n_wq > w_wq) tc::mbar_wait(&s.bar_wq, (uint32_t)(w_wq & 1));
            if (n_ka > w_ka) tc::mbar_wait(&s.bar_ka, (uint32_t)(w_ka & 1));
            tc::mbar_wait(&s.bar_m1, (uint32_t)(n_m1 & 1));
            tc::mbar_wait(&s.bar_m2, (uint32_t)(n_m2 & 1));
            atomicExch(status, -7);
        }
#pragma unroll
        for (int j = 0; j < 64; ++j) Sr[j] = __int_as_float(0x7fc00000);
    }
#pragma unroll
    for (int j = 0; j < 64; ++j) Sout[sbase + (int64_t)(hf * 64 + j) * kD + dv] = Sr[j];

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, kWalkTmemCols);
}

// ---------------------------------------------------------------------------------
// host-side launchers (called from kda_api.cu)
// ---------------------------------------------------------------------------------
size_t intra_smem_bytes() { return sizeof(IntraSmem); }
cudaError_t launch_plan(const int32_t *cu, int32_t N, int64_t seq_len, int64_t total, int32_t *status,
                        int32_t *seq_cu, int32_t *chunk_off, cudaStream_t st) {
    kda_plan_kernel<<<1, 256, 0, st>>>(cu, N, seq_len, total, status, seq_cu, chunk_off);
    return cudaGetLastError();
}

cudaError_t launch_intra(const __nv_bfloat16 *q, const __nv_bfloat16 *k, const __nv_bfloat16 *v, const float *z,
                         const float *A, const float *b, const int32_t *status, const int32_t *seq_cu,
                         const int32_t *chunk_off, int32_t N, int32_t H, int64_t nslots, uint8_t *records,
                         cudaStream_t st) {
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kda_intra_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)sizeof(IntraSmem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    if (nslots <= 0) return cudaSuccess;
    dim3 grid((unsigned)nslots, (unsigned)H);
    kda_intra_kernel<<<grid, kIntraThreads, sizeof(IntraSmem), st>>>(q, k, v, z, A, b, status, seq_cu, chunk_off, N,
                                                                     H, records);
    return cudaGetLastError();
}

cudaError_t launch_walk(int32_t *status, const int32_t *seq_cu, const int32_t *chunk_off, int32_t N, int32_t H,
                        const uint8_t *records, const float *S0, float *Sout, void *o, int o_f32, cudaStream_t st) {
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kda_walk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)sizeof(WalkSmem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    if (N <= 0) return cudaSuccess;
    dim3 grid((unsigned)N, (unsigned)H);
    kda_walk_kernel<<<grid, kWalkThreads, sizeof(WalkSmem), st>>>(status, seq_cu, chunk_off, H, records, S0, Sout,
                                                                   o, o_f32);
    return cudaGetLastError();
}

}  // namespace kda
