// KDA chunkwise prefill: three kernels on one stream.
//
//   kda_plan_kernel   validate cu_seqlens, tabulate sequence starts and chunk offsets
//   kda_intra_kernel  one CTA per (chunk, head), all chunks in parallel: gate and
//                     cumulative decay, decayed K K^T / Q K^T per 16-token tile row,
//                     UT transform T = (I + A_kk)^-1, W = T' Khat and U' = T' V
//   kda_inter_kernel  one CTA per (sequence, head, slice of value columns): walks the
//                     chunks in order with the state slice held in registers,
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
// Every product runs on the tensor cores (mma.sync m16n8k16 bf16, fp32 accumulate)
// with both operands split into bf16 hi + lo planes (three products per tile). A plain
// bf16 operand would cost about 2^-9 of relative error per product, which the
// prediction-error cancellation in U = U' - W S amplifies beyond the accuracy the
// outputs are held to; the split keeps about 16 mantissa bits.
//
// Decay factors never overflow: for tile row a (tokens 16a..16a+15) the reference
// point is r = 16a, and exp(G_i - G_j) = exp(G_i - G_r) * exp(G_r - G_j). The first
// factor is <= 1; the second is <= 1 for j <= r and at most e^75 (15 tokens of at most
// -5 each, §5.4 of the blog) inside the diagonal tile, within bf16/fp32 range.

#include "kda_common.cuh"

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
        // write -W (split) and U' (fp32, blocks of 16 columns) to the record
        __nv_bfloat16 *Wn = reinterpret_cast<__nv_bfloat16 *>(rec + kRecWn);
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
                    *reinterpret_cast<uint32_t *>(Wn + (size_t)i * kLd128 + c) = hi;
                    *reinterpret_cast<uint32_t *>(Wn + (size_t)kC * kLd128 + (size_t)i * kLd128 + c) = lo;
                    *reinterpret_cast<float2 *>(Up + (size_t)warp * kC * 16 + i * 16 + nt * 8 + 2 * t4) =
                        make_float2(accU[a][nt][2 * hr], accU[a][nt][2 * hr + 1]);
                }
    }

    // ---- Qhat, Kend^T, A_qk, gamma (elementwise) --------------------------------
    {
        __nv_bfloat16 *Qh = reinterpret_cast<__nv_bfloat16 *>(rec + kRecQh);
        for (int e = tid; e < kC * (kD / 2); e += kIntraThreads) {
            const int i = e / (kD / 2), c = (e % (kD / 2)) * 2;
            const float2 qq = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&s.qs[i][c]));
            uint32_t hi, lo;
            split_bf16x2(qq.x * expf(s.G[i][c]), qq.y * expf(s.G[i][c + 1]), hi, lo);
            *reinterpret_cast<uint32_t *>(Qh + (size_t)i * kLd128 + c) = hi;
            *reinterpret_cast<uint32_t *>(Qh + (size_t)kC * kLd128 + (size_t)i * kLd128 + c) = lo;
        }
        __nv_bfloat16 *KeT = reinterpret_cast<__nv_bfloat16 *>(rec + kRecKeT);
        for (int e = tid; e < kD * (kC / 2); e += kIntraThreads) {
            const int c = e / (kC / 2), j = (e % (kC / 2)) * 2;
            const float k0 = __bfloat162float(s.ks[j][c]);
            const float k1 = __bfloat162float(s.ks[j + 1][c]);
            const float gl = s.G[kC - 1][c];
            uint32_t hi, lo;
            split_bf16x2(k0 * expf(gl - s.G[j][c]), k1 * expf(gl - s.G[j + 1][c]), hi, lo);
            *reinterpret_cast<uint32_t *>(KeT + (size_t)c * kLd64 + j) = hi;
            *reinterpret_cast<uint32_t *>(KeT + (size_t)kD * kLd64 + (size_t)c * kLd64 + j) = lo;
        }
        __nv_bfloat16 *Aq = reinterpret_cast<__nv_bfloat16 *>(rec + kRecAqk);
        for (int e = tid; e < kC * (kC / 2); e += kIntraThreads) {
            const int i = e / (kC / 2), j = (e % (kC / 2)) * 2;
            uint32_t hi, lo;
            split_bf16x2(s.Aqk[i][j], s.Aqk[i][j + 1], hi, lo);
            *reinterpret_cast<uint32_t *>(Aq + (size_t)i * kLd64 + j) = hi;
            *reinterpret_cast<uint32_t *>(Aq + (size_t)kC * kLd64 + (size_t)i * kLd64 + j) = lo;
        }
        float *gam = reinterpret_cast<float *>(rec + kRecGam);
        if (tid < kD) gam[tid] = expf(s.G[kC - 1][tid]);
    }
}

// ---------------------------------------------------------------------------------
// inter-chunk kernel: the serial state walk of one (sequence, head, column slice)
// ---------------------------------------------------------------------------------
template <int CW>
struct InterSmem {
    __nv_bfloat16 Wn[2][kC][kLd128];
    __nv_bfloat16 Qh[2][kC][kLd128];
    __nv_bfloat16 KeT[2][kD][kLd64];
    __nv_bfloat16 Aqk[2][kC][kLd64];
    float gam[kD];
    float Up[CW / 16][kC][16];
    __nv_bfloat16 S[2][kD][CW + 8];  // state slice, split, [key channel][value column]
    __nv_bfloat16 U[2][kC][CW + 8];  // corrected values, split, [token][value column]
};

constexpr int kInterThreads = 256;

// B fragments of NTW adjacent n8 tiles (columns n0 .. n0 + 8*NTW - 1), k rows k0 .. k0+15,
// from a tile stored [k][n] row-major.
template <int NTW>
__device__ __forceinline__ void load_b_tiles(uint32_t (&r)[NTW][2], const __nv_bfloat16 *base, int ld, int k0,
                                             int n0, int lane) {
    if constexpr (NTW == 1) {
        ldsm_x2_t(r[0][0], r[0][1], base + (size_t)(k0 + (lane & 15)) * ld + n0);
    } else {
#pragma unroll
        for (int p = 0; p < NTW / 2; ++p) {
            uint32_t t[4];
            load_b_kn(t, base, ld, k0, n0 + 16 * p, lane);
            r[2 * p][0] = t[0];
            r[2 * p][1] = t[1];
            r[2 * p + 1][0] = t[2];
            r[2 * p + 1][1] = t[3];
        }
    }
}

// Eight warps. In the 64-row products (U, O) warp w owns rows 16*(w%4) .. +15 and half of
// the slice's columns; in the state update it owns key channels 16w .. 16w+15, all columns.
// The three split-bf16 products (hi*hi, hi*lo, lo*hi) accumulate separately, so each
// dependent chain of MMAs is one product per k-step long.
template <int CW>
__global__ void __launch_bounds__(kInterThreads, 1)
    kda_inter_kernel(const int32_t *__restrict__ status, const int32_t *__restrict__ seq_cu,
                     const int32_t *__restrict__ chunk_off, int32_t H, const uint8_t *__restrict__ records,
                     const float *__restrict__ S0, float *__restrict__ Sout, void *__restrict__ o, int o_f32) {
    static_assert(CW % 16 == 0 && CW >= 16 && CW <= 64, "column slice");
    constexpr int NT = CW / 8;   // n8 tiles in the slice
    constexpr int NTW = NT / 2;  // n8 tiles per warp in the 64-row products
    extern __shared__ __align__(16) unsigned char smem_raw[];
    InterSmem<CW> &s = *reinterpret_cast<InterSmem<CW> *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t4 = lane & 3;
    const int mrow = (warp & 3) * 16;         // rows of U and O owned by this warp
    const int ncol = (warp >> 2) * NTW * 8;   // first slice column of those
    const int srow = warp * 16;               // key channels of S owned by this warp
    const int n = blockIdx.x, h = blockIdx.y, col0 = blockIdx.z * CW;
    const int64_t sbase = ((int64_t)n * H + h) * kD * kD;

    if (*status != 0) {  // invalid batch table: make the failure visible in final_state
        for (int e = tid; e < kD * CW; e += kInterThreads)
            Sout[sbase + (int64_t)(e / CW) * kD + col0 + e % CW] = __int_as_float(0x7fc00000);
        return;
    }
    const int c_begin = chunk_off[n], c_end = chunk_off[n + 1];
    const int64_t t_begin = seq_cu[n], t_end = seq_cu[n + 1];

    float Sacc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const int row = srow + g + hr * 8;
            const int col = col0 + nt * 8 + 2 * t4;
            float2 x = make_float2(0.f, 0.f);
            if (S0) x = *reinterpret_cast<const float2 *>(S0 + sbase + (int64_t)row * kD + col);
            Sacc[nt][2 * hr] = x.x;
            Sacc[nt][2 * hr + 1] = x.y;
        }

    auto rec_of = [&](int c) { return records + ((int64_t)c * H + h) * (int64_t)kRecBytes; };
    auto issue_W = [&](int c) {
        if (c < c_end) {
            const uint8_t *r = rec_of(c);
            cp_async_block(&s.Wn[0][0][0], r + kRecWn, sizeof(s.Wn), tid, kInterThreads);
            for (int bblk = 0; bblk < CW / 16; ++bblk)
                cp_async_block(&s.Up[bblk][0][0], r + kRecUp + (size_t)(col0 / 16 + bblk) * kC * 16 * 4,
                               (size_t)kC * 16 * 4, tid, kInterThreads);
        }
        cp_async_commit();
    };
    auto issue_QA = [&](int c) {
        if (c < c_end) {
            const uint8_t *r = rec_of(c);
            cp_async_block(&s.Qh[0][0][0], r + kRecQh, sizeof(s.Qh), tid, kInterThreads);
            cp_async_block(&s.Aqk[0][0][0], r + kRecAqk, sizeof(s.Aqk), tid, kInterThreads);
        }
        cp_async_commit();
    };
    auto issue_K = [&](int c) {
        if (c < c_end) {
            const uint8_t *r = rec_of(c);
            cp_async_block(&s.KeT[0][0][0], r + kRecKeT, sizeof(s.KeT), tid, kInterThreads);
            cp_async_block(&s.gam[0], r + kRecGam, sizeof(s.gam), tid, kInterThreads);
        }
        cp_async_commit();
    };
    auto store_state_split = [&]() {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int row = srow + g + hr * 8;
                const int col = nt * 8 + 2 * t4;
                uint32_t hi, lo;
                split_bf16x2(Sacc[nt][2 * hr], Sacc[nt][2 * hr + 1], hi, lo);
                *reinterpret_cast<uint32_t *>(&s.S[0][row][col]) = hi;
                *reinterpret_cast<uint32_t *>(&s.S[1][row][col]) = lo;
            }
    };

    issue_W(c_begin);
    issue_QA(c_begin);
    issue_K(c_begin);
    store_state_split();

    for (int c = c_begin; c < c_end; ++c) {
        const int64_t t0 = t_begin + (int64_t)(c - c_begin) * kC;
        const int L = (int)min((int64_t)kC, t_end - t0);

        // ---- U = U' - W S (W is stored negated) ----
        cp_async_wait<2>();
        __syncthreads();
        float ua[3][NTW][4];
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int row = mrow + g + hr * 8;
                const int col = ncol + nt * 8 + 2 * t4;
                const float2 u = *reinterpret_cast<const float2 *>(&s.Up[col >> 4][row][col & 15]);
                ua[0][nt][2 * hr] = u.x;
                ua[0][nt][2 * hr + 1] = u.y;
                ua[1][nt][2 * hr] = ua[1][nt][2 * hr + 1] = 0.f;
                ua[2][nt][2 * hr] = ua[2][nt][2 * hr + 1] = 0.f;
            }
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
            uint32_t ah[4], al[4], bh[NTW][2], bl[NTW][2];
            load_a(ah, &s.Wn[0][0][0], kLd128, mrow, ks * 16, lane);
            load_a(al, &s.Wn[1][0][0], kLd128, mrow, ks * 16, lane);
            load_b_tiles<NTW>(bh, &s.S[0][0][0], CW + 8, ks * 16, ncol, lane);
            load_b_tiles<NTW>(bl, &s.S[1][0][0], CW + 8, ks * 16, ncol, lane);
#pragma unroll
            for (int nt = 0; nt < NTW; ++nt) {
                mma_bf16(ua[0][nt], ah, bh[nt][0], bh[nt][1]);
                mma_bf16(ua[1][nt], ah, bl[nt][0], bl[nt][1]);
                mma_bf16(ua[2][nt], al, bh[nt][0], bh[nt][1]);
            }
        }
        __syncthreads();
        issue_W(c + 1);
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int row = mrow + g + hr * 8;
                const int col = ncol + nt * 8 + 2 * t4;
                uint32_t hi, lo;
                split_bf16x2(ua[0][nt][2 * hr] + (ua[1][nt][2 * hr] + ua[2][nt][2 * hr]),
                             ua[0][nt][2 * hr + 1] + (ua[1][nt][2 * hr + 1] + ua[2][nt][2 * hr + 1]), hi, lo);
                *reinterpret_cast<uint32_t *>(&s.U[0][row][col]) = hi;
                *reinterpret_cast<uint32_t *>(&s.U[1][row][col]) = lo;
            }

        // ---- O = Qhat S + A_qk U ----
        cp_async_wait<2>();
        __syncthreads();
        {
            float oa[3][NTW][4];
#pragma unroll
            for (int p = 0; p < 3; ++p)
#pragma unroll
                for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) oa[p][nt][e] = 0.f;
#pragma unroll
            for (int ks = 0; ks < kD / 16; ++ks) {
                uint32_t ah[4], al[4], bh[NTW][2], bl[NTW][2];
                load_a(ah, &s.Qh[0][0][0], kLd128, mrow, ks * 16, lane);
                load_a(al, &s.Qh[1][0][0], kLd128, mrow, ks * 16, lane);
                load_b_tiles<NTW>(bh, &s.S[0][0][0], CW + 8, ks * 16, ncol, lane);
                load_b_tiles<NTW>(bl, &s.S[1][0][0], CW + 8, ks * 16, ncol, lane);
#pragma unroll
                for (int nt = 0; nt < NTW; ++nt) {
                    mma_bf16(oa[0][nt], ah, bh[nt][0], bh[nt][1]);
                    mma_bf16(oa[1][nt], ah, bl[nt][0], bl[nt][1]);
                    mma_bf16(oa[2][nt], al, bh[nt][0], bh[nt][1]);
                }
            }
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks) {
                if (ks > (warp & 3)) break;  // A_qk is lower triangular
                uint32_t ah[4], al[4], bh[NTW][2], bl[NTW][2];
                load_a(ah, &s.Aqk[0][0][0], kLd64, mrow, ks * 16, lane);
                load_a(al, &s.Aqk[1][0][0], kLd64, mrow, ks * 16, lane);
                load_b_tiles<NTW>(bh, &s.U[0][0][0], CW + 8, ks * 16, ncol, lane);
                load_b_tiles<NTW>(bl, &s.U[1][0][0], CW + 8, ks * 16, ncol, lane);
#pragma unroll
                for (int nt = 0; nt < NTW; ++nt) {
                    mma_bf16(oa[0][nt], ah, bh[nt][0], bh[nt][1]);
                    mma_bf16(oa[1][nt], ah, bl[nt][0], bl[nt][1]);
                    mma_bf16(oa[2][nt], al, bh[nt][0], bh[nt][1]);
                }
            }
#pragma unroll
            for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int row = mrow + g + hr * 8;
                    if (row < L) {
                        const float o0 = oa[0][nt][2 * hr] + (oa[1][nt][2 * hr] + oa[2][nt][2 * hr]);
                        const float o1 = oa[0][nt][2 * hr + 1] + (oa[1][nt][2 * hr + 1] + oa[2][nt][2 * hr + 1]);
                        const int64_t off = ((t0 + row) * H + h) * (int64_t)kD + col0 + ncol + nt * 8 + 2 * t4;
                        if (o_f32)
                            *reinterpret_cast<float2 *>(static_cast<float *>(o) + off) = make_float2(o0, o1);
                        else
                            *reinterpret_cast<__nv_bfloat162 *>(static_cast<__nv_bfloat16 *>(o) + off) =
                                __floats2bfloat162_rn(o0, o1);
                    }
                }
        }
        __syncthreads();
        issue_QA(c + 1);

        // ---- S = Diag(gamma) S + Kend^T U ----
        cp_async_wait<2>();
        __syncthreads();
        {
            float sx[NT][4];
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const float gm = s.gam[srow + g + hr * 8];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    Sacc[nt][2 * hr] *= gm;
                    Sacc[nt][2 * hr + 1] *= gm;
                    sx[nt][2 * hr] = sx[nt][2 * hr + 1] = 0.f;
                }
            }
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks) {
                uint32_t ah[4], al[4], bh[NT][2], bl[NT][2];
                load_a(ah, &s.KeT[0][0][0], kLd64, srow, ks * 16, lane);
                load_a(al, &s.KeT[1][0][0], kLd64, srow, ks * 16, lane);
                load_b_tiles<NT>(bh, &s.U[0][0][0], CW + 8, ks * 16, 0, lane);
                load_b_tiles<NT>(bl, &s.U[1][0][0], CW + 8, ks * 16, 0, lane);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    mma_bf16(sx[nt], ah, bl[nt][0], bl[nt][1]);
                    mma_bf16(sx[nt], al, bh[nt][0], bh[nt][1]);
                    mma_bf16(Sacc[nt], ah, bh[nt][0], bh[nt][1]);
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) Sacc[nt][e] += sx[nt][e];
        }
        __syncthreads();
        issue_K(c + 1);
        store_state_split();
    }
    cp_async_wait<0>();

#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const int row = srow + g + hr * 8;
            const int col = col0 + nt * 8 + 2 * t4;
            *reinterpret_cast<float2 *>(Sout + sbase + (int64_t)row * kD + col) =
                make_float2(Sacc[nt][2 * hr], Sacc[nt][2 * hr + 1]);
        }
}

// ---------------------------------------------------------------------------------
// host-side launchers (called from kda_api.cu)
// ---------------------------------------------------------------------------------
size_t intra_smem_bytes() { return sizeof(IntraSmem); }
template <int CW>
size_t inter_smem_bytes() {
    return sizeof(InterSmem<CW>);
}

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

template <int CW>
static cudaError_t launch_inter_cw(const int32_t *status, const int32_t *seq_cu, const int32_t *chunk_off,
                                   int32_t N, int32_t H, const uint8_t *records, const float *S0, float *Sout,
                                   void *o, int o_f32, cudaStream_t st) {
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kda_inter_kernel<CW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)sizeof(InterSmem<CW>));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    dim3 grid((unsigned)N, (unsigned)H, (unsigned)(kD / CW));
    kda_inter_kernel<CW><<<grid, kInterThreads, sizeof(InterSmem<CW>), st>>>(status, seq_cu, chunk_off, H, records,
                                                                            S0, Sout, o, o_f32);
    return cudaGetLastError();
}

cudaError_t launch_inter(int cw, const int32_t *status, const int32_t *seq_cu, const int32_t *chunk_off, int32_t N,
                         int32_t H, const uint8_t *records, const float *S0, float *Sout, void *o, int o_f32,
                         cudaStream_t st) {
    if (N <= 0) return cudaSuccess;
    switch (cw) {
        case 16: return launch_inter_cw<16>(status, seq_cu, chunk_off, N, H, records, S0, Sout, o, o_f32, st);
        case 32: return launch_inter_cw<32>(status, seq_cu, chunk_off, N, H, records, S0, Sout, o, o_f32, st);
        default: return launch_inter_cw<64>(status, seq_cu, chunk_off, N, H, records, S0, Sout, o, o_f32, st);
    }
}

}  // namespace kda
