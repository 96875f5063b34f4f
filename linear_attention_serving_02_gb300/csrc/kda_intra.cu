// KDA chunkwise prefill, intra-chunk part: every (chunk, head) item is independent of the
// state, so one persistent CTA per SM walks items b, b + grid, ... and writes, per item,
// the chunk record the state walk reads (layout in kda_common.cuh). Per item, on the
// tcgen05 tensor cores with TMEM accumulators:
//
//   gate        log a = g_min sigmoid(e^A z), beta = sigmoid(b), G = running sum of log a
//   Gram        A_kk[i,j] = beta_i sum_c k_i k_j e^(G_i - G_j)   (j <  i)
//               A_qk[i,j] =        sum_c q_i k_j e^(G_i - G_j)   (j <= i)
//   UT          T = (I + A_kk)^-1 (forward substitution, fp32), T' = T Diag(beta)
//   W, U'       [W | U'] = T' [Khat | V],  Khat = k * e^G
//
// ('From Linear Attention to KDA', §7.2-7.3 for the chunk algebra with the per-channel
// decay, §8 for tiles with the decay factored around a reference token inside them.)
//
// Decay factors. A product e^(G_i - G_j) is taken as (x_i e^(G_i - G_r)) . (k_j e^(G_r - G_j))
// around a reference token r. Where j < r <= i both factors are at most 1, so a factor
// that underflows belongs to a product that is smaller still. Where i and j lie on the
// same side of r, one factor may exceed 1, but only over the at most 16 tokens between r
// and that token (log a >= -5 per token, the page's §5.4): e^80 at most, and the other
// factor is then at least e^-80, inside the fp32 and bf16 range. So the 64-token chunk
// is cut into two 32-token halves: inside each half the reference is its middle token
// (16 or 48), and the off-diagonal block (i in the upper half, j in the lower one) uses
// r = 32. All three blocks come out of one MMA chain:
//
//   A (TMEM, M = 128 rows, K = 128 channels): key versions
//       rows  0..31  k_j e^(G_16 - G_j), j = 0..31
//       rows 32..63  k_j e^(G_48 - G_j), j = 32..63
//       rows 64..95  k_j e^(G_32 - G_j), j = 0..31          (rows 96..127 unused)
//   B (shared memory, N = 192 rows, K-major): row versions
//       n   0..31 q_i e^(G_i - G_16), i = 0..31   n  96..127 the same with k_i
//       n  32..63 q_i e^(G_i - G_48), i = 32..63  n 128..159 the same with k_i
//       n  64..95 q_i e^(G_i - G_32), i = 32..63  n 160..191 the same with k_i
//   D[m][n] (TMEM lanes m, columns n): the useful blocks are the diagonal ones of each
//   32-lane quarter; the others mix references and are never read (they may overflow).
//
// G is kept in units of log2 (G log2(e)), so every factor e^(G_x - G_y) is one 2^x on the
// special-function unit.
//
// Precision. Every product that the outputs are held to splits its operands into bf16
// hi + lo planes (hi*hi + hi*lo + lo*hi, about 16 bits). Two operands take one bf16
// plane: the k rows of A_kk and Khat in W. An emulation of this algorithm in fp64 with
// each operand rounded as here puts their rounding at about a sixth of the output
// tolerance on the 8192-token workload, where plain bf16 on the q rows, the key
// versions or T' would exceed it.
//
// Schedule of one item (16 warps):
//   all        Gram operands (A into TMEM, B into shared memory); MMA chain issued
//   all        Khat (the [W | U'] operand), Qhat, Kend^T, gamma (record), while the chain runs
//   12 warps   A_qk -> record, A_kk -> shared memory
//   warps 0-1  the UT solve's diagonal blocks (one column per thread) while the others
//              request the z of the item after next; then all warps the solve's other blocks
//   all        T' split; [W | U'] chain issued; while it runs, the next item's q and k
//              are requested and its gate computed
//   all        -W and U' staged in shared memory, two bulk stores
// Inputs arrive by cp.async; every thread arrives once per load on that load's mbarrier
// (count 512), so any warp can wait for a whole tile.

#include <algorithm>

#include "kda_common.cuh"
#include "kda_f32x2.cuh"
#include "kda_tc.cuh"

namespace kda {

namespace {

constexpr int kIntraThreads = 512;
constexpr int kLdG = kD + 4;    // G row stride (floats): 528 bytes, so rows start 4 banks apart
constexpr int kLdQK = kD + 8;   // q, k row stride (bf16): 272 bytes, likewise
constexpr float kLog2e = 1.4426950408889634f;  // log2(e): e^x = 2^(x log2(e))

struct Item {
    int slot, h;
    int64_t t0;
    int L;
};

struct IntraSmem {
    float G[2][kC * kLdG];  // z, then (in place) G log2(e); the other buffer is the next item's
    __nv_bfloat16 q[kC * kLdQK];  // q and k of the item (rows past the sequence end are zero)
    __nv_bfloat16 k[kC * kLdQK];
    alignas(1024) unsigned char kv[2 * kPlaneQK];  // B of [W | U'] = T' [Khat | V]: MN-major,
                                                   // N = 256 (Khat, then V channels), K = 64
    union {
        struct {  // B of the Gram chain (row versions), K-major, 8-channel groups outermost
            alignas(1024) unsigned char hi[192 * 256];
            alignas(1024) unsigned char lo[96 * 256];  // q rows only
        } g;
        struct {  // after the Gram chain has completed
            float Akk[kC][kC + 4];  // rows 16-byte aligned; the pad spreads rows over banks
            float T[kC][kC + 4];
            float X[2][kTile][kTile + 4];     // products of the solve's doubling steps (rows
            float Y[2 * kTile][2 * kTile + 4];  // 16-byte aligned for float4 access)
            alignas(1024) unsigned char tp[2][kC * kC * 2];  // A of [W | U']: T' hi and lo, K-major
        } s;
        struct {  // after the [W | U'] chain has completed: the record's -W and U'
            alignas(1024) unsigned char w[kPlaneQK];
            alignas(1024) float up[kC * kD];
        } e;
    } u;
    float beta[2][kC];
    Item nxt2;  // the item after next, looked up by an idle thread during the Gram operands
    uint64_t bar_z[2], bar_qk, bar_v, bar_gram, bar_wu;
    uint32_t tmem_base;
    int fail;
};

__device__ __forceinline__ const float *grow(const float *G, int i) { return G + i * kLdG; }
__device__ __forceinline__ void g_load8(const float *G, int i, int c, float (&x)[8]) {
    const float4 a = *reinterpret_cast<const float4 *>(grow(G, i) + c);
    const float4 b = *reinterpret_cast<const float4 *>(grow(G, i) + c + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ uint4 ld_unit(const __nv_bfloat16 *buf, int i, int c) {
    return *reinterpret_cast<const uint4 *>(buf + i * kLdQK + c);
}
// bf16 pair of (x0 f0, x1 f1), rounded to nearest
__device__ __forceinline__ uint32_t scale_bf16(uint32_t xbf2, float f0, float f1) {
    const float2 x = bf16x2_to_float2(xbf2);
    const float2 y = upk2(mul2(pk2(x.x, x.y), pk2(f0, f1)));
    return pack_bf16x2(__floats2bfloat162_rn(y.x, y.y));
}
// position of the 16-byte unit u (4 channels) of U' row i in the record: XOR-swizzled by
// i % 32, so that the 16 rows a warp stages at once fall on distinct banks
__device__ __forceinline__ int up_unit(int i, int u) { return u ^ (i & 31); }

// bounded mbarrier wait; a wait that gives up marks the CTA failed (reported at the end)
__device__ __forceinline__ bool intra_wait(uint64_t *bar, uint32_t parity, volatile int &fail, int32_t *) {
    if (fail) return false;  // after a failure nothing waits again: the kernel only runs out
    if (tc::mbar_wait(bar, parity)) return true;
    fail = 1;
    return false;
}

}  // namespace

__global__ void __launch_bounds__(kIntraThreads, 1)
    kda_intra_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                     const __nv_bfloat16 *__restrict__ v, const float *__restrict__ z, const float *__restrict__ A,
                     const float *__restrict__ bgate, int32_t *__restrict__ status,
                     const int32_t *__restrict__ seq_cu, const int32_t *__restrict__ chunk_off, int32_t N, int32_t H,
                     int64_t dense_len, uint8_t *__restrict__ records, int32_t item_lo, int32_t item_hi) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    IntraSmem &s = *reinterpret_cast<IntraSmem *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // N sequences of dense_len tokens each (dense_len > 0, no cu_seqlens): the sequence
    // tables are closed forms, so nothing here waits for the plan kernel before the end
    // (it writes only the walk's tables and a status of 0); every CTA waits for it before it
    // exits, which keeps its tables complete for the walk that waits for this kernel.
    const bool dense = dense_len > 0;
    const int cps = dense ? (int)((dense_len + kC - 1) / kC) : 0;  // chunks per sequence
    if (!dense) pdl_wait();
    pdl_trigger();
    if ((!dense && *status != 0) || N <= 0) {
        if (dense) pdl_wait();
        return;
    }
    // persistent: CTA b takes items lo + b, lo + b + gridDim.x, ... below hi, where [lo, hi)
    // is this launch's share of the items (item = slot * H + h)
    const int n_all = (dense ? N * cps : chunk_off[N]) * H;
    const int lo = min(item_lo, n_all), n_items = min(item_hi, n_all);
    if ((int)blockIdx.x >= n_items - lo) {
        if (dense) pdl_wait();
        return;
    }
    const int64_t rowstride = (int64_t)H * kD;  // elements between consecutive tokens

    if (warp == 0) {
        if (lane == 0) {
            tc::mbar_init(&s.bar_z[0], kIntraThreads);
            tc::mbar_init(&s.bar_z[1], kIntraThreads);
            tc::mbar_init(&s.bar_qk, kIntraThreads);
            tc::mbar_init(&s.bar_v, kIntraThreads);
            tc::mbar_init(&s.bar_gram, 1);
            tc::mbar_init(&s.bar_wu, 1);
            tc::mbar_init_fence();
            s.fail = 0;
        }
        __syncwarp();
        tc::tmem_alloc(&s.tmem_base, 512);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s.tmem_base;
    const uint32_t lanes = (uint32_t)((warp & 3) * 32) << 16;  // this warp's TMEM lane quarter
    // TMEM columns: [0, 128) the Gram's A operand (hi 0..63, lo 64..127), later [0, 256)
    // the [W | U'] accumulator (M = 64); [256, 448) the Gram accumulator (N = 192)
    const uint32_t D_W = tmem, D_G = tmem + 256;
    volatile int &fail = s.fail;

    auto item_of = [&](int it) {
        Item r;
        r.slot = it / H;
        r.h = it % H;
        if (dense) {
            const int n = r.slot / cps, ci = r.slot - n * cps;
            r.t0 = (int64_t)n * dense_len + (int64_t)ci * kC;
            r.L = (int)min((int64_t)kC, dense_len - (int64_t)ci * kC);
            return r;
        }
        const int n = find_seq(chunk_off, N, r.slot);
        r.t0 = (int64_t)seq_cu[n] + (int64_t)(r.slot - chunk_off[n]) * kC;
        r.L = (int)min((int64_t)kC, (int64_t)seq_cu[n + 1] - r.t0);
        return r;
    };
    // z of an item into G buffer b, q and k, v: every thread copies its 16-byte units with
    // cp.async and arrives on the load's mbarrier when they have landed. Rows of z past the
    // sequence end are not copied (the gate ignores them); those of q, k, v are zeroed.
    auto stage_z = [&](const Item &it, int b, int t0 = 0, int nt = kIntraThreads) {
#pragma unroll 4
        for (int e = tid - t0; e >= 0 && e < it.L * (kD / 4); e += nt) {
            const int i = e / (kD / 4), c = (e % (kD / 4)) * 4;
            cp_async16(s.G[b] + i * kLdG + c, z + (it.t0 + i) * rowstride + (int64_t)it.h * kD + c);
        }
        cp_async_arrive(&s.bar_z[b]);
    };
    auto stage_qk = [&](const Item &it) {
#pragma unroll 4
        for (int e = tid; e < 2 * kC * (kD / 8); e += kIntraThreads) {
            // 16 consecutive units of one row of q, then of k: q and k lie a multiple of 128
            // bytes apart, so alternating them per unit put two lanes on each bank group
            const int which = (e >> 4) & 1, i = e >> 5, c = (e & 15) * 8;
            __nv_bfloat16 *dst = (which ? s.k : s.q) + i * kLdQK + c;
            if (i < it.L)
                cp_async16(dst, (which ? k : q) + (it.t0 + i) * rowstride + (int64_t)it.h * kD + c);
            else
                *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
        cp_async_arrive(&s.bar_qk);
    };
    // v goes straight into the V half of the [Khat | V] operand (MN-major: the 16 bytes of
    // token j, channels 8 c8 .. 8 c8 + 7 are one core-matrix row)
    auto stage_v = [&](const Item &it) {
#pragma unroll 4
        for (int e = tid; e < kC * (kD / 8); e += kIntraThreads) {
            const int j = e & (kC - 1), c8 = e >> 6;  // consecutive threads: consecutive tokens
            unsigned char *dst = s.kv + ak_off(kD + 8 * c8, j);
            if (j < it.L)
                cp_async16(dst, v + (it.t0 + j) * rowstride + (int64_t)it.h * kD + c8 * 8);
            else
                *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
        cp_async_arrive(&s.bar_v);
    };
    // Gate of item it in G buffer b, beta into beta[b], by all 512 threads: thread (channel
    // quad cq, row quad ro) takes rows 4 ro .. 4 ro + 3 of channels 4 cq .. 4 cq + 3;
    // log a = g_min sigmoid(e^A z) (z = +inf gives -5), a running sum along its rows, and
    // the quads' totals scanned over the 16 lanes of the channel quad by shuffles. Stored
    // as G log2(e). The division is __fdividef: an infinite denominator (z = -inf) gives
    // 0, i.e. a = 1 exactly. pre holds the thread's b value (threads below it.L) and A_h,
    // loaded ahead of time by gate_inputs.
    auto gate = [&](const Item &it, int b, int par, float2 pre) {
        const float bv = pre.x, eA = expf(pre.y);
        intra_wait(&s.bar_z[b], (uint32_t)par, fail, status);
        float *Gb = s.G[b];
        // lane = 2 ro + (cq % 2): the 8 lanes of a shared-memory phase take 4 row quads of 2
        // channel quads, 4 distinct bank groups (row quads 4 rows apart share two)
        const int ro = lane >> 1, cq = 2 * warp + (lane & 1), r0 = 4 * ro, c0 = 4 * cq;
        const uint64_t mA = pk2(-eA * kLog2e, -eA * kLog2e), one = pk2(1.f, 1.f);
        uint64_t g[4][2];  // rows r0 + m, channel pairs (c0, c0 + 1), (c0 + 2, c0 + 3)
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float4 x = *reinterpret_cast<const float4 *>(Gb + (r0 + m) * kLdG + c0);
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                const float2 t = upk2(mul2(mA, p ? pk2(x.z, x.w) : pk2(x.x, x.y)));
                const float2 d = upk2(add2(one, pk2(tc::ex2(t.x), tc::ex2(t.y))));
                uint64_t la = pk2(__fdividef(kGMin, d.x), __fdividef(kGMin, d.y));
                if (r0 + m >= it.L) la = pk2(0.f, 0.f);  // rows past the end add nothing
                g[m][p] = m ? add2(g[m - 1][p], la) : la;
            }
        }
        // exclusive prefix of the quad totals over ro (the 16 lanes with the same cq, every
        // second lane)
        float tot[4];
        {
            const float2 x0 = upk2(g[3][0]), x1 = upk2(g[3][1]);
            tot[0] = x0.x; tot[1] = x0.y; tot[2] = x1.x; tot[3] = x1.y;
        }
        float inc[4] = {tot[0], tot[1], tot[2], tot[3]};
#pragma unroll
        for (int d = 1; d < 16; d <<= 1) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float y = __shfl_up_sync(0xffffffffu, inc[c], 2 * d);  // row quad ro - d
                if (ro >= d) inc[c] += y;
            }
        }
        const uint64_t pre0 = pk2(inc[0] - tot[0], inc[1] - tot[1]), pre1 = pk2(inc[2] - tot[2], inc[3] - tot[3]);
        const uint64_t l2e = pk2(kLog2e, kLog2e);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float2 x0 = upk2(mul2(add2(g[m][0], pre0), l2e)), x1 = upk2(mul2(add2(g[m][1], pre1), l2e));
            *reinterpret_cast<float4 *>(Gb + (r0 + m) * kLdG + c0) = make_float4(x0.x, x0.y, x1.x, x1.y);
        }
        if (tid < kC) s.beta[b][tid] = (tid < it.L) ? sigmoid_f(bv) : 0.f;
    };
    auto gate_inputs = [&](const Item &it) {
        return make_float2(tid < it.L ? bgate[(it.t0 + tid) * H + it.h] : 0.f, A[it.h]);
    };

    // ---- prologue: the first item's inputs and gate, the second item's z ---------------
    int item = lo + (int)blockIdx.x, iters = 0;
    Item cur = item_of(item);
    Item nxt = item + (int)gridDim.x < n_items ? item_of(item + gridDim.x) : cur;
    stage_z(cur, 0);
    if (item + (int)gridDim.x < n_items) stage_z(nxt, 1);
    stage_qk(cur);
    stage_v(cur);
    gate(cur, 0, 0, gate_inputs(cur));
    __syncthreads();

    for (; item < n_items; ++iters, item += gridDim.x) {
        const int b = iters & 1;
        const float *G = s.G[b];
        const int h = cur.h;
        uint8_t *rec = records + ((int64_t)cur.slot * H + h) * (int64_t)kRecBytes;
        const bool has_next = item + (int)gridDim.x < n_items;
        const bool has_next2 = item + 2 * (int)gridDim.x < n_items;
        const uint32_t ph = (uint32_t)(iters & 1);

        intra_wait(&s.bar_qk, ph, fail, status);  // this item's q and k have landed
        tc::fence_after_sync();

        // ---- Gram operands ---------------------------------------------------------------
        // A (key versions) into TMEM by the warps of lane quarters 0..2: warp w writes the
        // 32 rows of quarter w % 4, channels 32 (w / 4) .. +31, as split bf16 pairs (a
        // 32-bit TMEM column holds channels 2 col, 2 col + 1)
        if ((warp & 3) != 3) {
            const int qd = warp & 3, c0 = 32 * (warp >> 2);
            const int j = (qd == 1) ? 32 + lane : lane;
            const int ref = (qd == 0) ? 16 : (qd == 1 ? 48 : 32);
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c = c0 + 8 * u;
                float gj[8], gr[8];
                g_load8(G, j, c, gj);
                g_load8(G, ref, c, gr);
                const uint4 kr = ld_unit(s.k, j, c);
                const uint32_t kw[4] = {kr.x, kr.y, kr.z, kr.w};
#pragma unroll
                for (int p2 = 0; p2 < 4; ++p2)
                    scale_split_pk(kw[p2], tc::ex2(gr[2 * p2] - gj[2 * p2]), tc::ex2(gr[2 * p2 + 1] - gj[2 * p2 + 1]),
                                   hi[4 * u + p2], lo[4 * u + p2]);
            }
            tc::tmem_st16(tmem + lanes + (uint32_t)(c0 >> 1), hi);
            tc::tmem_st16(tmem + lanes + 64u + (uint32_t)(c0 >> 1), lo);
            tc::tmem_wait_st();
        } else if (warp == kIntraThreads / 32 - 1 && lane == 0 && has_next2) {
            s.nxt2 = item_of(item + 2 * gridDim.x);  // its dependent loads, off every other warp
        }
        // B (row versions) into shared memory by every thread: job (c8, nq) makes 8
        // channels of the q row version nq (split) and of the matching k row (hi only),
        // which share their factors. Consecutive threads take consecutive rows.
        if (tid == 0) tc::bulk_wait_read0();  // the last item's staged -W and U' have been read
        __syncthreads();
#pragma unroll
        for (int job = tid; job < 96 * (kD / 8); job += kIntraThreads) {
            const int c8 = job / 96, nq = job % 96;
            const int i = (nq < 64) ? nq : nq - 32;
            const int ref = (nq < 32) ? 16 : (nq < 64 ? 48 : 32);
            float gi[8], gr[8];
            g_load8(G, i, 8 * c8, gi);
            g_load8(G, ref, 8 * c8, gr);
            float f[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) f[m] = tc::ex2(gi[m] - gr[m]);
            const uint4 qr = ld_unit(s.q, i, 8 * c8), kr = ld_unit(s.k, i, 8 * c8);
            const uint32_t qw[4] = {qr.x, qr.y, qr.z, qr.w}, kw[4] = {kr.x, kr.y, kr.z, kr.w};
            uint32_t qh[4], ql[4], kh[4];
#pragma unroll
            for (int p2 = 0; p2 < 4; ++p2) {
                scale_split_pk(qw[p2], f[2 * p2], f[2 * p2 + 1], qh[p2], ql[p2]);
                kh[p2] = scale_bf16(kw[p2], f[2 * p2], f[2 * p2 + 1]);
            }
            *reinterpret_cast<uint4 *>(s.u.g.hi + c8 * 3072 + nq * 16) = make_uint4(qh[0], qh[1], qh[2], qh[3]);
            *reinterpret_cast<uint4 *>(s.u.g.hi + c8 * 3072 + (96 + nq) * 16) = make_uint4(kh[0], kh[1], kh[2], kh[3]);
            *reinterpret_cast<uint4 *>(s.u.g.lo + c8 * 1536 + nq * 16) = make_uint4(ql[0], ql[1], ql[2], ql[3]);
        }
        fence_proxy_async();  // the generic-proxy writes above are read by the tensor core
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            // 8 k-steps of 16 channels: A hi x B hi and A lo x B hi (N = 192), A hi x B lo on
            // the q rows (N = 96, the first 96 columns); unrolled, as issuing MMAs from one
            // thread in a loop cost ~90 cycles each
            tc::fence_after_sync();
            if (!fail) {
                const uint32_t idG = tc::idesc_bf16(128, 192, 0), idQ = tc::idesc_bf16(128, 96, 0);
                const uint32_t bh = tc::smem_addr(s.u.g.hi), bl = tc::smem_addr(s.u.g.lo);
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks) {
                    const uint64_t dh = tc::desc(bh + (uint32_t)ks * 6144u, 3072u, 128u);
                    const uint64_t dl = tc::desc(bl + (uint32_t)ks * 3072u, 1536u, 128u);
                    tc::mma_ts(D_G, tmem + 8u * ks, dh, idG, ks > 0);
                    tc::mma_ts(D_G, tmem + 64u + 8u * ks, dh, idG, 1);
                    tc::mma_ts(D_G, tmem + 8u * ks, dl, idQ, 1);
                }
            }
            tc::commit(&s.bar_gram);
        }

        const Item nxt2 = has_next2 ? s.nxt2 : nxt;  // the item after next

        // ---- while the Gram chain runs: Khat (the [W | U'] operand), Qhat and Kend^T (the
        // ---- record); Khat and Qhat share 2^(G_j log2 e). Job (c8, j): token j, 8 channels.
        // ---- Warp 0 issued the chain: its jobs go to warps 3 and 7, which read no Gram results.
        auto khat_job = [&](int job) {
            const int j = job & (kC - 1), c = 8 * (job >> 6);
            float gj[8], gl[8];
            g_load8(G, j, c, gj);
            g_load8(G, kC - 1, c, gl);
            float e[8], f[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                e[m] = tc::ex2(gj[m]);          // Khat, Qhat: e^(G_j)
                f[m] = tc::ex2(gl[m] - gj[m]);  // Kend: e^(G_last - G_j)
            }
            const uint4 qr = ld_unit(s.q, j, c), kr = ld_unit(s.k, j, c);
            const uint32_t qw[4] = {qr.x, qr.y, qr.z, qr.w}, kw[4] = {kr.x, kr.y, kr.z, kr.w};
            uint32_t kh[4], qh[4], ql[4], eh[4], el[4];
#pragma unroll
            for (int p2 = 0; p2 < 4; ++p2) {
                kh[p2] = scale_bf16(kw[p2], e[2 * p2], e[2 * p2 + 1]);
                scale_split_pk(qw[p2], e[2 * p2], e[2 * p2 + 1], qh[p2], ql[p2]);
                scale_split_pk(kw[p2], f[2 * p2], f[2 * p2 + 1], eh[p2], el[p2]);
            }
            *reinterpret_cast<uint4 *>(s.kv + ak_off(c, j)) = make_uint4(kh[0], kh[1], kh[2], kh[3]);
            // record stores stream past L2 (st.global.cs): the walk reads them only later
            __stcs(reinterpret_cast<uint4 *>(rec + kRecQh + il_off(j, c, kD)), make_uint4(qh[0], qh[1], qh[2], qh[3]));
            __stcs(reinterpret_cast<uint4 *>(rec + kRecQl + il_off(j, c, kD)), make_uint4(ql[0], ql[1], ql[2], ql[3]));
            __stcs(reinterpret_cast<uint4 *>(rec + kRecAK + ak_off(kC + c, j)), make_uint4(eh[0], eh[1], eh[2], eh[3]));
            __stcs(reinterpret_cast<uint4 *>(rec + kRecAK + kStackAK + ak_off(kC + c, j)),
                   make_uint4(el[0], el[1], el[2], el[3]));
        };
        static_assert(kC * (kD / 8) == 2 * kIntraThreads, "two Khat jobs per thread");
        if (warp != 0) {
            khat_job(tid);
            khat_job(tid + kIntraThreads);
        }
        if (warp == 3) khat_job(tid - 96);                  // jobs 0 .. 31
        if (warp == 7) khat_job(kIntraThreads + tid - 224);  // jobs 512 .. 543
        if (tid >= 128 && tid < 128 + kD)
            reinterpret_cast<float *>(rec + kRecGam)[tid - 128] = tc::ex2(grow(G, kC - 1)[tid - 128]);

        // ---- the Gram results: A_qk to the record, A_kk (times beta) to shared memory ----
        // Warp w of lane quarter qd = w % 4 < 3 reads 8 query columns 8 (w / 4) .. of its
        // block for its lane's key j.
        if ((warp & 3) != 3) {
            intra_wait(&s.bar_gram, ph, fail, status);
            tc::fence_after_sync();
            const int qd = warp & 3, cq = warp >> 2;
            const int j = (qd == 1) ? 32 + lane : lane;
            const int ib = ((qd == 0) ? 0 : 32) + 8 * cq;  // first of this thread's 8 query rows
            uint32_t dq[8], dk[8];
            tc::tmem_ld8_nowait(D_G + lanes + (uint32_t)(32 * qd + 8 * cq), dq);
            tc::tmem_ld8_nowait(D_G + lanes + (uint32_t)(96 + 32 * qd + 8 * cq), dk);
            tc::tmem_wait_ld();
            const bool diag = qd != 2;
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int p2 = 0; p2 < 4; ++p2) {
                const int i0 = ib + 2 * p2;
                const float a0 = (!diag || j <= i0) ? __uint_as_float(dq[2 * p2]) : 0.f;
                const float a1 = (!diag || j <= i0 + 1) ? __uint_as_float(dq[2 * p2 + 1]) : 0.f;
                split_pk(pk2(a0, a1), hi[p2], lo[p2]);
            }
            // 8 consecutive query rows of key j: one MN-major 16-byte unit per plane (none in
            // the blocks wholly above the diagonal, which the record leaves out)
            if (!aqk_zero_block(ib, j)) {
                __stcs(reinterpret_cast<uint4 *>(rec + kRecAqk + ak_off(ib, j)),
                       make_uint4(hi[0], hi[1], hi[2], hi[3]));
                __stcs(reinterpret_cast<uint4 *>(rec + kRecAqk + kStackAK + ak_off(ib, j)),
                       make_uint4(lo[0], lo[1], lo[2], lo[3]));
            }
            const float *be = s.beta[b];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const int i = ib + t;
                s.u.s.Akk[i][j] = (!diag || j < i) ? be[i] * __uint_as_float(dk[t]) : 0.f;
            }
        }
        // (the A_qk block above the diagonal, i < 32 <= j, is zero: the record leaves it out)
        tc::fence_before_sync();
        __syncthreads();
        const float2 pre = has_next ? gate_inputs(nxt) : make_float2(0.f, 0.f);

        // ---- UT transform: T = (I + A_kk)^-1, unit lower triangular ---------------------
        // The diagonal 16 x 16 blocks on warps 0-1, thread (block a, column j) solving
        // (I + A_aa) t = e_j by forward substitution: t_i = [i = j] - sum_{m < i} A[i][m] t_m,
        // each row of A_aa read with float4 broadcasts (the 16 threads of a block read the
        // same row). Every row's sum can start as soon as its first terms are known, so the
        // dependent chain is about one FMA per row. The other warps zero the blocks above
        // the diagonal.
        if (warp < 2) {
            const int base = (tid >> 4) * kTile, j = tid & 15;
            float t[kTile];
#pragma unroll
            for (int i = 0; i < kTile; ++i) {
                float acc = 0.f;
#pragma unroll
                for (int m4 = 0; m4 < i; m4 += 4) {
                    const float4 av = *reinterpret_cast<const float4 *>(&s.u.s.Akk[base + i][base + m4]);
                    const float am[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        if (m4 + u < i) acc = __fmaf_rn(am[u], t[m4 + u], acc);
                }
                t[i] = ((i == j) ? 1.f : 0.f) - acc;
            }
#pragma unroll
            for (int i = 0; i < kTile; ++i) s.u.s.T[base + i][base + j] = t[i];
        } else {
            for (int e = tid - 64; e < kC * kC; e += kIntraThreads - 64) {
                const int i = e / kC, j = e % kC;
                if ((j >> 4) > (i >> 4)) s.u.s.T[i][j] = 0.f;
            }
            // this item's G is read no more: the z of the item after next is requested into
            // its buffer by these warps while warps 0-1 solve (every thread still arrives on
            // the load's mbarrier)
            if (has_next2) stage_z(nxt2, b, 64, kIntraThreads - 64);
        }
        if (warp < 2 && has_next2) cp_async_arrive(&s.bar_z[b]);
        __syncthreads();
        // The blocks below the diagonal by doubling, the sums in k order:
        //   16 -> 32:  T_10 = -T_11 (A_10 T_00),  T_32 = -T_33 (A_32 T_22)
        //   32 -> 64:  T[32:64, 0:32] = -T[32:64, 32:64] (A[32:64, 0:32] T[0:32, 0:32])
        // (the inverse of a block lower triangular matrix, one halving of the block size at a
        // time: four dependent products instead of the six of a block-by-block solve). Each
        // thread makes 4 consecutive columns of one row with float4 loads; a warp spans a
        // few rows and all column quads, so its loads are broadcasts or one 128-byte row.
        auto dot4 = [&](const float *arow, const float *bmat, int ldb, int k0, int k1, float4 &acc) {
#pragma unroll 4
            for (int k = k0; k < k1; k += 4) {
                const float4 av = *reinterpret_cast<const float4 *>(arow + k);
                const float am[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float4 bv = *reinterpret_cast<const float4 *>(bmat + (k + u) * ldb);
                    acc.x = __fmaf_rn(am[u], bv.x, acc.x);
                    acc.y = __fmaf_rn(am[u], bv.y, acc.y);
                    acc.z = __fmaf_rn(am[u], bv.z, acc.z);
                    acc.w = __fmaf_rn(am[u], bv.w, acc.w);
                }
            }
        };
        if (tid < 128) {  // X[p] = A_(2p+1, 2p) T_(2p, 2p): thread (p, row r, column quad cq)
            const int p = tid >> 6, r = (tid >> 2) & 15, cq = tid & 3;
            const int r0 = 16 * (2 * p + 1), c0 = 32 * p;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            dot4(&s.u.s.Akk[r0 + r][c0], &s.u.s.T[c0][c0 + 4 * cq], kC + 4, 0, kTile, acc);
            *reinterpret_cast<float4 *>(&s.u.s.X[p][r][4 * cq]) = acc;
        }
        __syncthreads();
        if (tid < 128) {  // T_(2p+1, 2p) = -T_(2p+1, 2p+1) X[p]
            const int p = tid >> 6, r = (tid >> 2) & 15, cq = tid & 3;
            const int r0 = 16 * (2 * p + 1), c0 = 32 * p;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            dot4(&s.u.s.T[r0 + r][r0], &s.u.s.X[p][0][4 * cq], kTile + 4, 0, kTile, acc);
            *reinterpret_cast<float4 *>(&s.u.s.T[r0 + r][c0 + 4 * cq]) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
        }
        __syncthreads();
        if (tid < 256) {  // Y = A[32:64, 0:32] T[0:32, 0:32]: thread (row r, column quad cq);
                          // T[k][16 ..] = 0 for k < 16
            const int r = tid >> 3, cq = tid & 7;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            dot4(&s.u.s.Akk[2 * kTile + r][0], &s.u.s.T[0][4 * cq], kC + 4, cq < 4 ? 0 : kTile, 2 * kTile, acc);
            *reinterpret_cast<float4 *>(&s.u.s.Y[r][4 * cq]) = acc;
        }
        __syncthreads();
        if (tid < 256) {  // T[32 + r, 0:32] = -T[32 + r, 32:64] Y; T[32 + r][48 ..] = 0 for r < 16
            const int r = tid >> 3, cq = tid & 7;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            dot4(&s.u.s.T[2 * kTile + r][2 * kTile], &s.u.s.Y[0][4 * cq], 2 * kTile + 4, 0,
                 r < kTile ? kTile : 2 * kTile, acc);
            *reinterpret_cast<float4 *>(&s.u.s.T[2 * kTile + r][4 * cq]) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
        }
        __syncthreads();

        // ---- T' = T Diag(beta), split: the A operand of [W | U'] (K-major, M = 64 rows i,
        // ---- K = 64 tokens j; 8-token groups outermost) ------------------------------------
        {
            const int i = tid & (kC - 1), j8 = tid >> 6;
            const float4 t0v = *reinterpret_cast<const float4 *>(&s.u.s.T[i][8 * j8]);
            const float4 t1v = *reinterpret_cast<const float4 *>(&s.u.s.T[i][8 * j8 + 4]);
            const float4 b0 = *reinterpret_cast<const float4 *>(&s.beta[b][8 * j8]);
            const float4 b1 = *reinterpret_cast<const float4 *>(&s.beta[b][8 * j8 + 4]);
            uint32_t hi[4], lo[4];
            split_pk(mul2(pk2(t0v.x, t0v.y), pk2(b0.x, b0.y)), hi[0], lo[0]);
            split_pk(mul2(pk2(t0v.z, t0v.w), pk2(b0.z, b0.w)), hi[1], lo[1]);
            split_pk(mul2(pk2(t1v.x, t1v.y), pk2(b1.x, b1.y)), hi[2], lo[2]);
            split_pk(mul2(pk2(t1v.z, t1v.w), pk2(b1.z, b1.w)), hi[3], lo[3]);
            *reinterpret_cast<uint4 *>(s.u.s.tp[0] + j8 * 1024 + i * 16) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4 *>(s.u.s.tp[1] + j8 * 1024 + i * 16) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        intra_wait(&s.bar_v, ph, fail, status);  // this item's v
        fence_proxy_async();
        tc::fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            // [W | U'] (M = 64, N = 256) = T'hi [Khat | V] + T'lo [Khat | V], 4 k-steps each
            tc::fence_after_sync();
            if (!fail) {
                const uint32_t idW = tc::idesc_bf16(64, 256, 1);
                const uint32_t th = tc::smem_addr(s.u.s.tp[0]), tl = tc::smem_addr(s.u.s.tp[1]);
                const uint32_t kvb = tc::smem_addr(s.kv);
#pragma unroll
                for (int ks = 0; ks < kC / 16; ++ks) {
                    const uint64_t bd = tc::desc(kvb + (uint32_t)ks * 256u, 128u, 1024u);
                    tc::mma_ss(D_W, tc::desc(th + (uint32_t)ks * 2048u, 1024u, 128u), bd, idW, ks > 0);
                    tc::mma_ss(D_W, tc::desc(tl + (uint32_t)ks * 2048u, 1024u, 128u), bd, idW, 1);
                }
            }
            tc::commit(&s.bar_wu);
        }
        // while the [W | U'] chain runs: q and k are read no more, so the next item's are
        // requested; then the next item's gate (its z landed long before)
        if (has_next) stage_qk(nxt);
        if (has_next) gate(nxt, b ^ 1, ((iters + 1) >> 1) & 1, pre);
        intra_wait(&s.bar_wu, ph, fail, status);
        tc::fence_after_sync();
        // the V half of the operand is free: the next item's v comes in behind the epilogue
        if (has_next) stage_v(nxt);

        // ---- epilogue: -W (bf16, K-major) and U' (fp32, token-major, units swizzled) staged
        // ---- in shared memory, then two bulk stores. Accumulator row i sits in TMEM lane
        // ---- 32 (i / 16) + i % 16; warp w reads the 16 rows of its quarter, columns
        // ---- 64 (w / 4) .. +63 ------------------------------------------------------------
        {
            const int qd = warp & 3, cq = warp >> 2;
            const int i = 16 * qd + (lane & 15);
            uint32_t d0[32], d1[32];
            tc::tmem_ld32_nowait(D_W + lanes + (uint32_t)(64 * cq), d0);
            tc::tmem_ld32_nowait(D_W + lanes + (uint32_t)(64 * cq + 32), d1);
            tc::tmem_wait_ld();
            if (lane < 16) {
                if (cq < 2) {
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const uint32_t *d = (u < 4) ? &d0[8 * u] : &d1[8 * (u - 4)];
                        uint32_t w4[4];
#pragma unroll
                        for (int p2 = 0; p2 < 4; ++p2)
                            w4[p2] = pack_bf16x2(__floats2bfloat162_rn(-__uint_as_float(d[2 * p2]),
                                                                       -__uint_as_float(d[2 * p2 + 1])));
                        *reinterpret_cast<uint4 *>(s.u.e.w + il_off(i, 64 * cq + 8 * u, kD)) =
                            make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                } else {
                    float *row = s.u.e.up + i * kD;
                    const int u0 = 16 * (cq - 2);
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        *reinterpret_cast<float4 *>(row + 4 * up_unit(i, u0 + u)) =
                            make_float4(__uint_as_float(d0[4 * u]), __uint_as_float(d0[4 * u + 1]),
                                        __uint_as_float(d0[4 * u + 2]), __uint_as_float(d0[4 * u + 3]));
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        *reinterpret_cast<float4 *>(row + 4 * up_unit(i, u0 + 8 + u)) =
                            make_float4(__uint_as_float(d1[4 * u]), __uint_as_float(d1[4 * u + 1]),
                                        __uint_as_float(d1[4 * u + 2]), __uint_as_float(d1[4 * u + 3]));
                }
            }
        }
        fence_proxy_async();      // the staged tiles are read by the bulk copy engine
        tc::fence_before_sync();  // and the TMEM reads are ordered before the next item's writes
        __syncthreads();
        if (tid == 0) {
            tc::bulk_s2g_ef(rec + kRecW, s.u.e.w, (uint32_t)kPlaneQK);
            tc::bulk_s2g_ef(rec + kRecUp, s.u.e.up, (uint32_t)(kC * kD * 4));
            tc::bulk_commit();
        }
        cur = nxt;
        nxt = nxt2;
    }
    cp_async_commit();  // every copy was waited for through its mbarrier; nothing is left
    cp_async_wait<0>();
    if (tid == 0) tc::bulk_wait0();  // the last records are written before the CTA exits
    if (tid == 0 && fail && iters > 0) {
        // a wait gave up: let the tensor-core work still in flight finish (bounded) before
        // TMEM is released; each barrier's last phase is that of the last item
        tc::mbar_wait(&s.bar_gram, (uint32_t)((iters - 1) & 1));
        tc::mbar_wait(&s.bar_wu, (uint32_t)((iters - 1) & 1));
    }
    if (dense) pdl_wait();  // the plan kernel has finished (its status write comes first)
    if (tid == 0 && fail) atomicExch(status, -7);  // KDA_ERR_CUDA
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

size_t intra_smem_bytes() { return sizeof(IntraSmem); }

cudaError_t launch_intra(const __nv_bfloat16 *q, const __nv_bfloat16 *k, const __nv_bfloat16 *v, const float *z,
                         const float *A, const float *b, int32_t *status, const int32_t *seq_cu,
                         const int32_t *chunk_off, int32_t N, int32_t H, int64_t dense_len, int64_t items,
                         int32_t item_lo, int32_t item_hi, uint8_t *records, int num_sms, cudaStream_t st) {
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kda_intra_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)sizeof(IntraSmem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    // persistent: one CTA per SM (the shared memory and TMEM allow no more) walks the items;
    // items bounds this launch's share (at least one CTA runs, to keep the launch chain)
    const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>(items, (int64_t)num_sms));
    return launch_after(kda_intra_kernel, dim3(grid), dim3(kIntraThreads), sizeof(IntraSmem), st, q, k, v, z, A, b,
                        status, seq_cu, chunk_off, N, H, dense_len, records, item_lo, item_hi);
}

}  // namespace kda
