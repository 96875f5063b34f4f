// Device helpers shared by the KDA kernels: the gate, tile geometry, the layout of
// the per-chunk record that the intra-chunk kernel writes and the state walk reads, and
// thin wrappers over the PTX used (mma.sync, ldmatrix, cp.async).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_f32x2.cuh"

namespace kda {

constexpr int kD = 128;        // d_k = d_v
constexpr int kC = 64;         // chunk length (tokens)
constexpr int kTile = 16;      // sub-chunk tile ('From Linear Attention to KDA', §8)
constexpr float kGMin = -5.0f; // lower bound of log a (same page, §5.4)

// Row strides (in bf16 elements) of the 16-bit tiles kept in shared memory and in the
// chunk record. The 16-byte pad staggers rows across banks so that ldmatrix reads of
// 8 consecutive rows hit 32 distinct banks.
constexpr int kLd128 = kD + 8;  // 128-wide tiles: 272 B per row
constexpr int kLd64 = kC + 8;   // 64-wide tiles: 144 B per row

// ---------------------------------------------------------------------------------
// Chunk record: everything the serial state walk needs about one (chunk, head). The
// operand tiles are stored as the exact shared-memory images the tensor core reads,
// in the no-swizzle canonical layouts of kda_tc.cuh: core matrices of 8 rows x 16 bytes.
//   [ -W ; Qhat ]  K-major, 128 rows (row = token, K = key channel), three 16 KB planes
//          W    -W = -T' Khat in bf16 (rows 0..63). One bf16 plane is enough here: the
//               rounding of W moves the outputs by less than a tenth of their error bar.
//          Qh   q_i * exp(G_i), hi plane (rows 64..127)
//          Ql   the lo plane of the same (hi + lo = the fp32 value to ~16 bits)
//   AK  [ A_qk ; Kend^T ]  MN-major (N = 192, K = 64 tokens j), a hi and a lo plane
//          n 0..63    decayed causal Q K^T, diagonal included (n = query token i); its
//                     128-byte blocks of 8 query rows x 8 keys that lie wholly above the
//                     diagonal (key group > query group: 28 of 64) are zero and are
//                     neither written nor read: a reader keeps them zero on its side
//          n 64..191  k_j * exp(G_last - G_j), transposed     (n = key channel c)
//   gam  [128]   fp32   exp(G_last), the chunk's total decay
//   Up   [64][128] fp32 U' = T' V, token-major (row i, column = value channel); the
//        16-byte units (4 channels) of row i are XOR-swizzled by i % 32: channel c of row i
//        is at i * 128 + 4 ((c / 4) ^ (i % 32)) + c % 4
// ---------------------------------------------------------------------------------
constexpr size_t kPlaneQK = (size_t)kC * kD * 2;   // 64 x 128 bf16 tile
constexpr size_t kPlaneKT = (size_t)kD * kC * 2;   // 128 x 64 bf16 tile
constexpr size_t kPlaneCC = (size_t)kC * kC * 2;   // 64 x 64 bf16 tile
constexpr size_t kStackAK = kPlaneCC + kPlaneKT;   // one plane of [ A_qk ; Kend^T ]: 192 x 64
constexpr size_t kRecW = 0;                        // -W, then Qhat hi and lo: one 48 KB run
constexpr size_t kRecQh = kRecW + kPlaneQK;
constexpr size_t kRecQl = kRecQh + kPlaneQK;
constexpr size_t kRecWQBytes = 3 * kPlaneQK;
constexpr size_t kRecAK = kRecW + kRecWQBytes;
constexpr size_t kRecGam = kRecAK + 2 * kStackAK;
constexpr size_t kRecUp = kRecGam + kD * 4;
constexpr size_t kRecBytes = kRecUp + (size_t)kC * kD * 4;
// where each part of AK starts (its lo plane is one stack further)
constexpr size_t kRecAqk = kRecAK;
constexpr size_t kRecKeT = kRecAK + kPlaneCC;
static_assert(kRecBytes % 128 == 0, "chunk records must stay 128-byte aligned");
static_assert(kRecAK % 16 == 0 && kRecGam % 16 == 0 && kRecUp % 16 == 0, "record fields must be 16-byte aligned");

// byte offset of element (n, j) of the MN-major [ A_qk ; Kend^T ] plane: core matrices of
// 8 tokens j (K) x 8 consecutive n (16 bytes); the 8 K-groups of one n-group are adjacent
// (K-direction stride 128 B), n-groups are 1024 B apart
__host__ __device__ constexpr uint32_t ak_off(int n, int j) {
    return (uint32_t)((n >> 3) * 1024 + (j >> 3) * 128 + (j & 7) * 16 + (n & 7) * 2);
}
// whether the A_qk element (query row n, key j) lies in a 128-byte block of the plane that
// is wholly above the diagonal (its 8 keys all come after its 8 query rows): such blocks
// are zero and stay out of the record
__host__ __device__ constexpr bool aqk_zero_block(int n, int j) { return (j >> 3) > (n >> 3); }
// the same for the 16-byte unit u of an A_qk plane (u = ak_off / 16, u < 512)
__host__ __device__ constexpr bool aqk_zero_unit(int u) { return ((u >> 3) & 7) > (u >> 6); }
static_assert(aqk_zero_unit((int)(ak_off(7, 8) / 16)) && !aqk_zero_unit((int)(ak_off(8, 15) / 16)) &&
                  aqk_zero_block(0, 63) && !aqk_zero_block(63, 0),
              "zero blocks of A_qk");

// byte offset of element (r, k) in an interleaved K-major tile with K elements per row
__host__ __device__ constexpr uint32_t il_off(int r, int k, int K) {
    return (uint32_t)((r >> 3) * (K >> 3) * 128 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

// Workspace: [0, 256) header (int32 status at offset 0), then seq_cu[N+1] and
// chunk_off[N+1] (int32, 256-byte aligned each), then the chunk records.
constexpr size_t kWsHeader = 256;
__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
__host__ __device__ inline size_t ws_table_bytes(int64_t num_seqs) {
    return align_up((size_t)(num_seqs + 1) * 4, 256);
}
__host__ __device__ inline int64_t chunk_bound(int64_t total_tokens, int64_t num_seqs) {
    // sum_n ceil(len_n / C) <= (total + (C-1) * N) / C
    return (total_tokens + (int64_t)(kC - 1) * num_seqs) / kC;
}

// ---------------------------------------------------------------------------------
// Walk units: one CTA of the state walk (per head, blockIdx.y) carries a state across a
// run of chunks of one sequence. A plain walk has one unit per sequence. With few long
// sequences the chunks are cut into segments that run in parallel (the single-GPU form
// of KDA context parallelism): each segment's affine state map S_out = M S_in + R is
// found from walks started at zero and at the identity, the maps are chained per
// sequence, and every segment is walked again from its true input state.
// ---------------------------------------------------------------------------------
struct WalkUnit {
    const float *in;  // state at the start for head 0 ([128][128], row = key channel), head h
                      // at in + h * 128 * 128; nullptr: zero (or the identity, see flags)
    float *out;       // state at the end, same layout (or split planes, kUnitOutPlanes);
                      // nullptr: not kept
    // maps applied to the start state before the walk, in order: X <- M_j X + R_j for
    // j = 1 .. chain. M_j of head h is at maps + ((j - 1) H + h) * 128 * 128 floats, stored
    // as split bf16 planes (kUnitOutPlanes); R_j at offs, same indexing, in quads
    // (kUnitOutQuads)
    const float *maps, *offs;
    int32_t c_begin, c_end;  // chunk-record slots
    int32_t t_begin, t_end;  // tokens of those chunks (the last chunk may be partial)
    int32_t flags;
    int32_t chain;
};
constexpr int kUnitWriteO = 1;     // write the outputs o of these chunks
constexpr int kUnitAddUp = 2;      // U = U' - W S (else U = -W S: the homogeneous map)
constexpr int kUnitIdentity = 4;   // start from the identity when in == nullptr
constexpr int kUnitOutPlanes = 8;  // keep the end state S as the two bf16 planes (hi, then
                                   // lo = bf16(S - hi)) of the tensor-core operand B[n][k] =
                                   // S[n][k], interleaved K-major (il_off(n, k, 128)), 32 KB each
// the quad layout of a state: S[r][c] at ((r / 4) * 128 + c) * 4 + r % 4, so that the walk
// thread of value column c reads or writes four key rows with one 16-byte access, and a
// warp's 32 columns are 512 contiguous bytes
constexpr int kUnitOutQuads = 16;  // keep the end state in the quad layout
constexpr int kUnitInQuads = 32;   // the start state is in the quad layout
constexpr size_t kStateFloats = (size_t)kD * kD;

// Tables of the segmented walk, built by the plan kernel when P > 0 (segment length in
// chunks; P == 0: a plain walk, nothing else is read).
struct SegPlan {
    int32_t P;
    float *Sin, *Mseg, *Rseg;  // per (segment, head): input state, map M, offset R
    WalkUnit *unitsA, *unitsC;
    int32_t *nA, *nC;
    int32_t *chains;     // per sequence: first segment, number of segments (combine form)
    int32_t chain_mode;  // 1: each output walk chains the maps before it; 0: a combine kernel does
    int32_t E;           // end factor: a sequence of at least (2 E + 1) P chunks has first and
                         // last segments of E P chunks (1: every segment P chunks)
};

// Segment length (in chunks) of the segmented walk, or 0 for a plain walk. A pure
// function of the batch size, so that the workspace size can be computed without a
// device: segments pay when there are fewer (sequence, head) chains than about a wave
// of the GPU's 152 SMs and the chains are long. The length minimises a cost model of
// the three phases, in units of one output-walk chunk step, fitted to measured walks:
// with S segments of P chunks, phase A runs 2 S - 3 map walks per chain in
// ceil((2 S - 3) chains / 152) waves of P + 2 steps (a map step costs about 0.83 of an
// output step; the 2 covers a walk's start and end), the chain of S - 2 map products
// (about 1.2 steps each as the combine kernel's; the output walks' own chain, taken when
// phase C fits one wave, costs about 0.6 a map and keeps the same choice), and phase C S
// walks per chain in ceil(S chains / 152) waves of P + 2 steps. For 8192 tokens x 12
// heads this keeps 7 segments of at most 19 chunks (cut to even out the output walks' map
// chains in the chained form); for 1,048,576 tokens x 12 heads it takes 38
// segments of 432 chunks (phase A in six waves) before the long ends below are considered.
__host__ __device__ inline int walk_segment_uniform(int64_t total_tokens, int64_t num_seqs, int64_t num_heads) {
    const int64_t chains = num_seqs * num_heads;
    if (chains <= 0) return 0;
    const int64_t slots = chunk_bound(total_tokens, num_seqs);
    const int64_t avg = slots / num_seqs;
    if (chains * 2 >= 152 || avg < 24) return 0;
    int64_t best_p = 4;
    double best = 1e300;
    for (int64_t S = 2; S <= 64; ++S) {
        int64_t P = (avg + S - 1) / S;
        if (P < 4) P = 4;
        const int64_t segs = (avg + P - 1) / P;  // the segments a chain of avg chunks gets
        const int64_t waves_a = ((2 * segs - 3) * chains + 151) / 152, waves_c = (segs * chains + 151) / 152;
        const double cost = 0.83 * (double)(waves_a * (P + 2)) + 1.2 * (double)(segs - 2) + (double)(waves_c * (P + 2));
        if (cost < best) {
            best = cost;
            best_p = P;
        }
    }
    return (int)best_p;
}
__host__ __device__ inline int64_t segment_bound(int64_t total_tokens, int64_t num_seqs, int P) {
    return (chunk_bound(total_tokens, num_seqs) + (int64_t)(P - 1) * num_seqs) / P;
}
// How the segmented walk finds each segment's input state. When every output walk fits in
// one wave of the GPU (segments x heads <= 152), each one chains the maps of the segments
// before it on the tensor cores (M as split bf16 planes): the chain of the last segment,
// about 1.7 us per map, replaces a kernel launch and its serial chain on the critical path.
// With more segments that replicated chain costs more SM time than it saves, and a combine
// kernel chains the maps once per (sequence, head) in fp32 instead. A pure function of the
// sizes, like the segment length.
__host__ __device__ inline bool walk_chain_mode(int64_t total_tokens, int64_t num_seqs, int64_t num_heads) {
    const int P = walk_segment_uniform(total_tokens, num_seqs, num_heads);
    return P > 0 && segment_bound(total_tokens, num_seqs, P) * num_heads <= 152;
}
// Long ends (combine form only). The first segment of a chain needs one walk in phase A
// (from the initial state, no map) and the last none, while every other segment needs two
// (M and R). Making the two end segments E times as long as the others therefore takes
// map work off phase A, and in phase C their long walks run beside several waves of short
// ones. The walks of both phases are listed longest first. (P, E) minimises the cost model
// above with each phase's waves counted in units of P chunks per SM (a long walk fills E of
// them, and a phase lasts at least E); E = 1 is the uniform split. For 1,048,576 tokens x
// 12 heads: 42 segments of 328 chunks between two of 1,312 (phase A and phase C in seven
// and four such waves, against six and three waves of 432 chunks uniform).
struct SegShape {
    int P, E;
};
__host__ __device__ inline SegShape walk_segments(int64_t total_tokens, int64_t num_seqs, int64_t num_heads) {
    const int P1 = walk_segment_uniform(total_tokens, num_seqs, num_heads);
    if (P1 == 0 || walk_chain_mode(total_tokens, num_seqs, num_heads)) return SegShape{P1, 1};
    const int64_t chains = num_seqs * num_heads;
    const int64_t avg = chunk_bound(total_tokens, num_seqs) / num_seqs;
    auto cost = [&](int64_t P, int64_t E) {
        // the segments a chain of avg chunks gets, and each phase's walks in P-chunk units
        const int64_t segs = E > 1 ? 2 + (avg - 2 * E * P + P - 1) / P : (avg + P - 1) / P;
        const int64_t ua = chains * (E > 1 ? E + 2 * (segs - 2) : 2 * segs - 3);
        const int64_t uc = chains * (E > 1 ? 2 * E + segs - 2 : segs);
        int64_t waves_a = (ua + 151) / 152, waves_c = (uc + 151) / 152;
        if (waves_a < E) waves_a = E;
        if (waves_c < E) waves_c = E;
        return 0.83 * (double)(waves_a * (P + 2)) + 1.2 * (double)(segs - 2) + (double)(waves_c * (P + 2));
    };
    SegShape best{P1, 1};
    double best_cost = cost(P1, 1);
    for (int64_t E = 2; E <= 6; ++E) {
        for (int64_t S = 3; S <= 96; ++S) {
            int64_t P = (avg + 2 * E + S - 3) / (2 * E + S - 2);
            if (P < 4) P = 4;
            if (avg < (2 * E + 1) * P) continue;
            const double c = cost(P, E);
            if (c < best_cost) {
                best_cost = c;
                best = SegShape{(int)P, (int)E};
            }
        }
    }
    return best;
}
// Balanced cut (chained form). The output walk of segment k >= 1 first chains k - 1 maps,
// each about kChainStep16 / 16 of a chunk step (about 1.7 against 3.1 us, measured), so a
// sequence of len chunks in S = ceil(len / P) >= 3 segments is cut to even out chain plus
// chunks: segment k takes min(P, (t - kChainStep16 (k - 1)) / 16) chunks (segment 0:
// min(P, t / 16)), at least one, for the lowest level t (in 1/16 chunks) at which the
// lengths reach len; the segments that grew at that level give back the surplus, the last
// ones first. Used by the plan kernel and, for the last segment, by the host.
constexpr int32_t kChainStep16 = 9;
struct BalancedCut {
    int32_t P = 0, S = 0, level = 0, grown = 0, surplus = 0;
    __host__ __device__ static int32_t len_at(int32_t t16, int32_t k, int32_t P) {
        const int32_t x = t16 - kChainStep16 * (k > 1 ? k - 1 : 0);
        return x < 16 ? 1 : (P < (x >> 4) ? P : (x >> 4));
    }
    __host__ __device__ int32_t total(int32_t t16) const {
        int32_t sum = 0;
        for (int32_t k = 0; k < S; ++k) sum += len_at(t16, k, P);
        return sum;
    }
    __host__ __device__ BalancedCut(int32_t len, int32_t P_, int32_t S_) : P(P_), S(S_) {
        int32_t lo = 0, hi = 16 * P + kChainStep16 * S;  // total(hi) = S P >= len
        while (lo < hi) {
            const int32_t mid = (lo + hi) / 2;
            if (total(mid) >= len)
                hi = mid;
            else
                lo = mid + 1;
        }
        level = lo;
        surplus = total(level) - len;
        for (int32_t k = 0; k < S; ++k) grown += grew(k);
    }
    __host__ __device__ bool grew(int32_t k) const { return len_at(level, k, P) > len_at(level - 1, k, P); }
    // the last segment's length (it gives back first)
    __host__ __device__ int32_t last_len() const {
        return len_at(level, S - 1, P) - ((grew(S - 1) && surplus > 0) ? 1 : 0);
    }
};

// Segment length (in chunks) of the segmented walk, or 0 for a plain walk
__host__ __device__ inline int walk_segment_chunks(int64_t total_tokens, int64_t num_seqs, int64_t num_heads) {
    return walk_segments(total_tokens, num_seqs, num_heads).P;
}

// ---------------------------------------------------------------------------------
// Gate: log a = g_min * sigmoid(exp(A_h) * z), beta = sigmoid(b)
// ---------------------------------------------------------------------------------
__device__ __forceinline__ float gate_log_decay(float eA, float z) {
    return kGMin / (1.0f + expf(-eA * z));
}
__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + expf(-x)); }

// ---------------------------------------------------------------------------------
// Split-bf16: x = hi + lo with hi = bf16(x), lo = bf16(x - hi). A product of two split
// operands is taken as hi*hi + hi*lo + lo*hi, which carries about 16 mantissa bits.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_bf16x2(__nv_bfloat162 v) {
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ void split_bf16x2(float x, float y, uint32_t &hi, uint32_t &lo) {
    __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    float2 hf = __bfloat1622float2(h);
    __nv_bfloat162 l = __floats2bfloat162_rn(x - hf.x, y - hf.y);
    hi = pack_bf16x2(h);
    lo = pack_bf16x2(l);
}
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t u) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162 *>(&u);
    return __bfloat1622float2(h);
}

// ---------------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// D += A(16x16, row) * B(16x8, col), bf16 inputs, fp32 accumulate
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// split-bf16 product: d += ah*bh + ah*bl + al*bh
__device__ __forceinline__ void mma_split3(float (&d)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4],
                                           uint32_t bh0, uint32_t bh1, uint32_t bl0, uint32_t bl1) {
    mma_bf16(d, al, bh0, bh1);
    mma_bf16(d, ah, bl0, bl1);
    mma_bf16(d, ah, bh0, bh1);
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}

// A fragment (16x16) of a row-major bf16 tile at (row0, col0), row stride ld elements.
__device__ __forceinline__ void load_a(uint32_t (&r)[4], const __nv_bfloat16 *base, int ld, int row0, int col0,
                                       int lane) {
    ldsm_x4(r, base + (size_t)(row0 + (lane & 15)) * ld + col0 + ((lane >> 4) << 3));
}
// B fragments of two adjacent n8 tiles (cols n0..n0+15), k rows k0..k0+15, from a tile
// stored [k][n] row-major: r[0],r[1] = tile n0; r[2],r[3] = tile n0+8.
__device__ __forceinline__ void load_b_kn(uint32_t (&r)[4], const __nv_bfloat16 *base, int ld, int k0, int n0,
                                          int lane) {
    ldsm_x4_t(r, base + (size_t)(k0 + (lane & 7) + (((lane >> 3) & 1) << 3)) * ld + n0 + ((lane >> 4) << 3));
}

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem_dst)), "l"(gmem_src));
}
// the same with the shared-memory address given as such (unrolled copies add immediate
// offsets to one base)
__device__ __forceinline__ void cp_async16_s(uint32_t sdst, const void *gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sdst), "l"(gmem_src));
}
__device__ __forceinline__ void cp_async4(void *smem_dst, const void *gmem_src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_u32(smem_dst)), "l"(gmem_src));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
// one arrival on the mbarrier once all of this thread's earlier cp.async copies have landed
// (the arrival counts against the barrier's initial count)
__device__ __forceinline__ void cp_async_arrive(uint64_t *mbar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(smem_u32(mbar)) : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

// named barriers (bar.sync / bar.arrive) over a subset of a CTA's warps
__device__ __forceinline__ void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n)); }
__device__ __forceinline__ void named_arrive(int id, int n) {
    asm volatile("bar.arrive %0, %1;\n" ::"r"(id), "r"(n));
}

// Programmatic dependent launch: the kernels after the plan kernel are launched while
// their predecessor runs. Each waits for the predecessor to finish (and its memory to be
// visible) before anything else; each lets its successor launch once all its own CTAs
// are resident, so a waiting successor never holds an SM a predecessor CTA still needs.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

// a launch that may start while the previous kernel on the stream runs (the kernel
// waits for it with griddepcontrol.wait before touching its results)
template <typename... Params, typename... Args>
inline cudaError_t launch_after(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

// a packed pair y split into bf16 hi and lo pairs (one packed subtraction; the values of
// split_bf16x2)
__device__ __forceinline__ void split_pk(uint64_t y, uint32_t &hi, uint32_t &lo) {
    const float2 v = upk2(y);
    hi = pack_bf16x2(__floats2bfloat162_rn(v.x, v.y));
    const float2 d = upk2(sub2(y, pk2(__uint_as_float(hi << 16), __uint_as_float(hi & 0xffff0000u))));
    lo = pack_bf16x2(__floats2bfloat162_rn(d.x, d.y));
}
// (x0 f0, x1 f1) for a bf16 pair x and fp32 factors f, split into bf16 hi and lo pairs:
// one packed multiply and one packed subtraction
__device__ __forceinline__ void scale_split_pk(uint32_t xbf2, float f0, float f1, uint32_t &hi, uint32_t &lo) {
    const float2 x = bf16x2_to_float2(xbf2);
    split_pk(mul2(pk2(x.x, x.y), pk2(f0, f1)), hi, lo);
}

// largest n with chunk_off[n] <= slot (empty sequences share an offset and are skipped)
__device__ __forceinline__ int find_seq(const int32_t *chunk_off, int32_t N, int32_t slot) {
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

}  // namespace kda
