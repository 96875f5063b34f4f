/*
 * kda.h - C ABI of the GB300 Kimi Delta Attention (KDA) library.
 *
 * KDA is the gated delta-rule recurrence, per sequence n and head h, over tokens t:
 *
 *   log a_t = -5 * sigmoid(exp(A_h) * z_t)       (a vector over d_k; bounded decay,
 *                                                 'From Linear Attention to KDA', §5.4)
 *   beta_t  = sigmoid(b_t)                       (a scalar; same page, §5.3)
 *   S_t     = (I - beta_t k_t k_t^T) Diag(a_t) S_{t-1} + beta_t k_t v_t^T
 *   o_t     = S_t^T q_t                          (same page, §5.2; 'Kimi K3 attention deep
 *                                                 dive', §2.1; 'Kimi K3', section
 *                                                 "Kimi Delta Attention")
 *
 * S is a d_k x d_v fp32 matrix (row index = key channel). The library supports
 * d_k = d_v = 128 only. Inputs arrive already projected: q and k L2-normalised by the
 * caller, z and b the raw pre-activations of the decay and write-strength gates.
 * No 1/sqrt(d_k) scale is applied to q.
 *
 * Conventions for every entry point
 *   - Pointers named "device" are CUDA device pointers owned by the caller. The library
 *     allocates nothing and keeps no pointer after the call returns.
 *   - bf16 tensors are passed as uint16_t bit patterns (IEEE bfloat16).
 *   - Layouts are dense row-major with the last dimension contiguous.
 *   - 'stream' is a cudaStream_t (NULL = the legacy default stream). Work is enqueued
 *     asynchronously; a return of KDA_OK means the arguments were valid and the
 *     kernels were launched, not that they have finished.
 *   - The compute entry points only enqueue kernels on 'stream' (no allocation, copy or
 *     synchronisation), so they can be captured into a CUDA graph and replayed; a
 *     replay gives the bits of the same call made directly. The first call of a process
 *     sets kernel attributes and reads the device's properties: make one call before the
 *     first capture. kda_workspace_status synchronises and cannot be captured.
 *   - Errors are returned as kda_status codes; nothing is thrown across the ABI and no
 *     kernel traps. A failed argument check launches nothing and writes nothing.
 *   - Every pointer must be 16-byte aligned (the kernels use 128-bit accesses);
 *     the prefill workspace must be 256-byte aligned.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_NULL = -1,        /* a required pointer is NULL */
    KDA_ERR_SHAPE = -2,       /* a size is negative or inconsistent, or beyond the launch
                                 limits: num_seqs x num_heads >= 2^31, num_heads > 65535, or
                                 (prefill) chunk slots x num_heads >= 2^31 */
    KDA_ERR_UNSUPPORTED = -3, /* d_k or d_v other than 128, or an unknown output dtype */
    KDA_ERR_SEQLENS = -4,     /* cu_seqlens not rising from 0 to the token count */
    KDA_ERR_ALIGN = -5,       /* a pointer is not 16-byte (workspace: 256-byte) aligned */
    KDA_ERR_WORKSPACE = -6,   /* workspace smaller than kda_chunk_prefill_workspace_size() */
    KDA_ERR_CUDA = -7,        /* a CUDA launch or API call failed */
    KDA_ERR_DEVICE = -8       /* the device lacks what the kernels need (sm_103a, smem) */
} kda_status;

/* Output element type of the prefill. */
typedef enum {
    KDA_OUT_BF16 = 0, /* o rounded to bf16 (round to nearest even) */
    KDA_OUT_F32 = 1   /* o kept in fp32 */
} kda_out_dtype;

/* Short English text for a status code (static storage; never NULL). */
const char *kda_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int kda_version(void);

/*
 * Test hook for the state walk's failure path (no counterpart on the pages). On the
 * current device, every later kda_chunk_prefill call leaves out the MMA-completion signal
 * of chunk slot skip_commit_chunk in its state walks (-1: none; -2 - j: that of map j of
 * the map chain that a segmented walk's output walks run first, j = 0 the first), and
 * every wait of the walk gives up after wait_limit_ns nanoseconds of the GPU clock
 * (default 2e9). A walk
 * whose wait gives up skips the rest of its work, writes NaN into its final state and
 * sets the workspace status word to KDA_ERR_CUDA (see kda_workspace_status); no GPU fault
 * is involved and the context stays usable. Restore with (-1, 2000000000) before normal
 * use. The setting is global to the device and the process and not synchronised with
 * work in flight: call it with the device idle.
 *
 * Returns KDA_OK, KDA_ERR_SHAPE for wait_limit_ns == 0, or KDA_ERR_CUDA.
 */
int kda_debug_walk_fault(int32_t skip_commit_chunk, uint64_t wait_limit_ns);

/*
 * Test hook for the segmented walk's long end segments (no counterpart on the pages).
 * When a kda_chunk_prefill call takes the segmented walk with a combine kernel (walk
 * form 2, see kda_chunk_prefill_walk_form), a sequence of at least (2 E + 1) P chunks
 * (P the segment length the sizes give) is cut into a first and a last segment of E P
 * chunks and segments of P chunks between them; the sizes choose E themselves (1 = every segment P chunks), and
 * end_factor > 0 forces E = end_factor on every later call in this process (0 restores
 * the sizes' choice). The segment length, the workspace size and the launch count do not
 * change; only the cut of each sequence does, so the results agree with E = 1 up to
 * rounding. Process-global and not synchronised with calls in flight.
 *
 * Returns KDA_OK, or KDA_ERR_SHAPE for end_factor outside [0, 64].
 */
int kda_debug_segment_ends(int32_t end_factor);

/*
 * Bytes of device workspace kda_chunk_prefill() needs for a batch of total_tokens
 * tokens in num_seqs sequences and num_heads heads. The size is an upper bound that
 * depends only on these three numbers, so one buffer serves every batch up to them.
 * Returns 0 for negative arguments.
 */
size_t kda_chunk_prefill_workspace_size(int64_t total_tokens, int32_t num_seqs, int32_t num_heads);

/*
 * Number of kernels one kda_chunk_prefill() call with these sizes launches on its
 * stream: 0 when num_seqs is 0, 3 (plan, intra-chunk, state walk) when every
 * (sequence, head) chain walks its chunks in one pass, 5 when the chains are too few to
 * fill the GPU and the walk is split into segments: plan, intra-chunk, segment-map walk,
 * then either a second intra-chunk launch beside the map walk (the chained form, see
 * kda_chunk_prefill_walk_form) or a combine kernel, and the output walk. Depends only on
 * the three sizes, like the workspace. Returns -1 for negative arguments.
 */
int32_t kda_chunk_prefill_launch_count(int64_t total_tokens, int32_t num_seqs, int32_t num_heads);

/*
 * How a kda_chunk_prefill() call with these sizes walks the state: 0 in one pass per
 * (sequence, head) chain; 1 in segments whose output walks first chain the segment maps
 * before them on the tensor cores (every output walk fits in one wave of the GPU); 2 in
 * segments whose input states a combine kernel chains. In form 1 the intra-chunk items
 * past a whole number of rounds of the GPU's SMs that belong to the last segment of a
 * dense batch's last sequence run in a second intra-chunk launch beside the map walk.
 * Depends only on the three sizes. Returns -1 for negative arguments, 0 when num_seqs is 0.
 */
int32_t kda_chunk_prefill_walk_form(int64_t total_tokens, int32_t num_seqs, int32_t num_heads);

/*
 * kda_chunk_prefill - chunkwise-parallel KDA over whole sequences.
 *
 * Computes, for every sequence and head, all outputs o_t and the final state S_T of the
 * recurrence above, starting from initial_state. The work is the chunkwise form of
 * 'From Linear Attention to KDA', §7 (chunks of 64 tokens: per-chunk decayed K K^T and
 * Q K^T matrices, the UT/WY triangular solve that turns the chain of delta updates
 * into dense products, then a serial pass that carries S from chunk to chunk), with
 * the 16-token tiles of §8 inside each chunk. The gate and beta are computed from
 * z, A, b inside the kernels.
 *
 * Batch layouts (tokens packed row by row):
 *   dense   : cu_seqlens == NULL. batch sequences of seq_len tokens each; num_seqs must
 *             equal batch. Token (i, t) is row i * seq_len + t.
 *   varlen  : cu_seqlens != NULL. batch must be 1; seq_len is the total token count;
 *             sequence n owns rows cu_seqlens[n] .. cu_seqlens[n+1]-1. Empty sequences
 *             are allowed (their final state equals their initial state).
 *
 * Arguments (T_total = batch * seq_len rows, H = num_heads):
 *   q, k        device bf16 [T_total, H, 128]   queries, L2-normalised keys
 *   v           device bf16 [T_total, H, 128]   values
 *   z           device fp32 [T_total, H, 128]   decay pre-activation
 *   A           device fp32 [H]                 per-head log scale of the decay gate
 *   b           device fp32 [T_total, H]        write-strength pre-activation
 *   initial_state device fp32 [num_seqs, H, 128, 128] or NULL (zeros)
 *   cu_seqlens  device int32 [num_seqs + 1] or NULL (dense layout)
 *   cu_seqlens_host  host int32 [num_seqs + 1] or NULL. When given it must hold the same
 *               values as cu_seqlens; it is validated on the host before anything is
 *               launched (KDA_ERR_SEQLENS). Without it, cu_seqlens is validated on the
 *               device: a bad table makes the kernels fill final_state with NaN, leave o
 *               untouched, and record KDA_ERR_SEQLENS for kda_workspace_status().
 *   o           device [T_total, H, 128], bf16 or fp32 per o_dtype (written)
 *   final_state device fp32 [num_seqs, H, 128, 128] (written). May alias initial_state.
 *   workspace   device scratch of at least kda_chunk_prefill_workspace_size() bytes,
 *               256-byte aligned. Its contents need no initialisation and are dead after
 *               the kernels finish, except the status word read by kda_workspace_status().
 *   stream      cudaStream_t
 *
 * Calls that share a workspace must be ordered on one stream.
 */
int kda_chunk_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      const float *z, const float *A, const float *b,
                      const float *initial_state,
                      const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                      int32_t batch, int64_t seq_len, int32_t num_seqs, int32_t num_heads,
                      int32_t d_k, int32_t d_v,
                      void *o, int32_t o_dtype, float *final_state,
                      void *workspace, size_t workspace_bytes, void *stream);

/*
 * Status recorded on the device by the last kda_chunk_prefill() that used this
 * workspace. Synchronises 'stream'. Returns
 *   KDA_OK           the kernels ran to the end;
 *   KDA_ERR_SEQLENS  the device-side cu_seqlens check failed (final_state is NaN);
 *   KDA_ERR_CUDA     a bounded wait inside the state walk gave up (a copy or a tensor-core
 *                    group did not complete in time); the final states of the affected
 *                    (sequence, head) pairs are NaN and their outputs are not valid;
 *   or KDA_ERR_CUDA if the copy of the status word itself fails.
 */
int kda_workspace_status(const void *workspace, void *stream);

/*
 * kda_chunk_prefill_noalloc - the same prefill, for callers that cannot allocate.
 *
 * The pages have no counterpart to this entry point; it exists for callers that cannot
 * provide the device workspace kda_chunk_prefill() asks for: a plugin running inside an
 * engine that owns all device memory and passes it only the call's tensors, or code on
 * a latency-critical path where cudaMalloc, which may synchronise the whole device, is
 * not allowed. Instead of a workspace it uses a scratch area of
 * KDA_NOALLOC_SCRATCH_BYTES compiled into the library: a static device array that exists
 * on every GPU that loads the library, from load until process exit. The library still
 * allocates nothing at call time. Arguments, results and error codes are those of
 * kda_chunk_prefill() without the two workspace arguments; inputs and outputs are still
 * the caller's.
 *
 *   - A batch whose workspace (kda_chunk_prefill_workspace_size(total_tokens, num_seqs,
 *     num_heads)) exceeds KDA_NOALLOC_SCRATCH_BYTES is refused with KDA_ERR_WORKSPACE
 *     before anything is launched. 64 MiB holds, for example, 3072 tokens x 8 heads or
 *     2048 tokens x 12 heads.
 *   - The first call on a device looks up the scratch's device address on that device
 *     (cudaGetSymbolAddress, with the device current); make that first call before any
 *     stream capture. The address is kept for the life of the process, so do not use
 *     this entry point after cudaDeviceReset() on that device: the reset unloads the
 *     library's device code and the kept address no longer names the scratch.
 *   - All calls share the one scratch area and it keeps the last call's contents. The
 *     kernels need nothing in it to start at zero, but calls whose GPU work overlaps in
 *     time (different streams, or threads without ordering) race on it: order them.
 *   - The device-side cu_seqlens check still fills final_state with NaN on a bad table;
 *     there is no workspace to pass to kda_workspace_status(), so pass cu_seqlens_host
 *     to have the table checked on the host instead.
 */
#define KDA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int kda_chunk_prefill_noalloc(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                              const float *z, const float *A, const float *b,
                              const float *initial_state,
                              const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                              int32_t batch, int64_t seq_len, int32_t num_seqs, int32_t num_heads,
                              int32_t d_k, int32_t d_v,
                              void *o, int32_t o_dtype, float *final_state, void *stream);

/*
 * kda_recurrent_decode - one token per sequence, the recurrence applied in place.
 *
 * For every sequence n and head h: read S = state[n, h], apply
 *   S' = Diag(a) S;  p = S'^T k;  S = S' + beta k (v - p)^T;  o = S^T q
 * (the three-step diagonal-plus-low-rank update of 'Kimi K3 attention deep dive', §2.2;
 * the error form of 'Kimi K3', section "Kimi Delta Attention"), write S back and o out.
 * All arithmetic is fp32.
 *
 * Arguments (N = num_seqs, H = num_heads):
 *   q, k, v   device bf16 [N, H, 128]
 *   z         device fp32 [N, H, 128]
 *   A         device fp32 [H]
 *   b         device fp32 [N, H]
 *   state     device fp32 [N, H, 128, 128], read and overwritten in place
 *   o         device fp32 [N, H, 128] (written)
 *   stream    cudaStream_t
 */
int kda_recurrent_decode(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                         const float *z, const float *A, const float *b,
                         float *state, float *o,
                         int32_t num_seqs, int32_t num_heads, int32_t d_k, int32_t d_v,
                         void *stream);

/* Most draft tokens one kda_recurrent_verify() or kda_replay_fold() call takes. */
#define KDA_MAX_REPLAY_TOKENS 16

/*
 * kda_recurrent_verify - several tokens per sequence from a checkpoint state, with the
 * gate values logged for a later replay (ReplaySSM, 'Kimi K3 attention deep dive', §6.2).
 *
 * For every sequence n and head h, starting from S = state[n, h], the decode update of
 * kda_recurrent_decode() is applied to the m tokens of the sequence in order, and each
 * token's output o = S^T q (after its own write) is written. The checkpoint `state` is
 * only read. With state_out = state this is multi-token decode in place.
 *
 * Token t of sequence n is row n * m + t of the token-major inputs (m = num_tokens):
 *   q, k, v   device bf16 [N * m, H, 128]
 *   z         device fp32 [N * m, H, 128]
 *   A         device fp32 [H]
 *   b         device fp32 [N * m, H]
 *   state     device fp32 [N, H, 128, 128], read only
 *   state_out device fp32 [N, H, 128, 128] or NULL: the state after all m tokens
 *             (may be `state` itself)
 *   o         device fp32 [N * m, H, 128] (written)
 *   gk_log    device fp32 [N * m, H, 128] or NULL: each token's log a = -5 sigmoid(e^A z)
 *   beta_log  device fp32 [N * m, H] or NULL: each token's beta = sigmoid(b)
 *   num_tokens 0 .. KDA_MAX_REPLAY_TOKENS (larger: KDA_ERR_UNSUPPORTED)
 *
 * The per-element arithmetic, the column split and the order of the reductions are
 * those of kda_recurrent_decode() for the same num_seqs and num_heads, so o of token t
 * equals, bit for bit, the output of the (t+1)-th of m kda_recurrent_decode() calls on
 * a copy of the checkpoint, and state_out equals the state after the m-th call. That
 * (the ReplaySSM requirement) holds on one device for one (num_seqs, num_heads).
 * Pointers need 16-byte alignment (A, b, beta_log: 4). Stream-ordered, asynchronous.
 */
int kda_recurrent_verify(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                         const float *z, const float *A, const float *b,
                         const float *state, float *state_out, float *o,
                         float *gk_log, float *beta_log,
                         int32_t num_seqs, int32_t num_heads, int32_t num_tokens,
                         int32_t d_k, int32_t d_v, void *stream);

/*
 * kda_replay_fold - commit the accepted prefix of a verified draft window to the state.
 *
 * For every sequence n, the first a_n = clamp(num_accepted[n], 0, m) tokens of the
 * window are replayed, in order, on state[n, :] in place, from the caller's k, v and
 * the gate values that kda_recurrent_verify() logged (the fused fold of 'Kimi K3
 * attention deep dive', §6.2). The state must be the checkpoint the window was verified
 * from. No output is produced, and a sequence with a_n = 0 is not touched.
 *
 *   k, v          device bf16 [N * m, H, 128], the window's tokens as given to verify
 *   gk_log        device fp32 [N * m, H, 128] from kda_recurrent_verify()
 *   beta_log      device fp32 [N * m, H]      from kda_recurrent_verify()
 *   num_accepted  device int32 [N]
 *   state         device fp32 [N, H, 128, 128], updated in place
 *   num_tokens    the window length m, 0 .. KDA_MAX_REPLAY_TOKENS
 *
 * The result equals, bit for bit, a_n kda_recurrent_decode() calls with the same
 * (num_seqs, num_heads) on that sequence's tokens. Alignment: 16 bytes (beta_log and
 * num_accepted: 4).
 */
int kda_replay_fold(const uint16_t *k, const uint16_t *v, const float *gk_log, const float *beta_log,
                    const int32_t *num_accepted, float *state,
                    int32_t num_seqs, int32_t num_heads, int32_t num_tokens,
                    int32_t d_k, int32_t d_v, void *stream);

/*
 * kda_fused_decode - one decode token of the whole KDA layer step between the
 * projections: causal conv -> recurrent update -> gated RMSNorm in one launch ('Kimi K3
 * attention deep dive', §6.3), with the activations of the same page's §2.3:
 *
 *   q = L2Norm(Swish(ShortConv(x_q))),  k = L2Norm(Swish(ShortConv(x_k))),
 *   v = Swish(ShortConv(x_v))
 *   then the update of kda_recurrent_decode() on state[n, h] (in place), o = S^T q
 *   y = o / sqrt(mean(o^2) + eps_rms) * norm_w * sigmoid(g)
 *
 * ShortConv is depthwise and causal with 4 taps: output channel c is
 *   conv_w[s, h, c, 0] x_{t-3} + conv_w[s, h, c, 1] x_{t-2} + conv_w[s, h, c, 2] x_{t-1}
 *   + conv_w[s, h, c, 3] x_t,
 * with x_{t-3..t-1} read from the conv state, which afterwards holds x_{t-2}, x_{t-1}, x_t
 * (a new sequence starts from zeros). L2Norm(x) = x / sqrt(sum(x^2) + eps_l2) over the
 * head's 128 channels; Swish(x) = x sigmoid(x). There is no 1/sqrt(d) scale on q.
 *
 * Arguments (N = num_seqs, H = num_heads; all device pointers, caller-owned):
 *   x_q, x_k, x_v  bf16 [N, H, 128]      the projections before the convolution
 *   conv_state     bf16 [N, 3, 3, H, 128] per stream (q, k, v) the last three inputs,
 *                  oldest first; read and updated in place
 *   conv_w         fp32 [3, H, 128, 4]    taps per stream, head, channel, oldest first
 *   z, A, b        as kda_recurrent_decode()
 *   g              fp32 [N, H, 128]       output-gate pre-activation
 *   norm_w         fp32 [128]             RMSNorm weight (shared by the heads)
 *   eps_l2, eps_rms  >= 0 (negative or NaN: KDA_ERR_UNSUPPORTED)
 *   state          fp32 [N, H, 128, 128]  read and overwritten in place
 *   y              fp32 [N, H, 128]       written
 * Alignment: 16 bytes (A, b: 4). All arithmetic is fp32. Stream-ordered, asynchronous.
 */
int kda_fused_decode(const uint16_t *x_q, const uint16_t *x_k, const uint16_t *x_v,
                     uint16_t *conv_state, const float *conv_w,
                     const float *z, const float *A, const float *b,
                     const float *g, const float *norm_w, float eps_l2, float eps_rms,
                     float *state, float *y,
                     int32_t num_seqs, int32_t num_heads, int32_t d_k, int32_t d_v, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
