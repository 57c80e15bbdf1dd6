/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention library, libkda.so.
 *
 * The operation.  Per (sequence, head) the library keeps a fixed-size state
 * S in R^{dk x dv} (fp32) and applies, for every token t, in this order
 * ("Kimi K3 Architecture Explained", section 3 "Kimi Delta Attention": decay
 * stale context first, then erase conflicting memory, then write):
 *
 *     S <- Diag(exp(g_t)) S               decay, per key channel
 *     S <- S - beta_t k_t (k_t^T S)        erase
 *     S <- S + beta_t k_t v_t^T            write
 *     o_t = S^T q_t                        read, after the update
 *
 * g is the caller's log-decay, normally g = -5 sigmoid(x) so that g lies in
 * (-5, 0) (Kimi K3 technical-report digest, section 2.1 (1): bounded scaled
 * sigmoid, g_min = -5).  There is no positional input and no 1/sqrt(d) scale.
 *
 * Layouts (all row-major, innermost index last, no padding):
 *   q, k : [T_tot, H, dk]   activation dtype (fp32 or bf16)
 *   v    : [T_tot, H, dv]   activation dtype
 *   out  : [T_tot, H, dv]   activation dtype
 *   g    : [T_tot, H, dk]   fp32
 *   beta : [T_tot, H]       fp32
 *   states (S0, S_final, S_inout, zero-initial states) : [.., dk, dv] fp32
 *   transfer matrices : [.., dk, dk] fp32
 * Sequences are packed along T_tot and delimited by cu_seqlens (device int32
 * [N+1], cu[0] = 0, non-decreasing, cu[N] = T_tot).
 *
 * Ownership and execution.  Every pointer except the descriptor is a DEVICE
 * pointer owned by the caller.  The library allocates no memory, never
 * synchronises the host, and launches only on the given stream (a
 * cudaStream_t passed as void*, NULL = the legacy default stream).  Results
 * are ready when that stream reaches them.  Outputs must not alias inputs,
 * except that S_final may equal S0.
 *
 * Errors.  Argument checks that the host can make return a status at once and
 * launch nothing.  Problems only the device can see (a malformed cu_seqlens, a
 * bounded wait that ran out) are written to *dev_status (device int32, may be
 * NULL; the first error sticks, 0 means no error) and the affected work is
 * skipped.  A failed launch returns KDA_ERR_CUDA.  Nothing aborts or throws.
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
    KDA_ERR_INVALID_ARG = 1, /* null / misaligned pointer, bad size, bad cu_seqlens */
    KDA_ERR_UNSUPPORTED = 2, /* shape or dtype outside what the kernels cover      */
    KDA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required         */
    KDA_ERR_CUDA = 4,        /* a CUDA launch or runtime call failed               */
    KDA_ERR_TIMEOUT = 5      /* a bounded device-side wait gave up (dev_status)    */
} kda_status_t;

typedef enum { KDA_DTYPE_F32 = 0, KDA_DTYPE_BF16 = 1 } kda_dtype_t;

/* Problem description for the chunked prefill and the transfer pass. */
typedef struct {
    int32_t num_seqs;     /* N >= 0                                               */
    int32_t total_tokens; /* T_tot >= 0, equal to cu_seqlens[N]                   */
    int32_t num_heads;    /* H >= 1                                               */
    int32_t dk;           /* key / query width, 1..128                            */
    int32_t dv;           /* value width, 1..128                                  */
    int32_t act_dtype;    /* kda_dtype_t of q, k, v and out                       */
    int32_t chunk;        /* must be 16: the 16-token block of the digest, 2.1 (1) */
    int32_t num_segments; /* 0 = choose, 1 = one pass per (seq, head), S > 1 =     */
                          /* split every sequence into S chunk-aligned segments    */
                          /* joined by the transfer-matrix scan (digest 2.4 (1))   */
} kda_prefill_desc_t;

/*
 * Number of segments kda_prefill_chunked will use for desc (resolves
 * num_segments = 0 from the problem size and the current device's SM count).
 * Returns 0 for an invalid descriptor.
 */
int32_t kda_prefill_num_segments(const kda_prefill_desc_t *desc);

/*
 * Device workspace, in bytes, that kda_prefill_chunked needs for desc: zero
 * when it runs one pass, else room for N*H*S transfer matrices, zero-initial
 * states and segment start states (fp32), for BF16 at dk = dv = 128 also a BF16
 * copy of each start state laid out as a tensor-core operand (N*H*S x 128 x 128
 * x 2 bytes), and one dk-vector per token and head in the activation dtype;
 * each piece rounded up to 256 bytes.  Call with the same desc, on the same
 * device, as the prefill itself.
 */
size_t kda_prefill_workspace_size(const kda_prefill_desc_t *desc);

/*
 * Chunked prefill (the hot path): for every packed sequence and head, run the
 * recurrence above over its tokens starting from S0 (NULL = zeros), write o_t
 * for every token to out and, if S_final != NULL, the state after the last
 * token.  Chunked form: 16-token blocks, each turned into a WY/UT-transform
 * representation of its product of (I - beta k k^T) Diag(alpha) factors
 * ("intra-chunk parallel work"), then a sequential fp32 state step per block
 * ("cross-chunk state propagation"), overlapped as in the digest, section
 * 2.4 (1), FlashKDA.  With S > 1 segments every sequence is also split for
 * parallelism (digest 2.4 (1), KCP): kda_state_transfer on all S segments with
 * outputs (the zero-start outputs go straight to out), kda_state_compose (start
 * states and S_final), then kda_prefill_combine.  A zero-length sequence gives
 * S_final = S0.
 *
 *   desc            problem description (host pointer).
 *   q, k, v, g, beta, out   device arrays in the layouts above; q, k, v, g and
 *                   out 16-byte aligned, the rest 4-byte aligned.
 *   S0              [N, H, dk, dv] fp32 or NULL.
 *   cu_seqlens      [N+1] int32 (device).
 *   S_final         [N, H, dk, dv] fp32 or NULL; may equal S0.
 *   workspace       device buffer of workspace_bytes >= kda_prefill_workspace_size
 *                   (may be NULL when that is 0).  Contents on entry don't matter.
 *   dev_status      device int32 or NULL (see Errors).
 *   stream          cudaStream_t.
 */
kda_status_t kda_prefill_chunked(const kda_prefill_desc_t *desc, const void *q, const void *k,
                                 const void *v, const float *g, const float *beta,
                                 const float *S0, const int32_t *cu_seqlens, void *out,
                                 float *S_final, void *workspace, size_t workspace_bytes,
                                 int32_t *dev_status, void *stream);

/*
 * kda_prefill_chunked with stage timing, for measurement: identical launches
 * and results, and in addition records stage_events[0] (cudaEvent_t, created by
 * the caller) on the stream before the first launch, stage_events[1] after the
 * transfer pass (or the single output pass when the split is one segment),
 * stage_events[2] after the segment scan and stage_events[3] after the last
 * launch (with one segment 1, 2 and 3 follow each other).  Recording an event
 * between two launches keeps the next kernel from starting while the previous
 * one drains, so the call can take slightly longer than kda_prefill_chunked.
 * KDA_ERR_INVALID_ARG if stage_events or one of its four entries is NULL.
 */
kda_status_t kda_prefill_chunked_timed(const kda_prefill_desc_t *desc, const void *q,
                                       const void *k, const void *v, const float *g,
                                       const float *beta, const float *S0,
                                       const int32_t *cu_seqlens, void *out, float *S_final,
                                       void *workspace, size_t workspace_bytes,
                                       int32_t *dev_status, void *const *stage_events,
                                       void *stream);

/*
 * Fused gate prologue (digest, section 2.1 (1): g = -5 sigmoid(x), so g in
 * (-5, 0)): kda_prefill_chunked from the pre-activations, so the gates and the
 * normalised q, k are never written to memory.  The kernels take
 *     g = -5 sigmoid(x_g),  beta = sigmoid(x_beta),
 *     q <- q / ||q||,  k <- k / ||k||  per (token, head) over the key channels
 * (a zero row stays zero), in fp32, then run exactly as kda_prefill_chunked.
 * q, k [T_tot, H, dk] and v [T_tot, H, dv] as there (q, k not normalised); x_g
 * [T_tot, H, dk] in the activation dtype, 16-byte aligned; x_beta [T_tot, H]
 * fp32.  BF16 activations with dk = dv = 128 only (else KDA_ERR_UNSUPPORTED);
 * workspace as kda_prefill_workspace_size(desc).  HBM traffic per head-token
 * falls from 1540 to 1284 bytes at d = 128 (x_g in BF16 instead of fp32 g).
 */
kda_status_t kda_prefill_chunked_gated(const kda_prefill_desc_t *desc, const void *q,
                                       const void *k, const void *v, const void *x_g,
                                       const float *x_beta, const float *S0,
                                       const int32_t *cu_seqlens, void *out, float *S_final,
                                       void *workspace, size_t workspace_bytes,
                                       int32_t *dev_status, void *stream);

/*
 * Sparse state checkpoints during prefill (the fixed-size state is the unit of
 * the prefix cache: digest, section 2.4 (4)).  Everything kda_prefill_chunked
 * does, and in addition, for every sequence n and k = 0, 1, ... with
 * (k+1) * ckpt_interval <= len_n, the state after its first (k+1) * ckpt_interval
 * tokens is written to
 *     ckpt_states[(base_n + k) * H * dk * dv ...]   ([K, H, dk, dv] fp32),
 * base_n = sum over m < n of floor(len_m / ckpt_interval), K = that sum over all
 * sequences (the caller sizes ckpt_states for it; a checkpoint at a sequence's
 * last token equals its S_final).  ckpt_interval must be a positive multiple of
 * 16 (the block size), ckpt_states 4-byte aligned and not aliasing any other
 * argument.  With S > 1 segments the transfer pass also keeps the transfer matrix
 * so far at each checkpoint (floor(T_tot / ckpt_interval) * H * dk * dk fp32 of
 * extra workspace) and a last kernel adds its product with the segment's start
 * state once the scan has it.  Workspace: kda_prefill_ckpt_workspace_size(desc,
 * ckpt_interval) (0 on invalid arguments).  Errors as for kda_prefill_chunked;
 * a non-positive or unaligned interval returns KDA_ERR_INVALID_ARG.
 */
size_t kda_prefill_ckpt_workspace_size(const kda_prefill_desc_t *desc, int32_t ckpt_interval);
kda_status_t kda_prefill_chunked_ckpt(const kda_prefill_desc_t *desc, const void *q,
                                      const void *k, const void *v, const float *g,
                                      const float *beta, const float *S0,
                                      const int32_t *cu_seqlens, void *out, float *S_final,
                                      int32_t ckpt_interval, float *ckpt_states, void *workspace,
                                      size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * One decode step for `batch` independent sequences (one new token each): the
 * recurrence above applied once, in place on S_inout [batch, H, dk, dv] fp32,
 * with q, k [batch, H, dk], v, out [batch, H, dv] in act_dtype, g [batch, H,
 * dk] and beta [batch, H] fp32.  Streams each state through once.  dv must be
 * a multiple of 4 and S_inout 16-byte aligned (the others 4-byte aligned).
 * dev_status (device int32 or NULL, 4-byte aligned): KDA_ERR_TIMEOUT if a
 * bounded device-side wait gave up, in which case some states may not have
 * been stepped (S_inout is then partly old, partly new).
 */
kda_status_t kda_decode_step(int32_t batch, int32_t num_heads, int32_t dk, int32_t dv,
                             int32_t act_dtype, const void *q, const void *k, const void *v,
                             const float *g, const float *beta, float *S_inout, void *out,
                             int32_t *dev_status, void *stream);

/*
 * Transfer pass of the context-parallel split (digest, section 2.4 (1)): with
 * S = desc->num_segments >= 1, split every sequence into S chunk-aligned
 * segments (sequence n has c = ceil(len_n / 16) chunks; segment s takes chunks
 * [floor(s c / S), floor((s+1) c / S))) and compute for each (n, h, s)
 *     transfer        [N, H, S, dk, dk]  the matrix A with S_end = A S_start + B
 *     zero_init_state [N, H, S, dk, dv]  B, the state the segment reaches from 0.
 * Only segments s in [seg_begin, seg_end) are computed (0 <= seg_begin <=
 * seg_end <= S); the other slots are left untouched, so ranks or passes can
 * split the segments between them.  An empty segment gives A = I, B = 0.
 *
 * Outputs (optional: q, out_zero and out_transfer all NULL, or all given):
 * since S_t = A_t start + B_t inside a segment, o_t = B_t^T q_t + start^T (A_t^T
 * q_t).  The pass then also writes, for every token of those segments,
 *     out_zero     [T_tot, H, dv]  B_t^T q_t   (the output from a zero start)
 *     out_transfer [T_tot, H, dk]  A_t^T q_t
 * in the activation dtype; kda_prefill_combine adds the second term once the
 * start states are known.
 */
kda_status_t kda_state_transfer(const kda_prefill_desc_t *desc, int32_t seg_begin,
                                int32_t seg_end, const void *q, const void *k, const void *v,
                                const float *g, const float *beta, const int32_t *cu_seqlens,
                                float *transfer, float *zero_init_state, void *out_zero,
                                void *out_transfer, int32_t *dev_status, void *stream);

/*
 * Prefix scan that joins the segments (digest, section 2.4 (1)): for each of
 * `units` independent chains of `segments` (A_s, B_s) pairs,
 *     start_0 = S0 (NULL = zeros),  start_s = A_{s-1} start_{s-1} + B_{s-1},
 * written to seg_init_states [units, segments, dk, dv] (may be NULL), and
 * S_final [units, dk, dv] = A_{S-1} start_{S-1} + B_{S-1} (may be NULL; when it
 * is NULL the last pair is never read, so it need not have been computed).
 * transfer is [units, segments, dk, dk], zero_init_state [units, segments, dk,
 * dv]; all fp32, 16-byte aligned.  The scan is sequential over segments and
 * parallel over units and column blocks, in fp32.
 *
 * start_images (may be NULL; dk = dv = 128 only, else it must be NULL):
 * [units, segments, 128 * 128] BF16, 16-byte aligned, each start state rounded
 * to BF16 and laid out as the B operand of kda_prefill_combine's tensor-core
 * product (an internal layout: only kda_prefill_combine reads it).
 *
 * dev_status (device int32 or NULL, 4-byte aligned): KDA_ERR_TIMEOUT if a
 * bounded device-side wait of the scan gave up (its outputs are then
 * incomplete).
 */
kda_status_t kda_state_compose(int32_t units, int32_t segments, int32_t dk, int32_t dv,
                               const float *transfer, const float *zero_init_state,
                               const float *S0, float *seg_init_states, float *S_final,
                               void *start_images, int32_t *dev_status, void *stream);

/*
 * Output correction of the context-parallel split: for every token t of the
 * segments s in [first_segment, S) (S = desc->num_segments),
 *     out[t, h, :] += seg_init_states[n, h, s]^T out_transfer[t, h, :]
 * with seg_init_states [N, H, S, dk, dv] fp32 (from kda_state_compose) and
 * out_transfer [T_tot, H, dk] (from kda_state_transfer) in the activation
 * dtype.  out holds the zero-start outputs on entry and the outputs on exit.
 * first_segment = 1 skips the first segments' correction when they start from
 * zeros.  A dense product per segment on tensor cores for BF16 at d = 128: with
 * start_images (the BF16 images kda_state_compose wrote for the same states,
 * 16-byte aligned) through tcgen05, and seg_init_states may then be NULL;
 * without them from the fp32 states through mma.sync.  Other shapes: fp32 on
 * CUDA cores from seg_init_states.
 */
kda_status_t kda_prefill_combine(const kda_prefill_desc_t *desc, int32_t first_segment,
                                 const float *seg_init_states, const void *start_images,
                                 const void *out_transfer, const int32_t *cu_seqlens, void *out,
                                 int32_t *dev_status, void *stream);

/*
 * Output pass of the context-parallel split: with S = desc->num_segments >= 1
 * (segments as in kda_state_transfer), run segments [seg_begin, seg_end) of
 * every (sequence, head) from their given start states seg_init_states [N, H,
 * S, dk, dv] (as written by kda_state_compose; NULL = zeros), write o_t for
 * those segments' tokens to out and, if S_final != NULL and seg_end == S, the
 * state after the last segment.  With S = 1 and seg_init_states = S0 it is the
 * one-pass prefill; with S > 1 it is the alternative to kda_prefill_combine
 * (re-running every segment from its start state instead of correcting the
 * zero-start outputs).  Arguments otherwise as for kda_prefill_chunked.
 */
kda_status_t kda_prefill_segments(const kda_prefill_desc_t *desc, int32_t seg_begin,
                                  int32_t seg_end, const void *q, const void *k, const void *v,
                                  const float *g, const float *beta,
                                  const float *seg_init_states, const int32_t *cu_seqlens,
                                  void *out, float *S_final, int32_t *dev_status, void *stream);

/* Size of the device scratch compiled into the library for
 * kda_prefill_chunked_noalloc: 64 MiB, held on every GPU that loads it. */
#define KDA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/*
 * kda_prefill_chunked for callers that cannot allocate device memory (for
 * example an inference-engine plugin that may not call cudaMalloc while it
 * enqueues work, or a host whose device memory is all owned by another
 * framework's pool).  The source pages have no counterpart to this: it is a
 * convenience of this library.
 *
 * Same arguments and results as kda_prefill_chunked, minus the workspace: the
 * segment split's workspace comes from a fixed KDA_NOALLOC_SCRATCH_BYTES array
 * inside the library, and nothing is allocated.  A problem whose workspace
 * (kda_prefill_workspace_size) exceeds that returns KDA_ERR_WORKSPACE without
 * launching anything; pass desc->num_segments = 1 (no workspace) or a smaller
 * split instead.  The first call that needs the scratch on a device looks up
 * its address there (make that first call before any stream capture).  All
 * calls on a device share the one array and leave their data in it; nothing
 * has to be cleared between calls, but calls whose GPU work overlaps (e.g. on
 * two unordered streams) race on it and give wrong results.
 */
kda_status_t kda_prefill_chunked_noalloc(const kda_prefill_desc_t *desc, const void *q,
                                         const void *k, const void *v, const float *g,
                                         const float *beta, const float *S0,
                                         const int32_t *cu_seqlens, void *out, float *S_final,
                                         int32_t *dev_status, void *stream);

/*
 * Backward pass of the prefill ("Kimi K3 Architecture Explained", section 3: the
 * per-token recurrence, differentiated).  For the same inputs as
 * kda_prefill_chunked (q, k, v, g, beta, S0, cu_seqlens; q and k as the recurrence
 * uses them, i.e. already normalised) and the adjoints d_out [T_tot, H, dv] (the
 * activation dtype) and d_S_final [N, H, dk, dv] fp32 (NULL: zero), writes the
 * gradients of <d_out, o> + <d_S_final, S_final>:
 *     dq, dk, dg  [T_tot, H, dk] fp32,   dv [T_tot, H, dv] fp32,
 *     dbeta [T_tot, H] fp32,             dS0 [N, H, dk, dv] fp32 (NULL: skipped).
 * dg is the gradient with respect to the log-decay g (alpha = e^g).  All outputs
 * are overwritten; none may alias an input.
 *
 * BF16 activations at dk = dv = 128 take the chunked form on tensor cores (the
 * 16-token blocks of the prefill): the forward chain stores the BF16 state after
 * every 32 tokens, an adjoint chain runs every segment from its last block to its
 * first and stores the adjoint at every block end (BF16), and one CTA per SM then
 * walks the (block pair, head) items, forming every block's gradients from its
 * start state (stored, or one small product away inside the pair) and its end
 * adjoint, with no atomics.  q, k, v, g and d_out must then be 16-byte aligned
 * (KDA_ERR_INVALID_ARG otherwise).  Its results follow BF16 rounding of the
 * chain's operands and of the stored states (the BF16 tolerance of the prefill
 * applies).  Workspace: 32 KB per head and 32 tokens for the states and 32 KB per
 * head and 16 tokens (plus one block per sequence) for the adjoints, about 3 KB per
 * head-token, plus 256 KB per (sequence, head, segment) when segments are used,
 * part of it shared with the states.  Other dtypes and shapes take the token-level
 * form in fp32: one CTA per (sequence, head, 32 value columns) recomputes the
 * states from a checkpoint at every 4-token block start (16 KB of workspace per
 * head-token at d = 128); dq, dk, dg and dbeta are zeroed on the stream, then
 * accumulated.
 *
 * desc->num_segments (0: the library's choice, at most 64) splits every sequence
 * into segments run in parallel: each segment's transfer matrix A, zero-start
 * state and zero-end adjoint first, then scans for every segment's start state
 * and end adjoint (the adjoint map of a segment is A^T), then the chains per
 * segment.  The library's choice gives every SM one chain (chunked form: at least
 * 4 blocks per segment) or two (token-level form).  Workspace:
 * kda_prefill_backward_workspace_size(desc) (0 on invalid arguments).  A batch
 * too long for device memory is differentiated piece by piece, last piece first:
 * each piece from its start state (S0) with d_S_final = the next piece's dS0.
 * Pointers at least 4-byte aligned; KDA_ERR_INVALID_ARG on a missing or
 * misaligned pointer, KDA_ERR_WORKSPACE on a short workspace,
 * KDA_ERR_UNSUPPORTED as kda_prefill_chunked.
 */
size_t kda_prefill_backward_workspace_size(const kda_prefill_desc_t *desc);
/* Segments per sequence the backward pass uses for desc (0 on invalid arguments). */
int32_t kda_prefill_backward_num_segments(const kda_prefill_desc_t *desc);
kda_status_t kda_prefill_backward(const kda_prefill_desc_t *desc, const void *q, const void *k,
                                  const void *v, const float *g, const float *beta,
                                  const float *S0, const int32_t *cu_seqlens, const void *d_out,
                                  const float *d_S_final, float *dq, float *dk, float *dv,
                                  float *dg, float *dbeta, float *dS0, void *workspace,
                                  size_t workspace_bytes, int32_t *dev_status, void *stream);

/* Human-readable name of a status. Never NULL. */
const char *kda_status_string(kda_status_t status);

/* Build description (target architecture, library version). Never NULL. */
const char *kda_build_info(void);

/*
 * Self-test of the bounded device-side waits: one CTA waits, with a limit of
 * about limit_us microseconds of SM clocks, on an mbarrier that nothing arrives
 * on, then records KDA_ERR_TIMEOUT in dev_status (device int32, first error
 * wins) and returns, the same path every kernel takes when a wait gives up.
 * Nothing faults and the context stays usable.  limit_us in (0, 1e7].
 */
kda_status_t kda_selftest_wait_timeout(int32_t limit_us, int32_t *dev_status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
