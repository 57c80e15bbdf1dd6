// Internal declarations shared by the libkda translation units (not installed).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// ---------------------------------------------------------------------------
// Activation load / store in fp32 registers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float act_ld(const float *p, size_t i) { return p[i]; }
__device__ __forceinline__ float act_ld(const __nv_bfloat16 *p, size_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ void act_st(float *p, size_t i, float x) { p[i] = x; }
__device__ __forceinline__ void act_st(__nv_bfloat16 *p, size_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

// First error wins; 0 means "no error yet".
__device__ __forceinline__ void dev_fail(int32_t *status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// Blocks [c0, c1) of segment s (of Sg) of a sequence of c 16-token blocks.
// lead = 0: the blocks are split evenly, segment s takes [floor(s c / Sg),
// floor((s+1) c / Sg)).  lead > 0 (a fraction of 2^16; used with Sg >= 2):
// segment 0 takes the first floor(c lead / 2^16) blocks and segments 1 .. Sg-1
// split the rest evenly.
__host__ __device__ __forceinline__ void segment_blocks(long long c, int s, int Sg, int lead,
                                                        long long &c0, long long &c1) {
    if (lead <= 0 || Sg < 2) {
        c0 = (long long)s * c / Sg;
        c1 = (long long)(s + 1) * c / Sg;
        return;
    }
    const long long cl = c * lead >> 16, rest = c - cl;
    c0 = s == 0 ? 0 : cl + (long long)(s - 1) * rest / (Sg - 1);
    c1 = cl + (long long)s * rest / (Sg - 1);
}

// Token range [t_begin, t_end) of segment s (of Sg) of sequence n, from the
// block split above (c = ceil(len / 16) blocks).  Returns false (and records
// KDA_ERR_INVALID_ARG) if cu_seqlens is malformed.
__device__ __forceinline__ bool segment_range(const int32_t *cu, int n, int N, int T_tot,
                                              int s, int Sg, int32_t *status, int &t_begin,
                                              int &t_end, int lead = 0) {
    const int a = cu[n], b = cu[n + 1];
    if (a < 0 || b < a || b > T_tot || cu[0] != 0 || cu[N] != T_tot) {
        dev_fail(status, KDA_ERR_INVALID_ARG);
        return false;
    }
    const long long len = b - a;
    long long c0, c1;
    segment_blocks((len + 15) / 16, s, Sg, lead, c0, c1);
    t_begin = a + (int)min(len, c0 * 16);
    t_end = a + (int)min(len, c1 * 16);
    return true;
}

// ---------------------------------------------------------------------------
// Chunked prefill launch description (shared by the SIMT and tensor-core paths).
// ---------------------------------------------------------------------------
enum PrefillMode { MODE_OUTPUT = 0, MODE_TRANSFER = 1 };

struct PrefillArgs {
    const void *q, *k, *v;
    const float *g, *beta;
    const float *S0;        // [N,H,dk,dv] or null                (MODE_OUTPUT)
    const float *seg_init;  // [N,H,Sg,dk,dv] start states or null (MODE_OUTPUT, Sg > 1)
    const int32_t *cu;
    void *out;
    float *S_final;         // [N,H,dk,dv] or null; written by segment Sg-1
    float *transfer;        // [N,H,Sg,dk,dk] or null               (MODE_TRANSFER)
    // MODE_TRANSFER, dk = dv = 128: if set, the identity-start chain writes its
    // transfer matrix A as two BF16 images hi = bf16(A), lo = bf16(A - hi), each
    // stored transposed ([j][i], i contiguous): [N,H,Sg][2][128][128], instead of
    // the fp32 matrix (transfer is then ignored).
    __nv_bfloat16 *transfer_img;
    float *zero_state;      // [N,H,Sg,dk,dv]                       (MODE_TRANSFER)
    // MODE_TRANSFER with emit_out: the zero-start chain writes its outputs to
    // `out` [T,H,dv], the identity-start chain writes A_t^T q_t to `aux_out`
    // [T,H,dk] (both in the activation dtype); q is then required.
    void *aux_out;
    int emit_out;
    int32_t *dev_status;
    // Sparse state checkpoints (ckpt_interval = 0: none).  After every
    // ckpt_interval tokens of a sequence (a positive multiple of 16) the state goes
    // to ckpt [K][H][dk][dv] fp32, slot ckpt_base(n) + k for the (k+1)-th
    // checkpoint of sequence n.  MODE_OUTPUT writes the true state; in
    // MODE_TRANSFER the zero-start chain writes its state to ckpt and the
    // identity-start chain its transfer matrix so far to ckpt_a [K][H][dk][dk] (if
    // set), and launch_ckpt_fixup adds ckpt_a x start_s after the scan.
    int ckpt_interval;
    float *ckpt;
    float *ckpt_a;
    // Fused gate prologue (BF16, dk = dv = 128): g points to x_g [T_tot, H, dk] in
    // the activation dtype and beta to x_beta [T_tot, H] fp32; the kernels take
    // g = -5 sigmoid(x_g), beta = sigmoid(x_beta) and q, k divided by their L2 norm
    // per (token, head) (a zero row stays zero).
    int gate;
    // Backward (BF16, dk = dv = 128).  rev: the kernel runs the adjoint chain
    // instead (blocks last to first, v is d_out; the state is the adjoint dS of
    // the state, stepping dS <- Diag(e^{Gamma_C}) dS' + Qh^T dO - Kh^T dR with
    // dR = T^T (Mq^T dO + Kb dS')); in MODE_TRANSFER it runs only the chain from a
    // zero end adjoint (written to zero_state), in MODE_OUTPUT from seg_init (or
    // S0) and S_final receives the adjoint at the start of segment 0.
    // chunk_states (if set): [slots][H][dv][dk] BF16, the state transposed (row j
    // = value column, key channels contiguous): the forward chain writes the state
    // after every 32 tokens of a sequence (every second 16-token block) to slot
    // ckpt_base(n, 32) + done / 32 - 1; the adjoint chain writes the adjoint at the
    // end of every block, before stepping through it, to slot cbase(n) + block
    // (cbase(n) = sum over m < n of ceil(len_m / 16)).
    // In rev mode the segments' arrays run in reverse order: seg_init is read and
    // zero_state written at segment index Sg - 1 - s, so that the adjoint scan
    // Y_{s-1} = A_s^T Y_s + B^_s is the ordinary forward scan over reversed
    // segments.  transfer_img_t (MODE_TRANSFER, dk = dv = 128): the identity-start
    // chain also writes the hi/lo BF16 images of A^T in the layout transfer_img
    // uses for A ([N,H,Sg][2][128][128], i.e. A row-major), at segment index
    // Sg - 1 - s, for that reversed scan.
    int rev;
    __nv_bfloat16 *chunk_states;
    __nv_bfloat16 *transfer_img_t;
    // Lead segment (one-call split prefill, tensor-core path only): segment 0 takes
    // the first lead / 2^16 of every sequence's blocks (segment_blocks) and runs
    // from S0 as an output pass inside the transfer pass: its zero-start chain
    // starts from S0 and writes the final outputs, its end state goes to
    // zero_state and zero images to transfer_img, so the scan carries the end
    // state on unchanged and the combine skips the segment.  The lead CTAs come
    // first in the grid.  0: segments of equal length.
    int lead;
    int N, T_tot, H, dk, dv;
    int Sg;                 // segments per sequence (layout and bounds)
    int seg_begin;          // segments seg_begin .. seg_begin+seg_count-1 are
    int seg_count;          // processed by this launch
    int mode;
    int act;                // kda_dtype_t
};

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel in the stream drains, so it must call
// sm100::griddep_wait() before its first global memory access.  Used for the
// kernels of the split prefill, which run back to back.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t st, Args &&...args) {
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
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current device
// once: the attribute stays set in the context, so later launches skip the
// runtime call.  Thread-safe.
cudaError_t set_max_dynamic_smem(const void *kernel, int bytes);

// First 16-token block of sequence n when every sequence's blocks are numbered
// one after another (ceil(len / 16) of them per sequence).
__device__ __forceinline__ int block_base(const int32_t *cu, int n) {
    int b = 0;
    for (int m = 0; m < n; ++m) b += (cu[m + 1] - cu[m] + 15) / 16;
    return b;
}

// Slot of sequence n's first checkpoint: checkpoints of earlier sequences come
// first, floor(len / interval) of them per sequence.
__device__ __forceinline__ int ckpt_base(const int32_t *cu, int n, int interval) {
    int b = 0;
    for (int m = 0; m < n; ++m) b += (cu[m + 1] - cu[m]) / interval;
    return b;
}

// Launchers (return a cudaError_t from the launch).
cudaError_t launch_prefill_simt(const PrefillArgs &a, cudaStream_t st);
bool prefill_tc_supported(const PrefillArgs &a);
// Whether the tensor-core transfer pass runs both chains of a segment in one CTA.
bool prefill_tc_two_chain(const PrefillArgs &a);
cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t st);
// A (fp32) or, for BF16 at dk = dv = 128, a_img (the transfer pass's hi/lo
// images) gives the transfer matrices; exactly one of them is non-null.
cudaError_t launch_compose(int units, int Sg, int dk, int dv, const float *A,
                           const __nv_bfloat16 *a_img, const float *B, const float *S0,
                           float *seg_init, float *S_final, __nv_bfloat16 *start_img,
                           int32_t *dev_status, cudaStream_t st);
// Split path with checkpoints: ckpt[k] += ckpt_a[k] x start_s for every checkpoint
// k of every segment s with a nonzero start state (start_0 = S0, start_s for s >= 1
// from `starts` [N,H,Sg,dk,dv] written by the scan); max_ckpt bounds the number of
// checkpoints (floor(T_tot / ckpt_interval)).
cudaError_t launch_ckpt_fixup(const PrefillArgs &a, const float *S0, const float *starts,
                              int max_ckpt, cudaStream_t st);

// Backward pass (kda_backward.cu): workspace bytes, and the launch (zeroes the
// accumulated outputs on st first).
// Sg > 1 splits every sequence into Sg segments (pre-pass, scans, main pass).
size_t backward_workspace_bytes(int N, int T_tot, int H, int dk, int dv, int Sg);
cudaError_t launch_backward(const PrefillArgs &p, const void *dout, const float *dSF, float *dq,
                            float *dk, float *dv, float *dg, float *dbeta, float *dS0, int Sg,
                            void *workspace, cudaStream_t st);
// Chunked backward for BF16 activations at dk = dv = 128 (16-byte aligned rows):
// its workspace, the whole backward, and its last kernel (the per-block
// gradients from the forward states and adjoints at every block end).
size_t backward_chunked_workspace_bytes(int N, int T_tot, int H, int Sg);
cudaError_t launch_backward_chunked(const PrefillArgs &p, const void *dout, const float *dSF,
                                    float *dq, float *dk, float *dv, float *dg, float *dbeta,
                                    float *dS0, int Sg, void *workspace, cudaStream_t st);
cudaError_t launch_bwd_chunk(const PrefillArgs &p, const void *dout,
                             const __nv_bfloat16 *fwd_states, const __nv_bfloat16 *adj_states,
                             float *dq, float *dk, float *dv, float *dg, float *dbeta,
                             cudaStream_t st);
bool decode_tma_supported(int dk, int dv);
// dev_status (nullable) receives KDA_ERR_TIMEOUT if a bounded wait gives up.
cudaError_t launch_decode_tma(int batch, int H, int act, const void *q, const void *k,
                              const void *v, const float *g, const float *beta, float *S,
                              void *out, int32_t *dev_status, cudaStream_t st);
cudaError_t launch_combine(const PrefillArgs &a, const float *starts, const void *aux_out,
                           const __nv_bfloat16 *start_img, cudaStream_t st);
// True when launch_combine with these arguments reads only the start images (its
// tcgen05 path), so the fp32 start states need not be written.
bool combine_uses_images(const PrefillArgs &a, const void *aux_out,
                         const __nv_bfloat16 *start_img);

// BF16 image of a 128 x 128 start state as the B operand of a tensor-core
// product over its 128 key channels i (N = 128 columns j, K = 128 rows i),
// in the canonical K-major layout without swizzle: 8 x 8 core matrices of 128
// contiguous bytes (8 rows j of 16 bytes, 8 consecutive i each), core matrices
// adjacent along K (i) 2048 bytes apart, adjacent along N (j) 128 bytes apart.
// Element index of (j, i) within one image of 16384 elements:
__host__ __device__ constexpr int start_img_index(int j, int i) {
    return (i >> 3) * 1024 + (j >> 3) * 64 + (j & 7) * 8 + (i & 7);
}
constexpr int kStartImgElems = 128 * 128;
cudaError_t launch_decode(int batch, int H, int dk, int dv, int act, const void *q,
                          const void *k, const void *v, const float *g, const float *beta,
                          float *S, void *out, cudaStream_t st);

}  // namespace kda
