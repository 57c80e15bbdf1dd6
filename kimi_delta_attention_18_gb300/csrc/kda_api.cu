// C ABI of libkda: host-side argument checks, segment planning and dispatch.
// Nothing here allocates device memory or synchronises the host.
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "kda_internal.cuh"

namespace {

using namespace kda;

constexpr int kMaxDim = 128;
constexpr int kMaxSegments = 4096;

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
bool aligned4(const void *p) { return ((uintptr_t)p & 3u) == 0; }

kda_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA; }

kda_status_t check_desc(const kda_prefill_desc_t *d) {
    if (!d) return KDA_ERR_INVALID_ARG;
    if (d->num_seqs < 0 || d->total_tokens < 0 || d->num_heads < 1) return KDA_ERR_INVALID_ARG;
    if (d->dk < 1 || d->dv < 1 || d->num_segments < 0) return KDA_ERR_INVALID_ARG;
    if (d->chunk != 16) return KDA_ERR_UNSUPPORTED;
    if (d->act_dtype != KDA_DTYPE_F32 && d->act_dtype != KDA_DTYPE_BF16) return KDA_ERR_UNSUPPORTED;
    if (d->dk > kMaxDim || d->dv > kMaxDim) return KDA_ERR_UNSUPPORTED;
    if (d->num_segments > kMaxSegments) return KDA_ERR_UNSUPPORTED;
    // Every index the kernels form must fit the int/size_t arithmetic they use:
    // element offsets in 64 bits, and the (sequence, head, segment) unit count
    // (a grid dimension, formed in int) below 2^31.
    if ((long long)d->total_tokens * d->num_heads * (d->dk > d->dv ? d->dk : d->dv) >
        (1ll << 40))
        return KDA_ERR_UNSUPPORTED;
    const long long segs = d->num_segments > 0 ? d->num_segments : 64;
    if ((long long)d->num_seqs * d->num_heads * segs > 0x7fffffffll) return KDA_ERR_UNSUPPORTED;
    return KDA_OK;
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 148;
    return n;
}

PrefillArgs base_args(const kda_prefill_desc_t *d) {
    PrefillArgs a;
    memset(&a, 0, sizeof(a));
    a.N = d->num_seqs;
    a.T_tot = d->total_tokens;
    a.H = d->num_heads;
    a.dk = d->dk;
    a.dv = d->dv;
    a.act = d->act_dtype;
    return a;
}

// Segments per sequence when the caller leaves the choice to the library.
// Every (sequence, head) chain is sequential over its 16-token blocks, so with
// fewer chains than SMs the sequences are split.  The choice minimises a cost
// model in units of one block step of one CTA (one CTA per SM):
//   transfer pass : ceil(2 chains x S / SMs) waves x ceil(blocks / S)
//   scan          : S steps, each ~1.8 block steps
//   combine       : a dense correction, ~2 block steps
//   + ~4 block steps per extra launch;   S = 1: blocks (the longest chain)
// using the mean sequence length (the lengths live on the device).
int choose_segments(const kda_prefill_desc_t *d) {
    if (d->num_segments > 0) return d->num_segments;
    const long long chains = (long long)d->num_seqs * d->num_heads;
    if (chains == 0) return 1;
    const long long sms = sm_count();
    if (chains >= sms) return 1;
    const long long blocks = ((long long)d->total_tokens / d->num_seqs + 15) / 16;
    double best = (double)blocks;
    int best_s = 1;
    for (int S = 2; S <= 64 && S <= blocks; ++S) {
        const long long per = (blocks + S - 1) / S;
        const double cost =
            (double)((2 * chains * S + sms - 1) / sms) * per + 1.8 * S + 2.0 + 8.0;
        if (cost < best) {
            best = cost;
            best_s = S;
        }
    }
    return best_s;
}

// Segments per sequence of the backward pass (desc->num_segments, or the
// library's choice for 0).  Every (sequence, head, 32 value columns) unit of the
// backward is a token-sequential chain and its gradient pass runs two CTAs per
// SM; with fewer units than that the sequences are split (at least ~256 tokens
// per segment on average, at most 64 segments).
int backward_segments(const kda_prefill_desc_t *d) {
    if (d->num_segments > 0) return d->num_segments < 64 ? d->num_segments : 64;
    const long long units = (long long)d->num_seqs * d->num_heads * ((d->dv + 31) / 32);
    const int slots = 2 * sm_count();
    if (units <= 0 || units >= slots) return 1;
    long long sg = slots / units;
    const long long per_seq = d->num_seqs > 0 ? d->total_tokens / d->num_seqs : 0;
    const long long cap = per_seq / 256 > 1 ? per_seq / 256 : 1;
    if (sg > cap) sg = cap;
    if (sg > 64) sg = 64;
    return sg < 1 ? 1 : (int)sg;
}

// BF16 at dk = dv = 128: the chunked tensor-core backward (16-byte aligned rows);
// otherwise the token-level fp32 one.
bool backward_chunked(const kda_prefill_desc_t *d) {
    return d->act_dtype == KDA_DTYPE_BF16 && d->dk == 128 && d->dv == 128;
}
// Segments per sequence of the chunked backward.  It runs four sequential passes
// (transfer pass, zero-end adjoint pass, forward and adjoint passes from the
// scanned states) around two cheap tensor-core scans, so it splits further than
// the forward: the fewest segments that give every SM a one-chain CTA, with at
// least 4 blocks of 16 tokens per segment (mean length) and at most 64.
int backward_chunked_segments(const kda_prefill_desc_t *d) {
    if (d->num_segments > 0) return d->num_segments;
    const long long chains = (long long)d->num_seqs * d->num_heads;
    const long long sms = sm_count();
    if (chains == 0 || chains >= sms) return 1;
    long long S = (sms + chains - 1) / chains;
    const long long blocks = ((long long)d->total_tokens / d->num_seqs + 15) / 16;
    if (S > blocks / 4) S = blocks / 4;
    if (S > 64) S = 64;
    return S < 1 ? 1 : (int)S;
}

size_t act_bytes(const kda_prefill_desc_t *d) { return d->act_dtype == KDA_DTYPE_BF16 ? 2 : 4; }

// Split workspace: transfer matrices, zero-initial states and start states for
// every (sequence, head, segment) in fp32; for BF16 at dk = dv = 128 also each
// start state's BF16 operand image (kStartImgElems elements) for the tensor-core
// combine; then A_t^T q_t for every token (activation dtype).  Each piece
// starts on a 256-byte boundary.
size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }
bool wants_start_img(const kda_prefill_desc_t *d) {
    return d->act_dtype == KDA_DTYPE_BF16 && d->dk == 128 && d->dv == 128;
}
size_t states_bytes_for(const kda_prefill_desc_t *d, int Sg) {
    const size_t units = (size_t)d->num_seqs * d->num_heads * Sg;
    return round256(units * ((size_t)d->dk * d->dk + 2 * (size_t)d->dk * d->dv) * sizeof(float));
}
size_t img_bytes_for(const kda_prefill_desc_t *d, int Sg) {
    if (!wants_start_img(d)) return 0;
    return round256((size_t)d->num_seqs * d->num_heads * Sg * kStartImgElems * 2);
}
size_t workspace_bytes_for(const kda_prefill_desc_t *d, int Sg) {
    if (Sg <= 1) return 0;
    const size_t aux = round256((size_t)d->total_tokens * d->num_heads * d->dk * act_bytes(d));
    return states_bytes_for(d, Sg) + img_bytes_for(d, Sg) + aux;
}
// Checkpoints on the split path: at most floor(T_tot / interval) of them; each
// holds the identity-start chain's transfer matrix so far (dk x dk fp32 per head).
int max_checkpoints(const kda_prefill_desc_t *d, int interval) {
    return interval > 0 ? d->total_tokens / interval : 0;
}
size_t ckpt_scratch_bytes(const kda_prefill_desc_t *d, int Sg, int interval) {
    if (Sg <= 1 || interval <= 0) return 0;
    return round256((size_t)max_checkpoints(d, interval) * d->num_heads * d->dk * d->dk *
                    sizeof(float));
}

}  // namespace

cudaError_t kda::set_max_dynamic_smem(const void *kernel, int bytes) {
    struct Entry {
        const void *kernel;
        int device, bytes;
    };
    static std::mutex mu;
    static std::vector<Entry> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry &x : done)
        if (x.kernel == kernel && x.device == dev && x.bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.push_back({kernel, dev, bytes});
    return e;
}

namespace {

cudaError_t run_prefill_pass(const PrefillArgs &a, cudaStream_t st) {
    if (prefill_tc_supported(a)) return launch_prefill_tc(a, st);
    return launch_prefill_simt(a, st);
}

}  // namespace

extern "C" {

int32_t kda_prefill_num_segments(const kda_prefill_desc_t *desc) {
    if (check_desc(desc) != KDA_OK) return 0;
    return choose_segments(desc);
}

size_t kda_prefill_workspace_size(const kda_prefill_desc_t *desc) {
    if (check_desc(desc) != KDA_OK) return 0;
    return workspace_bytes_for(desc, choose_segments(desc));
}

}  // extern "C"

namespace {

// The one-call prefill, optionally with sparse state checkpoints (interval 0:
// none).
// Lead segment of the one-call split (see PrefillArgs::lead): with fewer chains
// (sequence, head) than SMs, every chain's first segment, whose start state S0 is
// known, runs as an output pass on an SM of its own while the remaining SMs run
// the transfer pass of the other segments, each of which costs both chains and
// a share of the combine.  The lead fraction f balances the two: f c1 = (1 - f)
// u c2 / (P - u) for u chains on P SMs, c1 the time of a 16-token block of a lead
// chain and c2 that of a block of the transfer pass's two chains together
// (measured on GB300, 56 heads x 256K tokens: c1 = 1.00 us, c2 = 1.57 us; with the
// fused gate prologue, whose heavier prep bounds the lead chain, c1 = 1.37 us,
// c2 = 1.89 us).  Only the tensor-core two-chain transfer pass supports it; 0
// elsewhere.
int lead_fraction(const PrefillArgs &t) {
    if (t.Sg < 2 || !prefill_tc_supported(t) || !prefill_tc_two_chain(t)) return 0;
    const double u = (double)t.N * t.H, P = (double)sm_count(), r = t.gate ? 1.38 : 1.57;
    if (u >= P) return 0;
    const double f = u * r / ((P - u) + u * r);
    return (int)(f * 65536.0);
}

kda_status_t prefill_one_call(const kda_prefill_desc_t *desc, const void *q, const void *k,
                              const void *v, const float *g, const float *beta, const float *S0,
                              const int32_t *cu_seqlens, void *out, float *S_final,
                              int32_t ckpt_interval, float *ckpt, void *workspace,
                              size_t workspace_bytes, int32_t *dev_status, void *stream,
                              int gate = 0, const cudaEvent_t *ev = nullptr) {
    kda_status_t rc = check_desc(desc);
    if (rc != KDA_OK) return rc;
    // the fused gate prologue runs in the tensor-core kernels only
    if (gate && !(desc->act_dtype == KDA_DTYPE_BF16 && desc->dk == 128 && desc->dv == 128))
        return KDA_ERR_UNSUPPORTED;
    if (desc->num_seqs == 0) return KDA_OK;
    if (!cu_seqlens) return KDA_ERR_INVALID_ARG;
    if (desc->total_tokens > 0 && (!q || !k || !v || !g || !beta || !out))
        return KDA_ERR_INVALID_ARG;
    // Row-wise bulk copies and vector stores need 16-byte bases; the rest is read
    // element by element.
    const void *rows[] = {q, k, v, g, out};
    for (const void *p : rows)
        if (p && !aligned16(p)) return KDA_ERR_INVALID_ARG;
    const void *elems[] = {beta, S0, S_final, cu_seqlens};
    for (const void *p : elems)
        if (p && !aligned4(p)) return KDA_ERR_INVALID_ARG;
    if (ckpt_interval < 0 || ckpt_interval % 16 != 0) return KDA_ERR_INVALID_ARG;
    if (ckpt_interval > 0 && (!ckpt || !aligned4(ckpt))) return KDA_ERR_INVALID_ARG;
    const int Sg = choose_segments(desc);
    const size_t need = workspace_bytes_for(desc, Sg) + ckpt_scratch_bytes(desc, Sg, ckpt_interval);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace)))
        return KDA_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;

    PrefillArgs a = base_args(desc);
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.cu = cu_seqlens;
    a.out = out; a.S_final = S_final; a.dev_status = dev_status;
    a.Sg = Sg;
    a.ckpt_interval = ckpt_interval;
    a.ckpt = ckpt_interval > 0 ? ckpt : nullptr;
    a.gate = gate;

    // ev (measurement only): ev[0] before the first launch, ev[1] after the
    // transfer pass (or the single pass), ev[2] after the scan, ev[3] at the end.
    auto mark = [&](int i) {
        return ev ? cudaEventRecord(ev[i], st) : cudaSuccess;
    };
    if (mark(0) != cudaSuccess) return KDA_ERR_CUDA;
    if (Sg == 1) {
        a.S0 = S0;
        a.seg_count = 1;
        a.mode = MODE_OUTPUT;
        cudaError_t e = run_prefill_pass(a, st);
        if (e != cudaSuccess) return KDA_ERR_CUDA;
        for (int i = 1; i < 4; ++i)
            if (mark(i) != cudaSuccess) return KDA_ERR_CUDA;
        return KDA_OK;
    }

    // Context-parallel split: the transfer pass runs every segment twice (from
    // the identity and from zeros), writing the zero-start outputs into out and
    // A_t^T q_t into the workspace; the scan joins the segments (and gives the
    // final state); the combine adds start_s^T (A_t^T q_t) to every output.
    const size_t units = (size_t)desc->num_seqs * desc->num_heads;
    float *A = (float *)workspace;
    float *B = A + units * Sg * desc->dk * desc->dk;
    float *starts = B + units * Sg * desc->dk * desc->dv;
    __nv_bfloat16 *img = wants_start_img(desc)
                             ? (__nv_bfloat16 *)((uint8_t *)workspace + states_bytes_for(desc, Sg))
                             : nullptr;
    void *aux = (uint8_t *)workspace + states_bytes_for(desc, Sg) + img_bytes_for(desc, Sg);

    PrefillArgs t = a;
    t.mode = MODE_TRANSFER;
    t.seg_begin = 0;
    t.seg_count = Sg;
    // BF16 at d = 128: A goes to the scan as hi/lo BF16 images (the same bytes)
    __nv_bfloat16 *a_img = wants_start_img(desc) ? (__nv_bfloat16 *)A : nullptr;
    t.transfer = a_img ? nullptr : A;
    t.transfer_img = a_img;
    t.zero_state = B;
    t.emit_out = 1;
    t.aux_out = aux;
    t.S_final = nullptr;
    t.lead = lead_fraction(t);
    if (t.lead) t.S0 = S0;  // the lead segment's zero-start chain starts from S0
    if (ckpt_interval > 0)  // partial transfer matrices at the checkpoints
        t.ckpt_a = (float *)((uint8_t *)workspace + workspace_bytes_for(desc, Sg));
    cudaError_t e = run_prefill_pass(t, st);
    if (e != cudaSuccess || mark(1) != cudaSuccess) return KDA_ERR_CUDA;
    PrefillArgs c = a;
    // from zeros (or run from S0 as the lead) the first segment needs no correction
    c.seg_begin = S0 && !t.lead ? 0 : 1;
    c.lead = t.lead;
    c.ckpt_interval = 0;
    // the tcgen05 combine reads the start states' BF16 images only: the scan then
    // skips the fp32 copies (unless checkpoints need them)
    float *starts_f32 =
        combine_uses_images(c, aux, img) && ckpt_interval == 0 ? nullptr : starts;
    e = launch_compose((int)units, Sg, desc->dk, desc->dv, a_img ? nullptr : A, a_img, B, S0,
                       starts_f32, S_final, img, dev_status, st);
    if (e != cudaSuccess || mark(2) != cudaSuccess) return KDA_ERR_CUDA;
    e = launch_combine(c, starts, aux, img, st);
    if (e == cudaSuccess && ckpt_interval > 0)
        e = launch_ckpt_fixup(t, S0, starts, max_checkpoints(desc, ckpt_interval), st);
    if (e != cudaSuccess || mark(3) != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
}

}  // namespace

extern "C" {

kda_status_t kda_prefill_chunked(const kda_prefill_desc_t *desc, const void *q, const void *k,
                                 const void *v, const float *g, const float *beta,
                                 const float *S0, const int32_t *cu_seqlens, void *out,
                                 float *S_final, void *workspace, size_t workspace_bytes,
                                 int32_t *dev_status, void *stream) {
    return prefill_one_call(desc, q, k, v, g, beta, S0, cu_seqlens, out, S_final, 0, nullptr,
                            workspace, workspace_bytes, dev_status, stream);
}

kda_status_t kda_prefill_chunked_timed(const kda_prefill_desc_t *desc, const void *q,
                                       const void *k, const void *v, const float *g,
                                       const float *beta, const float *S0,
                                       const int32_t *cu_seqlens, void *out, float *S_final,
                                       void *workspace, size_t workspace_bytes,
                                       int32_t *dev_status, void *const *stage_events,
                                       void *stream) {
    if (!stage_events) return KDA_ERR_INVALID_ARG;
    for (int i = 0; i < 4; ++i)
        if (!stage_events[i]) return KDA_ERR_INVALID_ARG;
    return prefill_one_call(desc, q, k, v, g, beta, S0, cu_seqlens, out, S_final, 0, nullptr,
                            workspace, workspace_bytes, dev_status, stream, 0,
                            (const cudaEvent_t *)stage_events);
}

kda_status_t kda_prefill_chunked_gated(const kda_prefill_desc_t *desc, const void *q,
                                       const void *k, const void *v, const void *x_g,
                                       const float *x_beta, const float *S0,
                                       const int32_t *cu_seqlens, void *out, float *S_final,
                                       void *workspace, size_t workspace_bytes,
                                       int32_t *dev_status, void *stream) {
    return prefill_one_call(desc, q, k, v, (const float *)x_g, x_beta, S0, cu_seqlens, out,
                            S_final, 0, nullptr, workspace, workspace_bytes, dev_status, stream,
                            1);
}

size_t kda_prefill_ckpt_workspace_size(const kda_prefill_desc_t *desc, int32_t ckpt_interval) {
    if (check_desc(desc) != KDA_OK || ckpt_interval < 0 || ckpt_interval % 16 != 0) return 0;
    const int Sg = choose_segments(desc);
    return workspace_bytes_for(desc, Sg) + ckpt_scratch_bytes(desc, Sg, ckpt_interval);
}

kda_status_t kda_prefill_chunked_ckpt(const kda_prefill_desc_t *desc, const void *q,
                                      const void *k, const void *v, const float *g,
                                      const float *beta, const float *S0,
                                      const int32_t *cu_seqlens, void *out, float *S_final,
                                      int32_t ckpt_interval, float *ckpt_states, void *workspace,
                                      size_t workspace_bytes, int32_t *dev_status, void *stream) {
    if (ckpt_interval <= 0) return KDA_ERR_INVALID_ARG;
    return prefill_one_call(desc, q, k, v, g, beta, S0, cu_seqlens, out, S_final, ckpt_interval,
                            ckpt_states, workspace, workspace_bytes, dev_status, stream);
}

size_t kda_prefill_backward_workspace_size(const kda_prefill_desc_t *desc) {
    if (check_desc(desc) != KDA_OK) return 0;
    if (backward_chunked(desc))
        return backward_chunked_workspace_bytes(desc->num_seqs, desc->total_tokens,
                                                desc->num_heads, backward_chunked_segments(desc));
    return backward_workspace_bytes(desc->num_seqs, desc->total_tokens, desc->num_heads, desc->dk,
                                    desc->dv, backward_segments(desc));
}

int32_t kda_prefill_backward_num_segments(const kda_prefill_desc_t *desc) {
    if (check_desc(desc) != KDA_OK) return 0;
    return backward_chunked(desc) ? backward_chunked_segments(desc) : backward_segments(desc);
}

kda_status_t kda_prefill_backward(const kda_prefill_desc_t *desc, const void *q, const void *k,
                                  const void *v, const float *g, const float *beta,
                                  const float *S0, const int32_t *cu_seqlens, const void *d_out,
                                  const float *d_S_final, float *dq, float *dk, float *dv,
                                  float *dg, float *dbeta, float *dS0, void *workspace,
                                  size_t workspace_bytes, int32_t *dev_status, void *stream) {
    kda_status_t rc = check_desc(desc);
    if (rc != KDA_OK) return rc;
    if (desc->num_seqs == 0) return KDA_OK;
    if (!cu_seqlens) return KDA_ERR_INVALID_ARG;
    if (desc->total_tokens > 0 &&
        (!q || !k || !v || !g || !beta || !d_out || !dq || !dk || !dv || !dg || !dbeta))
        return KDA_ERR_INVALID_ARG;
    const void *ptrs[] = {q, k, v, g, beta, S0, cu_seqlens, d_out, d_S_final,
                          dq, dk, dv, dg, dbeta, dS0};
    for (const void *p : ptrs)
        if (p && !aligned4(p)) return KDA_ERR_INVALID_ARG;
    if (backward_chunked(desc)) {
        // rows move as 16-byte pieces and tensor-map boxes
        const void *rows[] = {q, k, v, g, d_out};
        for (const void *p : rows)
            if (desc->total_tokens > 0 && !aligned16(p)) return KDA_ERR_INVALID_ARG;
        const int Sg = backward_chunked_segments(desc);
        const size_t need = backward_chunked_workspace_bytes(desc->num_seqs, desc->total_tokens,
                                                             desc->num_heads, Sg);
        if (!workspace || workspace_bytes < need || !aligned16(workspace)) return KDA_ERR_WORKSPACE;
        PrefillArgs a = base_args(desc);
        a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.S0 = S0; a.cu = cu_seqlens;
        a.dev_status = dev_status;
        return from_cuda(launch_backward_chunked(a, d_out, d_S_final, dq, dk, dv, dg, dbeta, dS0,
                                                 Sg, workspace, (cudaStream_t)stream));
    }
    const int Sg = backward_segments(desc);
    const size_t need = backward_workspace_bytes(desc->num_seqs, desc->total_tokens,
                                                 desc->num_heads, desc->dk, desc->dv, Sg);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return KDA_ERR_WORKSPACE;
    PrefillArgs a = base_args(desc);
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.S0 = S0; a.cu = cu_seqlens;
    a.dev_status = dev_status;
    return from_cuda(launch_backward(a, d_out, d_S_final, dq, dk, dv, dg, dbeta, dS0, Sg,
                                     workspace, (cudaStream_t)stream));
}

kda_status_t kda_prefill_segments(const kda_prefill_desc_t *desc, int32_t seg_begin,
                                  int32_t seg_end, const void *q, const void *k, const void *v,
                                  const float *g, const float *beta,
                                  const float *seg_init_states, const int32_t *cu_seqlens,
                                  void *out, float *S_final, int32_t *dev_status, void *stream) {
    kda_status_t rc = check_desc(desc);
    if (rc != KDA_OK) return rc;
    if (desc->num_segments < 1) return KDA_ERR_INVALID_ARG;
    if (seg_begin < 0 || seg_end < seg_begin || seg_end > desc->num_segments)
        return KDA_ERR_INVALID_ARG;
    if (seg_end == seg_begin) return KDA_OK;
    if (desc->num_seqs == 0) return KDA_OK;
    if (!cu_seqlens) return KDA_ERR_INVALID_ARG;
    if (desc->total_tokens > 0 && (!q || !k || !v || !g || !beta || !out))
        return KDA_ERR_INVALID_ARG;
    const void *rows[] = {q, k, v, g, out};
    for (const void *p : rows)
        if (p && !aligned16(p)) return KDA_ERR_INVALID_ARG;
    const void *elems[] = {beta, seg_init_states, S_final, cu_seqlens};
    for (const void *p : elems)
        if (p && !aligned4(p)) return KDA_ERR_INVALID_ARG;
    PrefillArgs a = base_args(desc);
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.cu = cu_seqlens;
    a.out = out; a.S_final = S_final; a.dev_status = dev_status;
    a.Sg = desc->num_segments;
    a.seg_begin = seg_begin;
    a.seg_count = seg_end - seg_begin;
    a.mode = MODE_OUTPUT;
    a.seg_init = seg_init_states;
    return from_cuda(run_prefill_pass(a, (cudaStream_t)stream));
}

kda_status_t kda_prefill_combine(const kda_prefill_desc_t *desc, int32_t first_segment,
                                 const float *seg_init_states, const void *start_images,
                                 const void *out_transfer, const int32_t *cu_seqlens, void *out,
                                 int32_t *dev_status, void *stream) {
    kda_status_t rc = check_desc(desc);
    if (rc != KDA_OK) return rc;
    if (desc->num_segments < 1 || first_segment < 0) return KDA_ERR_INVALID_ARG;
    if (start_images && !wants_start_img(desc)) return KDA_ERR_INVALID_ARG;
    if (desc->num_seqs == 0 || desc->total_tokens == 0 || first_segment >= desc->num_segments)
        return KDA_OK;
    if ((!seg_init_states && !start_images) || !out_transfer || !cu_seqlens || !out)
        return KDA_ERR_INVALID_ARG;
    if ((seg_init_states && !aligned16(seg_init_states)) ||
        (start_images && !aligned16(start_images)) || !aligned16(out_transfer) ||
        !aligned16(out) || !aligned4(cu_seqlens))
        return KDA_ERR_INVALID_ARG;
    PrefillArgs c = base_args(desc);
    c.cu = cu_seqlens;
    c.out = out;
    c.dev_status = dev_status;
    c.Sg = desc->num_segments;
    c.seg_begin = first_segment;
    return from_cuda(launch_combine(c, seg_init_states, out_transfer,
                                    (const __nv_bfloat16 *)start_images, (cudaStream_t)stream));
}

kda_status_t kda_decode_step(int32_t batch, int32_t num_heads, int32_t dk, int32_t dv,
                             int32_t act_dtype, const void *q, const void *k, const void *v,
                             const float *g, const float *beta, float *S_inout, void *out,
                             int32_t *dev_status, void *stream) {
    if (batch < 0 || num_heads < 1 || dk < 1 || dv < 1) return KDA_ERR_INVALID_ARG;
    if (act_dtype != KDA_DTYPE_F32 && act_dtype != KDA_DTYPE_BF16) return KDA_ERR_UNSUPPORTED;
    if (dk > kMaxDim || dv > kMaxDim || (dv & 3) != 0) return KDA_ERR_UNSUPPORTED;
    if ((long long)batch * num_heads > 0x7fffffffll) return KDA_ERR_UNSUPPORTED;
    if (batch == 0) return KDA_OK;
    // The state is streamed as float4; everything else is read element by element.
    const uintptr_t act_align = act_dtype == KDA_DTYPE_BF16 ? 2u : 4u;
    const void *acts[] = {q, k, v, out};
    for (const void *p : acts)
        if (!p || ((uintptr_t)p & (act_align - 1u)) != 0) return KDA_ERR_INVALID_ARG;
    if (!g || !beta || !aligned4(g) || !aligned4(beta)) return KDA_ERR_INVALID_ARG;
    if (!S_inout || !aligned16(S_inout)) return KDA_ERR_INVALID_ARG;
    if (dev_status && !aligned4(dev_status)) return KDA_ERR_INVALID_ARG;
    // dk = dv = 128 with 16-byte aligned rows: the TMA-streamed kernel; otherwise the
    // register-streamed one.
    if (decode_tma_supported(dk, dv) && aligned16(q) && aligned16(k) && aligned16(v) &&
        aligned16(g))
        return from_cuda(launch_decode_tma(batch, num_heads, act_dtype, q, k, v, g, beta,
                                           S_inout, out, dev_status, (cudaStream_t)stream));
    return from_cuda(launch_decode(batch, num_heads, dk, dv, act_dtype, q, k, v, g, beta,
                                   S_inout, out, (cudaStream_t)stream));
}

kda_status_t kda_state_transfer(const kda_prefill_desc_t *desc, int32_t seg_begin,
                                int32_t seg_end, const void *q, const void *k, const void *v,
                                const float *g, const float *beta, const int32_t *cu_seqlens,
                                float *transfer, float *zero_init_state, void *out_zero,
                                void *out_transfer, int32_t *dev_status, void *stream) {
    kda_status_t rc = check_desc(desc);
    if (rc != KDA_OK) return rc;
    if (desc->num_segments < 1) return KDA_ERR_INVALID_ARG;
    if (seg_begin < 0 || seg_end < seg_begin || seg_end > desc->num_segments)
        return KDA_ERR_INVALID_ARG;
    if (seg_end == seg_begin) return KDA_OK;
    if (desc->num_seqs == 0) return KDA_OK;
    if (!cu_seqlens || !transfer || !zero_init_state) return KDA_ERR_INVALID_ARG;
    if (desc->total_tokens > 0 && (!k || !v || !g || !beta)) return KDA_ERR_INVALID_ARG;
    const bool outputs = q || out_zero || out_transfer;
    if (outputs && (!q || !out_zero || !out_transfer)) return KDA_ERR_INVALID_ARG;
    const void *rows[] = {q, k, v, g, out_zero, out_transfer};
    for (const void *p : rows)
        if (p && !aligned16(p)) return KDA_ERR_INVALID_ARG;
    const void *elems[] = {beta, cu_seqlens, transfer, zero_init_state};
    for (const void *p : elems)
        if (p && !aligned4(p)) return KDA_ERR_INVALID_ARG;
    PrefillArgs t = base_args(desc);
    t.q = q;
    t.out = out_zero;
    t.aux_out = out_transfer;
    t.emit_out = outputs ? 1 : 0;
    t.k = k; t.v = v; t.g = g; t.beta = beta; t.cu = cu_seqlens; t.dev_status = dev_status;
    t.Sg = desc->num_segments;
    t.seg_begin = seg_begin;
    t.seg_count = seg_end - seg_begin;
    t.mode = MODE_TRANSFER;
    t.transfer = transfer;
    t.zero_state = zero_init_state;
    return from_cuda(run_prefill_pass(t, (cudaStream_t)stream));
}

kda_status_t kda_state_compose(int32_t units, int32_t segments, int32_t dk, int32_t dv,
                               const float *transfer, const float *zero_init_state,
                               const float *S0, float *seg_init_states, float *S_final,
                               void *start_images, int32_t *dev_status, void *stream) {
    if (units < 0 || segments < 1 || dk < 1 || dv < 1) return KDA_ERR_INVALID_ARG;
    if (dk > kMaxDim || dv > kMaxDim) return KDA_ERR_UNSUPPORTED;
    if (start_images && (dk != 128 || dv != 128)) return KDA_ERR_INVALID_ARG;
    if (units == 0) return KDA_OK;
    if (!transfer || !zero_init_state) return KDA_ERR_INVALID_ARG;
    const void *ptrs[] = {transfer, zero_init_state, S0, seg_init_states, S_final, start_images};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return KDA_ERR_INVALID_ARG;
    if (dev_status && !aligned4(dev_status)) return KDA_ERR_INVALID_ARG;
    return from_cuda(launch_compose(units, segments, dk, dv, transfer, nullptr, zero_init_state,
                                    S0, seg_init_states, S_final, (__nv_bfloat16 *)start_images,
                                    dev_status, (cudaStream_t)stream));
}

const char *kda_status_string(kda_status_t s) {
    switch (s) {
        case KDA_OK: return "ok";
        case KDA_ERR_INVALID_ARG: return "invalid argument";
        case KDA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case KDA_ERR_WORKSPACE: return "workspace missing or too small";
        case KDA_ERR_CUDA: return "CUDA launch or runtime error";
        case KDA_ERR_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

const char *kda_build_info(void) {
    return "libkda 0.1 sm_103a tc:1";
}

}  // extern "C"
