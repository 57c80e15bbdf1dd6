// Backward pass of the prefill: gradients of <d_out, o> + <d_S_final, S_final>
// with respect to q, k, v, g, beta and S0, for the recurrence of "Kimi K3
// Architecture Explained", section 3 (per token: decay, erase, write, read).
//
// Per token, with M = Diag(alpha) S_prev (alpha = e^g), u = v - M^T k and
// S = M + beta k u^T, o = S^T q, the adjoint dS of S (everything the later tokens
// and d_S_final contribute) gives
//     dS  += q do^T                     (the read)
//     dq   = S do
//     w    = dS^T k,   du = beta w,     dv = du
//     dbeta = w . u
//     dk   = beta dS u - M du
//     dM   = dS - k du^T
//     dg   = rowsum(dM o M)             (d alpha_i / d g_i = alpha_i)
//     dS_prev = Diag(alpha) dM
// and at the sequence start dS0 = dS.
//
// Columns of S and dS evolve independently (every step mixes rows only).  The
// gradient pass takes (sequence, head, segment, 32 value columns) per CTA: four
// consumer warps own 8 columns each and all dk <= 128 rows (4 rows per lane), so
// the column sums u and w of a token stay inside a warp (shuffles, no block
// barrier).  A producer warp stages every 4-token block's inputs (g, k, q, v,
// d_out, beta) into a 3-slot shared-memory ring ahead of use, by bulk copies
// where the rows allow, and forms alpha = e^g there once.  A forward pass keeps
// the state at every block start in the workspace; the reverse pass recomputes
// the block's token states into shared memory and walks them backwards.  dv and
// dS0 are column-local and written directly; the row sums dq, dk, dg and dbeta
// are summed over the consumer warps in shared memory once per block and added
// to zeroed fp32 outputs with global atomics.
//
// Segments: the adjoint step dS_prev = Diag(alpha)(I - beta k k^T)(dS + q do^T)
// is linear, and Diag(alpha)(I - beta k k^T) is the transpose of the forward
// token map (I - beta k k^T) Diag(alpha).  So a segment's adjoint map is A_s^T,
// A_s its transfer matrix, and its zero-end adjoint needs no forward state.  A
// pre-pass computes A_s, the zero-start state B_s and the zero-end adjoint of
// every segment in parallel; bwd_scan_kernel forms every segment's start state
// and end adjoint in fp32; the gradient pass then runs all segments at once.
// fp32 throughout: this token-level form serves fp32 activations and shapes
// other than dk = dv = 128.  BF16 activations at dk = dv = 128 take the chunked
// form on tensor cores (launch_backward_chunked at the end of this file).
#include <string.h>

#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int BB = 4;             // tokens per stored block
constexpr int WC = 8;             // state columns per consumer warp
constexpr int NWC = 4;            // consumer warps (one per SM sub-partition)
constexpr int CTC = WC * NWC;     // columns per CTA
constexpr int RPL = 4;            // rows per lane: dk <= 128
constexpr int NBUF = 3;           // ring slots (blocks staged ahead)
constexpr int BT = 32 * (NWC + 1);
constexpr long long kWaitLimit = 4000000000ll;  // ~2 s of SM clocks

// shared memory (floats): ring [NBUF] of {alpha = e^g [BB][128] fp32; k, q [BB][128] and v,
// d_out [BB][CTC] in the activation dtype (regions sized for fp32); beta [BB]};
// token states [NWC][BB][WC/4][128] float4; each consumer warp's row sums
// [NWC][BB][3][128] and dbeta [NWC][BB] of the block; u = v - M^T k of every
// token of the block [NWC][BB][WC]; then the mbarriers and the abort flag.
constexpr int R_G = 0, R_K = BB * 128, R_Q = 2 * BB * 128, R_V = 3 * BB * 128,
              R_D = R_V + BB * CTC, R_B = R_D + BB * CTC, R_SIZE = (R_B + BB + 3) / 4 * 4;
constexpr int SM_TOK = NBUF * R_SIZE;
constexpr int TOK_W = BB * 128 * WC;
constexpr int SM_PART = SM_TOK + NWC * TOK_W;
constexpr int SM_PB = SM_PART + NWC * BB * 3 * 128;
constexpr int SM_U = SM_PB + NWC * BB;
constexpr int SM_BAR = SM_U + NWC * BB * WC;  // 9 mbarriers (18 floats), then the flag
constexpr size_t BWD_SMEM = (size_t)(SM_BAR + 18 + 4) * sizeof(float);
// the pre-pass instantiation keeps only the ring; its barriers follow it
constexpr int SM_BAR_PRE = NBUF * R_SIZE;
constexpr size_t BWD_SMEM_PRE = (size_t)(SM_BAR_PRE + 18 + 4) * sizeof(float);
static_assert(R_B + BB <= R_SIZE && (R_SIZE % 4) == 0 && (R_D % 4) == 0, "ring layout");
static_assert((SM_BAR % 2) == 0 && (SM_TOK % 4) == 0 && (SM_U % 4) == 0, "alignment");
static_assert(BWD_SMEM <= 227 * 1024, "shared memory");
static_assert(WC % 4 == 0 && 32 % WC == 0, "columns per warp");

struct BwdArgs {
    const void *q, *k, *v, *dout;
    const float *g, *beta, *S0, *dSF;
    const int32_t *cu;
    float *gq, *gk, *gv, *gg, *gbeta, *gS0;  // dq, dk, dv, dg, dbeta, dS0
    float *blk_states;  // [blocks][H][ncw][dk][8]: the state at each BB-token block start
    int32_t *dev_status;
    int N, T_tot, H, dk, dv, ncw, act;
    int bulk;  // rows and column slices meet the bulk-copy rules (16-byte aligned)
    // Segments (Sg > 1): the main pass runs segment s from its start state X and
    // its end adjoint Y ([N][H][Sg][dk][dv] each, from the scan).  The pre-pass
    // (the PRE instantiation) takes roles by column block: the transfer matrix A_s (dk
    // columns, from the identity, v ignored) -> TA [N][H][Sg][dk][dk], the
    // zero-start state B_s -> TB, and the zero-end adjoint B^_s (the reverse
    // chain from dS = 0, which needs no forward state) -> TBh, both
    // [N][H][Sg][dk][dv].
    int Sg, ncbA, ncbB;
    float *X, *Y;
    float *TA, *TB, *TBh;
};

enum BwdRole { ROLE_MAIN = 0, ROLE_XFER_A = 1, ROLE_XFER_B = 2, ROLE_ADJ = 3 };

// Column sums of a WC-column block spread over the warp's lanes (p[j] of lane
// l: lane l's part of column j); lane l returns the total of column l % WC.
// log2(WC) halving steps trade half of the remaining columns with the partner
// lane, then log2(32 / WC) more add the lane groups.
__device__ __forceinline__ float colsum(float (&p)[WC]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int off = WC / 2; off >= 1; off >>= 1) {
        const bool up = lane & off;
#pragma unroll
        for (int j = 0; j < off; ++j) {
            const float send = up ? p[j] : p[j + off];
            const float keep = up ? p[j + off] : p[j];
            p[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    float s = p[0];
#pragma unroll
    for (int off = WC; off < 32; off <<= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    return s;
}

// WC consecutive activations (aligned to their size) as fp32
__device__ __forceinline__ void loadW(const float *p, float (&o)[WC]) {
#pragma unroll
    for (int i = 0; i < WC / 4; ++i) {
        const float4 a = ((const float4 *)p)[i];
        o[4 * i] = a.x; o[4 * i + 1] = a.y; o[4 * i + 2] = a.z; o[4 * i + 3] = a.w;
    }
}
__device__ __forceinline__ void loadW(const __nv_bfloat16 *p, float (&o)[WC]) {
#pragma unroll
    for (int i = 0; i < WC / 4; ++i) {
        const uint2 a = ((const uint2 *)p)[i];
        o[4 * i] = __uint_as_float(a.x << 16);
        o[4 * i + 1] = __uint_as_float(a.x & 0xffff0000u);
        o[4 * i + 2] = __uint_as_float(a.y << 16);
        o[4 * i + 3] = __uint_as_float(a.y & 0xffff0000u);
    }
}

// PRE: the segment pre-pass (transfer and adjoint roles only, 3 CTAs per SM);
// otherwise the gradient pass.
template <typename TA, bool PRE>
__global__ void __launch_bounds__(BT, PRE ? 3 : 2) backward_kernel(const BwdArgs a) {
    extern __shared__ __align__(16) float sm[];
    const int unit = blockIdx.x, s = blockIdx.z;
    const int n = unit / a.H, h = unit % a.H;
    int role = ROLE_MAIN, cb = blockIdx.y;  // column block within the role
    if (PRE) {
        if (cb < a.ncbA) {
            role = ROLE_XFER_A;
        } else if ((cb -= a.ncbA) < a.ncbB) {
            role = ROLE_XFER_B;
        } else {
            cb -= a.ncbB;
            role = ROLE_ADJ;
        }
    }
    const int c0 = cb * CTC;
    const int wp = threadIdx.x >> 5, l = threadIdx.x & 31;
    const int dk = a.dk, dv = a.dv, H = a.H;
    const int ncol = role == ROLE_XFER_A ? dk : dv;  // columns of this role's matrix
    // which inputs the role reads: v (forward steps), q and d_out (reverse steps)
    const bool want_v = role == ROLE_MAIN || role == ROLE_XFER_B;
    const bool want_qd = role == ROLE_MAIN || role == ROLE_ADJ;
    int t_begin, t_end;
    if (!segment_range(a.cu, n, a.N, a.T_tot, s, a.Sg, a.dev_status, t_begin, t_end)) return;
    int blk_base = 0;  // this sequence's first stored block
    for (int m = 0; m < n; ++m) {
        const int lm = a.cu[m + 1] - a.cu[m];
        if (lm < 0) {  // the earlier sequences' blocks must not overlap this one's
            dev_fail(a.dev_status, KDA_ERR_INVALID_ARG);
            return;
        }
        blk_base += (lm + BB - 1) / BB;
    }
    blk_base += (t_begin - a.cu[n]) / BB;  // segments start on 16-token boundaries
    const int nblk = (t_end - t_begin + BB - 1) / BB;
    // block visits f: forward (f < nblk) and reverse (f >= nblk); the main pass
    // makes both, the transfer roles the forward ones, the adjoint role the reverse
    const int fb = role == ROLE_ADJ ? nblk : 0;
    const int fe = (role == ROLE_XFER_A || role == ROLE_XFER_B) ? nblk : 2 * nblk;
    // full[NBUF] (ring slot ready), empty[NBUF] (slot consumed), landed[NBUF]
    // (bulk copies in)
    const uint32_t bar0 = smem_addr(sm + (PRE ? SM_BAR_PRE : SM_BAR));
    auto bar_full = [&](int b) { return bar0 + 8 * b; };
    auto bar_empty = [&](int b) { return bar0 + 8 * (NBUF + b); };
    auto bar_landed = [&](int b) { return bar0 + 8 * (2 * NBUF + b); };
    volatile int *abort = (volatile int *)(sm + (PRE ? SM_BAR_PRE : SM_BAR) + 18);
    // padded rows (past dk) and columns (past dv) of the ring stay zero: the
    // producer writes only the real ones
    for (int e = threadIdx.x; e < NBUF * R_SIZE; e += BT) sm[e] = 0.f;
    fence_async_smem();  // before the bulk copies overwrite these bytes
    if (threadIdx.x == 0) {
        for (int b = 0; b < NBUF; ++b) {
            mbar_init(bar_full(b), 32);          // producer lanes
            mbar_init(bar_empty(b), 32 * NWC);   // consumer threads
            mbar_init(bar_landed(b), 1);         // bulk bytes
        }
        *abort = 0;
        mbar_fence_init();
    }
    __syncthreads();
    // blocks are visited forward (c = 0 .. nblk-1), then backward (nblk-1 .. 0)
    auto block_of = [&](int f) { return f < nblk ? f : 2 * nblk - 1 - f; };

    if (wp == NWC) {  // ---------------------------------------------- producer
        const TA *q = (const TA *)a.q, *k = (const TA *)a.k, *v = (const TA *)a.v;
        const TA *dout = (const TA *)a.dout;
        // issue(f) stages block visit f into slot f % NBUF (bulk copies in flight,
        // or plain loads done); finish(f) waits for the copies, turns g into
        // alpha and releases the slot.  Visit f + 1 is issued before f finishes.
        bool pok = true;
        auto issue = [&](int f) {
            const int buf = (f - fb) % NBUF, use = (f - fb) / NBUF;
            const bool back = f >= nblk, qd = back && want_qd;
            if (use >= 1) pok = mbar_wait(bar_empty(buf), (use - 1) & 1, abort, kWaitLimit) && pok;
            if (!pok) return;
            {
                float *rb = sm + buf * R_SIZE;
                TA *rk = (TA *)(rb + R_K), *rq = (TA *)(rb + R_Q);
                TA *rv = (TA *)(rb + R_V), *rd = (TA *)(rb + R_D);
                const int tb = t_begin + block_of(f) * BB, nt = min(BB, t_end - tb);
                if (a.bulk) {  // one bulk copy per token row, counted in bytes on `landed`
                    const uint32_t landed = bar_landed(buf);
                    const int nvc = min(CTC, dv - c0);
                    const uint32_t es = sizeof(TA);
                    const uint32_t per_tok = dk * 4 + dk * es + (want_v ? nvc * es : 0) +
                                             (qd ? dk * es + nvc * es : 0);
                    fence_async_smem();  // this warp's earlier writes to the slot come first
                    if (l == 0) mbar_arrive_expect_tx(landed, nt * per_tok);
                    __syncwarp();
                    if (l < nt) {
                        const size_t row = (size_t)(tb + l) * H + h;
                        bulk_g2s(smem_addr(rb + R_G + l * 128), a.g + row * dk, dk * 4, landed);
                        bulk_g2s(smem_addr(rk + l * 128), k + row * dk, dk * es, landed);
                        if (want_v)
                            bulk_g2s(smem_addr(rv + l * CTC), v + row * dv + c0, nvc * es, landed);
                        if (qd) {
                            bulk_g2s(smem_addr(rq + l * 128), q + row * dk, dk * es, landed);
                            bulk_g2s(smem_addr(rd + l * CTC), dout + row * dv + c0, nvc * es,
                                     landed);
                        }
                        rb[R_B + l] = a.beta[row];
                    }
                } else {  // plain loads, a block's worth in flight
                    float gv_[BB][RPL], kv_[BB][RPL];
#pragma unroll
                    for (int j = 0; j < BB; ++j)
#pragma unroll
                        for (int rr = 0; rr < RPL; ++rr) {
                            const int r = l + 32 * rr;
                            const bool in = j < nt && r < dk;
                            const size_t ix = ((size_t)(tb + j) * H + h) * dk + r;
                            gv_[j][rr] = in ? a.g[ix] : 0.f;
                            kv_[j][rr] = in ? act_ld(k, ix) : 0.f;
                        }
#pragma unroll
                    for (int j = 0; j < BB; ++j)
#pragma unroll
                        for (int rr = 0; rr < RPL; ++rr) gv_[j][rr] = expf(gv_[j][rr]);  // alpha
                    float vv[BB], bv = 0.f;
#pragma unroll
                    for (int j = 0; j < BB; ++j) {
                        const bool in = want_v && j < nt && c0 + l < dv;
                        vv[j] = in ? act_ld(v, ((size_t)(tb + j) * H + h) * dv + c0 + l) : 0.f;
                    }
                    if (l < nt) bv = a.beta[(size_t)(tb + l) * H + h];
#pragma unroll
                    for (int j = 0; j < BB; ++j) {
#pragma unroll
                        for (int rr = 0; rr < RPL; ++rr) {
                            rb[R_G + j * 128 + l + 32 * rr] = gv_[j][rr];
                            act_st(rk, j * 128 + l + 32 * rr, kv_[j][rr]);
                        }
                        act_st(rv, j * CTC + l, vv[j]);
                    }
                    if (l < BB) rb[R_B + l] = bv;
                    if (qd) {  // the reverse walk also reads q and d_out
#pragma unroll
                        for (int j = 0; j < BB; ++j)
#pragma unroll
                            for (int rr = 0; rr < RPL; ++rr) {
                                const int r = l + 32 * rr;
                                const bool in = j < nt && r < dk;
                                gv_[j][rr] =
                                    in ? act_ld(q, ((size_t)(tb + j) * H + h) * dk + r) : 0.f;
                            }
#pragma unroll
                        for (int j = 0; j < BB; ++j) {
                            const bool in = j < nt && c0 + l < dv;
                            vv[j] = in ? act_ld(dout, ((size_t)(tb + j) * H + h) * dv + c0 + l)
                                       : 0.f;
                        }
#pragma unroll
                        for (int j = 0; j < BB; ++j) {
#pragma unroll
                            for (int rr = 0; rr < RPL; ++rr)
                                act_st(rq, j * 128 + l + 32 * rr, gv_[j][rr]);
                            act_st(rd, j * CTC + l, vv[j]);
                        }
                    }
                }
            }
        };
        auto finish = [&](int f) {
            const int buf = (f - fb) % NBUF, use = (f - fb) / NBUF;
            if (pok && a.bulk) {
                // alpha = e^g in place, once for all consumer warps and visits
                pok = mbar_wait(bar_landed(buf), use & 1, abort, kWaitLimit);
                if (pok) {
                    float *rb = sm + buf * R_SIZE;
                    const int tb = t_begin + block_of(f) * BB, nt = min(BB, t_end - tb);
#pragma unroll
                    for (int j = 0; j < BB; ++j)
#pragma unroll
                        for (int rr = 0; rr < RPL; ++rr)
                            if (j < nt && l + 32 * rr < dk)
                                rb[R_G + j * 128 + l + 32 * rr] = expf(rb[R_G + j * 128 + l + 32 * rr]);
                }
            }
            mbar_arrive(bar_full(buf));
        };
        if (fb < fe) issue(fb);
        for (int f = fb; f < fe; ++f) {
            if (f + 1 < fe) issue(f + 1);
            finish(f);
        }
        return;
    }

    // ------------------------------------------------------------------ consumers
    const int cw = cb * NWC + wp;  // this warp's WC-column group
    const int c0w = cw * WC;
    const bool has_cols = c0w < ncol;  // a warp past the last column keeps zeros only
    // start state and end adjoint of this segment (main), the identity (A), zeros
    const size_t seg_mat = ((size_t)unit * a.Sg + s) * dk;  // row 0 of segment s's matrices
    const bool main_role = !PRE && role == ROLE_MAIN;
    const float *S_in = !main_role ? nullptr : a.Sg > 1 ? a.X + seg_mat * dv : a.S0;
    const float *dS_in = !main_role ? nullptr : a.Sg > 1 ? a.Y + seg_mat * dv : a.dSF;
    if (a.Sg == 1) {
        S_in = S_in ? S_in + (size_t)unit * dk * dv : nullptr;
        dS_in = dS_in ? dS_in + (size_t)unit * dk * dv : nullptr;
    }
    float S[RPL][WC], dS[RPL][WC];
#pragma unroll
    for (int rr = 0; rr < RPL; ++rr)
#pragma unroll
        for (int j = 0; j < WC; ++j) {
            const int r = l + 32 * rr, c = c0w + j;
            const bool in = r < dk && c < ncol;
            S[rr][j] = role == ROLE_XFER_A ? (in && r == c ? 1.f : 0.f)
                                           : (S_in && in) ? S_in[(size_t)r * dv + c] : 0.f;
            dS[rr][j] = (dS_in && in) ? dS_in[(size_t)r * dv + c] : 0.f;
        }
    float4 *tokw = (float4 *)(sm + SM_TOK + wp * TOK_W);  // [BB][WC/4][128]
    float *part = sm + SM_PART, *pb = sm + SM_PB;
    float *us = sm + SM_U + wp * BB * WC;  // [BB][WC]: u of the block's tokens
    auto blk_ptr = [&](int c, int rr) {
        return (float4 *)(a.blk_states +
                          ((((size_t)(blk_base + c) * H + h) * a.ncw + cw) * dk + l + 32 * rr) * WC);
    };
    auto put_tok = [&](int j) {
#pragma unroll
        for (int rr = 0; rr < RPL; ++rr)
#pragma unroll
            for (int x = 0; x < WC / 4; ++x)
                tokw[(j * (WC / 4) + x) * 128 + l + 32 * rr] =
                    make_float4(S[rr][4 * x], S[rr][4 * x + 1], S[rr][4 * x + 2], S[rr][4 * x + 3]);
    };
    // one forward token step from ring slot j: S <- M + beta k u^T, M = Diag(alpha) S,
    // u = v - M^T k
    auto fstep = [&](const float *rb, int j, bool keep_u) {
        const TA *rk = (const TA *)(rb + R_K);
        float kr[RPL], al[RPL];
#pragma unroll
        for (int rr = 0; rr < RPL; ++rr) {
            kr[rr] = act_ld(rk, j * 128 + l + 32 * rr);
            al[rr] = rb[R_G + j * 128 + l + 32 * rr];
        }
        // column pairs (jj, jj + 1) as packed fp32x2 operations
        float p[WC];
#pragma unroll
        for (int jj = 0; jj < WC; ++jj) p[jj] = 0.f;
#pragma unroll
        for (int rr = 0; rr < RPL; ++rr)
#pragma unroll
            for (int jj = 0; jj < WC; jj += 2) {
                mul2_inplace(S[rr][jj], S[rr][jj + 1], make_float2(al[rr], al[rr]));
                fma2_acc(p[jj], p[jj + 1], S[rr][jj], S[rr][jj + 1], kr[rr], kr[rr]);
            }
        const float um =
            act_ld((const TA *)(rb + R_V), j * CTC + WC * wp + (l & (WC - 1))) - colsum(p);
        if (keep_u && l < WC) us[j * WC + l] = um;
        const float b = rb[R_B + j];
        float u[WC];
#pragma unroll
        for (int jj = 0; jj < WC; ++jj) u[jj] = b * __shfl_sync(0xffffffffu, um, jj);
#pragma unroll
        for (int rr = 0; rr < RPL; ++rr)
#pragma unroll
            for (int jj = 0; jj < WC; jj += 2)
                fma2_acc(S[rr][jj], S[rr][jj + 1], kr[rr], kr[rr], u[jj], u[jj + 1]);
    };
    bool ok = true;

    // forward: the state at every block start (main), or the segment's end state
    for (int f = 0; f < nblk && role != ROLE_ADJ; ++f) {
        const int buf = f % NBUF;
        ok = mbar_wait(bar_full(buf), (f / NBUF) & 1, abort, kWaitLimit) && ok;
        if (ok) {
            const float *rb = sm + buf * R_SIZE;
#pragma unroll
            for (int rr = 0; rr < RPL; ++rr) {
                if (!main_role || !has_cols || l + 32 * rr >= dk) continue;
                float4 *d = blk_ptr(f, rr);
#pragma unroll
                for (int x = 0; x < WC / 4; ++x)
                    d[x] = make_float4(S[rr][4 * x], S[rr][4 * x + 1], S[rr][4 * x + 2],
                                       S[rr][4 * x + 3]);
            }
            const int nt = min(BB, t_end - (t_begin + f * BB));
            for (int j = 0; j < nt; ++j) fstep(rb, j, false);
        }
        mbar_arrive(bar_empty(buf));
    }
    if (role == ROLE_XFER_A || role == ROLE_XFER_B) {  // A_s or B_s of this segment
        if (!ok) {
            dev_fail(a.dev_status, KDA_ERR_TIMEOUT);
            return;
        }
        float *out = role == ROLE_XFER_A ? a.TA + seg_mat * dk : a.TB + seg_mat * dv;
        const int ld = role == ROLE_XFER_A ? dk : dv;
#pragma unroll
        for (int rr = 0; rr < RPL; ++rr)
#pragma unroll
            for (int j = 0; j < WC; ++j) {
                const int r = l + 32 * rr, c = c0w + j;
                if (r < dk && c < ncol) out[(size_t)r * ld + c] = S[rr][j];
            }
        return;
    }
    auto load_start = [&](int c) {
#pragma unroll
        for (int rr = 0; rr < RPL; ++rr) {
            const bool in = has_cols && l + 32 * rr < dk;  // else the row stays zero
            const float4 *s = blk_ptr(c, rr);
#pragma unroll
            for (int x = 0; x < WC / 4; ++x) {
                const float4 v4 = in ? s[x] : make_float4(0.f, 0.f, 0.f, 0.f);
                S[rr][4 * x] = v4.x; S[rr][4 * x + 1] = v4.y;
                S[rr][4 * x + 2] = v4.z; S[rr][4 * x + 3] = v4.w;
            }
        }
    };
    if (main_role && nblk > 0 && ok) load_start(nblk - 1);

    // reverse
    for (int f = nblk; f < 2 * nblk; ++f) {
        const int buf = (f - fb) % NBUF, c = 2 * nblk - 1 - f;
        const int tb = t_begin + c * BB, nt = min(BB, t_end - tb);
        ok = mbar_wait(bar_full(buf), ((f - fb) / NBUF) & 1, abort, kWaitLimit) && ok;
        if (PRE) {  // ROLE_ADJ: the adjoint chain alone: dS <- Diag(alpha)(I - beta k k^T)(dS + q do^T)
            if (ok) {
                const float *rb = sm + buf * R_SIZE;
                for (int j = nt - 1; j >= 0; --j) {
                    float kr[RPL], qr[RPL], al[RPL], dov[WC], pw[WC];
#pragma unroll
                    for (int rr = 0; rr < RPL; ++rr) {
                        kr[rr] = act_ld((const TA *)(rb + R_K), j * 128 + l + 32 * rr);
                        qr[rr] = act_ld((const TA *)(rb + R_Q), j * 128 + l + 32 * rr);
                        al[rr] = rb[R_G + j * 128 + l + 32 * rr];
                    }
                    loadW((const TA *)(rb + R_D) + j * CTC + WC * wp, dov);
#pragma unroll
                    for (int jj = 0; jj < WC; ++jj) pw[jj] = 0.f;
#pragma unroll
                    for (int rr = 0; rr < RPL; ++rr)
#pragma unroll
                        for (int jj = 0; jj < WC; jj += 2) {
                            fma2_acc(dS[rr][jj], dS[rr][jj + 1], qr[rr], qr[rr], dov[jj],
                                     dov[jj + 1]);
                            fma2_acc(pw[jj], pw[jj + 1], dS[rr][jj], dS[rr][jj + 1], kr[rr],
                                     kr[rr]);
                        }
                    const float wm = colsum(pw);
                    const float nb = -rb[R_B + j];
                    float ndu[WC];
#pragma unroll
                    for (int jj = 0; jj < WC; ++jj) ndu[jj] = nb * __shfl_sync(0xffffffffu, wm, jj);
#pragma unroll
                    for (int rr = 0; rr < RPL; ++rr)
#pragma unroll
                        for (int jj = 0; jj < WC; jj += 2) {
                            fma2_acc(dS[rr][jj], dS[rr][jj + 1], kr[rr], kr[rr], ndu[jj],
                                     ndu[jj + 1]);
                            mul2_inplace(dS[rr][jj], dS[rr][jj + 1], make_float2(al[rr], al[rr]));
                        }
                }
            }
            mbar_arrive(bar_empty(buf));
            continue;
        }
        if (ok) {
            const float *rb = sm + buf * R_SIZE;
            for (int j = 0; j < nt; ++j) {  // the block's pre-token states
                put_tok(j);
                fstep(rb, j, true);
            }
            __syncwarp();  // u of lanes 0 .. WC-1 visible to the whole warp
            if (c > 0) load_start(c - 1);  // lands while this block is walked
            for (int j = nt - 1; j >= 0; --j) {
                float kr[RPL], qr[RPL], al[RPL];
#pragma unroll
                for (int rr = 0; rr < RPL; ++rr) {
                    kr[rr] = act_ld((const TA *)(rb + R_K), j * 128 + l + 32 * rr);
                    qr[rr] = act_ld((const TA *)(rb + R_Q), j * 128 + l + 32 * rr);
                    al[rr] = rb[R_G + j * 128 + l + 32 * rr];
                }
                float dov[WC];
                loadW((const TA *)(rb + R_D) + j * CTC + WC * wp, dov);
                float M[RPL][WC];
#pragma unroll
                for (int rr = 0; rr < RPL; ++rr)
#pragma unroll
                    for (int x = 0; x < WC / 4; ++x) {
                        const float4 s4 = tokw[(j * (WC / 4) + x) * 128 + l + 32 * rr];
                        M[rr][4 * x] = s4.x;
                        M[rr][4 * x + 1] = s4.y;
                        M[rr][4 * x + 2] = s4.z;
                        M[rr][4 * x + 3] = s4.w;
                    }
                // column pairs (jj, jj + 1) as packed fp32x2 operations
                float pw[WC];
#pragma unroll
                for (int jj = 0; jj < WC; ++jj) pw[jj] = 0.f;
#pragma unroll
                for (int rr = 0; rr < RPL; ++rr)
#pragma unroll
                    for (int jj = 0; jj < WC; jj += 2) {
                        // the read at t
                        fma2_acc(dS[rr][jj], dS[rr][jj + 1], qr[rr], qr[rr], dov[jj], dov[jj + 1]);
                        fma2_acc(pw[jj], pw[jj + 1], dS[rr][jj], dS[rr][jj + 1], kr[rr], kr[rr]);
                        mul2_inplace(M[rr][jj], M[rr][jj + 1], make_float2(al[rr], al[rr]));
                    }
                const float wm = colsum(pw);  // (dS^T k) of column l % WC
                const float b = rb[R_B + j];
                const int t = tb + j;
                if (l < WC && c0w + l < dv) a.gv[((size_t)t * H + h) * dv + c0w + l] = b * wm;
                float uj[WC];  // u = v - M^T k, kept by the recompute
                loadW(us + j * WC, uj);
                float bu[WC], ndu[WC], db = 0.f;  // beta u, -beta w
#pragma unroll
                for (int jj = 0; jj < WC; ++jj) {
                    const float w = __shfl_sync(0xffffffffu, wm, jj);
                    bu[jj] = b * uj[jj];
                    ndu[jj] = -b * w;
                    db = fmaf(w, uj[jj], db);
                }
                // per row, even and odd columns summed apart and added at the end
                float dq[RPL][2], dkr[RPL][2], dg[RPL][2];
#pragma unroll
                for (int rr = 0; rr < RPL; ++rr) {
                    dq[rr][0] = dq[rr][1] = dkr[rr][0] = dkr[rr][1] = dg[rr][0] = dg[rr][1] = 0.f;
#pragma unroll
                    for (int jj = 0; jj < WC; jj += 2) {
                        float s0 = M[rr][jj], s1 = M[rr][jj + 1];  // S_t = M + k (beta u)^T
                        fma2_acc(s0, s1, kr[rr], kr[rr], bu[jj], bu[jj + 1]);
                        fma2_acc(dq[rr][0], dq[rr][1], s0, s1, dov[jj], dov[jj + 1]);
                        // dk: beta dS u - M du
                        fma2_acc(dkr[rr][0], dkr[rr][1], M[rr][jj], M[rr][jj + 1], ndu[jj],
                                 ndu[jj + 1]);
                        fma2_acc(dkr[rr][0], dkr[rr][1], dS[rr][jj], dS[rr][jj + 1], bu[jj],
                                 bu[jj + 1]);
                        // dM = dS - k du^T, dg += dM o M, dS_prev = Diag(alpha) dM
                        fma2_acc(dS[rr][jj], dS[rr][jj + 1], kr[rr], kr[rr], ndu[jj], ndu[jj + 1]);
                        fma2_acc(dg[rr][0], dg[rr][1], dS[rr][jj], dS[rr][jj + 1], M[rr][jj],
                                 M[rr][jj + 1]);
                        mul2_inplace(dS[rr][jj], dS[rr][jj + 1], make_float2(al[rr], al[rr]));
                    }
                }
                float *pp = part + (wp * BB + j) * 3 * 128;
#pragma unroll
                for (int rr = 0; rr < RPL; ++rr) {
                    pp[l + 32 * rr] = dq[rr][0] + dq[rr][1];
                    pp[128 + l + 32 * rr] = dkr[rr][0] + dkr[rr][1];
                    pp[256 + l + 32 * rr] = dg[rr][0] + dg[rr][1];
                }
                if (l == 0) pb[wp * BB + j] = db;
            }
        }
        mbar_arrive(bar_empty(buf));
        // the consumer warps' row sums of this block, accumulated over column blocks
        const bool bad = named_bar_or(1, 32 * NWC, !ok);
        if (!bad) {
            const int x = threadIdx.x;  // row (32 * NWC = 128 consumer threads)
            if (x < dk) {
                for (int j = 0; j < nt; ++j) {
                    const size_t ix = ((size_t)(tb + j) * H + h) * dk + x;
                    float sq = 0.f, sk = 0.f, sg = 0.f;
#pragma unroll
                    for (int w = 0; w < NWC; ++w) {
                        const float *pp = part + (w * BB + j) * 3 * 128;
                        sq += pp[x];
                        sk += pp[128 + x];
                        sg += pp[256 + x];
                    }
                    atomicAdd(a.gq + ix, sq);
                    atomicAdd(a.gk + ix, sk);
                    atomicAdd(a.gg + ix, sg);
                }
            }
            if (x < nt) {
                float sb = 0.f;
#pragma unroll
                for (int w = 0; w < NWC; ++w) sb += pb[w * BB + x];
                atomicAdd(a.gbeta + (size_t)(tb + x) * H + h, sb);
            }
        }
        named_bar_sync(1, 32 * NWC);  // the partials are rewritten by the next block
        ok = ok && !bad;
    }
    if (!ok) {
        dev_fail(a.dev_status, KDA_ERR_TIMEOUT);
        return;
    }
    // the adjoint at the segment's start: dS0 (main, first segment) or B^_s
    float *dout_mat = role == ROLE_ADJ ? a.TBh + seg_mat * dv
                      : (main_role && s == 0 && a.gS0) ? a.gS0 + (size_t)unit * dk * dv
                                          : nullptr;
    if (dout_mat) {
#pragma unroll
        for (int rr = 0; rr < RPL; ++rr)
#pragma unroll
            for (int j = 0; j < WC; ++j) {
                const int r = l + 32 * rr, c = c0w + j;
                if (r < dk && c < dv) dout_mat[(size_t)r * dv + c] = dS[rr][j];
            }
    }
}

// The segment scans, fp32: start states X_0 = S0, X_{s+1} = A_s X_s + B_s, and
// end adjoints Y_{Sg-1} = d_S_final, Y_{s-1} = A_s^T Y_s + B^_s (the adjoint of a
// segment's linear map is the transpose of its transfer matrix: each token's
// adjoint step Diag(alpha)(I - beta k k^T) is the transpose of its forward map
// (I - beta k k^T) Diag(alpha)).  grid (N*H, ceil(dv / 32), 2): z = 0 the forward
// scan, z = 1 the adjoint scan.  Thread (r, g) keeps row r, columns 8g .. 8g + 7
// of a 32-column block; the next step's A is loaded into the other shared buffer
// while the current step's products run (A does not depend on the scan).
constexpr int SC_T = 512;
constexpr int SC_PER = 32;  // A elements per thread and step: 128 x 128 / 512
__global__ void __launch_bounds__(SC_T) bwd_scan_kernel(const BwdArgs a) {
    extern __shared__ __align__(16) float sm[];
    const int unit = blockIdx.x, c0 = blockIdx.y * 32, adj = blockIdx.z;
    const int dk = a.dk, dv = a.dv, Sg = a.Sg;
    const int r = threadIdx.x & 127, g8 = 8 * (threadIdx.x >> 7);
    const int nc = min(32, dv - c0);
    const int ald = dk + 1;             // padded rows against bank conflicts
    auto Abuf = [&](int i) { return sm + i * dk * ald; };  // two A buffers
    float *Z = sm + 2 * dk * ald;       // [dk][32]: the running matrix
    const size_t base = (size_t)unit * Sg * dk;  // row 0 of segment 0
    const float *init = adj ? a.dSF : a.S0;
    float *outm = adj ? a.Y : a.X;
    const bool row = r < dk;
    float z[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int c = g8 + j;
        z[j] = (init && row && c < nc) ? init[((size_t)unit * dk + r) * dv + c0 + c] : 0.f;
    }
    auto store_z = [&](int seg) {
        if (!row) return;
        float *o = outm + (base + (size_t)seg * dk + r) * dv + c0;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (g8 + j < nc) o[g8 + j] = z[j];
    };
    store_z(adj ? Sg - 1 : 0);
    auto seg_of = [&](int step) { return adj ? Sg - 1 - step : step; };  // the map applied
    float pre[SC_PER];
    auto fetch = [&](int step) {  // this thread's share of A_{seg_of(step)}
        const float *A = a.TA + (base + (size_t)seg_of(step) * dk) * dk;
#pragma unroll
        for (int i = 0; i < SC_PER; ++i) {
            const int e = threadIdx.x + i * SC_T;
            pre[i] = e < dk * dk ? A[e] : 0.f;
        }
    };
    auto put = [&](float *As) {
#pragma unroll
        for (int i = 0; i < SC_PER; ++i) {
            const int e = threadIdx.x + i * SC_T;
            if (e < dk * dk) As[(e / dk) * ald + e % dk] = pre[i];
        }
    };
    if (Sg > 1) {
        fetch(0);
        put(Abuf(0));
    }
    for (int step = 0; step < Sg - 1; ++step) {
        const int sa = seg_of(step);
        const float *As = Abuf(step & 1);
        if (row) {
#pragma unroll
            for (int j = 0; j < 8; ++j) Z[r * 32 + g8 + j] = z[j];
        }
        __syncthreads();  // A_sa and Z in place
        if (step + 1 < Sg - 1) fetch(step + 1);
        if (row) {
            const float *Bm = (adj ? a.TBh : a.TB) + (base + (size_t)sa * dk + r) * dv + c0;
#pragma unroll
            for (int j = 0; j < 8; ++j) z[j] = g8 + j < nc ? Bm[g8 + j] : 0.f;
            for (int kk = 0; kk < dk; ++kk) {
                const float av = adj ? As[kk * ald + r] : As[r * ald + kk];
                const float4 z0 = *(const float4 *)(Z + kk * 32 + g8);
                const float4 z1 = *(const float4 *)(Z + kk * 32 + g8 + 4);
                z[0] = fmaf(av, z0.x, z[0]);
                z[1] = fmaf(av, z0.y, z[1]);
                z[2] = fmaf(av, z0.z, z[2]);
                z[3] = fmaf(av, z0.w, z[3]);
                z[4] = fmaf(av, z1.x, z[4]);
                z[5] = fmaf(av, z1.y, z[5]);
                z[6] = fmaf(av, z1.z, z[6]);
                z[7] = fmaf(av, z1.w, z[7]);
            }
            store_z(adj ? sa - 1 : sa + 1);
        }
        __syncthreads();  // Z and this A read by everyone
        if (step + 1 < Sg - 1) put(Abuf((step + 1) & 1));
    }
}

}  // namespace

namespace {
size_t r256(size_t b) { return (b + 255) & ~(size_t)255; }
size_t blk_bytes(int N, int T_tot, int H, int dk, int dv) {
    const size_t blocks = (size_t)T_tot / BB + N;  // >= sum_n ceil(len_n / 8)
    const int ncw = (dv + WC - 1) / WC;
    return blocks * H * ncw * dk * WC * sizeof(float);
}
}  // namespace

size_t backward_workspace_bytes(int N, int T_tot, int H, int dk, int dv, int Sg) {
    size_t b = blk_bytes(N, T_tot, H, dk, dv);
    if (Sg > 1)  // A_s; B_s, B^_s, X_s, Y_s
        b = r256(b) + (size_t)N * H * Sg * ((size_t)dk * dk + 4 * (size_t)dk * dv) * sizeof(float);
    return b;
}

cudaError_t launch_backward(const PrefillArgs &p, const void *dout, const float *dSF, float *dq,
                            float *dk, float *dv, float *dg, float *dbeta, float *dS0, int Sg,
                            void *workspace, cudaStream_t st) {
    BwdArgs a;
    memset(&a, 0, sizeof(a));
    a.q = p.q; a.k = p.k; a.v = p.v; a.dout = dout;
    a.g = p.g; a.beta = p.beta; a.S0 = p.S0; a.dSF = dSF; a.cu = p.cu;
    a.gq = dq; a.gk = dk; a.gv = dv; a.gg = dg; a.gbeta = dbeta; a.gS0 = dS0;
    a.dev_status = p.dev_status;
    a.N = p.N; a.T_tot = p.T_tot; a.H = p.H; a.dk = p.dk; a.dv = p.dv; a.act = p.act;
    a.ncw = (p.dv + WC - 1) / WC;
    a.Sg = Sg < 1 ? 1 : Sg;
    a.blk_states = (float *)workspace;
    if (a.Sg > 1) {
        const size_t nhs = (size_t)p.N * p.H * a.Sg;
        a.TA = (float *)((uint8_t *)workspace + r256(blk_bytes(p.N, p.T_tot, p.H, p.dk, p.dv)));
        a.TB = a.TA + nhs * p.dk * p.dk;
        a.TBh = a.TB + nhs * p.dk * p.dv;
        a.X = a.TBh + nhs * p.dk * p.dv;
        a.Y = a.X + nhs * p.dk * p.dv;
    }
    {
        const int es = p.act == KDA_DTYPE_F32 ? 4 : 2;
        auto al16 = [](const void *x) { return ((uintptr_t)x & 15u) == 0; };
        a.bulk = al16(p.q) && al16(p.k) && al16(p.v) && al16(dout) && al16(p.g) &&
                 (p.dk * es) % 16 == 0 && (p.dk * 4) % 16 == 0 && (p.dv * es) % 16 == 0;
    }
    const size_t Tn = (size_t)p.T_tot * p.H;
    cudaError_t e;
    // the row sums are accumulated by every column block: start from zero
    if ((e = cudaMemsetAsync(dq, 0, Tn * p.dk * sizeof(float), st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dk, 0, Tn * p.dk * sizeof(float), st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dg, 0, Tn * p.dk * sizeof(float), st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dbeta, 0, Tn * sizeof(float), st)) != cudaSuccess) return e;
    if (p.N == 0 || p.H == 0) return cudaSuccess;
    const bool f32 = p.act == KDA_DTYPE_F32;
    auto run = [&](dim3 grid, bool pre) {
        const void *kern = pre ? (f32 ? (const void *)backward_kernel<float, true>
                                      : (const void *)backward_kernel<__nv_bfloat16, true>)
                               : (f32 ? (const void *)backward_kernel<float, false>
                                      : (const void *)backward_kernel<__nv_bfloat16, false>);
        const size_t smem = pre ? BWD_SMEM_PRE : BWD_SMEM;
        cudaError_t err = set_max_dynamic_smem(kern, (int)smem);
        if (err != cudaSuccess) return err;
        if (pre && f32) backward_kernel<float, true><<<grid, BT, smem, st>>>(a);
        else if (pre) backward_kernel<__nv_bfloat16, true><<<grid, BT, smem, st>>>(a);
        else if (f32) backward_kernel<float, false><<<grid, BT, smem, st>>>(a);
        else backward_kernel<__nv_bfloat16, false><<<grid, BT, smem, st>>>(a);
        return cudaGetLastError();
    };
    const int ncb = (p.dv + CTC - 1) / CTC;
    if (a.Sg > 1) {
        // pre-pass: A_s, B_s and B^_s of every segment, in parallel
        a.ncbA = (p.dk + CTC - 1) / CTC;
        a.ncbB = ncb;
        if ((e = run(dim3((unsigned)(p.N * p.H), (unsigned)(a.ncbA + 2 * ncb), (unsigned)a.Sg),
                      true)) != cudaSuccess)
            return e;
        // scans: every segment's start state and end adjoint
        const size_t ssm = (size_t)(2 * p.dk * (p.dk + 1) + p.dk * 32) * sizeof(float);
        if ((e = set_max_dynamic_smem((const void *)bwd_scan_kernel, (int)ssm)) != cudaSuccess)
            return e;
        bwd_scan_kernel<<<dim3((unsigned)(p.N * p.H), (unsigned)((p.dv + 31) / 32), 2), SC_T, ssm,
                          st>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return run(dim3((unsigned)(p.N * p.H), (unsigned)ncb, (unsigned)a.Sg), false);
}

// ---------------------------------------------------------------------------
// Chunked backward for BF16 activations at dk = dv = 128.
//
// The state at every 16-token block end and the adjoint at every block end are
// produced by the prefill kernels (forward chain with chunk states; adjoint
// chain run from the last block to the first), then every block's gradients
// come from kda_bwd_chunk.cu in parallel.  With Sg > 1 segments per sequence the
// two chains start from scanned segment states: the transfer pass gives A_s (as
// the BF16 hi/lo images of A_s for the forward scan and of A_s^T, segments
// reversed, for the adjoint scan) and B_s, the adjoint chain from a zero end
// adjoint gives B^_s (segments reversed), and the tensor-core scan runs twice:
// X_s = A_{s-1} X_{s-1} + B_{s-1} (start states) and, over the reversed segments,
// Y_s = A_{s+1}^T Y_{s+1} + B^_{s+1} (end adjoints).
// Workspace (each piece 256-byte aligned), in the order of the launches:
//   region A: with Sg > 1 first two of the four segment buffers (below), then,
//             once the scans have read them, the forward states [T_tot / 32][H]
//             [128][128] BF16 (the state after every 32 tokens of a sequence; the
//             gradient kernel forms the state after the 16 tokens in between);
//   with Sg > 1 the other two segment buffers;
//   the adjoints [ceil(T_tot / 16) + N][H][128][128] BF16.
// The four segment buffers are 128 x 128 fp32 per (sequence, head, segment):
// buf0 the images of A (hi, lo), then B^; buf2 the images of A^T; buf1 B, then Y;
// buf3 X.
static size_t seg_buffer_bytes(int N, int H, int Sg) {
    return r256((size_t)N * H * Sg * 128 * 128 * 4);
}
static size_t fwd_state_bytes(int T_tot, int H) {
    return r256((size_t)(T_tot / 32) * H * 128 * 128 * 2);
}
static size_t region_a_bytes(int N, int T_tot, int H, int Sg) {
    const size_t fwd = fwd_state_bytes(T_tot, H), two = 2 * seg_buffer_bytes(N, H, Sg);
    return Sg > 1 && two > fwd ? two : fwd;
}
size_t backward_chunked_workspace_bytes(int N, int T_tot, int H, int Sg) {
    const size_t adj = r256((size_t)((T_tot + 15) / 16 + N) * H * 128 * 128 * 2);
    return region_a_bytes(N, T_tot, H, Sg) + (Sg > 1 ? 2 * seg_buffer_bytes(N, H, Sg) : 0) + adj;
}

cudaError_t launch_backward_chunked(const PrefillArgs &p, const void *dout, const float *dSF,
                                    float *dq, float *dk, float *dv, float *dg, float *dbeta,
                                    float *dS0, int Sg, void *workspace, cudaStream_t st) {
    if (p.N == 0 || p.H == 0) return cudaSuccess;
    uint8_t *ws = (uint8_t *)workspace;
    const size_t ra = region_a_bytes(p.N, p.T_tot, p.H, Sg);
    const size_t seg = Sg > 1 ? seg_buffer_bytes(p.N, p.H, Sg) : 0;
    __nv_bfloat16 *fwd_states = (__nv_bfloat16 *)ws;  // written after the scans
    __nv_bfloat16 *adj_states = (__nv_bfloat16 *)(ws + ra + 2 * seg);
    PrefillArgs base = p;
    base.Sg = Sg;
    base.seg_begin = 0;
    base.seg_count = Sg;
    base.out = nullptr;
    base.S_final = nullptr;
    base.aux_out = nullptr;
    base.emit_out = 0;
    base.ckpt_interval = 0;
    base.gate = 0;
    PrefillArgs fwd = base, adj = base;
    fwd.mode = adj.mode = MODE_OUTPUT;
    fwd.chunk_states = fwd_states;
    adj.chunk_states = adj_states;
    adj.rev = 1;
    adj.v = dout;           // the adjoint chain reads d_out where the forward reads v
    adj.S_final = dS0;      // the adjoint at the start of segment 0
    cudaError_t e;
    if (Sg > 1) {
        // The launch order lets four buffers serve six arrays: the forward scan
        // reads A's images and B, after which the zero-end adjoint chain writes B^
        // over A's images and the adjoint scan writes Y over B.  buf0 and buf2 are
        // dead once the adjoint scan has run, and the forward states take their
        // place.
        const int units = p.N * p.H;
        uint8_t *buf0 = ws, *buf2 = ws + seg, *buf1 = ws + ra, *buf3 = ws + ra + seg;
        __nv_bfloat16 *a_img = (__nv_bfloat16 *)buf0, *a_img_t = (__nv_bfloat16 *)buf2;
        float *TB = (float *)buf1, *X = (float *)buf3;
        float *TBh = (float *)buf0, *Yr = (float *)buf1;
        PrefillArgs t = base;  // A_s (both images) and B_s
        t.mode = MODE_TRANSFER;
        t.transfer = nullptr;
        t.transfer_img = a_img;
        t.transfer_img_t = a_img_t;
        t.zero_state = TB;
        if ((e = launch_prefill_tc(t, st)) != cudaSuccess) return e;
        if ((e = launch_compose(units, Sg, 128, 128, nullptr, a_img, TB, p.S0, X, nullptr, nullptr,
                                p.dev_status, st)) != cudaSuccess)
            return e;
        PrefillArgs tz = base;  // B^_s: the adjoint chain from a zero end adjoint
        tz.mode = MODE_TRANSFER;
        tz.rev = 1;
        tz.v = dout;
        tz.zero_state = TBh;
        if ((e = launch_prefill_tc(tz, st)) != cudaSuccess) return e;
        if ((e = launch_compose(units, Sg, 128, 128, nullptr, a_img_t, TBh, dSF, Yr, nullptr,
                                nullptr, p.dev_status, st)) != cudaSuccess)
            return e;
        fwd.seg_init = X;
        adj.seg_init = Yr;  // read at the reversed segment index
    } else {
        adj.S0 = dSF;  // the adjoint chain starts from d_S_final (NULL: zero)
    }
    if ((e = launch_prefill_tc(fwd, st)) != cudaSuccess) return e;
    if ((e = launch_prefill_tc(adj, st)) != cudaSuccess) return e;
    return launch_bwd_chunk(p, dout, fwd_states, adj_states, dq, dk, dv, dg, dbeta, st);
}

}  // namespace kda
