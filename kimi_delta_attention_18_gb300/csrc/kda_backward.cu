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
// Columns of S and dS evolve independently (every step mixes rows only), so one
// CTA takes (sequence, head, 32-column block): thread i holds row i of both
// blocks in registers.  A forward pass stores the state at every 16-token block
// start (workspace); the reverse pass recomputes each block's 16 token states
// from its start and walks them backwards.  Column sums (u, w) go through
// shared memory; row sums (dq, dk, dg) and dbeta, which every column block
// contributes to, are accumulated with atomics into zeroed fp32 outputs.
// fp32 throughout: a first, token-level implementation of the row (the chunked
// tensor-core form of the backward is not built).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int BC = 16;   // tokens per stored block
constexpr int CB = 32;   // state columns per CTA
constexpr int BT = 128;  // threads: one state row each (dk <= 128)

struct BwdArgs {
    const void *q, *k, *v, *dout;
    const float *g, *beta, *S0, *dSF;
    const int32_t *cu;
    float *gq, *gk, *gv, *gg, *gbeta, *gS0;  // dq, dk, dv, dg, dbeta, dS0
    float *blk_states;   // [sum_n ceil(len_n / 16)][H][dk][dv]: state at each block start
    float *tok_states;   // [N*H*ncb][16][dk][CB]: one block's pre-token states
    int32_t *dev_status;
    int N, T_tot, H, dk, dv, ncb, act;
};

// Column sums of a 32 x 32 block held one row per lane: x[j] of lane l is entry
// (l, j); lane l returns the sum of column l.  Each halving step trades half of
// the remaining columns with the partner lane (16 + 8 + 4 + 2 + 1 shuffles).
__device__ __forceinline__ float warp_colsum(float (&x)[CB]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const bool up = lane & off;
#pragma unroll
        for (int j = 0; j < off; ++j) {
            const float send = up ? x[j] : x[j + off];
            const float keep = up ? x[j + off] : x[j];
            x[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    return x[0];
}

// One token's inputs as a thread needs them (row i of q, k, g; column i of v and
// d_out), loaded a token ahead of their use.
struct TokIn {
    float g, kv, qv, b, vj, dj;
};

template <typename TA>
__global__ void __launch_bounds__(BT) backward_kernel(const BwdArgs a) {
    __shared__ float part[2][BT / 32][CB];  // per-warp column sums
    __shared__ float col[2][CB];            // u, w after the cross-warp sum
    __shared__ float vs[CB], dos[CB];       // this token's v and d_out columns
    const int unit = blockIdx.x, cbk = blockIdx.y;
    const int n = unit / a.H, h = unit % a.H;
    const int c0 = cbk * CB, nc = min(CB, a.dv - c0);
    const int i = threadIdx.x, wp = i >> 5, lane = i & 31;
    const bool row = i < a.dk;
    const int dk = a.dk, dv = a.dv, H = a.H;
    int t_begin, t_end;
    if (!segment_range(a.cu, n, a.N, a.T_tot, 0, 1, a.dev_status, t_begin, t_end)) return;
    int blk_base = 0;  // this sequence's first stored block
    for (int m = 0; m < n; ++m) {
        const int lm = a.cu[m + 1] - a.cu[m];
        if (lm < 0) {  // the earlier sequences' blocks must not overlap this one's
            dev_fail(a.dev_status, KDA_ERR_INVALID_ARG);
            return;
        }
        blk_base += (lm + BC - 1) / BC;
    }
    const int nblk = (t_end - t_begin + BC - 1) / BC;
    const TA *q = (const TA *)a.q, *k = (const TA *)a.k, *v = (const TA *)a.v;
    const TA *dout = (const TA *)a.dout;
    // this CTA's token states [16][dk][CB] (256-byte aligned: whole float4 rows)
    float4 *tok = (float4 *)(a.tok_states + ((size_t)unit * a.ncb + cbk) * BC * dk * CB);
    auto blk_row = [&](int c) {
        return a.blk_states + (((size_t)(blk_base + c) * H + h) * dk + i) * dv + c0;
    };
    auto load = [&](int t, bool back) {
        TokIn r;
        const size_t ix = ((size_t)t * H + h) * dk + i;
        const size_t iv = ((size_t)t * H + h) * dv + c0 + i;
        r.g = row ? a.g[ix] : 0.f;
        r.kv = row ? act_ld(k, ix) : 0.f;
        r.qv = back && row ? act_ld(q, ix) : 0.f;
        r.b = a.beta[(size_t)t * H + h];
        r.vj = i < nc ? act_ld(v, iv) : 0.f;  // zero past the last column: those
        r.dj = back && i < nc ? act_ld(dout, iv) : 0.f;  // columns of S, dS stay 0
        return r;
    };

    float S[CB];
#pragma unroll
    for (int j = 0; j < CB; ++j)
        S[j] = (row && j < nc && a.S0) ? a.S0[((size_t)unit * dk + i) * dv + c0 + j] : 0.f;

    // one forward token step on this column block: S <- M + beta k u^T with
    // M = Diag(alpha) S, u = v - M^T k
    auto step = [&](const TokIn &x) {
        const float alpha = row ? expf(x.g) : 0.f;
        if (i < CB) vs[i] = x.vj;
        float y[CB];
#pragma unroll
        for (int j = 0; j < CB; ++j) {
            S[j] *= alpha;
            y[j] = S[j] * x.kv;
        }
        part[0][wp][lane] = warp_colsum(y);
        __syncthreads();
        if (i < CB) {
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < BT / 32; ++w) s += part[0][w][i];
            col[0][i] = vs[i] - s;
        }
        __syncthreads();
        const float bk = x.b * x.kv;
#pragma unroll
        for (int j = 0; j < CB; ++j) S[j] += bk * col[0][j];
        __syncthreads();  // part, col and vs are rewritten by the next step
    };

    // forward: the state at every block start
    {
        TokIn cur = t_begin < t_end ? load(t_begin, false) : TokIn{};
        for (int t = t_begin; t < t_end; ++t) {
            if (((t - t_begin) & (BC - 1)) == 0 && row) {
                float *d = blk_row((t - t_begin) / BC);
#pragma unroll
                for (int j = 0; j < CB; ++j)
                    if (j < nc) d[j] = S[j];
            }
            TokIn nxt = cur;
            if (t + 1 < t_end) nxt = load(t + 1, false);
            step(cur);
            cur = nxt;
        }
    }

    // reverse
    float dS[CB];
#pragma unroll
    for (int j = 0; j < CB; ++j)
        dS[j] = (row && j < nc && a.dSF) ? a.dSF[((size_t)unit * dk + i) * dv + c0 + j] : 0.f;
    const int ir = min(i, dk - 1);  // rows past dk read a valid row and discard it
    for (int c = nblk - 1; c >= 0; --c) {
        const int tb = t_begin + c * BC, te = min(tb + BC, t_end);
        {
            const float *s0 = blk_row(c);
#pragma unroll
            for (int j = 0; j < CB; ++j) S[j] = (row && j < nc) ? s0[j] : 0.f;
        }
        TokIn cur = load(tb, false);
        for (int t = tb; t < te; ++t) {  // the block's pre-token states
            if (row) {
                float4 *d = tok + ((size_t)(t - tb) * dk + i) * (CB / 4);
#pragma unroll
                for (int j = 0; j < CB / 4; ++j)
                    d[j] = make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]);
            }
            TokIn nxt = cur;
            if (t + 1 < te) nxt = load(t + 1, false);
            step(cur);
            cur = nxt;
        }
        cur = load(te - 1, true);
        float Sn[CB];  // the state before the token being processed, a token ahead
        {
            const float4 *s = tok + ((size_t)(te - 1 - tb) * dk + ir) * (CB / 4);
#pragma unroll
            for (int j = 0; j < CB / 4; ++j) {
                const float4 f = s[j];
                Sn[4 * j] = f.x; Sn[4 * j + 1] = f.y; Sn[4 * j + 2] = f.z; Sn[4 * j + 3] = f.w;
            }
        }
        for (int t = te - 1; t >= tb; --t) {
            const TokIn x = cur;
            float M[CB];
            const float alpha = row ? expf(x.g) : 0.f;
#pragma unroll
            for (int j = 0; j < CB; ++j) M[j] = row ? alpha * Sn[j] : 0.f;
            if (t > tb) {  // prefetch token t - 1
                cur = load(t - 1, true);
                const float4 *s = tok + ((size_t)(t - 1 - tb) * dk + ir) * (CB / 4);
#pragma unroll
                for (int j = 0; j < CB / 4; ++j) {
                    const float4 f = s[j];
                    Sn[4 * j] = f.x; Sn[4 * j + 1] = f.y; Sn[4 * j + 2] = f.z; Sn[4 * j + 3] = f.w;
                }
            }
            if (i < CB) {
                vs[i] = x.vj;
                dos[i] = x.dj;
            }
            __syncthreads();  // dos visible
            float y[CB], z[CB];
#pragma unroll
            for (int j = 0; j < CB; ++j) {
                dS[j] += x.qv * dos[j];  // the read at t
                y[j] = M[j] * x.kv;
                z[j] = dS[j] * x.kv;
            }
            part[0][wp][lane] = warp_colsum(y);
            part[1][wp][lane] = warp_colsum(z);
            __syncthreads();
            if (i < 2 * CB) {
                const int jj = i & (CB - 1), r = i >> 5;
                float s = 0.f;
#pragma unroll
                for (int w = 0; w < BT / 32; ++w) s += part[r][w][jj];
                col[r][jj] = r == 0 ? vs[jj] - s : s;  // u, w = dS^T k
            }
            __syncthreads();
            float dqi = 0.f, dki = 0.f, dgi = 0.f;
            const float bk = x.b * x.kv;
#pragma unroll
            for (int j = 0; j < CB; ++j) {
                const float u = col[0][j], du = x.b * col[1][j];
                dqi += (M[j] + bk * u) * dos[j];    // (S_t do)_i
                dki += x.b * dS[j] * u - M[j] * du;  // (beta dS u - M du)_i
                const float dM = dS[j] - x.kv * du;
                dgi += dM * M[j];
                dS[j] = alpha * dM;  // adjoint of the state before t
            }
            const size_t ix = ((size_t)t * H + h) * dk + i;
            if (row) {
                atomicAdd(a.gq + ix, dqi);
                atomicAdd(a.gk + ix, dki);
                atomicAdd(a.gg + ix, dgi);
            }
            if (i < nc) a.gv[((size_t)t * H + h) * dv + c0 + i] = x.b * col[1][i];
            if (i == CB * 2) {
                float db = 0.f;
#pragma unroll
                for (int j = 0; j < CB; ++j) db += col[1][j] * col[0][j];
                atomicAdd(a.gbeta + (size_t)t * H + h, db);
            }
            __syncthreads();  // part, col, vs, dos are rewritten by the next token
        }
    }
    if (a.gS0 && row) {
        float *d = a.gS0 + ((size_t)unit * dk + i) * dv + c0;
#pragma unroll
        for (int j = 0; j < CB; ++j)
            if (j < nc) d[j] = dS[j];
    }
}

}  // namespace

size_t backward_workspace_bytes(int N, int T_tot, int H, int dk, int dv) {
    const size_t blocks = (size_t)T_tot / BC + N;  // >= sum_n ceil(len_n / 16)
    const int ncb = (dv + CB - 1) / CB;
    const size_t a = ((blocks * H * dk * dv * sizeof(float)) + 255) & ~(size_t)255;
    const size_t b = (size_t)N * H * ncb * BC * dk * CB * sizeof(float);
    return a + b;
}

cudaError_t launch_backward(const PrefillArgs &p, const void *dout, const float *dSF, float *dq,
                            float *dk, float *dv, float *dg, float *dbeta, float *dS0,
                            void *workspace, cudaStream_t st) {
    BwdArgs a;
    a.q = p.q; a.k = p.k; a.v = p.v; a.dout = dout;
    a.g = p.g; a.beta = p.beta; a.S0 = p.S0; a.dSF = dSF; a.cu = p.cu;
    a.gq = dq; a.gk = dk; a.gv = dv; a.gg = dg; a.gbeta = dbeta; a.gS0 = dS0;
    a.dev_status = p.dev_status;
    a.N = p.N; a.T_tot = p.T_tot; a.H = p.H; a.dk = p.dk; a.dv = p.dv; a.act = p.act;
    a.ncb = (p.dv + CB - 1) / CB;
    const size_t blocks = (size_t)p.T_tot / BC + p.N;
    a.blk_states = (float *)workspace;
    a.tok_states = (float *)((uint8_t *)workspace +
                             (((blocks * p.H * p.dk * p.dv * sizeof(float)) + 255) & ~(size_t)255));
    const size_t Tn = (size_t)p.T_tot * p.H;
    cudaError_t e;
    // the row sums are accumulated by every column block: start from zero
    if ((e = cudaMemsetAsync(dq, 0, Tn * p.dk * sizeof(float), st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dk, 0, Tn * p.dk * sizeof(float), st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dg, 0, Tn * p.dk * sizeof(float), st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(dbeta, 0, Tn * sizeof(float), st)) != cudaSuccess) return e;
    if (p.N == 0 || p.H == 0) return cudaSuccess;
    dim3 grid((unsigned)(p.N * p.H), (unsigned)a.ncb);
    if (p.act == KDA_DTYPE_F32) backward_kernel<float><<<grid, BT, 0, st>>>(a);
    else backward_kernel<__nv_bfloat16><<<grid, BT, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
