// Chunked KDA prefill on CUDA cores, fp32 throughout: the path for fp32
// activations (where a 1e-4 relative bound rules out BF16/TF32 operands) and
// for shapes the tensor-core kernel does not take (dk or dv other than 128).
//
// Chunked form of the recurrence (decay, erase, write, read: "Kimi K3
// Architecture Explained", section 3), for one 16-token block starting from
// state S, with Gamma_r = g_1 + ... + g_r per key channel (|Gamma| < 80 because
// g > -5: Kimi K3 technical-report digest, section 2.1 (1)):
//   Kh = K e^{Gamma}, Kt = K e^{-Gamma}, Qh = Q e^{Gamma}, Kb = K e^{Gamma_C - Gamma}
//   L  = Diag(beta) strict_lower(Kh Kt^T),  Mq = lower(Qh Kt^T)
//   T  = (I + L)^{-1} Diag(beta),  W = T Kh,  Ut = T V
//   U  = Ut - W S,  O = Qh S + Mq U,  S <- e^{Gamma_C} * S + Kb^T U
// Columns of S are independent, so each CTA owns a block of them and redoes
// the (column-free) block preparation.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int C = 16;        // tokens per block
constexpr int NT = 256;      // threads per CTA

struct SimtSmem {
    int dk, cb, LD;
    float *S, *Kh, *Kt, *Qh, *Kb, *W, *V, *Ut, *U, *L, *Mq, *Tm, *decay, *bs;
    __device__ SimtSmem(float *base, int dk_, int cb_) : dk(dk_), cb(cb_), LD(dk_ + 1) {
        float *p = base;
        S = p; p += dk * cb;
        Kh = p; p += C * LD;
        Kt = p; p += C * LD;
        Qh = p; p += C * LD;
        Kb = p; p += C * LD;
        W = p; p += C * LD;
        V = p; p += C * cb;
        Ut = p; p += C * cb;
        U = p; p += C * cb;
        L = p; p += C * (C + 1);
        Mq = p; p += C * (C + 1);
        Tm = p; p += C * (C + 1);
        decay = p; p += dk;
        bs = p; p += C;
    }
    static size_t floats(int dk, int cb) {
        return (size_t)dk * cb + 5 * C * (dk + 1) + 3 * C * cb + 3 * C * (C + 1) + dk + C;
    }
};

template <typename TA>
__global__ void __launch_bounds__(NT) prefill_simt_kernel(PrefillArgs p, int cb, int ncb_a) {
    extern __shared__ float smem[];
    const int dk = p.dk, dv = p.dv, H = p.H, tid = threadIdx.x;
    SimtSmem sm(smem, dk, cb);
    const int LD = sm.LD;

    const int u = blockIdx.x;
    const int n = u / (H * p.seg_count);
    const int h = (u / p.seg_count) % H;
    const int s = p.seg_begin + u % p.seg_count;
    const bool transfer = p.mode == MODE_TRANSFER;
    const bool want_out = !transfer || p.emit_out;
    const bool partA = transfer && (int)blockIdx.y < ncb_a;
    const int b = partA ? (int)blockIdx.y : (int)blockIdx.y - ncb_a;
    const int c0 = b * cb;
    const int nc = min(cb, (partA ? dk : dv) - c0);
    if (nc <= 0) return;

    int t_begin, t_end;
    if (!segment_range(p.cu, n, p.N, p.T_tot, s, p.Sg, p.dev_status, t_begin, t_end)) return;

    const int seq0 = p.cu[n];
    const int cbase = p.ckpt_interval > 0 ? ckpt_base(p.cu, n, p.ckpt_interval) : 0;
    const TA *q = (const TA *)p.q;
    const TA *k = (const TA *)p.k;
    const TA *v = (const TA *)p.v;
    const size_t unit_hd = (size_t)n * H + h;

    // Initial state block.
    const float *src = nullptr;
    if (!transfer)
        src = p.seg_init ? p.seg_init + (unit_hd * p.Sg + s) * (size_t)dk * dv
                         : (p.S0 ? p.S0 + unit_hd * (size_t)dk * dv : nullptr);
    for (int e = tid; e < dk * cb; e += NT) {
        const int i = e / cb, c = e % cb;
        float x = 0.f;
        if (c < nc) {
            if (partA) x = (i == c0 + c) ? 1.f : 0.f;
            else if (src) x = src[(size_t)i * dv + c0 + c];
        }
        sm.S[e] = x;
    }
    __syncthreads();

    for (int t0 = t_begin; t0 < t_end; t0 += C) {
        const int nt = min(C, t_end - t0);
        // 1. cumulative log-decay and the scaled operands, one key channel per thread
        for (int i = tid; i < dk; i += NT) {
            float G = 0.f;
            for (int r = 0; r < C; ++r) {
                const bool ok = r < nt;
                const size_t ix = ((size_t)(t0 + r) * H + h) * dk + i;
                G += ok ? p.g[ix] : 0.f;
                const float kr = ok ? act_ld(k, ix) : 0.f;
                const float qr = (ok && want_out) ? act_ld(q, ix) : 0.f;
                const float eG = expf(G), eN = expf(-G);
                sm.Kh[r * LD + i] = kr * eG;
                sm.Kt[r * LD + i] = kr * eN;
                sm.Qh[r * LD + i] = qr * eG;
                sm.W[r * LD + i] = G;  // Gamma_r, consumed just below
            }
            sm.decay[i] = expf(G);
            for (int r = 0; r < C; ++r) {
                const bool ok = r < nt;
                const size_t ix = ((size_t)(t0 + r) * H + h) * dk + i;
                const float kr = ok ? act_ld(k, ix) : 0.f;
                sm.Kb[r * LD + i] = kr * expf(G - sm.W[r * LD + i]);
            }
        }
        for (int e = tid; e < C * cb; e += NT) {
            const int r = e / cb, c = e % cb;
            float x = 0.f;
            if (r < nt && c < nc && !partA) x = act_ld(v, ((size_t)(t0 + r) * H + h) * dv + c0 + c);
            sm.V[e] = x;
        }
        if (tid < C) sm.bs[tid] = tid < nt ? p.beta[(size_t)(t0 + tid) * H + h] : 0.f;
        __syncthreads();

        // 2. intra-block products: L (scaled by beta per row) and Mq
        for (int e = tid; e < C * C; e += NT) {
            const int r = e / C, i = e % C;
            float l = 0.f, m = 0.f;
            if (r > i) {
                for (int c = 0; c < dk; ++c) l += sm.Kh[r * LD + c] * sm.Kt[i * LD + c];
                l *= sm.bs[r];
            }
            if (want_out && r >= i)
                for (int c = 0; c < dk; ++c) m += sm.Qh[r * LD + c] * sm.Kt[i * LD + c];
            sm.L[r * (C + 1) + i] = l;
            sm.Mq[r * (C + 1) + i] = m;
        }
        __syncthreads();

        // 3. T = (I + L)^{-1} Diag(beta): forward substitution, one column per thread
        if (tid < C) {
            const int j = tid;
            float x[C];
#pragma unroll
            for (int r = 0; r < C; ++r) x[r] = 0.f;
            x[j] = 1.f;
            for (int r = j + 1; r < C; ++r) {
                float acc = 0.f;
                for (int m = j; m < r; ++m) acc += sm.L[r * (C + 1) + m] * x[m];
                x[r] = -acc;
            }
            const float bj = sm.bs[j];
            for (int r = 0; r < C; ++r) sm.Tm[r * (C + 1) + j] = r >= j ? x[r] * bj : 0.f;
        }
        __syncthreads();

        // 4. W = T Kh, Ut = T V
        for (int e = tid; e < C * dk; e += NT) {
            const int r = e / dk, c = e % dk;
            float acc = 0.f;
            for (int j = 0; j <= r; ++j) acc += sm.Tm[r * (C + 1) + j] * sm.Kh[j * LD + c];
            sm.W[r * LD + c] = acc;
        }
        for (int e = tid; e < C * cb; e += NT) {
            const int r = e / cb, c = e % cb;
            float acc = 0.f;
            for (int j = 0; j <= r; ++j) acc += sm.Tm[r * (C + 1) + j] * sm.V[j * cb + c];
            sm.Ut[e] = acc;
        }
        __syncthreads();

        // 5. U = Ut - W S
        for (int e = tid; e < C * cb; e += NT) {
            const int r = e / cb, c = e % cb;
            float acc = sm.Ut[e];
            for (int i = 0; i < dk; ++i) acc -= sm.W[r * LD + i] * sm.S[i * cb + c];
            sm.U[e] = acc;
        }
        __syncthreads();

        // 6. O = Qh S + Mq U (the identity-start chain's columns are dk wide)
        if (want_out) {
            TA *out = (TA *)(partA ? p.aux_out : p.out);
            const int ow = partA ? dk : dv;
            for (int e = tid; e < nt * cb; e += NT) {
                const int r = e / cb, c = e % cb;
                if (c >= nc) continue;
                float acc = 0.f;
                for (int i = 0; i < dk; ++i) acc += sm.Qh[r * LD + i] * sm.S[i * cb + c];
                for (int m = 0; m <= r; ++m) acc += sm.Mq[r * (C + 1) + m] * sm.U[m * cb + c];
                act_st(out, ((size_t)(t0 + r) * H + h) * ow + c0 + c, acc);
            }
            __syncthreads();
        }

        // 7. S <- e^{Gamma_C} * S + Kb^T U
        for (int e = tid; e < dk * cb; e += NT) {
            const int i = e / cb, c = e % cb;
            float acc = sm.decay[i] * sm.S[e];
            for (int r = 0; r < C; ++r) acc += sm.Kb[r * LD + i] * sm.U[r * cb + c];
            sm.S[e] = acc;
        }
        __syncthreads();

        if (p.ckpt_interval > 0) {  // state checkpoint after this block
            const int done = t0 + nt - seq0;
            float *d = partA ? p.ckpt_a : p.ckpt;
            const int ldd = partA ? dk : dv;
            if (done % p.ckpt_interval == 0 && d) {
                d += ((size_t)(cbase + done / p.ckpt_interval - 1) * H + h) * (size_t)dk * ldd;
                for (int e = tid; e < dk * cb; e += NT) {
                    const int i = e / cb, c = e % cb;
                    if (c < nc) d[(size_t)i * ldd + c0 + c] = sm.S[e];
                }
            }
        }
    }

    // Write the state block out.
    float *dst = nullptr;
    int ld = dv;
    if (!transfer) {
        if (s == p.Sg - 1 && p.S_final) dst = p.S_final + unit_hd * (size_t)dk * dv;
    } else if (partA) {
        dst = p.transfer + (unit_hd * p.Sg + s) * (size_t)dk * dk;
        ld = dk;
    } else {
        dst = p.zero_state + (unit_hd * p.Sg + s) * (size_t)dk * dv;
    }
    if (dst)
        for (int e = tid; e < dk * cb; e += NT) {
            const int i = e / cb, c = e % cb;
            if (c < nc) dst[(size_t)i * ld + c0 + c] = sm.S[e];
        }
}

}  // namespace

cudaError_t launch_prefill_simt(const PrefillArgs &a, cudaStream_t st) {
    const int cb = a.dv <= 32 ? a.dv : 32;
    const int ncb_v = (a.dv + cb - 1) / cb;
    const int ncb_a = a.mode == MODE_TRANSFER ? (a.dk + cb - 1) / cb : 0;
    const int units = a.N * a.H * a.seg_count;
    if (units == 0) return cudaSuccess;
    const size_t smem = SimtSmem::floats(a.dk, cb) * sizeof(float);
    dim3 grid(units, ncb_v + ncb_a);
    cudaError_t e;
    if (a.act == KDA_DTYPE_F32) {
        e = set_max_dynamic_smem((const void *)prefill_simt_kernel<float>, (int)smem);
        if (e != cudaSuccess) return e;
        prefill_simt_kernel<float><<<grid, NT, smem, st>>>(a, cb, ncb_a);
    } else {
        e = set_max_dynamic_smem((const void *)prefill_simt_kernel<__nv_bfloat16>, (int)smem);
        if (e != cudaSuccess) return e;
        prefill_simt_kernel<__nv_bfloat16><<<grid, NT, smem, st>>>(a, cb, ncb_a);
    }
    return cudaGetLastError();
}

}  // namespace kda
