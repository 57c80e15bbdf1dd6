// Gradient pass of the chunked backward (BF16, dk = dv = 128): one CTA per
// (16-token block, head), all blocks in parallel.
//
// The forward recurrence ("Kimi K3 Architecture Explained", section 3: decay,
// then erase, then write, then read), in the chunked form of its 16-token
// blocks (Kimi K3 technical-report digest, section 2.1 (1)): from the block's
// start state S,
//     Kh = K e^{Gamma}, Kt = K e^{-Gamma}, Qh = Q e^{Gamma}, Kb = K e^{Gamma_C - Gamma},
//     L = strict_lower(Kh Kt^T), Mq = lower(Qh Kt^T), Y = (I + Diag(beta) L)^{-1},
//     T = Y Diag(beta), R = V - Kh S, U = T R,
//     O = Qh S + Mq U,   S' = Diag(e^{Gamma_C}) S + Kb^T U.
// Given S (the forward chain's state at the block start) and dS' (the adjoint
// chain's adjoint of S'), every gradient of the block follows from the block's
// own inputs (the adjoint of the chunked form, term by term):
//     dU = Mq^T dO + Kb dS';   dR = T^T dU;  dv = dR;   dT = dU R^T;
//     dbeta_j = sum_i dT_ij Y_ij,  dMb = -Y^T (dT Diag(beta)) Y^T,
//     dbeta_i += sum_j dMb_ij L_ij,  dL = strict_lower(Diag(beta) dMb);
//     dMq = lower(dO U^T);
//     dQh = dO S^T + dMq Kt;  dKh = -dR S^T + dL Kt;  dKb = U dS'^T;
//     dKt = dL^T Kh + dMq^T Qh;  deC = rowsum(dS' o S);
//     dk = dKh e^{Gamma} + dKt e^{-Gamma} + dKb e^{Gamma_C - Gamma};  dq = dQh e^{Gamma};
//     dGamma = dKh o Kh - dKt o Kt + dQh o Qh - dKb o Kb, its last row plus
//              sum_r (dKb o Kb)_r + deC o e^{Gamma_C};  dg = reverse cumsum of dGamma.
// The products with S and dS' (16 x 128 x 128) and the 16 x 16 x 128 ones run on
// mma.sync with BF16 operands and fp32 accumulation; the 16 x 16 algebra (Y, T,
// dMb, dL) and the elementwise factors in fp32.  Warp w owns columns [16 w, 16 w +
// 16) of every 128-wide product.  Rows past the block's end (the last, partial
// block of a sequence) carry no decay, no key, query, value or output gradient, so
// they contribute nothing and are not written.
#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int C = 16, D = 128;
constexpr int GW = 8, GT = GW * 32;

// shared memory: BF16 tiles in 256-byte rows, 16-byte chunk c of row r at c ^ (r & 7)
constexpr int T_ST = 0;                   // S^T  [128 j][128 i]
constexpr int T_DS = T_ST + 32768;        // dS'^T [128 j][128 i]
constexpr int T_KH = T_DS + 32768;        // [16 r][128 i]
constexpr int T_KT = T_KH + 4096;
constexpr int T_QH = T_KT + 4096;
constexpr int T_KB = T_QH + 4096;
constexpr int T_R = T_KB + 4096;          // [16 r][128 j]
constexpr int T_U = T_R + 4096;
constexpr int T_DU = T_U + 4096;
constexpr int T_NDR = T_DU + 4096;        // -dR
// Row strides of the token-by-channel arrays that are read element-wise: BS BF16
// elements (272-byte rows) and FS floats (544-byte rows).  Lanes of a fragment read
// 8 rows at once; with dense rows those share banks (8-way conflicts), with 68- or
// 136-word rows their 4- and 8-byte reads fall on distinct banks.
constexpr int BS = 136, FS = 136;
// Input buffers, two, alternating between consecutive blocks of a CTA: raw q, k, v
// rows [16][BS] BF16, dO [16][128 j] BF16 (swizzled), g [16][FS] fp32, beta [16]
constexpr int IB_Q = 0, IB_K = IB_Q + C * BS * 2, IB_V = IB_K + C * BS * 2;
constexpr int IB_DO = IB_V + C * BS * 2, IB_G = IB_DO + 4096, IB_BETA = IB_G + C * FS * 4;
constexpr int IB_SIZE = IB_BETA + 128;
static_assert(IB_DO % 128 == 0 && IB_G % 128 == 0 && IB_SIZE % 128 == 0, "input buffer alignment");
constexpr int IB0 = T_NDR + 4096;
constexpr int F_EP = IB0 + 2 * IB_SIZE;   // e^{Gamma} [16][FS]
constexpr int F_EM = F_EP + C * FS * 4;   // e^{-Gamma} [16][FS]
constexpr int F_EB = F_EM + C * FS * 4;   // e^{Gamma_C - Gamma} [16][FS]
constexpr int F_DGAM = F_EB + C * FS * 4; // dGamma [16][FS] fp32
constexpr int F_PART = F_DGAM + C * FS * 4;  // partial 16 x 16 products [GW][2][16][16] fp32
constexpr int SQ = 17;                    // fp32 16 x 16 row stride
constexpr int F_SMALL = F_PART + GW * 2 * 256 * 4;   // fp32 16 x 16: L, Mq, Y, dT, dMq, P
enum { SM_L = 0, SM_MQ, SM_Y, SM_DT, SM_DMQ, SM_P, SM_DMB, NSMALL };
constexpr int TS = 24;                    // BF16 16 x 16 rows: 16 + pad (48 bytes)
constexpr int B_SMALL = F_SMALL + NSMALL * 16 * SQ * 4;  // BF16: T, Mq, dMq, dL
enum { SB_T = 0, SB_MQ, SB_DMQ, SB_DL, NSB };
constexpr int F_VEC = B_SMALL + NSB * 16 * TS * 2;       // eC [128], deC [128]
constexpr int SMEM_BYTES = F_VEC + (128 + 128) * 4;
static_assert(IB_SIZE % 128 == 0 && IB0 % 128 == 0, "input buffer alignment");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");

struct GradArgs {
    const __nv_bfloat16 *q, *k, *v, *dout;
    const float *g, *beta, *S0;
    const int32_t *cu;
    const __nv_bfloat16 *Sck;   // forward states after every 32 tokens: slot ckpt_base(n, 32) + m
    const __nv_bfloat16 *dSck;  // adjoints at every block end: slot block_base(n) + c
    float *dq, *dk, *dv, *dg, *dbeta;
    int N, T_tot, H;
};

__device__ __forceinline__ uint32_t sw(int row, int chunk) {
    return (uint32_t)(row * 256 + ((chunk ^ (row & 7)) << 4));
}

__global__ void __launch_bounds__(GT, 1) bwd_chunk_kernel(const __grid_constant__ GradArgs a) {
    extern __shared__ __align__(128) uint8_t sm[];
    const uint32_t sb = smem_addr(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g8 = lane >> 2, t4 = lane & 3;
    // The work: pairs of 16-token blocks (2p, 2p + 1) of a sequence, for every head,
    // pairs counted over all sequences.  CTA x takes pair items x, x + gridDim.x,
    // ..., and of each the even block, then the odd one.  The forward chain stored
    // the state after every 32 tokens, i.e. at the start of every even block; the
    // start state of an odd block is formed here from the even block's S, U and
    // Kb.  While one block is computed, the next one's inputs are in flight into
    // the other input buffer, and its tiles are requested as soon as this one's
    // last products have read them.
    int npair = 0;
    for (int m = 0; m < a.N; ++m) npair += ((a.cu[m + 1] - a.cu[m] + C - 1) / C + 1) / 2;
    const long long items = (long long)npair * a.H;
    const long long G = gridDim.x;
    const size_t row_stride = (size_t)a.H * D;  // elements between tokens
    struct Item {
        bool ok, odd;
        long long it;
        int n, c, h, t0, nt, cbase, sbase;
    };
    auto fill = [&](Item &w) {
        w.t0 = a.cu[w.n] + C * w.c;
        w.nt = min(C, a.cu[w.n + 1] - w.t0);
    };
    auto pair_item = [&](long long it) {  // the even block of pair item it
        Item w{};
        w.it = it;
        w.ok = it < items;
        if (!w.ok) return w;
        w.h = (int)(it / npair);
        int q = (int)(it % npair), n = 0, cb = 0, sbs = 0;
        for (;; ++n) {
            if (n >= a.N) {  // (only with inconsistent lengths)
                w.ok = false;
                return w;
            }
            const int len = a.cu[n + 1] - a.cu[n];
            const int nb = (len + C - 1) / C;
            if (q < (nb + 1) / 2) break;
            q -= (nb + 1) / 2;
            cb += nb;
            sbs += len / (2 * C);
        }
        w.n = n;
        w.c = 2 * q;
        w.cbase = cb;
        w.sbase = sbs;
        fill(w);
        return w;
    };
    auto next_of = [&](const Item &w) {
        if (!w.ok) return w;
        if (!w.odd && w.t0 + C < a.cu[w.n + 1]) {  // the odd block of the same pair
            Item v = w;
            v.odd = true;
            v.c = w.c + 1;
            fill(v);
            return v;
        }
        return pair_item(w.it + G);
    };
    // the block's inputs, rows past its end zero-filled
    auto issue_inputs = [&](const Item &w, int ibo) {
        const size_t base = ((size_t)w.t0 * a.H + w.h) * D;
        for (int e = tid; e < 4 * C * 16; e += GT) {  // q, k, v, dO: 16 rows x 16 chunks
            const int arr = e >> 8, r = (e >> 4) & 15, cc = e & 15;
            const __nv_bfloat16 *src = arr == 0 ? a.q : arr == 1 ? a.k : arr == 2 ? a.v : a.dout;
            const uint32_t dst = arr == 3 ? sb + ibo + IB_DO + sw(r, cc)
                                          : sb + ibo + (arr == 0 ? IB_Q : arr == 1 ? IB_K : IB_V) +
                                                r * (BS * 2) + 16 * cc;
            cp_async16(dst, src + base + (r < w.nt ? r : 0) * row_stride + 8 * cc, r < w.nt);
        }
        for (int e = tid; e < C * 32; e += GT) {  // g: 16 rows x 32 float4
            const int r = e >> 5, c4 = e & 31;
            cp_async16(sb + ibo + IB_G + r * (FS * 4) + 16 * c4,
                       a.g + base + (r < w.nt ? r : 0) * row_stride + 4 * c4, r < w.nt);
        }
        if (tid < C)
            cp_async4(sb + ibo + IB_BETA + 4 * tid,
                      a.beta + (size_t)(w.t0 + (tid < w.nt ? tid : 0)) * a.H + w.h, tid < w.nt);
    };
    // dS'^T (the adjoint at the block's end) and, for an even block, S^T (the forward
    // state after the previous block, or the sequence's initial state)
    auto issue_tiles = [&](const Item &w) {
        const __nv_bfloat16 *dsrc = a.dSck + ((size_t)(w.cbase + w.c) * a.H + w.h) * D * D;
        for (int e = tid; e < D * 16; e += GT) {
            const int j = e >> 4, cc = e & 15;
            cp_async16(sb + T_DS + sw(j, cc), dsrc + (size_t)j * D + 8 * cc, true);
        }
        if (w.odd) {
            // formed from the even block's data (next_state)
        } else if (w.c > 0) {
            const __nv_bfloat16 *ssrc = a.Sck + ((size_t)(w.sbase + w.c / 2 - 1) * a.H + w.h) * D * D;
            for (int e = tid; e < D * 16; e += GT) {
                const int j = e >> 4, cc = e & 15;
                cp_async16(sb + T_ST + sw(j, cc), ssrc + (size_t)j * D + 8 * cc, true);
            }
        } else {  // fp32 [i][j] or zeros, converted here
            const float *s0 = a.S0 ? a.S0 + ((size_t)w.n * a.H + w.h) * D * D : nullptr;
            for (int e = tid; e < D * D / 2; e += GT) {
                const int j = e & 127, i2 = e >> 7;  // channels 2 i2, 2 i2 + 1 of column j
                const float x0 = s0 ? s0[(size_t)(2 * i2) * D + j] : 0.f;
                const float x1 = s0 ? s0[(size_t)(2 * i2 + 1) * D + j] : 0.f;
                *(uint32_t *)(sm + T_ST + sw(j, i2 >> 2) + 4 * (i2 & 3)) = pack_bf16x2(x0, x1);
            }
        }
    };

    Item cur = pair_item(blockIdx.x), nxt = next_of(cur);
    if (!cur.ok) return;
    // copy groups in flight, oldest first: inputs(k), tiles(k), inputs(k + 1)
    issue_inputs(cur, IB0);
    cp_async_commit();
    issue_tiles(cur);
    cp_async_commit();
    if (nxt.ok) issue_inputs(nxt, IB0 + IB_SIZE);
    cp_async_commit();
    for (int k = 0;; ++k) {
    const int ibo = IB0 + (k & 1) * IB_SIZE;
    const int h = cur.h, t0 = cur.t0, nt = cur.nt;
    cp_async_wait_group<2>();  // this block's inputs
    __syncthreads();

    const float *fG = (const float *)(sm + ibo + IB_G);
    float *fEp = (float *)(sm + F_EP), *fEm = (float *)(sm + F_EM), *fEb = (float *)(sm + F_EB);
    float *beta = (float *)(sm + ibo + IB_BETA), *eC = (float *)(sm + F_VEC), *deC = eC + 128;
    auto small = [&](int which) { return (float *)(sm + F_SMALL) + which * 16 * SQ; };
    auto sbf = [&](int which) { return (__nv_bfloat16 *)(sm + B_SMALL) + which * 16 * TS; };

    // ---- elementwise factors, two threads per key channel: threads 0-127 take the
    // running product of alpha = e^g (e^{Gamma_r}: Kh, Qh), threads 128-255 the
    // reverse one (e^{Gamma_C - Gamma_r}: Kb; e^{-Gamma_r} = e^{Gamma_C - Gamma_r} /
    // e^{Gamma_C}: Kt; e^{Gamma_C} itself)
    {
        const int i = tid & (D - 1);
        const bool fwd_half = tid < D;
        float al[C];
#pragma unroll
        for (int r = 0; r < C; ++r) al[r] = __expf(fG[r * FS + i]);
        const __nv_bfloat16 *kr = (const __nv_bfloat16 *)(sm + ibo + IB_K);
        const __nv_bfloat16 *qr = (const __nv_bfloat16 *)(sm + ibo + IB_Q);
        if (fwd_half) {
            float run = 1.f;
#pragma unroll
            for (int r = 0; r < C; ++r) {
                run *= al[r];
                const float kv = __bfloat162float(kr[r * BS + i]), qv = __bfloat162float(qr[r * BS + i]);
                fEp[r * FS + i] = run;
                const uint32_t off = sw(r, i >> 3) + 2 * (i & 7);
                *(__nv_bfloat16 *)(sm + T_KH + off) = __float2bfloat16_rn(kv * run);
                *(__nv_bfloat16 *)(sm + T_QH + off) = __float2bfloat16_rn(qv * run);
            }
        } else {
            float rev[C];
            float b = 1.f;
#pragma unroll
            for (int r = C - 1; r >= 0; --r) { rev[r] = b; b *= al[r]; }
            const float einv = 1.f / b;  // b = e^{Gamma_C}
            eC[i] = b;
#pragma unroll
            for (int r = 0; r < C; ++r) {
                const float kv = __bfloat162float(kr[r * BS + i]);
                const float em = rev[r] * einv;
                fEm[r * FS + i] = em;
                fEb[r * FS + i] = rev[r];
                const uint32_t off = sw(r, i >> 3) + 2 * (i & 7);
                *(__nv_bfloat16 *)(sm + T_KT + off) = __float2bfloat16_rn(kv * em);
                *(__nv_bfloat16 *)(sm + T_KB + off) = __float2bfloat16_rn(kv * rev[r]);
            }
        }
    }
    __syncthreads();

    // fragment loaders (see the layout notes in the header of kda_prefill_tc.cu):
    // A 16 x 16 at k-step kk of a [16][128] tile
    auto lda = [&](int tile, int kk, uint32_t (&f)[4]) {
        const int row = (lane & 7) + 8 * ((lane >> 3) & 1);
        ldsm_x4(sb + tile + sw(row, 2 * kk + (lane >> 4)), f);
    };
    // B (k x 2 n-tiles) from rows = n with k contiguous: rows n0.., k chunks kc0, kc0 + 1
    auto ldb_nt = [&](int tile, int n0, int kc0, uint32_t (&f)[4]) {
        const int row = n0 + (lane & 7) + 8 * (lane >> 4);
        ldsm_x4(sb + tile + sw(row, kc0 + ((lane >> 3) & 1)), f);
    };
    // B (16 k x 2 n-tiles) from rows = k with n contiguous: k rows k0.., columns n0..
    auto ldb_t = [&](int tile, int k0, int n0, uint32_t (&f)[4]) {
        const int row = k0 + (lane & 7) + 8 * ((lane >> 3) & 1);
        ldsm_x4_t(sb + tile + sw(row, (n0 >> 3) + (lane >> 4)), f);
    };
    // A = M or M^T for a BF16 16 x 16 small matrix M ([16][TS])
    auto lda_small = [&](const __nv_bfloat16 *M, bool trans, uint32_t (&f)[4]) {
        const uint32_t base = smem_addr(M);
        if (!trans) {
            const int row = (lane & 7) + 8 * ((lane >> 3) & 1), col = 8 * (lane >> 4);
            ldsm_x4(base + (row * TS + col) * 2, f);
        } else {
            const int row = (lane & 7) + 8 * (lane >> 4), col = 8 * ((lane >> 3) & 1);
            ldsm_x4_t(base + (row * TS + col) * 2, f);
        }
    };
    float *part = (float *)(sm + F_PART) + warp * 2 * 256;
    auto put_part = [&](int which, const float (&acc)[2][4]) {  // 16 x 16 partial
#pragma unroll
        for (int nb = 0; nb < 2; ++nb)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                part[which * 256 + (g8 + 8 * (e >> 1)) * 16 + nb * 8 + 2 * t4 + (e & 1)] = acc[nb][e];
    };
    auto sum_parts = [&](int which, int r, int cc) {
        const float *p0 = (const float *)(sm + F_PART);
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < GW; ++w) s += p0[w * 512 + which * 256 + r * 16 + cc];
        return s;
    };

    // ---- L = strict_lower(Kh Kt^T), Mq = lower(Qh Kt^T) (16 x 16 x 128) and Y = (I +
    // Diag(beta) L)^{-1}, all in warp 0: the full products take it a few hundred
    // cycles, less than partial products summed across the warps behind a barrier
    if (warp == 0) {
        float accL[2][4] = {}, accM[2][4] = {};
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t af[4], aq[4], bf[4];
            lda(T_KH, kk, af);
            lda(T_QH, kk, aq);
            ldb_nt(T_KT, 0, 2 * kk, bf);  // B[k = i][n = r'] = Kt[r'][i]
            mma_bf16_16816(accL[0], af, bf[0], bf[1]);
            mma_bf16_16816(accL[1], af, bf[2], bf[3]);
            mma_bf16_16816(accM[0], aq, bf[0], bf[1]);
            mma_bf16_16816(accM[1], aq, bf[2], bf[3]);
        }
#pragma unroll
        for (int nb = 0; nb < 2; ++nb)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = g8 + 8 * (e >> 1), cc = nb * 8 + 2 * t4 + (e & 1);
                const float mq = cc <= r ? accM[nb][e] : 0.f;
                small(SM_L)[r * SQ + cc] = cc < r ? accL[nb][e] : 0.f;
                small(SM_MQ)[r * SQ + cc] = mq;
                sbf(SB_MQ)[r * TS + cc] = __float2bfloat16_rn(mq);
            }
        __syncwarp();
        // forward substitution, lane = column (fp32)
        if (lane < C) {
            const int j = lane;
            const float *L = small(SM_L);
            float y[C];
#pragma unroll
            for (int r = 0; r < C; ++r) {
                float s = r == j ? 1.f : 0.f;
#pragma unroll
                for (int m = 0; m < r; ++m) s -= beta[r] * L[r * SQ + m] * y[m];
                y[r] = r < j ? 0.f : s;
            }
#pragma unroll
            for (int r = 0; r < C; ++r) {
                small(SM_Y)[r * SQ + j] = y[r];
                sbf(SB_T)[r * TS + j] = __float2bfloat16_rn(y[r] * beta[j]);  // T = Y Diag(beta)
            }
        }
    }
    cp_async_wait_group<1>();  // this block's S^T and dS'^T
    __syncthreads();

    const int j0 = 16 * warp;  // this warp's 16 value columns (then key channels)
    // ---- R = V - Kh S and dU = Mq^T dO + Kb dS' over columns j0..j0+15
    float Rf[2][4] = {}, dUf[2][4] = {};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        uint32_t a1[4], a2[4], b1[4], b2[4];
        lda(T_KH, kk, a1);
        lda(T_KB, kk, a2);
        ldb_nt(T_ST, j0, 2 * kk, b1);  // B[k = i][n = j] = S^T[j][i]
        ldb_nt(T_DS, j0, 2 * kk, b2);
        mma_bf16_16816(Rf[0], a1, b1[0], b1[1]);
        mma_bf16_16816(Rf[1], a1, b1[2], b1[3]);
        mma_bf16_16816(dUf[0], a2, b2[0], b2[1]);
        mma_bf16_16816(dUf[1], a2, b2[2], b2[3]);
    }
    {
        uint32_t am[4], bd[4];
        lda_small(sbf(SB_MQ), true, am);  // Mq^T
        ldb_t(ibo + IB_DO, 0, j0, bd);    // B[k = r'][n = j] = dO[r'][j]
        mma_bf16_16816(dUf[0], am, bd[0], bd[1]);
        mma_bf16_16816(dUf[1], am, bd[2], bd[3]);
    }
    // R = V - Kh S (V from the raw rows), both to shared memory as BF16
    const __nv_bfloat16 *vr = (const __nv_bfloat16 *)(sm + ibo + IB_V);
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int r = g8 + 8 * hh, j = j0 + 8 * nb + 2 * t4;
            const float2 v2 = __bfloat1622float2(*(const __nv_bfloat162 *)(vr + r * BS + j));
            Rf[nb][2 * hh] = v2.x - Rf[nb][2 * hh];
            Rf[nb][2 * hh + 1] = v2.y - Rf[nb][2 * hh + 1];
            const uint32_t off = sw(r, j >> 3) + 2 * (j & 7);
            *(uint32_t *)(sm + T_R + off) = pack_bf16x2(Rf[nb][2 * hh], Rf[nb][2 * hh + 1]);
            *(uint32_t *)(sm + T_DU + off) = pack_bf16x2(dUf[nb][2 * hh], dUf[nb][2 * hh + 1]);
        }
    __syncwarp();  // this warp's columns of R and dU are in place
    // ---- U = T R, dR = T^T dU (columns j0..), dv = dR
    float Uf[2][4] = {}, dRf[2][4] = {};
    {
        uint32_t at[4], att[4], br[4], bu[4];
        lda_small(sbf(SB_T), false, at);
        lda_small(sbf(SB_T), true, att);
        ldb_t(T_R, 0, j0, br);
        ldb_t(T_DU, 0, j0, bu);
        mma_bf16_16816(Uf[0], at, br[0], br[1]);
        mma_bf16_16816(Uf[1], at, br[2], br[3]);
        mma_bf16_16816(dRf[0], att, bu[0], bu[1]);
        mma_bf16_16816(dRf[1], att, bu[2], bu[3]);
    }
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int r = g8 + 8 * hh, j = j0 + 8 * nb + 2 * t4;
            const uint32_t off = sw(r, j >> 3) + 2 * (j & 7);
            *(uint32_t *)(sm + T_U + off) = pack_bf16x2(Uf[nb][2 * hh], Uf[nb][2 * hh + 1]);
            *(uint32_t *)(sm + T_NDR + off) = pack_bf16x2(-dRf[nb][2 * hh], -dRf[nb][2 * hh + 1]);
            if (r < nt)
                *(float2 *)(a.dv + ((size_t)(t0 + r) * a.H + h) * D + j) =
                    make_float2(dRf[nb][2 * hh], dRf[nb][2 * hh + 1]);
        }
    __syncwarp();
    // ---- partial dT = dU R^T and dMq = dO U^T over this warp's columns
    {
        float accT[2][4] = {}, accM[2][4] = {};
        uint32_t adu[4], ado[4], br[4], bu[4];
        lda(T_DU, warp, adu);
        lda(ibo + IB_DO, warp, ado);
        ldb_nt(T_R, 0, 2 * warp, br);  // B[k = j][n = r'] = R[r'][j]
        ldb_nt(T_U, 0, 2 * warp, bu);
        mma_bf16_16816(accT[0], adu, br[0], br[1]);
        mma_bf16_16816(accT[1], adu, br[2], br[3]);
        mma_bf16_16816(accM[0], ado, bu[0], bu[1]);
        mma_bf16_16816(accM[1], ado, bu[2], bu[3]);
        put_part(0, accT);
        put_part(1, accM);
    }
    // deC[i] = sum_j dS'[i][j] S[i][j]: thread (chunk of 8 channels, group of 8
    // columns j) multiplies 16-byte pieces of both tiles; the 16 groups' partial
    // sums are added after the barrier
    {
        const int cc = tid & 15, jg = tid >> 4;
        float acc8[8] = {};
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
            const int j = 8 * jg + jj;
            const uint4 dsv = *(const uint4 *)(sm + T_DS + sw(j, cc));
            const uint4 stv = *(const uint4 *)(sm + T_ST + sw(j, cc));
            const __nv_bfloat162 *d2 = (const __nv_bfloat162 *)&dsv;
            const __nv_bfloat162 *s2 = (const __nv_bfloat162 *)&stv;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 a2 = __bfloat1622float2(d2[e]), b2 = __bfloat1622float2(s2[e]);
                acc8[2 * e] = fmaf(a2.x, b2.x, acc8[2 * e]);
                acc8[2 * e + 1] = fmaf(a2.y, b2.y, acc8[2 * e + 1]);
            }
        }
        float *part16 = (float *)(sm + F_DGAM);  // [16 groups][128 channels], scratch
        *(float4 *)(part16 + jg * D + 8 * cc) = make_float4(acc8[0], acc8[1], acc8[2], acc8[3]);
        *(float4 *)(part16 + jg * D + 8 * cc + 4) = make_float4(acc8[4], acc8[5], acc8[6], acc8[7]);
    }
    __syncthreads();
    {
        const int r = tid >> 4, cc = tid & 15;
        small(SM_DT)[r * SQ + cc] = sum_parts(0, r, cc);
        if (tid < D) {
            const float *part16 = (const float *)(sm + F_DGAM);
            float sdc = 0.f;
#pragma unroll
            for (int gq = 0; gq < 16; ++gq) sdc += part16[gq * D + tid];
            deC[tid] = sdc;
        }
        const float dmq = cc <= r ? sum_parts(1, r, cc) : 0.f;
        small(SM_DMQ)[r * SQ + cc] = dmq;
        sbf(SB_DMQ)[r * TS + cc] = __float2bfloat16_rn(dmq);

    }
    __syncthreads();
    // ---- the 16 x 16 algebra of T = Y Diag(beta), Y = (I + Diag(beta) L)^{-1}
    {
        const int r = tid >> 4, cc = tid & 15;
        const float *Y = small(SM_Y), *dT = small(SM_DT);
        // P = Y^T (dT Diag(beta))
        float pz = 0.f;
#pragma unroll
        for (int i = 0; i < C; ++i) pz += Y[i * SQ + r] * dT[i * SQ + cc] * beta[cc];
        small(SM_P)[r * SQ + cc] = pz;
    }
    __syncthreads();
    {
        const int r = tid >> 4, cc = tid & 15;
        const float *Y = small(SM_Y), *P = small(SM_P);
        float d = 0.f;  // dMb = -P Y^T
#pragma unroll
        for (int b = 0; b < C; ++b) d -= P[r * SQ + b] * Y[cc * SQ + b];
        small(SM_DMB)[r * SQ + cc] = d;
        sbf(SB_DL)[r * TS + cc] = __float2bfloat16_rn(cc < r ? beta[r] * d : 0.f);
    }
    __syncthreads();
    if (tid < C) {  // dbeta of row tid
        const int j = tid;
        const float *Y = small(SM_Y), *dT = small(SM_DT), *dMb = small(SM_DMB), *L = small(SM_L);
        float db = 0.f;
#pragma unroll
        for (int i = 0; i < C; ++i) db += dT[i * SQ + j] * Y[i * SQ + j] + dMb[j * SQ + i] * L[j * SQ + i];
        if (j < nt) a.dbeta[(size_t)(t0 + j) * a.H + h] = db;
    }

    // ---- over key channels i0..i0+15: dQh, dKh, dKb, dKt
    const int i0 = 16 * warp;
    float dQh[2][4] = {}, dKh[2][4] = {}, dKb[2][4] = {}, dKt[2][4] = {};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        uint32_t ad[4], an[4], au[4], bs[4], bd[4];
        lda(ibo + IB_DO, kk, ad);
        lda(T_NDR, kk, an);
        lda(T_U, kk, au);
        ldb_t(T_ST, 16 * kk, i0, bs);  // B[k = j][n = i] = S^T[j][i]
        ldb_t(T_DS, 16 * kk, i0, bd);
        mma_bf16_16816(dQh[0], ad, bs[0], bs[1]);
        mma_bf16_16816(dQh[1], ad, bs[2], bs[3]);
        mma_bf16_16816(dKh[0], an, bs[0], bs[1]);
        mma_bf16_16816(dKh[1], an, bs[2], bs[3]);
        mma_bf16_16816(dKb[0], au, bd[0], bd[1]);
        mma_bf16_16816(dKb[1], au, bd[2], bd[3]);
    }
    {
        uint32_t admq[4], adl[4], admqt[4], adlt[4], bkt[4], bkh[4], bqh[4];
        lda_small(sbf(SB_DMQ), false, admq);
        lda_small(sbf(SB_DL), false, adl);
        lda_small(sbf(SB_DMQ), true, admqt);
        lda_small(sbf(SB_DL), true, adlt);
        ldb_t(T_KT, 0, i0, bkt);  // B[k = r'][n = i] = Kt[r'][i]
        ldb_t(T_KH, 0, i0, bkh);
        ldb_t(T_QH, 0, i0, bqh);
        mma_bf16_16816(dQh[0], admq, bkt[0], bkt[1]);
        mma_bf16_16816(dQh[1], admq, bkt[2], bkt[3]);
        mma_bf16_16816(dKh[0], adl, bkt[0], bkt[1]);
        mma_bf16_16816(dKh[1], adl, bkt[2], bkt[3]);
        mma_bf16_16816(dKt[0], adlt, bkh[0], bkh[1]);
        mma_bf16_16816(dKt[1], adlt, bkh[2], bkh[3]);
        mma_bf16_16816(dKt[0], admqt, bqh[0], bqh[1]);
        mma_bf16_16816(dKt[1], admqt, bqh[2], bqh[3]);
    }
    // ---- elementwise: dk, dq and dGamma (fp32 factors), then dg per channel
    float *dgam = (float *)(sm + F_DGAM);
    float *kbk = (float *)(sm + F_PART);  // dKb o Kb [16][128] (the partials are consumed)
    const __nv_bfloat16 *kraw = (const __nv_bfloat16 *)(sm + ibo + IB_K);
    const __nv_bfloat16 *qraw = (const __nv_bfloat16 *)(sm + ibo + IB_Q);
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int r = g8 + 8 * hh, i = i0 + 8 * nb + 2 * t4;
            // channels i, i + 1 of row r: one 8-byte read per fp32 array, one 4-byte
            // read per BF16 row
            const float2 ep2 = *(const float2 *)(fEp + r * FS + i);
            const float2 em2 = *(const float2 *)(fEm + r * FS + i);
            const float2 eb2 = *(const float2 *)(fEb + r * FS + i);
            const float2 kv2 = __bfloat1622float2(*(const __nv_bfloat162 *)(kraw + r * BS + i));
            const float2 qv2 = __bfloat1622float2(*(const __nv_bfloat162 *)(qraw + r * BS + i));
            float dk2[2], dq2[2], dg2[2], kb2[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int q4 = 2 * hh + e;
                const float ep = e ? ep2.y : ep2.x, em = e ? em2.y : em2.x, eb = e ? eb2.y : eb2.x;
                const float kv = e ? kv2.y : kv2.x, qv = e ? qv2.y : qv2.x;
                dk2[e] = dKh[nb][q4] * ep + dKt[nb][q4] * em + dKb[nb][q4] * eb;
                dq2[e] = dQh[nb][q4] * ep;
                kb2[e] = dKb[nb][q4] * kv * eb;
                dg2[e] = dKh[nb][q4] * kv * ep - dKt[nb][q4] * kv * em + dQh[nb][q4] * qv * ep -
                         kb2[e];
            }
            *(float2 *)(dgam + r * FS + i) = make_float2(dg2[0], dg2[1]);
            *(float2 *)(kbk + r * FS + i) = make_float2(kb2[0], kb2[1]);
            if (r < nt) {
                const size_t o = ((size_t)(t0 + r) * a.H + h) * D + i;
                *(float2 *)(a.dk + o) = make_float2(dk2[0], dk2[1]);
                *(float2 *)(a.dq + o) = make_float2(dq2[0], dq2[1]);
            }
        }
    __syncthreads();  // every read of S^T and dS'^T is done: the next block's tiles
    const Item nx2 = next_of(nxt);
    if (nxt.ok) issue_tiles(nxt);
    cp_async_commit();
    if (nxt.ok && nxt.odd) {
        // S^T of the odd block: S^T Diag(e^{Gamma_C}) + U^T Kb of this one, this
        // warp's rows j of the S^T tile in place (every element is read and
        // written by the lane that holds it in the fragments)
        const int jw = 16 * warp;
        uint32_t au[4];  // A = U^T (rows j, k = r) from the [16 r][128 j] U tile
        {
            const int mi = lane >> 3, row = (lane & 7) + 8 * (mi >> 1);
            ldsm_x4_t(sb + T_U + sw(row, (jw >> 3) + (mi & 1)), au);
        }
        float acc[16][4];
#pragma unroll
        for (int nt8 = 0; nt8 < 16; ++nt8)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int j = jw + g8 + 8 * hh, i = 8 * nt8 + 2 * t4;
                const float2 sv = __bfloat1622float2(
                    *(const __nv_bfloat162 *)(sm + T_ST + sw(j, i >> 3) + 2 * (i & 7)));
                acc[nt8][2 * hh] = sv.x * eC[i];
                acc[nt8][2 * hh + 1] = sv.y * eC[i + 1];
            }
#pragma unroll
        for (int np = 0; np < 8; ++np) {
            uint32_t bk[4];
            ldb_t(T_KB, 0, 16 * np, bk);  // B[k = r][n = i] = Kb[r][i]
            mma_bf16_16816(acc[2 * np], au, bk[0], bk[1]);
            mma_bf16_16816(acc[2 * np + 1], au, bk[2], bk[3]);
        }
#pragma unroll
        for (int nt8 = 0; nt8 < 16; ++nt8)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int j = jw + g8 + 8 * hh, i = 8 * nt8 + 2 * t4;
                *(uint32_t *)(sm + T_ST + sw(j, i >> 3) + 2 * (i & 7)) =
                    pack_bf16x2(acc[nt8][2 * hh], acc[nt8][2 * hh + 1]);
            }
    }
    // dg[r] = sum over r' >= r of dGamma[r'], the last row taking sum_r (dKb o Kb)_r
    // (Gamma_C enters Kb of every row) and deC o e^{Gamma_C}
    if (tid < D) {
        const int i = tid;
        float acc = deC[i] * eC[i];
#pragma unroll
        for (int r = 0; r < C; ++r) acc += kbk[r * FS + i];
        float out[C];
#pragma unroll
        for (int r = C - 1; r >= 0; --r) {
            acc += dgam[r * FS + i];
            out[r] = acc;
        }
#pragma unroll
        for (int r = 0; r < C; ++r)
            if (r < nt) a.dg[((size_t)(t0 + r) * a.H + h) * D + i] = out[r];
    }
    __syncthreads();  // this input buffer is free: the block after next goes into it
    if (nx2.ok) issue_inputs(nx2, ibo);
    cp_async_commit();
    if (!nxt.ok) break;
    cur = nxt;
    nxt = nx2;
    }
}

}  // namespace

cudaError_t launch_bwd_chunk(const PrefillArgs &p, const void *dout,
                             const __nv_bfloat16 *fwd_states, const __nv_bfloat16 *adj_states,
                             float *dq, float *dk, float *dv, float *dg, float *dbeta,
                             cudaStream_t st) {
    if (p.N == 0 || p.T_tot == 0) return cudaSuccess;
    GradArgs a;
    a.q = (const __nv_bfloat16 *)p.q; a.k = (const __nv_bfloat16 *)p.k;
    a.v = (const __nv_bfloat16 *)p.v; a.dout = (const __nv_bfloat16 *)dout;
    a.g = p.g; a.beta = p.beta; a.S0 = p.S0; a.cu = p.cu;
    a.Sck = fwd_states; a.dSck = adj_states;
    a.dq = dq; a.dk = dk; a.dv = dv; a.dg = dg; a.dbeta = dbeta;
    a.N = p.N; a.T_tot = p.T_tot; a.H = p.H;
    cudaError_t e = set_max_dynamic_smem((const void *)bwd_chunk_kernel, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    // one CTA per SM walks the (block, head) list; at most T_tot / 16 + N blocks over
    // all sequences
    const long long bound = ((long long)(p.T_tot + C - 1) / C + p.N) * p.H;
    int sms = 148, dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const unsigned grid = (unsigned)(bound < sms ? bound : sms);
    bwd_chunk_kernel<<<grid, GT, SMEM_BYTES, st>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
