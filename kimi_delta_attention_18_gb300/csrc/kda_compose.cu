// Prefix scan joining context-parallel segments (Kimi K3 technical-report
// digest, section 2.4 (1), KCP: the recurrent state split into a transfer
// matrix and a zero-initial state, recombined by a prefix scan):
//     start_0 = S0,  start_s = A_{s-1} start_{s-1} + B_{s-1},
//     S_final = A_{S-1} start_{S-1} + B_{S-1}.
// Columns of the state never mix, so each CTA owns one (unit, column block)
// chain and runs it sequentially over the segments in fp32; different units
// and column blocks run on different SMs with no cross-CTA waiting.  Each step
// stages A_s (dk x dk) in shared memory with coalesced float4 loads.
#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int NT = 256;
constexpr int CB = 16;  // state columns per CTA

__global__ void __launch_bounds__(NT) compose_kernel(int Sg, int dk, int dv, const float *A,
                                                     const float *B, const float *S0,
                                                     float *seg_init, float *S_final,
                                                     __nv_bfloat16 *img) {
    extern __shared__ float smem[];
    const int LA = dk + 1;
    float *As = smem;              // [dk][dk+1]
    float *X = As + dk * LA;       // [dk][CB]
    float *Xn = X + dk * CB;       // [dk][CB]
    const int tid = threadIdx.x;
    const size_t u = blockIdx.x;
    const int c0 = blockIdx.y * CB;
    const int nc = min(CB, dv - c0);

    for (int e = tid; e < dk * CB; e += NT) {
        const int i = e / CB, c = e % CB;
        X[e] = (S0 && c < nc) ? S0[u * (size_t)dk * dv + (size_t)i * dv + c0 + c] : 0.f;
    }
    for (int s = 0; s < Sg; ++s) {
        const float *As_g = A + (u * Sg + s) * (size_t)dk * dk;
        const float *Bs_g = B + (u * Sg + s) * (size_t)dk * dv;
        __syncthreads();
        if (seg_init) {
            float *dst = seg_init + (u * Sg + s) * (size_t)dk * dv;
            for (int e = tid; e < dk * CB; e += NT) {
                const int i = e / CB, c = e % CB;
                if (c < nc) dst[(size_t)i * dv + c0 + c] = X[e];
            }
        }
        if (img) {  // dk = dv = 128 only
            __nv_bfloat16 *im = img + (u * Sg + s) * (size_t)kStartImgElems;
            for (int e = tid; e < dk * CB; e += NT) {
                const int i = e / CB, c = e % CB;
                if (c < nc) im[start_img_index(c0 + c, i)] = __float2bfloat16_rn(X[e]);
            }
        }
        if (s == Sg - 1 && !S_final) break;  // only the start states are wanted
        if ((dk & 3) == 0) {
            for (int e = tid; e < dk * dk / 4; e += NT) {
                const int i = (4 * e) / dk, m = (4 * e) % dk;
                const float4 a4 = *((const float4 *)As_g + e);
                As[i * LA + m] = a4.x; As[i * LA + m + 1] = a4.y;
                As[i * LA + m + 2] = a4.z; As[i * LA + m + 3] = a4.w;
            }
        } else {
            for (int e = tid; e < dk * dk; e += NT) As[(e / dk) * LA + e % dk] = As_g[e];
        }
        __syncthreads();
        for (int e = tid; e < dk * CB; e += NT) {
            const int i = e / CB, c = e % CB;
            float acc = c < nc ? Bs_g[(size_t)i * dv + c0 + c] : 0.f;
            for (int m = 0; m < dk; ++m) acc += As[i * LA + m] * X[m * CB + c];
            Xn[e] = acc;
        }
        __syncthreads();
        for (int e = tid; e < dk * CB; e += NT) X[e] = Xn[e];
    }
    __syncthreads();
    if (S_final)
        for (int e = tid; e < dk * CB; e += NT) {
            const int i = e / CB, c = e % CB;
            if (c < nc) S_final[u * (size_t)dk * dv + (size_t)i * dv + c0 + c] = X[e];
        }
}

// dk = 128, dv a multiple of 8, 16-byte aligned arrays.  One CTA per (unit,
// 8-column block), 256 threads.  A_s arrives by TMA two steps ahead into a
// double-buffered stage (four 128-row x 32-column fp32 boxes with 128-byte
// swizzle: the 16-byte chunk c of row i sits at chunk c ^ (i mod 8)); B_{s+1} is
// prefetched into registers.  The product A_s X is register-blocked: a thread
// takes rows r, r+32, r+64, r+96 (one swizzle phase, so the 16 rows a warp reads
// at once hit different banks) and 4 columns over one quarter of the 128 key
// channels; the four quarters' partial sums meet in shared memory, where each
// thread then adds up one row x 4 columns of the next state.  The running state
// is double-buffered, so each step needs two barriers.
constexpr int FD = 128, FT = 256, FCB = 8;
constexpr int ABOX = FD * 32 * 4;    // one 128 x 32 fp32 box, 16 KB
constexpr int ASTAGE = 4 * ABOX;     // A_s, 64 KB
constexpr int FX = 2 * FD * FCB;     // running state, two buffers [2][128][8]
constexpr int FP = 4 * FD * FCB;     // partial sums [4 quarters][128][8]
constexpr int FAST_SMEM = 2 * ASTAGE + (FX + FP) * 4 + 64 + 1024;
constexpr long long kWaitLimit = 4000000000ll;

__global__ void __launch_bounds__(FT) compose_tma_kernel(const __grid_constant__ CUtensorMap tmA,
                                                         int Sg, int dv, const float *B,
                                                         const float *S0, float *seg_init,
                                                         float *S_final, __nv_bfloat16 *img,
                                                         int32_t *dev_status) {
    extern __shared__ uint8_t smem_raw[];
    // Align by pointer arithmetic on the __shared__ array (not through an integer),
    // so accesses keep the shared address space instead of becoming generic.
    uint8_t *sm = smem_raw + ((1024u - (sm100::smem_addr(smem_raw) & 1023u)) & 1023u);
    float *X = (float *)(sm + 2 * ASTAGE);
    float *P = X + FX;
    uint64_t *bars = (uint64_t *)(P + FP);
    volatile int *abort = (volatile int *)(bars + 2);
    const uint32_t sb = smem_addr(sm), bar0 = smem_addr(&bars[0]), bar1 = smem_addr(&bars[1]);
    const uint64_t tmap = reinterpret_cast<uint64_t>(&tmA);
    const int t = threadIdx.x;
    const int kq = t >> 6, r = (t >> 1) & 31, cg = t & 1;  // product: quarter, rows r + 32 m
    const int oi = t >> 1, ocg = t & 1;                     // output: row oi, columns 4 ocg..
    const size_t u = blockIdx.x;
    const size_t row_off = (size_t)oi * dv + blockIdx.y * FCB + 4 * ocg;
    const int nsteps = S_final ? Sg : Sg - 1;  // without S_final the last pair is never read

    auto issue = [&](int s) {  // one thread: A_s into stage s % 2
        const uint32_t bar = (s & 1) ? bar1 : bar0;
        mbar_arrive_expect_tx(bar, ASTAGE);
        const int y = (int)((u * Sg + s) * FD);
#pragma unroll
        for (int b4 = 0; b4 < 4; ++b4)
            tma_load_2d(sb + (s & 1) * ASTAGE + b4 * ABOX, tmap, 32 * b4, y, bar);
    };
    int issued = 0;
    if (t == 0) {
        mbar_init(bar0, 1);
        mbar_init(bar1, 1);
        *abort = 0;
        mbar_fence_init();
    }
    __syncthreads();
    if (t == 0) {
        for (; issued < 2 && issued < nsteps; ++issued) issue(issued);
    }

    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (S0) x = *(const float4 *)(S0 + u * (size_t)FD * dv + row_off);
    *(float4 *)(X + oi * FCB + 4 * ocg) = x;
    float4 bcur = make_float4(0.f, 0.f, 0.f, 0.f);
    if (nsteps > 0) bcur = *(const float4 *)(B + (u * Sg) * (size_t)FD * dv + row_off);
    __syncthreads();

    const int xi = r & 7;  // swizzle phase shared by rows r + 32 m
    int s = 0;
    for (; s < Sg; ++s) {
        if (seg_init) *(float4 *)(seg_init + (u * Sg + s) * (size_t)FD * dv + row_off) = x;
        if (img) {  // dv = 128 only: columns jb..jb+3 of row oi
            __nv_bfloat16 *im = img + (u * Sg + s) * (size_t)kStartImgElems;
            const int jb = blockIdx.y * FCB + 4 * ocg;
            im[start_img_index(jb + 0, oi)] = __float2bfloat16_rn(x.x);
            im[start_img_index(jb + 1, oi)] = __float2bfloat16_rn(x.y);
            im[start_img_index(jb + 2, oi)] = __float2bfloat16_rn(x.z);
            im[start_img_index(jb + 3, oi)] = __float2bfloat16_rn(x.w);
        }
        if (s >= nsteps) break;
        float4 bnext = make_float4(0.f, 0.f, 0.f, 0.f);
        if (s + 1 < nsteps) bnext = *(const float4 *)(B + (u * Sg + s + 1) * (size_t)FD * dv + row_off);
        mbar_wait((s & 1) ? bar1 : bar0, (s >> 1) & 1, abort, kWaitLimit);
        const uint8_t *stage = sm + (s & 1) * ASTAGE;
        const float *Xc = X + (s & 1) * FD * FCB;
        float acc[4][4] = {};
#pragma unroll
        for (int k4h = 0; k4h < 8; ++k4h) {
            const int k4 = 8 * kq + k4h;
            const uint8_t *box = stage + (k4 >> 3) * ABOX + (((k4 & 7) ^ xi) << 4);
            float4 xr[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) xr[e] = *(const float4 *)(Xc + (4 * k4 + e) * FCB + 4 * cg);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float4 a = *(const float4 *)(box + (r + 32 * m) * 128);
                const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc[m][0] = fmaf(av[e], xr[e].x, acc[m][0]);
                    acc[m][1] = fmaf(av[e], xr[e].y, acc[m][1]);
                    acc[m][2] = fmaf(av[e], xr[e].z, acc[m][2]);
                    acc[m][3] = fmaf(av[e], xr[e].w, acc[m][3]);
                }
            }
        }
#pragma unroll
        for (int m = 0; m < 4; ++m)
            *(float4 *)(P + (kq * FD + r + 32 * m) * FCB + 4 * cg) =
                make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
        __syncthreads();  // partials written; every read of X and of stage s % 2 is done
        if (*abort) break;
        if (t == 0 && s + 2 < nsteps) {
            issue(s + 2);
            ++issued;
        }
        float4 sum = bcur;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 pp = *(const float4 *)(P + (q * FD + oi) * FCB + 4 * ocg);
            sum.x += pp.x; sum.y += pp.y; sum.z += pp.z; sum.w += pp.w;
        }
        x = sum;
        *(float4 *)(X + ((s + 1) & 1) * FD * FCB + oi * FCB + 4 * ocg) = x;
        bcur = bnext;
        __syncthreads();  // next state complete, partials free
    }
    if (*abort) {
        if (t == 0) {
            dev_fail(dev_status, KDA_ERR_TIMEOUT);
            volatile int never = 0;  // let copies already in flight land before exiting
            for (int c = s; c < issued; ++c)
                mbar_wait((c & 1) ? bar1 : bar0, (c >> 1) & 1, &never, kWaitLimit);
        }
        return;
    }
    if (S_final) *(float4 *)(S_final + u * (size_t)FD * dv + row_off) = x;
}

// BF16 workloads at dk = dv = 128, from the transfer pass's hi/lo BF16 images of
// A_s (A^T stored row-major, i.e. [j][i]).  One CTA per (unit, 8-column block):
// 8 compute warps and one producer warp.  Compute warp w owns rows [16w, 16w+16)
// of the next state over all 128 key channels, so no partial sums cross warps
// and a step needs one barrier among the compute warps.  The product runs on
// mma.sync with a three-term BF16 split,
//     A X ~ A_hi X_hi + A_hi X_lo + A_lo X_hi     (fp32 accumulation),
// whose dropped term and own rounding are ~2^-16 of |A| |X| per step.  The
// producer warp streams, two steps ahead, A_s hi and lo (64-channel x 128-row
// boxes, 128-byte swizzle: chunk q of row j sits at q ^ (j mod 8), so transposed
// ldmatrix rows hit different banks) and this CTA's 8 columns of B_s (one
// 8 x 128 fp32 box) into a stage; compute warps free a stage through an
// mbarrier, so neither the copy issue nor a global load sits on the step's
// critical path.  Each warp keeps its rows of the running state in fp32
// registers and publishes them, already split, as BF16 hi/lo images of X^T
// ([column j][key channel i], 272-byte rows so ldmatrix rows hit different
// banks), double-buffered: a k-step then needs one ldmatrix for both X splits.
constexpr int MB_T = 288;               // 8 compute warps + 1 producer warp
constexpr int MB_ABOX = 128 * 128;      // one 64-channel x 128-row BF16 box, 16 KB
constexpr int MB_BBOX = FD * FCB * 4;   // 8 columns x 128 rows of B_s, fp32, 4 KB
constexpr int MB_STAGE = 4 * MB_ABOX + MB_BBOX;  // hi (2 boxes), lo (2 boxes), B
constexpr int MB_XROW = 272;            // bytes per row of an X^T image (128 BF16 + pad)
constexpr int MB_X = 2 * MB_STAGE;
constexpr int MB_XSZ = 2 * FCB * MB_XROW;  // hi and lo images of one state
constexpr int MB_BAR = MB_X + 2 * MB_XSZ;
constexpr int MB_SMEM = MB_BAR + 64 + 1024;
static_assert(MB_STAGE % 1024 == 0, "stages keep the 128-byte swizzle's 1024-byte alignment");

__global__ void __launch_bounds__(MB_T) compose_mma_kernel(const __grid_constant__ CUtensorMap tmA,
                                                           const __grid_constant__ CUtensorMap tmB,
                                                           int Sg, const float *S0,
                                                           float *seg_init, float *S_final,
                                                           __nv_bfloat16 *img, int32_t *dev_status) {
    extern __shared__ uint8_t smem_raw[];
    griddep_wait();  // A_s, B_s come from the transfer pass just before
    griddep_launch_dependents();
    uint8_t *sm = smem_raw + ((1024u - (sm100::smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t *Xb = sm + MB_X;
    uint64_t *bars = (uint64_t *)(sm + MB_BAR);  // full[2], empty[2]
    volatile int *abort = (volatile int *)(bars + 4);
    const uint32_t sb = smem_addr(sm);
    auto full = [&](int s) { return smem_addr(&bars[s & 1]); };
    auto empty = [&](int s) { return smem_addr(&bars[2 + (s & 1)]); };
    const int t = threadIdx.x, w = t >> 5, lane = t & 31, g8 = lane >> 2, t4 = lane & 3;
    const size_t u = blockIdx.x;
    const int c0 = blockIdx.y * FCB;
    const int nsteps = S_final ? Sg : Sg - 1;  // without S_final the last pair is never read
    constexpr int dv = 128;
    constexpr int NCW = 8;  // compute warps

    if (t == 0) {
        mbar_init(full(0), 1);
        mbar_init(full(1), 1);
        mbar_init(empty(0), NCW);
        mbar_init(empty(1), NCW);
        *abort = 0;
        mbar_fence_init();
    }
    __syncthreads();

    if (w == NCW) {  // ---- producer: A_s hi / lo and B_s columns into stage s % 2
        if (lane != 0) return;
        const uint64_t ta = reinterpret_cast<uint64_t>(&tmA);
        const uint64_t tb = reinterpret_cast<uint64_t>(&tmB);
        int issued = 0;
        for (; issued < nsteps; ++issued) {
            const int s = issued;
            if (s >= 2 && !mbar_wait(empty(s), ((s >> 1) - 1) & 1, abort, kWaitLimit)) break;
            const uint32_t bar = full(s), dst = sb + (s & 1) * MB_STAGE;
            mbar_arrive_expect_tx(bar, MB_STAGE);
            const int y = (int)((u * Sg + s) * 2 * FD);
            tma_load_2d(dst, ta, 0, y, bar);
            tma_load_2d(dst + MB_ABOX, ta, 64, y, bar);
            tma_load_2d(dst + 2 * MB_ABOX, ta, 0, y + FD, bar);
            tma_load_2d(dst + 3 * MB_ABOX, ta, 64, y + FD, bar);
            tma_load_2d(dst + 4 * MB_ABOX, tb, c0, (int)((u * Sg + s) * FD), bar);
        }
        if (*abort) {
            dev_fail(dev_status, KDA_ERR_TIMEOUT);
            volatile int never = 0;  // let copies still in flight land before exiting
            for (int c = issued > 2 ? issued - 2 : 0; c < issued; ++c)
                mbar_wait(full(c), (c >> 1) & 1, &never, kWaitLimit);
        }
        return;
    }

    // ---- compute warps.  Running state: transposed copy for the products, this
    // thread's outputs (rows i0, i1; columns c0+cc, +1) in fp32.
    const int i0 = 16 * w + g8, i1 = i0 + 8, cc = 2 * t4;
    const float *s0 = S0 ? S0 + u * (size_t)FD * dv : nullptr;
    // X^T image element (column c, channel i) of buffer b, split img (0 hi, 1 lo)
    auto xb_at = [&](int b, int img, int c, int i) {
        return (__nv_bfloat16 *)(Xb + b * MB_XSZ + img * FCB * MB_XROW + c * MB_XROW) + i;
    };
    auto put_x = [&](int b, int c, int i, float v) {
        const __nv_bfloat16 h = __float2bfloat16_rn(v);
        *xb_at(b, 0, c, i) = h;
        *xb_at(b, 1, c, i) = __float2bfloat16_rn(v - __bfloat162float(h));
    };
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int idx = t + 256 * e, c = idx >> 7, i = idx & 127;
        put_x(0, c, i, s0 ? s0[(size_t)i * dv + c0 + c] : 0.f);
    }
    float2 xo0 = make_float2(0.f, 0.f), xo1 = xo0;
    if (s0) {  // S0 and S_final come from the caller, 4-byte aligned only: scalar accesses
        xo0 = make_float2(s0[(size_t)i0 * dv + c0 + cc], s0[(size_t)i0 * dv + c0 + cc + 1]);
        xo1 = make_float2(s0[(size_t)i1 * dv + c0 + cc], s0[(size_t)i1 * dv + c0 + cc + 1]);
    }
    named_bar_sync(1, NCW * 32);

    // A fragment rows: box (w >> 2) of hi / lo, channel chunks q0 = 2 (w & 3) (+1)
    const int abox = (w >> 2) * MB_ABOX, q0 = 2 * (w & 3);
    const int mi = lane >> 3, lr = lane & 7;
    bool aborted = false;
    // start state of segment s (this thread's four values)
    auto put_start = [&](int s) {
        const size_t us = u * Sg + s;
        if (seg_init) {
            float *d = seg_init + us * (size_t)FD * dv + c0 + cc;
            *(float2 *)(d + (size_t)i0 * dv) = xo0;
            *(float2 *)(d + (size_t)i1 * dv) = xo1;
        }
        if (img) {
            __nv_bfloat16 *im = img + us * (size_t)kStartImgElems;
            im[start_img_index(c0 + cc, i0)] = __float2bfloat16_rn(xo0.x);
            im[start_img_index(c0 + cc + 1, i0)] = __float2bfloat16_rn(xo0.y);
            im[start_img_index(c0 + cc, i1)] = __float2bfloat16_rn(xo1.x);
            im[start_img_index(c0 + cc + 1, i1)] = __float2bfloat16_rn(xo1.y);
        }
    };
    for (int s = 0; s < Sg; ++s) {
        put_start(s);
        if (s >= nsteps) break;
        // a failed wait still runs the step (on whatever the stage holds) up to the
        // barrier below, which makes the decision to stop the same for every warp
        const bool ok = mbar_wait(full(s), (s >> 1) & 1, abort, kWaitLimit);
        const uint32_t st_s = sb + (s & 1) * MB_STAGE;
        const float *Bs = (const float *)(sm + (s & 1) * MB_STAGE + 4 * MB_ABOX);
        // B fragments of X (hi: matrices 0, 1; lo: 2, 3) for k-step kk
        const uint32_t xb_s = sb + MB_X + (s & 1) * MB_XSZ + (mi >> 1) * FCB * MB_XROW +
                              lr * MB_XROW + 16 * (mi & 1);
        auto load_a = [&](int kk, uint32_t (&ahi)[4], uint32_t (&alo)[4]) {
            const int j = 16 * kk + lr + 8 * (mi >> 1), q = q0 + (mi & 1);
            const uint32_t off = abox + j * 128 + ((q ^ (j & 7)) << 4);
            ldsm_x4_t(st_s + off, ahi);
            ldsm_x4_t(st_s + 2 * MB_ABOX + off, alo);
        };
        float hh[4] = {}, hl[4] = {}, lh[4] = {};
        uint32_t ahi[2][4], alo[2][4], bx[2][4];
        load_a(0, ahi[0], alo[0]);
        ldsm_x4(xb_s, bx[0]);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            if (kk + 1 < 8) {
                load_a(kk + 1, ahi[(kk + 1) & 1], alo[(kk + 1) & 1]);
                ldsm_x4(xb_s + 32 * (kk + 1), bx[(kk + 1) & 1]);
            }
            const uint32_t(&b)[4] = bx[kk & 1];
            mma_bf16_16816(hh, ahi[kk & 1], b[0], b[1]);
            mma_bf16_16816(hl, ahi[kk & 1], b[2], b[3]);
            mma_bf16_16816(lh, alo[kk & 1], b[0], b[1]);
        }
        const float2 b0 = *(const float2 *)(Bs + i0 * FCB + cc);
        const float2 b1 = *(const float2 *)(Bs + i1 * FCB + cc);
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(s));  // this warp's reads of the stage are done
        xo0 = make_float2(hh[0] + hl[0] + lh[0] + b0.x, hh[1] + hl[1] + lh[1] + b0.y);
        xo1 = make_float2(hh[2] + hl[2] + lh[2] + b1.x, hh[3] + hl[3] + lh[3] + b1.y);
        const int nb = (s + 1) & 1;
        put_x(nb, cc, i0, xo0.x);
        put_x(nb, cc + 1, i0, xo0.y);
        put_x(nb, cc, i1, xo1.x);
        put_x(nb, cc + 1, i1, xo1.y);
        // next state complete; stop together if any wait (or the producer) gave up
        aborted = named_bar_or(1, NCW * 32, !ok || *abort);
        if (aborted) break;
    }
    if (aborted) {
        if (t == 0) dev_fail(dev_status, KDA_ERR_TIMEOUT);
        return;
    }
    if (S_final) {
        float *d = S_final + u * (size_t)FD * dv + c0 + cc;
        d[(size_t)i0 * dv] = xo0.x;
        d[(size_t)i0 * dv + 1] = xo0.y;
        d[(size_t)i1 * dv] = xo1.x;
        d[(size_t)i1 * dv + 1] = xo1.y;
    }
}

}  // namespace

cudaError_t launch_compose(int units, int Sg, int dk, int dv, const float *A,
                           const __nv_bfloat16 *a_img, const float *B, const float *S0,
                           float *seg_init, float *S_final, __nv_bfloat16 *start_img,
                           int32_t *dev_status, cudaStream_t st) {
    if (dk != 128 || dv != 128) start_img = nullptr;
    if (units == 0 || Sg == 0) return cudaSuccess;
    if (a_img) {
        // BF16 images of A_s: [units * Sg * 2 * 128 rows j, 128 channels i], boxes of
        // 64 channels x 128 rows with 128-byte swizzle
        auto al16 = [](const void *p) { return ((uintptr_t)p & 15u) == 0; };
        PFN_cuTensorMapEncodeTiled_v12000 enc = sm100::tensor_map_encoder();
        if (dk != 128 || dv != 128 || !enc || !al16(a_img) || !al16(B)) return cudaErrorInvalidValue;
        CUtensorMap tm, tmb;
        const cuuint64_t dims[2] = {(cuuint64_t)FD, (cuuint64_t)units * Sg * 2 * FD};
        const cuuint64_t strides[1] = {(cuuint64_t)FD * 2};
        const cuuint32_t box[2] = {64, (cuuint32_t)FD};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16 *>(a_img), dims,
                strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
            CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        // B viewed as [units * Sg * 128 rows, 128 fp32 columns], 8-column x 128-row boxes
        const cuuint64_t bdims[2] = {(cuuint64_t)dv, (cuuint64_t)units * Sg * FD};
        const cuuint64_t bstrides[1] = {(cuuint64_t)dv * 4};
        const cuuint32_t bbox[2] = {(cuuint32_t)FCB, (cuuint32_t)FD};
        if (enc(&tmb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(B), bdims, bstrides,
                bbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
            CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        cudaError_t e = set_max_dynamic_smem((const void *)compose_mma_kernel, MB_SMEM);
        if (e != cudaSuccess) return e;
        return launch_dependent(compose_mma_kernel, dim3(units, dv / FCB), dim3(MB_T), MB_SMEM, st,
                                tm, tmb, Sg, S0, seg_init, S_final, start_img, dev_status);
    }
    auto al16 = [](const void *p) { return ((uintptr_t)p & 15u) == 0; };
    PFN_cuTensorMapEncodeTiled_v12000 enc = sm100::tensor_map_encoder();
    if (dk == FD && dv % FCB == 0 && al16(A) && al16(B) && al16(S0) && al16(seg_init) &&
        al16(S_final) && enc) {
        // A viewed as [units * Sg * 128 rows, 128 fp32 columns], 128 x 32 boxes
        CUtensorMap tm;
        const cuuint64_t dims[2] = {(cuuint64_t)FD, (cuuint64_t)units * Sg * FD};
        const cuuint64_t strides[1] = {(cuuint64_t)FD * 4};
        const cuuint32_t box[2] = {32, (cuuint32_t)FD};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(A), dims, strides, box,
                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
            CUDA_SUCCESS) {
            cudaError_t e = set_max_dynamic_smem((const void *)compose_tma_kernel, FAST_SMEM);
            if (e != cudaSuccess) return e;
            compose_tma_kernel<<<dim3(units, dv / FCB), FT, FAST_SMEM, st>>>(
                tm, Sg, dv, B, S0, seg_init, S_final, start_img, dev_status);
            return cudaGetLastError();
        }
    }
    const size_t smem = ((size_t)dk * (dk + 1) + 2 * (size_t)dk * CB) * sizeof(float);
    cudaError_t e = set_max_dynamic_smem((const void *)compose_kernel, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(units, (dv + CB - 1) / CB);
    compose_kernel<<<grid, NT, smem, st>>>(Sg, dk, dv, A, B, S0, seg_init, S_final, start_img);
    return cudaGetLastError();
}

}  // namespace kda
