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

namespace kda {
namespace {

constexpr int NT = 256;
constexpr int CB = 16;  // state columns per CTA

__global__ void __launch_bounds__(NT) compose_kernel(int Sg, int dk, int dv, const float *A,
                                                     const float *B, const float *S0,
                                                     float *seg_init, float *S_final) {
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

// dk = 128, dv a multiple of 8, 16-byte aligned arrays: register-tiled form.
// One CTA per (unit, 8-column block), two threads per state row, each owning a
// row x 4-column tile of the running state; A_{s+1} is fetched into registers
// (16 float4 per thread, coalesced) while step s computes, then staged in shared
// memory with a padded row (conflict-free column walks).
constexpr int FD = 128, FT = 256, FCB = 8, LAP = FD + 1;

__global__ void __launch_bounds__(FT) compose_fast_kernel(int Sg, int dv, const float *A,
                                                          const float *B, const float *S0,
                                                          float *seg_init, float *S_final) {
    extern __shared__ float smem[];
    float *As = smem;              // [128][129]
    float *X = As + FD * LAP;      // [128][8]
    const int t = threadIdx.x, i = t >> 1, cg = t & 1;
    const size_t u = blockIdx.x;
    const int col = blockIdx.y * FCB + 4 * cg;
    const size_t row_off = (size_t)i * dv + col;
    const int nsteps = S_final ? Sg : Sg - 1;  // without S_final the last pair is never read

    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (S0) x = *(const float4 *)(S0 + u * (size_t)FD * dv + row_off);
    *(float4 *)(X + i * FCB + 4 * cg) = x;

    float4 ar[16];
    float4 bnext = make_float4(0.f, 0.f, 0.f, 0.f);
    auto fetch = [&](int s) {  // A_s (whole, coalesced) and this thread's tile of B_s
        const float4 *src = (const float4 *)(A + (u * Sg + s) * (size_t)FD * FD);
#pragma unroll
        for (int m = 0; m < 16; ++m) ar[m] = src[t + FT * m];
        bnext = *(const float4 *)(B + (u * Sg + s) * (size_t)FD * dv + row_off);
    };
    auto stage = [&]() {
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const int e = t + FT * m, r = e >> 5, c = (e & 31) * 4;
            float *d = As + r * LAP + c;
            d[0] = ar[m].x; d[1] = ar[m].y; d[2] = ar[m].z; d[3] = ar[m].w;
        }
    };
    float4 bcur = make_float4(0.f, 0.f, 0.f, 0.f);
    if (nsteps > 0) {
        fetch(0);
        stage();
        bcur = bnext;
    }
    __syncthreads();
    for (int s = 0; s < Sg; ++s) {
        if (seg_init) *(float4 *)(seg_init + (u * Sg + s) * (size_t)FD * dv + row_off) = x;
        if (s >= nsteps) break;
        if (s + 1 < nsteps) fetch(s + 1);  // in flight during the product below
        // two independent accumulation chains (even / odd k) halve the FMA latency chain
        float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
        const float *arow = As + i * LAP;
#pragma unroll 8
        for (int k = 0; k < FD; k += 2) {
            const float ae = arow[k], ao = arow[k + 1];
            const float4 xe = *(const float4 *)(X + k * FCB + 4 * cg);
            const float4 xo = *(const float4 *)(X + (k + 1) * FCB + 4 * cg);
            a0.x = fmaf(ae, xe.x, a0.x); a0.y = fmaf(ae, xe.y, a0.y);
            a0.z = fmaf(ae, xe.z, a0.z); a0.w = fmaf(ae, xe.w, a0.w);
            a1.x = fmaf(ao, xo.x, a1.x); a1.y = fmaf(ao, xo.y, a1.y);
            a1.z = fmaf(ao, xo.z, a1.z); a1.w = fmaf(ao, xo.w, a1.w);
        }
        float4 acc;
        acc.x = a0.x + a1.x + bcur.x; acc.y = a0.y + a1.y + bcur.y;
        acc.z = a0.z + a1.z + bcur.z; acc.w = a0.w + a1.w + bcur.w;
        __syncthreads();  // every read of X and of A_s is done
        x = acc;
        *(float4 *)(X + i * FCB + 4 * cg) = x;
        if (s + 1 < nsteps) {
            stage();
            bcur = bnext;
        }
        __syncthreads();
    }
    if (S_final) *(float4 *)(S_final + u * (size_t)FD * dv + row_off) = x;
}

}  // namespace

cudaError_t launch_compose(int units, int Sg, int dk, int dv, const float *A, const float *B,
                           const float *S0, float *seg_init, float *S_final, cudaStream_t st) {
    if (units == 0 || Sg == 0) return cudaSuccess;
    auto al16 = [](const void *p) { return ((uintptr_t)p & 15u) == 0; };
    if (dk == FD && dv % FCB == 0 && al16(A) && al16(B) && al16(S0) && al16(seg_init) &&
        al16(S_final)) {
        const size_t fsmem = ((size_t)FD * LAP + (size_t)FD * FCB) * sizeof(float);
        cudaError_t e = cudaFuncSetAttribute(compose_fast_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)fsmem);
        if (e != cudaSuccess) return e;
        compose_fast_kernel<<<dim3(units, dv / FCB), FT, fsmem, st>>>(Sg, dv, A, B, S0, seg_init,
                                                                       S_final);
        return cudaGetLastError();
    }
    const size_t smem = ((size_t)dk * (dk + 1) + 2 * (size_t)dk * CB) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(compose_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(units, (dv + CB - 1) / CB);
    compose_kernel<<<grid, NT, smem, st>>>(Sg, dk, dv, A, B, S0, seg_init, S_final);
    return cudaGetLastError();
}

}  // namespace kda
