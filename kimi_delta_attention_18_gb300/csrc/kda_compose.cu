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

}  // namespace

cudaError_t launch_compose(int units, int Sg, int dk, int dv, const float *A, const float *B,
                           const float *S0, float *seg_init, float *S_final, cudaStream_t st) {
    if (units == 0 || Sg == 0) return cudaSuccess;
    const size_t smem = ((size_t)dk * (dk + 1) + 2 * (size_t)dk * CB) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(compose_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(units, (dv + CB - 1) / CB);
    compose_kernel<<<grid, NT, smem, st>>>(Sg, dk, dv, A, B, S0, seg_init, S_final);
    return cudaGetLastError();
}

}  // namespace kda
