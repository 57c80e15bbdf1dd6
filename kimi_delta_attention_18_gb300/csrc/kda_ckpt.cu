// Sparse state checkpoints on the split prefill path.
//
// With S > 1 segments, the transfer pass runs every segment from the identity
// and from zeros, so at a checkpoint inside segment s it has the partial transfer
// matrix A_part and the zero-start state B_part (the state is linear in the
// segment's start state: "Kimi K3 Architecture Explained", section 3, the
// context-parallel split).  Once the scan has the segment's true start state,
// the checkpoint is
//     S = A_part start_s + B_part,
// the same composition the scan applies at segment ends.  The transfer pass left
// B_part in the caller's checkpoint slot and A_part in the workspace; this kernel
// adds the product in fp32 (sparse checkpoints: off the critical path).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int FX_ROWS = 16;   // rows i of one checkpoint per CTA
constexpr int FX_T = 256;

// grid (max_ckpt, H, ceil(dk / FX_ROWS)); CTA (k, h, r) updates rows
// [16 r, 16 r + 16) of checkpoint k of head h, if that checkpoint exists and its
// segment has a nonzero start state.
__global__ void __launch_bounds__(FX_T) ckpt_fixup_kernel(const PrefillArgs p, const float *S0,
                                                          const float *starts) {
    extern __shared__ float sm[];
    const int dk = p.dk, dv = p.dv, H = p.H, iv = p.ckpt_interval;
    const int kg = blockIdx.x, h = blockIdx.y, i0 = blockIdx.z * FX_ROWS;
    const int rows = min(FX_ROWS, dk - i0);
    if (rows <= 0) return;
    // the sequence that owns global checkpoint kg, and the checkpoint's position
    int n = -1, base = 0;
    for (int m = 0; m < p.N; ++m) {
        const int cnt = (p.cu[m + 1] - p.cu[m]) / iv;
        if (kg < base + cnt) {
            n = m;
            break;
        }
        base += cnt;
    }
    if (n < 0) return;  // fewer checkpoints than the bound
    const int len = p.cu[n + 1] - p.cu[n];
    const int done = (kg - base + 1) * iv;  // tokens of the sequence before the checkpoint
    // its segment: the one whose blocks [floor(s c / Sg), floor((s + 1) c / Sg)) hold
    // block done / 16 - 1 (the same split as every kernel of the split path)
    const long long c = (len + 15) / 16, blk = done / 16 - 1;
    int s = 0;
    while (s < p.Sg - 1 && blk >= (long long)(s + 1) * c / p.Sg) ++s;
    const size_t unit = (size_t)n * H + h;
    const float *start = s == 0 ? (S0 ? S0 + unit * dk * dv : nullptr)
                                : starts + (unit * p.Sg + s) * (size_t)dk * dv;
    if (!start) return;  // zero start: the zero-start state is the state
    const float *A = p.ckpt_a + ((size_t)kg * H + h) * dk * dk;
    float *out = p.ckpt + ((size_t)kg * H + h) * dk * dv;

    float *As = sm;                       // [FX_ROWS][dk]
    float *Xs = sm + FX_ROWS * dk;        // [dk][dv]
    for (int e = threadIdx.x; e < rows * dk; e += FX_T) As[e] = A[(size_t)(i0 + e / dk) * dk + e % dk];
    for (int e = threadIdx.x; e < dk * dv; e += FX_T) Xs[e] = start[e];
    __syncthreads();
    for (int e = threadIdx.x; e < rows * dv; e += FX_T) {
        const int r = e / dv, j = e % dv;
        float acc = 0.f;
        for (int q = 0; q < dk; ++q) acc += As[r * dk + q] * Xs[q * dv + j];
        out[(size_t)(i0 + r) * dv + j] += acc;
    }
}

}  // namespace

cudaError_t launch_ckpt_fixup(const PrefillArgs &a, const float *S0, const float *starts,
                              int max_ckpt, cudaStream_t st) {
    if (a.ckpt_interval <= 0 || !a.ckpt || !a.ckpt_a || max_ckpt <= 0 || a.H == 0) return cudaSuccess;
    const size_t smem = (size_t)(FX_ROWS * a.dk + a.dk * a.dv) * sizeof(float);
    cudaError_t e = set_max_dynamic_smem((const void *)ckpt_fixup_kernel, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)max_ckpt, (unsigned)a.H, (unsigned)((a.dk + FX_ROWS - 1) / FX_ROWS));
    ckpt_fixup_kernel<<<grid, FX_T, smem, st>>>(a, S0, starts);
    return cudaGetLastError();
}

}  // namespace kda
