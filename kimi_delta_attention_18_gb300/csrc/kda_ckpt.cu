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

constexpr int FX_ROWS = 32;   // rows i of one checkpoint per CTA
constexpr int FX_T = 256;     // 8 warps: warp w takes rows 4w..4w+3, lane l columns 4l..4l+3
constexpr int FX_ALD = FX_ROWS + 4;  // transposed A rows: 16-byte aligned, 4-way store conflicts

// grid (max_ckpt, H, ceil(dk / FX_ROWS)); CTA (k, h, r) updates rows
// [32 r, 32 r + 32) of checkpoint k of head h, if that checkpoint exists and its
// segment has a nonzero start state.  dv = 4 x 32 lanes = 128 at most: each
// thread keeps a 4 x 4 block of the product in registers; per key channel q one
// float4 of A^T (the warp's four rows, a broadcast) and one float4 of the start
// state row feed 16 fused multiply-adds.
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
    // its segment: the one whose blocks hold block done / 16 - 1 (the same split
    // as every kernel of the split path)
    const long long c = (len + 15) / 16, blk = done / 16 - 1;
    int s = 0;
    for (; s < p.Sg - 1; ++s) {
        long long c0, c1;
        segment_blocks(c, s, p.Sg, p.lead, c0, c1);
        if (blk < c1) break;
    }
    if (p.lead > 0 && s == 0) return;  // the lead segment ran from S0: already the state
    const size_t unit = (size_t)n * H + h;
    const float *start = s == 0 ? (S0 ? S0 + unit * dk * dv : nullptr)
                                : starts + (unit * p.Sg + s) * (size_t)dk * dv;
    if (!start) return;  // zero start: the zero-start state is the state
    const float *A = p.ckpt_a + ((size_t)kg * H + h) * dk * dk;
    float *out = p.ckpt + ((size_t)kg * H + h) * dk * dv;

    float *At = sm;                     // [dk][FX_ALD]: A^T of this CTA's rows (0 past `rows`)
    float *Xs = sm + dk * FX_ALD;       // [dk][dv]
    // fills with 16-byte loads where the rows allow (A_part lives in the
    // workspace; S0 is the caller's and only 4-byte aligned)
    if ((dk & 3) == 0) {
        for (int e = threadIdx.x; e < FX_ROWS * dk / 4; e += FX_T) {
            const int r = e / (dk / 4), q = 4 * (e % (dk / 4));
            const float4 v = r < rows ? *(const float4 *)(A + (size_t)(i0 + r) * dk + q)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
            At[q * FX_ALD + r] = v.x;
            At[(q + 1) * FX_ALD + r] = v.y;
            At[(q + 2) * FX_ALD + r] = v.z;
            At[(q + 3) * FX_ALD + r] = v.w;
        }
    } else {
        for (int e = threadIdx.x; e < FX_ROWS * dk; e += FX_T) {
            const int r = e / dk, q = e % dk;
            At[q * FX_ALD + r] = r < rows ? A[(size_t)(i0 + r) * dk + q] : 0.f;
        }
    }
    if (((uintptr_t)start & 15u) == 0 && ((dk * dv) & 3) == 0) {
        for (int e = threadIdx.x; e < dk * dv / 4; e += FX_T)
            ((float4 *)Xs)[e] = ((const float4 *)start)[e];
    } else {
        for (int e = threadIdx.x; e < dk * dv; e += FX_T) Xs[e] = start[e];
    }
    __syncthreads();
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    const int r0 = 4 * w, j0 = 4 * l;
    if (j0 >= dv) return;
    float acc[4][4] = {};
    auto fma_row = [&](int q, const float (&xr)[4]) {
        const float4 a = *(const float4 *)(At + q * FX_ALD + r0);
        const float ar[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int t = 0; t < 4; ++t) acc[r][t] += ar[r] * xr[t];
    };
    if ((dv & 3) == 0 && j0 + 4 <= dv) {  // 16-byte aligned rows of the start state
#pragma unroll 4
        for (int q = 0; q < dk; ++q) {
            const float4 x = *(const float4 *)(Xs + q * dv + j0);
            const float xr[4] = {x.x, x.y, x.z, x.w};
            fma_row(q, xr);
        }
    } else {
        for (int q = 0; q < dk; ++q) {
            float xr[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) xr[t] = j0 + t < dv ? Xs[q * dv + j0 + t] : 0.f;
            fma_row(q, xr);
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        if (r0 + r >= rows) break;
#pragma unroll
        for (int t = 0; t < 4; ++t)
            if (j0 + t < dv) out[(size_t)(i0 + r0 + r) * dv + j0 + t] += acc[r][t];
    }
}

}  // namespace

cudaError_t launch_ckpt_fixup(const PrefillArgs &a, const float *S0, const float *starts,
                              int max_ckpt, cudaStream_t st) {
    if (a.ckpt_interval <= 0 || !a.ckpt || !a.ckpt_a || max_ckpt <= 0 || a.H == 0) return cudaSuccess;
    const size_t smem = (size_t)(a.dk * FX_ALD + a.dk * a.dv) * sizeof(float);
    cudaError_t e = set_max_dynamic_smem((const void *)ckpt_fixup_kernel, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)max_ckpt, (unsigned)a.H, (unsigned)((a.dk + FX_ROWS - 1) / FX_ROWS));
    ckpt_fixup_kernel<<<grid, FX_T, smem, st>>>(a, S0, starts);
    return cudaGetLastError();
}

}  // namespace kda
