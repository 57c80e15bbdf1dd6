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
// B_part in the caller's checkpoint slot and A_part in the workspace; a kernel
// then adds the product: for dk = dv = 128 on tensor cores, each fp32 operand as
// a hi/lo pair of BF16 values and A X ~ Ah Xh + Ah Xl + Al Xh (the dropped Al Xl
// term and the splits' rounding are ~2^-16 of |A||X|, the same split the segment
// scan uses), otherwise in fp32 on CUDA cores.
#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

constexpr int FX_ROWS = 32;   // rows i of one checkpoint per CTA
constexpr int FX_T = 256;     // 8 warps: warp w takes rows 4w..4w+3, lane l columns 4l..4l+3
constexpr int FX_ALD = FX_ROWS + 4;  // transposed A rows: 16-byte aligned, 4-way store conflicts

// The checkpoint kg of head h: its slot of A_part and of the caller's array, and
// the start state of its segment; false if it does not exist or its segment
// starts from zeros (or is the lead segment, run from S0: its checkpoints are
// already the states).
__device__ __forceinline__ bool ckpt_operands(const PrefillArgs &p, const float *S0,
                                              const float *starts, int kg, int h,
                                              const float *&A, float *&out, const float *&start) {
    const int iv = p.ckpt_interval, dk = p.dk, dv = p.dv, H = p.H;
    int n = -1, base = 0;
    for (int m = 0; m < p.N; ++m) {  // the sequence that owns global checkpoint kg
        const int cnt = (p.cu[m + 1] - p.cu[m]) / iv;
        if (kg < base + cnt) {
            n = m;
            break;
        }
        base += cnt;
    }
    if (n < 0) return false;  // fewer checkpoints than the bound
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
    if (p.lead > 0 && s == 0) return false;
    const size_t unit = (size_t)n * H + h;
    start = s == 0 ? (S0 ? S0 + unit * dk * dv : nullptr) : starts + (unit * p.Sg + s) * (size_t)dk * dv;
    if (!start) return false;  // zero start: the zero-start state is the state
    A = p.ckpt_a + ((size_t)kg * H + h) * dk * dk;
    out = p.ckpt + ((size_t)kg * H + h) * dk * dv;
    return true;
}

// grid (max_ckpt, H, ceil(dk / FX_ROWS)); CTA (k, h, r) updates rows
// [32 r, 32 r + 32) of checkpoint k of head h, if that checkpoint exists and its
// segment has a nonzero start state.  dv = 4 x 32 lanes = 128 at most: each
// thread keeps a 4 x 4 block of the product in registers; per key channel q one
// float4 of A^T (the warp's four rows, a broadcast) and one float4 of the start
// state row feed 16 fused multiply-adds.
__global__ void __launch_bounds__(FX_T) ckpt_fixup_kernel(const PrefillArgs p, const float *S0,
                                                          const float *starts) {
    extern __shared__ float sm[];
    const int dk = p.dk, dv = p.dv;
    const int kg = blockIdx.x, h = blockIdx.y, i0 = blockIdx.z * FX_ROWS;
    const int rows = min(FX_ROWS, dk - i0);
    if (rows <= 0) return;
    const float *A, *start;
    float *out;
    if (!ckpt_operands(p, S0, starts, kg, h, A, out, start)) return;

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

// dk = dv = 128: one CTA of 8 warps per checkpoint.  The fp32 A_part and start
// state go to shared memory as hi/lo BF16 tiles (272-byte rows: the ldmatrix rows
// of every 8 x 8 matrix fall on distinct banks); warp w takes rows [16 w, 16 w +
// 16) of the product over all 128 columns, 3 x 8 x 16 mma.sync, and adds it to
// the zero-start state in the caller's slot.
constexpr int FM_ROW = 272;                 // bytes per BF16 tile row (128 + 8 pad)
constexpr int FM_TILE = 128 * FM_ROW;
constexpr int FM_SMEM = 4 * FM_TILE;        // A hi, A lo, X hi, X lo
__global__ void __launch_bounds__(256, 1) ckpt_fixup_mma_kernel(const __grid_constant__ PrefillArgs p,
                                                                const float *S0,
                                                                const float *starts) {
    extern __shared__ __align__(16) uint8_t smf[];
    const float *A, *X;
    float *out;
    if (!ckpt_operands(p, S0, starts, blockIdx.x, blockIdx.y, A, out, X)) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g8 = lane >> 2, t4 = lane & 3;
    const uint32_t sb = sm100::smem_addr(smf);
    const bool x16 = ((uintptr_t)X & 15u) == 0;  // S0 is the caller's, 4-byte aligned
    // fp32 [128][128] -> hi/lo BF16 tiles, four elements per thread and step
    auto split = [&](const float *src, bool v16, int hi_off) {
#pragma unroll 4
        for (int e = tid; e < 128 * 32; e += 256) {
            const int r = e >> 5, c4 = 4 * (e & 31);
            float4 v;
            if (v16) {
                v = *(const float4 *)(src + (size_t)r * 128 + c4);
            } else {
                const float *q = src + (size_t)r * 128 + c4;
                v = make_float4(q[0], q[1], q[2], q[3]);
            }
            const float f[4] = {v.x, v.y, v.z, v.w};
            uint32_t hw[2], lw[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(f[2 * u], f[2 * u + 1]);
                const float2 hf = __bfloat1622float2(h2);
                hw[u] = *(const uint32_t *)&h2;
                lw[u] = sm100::pack_bf16x2(f[2 * u] - hf.x, f[2 * u + 1] - hf.y);
            }
            *(uint2 *)(smf + hi_off + r * FM_ROW + 2 * c4) = make_uint2(hw[0], hw[1]);
            *(uint2 *)(smf + hi_off + FM_TILE + r * FM_ROW + 2 * c4) = make_uint2(lw[0], lw[1]);
        }
    };
    split(A, true, 0);            // A_part lives in the workspace: 16-byte aligned
    split(X, x16, 2 * FM_TILE);
    __syncthreads();
    float acc[16][4] = {};
    const int i0 = 16 * warp;
#pragma unroll 1
    for (int kk = 0; kk < 8; ++kk) {
        uint32_t ah[4], al[4];
        const uint32_t aoff = (i0 + (lane & 7) + 8 * ((lane >> 3) & 1)) * FM_ROW +
                              (16 * kk + 8 * (lane >> 4)) * 2;
        sm100::ldsm_x4(sb + aoff, ah);
        sm100::ldsm_x4(sb + FM_TILE + aoff, al);
#pragma unroll
        for (int np = 0; np < 8; ++np) {
            uint32_t bh[4], bl[4];
            const uint32_t boff = (16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1)) * FM_ROW +
                                  (16 * np + 8 * (lane >> 4)) * 2;
            sm100::ldsm_x4_t(sb + 2 * FM_TILE + boff, bh);
            sm100::ldsm_x4_t(sb + 3 * FM_TILE + boff, bl);
            sm100::mma_bf16_16816(acc[2 * np], ah, bh[0], bh[1]);
            sm100::mma_bf16_16816(acc[2 * np + 1], ah, bh[2], bh[3]);
            sm100::mma_bf16_16816(acc[2 * np], ah, bl[0], bl[1]);
            sm100::mma_bf16_16816(acc[2 * np + 1], ah, bl[2], bl[3]);
            sm100::mma_bf16_16816(acc[2 * np], al, bh[0], bh[1]);
            sm100::mma_bf16_16816(acc[2 * np + 1], al, bh[2], bh[3]);
        }
    }
    const bool o8 = ((uintptr_t)out & 7u) == 0;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float *d = out + (size_t)(i0 + g8 + 8 * hh) * 128 + 8 * nt + 2 * t4;
            if (o8) {
                float2 v = *(float2 *)d;
                v.x += acc[nt][2 * hh];
                v.y += acc[nt][2 * hh + 1];
                *(float2 *)d = v;
            } else {
                d[0] += acc[nt][2 * hh];
                d[1] += acc[nt][2 * hh + 1];
            }
        }
}

}  // namespace

cudaError_t launch_ckpt_fixup(const PrefillArgs &a, const float *S0, const float *starts,
                              int max_ckpt, cudaStream_t st) {
    if (a.ckpt_interval <= 0 || !a.ckpt || !a.ckpt_a || max_ckpt <= 0 || a.H == 0) return cudaSuccess;
    if (a.act == KDA_DTYPE_BF16 && a.dk == 128 && a.dv == 128) {
        cudaError_t e = set_max_dynamic_smem((const void *)ckpt_fixup_mma_kernel, FM_SMEM);
        if (e != cudaSuccess) return e;
        ckpt_fixup_mma_kernel<<<dim3((unsigned)max_ckpt, (unsigned)a.H), 256, FM_SMEM, st>>>(
            a, S0, starts);
        return cudaGetLastError();
    }
    const size_t smem = (size_t)(a.dk * FX_ALD + a.dk * a.dv) * sizeof(float);
    cudaError_t e = set_max_dynamic_smem((const void *)ckpt_fixup_kernel, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)max_ckpt, (unsigned)a.H, (unsigned)((a.dk + FX_ROWS - 1) / FX_ROWS));
    ckpt_fixup_kernel<<<grid, FX_T, smem, st>>>(a, S0, starts);
    return cudaGetLastError();
}

}  // namespace kda
