// Single-token KDA decode step: one pass over each fp32 state in HBM.
//
// For one (sequence, head) with state S (dk x dv) and a new token (q, k, v, g,
// beta), the recurrence ("Kimi K3 Architecture Explained", section 3: decay,
// then erase, then write; the eraser recalls with the key and writes the
// difference) becomes, with D = Diag(exp(g)):
//     r = (D S)^T k,  u = beta (v - r),  S' = D S + k u^T,
//     o = S'^T q = (D S)^T q + u (k . q)
// so the state is read once (decayed in registers while the two column
// reductions r and (DS)^T q are formed), and written once.
//
// Layout: one CTA per (sequence, head), 512 threads = 16 warps.  Lane l owns
// columns 4l..4l+3 (one float4), warp w owns rows w, w+16, ...; every thread
// issues all of its float4 loads before using any, so each CTA keeps up to
// 64 KB in flight.  The cross-warp column sums go through shared memory.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int NW = 16;                 // warps per CTA
constexpr int RPT = 128 / NW;          // rows per thread at dk = 128

__device__ __forceinline__ float4 ld_stream(const float4 *p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(float4 *p, float4 x) { __stcs(p, x); }

template <typename TA>
__global__ void __launch_bounds__(NW * 32) decode_kernel(int H, int dk, int dv, const TA *q,
                                                         const TA *k, const TA *v,
                                                         const float *g, const float *beta,
                                                         float *S, TA *out) {
    __shared__ float s_a[128], s_k[128], s_q[128], s_u[128];
    __shared__ __align__(16) float red_r[NW][128];
    __shared__ __align__(16) float red_p[NW][128];
    __shared__ float s_qk;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t bh = blockIdx.x;
    float *Sbh = S + bh * (size_t)dk * dv;
    const bool colok = 4 * lane < dv;

    // Issue the state loads first: they are the bulk of the traffic.
    float4 st[RPT];
#pragma unroll
    for (int m = 0; m < RPT; ++m) {
        const int i = warp + NW * m;
        if (i < dk && colok) st[m] = ld_stream((const float4 *)(Sbh + (size_t)i * dv) + lane);
        else st[m] = make_float4(0.f, 0.f, 0.f, 0.f);
    }

    if (tid < dk) {
        s_a[tid] = expf(g[bh * dk + tid]);
        s_k[tid] = act_ld(k, bh * dk + tid);
        s_q[tid] = act_ld(q, bh * dk + tid);
    }
    if (warp == NW - 1) {
        float acc = 0.f;
        for (int i = lane; i < dk; i += 32) acc += act_ld(q, bh * dk + i) * act_ld(k, bh * dk + i);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) s_qk = acc;
    }
    __syncthreads();

    // Decay in registers, partial column sums of (DS)^T k and (DS)^T q.
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f), pq = r;
#pragma unroll
    for (int m = 0; m < RPT; ++m) {
        const int i = warp + NW * m;
        if (i < dk) {
            const float a = s_a[i], ki = s_k[i], qi = s_q[i];
            st[m].x *= a; st[m].y *= a; st[m].z *= a; st[m].w *= a;
            r.x += ki * st[m].x; r.y += ki * st[m].y; r.z += ki * st[m].z; r.w += ki * st[m].w;
            pq.x += qi * st[m].x; pq.y += qi * st[m].y; pq.z += qi * st[m].z; pq.w += qi * st[m].w;
        }
    }
    if (colok) {
        *(float4 *)&red_r[warp][4 * lane] = r;
        *(float4 *)&red_p[warp][4 * lane] = pq;
    }
    __syncthreads();

    if (tid < dv) {
        float R = 0.f, P = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) { R += red_r[w][tid]; P += red_p[w][tid]; }
        const float uj = beta[bh] * (act_ld(v, bh * dv + tid) - R);
        s_u[tid] = uj;
        act_st(out, bh * dv + tid, P + uj * s_qk);
    }
    __syncthreads();

    if (colok) {
        const float4 uu = *(const float4 *)&s_u[4 * lane];
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            const int i = warp + NW * m;
            if (i < dk) {
                const float ki = s_k[i];
                float4 x = st[m];
                x.x += ki * uu.x; x.y += ki * uu.y; x.z += ki * uu.z; x.w += ki * uu.w;
                st_stream((float4 *)(Sbh + (size_t)i * dv) + lane, x);
            }
        }
    }
}

}  // namespace

cudaError_t launch_decode(int batch, int H, int dk, int dv, int act, const void *q,
                          const void *k, const void *v, const float *g, const float *beta,
                          float *S, void *out, cudaStream_t st) {
    const size_t units = (size_t)batch * H;
    if (units == 0) return cudaSuccess;
    if (act == KDA_DTYPE_F32)
        decode_kernel<float><<<(unsigned)units, NW * 32, 0, st>>>(
            H, dk, dv, (const float *)q, (const float *)k, (const float *)v, g, beta, S,
            (float *)out);
    else
        decode_kernel<__nv_bfloat16><<<(unsigned)units, NW * 32, 0, st>>>(
            H, dk, dv, (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k,
            (const __nv_bfloat16 *)v, g, beta, S, (__nv_bfloat16 *)out);
    return cudaGetLastError();
}

}  // namespace kda
