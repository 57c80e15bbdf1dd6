// Single-token KDA decode step at dk = dv = 128, streamed through shared memory
// by the TMA engine: a persistent CTA per SM walks its share of the (sequence,
// head) states; a producer warp moves each 64 KB fp32 state (plus the token's
// q, k, v, g) in with ONE bulk copy into a 3-stage ring, eight compute warps
// update it in place, and one bulk copy writes it back.  Loads of the next
// states are in flight while the current one is computed and the previous one
// drains, so HBM sees one continuous read stream and one write stream.
//
// Per state (decay, then erase, then write, then read: "Kimi K3 Architecture
// Explained", section 3), with D = Diag(exp(g)):
//     r = (D S)^T k,   p = (D S)^T q,   u = beta (v - r),
//     S' = D S + k u^T,   o = p + u (k . q)
// Thread t of the compute warps owns float4 column group (t mod 32) of rows
// (t div 32) + 8 m, m = 0..15: its 16 float4 stay in registers between the
// reduction and the update, so shared memory is read once and written once.
//
// Every wait is bounded.  A wait that gives up sets the CTA's abort flag; the
// compute warps decide together whether to stop (a barrier reduction right
// after each wait), so no warp is left at a named barrier the others never
// reach, and the CTA records KDA_ERR_TIMEOUT in dev_status before it exits
// (states it had not reached keep their old value: the step is then incomplete).
#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int D = 128;
constexpr int NSTG = 3;
constexpr int NCW = 8;                 // compute warps
constexpr int NT = (NCW + 1) * 32;     // + one producer warp
constexpr int STATE_B = D * D * 4;     // 64 KB
constexpr long long kWaitLimit = 4000000000ll;

template <typename TA>
struct Layout {
    static constexpr int VEC = D * (int)sizeof(TA);        // one q / k / v row
    static constexpr int Q = STATE_B, K = Q + VEC, V = K + VEC, G = V + VEC, BETA = G + 512;
    static constexpr int STAGE = (BETA + 16 + 127) & ~127;
    static constexpr int RED = NSTG * STAGE;                // fp32 [2][8][128]
    static constexpr int U = RED + 2 * NCW * D * 4;         // fp32 [128]
    static constexpr int BAR = U + D * 4;                   // full[NSTG], empty[NSTG]
    static constexpr int ABORT = BAR + 2 * NSTG * 8;
    static constexpr int BYTES = ABORT + 16 + 1024;
};

__device__ __forceinline__ void bulk_s2g(void *dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src),
                 "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_le1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

template <typename TA>
__global__ void __launch_bounds__(NT, 1) decode_tma_kernel(int units, const TA *q, const TA *k,
                                                           const TA *v, const float *g,
                                                           const float *beta, float *S, TA *out,
                                                           int32_t *dev_status) {
    using L = Layout<TA>;
    extern __shared__ uint8_t smem_raw[];
    // Align by pointer arithmetic on the __shared__ array (not through an integer),
    // so accesses keep the shared address space instead of becoming generic.
    uint8_t *sm = smem_raw + ((1024u - (sm100::smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_addr(sm);
    volatile int *abort = (volatile int *)(sm + L::ABORT);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto full = [&](int s) { return sb + L::BAR + 8 * s; };
    auto empty = [&](int s) { return sb + L::BAR + 8 * (NSTG + s); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTG; ++s) {
            mbar_init(full(s), 2);
            mbar_init(empty(s), 1);
        }
        *abort = 0;
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == NCW) {
        // ---------------- producer
        int i = 0;
        int issued = 0;
        // beta is one scalar per state: load the next one a step ahead so its
        // latency overlaps the wait for a free stage.
        float beta_next = (lane == 0 && (int)blockIdx.x < units) ? beta[blockIdx.x] : 0.f;
        for (int u = blockIdx.x; u < units; u += gridDim.x, ++i) {
            const int st = i % NSTG;
            const float beta_cur = beta_next;
            if (lane == 0 && u + (int)gridDim.x < units) beta_next = beta[u + gridDim.x];
            int ok = 1;
            if (lane == 0) ok = mbar_wait(empty(st), ((i / NSTG) & 1) ^ 1, abort, kWaitLimit);
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            const uint32_t base = sb + st * L::STAGE;
            if (lane == 0) {
                mbar_arrive_expect_tx(full(st), STATE_B + 3 * L::VEC + 512);
                bulk_g2s(base, S + (size_t)u * D * D, STATE_B, full(st));
                bulk_g2s(base + L::Q, q + (size_t)u * D, L::VEC, full(st));
                bulk_g2s(base + L::K, k + (size_t)u * D, L::VEC, full(st));
                bulk_g2s(base + L::V, v + (size_t)u * D, L::VEC, full(st));
                bulk_g2s(base + L::G, g + (size_t)u * D, 512, full(st));
                *(float *)(sm + st * L::STAGE + L::BETA) = beta_cur;
                mbar_arrive(full(st));
            }
            __syncwarp();
            issued = i + 1;
        }
        // On an abort, let loads already in flight land before the CTA can exit.
        if (*abort && lane == 0) {
            volatile int never = 0;
            for (int c = issued - NSTG > 0 ? issued - NSTG : 0; c < issued; ++c)
                mbar_wait(full(c % NSTG), (c / NSTG) & 1, &never, kWaitLimit);
        }
        return;
    }

    // ---------------- compute warps (256 threads)
    const int t = threadIdx.x;
    const int c4 = t & 31, rg = t >> 5;
    float *red_r = (float *)(sm + L::RED);
    float *red_p = red_r + NCW * D;
    float *su = (float *)(sm + L::U);
    int i = 0, prev_st = -1;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++i) {
        const int st = i % NSTG;
        int ok = 1;
        if (lane == 0) ok = mbar_wait(full(st), (i / NSTG) & 1, abort, kWaitLimit);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        // one decision for all compute warps: leave together or not at all
        if (named_bar_or(2, NCW * 32, !ok)) break;
        uint8_t *stg = sm + st * L::STAGE;
        float *Ss = (float *)stg;
        const TA *qs = (const TA *)(stg + L::Q);
        const TA *ks = (const TA *)(stg + L::K);
        const TA *vs = (const TA *)(stg + L::V);
        const float *gs = (const float *)(stg + L::G);
        const float bt = *(const float *)(stg + L::BETA);

        // k . q (every warp, redundantly: no extra barrier)
        float qk = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) qk += act_ld(qs, lane + 32 * e) * act_ld(ks, lane + 32 * e);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) qk += __shfl_xor_sync(0xffffffffu, qk, o);

        float4 x[16];
        float4 r = make_float4(0.f, 0.f, 0.f, 0.f), p = r;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const int row = rg + 8 * m;
            x[m] = *(const float4 *)(Ss + row * D + 4 * c4);
            const float a = __expf(gs[row]), kr = act_ld(ks, row), qr = act_ld(qs, row);
            x[m].x *= a; x[m].y *= a; x[m].z *= a; x[m].w *= a;
            r.x += kr * x[m].x; r.y += kr * x[m].y; r.z += kr * x[m].z; r.w += kr * x[m].w;
            p.x += qr * x[m].x; p.y += qr * x[m].y; p.z += qr * x[m].z; p.w += qr * x[m].w;
        }
        *(float4 *)(red_r + rg * D + 4 * c4) = r;
        *(float4 *)(red_p + rg * D + 4 * c4) = p;
        named_bar_sync(1, NCW * 32);
        if (t < D) {
            float R = 0.f, P = 0.f;
#pragma unroll
            for (int w = 0; w < NCW; ++w) { R += red_r[w * D + t]; P += red_p[w * D + t]; }
            const float uj = bt * (act_ld(vs, t) - R);
            su[t] = uj;
            act_st(out, (size_t)u * D + t, P + uj * qk);
        }
        named_bar_sync(1, NCW * 32);
        const float4 uu = *(const float4 *)(su + 4 * c4);
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const int row = rg + 8 * m;
            const float kr = act_ld(ks, row);
            x[m].x += kr * uu.x; x[m].y += kr * uu.y; x[m].z += kr * uu.z; x[m].w += kr * uu.w;
            *(float4 *)(Ss + row * D + 4 * c4) = x[m];
        }
        fence_async_smem();
        named_bar_sync(1, NCW * 32);
        if (t == 0) {
            bulk_s2g(S + (size_t)u * D * D, smem_addr(Ss), STATE_B);
            // the previous stage's store has finished reading shared memory: hand it back
            bulk_wait_read_le1();
            if (prev_st >= 0) mbar_arrive(empty(prev_st));
        }
        prev_st = st;
    }
    if (t == 0) {
        bulk_wait_all();
        if (prev_st >= 0) mbar_arrive(empty(prev_st));
        if (*abort) dev_fail(dev_status, KDA_ERR_TIMEOUT);
    }
}

}  // namespace

bool decode_tma_supported(int dk, int dv) { return dk == D && dv == D; }

cudaError_t launch_decode_tma(int batch, int H, int act, const void *q, const void *k,
                              const void *v, const float *g, const float *beta, float *S,
                              void *out, int32_t *dev_status, cudaStream_t st) {
    const int units = batch * H;
    if (units == 0) return cudaSuccess;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int grid = units < sms ? units : sms;
    if (act == KDA_DTYPE_F32) {
        const int bytes = Layout<float>::BYTES;
        cudaError_t e = set_max_dynamic_smem((const void *)decode_tma_kernel<float>, bytes);
        if (e != cudaSuccess) return e;
        decode_tma_kernel<float><<<grid, NT, bytes, st>>>(units, (const float *)q, (const float *)k,
                                                          (const float *)v, g, beta, S,
                                                          (float *)out, dev_status);
    } else {
        const int bytes = Layout<__nv_bfloat16>::BYTES;
        cudaError_t e = set_max_dynamic_smem((const void *)decode_tma_kernel<__nv_bfloat16>, bytes);
        if (e != cudaSuccess) return e;
        decode_tma_kernel<__nv_bfloat16><<<grid, NT, bytes, st>>>(
            units, (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v, g,
            beta, S, (__nv_bfloat16 *)out, dev_status);
    }
    return cudaGetLastError();
}

}  // namespace kda
