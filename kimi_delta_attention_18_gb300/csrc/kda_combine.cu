// Output correction of the context-parallel split.
//
// Within segment s of a sequence the state after token t is S_t = A_t start_s +
// B_t (transfer matrix and zero-initial state so far: Kimi K3 technical-report
// digest, section 2.4 (1)), so the output is linear in the segment's start state:
//     o_t = S_t^T q_t = B_t^T q_t + start_s^T (A_t^T q_t).
// The transfer pass writes the first term into out and A_t^T q_t into aux_out;
// once the scan has produced start_s, this kernel adds the second term:
//     out[t, h, :] += start_s^T aux_out[t, h, :]
// a dense (tokens x dk) x (dk x dv) product per segment, fully parallel.
//   BF16, dk = dv = 128, with the scan's BF16 start images: tcgen05 (one CTA per
//       (sequence, head, segment, 128-token tile): A_t^T q_t rows by TMA and the
//       start image by one bulk copy into shared memory, eight MMAs into 128
//       TMEM columns, fp32 read-back and correction of out).
//   BF16, dk = dv = 128, from fp32 start states: mma.sync m16n8k16 (start_s
//       rounded to BF16, fp32 accumulation); one CTA per (sequence, head,
//       segment, group of 64-token tiles), so each start state is converted once
//       per group.
//   fp32 (any dk, dv <= 128): CUDA cores, fp32 throughout.
#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int TILE = 64;

// Token range of this CTA's tile within its segment; false if nothing to do.
__device__ __forceinline__ bool tile_range(const PrefillArgs &p, int u, int tile, int &h,
                                           int &s, int &t0, int &t1) {
    const int n = u / (p.H * p.Sg);
    h = (u / p.Sg) % p.H;
    s = u % p.Sg;
    if (s < p.seg_begin) return false;  // segments before seg_begin start from zeros
    int a, b;
    if (!segment_range(p.cu, n, p.N, p.T_tot, s, p.Sg, p.dev_status, a, b)) return false;
    t0 = a + tile * TILE;
    t1 = min(b, t0 + TILE);
    return t0 < t1;
}

constexpr int SB_LD = 136;  // padded bf16 row (272 bytes): ldmatrix rows hit distinct banks
constexpr int BF_WARPS = 8;
constexpr int BF16_SMEM = (128 + BF_WARPS * 16) * SB_LD * 2;

// One CTA per (sequence, head, segment, group of `gtiles` 64-token tiles): start_s
// is converted to BF16 in shared memory once, then each warp takes 16-token slabs
// of the group on its own (aux rows staged in its private shared rows, the
// product on mma.sync, out read, corrected in fp32 and rewritten).
__global__ void __launch_bounds__(BF_WARPS * 32) combine_bf16_kernel(
    const __grid_constant__ PrefillArgs p, const float *starts, const __nv_bfloat16 *aux,
    int group_base, int gtiles) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    __nv_bfloat16 *Sb = (__nv_bfloat16 *)smem_raw;  // start_s, [i][j]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    __nv_bfloat16 *Ab = Sb + 128 * SB_LD + warp * 16 * SB_LD;  // this warp's aux rows [t][i]
    const int u = blockIdx.x;
    const int n = u / (p.H * p.Sg), h = (u / p.Sg) % p.H, s = u % p.Sg;
    if (s < p.seg_begin) return;  // segments before seg_begin start from zeros
    int a, b;
    if (!segment_range(p.cu, n, p.N, p.T_tot, s, p.Sg, p.dev_status, a, b)) return;
    const int t0 = a + (group_base + blockIdx.y) * gtiles * TILE;
    const int t1 = min(b, t0 + gtiles * TILE);
    if (t0 >= t1) return;
    const size_t unit = (size_t)(u / p.Sg);  // (n, h)
    const float *st = starts + (unit * p.Sg + s) * 128 * 128;
    // Loads are issued in batches (all in flight at once), then converted and stored.
#pragma unroll 1
    for (int base = 0; base < 128 * 32; base += BF_WARPS * 32 * 8) {  // 128 rows x 32 float4
        float4 v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = base + tid + BF_WARPS * 32 * q;
            v[q] = *(const float4 *)(st + (e >> 5) * 128 + 4 * (e & 31));
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = base + tid + BF_WARPS * 32 * q;
            uint2 w;
            w.x = pack_bf16x2(v[q].x, v[q].y);
            w.y = pack_bf16x2(v[q].z, v[q].w);
            *(uint2 *)(Sb + (e >> 5) * SB_LD + 4 * (e & 31)) = w;
        }
    }
    __syncthreads();

    const uint32_t ab = smem_addr(Ab), sbb = smem_addr(Sb);
    __nv_bfloat16 *out = (__nv_bfloat16 *)p.out;
    const int g8 = lane >> 2, t4 = lane & 3;
#pragma unroll 1
    for (int r0 = t0 + 16 * warp; r0 < t1; r0 += 16 * BF_WARPS) {
        const int nt = min(16, t1 - r0);
        {
            uint4 w[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {  // 16 rows x 16 chunks of 16 bytes
                const int e = lane + 32 * q, r = e >> 4, c8 = e & 15;
                w[q] = r < nt ? *(const uint4 *)(aux + ((size_t)(r0 + r) * p.H + h) * 128 + 8 * c8)
                              : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int e = lane + 32 * q, r = e >> 4, c8 = e & 15;
                *(uint4 *)(Ab + r * SB_LD + 8 * c8) = w[q];
            }
        }
        __syncwarp();
        float acc[16][4];
#pragma unroll
        for (int q = 0; q < 16; ++q) acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t af[4];
            ldsm_x4(ab + ((lane & 15) * SB_LD + kk * 16 + (lane >> 4) * 8) * 2, af);
#pragma unroll
            for (int np = 0; np < 8; ++np) {
                uint32_t bf[4];
                ldsm_x4_t(sbb + ((kk * 16 + (lane & 15)) * SB_LD + np * 16 + (lane >> 4) * 8) * 2, bf);
                mma_bf16_16816(acc[2 * np], af, bf[0], bf[1]);
                mma_bf16_16816(acc[2 * np + 1], af, bf[2], bf[3]);
            }
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int r = g8 + 8 * hh;
            if (r >= nt) continue;
            __nv_bfloat162 *orow =
                (__nv_bfloat162 *)(out + ((size_t)(r0 + r) * p.H + h) * 128 + 2 * t4);
            __nv_bfloat162 cur[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) cur[q] = orow[4 * q];  // all 16 reads in flight
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const float2 c = __bfloat1622float2(cur[q]);
                orow[4 * q] = __floats2bfloat162_rn(c.x + acc[q][2 * hh], c.y + acc[q][2 * hh + 1]);
            }
        }
        __syncwarp();  // the staging rows are rewritten for the next slab
    }
}

// ---- tcgen05 path: D[t][j] = sum_i aux[t][i] start_s[i][j] over a 128-token tile
constexpr int TC_TILE = 128;
constexpr int TC_A = 0;         // aux tile: 2 TMA boxes of 64 channels x 128 rows, 128-byte swizzle
constexpr int TC_B = 32768;     // start image: K-major core matrices without swizzle (rows j)
constexpr int TC_O = 65536;     // out tile: 2 TMA boxes of 64 columns x 128 rows, 128-byte swizzle
constexpr int TC_BAR = 98304;   // [0] operands landed, [8] products done, [16] abort, [24] TMEM base
constexpr int TC_SMEM = TC_BAR + 32 + 1024;  // + slack for the 1024-byte alignment of the base
constexpr uint32_t TC_COLS = 128;
constexpr long long kTcWaitLimit = 4000000000ll;  // ~2 s of SM clocks

// A (the tile's A_t^T q_t rows) and the tile's out rows arrive as two 64-column
// TMA boxes each with 128-byte swizzle, so every copy moves whole 128-byte row
// pieces; B, the start image, is K-major without swizzle (core matrices 8 rows x
// 16 bytes, adjacent along K 2048 bytes apart, 8-row groups 128 bytes apart).
// The accumulator row m is TMEM lane m, so warp w reads the products of tokens
// 32w..32w+31 and corrects their out rows in fp32 (each thread reads its row's
// swizzled chunks: conflict-free).  All waits are bounded; a CTA that gives up
// records KDA_ERR_TIMEOUT, lets its copies land and frees its TMEM.
__global__ void __launch_bounds__(128) combine_tc_kernel(const __grid_constant__ PrefillArgs p,
                                                         const __grid_constant__ CUtensorMap tm_aux,
                                                         const __grid_constant__ CUtensorMap tm_out,
                                                         const __nv_bfloat16 *img, int tile_base) {
    extern __shared__ uint8_t smem_raw[];
    griddep_wait();  // out, A_t^T q_t and the start images come from earlier kernels
    griddep_launch_dependents();
    uint8_t *sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_addr(sm);
    const uint32_t full = sb + TC_BAR, mmad = sb + TC_BAR + 8;
    volatile int *abort = (volatile int *)(sm + TC_BAR + 16);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int u = blockIdx.x;
    const int n = u / (p.H * p.Sg), h = (u / p.Sg) % p.H, s = u % p.Sg;
    if (s < p.seg_begin) return;  // segments before seg_begin start from zeros
    int a, b;
    if (!segment_range(p.cu, n, p.N, p.T_tot, s, p.Sg, p.dev_status, a, b)) return;
    const int t0 = a + (tile_base + blockIdx.y) * TC_TILE;
    if (t0 >= b) return;
    const int nt = min(TC_TILE, b - t0);
    const size_t unit = (size_t)(u / p.Sg);  // (n, h)

    const int row = 32 * warp + lane;  // this thread's token in the tile
    const bool live = row < nt;
    uint4 *orow = (uint4 *)((__nv_bfloat16 *)p.out + ((size_t)(t0 + row) * p.H + h) * 128);

    if (tid == 0) {
        mbar_init(full, 1);
        mbar_init(mmad, 1);
        *abort = 0;
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(sb + TC_BAR + 24, TC_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *(volatile uint32_t *)(sm + TC_BAR + 24);

    bool landed = false;
    if (tid == 0) {
        mbar_arrive_expect_tx(full, 3 * 32768);
        const uint64_t ta = reinterpret_cast<uint64_t>(&tm_aux);
        const uint64_t to = reinterpret_cast<uint64_t>(&tm_out);
        // rows past the segment's end come along (the next segment's, or zero fill
        // past the array); they are never used
#pragma unroll
        for (int bx = 0; bx < 2; ++bx) {
            tma_load_2d(sb + TC_A + bx * 16384, ta, h * 128 + 64 * bx, t0, full);
            tma_load_2d(sb + TC_O + bx * 16384, to, h * 128 + 64 * bx, t0, full);
        }
        bulk_g2s(sb + TC_B, img + (unit * p.Sg + s) * (size_t)kStartImgElems, 32768, full);
        landed = mbar_wait(full, 0, abort, kTcWaitLimit);
        if (landed) {
            tc_fence_after();
            const uint32_t idesc = umma_idesc_bf16(128, 128);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                umma_bf16(tmem, umma_desc_sw128(sb + TC_A + (kk >> 2) * 16384 + (kk & 3) * 32, 1024),
                          umma_desc(sb + TC_B + kk * 4096, 2048, 128), idesc, kk > 0);
            umma_commit(mmad);
        }
    }
    // products done; the operand barrier (long complete) orders the out tile's
    // landing before this thread's reads of it
    const bool done = mbar_wait(mmad, 0, abort, kTcWaitLimit) && mbar_wait(full, 0, abort, kTcWaitLimit);
    if (__all_sync(0xffffffffu, done)) {
        tc_fence_after();
        uint4 ov[16];  // this thread's out row from the swizzled tile
#pragma unroll
        for (int q = 0; q < 16; ++q)
            ov[q] = *(const uint4 *)(sm + TC_O + (q >> 3) * 16384 + row * 128 +
                                     (((q & 7) ^ (row & 7)) << 4));
#pragma unroll
        for (int c = 0; c < 4; ++c) {  // 32 columns j at a time
            float d[32];
            tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + 32 * c, d);
            if (live) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const __nv_bfloat162 *o2 = (const __nv_bfloat162 *)&ov[4 * c + q4];
                    const float *dd = d + 8 * q4;
                    uint4 w;
                    const float2 f0 = __bfloat1622float2(o2[0]), f1 = __bfloat1622float2(o2[1]);
                    const float2 f2 = __bfloat1622float2(o2[2]), f3 = __bfloat1622float2(o2[3]);
                    w.x = pack_bf16x2(f0.x + dd[0], f0.y + dd[1]);
                    w.y = pack_bf16x2(f1.x + dd[2], f1.y + dd[3]);
                    w.z = pack_bf16x2(f2.x + dd[4], f2.y + dd[5]);
                    w.w = pack_bf16x2(f3.x + dd[6], f3.y + dd[7]);
                    orow[4 * c + q4] = w;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && *abort) {
        dev_fail(p.dev_status, KDA_ERR_TIMEOUT);
        if (!landed) {  // let the copies in flight land before the CTA exits
            volatile int never = 0;
            mbar_wait(full, 0, &never, kTcWaitLimit);
        }
    }
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TC_COLS);
    }
}

template <typename TA>
__global__ void __launch_bounds__(256) combine_simt_kernel(const __grid_constant__ PrefillArgs p,
                                                           const float *starts, const TA *aux,
                                                           int tile) {
    extern __shared__ float sm[];
    const int dk = p.dk, dv = p.dv;
    float *Ss = sm;             // [dk][dv]
    float *As = sm + dk * dv;   // [TILE][dk]
    int h, s, t0, t1;
    if (!tile_range(p, blockIdx.x, tile + blockIdx.y, h, s, t0, t1)) return;
    const size_t unit = (size_t)(blockIdx.x / p.Sg);
    const float *st = starts + (unit * p.Sg + s) * (size_t)dk * dv;
    for (int e = threadIdx.x; e < dk * dv; e += 256) Ss[e] = st[e];
    const int nt = t1 - t0;
    for (int e = threadIdx.x; e < nt * dk; e += 256) {
        const int r = e / dk, i = e % dk;
        As[e] = act_ld(aux, ((size_t)(t0 + r) * p.H + h) * dk + i);
    }
    __syncthreads();
    TA *out = (TA *)p.out;
    for (int e = threadIdx.x; e < nt * dv; e += 256) {
        const int r = e / dv, j = e % dv;
        float acc = 0.f;
        for (int i = 0; i < dk; ++i) acc = fmaf(As[r * dk + i], Ss[i * dv + j], acc);
        const size_t o = ((size_t)(t0 + r) * p.H + h) * dv + j;
        act_st(out, o, act_ld(out, o) + acc);
    }
}

}  // namespace

bool combine_uses_images(const PrefillArgs &a, const void *aux_out,
                         const __nv_bfloat16 *start_img) {
    return a.act == KDA_DTYPE_BF16 && a.dk == 128 && a.dv == 128 && start_img &&
           sm100::tensor_map_encoder() && ((uintptr_t)start_img & 15u) == 0 &&
           ((uintptr_t)aux_out & 15u) == 0 && ((uintptr_t)a.out & 15u) == 0;
}

cudaError_t launch_combine(const PrefillArgs &a, const float *starts, const void *aux_out,
                           const __nv_bfloat16 *start_img, cudaStream_t st) {
    const long long units = (long long)a.N * a.H * a.Sg;
    if (units == 0 || a.T_tot == 0) return cudaSuccess;
    // tokens of one segment: at most ceil(ceil(T_tot / 16) / Sg) blocks of 16
    const long long blocks = ((long long)a.T_tot + 15) / 16;
    const long long seg_tokens = 16 * ((blocks + a.Sg - 1) / a.Sg);
    const long long tiles = (seg_tokens + TILE - 1) / TILE;
    PFN_cuTensorMapEncodeTiled_v12000 enc = sm100::tensor_map_encoder();
    if (combine_uses_images(a, aux_out, start_img)) {
        // aux and out viewed as [T_tot, H * 128] BF16, boxes of 64 columns x 128
        // tokens with 128-byte swizzle
        CUtensorMap tm, tmo;
        const cuuint64_t dims[2] = {(cuuint64_t)a.H * 128, (cuuint64_t)a.T_tot};
        const cuuint64_t strides[1] = {(cuuint64_t)a.H * 128 * 2};
        const cuuint32_t box[2] = {64, (cuuint32_t)TC_TILE};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(aux_out), dims,
                strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
                CUDA_SUCCESS ||
            enc(&tmo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.out, dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
                CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        cudaError_t e = set_max_dynamic_smem((const void *)combine_tc_kernel, TC_SMEM);
        if (e != cudaSuccess) return e;
        const long long tc_tiles = (seg_tokens + TC_TILE - 1) / TC_TILE;
        for (long long base = 0; base < tc_tiles; base += 65535) {
            const unsigned ny = (unsigned)(tc_tiles - base < 65535 ? tc_tiles - base : 65535);
            e = launch_dependent(combine_tc_kernel, dim3((unsigned)units, ny), dim3(128), TC_SMEM, st,
                                 a, tm, tmo, start_img, (int)base);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    if (a.act == KDA_DTYPE_BF16 && a.dk == 128 && a.dv == 128) {
        // Tiles per CTA: about one CTA per SM, each reusing its converted start
        // state for as many tiles as that allows (at least two: the eight warps
        // take 128 tokens per pass).
        int dev = 0, sms = 148;
        if (cudaGetDevice(&dev) == cudaSuccess)
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const long long active = units - (long long)a.N * a.H * a.seg_begin;
        long long gtiles = active > 0 ? (active * tiles) / sms : 2;
        gtiles = gtiles < 2 ? 2 : gtiles;
        gtiles = gtiles > tiles ? tiles : gtiles;
        const long long groups = (tiles + gtiles - 1) / gtiles;
        cudaError_t e = set_max_dynamic_smem((const void *)combine_bf16_kernel, BF16_SMEM);
        if (e != cudaSuccess) return e;
        // grid.y is limited to 65535: launch group ranges one after another
        for (long long base = 0; base < groups; base += 65535) {
            const unsigned ny = (unsigned)(groups - base < 65535 ? groups - base : 65535);
            combine_bf16_kernel<<<dim3((unsigned)units, ny), BF_WARPS * 32, BF16_SMEM, st>>>(
                a, starts, (const __nv_bfloat16 *)aux_out, (int)base, (int)gtiles);
            e = cudaGetLastError();
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    for (long long base = 0; base < tiles; base += 65535) {
        const unsigned ny = (unsigned)(tiles - base < 65535 ? tiles - base : 65535);
        dim3 grid((unsigned)units, ny);
        const size_t smem = ((size_t)a.dk * a.dv + (size_t)TILE * a.dk) * sizeof(float);
        cudaError_t e;
        if (a.act == KDA_DTYPE_F32) {
            e = set_max_dynamic_smem((const void *)combine_simt_kernel<float>, (int)smem);
            if (e != cudaSuccess) return e;
            combine_simt_kernel<float><<<grid, 256, smem, st>>>(a, starts, (const float *)aux_out,
                                                                (int)base);
        } else {
            e = set_max_dynamic_smem((const void *)combine_simt_kernel<__nv_bfloat16>, (int)smem);
            if (e != cudaSuccess) return e;
            combine_simt_kernel<__nv_bfloat16><<<grid, 256, smem, st>>>(
                a, starts, (const __nv_bfloat16 *)aux_out, (int)base);
        }
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace kda
