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
    if (!segment_range(p.cu, n, p.N, p.T_tot, s, p.Sg, p.dev_status, a, b, p.lead)) return false;
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
    if (!segment_range(p.cu, n, p.N, p.T_tot, s, p.Sg, p.dev_status, a, b, p.lead)) return;
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

// ---- tcgen05 path: D[t][j] = sum_i aux[t][i] start_s[i][j] over 128-token tiles.
// A persistent CTA per SM walks a contiguous range of the (sequence, head,
// segment, tile) list, so consecutive tiles share a segment and its start image
// is loaded once per segment.  Warp roles:
//   warp 0   producer: per tile, the A_t^T q_t rows and the out rows as two TMA
//            boxes each (64 columns x 128 tokens, 128-byte swizzle) into one of
//            three stages; per segment, the start image (K-major core matrices
//            without swizzle) by one bulk copy.
//   warp 1   one thread issues eight tcgen05.mma (M = N = 128, K = 16) per tile
//            into one of two TMEM accumulators and commits.
//   warps 2-9 epilogue: thread = (token row = TMEM lane, 64-column half): reads
//            its 64 products with one tcgen05.ld, adds its zero-start out values
//            from the stage in fp32 and puts the results back in place; then one
//            thread stores the tile with one TMA store per 64-column box (a tile
//            that ends inside the segment is written row by row instead, only its
//            live rows).
// A stage is free once its products are done (commit) and its tile has been
// stored (the bulk store has read the stage); an accumulator once the epilogue
// has loaded it; the image once the last products of its segment are done.  Every wait is
// bounded; on an abort the roles stop, copies and products in flight complete
// before the CTA frees its TMEM, and dev_status records KDA_ERR_TIMEOUT.
constexpr int TC_TILE = 128;
constexpr int TC_NST = 3;
constexpr int TC_STAGE = 65536;                     // aux (2 x 16 KB) then out (2 x 16 KB)
constexpr int TC_IMG = TC_NST * TC_STAGE;           // start image, 32 KB
constexpr int TC_BAR = TC_IMG + 32768;
enum { PB_FULL = 0, PB_EMPTY = PB_FULL + TC_NST, PB_ACCF = PB_EMPTY + TC_NST, PB_ACCE = PB_ACCF + 2,
       PB_IMGF = PB_ACCE + 2, PB_IMGE = PB_IMGF + 1, PB_FIN = PB_IMGE + 1, PB_N = PB_FIN + 1 };
constexpr int TC_MISC = TC_BAR + PB_N * 8;          // [0] abort, [4] TMEM base
constexpr int TC_SMEM = TC_MISC + 16 + 1024;        // + slack for the 1024-byte alignment
constexpr uint32_t TC_COLS = 256;                   // two 128-column accumulators
constexpr long long kTcWaitLimit = 4000000000ll;    // ~2 s of SM clocks
static_assert(TC_SMEM <= 227 * 1024, "shared memory budget");

struct TileRef {
    int us;       // (sequence, head, segment) index: (n H + h) Sg + s
    int h, t0, nt;
    bool ok;      // the tile has tokens
};

// Tile f of the list (segments from seg_begin on, ntile tiles reserved per segment).
__device__ __forceinline__ TileRef tile_ref(const PrefillArgs &p, long long f, int ntile) {
    TileRef r;
    const int sact = p.Sg - p.seg_begin;
    const long long us_act = f / ntile;
    const int tile = (int)(f % ntile);
    const int unit = (int)(us_act / sact), s = p.seg_begin + (int)(us_act % sact);
    const int n = unit / p.H;
    r.h = unit % p.H;
    r.us = unit * p.Sg + s;
    int a, b;
    r.ok = segment_range(p.cu, n, p.N, p.T_tot, s, p.Sg, p.dev_status, a, b, p.lead);
    r.t0 = a + tile * TC_TILE;
    r.nt = min(TC_TILE, b - r.t0);
    r.ok = r.ok && r.t0 < b;
    return r;
}

constexpr int TC_EPI = 8;  // epilogue warps
__global__ void __launch_bounds__(32 * (2 + TC_EPI), 1) combine_tc_kernel(const __grid_constant__ PrefillArgs p,
                                                            const __grid_constant__ CUtensorMap tm_aux,
                                                            const __grid_constant__ CUtensorMap tm_out,
                                                            const __nv_bfloat16 *img, int ntile,
                                                            long long total) {
    extern __shared__ uint8_t smem_raw[];
    griddep_wait();  // out, A_t^T q_t and the start images come from earlier kernels
    griddep_launch_dependents();
    uint8_t *sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_addr(sm);
    auto bar = [&](int i) { return sb + TC_BAR + 8 * i; };
    volatile int *abort = (volatile int *)(sm + TC_MISC);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long f0 = (long long)blockIdx.x * total / gridDim.x;
    const long long f1 = (long long)(blockIdx.x + 1) * total / gridDim.x;

    if (threadIdx.x == 0) {
        for (int i = 0; i < TC_NST; ++i) {
            mbar_init(bar(PB_FULL + i), 1);
            mbar_init(bar(PB_EMPTY + i), 1 + 1);  // products done + tile stored
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(PB_ACCF + i), 1);
            mbar_init(bar(PB_ACCE + i), TC_EPI);
        }
        mbar_init(bar(PB_IMGF), 1);
        mbar_init(bar(PB_IMGE), 1);
        mbar_init(bar(PB_FIN), 1);
        *abort = 0;
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(sb + TC_MISC + 4, TC_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *(volatile uint32_t *)(sm + TC_MISC + 4);

    if (warp == 0) {
        // ---- producer
        if (lane == 0) {
            const uint64_t ta = reinterpret_cast<uint64_t>(&tm_aux);
            const uint64_t to = reinterpret_cast<uint64_t>(&tm_out);
            int i = 0, nimg = 0, cur = -1, pending = 0;
            for (long long f = f0; f < f1; ++f) {
                const TileRef t = tile_ref(p, f, ntile);
                if (!t.ok) continue;
                if (t.us != cur) {  // a new segment: its start image, once the old one is free
                    if (nimg > 0 && !mbar_wait(bar(PB_IMGE), (nimg - 1) & 1, abort, kTcWaitLimit))
                        break;
                    mbar_arrive_expect_tx(bar(PB_IMGF), 32768);
                    bulk_g2s(sb + TC_IMG, img + (size_t)t.us * kStartImgElems, 32768, bar(PB_IMGF));
                    cur = t.us;
                    ++nimg;
                }
                const int stg = i % TC_NST;
                if (!mbar_wait(bar(PB_EMPTY + stg), ((i / TC_NST) & 1) ^ 1, abort, kTcWaitLimit))
                    break;
                const uint32_t st = sb + stg * TC_STAGE;
                mbar_arrive_expect_tx(bar(PB_FULL + stg), 4 * 16384);
                // rows past the segment's end come along (the next segment's, or zero
                // fill past the array); they are never used
#pragma unroll
                for (int bx = 0; bx < 2; ++bx) {
                    tma_load_2d(st + bx * 16384, ta, t.h * 128 + 64 * bx, t.t0, bar(PB_FULL + stg));
                    tma_load_2d(st + 32768 + bx * 16384, to, t.h * 128 + 64 * bx, t.t0,
                                bar(PB_FULL + stg));
                }
                ++i;
                pending = i;
            }
            // on an abort, let the copies in flight land before the CTA exits
            if (*abort) {
                volatile int never = 0;
                for (int k = pending - TC_NST > 0 ? pending - TC_NST : 0; k < pending; ++k)
                    mbar_wait(bar(PB_FULL + k % TC_NST), (k / TC_NST) & 1, &never, kTcWaitLimit);
                if (nimg > 0) mbar_wait(bar(PB_IMGF), (nimg - 1) & 1, &never, kTcWaitLimit);
            }
        }
    } else if (warp == 1) {
        // ---- products
        if (lane == 0) {
            const uint32_t idesc = umma_idesc_bf16(128, 128);
            int i = 0, nimg = 0, cur = -1;
            for (long long f = f0; f < f1; ++f) {
                const TileRef t = tile_ref(p, f, ntile);
                if (!t.ok) continue;
                if (t.us != cur) {
                    if (!mbar_wait(bar(PB_IMGF), nimg & 1, abort, kTcWaitLimit)) break;
                    cur = t.us;
                    ++nimg;
                }
                const int stg = i % TC_NST, acc = i & 1;
                if (!mbar_wait(bar(PB_FULL + stg), (i / TC_NST) & 1, abort, kTcWaitLimit)) break;
                if (!mbar_wait(bar(PB_ACCE + acc), ((i >> 1) & 1) ^ 1, abort, kTcWaitLimit)) break;
                tc_fence_after();
                const uint32_t st = sb + stg * TC_STAGE;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    umma_bf16(tmem + 128 * acc,
                              umma_desc_sw128(st + (kk >> 2) * 16384 + (kk & 3) * 32, 1024),
                              umma_desc(sb + TC_IMG + kk * 4096, 2048, 128), idesc, kk > 0);
                umma_commit(bar(PB_ACCF + acc));
                umma_commit(bar(PB_EMPTY + stg));
                // the last tile of this segment in the range frees the image
                bool last = true;
                for (long long g = f + 1; g < f1; ++g) {
                    const TileRef u = tile_ref(p, g, ntile);
                    if (u.ok) {
                        last = u.us != cur;
                        break;
                    }
                }
                if (last) umma_commit(bar(PB_IMGE));
                ++i;
            }
            if (*abort) {  // products in flight complete before TMEM is freed
                umma_commit(bar(PB_FIN));
                volatile int never = 0;
                mbar_wait(bar(PB_FIN), 0, &never, kTcWaitLimit);
            }
        }
    } else {
        // ---- epilogue: thread = (token row = TMEM lane 32 (warp % 4) + lane, columns
        // 64 half .. 64 half + 63 = TMA box `half` of the out tile)
        const int row = 32 * (warp & 3) + lane, half = (warp - 2) >> 2;
        const bool leader = warp == 2 && lane == 0;
        const uint64_t to = reinterpret_cast<uint64_t>(&tm_out);
        int i = 0, pending = -1;  // stage whose bulk store may still read shared memory
        for (long long f = f0; f < f1; ++f) {
            const TileRef t = tile_ref(p, f, ntile);
            if (!t.ok) continue;
            const int stg = i % TC_NST, acc = i & 1;
            bool ok = mbar_wait(bar(PB_ACCF + acc), (i >> 1) & 1, abort, kTcWaitLimit) &&
                      mbar_wait(bar(PB_FULL + stg), (i / TC_NST) & 1, abort, kTcWaitLimit);
            // one decision for the eight warps (they meet at a named barrier below)
            if (named_bar_or(1, 32 * TC_EPI, !ok)) break;
            tc_fence_after();
            float d[64];
            tmem_ld64(tmem + 128 * acc + ((uint32_t)(32 * (warp & 3)) << 16) + 64 * half, d);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(PB_ACCE + acc));  // the accumulator is in registers
            uint8_t *obox = sm + stg * TC_STAGE + 32768 + half * 16384 + row * 128;
#pragma unroll
            for (int q = 0; q < 8; ++q) {  // 16-byte chunk q of this row's box, swizzled
                uint4 *ptr = (uint4 *)(obox + ((q ^ (row & 7)) << 4));
                const uint4 ov = *ptr;
                const __nv_bfloat162 *o2 = (const __nv_bfloat162 *)&ov;
                const float *dd = d + 8 * q;
                const float2 a0 = __bfloat1622float2(o2[0]), a1 = __bfloat1622float2(o2[1]);
                const float2 a2 = __bfloat1622float2(o2[2]), a3 = __bfloat1622float2(o2[3]);
                *ptr = make_uint4(pack_bf16x2(a0.x + dd[0], a0.y + dd[1]),
                                  pack_bf16x2(a1.x + dd[2], a1.y + dd[3]),
                                  pack_bf16x2(a2.x + dd[4], a2.y + dd[5]),
                                  pack_bf16x2(a3.x + dd[6], a3.y + dd[7]));
            }
            const bool full_tile = t.nt == TC_TILE;
            if (full_tile) fence_async_smem();  // the tile goes out through the TMA engine
            named_bar_sync(1, 32 * TC_EPI);
            if (!full_tile && row < t.nt) {  // a partial tile: its live rows, row by row
                uint4 *orow = (uint4 *)((__nv_bfloat16 *)p.out +
                                        ((size_t)(t.t0 + row) * p.H + t.h) * 128 + 64 * half);
#pragma unroll
                for (int q = 0; q < 8; ++q) orow[q] = *(const uint4 *)(obox + ((q ^ (row & 7)) << 4));
            }
            if (!full_tile) named_bar_sync(1, 32 * TC_EPI);  // the stage has been read
            if (leader) {
                if (full_tile) {
#pragma unroll
                    for (int bx = 0; bx < 2; ++bx)
                        tma_store_2d(to, sb + stg * TC_STAGE + 32768 + bx * 16384,
                                     t.h * 128 + 64 * bx, t.t0);
                    cp_bulk_commit();
                    cp_bulk_wait_read<1>();  // the previous tile's store has read its stage
                    if (pending >= 0) mbar_arrive(bar(PB_EMPTY + pending));
                    pending = stg;
                } else {
                    cp_bulk_wait_read<0>();
                    if (pending >= 0) mbar_arrive(bar(PB_EMPTY + pending));
                    pending = -1;
                    mbar_arrive(bar(PB_EMPTY + stg));
                }
            }
            ++i;
        }
        if (leader) {  // every store has completed before the CTA ends
            cp_bulk_wait<0>();
            if (pending >= 0) mbar_arrive(bar(PB_EMPTY + pending));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abort) dev_fail(p.dev_status, KDA_ERR_TIMEOUT);
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
    // tokens of one segment: at most ceil(ceil(T_tot / 16) / Sg) blocks of 16; with a
    // lead segment (skipped here) the others split what the lead leaves of the
    // longest possible sequence
    const long long blocks = ((long long)a.T_tot + 15) / 16;
    long long seg_blocks = (blocks + a.Sg - 1) / a.Sg;
    if (a.lead > 0 && a.Sg >= 2 && a.seg_begin >= 1) {
        const long long rest = blocks - (blocks * a.lead >> 16);
        seg_blocks = (rest + a.Sg - 2) / (a.Sg - 1);
    }
    const long long seg_tokens = 16 * seg_blocks;
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
        // (sequence, head, segment) x tiles from seg_begin on; one persistent CTA per SM
        const long long ntile = (seg_tokens + TC_TILE - 1) / TC_TILE;
        const long long total = (long long)a.N * a.H * (a.Sg - a.seg_begin) * ntile;
        if (total <= 0) return cudaSuccess;
        int dev = 0, sms = 148;
        if (cudaGetDevice(&dev) == cudaSuccess)
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const unsigned grid = (unsigned)(total < sms ? total : sms);
        return launch_dependent(combine_tc_kernel, dim3(grid), dim3(32 * (2 + TC_EPI)), TC_SMEM, st,
                                a, tm, tmo, start_img, (int)ntile, total);
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
