// Tensor-memory chunked KDA prefill for BF16 activations at dk = dv = 128 (sm_103a).
//
// What it computes: the chunked form of the KDA recurrence (decay, then erase,
// then write, then read: "Kimi K3 Architecture Explained", section 3).  The
// bounded log-decay g > -5 keeps every in-block factor exp(+-Gamma), |Gamma| <
// 80, inside BF16 range, so both the intra-block ("diagonal") and the state
// ("off-diagonal") products run on tensor cores with BF16 operands and fp32
// accumulation (Kimi K3 technical-report digest, section 2.1 (1)).  Per 16-token
// block, from the state S (128 x 128, fp32, rows = key channels i, columns =
// value columns j):
//   prep (state-free):  Gamma = cumsum g;  Kh = K e^{Gamma};  Kt = K e^{-Gamma};
//                       Qh = Q e^{Gamma};  Kb = K e^{Gamma_C - Gamma};
//                       L = Diag(beta) strict_lower(Kh Kt^T);  Mq = lower(Qh Kt^T);
//                       T = (I + L)^{-1} Diag(beta)
//   chain (sequential): U = T (V - Kh S);  O = Qh S + Mq U;  S <- e^{Gamma_C} S + Kb^T U
// The digest's FlashKDA overlaps intra-block work with cross-block state
// propagation (section 2.4 (1)); here that is warp specialisation in a CTA of
// three warpgroups:
//
//   warpgroup 0   prep: each warp prepares whole blocks on its own (TMA loads of
//                 q, k, v, g into its input stage, the elementwise factors, L and
//                 Mq on mma.sync, T by forward substitution) and writes them into
//                 a record slot: [Kh; Qh] as the B operand of the first tensor-core
//                 product (K-major, 128-byte swizzle), Kb^T as the B operand of the
//                 second (K-major), V, T, Mq and e^{Gamma_C}.
//   warpgroups 1, 2   one chain each: thread j owns value column j of S (S^T row j
//                 = TMEM lane j) as 128 fp32 registers.  Per block:
//       MMA1 (tcgen05, M=128 N=32 K=128):  [E^T | P^T] = S^T [Kh^T | Qh^T], with S^T
//            in BF16 read as the A operand straight from tensor memory;
//       U^T = (V^T - E^T) T^T and O^T = P^T + U^T Mq^T on mma.sync (16 x 16 blocks,
//            loaded from tensor memory in the accumulator fragment layout);
//       MMA2 (tcgen05, M=128 N=128 K=16):  dS^T = U^T Kb;
//       S^T <- S^T Diag(e^{Gamma_C}) + dS^T in fp32 registers, and its BF16 copy back
//            into tensor memory for the next block's MMA1.
//   The fp32 master state never leaves registers; only its BF16 rounding feeds
//   the products, so the decay term stays exact in fp32.  Each chain uses 128
//   TMEM columns: dS^T in all of them while the update reads it, the BF16 S^T
//   in the first 64 and [E^T | P^T] in the next 32 while those live.
//
// CTA layouts: in the transfer pass one CTA runs both chains of a (sequence,
// head, segment) from one prep (identity start without values: the transfer
// matrix; zero start: the zero-initial state), so the inputs are read once; in
// the output pass a CTA runs one (sequence, head, segment) or, when there are
// more of them than SMs, two, each with half the prep warps.
//
// Every wait is bounded: a stalled barrier sets an abort flag, records
// KDA_ERR_TIMEOUT in dev_status, and all roles leave their loops (the chains
// decide together through barrier reductions) and return.
#include <string.h>

#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int C = 16;    // tokens per block
constexpr int D = 128;   // dk = dv
constexpr int N_PREP = 4;
constexpr int NCH = 2;   // chains per CTA
constexpr int NTHREADS = 128 * (1 + NCH);
constexpr int NSLOT = 6;
constexpr long long kWaitLimit = 4000000000ll;  // ~2 s of SM clocks
// 384 threads launch with 168 registers each; the prep warpgroup gives 48 of them
// back and each chain warpgroup takes 24 more (128 x 120 + 256 x 192 = 384 x 168).
constexpr int PREP_REGS = 120, CHAIN_REGS = 192;

enum Layout { LAYOUT_SHARED = 0, LAYOUT_SINGLE = 1, LAYOUT_PAIR = 2 };

// ---- shared memory (offsets from a 1024-byte aligned base)
// input stage of prep warp p: TMA boxes (dense rows)
constexpr int IN_Q = 0, IN_K = 4096, IN_V = 8192, IN_G = 12288, IN_SIZE = 20480;
constexpr int IN_OFF = 0;
// record slot: the chain's operands for one block
constexpr int R_KQ = 0;      // [Kh (rows 0-15); Qh (rows 16-31)] x 128 channels, K-major, 128-byte
                             // swizzle: two 4 KB atom columns (channels 0-63, 64-127)
constexpr int R_KB = 8192;   // Kb as [i][r], K-major without swizzle: core matrices of 8 i x 8 r,
                             // r halves 2048 bytes apart, 8-channel groups 128 bytes apart
constexpr int R_V = 12288;   // V [r][j] in 256-byte rows, 16-byte chunk c of row r at c ^ (r & 7);
                             // before V is copied in, Kt [r][i] in the same layout
constexpr int TL = 24;       // T and Mq rows: 16 BF16 + pad (48 bytes)
constexpr int R_T = 16384;   // T [r][r']
constexpr int R_MQ = R_T + C * TL * 2;   // Mq [r][r']
constexpr int R_DEC = R_MQ + C * TL * 2; // e^{Gamma_C} fp32 [128]
constexpr int R_SIZE = R_DEC + D * 4;    // 18432
constexpr int REC_OFF = IN_OFF + N_PREP * IN_SIZE;
constexpr int LS = 20;                   // Diag(beta) L, fp32 [16][LS] per prep warp
constexpr int L_SIZE = C * LS * 4;
constexpr int L_OFF = REC_OFF + NSLOT * R_SIZE;
constexpr int U_SIZE = 4096;             // U^T as MMA2's A operand, layout as R_KB (rows j)
constexpr int U_OFF = L_OFF + N_PREP * L_SIZE;
constexpr int OST_SIZE = 1024;           // per chain warp: O^T staging [2 m-tiles][16 r][16 j]
constexpr int OST_OFF = U_OFF + NCH * U_SIZE;
constexpr int BAR_OFF = OST_OFF + NCH * 4 * OST_SIZE;
enum {
    B_IN = 0,
    B_FULL = B_IN + N_PREP,
    B_EMPTY = B_FULL + NSLOT,
    B_EO = B_EMPTY + NSLOT,
    B_DS = B_EO + NCH,
    B_FIN = B_DS + NCH,
    NBARS = B_FIN + NCH
};
constexpr int MISC_OFF = BAR_OFF + NBARS * 8;  // [0] abort flag, [4] TMEM base
constexpr int SMEM_USED = MISC_OFF + 16;
constexpr int SMEM_BYTES = SMEM_USED + 1024;   // slack for the 1024-byte alignment
constexpr uint32_t TMEM_COLS = 128 * NCH;

static_assert(R_SIZE == 18432 && REC_OFF % 1024 == 0 && R_SIZE % 1024 == 0, "record alignment");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(128 * PREP_REGS + 128 * NCH * CHAIN_REGS <= NTHREADS * 168, "register split");

struct Unit {
    int n, h, s;
    int t_begin, t_end, nchunks;
    int seq0, ckpt_base;
    bool valid;
};

struct Ctx {
    const PrefillArgs *p;
    uint64_t tm_q, tm_k, tm_v, tm_g;  // generic addresses of the tensor maps
    uint8_t *smem;
    uint32_t sbase;
    volatile int *abort;
    int layout;
    bool transfer, want_q;
    __device__ uint32_t bar(int i) const { return sbase + BAR_OFF + 8 * i; }
};

// Every lane polls (each with acquire semantics), so the warp does not split
// around the wait.
__device__ __forceinline__ bool warp_wait(const Ctx &x, int b, uint32_t parity) {
    const bool ok = mbar_wait(x.bar(b), parity, x.abort, kWaitLimit);
    return __all_sync(0xffffffffu, ok);
}

// Byte offset in R_KQ of channels (c, c + 1) of row n (c even).
__device__ __forceinline__ uint32_t kq_off(int n, int c) {
    return (uint32_t)((c >> 6) * 4096 + n * 128 + ((((c & 63) >> 3) ^ (n & 7)) << 4) + (c & 7) * 2);
}
// Byte offset in R_V of 16-byte chunk cc (0..15) of row r.
__device__ __forceinline__ uint32_t v_off(int r, int cc) {
    return (uint32_t)(r * 256 + ((cc ^ (r & 7)) << 4));
}

// ------------------------------------------------------------------ prep
// Elementwise factors of one block; lane takes channels c0 = 64 m + 2 lane and
// c0 + 1 (m = 0, 1), so neighbouring channels share packed fp32x2 arithmetic and
// 4-byte BF16 pairs.  e^{Gamma_r} comes from the running product of alpha = e^g,
// e^{-Gamma_r} from its reciprocal and e^{Gamma_C - Gamma_r} = e^{Gamma_C}
// e^{-Gamma_r}.  With MASK (the last, partial block of a sequence) rows past its
// end get no decay, no key and no query.  With GATE the box at IN_G holds x_g in
// BF16 (g = -5 sigmoid(x_g) is formed here) and k, q are scaled by their rows'
// inverse L2 norms rk, rq.
template <bool WANT_Q, bool MASK, bool GATE>
__device__ __forceinline__ void elementwise(const uint8_t *in, uint8_t *rec, int nt, int lane,
                                            const float *rk, const float *rq) {
#pragma unroll 1
    for (int m = 0; m < 2; ++m) {
        const int c0 = 64 * m + 2 * lane;
        float2 fwd[C];
        float2 run = make_float2(1.f, 1.f);
#pragma unroll
        for (int r = 0; r < C; ++r) {
            float2 gg;
            if (GATE) {
                const float2 xg = __bfloat1622float2(
                    *(const __nv_bfloat162 *)(in + IN_G + r * 256 + c0 * 2));
                // g = -5 sigmoid(x_g); the fast divide (reciprocal and multiply,
                // ~2 ulp) is far below the BF16 rounding of the operands g feeds
                gg = make_float2(__fdividef(-5.f, 1.f + __expf(-xg.x)),
                                 __fdividef(-5.f, 1.f + __expf(-xg.y)));
            } else {
                gg = *(const float2 *)(in + IN_G + r * 512 + c0 * 4);
            }
            if (MASK && r >= nt) gg = make_float2(0.f, 0.f);
            const float2 al = make_float2(__expf(gg.x), __expf(gg.y));  // alpha = e^g
            mul2_inplace(run.x, run.y, al);
            fwd[r] = run;
        }
        const float2 eGC = fwd[C - 1];
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // positions 8 h .. 8 h + 7
            float2 kb[8];
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
                const int r = 8 * h + rr;
                float2 k2 =
                    __bfloat1622float2(*(const __nv_bfloat162 *)(in + IN_K + r * 256 + c0 * 2));
                if (GATE) {
                    const float s = rk[r];
                    k2 = make_float2(k2.x * s, k2.y * s);
                }
                if (MASK && r >= nt) k2 = make_float2(0.f, 0.f);
                const float2 inv =
                    make_float2(__fdividef(1.f, fwd[r].x), __fdividef(1.f, fwd[r].y));
                float2 rev = inv;
                mul2_inplace(rev.x, rev.y, eGC);
                float2 kh = k2, kt = k2;
                mul2_inplace(kh.x, kh.y, fwd[r]);
                mul2_inplace(kt.x, kt.y, inv);
                kb[rr] = k2;
                mul2_inplace(kb[rr].x, kb[rr].y, rev);
                *(uint32_t *)(rec + R_KQ + kq_off(r, c0)) = pack_bf16x2(kh.x, kh.y);
                *(uint32_t *)(rec + R_V + v_off(r, c0 >> 3) + (c0 & 7) * 2) =
                    pack_bf16x2(kt.x, kt.y);
                if (WANT_Q) {
                    float2 q2 = __bfloat1622float2(
                        *(const __nv_bfloat162 *)(in + IN_Q + r * 256 + c0 * 2));
                    if (GATE) {
                        const float s = rq[r];
                        q2 = make_float2(q2.x * s, q2.y * s);
                    }
                    if (MASK && r >= nt) q2 = make_float2(0.f, 0.f);
                    mul2_inplace(q2.x, q2.y, fwd[r]);
                    *(uint32_t *)(rec + R_KQ + kq_off(16 + r, c0)) = pack_bf16x2(q2.x, q2.y);
                }
            }
            // this half of the Kb^T rows of channels c0 and c0 + 1
            *(uint4 *)(rec + R_KB + 2048 * h + c0 * 16) =
                make_uint4(pack_bf16x2(kb[0].x, kb[1].x), pack_bf16x2(kb[2].x, kb[3].x),
                           pack_bf16x2(kb[4].x, kb[5].x), pack_bf16x2(kb[6].x, kb[7].x));
            *(uint4 *)(rec + R_KB + 2048 * h + (c0 + 1) * 16) =
                make_uint4(pack_bf16x2(kb[0].y, kb[1].y), pack_bf16x2(kb[2].y, kb[3].y),
                           pack_bf16x2(kb[4].y, kb[5].y), pack_bf16x2(kb[6].y, kb[7].y));
        }
        *(float2 *)(rec + R_DEC + c0 * 4) = eGC;
    }
}

// Prep warp p: prepares blocks first, first + stride, ... of its ring's unit.
template <bool WANT_Q, bool GATE>
__device__ __forceinline__ void prep_role(const Ctx &x, const Unit u) {
    const PrefillArgs &p = *x.p;
    const int pw = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31, g8 = lane >> 2, t4 = lane & 3;
    const bool pair = x.layout == LAYOUT_PAIR;
    const int ring = pair ? pw >> 1 : 0;
    const int stride = pair ? 2 : N_PREP;
    const int first = pair ? pw & 1 : pw;
    const int nslot = pair ? NSLOT / 2 : NSLOT;
    const int slot0 = pair ? ring * (NSLOT / 2) : 0;
    if (!u.valid) return;
    float *Lf = (float *)(x.smem + L_OFF + pw * L_SIZE);
    const uint32_t full = x.bar(B_IN + pw);
    const uint32_t in_s = x.sbase + IN_OFF + pw * IN_SIZE;
    const uint8_t *in = x.smem + IN_OFF + pw * IN_SIZE;

    // One 2D tensor-map TMA copy per array (whole 16-row boxes; rows past the
    // block's end hold the next sequence's tokens, masked below, or past the
    // array zero fill).
    auto issue = [&](int c) {
        if (lane == 0) {
            const uint32_t bytes = (WANT_Q ? 4096u : 0u) + 8192u + (GATE ? 4096u : 8192u);
            mbar_arrive_expect_tx(full, bytes);
            const int xc = u.h * D, t0 = u.t_begin + C * c;
            if (WANT_Q) tma_load_2d(in_s + IN_Q, x.tm_q, xc, t0, full);
            tma_load_2d(in_s + IN_K, x.tm_k, xc, t0, full);
            tma_load_2d(in_s + IN_V, x.tm_v, xc, t0, full);
            tma_load_2d(in_s + IN_G, x.tm_g, xc, t0, full);
        }
    };
    // beta of rows g8 and g8 + 8 (for L) and of column lane (for T), zero past the
    // block's end; loaded one block ahead
    auto load_beta = [&](int c, float &lo, float &hi, float &col) {
        const int t0 = u.t_begin + C * c, nt = min(C, u.t_end - t0);
        const float *bp = p.beta + (size_t)t0 * p.H + u.h;
        auto b = [&](int r) {  // beta, or sigmoid(x_beta) with the fused prologue
            const float v = bp[(size_t)r * p.H];
            return GATE ? __fdividef(1.f, 1.f + __expf(-v)) : v;
        };
        lo = g8 < nt ? b(g8) : 0.f;
        hi = g8 + 8 < nt ? b(g8 + 8) : 0.f;
        col = (lane & 15) < nt ? b(lane & 15) : 0.f;
    };
    int issued = 0, uses = 0;
    float b_lo = 0.f, b_hi = 0.f, b_col = 0.f;
    if (first < u.nchunks) {
        issue(first);
        issued = 1;
        load_beta(first, b_lo, b_hi, b_col);
    }
    for (int c = first; c < u.nchunks; c += stride, ++uses) {
        const int slot = slot0 + c % nslot;
        const float beta_lo = b_lo, beta_hi = b_hi, beta_col = b_col;
        if (c + stride < u.nchunks) load_beta(c + stride, b_lo, b_hi, b_col);
        if (!warp_wait(x, B_EMPTY + slot, ((c / nslot) & 1) ^ 1)) break;
        if (!warp_wait(x, B_IN + pw, uses & 1)) break;
        uint8_t *rec = x.smem + REC_OFF + slot * R_SIZE;
        const uint32_t rec_s = x.sbase + REC_OFF + slot * R_SIZE;
        const int nt = min(C, u.t_end - (u.t_begin + C * c));

        // ---- fused prologue: inverse L2 norms of this block's k and q rows (a zero
        // row keeps scale 0), over the 128 channels = 4 per lane, then the warp;
        // kept in the warp's L scratch, which L overwrites only after the
        // elementwise pass
        float *rk = Lf, *rq = Lf + C;
        if (GATE) {
#pragma unroll
            for (int r = 0; r < C; ++r) {
                float sk = 0.f, sq = 0.f;
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    const float2 kv = __bfloat1622float2(
                        *(const __nv_bfloat162 *)(in + IN_K + r * 256 + (64 * m + 2 * lane) * 2));
                    sk += kv.x * kv.x + kv.y * kv.y;
                    if (WANT_Q) {
                        const float2 qv = __bfloat1622float2(*(
                            const __nv_bfloat162 *)(in + IN_Q + r * 256 + (64 * m + 2 * lane) * 2));
                        sq += qv.x * qv.x + qv.y * qv.y;
                    }
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    sk += __shfl_xor_sync(0xffffffffu, sk, off);
                    if (WANT_Q) sq += __shfl_xor_sync(0xffffffffu, sq, off);
                }
                if (lane == 0) {
                    rk[r] = sk > 0.f ? rsqrtf(sk) : 0.f;
                    rq[r] = sq > 0.f ? rsqrtf(sq) : 0.f;
                }
            }
            __syncwarp();
        }

        if (nt == C) elementwise<WANT_Q, false, GATE>(in, rec, nt, lane, rk, rq);
        else elementwise<WANT_Q, true, GATE>(in, rec, nt, lane, rk, rq);
        __syncwarp();

        // ---- L = Diag(beta) strict_lower(Kh Kt^T) and Mq = lower(Qh Kt^T), 16 x 16 x 128
        {
            float accL[2][4] = {}, accM[2][4] = {};
            const int arow = (lane & 7) + 8 * ((lane >> 3) & 1);
            const int brow = (lane & 7) + 8 * (lane >> 4);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const int gc = 2 * kk + (lane >> 4);
                const uint32_t aoff = (gc >> 3) * 4096 + ((gc & 7) ^ (arow & 7)) * 16;
                uint32_t af[4], bf[4];
                ldsm_x4(rec_s + R_KQ + aoff + arow * 128, af);
                ldsm_x4(rec_s + R_V + v_off(brow, 2 * kk + ((lane >> 3) & 1)), bf);
                mma_bf16_16816(accL[0], af, bf[0], bf[1]);
                mma_bf16_16816(accL[1], af, bf[2], bf[3]);
                if (WANT_Q) {
                    uint32_t aq[4];
                    ldsm_x4(rec_s + R_KQ + aoff + (arow + 16) * 128, aq);
                    mma_bf16_16816(accM[0], aq, bf[0], bf[1]);
                    mma_bf16_16816(accM[1], aq, bf[2], bf[3]);
                }
            }
#pragma unroll
            for (int nb = 0; nb < 2; ++nb)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int r = g8 + 8 * hh;
                    const int i0 = nb * 8 + 2 * t4;
                    const float br = hh ? beta_hi : beta_lo;
                    *(float2 *)(Lf + r * LS + i0) =
                        make_float2(i0 < r ? br * accL[nb][2 * hh] : 0.f,
                                    i0 + 1 < r ? br * accL[nb][2 * hh + 1] : 0.f);
                    if (WANT_Q)
                        *(uint32_t *)(rec + R_MQ + (r * TL + i0) * 2) =
                            pack_bf16x2(i0 <= r ? accM[nb][2 * hh] : 0.f,
                                        i0 + 1 <= r ? accM[nb][2 * hh + 1] : 0.f);
                }
        }
        __syncwarp();
        // V into the record over Kt.  Rows past the block's end become zero: they are
        // weighted by zero in the chain's products, and the next sequence's values
        // (or anything non-finite in them) must not leak in.
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int idx = lane + 32 * i, r = idx >> 4, cc = idx & 15;
            uint4 v = *(const uint4 *)(in + IN_V + r * 256 + cc * 16);
            if (r >= nt) v = make_uint4(0u, 0u, 0u, 0u);
            *(uint4 *)(rec + R_V + v_off(r, cc)) = v;
        }
        __syncwarp();
        // Input stage read: load this warp's next block into it (the generic reads
        // above are ordered before the copy's writes by the proxy fence).
        if (c + stride < u.nchunks) {
            if (lane == 0) fence_async_smem();
            issue(c + stride);
            ++issued;
        }

        // ---- T = (I + Diag(beta) L)^{-1} Diag(beta): forward substitution, lane = column
        if (lane < C) {
            const int j = lane;
            float xv[C];
#pragma unroll
            for (int r = 0; r < C; ++r) xv[r] = (r == j) ? 1.f : 0.f;
#pragma unroll
            for (int r = 1; r < C; ++r) {
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int c4 = 0; 4 * c4 < r; ++c4) {
                    const float4 lv = *(const float4 *)(Lf + r * LS + 4 * c4);
                    const float l4[4] = {lv.x, lv.y, lv.z, lv.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int m = 4 * c4 + q;
                        if (m < r) {
                            if (m & 1) s1 += l4[q] * xv[m];
                            else s0 += l4[q] * xv[m];
                        }
                    }
                }
                xv[r] = r > j ? -(s0 + s1) : xv[r];
            }
            __nv_bfloat16 *Tb = (__nv_bfloat16 *)(rec + R_T);
#pragma unroll
            for (int r = 0; r < C; ++r) Tb[r * TL + j] = __float2bfloat16_rn(xv[r] * beta_col);
        }
        // the tensor cores read [Kh; Qh] and Kb^T through the async proxy
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(x.bar(B_FULL + slot));
    }
    // On an abort, let this warp's copy in flight land before the CTA can exit.
    if (*x.abort && lane == 0 && issued > uses) {
        volatile int never = 0;
        mbar_wait(full, uses & 1, &never, kWaitLimit);
    }
}

// ------------------------------------------------------------------ chain
// Chain ch (warpgroup 1 + ch): thread j owns S^T row j (TMEM lane j).
template <bool WANT_Q>
__device__ __forceinline__ void chain_role(const Ctx &x, const Unit u, int ch, uint32_t tmem) {
    const PrefillArgs &p = *x.p;
    const int tid = threadIdx.x - 128 * (1 + ch);
    const int cw = tid >> 5, lane = tid & 31, g8 = lane >> 2, t4 = lane & 3;
    const int j = tid;
    const bool pair = x.layout == LAYOUT_PAIR;
    const int nslot = pair ? NSLOT / 2 : NSLOT;
    const int slot0 = pair ? ch * (NSLOT / 2) : 0;
    const bool partA = x.transfer && ch == 0;  // identity start, no values
    const bool want_v = !partA;
    const int bar_id = 1 + ch;
    const size_t unit_hn = (size_t)u.n * p.H + u.h;
    // this chain's 128 columns; lane field = the warp's quarter
    const uint32_t tc = tmem + 128 * ch;
    const uint32_t tl = tc + ((uint32_t)(32 * cw) << 16);
    const uint32_t eo_col = 64;  // [E^T | P^T] at columns 64 .. 95 of the chain
    const uint32_t mbar_eo = x.bar(B_EO + ch), mbar_ds = x.bar(B_DS + ch);

    // S[i] = S^T[j][i] = S_start[i][j]
    float S[D];
    {
        const float *src = nullptr;
        if (!x.transfer)
            src = p.seg_init ? p.seg_init + (unit_hn * p.Sg + u.s) * (size_t)D * D
                             : (p.S0 ? p.S0 + unit_hn * (size_t)D * D : nullptr);
#pragma unroll
        for (int i = 0; i < D; ++i)
            S[i] = partA ? (i == j ? 1.f : 0.f) : (src ? src[(size_t)i * D + j] : 0.f);
    }
    // the BF16 copy of S^T row j -> columns [0, 64) (two channels per column)
    auto store_sbf = [&](int piece) {  // channels 16 piece .. 16 piece + 15
        uint32_t w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = pack_bf16x2(S[16 * piece + 2 * e], S[16 * piece + 2 * e + 1]);
        tmem_st8(tl + 8 * piece, w);
    };
#pragma unroll
    for (int pc = 0; pc < 8; ++pc) store_sbf(pc);
    tmem_wait_st();
    tc_fence_before();

    __nv_bfloat16 *out = (__nv_bfloat16 *)(partA ? p.aux_out : p.out);
    uint8_t *ust = x.smem + U_OFF + ch * U_SIZE;
    const uint32_t ust_s = x.sbase + U_OFF + ch * U_SIZE;
    const uint32_t ost_s = x.sbase + OST_OFF + (ch * 4 + cw) * OST_SIZE;
    const uint8_t *ost = x.smem + OST_OFF + (ch * 4 + cw) * OST_SIZE;
    const uint32_t idesc1 = umma_idesc_bf16(128, WANT_Q ? 32 : 16);
    const uint32_t idesc2 = umma_idesc_bf16(128, 128);
    bool ok = true;
    for (int c = 0; c < u.nchunks; ++c) {
        const int slot = slot0 + c % nslot;
        const uint32_t rec_s = x.sbase + REC_OFF + slot * R_SIZE;
        const float *dec = (const float *)(x.smem + REC_OFF + slot * R_SIZE + R_DEC);
        ok = warp_wait(x, B_FULL + slot, (c / nslot) & 1);
        // all of S^T in BF16 is in tensor memory and the record is full
        if (named_bar_or(bar_id, 128, !ok)) break;
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                umma_bf16_ts(tc + eo_col, tc + 8 * kk,
                             umma_desc_sw128(rec_s + R_KQ + (kk >> 2) * 4096 + (kk & 3) * 32, 1024),
                             idesc1, kk > 0);
            umma_commit(mbar_eo);
        }
        ok = warp_wait(x, B_EO + ch, c & 1);
        tc_fence_after();
        if (ok) {
            uint32_t tb[4], mq[4];
            ldsm_x4(rec_s + R_T + (8 * (lane >> 4) + (lane & 7)) * (TL * 2) + 16 * ((lane >> 3) & 1),
                    tb);
            if (WANT_Q)
                ldsm_x4(rec_s + R_MQ + (8 * (lane >> 4) + (lane & 7)) * (TL * 2) +
                            16 * ((lane >> 3) & 1),
                        mq);
#pragma unroll 1
            for (int m = 0; m < 2; ++m) {  // 16 value columns at a time: j in jb .. jb + 15
                const int jb = 32 * cw + 16 * m;
                float e[16];
                tmem_ld_16x256b_x4(tc + ((uint32_t)jb << 16) + eo_col, e);
                // W = V^T - E^T (rows j, columns r), from V^T as an A fragment
                float w[2][4];
#pragma unroll
                for (int q = 0; q < 8; ++q) w[q >> 2][q & 3] = -e[q];
                if (want_v) {
                    uint32_t va[4];
                    const int vr = 8 * (lane >> 4) + (lane & 7);
                    ldsm_x4_t(rec_s + R_V + v_off(vr, (jb >> 3) + ((lane >> 3) & 1)), va);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float2 v2 =
                            __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&va[q]));
                        w[q >> 1][2 * (q & 1)] += v2.x;
                        w[q >> 1][2 * (q & 1) + 1] += v2.y;
                    }
                }
                const uint32_t wa[4] = {pack_bf16x2(w[0][0], w[0][1]), pack_bf16x2(w[0][2], w[0][3]),
                                        pack_bf16x2(w[1][0], w[1][1]), pack_bf16x2(w[1][2], w[1][3])};
                float U[2][4] = {};
                mma_bf16_16816(U[0], wa, tb[0], tb[1]);
                mma_bf16_16816(U[1], wa, tb[2], tb[3]);
                const uint32_t ua[4] = {pack_bf16x2(U[0][0], U[0][1]), pack_bf16x2(U[0][2], U[0][3]),
                                        pack_bf16x2(U[1][0], U[1][1]), pack_bf16x2(U[1][2], U[1][3])};
                // U^T into MMA2's A operand (rows j, K-major without swizzle)
                const uint32_t uo = (jb >> 3) * 128 + g8 * 16 + 4 * t4;
                *(uint32_t *)(ust + uo) = ua[0];
                *(uint32_t *)(ust + uo + 128) = ua[1];
                *(uint32_t *)(ust + uo + 2048) = ua[2];
                *(uint32_t *)(ust + uo + 2048 + 128) = ua[3];
                if (WANT_Q) {
                    float O[2][4];
#pragma unroll
                    for (int q = 0; q < 8; ++q) O[q >> 2][q & 3] = e[8 + q];
                    mma_bf16_16816(O[0], ua, mq[0], mq[1]);
                    mma_bf16_16816(O[1], ua, mq[2], mq[3]);
                    // O^T (j x r) -> staging [r][j]
                    stsm_x4_t(ost_s + m * 512 + ((lane & 7) + 8 * (lane >> 4)) * 32 +
                                  16 * ((lane >> 3) & 1),
                              pack_bf16x2(O[0][0], O[0][1]), pack_bf16x2(O[0][2], O[0][3]),
                              pack_bf16x2(O[1][0], O[1][1]), pack_bf16x2(O[1][2], O[1][3]));
                }
            }
            if (WANT_Q) {
                __syncwarp();
                const int t0 = u.t_begin + C * c;
                const int r = lane >> 1, half = lane & 1;
                if (r < u.t_end - t0) {
#pragma unroll
                    for (int m = 0; m < 2; ++m)
                        *(uint4 *)(out + ((size_t)(t0 + r) * p.H + u.h) * D + 32 * cw + 16 * m +
                                   8 * half) = *(const uint4 *)(ost + m * 512 + r * 32 + half * 16);
                }
            }
            fence_async_smem();  // U^T is read by the tensor core
        }
        tc_fence_before();
        if (named_bar_or(bar_id, 128, !ok)) break;
        if (tid == 0) {
            tc_fence_after();
            umma_bf16(tc, umma_desc(ust_s, 2048, 128), umma_desc(rec_s + R_KB, 2048, 128), idesc2, 0);
            umma_commit(mbar_ds);
        }
        ok = warp_wait(x, B_DS + ch, c & 1);
        tc_fence_after();
        if (ok) {
            // S^T <- S^T Diag(e^{Gamma_C}) + dS^T in fp32, 16 channels at a time; the
            // BF16 copy of piece pc goes to columns [8 pc, 8 pc + 8), which lie in dS^T
            // pieces already read
#pragma unroll
            for (int pc = 0; pc < 8; ++pc) {
                float d[16];
                tmem_ld16(tl + 16 * pc, d);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 dv = *(const float4 *)(dec + 16 * pc + 4 * q);
                    const int i0 = 16 * pc + 4 * q;
                    fma2_scale_add(S[i0], S[i0 + 1], dv.x, dv.y, d[4 * q], d[4 * q + 1]);
                    fma2_scale_add(S[i0 + 2], S[i0 + 3], dv.z, dv.w, d[4 * q + 2], d[4 * q + 3]);
                }
                store_sbf(pc);
            }
        }
        // the record (last read: e^{Gamma_C}) goes back to the prep warps
        __syncwarp();
        if (lane == 0) mbar_arrive(x.bar(B_EMPTY + slot));
        tmem_wait_st();
        tc_fence_before();
        if (ok && p.ckpt_interval > 0) {  // state checkpoint after this block
            const int done = min(u.t_begin + C * (c + 1), u.t_end) - u.seq0;
            float *dst = partA ? p.ckpt_a : p.ckpt;
            if (done % p.ckpt_interval == 0 && dst) {
                dst += ((size_t)(u.ckpt_base + done / p.ckpt_interval - 1) * p.H + u.h) * D * D + j;
#pragma unroll
                for (int i = 0; i < D; ++i) dst[(size_t)i * D] = S[i];
            }
        }
    }
    if (*x.abort) {
        // let the products this chain issued finish before the CTA frees its TMEM
        if (tid == 0) {
            umma_commit(x.bar(B_FIN + ch));
            volatile int never = 0;
            mbar_wait(x.bar(B_FIN + ch), 0, &never, kWaitLimit);
        }
        return;
    }

    // final writes: thread j holds column j of the state, so every store of row i
    // is 128 consecutive floats across the warpgroup
    if (!x.transfer) {
        if (u.s == p.Sg - 1 && p.S_final) {
            float *dst = p.S_final + unit_hn * (size_t)D * D + j;
#pragma unroll
            for (int i = 0; i < D; ++i) dst[(size_t)i * D] = S[i];
        }
    } else if (partA && p.transfer_img) {
        // A[i][j] as hi/lo BF16 images, transposed ([j][i], i contiguous): row j is
        // this thread's registers in order
        __nv_bfloat16 *hi = p.transfer_img + (unit_hn * p.Sg + u.s) * (size_t)2 * D * D + (size_t)j * D;
        __nv_bfloat16 *lo = hi + (size_t)D * D;
#pragma unroll
        for (int i8 = 0; i8 < D / 8; ++i8) {
            uint32_t wh[4], wl[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float v0 = S[8 * i8 + 2 * e], v1 = S[8 * i8 + 2 * e + 1];
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(v0, v1);
                const float2 hf = __bfloat1622float2(h2);
                wh[e] = *(const uint32_t *)&h2;
                wl[e] = pack_bf16x2(v0 - hf.x, v1 - hf.y);
            }
            *(uint4 *)(hi + 8 * i8) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
            *(uint4 *)(lo + 8 * i8) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
        }
    } else {
        float *base = partA ? p.transfer : p.zero_state;
        if (base) {
            float *dst = base + (unit_hn * p.Sg + u.s) * (size_t)D * D + j;
#pragma unroll
            for (int i = 0; i < D; ++i) dst[(size_t)i * D] = S[i];
        }
    }
}

__device__ __forceinline__ bool load_unit(const PrefillArgs &p, int idx, Unit &u) {
    u.valid = false;
    const int units = p.N * p.H * p.seg_count;
    if (idx >= units) return true;
    u.n = idx / (p.H * p.seg_count);
    u.h = (idx / p.seg_count) % p.H;
    u.s = p.seg_begin + idx % p.seg_count;
    if (!segment_range(p.cu, u.n, p.N, p.T_tot, u.s, p.Sg, p.dev_status, u.t_begin, u.t_end))
        return false;
    u.nchunks = (u.t_end - u.t_begin + C - 1) / C;
    u.seq0 = p.cu[u.n];
    u.ckpt_base = p.ckpt_interval > 0 ? ckpt_base(p.cu, u.n, p.ckpt_interval) : 0;
    u.valid = true;
    return true;
}

template <bool GATE>
__global__ void __launch_bounds__(NTHREADS, 1)
    prefill_tm_kernel(const __grid_constant__ PrefillArgs p, int layout,
                      const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_g) {
    extern __shared__ uint8_t smem_raw[];
    griddep_wait();  // inputs may come from the previous kernel in the stream
    griddep_launch_dependents();
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_addr(smem);
    const int first_unit = layout == LAYOUT_PAIR ? 2 * blockIdx.x : blockIdx.x;
    {
        Unit t;
        bool good = load_unit(p, first_unit, t);
        if (layout == LAYOUT_PAIR) good = load_unit(p, first_unit + 1, t) && good;
        if (!good) return;  // malformed cu_seqlens (recorded in dev_status)
    }
    const int nconsumers = layout == LAYOUT_SHARED ? 2 : 1;
    const int warp = threadIdx.x >> 5;
    volatile int *abort = (volatile int *)(smem + MISC_OFF);
    if (threadIdx.x == 0) {
        const uint32_t bar = sbase + BAR_OFF;
        for (int i = 0; i < N_PREP; ++i) mbar_init(bar + 8 * (B_IN + i), 1);
        for (int i = 0; i < NSLOT; ++i) {
            mbar_init(bar + 8 * (B_FULL + i), 1);
            mbar_init(bar + 8 * (B_EMPTY + i), 4 * nconsumers);
        }
        for (int i = 0; i < NCH; ++i) {
            mbar_init(bar + 8 * (B_EO + i), 1);
            mbar_init(bar + 8 * (B_DS + i), 1);
            mbar_init(bar + 8 * (B_FIN + i), 1);
        }
        *abort = 0;
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(sbase + MISC_OFF + 4, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // Each role builds its own context and decodes its own unit, so that little
    // stays live across the branch (the warpgroups run with different register
    // budgets).
    auto make_ctx = [&]() {
        Ctx x;
        x.p = &p;
        x.tm_q = reinterpret_cast<uint64_t>(&tm_q);
        x.tm_k = reinterpret_cast<uint64_t>(&tm_k);
        x.tm_v = reinterpret_cast<uint64_t>(&tm_v);
        x.tm_g = reinterpret_cast<uint64_t>(&tm_g);
        x.smem = smem;
        x.sbase = sbase;
        x.abort = abort;
        x.layout = layout;
        x.transfer = p.mode == MODE_TRANSFER;
        x.want_q = !x.transfer || p.emit_out;
        return x;
    };
    if (warp < 4) {
        regs_dealloc<PREP_REGS>();
        const Ctx x = make_ctx();
        // in the pair layout warps 2 and 3 prepare the second unit's blocks
        Unit u;
        load_unit(p, first_unit + ((layout == LAYOUT_PAIR && warp >= 2) ? 1 : 0), u);
        if (GATE) prep_role<true, true>(x, u);
        else if (x.want_q) prep_role<true, false>(x, u);
        else prep_role<false, false>(x, u);
    } else {
        regs_alloc<CHAIN_REGS>();
        const Ctx x = make_ctx();
        const int ch = (warp >> 2) - 1;
        Unit u;
        load_unit(p, first_unit + ((layout == LAYOUT_PAIR && ch == 1) ? 1 : 0), u);
        const bool active = u.valid && (layout != LAYOUT_SINGLE || ch == 0);
        if (active) {
            const uint32_t tmem = *(volatile uint32_t *)(smem + MISC_OFF + 4);
            if (x.want_q) chain_role<true>(x, u, ch, tmem);
            else chain_role<false>(x, u, ch, tmem);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abort) dev_fail(p.dev_status, KDA_ERR_TIMEOUT);
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(*(volatile uint32_t *)(smem + MISC_OFF + 4), TMEM_COLS);
    }
}

// [T_tot, H * 128] row-major view of a token-major array, 16 x 128 boxes.
bool encode_rows(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap *m, const void *ptr, int T,
                 int H, bool fp32) {
    const cuuint64_t dims[2] = {(cuuint64_t)H * D, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)H * D * (fp32 ? 4 : 2)};
    const cuuint32_t box[2] = {(cuuint32_t)D, (cuuint32_t)C};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
               const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool prefill_tc_supported(const PrefillArgs &a) {
    if (a.gate && !(a.q && (a.mode == MODE_OUTPUT || a.emit_out))) return false;
    return a.act == KDA_DTYPE_BF16 && a.dk == D && a.dv == D;
}

cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t st) {
    const long long units = (long long)a.N * a.H * a.seg_count;
    if (units == 0) return cudaSuccess;
    CUtensorMap tq, tk, tv, tg;
    memset(&tq, 0, sizeof(tq)); memset(&tk, 0, sizeof(tk));
    memset(&tv, 0, sizeof(tv)); memset(&tg, 0, sizeof(tg));
    if (a.T_tot > 0) {  // with no tokens no CTA loads anything (and the pointers may be null)
        PFN_cuTensorMapEncodeTiled_v12000 enc = sm100::tensor_map_encoder();
        if (!enc) return cudaErrorNotSupported;
        const void *qp = a.q ? a.q : a.k;  // the transfer pass may have no q
        if (!encode_rows(enc, &tq, qp, a.T_tot, a.H, false) ||
            !encode_rows(enc, &tk, a.k, a.T_tot, a.H, false) ||
            !encode_rows(enc, &tv, a.v, a.T_tot, a.H, false) ||
            !encode_rows(enc, &tg, a.g, a.T_tot, a.H, !a.gate))
            return cudaErrorInvalidValue;
    }
    int layout = LAYOUT_SHARED;
    long long grid = units;
    if (a.mode != MODE_TRANSFER) {
        int dev = 0, sms = 148;
        if (cudaGetDevice(&dev) == cudaSuccess)
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        // two (sequence, head, segment) chains per CTA once there are more than SMs
        layout = units > sms ? LAYOUT_PAIR : LAYOUT_SINGLE;
        grid = layout == LAYOUT_PAIR ? (units + 1) / 2 : units;
    }
    if (a.gate) {
        cudaError_t e = set_max_dynamic_smem((const void *)prefill_tm_kernel<true>, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        return launch_dependent(prefill_tm_kernel<true>, dim3((unsigned)grid), dim3(NTHREADS),
                                SMEM_BYTES, st, a, layout, tq, tk, tv, tg);
    }
    cudaError_t e = set_max_dynamic_smem((const void *)prefill_tm_kernel<false>, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return launch_dependent(prefill_tm_kernel<false>, dim3((unsigned)grid), dim3(NTHREADS),
                            SMEM_BYTES, st, a, layout, tq, tk, tv, tg);
}

}  // namespace kda
