// Tensor-core chunked KDA prefill for BF16 activations at dk = dv = 128 (sm_103a).
//
// What it computes: the chunked form of the KDA recurrence (decay, then erase,
// then write, then read: "Kimi K3 Architecture Explained", section 3), with the
// bounded log-decay g > -5 keeping every in-block factor exp(+-Gamma), |Gamma| <
// 80, inside BF16 range so that both the intra-block ("diagonal") and the
// state ("off-diagonal") products run on tensor cores with BF16 operands and
// fp32 accumulation (Kimi K3 technical-report digest, section 2.1 (1)).  Per
// 16-token block, from state S (128 x 128, fp32):
//   prep (state-free):  Gamma = cumsum g;  Kh = K e^{Gamma};  Kt = K e^{-Gamma};
//                       Qh = Q e^{Gamma};  Kb = K e^{Gamma_C - Gamma};
//                       L = Diag(beta) strict_lower(Kh Kt^T);  Mq = lower(Qh Kt^T);
//                       T = (I + L)^{-1} Diag(beta)
//   chain (sequential): U = T (V - Kh S);  O = Qh S + Mq U;  S <- e^{Gamma_C} S + Kb^T U
// The digest's FlashKDA overlaps the intra-block work with the cross-block state
// propagation (section 2.4 (1)); here that is warp specialisation in one CTA per
// (sequence, head, segment):
//
//   warps 0-3   prep: warp p owns input stage p and prepares blocks p, p+4, p+8,
//               ... on its own (no barrier between prep warps), so four blocks are
//               in preparation at once.  It loads its own blocks (one 2D
//               tensor-map TMA copy per array: q, k, v as 16 x 128 BF16 boxes, g
//               as a 16 x 128 fp32 box; beta by loads one block ahead), issuing
//               the next block's copy into its stage as soon as it has read the
//               current one, and writes each block's chain operands, V included,
//               into one of five record slots.
//   warps 4-7   chain: warp w owns the state columns j in [32w, 32w+32): rows j of
//               S^T, all 128 key channels, held as fp32 mma.sync accumulators in
//               two 16-row m-tiles that share every operand fragment.  Columns of
//               S never mix, so each warp runs the recurrence of its columns
//               entirely in its own registers; per block it reads only the record
//               and signals when it is done with it.
//
// In the throughput regime the transfer pass runs both of a segment's chains in
// one CTA (NCH = 2): a second group of four chain warps (warps 8-11) consumes the
// same records, so each block is loaded and prepared once for the identity-start
// and the zero-start chain.  The warpgroups then run with different register
// budgets (setmaxnreg): the prep warps give registers to the chain warps.  There
// the one-call split may also have a lead segment (PrefillArgs::lead): segment 0
// of every chain, whose start state S0 is known, runs in a lead CTA as an output
// pass (the zero-start chain from S0, the identity-start warps idle and writing a
// zero transfer matrix), and the lead CTAs come first in the grid.
//
// Two more instantiations serve the chunked backward: the forward chain writing
// its BF16 state after every 32 tokens (chunk states), and the adjoint chain,
// which takes the blocks from the last to the first with d_out in place of v.
//
// The chain is a strict sequence of small products (16 x 128 x 128 per block).
// Kept in registers, one step costs a handful of dependent mma.sync issues and
// no round trip through shared or tensor memory, no commit and no cross-warp
// barrier; the fp32 master state never leaves registers and only its BF16
// rounding feeds the products, so the decay term e^{Gamma_C} S stays exact in
// fp32.  In the transfer pass the same recurrence runs from the identity with zero
// values (transfer matrix) and from zeros (zero-initial state): in one CTA (NCH =
// 2) or, below the throughput regime, in two CTAs per unit.
//
// mma.sync m16n8k16 fragments (g8 = lane / 4, t4 = lane % 4):
//   A (16x16): a0 = A[g8][2t4..+1], a1 = A[g8+8][2t4..+1], a2 = A[g8][2t4+8..+9],
//              a3 = A[g8+8][2t4+8..+9];  B (16x8): b0 = B[2t4..+1][g8], b1 = B[2t4+8..+9][g8];
//   C (16x8):  c0,c1 = C[g8][2t4..+1], c2,c3 = C[g8+8][2t4..+1].
// A chain warp's S^T accumulator n (n = 0..15) of an m-tile covers key channels
// [8n, 8n+8); two adjacent accumulators are exactly the A fragment of one
// 16-channel k-step.
//
// Every wait is bounded: a stalled barrier sets an abort flag, records
// KDA_ERR_TIMEOUT in dev_status, and all roles leave their loops and return.
#include <string.h>

#include "kda_internal.cuh"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int C = 16;    // tokens per block
constexpr int D = 128;   // dk = dv
// Input stage i belongs to prep warp i (blocks i, i + 4, ...): a waiter must
// know that the barrier's previous phase has completed, or the parity test
// cannot tell that phase from the one it waits for.  A prep warp consumed its
// stage's previous phase itself; a stage shared between prep warps could still
// be one phase behind.  Record slots need no such ownership: with at least
// N_PREP of them, the release a prep warp waits for is always the barrier's
// next phase.
constexpr int N_PREP = 4;
constexpr int NS = N_PREP;  // input stages (TMA ring)
constexpr int NR = N_PREP + 1;  // record slots (prepared blocks waiting for the chain)
constexpr int W_PREP0 = 0, W_CHAIN0 = W_PREP0 + N_PREP, N_CHAIN = 4;
// threads of a CTA with nch chains (four chain warps each)
__host__ __device__ constexpr int cta_threads(int nch) { return (W_CHAIN0 + N_CHAIN * nch) * 32; }
// Register split of the two-chain CTA: 384 threads launch with 168 registers each;
// the prep warpgroup gives back what the two chain warpgroups take.  Measured on
// GB300 (16-token block of the two-chain transfer pass / of a lead chain):
// 136 / 184: 1.65 / 1.20 us; 120 / 192: 1.57 / 1.12 us (a few spilled prep
// registers); 104 / 200: 1.60 / 1.08 us.
constexpr int PREP_REGS = 120, CHAIN_REGS = 192;
static_assert(128 * PREP_REGS + 256 * CHAIN_REGS <= 384 * 168, "register split");
// In a lead CTA only the zero-start chain runs: the identity-start warpgroup keeps
// just what writing a zero transfer matrix takes, and the running chain gets the
// rest (a separate instantiation, compiled for that budget).
constexpr int LEAD_IDLE_REGS = 40, LEAD_CHAIN_REGS = 232;
static_assert(128 * (PREP_REGS + LEAD_IDLE_REGS + LEAD_CHAIN_REGS) <= 384 * 168,
              "lead register split");
constexpr long long kWaitLimit = 4000000000ll;  // ~2 s of SM clocks

// ---- shared memory: [NS input stages | NR records | N_PREP prep scratches | O staging]
// input stage (TMA boxes, dense rows); released by the prep warp once read
constexpr int IN_ROWB = 256;                    // one 128-element BF16 row
constexpr int IN_Q = 0;                         // BF16 [16][128]
constexpr int IN_K = IN_Q + C * IN_ROWB;
constexpr int IN_V = IN_K + C * IN_ROWB;
constexpr int IN_G = IN_V + C * IN_ROWB;        // fp32 [16][128]
constexpr int IN_SIZE = IN_G + C * 512;
// record: the chain's operands for one block; released by the chain warps
constexpr int RL = 56;                          // BF16 elements per channel row (112 B):
constexpr int RLB = RL * 2;                     //   [Kh^T (16) | Qh^T (16) | Kb^T (16) | pad]
constexpr int RC_KH = 0, RC_Q = 16, RC_K = 32;
constexpr int TL = 24;                          // T and Mq rows: 16 BF16 + pad (48 B)
constexpr int VROWB = 272;                      // V rows: 128 BF16 + pad
constexpr int R_T = D * RLB;                    // T  [r][r'] BF16
constexpr int R_MQ = R_T + C * TL * 2;          // Mq [r][r'] BF16
constexpr int R_DECAY = R_MQ + C * TL * 2;      // e^{Gamma_C} fp32 [128]
constexpr int R_V = R_DECAY + D * 4;            // V  [r][j] BF16 (rows past the block: 0)
constexpr int R_SIZE = R_V + C * VROWB;
// prep scratch (private to one prep warp)
constexpr int TROW = 48;                        // one channel's 16 positions, BF16, padded
constexpr int X_KT = 0;                         // Kt^T [128 ch][24]
constexpr int LS = 20;                          // row stride of L: 16-byte aligned rows
constexpr int X_L = X_KT + D * TROW;            // Diag(beta) L fp32 [16][LS]
constexpr int X_SIZE = (X_L + C * LS * 4 + 127) & ~127;
constexpr int IN_OFF = 0;
constexpr int REC_OFF = IN_OFF + NS * IN_SIZE;
constexpr int X_OFF = REC_OFF + NR * R_SIZE;
constexpr int OST_OFF = X_OFF + N_PREP * X_SIZE;  // per chain warp: O^T staging [16 r][16 j]
constexpr int OST_SIZE = 2 * C * 16 * 2;  // two m-tiles
constexpr int BAR_OFF = OST_OFF + 2 * N_CHAIN * OST_SIZE;
enum {
    B_IN_FULL = 0,
    B_REC_FULL = B_IN_FULL + NS,
    B_REC_EMPTY = B_REC_FULL + NR,
    NBARS = B_REC_EMPTY + NR
};
constexpr int MISC_OFF = BAR_OFF + NBARS * 8;   // [0] abort flag
constexpr int SMEM_USED = MISC_OFF + 16;
constexpr int SMEM_BYTES = SMEM_USED + 128;     // slack for aligning the base

static_assert(IN_SIZE % 128 == 0 && R_SIZE % 128 == 0 && X_SIZE % 128 == 0, "stage alignment");
// Final-write staging per chain warp, in the input stages once they are idle: the
// BF16 hi/lo images of its 32 columns ([32 j][FW_IROW bytes] each; 272-byte rows
// keep stmatrix rows on distinct banks) or its fp32 state columns ([128 i][FW_JROW]
// floats; 36-float rows make the transposing scalar stores conflict-free).
constexpr int FW_IROW = 272;
constexpr int FW_JROW = 36;
constexpr int FW_SIZE = 128 * FW_JROW * 4;
static_assert(2 * 32 * FW_IROW <= FW_SIZE && N_CHAIN * FW_SIZE <= NS * IN_SIZE,
              "final-write staging fits in the input stages");
static_assert(2 * N_CHAIN * FW_SIZE <= NS * IN_SIZE + NR * R_SIZE,
              "two chains' final-write staging fits in the input stages and records");
static_assert(RLB % 16 == 0 && (RLB / 16) % 2 == 1, "record rows: 16-byte aligned, odd stride");
static_assert(VROWB % 16 == 0 && (VROWB / 16) % 2 == 1, "V rows: 16-byte aligned, odd stride");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

struct Ctx {
    const PrefillArgs *p;
    uint64_t tm_q, tm_k, tm_v, tm_g;  // generic addresses of the tensor maps
    uint8_t *smem;
    uint32_t sbase;
    volatile int *abort;
    int n, h, s;
    int seq0, ckpt_base;  // the sequence's first token; its first checkpoint slot
    int cs_base;          // first chunk-state slot of the sequence (chunk_states)
    int t_begin, t_end, nchunks;
    bool transfer, partA, want_q, want_v;
    bool lead;  // a lead CTA: segment 0 run from S0 by the zero-start chain only
    __device__ uint32_t bar(int i) const { return sbase + BAR_OFF + 8 * i; }
};

// Index of the sequence with the r-th longest length (ties: lower index first),
// for N <= 32; every lane of the warp takes part.  CTAs are handed out in
// launch order, so giving the first CTAs the longest sequences' chains starts
// the critical path first (longest processing time first): with more chains
// than SMs a long sequence would otherwise wait for a wave of short ones.
__device__ __forceinline__ int longest_first(const PrefillArgs &p, int r) {
    const int lane = threadIdx.x & 31;
    const int len = lane < p.N ? p.cu[lane + 1] - p.cu[lane] : -1;
    int rank = 0;
    for (int m = 0; m < p.N; ++m) {
        const int lm = __shfl_sync(0xffffffffu, len, m);
        rank += (lm > len) || (lm == len && m < lane);
    }
    const unsigned hit = __ballot_sync(0xffffffffu, lane < p.N && rank == r);
    return hit ? __ffs(hit) - 1 : r;
}

// Every lane polls the barrier (each with acquire semantics), so the warp does
// not split around the wait: a lane-0 wait with the other lanes parked at a
// shuffle cost thousands of cycles of reconvergence per wait on sm_103a.
__device__ __forceinline__ bool warp_wait(const Ctx &x, int b, uint32_t parity) {
    const bool ok = mbar_wait(x.bar(b), parity, x.abort, kWaitLimit);
    return __all_sync(0xffffffffu, ok);
}

// ------------------------------------------------------------------ prep
// Elementwise factors of one block for the key channels lane + 32 m (m = 0..3):
// Kt^T rows into the prep scratch, Kh^T, Qh^T and Kb^T rows and e^{Gamma_C}
// into the record.  Every row of the boxes is in shared memory, so the loads are
// unconditional; with MASK (the sequence's last, partial block) rows past its
// end get no decay, no key and no query.  Full blocks take the unmasked form,
// whose dependency chains are about half as long.
// With GATE the box at IN_G holds x_g in BF16, g = -5 sigmoid(x_g) is formed
// here, and k, q are scaled by their rows' inverse L2 norms rk, rq.
template <bool WANT_Q, bool MASK, bool GATE>
__device__ __forceinline__ void elementwise(const uint8_t *in, uint8_t *scr, uint8_t *rec, int nt,
                                            int lane, const float (&rk)[C], const float (&rq)[C]) {
    const float *gin = (const float *)(in + IN_G);
    const __nv_bfloat16 *xin = (const __nv_bfloat16 *)(in + IN_G);
    const __nv_bfloat16 *kin = (const __nv_bfloat16 *)(in + IN_K);
    const __nv_bfloat16 *qin = (const __nv_bfloat16 *)(in + IN_Q);
#pragma unroll 1
    for (int m = 0; m < 4; ++m) {
        const int ch = lane + 32 * m;
        float al[C], kv[C];
#pragma unroll
        for (int r = 0; r < C; ++r) {
            if (GATE) {
                const float xg = __bfloat162float(xin[r * D + ch]);
                // g = -5 sigmoid(x_g); the fast divide (reciprocal and multiply, ~2 ulp)
                // is far below the BF16 rounding of the operands g feeds
                al[r] = __fdividef(-5.f, 1.f + __expf(-xg));
                kv[r] = __bfloat162float(kin[r * D + ch]) * rk[r];
            } else {
                al[r] = gin[r * D + ch];
                kv[r] = __bfloat162float(kin[r * D + ch]);
            }
        }
        if (MASK) {
#pragma unroll
            for (int r = 0; r < C; ++r) {
                al[r] = r < nt ? al[r] : 0.f;
                kv[r] = r < nt ? kv[r] : 0.f;
            }
        }
#pragma unroll
        for (int r = 0; r < C; ++r) al[r] = __expf(al[r]);  // alpha = e^g
        float fwd[C], rev[C];  // e^{Gamma_r}, e^{Gamma_C - Gamma_r}
        float a = 1.f;
#pragma unroll
        for (int r = 0; r < C; ++r) { a *= al[r]; fwd[r] = a; }
        float b = 1.f;
#pragma unroll
        for (int r = C - 1; r >= 0; --r) { rev[r] = b; b *= al[r]; }
        const float eGC = fwd[C - 1];
        const float einv = 1.f / eGC;
        // One operand's 16 positions for this channel as one 32-byte row.
        auto put_row = [&](uint8_t *dst, const float (&val)[C]) {
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) w[e] = pack_bf16x2(val[2 * e], val[2 * e + 1]);
            *(uint4 *)dst = make_uint4(w[0], w[1], w[2], w[3]);
            *(uint4 *)(dst + 16) = make_uint4(w[4], w[5], w[6], w[7]);
        };
        // products over adjacent token pairs as packed f32x2 multiplies
        auto vmul = [&](float (&o)[C], const float (&x)[C], const float (&y)[C]) {
#pragma unroll
            for (int e = 0; e < C / 2; ++e) {
                o[2 * e] = x[2 * e];
                o[2 * e + 1] = x[2 * e + 1];
                mul2_inplace(o[2 * e], o[2 * e + 1], make_float2(y[2 * e], y[2 * e + 1]));
            }
        };
        // the products with e^{Gamma} first (Kh, Qh), so that fwd is dead before the
        // reverse factors are used: fewer arrays live at once
        float tmp[C];
        vmul(tmp, kv, fwd);
        put_row(rec + ch * RLB + RC_KH * 2, tmp);
        if (WANT_Q) {
            float qv[C];
#pragma unroll
            for (int r = 0; r < C; ++r) {
                const float q1 = __bfloat162float(qin[r * D + ch]) * (GATE ? rq[r] : 1.f);
                qv[r] = MASK && r >= nt ? 0.f : q1;
            }
            vmul(tmp, qv, fwd);
            put_row(rec + ch * RLB + RC_Q * 2, tmp);
        }
        vmul(tmp, kv, rev);
        put_row(rec + ch * RLB + RC_K * 2, tmp);
        // Kt = K e^{-Gamma_r} = Kb / e^{Gamma_C}, in place
#pragma unroll
        for (int e = 0; e < C / 2; ++e) mul2_inplace(tmp[2 * e], tmp[2 * e + 1], make_float2(einv, einv));
        put_row(scr + X_KT + ch * TROW, tmp);
        ((float *)(rec + R_DECAY))[ch] = eGC;
    }
}

// One warp prepares one whole block: elementwise factors, L and Mq and the
// solve for T, written with V into a record slot.  Prep warp p takes
// blocks p, p + 4, p + 8, ...; it frees the input stage as soon as it has read it.
template <bool WANT_Q, bool GATE, bool REV>
__device__ __forceinline__ void prep_role(const Ctx &x) {
    const PrefillArgs &p = *x.p;
    const int pw = (threadIdx.x >> 5) - W_PREP0;
    const int lane = threadIdx.x & 31, g8 = lane >> 2, t4 = lane & 3;
    uint8_t *scr = x.smem + X_OFF + pw * X_SIZE;
    const uint32_t scr_s = x.sbase + X_OFF + pw * X_SIZE;
    float *Lf = (float *)(scr + X_L);
    const int st = pw;  // this warp's input stage
    const uint32_t full = x.bar(B_IN_FULL + st);
    const uint32_t in_s = x.sbase + IN_OFF + st * IN_SIZE;
    const uint8_t *in = x.smem + IN_OFF + st * IN_SIZE;

    // The warp loads its own blocks: one 2D tensor-map TMA copy per array (whole
    // 16-row boxes; rows past the block's end hold the next sequence's tokens,
    // masked below, or past the array zero fill).
    // the c-th block prepared is block c of the segment, or with REV block
    // nchunks - 1 - c (the adjoint chain runs from the last block to the first)
    auto first_token = [&](int c) { return x.t_begin + C * (REV ? x.nchunks - 1 - c : c); };
    auto issue = [&](int c) {
        if (lane == 0) {
            const uint32_t bytes =
                (WANT_Q ? 4096u : 0u) + 4096u + (x.want_v ? 4096u : 0u) + (GATE ? 4096u : 8192u);
            mbar_arrive_expect_tx(full, bytes);
            const int xc = x.h * D, t0 = first_token(c);
            if (WANT_Q) tma_load_2d(in_s + IN_Q, x.tm_q, xc, t0, full);
            tma_load_2d(in_s + IN_K, x.tm_k, xc, t0, full);
            if (x.want_v) tma_load_2d(in_s + IN_V, x.tm_v, xc, t0, full);
            tma_load_2d(in_s + IN_G, x.tm_g, xc, t0, full);
        }
    };
    // beta (or with the fused prologue its pre-activation) of rows g8 and g8 + 8
    // (for L) and of column lane (for T), loaded one block ahead; rows past the
    // block's end read nothing
    auto load_beta = [&](int c, float &lo, float &hi, float &col) {
        const int t0 = first_token(c), nt = min(C, x.t_end - t0);
        const float *bp = p.beta + (size_t)t0 * p.H + x.h;
        lo = g8 < nt ? bp[(size_t)g8 * p.H] : 0.f;
        hi = g8 + 8 < nt ? bp[(size_t)(g8 + 8) * p.H] : 0.f;
        col = (lane & 15) < nt ? bp[(size_t)(lane & 15) * p.H] : 0.f;
    };
    // The sigmoid of the fused prologue is taken a block after the load, when the
    // value is used, so that no instruction waits on the load in flight; rows past
    // the block's end get beta = 0.
    auto act = [&](float v, int r, int nt) {
        return r < nt ? (GATE ? __fdividef(1.f, 1.f + __expf(-v)) : v) : 0.f;
    };
    int issued = 0;  // blocks whose copies were issued (for an orderly abort)
    float b_lo = 0.f, b_hi = 0.f, b_col = 0.f;
    if (pw < x.nchunks) {
        issue(pw);
        issued = 1;
        load_beta(pw, b_lo, b_hi, b_col);
    }

    int uses = 0;  // completed uses of the input stage
    for (int c = pw; c < x.nchunks; c += N_PREP, ++uses) {
        const int slot = c % NR;
        const int nt = min(C, x.t_end - first_token(c));
        const float beta_lo = act(b_lo, g8, nt), beta_hi = act(b_hi, g8 + 8, nt),
                    beta_col = act(b_col, lane & 15, nt);
        if (c + N_PREP < x.nchunks) load_beta(c + N_PREP, b_lo, b_hi, b_col);
        if (!warp_wait(x, B_REC_EMPTY + slot, ((c / NR) & 1) ^ 1)) break;
        if (!warp_wait(x, B_IN_FULL + st, uses & 1)) break;
        uint8_t *rec = x.smem + REC_OFF + slot * R_SIZE;
        const uint32_t rec_s = x.sbase + REC_OFF + slot * R_SIZE;

        // ---- fused prologue: inverse L2 norms of this block's k and q rows (a zero
        // row keeps scale 0), in fp32 FMAs: lane (r, half) sums the squares of 64
        // channels of row r = lane / 2, reading its 16-byte chunks in a rotated order
        // so that the eight lanes of each quarter-warp hit eight different banks,
        // then adds its partner's half.  The row scales reach every lane through the
        // L scratch, which is free until L is formed below.  (The diagonal of K K^T
        // on the tensor cores took several times longer per block: its 32 small
        // products waited behind the chain warps' products on the same pipe.)
        float rk[C], rq[C];
        if (GATE) {
            const int rr = lane >> 1, hf = lane & 1;
            float2 ak = make_float2(0.f, 0.f), aq = make_float2(0.f, 0.f);
#pragma unroll
            for (int v = 0; v < 8; ++v) {
                const int off = rr * IN_ROWB + hf * 128 + 16 * ((v + lane) & 7);
                const uint4 wk = *(const uint4 *)(in + IN_K + off);
                const uint32_t k4[4] = {wk.x, wk.y, wk.z, wk.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&k4[e]));
                    fma2_acc(ak.x, ak.y, f.x, f.y, f.x, f.y);
                }
                if (WANT_Q) {
                    const uint4 wq = *(const uint4 *)(in + IN_Q + off);
                    const uint32_t q4[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&q4[e]));
                        fma2_acc(aq.x, aq.y, f.x, f.y, f.x, f.y);
                    }
                }
            }
            float sk = ak.x + ak.y, sq = aq.x + aq.y;
            sk += __shfl_xor_sync(0xffffffffu, sk, 1);
            sq += __shfl_xor_sync(0xffffffffu, sq, 1);
            if (hf == 0) {
                Lf[rr] = sk > 0.f ? rsqrtf(sk) : 0.f;
                Lf[C + rr] = sq > 0.f ? rsqrtf(sq) : 0.f;
            }
            __syncwarp();
#pragma unroll
            for (int r4 = 0; r4 < C / 4; ++r4) {
                const float4 a4 = *(const float4 *)(Lf + 4 * r4);
                const float4 b4 = *(const float4 *)(Lf + C + 4 * r4);
                rk[4 * r4] = a4.x;
                rk[4 * r4 + 1] = a4.y;
                rk[4 * r4 + 2] = a4.z;
                rk[4 * r4 + 3] = a4.w;
                rq[4 * r4] = WANT_Q ? b4.x : 0.f;
                rq[4 * r4 + 1] = WANT_Q ? b4.y : 0.f;
                rq[4 * r4 + 2] = WANT_Q ? b4.z : 0.f;
                rq[4 * r4 + 3] = WANT_Q ? b4.w : 0.f;
            }
        }

        // ---- elementwise: lane handles key channels lane + 32 m
        if (nt == C) elementwise<WANT_Q, false, GATE>(in, scr, rec, nt, lane, rk, rq);
        else elementwise<WANT_Q, true, GATE>(in, scr, rec, nt, lane, rk, rq);
        // V into the record (padded rows).  Rows past the block's end become zero:
        // they are weighted by zero in the chain's products, and the next
        // sequence's values (or anything non-finite in them) must not leak in.
        if (x.want_v) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int idx = lane + 32 * i, r = idx >> 4, q16 = idx & 15;
                uint4 v = *(const uint4 *)(in + IN_V + r * IN_ROWB + q16 * 16);
                if (r >= nt) v = make_uint4(0u, 0u, 0u, 0u);
                *(uint4 *)(rec + R_V + r * VROWB + q16 * 16) = v;
            }
        }
        __syncwarp();
        // Input stage read: load this warp's next block into it (the generic reads
        // above are ordered before the copy's writes by the proxy fence).
        if (c + N_PREP < x.nchunks) {
            if (lane == 0) fence_async_smem();
            issue(c + N_PREP);
            ++issued;
        }

        // ---- L = Diag(beta) strict_lower(Kh Kt^T) and Mq = lower(Qh Kt^T), 16 x 16 x 128
        {
            float accL[2][4] = {}, accM[2][4] = {};
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                uint32_t bf[4], af[4];
                // B (channels x positions) from Kt^T rows, transposed
                ldsm_x4_t(scr_s + X_KT + (kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * TROW +
                              (lane >> 4) * 16,
                          bf);
                // A (positions x channels) from the record's Kh^T rows, transposed
                ldsm_x4_t(rec_s + (kk * 16 + (lane & 7) + ((lane >> 4) << 3)) * RLB + RC_KH * 2 +
                              ((lane >> 3) & 1) * 16,
                          af);
                mma_bf16_16816(accL[0], af, bf[0], bf[1]);
                mma_bf16_16816(accL[1], af, bf[2], bf[3]);
                if (WANT_Q) {
                    uint32_t aq[4];
                    ldsm_x4_t(rec_s + (kk * 16 + (lane & 7) + ((lane >> 4) << 3)) * RLB + RC_Q * 2 +
                                  ((lane >> 3) & 1) * 16,
                              aq);
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

        // ---- T = (I + Diag(beta) L)^{-1} Diag(beta): forward substitution, lane = column
        if (lane < C) {
            const int j = lane;
            float xv[C];
#pragma unroll
            for (int r = 0; r < C; ++r) xv[r] = (r == j) ? 1.f : 0.f;
#pragma unroll
            for (int r = 1; r < C; ++r) {
                float s0 = 0.f, s1 = 0.f;
                // row r of L in 16-byte pieces (one broadcast load per four entries)
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
        __syncwarp();

        if (lane == 0) mbar_arrive(x.bar(B_REC_FULL + slot));
    }
    // On an abort, let this warp's copies in flight land before the CTA can exit.
    if (*x.abort && lane == 0 && issued > uses) {
        volatile int never = 0;
        mbar_wait(full, uses & 1, &never, kWaitLimit);
    }
}

// ------------------------------------------------------------------ chain
// Chain warp w owns state columns [32w, 32w+32) as two 16-column m-tiles, which
// share every B fragment the warp loads from the record.
constexpr int MT = 2;  // m-tiles per chain warp

template <bool WANT_Q, int NCH, bool REV, bool CKS, bool LEAD = false>
__device__ __forceinline__ void chain_role(const Ctx &x) {
    const PrefillArgs &p = *x.p;
    const int chain = ((threadIdx.x >> 5) - W_CHAIN0) / N_CHAIN;  // 0 unless NCH = 2
    const int cw = ((threadIdx.x >> 5) - W_CHAIN0) % N_CHAIN;
    // with two chains per CTA, chain 0 starts from the identity (transfer matrix)
    // and chain 1 from zeros with the values (zero-initial state)
    // (LEAD: the zero-start chain of a lead CTA, which starts from S0)
    const bool partA = !REV && !LEAD && (NCH == 2 ? chain == 0 : x.partA);
    const bool want_v = !partA;
    const int lane = threadIdx.x & 31, g8 = lane >> 2, t4 = lane & 3;
    const int j0 = 16 * MT * cw;
    const size_t unit = (size_t)x.n * p.H + x.h;

    // S^T[j][i] for j = j0 + 16 m + g8 (+8), i = 8n + 2t4 (+1)
    float S[MT][16][4];
    {
        const float *src = nullptr;
        const int sidx = REV ? p.Sg - 1 - x.s : x.s;  // the adjoint's arrays run reversed
        if (!x.transfer)
            src = p.seg_init ? p.seg_init + (unit * p.Sg + sidx) * (size_t)D * D
                             : (p.S0 ? p.S0 + unit * (size_t)D * D : nullptr);
        else if (LEAD && p.S0)
            src = p.S0 + unit * (size_t)D * D;
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int n = 0; n < 16; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = 8 * n + 2 * t4 + (e & 1), j = j0 + 16 * m + g8 + 8 * (e >> 1);
                    S[m][n][e] = partA ? (i == j ? 1.f : 0.f)
                                         : (src ? src[(size_t)i * D + j] : 0.f);
                }
    }

    // output destination: the prefill's out, or in the transfer pass the zero-start
    // chain's outputs (out) and the identity-start chain's A_t^T q_t (aux_out)
    __nv_bfloat16 *out = (__nv_bfloat16 *)(partA ? p.aux_out : p.out);
    const uint32_t ost_s = x.sbase + OST_OFF + (chain * N_CHAIN + cw) * OST_SIZE;
    const uint8_t *ost = x.smem + OST_OFF + (chain * N_CHAIN + cw) * OST_SIZE;
    // The state, transposed and in BF16, into chunk-state slot `slot` ([dv][dk]:
    // the two channels a lane holds per row are adjacent, one 4-byte store each).
    auto store_chunk_state = [&](int cslot) {
        __nv_bfloat16 *d = p.chunk_states + ((size_t)cslot * p.H + x.h) * D * D;
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int n = 0; n < 16; ++n)
#pragma unroll
                for (int hi = 0; hi < 2; ++hi)
                    *(uint32_t *)(d + (size_t)(j0 + 16 * m + g8 + 8 * hi) * D + 8 * n + 2 * t4) =
                        pack_bf16x2(S[m][n][2 * hi], S[m][n][2 * hi + 1]);
    };
    // Checkpoints fall on the blocks whose end is a multiple of ckpt_interval tokens
    // into the sequence (a multiple of 16; segments start on block boundaries):
    // every ck_step-th block from ck_c on, the k-th of the sequence being ck_k.
    const int ck_step = p.ckpt_interval > 0 ? p.ckpt_interval / C : 0;
    const int blk0 = (x.t_begin - x.seq0) / C;
    int ck_c = ck_step > 0 ? ck_step - 1 - blk0 % ck_step : -1;
    int ck_k = ck_step > 0 ? (blk0 + ck_c + 1) / ck_step : 0;
    for (int c = 0; c < x.nchunks; ++c) {
        const int slot = c % NR;
        if (!warp_wait(x, B_REC_FULL + slot, (c / NR) & 1)) break;
        const uint32_t rec_s = x.sbase + REC_OFF + slot * R_SIZE;
        const float *decay = (const float *)(x.smem + REC_OFF + slot * R_SIZE + R_DECAY);
        if constexpr (REV) {
            // ---- adjoint chain, block nchunks - 1 - c: the state is dS', the
            // adjoint of the state after the block (written out first)
            if (p.chunk_states)
                store_chunk_state(x.cs_base + (x.t_begin - x.seq0) / C + x.nchunks - 1 - c);
            // dU^T = dO^T Mq + dS'^T Kb^T (j x r): seeded with dO^T Mq
            float E[MT][2][4] = {};
            uint32_t doa[MT][4];  // dO^T as A fragments (rows j, k = r)
            {
                uint32_t mqt[4];
                ldsm_x4_t(rec_s + R_MQ + ((lane & 7) + 8 * ((lane >> 3) & 1)) * (TL * 2) +
                              16 * (lane >> 4),
                          mqt);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    ldsm_x4_t(rec_s + R_V + (8 * (lane >> 4) + (lane & 7)) * VROWB +
                                  (j0 + 16 * m + 8 * ((lane >> 3) & 1)) * 2,
                              doa[m]);
                    mma_bf16_16816(E[m][0], doa[m], mqt[0], mqt[1]);
                    mma_bf16_16816(E[m][1], doa[m], mqt[2], mqt[3]);
                }
            }
            {
                uint32_t bk[2][4];
                auto load_b = [&](int kk, uint32_t (&w)[4]) {
                    ldsm_x4_t(rec_s + (16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1)) * RLB +
                                  16 * (lane >> 4) + RC_K * 2,
                              w);
                };
                load_b(0, bk[0]);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    if (kk + 1 < 8) load_b(kk + 1, bk[(kk + 1) & 1]);
                    const uint32_t(&w)[4] = bk[kk & 1];
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        const uint32_t a[4] = {
                            pack_bf16x2(S[m][2 * kk][0], S[m][2 * kk][1]),
                            pack_bf16x2(S[m][2 * kk][2], S[m][2 * kk][3]),
                            pack_bf16x2(S[m][2 * kk + 1][0], S[m][2 * kk + 1][1]),
                            pack_bf16x2(S[m][2 * kk + 1][2], S[m][2 * kk + 1][3])};
                        mma_bf16_16816(E[m][0], a, w[0], w[1]);
                        mma_bf16_16816(E[m][1], a, w[2], w[3]);
                    }
                }
            }
            // dR^T = dU^T T (j x r), kept negated as A fragments
            uint32_t ndra[MT][4];
            {
                uint32_t tt[4];
                ldsm_x4_t(rec_s + R_T + ((lane & 7) + 8 * ((lane >> 3) & 1)) * (TL * 2) +
                              16 * (lane >> 4),
                          tt);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const uint32_t dua[4] = {pack_bf16x2(E[m][0][0], E[m][0][1]),
                                             pack_bf16x2(E[m][0][2], E[m][0][3]),
                                             pack_bf16x2(E[m][1][0], E[m][1][1]),
                                             pack_bf16x2(E[m][1][2], E[m][1][3])};
                    float R[2][4] = {};
                    mma_bf16_16816(R[0], dua, tt[0], tt[1]);
                    mma_bf16_16816(R[1], dua, tt[2], tt[3]);
                    ndra[m][0] = pack_bf16x2(-R[0][0], -R[0][1]);
                    ndra[m][1] = pack_bf16x2(-R[0][2], -R[0][3]);
                    ndra[m][2] = pack_bf16x2(-R[1][0], -R[1][1]);
                    ndra[m][3] = pack_bf16x2(-R[1][2], -R[1][3]);
                }
            }
            // dS^T <- dS'^T Diag(e^{Gamma_C}) + dO^T Qh - dR^T Kh
#pragma unroll
            for (int np = 0; np < 8; ++np) {
                uint32_t fq[4], fk[4];
                const uint32_t row = rec_s + (16 * np + (lane & 7) + 8 * (lane >> 4)) * RLB +
                                     16 * ((lane >> 3) & 1);
                ldsm_x4(row + RC_Q * 2, fq);
                ldsm_x4(row + RC_KH * 2, fk);
                const float2 d0 = *(const float2 *)(decay + 16 * np + 2 * t4);
                const float2 d1 = *(const float2 *)(decay + 16 * np + 8 + 2 * t4);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    mul2_inplace(S[m][2 * np][0], S[m][2 * np][1], d0);
                    mul2_inplace(S[m][2 * np][2], S[m][2 * np][3], d0);
                    mul2_inplace(S[m][2 * np + 1][0], S[m][2 * np + 1][1], d1);
                    mul2_inplace(S[m][2 * np + 1][2], S[m][2 * np + 1][3], d1);
                    mma_bf16_16816(S[m][2 * np], doa[m], fq[0], fq[1]);
                    mma_bf16_16816(S[m][2 * np], ndra[m], fk[0], fk[1]);
                    mma_bf16_16816(S[m][2 * np + 1], doa[m], fq[2], fq[3]);
                    mma_bf16_16816(S[m][2 * np + 1], ndra[m], fk[2], fk[3]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(x.bar(B_REC_EMPTY + slot));
            continue;
        }

        // E^T = S^T Kh^T - V^T (j x r) = -(V - Kh S)^T in fp32.  V^T is loaded as
        // an A fragment, whose element positions are those of the 16 x 16
        // accumulator pair, so it seeds E directly.
        float E[MT][2][4] = {};
        if (want_v) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                uint32_t va[4];
                ldsm_x4_t(rec_s + R_V + (8 * (lane >> 4) + (lane & 7)) * VROWB +
                              (j0 + 16 * m + 8 * ((lane >> 3) & 1)) * 2,
                          va);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 v2 =
                        __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&va[q]));
                    E[m][q >> 1][2 * (q & 1)] = -v2.x;
                    E[m][q >> 1][2 * (q & 1) + 1] = -v2.y;
                }
            }
        }
        float O[MT][2][4] = {};  // (Qh S)^T, then + (Mq U)^T
        {
            uint32_t bk[2][4], bq[2][4];
            auto load_b = [&](int kk, uint32_t (&w)[4], uint32_t (&q)[4]) {
                const uint32_t brow =
                    rec_s + (16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1)) * RLB + 16 * (lane >> 4);
                ldsm_x4_t(brow + RC_KH * 2, w);
                if (WANT_Q) ldsm_x4_t(brow + RC_Q * 2, q);
            };
            load_b(0, bk[0], bq[0]);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                if (kk + 1 < 8) load_b(kk + 1, bk[(kk + 1) & 1], bq[(kk + 1) & 1]);
                const uint32_t(&w)[4] = bk[kk & 1];
                const uint32_t(&q)[4] = bq[kk & 1];
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const uint32_t a[4] = {pack_bf16x2(S[m][2 * kk][0], S[m][2 * kk][1]),
                                           pack_bf16x2(S[m][2 * kk][2], S[m][2 * kk][3]),
                                           pack_bf16x2(S[m][2 * kk + 1][0], S[m][2 * kk + 1][1]),
                                           pack_bf16x2(S[m][2 * kk + 1][2], S[m][2 * kk + 1][3])};
                    mma_bf16_16816(E[m][0], a, w[0], w[1]);
                    mma_bf16_16816(E[m][1], a, w[2], w[3]);
                    if (WANT_Q) {
                        mma_bf16_16816(O[m][0], a, q[0], q[1]);
                        mma_bf16_16816(O[m][1], a, q[2], q[3]);
                    }
                }
            }
        }
        // U^T = (V - Kh S)^T T^T = -E^T T^T
        uint32_t ua[MT][4];
        {
            uint32_t tb[4];
            ldsm_x4(rec_s + R_T + (8 * (lane >> 4) + (lane & 7)) * (TL * 2) + 16 * ((lane >> 3) & 1),
                    tb);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const uint32_t ea[4] = {pack_bf16x2(-E[m][0][0], -E[m][0][1]),
                                        pack_bf16x2(-E[m][0][2], -E[m][0][3]),
                                        pack_bf16x2(-E[m][1][0], -E[m][1][1]),
                                        pack_bf16x2(-E[m][1][2], -E[m][1][3])};
                float U[2][4] = {};
                mma_bf16_16816(U[0], ea, tb[0], tb[1]);
                mma_bf16_16816(U[1], ea, tb[2], tb[3]);
                ua[m][0] = pack_bf16x2(U[0][0], U[0][1]);
                ua[m][1] = pack_bf16x2(U[0][2], U[0][3]);
                ua[m][2] = pack_bf16x2(U[1][0], U[1][1]);
                ua[m][3] = pack_bf16x2(U[1][2], U[1][3]);
            }
        }

        // S^T <- S^T Diag(e^{Gamma_C}) + U^T Kb.  Kb fragments and the decay pairs are
        // loaded one tile pair ahead; the decay runs as packed f32x2 multiplies
        // (the two channels a lane holds per row are adjacent).
        {
            uint32_t kb[2][4];
            float2 dd[2][2];
            auto load_kb = [&](int np, uint32_t (&f)[4], float2 (&d)[2]) {
                ldsm_x4(rec_s + (16 * np + (lane & 7) + 8 * (lane >> 4)) * RLB + RC_K * 2 +
                            16 * ((lane >> 3) & 1),
                        f);
                d[0] = *(const float2 *)(decay + 16 * np + 2 * t4);
                d[1] = *(const float2 *)(decay + 16 * np + 8 + 2 * t4);
            };
            load_kb(0, kb[0], dd[0]);
#pragma unroll
            for (int np = 0; np < 8; ++np) {
                if (np + 1 < 8) load_kb(np + 1, kb[(np + 1) & 1], dd[(np + 1) & 1]);
                const float2 d0 = dd[np & 1][0], d1 = dd[np & 1][1];
                const uint32_t(&f)[4] = kb[np & 1];
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    mul2_inplace(S[m][2 * np][0], S[m][2 * np][1], d0);
                    mul2_inplace(S[m][2 * np][2], S[m][2 * np][3], d0);
                    mul2_inplace(S[m][2 * np + 1][0], S[m][2 * np + 1][1], d1);
                    mul2_inplace(S[m][2 * np + 1][2], S[m][2 * np + 1][3], d1);
                    mma_bf16_16816(S[m][2 * np], ua[m], f[0], f[1]);
                    mma_bf16_16816(S[m][2 * np + 1], ua[m], f[2], f[3]);
                }
            }
        }

        if (WANT_Q) {
            uint32_t mq[4];
            ldsm_x4(rec_s + R_MQ + (8 * (lane >> 4) + (lane & 7)) * (TL * 2) + 16 * ((lane >> 3) & 1),
                    mq);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                mma_bf16_16816(O[m][0], ua[m], mq[0], mq[1]);
                mma_bf16_16816(O[m][1], ua[m], mq[2], mq[3]);
                // O^T (j x r) -> staging [r][j], then one 16-byte store per (token, half)
                stsm_x4_t(ost_s + m * 512 + ((lane & 7) + 8 * (lane >> 4)) * 32 +
                              16 * ((lane >> 3) & 1),
                          pack_bf16x2(O[m][0][0], O[m][0][1]), pack_bf16x2(O[m][0][2], O[m][0][3]),
                          pack_bf16x2(O[m][1][0], O[m][1][1]), pack_bf16x2(O[m][1][2], O[m][1][3]));
            }
            __syncwarp();
            const int t0 = x.t_begin + C * c;
            const int r = lane >> 1, half = lane & 1;
            if (r < x.t_end - t0) {
#pragma unroll
                for (int m = 0; m < MT; ++m)
                    *(uint4 *)(out + ((size_t)(t0 + r) * p.H + x.h) * D + j0 + 16 * m + 8 * half) =
                        *(const uint4 *)(ost + m * 512 + r * 32 + half * 16);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(x.bar(B_REC_EMPTY + slot));
        if (CKS) {  // the state after every 32 tokens, BF16 transposed
            const int done = min(x.t_begin + C * (c + 1), x.t_end) - x.seq0;
            if (done % (2 * C) == 0) store_chunk_state(x.cs_base + done / (2 * C) - 1);
        }
        if (c == ck_c) {  // state checkpoint after this block
            float *d = partA ? p.ckpt_a : p.ckpt;
            if (x.t_begin + C * (c + 1) <= x.t_end && d) {
                d += ((size_t)(x.ckpt_base + ck_k - 1) * p.H + x.h) * D * D;
#pragma unroll
                for (int m = 0; m < MT; ++m)
#pragma unroll
                    for (int n = 0; n < 16; ++n)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            d[(size_t)(8 * n + 2 * t4 + (e & 1)) * D + j0 + 16 * m + g8 + 8 * (e >> 1)] =
                                S[m][n][e];
            }
            ck_c += ck_step;
            ++ck_k;
        }
    }
    // Both chains of a two-chain CTA have consumed every record before either
    // stages its final writes over the records; the decision to stop after an
    // abort is taken together.
    if (NCH == 2) {
        if (named_bar_or(1, N_CHAIN * 64, *x.abort != 0)) return;
    } else if (*x.abort) {
        return;
    }

    float *dst = nullptr;
    if (!x.transfer) {
        // the adjoint chain ends at the segment's start: segment 0 gives dS0
        if (x.s == (REV ? 0 : p.Sg - 1) && p.S_final) dst = p.S_final + unit * (size_t)D * D;
    } else {
        float *base = partA ? p.transfer : p.zero_state;
        const int sidx = REV ? p.Sg - 1 - x.s : x.s;
        if (base) dst = base + (unit * p.Sg + sidx) * (size_t)D * D;
    }
    // Final writes go through shared memory so that every global store is a fully
    // used 16-byte piece of a contiguous run.  Every record has been consumed, so
    // the prep warps are done with the input stages; each chain warp stages its
    // 32 columns j in a private FW_SIZE slice of them.
    uint8_t *fw = x.smem + IN_OFF + (chain * N_CHAIN + cw) * FW_SIZE;
    const uint32_t fw_s = x.sbase + IN_OFF + (chain * N_CHAIN + cw) * FW_SIZE;
    if (partA && p.transfer_img) {
        // A[i][j] as hi/lo BF16 images, transposed ([j][i], i contiguous): the
        // accumulator fragments are already j-row / i-column, so stmatrix writes
        // 16 x 16 blocks of each image into [32 j][FW_IROW bytes] rows.
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int pb = 0; pb < 8; ++pb) {  // one 16 x 16 block of both images
                uint32_t rh[4], rl[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {  // matrix k: rows +8 (k & 1), cols +8 (k >> 1)
                    const float v0 = S[m][2 * pb + (k >> 1)][2 * (k & 1)];
                    const float v1 = S[m][2 * pb + (k >> 1)][2 * (k & 1) + 1];
                    const __nv_bfloat162 h2 = __floats2bfloat162_rn(v0, v1);
                    const float2 hf = __bfloat1622float2(h2);
                    rh[k] = *(const uint32_t *)&h2;
                    rl[k] = pack_bf16x2(v0 - hf.x, v1 - hf.y);
                }
                const int mk = lane >> 3, row = 16 * m + (lane & 7) + 8 * (mk & 1);
                const uint32_t o = row * FW_IROW + (16 * pb + 8 * (mk >> 1)) * 2;
                stsm_x4(fw_s + o, rh[0], rh[1], rh[2], rh[3]);
                stsm_x4(fw_s + 32 * FW_IROW + o, rl[0], rl[1], rl[2], rl[3]);
            }
        __syncwarp();
        // rows j0 .. j0+31 of each image are 8 KB contiguous in global memory
        __nv_bfloat16 *hi = p.transfer_img + (unit * p.Sg + x.s) * (size_t)2 * D * D;
#pragma unroll
        for (int img = 0; img < 2; ++img)
#pragma unroll 4
            for (int it = 0; it < 16; ++it) {
                const int idx = 32 * it + lane, row = idx >> 4, c16 = idx & 15;
                *(uint4 *)(hi + (size_t)img * D * D + (size_t)(j0 + row) * D + 8 * c16) =
                    *(const uint4 *)(fw + img * 32 * FW_IROW + row * FW_IROW + 16 * c16);
            }
    }
    if (partA && p.transfer_img_t) {
        // A[i][j] row-major as hi/lo BF16 images (the images of A^T in the layout
        // above) at the reversed segment index: stage fp32 [128 i][FW_JROW] as for
        // the states below, then each row's 32 columns as 64-byte pieces
        if (p.transfer_img) __syncwarp();  // the staging above has been read
        float *f = (float *)fw;
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int n = 0; n < 16; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    f[(8 * n + 2 * t4 + (e & 1)) * FW_JROW + 16 * m + g8 + 8 * (e >> 1)] = S[m][n][e];
        __syncwarp();
        __nv_bfloat16 *hi = p.transfer_img_t + (unit * p.Sg + p.Sg - 1 - x.s) * (size_t)2 * D * D;
#pragma unroll 4
        for (int it = 0; it < 16; ++it) {  // 128 rows x 4 pieces of 8 columns
            const int idx = 32 * it + lane, i = idx >> 2, c = idx & 3;
            const float4 v0 = *(const float4 *)(f + i * FW_JROW + 8 * c);
            const float4 v1 = *(const float4 *)(f + i * FW_JROW + 8 * c + 4);
            const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
            uint32_t wh[4], wl[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
                const float2 hf = __bfloat1622float2(h2);
                wh[e] = *(const uint32_t *)&h2;
                wl[e] = pack_bf16x2(v[2 * e] - hf.x, v[2 * e + 1] - hf.y);
            }
            const size_t o = (size_t)i * D + j0 + 8 * c;
            *(uint4 *)(hi + o) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
            *(uint4 *)(hi + (size_t)D * D + o) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
        }
    } else if (dst && !(partA && p.transfer_img)) {
        // S[i][j] (j contiguous) is the transpose of the accumulator layout: stage
        // this warp's columns as [128 i][FW_JROW floats] (conflict-free scalar
        // stores), then write 128-byte row segments.
        float *f = (float *)fw;
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int n = 0; n < 16; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    f[(8 * n + 2 * t4 + (e & 1)) * FW_JROW + 16 * m + g8 + 8 * (e >> 1)] = S[m][n][e];
        __syncwarp();
        const bool v16 = ((uintptr_t)dst & 15u) == 0;  // S_final is only 4-byte aligned
#pragma unroll 4
        for (int it = 0; it < 32; ++it) {
            const int idx = 32 * it + lane, i = idx >> 3, c = idx & 7;
            const float4 v = *(const float4 *)(f + i * FW_JROW + 4 * c);
            float *d = dst + (size_t)i * D + j0 + 4 * c;
            if (v16) {
                *(float4 *)d = v;
            } else {
                d[0] = v.x;
                d[1] = v.y;
                d[2] = v.z;
                d[3] = v.w;
            }
        }
    }
}

// With or without V is a runtime switch (uniform per CTA), not a template
// parameter: the identity-start and zero-start CTAs of the transfer pass then
// run the same instructions, so the code that the first of them fetches into the
// instruction caches serves the other, and the kernel's code footprint halves.
// REV: the adjoint chain; CKS: the forward chain also writes chunk states (the
// backward's forward pass).  Both are separate instantiations, so the prefill's
// own kernels carry none of their code.
// The identity-start warpgroup of a lead CTA: the lead segment runs from S0, so its
// transfer matrix is zero (the scan then passes the segment's end state on as the
// next start state).  Each warp zeroes its 32 rows of both images (or its 32
// columns of the fp32 matrix) and meets the running chain at its final barrier.
__device__ __forceinline__ void lead_idle_role(const Ctx &x) {
    const PrefillArgs &p = *x.p;
    const int cw = ((threadIdx.x >> 5) - W_CHAIN0) % N_CHAIN, lane = threadIdx.x & 31;
    const int j0 = 32 * cw;
    const size_t unit = (size_t)x.n * p.H + x.h;
    if (p.transfer_img) {
        __nv_bfloat16 *img = p.transfer_img + (unit * p.Sg + x.s) * (size_t)2 * D * D;
#pragma unroll 4
        for (int it = 0; it < 32; ++it) {  // 2 images x 32 rows x 16 pieces of 16 bytes
            const int idx = 32 * it + lane, im = idx >> 9, row = (idx >> 4) & 31, c16 = idx & 15;
            *(uint4 *)(img + (size_t)im * D * D + (size_t)(j0 + row) * D + 8 * c16) =
                make_uint4(0u, 0u, 0u, 0u);
        }
    } else if (p.transfer) {
        float *t = p.transfer + (unit * p.Sg + x.s) * (size_t)D * D;  // [i][j]
#pragma unroll 4
        for (int it = 0; it < 32; ++it) {  // 128 rows x 32 columns
            const int idx = 32 * it + lane, i = idx >> 3, c = idx & 7;
            float *d = t + (size_t)i * D + j0 + 4 * c;
            d[0] = d[1] = d[2] = d[3] = 0.f;
        }
    }
    named_bar_or(1, N_CHAIN * 64, *x.abort != 0);
}

template <bool WANT_Q, bool GATE, int NCH, bool REV = false, bool CKS = false>
__device__ __forceinline__ void run_role(const Ctx &x, int warp) {
    if (warp < W_CHAIN0) {
        if (NCH == 2) regs_dealloc<PREP_REGS>();
        prep_role<WANT_Q, GATE, REV>(x);
    } else if (NCH == 2 && !REV && !CKS && x.lead) {
        if ((warp - W_CHAIN0) / N_CHAIN == 0) {
            regs_dealloc<LEAD_IDLE_REGS>();
            lead_idle_role(x);
        } else {
            regs_alloc<LEAD_CHAIN_REGS>();
            chain_role<WANT_Q, NCH, REV, CKS, true>(x);
        }
    } else {
        if (NCH == 2) regs_alloc<CHAIN_REGS>();
        chain_role<WANT_Q, NCH, REV, CKS>(x);
    }
}

// GATE (the fused prologue) is a separate kernel: the plain kernel's code is then
// only its own, which matters because the kernel starts with cold instruction
// caches after the scan and the combine of the previous call.
// VAR: 0 the prefill, 1 the adjoint chain of the backward, 2 the backward's
// forward chain with chunk states.  Separate kernels, so that each one's code is
// only its own (the prefill starts with cold instruction caches after the scan
// and the combine of the previous call).
enum { VAR_PREFILL = 0, VAR_ADJOINT = 1, VAR_CHUNK_STATES = 2 };
template <bool GATE, int NCH, int VAR = VAR_PREFILL>
__global__ void __launch_bounds__(cta_threads(NCH), 1)
    prefill_tc_kernel(const __grid_constant__ PrefillArgs p, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_g) {
    extern __shared__ uint8_t smem_raw[];
    griddep_wait();  // inputs may come from the previous kernel in the stream
    griddep_launch_dependents();
    // Align by pointer arithmetic on the __shared__ array (not through an integer),
    // so accesses keep the shared address space instead of becoming generic.
    uint8_t *smem = smem_raw + ((128u - (smem_addr(smem_raw) & 127u)) & 127u);
    Ctx x;
    x.p = &p;
    x.tm_q = reinterpret_cast<uint64_t>(&tm_q);
    x.tm_k = reinterpret_cast<uint64_t>(&tm_k);
    x.tm_v = reinterpret_cast<uint64_t>(&tm_v);
    x.tm_g = reinterpret_cast<uint64_t>(&tm_g);
    x.smem = smem;
    x.sbase = smem_addr(smem);
    x.abort = (volatile int *)(smem + MISC_OFF);
    const int u = blockIdx.x;
    x.transfer = p.mode == MODE_TRANSFER;
    if (NCH == 2 && p.lead && x.transfer) {
        // the lead units (segment 0 of every chain, the longest) first, then
        // segments 1 .. Sg-1 of every chain
        const int nh = p.N * p.H, sc = p.Sg - 1;
        if (u < nh) {
            x.n = u / p.H;
            x.h = u % p.H;
            x.s = 0;
        } else {
            const int v = u - nh;
            x.n = v / (p.H * sc);
            x.h = (v / sc) % p.H;
            x.s = 1 + v % sc;
        }
    } else {
        x.n = u / (p.H * p.seg_count);
        x.h = (u / p.seg_count) % p.H;
        x.s = p.seg_begin + u % p.seg_count;
    }
    if (p.N <= 32) x.n = longest_first(p, x.n);
    x.lead = NCH == 2 && p.lead && x.transfer && x.s == 0;
    x.partA = NCH == 1 && x.transfer && blockIdx.y == 0 && !p.rev;
    // outputs (and q) only where they are written: the prefill's out, or the
    // transfer pass's outputs; the adjoint chain always needs q
    x.want_q = (!x.transfer && p.out) || p.emit_out || p.rev;
    x.want_v = !x.partA;  // the prep loads V whenever a chain of the CTA uses it
    if (!segment_range(p.cu, x.n, p.N, p.T_tot, x.s, p.Sg, p.dev_status, x.t_begin, x.t_end,
                       NCH == 2 ? p.lead : 0))
        return;
    x.nchunks = (x.t_end - x.t_begin + C - 1) / C;
    x.seq0 = p.cu[x.n];
    x.ckpt_base = p.ckpt_interval > 0 ? ckpt_base(p.cu, x.n, p.ckpt_interval) : 0;
    x.cs_base = !p.chunk_states ? 0 : (p.rev ? block_base(p.cu, x.n) : ckpt_base(p.cu, x.n, 2 * C));

    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) mbar_init(x.bar(B_IN_FULL + i), 1);
        for (int i = 0; i < NR; ++i) {
            mbar_init(x.bar(B_REC_FULL + i), 1);
            mbar_init(x.bar(B_REC_EMPTY + i), N_CHAIN * (x.lead ? 1 : NCH));
        }
        *x.abort = 0;
        mbar_fence_init();
    }
    __syncthreads();

    if (VAR == VAR_ADJOINT) run_role<true, false, 1, true>(x, warp);
    else if (VAR == VAR_CHUNK_STATES) run_role<false, false, 1, false, true>(x, warp);
    else if (GATE) run_role<true, true, NCH>(x, warp);  // (the fused prologue always has q)
    else if (x.want_q) run_role<true, false, NCH>(x, warp);
    else run_role<false, false, NCH>(x, warp);

    __syncthreads();
    if (threadIdx.x == 0 && *x.abort) dev_fail(p.dev_status, KDA_ERR_TIMEOUT);
}

}  // namespace

// The transfer pass runs both chains of a segment in one CTA once there are at
// least as many segments as SMs (the throughput regime: inputs read and prepared
// once); with fewer, each chain gets its own CTA and SM.
bool prefill_tc_two_chain(const PrefillArgs &a) {
    int sms = 148, dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return a.mode == MODE_TRANSFER && (long long)a.N * a.H * a.seg_count >= sms && !a.rev;
}

bool prefill_tc_supported(const PrefillArgs &a) {
    if (a.gate && !(a.q && (a.mode == MODE_OUTPUT || a.emit_out))) return false;
    return a.act == KDA_DTYPE_BF16 && a.dk == D && a.dv == D;
}

namespace {

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

cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t st) {
    const int units = a.N * a.H * a.seg_count;
    if (units == 0) return cudaSuccess;
    CUtensorMap tq, tk, tv, tg;
    memset(&tq, 0, sizeof(tq)); memset(&tk, 0, sizeof(tk));
    memset(&tv, 0, sizeof(tv)); memset(&tg, 0, sizeof(tg));
    if (a.T_tot > 0) {  // with no tokens no CTA loads anything (and the pointers may be null)
        PFN_cuTensorMapEncodeTiled_v12000 enc = sm100::tensor_map_encoder();
        if (!enc) return cudaErrorNotSupported;
        const void *qp = a.q ? a.q : a.k;  // the transfer pass has no q
        if (!encode_rows(enc, &tq, qp, a.T_tot, a.H, false) ||
            !encode_rows(enc, &tk, a.k, a.T_tot, a.H, false) ||
            !encode_rows(enc, &tv, a.v, a.T_tot, a.H, false) ||
            !encode_rows(enc, &tg, a.g, a.T_tot, a.H, !a.gate))
            return cudaErrorInvalidValue;
    }
    const bool two = prefill_tc_two_chain(a);
    if (a.lead && !(two && a.seg_begin == 0 && a.seg_count == a.Sg && a.Sg >= 2))
        return cudaErrorInvalidValue;  // lead segments exist only in the full two-chain pass
    const dim3 grid(units, a.mode == MODE_TRANSFER && !two && !a.rev ? 2 : 1);
    auto go = [&](auto kernel, int threads) -> cudaError_t {
        cudaError_t e = set_max_dynamic_smem((const void *)kernel, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        return launch_dependent(kernel, grid, dim3(threads), SMEM_BYTES, st, a, tq, tk, tv, tg);
    };
    if (a.gate)
        return two ? go(prefill_tc_kernel<true, 2>, cta_threads(2))
                   : go(prefill_tc_kernel<true, 1>, cta_threads(1));
    if (a.rev) return go(prefill_tc_kernel<false, 1, VAR_ADJOINT>, cta_threads(1));
    if (a.chunk_states) return go(prefill_tc_kernel<false, 1, VAR_CHUNK_STATES>, cta_threads(1));
    return two ? go(prefill_tc_kernel<false, 2>, cta_threads(2))
               : go(prefill_tc_kernel<false, 1>, cta_threads(1));
}

}  // namespace kda
