// dash_bwd.cuh -- the persistent, KV-stationary deterministic attention
// backward kernel for sm_103a, and the tile building blocks it shares with
// the single-tile probe.
//
// One CTA per SM.  A CTA takes tasks (one KV tile, or a symmetric pair of KV
// tiles) either from a static round-robin assignment (shift, symmetric shift)
// or from a global counter in task order (the other schedules).  For each
// pair (KV tile j, Q tile i) of a task:
//
//   S^T  = K_j Q_i^T            (tcgen05, both operands K-major in smem)
//   P^T  = exp(scale S^T - LSE_i)      (masked on the causal diagonal)
//   dV_j += P^T dO_i            (A = P^T from tensor memory, packed bf16)
//   dP^T = V_j dO_i^T
//   dS^T = scale * P^T o (dP^T - delta_i)   (bf16, smem)
//   dK_j += dS^T Q_i            (B = Q MN-major)
//   dQ_i^(j) = dS K_j           (A = dS^T read MN-major, B = K MN-major)
//   dq[tile i] += dQ_i^(j)      (fp32, after waiting for this pair's turn)
//
// The ordered reduction is the one the DASH pages describe: a per-dQ-tile
// counter (the release side is the "safe_signal" counter of the pwwt.cn
// write-up, section 3.1), each contributor waiting until the counter equals
// its rank in the schedule's accumulation order (gist.science DASH summary,
// section 1: a fixed accumulation order makes dQ reproducible).
//
// Warp roles (20 warps, 640 threads, five warpgroups):
//   WG0  warp 0 producer (task dispatch, pair descriptors, TMA loads),
//        warp 1 MMA issuer (one thread) and TMEM owner, warps 2-3 idle;
//   WG1  warps 4-7   dQ drain, TMEM lanes 32*(w%4) + 0..15;
//   WG2  warps 8-11  softmax / dS, Q columns 0..63;
//   WG3  warps 12-15 softmax / dS, Q columns 64..127;
//   WG4  warps 16-19 dQ drain, TMEM lanes 32*(w%4) + 16..31.
// A drain warp owns 16 rows of the dQ tile (a sub-tile): it reads them out
// of tensor memory (16x256b shape), hands the columns back to the MMA issuer,
// waits for the pair's turn on its own sub-tile counter and adds its rows
// into global dq with 64-byte-per-row fp32 vector reductions straight from
// registers.  Nothing but the tensor core reads shared memory in the steady
// state: thread loads from shared memory and TMA stores from it are starved
// while the tensor core streams its operands, so LSE and delta reach the
// softmax warps through global loads and warp shuffles.  The eight
// sub-tiles of a dQ tile carry the same accumulation rank, so the order of
// the additions into every element is the schedule's.
//
// Tensor memory (512 columns): dK [0,D), dV [D,2D), S/P [2D, 2D+128),
// dP [2D+128, 2D+256); dQ aliases dP when D = 128 and has its own 64
// columns when D = 64.  dQ is issued before dK, so the drain warps get it
// one product earlier.
//
// Every wait is bounded (%globaltimer); a wait that runs out records the
// failure in the status word, raises a CTA-wide and a grid-wide abort flag,
// and every role then leaves its loop; the CTA waits for its own TMA loads
// and MMAs to land, frees tensor memory and exits.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "dash_ptx.cuh"
#include "dash_schedule.h"

namespace dash {

constexpr int kThreads = 640;
constexpr int kSubTiles = 8;        // dQ sub-tiles (16 rows each) with their own turn counters
constexpr int kBox = 16384;        // 128 rows x 128 B
constexpr int kNDesc = 8;          // pair-descriptor ring depth
constexpr float kLog2e = 1.4426950408889634f;

enum Role : int { kRoleDrain = 0, kRoleProducer = 1, kRoleMma = 2, kRoleSoftmax = 3 };
// kPartial: the pair touches the partial last tile (S % 128 != 0) in KV or Q.
enum DescFlags : int { kKvFirst = 1, kKvLast = 2, kDiag = 4, kEnd = 8, kPartial = 16 };

// Barrier slots (8 bytes each) at the start of the control area.
enum Bar : int {
    B_DESC_FULL = 0,
    B_DESC_EMPTY = B_DESC_FULL + kNDesc,
    B_KV_FULL = B_DESC_EMPTY + kNDesc,
    B_KV_EMPTY,
    B_Q_FULL,
    B_Q_EMPTY = B_Q_FULL + 2,
    B_DO_FULL = B_Q_EMPTY + 2,
    B_DO_EMPTY = B_DO_FULL + 2,
    B_S_FULL = B_DO_EMPTY + 2,
    B_DP_FULL,
    B_P_READY,
    B_DS_READY,
    B_DS_FREE,
    B_DQ_FULL,
    B_DQ_EMPTY,
    B_ACC_FULL,
    B_ACC_EMPTY,
    B_DRAIN,
    B_COUNT
};

// Control area: barriers [0, 320), descriptors [320, 576), TMEM address
// 576, abort flag 580, cycle counters [584, ...).
constexpr int kCtlBars = 0, kCtlDescs = 320, kCtlTmem = 576, kCtlAbort = 580, kCtlProf = 584;
constexpr int kProfPerRole = 10;
constexpr int kProfSmem = 4 * kProfPerRole + 1;   // + whole-CTA cycles
constexpr int kProfOut = 64;                       // per-CTA entries in the debug buffer
constexpr int kTracePairs = 64;                    // event trace of the first pairs of CTA 0
constexpr int kTraceEvents = 32;
enum TraceEv : int {
    EV_S_ISSUE = 0, EV_DP_ISSUE, EV_DV_ISSUE, EV_DK_ISSUE, EV_DQ_ISSUE,         // MMA issuer
    EV_SM_S_SEEN = 5, EV_SM_P_DONE, EV_SM_DP_SEEN, EV_SM_DS_DONE,               // softmax warp 8
    EV_DR_DQ_SEEN = 10, EV_DR_DQ_EMPTY, EV_DR_TURN, EV_DR_REDS, EV_DR_DONE,     // drain warp 4
    EV_PR_DESC = 22, EV_PR_Q_ISSUED, EV_PR_DO_ISSUED                            // producer
};
static_assert(B_COUNT * 8 <= kCtlDescs, "barrier area");
// multi-slot barriers: every range ends before the next name starts
static_assert(B_DESC_EMPTY == B_DESC_FULL + kNDesc && B_KV_FULL == B_DESC_EMPTY + kNDesc, "descriptor slots");
static_assert(B_Q_EMPTY == B_Q_FULL + 2 && B_DO_FULL == B_Q_EMPTY + 2 && B_DO_EMPTY == B_DO_FULL + 2 &&
                  B_S_FULL == B_DO_EMPTY + 2, "stage slots");
static_assert(kCtlProf + kProfSmem * 8 <= 1024, "control area");

struct PairDesc {
    int b, hq, hkv, q, kv, flags, rank, pad;
};
static_assert(sizeof(PairDesc) * kNDesc <= kCtlTmem - kCtlDescs, "descriptor ring area");

template <int D>
struct Cfg {
    static constexpr int kTile = D * 128 * 2;         // 128 x D bf16
    static constexpr int kNBox = D / 64;
    static constexpr int kQStages = 2;
    // Two dO stages at both head dimensions (225 KB of shared memory at
    // D = 128; one stage measured 0.5% slower on the current kernel).
    static constexpr int kDoStages = 2;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + kTile;
    static constexpr int OFF_Q = OFF_V + kTile;
    static constexpr int OFF_DO = OFF_Q + kQStages * kTile;
    static constexpr int OFF_DS = OFF_DO + kDoStages * kTile;
    static constexpr int OFF_CTL = OFF_DS + 2 * kBox;
    static constexpr int kSmem = OFF_CTL + 1024;
    static constexpr uint32_t COL_DK = 0;
    static constexpr uint32_t COL_DV = D;
    static constexpr uint32_t COL_S = 2 * D;
    static constexpr uint32_t COL_DP = 2 * D + 128;
    static constexpr bool kDqAlias = (D == 128);
    static constexpr uint32_t COL_DQ = kDqAlias ? COL_DP : 2 * D + 256;
    static constexpr uint32_t kQBytes = kTile;
    static constexpr uint32_t kDoBytes = kTile;
    static constexpr uint32_t kKvBytes = 2 * kTile;
    static_assert(kSmem <= 232448, "shared memory budget");
    static_assert(COL_DQ + D <= 512, "tensor memory budget");
};

// Register split of the five warpgroups (setmaxnreg); the launch must grant
// kRegsLaunch registers per thread so that the split fits the block's pool.
// At D = 128 the producer / MMA warpgroup gets 80: at 64 its spilled values
// are reloaded through the load/store path that the drain warps' reductions
// keep busy, which delays every MMA issue (measured: 8% on the unordered
// kernel); the softmax warps give up the 8 registers.
constexpr int kRegsLaunch = 96;
template <int D>
struct Regs {
    static constexpr int kCtl = (D == 128) ? 80 : 64;
    static constexpr int kDrain = (D == 128) ? 96 : 80;
    static constexpr int kSoftmax = (D == 128) ? 104 : 120;
    static_assert(128 * kCtl + 256 * kDrain + 256 * kSoftmax <= kThreads * kRegsLaunch, "register split");
};

struct BwdParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_do;   // 3D [heads][S][D] bf16, box 64 x 128 x 1, SWIZZLE_128B
    const float* lse;
    const float* delta;
    float* dq;
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    const uint16_t* ranks;                  // static schedules: [B*Hq*n][n]
    int* sem;                               // [B*Hq*n][kSubTiles] accumulation counters
    int* logcnt;                            // [B*Hq*n] order-log cursors
    int* task_counter;                      // dynamic dispatch
    int* status;                            // [8]: code, info[4]
    int* abort_flag;                        // grid-wide abort
    int32_t* order_log;                     // debug, may be null
    float* partials;                        // debug, may be null
    const int32_t* cta_perm;                // debug, may be null
    const int64_t* delay_ns;                // debug, may be null
    unsigned long long* prof;               // debug, may be null: [P][kProfOut] cycle counters
    unsigned long long* trace;              // debug, may be null: [kTracePairs][kTraceEvents] clock64 of CTA 0
    unsigned long long timeout_ns;
    long long ntasks;
    int B, Hq, Hkv, S, n, G, causal, sched, P;
    float scale, scale_log2e;
    int window;                             // causal sliding window in tokens (0 = none)
    int win;                                // its tile diagonals (band_tiles), 0 = none
    int Skv;                                // key/value length (S is the query length)
    int nk;                                 // key/value tiles when they differ from n, else 0
    int nkv;                                // key/value tiles per head (n or nk)
    // Grouped-query heads.  Hkv and G above describe the tasks (with one task
    // per query head they are Hq and 1); kvh and kvg are the key/value heads
    // of the tensors and the query heads per key/value head.
    int kvh, kvg;
    // One task per query head: fp32 [B, Hq, Skv, D] dK / dV of each query
    // head, summed over the group afterwards; null: bf16 dk / dv directly.
    float* part_dk;
    float* part_dv;
};

// ------------------------------------------------------------------ MMA issue
// All operand addresses are shared-window byte addresses of 1024-aligned
// 128-row boxes.  One thread issues.  kUnroll: the backward keeps the K-step
// loops rolled (1): with its five products (and their call sites) unrolled,
// its code no longer fits the SM's instruction cache (about 26% of the
// requests missed and instruction fetch was the second-largest stall), and
// the extra issue cycles hide behind each 512-cycle product.  The forward,
// whose code fits, unrolls them.

template <int D, int kUnroll = 1>
__device__ __forceinline__ void issue_s(uint32_t d_tmem, uint32_t sA, uint32_t sB) {
    // [128 x 128] = A[128 x D] * B[128 x D]^T, both K-major
    constexpr uint32_t idesc = ptx::idesc_bf16(128, 128, 0, 0);
#pragma unroll kUnroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
        ptx::mma_ss(d_tmem, ptx::sdesc(sA + off, 16, 1024), ptx::sdesc(sB + off, 16, 1024), idesc,
                    kk > 0);
    }
}

template <int D, int kUnroll = 1>
__device__ __forceinline__ void issue_dv(uint32_t d_tmem, uint32_t p_tmem, uint32_t sDo,
                                         uint32_t acc) {
    // dV[128 x D] (+)= P^T[128 x 128] (tmem, K-major) * dO[128 x D] (MN-major)
    constexpr uint32_t idesc = ptx::idesc_bf16(128, D, 0, 1);
#pragma unroll kUnroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t a = p_tmem + (kk >> 2) * 64 + (kk & 3) * 8;
        ptx::mma_ts(d_tmem, a, ptx::sdesc(sDo + kk * 2048, kBox, 1024), idesc, acc | (kk > 0));
    }
}

template <int D>
__device__ __forceinline__ void issue_dk(uint32_t d_tmem, uint32_t sDsT, uint32_t sQ, uint32_t acc) {
    // dK[128 x D] (+)= dS^T[128 x 128] (K-major) * Q[128 x D] (MN-major)
    constexpr uint32_t idesc = ptx::idesc_bf16(128, D, 0, 1);
#pragma unroll 1
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t aoff = (kk >> 2) * kBox + (kk & 3) * 32;
        ptx::mma_ss(d_tmem, ptx::sdesc(sDsT + aoff, 16, 1024), ptx::sdesc(sQ + kk * 2048, kBox, 1024),
                    idesc, acc | (kk > 0));
    }
}

template <int D>
__device__ __forceinline__ void issue_dq(uint32_t d_tmem, uint32_t sDsT, uint32_t sK) {
    // dQ[128 x D] = dS[128 x 128] (dS^T read MN-major) * K[128 x D] (MN-major)
    constexpr uint32_t idesc = ptx::idesc_bf16(128, D, 1, 1);
#pragma unroll 1
    for (int kk = 0; kk < 8; ++kk) {
        ptx::mma_ss(d_tmem, ptx::sdesc(sDsT + kk * 2048, kBox, 1024),
                    ptx::sdesc(sK + kk * 2048, kBox, 1024), idesc, kk > 0);
    }
}

// ------------------------------------------------------------ softmax / dS
// Executed by one warp that owns TMEM lanes [lane_base, lane_base+32) (KV rows)
// and Q columns [c0, c0+64) of the pair.  Lane l holds the per-column
// statistics of columns c0 + l (x_a) and c0 + 32 + l (x_b); column k's value
// reaches every lane through a shuffle.

// P for 64 columns: reads S^T, writes P (fp32, registers) and the packed
// bf16 P^T back into tensor memory at columns [c0, c0+32) of its own
// 64-column span (so the MMA reads it as a K-major A operand).  lse2_* are
// LSE * log2(e).  Works in 32-column halves to keep few registers live.
// P is zero where row > column on a diagonal tile (`diag`) and, when `mask`
// is set, where row >= lim_row (keys past S), column >= lim_col (queries
// past S) or column - row >= wlim (query - key at or beyond a sliding
// window: wlim = window - 128 * (q tile - kv tile)).  kBranchMask: apply the masks in a branch taken only by masked
// pairs (needed for partial tiles; measured faster at D = 64); otherwise the
// diagonal is applied with a per-element select (measured faster at D = 128
// and then lim_row, lim_col must be >= 128).
template <bool kBranchMask>
__device__ __forceinline__ void softmax_64(uint32_t tmem_s_lane, int c0, float lse2_a, float lse2_b,
                                           float scale_log2e, bool mask, bool diag, int row, int lim_row,
                                           int lim_col, int wlim, float (&P)[64]) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t r[32];
        ptx::tmem_ld32(tmem_s_lane + c0 + 32 * h, r);
        ptx::tmem_ld_wait();
        // -LSE of the columns (negated once, exactly), broadcast two at a
        // time; the exponent scale*log2e*S - LSE as one packed fma per pair
        const float nsrc = -(h ? lse2_b : lse2_a);
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
            const ptx::f2 nl{__shfl_sync(0xffffffffu, nsrc, k), __shfl_sync(0xffffffffu, nsrc, k + 1)};
            const ptx::f2 y = ptx::fma2({__uint_as_float(r[k]), __uint_as_float(r[k + 1])}, {scale_log2e, scale_log2e}, nl);
            const float x0 = ptx::ex2(y.x), x1 = ptx::ex2(y.y);
            P[32 * h + k] = (!kBranchMask && diag && row > c0 + 32 * h + k) ? 0.f : x0;
            P[32 * h + k + 1] = (!kBranchMask && diag && row > c0 + 32 * h + k + 1) ? 0.f : x1;
        }
        if (kBranchMask && mask) {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const int col = c0 + 32 * h + k;
                if ((diag && row > col) || row >= lim_row || col >= lim_col || col - row >= wlim) P[32 * h + k] = 0.f;
            }
        }
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn(P[32 * h + 2 * k], P[32 * h + 2 * k + 1]);
            pk[k] = *reinterpret_cast<uint32_t*>(&h2);
        }
        // packed columns [c0 + 16h, c0 + 16h + 16): S values there were already read
        ptx::tmem_st16(tmem_s_lane + c0 + 16 * h, pk);
    }
    ptx::tmem_st_wait();
}

// dS^T = scale * P o (dP^T - delta) for 64 columns, written as bf16 into row
// `row` of the K-major swizzled box `box` (box c0/64 of dS^T), 16 columns
// (two 16-byte chunks) at a time.
__device__ __forceinline__ void ds_64(uint32_t tmem_dp_lane, int c0, float delta_a, float delta_b, float scale,
                                      const float (&P)[64], uint8_t* box, int row) {
    uint8_t* rp = box + row * 128;
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t r[16];
        ptx::tmem_ld16(tmem_dp_lane + c0 + 16 * q4, r);
        ptx::tmem_ld_wait();
        const float dsrc = (q4 < 2) ? delta_a : delta_b;
        uint32_t pk[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int a = 16 * q4 + 2 * k;
            const ptx::f2 e{__shfl_sync(0xffffffffu, dsrc, (a & 31)), __shfl_sync(0xffffffffu, dsrc, (a & 31) + 1)};
            // (P * (dP - delta)) * scale, in that order, two columns per instruction
            const ptx::f2 d = ptx::mul2(ptx::mul2({P[a], P[a + 1]}, ptx::sub2({__uint_as_float(r[2 * k]), __uint_as_float(r[2 * k + 1])}, e)),
                                        {scale, scale});
            __nv_bfloat162 h2 = __floats2bfloat162_rn(d.x, d.y);
            pk[k] = *reinterpret_cast<uint32_t*>(&h2);
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int chunk = 2 * q4 + c;   // 16-byte chunk (8 columns) within the 128-byte row
            *reinterpret_cast<uint4*>(rp + ((chunk ^ (row & 7)) << 4)) =
                make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
    }
}

}  // namespace dash
