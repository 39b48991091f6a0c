// dash_fwd.cu -- the attention forward pass (O and the log-sum-exp LSE) on
// sm_103a, producing exactly the inputs the deterministic backward consumes,
// so that a training step runs on one GPU without another library.
//
// One CTA per 128-row Q tile (head-major over the grid, so that resident
// CTAs share K/V in L2; within a head, causal tiles longest first).  For KV tiles j = 0 .. (causal ? i : n-1):
//
//   S = Q K_j^T                 (tcgen05, both operands K-major, two TMEM buffers)
//   m = running row max of scale*log2e*S, l = running row sum of
//   P = exp2(scale*log2e*S - m) (zero right of the diagonal on the diagonal tile)
//   O += P V_j                  (A = P packed bf16 in tensor memory, B = V MN-major)
//
// The row max is only raised (and O, l rescaled) when a row's new maximum
// exceeds the reference by more than 8 (a factor 2^8), which keeps P <= 256
// and makes rescaling rare; the final O / l and LSE = ln2 * (m + log2 l) do
// not depend on when it happens.  No CTA reads another's results, so the
// outputs are bitwise reproducible.  This is the textbook softmax attention
// that the gist.science DASH summary (section 1) takes as the forward pass
// whose backward it schedules.
//
// Warps: 0 producer (TMA: Q once, K and V double-buffered; a K stage is
// released as soon as its S product completes, a V stage after its PV), 1 MMA
// issuer and TMEM owner, 2-3 idle, 4-7 softmax and epilogue (one Q row per
// thread, TMEM lanes 32*(w%4) ..).  Tensor memory: O [0, D), S/P buffers at columns
// 256 and 384.  Every wait is bounded (%globaltimer); on expiry the status
// word records DASH_ERR_TIMEOUT and the CTA drains and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "dash_bwd.cuh"
#include "dash_internal.h"

namespace dash {

namespace {

struct FwdParams {
    CUtensorMap tm_q, tm_k, tm_v;   // 3D [heads][S][D] bf16, box 64 x 128 x 1, SWIZZLE_128B
    __nv_bfloat16* o;
    float* lse;
    int* status;                    // [8]: code, info[4]
    unsigned long long timeout_ns;
    int B, Hq, Hkv, S, n, G, causal;
    float scale_log2e;
    int window;                     // causal sliding window in tokens (0 = none)
    int win;                        // its tile diagonals (band_tiles), 0 = none
    int Skv, nkv;                   // key/value length and tiles (S, n: the query's)
};

enum FwdBar : int {
    F_Q_FULL = 0,
    F_K_FULL = 1,      // 2 stages
    F_V_FULL = 3,      // 2 stages
    F_K_EMPTY = 5,     // 2 stages: K stage free once S(j) is done
    F_S_FULL = 7,      // 2 buffers
    F_P_READY = 9,     // 2 buffers
    F_O_DONE = 11,
    F_DRAIN = 12,
    F_V_EMPTY = 13,     // 2 stages: V stage free once PV(j) is done
    F_COUNT = 15
};

template <int D>
struct FwdCfg {
    static constexpr int kTile = D * 128 * 2;
    static constexpr int kNBox = D / 64;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = kTile;                 // 2 stages
    static constexpr int OFF_V = OFF_K + 2 * kTile;     // 2 stages
    static constexpr int OFF_CTL = OFF_V + 2 * kTile;
    // at least ~117 KB so that one CTA (and its 512 TMEM columns) holds an SM
    static constexpr int kSmem = (OFF_CTL + 256 > 120000) ? OFF_CTL + 256 : 120000;
    static constexpr uint32_t COL_O = 0;
    static constexpr uint32_t COL_S = 256;              // buffers at 256 and 384
    static_assert(D <= 256, "tensor memory budget");
};

constexpr int kCtlTmemF = 128, kCtlAbortF = 132;
constexpr float kLn2 = 0.69314718055994531f;

struct FwdWait {
    volatile int* abort_smem;
    int* status;
    unsigned long long timeout;
};

__device__ __noinline__ void fwd_timeout(const FwdWait& w, int role, int i0) {
    if (atomicCAS(w.status, 0, -4) == 0) {   // DASH_ERR_TIMEOUT, first failure wins
        w.status[1] = i0;
        w.status[2] = (int)blockIdx.x;
        w.status[3] = -1;
        w.status[4] = role;
        __threadfence();
    }
    *w.abort_smem = 1;
}

__device__ bool fwait1(uint32_t bar, uint32_t parity, const FwdWait& w, int role, int i0) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (*w.abort_smem) return false;
        if (ptx::globaltimer() - t0 > w.timeout) {
            fwd_timeout(w, role, i0);
            return false;
        }
    }
    return true;
}

// Every lane's own poll after lane 0 saw the phase complete: normally no
// iteration at all; bounded all the same (role + 8 in the status if it runs out).
__device__ __noinline__ int fwait_lanes(uint32_t bar, uint32_t parity, const FwdWait& w, int role, int i0) {
    for (int n = 0; !ptx::mbar_try_wait(bar, parity); ++n) {
        if (n == (1 << 24)) {
            fwd_timeout(w, role + 8, i0);
            return 0;
        }
    }
    return 1;
}

// Whole warp: lane 0 polls, then every lane observes the phase (acquire).
__device__ __forceinline__ bool fwaitw(uint32_t bar, uint32_t parity, const FwdWait& w, int role, int i0) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = fwait1(bar, parity, w, role, i0) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok && !ptx::mbar_try_wait(bar, parity)) ok = fwait_lanes(bar, parity, w, role, i0);
    return __all_sync(0xffffffffu, ok != 0);
}

// kMasked: compiled for a partial last tile (S % 128 != 0) or a sliding
// window (their masks and guards); the instantiation for whole tiles and
// plain masks carries none of that code.
template <int D, bool kMasked>
__global__ void __launch_bounds__(256, 1) dash_fwd_kernel(const __grid_constant__ FwdParams p) {
    using C = FwdCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint8_t* ctl = smem + C::OFF_CTL;
    const uint32_t bar0 = ptx::smem_u32(ctl);
    auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(ctl + kCtlTmemF);
    volatile int* abort_smem = reinterpret_cast<volatile int*>(ctl + kCtlAbortF);
    const FwdWait fw{abort_smem, p.status, p.timeout_ns};
    const uint32_t sbase = ptx::smem_u32(smem);

    // work item: head-major, so that the CTAs resident together share their
    // heads' K/V in L2 (query heads of one group are adjacent); within a head
    // the Q tiles run in descending order (longest causal rows first)
    const int qt = p.n - 1 - (int)(blockIdx.x % p.n);
    const int bh = (int)(blockIdx.x / p.n);
    const int b = bh / p.Hq, hq = bh % p.Hq, hkv = hq / p.G;
    // KV tiles j0 .. j0 + nkv - 1 (a window starts the range at its far edge);
    // loops count j from 0 and address the tile j0 + j
    const int j0 = (p.causal && p.win && qt >= p.win) ? qt - p.win + 1 : 0;
    const int nkv = p.causal ? qt - j0 + 1 : p.nkv;
    const int qrow = (b * p.Hq + hq) * p.S + qt * 128;   // first row of this tile in o / lse
    const int hqi = b * p.Hq + hq, hki = b * p.Hkv + hkv;  // head indices of the 3-D tensor maps

    if (threadIdx.x == 0) {
        *abort_smem = (sbase & 1023u) ? 1 : 0;
        if (sbase & 1023u) fwd_timeout(fw, -1, (int)sbase);
        ptx::mbar_init(BAR(F_Q_FULL), 1);
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(BAR(F_K_FULL + s), 1);
            ptx::mbar_init(BAR(F_V_FULL + s), 1);
            ptx::mbar_init(BAR(F_K_EMPTY + s), 1);
            ptx::mbar_init(BAR(F_V_EMPTY + s), 1);
            ptx::mbar_init(BAR(F_S_FULL + s), 1);
            ptx::mbar_init(BAR(F_P_READY + s), 4);
        }
        ptx::mbar_init(BAR(F_O_DONE), 1);
        ptx::mbar_init(BAR(F_DRAIN), 1);
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32((const void*)tmem_slot), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ================================================== producer
        if (lane == 0 && !*abort_smem) {
            ptx::prefetch_tensormap(&p.tm_q);
            ptx::prefetch_tensormap(&p.tm_k);
            ptx::prefetch_tensormap(&p.tm_v);
            ptx::mbar_arrive_expect_tx(BAR(F_Q_FULL), C::kTile);
#pragma unroll
            for (int bx = 0; bx < C::kNBox; ++bx)
                ptx::tma_load_3d(sbase + C::OFF_Q + bx * kBox, &p.tm_q, 64 * bx, qt * 128, hqi, BAR(F_Q_FULL));
            int issued = 0;
            for (int j = 0; j < nkv; ++j) {
                const int st = j & 1;
                if (j >= 2 && !fwait1(BAR(F_K_EMPTY + st), (uint32_t)((j / 2 - 1) & 1), fw, 1, j)) break;
                ptx::mbar_arrive_expect_tx(BAR(F_K_FULL + st), C::kTile);
#pragma unroll
                for (int bx = 0; bx < C::kNBox; ++bx)
                    ptx::tma_load_3d(sbase + C::OFF_K + st * C::kTile + bx * kBox, &p.tm_k, 64 * bx, (j0 + j) * 128, hki,
                                     BAR(F_K_FULL + st));
                if (j >= 2 && !fwait1(BAR(F_V_EMPTY + st), (uint32_t)((j / 2 - 1) & 1), fw, 1, j)) break;
                ptx::mbar_arrive_expect_tx(BAR(F_V_FULL + st), C::kTile);
#pragma unroll
                for (int bx = 0; bx < C::kNBox; ++bx)
                    ptx::tma_load_3d(sbase + C::OFF_V + st * C::kTile + bx * kBox, &p.tm_v, 64 * bx, (j0 + j) * 128, hki,
                                     BAR(F_V_FULL + st));
                issued = j + 1;
            }
            // let every issued load land before the CTA can exit (bounded)
            const uint64_t t0 = ptx::globaltimer();
            auto drain = [&](uint32_t bar, uint32_t parity) {
                while (!ptx::mbar_try_wait(bar, parity) && ptx::globaltimer() - t0 < 100000000ull) {
                }
            };
            drain(BAR(F_Q_FULL), 0);
            for (int j = (issued > 2 ? issued - 2 : 0); j < issued; ++j) {
                drain(BAR(F_K_FULL + (j & 1)), (uint32_t)((j / 2) & 1));
                drain(BAR(F_V_FULL + (j & 1)), (uint32_t)((j / 2) & 1));
            }
        }
    } else if (warp == 1) {
        // ================================================== MMA issuer
        if (lane == 0 && !*abort_smem) {
            const uint32_t sQ = sbase + C::OFF_Q;
            auto tS = [&](int j) { return tmem + C::COL_S + 128u * (uint32_t)(j & 1); };
            auto sK = [&](int j) { return sbase + C::OFF_K + (uint32_t)(j & 1) * C::kTile; };
            auto sV = [&](int j) { return sbase + C::OFF_V + (uint32_t)(j & 1) * C::kTile; };
            bool ok = fwait1(BAR(F_Q_FULL), 0, fw, 2, 0) && fwait1(BAR(F_K_FULL), 0, fw, 2, 0);
            if (ok) {
                ptx::tc_fence_after();
                issue_s<D, D / 16>(tS(0), sQ, sK(0));
                ptx::tc_commit(BAR(F_S_FULL));
                ptx::tc_commit(BAR(F_K_EMPTY));
            }
            for (int j = 0; ok && j < nkv; ++j) {
                if (j + 1 < nkv) {
                    // S(j+1) overwrites the buffer PV(j-1) read; MMAs run in issue order
                    if (!fwait1(BAR(F_K_FULL + ((j + 1) & 1)), (uint32_t)(((j + 1) / 2) & 1), fw, 2, j)) break;
                    ptx::tc_fence_after();
                    issue_s<D, D / 16>(tS(j + 1), sQ, sK(j + 1));
                    ptx::tc_commit(BAR(F_S_FULL + ((j + 1) & 1)));
                    ptx::tc_commit(BAR(F_K_EMPTY + ((j + 1) & 1)));
                }
                if (!fwait1(BAR(F_P_READY + (j & 1)), (uint32_t)((j / 2) & 1), fw, 2, j)) break;
                if (!fwait1(BAR(F_V_FULL + (j & 1)), (uint32_t)((j / 2) & 1), fw, 2, j)) break;
                ptx::tc_fence_after();
                issue_dv<D, 8>(tmem + C::COL_O, tS(j), sV(j), j > 0 ? 1u : 0u);   // O (+)= P V_j
                ptx::tc_commit(BAR(F_V_EMPTY + (j & 1)));
                ptx::tc_commit(BAR(F_O_DONE));
            }
            // wait for every issued MMA before tensor memory can be freed
            ptx::tc_commit(BAR(F_DRAIN));
            const uint64_t t0 = ptx::globaltimer();
            while (!ptx::mbar_try_wait(BAR(F_DRAIN), 0) && ptx::globaltimer() - t0 < 100000000ull) {
            }
        }
    } else if (warp >= 4) {
        // ================================================== softmax + epilogue (one Q row per thread)
        const int sub = warp & 3;
        const int row = 32 * sub + lane;
        const uint32_t lane_off = (uint32_t)(32 * sub) << 16;
        const float c = p.scale_log2e;
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nkv; ++j) {
            const int buf = j & 1;
            if (!fwaitw(BAR(F_S_FULL + buf), (uint32_t)((j / 2) & 1), fw, 3, j)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t ts = tmem + lane_off + C::COL_S + 128u * (uint32_t)buf;
            float x[128];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                uint32_t r[32];
                ptx::tmem_ld32(ts + 32 * h, r);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 32; ++k) x[32 * h + k] = __uint_as_float(r[k]);   // raw scores
            }
            const int jt = j0 + j;   // the KV tile
            if (p.causal && jt == qt) {   // diagonal tile: key k visible to query row iff k <= row
#pragma unroll
                for (int k = 0; k < 128; ++k)
                    if (k > row) x[k] = -INFINITY;
            }
            if (kMasked && p.window && 128 * (qt - jt) + 127 >= p.window) {   // the window's far edge
                const int wlim = p.window - 128 * (qt - jt);   // key k hidden from row iff row - k >= wlim
#pragma unroll
                for (int k = 0; k < 128; ++k)
                    if (row - k >= wlim) x[k] = -INFINITY;
            }
            if (kMasked && jt == p.nkv - 1 && (p.Skv & 127)) {   // keys past S_kv of the partial last tile
                const int lim = p.Skv - jt * 128;
#pragma unroll
                for (int k = 0; k < 128; ++k)
                    if (k >= lim) x[k] = -INFINITY;
            }
            // row max and (below) row sum over 8 interleaved partials: short
            // dependency chains, and a fixed order of the additions
            float part[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) part[i] = x[i];
#pragma unroll
            for (int k = 8; k < 128; ++k) part[k & 7] = fmaxf(part[k & 7], x[k]);
            const float mx = c * fmaxf(fmaxf(fmaxf(part[0], part[1]), fmaxf(part[2], part[3])),
                                       fmaxf(fmaxf(part[4], part[5]), fmaxf(part[6], part[7])));
            // raise the reference maximum only when some row of the warp grew by > 2^8
            const bool raise = __any_sync(0xffffffffu, mx > m_ref + 8.f);
            float alpha = 1.f;
            if (raise) {
                const float m_new = fmaxf(m_ref, mx);
                // 0 once the row has a first visible key (m_ref = -inf); a row
                // with none yet (the window's far edge) stays at -inf, alpha 1
                alpha = (m_new == -INFINITY) ? 1.f : ptx::ex2(m_ref - m_new);
                m_ref = m_new;
            }
            const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;   // P = 0, not NaN, for such a row
#pragma unroll
            for (int i = 0; i < 8; ++i) part[i] = 0.f;
            // the exponents and the partial sums two columns per instruction
            // (packed fp32 pairs round each lane as the scalar ops would)
#pragma unroll
            for (int k = 0; k < 128; k += 2) {
                const ptx::f2 y = ptx::fma2({x[k], x[k + 1]}, {c, c}, {-m_use, -m_use});
                x[k] = ptx::ex2(y.x);
                x[k + 1] = ptx::ex2(y.y);
                const ptx::f2 s = ptx::add2({part[k & 7], part[(k + 1) & 7]}, {x[k], x[k + 1]});
                part[k & 7] = s.x;
                part[(k + 1) & 7] = s.y;
            }
            const float rs = ((part[0] + part[1]) + (part[2] + part[3])) + ((part[4] + part[5]) + (part[6] + part[7]));
            l = l * alpha + rs;
            if (raise && j > 0) {
                // O holds the sum through PV(j-1): wait for it, then rescale in place
                // (S(j) was committed after PV(j-2), so phase j-1 is the next one)
                if (!fwaitw(BAR(F_O_DONE), (uint32_t)((j - 1) & 1), fw, 3, j)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t r[32];
                    ptx::tmem_ld32(tmem + lane_off + C::COL_O + 32 * cc, r);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha);
                    ptx::tmem_st32(tmem + lane_off + C::COL_O + 32 * cc, r);
                }
            }
            // packed bf16 P: keys [0,64) -> columns [0,32), keys [64,128) -> [64,96)
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t pk[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    __nv_bfloat162 h2 = __floats2bfloat162_rn(x[32 * q4 + 2 * k], x[32 * q4 + 2 * k + 1]);
                    pk[k] = *reinterpret_cast<uint32_t*>(&h2);
                }
                ptx::tmem_st16(ts + 64 * (q4 >> 1) + 16 * (q4 & 1), pk);
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(BAR(F_P_READY + buf));
        }
        // O is complete once every MMA is: F_DRAIN, committed once after the
        // last one, has a single phase, so this wait cannot alias (a wait on
        // O_DONE could see its parity pass on between two lanes' polls)
        if (ok) ok = fwaitw(BAR(F_DRAIN), 0u, fw, 3, nkv);
        if (ok) {
            ptx::tc_fence_after();
            const bool row_ok = !kMasked || qt * 128 + row < p.S;   // rows past S are not stored (loads stay warp-wide)
            const float inv = 1.f / l;
            __nv_bfloat16* orow = p.o + ((size_t)qrow + row) * D;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t r[32];
                ptx::tmem_ld32(tmem + lane_off + C::COL_O + 32 * cc, r);
                ptx::tmem_ld_wait();
                uint32_t pk[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    __nv_bfloat162 h2 =
                        __floats2bfloat162_rn(__uint_as_float(r[2 * k]) * inv, __uint_as_float(r[2 * k + 1]) * inv);
                    pk[k] = *reinterpret_cast<uint32_t*>(&h2);
                }
                if (row_ok) {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        *reinterpret_cast<uint4*>(orow + 32 * cc + 8 * e) =
                            make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                }
            }
            if (row_ok) p.lse[qrow + row] = (m_ref + log2f(l)) * kLn2;
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

template <int D, bool kMasked>
int launch_fwd_t(const FwdParams& prm, int grid, cudaStream_t stream) {
    static bool attr_done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -2;
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(dash_fwd_kernel<D, kMasked>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 FwdCfg<D>::kSmem) != cudaSuccess)
            return -2;
        attr_done[dev] = true;
    }
    dash_fwd_kernel<D, kMasked><<<grid, 256, FwdCfg<D>::kSmem, stream>>>(prm);
    return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

}  // namespace

int launch_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int* status, int B, int Hq,
               int Hkv, int S, int D, int causal, int window, unsigned long long timeout_ns, cudaStream_t stream,
               int Skv) {
    if (Skv == 0) Skv = S;
    FwdParams prm;
    if (make_tmap_3d(&prm.tm_q, q, (long long)B * Hq, S, D) || make_tmap_3d(&prm.tm_k, k, (long long)B * Hkv, Skv, D) ||
        make_tmap_3d(&prm.tm_v, v, (long long)B * Hkv, Skv, D))
        return -2;
    prm.o = (__nv_bfloat16*)o;
    prm.lse = lse;
    prm.status = status;
    prm.timeout_ns = timeout_ns;
    prm.B = B;
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.S = S;
    prm.n = (S + 127) / 128;   // the last tile may be partial
    prm.G = Hq / Hkv;
    prm.causal = causal;
    prm.scale_log2e = (1.0f / sqrtf((float)D)) * kLog2e;
    prm.window = window;
    prm.win = window ? band_tiles(window) : 0;
    prm.Skv = Skv;
    prm.nkv = (Skv + 127) / 128;
    const long long grid = (long long)B * Hq * ((S + 127) / 128);
    if (grid <= 0 || grid > 0x7fffffffll) return -1;
    if ((S % 128) || (Skv % 128) || window)
        return D == 64 ? launch_fwd_t<64, true>(prm, (int)grid, stream) : launch_fwd_t<128, true>(prm, (int)grid, stream);
    return D == 64 ? launch_fwd_t<64, false>(prm, (int)grid, stream) : launch_fwd_t<128, false>(prm, (int)grid, stream);
}

}  // namespace dash
