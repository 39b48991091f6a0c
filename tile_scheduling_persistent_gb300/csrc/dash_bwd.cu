// dash_bwd.cu -- the persistent deterministic attention backward kernel
// (see dash_bwd.cuh for the design) and its launcher.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dash_bwd.cuh"
#include "dash_internal.h"

namespace dash {

namespace {

struct Ctl {
    volatile int* abort_smem;
    int* status;
    int* abort_global;
    unsigned long long timeout;
    unsigned long long* prof;   // per-CTA cycle counters in shared memory, or null
    uint32_t suspend_ns;        // mbarrier waits: suspend-time hint (0 = plain polls)
    int poll_ns;                // accumulation-turn polls: sleep between two reads
};

// Cycle counters (debug): slot = role * kProfPerRole + site.  One thread per
// role records: the producer, MMA and reduce-issuer lanes, warp 0 lane 0 of
// the drain warps and warp 8 lane 0 of the softmax warps.
__device__ __forceinline__ void prof_add(const Ctl& c, int role, int site, unsigned long long t0) {
    if (c.prof) c.prof[role * kProfPerRole + site] += clock64() - t0;
}

// Event trace (debug instantiation only): clock64 of CTA 0 for the first pairs.
template <bool kProf>
__device__ __forceinline__ void trace_ev(const BwdParams& p, long long pair, int ev) {
    if (kProf && p.trace && blockIdx.x == 0 && pair >= 0 && pair < kTracePairs)
        p.trace[pair * kTraceEvents + ev] = clock64();
}

__device__ __noinline__ void report_timeout(const Ctl& c, int role, int i0, int i1, int i2) {
    if (atomicCAS(c.status, 0, -4) == 0) {   // DASH_ERR_TIMEOUT, first failure wins
        c.status[1] = i0;
        c.status[2] = i1;
        c.status[3] = i2;
        c.status[4] = role;
        __threadfence();
    }
    *c.abort_smem = 1;
    atomicExch(c.abort_global, 1);
}

// Single-thread bounded wait; `site` names the wait in the cycle counters.
__device__ __forceinline__ bool wait1(uint32_t bar, uint32_t parity, const Ctl& c, int role, int i0, int site) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const unsigned long long c0 = clock64();
    const uint64_t t0 = ptx::globaltimer();
    while (!(c.suspend_ns ? ptx::mbar_try_wait_hint(bar, parity, c.suspend_ns) : ptx::mbar_try_wait(bar, parity))) {
        if (*c.abort_smem) return false;
        if (ptx::globaltimer() - t0 > c.timeout) {
            report_timeout(c, role, i0, site, (int)bar);
            return false;
        }
    }
    prof_add(c, role, site, c0);
    return true;
}

// Whole-warp bounded wait with a warp-uniform outcome: lane 0 polls (its
// try_wait acquires the phase), the outcome is broadcast, and the warp
// barrier orders every other lane's later accesses after lane 0's acquire.
// kFast: first one try_wait by every lane and a vote, which returns at once
// when the phase has already completed (one shared-memory round trip instead
// of two); the polled path only when it has not.
template <bool kFast = false>
__device__ __forceinline__ bool waitw(uint32_t bar, uint32_t parity, const Ctl& c, int role, int i0, int site) {
    if (kFast && __all_sync(0xffffffffu, ptx::mbar_try_wait(bar, parity))) return true;
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = wait1(bar, parity, c, role, i0, site) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

__device__ __forceinline__ int64_t next_task(const BwdParams& p, int slot, int& w) {
    if (is_static(p.sched)) {
        const int64_t k = (int64_t)slot + (int64_t)w * p.P;
        ++w;
        return k;
    }
    return (int64_t)atomicAdd(p.task_counter, 1);
}

// Spin until an accumulation counter equals `rank` (acquire).
__device__ bool wait_turn(const BwdParams& p, const Ctl& c, volatile int* abort_smem, int* sem, int rank, int head,
                          int qtile) {
    if (ptx::ld_acquire(sem) == rank) return true;
    const uint64_t t0 = ptx::globaltimer();
    int spins = 0;
    for (;;) {
        if (ptx::ld_acquire(sem) == rank) return true;
        if ((++spins & 63) == 0) {
            if (ptx::ld_volatile(p.abort_flag) || *abort_smem) return false;
            if (ptx::globaltimer() - t0 > c.timeout) {
                report_timeout(c, kRoleDrain, head, qtile, rank);
                return false;
            }
        }
        __nanosleep(c.poll_ns);
    }
}

}  // namespace

// kMasked: compiled for a partial last tile (S % 128 != 0) or a sliding
// window (their masks and guards); the instantiation for whole tiles and
// plain masks carries none of that code.
template <int D, bool kProf, bool kMasked>
__global__ void __launch_bounds__(kThreads, 1) dash_bwd_kernel(const __grid_constant__ BwdParams p) {
    using C = Cfg<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int wg = warp >> 2;

    uint8_t* ctl = smem + C::OFF_CTL;
    const uint32_t bar0 = ptx::smem_u32(ctl + kCtlBars);
    auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
    PairDesc* descs = reinterpret_cast<PairDesc*>(ctl + kCtlDescs);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(ctl + kCtlTmem);
    volatile int* abort_smem = reinterpret_cast<volatile int*>(ctl + kCtlAbort);
    unsigned long long* prof_smem = reinterpret_cast<unsigned long long*>(ctl + kCtlProf);

    constexpr bool prof_on = kProf;   // cycle counters compiled in only for the debug instantiation
    const bool prof_rec = prof_on && lane == 0 && (warp == 0 || warp == 1 || warp == 4 || warp == 8);
    // At D = 128 waiting warps sleep in their mbarrier waits (1 us hint) and
    // poll the accumulation turn every 256 ns, leaving issue slots and the
    // load/store path to the working warps (+4% deterministic on the full
    // S = 4096 workload); at D = 64 the plain polls measured faster.
    const Ctl c{abort_smem, p.status, p.abort_flag, p.timeout_ns, prof_rec ? prof_smem : nullptr,
                D == 128 ? 1000u : 0u, D == 128 ? 256 : 32};
    const unsigned long long t_start = kProf ? clock64() : 0ull;
    const uint32_t sbase = ptx::smem_u32(smem);

    if (threadIdx.x == 0) {
        *abort_smem = ((sbase & 1023u) != 0) ? 1 : 0;
        if (sbase & 1023u) report_timeout(c, -1, (int)sbase, 0, 0);
        for (int i = 0; i < kNDesc; ++i) {
            ptx::mbar_init(BAR(B_DESC_FULL + i), 1);
            ptx::mbar_init(BAR(B_DESC_EMPTY + i), kSubTiles);   // the drain warps read it last
        }
        ptx::mbar_init(BAR(B_KV_FULL), 1);
        ptx::mbar_init(BAR(B_KV_EMPTY), 1);
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(BAR(B_Q_FULL + s), 1);
            ptx::mbar_init(BAR(B_Q_EMPTY + s), 1);
            ptx::mbar_init(BAR(B_DO_FULL + s), 1);
            ptx::mbar_init(BAR(B_DO_EMPTY + s), 1);
        }
        ptx::mbar_init(BAR(B_S_FULL), 1);
        ptx::mbar_init(BAR(B_DP_FULL), 1);
        ptx::mbar_init(BAR(B_P_READY), 8);
        ptx::mbar_init(BAR(B_DS_READY), 8);
        ptx::mbar_init(BAR(B_DS_FREE), 1);
        ptx::mbar_init(BAR(B_DQ_FULL), 1);
        ptx::mbar_init(BAR(B_DQ_EMPTY), kSubTiles);
        ptx::mbar_init(BAR(B_ACC_FULL), 1);
        ptx::mbar_init(BAR(B_ACC_EMPTY), 8);
        ptx::mbar_init(BAR(B_DRAIN), 1);
        ptx::fence_mbar_init();
        if (prof_on)
            for (int i = 0; i < kProfSmem; ++i) prof_smem[i] = 0;
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32((const void*)tmem_slot), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int slot = p.cta_perm ? p.cta_perm[blockIdx.x] : (int)blockIdx.x;
    const Shape sh{p.B, p.Hq, p.Hkv, p.n, p.G, p.causal, p.sched, p.win, p.nk};
    const bool ordered = is_ordered(p.sched);

    // Each warpgroup first re-sizes its registers (all four warps execute the
    // same setmaxnreg), then runs its role.
    if (wg == 0) {
    ptx::setmaxnreg_dec<Regs<D>::kCtl>();
    if (warp == 0) {
        // ================================================== producer
        if (lane == 0 && !*abort_smem) {
            ptx::prefetch_tensormap(&p.tm_q);
            ptx::prefetch_tensormap(&p.tm_k);
            ptx::prefetch_tensormap(&p.tm_v);
            ptx::prefetch_tensormap(&p.tm_do);
            if (p.delay_ns) {
                const uint64_t t0 = ptx::globaltimer();
                while (ptx::globaltimer() - t0 < (uint64_t)p.delay_ns[slot]) {
                }
            }
            int w = 0;
            long long pc = 0;   // pairs produced
            int kvc = 0;        // KV tiles loaded
            int q_armed[2] = {0, 0}, do_armed[2] = {0, 0};
            bool ok = true;
            for (;;) {
                const int64_t k = next_task(p, slot, w);
                const bool have = k < p.ntasks;
                const TaskRef tr = task_ref(sh, have ? k : 0);   // once per task
                const int L = have ? task_len_at(sh, tr) : 1;
                for (int u = 0; u < L && ok; ++u) {
                    const int ds = (int)(pc % kNDesc);
                    if (pc >= kNDesc && !wait1(BAR(B_DESC_EMPTY + ds), (uint32_t)((pc / kNDesc - 1) & 1), c,
                                               kRoleProducer, (int)pc, 0)) {
                        ok = false;
                        break;
                    }
                    PairDesc d;
                    if (!have) {
                        d = PairDesc{0, 0, 0, 0, 0, kEnd, -1, 0};
                        descs[ds] = d;
                        ptx::mbar_arrive(BAR(B_DESC_FULL + ds));
                        break;
                    }
                    const Visit v = visit_at(sh, tr, u);
                    const bool first = (u == 0) || visit_at(sh, tr, u - 1).kv != v.kv;
                    const bool last = (u == L - 1) || visit_at(sh, tr, u + 1).kv != v.kv;
                    int rank = -1;
                    if (ordered)
                        rank = p.ranks ? (int)p.ranks[rank_index(sh, v.b, v.hq, v.q, v.kv)] : v.kv - first_kv(sh, v.q);
                    d.b = v.b;
                    d.hq = v.hq;
                    d.hkv = v.hkv;
                    d.q = v.q;
                    d.kv = v.kv;
                    d.flags = (first ? kKvFirst : 0) | (last ? kKvLast : 0) |
                              ((p.causal && v.q == v.kv) ? kDiag : 0) |
                              ((kMasked && (((p.S & 127) && v.q == p.n - 1) || ((p.Skv & 127) && v.kv == p.nkv - 1) ||
                                            (p.window && 128 * (v.q - v.kv) + 127 >= p.window)))
                                   ? kPartial : 0);   // partial last tile, or the far edge of the window
                    d.rank = rank;
                    d.pad = 0;
                    descs[ds] = d;
                    ptx::mbar_arrive(BAR(B_DESC_FULL + ds));
                    trace_ev<kProf>(p, pc, EV_PR_DESC);
                    if (first) {
                        if (kvc > 0 && !wait1(BAR(B_KV_EMPTY), (uint32_t)((kvc - 1) & 1), c, kRoleProducer,
                                              (int)pc, 1)) {
                            ok = false;
                            break;
                        }
                        const uint32_t fb = BAR(B_KV_FULL);
                        ptx::mbar_arrive_expect_tx(fb, C::kKvBytes);
                        // the tensors' key/value head (D = 128 may run one task per query head)
                        const int hk = (D == 128) ? v.b * p.kvh + v.hq / p.kvg : v.b * p.Hkv + v.hkv;
#pragma unroll
                        for (int bx = 0; bx < C::kNBox; ++bx) {
                            ptx::tma_load_3d(sbase + C::OFF_K + bx * kBox, &p.tm_k, 64 * bx, v.kv * 128, hk, fb);
                            ptx::tma_load_3d(sbase + C::OFF_V + bx * kBox, &p.tm_v, 64 * bx, v.kv * 128, hk, fb);
                        }
                        ++kvc;
                    }
                    const int hqi = v.b * p.Hq + v.hq;
                    const int st = (int)(pc % C::kQStages);
                    if (q_armed[st] > 0 && !wait1(BAR(B_Q_EMPTY + st), (uint32_t)((q_armed[st] - 1) & 1), c,
                                                  kRoleProducer, (int)pc, 2)) {
                        ok = false;
                        break;
                    }
                    uint32_t fb = BAR(B_Q_FULL + st);
                    ptx::mbar_arrive_expect_tx(fb, C::kQBytes);
                    const uint32_t sq = sbase + C::OFF_Q + st * C::kTile;
#pragma unroll
                    for (int bx = 0; bx < C::kNBox; ++bx)
                        ptx::tma_load_3d(sq + bx * kBox, &p.tm_q, 64 * bx, v.q * 128, hqi, fb);
                    ++q_armed[st];
                    trace_ev<kProf>(p, pc, EV_PR_Q_ISSUED);
                    const int so = (int)(pc % C::kDoStages);
                    if (do_armed[so] > 0 && !wait1(BAR(B_DO_EMPTY + so), (uint32_t)((do_armed[so] - 1) & 1), c,
                                                   kRoleProducer, (int)pc, 3)) {
                        ok = false;
                        break;
                    }
                    fb = BAR(B_DO_FULL + so);
                    ptx::mbar_arrive_expect_tx(fb, C::kDoBytes);
                    const uint32_t sd = sbase + C::OFF_DO + so * C::kTile;
#pragma unroll
                    for (int bx = 0; bx < C::kNBox; ++bx)
                        ptx::tma_load_3d(sd + bx * kBox, &p.tm_do, 64 * bx, v.q * 128, hqi, fb);
                    ++do_armed[so];
                    trace_ev<kProf>(p, pc, EV_PR_DO_ISSUED);
                    ++pc;
                }
                if (!have || !ok) break;
            }
            // Let every issued load land before the CTA can exit (bounded).
            constexpr uint64_t kDrainNs = 100000000ull;
            auto drain = [&](uint32_t bar, int armed) {
                if (armed == 0) return;
                const uint64_t t0 = ptx::globaltimer();
                while (!ptx::mbar_try_wait(bar, (uint32_t)((armed - 1) & 1)) && ptx::globaltimer() - t0 < kDrainNs) {
                }
            };
            drain(BAR(B_KV_FULL), kvc);
            for (int s = 0; s < 2; ++s) {
                drain(BAR(B_Q_FULL + s), q_armed[s]);
                drain(BAR(B_DO_FULL + s), do_armed[s]);
            }
        }
    } else if (warp == 1) {
        // ================================================== MMA issuer
        if (lane == 0 && !*abort_smem) {
            const uint32_t tS = tmem + C::COL_S, tDP = tmem + C::COL_DP, tDQ = tmem + C::COL_DQ;
            const uint32_t tDK = tmem + C::COL_DK, tDV = tmem + C::COL_DV;
            const uint32_t sK = sbase + C::OFF_K, sV = sbase + C::OFF_V, sDS = sbase + C::OFF_DS;
            auto sQ = [&](long long i) { return sbase + C::OFF_Q + (uint32_t)(i % C::kQStages) * C::kTile; };
            auto sDO = [&](long long i) { return sbase + C::OFF_DO + (uint32_t)(i % C::kDoStages) * C::kTile; };
            auto wait_q = [&](long long i, int site) {
                return wait1(BAR(B_Q_FULL + (int)(i % C::kQStages)), (uint32_t)((i / C::kQStages) & 1), c, kRoleMma,
                             (int)i, site);
            };
            auto wait_do = [&](long long i, int site) {
                return wait1(BAR(B_DO_FULL + (int)(i % C::kDoStages)), (uint32_t)((i / C::kDoStages) & 1), c,
                             kRoleMma, (int)i, site);
            };
            long long pp = 0;
            int kvc = 0;
            bool ok = wait1(BAR(B_DESC_FULL), 0, c, kRoleMma, 0, 0);
            PairDesc d = descs[0];
            if (ok && !(d.flags & kEnd)) {
                ok = wait1(BAR(B_KV_FULL), 0, c, kRoleMma, 0, 0) && wait_q(0, 0);
                if (ok) {
                    ptx::tc_fence_after();
                    issue_s<D>(tS, sK, sQ(0));
                    ptx::tc_commit(BAR(B_S_FULL));
                    trace_ev<kProf>(p, 0, EV_S_ISSUE);
                    ok = wait_do(0, 2);
                }
                if (ok) {
                    ptx::tc_fence_after();
                    issue_s<D>(tDP, sV, sDO(0));
                    ptx::tc_commit(BAR(B_DP_FULL));
                    trace_ev<kProf>(p, 0, EV_DP_ISSUE);
                }
                while (ok) {
                    const bool kv_first = d.flags & kKvFirst;
                    if (!wait1(BAR(B_P_READY), (uint32_t)(pp & 1), c, kRoleMma, (int)pp, 3)) break;
                    if (kv_first && kvc > 0 &&
                        !wait1(BAR(B_ACC_EMPTY), (uint32_t)((kvc - 1) & 1), c, kRoleMma, (int)pp, 4))
                        break;
                    ptx::tc_fence_after();
                    issue_dv<D>(tDV, tS, sDO(pp), kv_first ? 0u : 1u);
                    ptx::tc_commit(BAR(B_DO_EMPTY + (int)(pp % C::kDoStages)));
                    trace_ev<kProf>(p, pp, EV_DV_ISSUE);
                    const int nslot = (int)((pp + 1) % kNDesc);
                    if (!wait1(BAR(B_DESC_FULL + nslot), (uint32_t)(((pp + 1) / kNDesc) & 1), c, kRoleMma, (int)pp, 5))
                        break;
                    const PairDesc nd = descs[nslot];
                    const bool has_next = !(nd.flags & kEnd);
                    const bool next_new_kv = has_next && (nd.flags & kKvFirst);
                    if (has_next && !next_new_kv) {
                        if (!wait_q(pp + 1, 6)) break;
                        ptx::tc_fence_after();
                        issue_s<D>(tS, sK, sQ(pp + 1));
                        ptx::tc_commit(BAR(B_S_FULL));
                        trace_ev<kProf>(p, pp + 1, EV_S_ISSUE);
                    }
                    if (!wait1(BAR(B_DS_READY), (uint32_t)(pp & 1), c, kRoleMma, (int)pp, 7)) break;
                    // dQ is issued before dK, so that the drain warps get it one product
                    // earlier (at D = 128 it reuses the dP columns, which dS has just freed)
                    if (!C::kDqAlias && pp > 0 &&
                        !wait1(BAR(B_DQ_EMPTY), (uint32_t)((pp - 1) & 1), c, kRoleMma, (int)pp, 8))
                        break;
                    ptx::tc_fence_after();
                    issue_dq<D>(tDQ, sDS, sK);
                    ptx::tc_commit(BAR(B_DQ_FULL));
                    trace_ev<kProf>(p, pp, EV_DQ_ISSUE);
                    issue_dk<D>(tDK, sDS, sQ(pp), kv_first ? 0u : 1u);
                    ptx::tc_commit(BAR(B_Q_EMPTY + (int)(pp % C::kQStages)));
                    trace_ev<kProf>(p, pp, EV_DK_ISSUE);
                    ptx::tc_commit(BAR(B_DS_FREE));
                    if (d.flags & kKvLast) {
                        ptx::tc_commit(BAR(B_ACC_FULL));
                        ptx::tc_commit(BAR(B_KV_EMPTY));
                    }
                    if (!has_next) break;
                    if (next_new_kv) {
                        ++kvc;
                        if (!wait1(BAR(B_KV_FULL), (uint32_t)(kvc & 1), c, kRoleMma, (int)pp, 1)) break;
                        if (!wait_q(pp + 1, 6)) break;
                        ptx::tc_fence_after();
                        issue_s<D>(tS, sK, sQ(pp + 1));
                        ptx::tc_commit(BAR(B_S_FULL));
                        trace_ev<kProf>(p, pp + 1, EV_S_ISSUE);
                    }
                    if (C::kDqAlias && !wait1(BAR(B_DQ_EMPTY), (uint32_t)(pp & 1), c, kRoleMma, (int)pp, 8)) break;
                    if (!wait_do(pp + 1, 9)) break;
                    ptx::tc_fence_after();
                    issue_s<D>(tDP, sV, sDO(pp + 1));
                    ptx::tc_commit(BAR(B_DP_FULL));
                    trace_ev<kProf>(p, pp + 1, EV_DP_ISSUE);
                    ++pp;
                    d = nd;
                }
            }
            // Wait for every issued MMA before tensor memory can be freed.
            ptx::tc_commit(BAR(B_DRAIN));
            const uint64_t t0 = ptx::globaltimer();
            while (!ptx::mbar_try_wait(BAR(B_DRAIN), 0) && ptx::globaltimer() - t0 < 100000000ull) {
            }
        }
    }
    } else if (wg == 2 || wg == 3) {
        ptx::setmaxnreg_inc<Regs<D>::kSoftmax>();
        // ================================================== softmax / dS
        const int sub = warp & 3;
        const int c0 = 64 * (wg - 2);
        const int row = 32 * sub + lane;                   // KV row within the tile
        const uint32_t lane_off = (uint32_t)(32 * sub) << 16;
        uint8_t* ds_box = smem + C::OFF_DS + (c0 >> 6) * kBox;
        const bool rec = warp == 8 && lane == 0;
        // Per-column statistics of a pair's Q tile: lane l holds LSE and delta
        // of columns c0+l and c0+32+l (columns past S of a partial last tile
        // read 0 and are masked).
        // sv: LSE of the two columns, then their delta.
        constexpr bool kAhead = true;
        constexpr float kLseMul = kAhead ? 1.f : kLog2e;
        auto fetch = [&](const PairDesc& fd, float (&sv)[4]) {
            const int qcol = fd.q * 128 + c0 + lane;
            const size_t qrow = (size_t)(fd.b * p.Hq + fd.hq) * p.S + (size_t)qcol;
            const bool va = !kMasked || qcol < p.S, vb = !kMasked || qcol + 32 < p.S;
            sv[0] = va ? ptx::ld_nc(p.lse + qrow) * kLseMul : 0.f;
            sv[1] = vb ? ptx::ld_nc(p.lse + qrow + 32) * kLseMul : 0.f;
            sv[2] = va ? ptx::ld_nc(p.delta + qrow) : 0.f;
            sv[3] = vb ? ptx::ld_nc(p.delta + qrow + 32) : 0.f;
        };
        // kAhead: the next pair's descriptor is read at the top of this pair
        // and its statistics are loaded after this pair's P phase, so that the
        // shared-memory read and the global loads overlap the dP wait and the
        // dS phase (both head dimensions on the current kernel; the other
        // order reads a pair's descriptor and statistics at the top of its
        // own iteration).
        PairDesc d{};
        float sv[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (kAhead) {
            if (waitw<true>(BAR(B_DESC_FULL), 0u, c, kRoleSoftmax, 0, 0)) {
                d = descs[0];
                if (!(d.flags & kEnd)) fetch(d, sv);
            } else {
                d.flags = kEnd;
            }
        }
        for (long long pp = 0;; ++pp) {
            PairDesc nd{};
            if constexpr (kAhead) {
                if (d.flags & kEnd) break;
                const int ns = (int)((pp + 1) % kNDesc);
                if (!waitw<true>(BAR(B_DESC_FULL + ns), (uint32_t)(((pp + 1) / kNDesc) & 1), c, kRoleSoftmax, (int)pp, 0))
                    break;
                nd = descs[ns];
            } else {
                const int ds = (int)(pp % kNDesc);
                if (!waitw<true>(BAR(B_DESC_FULL + ds), (uint32_t)((pp / kNDesc) & 1), c, kRoleSoftmax, (int)pp, 0)) break;
                d = descs[ds];
                if (d.flags & kEnd) break;
                fetch(d, sv);
            }
            const float lse2_a = kAhead ? sv[0] * kLog2e : sv[0], lse2_b = kAhead ? sv[1] * kLog2e : sv[1];
            const float delta_a = sv[2], delta_b = sv[3];
            if (!waitw<true>(BAR(B_S_FULL), (uint32_t)(pp & 1), c, kRoleSoftmax, (int)pp, 1)) break;
            if (rec) trace_ev<kProf>(p, pp, EV_SM_S_SEEN);
            ptx::tc_fence_after();
            float P[64];
            unsigned long long tc0 = kProf ? clock64() : 0ull;
            softmax_64<kMasked || D == 64>(tmem + lane_off + C::COL_S, c0, lse2_a, lse2_b, p.scale_log2e, (d.flags & (kDiag | kPartial)) != 0,
                       (d.flags & kDiag) != 0, row, p.Skv - d.kv * 128, p.S - d.q * 128,
                       p.window ? p.window - 128 * (d.q - d.kv) : (1 << 30), P);
            prof_add(c, kRoleSoftmax, 8, tc0);
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(BAR(B_P_READY));
            if (rec) trace_ev<kProf>(p, pp, EV_SM_P_DONE);
            float svn[4] = {0.f, 0.f, 0.f, 0.f};
            if (kAhead && !(nd.flags & kEnd)) fetch(nd, svn);
            if (!waitw<true>(BAR(B_DP_FULL), (uint32_t)(pp & 1), c, kRoleSoftmax, (int)pp, 2)) break;
            if (rec) trace_ev<kProf>(p, pp, EV_SM_DP_SEEN);
            ptx::tc_fence_after();
            if (pp > 0 && !waitw<true>(BAR(B_DS_FREE), (uint32_t)((pp - 1) & 1), c, kRoleSoftmax, (int)pp, 3)) break;
            tc0 = kProf ? clock64() : 0ull;
            ds_64(tmem + lane_off + C::COL_DP, c0, delta_a, delta_b, p.scale, P, ds_box, row);
            prof_add(c, kRoleSoftmax, 9, tc0);
            ptx::tc_fence_before();
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(BAR(B_DS_READY));
            if (rec) trace_ev<kProf>(p, pp, EV_SM_DS_DONE);
            if constexpr (kAhead) {
                d = nd;
#pragma unroll
                for (int k = 0; k < 4; ++k) sv[k] = svn[k];
            }
        }
    } else {
        if constexpr (Regs<D>::kDrain < kRegsLaunch) ptx::setmaxnreg_dec<Regs<D>::kDrain>();   // 96 at D = 128: as launched
        // ================================================== dQ drain + ordered reduction + dK/dV epilogue
        // Fast-path waits (every lane tries once, then a vote) at both head
        // dimensions: once the kernel's hot code fitted the instruction cache
        // they measured +0.5% ordered and +5% unordered at D = 128 (with the
        // unrolled MMA loops they had cost the ordered schedules 5-9%).
        constexpr bool kDrainFast = true;
        const int sub = warp & 3;
        const int half = (wg == 4) ? 1 : 0;
        const int st = 2 * sub + half;                     // dQ sub-tile: rows 16*st .. 16*st+15
        const uint32_t q_lanes = (uint32_t)(32 * sub + 16 * half) << 16;
        const uint32_t kv_lanes = (uint32_t)(32 * sub) << 16;
        const int qa = 16 * st + (lane >> 2);              // rows of this lane's fragments: qa, qa + 8
        const int ca = 2 * (lane & 3);                     // column of the first fragment element
        const bool odd = lane & 1;
        const bool rec = warp == 4 && lane == 0;
        int kvc = 0;
        for (long long pp = 0;; ++pp) {
            const int ds = (int)(pp % kNDesc);
            if (!waitw<kDrainFast>(BAR(B_DESC_FULL + ds), (uint32_t)((pp / kNDesc) & 1), c, kRoleDrain, (int)pp, 0)) break;
            const PairDesc d = descs[ds];
            if (d.flags & kEnd) break;
            if (!waitw<kDrainFast>(BAR(B_DQ_FULL), (uint32_t)(pp & 1), c, kRoleDrain, (int)pp, 1)) break;
            if (rec) trace_ev<kProf>(p, pp, EV_DR_DQ_SEEN);
            ptx::tc_fence_after();
            // Read the sub-tile (16 rows x D) out of tensor memory, then hand the
            // columns back to the MMA issuer.
            uint32_t r[D / 2];
#pragma unroll
            for (int b = 0; b < D / 64; ++b)
                ptx::tmem_ld16x256_x8(tmem + q_lanes + C::COL_DQ + 64 * b,
                                      *reinterpret_cast<uint32_t(*)[32]>(&r[32 * b]));
            ptx::tmem_ld_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(BAR(B_DQ_EMPTY));
            if (rec) trace_ev<kProf>(p, pp, EV_DR_DQ_EMPTY);
            const int tile = (d.b * p.Hq + d.hq) * p.n + d.q;
            if (p.partials) {
                float* gp = p.partials + ((size_t)tile * p.nkv + d.kv) * 128 * D;
#pragma unroll
                for (int j = 0; j < D / 8; ++j) {
                    *reinterpret_cast<float2*>(gp + (size_t)qa * D + 8 * j + ca) =
                        make_float2(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]));
                    *reinterpret_cast<float2*>(gp + (size_t)(qa + 8) * D + 8 * j + ca) =
                        make_float2(__uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
                }
            }
            // Pair exchange inside each lane quad: afterwards a lane holds 4
            // consecutive columns of one 8-column chunk (even lanes: chunk j,
            // odd lanes: chunk j+1) for its two rows.
#pragma unroll
            for (int j = 0; j < D / 8; j += 2) {
                const uint32_t s0 = odd ? r[4 * j] : r[4 * (j + 1)];
                const uint32_t s1 = odd ? r[4 * j + 1] : r[4 * (j + 1) + 1];
                const uint32_t s2 = odd ? r[4 * j + 2] : r[4 * (j + 1) + 2];
                const uint32_t s3 = odd ? r[4 * j + 3] : r[4 * (j + 1) + 3];
                const uint32_t g0 = __shfl_xor_sync(0xffffffffu, s0, 1);
                const uint32_t g1 = __shfl_xor_sync(0xffffffffu, s1, 1);
                const uint32_t g2 = __shfl_xor_sync(0xffffffffu, s2, 1);
                const uint32_t g3 = __shfl_xor_sync(0xffffffffu, s3, 1);
                if (odd) {   // keeps chunk j+1: partner's lower pair first
                    r[4 * j] = g0;
                    r[4 * j + 1] = g1;
                    r[4 * j + 2] = r[4 * (j + 1)];
                    r[4 * j + 3] = r[4 * (j + 1) + 1];
                    const uint32_t b2 = r[4 * (j + 1) + 2], b3 = r[4 * (j + 1) + 3];
                    r[4 * (j + 1)] = g2;
                    r[4 * (j + 1) + 1] = g3;
                    r[4 * (j + 1) + 2] = b2;
                    r[4 * (j + 1) + 3] = b3;
                } else {     // keeps chunk j: own pair first
                    const uint32_t a2 = r[4 * j + 2], a3 = r[4 * j + 3];
                    r[4 * j + 2] = g0;
                    r[4 * j + 3] = g1;
                    r[4 * (j + 1)] = a2;
                    r[4 * (j + 1) + 1] = a3;
                    r[4 * (j + 1) + 2] = g2;
                    r[4 * (j + 1) + 3] = g3;
                }
            }
            // this lane now holds, for chunk pair (j, j+1): row qa cols cb..cb+3 in
            // r[4j..4j+3] and row qa+8 cols cb..cb+3 in r[4(j+1)..4(j+1)+3],
            // cb = 8*(j + odd) + 2*(lane & 2)
            bool ok = true;
            if (ordered) {
                int* sem = p.sem + (size_t)tile * kSubTiles + st;
                int good = 1;
                if (lane == 0) {
                    const unsigned long long t0 = kProf ? clock64() : 0ull;
                    good = wait_turn(p, c, abort_smem, sem, d.rank, d.b * p.Hq + d.hq, tile % p.n) ? 1 : 0;
                    prof_add(c, kRoleDrain, 8, t0);
                    if (good && st == 0 && p.order_log) {
                        const int s = atomicAdd(p.logcnt + tile, 1);
                        if (s >= 0 && s < p.nkv) p.order_log[(size_t)tile * p.nkv + s] = d.kv;
                    }
                }
                ok = __shfl_sync(0xffffffffu, good, 0) != 0;
                // the barrier orders the other lanes' reductions after lane 0's
                // acquire (a shuffle alone carries no memory ordering)
                __syncwarp();
            } else if (st == 0 && p.order_log && lane == 0) {
                const int s = atomicAdd(p.logcnt + tile, 1);
                if (s >= 0 && s < p.nkv) p.order_log[(size_t)tile * p.nkv + s] = d.kv;
            }
            if (!ok) break;
            if (rec) trace_ev<kProf>(p, pp, EV_DR_TURN);
            float* gdq = p.dq + ((size_t)(d.b * p.Hq + d.hq) * p.S + (size_t)d.q * 128) * D;
            const bool row_a = !kMasked || d.q * 128 + qa < p.S;   // rows past S
            const bool row_b = !kMasked || d.q * 128 + qa + 8 < p.S;
            const int cofs = 2 * (lane & 2);
#pragma unroll
            for (int j = 0; j < D / 8; j += 2) {
                const int cb = 8 * (j + (odd ? 1 : 0)) + cofs;
                if (row_a)
                    ptx::red_add_v4(gdq + (size_t)qa * D + cb, __uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                    __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
                if (row_b)
                    ptx::red_add_v4(gdq + (size_t)(qa + 8) * D + cb, __uint_as_float(r[4 * (j + 1)]),
                                __uint_as_float(r[4 * (j + 1) + 1]), __uint_as_float(r[4 * (j + 1) + 2]),
                                __uint_as_float(r[4 * (j + 1) + 3]));
            }
            if (rec) trace_ev<kProf>(p, pp, EV_DR_REDS);
            if (ordered) {
                __threadfence();
                __syncwarp();
                if (lane == 0) ptx::st_release(p.sem + (size_t)tile * kSubTiles + st, d.rank + 1);
            }
            if (rec) trace_ev<kProf>(p, pp, EV_DR_DONE);
            if (lane == 0) ptx::mbar_arrive(BAR(B_DESC_EMPTY + ds));
            if (d.flags & kKvLast) {
                // dK (drain warps of WG1) and dV (WG4) of the finished KV tile
                if (!waitw<kDrainFast>(BAR(B_ACC_FULL), (uint32_t)(kvc & 1), c, kRoleDrain, (int)pp, 2)) break;
                ptx::tc_fence_after();
                const int krow = 32 * sub + lane;
                const bool krow_ok = !kMasked || d.kv * 128 + krow < p.Skv;   // rows past S_kv are not stored
                // task head d.hkv: the key/value head, or the query head when
                // every query head is its own task (fp32 partial, summed later)
                const size_t grow = ((size_t)(d.b * p.Hkv + d.hkv) * p.Skv + (size_t)d.kv * 128 + krow) * D;
                const uint32_t col = half == 0 ? C::COL_DK : C::COL_DV;
                // The epilogue runs once per KV tile: its column loop stays
                // rolled, which keeps it out of the instruction cache's way.
                if constexpr (D == 128) {
                    // bf16 dK / dV, or the fp32 partials of one query head
                    const bool f32 = p.part_dk != nullptr;
                    uint8_t* outb = f32 ? reinterpret_cast<uint8_t*>((half == 0 ? p.part_dk : p.part_dv) + grow)
                                        : reinterpret_cast<uint8_t*>((half == 0 ? p.dk : p.dv) + grow);
#pragma unroll 1
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t v[32];
                        ptx::tmem_ld16(tmem + kv_lanes + col + 32 * cc, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                        ptx::tmem_ld16(tmem + kv_lanes + col + 32 * cc + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
                        ptx::tmem_ld_wait();
                        if (!krow_ok) continue;
                        if (f32) {
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                *reinterpret_cast<uint4*>(outb + 4 * (32 * cc + 4 * e)) =
                                    make_uint4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
                        } else {
                            uint32_t pk[16];
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                __nv_bfloat162 h2 =
                                    __floats2bfloat162_rn(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
                                pk[e] = *reinterpret_cast<uint32_t*>(&h2);
                            }
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                *reinterpret_cast<uint4*>(outb + 2 * (32 * cc + 8 * e)) =
                                    make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                        }
                    }
                } else {
                    // D = 64: always one task per key/value head group, bf16 out
                    __nv_bfloat16* out = (half == 0 ? p.dk : p.dv) + grow;
#pragma unroll 1
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t v[32];
                        ptx::tmem_ld16(tmem + kv_lanes + col + 32 * cc, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                        ptx::tmem_ld16(tmem + kv_lanes + col + 32 * cc + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
                        ptx::tmem_ld_wait();
                        uint32_t pk[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            __nv_bfloat162 h2 =
                                __floats2bfloat162_rn(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
                            pk[e] = *reinterpret_cast<uint32_t*>(&h2);
                        }
                        if (krow_ok) {
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                *reinterpret_cast<uint4*>(out + 32 * cc + 8 * e) =
                                    make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
                        }
                    }
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(BAR(B_ACC_EMPTY));
                ++kvc;
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
    if (prof_on && threadIdx.x == 0) {
        prof_smem[kProfSmem - 1] = clock64() - t_start;
        unsigned long long* out = p.prof + (size_t)blockIdx.x * kProfOut;
        for (int i = 0; i < kProfSmem - 1; ++i) out[i] = prof_smem[i];
        out[kProfOut - 1] = prof_smem[kProfSmem - 1];
    }
}

template <int D, bool kProf, bool kMasked>
int launch_bwd(const BwdParams& prm, int grid, cudaStream_t stream) {
    using C = Cfg<D>;
    static bool attr_done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -2;
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(dash_bwd_kernel<D, kProf, kMasked>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kSmem) != cudaSuccess)
            return -2;
        attr_done[dev] = true;
    }
    // The warpgroups re-split the block's registers with setmaxnreg; that is
    // only safe if the compiled kernel was granted the registers it assumes.
    static int regs_ok[64] = {};
    if (dev >= 0 && dev < 64 && regs_ok[dev] == 0) {
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, dash_bwd_kernel<D, kProf, kMasked>) != cudaSuccess) return -2;
        regs_ok[dev] = (fa.numRegs >= kRegsLaunch) ? 1 : -1;
    }
    if (dev < 0 || dev >= 64 || regs_ok[dev] != 1) return -3;
    void* args[] = {(void*)&prm};
    cudaError_t e = cudaLaunchCooperativeKernel((const void*)dash_bwd_kernel<D, kProf, kMasked>, dim3(grid),
                                                dim3(kThreads), args, C::kSmem, stream);
    if (e == cudaErrorCooperativeLaunchTooLarge) {
        (void)cudaGetLastError();
        return -3;
    }
    return e == cudaSuccess ? 0 : -2;
}

int bwd_max_ctas(int D, int device, int* P) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return -2;
    int per_sm = 0;
    cudaError_t e;
    if (D == 64) {
        cudaFuncSetAttribute(dash_bwd_kernel<64, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg<64>::kSmem);
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dash_bwd_kernel<64, false, false>, kThreads,
                                                          Cfg<64>::kSmem);
    } else {
        cudaFuncSetAttribute(dash_bwd_kernel<128, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg<128>::kSmem);
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dash_bwd_kernel<128, false, false>, kThreads,
                                                          Cfg<128>::kSmem);
    }
    if (e != cudaSuccess) return -2;
    if (per_sm < 1) return -3;
    *P = sms;   // one persistent CTA per SM
    return 0;
}

int launch_bwd_dispatch(int D, const BwdParams& prm, int grid, cudaStream_t stream) {
    if ((prm.S % 128) || (prm.Skv % 128) || prm.window) {   // a partial last tile or a window: masked
        if (prm.prof)
            return D == 64 ? launch_bwd<64, true, true>(prm, grid, stream) : launch_bwd<128, true, true>(prm, grid, stream);
        return D == 64 ? launch_bwd<64, false, true>(prm, grid, stream) : launch_bwd<128, false, true>(prm, grid, stream);
    }
    if (prm.prof)
        return D == 64 ? launch_bwd<64, true, false>(prm, grid, stream) : launch_bwd<128, true, false>(prm, grid, stream);
    return D == 64 ? launch_bwd<64, false, false>(prm, grid, stream) : launch_bwd<128, false, false>(prm, grid, stream);
}

// Loads (on the current device) every production variant of the persistent
// kernel; under lazy module loading it would otherwise load at its first launch.
int load_bwd_kernels() {
    cudaFuncAttributes fa;
    const void* fns[] = {(const void*)dash_bwd_kernel<64, false, false>, (const void*)dash_bwd_kernel<64, false, true>,
                         (const void*)dash_bwd_kernel<128, false, false>,
                         (const void*)dash_bwd_kernel<128, false, true>};
    for (const void* f : fns)
        if (cudaFuncGetAttributes(&fa, f) != cudaSuccess) return -2;
    return 0;
}

int bwd_smem_bytes(int D) { return D == 64 ? Cfg<64>::kSmem : Cfg<128>::kSmem; }

}  // namespace dash
