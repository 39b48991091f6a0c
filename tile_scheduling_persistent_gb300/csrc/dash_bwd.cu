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
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (*c.abort_smem) return false;
        if (ptx::globaltimer() - t0 > c.timeout) {
            report_timeout(c, role, i0, site, (int)bar);
            return false;
        }
    }
    prof_add(c, role, site, c0);
    return true;
}

// Whole-warp bounded wait with a warp-uniform outcome: lane 0 polls, then
// every lane observes the completed phase itself (acquire per thread).
__device__ __forceinline__ bool waitw(uint32_t bar, uint32_t parity, const Ctl& c, int role, int i0, int site) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = wait1(bar, parity, c, role, i0, site) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) {
        while (!ptx::mbar_try_wait(bar, parity)) {
        }
    }
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

// Spin until the accumulation counter of a dQ tile equals `rank` (acquire).
__device__ bool wait_turn(const BwdParams& p, const Ctl& c, volatile int* abort_smem, int tile, int rank,
                          int head) {
    int* sem = p.sem + tile;
    if (ptx::ld_acquire(sem) == rank) return true;
    const uint64_t t0 = ptx::globaltimer();
    int spins = 0;
    for (;;) {
        if (ptx::ld_acquire(sem) == rank) return true;
        if ((++spins & 63) == 0) {
            if (ptx::ld_volatile(p.abort_flag) || *abort_smem) return false;
            if (ptx::globaltimer() - t0 > c.timeout) {
                report_timeout(c, kRoleReducer, head, tile % p.n, rank);
                return false;
            }
        }
        __nanosleep(64);
    }
}

}  // namespace

template <int D, bool kProf>
__global__ void __launch_bounds__(kThreads, 1) dash_bwd_kernel(const __grid_constant__ BwdParams p) {
    using C = Cfg<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    uint8_t* ctl = smem + C::OFF_CTL;
    const uint32_t bar0 = ptx::smem_u32(ctl + kCtlBars);
    auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
    PairDesc* descs = reinterpret_cast<PairDesc*>(ctl + kCtlDescs);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(ctl + kCtlTmem);
    volatile int* abort_smem = reinterpret_cast<volatile int*>(ctl + kCtlAbort);
    unsigned long long* prof_smem = reinterpret_cast<unsigned long long*>(ctl + kCtlProf);

    constexpr bool prof_on = kProf;   // cycle counters compiled in only for the debug instantiation
    const bool prof_rec =
        prof_on && lane == 0 && (warp == 0 || warp == 4 || warp == 5 || warp == 6 || warp == 8);
    const Ctl c{abort_smem, p.status, p.abort_flag, p.timeout_ns, prof_rec ? prof_smem : nullptr};
    const unsigned long long t_start = kProf ? clock64() : 0ull;
    const uint32_t sbase = ptx::smem_u32(smem);

    if (threadIdx.x == 0) {
        *abort_smem = ((sbase & 1023u) != 0) ? 1 : 0;
        if (sbase & 1023u) report_timeout(c, -1, (int)sbase, 0, 0);
        for (int i = 0; i < kNDesc; ++i) {
            ptx::mbar_init(BAR(B_DESC_FULL + i), 1);
            ptx::mbar_init(BAR(B_DESC_EMPTY + i), 1);
        }
        ptx::mbar_init(BAR(B_KV_FULL), 1);
        ptx::mbar_init(BAR(B_KV_EMPTY), 1);
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(BAR(B_Q_FULL + s), 1);
            ptx::mbar_init(BAR(B_Q_EMPTY + s), 9);   // MMA commit + 8 softmax warps (LSE/delta)
            ptx::mbar_init(BAR(B_DO_FULL + s), 1);
            ptx::mbar_init(BAR(B_DO_EMPTY + s), 1);
        }
        ptx::mbar_init(BAR(B_S_FULL), 1);
        ptx::mbar_init(BAR(B_DP_FULL), 1);
        ptx::mbar_init(BAR(B_P_READY), 8);
        ptx::mbar_init(BAR(B_DS_READY), 8);
        ptx::mbar_init(BAR(B_DS_FREE), 1);
        ptx::mbar_init(BAR(B_DQ_FULL), 1);
        ptx::mbar_init(BAR(B_DQ_EMPTY), 4);
        ptx::mbar_init(BAR(B_ACC_FULL), 1);
        ptx::mbar_init(BAR(B_ACC_EMPTY), 4);
        ptx::mbar_init(BAR(B_STG_FULL), 4);
        ptx::mbar_init(BAR(B_STG_EMPTY), 1);
        ptx::mbar_init(BAR(B_DRAIN), 1);
        ptx::fence_mbar_init();
        if (prof_on)
            for (int i = 0; i < kProfSmem; ++i) prof_smem[i] = 0;
    }
    if (warp == 5) {
        ptx::tmem_alloc(ptx::smem_u32((const void*)tmem_slot), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int slot = p.cta_perm ? p.cta_perm[blockIdx.x] : (int)blockIdx.x;
    const Shape sh{p.B, p.Hq, p.Hkv, p.n, p.G, p.causal, p.sched};
    const bool ordered = is_ordered(p.sched);

    if (warp == 4) {
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
                const int L = have ? task_len(sh, k) : 1;
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
                    const Visit v = task_visit(sh, k, u);
                    const bool first = (u == 0) || task_visit(sh, k, u - 1).kv != v.kv;
                    const bool last = (u == L - 1) || task_visit(sh, k, u + 1).kv != v.kv;
                    int rank = -1;
                    if (ordered)
                        rank = p.ranks ? (int)p.ranks[rank_index(sh, v.b, v.hq, v.q, v.kv)] : v.kv;
                    d.b = v.b;
                    d.hq = v.hq;
                    d.hkv = v.hkv;
                    d.q = v.q;
                    d.kv = v.kv;
                    d.flags = (first ? kKvFirst : 0) | (last ? kKvLast : 0) |
                              ((p.causal && v.q == v.kv) ? kDiag : 0);
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
                        const int row = (v.b * p.Hkv + v.hkv) * p.S + v.kv * 128;
#pragma unroll
                        for (int bx = 0; bx < C::kNBox; ++bx) {
                            ptx::tma_load_2d(sbase + C::OFF_K + bx * kBox, &p.tm_k, 64 * bx, row, fb);
                            ptx::tma_load_2d(sbase + C::OFF_V + bx * kBox, &p.tm_v, 64 * bx, row, fb);
                        }
                        ++kvc;
                    }
                    const int qrow = (v.b * p.Hq + v.hq) * p.S + v.q * 128;
                    // Q, LSE, delta
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
                    for (int bx = 0; bx < C::kNBox; ++bx) ptx::tma_load_2d(sq + bx * kBox, &p.tm_q, 64 * bx, qrow, fb);
                    const uint32_t sv = sbase + C::OFF_VEC + st * 1024;
                    ptx::bulk_load(sv, p.lse + qrow, 512, fb);
                    ptx::bulk_load(sv + 512, p.delta + qrow, 512, fb);
                    ++q_armed[st];
                    trace_ev<kProf>(p, pc, EV_PR_Q_ISSUED);
                    // dO
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
                        ptx::tma_load_2d(sd + bx * kBox, &p.tm_do, 64 * bx, qrow, fb);
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
    } else if (warp == 5) {
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
                    ptx::tc_fence_after();
                    issue_dk<D>(tDK, sDS, sQ(pp), kv_first ? 0u : 1u);
                    trace_ev<kProf>(p, pp, EV_DK_ISSUE);
                    if (!C::kDqAlias && pp > 0 &&
                        !wait1(BAR(B_DQ_EMPTY), (uint32_t)((pp - 1) & 1), c, kRoleMma, (int)pp, 8))
                        break;
                    ptx::tc_fence_after();
                    issue_dq<D>(tDQ, sDS, sK);
                    trace_ev<kProf>(p, pp, EV_DQ_ISSUE);
                    ptx::tc_commit(BAR(B_DS_FREE));
                    ptx::tc_commit(BAR(B_DQ_FULL));
                    ptx::tc_commit(BAR(B_Q_EMPTY + (int)(pp % C::kQStages)));
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
    } else if (warp == 6) {
        // ================================================== reduce issuer
        if (lane == 0 && !*abort_smem) {
            ptx::prefetch_tensormap(&p.tm_dq);
            const uint32_t sstg = sbase + C::OFF_STG;
            long long u = 0;   // staging-buffer uses
            for (long long pp = 0;; ++pp) {
                const int ds = (int)(pp % kNDesc);
                if (!wait1(BAR(B_DESC_FULL + ds), (uint32_t)((pp / kNDesc) & 1), c, kRoleIssuer, (int)pp, 0)) break;
                const PairDesc d = descs[ds];
                if (d.flags & kEnd) break;
                const int tile = (d.b * p.Hq + d.hq) * p.n + d.q;
                const int row0 = (d.b * p.Hq + d.hq) * p.S + d.q * 128;
                bool ok = true;
                for (int h = 0; h < C::kHalves; ++h) {
                    if (!wait1(BAR(B_STG_FULL), (uint32_t)(u & 1), c, kRoleIssuer, (int)pp, 1)) {
                        ok = false;
                        break;
                    }
                    if (h == 0) trace_ev<kProf>(p, pp, EV_IS_STG_SEEN);
                    if (h == 0) {
                        const unsigned long long t0 = kProf ? clock64() : 0ull;
                        if (ordered && !wait_turn(p, c, abort_smem, tile, d.rank, d.b * p.Hq + d.hq)) {
                            ok = false;
                            break;
                        }
                        prof_add(c, kRoleIssuer, 8, t0);
                        trace_ev<kProf>(p, pp, EV_IS_TURN);
                        if (p.order_log) {
                            const int s = atomicAdd(p.logcnt + tile, 1);
                            if (s >= 0 && s < p.n) p.order_log[(size_t)tile * p.n + s] = d.kv;
                        }
                        ptx::fence_proxy_async_global();
                    }
                    const unsigned long long t1 = kProf ? clock64() : 0ull;
                    ptx::tma_reduce_add_2d(&p.tm_dq, 64 * h, row0, sstg);
                    ptx::tma_reduce_add_2d(&p.tm_dq, 64 * h + 32, row0, sstg + kBox);
                    ptx::bulk_commit();
                    ptx::bulk_wait_read0();
                    trace_ev<kProf>(p, pp, EV_IS_READ0 + (h & 1));
                    prof_add(c, kRoleIssuer, 9, t1);
                    ptx::mbar_arrive(BAR(B_STG_EMPTY));
                    ++u;
                }
                if (!ok) break;
                if (ordered) {
                    const unsigned long long t2 = kProf ? clock64() : 0ull;
                    ptx::bulk_wait0();
                    ptx::fence_proxy_async_global();
                    ptx::st_release(p.sem + tile, d.rank + 1);
                    prof_add(c, kRoleIssuer, 2, t2);
                }
                trace_ev<kProf>(p, pp, EV_IS_DONE);
                ptx::mbar_arrive(BAR(B_DESC_EMPTY + ds));
            }
            ptx::bulk_wait0();
        }
    } else if (warp >= 8) {
        // ================================================== softmax / dS
        const int sub = warp & 3;
        const int c0 = 64 * ((warp - 8) >> 2);
        const int row = 32 * sub + lane;                   // KV row within the tile
        const uint32_t lane_off = (uint32_t)(32 * sub) << 16;
        uint8_t* ds_box = smem + C::OFF_DS + (c0 >> 6) * kBox;
        for (long long pp = 0;; ++pp) {
            const int ds = (int)(pp % kNDesc);
            if (!waitw(BAR(B_DESC_FULL + ds), (uint32_t)((pp / kNDesc) & 1), c, kRoleSoftmax, (int)pp, 0)) break;
            const PairDesc d = descs[ds];
            if (d.flags & kEnd) break;
            const int st = (int)(pp % C::kQStages);
            const float* vec = reinterpret_cast<const float*>(smem + C::OFF_VEC + st * 1024);
            if (!waitw(BAR(B_S_FULL), (uint32_t)(pp & 1), c, kRoleSoftmax, (int)pp, 1)) break;
            if (warp == 8 && lane == 0) trace_ev<kProf>(p, pp, EV_SM_S_SEEN);
            ptx::tc_fence_after();
            float P[64];
            unsigned long long tc0 = kProf ? clock64() : 0ull;
            softmax_64(tmem + lane_off + C::COL_S, c0, vec, p.scale_log2e, (d.flags & kDiag) != 0, row, P);
            prof_add(c, kRoleSoftmax, 8, tc0);
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(BAR(B_P_READY));
            if (warp == 8 && lane == 0) trace_ev<kProf>(p, pp, EV_SM_P_DONE);
            if (!waitw(BAR(B_DP_FULL), (uint32_t)(pp & 1), c, kRoleSoftmax, (int)pp, 2)) break;
            if (warp == 8 && lane == 0) trace_ev<kProf>(p, pp, EV_SM_DP_SEEN);
            ptx::tc_fence_after();
            uint32_t pk[32];
            tc0 = kProf ? clock64() : 0ull;
            ds_64(tmem + lane_off + C::COL_DP, c0, vec + 128, p.scale, P, pk);
            prof_add(c, kRoleSoftmax, 9, tc0);
            ptx::tc_fence_before();
            if (pp > 0 && !waitw(BAR(B_DS_FREE), (uint32_t)((pp - 1) & 1), c, kRoleSoftmax, (int)pp, 3)) break;
            store_row_sw128(ds_box, row, pk);
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(BAR(B_DS_READY));
                ptx::mbar_arrive(BAR(B_Q_EMPTY + st));
            }
            if (warp == 8 && lane == 0) trace_ev<kProf>(p, pp, EV_SM_DS_DONE);
        }
    } else if (warp < 4) {
        // ================================================== dQ drain + dK/dV epilogue
        const int row = 32 * warp + lane;
        const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
        uint8_t* stg = smem + C::OFF_STG;
        int kvc = 0;
        long long u = 0;   // staging-buffer uses
        for (long long pp = 0;; ++pp) {
            const int ds = (int)(pp % kNDesc);
            if (!waitw(BAR(B_DESC_FULL + ds), (uint32_t)((pp / kNDesc) & 1), c, kRoleReducer, (int)pp, 0)) break;
            const PairDesc d = descs[ds];
            if (d.flags & kEnd) break;
            if (!waitw(BAR(B_DQ_FULL), (uint32_t)(pp & 1), c, kRoleReducer, (int)pp, 1)) break;
            if (warp == 0 && lane == 0) trace_ev<kProf>(p, pp, EV_DR_DQ_SEEN);
            ptx::tc_fence_after();
            const int tile = (d.b * p.Hq + d.hq) * p.n + d.q;
            float* gpart = p.partials ? p.partials + (((size_t)tile * p.n + d.kv) * 128 + row) * D : nullptr;
            bool ok = true;
#pragma unroll 1
            for (int h = 0; h < C::kHalves; ++h) {
                uint32_t r0[32], r1[32];
                ptx::tmem_ld32(tmem + lane_off + C::COL_DQ + 64 * h, r0);
                ptx::tmem_ld32(tmem + lane_off + C::COL_DQ + 64 * h + 32, r1);
                ptx::tmem_ld_wait();
                if (h == C::kHalves - 1) {   // dQ columns go back to the MMA issuer
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(BAR(B_DQ_EMPTY));
                    if (warp == 0 && lane == 0) trace_ev<kProf>(p, pp, EV_DR_DQ_EMPTY);
                }
                if (gpart) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        *reinterpret_cast<uint4*>(gpart + 64 * h + 4 * e) =
                            make_uint4(r0[4 * e], r0[4 * e + 1], r0[4 * e + 2], r0[4 * e + 3]);
                        *reinterpret_cast<uint4*>(gpart + 64 * h + 32 + 4 * e) =
                            make_uint4(r1[4 * e], r1[4 * e + 1], r1[4 * e + 2], r1[4 * e + 3]);
                    }
                }
                const unsigned long long t0 = kProf ? clock64() : 0ull;
                if (u > 0 && !waitw(BAR(B_STG_EMPTY), (uint32_t)((u - 1) & 1), c, kRoleReducer, (int)pp, 3)) {
                    ok = false;
                    break;
                }
                store_row_f32_sw128(stg, row, r0);
                store_row_f32_sw128(stg + kBox, row, r1);
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(BAR(B_STG_FULL));
                if (warp == 0 && lane == 0) trace_ev<kProf>(p, pp, EV_DR_STAGED0 + (h & 1));
                prof_add(c, kRoleReducer, 8, t0);
                ++u;
            }
            if (!ok) break;
            if (d.flags & kKvLast) {
                if (!waitw(BAR(B_ACC_FULL), (uint32_t)(kvc & 1), c, kRoleReducer, (int)pp, 2)) break;
                ptx::tc_fence_after();
                const size_t grow = ((size_t)(d.b * p.Hkv + d.hkv) * p.S + (size_t)d.kv * 128 + row) * D;
#pragma unroll
                for (int which = 0; which < 2; ++which) {
                    __nv_bfloat16* out = (which == 0 ? p.dk : p.dv) + grow;
                    const uint32_t col = which == 0 ? C::COL_DK : C::COL_DV;
#pragma unroll
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t r[32];
                        ptx::tmem_ld32(tmem + lane_off + col + 32 * cc, r);
                        ptx::tmem_ld_wait();
                        uint32_t pk[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            __nv_bfloat162 h2 =
                                __floats2bfloat162_rn(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
                            pk[e] = *reinterpret_cast<uint32_t*>(&h2);
                        }
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
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
    if (warp == 5) {
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

template <int D, bool kProf>
int launch_bwd(const BwdParams& prm, int grid, cudaStream_t stream) {
    using C = Cfg<D>;
    static bool attr_done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -2;
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(dash_bwd_kernel<D, kProf>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kSmem) != cudaSuccess)
            return -2;
        attr_done[dev] = true;
    }
    void* args[] = {(void*)&prm};
    cudaError_t e = cudaLaunchCooperativeKernel((const void*)dash_bwd_kernel<D, kProf>, dim3(grid),
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
        cudaFuncSetAttribute(dash_bwd_kernel<64, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg<64>::kSmem);
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dash_bwd_kernel<64, false>, kThreads,
                                                          Cfg<64>::kSmem);
    } else {
        cudaFuncSetAttribute(dash_bwd_kernel<128, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg<128>::kSmem);
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dash_bwd_kernel<128, false>, kThreads,
                                                          Cfg<128>::kSmem);
    }
    if (e != cudaSuccess) return -2;
    if (per_sm < 1) return -3;
    *P = sms;   // one persistent CTA per SM
    return 0;
}

int launch_bwd_dispatch(int D, const BwdParams& prm, int grid, cudaStream_t stream) {
    if (prm.prof)
        return D == 64 ? launch_bwd<64, true>(prm, grid, stream) : launch_bwd<128, true>(prm, grid, stream);
    return D == 64 ? launch_bwd<64, false>(prm, grid, stream) : launch_bwd<128, false>(prm, grid, stream);
}

int bwd_smem_bytes(int D) { return D == 64 ? Cfg<64>::kSmem : Cfg<128>::kSmem; }

}  // namespace dash
