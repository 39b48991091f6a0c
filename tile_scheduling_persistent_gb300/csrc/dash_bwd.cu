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
};

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

// Single-thread bounded wait.
__device__ __forceinline__ bool wait1(uint32_t bar, uint32_t parity, const Ctl& c, int role, int i0,
                                      int i1) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (*c.abort_smem) return false;
        if (ptx::globaltimer() - t0 > c.timeout) {
            report_timeout(c, role, i0, i1, (int)bar);
            return false;
        }
    }
    return true;
}

// Whole-warp bounded wait with a warp-uniform outcome: lane 0 polls, then
// every lane observes the completed phase itself (acquire per thread).
__device__ __forceinline__ bool waitw(uint32_t bar, uint32_t parity, const Ctl& c, int role, int i0,
                                      int i1) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = wait1(bar, parity, c, role, i0, i1) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) {
        while (!ptx::mbar_try_wait(bar, parity)) {
        }
    }
    return ok != 0;
}

// Barrier among the 4 reducer warps that also ORs a predicate.
__device__ __forceinline__ bool reducer_bar_or(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ int64_t next_task(const BwdParams& p, int slot, int& w) {
    if (is_static(p.sched)) {
        const int64_t k = (int64_t)slot + (int64_t)w * p.P;
        ++w;
        return k;
    }
    return (int64_t)atomicAdd(p.task_counter, 1);
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(kThreads, 1) dash_bwd_kernel(const __grid_constant__ BwdParams p) {
    using C = Cfg<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    uint8_t* ctl = smem + C::OFF_CTL;
    const uint32_t bar0 = ptx::smem_u32(ctl);
    auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
    PairDesc* descs = reinterpret_cast<PairDesc*>(ctl + 256);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(ctl + 512);
    volatile int* abort_smem = reinterpret_cast<volatile int*>(ctl + 516);

    const Ctl c{abort_smem, p.status, p.abort_flag, p.timeout_ns};
    const uint32_t sbase = ptx::smem_u32(smem);

    if (threadIdx.x == 0) {
        *abort_smem = ((sbase & 1023u) != 0) ? 1 : 0;
        if (sbase & 1023u) report_timeout(c, -1, (int)sbase, 0, 0);
        for (int i = 0; i < kNDesc; ++i) {
            ptx::mbar_init(BAR(B_DESC_FULL + i), 1);
            ptx::mbar_init(BAR(B_DESC_EMPTY + i), 4);
        }
        ptx::mbar_init(BAR(B_KV_FULL), 1);
        ptx::mbar_init(BAR(B_KV_EMPTY), 1);
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(BAR(B_Q_FULL + s), 1);
            ptx::mbar_init(BAR(B_Q_EMPTY + s), 9);
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
        ptx::mbar_init(BAR(B_DRAIN), 1);
        ptx::fence_mbar_init();
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
            long long pc = 0;            // pairs produced
            int kvc = 0;                 // KV tiles loaded
            int q_armed[kStages] = {0, 0};
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
                    if (ordered) {
                        rank = is_static(p.sched) ? (int)p.ranks[rank_index(sh, v.b, v.hq, v.q, v.kv)] : v.kv;
                    }
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
                    const int st = (int)(pc % kStages);
                    if (q_armed[st] > 0 && !wait1(BAR(B_Q_EMPTY + st), (uint32_t)((q_armed[st] - 1) & 1), c,
                                                  kRoleProducer, (int)pc, 2)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = BAR(B_Q_FULL + st);
                    ptx::mbar_arrive_expect_tx(fb, C::kStageBytes);
                    const int qrow = (v.b * p.Hq + v.hq) * p.S + v.q * 128;
                    const uint32_t sq = sbase + C::OFF_STAGE + st * 2 * C::kTile;
#pragma unroll
                    for (int bx = 0; bx < C::kNBox; ++bx) {
                        ptx::tma_load_2d(sq + bx * kBox, &p.tm_q, 64 * bx, qrow, fb);
                        ptx::tma_load_2d(sq + C::kTile + bx * kBox, &p.tm_do, 64 * bx, qrow, fb);
                    }
                    const uint32_t sv = sbase + C::OFF_VEC + st * 1024;
                    ptx::bulk_load(sv, p.lse + qrow, 512, fb);
                    ptx::bulk_load(sv + 512, p.delta + qrow, 512, fb);
                    ++q_armed[st];
                    ++pc;
                }
                if (!have || !ok) break;
            }
            // Let every issued load land before the CTA can exit (bounded).
            constexpr uint64_t kDrainNs = 100000000ull;
            if (kvc > 0) {
                const uint64_t t0 = ptx::globaltimer();
                while (!ptx::mbar_try_wait(BAR(B_KV_FULL), (uint32_t)((kvc - 1) & 1)) &&
                       ptx::globaltimer() - t0 < kDrainNs) {
                }
            }
            for (int s = 0; s < kStages; ++s) {
                if (q_armed[s] == 0) continue;
                const uint64_t t0 = ptx::globaltimer();
                while (!ptx::mbar_try_wait(BAR(B_Q_FULL + s), (uint32_t)((q_armed[s] - 1) & 1)) &&
                       ptx::globaltimer() - t0 < kDrainNs) {
                }
            }
        }
    } else if (warp == 5) {
        // ================================================== MMA issuer
        if (lane == 0 && !*abort_smem) {
            const uint32_t tS = tmem + C::COL_S, tDP = tmem + C::COL_DP, tDQ = tmem + C::COL_DQ;
            const uint32_t tDK = tmem + C::COL_DK, tDV = tmem + C::COL_DV;
            const uint32_t sK = sbase + C::OFF_K, sV = sbase + C::OFF_V, sDS = sbase + C::OFF_DS;
            auto sQ = [&](long long pp) { return sbase + C::OFF_STAGE + (uint32_t)(pp % kStages) * 2 * C::kTile; };
            auto q_par = [&](long long pp) { return (uint32_t)((pp / kStages) & 1); };
            long long pp = 0;
            int kvc = 0;
            bool ok = wait1(BAR(B_DESC_FULL), 0, c, kRoleMma, 0, 0);
            PairDesc d = descs[0];
            if (ok && !(d.flags & kEnd)) {
                ok = wait1(BAR(B_KV_FULL), 0, c, kRoleMma, 0, 1) && wait1(BAR(B_Q_FULL), 0, c, kRoleMma, 0, 2);
                if (ok) {
                    ptx::tc_fence_after();
                    issue_s<D>(tS, sK, sQ(0));
                    ptx::tc_commit(BAR(B_S_FULL));
                    issue_s<D>(tDP, sV, sQ(0) + C::kTile);
                    ptx::tc_commit(BAR(B_DP_FULL));
                }
                while (ok) {
                    const bool kv_first = d.flags & kKvFirst;
                    if (!wait1(BAR(B_P_READY), (uint32_t)(pp & 1), c, kRoleMma, (int)pp, 3)) break;
                    if (kv_first && kvc > 0 &&
                        !wait1(BAR(B_ACC_EMPTY), (uint32_t)((kvc - 1) & 1), c, kRoleMma, (int)pp, 4))
                        break;
                    ptx::tc_fence_after();
                    issue_dv<D>(tDV, tS, sQ(pp) + C::kTile, kv_first ? 0u : 1u);
                    const int nslot = (int)((pp + 1) % kNDesc);
                    if (!wait1(BAR(B_DESC_FULL + nslot), (uint32_t)(((pp + 1) / kNDesc) & 1), c, kRoleMma,
                               (int)pp, 5))
                        break;
                    const PairDesc nd = descs[nslot];
                    const bool has_next = !(nd.flags & kEnd);
                    const bool next_new_kv = has_next && (nd.flags & kKvFirst);
                    if (has_next && !next_new_kv) {
                        if (!wait1(BAR(B_Q_FULL + (int)((pp + 1) % kStages)), q_par(pp + 1), c, kRoleMma,
                                   (int)pp, 6))
                            break;
                        ptx::tc_fence_after();
                        issue_s<D>(tS, sK, sQ(pp + 1));
                        ptx::tc_commit(BAR(B_S_FULL));
                    }
                    if (!wait1(BAR(B_DS_READY), (uint32_t)(pp & 1), c, kRoleMma, (int)pp, 7)) break;
                    ptx::tc_fence_after();
                    issue_dk<D>(tDK, sDS, sQ(pp), kv_first ? 0u : 1u);
                    if (!C::kDqAlias && pp > 0 &&
                        !wait1(BAR(B_DQ_EMPTY), (uint32_t)((pp - 1) & 1), c, kRoleMma, (int)pp, 8))
                        break;
                    ptx::tc_fence_after();
                    issue_dq<D>(tDQ, sDS, sK);
                    ptx::tc_commit(BAR(B_DS_FREE));
                    ptx::tc_commit(BAR(B_DQ_FULL));
                    ptx::tc_commit(BAR(B_Q_EMPTY + (int)(pp % kStages)));
                    if (d.flags & kKvLast) {
                        ptx::tc_commit(BAR(B_ACC_FULL));
                        ptx::tc_commit(BAR(B_KV_EMPTY));
                    }
                    if (!has_next) break;
                    if (next_new_kv) {
                        ++kvc;
                        if (!wait1(BAR(B_KV_FULL), (uint32_t)(kvc & 1), c, kRoleMma, (int)pp, 9)) break;
                        if (!wait1(BAR(B_Q_FULL + (int)((pp + 1) % kStages)), q_par(pp + 1), c, kRoleMma,
                                   (int)pp, 6))
                            break;
                        ptx::tc_fence_after();
                        issue_s<D>(tS, sK, sQ(pp + 1));
                        ptx::tc_commit(BAR(B_S_FULL));
                    }
                    if (C::kDqAlias &&
                        !wait1(BAR(B_DQ_EMPTY), (uint32_t)(pp & 1), c, kRoleMma, (int)pp, 10))
                        break;
                    ptx::tc_fence_after();
                    issue_s<D>(tDP, sV, sQ(pp + 1) + C::kTile);
                    ptx::tc_commit(BAR(B_DP_FULL));
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
            const int st = (int)(pp % kStages);
            const float* vec = reinterpret_cast<const float*>(smem + C::OFF_VEC + st * 1024);
            if (!waitw(BAR(B_S_FULL), (uint32_t)(pp & 1), c, kRoleSoftmax, (int)pp, 1)) break;
            ptx::tc_fence_after();
            float P[64];
            softmax_64(tmem + lane_off + C::COL_S, c0, vec, p.scale_log2e, (d.flags & kDiag) != 0, row, P);
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(BAR(B_P_READY));
            if (!waitw(BAR(B_DP_FULL), (uint32_t)(pp & 1), c, kRoleSoftmax, (int)pp, 2)) break;
            ptx::tc_fence_after();
            uint32_t pk[32];
            ds_64(tmem + lane_off + C::COL_DP, c0, vec + 128, p.scale, P, pk);
            ptx::tc_fence_before();
            if (pp > 0 && !waitw(BAR(B_DS_FREE), (uint32_t)((pp - 1) & 1), c, kRoleSoftmax, (int)pp, 3)) break;
            store_row_sw128(ds_box, row, pk);
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(BAR(B_DS_READY));
                ptx::mbar_arrive(BAR(B_Q_EMPTY + st));
            }
        }
    } else if (warp < 4) {
        // ================================================== reducer + dK/dV epilogue
        const int row = 32 * warp + lane;
        const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
        int kvc = 0;
        for (long long pp = 0;; ++pp) {
            const int ds = (int)(pp % kNDesc);
            bool fail = !waitw(BAR(B_DESC_FULL + ds), (uint32_t)((pp / kNDesc) & 1), c, kRoleReducer, (int)pp, 0);
            if (reducer_bar_or(fail)) break;
            const PairDesc d = descs[ds];
            if (d.flags & kEnd) break;
            fail = !waitw(BAR(B_DQ_FULL), (uint32_t)(pp & 1), c, kRoleReducer, (int)pp, 1);
            if (reducer_bar_or(fail)) break;
            ptx::tc_fence_after();
            const int tile = (d.b * p.Hq + d.hq) * p.n + d.q;
            fail = false;
            if (ordered && warp == 0 && lane == 0) {
                int* sem = p.sem + tile;
                if (ptx::ld_acquire(sem) != d.rank) {
                    const uint64_t t0 = ptx::globaltimer();
                    int spins = 0;
                    for (;;) {
                        if (ptx::ld_acquire(sem) == d.rank) break;
                        if ((++spins & 63) == 0) {
                            if (ptx::ld_volatile(p.abort_flag) || *abort_smem) {
                                fail = true;
                                break;
                            }
                            if (ptx::globaltimer() - t0 > c.timeout) {
                                report_timeout(c, kRoleReducer, d.b * p.Hq + d.hq, d.q, d.rank);
                                fail = true;
                                break;
                            }
                        }
                        __nanosleep(64);
                    }
                }
                __threadfence();
            }
            if (reducer_bar_or(fail)) break;
            float* gdq = p.dq + ((size_t)(d.b * p.Hq + d.hq) * p.S + (size_t)d.q * 128 + row) * D;
            float* gpart = p.partials
                               ? p.partials + (((size_t)tile * p.n + d.kv) * 128 + row) * D
                               : nullptr;
            // Drain dQ from tensor memory 64 columns per wait; the columns are
            // handed back to the MMA issuer before the last reductions go out.
#pragma unroll 1
            for (int cc = 0; cc < D / 64; ++cc) {
                uint32_t r0[32], r1[32];
                ptx::tmem_ld32(tmem + lane_off + C::COL_DQ + 64 * cc, r0);
                ptx::tmem_ld32(tmem + lane_off + C::COL_DQ + 64 * cc + 32, r1);
                ptx::tmem_ld_wait();
                if (cc == D / 64 - 1) {
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(BAR(B_DQ_EMPTY));
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float* g = gdq + 64 * cc + 4 * e;
                    ptx::red_add_v4(g, __uint_as_float(r0[4 * e]), __uint_as_float(r0[4 * e + 1]),
                                    __uint_as_float(r0[4 * e + 2]), __uint_as_float(r0[4 * e + 3]));
                    ptx::red_add_v4(g + 32, __uint_as_float(r1[4 * e]), __uint_as_float(r1[4 * e + 1]),
                                    __uint_as_float(r1[4 * e + 2]), __uint_as_float(r1[4 * e + 3]));
                    if (gpart) {
                        float* gp = gpart + 64 * cc + 4 * e;
                        *reinterpret_cast<float4*>(gp) =
                            make_float4(__uint_as_float(r0[4 * e]), __uint_as_float(r0[4 * e + 1]),
                                        __uint_as_float(r0[4 * e + 2]), __uint_as_float(r0[4 * e + 3]));
                        *reinterpret_cast<float4*>(gp + 32) =
                            make_float4(__uint_as_float(r1[4 * e]), __uint_as_float(r1[4 * e + 1]),
                                        __uint_as_float(r1[4 * e + 2]), __uint_as_float(r1[4 * e + 3]));
                    }
                }
            }
            if (ordered || p.order_log) {
                __threadfence();
                ptx::named_bar_sync(1, 128);
                if (warp == 0 && lane == 0) {
                    if (p.order_log) {
                        const int s = atomicAdd(p.logcnt + tile, 1);
                        if (s >= 0 && s < p.n) p.order_log[(size_t)tile * p.n + s] = d.kv;
                    }
                    if (ordered) ptx::st_release(p.sem + tile, d.rank + 1);
                }
            }
            if (lane == 0) ptx::mbar_arrive(BAR(B_DESC_EMPTY + ds));
            if (d.flags & kKvLast) {
                fail = !waitw(BAR(B_ACC_FULL), (uint32_t)(kvc & 1), c, kRoleReducer, (int)pp, 2);
                if (reducer_bar_or(fail)) break;
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
                            __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(r[2 * e]),
                                                                      __uint_as_float(r[2 * e + 1]));
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
}

template <int D>
int launch_bwd(const BwdParams& prm, int grid, cudaStream_t stream) {
    using C = Cfg<D>;
    static bool attr_done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -2;
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(dash_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) !=
            cudaSuccess)
            return -2;
        attr_done[dev] = true;
    }
    void* args[] = {(void*)&prm};
    cudaError_t e = cudaLaunchCooperativeKernel((const void*)dash_bwd_kernel<D>, dim3(grid), dim3(kThreads),
                                                args, C::kSmem, stream);
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
        cudaFuncSetAttribute(dash_bwd_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<64>::kSmem);
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dash_bwd_kernel<64>, kThreads, Cfg<64>::kSmem);
    } else {
        cudaFuncSetAttribute(dash_bwd_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<128>::kSmem);
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dash_bwd_kernel<128>, kThreads,
                                                          Cfg<128>::kSmem);
    }
    if (e != cudaSuccess) return -2;
    if (per_sm < 1) return -3;
    *P = sms;   // one persistent CTA per SM
    return 0;
}

int launch_bwd_dispatch(int D, const BwdParams& prm, int grid, cudaStream_t stream) {
    return D == 64 ? launch_bwd<64>(prm, grid, stream) : launch_bwd<128>(prm, grid, stream);
}

int bwd_smem_bytes(int D) { return D == 64 ? Cfg<64>::kSmem : Cfg<128>::kSmem; }

}  // namespace dash
