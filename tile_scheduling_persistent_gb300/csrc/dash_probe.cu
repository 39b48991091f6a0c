// dash_probe.cu -- one (KV tile, Q tile) pair through the same device building
// blocks as the persistent kernel (TMA boxes, the five tcgen05 products, the
// softmax / dS warps), one CTA, no pipelining.  Every intermediate is written
// out so that tests can check each operand layout on its own.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dash_bwd.cuh"
#include "dash_internal.h"

namespace dash {

namespace {

struct ProbeParams {
    CUtensorMap tm_k, tm_v, tm_q, tm_do;
    const float* lse;
    const float* delta;
    float *sT, *pT, *dpT, *dsT, *dv, *dk, *dq;
    int* err;
    int diag;
    float scale, scale_log2e;
};

__device__ bool probe_wait(uint32_t bar, uint32_t parity, int* err) {
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer() - t0 > 1000000000ull) {
            atomicExch(err, 1);
            return false;
        }
    }
    return true;
}

template <int D>
__global__ void __launch_bounds__(256, 1) probe_kernel(const __grid_constant__ ProbeParams p) {
    using C = Cfg<D>;
    constexpr int T = C::kTile;
    extern __shared__ __align__(1024) uint8_t smem[];
    // layout: K, V, Q, dO tiles, dS^T (2 boxes), LSE/delta, barriers
    const uint32_t sbase = ptx::smem_u32(smem);
    const uint32_t sK = sbase, sV = sbase + T, sQ = sbase + 2 * T, sDO = sbase + 3 * T, sDS = sbase + 4 * T;
    uint8_t* ctl = smem + 4 * T + 2 * kBox + 1024;
    const uint32_t bar_tma = ptx::smem_u32(ctl), bar_mma = bar_tma + 8;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(ctl + 64);
    volatile int* bad = reinterpret_cast<volatile int*>(ctl + 68);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        *bad = (sbase & 1023u) ? 1 : 0;
        if (sbase & 1023u) atomicExch(p.err, 2);
        ptx::mbar_init(bar_tma, 1);
        ptx::mbar_init(bar_mma, 1);
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(ptx::smem_u32((const void*)tmem_slot), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = *bad == 0;
    if (ok && threadIdx.x == 0) {
        ptx::mbar_arrive_expect_tx(bar_tma, 4 * T);
        for (int bx = 0; bx < C::kNBox; ++bx) {
            ptx::tma_load_2d(sK + bx * kBox, &p.tm_k, 64 * bx, 0, bar_tma);
            ptx::tma_load_2d(sV + bx * kBox, &p.tm_v, 64 * bx, 0, bar_tma);
            ptx::tma_load_2d(sQ + bx * kBox, &p.tm_q, 64 * bx, 0, bar_tma);
            ptx::tma_load_2d(sDO + bx * kBox, &p.tm_do, 64 * bx, 0, bar_tma);
        }
    }
    if (ok) ok = probe_wait(bar_tma, 0, p.err);
    ok = __syncthreads_and(ok);
    if (ok && threadIdx.x == 0) {
        ptx::tc_fence_after();
        issue_s<D>(tmem + C::COL_S, sK, sQ);
        issue_s<D>(tmem + C::COL_DP, sV, sDO);
        ptx::tc_commit(bar_mma);
    }
    if (ok) ok = probe_wait(bar_mma, 0, p.err);
    ok = __syncthreads_and(ok);

    const int sub = warp & 3, c0 = 64 * (warp >> 2), row = 32 * sub + lane;
    const uint32_t lane_off = (uint32_t)(32 * sub) << 16;
    const float lse2_a = p.lse[c0 + lane] * kLog2e, lse2_b = p.lse[c0 + 32 + lane] * kLog2e;
    const float delta_a = p.delta[c0 + lane], delta_b = p.delta[c0 + 32 + lane];
    float P[64];
    if (ok) {
        ptx::tc_fence_after();
        uint32_t r[32];
        for (int h = 0; h < 2; ++h) {
            ptx::tmem_ld32(tmem + lane_off + C::COL_S + c0 + 32 * h, r);
            ptx::tmem_ld_wait();
            for (int k = 0; k < 32; ++k) p.sT[row * 128 + c0 + 32 * h + k] = __uint_as_float(r[k]);
        }
        softmax_64<false>(tmem + lane_off + C::COL_S, c0, lse2_a, lse2_b, p.scale_log2e, p.diag != 0, p.diag != 0, row, 128,
                   128, 1 << 30, P);
        for (int k = 0; k < 64; ++k) p.pT[row * 128 + c0 + k] = P[k];
        ptx::tc_fence_before();
    }
    ok = __syncthreads_and(ok);
    if (ok && threadIdx.x == 0) {
        ptx::tc_fence_after();
        issue_dv<D>(tmem + C::COL_DV, tmem + C::COL_S, sDO, 0);
        ptx::tc_commit(bar_mma);
    }
    if (ok) ok = probe_wait(bar_mma, 1, p.err);
    ok = __syncthreads_and(ok);
    if (ok) {
        ptx::tc_fence_after();
        uint32_t r[32];
        for (int h = 0; h < 2; ++h) {
            ptx::tmem_ld32(tmem + lane_off + C::COL_DP + c0 + 32 * h, r);
            ptx::tmem_ld_wait();
            for (int k = 0; k < 32; ++k) p.dpT[row * 128 + c0 + 32 * h + k] = __uint_as_float(r[k]);
        }
        uint8_t* box = smem + 4 * T + (c0 >> 6) * kBox;
        ds_64(tmem + lane_off + C::COL_DP, c0, delta_a, delta_b, p.scale, P, box, row);
        ptx::tc_fence_before();
        ptx::fence_proxy_async_smem();
        // read the bf16 dS^T row back (unswizzled) for the dump
        for (int cc = 0; cc < 8; ++cc) {
            const uint4 v4 = *reinterpret_cast<const uint4*>(box + row * 128 + ((cc ^ (row & 7)) << 4));
            const uint32_t w4[4] = {v4.x, v4.y, v4.z, v4.w};
            for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[e]));
                p.dsT[row * 128 + c0 + 8 * cc + 2 * e] = f.x;
                p.dsT[row * 128 + c0 + 8 * cc + 2 * e + 1] = f.y;
            }
        }
    }
    ok = __syncthreads_and(ok);
    if (ok && threadIdx.x == 0) {
        ptx::tc_fence_after();
        issue_dk<D>(tmem + C::COL_DK, sDS, sQ, 0);
        issue_dq<D>(tmem + C::COL_DQ, sDS, sK);
        ptx::tc_commit(bar_mma);
    }
    if (ok) ok = probe_wait(bar_mma, 0, p.err);
    ok = __syncthreads_and(ok);
    if (ok && warp < 4) {
        ptx::tc_fence_after();
        const uint32_t cols[3] = {C::COL_DV, C::COL_DK, C::COL_DQ};
        float* outs[3] = {p.dv, p.dk, p.dq};
        for (int m = 0; m < 3; ++m) {
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t r[32];
                ptx::tmem_ld32(tmem + lane_off + cols[m] + 32 * cc, r);
                ptx::tmem_ld_wait();
                for (int k = 0; k < 32; ++k) outs[m][row * D + 32 * cc + k] = __uint_as_float(r[k]);
            }
        }
    }
    // Every commit was waited for (or timed out); make sure the MMAs are done.
    if (threadIdx.x == 0) {
        ptx::tc_commit(bar_tma);   // reuse: phase 1 of bar_tma
        const uint64_t t0 = ptx::globaltimer();
        while (!ptx::mbar_try_wait(bar_tma, 1) && ptx::globaltimer() - t0 < 100000000ull) {
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

template <int D>
int run_probe_t(const void* k, const void* v, const void* q, const void* dO, const float* lse, const float* delta,
                int diag, float* sT, float* pT, float* dpT, float* dsT, float* dv, float* dk, float* dq) {
    ProbeParams prm;
    if (make_tmap_2d(&prm.tm_k, k, 128, D) || make_tmap_2d(&prm.tm_v, v, 128, D) ||
        make_tmap_2d(&prm.tm_q, q, 128, D) || make_tmap_2d(&prm.tm_do, dO, 128, D))
        return -2;
    int* err = nullptr;
    if (cudaMalloc(&err, sizeof(int)) != cudaSuccess) return -6;
    cudaMemset(err, 0, sizeof(int));
    prm.lse = lse;
    prm.delta = delta;
    prm.sT = sT;
    prm.pT = pT;
    prm.dpT = dpT;
    prm.dsT = dsT;
    prm.dv = dv;
    prm.dk = dk;
    prm.dq = dq;
    prm.err = err;
    prm.diag = diag;
    prm.scale = 1.0f / sqrtf((float)D);
    prm.scale_log2e = prm.scale * kLog2e;
    const int smem = 4 * Cfg<D>::kTile + 2 * kBox + 1024 + 128;
    cudaFuncSetAttribute(probe_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    probe_kernel<D><<<1, 256, smem>>>(prm);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    int h_err = 0;
    if (e == cudaSuccess) cudaMemcpy(&h_err, err, sizeof(int), cudaMemcpyDeviceToHost);
    cudaFree(err);
    if (e != cudaSuccess) return -2;
    return h_err ? -4 : 0;
}

}  // namespace

int run_tile_probe(const void* k, const void* v, const void* q, const void* dO, const float* lse,
                   const float* delta, int D, int diag, float* sT, float* pT, float* dpT, float* dsT,
                   float* dv, float* dk, float* dq) {
    if (D == 64) return run_probe_t<64>(k, v, q, dO, lse, delta, diag, sT, pT, dpT, dsT, dv, dk, dq);
    if (D == 128) return run_probe_t<128>(k, v, q, dO, lse, delta, diag, sT, pT, dpT, dsT, dv, dk, dq);
    return -1;
}

}  // namespace dash
