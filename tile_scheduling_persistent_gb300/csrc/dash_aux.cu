// dash_aux.cu -- the small kernels around the persistent backward:
//   preprocess  delta = rowsum(dO o O)            (memory bound)
//   finalize    dq_bf16 = round_to_nearest_even(dq_fp32)
//   build_ranks accumulation ranks of the static schedules (integer only)
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dash_internal.h"
#include "dash_schedule.h"

namespace dash {

namespace {

// ---------------------------------------------------------------- delta
// A group of L = D/8 lanes owns one row: each lane loads 16 B of dO and of O,
// sums its 8 products in order, then the group reduces with a fixed
// butterfly, so every row is summed in one fixed order.
template <int D>
__global__ void __launch_bounds__(256) preprocess_kernel(const uint4* __restrict__ o,
                                                         const uint4* __restrict__ dO,
                                                         float* __restrict__ delta, long long rows) {
    constexpr int L = D / 8;
    constexpr int RPW = 32 / L;   // rows per warp
    const long long warp_global = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const long long row = warp_global * RPW + lane / L;
    const int sub = lane % L;
    float acc = 0.f;
    if (row < rows) {
        const uint4 a = o[row * L + sub];
        const uint4 b = dO[row * L + sub];
        const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 fa = __bfloat1622float2(pa[e]);
            const float2 fb = __bfloat1622float2(pb[e]);
            acc = fmaf(fa.x, fb.x, acc);
            acc = fmaf(fa.y, fb.y, acc);
        }
    }
#pragma unroll
    for (int m = L / 2; m >= 1; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (row < rows && sub == 0) delta[row] = acc;
}

// ---------------------------------------------------------------- finalize
__global__ void __launch_bounds__(256) finalize_kernel(const float4* __restrict__ src, uint2* __restrict__ dst,
                                                       size_t n4) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
        const float4 v = src[i];
        __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
        __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
        dst[i] = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
    }
}

__global__ void finalize_tail_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst, size_t begin,
                                     size_t end) {
    const size_t i = begin + threadIdx.x;
    if (i < end) dst[i] = __float2bfloat16_rn(src[i]);
}

// ---------------------------------------------------------------- GQA group sum
// out[b, hk, s, :] = bf16_rn(((part[b, hk*G] + part[b, hk*G+1]) + ...) + part[b, hk*G+G-1])
// for the fp32 per-query-head dK / dV of a backward run with one task per
// query head: the group's heads are added in ascending order.  One thread per
// four consecutive elements of a key/value row (D is a multiple of 4).
__global__ void __launch_bounds__(256) group_sum_kernel(const float4* __restrict__ part, uint2* __restrict__ out,
                                                       long long rows_out, int G, long long head4) {
    // head4: float4s per head (Skv * D / 4); a head's rows are contiguous
    const long long n4 = rows_out;   // float4s in the output
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x) {
        const long long bh = i / head4, r = i - bh * head4;   // output head (b * Hkv + hk), offset
        const float4* src = part + bh * G * head4 + r;
        float4 a = src[0];
        for (int g = 1; g < G; ++g) {
            const float4 v = src[(long long)g * head4];
            a.x += v.x;
            a.y += v.y;
            a.z += v.z;
            a.w += v.w;
        }
        __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(a.z, a.w);
        out[i] = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
    }
}

// ---------------------------------------------------------------- key blocks
// Inputs of the key-block split of the backward with different query and key
// lengths: dst[bh][g][e] = src[bh][e] for g < G (T = uint4 when a head's
// array is a whole number of 16-byte words, else uint32_t).
template <typename T>
__global__ void __launch_bounds__(256) replicate_kernel(const T* __restrict__ src, T* __restrict__ dst,
                                                       long long per_head, int G, long long total) {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long bh = i / ((long long)G * per_head);
        const long long e = (i - bh * G * per_head) % per_head;
        dst[i] = src[bh * per_head + e];
    }
}

// out[bh][e] = ((part[bh][0][e] + part[bh][1][e]) + ...) + part[bh][G-1][e]
// (fp32, round to nearest): the G key blocks' dQ partial sums added in
// ascending block order.
__global__ void __launch_bounds__(256) block_sum_kernel(const float4* __restrict__ part, float4* __restrict__ out,
                                                       long long n4, int G, long long head4) {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
         i += (long long)gridDim.x * blockDim.x) {
        const long long bh = i / head4, r = i - bh * head4;
        const float4* src = part + bh * G * head4 + r;
        float4 a = src[0];
        for (int g = 1; g < G; ++g) {
            const float4 v = src[(long long)g * head4];
            a.x = __fadd_rn(a.x, v.x);
            a.y = __fadd_rn(a.y, v.y);
            a.z = __fadd_rn(a.z, v.z);
            a.w = __fadd_rn(a.w, v.w);
        }
        out[i] = a;
    }
}

// ---------------------------------------------------------------- ranks
// Model time of a pair = its position in its worker's unit-step sequence
// (worker = task % P, tasks taken in order); the accumulation rank of KV
// tile j in dQ tile t = number of contributors of t with a smaller
// (model time, KV index).
__global__ void task_start_kernel(Shape s, int P, long long ntasks, uint32_t* task_start) {
    const int w = blockIdx.x * blockDim.x + threadIdx.x;
    if (w >= P) return;
    uint32_t t = 0;
    for (long long k = w; k < ntasks; k += P) {
        task_start[k] = t;
        t += (uint32_t)task_len(s, k);
    }
}

__global__ void pair_time_kernel(Shape s, long long ntasks, const uint32_t* task_start, uint32_t* time) {
    const long long k = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= ntasks) return;
    const int L = task_len(s, k);
    const uint32_t t0 = task_start[k];
    for (int u = 0; u < L; ++u) {
        const Visit v = task_visit(s, k, u);
        time[rank_index(s, v.b, v.hq, v.q, v.kv)] = t0 + (uint32_t)u;
    }
}

__global__ void rank_kernel(int n, long long entries, const uint32_t* time, uint16_t* ranks) {
    // n: key/value tiles per head (the row length of the tables)
    const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= entries) return;
    const long long tile = e / n;
    const int j = (int)(e % n);
    const uint32_t* row = time + tile * n;
    const uint32_t tj = row[j];
    if (tj == 0xFFFFFFFFu) {
        ranks[e] = 0xFFFF;
        return;
    }
    int r = 0;
    for (int x = 0; x < n; ++x) {
        const uint32_t tx = row[x];
        if (tx == 0xFFFFFFFFu) continue;
        r += (tx < tj) || (tx == tj && x < j);
    }
    ranks[e] = (uint16_t)r;
}

}  // namespace

int launch_preprocess(const void* o, const void* dO, float* delta, long long rows, int D, cudaStream_t s) {
    if (rows <= 0) return 0;
    const int L = D / 8;
    const long long warps = (rows * L + 31) / 32;
    const long long blocks = (warps * 32 + 255) / 256;
    if (D == 64)
        preprocess_kernel<64><<<(unsigned)blocks, 256, 0, s>>>((const uint4*)o, (const uint4*)dO, delta, rows);
    else if (D == 128)
        preprocess_kernel<128><<<(unsigned)blocks, 256, 0, s>>>((const uint4*)o, (const uint4*)dO, delta, rows);
    else
        return -1;
    return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

int launch_finalize(const float* src, void* dst, size_t numel, cudaStream_t s) {
    const size_t n4 = numel / 4;
    if (n4) {
        int dev = 0, sms = 148;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        size_t blocks = (n4 + 255) / 256;
        const size_t cap = (size_t)sms * 8;
        if (blocks > cap) blocks = cap;
        finalize_kernel<<<(unsigned)blocks, 256, 0, s>>>((const float4*)src, (uint2*)dst, n4);
    }
    if (numel % 4) finalize_tail_kernel<<<1, 32, 0, s>>>(src, (__nv_bfloat16*)dst, n4 * 4, numel);
    return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

int launch_group_sum(const float* part, void* out, int B, int Hkv, int G, int Skv, int D, cudaStream_t s) {
    const long long head4 = (long long)Skv * D / 4;
    const long long n4 = (long long)B * Hkv * head4;
    if (n4 == 0) return 0;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    long long blocks = (n4 + 255) / 256;
    const long long cap = (long long)sms * 8;
    if (blocks > cap) blocks = cap;
    group_sum_kernel<<<(unsigned)blocks, 256, 0, s>>>((const float4*)part, (uint2*)out, n4, G, head4);
    return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

namespace {
long long grid_for(long long n) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long blocks = (n + 255) / 256, cap = (long long)sms * 8;
    return blocks < cap ? blocks : cap;
}
}  // namespace

int launch_replicate(const void* src, void* dst, long long bytes_per_head, long long BH, int G, cudaStream_t s) {
    if (BH <= 0 || bytes_per_head <= 0 || bytes_per_head % 4) return -1;
    if (bytes_per_head % 16 == 0) {
        const long long per = bytes_per_head / 16, total = BH * G * per;
        replicate_kernel<uint4><<<(unsigned)grid_for(total), 256, 0, s>>>((const uint4*)src, (uint4*)dst, per, G, total);
    } else {
        const long long per = bytes_per_head / 4, total = BH * G * per;
        replicate_kernel<uint32_t><<<(unsigned)grid_for(total), 256, 0, s>>>((const uint32_t*)src, (uint32_t*)dst, per,
                                                                             G, total);
    }
    return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

int launch_block_sum(const float* part, float* out, long long BH, int G, long long elems_per_head, cudaStream_t s) {
    if (elems_per_head % 4) return -1;
    const long long head4 = elems_per_head / 4, n4 = BH * head4;
    if (n4 == 0) return 0;
    block_sum_kernel<<<(unsigned)grid_for(n4), 256, 0, s>>>((const float4*)part, (float4*)out, n4, G, head4);
    return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

// Loads (on the current device) the auxiliary kernels of the backward pass:
// under lazy module loading a kernel's module is otherwise loaded at its first
// launch.
int load_aux_kernels() {
    cudaFuncAttributes fa;
    const void* fns[] = {(const void*)preprocess_kernel<64>, (const void*)preprocess_kernel<128>,
                         (const void*)finalize_kernel, (const void*)finalize_tail_kernel,
                         (const void*)task_start_kernel, (const void*)pair_time_kernel, (const void*)rank_kernel};
    for (const void* f : fns)
        if (cudaFuncGetAttributes(&fa, f) != cudaSuccess) return -2;
    return 0;
}

int launch_build_ranks(int B, int Hq, int Hkv, int n, int causal, int sched, int P, uint16_t* ranks,
                       uint32_t* time, uint32_t* task_start, cudaStream_t st, int win, int nk) {
    const Shape s{B, Hq, Hkv, n, Hq / Hkv, causal, sched, win, nk};
    const int nkv = num_kv(s);
    const long long ntasks = num_tasks(s);
    const long long entries = (long long)B * Hq * n * nkv;
    if (cudaMemsetAsync(time, 0xFF, (size_t)entries * sizeof(uint32_t), st) != cudaSuccess) return -2;
    task_start_kernel<<<(P + 127) / 128, 128, 0, st>>>(s, P, ntasks, task_start);
    pair_time_kernel<<<(unsigned)((ntasks + 127) / 128), 128, 0, st>>>(s, ntasks, task_start, time);
    rank_kernel<<<(unsigned)((entries + 255) / 256), 256, 0, st>>>(nkv, entries, time, ranks);
    return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

}  // namespace dash
