// dash_internal.h -- declarations shared by the translation units of libdash.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace dash {

struct BwdParams;

// Persistent backward kernel (dash_bwd.cu).
int launch_bwd_dispatch(int D, const BwdParams& prm, int grid, cudaStream_t stream);
int bwd_max_ctas(int D, int device, int* P);
int bwd_smem_bytes(int D);
int load_bwd_kernels();   // load every production variant on the current device

// Auxiliary kernels (dash_aux.cu).
int launch_preprocess(const void* o, const void* dO, float* delta, long long rows, int D, cudaStream_t s);
int launch_finalize(const float* src, void* dst, size_t numel, cudaStream_t s);
// dK / dV of a backward run with one task per query head: out bf16
// [B, Hkv, Skv, D] = the fp32 part [B, Hkv*G, Skv, D] summed over each group
// of G query heads in ascending order.
int load_aux_kernels();   // load the auxiliary backward kernels on the current device
int launch_group_sum(const float* part, void* out, int B, int Hkv, int G, int Skv, int D, cudaStream_t s);
// Key-block split of the backward with different query and key lengths:
// dst [BH][G][bytes_per_head] = G copies of each head's src [BH][bytes_per_head];
// out fp32 [BH][elems] = part [BH][G][elems] summed over G in ascending order.
int launch_replicate(const void* src, void* dst, long long bytes_per_head, long long BH, int G, cudaStream_t s);
int launch_block_sum(const float* part, float* out, long long BH, int G, long long elems_per_head, cudaStream_t s);
// Accumulation ranks of a static schedule, built on the device:
// ranks [B*Hq*n][n] (uint16), scratch `time` [B*Hq*n][n] (uint32),
// `task_start` [num_tasks] (uint32).
int launch_build_ranks(int B, int Hq, int Hkv, int n, int causal, int sched, int P, uint16_t* ranks,
                       uint32_t* time, uint32_t* task_start, cudaStream_t s, int win = 0, int nk = 0);

// Attention forward (dash_fwd.cu): O bf16 [B,Hq,S,D], LSE fp32 [B,Hq,S];
// status = the stream workspace's status word (cleared by the caller).
int launch_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int* status, int B, int Hq,
               int Hkv, int S, int D, int causal, int window, unsigned long long timeout_ns, cudaStream_t stream,
               int Skv = 0);

// Single-tile probe (dash_probe.cu).
int run_tile_probe(const void* k, const void* v, const void* q, const void* dO, const float* lse,
                   const float* delta, int D, int diag, float* sT, float* pT, float* dpT, float* dsT,
                   float* dv, float* dk, float* dq);

// Timeout of every device-side wait, in ns, as dash_set_timeout_ns set it (dash_api.cu).
unsigned long long timeout_ns();

// Tensor maps (dash_api.cu).
int make_tmap_2d(void* map_out, const void* base, long long rows, int D);
int make_tmap_3d(void* map_out, const void* base, long long heads, int S, int D);
int make_tmap_2d_f32(void* map_out, const void* base, long long rows, int D);

}  // namespace dash
