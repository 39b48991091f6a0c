// dash_noalloc.cu -- dash_attn_bwd_noalloc: the deterministic backward pass
// for callers that cannot allocate device memory, with all library scratch
// taken from one fixed file-scope device array.
//
// Who needs this: a caller that has handed the whole device to its own pool
// allocator (so cudaMalloc would fail or fragment that pool), or one on a
// latency-critical path where the implicit device synchronization of
// cudaMalloc / cudaFree is not acceptable, or one that must not allocate at
// all after initialisation.  dash_attn_bwd grows a per-(device, stream)
// workspace with cudaMalloc on first use; this entry point never allocates.
//
// The scratch (delta, the per-tile accumulation counters, the status word
// and the schedule's rank tables) lives in g_scratch below: kScratchBytes on
// every GPU that loads the library, held until the process exits.  The
// array keeps whatever the previous call left in it, so everything that
// must start at zero is cleared on the stream at the start of each call, and
// two calls whose executions overlap on the GPU (different streams, or
// different host threads) race on the array.
//
// Set-up, once per device: dash_noalloc_init (or else the first call) looks
// up the device address of g_scratch with that device current and loads the
// backward kernels.  Under lazy module loading that is when the driver loads
// the library's module and reserves the array's memory, so it belongs before
// a caller's pool takes the device and before its latency-critical path or
// any stream capture.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "../../include/dash.h"
#include "dash_bwd.cuh"
#include "dash_internal.h"
#include "dash_schedule.h"

namespace dash {
namespace {

constexpr size_t kScratchBytes = 8u << 20;   // 8 MiB per device
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Looks up the device address of g_scratch on `dev` (the current device) and
// loads the kernels this entry point launches.  In host code the symbol is
// only a host-side stand-in; the kernels get the looked-up address.
int setup_device(int dev) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) {
        (void)cudaGetLastError();
        return DASH_ERR_CUDA;
    }
    int P = 0;
    if (bwd_max_ctas(64, dev, &P) || bwd_max_ctas(128, dev, &P) || load_bwd_kernels() || load_aux_kernels()) {
        (void)cudaGetLastError();
        return DASH_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
    return DASH_OK;
}

// Device address of g_scratch on `dev`, set up on first use.
int scratch_for_device(int dev, unsigned char** out) {
    if (dev < 0 || dev >= kMaxDevices) return DASH_ERR_DEVICE;
    std::lock_guard<std::mutex> lk(g_setup_mu);
    if (!g_scratch_ptr[dev]) {
        const int rc = setup_device(dev);
        if (rc) return rc;
    }
    *out = static_cast<unsigned char*>(g_scratch_ptr[dev]);
    return DASH_OK;
}

int current_sm103(int* dev) {
    int major = 0, minor = 0;
    if (cudaGetDevice(dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev) != cudaSuccess)
        return DASH_ERR_CUDA;
    return (major == 10 && minor == 3) ? DASH_OK : DASH_ERR_DEVICE;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace
}  // namespace dash

using namespace dash;

extern "C" int dash_attn_bwd_noalloc(const dash_bf16* q, const dash_bf16* k, const dash_bf16* v, const dash_bf16* o,
                                     const dash_bf16* dO, const float* lse, float* dq, dash_bf16* dk, dash_bf16* dv,
                                     int B, int Hq, int Hkv, int S, int D, int causal, int schedule,
                                     dash_stream_t stream_) {
    cudaStream_t stream = (cudaStream_t)stream_;
    const void* ptrs[] = {q, k, v, o, dO, lse, dq, dk, dv};
    for (const void* ptr : ptrs)
        if (!ptr || ((uintptr_t)ptr & 15u)) return DASH_ERR_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || S <= 0 || (D != 64 && D != 128) || Hq % Hkv ||
        (causal != 0 && causal != 1) || schedule < 0 || schedule > kAuto || (long long)B * Hq * S >= (1ll << 31) ||
        (S + 127) / 128 > 65535)
        return DASH_ERR_ARG;
    if (schedule == kAuto) schedule = select_schedule(D, causal);
    int dev = 0;
    int rc = current_sm103(&dev);
    if (rc) return rc;
    int P = 0;
    rc = bwd_max_ctas(D, dev, &P);
    if (rc == -3) return DASH_ERR_LAUNCH;
    if (rc) return DASH_ERR_CUDA;

    const int n = (S + 127) / 128;   // the last tile may be partial
    const Shape sh{B, Hq, Hkv, n, Hq / Hkv, causal, schedule, 0, 0};   // no window, equal lengths
    const long long tiles = (long long)B * Hq * n;
    const long long entries = tiles * n;
    const long long ntasks = num_tasks(sh);
    const bool tables = is_static(schedule);

    // Carve the scratch: counters (cleared every call), delta, rank tables.
    const size_t n_ints = 16 + (size_t)(kSubTiles + 1) * tiles;
    const size_t off_ints = 0;
    const size_t off_delta = align256(off_ints + n_ints * sizeof(int));
    const size_t off_ranks = align256(off_delta + (size_t)tiles * 128 * sizeof(float));
    const size_t off_time = align256(off_ranks + (tables ? (size_t)entries * sizeof(uint16_t) : 0));
    const size_t off_start = align256(off_time + (tables ? (size_t)entries * sizeof(uint32_t) : 0));
    const size_t need = off_start + (tables ? (size_t)ntasks * sizeof(uint32_t) : 0);
    if (need > kScratchBytes) return DASH_ERR_SCRATCH;

    unsigned char* base = nullptr;
    if ((rc = scratch_for_device(dev, &base))) return rc;
    int* ints = reinterpret_cast<int*>(base + off_ints);
    float* delta = reinterpret_cast<float*>(base + off_delta);
    uint16_t* ranks = tables ? reinterpret_cast<uint16_t*>(base + off_ranks) : nullptr;

    if (tables && launch_build_ranks(B, Hq, Hkv, n, causal, schedule, P, ranks,
                                     reinterpret_cast<uint32_t*>(base + off_time),
                                     reinterpret_cast<uint32_t*>(base + off_start), stream))
        return DASH_ERR_CUDA;
    if (cudaMemsetAsync(ints, 0, n_ints * sizeof(int), stream) != cudaSuccess ||
        cudaMemsetAsync(dq, 0, (size_t)B * Hq * S * D * sizeof(float), stream) != cudaSuccess)
        return DASH_ERR_CUDA;
    if (launch_preprocess(o, dO, delta, (long long)B * Hq * S, D, stream)) return DASH_ERR_CUDA;

    BwdParams prm;
    memset(&prm, 0, sizeof(prm));
    if (make_tmap_3d(&prm.tm_q, q, (long long)B * Hq, S, D) || make_tmap_3d(&prm.tm_k, k, (long long)B * Hkv, S, D) ||
        make_tmap_3d(&prm.tm_v, v, (long long)B * Hkv, S, D) || make_tmap_3d(&prm.tm_do, dO, (long long)B * Hq, S, D))
        return DASH_ERR_CUDA;
    prm.lse = lse;
    prm.delta = delta;
    prm.dq = dq;
    prm.dk = (__nv_bfloat16*)dk;
    prm.dv = (__nv_bfloat16*)dv;
    prm.ranks = ranks;
    prm.status = ints;
    prm.task_counter = ints + 8;
    prm.abort_flag = ints + 9;
    prm.sem = ints + 16;
    prm.logcnt = ints + 16 + kSubTiles * tiles;
    prm.timeout_ns = timeout_ns();   // as dash_set_timeout_ns set it
    prm.ntasks = ntasks;
    prm.B = B;
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.kvh = Hkv;   // one task per key/value head group (no per-head partials here)
    prm.kvg = Hq / Hkv;
    prm.S = S;
    prm.n = n;
    prm.G = Hq / Hkv;
    prm.causal = causal;
    prm.sched = schedule;
    prm.P = P;
    prm.scale = 1.0f / sqrtf((float)D);
    prm.scale_log2e = prm.scale * kLog2e;
    prm.Skv = S;   // equal query and key lengths, no window
    prm.nkv = n;
    rc = launch_bwd_dispatch(D, prm, P, stream);
    if (rc == -3) return DASH_ERR_LAUNCH;
    return rc ? DASH_ERR_CUDA : DASH_OK;
}

extern "C" int dash_noalloc_init(void) {
    int dev = 0;
    int rc = current_sm103(&dev);
    if (rc) return rc;
    if (dev >= kMaxDevices) return DASH_ERR_DEVICE;
    std::lock_guard<std::mutex> lk(g_setup_mu);
    return setup_device(dev);
}

extern "C" int dash_get_status_noalloc(dash_stream_t stream, int* code, int* info) {
    if (!code) return DASH_ERR_ARG;
    int dev = 0;
    int rc = current_sm103(&dev);
    if (rc) return rc;
    unsigned char* base = nullptr;
    if ((rc = scratch_for_device(dev, &base))) return rc;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return DASH_ERR_CUDA;
    int h[8] = {0};
    if (cudaMemcpy(h, base, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return DASH_ERR_CUDA;
    *code = h[0];
    if (info)
        for (int i = 0; i < 4; ++i) info[i] = h[1 + i];
    return DASH_OK;
}
