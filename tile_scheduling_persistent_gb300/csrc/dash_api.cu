// dash_api.cu -- the C ABI of libdash.so (declared in include/dash.h):
// argument validation, the per-(device, stream) workspace, tensor maps and
// the launch sequence  tables (cached) -> zero dq / counters -> delta ->
// persistent backward.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/dash.h"
#include "dash_bwd.cuh"
#include "dash_internal.h"
#include "dash_schedule.h"

namespace dash {

namespace {

std::atomic<unsigned long long> g_timeout_ns{2000000000ull};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Growable device buffer.
struct DevBuf {
    void* p = nullptr;
    size_t cap = 0;
    int ensure(size_t bytes) {
        if (bytes <= cap) return 0;
        if (p) cudaFree(p);
        p = nullptr;
        cap = 0;
        size_t want = bytes < 4096 ? 4096 : bytes;
        if (cudaMalloc(&p, want) != cudaSuccess) {
            (void)cudaGetLastError();
            return -6;
        }
        cap = want;
        return 0;
    }
    void release() {
        if (p) cudaFree(p);
        p = nullptr;
        cap = 0;
    }
};

// ints layout: [0..7] status, [8] task counter, [9] abort, then the
// accumulation counters [T][kSubTiles] and the order-log cursors [T].
constexpr int kIntHeader = 16;

struct Workspace {
    DevBuf delta, ints, ranks, time, task_start, dbg_ranks, part, kb;
    long long table_key[8] = {-1, -1, -1, -1, -1, -1, -1, -1};
    void release() {
        delta.release();
        ints.release();
        ranks.release();
        time.release();
        task_start.release();
        dbg_ranks.release();
        part.release();
        kb.release();
        for (auto& k : table_key) k = -1;
    }
};

std::mutex g_mu;
std::map<std::pair<int, uintptr_t>, Workspace*>& workspaces() {
    static auto* m = new std::map<std::pair<int, uintptr_t>, Workspace*>();
    return *m;
}

Workspace* get_ws(int dev, cudaStream_t s) {
    std::lock_guard<std::mutex> lk(g_mu);
    auto key = std::make_pair(dev, (uintptr_t)s);
    auto& m = workspaces();
    auto it = m.find(key);
    if (it != m.end()) return it->second;
    Workspace* w = new Workspace();
    m[key] = w;
    return w;
}

bool aligned16(const void* p) { return p && (((uintptr_t)p) & 15u) == 0; }

int check_device(int* dev_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DASH_ERR_CUDA;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return DASH_ERR_CUDA;
    if (major != 10 || minor != 3) return DASH_ERR_DEVICE;
    *dev_out = dev;
    return DASH_OK;
}

int validate_shape(int B, int Hq, int Hkv, int S, int D, int causal, int schedule) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || S <= 0) return DASH_ERR_ARG;
    if (D != 64 && D != 128) return DASH_ERR_ARG;
    if (Hq % Hkv != 0) return DASH_ERR_ARG;
    if (causal != 0 && causal != 1) return DASH_ERR_ARG;
    if (schedule < 0 || schedule > kAuto) return DASH_ERR_ARG;
    if ((long long)B * Hq * S >= (1ll << 31)) return DASH_ERR_ARG;
    if ((S + 127) / 128 > 65535) return DASH_ERR_ARG;
    return DASH_OK;
}

// Pairs on the busiest of P workers when the tasks of `s` are dealt round-robin.
long long max_worker_load(const Shape& s, int P) {
    std::vector<long long> load((size_t)P, 0);
    const long long nt = num_tasks(s);
    for (long long k = 0; k < nt; ++k) load[(size_t)(k % P)] += task_len(s, k);
    long long m = 0;
    for (long long x : load) m = x > m ? x : m;
    return m;
}

// Grouped-query heads on a static schedule (D = 128): run one task per query head
// (instead of one per key/value head group) when that takes more than 2% off
// the busiest worker's pair count.  With few, long group tasks the last wave
// leaves many SMs idle (causal Hq = 32, Hkv = 8, S = 16384, symmetric shift:
// 512 tasks of 516 pairs on 152 SMs, the busiest worker at 1.19x the mean);
// per-head tasks fill it (2048 tasks, 1.04x).  A pure function of the shape
// and P, like the schedule itself.
int head_split_helps(const Shape& grouped, int P, int D) {
    if (D != 128 || grouped.G <= 1 || !is_static(grouped.sched) || P <= 0) return 0;   // partials: D = 128
    Shape split = grouped;
    split.Hkv = grouped.Hq;
    split.G = 1;
    return max_worker_load(split, P) * 102 < max_worker_load(grouped, P) * 100 ? 1 : 0;
}

// head_split_helps, remembered per (shape, P): the decision walks every task
// twice, which should not be paid again on every call of the same shape.
int head_split_cached(const Shape& g, int P, int D) {
    if (D != 128 || g.G <= 1 || !is_static(g.sched) || P <= 0) return 0;
    static std::mutex mu;
    static std::map<std::vector<long long>, int> memo;
    const std::vector<long long> key{g.B, g.Hq, g.Hkv, g.n, g.causal, g.sched, g.win, g.nk, P, D};
    std::lock_guard<std::mutex> lk(mu);
    auto it = memo.find(key);
    if (it != memo.end()) return it->second;
    if (memo.size() >= 4096) memo.clear();
    const int v = head_split_helps(g, P, D);
    memo[key] = v;
    return v;
}

// delta_in: delta [B*Hq][S] computed by the caller (o is then not read), or null.
int bwd_impl(const dash_bf16* q, const dash_bf16* k, const dash_bf16* v, const dash_bf16* o, const dash_bf16* dO,
             const float* lse, float* dq, dash_bf16* dk, dash_bf16* dv, int B, int Hq, int Hkv, int S, int D,
             int causal, int schedule, cudaStream_t stream, const dash_debug_opts* dbg, int window = 0,
             int Skv = 0, const float* delta_in = nullptr) {
    const void* ptrs[] = {q, k, v, o, dO, lse, dq, dk, dv};
    for (const void* ptr : ptrs)
        if (!aligned16(ptr)) return DASH_ERR_ARG;
    int rc = validate_shape(B, Hq, Hkv, S, D, causal, schedule);
    if (rc) return rc;
    if (window < 0 || (window > 0 && !causal)) return DASH_ERR_ARG;
    if (window >= S) window = 0;   // a window that covers the sequence is the causal mask
    const int win = window ? band_tiles(window) : 0;
    if (win && dbg && dbg->ranks_host) return DASH_ERR_ARG;   // the table check knows no window
    if (Skv == 0) Skv = S;
    if (Skv < 0 || (Skv != S && (causal || (dbg && dbg->ranks_host))) || (Skv + 127) / 128 > 65535 ||
        (long long)B * Hkv * Skv >= (1ll << 31))
        return DASH_ERR_ARG;   // different lengths: full mask only
    // auto: different lengths run descending Q (with one ordered chain per dQ tile, measured best for 1K
    // queries x 8K keys on GB300: descending 153, ascending 148, shift 85 TFLOP/s; the key-block path of
    // dash_attn_bwd_cross calls this with the square block shape, where the shape table applies)
    if (schedule == kAuto) schedule = (Skv != S) ? kDescending : select_schedule(D, causal);
    int dev = 0;
    if ((rc = check_device(&dev))) return rc;
    int P = 0;
    rc = bwd_max_ctas(D, dev, &P);
    if (rc == -3) return DASH_ERR_LAUNCH;
    if (rc) return DASH_ERR_CUDA;

    const int n = (S + 127) / 128;   // the last tile may be partial
    const int nkv = (Skv + 127) / 128;
    // tasks: one per key/value head group, or one per query head (head split)
    const Shape grouped{B, Hq, Hkv, n, Hq / Hkv, causal, schedule, win, nkv == n ? 0 : nkv};
    int split = 0;
    if (!(dbg && dbg->ranks_host)) {   // a supplied table is laid out for group tasks
        const int mode = dbg ? dbg->head_split : 0;
        split = (mode == 1) ? (D == 128 && grouped.G > 1 && is_static(schedule))
                : (mode == 2) ? 0
                              : head_split_cached(grouped, P, D);
    }
    const int Ht = split ? Hq : Hkv;   // task heads
    const Shape sh{B, Hq, Ht, n, Hq / Ht, causal, schedule, win, nkv == n ? 0 : nkv};
    const long long tiles = (long long)B * Hq * n;
    const long long entries = tiles * nkv;
    const long long ntasks = num_tasks(sh);
    const bool use_table = dbg && dbg->ranks_host;
    if (use_table && !is_static(schedule)) return DASH_ERR_ARG;
    if (use_table && !dbg->skip_table_check &&
        dash_sim_check_ranks(schedule, causal, B, Hq, Hkv, n, P, dbg->ranks_host) != DASH_OK)
        return DASH_ERR_DEADLOCK;

    Workspace* ws = get_ws(dev, stream);
    const size_t part_elems = split ? (size_t)B * Hq * Skv * D : 0;   // per-query-head dK (then dV), fp32
    if (ws->delta.ensure((size_t)tiles * 128 * sizeof(float)) ||
        ws->ints.ensure((size_t)(kIntHeader + (kSubTiles + 1) * tiles) * sizeof(int)) ||
        (split && ws->part.ensure(2 * part_elems * sizeof(float))))
        return DASH_ERR_NOMEM;

    const uint16_t* ranks = nullptr;
    if (use_table) {
        if (ws->dbg_ranks.ensure((size_t)entries * sizeof(uint16_t))) return DASH_ERR_NOMEM;
        if (cudaMemcpyAsync(ws->dbg_ranks.p, dbg->ranks_host, (size_t)entries * sizeof(uint16_t),
                            cudaMemcpyHostToDevice, stream) != cudaSuccess)
            return DASH_ERR_CUDA;
        ranks = (const uint16_t*)ws->dbg_ranks.p;
    } else if (is_static(schedule)) {
        const long long key[8] = {B, Hq, Ht, n, causal, is_symmetric(sh) ? kSymmetric : kShift, P,
                                  (long long)win * 65536 + nkv};
        if (memcmp(key, ws->table_key, sizeof(key)) != 0) {
            if (ws->ranks.ensure((size_t)entries * sizeof(uint16_t)) ||
                ws->time.ensure((size_t)entries * sizeof(uint32_t)) ||
                ws->task_start.ensure((size_t)ntasks * sizeof(uint32_t)))
                return DASH_ERR_NOMEM;
            if (launch_build_ranks(B, Hq, Ht, n, causal, schedule, P, (uint16_t*)ws->ranks.p,
                                   (uint32_t*)ws->time.p, (uint32_t*)ws->task_start.p, stream, win, sh.nk))
                return DASH_ERR_CUDA;
            memcpy(ws->table_key, key, sizeof(key));
        }
        ranks = (const uint16_t*)ws->ranks.p;
    }

    int* ints = (int*)ws->ints.p;
    if (cudaMemsetAsync(ints, 0, (size_t)(kIntHeader + (kSubTiles + 1) * tiles) * sizeof(int), stream) != cudaSuccess ||
        cudaMemsetAsync(dq, 0, (size_t)B * Hq * S * D * sizeof(float), stream) != cudaSuccess)
        return DASH_ERR_CUDA;
    if (!delta_in && launch_preprocess(o, dO, (float*)ws->delta.p, (long long)B * Hq * S, D, stream))
        return DASH_ERR_CUDA;

    BwdParams prm;
    memset(&prm, 0, sizeof(prm));
    if (make_tmap_3d(&prm.tm_q, q, (long long)B * Hq, S, D) || make_tmap_3d(&prm.tm_k, k, (long long)B * Hkv, Skv, D) ||
        make_tmap_3d(&prm.tm_v, v, (long long)B * Hkv, Skv, D) || make_tmap_3d(&prm.tm_do, dO, (long long)B * Hq, S, D))
        return DASH_ERR_CUDA;
    prm.lse = lse;
    prm.delta = delta_in ? delta_in : (const float*)ws->delta.p;
    prm.dq = dq;
    prm.dk = (__nv_bfloat16*)dk;
    prm.dv = (__nv_bfloat16*)dv;
    prm.ranks = ranks;
    prm.status = ints;
    prm.task_counter = ints + 8;
    prm.abort_flag = ints + 9;
    prm.sem = ints + kIntHeader;
    prm.logcnt = ints + kIntHeader + kSubTiles * tiles;
    if (dbg) {
        prm.order_log = dbg->order_log;
        prm.partials = dbg->dq_partials;
        prm.cta_perm = dbg->cta_perm;
        prm.delay_ns = dbg->start_delay_ns;
        prm.prof = dbg->wait_cycles;
        prm.trace = dbg->event_trace;
        if (prm.trace && !prm.prof) return DASH_ERR_ARG;   // the trace needs the instrumented build
    }
    prm.timeout_ns = g_timeout_ns.load();
    prm.ntasks = ntasks;
    prm.B = B;
    prm.Hq = Hq;
    prm.Hkv = Ht;
    prm.kvh = Hkv;
    prm.kvg = Hq / Hkv;
    prm.S = S;
    prm.n = n;
    prm.G = Hq / Ht;
    prm.causal = causal;
    prm.sched = schedule;
    prm.P = P;
    prm.scale = 1.0f / sqrtf((float)D);
    prm.scale_log2e = prm.scale * kLog2e;
    prm.window = window;
    prm.win = win;
    prm.Skv = Skv;
    prm.nk = sh.nk;
    prm.nkv = nkv;
    if (dbg && dbg->kernel_event_begin &&
        cudaEventRecord((cudaEvent_t)dbg->kernel_event_begin, stream) != cudaSuccess)
        return DASH_ERR_CUDA;
    if (split) {
        prm.part_dk = (float*)ws->part.p;
        prm.part_dv = prm.part_dk + part_elems;
    }
    rc = launch_bwd_dispatch(D, prm, P, stream);
    if (rc == 0 && dbg && dbg->kernel_event_end &&
        cudaEventRecord((cudaEvent_t)dbg->kernel_event_end, stream) != cudaSuccess)
        return DASH_ERR_CUDA;
    if (rc == -3) return DASH_ERR_LAUNCH;
    if (rc) return DASH_ERR_CUDA;
    // one task per query head: dK, dV = the group's per-head partials, ascending head order
    if (split && (launch_group_sum(prm.part_dk, dk, B, Hkv, Hq / Hkv, Skv, D, stream) ||
                  launch_group_sum(prm.part_dv, dv, B, Hkv, Hq / Hkv, Skv, D, stream)))
        return DASH_ERR_CUDA;
    return DASH_OK;
}

// Key blocks of the backward with more key tiles than query tiles (full mask,
// as many key/value heads as query heads, whole key tiles): G, the largest
// divisor of the key tile count that leaves at least as many key tiles per
// block as query tiles, so that each dQ tile's ordered chain is at most about
// as long as in a square problem, and keeps the block shape's B*Hq*G*Sq
// within the index range; 1 = no split.
int key_blocks(int B, int Hq, int Hkv, int Sq, int Skv) {
    if (Hq != Hkv || Skv % 128 != 0) return 1;
    const int nq = (Sq + 127) / 128, nkv = Skv / 128;
    int best = 1;
    for (int g = 2; g <= nkv; ++g)
        if (nkv % g == 0 && nkv / g >= nq && (long long)B * Hq * g * Sq < (1ll << 31)) best = g;
    return best;
}

// The backward with different lengths, the keys cut into G blocks: block g of
// head h runs as head h*G + g of one backward with B*H*G heads and Skv/G keys
// (those are the contiguous rows g*Skv/G.. of the head's K, V, dK and dV, so
// dK and dV are written in place), each with a copy of the head's Q, dO, LSE
// and delta (delta from the full O and dO); then dq = the G blocks' fp32
// partial sums added in ascending block order.  Each dQ tile thus takes G
// ordered chains of Skv/G/128 contributions instead of one of Skv/128.
// Returns DASH_ERR_NOMEM (nothing launched) when the copies do not fit.
int bwd_cross_blocks(const dash_bf16* q, const dash_bf16* k, const dash_bf16* v, const dash_bf16* o,
                     const dash_bf16* dO, const float* lse, float* dq, dash_bf16* dk, dash_bf16* dv, int B, int H,
                     int Sq, int Skv, int D, int schedule, cudaStream_t stream, int G) {
    const void* ptrs[] = {q, k, v, o, dO, lse, dq, dk, dv};
    for (const void* ptr : ptrs)
        if (!aligned16(ptr)) return DASH_ERR_ARG;
    int rc = validate_shape(B, H, H, Sq, D, 0, schedule);
    if (rc) return rc;
    if ((long long)B * H * Skv >= (1ll << 31) || (long long)B * H * G * Sq >= (1ll << 31)) return DASH_ERR_ARG;   // key_blocks keeps G below
    int dev = 0;
    if ((rc = check_device(&dev))) return rc;
    const long long BH = (long long)B * H;
    auto up = [](long long x) { return (x + 255) & ~255ll; };
    const long long b_x = up(BH * G * Sq * D * 2), b_r = up(BH * G * Sq * 4), b_d = up(BH * Sq * 4);
    const long long b_q = up(BH * G * Sq * D * 4);
    Workspace* ws = get_ws(dev, stream);
    if (ws->kb.ensure((size_t)(2 * b_x + 2 * b_r + b_d + b_q))) return DASH_ERR_NOMEM;
    char* base = (char*)ws->kb.p;
    dash_bf16* qv = (dash_bf16*)base;
    dash_bf16* dov = (dash_bf16*)(base + b_x);
    float* lsev = (float*)(base + 2 * b_x);
    float* dlv = (float*)(base + 2 * b_x + b_r);
    float* delta = (float*)(base + 2 * b_x + 2 * b_r);
    float* dqv = (float*)(base + 2 * b_x + 2 * b_r + b_d);
    if (launch_preprocess(o, dO, delta, BH * Sq, D, stream) ||
        launch_replicate(q, qv, (long long)Sq * D * 2, BH, G, stream) ||
        launch_replicate(dO, dov, (long long)Sq * D * 2, BH, G, stream) ||
        launch_replicate(lse, lsev, (long long)Sq * 4, BH, G, stream) ||
        launch_replicate(delta, dlv, (long long)Sq * 4, BH, G, stream))
        return DASH_ERR_CUDA;
    rc = bwd_impl(qv, k, v, o, dov, lsev, dqv, dk, dv, B, H * G, H * G, Sq, D, 0, schedule, stream, nullptr, 0,
                  Skv / G, dlv);
    if (rc) return rc;
    return launch_block_sum(dqv, dq, BH, G, (long long)Sq * D, stream) ? DASH_ERR_CUDA : DASH_OK;
}

}  // namespace

namespace {
int encode_2d(void* map_out, CUtensorMapDataType dt, int esize, const void* base, long long rows, int D,
              unsigned box_cols) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return -2;
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)D * esize};
    const cuuint32_t box[2] = {box_cols, 128};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(reinterpret_cast<CUtensorMap*>(map_out), dt, 2, const_cast<void*>(base), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : -2;
}
}  // namespace

unsigned long long timeout_ns() { return g_timeout_ns.load(); }

// bf16 [heads][S][D], boxes of 64 columns x 128 rows x 1 head (128 B rows,
// swizzled).  Rows past S inside a head read as zero, so a ragged last tile
// never touches the next head.  Strides S*D*2 and D*2 are multiples of 16.
int make_tmap_3d(void* map_out, const void* base, long long heads, int S, int D) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return -2;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)heads};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)S * D * 2};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(reinterpret_cast<CUtensorMap*>(map_out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                    const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : -2;
}

// bf16 [rows, D], boxes of 64 columns x 128 rows (128 B rows, swizzled).
int make_tmap_2d(void* map_out, const void* base, long long rows, int D) {
    return encode_2d(map_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, rows, D, 64);
}

// fp32 [rows, D], boxes of 32 columns x 128 rows (128 B rows, swizzled).
int make_tmap_2d_f32(void* map_out, const void* base, long long rows, int D) {
    return encode_2d(map_out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, rows, D, 32);
}

}  // namespace dash

using namespace dash;

extern "C" {

int dash_attn_bwd_preprocess(const dash_bf16* o, const dash_bf16* dO, float* delta, int B, int Hq, int S, int D,
                             dash_stream_t stream) {
    if (!aligned16(o) || !aligned16(dO) || !aligned16(delta)) return DASH_ERR_ARG;
    if (B <= 0 || Hq <= 0 || S <= 0 || (D != 64 && D != 128)) return DASH_ERR_ARG;
    int dev = 0;
    int rc = check_device(&dev);
    if (rc) return rc;
    return launch_preprocess(o, dO, delta, (long long)B * Hq * S, D, (cudaStream_t)stream) ? DASH_ERR_CUDA : DASH_OK;
}

int dash_attn_bwd(const dash_bf16* q, const dash_bf16* k, const dash_bf16* v, const dash_bf16* o,
                  const dash_bf16* dO, const float* lse, float* dq, dash_bf16* dk, dash_bf16* dv, int B, int Hq,
                  int Hkv, int S, int D, int causal, int schedule, dash_stream_t stream) {
    return bwd_impl(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, S, D, causal, schedule, (cudaStream_t)stream,
                    nullptr);
}

int dash_attn_bwd_debug(const dash_bf16* q, const dash_bf16* k, const dash_bf16* v, const dash_bf16* o,
                        const dash_bf16* dO, const float* lse, float* dq, dash_bf16* dk, dash_bf16* dv, int B,
                        int Hq, int Hkv, int S, int D, int causal, int schedule, dash_stream_t stream,
                        const dash_debug_opts* opts) {
    return bwd_impl(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, S, D, causal, schedule, (cudaStream_t)stream,
                    opts, opts ? opts->window : 0, opts ? opts->skv : 0);
}

static int fwd_impl(const dash_bf16* q, const dash_bf16* k, const dash_bf16* v, dash_bf16* o, float* lse, int B,
                    int Hq, int Hkv, int S, int D, int causal, int window, dash_stream_t stream_, int Skv = 0) {
    cudaStream_t stream = (cudaStream_t)stream_;
    const void* ptrs[] = {q, k, v, o, lse};
    for (const void* ptr : ptrs)
        if (!aligned16(ptr)) return DASH_ERR_ARG;
    int rc = validate_shape(B, Hq, Hkv, S, D, causal, 0);
    if (rc) return rc;
    if (window < 0 || (window > 0 && !causal)) return DASH_ERR_ARG;
    if (window >= S) window = 0;
    if (Skv == 0) Skv = S;
    if (Skv < 0 || (Skv != S && causal) || (Skv + 127) / 128 > 65535) return DASH_ERR_ARG;
    int dev = 0;
    if ((rc = check_device(&dev))) return rc;
    Workspace* ws = get_ws(dev, stream);
    if (ws->ints.ensure((size_t)kIntHeader * sizeof(int))) return DASH_ERR_NOMEM;
    if (cudaMemsetAsync(ws->ints.p, 0, 8 * sizeof(int), stream) != cudaSuccess) return DASH_ERR_CUDA;
    rc = launch_fwd(q, k, v, o, lse, (int*)ws->ints.p, B, Hq, Hkv, S, D, causal, window, g_timeout_ns.load(),
                    stream, Skv);
    if (rc == -1) return DASH_ERR_ARG;
    return rc ? DASH_ERR_CUDA : DASH_OK;
}

int dash_attn_fwd(const dash_bf16* q, const dash_bf16* k, const dash_bf16* v, dash_bf16* o, float* lse, int B,
                  int Hq, int Hkv, int S, int D, int causal, dash_stream_t stream) {
    return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, S, D, causal, 0, stream);
}

int dash_attn_fwd_window(const dash_bf16* q, const dash_bf16* k, const dash_bf16* v, dash_bf16* o, float* lse,
                         int B, int Hq, int Hkv, int S, int D, int window, dash_stream_t stream) {
    if (window < 1) return DASH_ERR_ARG;
    return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, S, D, 1, window, stream);
}

int dash_attn_fwd_cross(const dash_bf16* q, const dash_bf16* k, const dash_bf16* v, dash_bf16* o, float* lse,
                        int B, int Hq, int Hkv, int Sq, int Skv, int D, dash_stream_t stream) {
    if (Skv < 1) return DASH_ERR_ARG;
    return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Sq, D, 0, 0, stream, Skv);
}

int dash_attn_bwd_cross(const dash_bf16* q, const dash_bf16* k, const dash_bf16* v, const dash_bf16* o,
                        const dash_bf16* dO, const float* lse, float* dq, dash_bf16* dk, dash_bf16* dv, int B,
                        int Hq, int Hkv, int Sq, int Skv, int D, int schedule, dash_stream_t stream) {
    if (Skv < 1) return DASH_ERR_ARG;
    const int G = (Skv != Sq && B > 0 && Hq > 0 && Sq > 0) ? key_blocks(B, Hq, Hkv, Sq, Skv) : 1;
    if (G > 1) {
        const int rc = bwd_cross_blocks(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Sq, Skv, D, schedule,
                                        (cudaStream_t)stream, G);
        if (rc != DASH_ERR_NOMEM) return rc;   // else one chain per dQ tile, as below
    }
    return bwd_impl(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, Sq, D, 0, schedule, (cudaStream_t)stream, nullptr, 0,
                    Skv);
}

int dash_attn_bwd_window(const dash_bf16* q, const dash_bf16* k, const dash_bf16* v, const dash_bf16* o,
                         const dash_bf16* dO, const float* lse, float* dq, dash_bf16* dk, dash_bf16* dv, int B,
                         int Hq, int Hkv, int S, int D, int window, int schedule, dash_stream_t stream) {
    if (window < 1) return DASH_ERR_ARG;
    return bwd_impl(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, S, D, 1, schedule, (cudaStream_t)stream, nullptr,
                    window);
}

int dash_key_blocks(int B, int Hq, int Hkv, int Sq, int Skv) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Skv <= 0) return DASH_ERR_ARG;
    return Skv != Sq ? key_blocks(B, Hq, Hkv, Sq, Skv) : 1;
}

int dash_select_schedule(int B, int Hq, int Hkv, int S, int D, int causal) {
    const int rc = validate_shape(B, Hq, Hkv, S, D, causal, kAuto);
    return rc ? rc : select_schedule(D, causal);
}

int dash_head_split(int schedule, int causal, int B, int Hq, int Hkv, int S, int D, int window, int Skv, int P) {
    int rc = validate_shape(B, Hq, Hkv, S, D, causal, schedule);
    if (rc) return rc;
    if (P <= 0 || window < 0 || (window > 0 && !causal)) return DASH_ERR_ARG;
    if (Skv == 0) Skv = S;
    if (Skv < 0 || (Skv != S && causal)) return DASH_ERR_ARG;
    if (window >= S) window = 0;
    if (schedule == kAuto) schedule = (Skv != S) ? kDescending : select_schedule(D, causal);
    const int n = (S + 127) / 128, nkv = (Skv + 127) / 128;
    const Shape grouped{B, Hq, Hkv, n, Hq / Hkv, causal, schedule, window ? band_tiles(window) : 0,
                        nkv == n ? 0 : nkv};
    return head_split_helps(grouped, P, D);
}

int dash_dq_finalize(const float* dq_accum, dash_bf16* dq, size_t numel, dash_stream_t stream) {
    if (!aligned16(dq_accum) || !aligned16(dq)) return DASH_ERR_ARG;
    if (numel == 0) return DASH_OK;
    int dev = 0;
    int rc = check_device(&dev);
    if (rc) return rc;
    return launch_finalize(dq_accum, dq, numel, (cudaStream_t)stream) ? DASH_ERR_CUDA : DASH_OK;
}

int dash_get_status(dash_stream_t stream, int* code, int* info) {
    if (!code) return DASH_ERR_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DASH_ERR_CUDA;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return DASH_ERR_CUDA;
    Workspace* ws = get_ws(dev, (cudaStream_t)stream);
    int h[8] = {0};
    if (ws->ints.p && cudaMemcpy(h, ws->ints.p, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
        return DASH_ERR_CUDA;
    *code = h[0];
    if (info)
        for (int i = 0; i < 4; ++i) info[i] = h[1 + i];
    return DASH_OK;
}

int dash_set_timeout_ns(uint64_t ns) {
    g_timeout_ns.store(ns ? ns : 1);
    return DASH_OK;
}

int dash_release_workspaces(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    for (auto& kv : workspaces()) {
        cudaSetDevice(kv.first.first);
        kv.second->release();
        delete kv.second;
    }
    workspaces().clear();
    cudaSetDevice(cur);
    return DASH_OK;
}

int dash_num_ctas(int device, int* P) {
    if (!P) return DASH_ERR_ARG;
    int cur = 0;
    if (cudaGetDevice(&cur) != cudaSuccess) return DASH_ERR_CUDA;
    if (cudaSetDevice(device) != cudaSuccess) return DASH_ERR_ARG;
    int rc = bwd_max_ctas(128, device, P);
    cudaSetDevice(cur);
    if (rc == -3) return DASH_ERR_LAUNCH;
    return rc ? DASH_ERR_CUDA : DASH_OK;
}

int dash_debug_tile_probe(const dash_bf16* k, const dash_bf16* v, const dash_bf16* q, const dash_bf16* dO,
                          const float* lse, const float* delta, int D, int diag, float* sT, float* pT, float* dpT,
                          float* dsT, float* dv, float* dk, float* dq) {
    const void* ptrs[] = {k, v, q, dO, lse, delta, sT, pT, dpT, dsT, dv, dk, dq};
    for (const void* ptr : ptrs)
        if (!aligned16(ptr)) return DASH_ERR_ARG;
    if (D != 64 && D != 128) return DASH_ERR_ARG;
    int dev = 0;
    int rc = check_device(&dev);
    if (rc) return rc;
    rc = run_tile_probe(k, v, q, dO, lse, delta, D, diag, sT, pT, dpT, dsT, dv, dk, dq);
    if (rc == -4) return DASH_ERR_TIMEOUT;
    if (rc == -6) return DASH_ERR_NOMEM;
    return rc ? DASH_ERR_CUDA : DASH_OK;
}

}  // extern "C"
