// dash_schedule.h -- the tile schedules of DASH as closed-form functions.
//
// Shared by the persistent kernel (the producer warp walks a task's visit
// list), the device table builder and the host simulator.  Definitions
// follow "DASH: Deterministic Attention Scheduling for High-Throughput"
// (gist.science technical summary), section 2.2:
//   - descending Q-tile iteration (2.2.A): Q tiles visited n-1 .. 0;
//   - shift scheduling (2.2.B, full masks): the worker that owns KV tile j
//     visits Q tiles j, j+1, ..., n-1, 0, ..., j-1 (the summary words it as
//     "SM i processes i, i+1, ..., N-1, 0, ..., i-1"; with the KV tile kept
//     resident it is the Q tiles that rotate);
//   - symmetric shift (2.2.B, causal masks): KV tiles jp and n-1-jp form one
//     task; phase 1 is the dense rectangle (KV jp against the last h = n/2 Q
//     tiles, rotated by jp), phase 2 the folded triangle (KV jp against Q
//     jp .. n-h-1 ascending, then KV n-1-jp against Q n-1 .. n-1-jp).
// and the FlashAttention-3-style baseline (ascending visits, ascending-KV
// accumulation order) that the summary's section 1 describes.
//
// A task is one KV tile (b, hkv, j) -- or one symmetric pair -- and runs the
// pairs of every query head of its group (ascending) back to back on one
// CTA, so dK/dV stay in tensor memory for the whole task.  (The library may
// describe a grouped-query problem with Hkv = Hq, G = 1, i.e. one task per
// query head, to fill the last wave; its host side then sums the group.)
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define DASH_HD __host__ __device__ __forceinline__
#else
#define DASH_HD inline
#endif

namespace dash {

enum Sched : int {
    kAtomic = 0,
    kAscending = 1,
    kDescending = 2,
    kShift = 3,
    kSymmetric = 4,
    kAuto = 5,   // resolved on the host by select_schedule before anything runs
};

// The deterministic schedule run for kAuto: a function of the shape only, so
// that kAuto is as reproducible as the schedule it names.  Measured on GB300
// (kernel-only): full masks run shift (symmetric shift is the same schedule);
// causal masks run symmetric shift at D = 128 (ahead of shift by 9%, of
// descending by 2x) and shift at D = 64 (ahead of symmetric shift by 30%).
inline int select_schedule(int D, int causal) {
    if (!causal) return kShift;
    return D == 128 ? kSymmetric : kShift;
}

struct Shape {
    int B, Hq, Hkv, n, G, causal, sched;   // n: query tiles per head
    int win;   // causal sliding window: tile diagonals 0 <= q - kv < win visited; 0 = none
    int nk;    // key/value tiles per head when they differ from n (full masks only); 0 = n
};

// Key/value tiles per head.
DASH_HD int num_kv(const Shape& s) { return s.nk ? s.nk : s.n; }

// Tile diagonals touched by a causal sliding window of `window` tokens: tile
// pair (q, kv) holds a visible element iff 0 <= q - kv < band_tiles(window)
// (the smallest query-key distance on diagonal t >= 1 is 128 t - 127).
inline int band_tiles(int window) { return (window + 126) / 128 + 1; }

// Symmetric shift only exists on causal masks without a window; otherwise it
// is shift (a band leaves no triangle to fold).
DASH_HD bool is_symmetric(const Shape& s) { return s.sched == kSymmetric && s.causal && !s.win; }
DASH_HD bool is_static(int sched) { return sched == kShift || sched == kSymmetric; }
DASH_HD bool is_ordered(int sched) { return sched != kAtomic; }

// Tasks per (b, hkv) and in total.
DASH_HD int tasks_per_group(const Shape& s) { return is_symmetric(s) ? (s.n + 1) / 2 : num_kv(s); }
DASH_HD int64_t num_tasks(const Shape& s) {
    return (int64_t)s.B * s.Hkv * tasks_per_group(s);
}

// Visits of one KV tile j for ONE query head (non-symmetric schedules).
DASH_HD int kv_len(const Shape& s, int j) {
    if (!s.causal) return s.n;
    return (s.win && s.win < s.n - j) ? s.win : s.n - j;
}

// First KV tile that adds into dQ tile q (the rank base of the schedules
// whose accumulation order is ascending KV).
DASH_HD int first_kv(const Shape& s, int q) { return (s.causal && s.win && q >= s.win) ? q - s.win + 1 : 0; }

// Task numbering (the dealing rule is task k -> worker k mod P throughout).
//  - Causal shift without a window is KV-tile-major (tile k / (B*Hkv) of group
//    k % (B*Hkv)): a causal KV tile j has n - j pairs, and dealing the tasks
//    round-robin in that order gives every wave tiles of nearly equal length
//    (busiest of 152 workers at 1.035x the mean instead of 1.09x for B1 H32
//    S16384) and spaces the contributions to a dQ tile about a wave apart.
//  - Shift on a full mask or a sliding-window band, and symmetric shift
//    (full or causal; on a band it is shift), with equal query and key
//    lengths, are parity-major: the even tiles (pairs) of every head group,
//    head group by head group, then the odd ones.  All of a head's tiles in
//    one wave would add into each of its dQ tiles at every step of the
//    rotation; a wave of one parity adds at every second step, which leaves
//    each ordered link two steps to complete.
//  - Everything else is head-group-major (tile k % T of group k / T).
// (A band with win >= n visits every tile of the causal triangle and is dealt
// as the causal mask is.)
DASH_HD bool banded(const Shape& s) { return s.win && s.win < s.n; }
DASH_HD bool kv_major(const Shape& s) { return s.sched == kShift && s.causal && !banded(s); }
DASH_HD bool parity_major(const Shape& s) {
    return !s.nk && (s.sched == kShift || s.sched == kSymmetric) &&
           (!s.causal || banded(s) || s.sched == kSymmetric);
}

// A task's tile (or symmetric pair) and head group (b * Hkv + hkv); callers
// that walk a task's pairs compute it once per task.  Task counts are below
// 2^31 because B*Hq*S is.
struct TaskRef {
    int t, bh;
};
DASH_HD TaskRef task_ref(const Shape& s, int64_t k) {
    const int kk = (int)k;
    TaskRef r;
    if (kv_major(s)) {
        const int g = s.B * s.Hkv;
        r.t = kk / g;
        r.bh = kk - r.t * g;
    } else if (parity_major(s)) {
        const int g = s.B * s.Hkv, T = tasks_per_group(s);
        const int even = (T + 1) / 2;   // even tiles per group, then T / 2 odd ones
        if (kk < g * even) {
            r.bh = kk / even;
            r.t = 2 * (kk - r.bh * even);
        } else {
            const int x = kk - g * even, odd = T / 2;
            r.bh = x / odd;
            r.t = 2 * (x - r.bh * odd) + 1;
        }
    } else {
        const int T = tasks_per_group(s);
        r.bh = kk / T;
        r.t = kk - r.bh * T;
    }
    return r;
}

// Pairs in a task (all heads of the group).
DASH_HD int task_len_at(const Shape& s, TaskRef r) {
    const int t = r.t;
    if (!is_symmetric(s)) return s.G * kv_len(s, t);
    const int h = s.n / 2;
    if ((s.n & 1) && t == h) return s.G * (s.n - h);   // middle tile of an odd n
    return s.G * (s.n + 1);
}
DASH_HD int task_len(const Shape& s, int64_t k) { return task_len_at(s, task_ref(s, k)); }

struct Visit {
    int b, hkv, hq, kv, q;   // dQ tile (b, hq, q) receives the partial of KV tile (b, hkv, kv)
};

// The u-th pair of a task, 0 <= u < task_len_at(s, r).
DASH_HD Visit visit_at(const Shape& s, TaskRef r, int u) {
    Visit v;
    const int t = r.t;
    v.hkv = r.bh % s.Hkv;
    v.b = r.bh / s.Hkv;
    const int n = s.n;
    if (!is_symmetric(s)) {
        const int j = t;
        const int L = kv_len(s, j);
        const int g = u / L, w = u % L;
        v.hq = v.hkv * s.G + g;
        v.kv = j;
        switch (s.sched) {
            case kDescending: v.q = (s.causal ? j : 0) + L - 1 - w; break;
            case kShift:
            case kSymmetric:  v.q = s.causal ? j + w : (j + w) % n; break;   // symmetric on a full mask = shift
            default:          v.q = (s.causal ? j : 0) + w; break;   // ascending, atomic
        }
        return v;
    }
    const int h = n / 2;
    const int jp = t;
    if ((n & 1) && jp == h) {                   // middle tile: descending visits
        const int L = n - h;
        v.hq = v.hkv * s.G + u / L;
        v.kv = h;
        v.q = n - 1 - (u % L);
        return v;
    }
    const int La = n - jp;                      // phase 1 (h) + phase 2a (n-h-jp)
    if (u < s.G * La) {
        const int g = u / La, w = u % La;
        v.hq = v.hkv * s.G + g;
        v.kv = jp;
        v.q = (w < h) ? (n - h) + (jp + w) % h : jp + (w - h);
        return v;
    }
    const int ub = u - s.G * La;                // phase 2b: KV n-1-jp, descending Q
    const int Lb = jp + 1;
    v.hq = v.hkv * s.G + ub / Lb;
    v.kv = n - 1 - jp;
    v.q = n - 1 - (ub % Lb);
    return v;
}
DASH_HD Visit task_visit(const Shape& s, int64_t k, int u) { return visit_at(s, task_ref(s, k), u); }

// Index of the accumulation-rank entry of pair (b, hq, q, kv).
DASH_HD int64_t rank_index(const Shape& s, int b, int hq, int q, int kv) {
    return (((int64_t)b * s.Hq + hq) * s.n + q) * num_kv(s) + kv;
}

}  // namespace dash
