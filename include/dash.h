/*
 * dash.h -- C ABI of libdash.so: deterministic attention backward (dQ, dK, dV)
 * under the DASH tile schedules, for one GB300 (sm_103a) GPU.
 *
 * Source of the method: "DASH: Deterministic Attention Scheduling for
 * High-Throughput" (gist.science technical summary of arXiv 2601.21824),
 * sections 1 (fixed dQ accumulation order), 2.1 (DAG model) and 2.2
 * (descending Q-tile iteration, shift and symmetric shift scheduling); and
 * the pwwt.cn write-up "DASH: how it changes deterministic LLM training",
 * sections 2.2-2.3 (chain model, shift rotation, closed forms) and 3.1 (the
 * release-side counter of an ordered reduction).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Tensor pointers are DEVICE pointers owned by the caller, contiguous
 *    row-major [B, H, S, D] (LSE and delta: [B, H, S]), 16-byte aligned.
 *  - dash_bf16 is the raw 16-bit storage of a bfloat16 value.
 *  - S is any positive length; the kernels work on 128 x 128 tiles, n =
 *    ceil(S / 128) per head, and mask the rows and columns of a partial last
 *    tile (the schedules and accumulation orders are those of n tiles).  D
 *    is 64 or 128; Hq must be a multiple of Hkv (query heads hq = g*G ..
 *    g*G+G-1 share key/value head g, G = Hq / Hkv).
 *  - LSE is the natural-log log-sum-exp of scale * Q K^T per query row with
 *    scale = 1/sqrt(D) (the forward's statistic); masks are "full" or
 *    top-left causal (key j visible to query i iff j <= i).
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and returns a dash_status; errors never throw.
 *  - Library-owned scratch (delta, per-tile semaphores, schedule tables, the
 *    status word) lives in a workspace cached per (device, stream) and grown
 *    on demand; dash_release_workspaces() frees it.  Calls on the same stream
 *    are ordered; concurrent calls that share a stream from several host
 *    threads are not supported.  Different devices/streams are independent.
 */
#ifndef DASH_H
#define DASH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t dash_bf16;
typedef struct CUstream_st* dash_stream_t;

typedef enum {
    DASH_OK = 0,
    DASH_ERR_ARG = -1,        /* invalid argument (null, misaligned, bad shape, unknown schedule) */
    DASH_ERR_CUDA = -2,       /* a CUDA runtime/driver call failed */
    DASH_ERR_LAUNCH = -3,     /* the persistent grid cannot be co-resident on this device */
    DASH_ERR_TIMEOUT = -4,    /* device-side wait exceeded the timeout (reported by dash_get_status) */
    DASH_ERR_DEADLOCK = -5,   /* a schedule table cannot complete (cycle or missing predecessor) */
    DASH_ERR_NOMEM = -6,      /* workspace allocation failed */
    DASH_ERR_DEVICE = -7,     /* device is not sm_103 / lacks the needed shared memory */
    DASH_ERR_SCRATCH = -8     /* problem needs more than dash_attn_bwd_noalloc's fixed scratch */
} dash_status;

typedef enum {
    DASH_SCHED_ATOMIC_NONDET = 0,        /* unordered fp32 atomics: fast, NOT reproducible */
    DASH_SCHED_SERIALIZED_ASCENDING = 1, /* ascending Q visits, ascending-KV accumulation order */
    DASH_SCHED_DESCENDING_Q = 2,         /* descending Q visits, ascending-KV accumulation order */
    DASH_SCHED_SHIFT = 3,                /* cyclic Q rotation per KV tile, model-time order */
    DASH_SCHED_SYMMETRIC_SHIFT = 4,      /* causal: KV pairs (j, n-1-j), two phases; full mask = SHIFT */
    DASH_SCHED_AUTO = 5                  /* the deterministic schedule dash_select_schedule picks */
} dash_schedule;

/*
 * dash_attn_fwd -- the attention forward pass whose backward dash_attn_bwd
 * computes (the textbook softmax attention that the gist.science DASH
 * summary, section 1, takes as given; the pages schedule only the backward):
 *   o[b,h,i,:]  = sum_j P[i,j] v[b,hk,j,:],  P = softmax_j(scale <q_i, k_j>),
 *   lse[b,h,i]  = log sum_j exp(scale <q_i, k_j>)   (natural log),
 * with scale = 1/sqrt(D), hk = h / (Hq/Hkv), and the sum over j <= i when
 * causal (top-left aligned).  Outputs are exactly the o and lse arguments
 * that dash_attn_bwd expects.
 *   q: device bf16 [B,Hq,S,D]; k, v: device bf16 [B,Hkv,S,D] (caller-owned,
 *   contiguous, 16-byte aligned).  o: device bf16 [B,Hq,S,D] (written,
 *   rounded to nearest even); lse: device fp32 [B,Hq,S] (written).
 * One CTA per 128-row query tile; no cross-CTA reduction, so the outputs are
 * bitwise reproducible.  Same shape rules as dash_attn_bwd (any S > 0,
 * D in {64, 128}, Hq % Hkv == 0).  Asynchronous on `stream`; returns
 * DASH_OK, DASH_ERR_ARG, DASH_ERR_DEVICE, DASH_ERR_NOMEM or DASH_ERR_CUDA;
 * a device-side timeout is reported by dash_get_status on the same stream.
 */
int dash_attn_fwd(const dash_bf16* q, const dash_bf16* k, const dash_bf16* v, dash_bf16* o, float* lse,
                  int B, int Hq, int Hkv, int S, int D, int causal, dash_stream_t stream);

/*
 * dash_attn_bwd_window, dash_attn_fwd_window -- dash_attn_bwd and
 * dash_attn_fwd for a causal sliding window of `window` tokens (>= 1): key
 * j is visible to query i iff i - window < j <= i.  This is the band mask of
 * the Ascend FlashAttentionGrad plan (ocdem.com, section 2.3.5, with tiles
 * that are entirely masked skipped, section 3.1): a KV tile is visited only
 * by the Q tiles of its band (band = ceil((window + 127) / 128) tile
 * diagonals), the two edge diagonals are masked element by element, and
 * the schedules, accumulation orders and rank tables are those of the band
 * (symmetric shift runs as shift).  window >= S is the causal mask.  Same
 * arguments (with `window` in place of `causal`), layouts, determinism and
 * errors as the calls without a window; DASH_ERR_ARG also for window < 1.
 */
int dash_attn_bwd_window(const dash_bf16* q, const dash_bf16* k, const dash_bf16* v,
                         const dash_bf16* o, const dash_bf16* dO, const float* lse,
                         float* dq, dash_bf16* dk, dash_bf16* dv,
                         int B, int Hq, int Hkv, int S, int D, int window, int schedule,
                         dash_stream_t stream);
int dash_attn_fwd_window(const dash_bf16* q, const dash_bf16* k, const dash_bf16* v, dash_bf16* o, float* lse,
                         int B, int Hq, int Hkv, int S, int D, int window, dash_stream_t stream);

/*
 * dash_attn_bwd_cross, dash_attn_fwd_cross -- dash_attn_bwd and dash_attn_fwd
 * with a key/value length Skv different from the query length Sq (full mask):
 * q, o, dO, dq: [B,Hq,Sq,D]; lse: [B,Hq,Sq]; k, v, dk, dv: [B,Hkv,Skv,D].  The
 * Ascend plan's tiling (ocdem.com, section 2.3.1): ceil(Sq/128) query tiles
 * by ceil(Skv/128) key tiles; each KV tile is one task that visits every
 * query tile (shift rotates from query tile kv mod nq; symmetric shift is
 * shift).  Same arguments otherwise (no causal flag), same determinism and
 * errors.
 *   Key blocks (backward only; the pages give no schedule for more key tiles
 * than query tiles, where every dQ tile would take one ordered chain of
 * Skv/128 contributions): when dash_key_blocks returns G > 1 the keys are cut
 * into G blocks of Skv/G keys.  Block g of head h runs as head h*G + g of one
 * backward with B*Hq*G heads and Skv/G keys (its K, V, dK and dV rows are the
 * head's rows g*Skv/G .. (g+1)*Skv/G - 1, used in place; Q, dO, LSE and delta
 * are copied per block into a library workspace), with the schedule's tasks
 * and accumulation order of that shape (DASH_SCHED_AUTO then picks for it);
 * dq = the G blocks' fp32 dQ sums added in ascending block order.  If the
 * workspace cannot be allocated the call runs unsplit.  The debug entry
 * (dash_attn_bwd_debug) never splits.
 */
int dash_attn_bwd_cross(const dash_bf16* q, const dash_bf16* k, const dash_bf16* v,
                        const dash_bf16* o, const dash_bf16* dO, const float* lse,
                        float* dq, dash_bf16* dk, dash_bf16* dv,
                        int B, int Hq, int Hkv, int Sq, int Skv, int D, int schedule,
                        dash_stream_t stream);
int dash_attn_fwd_cross(const dash_bf16* q, const dash_bf16* k, const dash_bf16* v, dash_bf16* o, float* lse,
                        int B, int Hq, int Hkv, int Sq, int Skv, int D, dash_stream_t stream);

/*
 * dash_select_schedule -- the deterministic schedule that DASH_SCHED_AUTO
 * runs for this shape.  The DASH pages make the choice of strategy a matter
 * of the hardware: on H800 symmetric shift falls behind descending Q-tile
 * iteration for causal masks at D = 128 because of register spills
 * (gist.science summary, section 4), and the pwwt.cn write-up (section 3.1)
 * switches to descending automatically when head_dim > 64.  On GB300 dK/dV
 * live in tensor memory and that pressure does not arise; the choice
 * measured there (152 SMs, kernel-only TFLOP/s) is:
 *   full mask            -> DASH_SCHED_SHIFT (symmetric shift is the same
 *                           schedule; ascending is 26% slower)
 *   causal, D = 128      -> DASH_SCHED_SYMMETRIC_SHIFT (9% ahead of shift,
 *                           also with grouped-query heads; descending 2x slower)
 *   causal, D = 64       -> DASH_SCHED_SHIFT (30% ahead of symmetric shift)
 * With a sliding window symmetric shift is shift; with different query and
 * key lengths (dash_attn_bwd_cross) AUTO runs DASH_SCHED_DESCENDING_Q
 * (measured best there).
 * A pure function of the shape, never of timing, so that AUTO stays bitwise
 * reproducible from run to run and process to process.  Returns the
 * schedule (1..4), or DASH_ERR_ARG for a shape dash_attn_bwd rejects.
 */
int dash_select_schedule(int B, int Hq, int Hkv, int S, int D, int causal);

/*
 * dash_head_split -- does the backward of this shape, with grouped-query
 * heads (Hq > Hkv) on a static schedule (shift, symmetric shift, or AUTO
 * resolving to one), run one task per query head instead of one task per
 * key/value head group?  The pages' task is one KV tile (or symmetric pair)
 * with every query head of its group; with few, long group tasks the last
 * wave of the P persistent CTAs runs part-empty, so the library splits the
 * tasks per query head when that takes more than 2% off the busiest CTA's pair
 * count (a pure function of the shape and P).  A split run has the tasks and
 * accumulation order of the same shape with Hkv = Hq (simulate it with
 * dash_sim_schedule(..., Hkv = Hq, ...)); each task writes its query head's
 * dK and dV in fp32 to a library workspace, and a second kernel sums every
 * group's heads in ascending head order before rounding to bf16.
 *   window: causal sliding window in tokens (0 = none); Skv: key/value length
 *   (0 = S); P: the number of persistent CTAs (dash_num_ctas).
 * Only D = 128 splits (the per-head partial path is compiled into the D = 128
 * kernel alone).  Returns 1 (split) or 0, or DASH_ERR_ARG for a shape
 * dash_attn_bwd rejects.  Host only; needs no GPU.
 */
int dash_head_split(int schedule, int causal, int B, int Hq, int Hkv, int S, int D, int window, int Skv, int P);

/*
 * dash_key_blocks -- the number of key blocks G that dash_attn_bwd_cross
 * cuts the keys into (no counterpart on the pages): with Hq == Hkv and Skv a
 * multiple of 128, the largest divisor of Skv/128 that leaves at least
 * ceil(Sq/128) key tiles per block (so that each dQ tile's ordered chains are
 * no longer than its query tile count) and keeps B*Hq*G*Sq < 2^31; else 1 (no
 * split).  Returns G >= 1, or DASH_ERR_ARG for non-positive sizes.  Host
 * only; needs no GPU.
 */
int dash_key_blocks(int B, int Hq, int Hkv, int Sq, int Skv);

/*
 * dash_attn_bwd_preprocess -- delta[b,h,s] = sum_d dO[b,h,s,d] * O[b,h,s,d].
 *
 * The per-row statistic of the softmax backward (dS = P o (dP - delta)),
 * consumed by every tile pair of the backward pass whose dQ accumulation the
 * gist.science DASH summary (section 1) orders.  The pages do not print it:
 * it is the textbook softmax-gradient identity (rowsum of P o dP equals
 * rowsum of dO o O), computed once per row before the tile loop.
 * o, dO: bf16 [B,Hq,S,D]; delta: fp32 [B,Hq,S] written by the
 * call (caller-owned device buffers, 16-byte aligned).  Each row is summed
 * in fp32 in one fixed order, so the result is bitwise reproducible.
 * Returns DASH_ERR_ARG on null/misaligned pointers or bad sizes (any S > 0,
 * D in {64, 128}), DASH_ERR_DEVICE off sm_103, DASH_ERR_CUDA on launch
 * failure.
 */
int dash_attn_bwd_preprocess(const dash_bf16* o, const dash_bf16* dO, float* delta,
                             int B, int Hq, int S, int D, dash_stream_t stream);

/*
 * dash_attn_bwd -- the deterministic attention backward pass.
 *
 * What the DASH pages define: the backward pass of softmax attention whose
 * dQ tiles are each a sum over KV tiles that must be added in one fixed
 * order to be reproducible (gist.science DASH summary, section 1), with each
 * KV tile resident on one SM while it visits the Q tiles (section 2.1), and
 * the visit / accumulation orders of the schedules in section 2.2 (descending
 * Q-tile iteration; shift scheduling for full masks; two-phase symmetric
 * shift for causal masks).  The gradient accumulation is fp32 with bf16
 * storage (pwwt.cn write-up, section 3.2, mixed-precision configuration),
 * gated per dQ tile by a counter that each contributor waits on and then
 * advances (the write-up's release-side counter, section 3.1).
 *
 * Inputs: q, o, dO bf16 [B,Hq,S,D]; k, v bf16 [B,Hkv,S,D]; lse fp32 [B,Hq,S].
 * Outputs:
 *   dq  fp32 [B,Hq,S,D] -- the fp32 dQ accumulator.  The library zeroes it
 *       and leaves the final, scaled dQ in it (dash_dq_finalize rounds it to
 *       bf16).  Each dQ tile (128 rows of one head) is the fp32 sum of its
 *       KV-tile partials added in the order the schedule fixes.
 *   dk, dv bf16 [B,Hkv,S,D] -- accumulated on chip per KV tile over the
 *       tile's pairs in the schedule's visit order and over the query heads
 *       of its group in ascending head order; rounded to nearest even.  When
 *       dash_head_split returns 1 for the shape, each query head is its own
 *       task and the group's fp32 per-head results are added in ascending
 *       head order by a second kernel instead (workspace: 2 x B*Hq*S*D*4
 *       bytes).
 * All buffers are caller-owned device memory, contiguous, 16-byte aligned.
 * schedule: a dash_schedule value (DASH_SCHED_AUTO runs the schedule
 * dash_select_schedule returns).  causal: 0 (full) or 1 (top-left causal).
 *
 * For every schedule except DASH_SCHED_ATOMIC_NONDET the three outputs are
 * bitwise identical across runs on the same device model and SM count,
 * whatever the launch timing.  The call computes delta itself (o is an
 * argument), zeroes dq, builds or reuses the schedule tables, and launches
 * one persistent CTA per SM (cooperative launch).
 *
 * Errors: DASH_ERR_ARG (null or non-16-byte-aligned pointer, S <= 0,
 * more than 65535 tiles per head, D not in {64,128}, Hq % Hkv != 0, non-positive sizes, unknown schedule or
 * causal flag), DASH_ERR_DEVICE, DASH_ERR_LAUNCH, DASH_ERR_NOMEM,
 * DASH_ERR_CUDA.  A device-side wait that exceeds the timeout does not hang:
 * the kernel stops, leaves dq/dk/dv undefined and records DASH_ERR_TIMEOUT,
 * which dash_get_status reports.
 */
int dash_attn_bwd(const dash_bf16* q, const dash_bf16* k, const dash_bf16* v,
                  const dash_bf16* o, const dash_bf16* dO, const float* lse,
                  float* dq, dash_bf16* dk, dash_bf16* dv,
                  int B, int Hq, int Hkv, int S, int D, int causal, int schedule,
                  dash_stream_t stream);

/*
 * dash_attn_bwd_noalloc -- dash_attn_bwd for callers that cannot allocate.
 *
 * No counterpart on the DASH pages: this is a deployment variant.  Same
 * arguments, outputs and determinism as dash_attn_bwd, but it never calls
 * cudaMalloc/cudaFree or any allocating routine.  It is meant for callers
 * that have given all device memory to their own pool allocator, or that
 * run on a latency-critical path where the implicit synchronization of
 * cudaMalloc/cudaFree is not acceptable.  The caller still provides every
 * input and output buffer.  With grouped-query heads it always runs one task
 * per key/value head group (no room for per-query-head partials), so where
 * dash_head_split returns 1 its dK and dV bits are those of
 * dash_attn_bwd_debug with head_split = 2, not of dash_attn_bwd (both are
 * reproducible).
 *
 * Scratch (delta, the accumulation counters, the status word, the rank
 * tables) comes from one 8 MiB file-scope device array that every GPU loading
 * the library keeps until the process exits.  A problem needing more returns
 * DASH_ERR_SCRATCH (roughly: B*Hq*S*4 bytes of delta plus, for the shift
 * schedules, B*Hq*(S/128)^2*6 bytes of tables must fit).
 *
 * Set-up: the first call on a device (or dash_noalloc_init) looks up that
 * device's address of the array, with the device current, and loads the
 * kernels.  Under lazy module loading (the CUDA default) that is when the
 * driver loads the library's module and reserves the array, so do it before
 * a pool allocator takes the whole device, before a latency-critical path and
 * before any stream capture, or run with CUDA_MODULE_LOADING=EAGER.  After a
 * cudaDeviceReset, call dash_noalloc_init again before the next call.
 *
 * All calls share the array and it keeps the previous call's contents: each
 * call clears what must start at zero on its stream, so calls must not
 * overlap on the GPU (different streams or host threads racing on the array
 * give undefined results).  Device-side waits use the dash_set_timeout_ns
 * limit; one that runs out leaves the outputs undefined and is reported by
 * dash_get_status_noalloc (not by dash_get_status).
 *
 * Errors: DASH_ERR_ARG (as dash_attn_bwd), DASH_ERR_DEVICE (not sm_103),
 * DASH_ERR_LAUNCH, DASH_ERR_SCRATCH, DASH_ERR_CUDA.
 */
int dash_attn_bwd_noalloc(const dash_bf16* q, const dash_bf16* k, const dash_bf16* v,
                          const dash_bf16* o, const dash_bf16* dO, const float* lse,
                          float* dq, dash_bf16* dk, dash_bf16* dv,
                          int B, int Hq, int Hkv, int S, int D, int causal, int schedule,
                          dash_stream_t stream);

/*
 * dash_noalloc_init -- set-up of dash_attn_bwd_noalloc on the current device
 * (no counterpart on the pages): looks up the device address of its scratch
 * array and loads every kernel it launches, so that later calls do neither.
 * Allocates nothing itself; the driver reserves the array when it loads the
 * module.  Calling it again refreshes the address (needed after a
 * cudaDeviceReset).  Returns DASH_OK, DASH_ERR_DEVICE or DASH_ERR_CUDA.
 */
int dash_noalloc_init(void);

/*
 * dash_get_status_noalloc -- dash_get_status for dash_attn_bwd_noalloc (no
 * counterpart on the pages): synchronizes `stream` and reports the status
 * word of the last call on the current device, *code = DASH_OK or
 * DASH_ERR_TIMEOUT, info[0..3] as dash_get_status (info may be NULL).  Reads
 * the shared scratch array, so it describes whichever call last wrote it.
 * Returns DASH_OK, DASH_ERR_ARG (code NULL), DASH_ERR_DEVICE or DASH_ERR_CUDA.
 */
int dash_get_status_noalloc(dash_stream_t stream, int* code, int* info);

/*
 * dash_dq_finalize -- dq[i] = bf16_round_to_nearest_even(dq_accum[i]) for
 * i < numel: the last step of the backward, after the fp32 accumulation of
 * every dQ tile (pwwt.cn write-up, section 3.2: the backward's accumulations
 * run in fp32 and tensors are stored as bf16).  dq_accum fp32 (read), dq bf16 (written); both
 * caller-owned device pointers, 16-byte aligned, numel elements each.
 * Returns DASH_OK (also for numel = 0), DASH_ERR_ARG (null or misaligned),
 * DASH_ERR_DEVICE off sm_103, DASH_ERR_CUDA on launch failure.
 */
int dash_dq_finalize(const float* dq_accum, dash_bf16* dq, size_t numel, dash_stream_t stream);

/* ---------------------------------------------------------------------------
 * Status and configuration
 * ------------------------------------------------------------------------- */

/*
 * dash_get_status -- synchronizes `stream` and reports the device status of
 * the last dash_attn_bwd on (current device, stream): *code = DASH_OK or
 * DASH_ERR_TIMEOUT; info[0..3] = {b*Hq+hq, Q tile, expected turn, role} of
 * the first wait that timed out (role 0 reducer, 1 producer, 2 MMA,
 * 3 softmax/dS).  info may be NULL.  Returns DASH_OK or DASH_ERR_CUDA.
 */
int dash_get_status(dash_stream_t stream, int* code, int* info);

/* Timeout of every device-side wait, in ns (default 2e9).  Returns DASH_OK. */
int dash_set_timeout_ns(uint64_t ns);

/* Frees every cached workspace of the calling process (all devices).  The
 * caller must ensure no dash call is in flight.  Returns DASH_OK. */
int dash_release_workspaces(void);

/* *P = number of persistent CTAs (one per SM) dash_attn_bwd uses on `device`;
 * the static schedules' accumulation order depends on it. */
int dash_num_ctas(int device, int* P);

/* ---------------------------------------------------------------------------
 * Schedule simulator (host only, no GPU needed)
 *
 * The DAG model of the DASH summary, section 2.1: each pair (KV tile j,
 * Q tile i) is a compute of cost c followed by a reduce of cost r; the pairs
 * of one task run back to back on one SM; the reduces into one dQ tile follow
 * the accumulation order.  Static schedules (shift, symmetric shift) give
 * task k to SM k % P; the others dispatch greedily in task order.
 * ------------------------------------------------------------------------- */

/*
 * dash_sim_schedule -- simulate `schedule` for the shape (B,Hq,Hkv,n tiles
 * per head, causal) on P SMs.
 *   makespan (out, may be NULL): the critical-path length.
 *   turn_order (out, may be NULL): int32 [B*Hq*n][n]; row ((b*Hq+hq)*n+i)
 *     lists the KV tiles accumulated into dQ tile i of head (b,hq), in order,
 *     padded with -1 (for DASH_SCHED_ATOMIC_NONDET: the order of the
 *     simulated reduce completions).
 *   num_tasks (out, may be NULL).
 * Returns DASH_OK, DASH_ERR_ARG, DASH_ERR_NOMEM or DASH_ERR_DEADLOCK.
 */
int dash_sim_schedule(int schedule, int causal, int B, int Hq, int Hkv, int n, int P,
                      double c, double r, double* makespan, int32_t* turn_order,
                      int64_t* num_tasks);

/*
 * dash_sim_schedule_band -- dash_sim_schedule for a causal sliding window
 * that touches `band` tile diagonals (tile pair (q, kv) visited iff
 * 0 <= q - kv < band; band >= 1).  The tiles outside the band are skipped the
 * way the masked tiles of a causal mask are; symmetric shift is shift there.
 * Same outputs and errors as dash_sim_schedule.
 */
int dash_sim_schedule_band(int schedule, int B, int Hq, int Hkv, int n, int band, int P,
                           double c, double r, double* makespan, int32_t* turn_order,
                           int64_t* num_tasks);

/*
 * dash_sim_schedule_cross -- dash_sim_schedule for a full mask with nq query
 * tiles and nkv key/value tiles per head (S_q != S_kv): each KV tile is one
 * task that visits every query tile (shift rotates from tile kv mod nq).
 * turn_order is int32 [B*Hq*nq][nkv].  Same outputs and errors otherwise.
 */
int dash_sim_schedule_cross(int schedule, int B, int Hq, int Hkv, int nq, int nkv, int P,
                            double c, double r, double* makespan, int32_t* turn_order,
                            int64_t* num_tasks);

/*
 * dash_sim_check_ranks -- would the kernel complete with this accumulation
 * table?  ranks: host uint16 [B*Hq*n][n], rank of KV tile j's partial in dQ
 * tile i (entries of masked pairs are ignored).  The visit lists and SM
 * assignment are those of `schedule` on P SMs.  Returns DASH_OK if every
 * tile's ranks are exactly 0..m-1 and the chain + order DAG is acyclic,
 * DASH_ERR_DEADLOCK otherwise, DASH_ERR_ARG on bad input.
 */
int dash_sim_check_ranks(int schedule, int causal, int B, int Hq, int Hkv, int n, int P,
                         const uint16_t* ranks);

/* ---------------------------------------------------------------------------
 * Debug and test hooks (used by the test-suite; not needed for normal use)
 * ------------------------------------------------------------------------- */

typedef struct {
    /* device int32 [B*Hq*n][nkv] or NULL (n, nkv: query and key/value tiles
     * per head): slot k of dQ tile t receives the KV index of the k-th
     * partial actually added (log written as it happens). */
    int32_t* order_log;
    /* device fp32 [B*Hq*n*nkv][128][D] or NULL: the fp32 dQ partial of pair
     * (b,hq,i,j) at index ((b*Hq+hq)*n+i)*nkv+j, as produced by the MMA. */
    float* dq_partials;
    /* device int32 [P] or NULL: worker slot used by CTA blockIdx.x (a
     * permutation of 0..P-1). */
    const int32_t* cta_perm;
    /* device int64 [P] or NULL: ns each worker slot waits before starting. */
    const int64_t* start_delay_ns;
    /* host uint16 [B*Hq*n][n] or NULL: replaces the accumulation ranks of a
     * deterministic schedule (checked by dash_sim_check_ranks first unless
     * skip_table_check is nonzero). */
    const uint16_t* ranks_host;
    int skip_table_check;
    /* two cudaEvent_t or NULL: recorded on `stream` immediately before and
     * after the persistent kernel's launch (for timing that kernel alone). */
    void* kernel_event_begin;
    void* kernel_event_end;
    /* device uint64 [P][64] or NULL: per-CTA clock64 cycles spent in each
     * wait / phase of the persistent kernel, slot = role*10 + site (role 0
     * dQ drain, 1 producer, 2 MMA issuer, 3 softmax/dS, 4 reduce issuer);
     * slot 63 = the CTA's total cycles.  Sites are named in the kernel
     * source.  Selects an instrumented build of the kernel. */
    unsigned long long* wait_cycles;
    /* device uint64 [64][32] or NULL (needs wait_cycles): clock64 of named
     * events (MMA issues, softmax/drain/reduce milestones) for the first 64
     * pairs of CTA 0; event ids are listed in the kernel source. */
    unsigned long long* event_trace;
    /* causal sliding window in tokens (as dash_attn_bwd_window), 0 = none;
     * needs causal = 1 and no ranks_host. */
    int window;
    /* key/value length when it differs from S (as dash_attn_bwd_cross),
     * 0 = S; needs causal = 0 and no ranks_host. */
    int skv;
    /* grouped-query heads on shift / symmetric shift: 0 = as dash_head_split
     * decides, 1 = one task per query head (D = 128 only), 2 = one task per
     * key/value head group.  Ignored with ranks_host (its table is laid out
     * for group tasks). */
    int head_split;
} dash_debug_opts;

/* dash_attn_bwd with debug hooks; same arguments and errors, plus
 * DASH_ERR_DEADLOCK when a supplied table fails the simulator check. */
int dash_attn_bwd_debug(const dash_bf16* q, const dash_bf16* k, const dash_bf16* v,
                        const dash_bf16* o, const dash_bf16* dO, const float* lse,
                        float* dq, dash_bf16* dk, dash_bf16* dv,
                        int B, int Hq, int Hkv, int S, int D, int causal, int schedule,
                        dash_stream_t stream, const dash_debug_opts* opts);

/*
 * dash_debug_tile_probe -- one (KV tile, Q tile) pair computed by the same
 * device building blocks as the persistent kernel, one CTA, no pipelining:
 * k, v, q, dO bf16 [128][D]; lse, delta fp32 [128]; outputs fp32 [128][128]
 * sT (S^T), pT (P^T), dpT (dP^T), dsT (dS^T incl. scale), and fp32 [128][D]
 * dv (P^T dO), dk (dS^T Q), dq (dS K).  diag=1 applies the causal mask of a
 * diagonal tile.  Synchronous.  For unit tests of the MMA operand layouts.
 */
int dash_debug_tile_probe(const dash_bf16* k, const dash_bf16* v, const dash_bf16* q,
                          const dash_bf16* dO, const float* lse, const float* delta,
                          int D, int diag, float* sT, float* pT, float* dpT, float* dsT,
                          float* dv, float* dk, float* dq);

#ifdef __cplusplus
}
#endif

#endif /* DASH_H */
