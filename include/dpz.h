/*
 * dpz — the data-parallel / ZeRO-1 gradient-synchronisation and optimizer step
 * for N simulated ranks whose replicas all live in one GPU's memory.
 *
 * A "rank" is a replica slab of an arena.  The collectives of the pages become
 * in-memory kernels: a ring "send" of a chunk is a load from another slab, the
 * ring's hop order is a fixed per-element fold order, and an all-gather is N
 * coalesced stores.  Every compute call is asynchronous on the caller's CUDA
 * stream, never synchronises the host, allocates nothing, and launches only
 * this library's own kernels (dpz_device_status, a read of a device flag, is
 * the one synchronous call).
 *
 * ------------------------------------------------------------------------
 * Layout (all buffers are owned and allocated by the caller, device memory)
 *
 *   N   number of ranks, 1 <= N <= 64
 *   P   elements per replica (a flat parameter / gradient arena), P % (8N) == 0
 *   C   chunk = shard = P / N; chunk c is elements [c*C, (c+1)*C)
 *   grads    [N][P] gradient dtype: slab r = grads + r*P = rank r's gradients
 *   weights  [N][P] weight dtype:   slab r = rank r's weight replica
 *   master, m, v   [P] fp32 each: the N ranks' shards laid end to end, so rank
 *            r's shard (A4 — Multi-GPU with NCCL and ZeRO-1, Part 2:
 *            shard_offset = rank * shard_size) is elements [r*C, (r+1)*C)
 *   ws       dpz_workspace_bytes(P, N) bytes, 16-byte aligned: norm partials
 *            and the global norm, written and read only by this library
 *
 * Chunk ownership: rank c owns chunk c.  The reduce-scatter is the ring of
 * "Lab 09 — Parallelism, simulated", §1, rotated so that its last receiver of
 * chunk c is rank c; element i of chunk c is therefore summed as the left fold
 *     acc = x[(c+1)%N][i];  acc = R(acc + x[(c+j)%N][i]) for j = 2..N
 * where R rounds to the gradient dtype (identity for fp32; round to nearest
 * even for bf16, so a bf16 ring rounds once per hop: 13.5 Multi-GPU from First
 * Principles, Exercise 8).  The average is R(acc / N): sum, then divide by N
 * (Lab 09 §2; A4 Part 3, ncclAvg).  The fold order never depends on the
 * launch configuration, so results are bit-for-bit reproducible.
 *
 * Alignment: bf16 buffers 16-byte aligned, fp32 buffers (master, m, v and
 * fp32 gradients or weights) 32-byte aligned, the workspace 16-byte aligned;
 * P % (8N) == 0, so that every chunk is a whole number of 8-element groups
 * (each lane moves 8 elements with one 128- or 256-bit access).
 *
 * Status: every call returns DPZ_OK or an error code without launching
 * anything when an argument is invalid (null pointer, N out of range,
 * P <= 0, P % N != 0, bad dtype, step < 1, overlapping buffers), and
 * DPZ_ERR_ALIGN for misaligned pointers or chunks (P/N not a multiple of 8).
 * A CUDA launch failure returns DPZ_ERR_CUDA.  dpz_last_error() gives the
 * calling thread's last message.  NaN and Inf inputs are not special-cased:
 * they propagate.
 *
 * Streams: the caller orders producers of `grads` before the call with
 * events (A4 Part 3: record an event on the compute stream, make the
 * communication stream wait on it), and consumers after it.  Every kernel is
 * launched with programmatic stream serialisation: its blocks may be placed
 * while the kernel before it on the same stream still runs, and they wait
 * for that kernel to complete (its writes visible) before they touch memory.
 * So the calls keep the stream's order after a kernel, a copy or an event
 * wait alike.
 *
 * CUDA graphs: every compute call except dp_grad_global_norm_static only
 * enqueues kernels on `stream`, so it can be captured into a CUDA graph and
 * replayed.  Call each once outside capture first (its launch configuration
 * is cached per device) and keep profiling off while capturing.
 */
#ifndef DPZ_H
#define DPZ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define DPZ_API __attribute__((visibility("default")))
#else
#define DPZ_API
#endif

/* element types */
#define DPZ_F32 0
#define DPZ_BF16 1
/* Gradients only: bf16 storage whose ring accumulates in fp32 (13.5 Multi-GPU
 * from First Principles, Exercise 8, second variant: each rank's vector is
 * rounded to bf16 once and the sum is accumulated in fp32).  The fold is
 *     acc = x[(c+1)%N][i];  acc = acc + x[(c+j)%N][i]  (fp32, j = 2..N)
 * and the stored average is RNE_bf16(acc / N), one rounding in all.  The
 * arena, the stored averages and every byte moved are those of DPZ_BF16; in
 * a ring of processes the partial sums would travel as fp32 (twice the
 * reduce-scatter's bytes), here they stay in registers. */
#define DPZ_BF16_ACC32 2

/* status codes */
#define DPZ_OK 0
#define DPZ_ERR_INVALID_ARG 1
#define DPZ_ERR_ALIGN 2
#define DPZ_ERR_CUDA 3

#define DPZ_MAX_RANKS 64

/* Per-call status in the workspace.  Three kernels stage their tiles through
 * shared memory with asynchronous bulk copies and wait for them on a barrier,
 * bounded by the SM clock (about two seconds): the norm of the owner chunks
 * (dp_grad_global_norm, dp_grad_global_norm_static), the one-kernel step
 * without clip (dp_zero1_step), and the AdamW + all-gather update from stored
 * averages (dp_zero1_step with clip, dp_zero1_update, dp_zero2_update).  If a
 * wait runs out the kernel gives up on that tile instead of hanging, and says
 * so in stream order, for a consumer on the same stream to see without
 * synchronising:
 *   - the uint32 at byte DPZ_WS_STATUS_OFFSET of the call's workspace holds
 *     DPZ_STATUS_* bits.  Every norm finalisation (dp_grad_global_norm,
 *     dp_grad_norm_finalize, dp_zero1_step with clip or with norm_out) writes
 *     the whole word; the update kernels that follow it only set
 *     DPZ_STATUS_UPDATE_SKIPPED.  So after dp_zero1_step with a workspace and
 *     a clip or a norm_out, and after dp_grad_norm_finalize followed by
 *     dp_zero1_update / dp_zero2_update, the word describes that step alone;
 *   - the norm written to the workspace and to norm_out is NaN;
 *   - an update with clipping whose norm has DPZ_STATUS_NORM_SKIPPED set is not
 *     applied at all: master/m/v and the weights keep their values and
 *     DPZ_STATUS_UPDATE_SKIPPED is set.
 * dp_zero1_step without clip and without norm_out runs no finalisation and
 * has no per-call word; there, and in every case, the device-wide flag of
 * dpz_device_status is raised as well.  NaN or Inf in the data is not a
 * status: it propagates into the norm and the update as any value does. */
#define DPZ_WS_STATUS_OFFSET 20
#define DPZ_STATUS_NORM_SKIPPED 1u   /* a tile of the norm's input was not read */
#define DPZ_STATUS_UPDATE_SKIPPED 2u /* a tile of master/m/v and the weights was
                                        not updated (it keeps the old values) */

/* AdamW hyperparameters for one step (A4 Part 4: the optimizer runs on the
 * owned shard).  The update, in fp32 with every operation rounded:
 *   g  = avg * s          s = clip/norm if clip_norm > 0 and norm > clip_norm,
 *                         else 1 (norm: of the averaged gradient, before the
 *                         step)
 *   m  = beta1*m + (1-beta1)*g
 *   v  = beta2*v + (1-beta2)*(g*g)
 *   mh = m / bc1,  vh = v / bc2,  bc = 1 - beta^step (host, double -> float)
 *   theta = theta - lr * (mh / (sqrt(vh) + eps) + weight_decay * theta)
 * weights = theta cast to the weight dtype (round to nearest even for bf16). */
typedef struct dpz_adamw_cfg {
    float lr;
    float beta1;
    float beta2;
    float eps;
    float weight_decay;
    int64_t step;        /* t >= 1, passed by the caller; the library keeps no state */
    float clip_norm;     /* > 0: global-norm clip to this value; <= 0: no clip */
    int store_avg;       /* dp_zero1_step without clip: nonzero also stores the
                            averaged gradient into chunk c of slab c */
} dpz_adamw_cfg;

/* Per-kernel timing collected while profiling is on (see dpz_profile_start). */
typedef struct dpz_kernel_stat {
    char name[48];
    int64_t launches;
    double total_ms;     /* sum of per-launch CUDA-event durations */
} dpz_kernel_stat;

/* Bytes of device workspace `ws` must provide for an arena of N slabs of P
 * elements: a 256-byte header (the norm), 256 first-stage sums and one fp64
 * sum of squares per 256-element segment of every chunk (about P/32 bytes).
 * Returns 0 for invalid P or N. */
DPZ_API size_t dpz_workspace_bytes(int64_t P, int N);

/* Ring reduce-scatter + average, in place (A4 Part 3: ncclReduceScatter of
 * pointers[i] into pointers[i] + shard_offset with ncclAvg; Lab 09 §1 ring).
 * grads: [N][P] device, dtype gdtype.  On return chunk c of slab c holds the
 * average of chunk c over the N ranks; every other chunk of every slab is
 * untouched.  Reads N*P and writes P elements. */
DPZ_API int dp_reduce_scatter_avg(void* grads, int64_t P, int N, int gdtype,
                                  void* stream);

/* Ring all-reduce + average (ZeRO-0), in place (A4 Part 3, zero_stage 0:
 * ncclAllReduce with ncclAvg; Lab 09 §1: reduce-scatter then all-gather).
 * On return every slab holds the average; chunk c equals what the
 * reduce-scatter leaves in chunk c of slab c.  Reads and writes N*P. */
DPZ_API int dp_allreduce_avg(void* grads, int64_t P, int N, int gdtype,
                             void* stream);

/* Global L2 norm of the averaged gradient held in the owner chunks (chunk c of
 * slab c, as left by dp_reduce_scatter_avg): each rank's sum of squares of its
 * shard, then the sum over ranks ("Distributed training", Gates: ZeRO stages
 * differ from DDP only in the order the global norm is summed).  Squares are
 * summed in fp32 within each 256-element segment (a fixed pairwise tree); the
 * segment sums are then added in a fixed two-level order (compensated fp32
 * chains, fp64 beyond them), which depends on P and N alone, so every entry
 * point and every launch configuration gives the same bits.
 * Writes the norm into ws (for zero1_adamw_step) and, if norm_out is not
 * NULL, to *norm_out (device pointer to one float). */
DPZ_API int dp_grad_global_norm(const void* grads, int64_t P, int N, int gdtype,
                                void* ws, float* norm_out, void* stream);

/* Sharded AdamW (A4 Part 4, step 1: adamw_update on this rank's shard only).
 * For every rank c: reads the averaged chunk c of slab c, updates master/m/v
 * elements [c*C, (c+1)*C) and writes the cast weights into chunk c of slab c
 * of `weights` only (the all-gather is dp_allgather).  If cfg->clip_norm > 0
 * the clip scale uses the norm that dp_grad_global_norm left in ws (ws may be
 * NULL otherwise).  gdtype/wdtype: DPZ_F32 or DPZ_BF16. */
DPZ_API int zero1_adamw_step(const void* grads, float* master, float* m,
                             float* v, void* weights, int64_t P, int N,
                             int gdtype, int wdtype, const dpz_adamw_cfg* cfg,
                             const void* ws, void* stream);

/* All-gather (A4 Part 4, step 2: ncclAllGather of the updated shards; Lab 09
 * §1 all-gather phase): chunk c of slab c is copied into chunk c of every
 * other slab, in place.  Reads P and writes (N-1)*P elements. */
DPZ_API int dp_allgather(void* weights, int64_t P, int N, int wdtype,
                         void* stream);

/* The whole ZeRO-1 step, fused: reduce-scatter + average -> (global norm and
 * clip) -> AdamW on each rank's shard -> cast -> all-gather into all N weight
 * slabs.  Bit-identical to calling dp_reduce_scatter_avg,
 * dp_grad_global_norm (when clipping), zero1_adamw_step and dp_allgather in
 * turn.  Without clipping it is one kernel that reads each gradient byte once
 * and writes the averages only if cfg->store_avg, plus the norm's
 * finalisation when norm_out is given (for arenas of at most 32 segments of
 * 256 elements, one kernel on a thread-block cluster does both); with clipping it is three
 * (reduce + norm partials and averages store, norm finalize, AdamW + cast +
 * broadcast), because the clip scale depends on every element.  norm_out
 * (device, may be NULL) receives the global norm; ws is required when
 * clipping or when norm_out is given. */
DPZ_API int dp_zero1_step(void* grads, float* master, float* m, float* v,
                          void* weights, int64_t P, int N, int gdtype,
                          int wdtype, const dpz_adamw_cfg* cfg, void* ws,
                          float* norm_out, void* stream);

/* ---------------------------------------------------------------------
 * Buckets (overlap with the backward pass) and ZeRO-2 (sharded gradients)
 *
 * A backward pass produces the gradients layer by layer, from the last layer
 * to the first, so a bucket of the arena can be reduced while the rest is
 * still being computed ("A4 — Multi-GPU with NCCL and ZeRO-1", Part 3: each
 * layer's reduction runs on a separate stream after an event recorded on the
 * compute stream; "Lab 09 — Parallelism, simulated", §2: DDP all-reduces 25
 * MB buckets as backward produces them; "Distributed training", "Overlap and
 * graphs").  Record an event on the producing stream after each bucket is
 * written and make the stream of these calls wait on it.
 *
 * Buckets reduce element ranges [lo, lo+n) of the arena (lo and n multiples
 * of 8; any ranges, in any order, each element once per step).  With ws,
 * each range must start and end on 256-element segment boundaries of its
 * chunks ((lo mod C) and ((lo+n) mod C) multiples of 256) and its norm
 * partials are written; once every bucket is reduced, dp_grad_norm_finalize
 * gives the same norm, bit for bit, as the whole-arena calls.
 *
 * max_ctas bounds the thread blocks of the reduction kernel.  0: one pass
 * with as many blocks as the range needs, the fastest when nothing else runs.
 * > 0: at most max(max_ctas, c) blocks, where c is the number of chunks the
 * range touches, each looping over its part of the range.  A reduction that
 * runs beside compute kernels on other streams (a backward pass) should leave
 * them most of the GPU: with one block per SM it hid about 60 % of its time
 * behind a compute-bound stand-in on GB300, against about 10 % with 0, whose
 * blocks take every SM slot that the compute kernels free.  The result is the
 * same, bit for bit, for every max_ctas.  Negative: DPZ_ERR_INVALID_ARG.
 * ------------------------------------------------------------------- */

/* ZeRO-1 with buckets: reduce + average elements [lo, lo+n) of the arena in
 * place (the average of element e of chunk c goes to slab c), as
 * dp_reduce_scatter_avg does for the whole arena.  ws may be NULL (no norm
 * partials). */
DPZ_API int dp_reduce_scatter_avg_range(void* grads, int64_t P, int N, int gdtype,
                                        int64_t lo, int64_t n, void* ws, int max_ctas,
                                        void* stream);

/* ZeRO-2: gradients are sharded too ("Lab 09 — Parallelism, simulated", §4:
 * stage 2 shards the gradients, 2Ψ + 14Ψ/N bytes per rank; "Distributed
 * training": ZeroSharded[M, N, 2]).  Reduce + average a bucket of N ranks' gradients for
 * arena elements [lo, lo+n), held in a staging buffer [N][n] (rank r's
 * values at staging + r*n), into `shards` [P]: the average of element e is
 * written at shards[e], which belongs to rank e / C's shard.  The staging
 * buffer can be reused for the next bucket once this call has run, so no
 * rank keeps a full gradient replica. */
DPZ_API int dp_reduce_scatter_avg_bucket(const void* staging, int64_t lo, int64_t n,
                                         void* shards, int64_t P, int N, int gdtype,
                                         void* ws, int max_ctas, void* stream);

/* The global norm from the partials that the range or bucket calls left in
 * ws (all of [0, P) reduced, with ws); writes it into ws and, if not NULL,
 * *norm_out. */
DPZ_API int dp_grad_norm_finalize(void* ws, int64_t P, int N, float* norm_out,
                                  void* stream);

/* The second half of dp_zero1_step: AdamW on every rank's shard reading the
 * averaged chunk c of slab c, cast, and the all-gather into all N weight
 * slabs (one kernel).  Clip scale from the norm in ws when clip_norm > 0. */
DPZ_API int dp_zero1_update(const void* grads, float* master, float* m, float* v,
                            void* weights, int64_t P, int N, int gdtype, int wdtype,
                            const dpz_adamw_cfg* cfg, const void* ws, void* stream);

/* The same for ZeRO-2: the averages are read from shards [P]. */
DPZ_API int dp_zero2_update(const void* shards, float* master, float* m, float* v,
                            void* weights, int64_t P, int N, int gdtype, int wdtype,
                            const dpz_adamw_cfg* cfg, const void* ws, void* stream);

/* The global norm of dp_grad_global_norm for callers that cannot allocate
 * device memory.  The pages have no counterpart to this call.  It serves code
 * that must not call cudaMalloc or any allocator of its own: a plug-in running
 * inside a host framework whose caching allocator owns all device memory, or
 * a service that reserves its whole memory budget up front.  Such a caller
 * cannot provide the workspace of dp_grad_global_norm.  Here the partial sums
 * live in a fixed 4 MiB array of device memory that the library declares at
 * file scope, so the call allocates nothing; it needs
 * dpz_workspace_bytes(P, N) <= 4 MiB (for example the GPT-2 124M arena at
 * N = 8) and returns DPZ_ERR_INVALID_ARG with a clear message beyond that.
 * Inputs and output are as in dp_grad_global_norm; norm_out (one float of
 * device memory) is required.
 *
 * The first call on a device looks up the array's address on that device
 * (cudaGetSymbolAddress), so make that first call before any stream capture.
 * Every later call made outside a stream capture looks it up again (after a
 * device reset the array may sit elsewhere).
 * Every GPU that loads the library holds the 4 MiB array until the process
 * exits.  All calls share it: each call clears what must start at zero, but
 * calls whose kernels overlap on the GPU (unordered streams) race with each
 * other and give wrong results. */
DPZ_API int dp_grad_global_norm_static(const void* grads, int64_t P, int N,
                                       int gdtype, float* norm_out, void* stream);

/* The calling thread's last error message ("" if none). */
DPZ_API const char* dpz_last_error(void);

/* Library version string. */
DPZ_API const char* dpz_version(void);

/* Device-side error flag of the current device, read and cleared: 1 if any
 * bulk-copy staged kernel (see DPZ_WS_STATUS_OFFSET) gave up on a tile since
 * the last call, else 0.  Synchronous: call it after the work in question has
 * finished (for example after cudaStreamSynchronize), not inside a stream
 * capture.  Returns DPZ_ERR_INVALID_ARG for a NULL flag_out, DPZ_ERR_CUDA if
 * the read fails. */
DPZ_API int dpz_device_status(int* flag_out);

/* Self-test of the timeout path (no counterpart on the pages).  Launches, on
 * `stream`, one of the staged kernels on a one-tile arena (N = 1, P = 8) laid
 * out in `buf`, DPZ_SELFTEST_BUF_BYTES bytes of caller device memory, 256-byte
 * aligned:
 *   +0     the arena's workspace (DPZ_WS_STATUS_OFFSET is relative to it)
 *   +2560  norm_out, one float
 *   +2816  gradients (bf16, 8 elements); +2848, +2880, +2912 master, m, v
 *          (fp32, 8 each); +2944 weights (bf16, 8)
 * The kernel's barrier expects 16 bytes more than its bulk loads deliver and
 * its wait is bounded by about 10^8 SM cycles (some 0.05 to 0.1 s) instead of
 * the usual two seconds.  Every copy it issues completes, so the wait runs out
 * and nothing is in flight when the kernel gives up.  kernel:
 *   DPZ_SELFTEST_UPDATE  the AdamW + all-gather update (without clip): sets
 *                        DPZ_STATUS_UPDATE_SKIPPED in the workspace's status
 *                        word and NaN in norm_out;
 *   DPZ_SELFTEST_NORM    the norm of the owner chunks, then the finalisation:
 *                        status DPZ_STATUS_NORM_SKIPPED, norm_out NaN;
 *   DPZ_SELFTEST_STEP    the step without clip with norm partials, then the
 *                        finalisation: status NORM_SKIPPED | UPDATE_SKIPPED,
 *                        norm_out NaN.
 * No kernel writes the arena's gradients, master/m/v or weights, and each
 * raises the device flag of dpz_device_status; the context stays usable.
 * Returns DPZ_ERR_INVALID_ARG for a NULL buf or an unknown kernel,
 * DPZ_ERR_ALIGN for a buf not 256-byte aligned, DPZ_ERR_CUDA if a launch
 * fails. */
#define DPZ_SELFTEST_BUF_BYTES 4096
#define DPZ_SELFTEST_UPDATE 0
#define DPZ_SELFTEST_NORM 1
#define DPZ_SELFTEST_STEP 2
DPZ_API int dpz_selftest_staged_timeout(int kernel, void* buf, void* stream);

/* Self-test of the division inside the average (no counterpart on the pages,
 * which fix only that the reduced sum is divided by N).  For N not a power of
 * two the library divides with Markstein's correction of a reciprocal
 * product instead of an IEEE division; this call checks that the two agree
 * for every float.  It sets, on `stream`, the 8-byte device counter
 * `mismatches` (caller memory, 16-byte aligned) to the number of (pattern,
 * path) cases, over all 2^32 float bit patterns a, where the library's
 * quotient a/N differs bit for bit from the IEEE round-to-nearest quotient
 * (two NaNs count as equal).  Each pattern is checked twice: in a group of
 * 8 consecutive patterns, as the streaming kernels divide them, and in a
 * group of 8 copies of itself.  0 means the average is correctly rounded for
 * this N.  It takes a few milliseconds.  Returns DPZ_ERR_INVALID_ARG for
 * N outside [1, DPZ_MAX_RANKS] or a NULL pointer, DPZ_ERR_ALIGN for one not 16-byte aligned,
 * DPZ_ERR_CUDA if the launch fails. */
DPZ_API int dpz_selftest_average_division(int N, unsigned long long* mismatches,
                                          void* stream);

/* Number of kernels this library has launched since it was loaded. */
DPZ_API int64_t dpz_launch_count(void);

/* Profiling: while on, every kernel launch is bracketed by a pair of CUDA
 * events recorded on the launch's own stream (capacity: max_launches
 * launches; later launches are not timed).  dpz_profile_stop synchronises
 * those events, fills up to max_stats per-kernel totals, sets *n_stats and
 * turns profiling off. */
DPZ_API int dpz_profile_start(int max_launches);
DPZ_API int dpz_profile_stop(dpz_kernel_stat* stats, int max_stats, int* n_stats);

#ifdef __cplusplus
}
#endif

#endif /* DPZ_H */
