/*
 * CPU oracle for the data-parallel / ZeRO-1 step.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may include, link or
 * call this code: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it. It shares no code with the CUDA library.
 *
 * Every function is a plain, slow, literal restatement of the pages:
 *   - "Lab 09 — Parallelism, simulated", §1 Ring all-reduce (the N = 3 table,
 *     the byte counts, and the Tips: build every message, then deliver);
 *   - "A4 — Multi-GPU with NCCL and ZeRO-1", Part 2 (shard offset
 *     rank * shard_size), Part 3 (ReduceScatter with ncclAvg), Part 4
 *     (adamw_update on the shard, then AllGather);
 *   - "13.5 Multi-GPU from First Principles", §13.5.3 (Eq. 13.5.1) and
 *     Exercise 8 (a bf16 ring rounds the partial sum once per hop);
 *   - "Distributed training" (noeira), "Gates" (ZeRO stages equal DDP bit for
 *     bit without clipping; with clipping only the norm's summation order
 *     differs).
 *
 * Values are carried in their storage type: ORC_F64 as double, ORC_F32 as
 * float, ORC_BF16 as the upper 16 bits of an IEEE float (uint16_t).
 */
#ifndef DPZ_ORACLE_H
#define DPZ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F64 = 2, ORC_BF16_ACC32 = 3 };

/* ORC_BF16_ACC32: bf16 storage whose ring carries fp32 partial sums ("13.5
 * Multi-GPU from First Principles", Exercise 8, second variant: each vector
 * is rounded to bf16 once and the sum is accumulated in fp32).  The rank
 * buffers hold the bf16 values as floats, reduce-scatter messages are fp32
 * (4 bytes per element), the owner's average is rounded to bf16 once, and
 * all-gather messages carry those bf16 averages (2 bytes per element). */

typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
    int64_t step;       /* t >= 1 */
    float clip_norm;    /* <= 0: no clipping */
} orc_adamw_cfg;

/* float -> bf16, round to nearest, ties to even; NaN stays a (quiet) NaN. */
uint16_t orc_f32_to_bf16(float x);
float orc_bf16_to_f32(uint16_t h);
void orc_f32_to_bf16_array(const float* x, uint16_t* out, int64_t n);

/* Ring reduce-scatter over an arena of N replica slabs of P elements
 * (slab r = rank r's buffer).  Runs `steps` (<= N-1) steps.  In step t rank r
 * sends chunk (r - t - rho) mod N to rank r+1, which adds it into its own copy
 * of that chunk (rounding to the storage type).  rho = 0 is the lab's table;
 * rho = 1 makes rank c the owner of chunk c (ZeRO-1 offset rank*shard_size).
 * sent[r] accumulates the bytes rank r sends (may be NULL). Returns 0 or -1. */
int orc_ring_reduce_scatter(void* arena, int N, int64_t P, int dtype, int rho,
                            int steps, int64_t* sent);

/* Ring all-gather: step t, rank r sends chunk (r + 1 - rho - t) mod N and the
 * receiver overwrites its copy. */
int orc_ring_allgather(void* arena, int N, int64_t P, int dtype, int rho,
                       int steps, int64_t* sent);

/* Owner of chunk c after a full reduce-scatter with rotation rho. */
int orc_owner(int c, int N, int rho);

/* The owner of every chunk divides its fully reduced chunk by N (sum, then
 * divide), rounding to the storage type. */
int orc_average_owned(void* arena, int N, int64_t P, int dtype, int rho);

/* Reduce-scatter then owner average in one ring session (the partial sums of
 * the fp32-accumulating bf16 ring exist only inside the ring). */
int orc_reduce_scatter_avg(void* arena, int N, int64_t P, int dtype, int rho,
                           int64_t* sent);

/* Full ring all-reduce-average: reduce-scatter, owner average, all-gather. */
int orc_ring_allreduce_avg(void* arena, int N, int64_t P, int dtype, int rho,
                           int64_t* sent);

/* Star all-reduce (sum onto rank 0, broadcast back), only to count bytes:
 * recv[r] = bytes rank r receives. Sums into slab 0 and copies back. */
int orc_star_allreduce(void* arena, int N, int64_t P, int dtype, int64_t* recv);

/* Sum of squares of the owned (averaged) chunks, chunk 0..N-1 in order, each
 * chunk summed sequentially in double. */
double orc_sumsq_owned(const void* arena, int N, int64_t P, int dtype, int rho);

/* norm = (float)sqrt(sumsq); scale = clip/norm if clip > 0 and norm > clip,
 * else 1. */
void orc_clip_scale(double sumsq, float clip, float* norm, float* scale);

/* AdamW with decoupled weight decay on n elements, fp32 arithmetic:
 *   g  = grad * scale
 *   m  = b1*m + (1-b1)*g ;  v = b2*v + (1-b2)*(g*g)
 *   mh = m/bc1 ; vh = v/bc2      (bc = 1 - beta^t, host double, to float)
 *   theta = theta - lr*(mh/(sqrt(vh)+eps) + wd*theta)          */
void orc_adamw(float* theta, float* m, float* v, const void* grad, int gdtype,
               int64_t n, const orc_adamw_cfg* cfg, float scale);

/* Bias corrections as the oracle computes them. */
void orc_bias_corrections(const orc_adamw_cfg* cfg, float* bc1, float* bc2);

/* ZeRO-1 step over N ranks (rho = 1):
 *   ring reduce-scatter of grads[N][P] -> owner average -> (norm, clip scale)
 *   -> AdamW on each rank's shard r of master/m/v (the P-long arrays are the
 *   N shards laid end to end) -> cast to the weight dtype into rank r's chunk
 *   r of weights[N][P] -> ring all-gather of weights.
 * ext_sumsq >= 0 replaces the arena's own sum of squares (for checking a
 * window of a larger arena).  Outputs: grads (owner chunks hold averages;
 * other chunks hold ring partials), master/m/v, weights, norm, scale, bytes
 * sent per rank in each phase (may be NULL). */
int orc_zero1_step(void* grads, float* master, float* m, float* v,
                   void* weights, int N, int64_t P, int gdtype, int wdtype,
                   const orc_adamw_cfg* cfg, double ext_sumsq,
                   float* norm_out, float* scale_out,
                   int64_t* sent_rs, int64_t* sent_ag);

/* ZeRO-0 (plain data parallel) step: ring all-reduce-average of grads, then
 * every rank keeps a full copy of master/m/v (master_full etc. are [N][P]) and
 * updates all P elements; weights[N][P] are each rank's cast. The norm is
 * taken from each rank's full averaged vector in chunk order. */
int orc_zero0_step(void* grads, float* master_full, float* m_full,
                   float* v_full, void* weights, int N, int64_t P, int gdtype,
                   int wdtype, const orc_adamw_cfg* cfg, float* norm_out,
                   int64_t* sent);

#ifdef __cplusplus
}
#endif
#endif
