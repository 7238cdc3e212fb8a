// Optimizer-side kernel: sharded AdamW on every rank's owned chunk, the cast
// to the weight dtype, and the write of the new weights into the owner slab
// (zero1_adamw_step, averages loaded from the owner slab) or into all N slabs
// (the single-kernel step without clip, averages computed in place by the
// ring fold).  AdamW + all-gather from stored averages (the clipped step,
// dp_zero1_update, dp_zero2_update) is the bulk-copy staged kernel of
// staged.cu, to which launch_adamw hands that case.
#include "bulk.cuh"
#include "device.cuh"
#include "internal.h"

namespace dpz {

// NT > 0: N == NT known at compile time (the fold and the broadcast unroll);
// NT == 0: any N, read from n_rt.
// Without FOLD the average of element e (chunk c) is read at
// grads + (c*avg_stride + e) elements: avg_stride = P for the owner slabs of
// the arena, 0 for a compact [P] buffer of gradient shards.
// One-shot grid, one segment per warp (device.cuh).  Register caps that keep
// more blocks, hence more loads, in flight without spilling: 64 registers
// (four blocks per SM) for the load-owner variant, 80 (three blocks) for the
// fold.  The launchers instantiate this kernel with NT == 0 only: the step
// without clip for N <= 8, and for larger N where its tiles fit, is the
// staged kernel of staged.cu, and small arenas take k_zero1_small.
template <bool FOLD>
struct AdamwBlocksPerSm {
    static constexpr int value = FOLD ? 3 : 4;
};

// The work of one lane: group gi of chunk c (nothing if gi is past the chunk
// end).  Returns the lane's sum of squares of its averaged values (SUMSQ),
// else 0.
template <int GDT, int WDT, int NT, bool FOLD, bool BCAST, bool SUMSQ>
__device__ __forceinline__ float adamw_group(char* __restrict__ grads, float* __restrict__ master,
                                             float* __restrict__ mom, float* __restrict__ var,
                                             char* __restrict__ weights, int64_t P, int64_t C,
                                             int N, int c, int64_t gi, const Avg& avg,
                                             const AdamArgs& h, int store_avg, bool do_scale,
                                             float scale, int64_t avg_stride)
{
    constexpr int GES = Group<GDT>::kBytes;
    constexpr int WES = Group<WDT>::kBytes;
    const int64_t gslab = P * GES;
    const int64_t wslab = P * WES;
    float ss = 0.0f;
    if (gi >= C / kGroup) return ss;
    const int64_t e = c * C + gi * kGroup;      // element index (same in every slab)
    constexpr int NS = NT > 0 ? NT : 1;
    const char* src[NS];
    if constexpr (NT > 0) ring_sources<NT>(grads, gslab, c, src);
    float g[8];
    if (FOLD) {
        if constexpr (NT > 0) {
            typename Group<GDT>::Raw raw[NT];
#pragma unroll
            for (int j = 0; j < NT; ++j) raw[j] = Group<GDT>::load_raw(src[j] + e * GES);
            fold_loaded<GDT, NT>(raw, g);
        } else {
            ring_fold<GDT>(grads, gslab, e * GES, c, N, g);
        }
        average8<GDT, NT>(g, avg);
        if (SUMSQ) ss = sumsq8(g);
        if (store_avg) store_group<GDT>(grads + c * gslab + e * GES, g);
    } else {
        load_group<GDT>(grads + (c * avg_stride + e) * GES, g);
    }
    float th[8], mm[8], vv[8];
    load_group<0>(reinterpret_cast<const char*>(master + e), th);
    load_group<0>(reinterpret_cast<const char*>(mom + e), mm);
    load_group<0>(reinterpret_cast<const char*>(var + e), vv);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float gq = do_scale ? __fmul_rn(g[q], scale) : g[q];
        adamw_elem(th[q], mm[q], vv[q], gq, h);
    }
    store_group<0>(reinterpret_cast<char*>(master + e), th);
    store_group<0>(reinterpret_cast<char*>(mom + e), mm);
    store_group<0>(reinterpret_cast<char*>(var + e), vv);
    const typename Group<WDT>::Raw w = Group<WDT>::pack(th);
    if (BCAST) {
        if constexpr (NT > 0) {
#pragma unroll
            for (int r = 0; r < NT; ++r) Group<WDT>::store_raw(weights + r * wslab + e * WES, w);
        } else {
            for (int r = 0; r < N; ++r) Group<WDT>::store_raw(weights + r * wslab + e * WES, w);
        }
    } else {
        Group<WDT>::store_raw(weights + c * wslab + e * WES, w);
    }
    return ss;
}

template <int GDT, int WDT, int NT, bool FOLD, bool BCAST, bool SUMSQ>
__global__ void __launch_bounds__(kBlock, AdamwBlocksPerSm<FOLD>::value)
k_adamw(char* __restrict__ grads, float* __restrict__ master, float* __restrict__ mom,
        float* __restrict__ var, char* __restrict__ weights, int64_t P, int64_t C, int n_rt,
        Avg avg, AdamArgs h, int store_avg, WsHeader* __restrict__ hdr,
        double* __restrict__ partials, int64_t avg_stride)
{
    const int N = NT > 0 ? NT : n_rt;
    const int64_t segs = segments_per_chunk(C);
    const int lane = threadIdx.x & 31;
    pdl_enter();
    if (SUMSQ && blockIdx.x == 0 && threadIdx.x == 0) hdr->arrive = 0u;
    const int64_t sw = global_warp();
    if (sw >= (int64_t)N * segs) return;                 // whole warps
    const SegPos p = seg_pos(sw, segs);

    // clip scale from the global norm of the averaged gradient; a norm whose
    // input was not read in full is unknown, and then nothing is updated
    float scale = 1.0f;
    bool do_scale = false;
    if (!FOLD && h.clip > 0.0f) {
        if (hdr->status & DPZ_STATUS_NORM_SKIPPED) {
            if (threadIdx.x == 0) atomicOr(&hdr->status, DPZ_STATUS_UPDATE_SKIPPED);
            return;
        }
        const float nrm = hdr->norm;
        if (nrm > h.clip) {
            scale = __fdiv_rn(h.clip, nrm);
            do_scale = true;
        }
    }

    const float ss = adamw_group<GDT, WDT, NT, FOLD, BCAST, SUMSQ>(
        grads, master, mom, var, weights, P, C, N, p.c, p.seg * 32 + lane, avg, h, store_avg,
        do_scale, scale, avg_stride);
    if (SUMSQ) {
        const float t = warp_sum_f32(ss);
        if (lane == 0) partials[p.c * segs + p.seg] = (double)t;
    }
}

// The whole step without clip for a small arena, norm included, in one
// launch: a thread-block cluster of up to 8 CTAs (one per SM).  Each
// 256-element segment of the list gets a team of four warps, and each thread
// two consecutive elements of one 8-element group (lanes 4k .. 4k+3 of a warp
// share group k), so every thread's serial chain of loads, ring fold,
// average, AdamW and stores covers 2 elements instead of 8.  The segment's
// partial is the same fixed tree as everywhere else: each thread squares and
// adds its pair (sumsq8's first level), the 4-lane shuffles add the pairs as
// sumsq8's second and third levels do, and the first warp of the team adds the
// 32 group sums with warp_sum_f32, group g in lane g.  Every team writes its
// partial to the workspace and, over distributed shared memory, into CTA 0's
// copy of sp.  After a cluster barrier, warp 0 of CTA 0 adds the partials
// exactly as k_norm_finalize does when it runs as one block: thread t holds
// partial t (t < total, else 0; a chain of one term gives its term back, by
// Sum2 or in fp64) and block_sum adds them with warp_sum in each warp, then
// adds the warp sums with warp_sum again.  With at most 32
// partials every partial sits in warp 0, the other warps' sums are +0, and
// adding +0 to a sum of squares leaves it unchanged, so warp 0's warp_sum
// alone has the same bits.  So the step and its norm equal the two-kernel
// path's bit for bit, in one launch instead of two, for arenas of at most
// kSmallStepSegments segments, where latency is the cost.  The average takes
// the correctly rounded quotient element by element (Markstein's correction
// where its theorem holds, else IEEE division), the same value divide8 gives.
// Device time per step (20 steps per CUDA graph), tiny arena (N = 4, 16
// segments): one 512-thread block 5.1 us, a cluster with one warp per
// segment 3.9 us, four warps per segment 3.4 us (32 segments: 4.3-4.7 and
// 3.7-4.1 us; one segment: 4.1 and 3.2 us).
static_assert(kSmallStepSegments <= 32, "every partial is held by warp 0 of CTA 0");
constexpr int kClusterCtas = 8;                                 // portable cluster size
constexpr int kTeam = 128;                                      // threads per segment
constexpr int kSmallMaxThreads =
    kTeam * (int)((kSmallStepSegments + kClusterCtas - 1) / kClusterCtas);

// Two consecutive elements of one storage type, as Group does for eight.
template <int DT>
struct Pair;

template <>
struct Pair<0> {
    static __device__ __forceinline__ void load(const char* p, float x[2])
    {
        const float2 v = *reinterpret_cast<const float2*>(p);
        x[0] = v.x;
        x[1] = v.y;
    }
    static __device__ __forceinline__ void store(char* p, const float x[2])
    {
        *reinterpret_cast<float2*>(p) = make_float2(x[0], x[1]);
    }
    static __device__ __forceinline__ void round2(float[2]) {}
    static __device__ __forceinline__ void hop_round2(float[2]) {}
};

template <>
struct Pair<1> {
    static __device__ __forceinline__ void load(const char* p, float x[2])
    {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
        x[0] = bf16_lo(w);
        x[1] = bf16_hi(w);
    }
    static __device__ __forceinline__ void store(char* p, const float x[2])
    {
        *reinterpret_cast<uint32_t*>(p) = pack_bf16x2(x[0], x[1]);
    }
    static __device__ __forceinline__ void round2(float x[2]) { round_bf16x2(x[0], x[1]); }
    static __device__ __forceinline__ void hop_round2(float x[2]) { round2(x); }
};

template <>
struct Pair<2> : Pair<1> {
    static __device__ __forceinline__ void hop_round2(float[2]) {}
};

// a / N correctly rounded, one element at a time: the value divide8 gives
// (its two paths agree with IEEE division for every float, so which path an
// element takes does not change its bits).
template <int NT>
__device__ __forceinline__ float divide1(float a, const Avg& avg)
{
    constexpr bool kPow2 = NT > 0 && (NT & (NT - 1)) == 0;
    if (kPow2 || (NT == 0 && avg.pow2)) return __fmul_rn(a, avg.invN);
    return markstein_ok(a) ? div_markstein(a, avg.fN, avg.invN) : __fdiv_rn(a, avg.fN);
}

// The work of one thread: elements e and e + 1 of chunk c (the step without
// clip); returns their sum of squares, x0*x0 + x1*x1 (0 if nothing to do).
template <int GDT, int WDT, int NT>
__device__ __forceinline__ float small_pair(char* __restrict__ grads, float* __restrict__ master,
                                            float* __restrict__ mom, float* __restrict__ var,
                                            char* __restrict__ weights, int64_t P, int N, int c,
                                            int64_t e, const Avg& avg, const AdamArgs& h,
                                            int store_avg)
{
    using G = Pair<GDT>;
    constexpr int GES = Group<GDT>::kBytes;
    constexpr int WES = Group<WDT>::kBytes;
    const int64_t gslab = P * GES;
    float g[2];
    if constexpr (NT > 0) {
        float x[NT][2];
#pragma unroll
        for (int j = 0; j < NT; ++j) {                  // ring order: slabs c+1, ..., c
            int r = c + 1 + j;
            if (r >= NT) r -= NT;
            G::load(grads + r * gslab + e * GES, x[j]);
        }
        g[0] = x[0][0];
        g[1] = x[0][1];
#pragma unroll
        for (int j = 1; j < NT; ++j) {
            g[0] = __fadd_rn(g[0], x[j][0]);
            g[1] = __fadd_rn(g[1], x[j][1]);
            G::hop_round2(g);
        }
    } else {
        int r = c + 1;
        if (r >= N) r -= N;
        G::load(grads + r * gslab + e * GES, g);
        for (int j = 2; j <= N; ++j) {
            ++r;
            if (r >= N) r -= N;
            float x[2];
            G::load(grads + r * gslab + e * GES, x);
            g[0] = __fadd_rn(g[0], x[0]);
            g[1] = __fadd_rn(g[1], x[1]);
            G::hop_round2(g);
        }
    }
    g[0] = divide1<NT>(g[0], avg);
    g[1] = divide1<NT>(g[1], avg);
    G::round2(g);
    if (store_avg) G::store(grads + c * gslab + e * GES, g);
    const float ss = __fadd_rn(__fmul_rn(g[0], g[0]), __fmul_rn(g[1], g[1]));
    float th[2], mm[2], vv[2];
    Pair<0>::load(reinterpret_cast<const char*>(master + e), th);
    Pair<0>::load(reinterpret_cast<const char*>(mom + e), mm);
    Pair<0>::load(reinterpret_cast<const char*>(var + e), vv);
#pragma unroll
    for (int q = 0; q < 2; ++q) adamw_elem(th[q], mm[q], vv[q], g[q], h);
    Pair<0>::store(reinterpret_cast<char*>(master + e), th);
    Pair<0>::store(reinterpret_cast<char*>(mom + e), mm);
    Pair<0>::store(reinterpret_cast<char*>(var + e), vv);
    const int64_t wslab = P * WES;
    if constexpr (NT > 0) {
#pragma unroll
        for (int r = 0; r < NT; ++r) Pair<WDT>::store(weights + r * wslab + e * WES, th);
    } else {
        for (int r = 0; r < N; ++r) Pair<WDT>::store(weights + r * wslab + e * WES, th);
    }
    return ss;
}

template <int GDT, int WDT, int NT>
__global__ void __launch_bounds__(kSmallMaxThreads)
k_zero1_small(char* __restrict__ grads, float* __restrict__ master, float* __restrict__ mom,
              float* __restrict__ var, char* __restrict__ weights, int64_t P, int64_t C, int N,
              Avg avg, AdamArgs h, int store_avg, WsHeader* __restrict__ hdr,
              double* __restrict__ partials, float* __restrict__ norm_out)
{
    __shared__ double sp[kSmallStepSegments];       // CTA 0's copy receives the partials
    __shared__ float gsum[kSmallMaxThreads / kTeam][32];   // each team's 32 group sums
    const int64_t segs = segments_per_chunk(C);
    const int64_t total = (int64_t)N * segs;        // <= kSmallStepSegments
    const int tid = threadIdx.x, lane = tid & 31;
    const int team = tid / kTeam, tt = tid % kTeam;
    const int grp = tt >> 2, quarter = tt & 3;       // group of the segment, pair of the group
    const int64_t sw = (int64_t)blockIdx.x * (blockDim.x / kTeam) + team;
    pdl_enter();
    cluster_arrive_relaxed();      // CTA 0 has started before anyone writes its shared memory
    float s = 0.0f;
    if (sw < total) {                               // whole teams
        const SegPos p = seg_pos(sw, segs);
        const int64_t gi = p.seg * 32 + grp;
        if (gi < C / kGroup)
            s = small_pair<GDT, WDT, NT>(grads, master, mom, var, weights, P, N, p.c,
                                         p.c * C + gi * kGroup + 2 * quarter, avg, h, store_avg);
    }
    // the group's sum of squares in sumsq8's tree: (p0 + p1) + (p2 + p3)
    s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, 1));
    s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, 2));
    if (quarter == 0) gsum[team][grp] = s;
    __syncthreads();
    float t = 0.0f;
    if (tt < 32 && sw < total) t = warp_sum_f32(gsum[team][lane]);   // whole warps
    cluster_wait();
    if (sw < total && tt == 0) {
        partials[sw] = (double)t;                   // sw = p.c * segs + p.seg
        store_shared_of_rank(&sp[sw], 0, (double)t);
    }
    cluster_arrive_release();
    cluster_wait();                                 // every partial is in CTA 0's sp
    if (blockIdx.x != 0 || threadIdx.x >= 32) return;
    const double r = warp_sum(threadIdx.x < total ? 0.0 + sp[threadIdx.x] : 0.0);
    if (threadIdx.x == 0) {
        const float nrm = __double2float_rn(__dsqrt_rn(r));
        hdr->sumsq = r;
        hdr->norm = nrm;
        hdr->nparts = (uint32_t)total;
        hdr->status = 0u;          // plain loads: no tile is ever skipped here
        hdr->arrive = 0u;
        if (norm_out) *norm_out = nrm;
    }
}

template <int GDT, int WDT, int NT, bool FOLD, bool BCAST, bool SUMSQ>
static cudaError_t adamw_t(const Arena& a, const Avg& avg, const AdamArgs& h, bool store_avg,
                           void* grads, float* master, float* m, float* v, void* weights,
                           void* ws, cudaStream_t s, int64_t avg_stride)
{
    const unsigned blocks = blocks_for_segments(int64_t(a.N) * segments_per_chunk(a.C), 1);
    set_last_kernel_name(FOLD ? (SUMSQ ? "dpz_zero1_fused_sumsq" : "dpz_zero1_fused")
                              : (BCAST ? "dpz_adamw_bcast" : "dpz_adamw_owner"));
    return launch_kernel(k_adamw<GDT, WDT, NT, FOLD, BCAST, SUMSQ>, dim3(blocks), dim3(kBlock), 0, s,
                         true, 0u, static_cast<char*>(grads), master, m, v,
                         static_cast<char*>(weights), a.P, a.C, a.N, avg, h, store_avg ? 1 : 0,
                         static_cast<WsHeader*>(ws), SUMSQ ? ws_partials(ws) : nullptr,
                         avg_stride);
}

// The fold kernel for the arenas the staged kernel does not take (large N
// whose slab tiles cannot stay resident, zero1_fused_staged).
template <int GDT, int WDT, bool SUMSQ>
static cudaError_t fused_n(const Arena& a, const Avg& avg, const AdamArgs& h, bool store_avg,
                           void* grads, float* master, float* m, float* v, void* weights,
                           void* ws, cudaStream_t s)
{
    return adamw_t<GDT, WDT, 0, true, true, SUMSQ>(a, avg, h, store_avg, grads, master, m, v,
                                                  weights, ws, s, a.P);
}

template <int GDT, int WDT>
static cudaError_t adamw_dt(const Arena& a, const Avg& avg, const AdamArgs& h, AdamSrc src,
                            bool bcast, bool store_avg, void* grads, float* master, float* m,
                            float* v, void* weights, void* ws, cudaStream_t s,
                            int64_t avg_stride, float* norm_out)
{
    if (src == AdamSrc::kFold) {
        if (zero1_fused_staged(a))   // staged through shared memory by bulk copies (staged.cu)
            return launch_zero1_fused_tma(a, avg, h, store_avg, grads, master, m, v, weights, ws,
                                          s);
        if (ws != nullptr)
            return fused_n<GDT, WDT, true>(a, avg, h, store_avg, grads, master, m, v, weights, ws,
                                           s);
        return fused_n<GDT, WDT, false>(a, avg, h, store_avg, grads, master, m, v, weights, ws,
                                        s);
    }
    if (bcast)      // staged through shared memory by bulk copies (staged.cu)
        return launch_adamw_bcast_tma(a, h, grads, avg_stride, master, m, v, weights, ws,
                                      norm_out, s);
    return adamw_t<GDT, WDT, 0, false, false, false>(a, avg, h, false, grads, master, m, v,
                                                    weights, ws, s, avg_stride);
}

bool zero1_fits_small_step(const Arena& a)
{
    return int64_t(a.N) * segments_per_chunk(a.C) <= kSmallStepSegments;
}

template <int GDT, int WDT, int NT>
static cudaError_t small_t(const Arena& a, const Avg& avg, const AdamArgs& h, bool store_avg,
                           void* grads, float* master, float* m, float* v, void* weights,
                           void* ws, float* norm_out, cudaStream_t s)
{
    const int64_t total = int64_t(a.N) * segments_per_chunk(a.C);
    const unsigned teams = (unsigned)((total + kClusterCtas - 1) / kClusterCtas);   // per CTA
    const unsigned ctas = (unsigned)((total + teams - 1) / teams);                  // <= 8
    return launch_kernel(k_zero1_small<GDT, WDT, NT>, dim3(ctas), dim3(kTeam * teams), 0, s, true,
                         ctas, static_cast<char*>(grads), master, m, v,
                         static_cast<char*>(weights), a.P, a.C, a.N, avg, h, store_avg ? 1 : 0,
                         static_cast<WsHeader*>(ws), ws_partials(ws), norm_out);
}

template <int GDT, int WDT>
static cudaError_t small_n(const Arena& a, const Avg& avg, const AdamArgs& h, bool store_avg,
                           void* grads, float* master, float* m, float* v, void* weights,
                           void* ws, float* norm_out, cudaStream_t s)
{
    switch (a.N) {
    case 1: return small_t<GDT, WDT, 1>(a, avg, h, store_avg, grads, master, m, v, weights, ws, norm_out, s);
    case 2: return small_t<GDT, WDT, 2>(a, avg, h, store_avg, grads, master, m, v, weights, ws, norm_out, s);
    case 3: return small_t<GDT, WDT, 3>(a, avg, h, store_avg, grads, master, m, v, weights, ws, norm_out, s);
    case 4: return small_t<GDT, WDT, 4>(a, avg, h, store_avg, grads, master, m, v, weights, ws, norm_out, s);
    case 5: return small_t<GDT, WDT, 5>(a, avg, h, store_avg, grads, master, m, v, weights, ws, norm_out, s);
    case 6: return small_t<GDT, WDT, 6>(a, avg, h, store_avg, grads, master, m, v, weights, ws, norm_out, s);
    case 7: return small_t<GDT, WDT, 7>(a, avg, h, store_avg, grads, master, m, v, weights, ws, norm_out, s);
    case 8: return small_t<GDT, WDT, 8>(a, avg, h, store_avg, grads, master, m, v, weights, ws, norm_out, s);
    default: return small_t<GDT, WDT, 0>(a, avg, h, store_avg, grads, master, m, v, weights, ws, norm_out, s);
    }
}

cudaError_t launch_zero1_small(const Arena& a, const Avg& avg, const AdamArgs& h, bool store_avg,
                               void* grads, float* master, float* m, float* v, void* weights,
                               void* ws, float* norm_out, cudaStream_t s)
{
    set_last_kernel_name("dpz_zero1_small");
    const bool wb = a.wdt == 1;
    switch (a.gdt) {
    case 0:
        return wb ? small_n<0, 1>(a, avg, h, store_avg, grads, master, m, v, weights, ws, norm_out, s)
                  : small_n<0, 0>(a, avg, h, store_avg, grads, master, m, v, weights, ws, norm_out, s);
    case 1:
        return wb ? small_n<1, 1>(a, avg, h, store_avg, grads, master, m, v, weights, ws, norm_out, s)
                  : small_n<1, 0>(a, avg, h, store_avg, grads, master, m, v, weights, ws, norm_out, s);
    default:
        return wb ? small_n<2, 1>(a, avg, h, store_avg, grads, master, m, v, weights, ws, norm_out, s)
                  : small_n<2, 0>(a, avg, h, store_avg, grads, master, m, v, weights, ws, norm_out, s);
    }
}

cudaError_t launch_adamw(const Arena& a, const Avg& avg, const AdamArgs& h, AdamSrc src,
                         bool bcast, bool store_avg, void* grads, float* master, float* m,
                         float* v, void* weights, void* ws, cudaStream_t s, int64_t avg_stride,
                         float* norm_out)
{
    if (a.gdt == 2) {
        // fp32-accumulating bf16 ring: only the fold differs; stored averages
        // are plain bf16
        if (src == AdamSrc::kFold) {
            if (a.wdt == 1)
                return adamw_dt<2, 1>(a, avg, h, src, bcast, store_avg, grads, master, m, v,
                                      weights, ws, s, avg_stride, norm_out);
            return adamw_dt<2, 0>(a, avg, h, src, bcast, store_avg, grads, master, m, v,
                                  weights, ws, s, avg_stride, norm_out);
        }
        Arena b = a;
        b.gdt = 1;
        return launch_adamw(b, avg, h, src, bcast, store_avg, grads, master, m, v, weights, ws, s,
                            avg_stride, norm_out);
    }
    if (a.gdt == 1 && a.wdt == 1)
        return adamw_dt<1, 1>(a, avg, h, src, bcast, store_avg, grads, master, m, v,
                              weights, ws, s, avg_stride, norm_out);
    if (a.gdt == 1 && a.wdt == 0)
        return adamw_dt<1, 0>(a, avg, h, src, bcast, store_avg, grads, master, m, v,
                              weights, ws, s, avg_stride, norm_out);
    if (a.gdt == 0 && a.wdt == 1)
        return adamw_dt<0, 1>(a, avg, h, src, bcast, store_avg, grads, master, m, v,
                              weights, ws, s, avg_stride, norm_out);
    return adamw_dt<0, 0>(a, avg, h, src, bcast, store_avg, grads, master, m, v,
                          weights, ws, s, avg_stride, norm_out);
}

}  // namespace dpz
