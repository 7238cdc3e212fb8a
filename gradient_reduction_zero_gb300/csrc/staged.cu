// Kernels staged through shared memory by the Blackwell bulk-copy engine
// (TMA, 1-D cp.async.bulk; bulk.cuh), all three on one-shot, chunk-major grids:
//
// - AdamW + cast + all-gather of the new weights from the stored averages:
//   one 2048-element tile per 256-thread CTA.  Thread 0 issues the bulk loads
//   of the tile's averaged gradient and master/m/v, completing on one
//   mbarrier; every thread updates 8 elements in shared memory; thread 0 then
//   bulk-stores master/m/v and the cast weights into the N weight slabs and
//   waits until those stores have read shared memory.  The arithmetic is
//   adamw_elem, so the results are bit-identical to k_adamw.
// - The whole step without clip (ring fold of the N slabs, average, AdamW,
//   cast, N weight stores, optional averages store and norm partials): one
//   1024-element tile of every slab plus master/m/v per 128-thread CTA, the
//   same load / update / store shape.  N up to 8 is compiled in; larger N
//   fold at run time, on 1024- or 512-element tiles (64 threads), where
//   enough of their tiles stay resident per SM (zero1_fused_tile).
// - Sums of squares of the owner chunks (the standalone norm): one tile of
//   4,096 elements per 64-thread CTA, one bulk load, then each warp takes eight
//   segments of the tile at once.  Small tiles keep ~200 KB of loads in flight
//   per SM (25 resident CTAs) and turn over quickly.
//
// Every wait on an mbarrier is bounded by the SM clock: if a tile has not
// arrived after about two seconds the CTA sets the device error flag that
// dpz_device_status reads, reports the tile in the call's workspace (negative
// markers in the tile's norm partials, which the finalisation turns into a
// NaN norm and status bits; the update sets DPZ_STATUS_UPDATE_SKIPPED and a
// NaN norm_out), waits (again bounded) for its loads in flight, and returns
// without writing the tile.
#include <atomic>

#include "bulk.cuh"
#include "device.cuh"
#include "internal.h"

namespace dpz {

constexpr int kTmaTile = 1024;                     // elements per CTA of the step without clip
constexpr int kTmaThreads = kTmaTile / kGroup;     // 128: 8 elements each
// The AdamW + broadcast kernel's tile: 2048 elements per 256-thread CTA, five
// CTAs per SM.  Against 1024-element tiles (128 threads, ten per SM), same
// bits, the clipped steps measured 8-11 us faster at 1.5B and 3 us at 124M
// on two boxes; 512-element tiles were slower, and 4096-element tiles (two
// CTAs per SM) much slower.
constexpr int kUpdateTile = 2048;
constexpr int kUpdateThreads = kUpdateTile / kGroup;

__device__ unsigned g_pipeline_error;

// A tile whose loads did not arrive in time: raise the device flag and give
// the loads (bounded) time to land, since shared memory must outlive them.
__device__ __forceinline__ void abandon_tile(uint64_t* bar, long long limit)
{
    atomicExch(&g_pipeline_error, 1u);
    mbar_wait_bounded(bar, limit);
}

__device__ __forceinline__ float quiet_nan() { return __int_as_float(0x7fc00000); }

template <int GDT, int WDT>
struct TmaTile {
    unsigned char avg[kUpdateTile * Group<GDT>::kBytes];
    float th[kUpdateTile];
    float m[kUpdateTile];
    float v[kUpdateTile];
    unsigned char w[kUpdateTile * Group<WDT>::kBytes];
};

// grads: the averaged gradient of element e (chunk c) at grads + (c*avg_stride
// + e) elements; hdr: the workspace header (the norm, read when clip > 0; the
// status word, where a skipped tile is reported; may be NULL without clip);
// norm_out: set to NaN if this kernel gives up on a tile (may be NULL).
// NT > 0: N == NT known at compile time; NT == 0: any N, read from n_rt.
// Five CTAs per SM (at most 51 registers a thread).
template <int GDT, int WDT, int NT>
__global__ void __launch_bounds__(kUpdateThreads, 5)
k_adamw_bcast_tma(const char* __restrict__ grads, int64_t avg_stride, float* __restrict__ master,
                  float* __restrict__ mom, float* __restrict__ var, char* __restrict__ weights,
                  int64_t P, int64_t C, int n_rt, AdamArgs h, WsHeader* __restrict__ hdr,
                  float* __restrict__ norm_out, WaitSpec wait)
{
    using GS = Group<GDT>;
    using WS = Group<WDT>;
    constexpr int GES = GS::kBytes;
    constexpr int WES = WS::kBytes;
    const int N = NT > 0 ? NT : n_rt;
    extern __shared__ __align__(128) unsigned char dsmem[];
    TmaTile<GDT, WDT>& t = *reinterpret_cast<TmaTile<GDT, WDT>*>(dsmem);
    __shared__ __align__(8) uint64_t full;
    __shared__ int timed_out;

    // tile b of the chunk-major tile list: chunk c, first element e, n elements
    const int64_t tiles_per_chunk = (C + kUpdateTile - 1) / kUpdateTile;
    const int c = (int)(blockIdx.x / tiles_per_chunk);
    const int64_t tc = blockIdx.x - (int64_t)c * tiles_per_chunk;
    const int64_t e = (int64_t)c * C + tc * kUpdateTile;
    const int64_t left = C - tc * kUpdateTile;
    const int n = (int)(left < kUpdateTile ? left : kUpdateTile);   // a multiple of 8
    const int tid = threadIdx.x;

    pdl_enter();
    if (tid == 0) {
        mbar_init_one(&full);
        timed_out = 0;
        mbar_expect_tx(&full, (uint32_t)n * (GES + 12u) + wait.extra_tx);
        bulk_load(t.avg, grads + ((int64_t)c * avg_stride + e) * GES, (uint32_t)n * GES, &full);
        bulk_load(t.th, master + e, (uint32_t)n * 4u, &full);
        bulk_load(t.m, mom + e, (uint32_t)n * 4u, &full);
        bulk_load(t.v, var + e, (uint32_t)n * 4u, &full);
    }
    __syncthreads();     // the barrier is initialised before anyone waits on it

    float scale = 1.0f;
    bool do_scale = false, skip = false;
    if (h.clip > 0.0f) {
        // a norm whose input was not read in full is unknown: no update at all
        skip = (hdr->status & DPZ_STATUS_NORM_SKIPPED) != 0u;
        const float nrm = hdr->norm;
        if (nrm > h.clip) {
            scale = __fdiv_rn(h.clip, nrm);
            do_scale = true;
        }
    }

    if (!mbar_wait_bounded(&full, wait.limit)) atomicExch(&timed_out, 1);
    __syncthreads();
    if (timed_out || skip) {
        if (tid == 0) {
            if (timed_out) abandon_tile(&full, wait.limit);
            if (hdr != nullptr) atomicOr(&hdr->status, DPZ_STATUS_UPDATE_SKIPPED);
            if (timed_out && norm_out != nullptr) *norm_out = quiet_nan();
        }
        return;
    }

    const int i0 = tid * kGroup;
    if (i0 < n) {
        float g[8], th[8], mm[8], vv[8];
        GS::unpack(*reinterpret_cast<const typename GS::Raw*>(t.avg + i0 * GES), g);
        Group<0>::unpack(*reinterpret_cast<const U8*>(&t.th[i0]), th);
        Group<0>::unpack(*reinterpret_cast<const U8*>(&t.m[i0]), mm);
        Group<0>::unpack(*reinterpret_cast<const U8*>(&t.v[i0]), vv);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float gq = do_scale ? __fmul_rn(g[q], scale) : g[q];
            adamw_elem(th[q], mm[q], vv[q], gq, h);
        }
        *reinterpret_cast<U8*>(&t.th[i0]) = Group<0>::pack(th);
        *reinterpret_cast<U8*>(&t.m[i0]) = Group<0>::pack(mm);
        *reinterpret_cast<U8*>(&t.v[i0]) = Group<0>::pack(vv);
        *reinterpret_cast<typename WS::Raw*>(t.w + i0 * WES) = WS::pack(th);
    }
    // the threads' shared-memory writes become visible to the bulk stores
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (tid == 0) {
        bulk_store(master + e, t.th, (uint32_t)n * 4u);
        bulk_store(mom + e, t.m, (uint32_t)n * 4u);
        bulk_store(var + e, t.v, (uint32_t)n * 4u);
        if constexpr (NT > 0) {
#pragma unroll
            for (int r = 0; r < NT; ++r)
                bulk_store(weights + ((int64_t)r * P + e) * WES, t.w, (uint32_t)n * WES);
        } else {
            for (int r = 0; r < N; ++r)
                bulk_store(weights + ((int64_t)r * P + e) * WES, t.w, (uint32_t)n * WES);
        }
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        // shared memory is released when the CTA exits: wait until the stores
        // have read it (their writes to global memory complete on their own)
        asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    }
}

// ------------------------------------------------------------ fold step

// Shared memory of one fold tile of `tile` elements: the tiles of the nr
// slabs (slab r's at r * fold_slab_tile(GDT, tile)), then master, m and v
// (fp32), then the cast weights.
__host__ __device__ constexpr size_t fold_slab_tile(int GDT, int tile)
{
    return (size_t)tile * (GDT == 0 ? 4 : 2);
}
constexpr size_t fold_tile_bytes(int GDT, int WDT, int nr, int tile)
{
    return (size_t)nr * fold_slab_tile(GDT, tile) + (size_t)tile * (12 + (WDT == 0 ? 4 : 2));
}

// Largest fold tile the run-time-N kernel takes: two CTAs still fit an SM's
// 228 KB (1024-element tiles: bf16 gradients up to N = 47, fp32 up to
// N = 23; 512-element tiles: fp32 up to N = 51; one more with bf16 weights).
constexpr size_t kFoldTileMaxBytes = 110 * 1024;

// The step without clip: every lane folds its 8 elements over the slab tiles
// in ring order (for NT > 0 with fold_loaded, for NT == 0 over the n_rt tiles
// one at a time; both the same arithmetic as k_adamw), averages, adds its sum
// of squares to its warp's segment partial (a warp covers one 256-element
// segment of the tile), runs AdamW and casts.  With store_avg the averages
// replace slab c's tile and are stored into slab c.  TILE elements per CTA
// (1024 or 512), 8 per thread.
template <int GDT, int WDT, int NT, bool SUMSQ, int TILE>
__global__ void __launch_bounds__(TILE / kGroup)
k_zero1_fused_tma(char* __restrict__ grads, float* __restrict__ master, float* __restrict__ mom,
                  float* __restrict__ var, char* __restrict__ weights, int64_t P, int64_t C,
                  int n_rt, Avg avg, AdamArgs h, int store_avg, WsHeader* __restrict__ hdr,
                  double* __restrict__ partials, WaitSpec wait)
{
    using GS = Group<GDT>;
    using WS = Group<WDT>;
    constexpr int GES = GS::kBytes;
    constexpr int WES = WS::kBytes;
    constexpr size_t kSlabTile = fold_slab_tile(GDT, TILE);
    extern __shared__ __align__(128) unsigned char dsmem[];
    __shared__ __align__(8) uint64_t full;
    __shared__ int timed_out;

    const int nr = NT > 0 ? NT : n_rt;
    unsigned char* const tg = dsmem;
    float* const tth = reinterpret_cast<float*>(dsmem + (size_t)nr * kSlabTile);
    float* const tm = tth + TILE;
    float* const tv = tm + TILE;
    unsigned char* const tw = reinterpret_cast<unsigned char*>(tv + TILE);

    const int64_t tiles_per_chunk = (C + TILE - 1) / TILE;
    const int c = (int)(blockIdx.x / tiles_per_chunk);
    const int64_t tc = blockIdx.x - (int64_t)c * tiles_per_chunk;
    const int64_t e = (int64_t)c * C + tc * TILE;
    const int64_t left = C - tc * TILE;
    const int n = (int)(left < TILE ? left : TILE);   // a multiple of 8
    const int tid = threadIdx.x, lane = tid & 31;
    const int64_t gslab = P * GES;

    pdl_enter();
    if (SUMSQ && blockIdx.x == 0 && tid == 0) hdr->arrive = 0u;
    if (tid == 0) {
        mbar_init_one(&full);
        timed_out = 0;
        mbar_expect_tx(&full, (uint32_t)n * ((uint32_t)nr * GES + 12u) + wait.extra_tx);
#pragma unroll
        for (int r = 0; r < nr; ++r)
            bulk_load(tg + r * kSlabTile, grads + r * gslab + e * GES, (uint32_t)n * GES, &full);
        bulk_load(tth, master + e, (uint32_t)n * 4u, &full);
        bulk_load(tm, mom + e, (uint32_t)n * 4u, &full);
        bulk_load(tv, var + e, (uint32_t)n * 4u, &full);
    }
    __syncthreads();     // the barrier is initialised before anyone waits on it
    if (!mbar_wait_bounded(&full, wait.limit)) atomicExch(&timed_out, 1);
    __syncthreads();
    if (timed_out) {
        // the tile's partials say that neither its norm terms nor its update exist
        const int seg = tid >> 5;
        if (SUMSQ && lane == 0 && seg * kSegment < n)
            partials[c * segments_per_chunk(C) + tc * (TILE / kSegment) + seg] =
                kPartialStepSkipped;
        if (tid == 0) abandon_tile(&full, wait.limit);
        return;
    }

    const int i0 = tid * kGroup;
    float ss = 0.0f;
    if (i0 < n) {
        const unsigned char* const gi = tg + i0 * GES;   // this lane's group in slab 0's tile
        float g[8];
        if constexpr (NT > 0) {
            typename GS::Raw raw[NT];
#pragma unroll
            for (int j = 0; j < NT; ++j) {               // ring order: slabs c+1, ..., c
                int r = c + 1 + j;
                if (r >= NT) r -= NT;
                raw[j] = *reinterpret_cast<const typename GS::Raw*>(gi + r * kSlabTile);
            }
            fold_loaded<GDT, NT>(raw, g);
        } else {
            int r = c + 1;
            if (r >= nr) r -= nr;
            GS::unpack(*reinterpret_cast<const typename GS::Raw*>(gi + r * kSlabTile), g);
            for (int j = 2; j <= nr; ++j) {
                ++r;
                if (r >= nr) r -= nr;
                float x[8];
                GS::unpack(*reinterpret_cast<const typename GS::Raw*>(gi + r * kSlabTile), x);
#pragma unroll
                for (int q = 0; q < 8; ++q) g[q] = __fadd_rn(g[q], x[q]);
                GS::hop_round8(g);
            }
        }
        average8<GDT, NT>(g, avg);
        if (SUMSQ) ss = sumsq8(g);
        if (store_avg)
            *reinterpret_cast<typename GS::Raw*>(tg + c * kSlabTile + i0 * GES) = GS::pack(g);
        float th[8], mm[8], vv[8];
        Group<0>::unpack(*reinterpret_cast<const U8*>(&tth[i0]), th);
        Group<0>::unpack(*reinterpret_cast<const U8*>(&tm[i0]), mm);
        Group<0>::unpack(*reinterpret_cast<const U8*>(&tv[i0]), vv);
#pragma unroll
        for (int q = 0; q < 8; ++q) adamw_elem(th[q], mm[q], vv[q], g[q], h);
        *reinterpret_cast<U8*>(&tth[i0]) = Group<0>::pack(th);
        *reinterpret_cast<U8*>(&tm[i0]) = Group<0>::pack(mm);
        *reinterpret_cast<U8*>(&tv[i0]) = Group<0>::pack(vv);
        *reinterpret_cast<typename WS::Raw*>(tw + i0 * WES) = WS::pack(th);
    }
    if (SUMSQ) {
        const float tsum = warp_sum_f32(ss);                // whole warps
        const int seg = tid >> 5;
        if (lane == 0 && seg * kSegment < n)
            partials[c * segments_per_chunk(C) + tc * (TILE / kSegment) + seg] = (double)tsum;
    }
    // the threads' shared-memory writes become visible to the bulk stores
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (tid == 0) {
        bulk_store(master + e, tth, (uint32_t)n * 4u);
        bulk_store(mom + e, tm, (uint32_t)n * 4u);
        bulk_store(var + e, tv, (uint32_t)n * 4u);
        const int64_t wslab = P * WES;
#pragma unroll
        for (int r = 0; r < nr; ++r)
            bulk_store(weights + r * wslab + e * WES, tw, (uint32_t)n * WES);
        if (store_avg)
            bulk_store(grads + c * gslab + e * GES, tg + c * kSlabTile, (uint32_t)n * GES);
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        // shared memory is released when the CTA exits: wait until the stores
        // have read it (their writes to global memory complete on their own)
        asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    }
}

// ------------------------------------------------------------ norm

// Two warps per CTA, each taking eight consecutive 256-element segments of
// the CTA's tile: 4,096 elements (8 KB of bf16, 16 KB of fp32).
constexpr int kNormWarps = 2;
constexpr int kNormThreads = 32 * kNormWarps;
constexpr int kNormTile = 8 * kSegment * kNormWarps;

// Sums of squares of the owner chunks (chunk c of slab c), one per 256-element
// segment, from one kNormTile-element tile per CTA loaded by one bulk copy.
// The partial of a segment is the same fixed shuffle tree over the same
// values as in every other kernel that writes partials: a warp holds the
// terms of its eight segments at once and adds them with warp_sum8_f32, whose
// nine shuffles replace eight trees of five.  With the one tree per warp at a
// time the kernel read the 1.5B arena's owner chunks at 6.78 TB/s; with the
// eight trees interleaved 7.08, and with warp_sum8_f32 7.11 TB/s, against
// 7.47 for the same bulk copies with no arithmetic.  Tiles of 4 to 32 KB ran
// within 0.2 % of each other there; the small tiles were faster on small
// arenas (the GPT-2 124M one: 5.46, 5.95 and 5.97 TB/s for 32 KB tiles with
// one tree at a time, 32 KB and 8 KB tiles with warp_sum8_f32).
template <int GDT>
__global__ void __launch_bounds__(kNormThreads)
k_norm_owned_tma(const char* __restrict__ grads, int64_t P, int64_t C,
                 WsHeader* __restrict__ hdr, double* __restrict__ partials, WaitSpec wait)
{
    using G = Group<GDT>;
    constexpr int ES = G::kBytes;
    constexpr int T = kNormTile;
    extern __shared__ __align__(128) unsigned char dsmem[];
    __shared__ __align__(8) uint64_t full;
    __shared__ int timed_out;

    const int64_t tiles_per_chunk = (C + T - 1) / T;
    const int c = (int)(blockIdx.x / tiles_per_chunk);
    const int64_t tc = blockIdx.x - (int64_t)c * tiles_per_chunk;
    const int64_t e = (int64_t)c * C + tc * T;
    const int64_t left = C - tc * T;
    const int n = (int)(left < T ? left : T);           // a multiple of 8
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    double* const tile_parts = partials + c * segments_per_chunk(C) + tc * (T / kSegment);

    pdl_enter();
    if (blockIdx.x == 0 && tid == 0) hdr->arrive = 0u;
    if (tid == 0) {
        mbar_init_one(&full);
        timed_out = 0;
        mbar_expect_tx(&full, (uint32_t)n * ES + wait.extra_tx);
        bulk_load(dsmem, grads + ((int64_t)c * P + e) * ES, (uint32_t)n * ES, &full);
    }
    __syncthreads();
    if (!mbar_wait_bounded(&full, wait.limit)) atomicExch(&timed_out, 1);
    __syncthreads();
    // lane 4u of warp w writes the partial of the tile's segment 8w + u
    const int sg_out = warp * 8 + (lane >> 2);
    const bool writes = (lane & 3) == 0 && sg_out * kSegment < n;
    if (timed_out) {
        // the tile's partials say that its terms of the norm are missing
        if (writes) tile_parts[sg_out] = kPartialNormSkipped;
        if (tid == 0) abandon_tile(&full, wait.limit);
        return;
    }
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int i0 = (warp * 8 + u) * kSegment + lane * kGroup;
        v[u] = 0.0f;
        if (i0 < n) {
            float x[8];
            G::unpack(*reinterpret_cast<const typename G::Raw*>(dsmem + (int64_t)i0 * ES), x);
            v[u] = sumsq8(x);
        }
    }
    const float t = warp_sum8_f32(v);
    if (writes) tile_parts[sg_out] = (double)t;
}

namespace {

// Devices on which a kernel's dynamic shared memory limit has been raised,
// one bit per device (0..255): each launcher keeps one of these per kernel,
// so a launch after the first costs one atomic load.
struct SmemRaised {
    std::atomic<uint64_t> dev[4];
};

// Raise the kernel's dynamic shared memory limit on the current device, once.
cudaError_t allow_smem(SmemRaised& done, const void* fn, size_t smem)
{
    int d = 0;
    cudaError_t e = cudaGetDevice(&d);
    if (e != cudaSuccess) return e;
    const bool cached = d >= 0 && d < 256;
    const uint64_t bit = cached ? uint64_t(1) << (d & 63) : 0;
    if (cached && (done.dev[d >> 6].load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess && cached) done.dev[d >> 6].fetch_or(bit, std::memory_order_release);
    return e;
}

// The arguments of one launch of the AdamW + all-gather kernel.
struct UpdateLaunch {
    const void* grads;
    int64_t avg_stride;
    float* master;
    float* m;
    float* v;
    void* weights;
    void* ws;
    float* norm_out;
};

template <int GDT, int WDT, int NT>
cudaError_t tma_t(const Arena& a, const AdamArgs& h, const UpdateLaunch& u, cudaStream_t s)
{
    static SmemRaised raised;
    auto fn = k_adamw_bcast_tma<GDT, WDT, NT>;
    const size_t smem = sizeof(TmaTile<GDT, WDT>);
    const cudaError_t e = allow_smem(raised, reinterpret_cast<const void*>(fn), smem);
    if (e != cudaSuccess) return e;
    const int64_t tiles = (a.C + kUpdateTile - 1) / kUpdateTile * a.N;
    set_last_kernel_name("dpz_adamw_bcast");
    return launch_kernel(fn, dim3((unsigned)tiles), dim3(kUpdateThreads), smem, s, true, 0u,
                         static_cast<const char*>(u.grads), u.avg_stride, u.master, u.m, u.v,
                         static_cast<char*>(u.weights), a.P, a.C, a.N, h,
                         static_cast<WsHeader*>(u.ws), u.norm_out, kWaitNormal);
}

template <int GDT, int WDT>
cudaError_t tma_n(const Arena& a, const AdamArgs& h, const UpdateLaunch& u, cudaStream_t s)
{
    switch (a.N) {
    case 1: return tma_t<GDT, WDT, 1>(a, h, u, s);
    case 2: return tma_t<GDT, WDT, 2>(a, h, u, s);
    case 3: return tma_t<GDT, WDT, 3>(a, h, u, s);
    case 4: return tma_t<GDT, WDT, 4>(a, h, u, s);
    case 5: return tma_t<GDT, WDT, 5>(a, h, u, s);
    case 6: return tma_t<GDT, WDT, 6>(a, h, u, s);
    case 7: return tma_t<GDT, WDT, 7>(a, h, u, s);
    case 8: return tma_t<GDT, WDT, 8>(a, h, u, s);
    default: return tma_t<GDT, WDT, 0>(a, h, u, s);
    }
}

}  // namespace

cudaError_t launch_adamw_bcast_tma(const Arena& a, const AdamArgs& h, const void* grads,
                                   int64_t avg_stride, float* master, float* m, float* v,
                                   void* weights, void* ws, float* norm_out, cudaStream_t s)
{
    const UpdateLaunch u{grads, avg_stride, master, m, v, weights, ws, norm_out};
    const bool gbf = a.gdt != 0;       // stored averages: bf16 in both bf16 modes
    if (gbf && a.wdt == 1) return tma_n<1, 1>(a, h, u, s);
    if (gbf) return tma_n<1, 0>(a, h, u, s);
    if (a.wdt == 1) return tma_n<0, 1>(a, h, u, s);
    return tma_n<0, 0>(a, h, u, s);
}

// Shared memory of an SM (sm_103a), and what each resident CTA costs beyond
// its tile: the runtime's 1 KB reservation and the kernel's static barrier.
constexpr size_t kSmemPerSm = 228 * 1024;
constexpr size_t kCtaSmemOverhead = 1024 + 16;

// Staged tiles resident on one SM when the grid fills it.
static size_t fold_bytes_resident(size_t tile)
{
    return kSmemPerSm / (tile + kCtaSmemOverhead) * tile;
}

// The staged kernel keeps a stream going only with enough bytes in flight per
// SM.  Measured on the 1.5B-class arenas without clip: tiles resident at 184
// KB per SM and more ran at 7.08-7.18 TB/s, ahead of the fold kernel by 3-22
// %; at 156 KB (two 78 KB tiles, e.g. N = 32 bf16 or N = 16 fp32) the fold
// kernel was as fast or faster.  So for N > 8 the staged kernel is taken when
// the resident tiles reach 176 KB.
constexpr size_t kFoldMinResident = 176 * 1024;

// Elements per CTA of the staged step for this arena: 1024 for N <= 8, and
// for larger N the larger of 1024 and 512 whose tiles fit and stay resident
// at kFoldMinResident; 0 when neither does (the fold kernel then runs).
static int zero1_fused_tile(const Arena& a)
{
    if (a.N < 1) return 0;
    if (a.N <= 8) return kTmaTile;
    const int gdt = a.gdt == 0 ? 0 : 1;
    for (int tile = kTmaTile; tile >= kTmaTile / 2; tile /= 2) {
        const size_t bytes = fold_tile_bytes(gdt, a.wdt, a.N, tile);
        if (bytes <= kFoldTileMaxBytes && fold_bytes_resident(bytes) >= kFoldMinResident)
            return tile;
    }
    return 0;
}

bool zero1_fused_staged(const Arena& a)
{
    return zero1_fused_tile(a) != 0;
}

template <int GDT, int WDT, int NT, bool SUMSQ, int TILE = kTmaTile>
static cudaError_t fused_tma_t(const Arena& a, const Avg& avg, const AdamArgs& h, bool store_avg,
                               void* grads, float* master, float* m, float* v, void* weights,
                               void* ws, cudaStream_t s)
{
    static SmemRaised raised;
    auto fn = k_zero1_fused_tma<GDT, WDT, NT, SUMSQ, TILE>;
    const size_t smem = fold_tile_bytes(GDT, WDT, NT > 0 ? NT : a.N, TILE);
    // the run-time-N kernel may take any tile up to kFoldTileMaxBytes
    const cudaError_t e = allow_smem(raised, reinterpret_cast<const void*>(fn),
                                     NT > 0 ? smem : kFoldTileMaxBytes);
    if (e != cudaSuccess) return e;
    const int64_t tiles = (a.C + TILE - 1) / TILE * a.N;
    set_last_kernel_name(SUMSQ ? "dpz_zero1_fused_sumsq" : "dpz_zero1_fused");
    return launch_kernel(fn, dim3((unsigned)tiles), dim3(TILE / kGroup), smem, s, true, 0u,
                         static_cast<char*>(grads), master, m, v, static_cast<char*>(weights), a.P,
                         a.C, a.N, avg, h, store_avg ? 1 : 0, static_cast<WsHeader*>(ws),
                         SUMSQ ? ws_partials(ws) : nullptr, kWaitNormal);
}

template <int GDT, int WDT, bool SUMSQ>
static cudaError_t fused_tma_n(const Arena& a, const Avg& avg, const AdamArgs& h, bool store_avg,
                               void* grads, float* master, float* m, float* v, void* weights,
                               void* ws, cudaStream_t s)
{
    switch (a.N) {
    case 1:
        return fused_tma_t<GDT, WDT, 1, SUMSQ>(a, avg, h, store_avg, grads, master, m, v,
                                                weights, ws, s);
    case 2:
        return fused_tma_t<GDT, WDT, 2, SUMSQ>(a, avg, h, store_avg, grads, master, m, v,
                                                weights, ws, s);
    case 3:
        return fused_tma_t<GDT, WDT, 3, SUMSQ>(a, avg, h, store_avg, grads, master, m, v,
                                                weights, ws, s);
    case 4:
        return fused_tma_t<GDT, WDT, 4, SUMSQ>(a, avg, h, store_avg, grads, master, m, v,
                                                weights, ws, s);
    case 5:
        return fused_tma_t<GDT, WDT, 5, SUMSQ>(a, avg, h, store_avg, grads, master, m, v,
                                                weights, ws, s);
    case 6:
        return fused_tma_t<GDT, WDT, 6, SUMSQ>(a, avg, h, store_avg, grads, master, m, v,
                                                weights, ws, s);
    case 7:
        return fused_tma_t<GDT, WDT, 7, SUMSQ>(a, avg, h, store_avg, grads, master, m, v,
                                                weights, ws, s);
    case 8:
        return fused_tma_t<GDT, WDT, 8, SUMSQ>(a, avg, h, store_avg, grads, master, m, v,
                                                weights, ws, s);
    default:
        if (zero1_fused_tile(a) == kTmaTile)
            return fused_tma_t<GDT, WDT, 0, SUMSQ>(a, avg, h, store_avg, grads, master, m, v,
                                                    weights, ws, s);
        return fused_tma_t<GDT, WDT, 0, SUMSQ, kTmaTile / 2>(a, avg, h, store_avg, grads, master,
                                                              m, v, weights, ws, s);
    }
}

template <int GDT, int WDT>
static cudaError_t fused_tma_dt(const Arena& a, const Avg& avg, const AdamArgs& h, bool store_avg,
                                void* grads, float* master, float* m, float* v, void* weights,
                                void* ws, cudaStream_t s)
{
    if (ws != nullptr)
        return fused_tma_n<GDT, WDT, true>(a, avg, h, store_avg, grads, master, m, v, weights,
                                           ws, s);
    return fused_tma_n<GDT, WDT, false>(a, avg, h, store_avg, grads, master, m, v, weights, ws,
                                        s);
}

cudaError_t launch_zero1_fused_tma(const Arena& a, const Avg& avg, const AdamArgs& h,
                                   bool store_avg, void* grads, float* master, float* m, float* v,
                                   void* weights, void* ws, cudaStream_t s)
{
    if (!zero1_fused_staged(a)) return cudaErrorInvalidValue;
    const bool wb = a.wdt == 1;
    switch (a.gdt) {
    case 0:
        return wb ? fused_tma_dt<0, 1>(a, avg, h, store_avg, grads, master, m, v, weights, ws, s)
                  : fused_tma_dt<0, 0>(a, avg, h, store_avg, grads, master, m, v, weights, ws, s);
    case 1:
        return wb ? fused_tma_dt<1, 1>(a, avg, h, store_avg, grads, master, m, v, weights, ws, s)
                  : fused_tma_dt<1, 0>(a, avg, h, store_avg, grads, master, m, v, weights, ws, s);
    default:
        return wb ? fused_tma_dt<2, 1>(a, avg, h, store_avg, grads, master, m, v, weights, ws, s)
                  : fused_tma_dt<2, 0>(a, avg, h, store_avg, grads, master, m, v, weights, ws, s);
    }
}

template <int GDT>
static cudaError_t norm_t(const Arena& a, const void* grads, void* ws, cudaStream_t s)
{
    auto fn = k_norm_owned_tma<GDT>;
    constexpr size_t smem = (size_t)kNormTile * Group<GDT>::kBytes;   // at most 48 KB
    const int64_t tiles = (a.C + kNormTile - 1) / kNormTile * a.N;
    return launch_kernel(fn, dim3((unsigned)tiles), dim3(kNormThreads), smem, s, true, 0u,
                         static_cast<const char*>(grads), a.P, a.C, static_cast<WsHeader*>(ws),
                         ws_partials(ws), kWaitNormal);
}

cudaError_t launch_norm_owned(const Arena& a, const void* grads, void* ws, cudaStream_t s)
{
    set_last_kernel_name("dpz_norm_owned");
    // both bf16 modes store bf16 averages
    return a.gdt != 0 ? norm_t<1>(a, grads, ws, s) : norm_t<0>(a, grads, ws, s);
}

// The self-test of the timeout path: one staged kernel on a one-tile arena
// (N = 1, P = 8, bf16 gradients and weights, fp32 state) laid out in the
// caller's buffer as dpz.h describes, with a barrier that expects 16 bytes
// more than the kernel's loads deliver and a wait bound of
// kSelftestWaitCycles.  Every copy it issues completes, so nothing is in
// flight when the CTA gives up; the bounded wait runs out (and then the
// bounded wait of the abandon path), the device flag is set, the tile is
// reported in the workspace, and the kernel returns without writing the
// arena.  The caller follows the norm and the step kernels with the
// finalisation, which turns their markers into status bits and a NaN norm.
constexpr long long kSelftestWaitCycles = 100000000LL;

cudaError_t launch_staged_timeout_selftest(int kernel, void* buf, cudaStream_t s)
{
    char* b = static_cast<char*>(buf);
    void* ws = b;
    WsHeader* hdr = static_cast<WsHeader*>(ws);
    float* norm_out = reinterpret_cast<float*>(b + kSelftestNormOut);
    char* grads = b + kSelftestGrads;
    float* master = reinterpret_cast<float*>(b + kSelftestGrads + 32);
    float* m = reinterpret_cast<float*>(b + kSelftestGrads + 64);
    float* v = reinterpret_cast<float*>(b + kSelftestGrads + 96);
    char* weights = b + kSelftestGrads + 128;
    const Arena a = kSelftestArena;
    const WaitSpec wait{kSelftestWaitCycles, 16u};
    AdamArgs h{};
    h.lr = 1e-3f;
    h.b1 = 0.9f;
    h.b2 = 0.999f;
    h.omb1 = 0.1f;
    h.omb2 = 0.001f;
    h.bc1 = 0.1f;
    h.bc2 = 0.001f;
    h.eps = 1e-8f;
    static_assert(kSelftestGrads + 144 <= DPZ_SELFTEST_BUF_BYTES, "the arena fits the buffer");
    cudaError_t e = cudaSuccess;
    if (kernel == DPZ_SELFTEST_UPDATE) {
        static SmemRaised raised;
        auto fn = k_adamw_bcast_tma<1, 1, 1>;
        const size_t smem = sizeof(TmaTile<1, 1>);
        e = allow_smem(raised, reinterpret_cast<const void*>(fn), smem);
        if (e != cudaSuccess) return e;
        set_last_kernel_name("dpz_selftest_staged_timeout");
        fn<<<1, kUpdateThreads, smem, s>>>(grads, a.P, master, m, v, weights, a.P, a.C, 1, h, hdr,
                                       norm_out, wait);
        return cudaGetLastError();
    }
    if (kernel == DPZ_SELFTEST_NORM) {
        auto fn = k_norm_owned_tma<1>;
        fn<<<1, kNormThreads, (size_t)kNormTile * 2, s>>>(grads, a.P, a.C, hdr, ws_partials(ws),
                                                         wait);
    } else if (kernel == DPZ_SELFTEST_STEP) {
        static SmemRaised raised;
        auto fn = k_zero1_fused_tma<1, 1, 1, true, kTmaTile>;
        const size_t smem = fold_tile_bytes(1, 1, 1, kTmaTile);
        e = allow_smem(raised, reinterpret_cast<const void*>(fn), smem);
        if (e != cudaSuccess) return e;
        Avg avg;
        avg.fN = 1.0f;
        avg.invN = 1.0f;
        avg.pow2 = 1;
        fn<<<1, kTmaThreads, smem, s>>>(grads, master, m, v, weights, a.P, a.C, 1, avg, h, 0, hdr,
                                       ws_partials(ws), wait);
    } else {
        return cudaErrorInvalidValue;
    }
    set_last_kernel_name("dpz_selftest_staged_timeout");
    return cudaGetLastError();
}

cudaError_t read_and_clear_pipeline_error(unsigned* flag)
{
    cudaError_t e = cudaMemcpyFromSymbol(flag, g_pipeline_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_pipeline_error, &zero, sizeof(unsigned));
}

}  // namespace dpz
