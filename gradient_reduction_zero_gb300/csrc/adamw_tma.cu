// AdamW + cast + all-gather of the new weights, staged through shared memory
// by the Blackwell bulk-copy engine (TMA, 1-D cp.async.bulk).
//
// Persistent CTAs (as many as are resident), each with a 4-stage pipeline of
// 1024-element tiles.  Thread 0 issues the bulk loads of a tile (the averaged
// gradient and master/m/v) into a stage, completing on that stage's mbarrier;
// all threads update the tile in shared memory; thread 0 then bulk-stores
// master/m/v and the cast weights into every rank's slab, and refills the
// stage of the previous tile once its stores have read shared memory.  The
// arithmetic is adamw_elem, so the results are bit-identical to k_adamw.
//
// Waits on an mbarrier are bounded by the SM clock: if a tile has not
// arrived after ~2 s the CTA sets a device error flag (dpz_device_status),
// waits again (bounded) for its copies in flight, and returns.
#include <map>
#include <mutex>
#include <utility>

#include "device.cuh"
#include "internal.h"

namespace dpz {

constexpr int kTmaTile = 1024;
constexpr int kTmaStages = 4;
constexpr int kTmaThreads = 256;
constexpr long long kWaitLimitCycles = 4000000000LL;

__device__ unsigned g_pipeline_error;

template <int GDT, int WDT>
struct TmaStage {
    unsigned char avg[kTmaTile * Group<GDT>::kBytes];
    float th[kTmaTile];
    float m[kTmaTile];
    float v[kTmaTile];
    unsigned char w[kTmaTile * Group<WDT>::kBytes];
};

namespace {

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// global -> shared, completing `bytes` on the mbarrier
__device__ __forceinline__ void bulk_load(void* sdst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(sdst)),
        "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// shared -> global, in the current bulk group
__device__ __forceinline__ void bulk_store(void* gdst, const void* ssrc, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
                 "r"(smem_addr(ssrc)), "r"(bytes)
                 : "memory");
}

}  // namespace

// grads: the averaged gradient of element e (chunk c) at grads + (c*avg_stride + e)
// elements; hdr: the workspace header (the norm), NULL when clip <= 0.
template <int GDT, int WDT>
__global__ void __launch_bounds__(kTmaThreads, 3)
k_adamw_bcast_tma(const char* __restrict__ grads, int64_t avg_stride, float* __restrict__ master,
                  float* __restrict__ mom, float* __restrict__ var, char* __restrict__ weights,
                  int64_t P, int64_t C, int N, AdamArgs h, const WsHeader* __restrict__ hdr)
{
    using GS = Group<GDT>;
    using WS = Group<WDT>;
    using Stage = TmaStage<GDT, WDT>;
    constexpr int GES = GS::kBytes;
    constexpr int WES = WS::kBytes;
    extern __shared__ __align__(128) unsigned char dsmem[];
    Stage* st = reinterpret_cast<Stage*>(dsmem);
    __shared__ __align__(8) uint64_t full[kTmaStages];
    __shared__ int abort_flag;

    const int tid = threadIdx.x;
    const int64_t tiles_per_chunk = (C + kTmaTile - 1) / kTmaTile;
    const int64_t ntiles = tiles_per_chunk * N;
    const int64_t mine =
        (int64_t)blockIdx.x < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    float scale = 1.0f;
    bool do_scale = false;
    if (h.clip > 0.0f) {
        const float nrm = hdr->norm;
        if (nrm > h.clip) {
            scale = __fdiv_rn(h.clip, nrm);
            do_scale = true;
        }
    }

    if (tid == 0) {
        for (int s = 0; s < kTmaStages; ++s) mbar_init(&full[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        abort_flag = 0;
    }
    __syncthreads();

    // tile k of this CTA: chunk c, first element e, n elements
    auto tile = [&](int64_t k, int& c, int64_t& e, int& n) {
        const int64_t g = (int64_t)blockIdx.x + k * gridDim.x;
        c = (int)(g / tiles_per_chunk);
        const int64_t t = g - (int64_t)c * tiles_per_chunk;
        e = (int64_t)c * C + t * kTmaTile;
        const int64_t left = C - t * kTmaTile;
        n = (int)(left < kTmaTile ? left : kTmaTile);
    };
    int64_t issued = 0;   // tiles whose loads thread 0 has issued, in order
    auto issue_load = [&](int64_t k) {
        int c;
        int64_t e;
        int n;
        tile(k, c, e, n);
        Stage& sg = st[k % kTmaStages];
        uint64_t* bar = &full[k % kTmaStages];
        mbar_expect_tx(bar, (uint32_t)n * (GES + 12u));
        bulk_load(sg.avg, grads + ((int64_t)c * avg_stride + e) * GES, (uint32_t)n * GES, bar);
        bulk_load(sg.th, master + e, (uint32_t)n * 4u, bar);
        bulk_load(sg.m, mom + e, (uint32_t)n * 4u, bar);
        bulk_load(sg.v, var + e, (uint32_t)n * 4u, bar);
        issued = k + 1;
    };

    if (tid == 0)
        for (int64_t k = 0; k < kTmaStages && k < mine; ++k) issue_load(k);

    int64_t k = 0;
    for (; k < mine; ++k) {
        const int s = (int)(k % kTmaStages);
        const uint32_t parity = (uint32_t)((k / kTmaStages) & 1);
        if (!mbar_try_wait(&full[s], parity)) {
            const long long t0 = clock64();
            while (!mbar_try_wait(&full[s], parity)) {
                if (clock64() - t0 > kWaitLimitCycles) {
                    atomicExch(&abort_flag, 1);
                    break;
                }
            }
        }
        __syncthreads();
        if (abort_flag) break;

        int c;
        int64_t e;
        int n;
        tile(k, c, e, n);
        Stage& sg = st[s];
        for (int i0 = tid * kGroup; i0 < n; i0 += kTmaThreads * kGroup) {
            float g[8], th[8], mm[8], vv[8];
            GS::unpack(*reinterpret_cast<const typename GS::Raw*>(sg.avg + i0 * GES), g);
            Group<0>::unpack(*reinterpret_cast<const U8*>(&sg.th[i0]), th);
            Group<0>::unpack(*reinterpret_cast<const U8*>(&sg.m[i0]), mm);
            Group<0>::unpack(*reinterpret_cast<const U8*>(&sg.v[i0]), vv);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float gq = do_scale ? __fmul_rn(g[q], scale) : g[q];
                adamw_elem(th[q], mm[q], vv[q], gq, h);
            }
            *reinterpret_cast<U8*>(&sg.th[i0]) = Group<0>::pack(th);
            *reinterpret_cast<U8*>(&sg.m[i0]) = Group<0>::pack(mm);
            *reinterpret_cast<U8*>(&sg.v[i0]) = Group<0>::pack(vv);
            *reinterpret_cast<typename WS::Raw*>(sg.w + i0 * WES) = WS::pack(th);
        }
        // the threads' shared-memory writes become visible to the bulk stores
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (tid == 0) {
            bulk_store(master + e, sg.th, (uint32_t)n * 4u);
            bulk_store(mom + e, sg.m, (uint32_t)n * 4u);
            bulk_store(var + e, sg.v, (uint32_t)n * 4u);
            for (int r = 0; r < N; ++r)
                bulk_store(weights + ((int64_t)r * P + e) * WES, sg.w, (uint32_t)n * WES);
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            // refill the previous tile's stage once its stores have read it
            if (k >= 1 && k - 1 + kTmaStages < mine) {
                asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
                issue_load(k - 1 + kTmaStages);
            }
        }
    }
    if (tid == 0) {
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        if (abort_flag) {
            atomicExch(&g_pipeline_error, 1u);
            // tiles k .. issued-1 may still have loads in flight: wait for
            // each stage's phase, under one overall limit
            const long long t0 = clock64();
            for (int64_t j = k; j < issued; ++j) {
                const uint32_t par = (uint32_t)((j / kTmaStages) & 1);
                while (!mbar_try_wait(&full[j % kTmaStages], par))
                    if (clock64() - t0 > kWaitLimitCycles) break;
            }
        }
    }
}

namespace {

std::mutex g_tma_mu;
std::map<std::pair<int, const void*>, int> g_tma_resident;   // (device, kernel) -> CTAs per SM

// Resident CTAs per SM of `fn` with `smem` bytes of dynamic shared memory on
// the current device, after raising the kernel's dynamic shared memory limit
// there (once per device).
cudaError_t tma_residency(const void* fn, size_t smem, int* resident)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_tma_mu);
    auto it = g_tma_resident.find({dev, fn});
    if (it != g_tma_resident.end()) {
        *resident = it->second;
        return cudaSuccess;
    }
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int nb = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, kTmaThreads, smem);
    if (e != cudaSuccess) return e;
    if (nb < 1) nb = 1;
    g_tma_resident[{dev, fn}] = nb;
    *resident = nb;
    return cudaSuccess;
}

template <int GDT, int WDT>
cudaError_t tma_t(const Arena& a, const AdamArgs& h, const void* grads, int64_t avg_stride,
                  float* master, float* m, float* v, void* weights, const void* ws,
                  cudaStream_t s)
{
    auto fn = k_adamw_bcast_tma<GDT, WDT>;
    const size_t smem = sizeof(TmaStage<GDT, WDT>) * kTmaStages;
    int resident = 1;
    const cudaError_t e = tma_residency(reinterpret_cast<const void*>(fn), smem, &resident);
    if (e != cudaSuccess) return e;
    const int64_t tiles = (a.C + kTmaTile - 1) / kTmaTile * a.N;
    // persistent: one wave of resident CTAs, each walking its tiles in turn
    int64_t grid = (int64_t)device_sms() * resident;
    if (grid > tiles) grid = tiles;
    if (grid < 1) grid = 1;
    set_last_kernel_name("dpz_adamw_bcast");
    fn<<<(unsigned)grid, kTmaThreads, smem, s>>>(static_cast<const char*>(grads), avg_stride, master,
                                                 m, v, static_cast<char*>(weights), a.P, a.C, a.N,
                                                 h, static_cast<const WsHeader*>(ws));
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_adamw_bcast_tma(const Arena& a, const AdamArgs& h, const void* grads,
                                   int64_t avg_stride, float* master, float* m, float* v,
                                   void* weights, const void* ws, cudaStream_t s)
{
    const int gdt = a.gdt == 0 ? 0 : 1;      // stored averages: fp32 or bf16
    if (gdt == 1 && a.wdt == 1) return tma_t<1, 1>(a, h, grads, avg_stride, master, m, v, weights, ws, s);
    if (gdt == 1 && a.wdt == 0) return tma_t<1, 0>(a, h, grads, avg_stride, master, m, v, weights, ws, s);
    if (gdt == 0 && a.wdt == 1) return tma_t<0, 1>(a, h, grads, avg_stride, master, m, v, weights, ws, s);
    return tma_t<0, 0>(a, h, grads, avg_stride, master, m, v, weights, ws, s);
}

cudaError_t read_and_clear_pipeline_error(unsigned* flag)
{
    cudaError_t e = cudaMemcpyFromSymbol(flag, g_pipeline_error, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_pipeline_error, &zero, sizeof(unsigned));
}

}  // namespace dpz
