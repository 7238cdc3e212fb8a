// The C-ABI of include/dpz.h: argument checks, status codes, the last-error
// message, launch accounting and optional per-launch event timing.  Every
// entry point validates all of its arguments before it launches anything.
#include "dpz.h"

#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"

using namespace dpz;

namespace {

thread_local std::string g_err;
std::atomic<int64_t> g_launches{0};

int fail(int code, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

int ok()
{
    g_err.clear();
    return DPZ_OK;
}

int elem_bytes(int dt) { return dt == DPZ_F32 ? 4 : 2; }

// ------------------------------------------------------------ validation

int check_dims(int64_t P, int N)
{
    if (N < 1 || N > DPZ_MAX_RANKS)
        return fail(DPZ_ERR_INVALID_ARG, "N = %d is outside 1..%d", N, DPZ_MAX_RANKS);
    if (P <= 0) return fail(DPZ_ERR_INVALID_ARG, "P = %lld must be positive", (long long)P);
    if (P > (int64_t(1) << 40))
        return fail(DPZ_ERR_INVALID_ARG, "P = %lld exceeds 2^40", (long long)P);
    if (P % N != 0)
        return fail(DPZ_ERR_INVALID_ARG,
                    "P = %lld is not divisible by N = %d: the arena cannot be sharded equally",
                    (long long)P, N);
    if ((P / N) % kGroup != 0)
        return fail(DPZ_ERR_ALIGN,
                    "chunk P/N = %lld is not a multiple of 8 elements (16-byte chunks); "
                    "pad P to a multiple of 8*N",
                    (long long)(P / N));
    return DPZ_OK;
}

// Gradients: DPZ_F32, DPZ_BF16 or DPZ_BF16_ACC32; weights: DPZ_F32 or DPZ_BF16.
int check_dtype(int dt, const char* what, bool gradient)
{
    if (dt != DPZ_F32 && dt != DPZ_BF16 && !(gradient && dt == DPZ_BF16_ACC32))
        return fail(DPZ_ERR_INVALID_ARG, "%s dtype %d is not supported", what, dt);
    return DPZ_OK;
}

// bf16 buffers must be 16-byte aligned, fp32 buffers 32-byte aligned (the
// kernels move 8 elements per lane in one 128- or 256-bit access).
int check_ptr(const void* p, const char* what, int dt = DPZ_BF16)
{
    if (p == nullptr) return fail(DPZ_ERR_INVALID_ARG, "%s is NULL", what);
    const uintptr_t align = dt == DPZ_F32 ? 32 : 16;
    if (reinterpret_cast<uintptr_t>(p) % align != 0)
        return fail(DPZ_ERR_ALIGN, "%s is not %d-byte aligned", what, (int)align);
    return DPZ_OK;
}

struct Range {
    const char* name;
    uintptr_t lo, hi;
};

Range range(const char* name, const void* p, int64_t bytes)
{
    uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return {name, lo, lo + static_cast<uintptr_t>(bytes)};
}

// The byte ranges of one call's buffers, held on the stack (no allocation on
// the launch path).  A NULL buffer is not added.  No call has more than seven
// buffers; one past kMax would be dropped, never written out of bounds.
struct Ranges {
    static constexpr int kMax = 8;
    Range r[kMax];
    int n = 0;
    Ranges(std::initializer_list<Range> rs)
    {
        for (const Range& x : rs)
            if (n < kMax) r[n++] = x;
    }
    void add(const char* name, const void* p, int64_t bytes)
    {
        if (p != nullptr && n < kMax) r[n++] = range(name, p, bytes);
    }
};

int check_disjoint(const Ranges& rs)
{
    for (int i = 0; i < rs.n; ++i)
        for (int j = i + 1; j < rs.n; ++j)
            if (rs.r[i].lo < rs.r[j].hi && rs.r[j].lo < rs.r[i].hi)
                return fail(DPZ_ERR_INVALID_ARG, "buffers %s and %s overlap", rs.r[i].name,
                            rs.r[j].name);
    return DPZ_OK;
}

int check_cfg(const dpz_adamw_cfg* cfg)
{
    if (cfg == nullptr) return fail(DPZ_ERR_INVALID_ARG, "cfg is NULL");
    if (cfg->step < 1)
        return fail(DPZ_ERR_INVALID_ARG, "step = %lld must be >= 1", (long long)cfg->step);
    return DPZ_OK;
}

#define DPZ_TRY(x)                     \
    do {                               \
        int rc_ = (x);                 \
        if (rc_ != DPZ_OK) return rc_; \
    } while (0)

Arena make_arena(int64_t P, int N, int gdt, int wdt)
{
    return Arena{P, P / N, N, gdt, wdt};
}

Avg make_avg(int N)
{
    Avg a;
    a.fN = static_cast<float>(N);
    a.pow2 = (N & (N - 1)) == 0;
    a.invN = 1.0f / static_cast<float>(N);
    return a;
}

AdamArgs make_adam(const dpz_adamw_cfg* cfg)
{
    AdamArgs h;
    h.lr = cfg->lr;
    h.b1 = cfg->beta1;
    h.b2 = cfg->beta2;
    h.omb1 = 1.0f - cfg->beta1;
    h.omb2 = 1.0f - cfg->beta2;
    h.bc1 = static_cast<float>(1.0 - std::pow(static_cast<double>(cfg->beta1),
                                              static_cast<double>(cfg->step)));
    h.bc2 = static_cast<float>(1.0 - std::pow(static_cast<double>(cfg->beta2),
                                              static_cast<double>(cfg->step)));
    h.eps = cfg->eps;
    h.wd = cfg->weight_decay;
    h.clip = cfg->clip_norm;
    return h;
}

// ------------------------------------------------------------ profiling

struct Profiler {
    std::mutex mu;
    std::atomic<bool> on{false};     // read without the lock on every launch
    int cap = 0;
    int used = 0;
    std::vector<cudaEvent_t> ev;
    std::vector<std::string> names;
};
Profiler g_prof;

template <class F>
int launch(cudaStream_t s, F&& f)
{
    int slot = -1;
    if (g_prof.on.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lk(g_prof.mu);
        if (g_prof.on.load(std::memory_order_relaxed) && g_prof.used < g_prof.cap)
            slot = g_prof.used++;
    }
    if (slot >= 0) cudaEventRecord(g_prof.ev[2 * slot], s);
    cudaError_t e = f();
    const char* name = last_kernel_name();
    if (slot >= 0) {
        cudaEventRecord(g_prof.ev[2 * slot + 1], s);
        std::lock_guard<std::mutex> lk(g_prof.mu);
        g_prof.names[slot] = name;
    }
    if (e != cudaSuccess)
        return fail(DPZ_ERR_CUDA, "launch of %s failed: %s", name, cudaGetErrorString(e));
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return DPZ_OK;
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

}  // namespace

// ====================================================================== ABI

extern "C" {

DPZ_API size_t dpz_workspace_bytes(int64_t P, int N)
{
    if (N < 1 || N > DPZ_MAX_RANKS || P <= 0 || P % N != 0) return 0;
    return ws_bytes_for(P, N);
}

DPZ_API const char* dpz_last_error(void) { return g_err.c_str(); }

DPZ_API const char* dpz_version(void) { return "dpz 0.2 (sm_103a)"; }

DPZ_API int64_t dpz_launch_count(void) { return g_launches.load(); }

DPZ_API int dpz_selftest_staged_timeout(int kernel, void* buf, void* stream)
{
    if (kernel != DPZ_SELFTEST_UPDATE && kernel != DPZ_SELFTEST_NORM &&
        kernel != DPZ_SELFTEST_STEP)
        return fail(DPZ_ERR_INVALID_ARG, "unknown self-test kernel %d", kernel);
    if (buf == nullptr) return fail(DPZ_ERR_INVALID_ARG, "buf is NULL");
    if (reinterpret_cast<uintptr_t>(buf) % 256 != 0)
        return fail(DPZ_ERR_ALIGN, "buf is not 256-byte aligned");
    cudaStream_t s = as_stream(stream);
    DPZ_TRY(launch(s, [&] { return launch_staged_timeout_selftest(kernel, buf, s); }));
    if (kernel != DPZ_SELFTEST_UPDATE) {
        // the finalisation turns the skipped tile's markers into the status
        float* nrm = reinterpret_cast<float*>(static_cast<char*>(buf) + kSelftestNormOut);
        DPZ_TRY(launch(s, [&] { return launch_norm_finalize(kSelftestArena, buf, nrm, s); }));
    }
    return ok();
}

DPZ_API int dpz_selftest_average_division(int N, unsigned long long* mismatches, void* stream)
{
    if (N < 1 || N > DPZ_MAX_RANKS)
        return fail(DPZ_ERR_INVALID_ARG, "N must be in [1, %d] (got %d)", DPZ_MAX_RANKS, N);
    DPZ_TRY(check_ptr(mismatches, "mismatches"));
    cudaStream_t s = as_stream(stream);
    const Avg avg = make_avg(N);
    DPZ_TRY(launch(s, [&] { return launch_selftest_division(avg, mismatches, s); }));
    return ok();
}

DPZ_API int dpz_device_status(int* flag_out)
{
    if (flag_out == nullptr) return fail(DPZ_ERR_INVALID_ARG, "flag_out is NULL");
    unsigned f = 0;
    const cudaError_t e = read_and_clear_pipeline_error(&f);
    if (e != cudaSuccess)
        return fail(DPZ_ERR_CUDA, "reading the device error flag failed: %s",
                    cudaGetErrorString(e));
    *flag_out = f != 0;
    return ok();
}

DPZ_API int dp_reduce_scatter_avg(void* grads, int64_t P, int N, int gdtype, void* stream)
{
    DPZ_TRY(check_dims(P, N));
    DPZ_TRY(check_dtype(gdtype, "gradient", true));
    DPZ_TRY(check_ptr(grads, "grads", gdtype));
    const Arena a = make_arena(P, N, gdtype, gdtype);
    const Avg avg = make_avg(N);
    DPZ_TRY(launch(as_stream(stream), [&] {
        return launch_reduce(a, avg, grads, false, nullptr, as_stream(stream));
    }));
    return ok();
}

DPZ_API int dp_allreduce_avg(void* grads, int64_t P, int N, int gdtype, void* stream)
{
    DPZ_TRY(check_dims(P, N));
    DPZ_TRY(check_dtype(gdtype, "gradient", true));
    DPZ_TRY(check_ptr(grads, "grads", gdtype));
    const Arena a = make_arena(P, N, gdtype, gdtype);
    const Avg avg = make_avg(N);
    DPZ_TRY(launch(as_stream(stream), [&] {
        return launch_reduce(a, avg, grads, true, nullptr, as_stream(stream));
    }));
    return ok();
}

DPZ_API int dp_grad_global_norm(const void* grads, int64_t P, int N, int gdtype, void* ws,
                                float* norm_out, void* stream)
{
    DPZ_TRY(check_dims(P, N));
    DPZ_TRY(check_dtype(gdtype, "gradient", true));
    DPZ_TRY(check_ptr(grads, "grads", gdtype));
    DPZ_TRY(check_ptr(ws, "ws"));
    Ranges rs = {range("grads", grads, int64_t(N) * P * elem_bytes(gdtype)),
                 range("ws", ws, (int64_t)dpz_workspace_bytes(P, N))};
    rs.add("norm_out", norm_out, 4);
    DPZ_TRY(check_disjoint(rs));
    const Arena a = make_arena(P, N, gdtype, gdtype);
    cudaStream_t s = as_stream(stream);
    DPZ_TRY(launch(s, [&] { return launch_norm_owned(a, grads, ws, s); }));
    DPZ_TRY(launch(s, [&] { return launch_norm_finalize(a, ws, norm_out, s); }));
    return ok();
}

static int check_step_buffers(const void* grads, const float* master, const float* m,
                              const float* v, const void* weights, int64_t P, int N, int gdtype,
                              int wdtype, const dpz_adamw_cfg* cfg, const void* ws, bool need_ws,
                              const float* norm_out)
{
    DPZ_TRY(check_dims(P, N));
    DPZ_TRY(check_dtype(gdtype, "gradient", true));
    DPZ_TRY(check_dtype(wdtype, "weight", false));
    DPZ_TRY(check_cfg(cfg));
    DPZ_TRY(check_ptr(grads, "grads", gdtype));
    DPZ_TRY(check_ptr(master, "master", DPZ_F32));
    DPZ_TRY(check_ptr(m, "m", DPZ_F32));
    DPZ_TRY(check_ptr(v, "v", DPZ_F32));
    DPZ_TRY(check_ptr(weights, "weights", wdtype));
    if (need_ws) DPZ_TRY(check_ptr(ws, "ws"));
    Ranges rs = {range("grads", grads, int64_t(N) * P * elem_bytes(gdtype)),
                 range("master", master, P * 4), range("m", m, P * 4), range("v", v, P * 4),
                 range("weights", weights, int64_t(N) * P * elem_bytes(wdtype))};
    rs.add("ws", ws, (int64_t)dpz_workspace_bytes(P, N));
    rs.add("norm_out", norm_out, 4);
    return check_disjoint(rs);
}

DPZ_API int zero1_adamw_step(const void* grads, float* master, float* m, float* v,
                             void* weights, int64_t P, int N, int gdtype, int wdtype,
                             const dpz_adamw_cfg* cfg, const void* ws, void* stream)
{
    const bool clip = cfg != nullptr && cfg->clip_norm > 0.0f;
    DPZ_TRY(check_step_buffers(grads, master, m, v, weights, P, N, gdtype, wdtype, cfg, ws, clip,
                               nullptr));
    const Arena a = make_arena(P, N, gdtype, wdtype);
    const Avg avg = make_avg(N);
    const AdamArgs h = make_adam(cfg);
    cudaStream_t s = as_stream(stream);
    DPZ_TRY(launch(s, [&] {
        return launch_adamw(a, avg, h, AdamSrc::kLoadOwner, false, false,
                            const_cast<void*>(grads), master, m, v, weights,
                            const_cast<void*>(ws), s, P);
    }));
    return ok();
}

DPZ_API int dp_allgather(void* weights, int64_t P, int N, int wdtype, void* stream)
{
    DPZ_TRY(check_dims(P, N));
    DPZ_TRY(check_dtype(wdtype, "weight", false));
    DPZ_TRY(check_ptr(weights, "weights", wdtype));
    const Arena a = make_arena(P, N, wdtype, wdtype);
    cudaStream_t s = as_stream(stream);
    DPZ_TRY(launch(s, [&] { return launch_allgather(a, weights, s); }));
    return ok();
}

DPZ_API int dp_zero1_step(void* grads, float* master, float* m, float* v, void* weights,
                          int64_t P, int N, int gdtype, int wdtype, const dpz_adamw_cfg* cfg,
                          void* ws, float* norm_out, void* stream)
{
    const bool clip = cfg != nullptr && cfg->clip_norm > 0.0f;
    DPZ_TRY(check_step_buffers(grads, master, m, v, weights, P, N, gdtype, wdtype, cfg, ws,
                               clip || norm_out != nullptr, norm_out));
    const Arena a = make_arena(P, N, gdtype, wdtype);
    const Avg avg = make_avg(N);
    const AdamArgs h = make_adam(cfg);
    cudaStream_t s = as_stream(stream);
    if (clip) {
        // reduce-scatter + average + norm partials, then the norm, then AdamW +
        // cast + all-gather reading the stored averages
        DPZ_TRY(launch(s, [&] { return launch_reduce(a, avg, grads, false, ws, s); }));
        DPZ_TRY(launch(s, [&] { return launch_norm_finalize(a, ws, norm_out, s); }));
        DPZ_TRY(launch(s, [&] {
            return launch_adamw(a, avg, h, AdamSrc::kLoadOwner, true, false, grads, master, m, v,
                                weights, ws, s, P, norm_out);
        }));
    } else if (norm_out && zero1_fits_small_step(a)) {
        // a small arena: the step and its norm in one launch (a thread-block cluster)
        DPZ_TRY(launch(s, [&] {
            return launch_zero1_small(a, avg, h, cfg->store_avg != 0, grads, master, m, v,
                                      weights, ws, norm_out, s);
        }));
    } else {
        void* sws = norm_out ? ws : nullptr;
        DPZ_TRY(launch(s, [&] {
            return launch_adamw(a, avg, h, AdamSrc::kFold, true, cfg->store_avg != 0, grads,
                                master, m, v, weights, sws, s, P);
        }));
        if (norm_out)
            DPZ_TRY(launch(s, [&] { return launch_norm_finalize(a, ws, norm_out, s); }));
    }
    return ok();
}

// ---------------------------------------------------------- buckets, ZeRO-2

static int check_range(int64_t P, int N, int64_t lo, int64_t n, bool segment_aligned)
{
    if (lo < 0 || n <= 0 || lo > P - n)
        return fail(DPZ_ERR_INVALID_ARG, "range [%lld, %lld) is not inside [0, %lld)",
                    (long long)lo, (long long)(lo + n), (long long)P);
    if (lo % kGroup != 0 || n % kGroup != 0)
        return fail(DPZ_ERR_ALIGN, "range start %lld and length %lld must be multiples of 8",
                    (long long)lo, (long long)n);
    const int64_t C = P / N;
    if (segment_aligned && (((lo % C) % kSegment) != 0 || (((lo + n) % C) % kSegment) != 0))
        return fail(DPZ_ERR_ALIGN,
                    "with norm partials the range [%lld, %lld) must start and end on "
                    "256-element segment boundaries of its chunks (chunk = %lld)",
                    (long long)lo, (long long)(lo + n), (long long)C);
    return DPZ_OK;
}

static int check_max_ctas(int max_ctas)
{
    if (max_ctas < 0) return fail(DPZ_ERR_INVALID_ARG, "max_ctas = %d is negative", max_ctas);
    return DPZ_OK;
}

DPZ_API int dp_reduce_scatter_avg_range(void* grads, int64_t P, int N, int gdtype, int64_t lo,
                                        int64_t n, void* ws, int max_ctas, void* stream)
{
    DPZ_TRY(check_dims(P, N));
    DPZ_TRY(check_max_ctas(max_ctas));
    DPZ_TRY(check_dtype(gdtype, "gradient", true));
    DPZ_TRY(check_ptr(grads, "grads", gdtype));
    DPZ_TRY(check_range(P, N, lo, n, ws != nullptr));
    if (ws) {
        DPZ_TRY(check_ptr(ws, "ws"));
        DPZ_TRY(check_disjoint({range("grads", grads, int64_t(N) * P * elem_bytes(gdtype)),
                                range("ws", ws, (int64_t)dpz_workspace_bytes(P, N))}));
    }
    const Arena a = make_arena(P, N, gdtype, gdtype);
    const Avg avg = make_avg(N);
    const int es = elem_bytes(gdtype);
    const RangeArgs g{static_cast<char*>(grads) + lo * es, P, grads, P, lo, lo + n, max_ctas};
    cudaStream_t s = as_stream(stream);
    DPZ_TRY(launch(s, [&] { return launch_reduce_range(a, avg, g, ws, s); }));
    return ok();
}

DPZ_API int dp_reduce_scatter_avg_bucket(const void* staging, int64_t lo, int64_t n, void* shards,
                                         int64_t P, int N, int gdtype, void* ws, int max_ctas,
                                         void* stream)
{
    DPZ_TRY(check_dims(P, N));
    DPZ_TRY(check_max_ctas(max_ctas));
    DPZ_TRY(check_dtype(gdtype, "gradient", true));
    DPZ_TRY(check_ptr(staging, "staging", gdtype));
    DPZ_TRY(check_ptr(shards, "shards", gdtype));
    DPZ_TRY(check_range(P, N, lo, n, ws != nullptr));
    const int es = elem_bytes(gdtype);
    Ranges rs = {range("staging", staging, int64_t(N) * n * es),
                 range("shards", shards, P * es)};
    if (ws) DPZ_TRY(check_ptr(ws, "ws"));
    rs.add("ws", ws, (int64_t)dpz_workspace_bytes(P, N));
    DPZ_TRY(check_disjoint(rs));
    const Arena a = make_arena(P, N, gdtype, gdtype);
    const Avg avg = make_avg(N);
    const RangeArgs g{staging, n, shards, 0, lo, lo + n, max_ctas};
    cudaStream_t s = as_stream(stream);
    DPZ_TRY(launch(s, [&] { return launch_reduce_range(a, avg, g, ws, s); }));
    return ok();
}

DPZ_API int dp_grad_norm_finalize(void* ws, int64_t P, int N, float* norm_out, void* stream)
{
    DPZ_TRY(check_dims(P, N));
    DPZ_TRY(check_ptr(ws, "ws"));
    if (norm_out)
        DPZ_TRY(check_disjoint({range("ws", ws, (int64_t)dpz_workspace_bytes(P, N)),
                                range("norm_out", norm_out, 4)}));
    const Arena a = make_arena(P, N, DPZ_BF16, DPZ_BF16);
    cudaStream_t s = as_stream(stream);
    DPZ_TRY(launch(s, [&] { return launch_norm_finalize(a, ws, norm_out, s); }));
    return ok();
}

static int update_common(const void* avg_src, int64_t avg_stride, int64_t avg_elems,
                         float* master, float* m, float* v, void* weights, int64_t P, int N,
                         int gdtype, int wdtype, const dpz_adamw_cfg* cfg, const void* ws,
                         void* stream, const char* what)
{
    DPZ_TRY(check_dims(P, N));
    DPZ_TRY(check_dtype(gdtype, "gradient", true));
    DPZ_TRY(check_dtype(wdtype, "weight", false));
    DPZ_TRY(check_cfg(cfg));
    DPZ_TRY(check_ptr(avg_src, what, gdtype));
    DPZ_TRY(check_ptr(master, "master", DPZ_F32));
    DPZ_TRY(check_ptr(m, "m", DPZ_F32));
    DPZ_TRY(check_ptr(v, "v", DPZ_F32));
    DPZ_TRY(check_ptr(weights, "weights", wdtype));
    const bool clip = cfg->clip_norm > 0.0f;
    if (clip) DPZ_TRY(check_ptr(ws, "ws"));
    Ranges rs = {range(what, avg_src, avg_elems * elem_bytes(gdtype)),
                 range("master", master, P * 4), range("m", m, P * 4), range("v", v, P * 4),
                 range("weights", weights, int64_t(N) * P * elem_bytes(wdtype))};
    rs.add("ws", ws, (int64_t)dpz_workspace_bytes(P, N));
    DPZ_TRY(check_disjoint(rs));
    const Arena a = make_arena(P, N, gdtype, wdtype);
    const Avg avg = make_avg(N);
    const AdamArgs h = make_adam(cfg);
    cudaStream_t s = as_stream(stream);
    DPZ_TRY(launch(s, [&] {
        return launch_adamw(a, avg, h, AdamSrc::kLoadOwner, true, false,
                            const_cast<void*>(avg_src), master, m, v, weights,
                            const_cast<void*>(ws), s, avg_stride);
    }));
    return ok();
}

DPZ_API int dp_zero1_update(const void* grads, float* master, float* m, float* v, void* weights,
                            int64_t P, int N, int gdtype, int wdtype, const dpz_adamw_cfg* cfg,
                            const void* ws, void* stream)
{
    return update_common(grads, P, int64_t(N) * P, master, m, v, weights, P, N, gdtype, wdtype,
                         cfg, ws, stream, "grads");
}

DPZ_API int dp_zero2_update(const void* shards, float* master, float* m, float* v, void* weights,
                            int64_t P, int N, int gdtype, int wdtype, const dpz_adamw_cfg* cfg,
                            const void* ws, void* stream)
{
    return update_common(shards, 0, P, master, m, v, weights, P, N, gdtype, wdtype, cfg, ws,
                         stream, "shards");
}

DPZ_API int dp_grad_global_norm_static(const void* grads, int64_t P, int N, int gdtype,
                                       float* norm_out, void* stream)
{
    DPZ_TRY(check_dims(P, N));
    DPZ_TRY(check_dtype(gdtype, "gradient", true));
    DPZ_TRY(check_ptr(grads, "grads", gdtype));
    if (norm_out == nullptr) return fail(DPZ_ERR_INVALID_ARG, "norm_out is NULL");
    const size_t need = ws_bytes_for(P, N);
    if (need > static_scratch_bytes())
        return fail(DPZ_ERR_INVALID_ARG,
                    "N = %d slabs of P = %lld elements need %zu bytes of norm scratch, more than "
                    "the %zu-byte static scratch; use dp_grad_global_norm with a workspace",
                    N, (long long)P, need, static_scratch_bytes());
    DPZ_TRY(check_disjoint({range("grads", grads, int64_t(N) * P * elem_bytes(gdtype)),
                            range("norm_out", norm_out, 4)}));
    cudaStream_t s = as_stream(stream);
    void* ws = nullptr;
    const cudaError_t e = static_scratch_address(&ws, s);
    if (e != cudaSuccess)
        return fail(DPZ_ERR_CUDA, "address of the static norm scratch: %s", cudaGetErrorString(e));
    const Arena a = make_arena(P, N, gdtype, gdtype);
    DPZ_TRY(launch(s, [&] { return launch_norm_owned(a, grads, ws, s); }));
    DPZ_TRY(launch(s, [&] { return launch_norm_finalize(a, ws, norm_out, s); }));
    return ok();
}

DPZ_API int dpz_profile_start(int max_launches)
{
    if (max_launches < 1 || max_launches > (1 << 20))
        return fail(DPZ_ERR_INVALID_ARG, "max_launches = %d is outside 1..2^20", max_launches);
    std::lock_guard<std::mutex> lk(g_prof.mu);
    for (cudaEvent_t e : g_prof.ev) cudaEventDestroy(e);
    g_prof.ev.assign(2 * static_cast<size_t>(max_launches), nullptr);
    g_prof.names.assign(static_cast<size_t>(max_launches), std::string());
    for (auto& e : g_prof.ev) {
        cudaError_t rc = cudaEventCreate(&e);
        if (rc != cudaSuccess) {
            g_prof.on = false;
            return fail(DPZ_ERR_CUDA, "cudaEventCreate failed: %s", cudaGetErrorString(rc));
        }
    }
    g_prof.cap = max_launches;
    g_prof.used = 0;
    g_prof.on = true;
    return ok();
}

DPZ_API int dpz_profile_stop(dpz_kernel_stat* stats, int max_stats, int* n_stats)
{
    std::lock_guard<std::mutex> lk(g_prof.mu);
    g_prof.on = false;
    std::vector<dpz_kernel_stat> out;
    for (int i = 0; i < g_prof.used; ++i) {
        cudaError_t rc = cudaEventSynchronize(g_prof.ev[2 * i + 1]);
        if (rc != cudaSuccess)
            return fail(DPZ_ERR_CUDA, "cudaEventSynchronize failed: %s", cudaGetErrorString(rc));
        float ms = 0.0f;
        rc = cudaEventElapsedTime(&ms, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]);
        if (rc != cudaSuccess)
            return fail(DPZ_ERR_CUDA, "cudaEventElapsedTime failed: %s", cudaGetErrorString(rc));
        const std::string& nm = g_prof.names[i];
        dpz_kernel_stat* hit = nullptr;
        for (auto& st : out)
            if (nm == st.name) hit = &st;
        if (!hit) {
            dpz_kernel_stat st{};
            std::snprintf(st.name, sizeof st.name, "%s", nm.c_str());
            out.push_back(st);
            hit = &out.back();
        }
        hit->launches += 1;
        hit->total_ms += ms;
    }
    const int n = static_cast<int>(out.size());
    if (n_stats) *n_stats = n;
    if (stats)
        for (int i = 0; i < n && i < max_stats; ++i) stats[i] = out[i];
    return ok();
}

}  // extern "C"
