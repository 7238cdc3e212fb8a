/*
 * CPU oracle for the data-parallel / ZeRO-1 step — TEST INFRASTRUCTURE ONLY.
 * See oracle.h for the contract and the pages each function follows.
 *
 * Build: gcc -std=c11 -O2 -ffp-contract=off -fno-fast-math -fPIC -shared
 * (no contraction into FMA, no fast-math, no flush-to-zero), so every float
 * operation below is one IEEE operation rounded to nearest even.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* storage types                                                        */
/* ------------------------------------------------------------------ */

static size_t elem_bytes(int dt)
{
    return dt == ORC_F64 ? 8u : dt == ORC_F32 ? 4u : 2u;
}

/* bytes of one element in a rank's working buffer and in a reduce-scatter
 * message: the fp32-accumulating bf16 ring works in fp32 */
static size_t work_bytes(int dt)
{
    return dt == ORC_BF16_ACC32 ? 4u : elem_bytes(dt);
}

static int valid_dtype(int dt)
{
    return dt == ORC_F32 || dt == ORC_BF16 || dt == ORC_F64 || dt == ORC_BF16_ACC32;
}

uint16_t orc_f32_to_bf16(float x)
{
    uint32_t b;
    memcpy(&b, &x, 4);
    if ((b & 0x7fffffffu) > 0x7f800000u)            /* NaN: keep it a NaN */
        return (uint16_t)((b >> 16) | 0x0040u);
    /* round to nearest, ties to even, on the 16 bits that are dropped */
    b += 0x7fffu + ((b >> 16) & 1u);
    return (uint16_t)(b >> 16);
}

float orc_bf16_to_f32(uint16_t h)
{
    uint32_t b = (uint32_t)h << 16;
    float x;
    memcpy(&x, &b, 4);
    return x;
}

void orc_f32_to_bf16_array(const float* x, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(x[i]);
}

/* local[i] = R(local[i] + msg[i]): the receiver adds the incoming partial sum
 * into its own chunk and stores the result in the storage type.  For bf16 the
 * two bf16 values are added in fp32 and the sum is rounded back to bf16 once
 * per hop (13.5 Multi-GPU from First Principles, Exercise 8). */
static void add_into(int dt, void* local, const void* msg, int64_t n)
{
    if (dt == ORC_F64) {
        double* a = (double*)local;
        const double* b = (const double*)msg;
        for (int64_t i = 0; i < n; ++i) a[i] = a[i] + b[i];
    } else if (dt == ORC_F32 || dt == ORC_BF16_ACC32) {
        float* a = (float*)local;
        const float* b = (const float*)msg;
        for (int64_t i = 0; i < n; ++i) a[i] = a[i] + b[i];
    } else {
        uint16_t* a = (uint16_t*)local;
        const uint16_t* b = (const uint16_t*)msg;
        for (int64_t i = 0; i < n; ++i) {
            float s = orc_bf16_to_f32(a[i]) + orc_bf16_to_f32(b[i]);
            a[i] = orc_f32_to_bf16(s);
        }
    }
}

static double load_as_double(int dt, const void* p, int64_t i)
{
    if (dt == ORC_F64) return ((const double*)p)[i];
    if (dt == ORC_F32 || dt == ORC_BF16_ACC32) return (double)((const float*)p)[i];
    return (double)orc_bf16_to_f32(((const uint16_t*)p)[i]);
}

static int64_t pmod(int64_t a, int64_t n)
{
    int64_t r = a % n;
    return r < 0 ? r + n : r;
}

/* ------------------------------------------------------------------ */
/* the ring: N separate rank buffers, messages built, then delivered    */
/* ------------------------------------------------------------------ */

typedef struct {
    int N;
    int64_t P, C;
    int dt;
    size_t es;              /* bytes per element in the working buffers */
    unsigned char** rank;   /* rank[r] = rank r's own full buffer */
    unsigned char** msg;    /* msg[r]  = the chunk rank r sends this step */
} ring_t;

static int ring_open(ring_t* R, const void* arena, int N, int64_t P, int dt)
{
    if (!arena || N < 1 || P < 1 || P % N != 0 || !valid_dtype(dt)) return -1;
    R->N = N;
    R->P = P;
    R->C = P / N;
    R->dt = dt;
    R->es = work_bytes(dt);
    R->rank = (unsigned char**)calloc((size_t)N, sizeof(void*));
    R->msg = (unsigned char**)calloc((size_t)N, sizeof(void*));
    if (!R->rank || !R->msg) return -1;
    for (int r = 0; r < N; ++r) {
        R->rank[r] = (unsigned char*)malloc((size_t)P * R->es);
        R->msg[r] = (unsigned char*)malloc((size_t)R->C * R->es);
        if (!R->rank[r] || !R->msg[r]) return -1;
        if (dt == ORC_BF16_ACC32) {
            const uint16_t* src = (const uint16_t*)arena + (size_t)r * P;
            float* dst = (float*)R->rank[r];
            for (int64_t i = 0; i < P; ++i) dst[i] = orc_bf16_to_f32(src[i]);
        } else {
            memcpy(R->rank[r], (const unsigned char*)arena + (size_t)r * P * R->es,
                   (size_t)P * R->es);
        }
    }
    return 0;
}

static void ring_close(ring_t* R, void* arena)
{
    for (int r = 0; r < R->N; ++r) {
        if (arena && R->rank[r] && R->dt == ORC_BF16_ACC32) {
            /* working fp32 values back to bf16 storage */
            uint16_t* dst = (uint16_t*)arena + (size_t)r * R->P;
            const float* src = (const float*)R->rank[r];
            for (int64_t i = 0; i < R->P; ++i) dst[i] = orc_f32_to_bf16(src[i]);
        } else if (arena && R->rank[r]) {
            memcpy((unsigned char*)arena + (size_t)r * R->P * R->es, R->rank[r],
                   (size_t)R->P * R->es);
        }
        free(R->rank[r]);
        free(R->msg[r]);
    }
    free(R->rank);
    free(R->msg);
}

static unsigned char* chunk_ptr(const ring_t* R, int r, int64_t c)
{
    return R->rank[r] + (size_t)c * R->C * R->es;
}

int orc_owner(int c, int N, int rho)
{
    /* the last receiver of chunk c: rank c - 1 + rho (mod N) */
    return (int)pmod((int64_t)c - 1 + rho, N);
}

static void rs_steps(ring_t* R, int rho, int steps, int64_t* sent)
{
    const int N = R->N;
    int64_t* ch = (int64_t*)malloc((size_t)N * sizeof(int64_t));
    const size_t bytes = (size_t)R->C * R->es;
    for (int t = 0; t < steps; ++t) {
        /* every rank builds its message first: all sends are simultaneous */
        for (int r = 0; r < N; ++r) {
            ch[r] = pmod((int64_t)r - t - rho, N);
            memcpy(R->msg[r], chunk_ptr(R, r, ch[r]), bytes);
            if (sent) sent[r] += (int64_t)bytes;
        }
        /* then every message is delivered to the right neighbour */
        for (int r = 0; r < N; ++r) {
            int dst = (r + 1) % N;
            add_into(R->dt, chunk_ptr(R, dst, ch[r]), R->msg[r], R->C);
        }
    }
    free(ch);
}

static void ag_steps(ring_t* R, int rho, int steps, int64_t* sent)
{
    const int N = R->N;
    int64_t* ch = (int64_t*)malloc((size_t)N * sizeof(int64_t));
    const size_t bytes = (size_t)R->C * R->es;
    /* what a message carries on the wire: the storage type (the averages of
     * the fp32-accumulating bf16 ring are bf16 values) */
    const size_t wire = (size_t)R->C * elem_bytes(R->dt);
    for (int t = 0; t < steps; ++t) {
        for (int r = 0; r < N; ++r) {
            ch[r] = pmod((int64_t)r + 1 - rho - t, N);
            memcpy(R->msg[r], chunk_ptr(R, r, ch[r]), bytes);
            if (sent) sent[r] += (int64_t)wire;
        }
        for (int r = 0; r < N; ++r) {
            int dst = (r + 1) % N;
            memcpy(chunk_ptr(R, dst, ch[r]), R->msg[r], bytes);   /* overwrite */
        }
    }
    free(ch);
}

static void average_owned_ring(ring_t* R, int rho)
{
    const int N = R->N;
    for (int c = 0; c < N; ++c) {
        unsigned char* p = chunk_ptr(R, orc_owner(c, N, rho), c);
        for (int64_t i = 0; i < R->C; ++i) {
            if (R->dt == ORC_F64) {
                double* a = (double*)p;
                a[i] = a[i] / (double)N;
            } else if (R->dt == ORC_F32) {
                float* a = (float*)p;
                a[i] = a[i] / (float)N;
            } else if (R->dt == ORC_BF16_ACC32) {
                float* a = (float*)p;
                a[i] = orc_bf16_to_f32(orc_f32_to_bf16(a[i] / (float)N));
            } else {
                uint16_t* a = (uint16_t*)p;
                a[i] = orc_f32_to_bf16(orc_bf16_to_f32(a[i]) / (float)N);
            }
        }
    }
}

int orc_ring_reduce_scatter(void* arena, int N, int64_t P, int dtype, int rho,
                            int steps, int64_t* sent)
{
    ring_t R;
    if (steps < 0 || steps > N - 1 || ring_open(&R, arena, N, P, dtype)) return -1;
    rs_steps(&R, rho, steps, sent);
    ring_close(&R, arena);
    return 0;
}

int orc_ring_allgather(void* arena, int N, int64_t P, int dtype, int rho,
                       int steps, int64_t* sent)
{
    ring_t R;
    if (steps < 0 || steps > N - 1 || ring_open(&R, arena, N, P, dtype)) return -1;
    ag_steps(&R, rho, steps, sent);
    ring_close(&R, arena);
    return 0;
}

int orc_average_owned(void* arena, int N, int64_t P, int dtype, int rho)
{
    ring_t R;
    if (ring_open(&R, arena, N, P, dtype)) return -1;
    average_owned_ring(&R, rho);
    ring_close(&R, arena);
    return 0;
}

int orc_reduce_scatter_avg(void* arena, int N, int64_t P, int dtype, int rho,
                           int64_t* sent)
{
    ring_t R;
    if (ring_open(&R, arena, N, P, dtype)) return -1;
    rs_steps(&R, rho, N - 1, sent);
    average_owned_ring(&R, rho);
    ring_close(&R, arena);
    return 0;
}

int orc_ring_allreduce_avg(void* arena, int N, int64_t P, int dtype, int rho,
                           int64_t* sent)
{
    ring_t R;
    if (ring_open(&R, arena, N, P, dtype)) return -1;
    rs_steps(&R, rho, N - 1, sent);
    average_owned_ring(&R, rho);
    ag_steps(&R, rho, N - 1, sent);
    ring_close(&R, arena);
    return 0;
}

int orc_star_allreduce(void* arena, int N, int64_t P, int dtype, int64_t* recv)
{
    ring_t R;
    if (ring_open(&R, arena, N, P, dtype)) return -1;
    const size_t bytes = (size_t)P * R.es;
    unsigned char* buf = (unsigned char*)malloc(bytes);
    /* gather: every other rank sends its whole buffer to rank 0, which sums */
    for (int r = 1; r < N; ++r) {
        memcpy(buf, R.rank[r], bytes);
        if (recv) recv[0] += (int64_t)bytes;
        add_into(dtype, R.rank[0], buf, P);
    }
    /* broadcast the sum back */
    for (int r = 1; r < N; ++r) {
        memcpy(R.rank[r], R.rank[0], bytes);
        if (recv) recv[r] += (int64_t)bytes;
    }
    free(buf);
    ring_close(&R, arena);
    return 0;
}

static double sumsq_ring(const ring_t* R, int rho)
{
    double ss = 0.0;
    for (int c = 0; c < R->N; ++c) {
        const unsigned char* p = chunk_ptr(R, orc_owner(c, R->N, rho), c);
        for (int64_t i = 0; i < R->C; ++i) {
            double g = load_as_double(R->dt, p, i);
            ss += g * g;
        }
    }
    return ss;
}

double orc_sumsq_owned(const void* arena, int N, int64_t P, int dtype, int rho)
{
    ring_t R;
    if (ring_open(&R, arena, N, P, dtype)) return NAN;
    double ss = sumsq_ring(&R, rho);
    ring_close(&R, NULL);
    return ss;
}

void orc_clip_scale(double sumsq, float clip, float* norm, float* scale)
{
    float n = (float)sqrt(sumsq);
    float s = 1.0f;
    if (clip > 0.0f && n > clip) s = clip / n;
    if (norm) *norm = n;
    if (scale) *scale = s;
}

/* ------------------------------------------------------------------ */
/* AdamW                                                                */
/* ------------------------------------------------------------------ */

void orc_bias_corrections(const orc_adamw_cfg* cfg, float* bc1, float* bc2)
{
    *bc1 = (float)(1.0 - pow((double)cfg->beta1, (double)cfg->step));
    *bc2 = (float)(1.0 - pow((double)cfg->beta2, (double)cfg->step));
}

void orc_adamw(float* theta, float* m, float* v, const void* grad, int gdtype,
               int64_t n, const orc_adamw_cfg* cfg, float scale)
{
    float bc1, bc2;
    orc_bias_corrections(cfg, &bc1, &bc2);
    const float b1 = cfg->beta1, b2 = cfg->beta2;
    const float omb1 = 1.0f - b1, omb2 = 1.0f - b2;
    const float lr = cfg->lr, eps = cfg->eps, wd = cfg->weight_decay;
    for (int64_t i = 0; i < n; ++i) {
        float g = (float)load_as_double(gdtype, grad, i);
        g = g * scale;
        float mi = b1 * m[i] + omb1 * g;
        float vi = b2 * v[i] + omb2 * (g * g);
        float mhat = mi / bc1;
        float vhat = vi / bc2;
        float upd = mhat / (sqrtf(vhat) + eps);
        float th = theta[i];
        theta[i] = th - lr * (upd + wd * th);
        m[i] = mi;
        v[i] = vi;
    }
}

static void cast_weights(const float* theta, void* w, int wdtype, int64_t n)
{
    if (wdtype == ORC_F32) {
        memcpy(w, theta, (size_t)n * 4u);
    } else {
        uint16_t* o = (uint16_t*)w;
        for (int64_t i = 0; i < n; ++i) o[i] = orc_f32_to_bf16(theta[i]);
    }
}

/* ------------------------------------------------------------------ */
/* the two steps                                                        */
/* ------------------------------------------------------------------ */

int orc_zero1_step(void* grads, float* master, float* m, float* v,
                   void* weights, int N, int64_t P, int gdtype, int wdtype,
                   const orc_adamw_cfg* cfg, double ext_sumsq,
                   float* norm_out, float* scale_out,
                   int64_t* sent_rs, int64_t* sent_ag)
{
    const int rho = 1;
    if (!master || !m || !v || !weights || !cfg || cfg->step < 1) return -1;
    if (gdtype == ORC_F64 || (wdtype != ORC_F32 && wdtype != ORC_BF16)) return -1;

    ring_t G;
    if (ring_open(&G, grads, N, P, gdtype)) return -1;
    const int64_t C = G.C;
    /* AdamW reads the averaged chunk from the working buffer: fp32 words for
     * the fp32-accumulating ring (bf16 values after the owner's rounding) */
    const int gwork = gdtype == ORC_BF16_ACC32 ? ORC_F32 : gdtype;

    /* 1. reduce-scatter, 2. the owner averages its chunk */
    rs_steps(&G, rho, N - 1, sent_rs);
    average_owned_ring(&G, rho);

    /* 3. global norm of the averaged gradient, clip scale */
    double ss = ext_sumsq >= 0.0 ? ext_sumsq : sumsq_ring(&G, rho);
    float norm, scale;
    orc_clip_scale(ss, cfg->clip_norm, &norm, &scale);
    if (cfg->clip_norm <= 0.0f) scale = 1.0f;

    /* 4. each rank r updates only its own shard r of master/m/v */
    ring_t W;
    if (ring_open(&W, weights, N, P, wdtype)) { ring_close(&G, NULL); return -1; }
    float* sh_t = (float*)malloc((size_t)C * 4u);
    float* sh_m = (float*)malloc((size_t)C * 4u);
    float* sh_v = (float*)malloc((size_t)C * 4u);
    for (int r = 0; r < N; ++r) {
        const int64_t off = (int64_t)r * C;             /* rank * shard_size */
        memcpy(sh_t, master + off, (size_t)C * 4u);
        memcpy(sh_m, m + off, (size_t)C * 4u);
        memcpy(sh_v, v + off, (size_t)C * 4u);
        orc_adamw(sh_t, sh_m, sh_v, chunk_ptr(&G, r, r), gwork, C, cfg, scale);
        cast_weights(sh_t, chunk_ptr(&W, r, r), wdtype, C);
        memcpy(master + off, sh_t, (size_t)C * 4u);
        memcpy(m + off, sh_m, (size_t)C * 4u);
        memcpy(v + off, sh_v, (size_t)C * 4u);
    }
    free(sh_t);
    free(sh_m);
    free(sh_v);

    /* 5. all-gather the updated weights */
    ag_steps(&W, rho, N - 1, sent_ag);

    ring_close(&W, weights);
    ring_close(&G, grads);
    if (norm_out) *norm_out = norm;
    if (scale_out) *scale_out = scale;
    return 0;
}

int orc_zero0_step(void* grads, float* master_full, float* m_full,
                   float* v_full, void* weights, int N, int64_t P, int gdtype,
                   int wdtype, const orc_adamw_cfg* cfg, float* norm_out,
                   int64_t* sent)
{
    const int rho = 1;
    if (!master_full || !m_full || !v_full || !weights || !cfg || cfg->step < 1)
        return -1;
    if (gdtype == ORC_F64 || (wdtype != ORC_F32 && wdtype != ORC_BF16)) return -1;

    ring_t G;
    if (ring_open(&G, grads, N, P, gdtype)) return -1;
    rs_steps(&G, rho, N - 1, sent);
    average_owned_ring(&G, rho);
    ag_steps(&G, rho, N - 1, sent);

    float norm0 = 0.0f;
    for (int r = 0; r < N; ++r) {
        /* every rank takes the norm of its own full averaged vector, chunk
         * by chunk in order 0..N-1 */
        double ss = 0.0;
        for (int c = 0; c < N; ++c) {
            const unsigned char* p = chunk_ptr(&G, r, c);
            for (int64_t i = 0; i < G.C; ++i) {
                double g = load_as_double(gdtype, p, i);
                ss += g * g;
            }
        }
        float norm, scale;
        orc_clip_scale(ss, cfg->clip_norm, &norm, &scale);
        if (cfg->clip_norm <= 0.0f) scale = 1.0f;
        if (r == 0) norm0 = norm;
        float* th = master_full + (size_t)r * P;
        float* mm = m_full + (size_t)r * P;
        float* vv = v_full + (size_t)r * P;
        orc_adamw(th, mm, vv, G.rank[r], gdtype == ORC_BF16_ACC32 ? ORC_F32 : gdtype, P, cfg,
                  scale);
        cast_weights(th, (unsigned char*)weights + (size_t)r * P * elem_bytes(wdtype),
                     wdtype, P);
    }
    ring_close(&G, grads);
    if (norm_out) *norm_out = norm0;
    return 0;
}
