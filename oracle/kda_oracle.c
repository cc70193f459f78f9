/*
 * Plain fp64 CPU oracle for the Kimi Delta Attention (KDA) serving hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link,
 * load or call this file: only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * What it computes, and where each definition comes from:
 *
 *   oracle_gather   "vllm-ascend KDA state copy" page, section "Numeric
 *                   contract / Gather side": packed row s is cache row idx[s]
 *                   when 0 <= idx[s] < N and the row's flag is true (or no
 *                   flags are given); otherwise it is all zeros.  Duplicate
 *                   indices are legal.  Gap elements between stride(0) and
 *                   the payload are never read.
 *   oracle_scatter  same page, "Numeric contract / Scatter side" and "Memory
 *                   and addressing": every packed row whose index is valid is
 *                   converted to the cache dtype and written over the
 *                   payload of that row; invalid indices are skipped, flags
 *                   play no part, gap elements are never written.
 *   oracle_prefill  the recurrence of the "KDA's challenges for AI infra"
 *                   page, section 1.1 (S_t = M_t S_{t-1} + b_t), with
 *                   M_t = (I - beta_t k_t k_t^T) Diag(exp g_t),
 *                   b_t = beta_t k_t v_t^T and o_t = scale * S_t^T q_t, run
 *                   token by token per (sequence, head) over a cu_seqlens
 *                   varlen batch.  q and k are L2-normalised per (token,
 *                   head) first, as the "Support Kimi-K3 on NPU" report's
 *                   extend listing does before its chunk math.
 *   oracle_prefill_ckpt  oracle_prefill plus the state after every `every`
 *                   tokens of each sequence (chunk-boundary checkpoints).
 *   oracle_ckpt_store_int8 / oracle_ckpt_load_int8
 *                   the INT8 checkpoint of the infra page, section 6.6.2
 *                   (Int8CheckpointStore): per (slot, head, k) a scale from
 *                   the max-abs over d_v, symmetric codes in [-127, 127];
 *                   loading multiplies back into an active state row.
 *   oracle_conv1d_varlen / oracle_conv1d_update
 *                   the short causal convolution applied to q, k and v
 *                   before the recurrence (infra page, sections 6.5 and
 *                   8.2.3: causal_conv1d_fn for prefill, causal_conv1d_update
 *                   for decode, with a convolution state per request).  The
 *                   pages give no formula; the textbook depthwise causal
 *                   convolution is taken: per channel c and width W,
 *                   y_t = act(bias_c + sum_{i<W} w[c][i] x_{t-(W-1)+i}),
 *                   inputs before a sequence start coming from its state
 *                   (the last W-1 inputs seen, oldest first; zeros when
 *                   absent), act = identity or SiLU (y * sigmoid(y)).
 *   oracle_target_verify
 *                   speculative target verification (infra page, section
 *                   6.4, target_verify, and 6.5's verify intermediate state
 *                   indices): L draft tokens per request run through the
 *                   recurrence from the request's cached state, the output of
 *                   every token is returned and the state after each token
 *                   goes to its own slot of an intermediate-state pool; the
 *                   cached state itself is not changed (a caller commits the
 *                   accepted prefix by copying one intermediate slot).
 *   oracle_decode   one token of the same recurrence per request, reading
 *                   the state from a cache row by index and writing it back
 *                   in the cache dtype (the decode route named on the state
 *                   copy page, "Background").  An invalid index starts from
 *                   a zero state and writes nothing back.
 *
 * Readings where the pages are silent:
 *   - the state S is K x V; a cache row [H, V, K] holds element (v, k) of
 *     head h at ((h * V) + v) * K + k, i.e. S stored transposed;
 *   - L2 normalisation is x / sqrt(sum(x^2) + eps);
 *   - decay is applied before the delta-rule erase (M_t's factor order);
 *   - an empty sequence leaves its state unchanged and emits no output;
 *   - fp32 -> bf16 conversion rounds to nearest, ties to even.
 *
 * All floating-point work is fp64.  Inputs arrive already upcast to fp64 by
 * the caller, so the oracle sees exactly the values the GPU sees.
 * Parity status: pinned (see tests/test_oracle_pins.py for each pin).
 */
#include <float.h>
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_BF16 = 1 };

/* ---- bf16 conversion: round to nearest, ties to even, on the fp32 bits ---- */
static uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u); /* NaN stays a quiet NaN */
    /* add half an ulp of the kept part, plus one more when the kept part is odd */
    uint32_t keep_lsb = (u >> 16) & 1u;
    u += 0x7fffu + keep_lsb;
    return (uint16_t)(u >> 16);
}

static float orc_bf16_to_f32(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Exported for the bf16 rounding pins. */
void oracle_f32_to_bf16(const float *x, uint16_t *y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = orc_f32_to_bf16(x[i]);
}

static double orc_load(const void *base, int dtype, int64_t e)
{
    if (dtype == ORC_F32) return (double)((const float *)base)[e];
    return (double)orc_bf16_to_f32(((const uint16_t *)base)[e]);
}

/* fp64 -> cache dtype: first to fp32 (round to nearest), then to bf16 (RNE). */
static void orc_store(void *base, int dtype, int64_t e, double x)
{
    float f = (float)x;
    if (dtype == ORC_F32) ((float *)base)[e] = f;
    else ((uint16_t *)base)[e] = orc_f32_to_bf16(f);
}

static int orc_esize(int dtype) { return dtype == ORC_F32 ? 4 : 2; }

/* ------------------------------- state copy ------------------------------- */

/* packed[s, :] = cache[idx[s], :payload] if valid, else zeros.  Element by
 * element, bitwise.  Returns 0, or -1 on a bad argument. */
int oracle_gather(const void *cache, int dtype, int64_t n_rows, int64_t payload,
                  int64_t row_stride, const int64_t *idx, const uint8_t *flags,
                  int64_t selected, void *packed)
{
    if (dtype != ORC_F32 && dtype != ORC_BF16) return -1;
    if (n_rows <= 0 || payload <= 0 || row_stride < payload || selected < 0) return -1;
    const int es = orc_esize(dtype);
    for (int64_t s = 0; s < selected; ++s) {
        const int64_t r = idx[s];
        const int valid = r >= 0 && r < n_rows && (flags == NULL || flags[s] != 0);
        char *dst = (char *)packed + s * payload * es;
        for (int64_t e = 0; e < payload; ++e) {
            if (valid)
                memcpy(dst + e * es, (const char *)cache + (r * row_stride + e) * es, (size_t)es);
            else
                memset(dst + e * es, 0, (size_t)es);
        }
    }
    return 0;
}

/* cache[idx[s], :payload] = to_cache_dtype(packed[s, :]) for valid idx[s]. */
int oracle_scatter(void *cache, int cache_dtype, int64_t n_rows, int64_t payload,
                   int64_t row_stride, const int64_t *idx, int64_t selected,
                   const void *packed, int packed_dtype)
{
    if ((cache_dtype != ORC_F32 && cache_dtype != ORC_BF16) ||
        (packed_dtype != ORC_F32 && packed_dtype != ORC_BF16))
        return -1;
    if (n_rows <= 0 || payload <= 0 || row_stride < payload || selected < 0) return -1;
    for (int64_t s = 0; s < selected; ++s) {
        const int64_t r = idx[s];
        if (r < 0 || r >= n_rows) continue;
        for (int64_t e = 0; e < payload; ++e) {
            const int64_t src = s * payload + e;
            const int64_t dst = r * row_stride + e;
            if (packed_dtype == cache_dtype) {
                const int es = orc_esize(cache_dtype);
                memcpy((char *)cache + dst * es, (const char *)packed + src * es, (size_t)es);
            } else if (cache_dtype == ORC_F32) {
                ((float *)cache)[dst] = orc_bf16_to_f32(((const uint16_t *)packed)[src]);
            } else {
                ((uint16_t *)cache)[dst] = orc_f32_to_bf16(((const float *)packed)[src]);
            }
        }
    }
    return 0;
}

/* ---------------------------- INT8 checkpoints ---------------------------- */

static float orc_load_f32(const void *base, int dtype, int64_t e)
{
    return dtype == ORC_F32 ? ((const float *)base)[e] : orc_bf16_to_f32(((const uint16_t *)base)[e]);
}

/* Quantise active state rows into checkpoint slots: for each pair s with
 * 0 <= src[s] < n_rows and 0 <= dst[s] < n_slots, and each head h and key
 * channel k of the row's [H, V, K] block x (upcast to fp32):
 *   amax = max over v of |x[h][v][k]|;  scale = amax / 127;
 *   code[v] = round_half_even(x[h][v][k] / scale), clamped to [-127, 127];
 *   a scale below FLT_MIN (amax == 0, or amax < 127 * 2^-126) is stored
 *   as 0 with all codes 0 (a reading: the page does not say);
 * qdata[dst][h][v][k] = code, scale_out[dst][h][k] = scale.  Every operation
 * is one correctly rounded fp32 operation (the precision in which the codes
 * are decided on the GPU as well).  Pairs with an invalid index are skipped. */
int oracle_ckpt_store_int8(const void *active, int dtype, int64_t n_rows, int64_t row_stride,
                           int64_t H, int64_t V, int64_t K, const int64_t *src, const int64_t *dst,
                           int64_t count, int8_t *qdata, float *scale_out, int64_t n_slots)
{
    if (dtype != ORC_F32 && dtype != ORC_BF16) return -1;
    if (n_rows <= 0 || H <= 0 || V <= 0 || K <= 0 || row_stride < H * V * K || count < 0) return -1;
    for (int64_t s = 0; s < count; ++s) {
        const int64_t r = src[s], c = dst[s];
        if (r < 0 || r >= n_rows || c < 0 || c >= n_slots) continue;
        for (int64_t h = 0; h < H; ++h) {
            for (int64_t k = 0; k < K; ++k) {
                float amax = 0.0f;
                for (int64_t v = 0; v < V; ++v) {
                    const float a = fabsf(orc_load_f32(active, dtype, r * row_stride + (h * V + v) * K + k));
                    if (a > amax) amax = a;
                }
                float sc = amax / 127.0f;
                /* Reading where the page is silent: a scale below the smallest normal
                 * float (every |x| < 127 * 2^-126) is stored as 0 with all codes 0, so
                 * no code is ever formed by dividing by a subnormal scale. */
                if (sc < FLT_MIN) sc = 0.0f;
                scale_out[(c * H + h) * K + k] = sc;
                for (int64_t v = 0; v < V; ++v) {
                    int q = 0;
                    if (sc > 0.0f) {
                        const float y = orc_load_f32(active, dtype, r * row_stride + (h * V + v) * K + k) / sc;
                        const float rq = nearbyintf(y); /* default rounding: to nearest, ties to even */
                        q = rq > 127.0f ? 127 : rq < -127.0f ? -127 : (int)rq;
                    }
                    qdata[((c * H + h) * V + v) * K + k] = (int8_t)q;
                }
            }
        }
    }
    return 0;
}

/* Dequantise checkpoint slots into active state rows: for each pair s with
 * 0 <= src_slot[s] < n_slots and 0 <= dst_row[s] < n_rows,
 *   active[dst][h][v][k] = to_dtype(code[src][h][v][k] * scale[src][h][k])
 * (one fp32 multiply; bf16 rows round to nearest even).  Other rows and the
 * gaps between rows are not touched. */
int oracle_ckpt_load_int8(const int8_t *qdata, const float *scale, int64_t n_slots,
                          const int64_t *src_slot, const int64_t *dst_row, int64_t count, void *active,
                          int dtype, int64_t n_rows, int64_t row_stride, int64_t H, int64_t V, int64_t K)
{
    if (dtype != ORC_F32 && dtype != ORC_BF16) return -1;
    if (n_rows <= 0 || H <= 0 || V <= 0 || K <= 0 || row_stride < H * V * K || count < 0) return -1;
    for (int64_t s = 0; s < count; ++s) {
        const int64_t c = src_slot[s], r = dst_row[s];
        if (c < 0 || c >= n_slots || r < 0 || r >= n_rows) continue;
        for (int64_t h = 0; h < H; ++h)
            for (int64_t v = 0; v < V; ++v)
                for (int64_t k = 0; k < K; ++k) {
                    const float x = (float)qdata[((c * H + h) * V + v) * K + k] * scale[(c * H + h) * K + k];
                    const int64_t e = r * row_stride + (h * V + v) * K + k;
                    if (dtype == ORC_F32) ((float *)active)[e] = x;
                    else ((uint16_t *)active)[e] = orc_f32_to_bf16(x);
                }
    }
    return 0;
}

/* ------------------------- short causal convolution ------------------------ */

static double orc_act(double y, int act) { return act == 1 ? y / (1.0 + exp(-y)) : y; }

/* x: [T, C]; cu_seqlens: [B + 1]; weight: [C, W] (weight[c][W-1] multiplies the
 * current token); bias: [C] or NULL; init: [B, W-1, C] or NULL (zeros);
 * y: [T, C]; final_state: [B, W-1, C] = the last W-1 inputs of each sequence's
 * window, oldest first (init's rows when the sequence is shorter). */
int oracle_conv1d_varlen(const double *x, const int64_t *cu_seqlens, int64_t B, int64_t C, int64_t W,
                         const double *weight, const double *bias, int act, const double *init,
                         double *y, double *final_state)
{
    if (B < 0 || C <= 0 || W < 1 || (act != 0 && act != 1)) return -1;
    double *win = (double *)malloc(sizeof(double) * (size_t)W);
    if (!win) return -2;
    for (int64_t b = 0; b < B; ++b) {
        if (cu_seqlens[b + 1] < cu_seqlens[b]) { free(win); return -1; }
        for (int64_t c = 0; c < C; ++c) {
            /* window = (state oldest .. newest, current); the state part first */
            for (int64_t i = 0; i + 1 < W; ++i) win[i] = init ? init[(b * (W - 1) + i) * C + c] : 0.0;
            for (int64_t t = cu_seqlens[b]; t < cu_seqlens[b + 1]; ++t) {
                win[W - 1] = x[t * C + c];
                double acc = bias ? bias[c] : 0.0;
                for (int64_t i = 0; i < W; ++i) acc += weight[c * W + i] * win[i];
                y[t * C + c] = orc_act(acc, act);
                for (int64_t i = 0; i + 1 < W; ++i) win[i] = win[i + 1]; /* slide by one token */
            }
            for (int64_t i = 0; i + 1 < W; ++i) final_state[(b * (W - 1) + i) * C + c] = win[i];
        }
    }
    free(win);
    return 0;
}

/* One token per request on conv-state cache rows, in place: row idx[r] holds
 * [W-1, C] (oldest first) in the cache dtype; an invalid index starts from
 * zeros and writes nothing back.  x: [R, C]; y: [R, C]. */
int oracle_conv1d_update(const double *x, int64_t R, int64_t C, int64_t W, const double *weight,
                         const double *bias, int act, void *cache, int cache_dtype, int64_t n_rows,
                         int64_t row_stride, const int64_t *idx, double *y)
{
    if (R < 0 || C <= 0 || W < 2 || (act != 0 && act != 1)) return -1;
    if (cache_dtype != ORC_F32 && cache_dtype != ORC_BF16) return -1;
    double *win = (double *)malloc(sizeof(double) * (size_t)W);
    if (!win) return -2;
    for (int64_t r = 0; r < R; ++r) {
        const int64_t row = idx[r];
        const int valid = row >= 0 && row < n_rows;
        for (int64_t c = 0; c < C; ++c) {
            for (int64_t i = 0; i + 1 < W; ++i)
                win[i] = valid ? orc_load(cache, cache_dtype, row * row_stride + i * C + c) : 0.0;
            win[W - 1] = x[r * C + c];
            double acc = bias ? bias[c] : 0.0;
            for (int64_t i = 0; i < W; ++i) acc += weight[c * W + i] * win[i];
            y[r * C + c] = orc_act(acc, act);
            if (valid)
                for (int64_t i = 0; i + 1 < W; ++i)
                    orc_store(cache, cache_dtype, row * row_stride + i * C + c, win[i + 1]);
        }
    }
    free(win);
    return 0;
}

/* ------------------------------- recurrence ------------------------------- */

/* One token of S_t = (I - beta k k^T) Diag(exp g) S_{t-1} + beta k v^T and
 * o_t = scale * S_t^T q, on S (K x V, row-major S[k * V + v]).
 * qn, kn: K-long scratch; p: V-long scratch. */
static void orc_token_step(double *S, int64_t K, int64_t V, const double *q, const double *k,
                           const double *v, const double *g, double beta, double scale,
                           int l2norm, double eps, double *o, double *qn, double *kn, double *p)
{
    if (l2norm) {
        double sq = 0.0, sk = 0.0;
        for (int64_t c = 0; c < K; ++c) {
            sq += q[c] * q[c];
            sk += k[c] * k[c];
        }
        const double rq = 1.0 / sqrt(sq + eps), rk = 1.0 / sqrt(sk + eps);
        for (int64_t c = 0; c < K; ++c) {
            qn[c] = q[c] * rq;
            kn[c] = k[c] * rk;
        }
    } else {
        for (int64_t c = 0; c < K; ++c) {
            qn[c] = q[c];
            kn[c] = k[c];
        }
    }
    /* Diag(exp g) S */
    for (int64_t c = 0; c < K; ++c) {
        const double d = exp(g[c]);
        for (int64_t j = 0; j < V; ++j) S[c * V + j] *= d;
    }
    /* (I - beta k k^T) applied to the decayed state: S -= beta k (k^T S) */
    for (int64_t j = 0; j < V; ++j) {
        double acc = 0.0;
        for (int64_t c = 0; c < K; ++c) acc += kn[c] * S[c * V + j];
        p[j] = acc;
    }
    for (int64_t c = 0; c < K; ++c)
        for (int64_t j = 0; j < V; ++j) S[c * V + j] -= beta * kn[c] * p[j];
    /* + b_t = beta k v^T */
    for (int64_t c = 0; c < K; ++c)
        for (int64_t j = 0; j < V; ++j) S[c * V + j] += beta * kn[c] * v[j];
    /* o_t = scale * S_t^T q */
    for (int64_t j = 0; j < V; ++j) {
        double acc = 0.0;
        for (int64_t c = 0; c < K; ++c) acc += qn[c] * S[c * V + j];
        o[j] = scale * acc;
    }
}

typedef struct {
    const double *q, *k, *v, *g, *beta;
    const int64_t *cu_seqlens;
    const double *init; /* [B, H, V, K] or NULL */
    double *out;        /* [T, H, V] */
    double *final_state;/* [B, H, V, K] */
    int64_t B, H, K, V;
    double scale, eps;
    int l2norm;
    int64_t every;            /* checkpoint interval in tokens, 0: none */
    double *ckpt;             /* [slots, H, V, K] or NULL */
    const int64_t *ckpt_first;/* [B] first checkpoint slot of each sequence */
    int64_t n_items;
    int64_t next; /* work counter, atomically advanced */
} orc_prefill_job;

static void orc_prefill_item(orc_prefill_job *a, int64_t item, double *S, double *qn, double *kn,
                             double *p)
{
    const int64_t H = a->H, K = a->K, V = a->V;
    const int64_t b = item / H, h = item % H;
    for (int64_t j = 0; j < V; ++j)
        for (int64_t c = 0; c < K; ++c)
            S[c * V + j] = a->init ? a->init[((b * H + h) * V + j) * K + c] : 0.0;
    for (int64_t t = a->cu_seqlens[b]; t < a->cu_seqlens[b + 1]; ++t) {
        orc_token_step(S, K, V, a->q + (t * H + h) * K, a->k + (t * H + h) * K,
                       a->v + (t * H + h) * V, a->g + (t * H + h) * K, a->beta[t * H + h],
                       a->scale, a->l2norm, a->eps, a->out + (t * H + h) * V, qn, kn, p);
        const int64_t done = t - a->cu_seqlens[b] + 1; /* tokens of sequence b processed */
        if (a->ckpt && done % a->every == 0) {
            const int64_t slot = a->ckpt_first[b] + done / a->every - 1;
            for (int64_t j = 0; j < V; ++j)
                for (int64_t c = 0; c < K; ++c)
                    a->ckpt[((slot * H + h) * V + j) * K + c] = S[c * V + j];
        }
    }
    for (int64_t j = 0; j < V; ++j)
        for (int64_t c = 0; c < K; ++c)
            a->final_state[((b * H + h) * V + j) * K + c] = S[c * V + j];
}

static void *orc_prefill_worker(void *arg)
{
    orc_prefill_job *a = (orc_prefill_job *)arg;
    double *S = (double *)malloc(sizeof(double) * (size_t)(a->K * a->V + 2 * a->K + a->V));
    if (!S) return (void *)1;
    double *qn = S + a->K * a->V, *kn = qn + a->K, *p = kn + a->K;
    for (;;) {
        const int64_t item = __atomic_fetch_add(&a->next, 1, __ATOMIC_RELAXED);
        if (item >= a->n_items) break;
        orc_prefill_item(a, item, S, qn, kn, p);
    }
    free(S);
    return NULL;
}

static int orc_run_threads(void *(*fn)(void *), void *job, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    int started = 0, rc = 0;
    for (int i = 0; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, fn, job) != 0) break;
        ++started;
    }
    if (started == 0) return fn(job) == NULL ? 0 : -2;
    for (int i = 0; i < started; ++i) {
        void *ret = NULL;
        pthread_join(th[i], &ret);
        if (ret != NULL) rc = -2;
    }
    return rc;
}

/* Token-by-token prefill over a varlen batch.  q, k, g: [T, H, K]; v: [T, H, V];
 * beta: [T, H]; cu_seqlens: [B + 1]; init: [B, H, V, K] or NULL (zeros);
 * out: [T, H, V]; final_state: [B, H, V, K].  Returns 0 or a negative code. */
int oracle_prefill(const double *q, const double *k, const double *v, const double *g,
                   const double *beta, const int64_t *cu_seqlens, int64_t B, int64_t H,
                   int64_t K, int64_t V, const double *init, double scale, int l2norm,
                   double eps, double *out, double *final_state, int nthreads)
{
    if (B < 0 || H <= 0 || K <= 0 || V <= 0) return -1;
    for (int64_t b = 0; b < B; ++b)
        if (cu_seqlens[b + 1] < cu_seqlens[b]) return -1;
    orc_prefill_job a = {q, k, v, g, beta, cu_seqlens, init, out, final_state,
                         B, H, K, V, scale, eps, l2norm, 0, NULL, NULL, B * H, 0};
    return orc_run_threads(orc_prefill_worker, &a, nthreads);
}

/* oracle_prefill that also records checkpoints: the state after the first
 * m * every tokens of sequence b, m = 1 .. len_b / every, goes to slot
 * first_b + m - 1 of ckpt [slots, H, V, K], first_b = sum over b' < b of
 * len_b' / every (sequence-major).  The chunk-boundary states that the
 * "Support Kimi-K3 on NPU" report's extend listing returns for state
 * tracking, and the recurrent checkpoints written during prefill on the
 * infra page (section 8.2.4), at a fixed token interval. */
int oracle_prefill_ckpt(const double *q, const double *k, const double *v, const double *g,
                        const double *beta, const int64_t *cu_seqlens, int64_t B, int64_t H,
                        int64_t K, int64_t V, const double *init, double scale, int l2norm,
                        double eps, double *out, double *final_state, int64_t every, double *ckpt,
                        int nthreads)
{
    if (B < 0 || H <= 0 || K <= 0 || V <= 0 || every <= 0 || ckpt == NULL) return -1;
    for (int64_t b = 0; b < B; ++b)
        if (cu_seqlens[b + 1] < cu_seqlens[b]) return -1;
    int64_t *first = (int64_t *)malloc(sizeof(int64_t) * (size_t)(B > 0 ? B : 1));
    if (!first) return -2;
    int64_t n = 0;
    for (int64_t b = 0; b < B; ++b) {
        first[b] = n;
        n += (cu_seqlens[b + 1] - cu_seqlens[b]) / every;
    }
    orc_prefill_job a = {q, k, v, g, beta, cu_seqlens, init, out, final_state,
                         B, H, K, V, scale, eps, l2norm, every, ckpt, first, B * H, 0};
    const int rc = orc_run_threads(orc_prefill_worker, &a, nthreads);
    free(first);
    return rc;
}

typedef struct {
    const double *q, *k, *v, *g, *beta;
    int64_t R, H, K, V;
    double scale, eps;
    int l2norm;
    void *cache;
    int cache_dtype;
    int64_t n_rows, row_stride;
    const int64_t *idx;
    double *out;
    int64_t n_items, next;
} orc_decode_job;

static void *orc_decode_worker(void *arg)
{
    orc_decode_job *a = (orc_decode_job *)arg;
    const int64_t H = a->H, K = a->K, V = a->V;
    double *S = (double *)malloc(sizeof(double) * (size_t)(K * V + 2 * K + V));
    if (!S) return (void *)1;
    double *qn = S + K * V, *kn = qn + K, *p = kn + K;
    for (;;) {
        const int64_t item = __atomic_fetch_add(&a->next, 1, __ATOMIC_RELAXED);
        if (item >= a->n_items) break;
        const int64_t r = item / H, h = item % H;
        const int64_t row = a->idx[r];
        const int valid = row >= 0 && row < a->n_rows;
        const int64_t base = row * a->row_stride + h * V * K; /* used only when valid */
        for (int64_t j = 0; j < V; ++j)
            for (int64_t c = 0; c < K; ++c)
                S[c * V + j] = valid ? orc_load(a->cache, a->cache_dtype, base + j * K + c) : 0.0;
        orc_token_step(S, K, V, a->q + (r * H + h) * K, a->k + (r * H + h) * K,
                       a->v + (r * H + h) * V, a->g + (r * H + h) * K, a->beta[r * H + h],
                       a->scale, a->l2norm, a->eps, a->out + (r * H + h) * V, qn, kn, p);
        if (valid)
            for (int64_t j = 0; j < V; ++j)
                for (int64_t c = 0; c < K; ++c)
                    orc_store(a->cache, a->cache_dtype, base + j * K + c, S[c * V + j]);
    }
    free(S);
    return NULL;
}

/* One decode token per request on cache rows, in place.  q, k, g: [R, H, K];
 * v: [R, H, V]; beta: [R, H]; cache: n_rows rows of row_stride elements, each
 * holding [H, V, K]; idx: [R]; out: [R, H, V].  Valid indices must be unique. */
typedef struct {
    const double *q, *k, *v, *g, *beta;
    int64_t R, L, H, K, V;
    double scale, eps;
    int l2norm;
    const void *cache;
    int cache_dtype;
    int64_t n_rows, row_stride;
    const int64_t *idx;
    void *pool;
    int pool_dtype;
    int64_t pool_rows, pool_stride;
    const int64_t *inter_idx; /* [R, L] */
    double *out;              /* [R, L, H, V] */
    int64_t n_items, next;
} orc_verify_job;

static void *orc_verify_worker(void *arg)
{
    orc_verify_job *a = (orc_verify_job *)arg;
    const int64_t H = a->H, K = a->K, V = a->V, L = a->L;
    double *S = (double *)malloc(sizeof(double) * (size_t)(K * V + 2 * K + V));
    if (!S) return (void *)1;
    double *qn = S + K * V, *kn = qn + K, *p = kn + K;
    for (;;) {
        const int64_t item = __atomic_fetch_add(&a->next, 1, __ATOMIC_RELAXED);
        if (item >= a->n_items) break;
        const int64_t r = item / H, h = item % H;
        const int64_t row = a->idx[r];
        const int valid = row >= 0 && row < a->n_rows;
        for (int64_t j = 0; j < V; ++j)
            for (int64_t c = 0; c < K; ++c)
                S[c * V + j] = valid ? orc_load(a->cache, a->cache_dtype, row * a->row_stride + (h * V + j) * K + c)
                                     : 0.0;
        for (int64_t t = 0; t < L; ++t) {
            const int64_t tok = r * L + t;
            orc_token_step(S, K, V, a->q + (tok * H + h) * K, a->k + (tok * H + h) * K, a->v + (tok * H + h) * V,
                           a->g + (tok * H + h) * K, a->beta[tok * H + h], a->scale, a->l2norm, a->eps,
                           a->out + (tok * H + h) * V, qn, kn, p);
            const int64_t slot = a->inter_idx[tok];
            if (slot >= 0 && slot < a->pool_rows)
                for (int64_t j = 0; j < V; ++j)
                    for (int64_t c = 0; c < K; ++c)
                        orc_store(a->pool, a->pool_dtype, slot * a->pool_stride + (h * V + j) * K + c, S[c * V + j]);
        }
    }
    free(S);
    return NULL;
}

/* L tokens per request from cache row idx[r] (zeros when invalid; the cache is
 * only read).  q, k, g: [R, L, H, K]; v: [R, L, H, V]; beta: [R, L, H];
 * inter_idx: [R, L] pool rows (invalid: not written); out: [R, L, H, V]. */
int oracle_target_verify(const double *q, const double *k, const double *v, const double *g,
                         const double *beta, int64_t R, int64_t L, int64_t H, int64_t K, int64_t V,
                         double scale, int l2norm, double eps, const void *cache, int cache_dtype,
                         int64_t n_rows, int64_t row_stride, const int64_t *idx, void *pool, int pool_dtype,
                         int64_t pool_rows, int64_t pool_stride, const int64_t *inter_idx, double *out,
                         int nthreads)
{
    if (R < 0 || L < 1 || H <= 0 || K <= 0 || V <= 0 || n_rows <= 0 || row_stride < H * V * K) return -1;
    if (pool_rows < 0 || pool_stride < H * V * K) return -1;
    if ((cache_dtype != ORC_F32 && cache_dtype != ORC_BF16) || (pool_dtype != ORC_F32 && pool_dtype != ORC_BF16))
        return -1;
    orc_verify_job a = {q, k, v, g, beta, R, L, H, K, V, scale, eps, l2norm, cache, cache_dtype, n_rows,
                        row_stride, idx, pool, pool_dtype, pool_rows, pool_stride, inter_idx, out, R * H, 0};
    return orc_run_threads(orc_verify_worker, &a, nthreads);
}

int oracle_decode(const double *q, const double *k, const double *v, const double *g,
                  const double *beta, int64_t R, int64_t H, int64_t K, int64_t V, double scale,
                  int l2norm, double eps, void *cache, int cache_dtype, int64_t n_rows,
                  int64_t row_stride, const int64_t *idx, double *out, int nthreads)
{
    if (R < 0 || H <= 0 || K <= 0 || V <= 0 || n_rows <= 0 || row_stride < H * V * K) return -1;
    if (cache_dtype != ORC_F32 && cache_dtype != ORC_BF16) return -1;
    orc_decode_job a = {q, k, v, g, beta, R, H, K, V, scale, eps, l2norm, cache, cache_dtype,
                        n_rows, row_stride, idx, out, R * H, 0};
    return orc_run_threads(orc_decode_worker, &a, nthreads);
}
