/*
 * oracle.c -- float64 CPU oracle of one masked multi-head attention decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline / reference arm may load this library.  The product path (the
 * CUDA library) shares no code, header, table or helper with this file.
 *
 * What it computes, for every batch slot b with L = seq_lens[b] cached tokens:
 *
 *   1. Fused QKV bias (FasterTransformer practice notes, lpnh.cn, section 2.1:
 *      the QKV projection output is split into Q, K, V and the bias is added
 *      inside the fused attention step):
 *         q' = f32(q) + f32(b_q),  k' = f32(k_new) + f32(b_k),  v' likewise,
 *      each a single binary32 addition.
 *   2. KV-cache append (lpnh.cn section 2.2; "FasterTransformer source
 *      analysis", framerc.cn, section 3.2; intelliparadigm.com section 2.1):
 *      the cache is pre-allocated with layout [B, Hkv, Lmax, D] and the new
 *      token's K/V is written at position L.  fp32 stores k' as is; fp16/bf16
 *      store k' rounded to nearest-even; int8 stores the symmetric absmax code
 *      (pptc.cn section 3.1 "quantise K and V to INT8"):
 *         s = f32(max_d |k'_d|) / 127 (binary32 division),
 *         code_d = clamp(rint_even(k'_d / s), -127, 127) (binary32 division),
 *         s = 1 and code = 0 when the row is all zero;
 *      the scale goes to scales[0 for K / 1 for V][b][h][L].
 *      A slot with L < 0 is inactive; L >= Lmax is an overflow (framerc.cn
 *      section 3.2: a sequence longer than the preset maximum is an error).
 *      Both leave the cache untouched and give an all-zero output.
 *   3. Attention of the current token over positions 0..L inclusive (the
 *      causal mask ends at the current position; intelliparadigm.com section 1
 *      and lpnh.cn section 2.2: decode computes only the new token's Q and
 *      attends to every cached K, V), reading the cache after the append:
 *         s_t = scale * sum_d q'_d * K[t][d],   scale = 1/sqrt(D) by default,
 *         p_t = exp(s_t - max_u s_u) / sum_u exp(s_u - max_u s_u),
 *         o_d = sum_t p_t * V[t][d],
 *      With a sliding window of W > 0 positions ("10 tricks", pptc.cn,
 *      section 3.1: keep only the most recent history) the sums run over
 *      t = max(0, L + 1 - W) .. L instead.
 *      with q head h reading kv head h / (Hq / Hkv) (contiguous groups,
 *      pptc.cn section 3.4 on MQA/GQA).  int8 rows are dequantised as
 *      scale[t] * code before use.  Everything after the binary32 bias add is
 *      computed in float64.
 *   4. Several new tokens per step (q_len = T > 1; pptc.cn section 4.3,
 *      speculative decoding: the large model checks a run of draft tokens in
 *      one forward pass).  Token j of slot b is appended at position L + j,
 *      and its query attends to positions 0 .. L + j (with a window W, from
 *      max(0, L + j + 1 - W)): each draft token sees the cache and the draft
 *      tokens before it, as T single-token steps in a row would.  A slot with
 *      L + T > Lmax is an overflow.
 *   5. Output projection (lpnh.cn section 2.1: the fused kernels hand their
 *      result straight to the next projection): oracle_out_proj computes
 *         y[t][f] = sum_k W[f][k] * x[t][k],
 *      for the step's output x flattened to one row of Hq * D values per token
 *      and a weight W laid out as a linear layer's [F][Hq * D], in float64.
 *
 * Plain loops, no blocking, no fusion: a reader can check each line against
 * the formulas above.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2, OR_I8 = 3 };

typedef struct {
    int B, Hq, Hkv, D, Lmax;
    int qkv_dtype;    /* q, k_new, v_new, bias: OR_F32 / OR_F16 / OR_BF16 */
    int cache_dtype;  /* OR_F32 / OR_F16 / OR_BF16 / OR_I8 */
    double softmax_scale; /* <= 0 selects 1/sqrt(D) */
    int window;           /* > 0: attend only the last `window` positions (sliding window) */
    int q_len;            /* new tokens per slot in this step; 0 counts as 1 */
} oracle_cfg;

/* ---- storage formats (IEEE-754 definitions) ---------------------------- */

float oracle_bf16_to_f32(uint16_t h) {
    /* bfloat16 is the upper half of a binary32 pattern */
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

uint16_t oracle_f32_to_bf16(float f) {
    /* round to nearest, ties to even, on the 16 dropped bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u); /* NaN stays NaN */
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

float oracle_f16_to_f32(uint16_t h) {
    _Float16 x;
    memcpy(&x, &h, 2);
    return (float)x;
}

uint16_t oracle_f32_to_f16(float f) {
    _Float16 x = (_Float16)f; /* IEEE conversion, round to nearest even */
    uint16_t h;
    memcpy(&h, &x, 2);
    return h;
}

static float load_elem(const void* base, int dt, size_t i) {
    switch (dt) {
    case OR_F32: return ((const float*)base)[i];
    case OR_F16: return oracle_f16_to_f32(((const uint16_t*)base)[i]);
    case OR_BF16: return oracle_bf16_to_f32(((const uint16_t*)base)[i]);
    default: return (float)((const int8_t*)base)[i];
    }
}

static void store_elem(void* base, int dt, size_t i, float x) {
    switch (dt) {
    case OR_F32: ((float*)base)[i] = x; break;
    case OR_F16: ((uint16_t*)base)[i] = oracle_f32_to_f16(x); break;
    case OR_BF16: ((uint16_t*)base)[i] = oracle_f32_to_bf16(x); break;
    default: break;
    }
}

/* ---- INT8 symmetric absmax quantiser for one row ----------------------- */

void oracle_quant_i8(const float* x, int D, int8_t* code, float* scale) {
    float amax = 0.0f;
    for (int d = 0; d < D; ++d) {
        float a = fabsf(x[d]);
        if (a > amax) amax = a;
    }
    if (amax == 0.0f) {
        for (int d = 0; d < D; ++d) code[d] = 0;
        *scale = 1.0f;
        return;
    }
    float s = amax / 127.0f;
    for (int d = 0; d < D; ++d) {
        float r = rintf(x[d] / s);
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        code[d] = (int8_t)r;
    }
    *scale = s;
}

/* ---- attention of one query over n cached rows (all float64) ---------- */

/* o[D] = softmax(scale * K q) V ;  K, V are [n][D] row-major; p (optional) gets the weights. */
void oracle_attend(const double* q, const double* K, const double* V, int n, int D,
                   double scale, double* o, double* p) {
    double m = -INFINITY;
    for (int t = 0; t < n; ++t) {
        double s = 0.0;
        for (int d = 0; d < D; ++d) s += q[d] * K[(size_t)t * D + d];
        s *= scale;
        if (p) p[t] = s;
        if (s > m) m = s;
    }
    double denom = 0.0;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    for (int t = 0; t < n; ++t) {
        double s = 0.0;
        for (int d = 0; d < D; ++d) s += q[d] * K[(size_t)t * D + d];
        s *= scale;
        double w = exp(s - m);
        denom += w;
        for (int d = 0; d < D; ++d) o[d] += w * V[(size_t)t * D + d];
        if (p) p[t] = w;
    }
    for (int d = 0; d < D; ++d) o[d] /= denom;
    if (p)
        for (int t = 0; t < n; ++t) p[t] /= denom;
}

/* ---- one decode step -------------------------------------------------- */

static size_t cache_index(const oracle_cfg* c, int b, int h, int pos, int d) {
    return (((size_t)b * c->Hkv + h) * c->Lmax + pos) * c->D + d;
}

static double dequant(const oracle_cfg* c, const void* cache, const float* scale_plane,
                      int b, int h, int pos, int d) {
    size_t i = cache_index(c, b, h, pos, d);
    if (c->cache_dtype == OR_I8) {
        double s = scale_plane[((size_t)b * c->Hkv + h) * c->Lmax + pos];
        return s * (double)((const int8_t*)cache)[i];
    }
    return (double)load_elem(cache, c->cache_dtype, i);
}

/* Appends k_new/v_new (+ bias) into the caches, then writes out[B][T][Hq][D].
 * q: [B][T][Hq][D]; k_new, v_new: [B][T][Hkv][D] (T = q_len).
 * bias: NULL or [(Hq + 2*Hkv) * D] laid out as q | k | v, the same for every token.
 * scales: [2][B][Hkv][Lmax] fp32 when cache_dtype is int8, else ignored.
 * Returns 1 when some slot had seq_lens[b] + T > Lmax, else 0. */
int oracle_decode_step(const oracle_cfg* c, const void* q, const void* k_new, const void* v_new,
                       const void* bias, void* k_cache, void* v_cache, const int32_t* seq_lens,
                       float* scales, double* out, int nthreads) {
    const int B = c->B, Hq = c->Hq, Hkv = c->Hkv, D = c->D, Lmax = c->Lmax;
    const int T = c->q_len > 1 ? c->q_len : 1;
    const int g = Hq / Hkv;
    const double scale = c->softmax_scale > 0.0 ? c->softmax_scale : 1.0 / sqrt((double)D);
    const size_t plane = (size_t)B * Hkv * Lmax;
    int overflow = 0;

    /* step 2: append */
    float kf[1024], vf[1024];
    int8_t code[1024];
    for (int b = 0; b < B; ++b) {
        if (seq_lens[b] < 0) continue;
        if (seq_lens[b] > Lmax - T) { overflow = 1; continue; }
        for (int j = 0; j < T; ++j)
        for (int h = 0; h < Hkv; ++h) {
            const int L = seq_lens[b] + j; /* position of token j */
            for (int d = 0; d < D; ++d) {
                size_t i = (((size_t)b * T + j) * Hkv + h) * D + d;
                float kb = bias ? load_elem(bias, c->qkv_dtype, (size_t)(Hq + h) * D + d) : 0.0f;
                float vb = bias ? load_elem(bias, c->qkv_dtype, (size_t)(Hq + Hkv + h) * D + d) : 0.0f;
                kf[d] = load_elem(k_new, c->qkv_dtype, i) + kb;
                vf[d] = load_elem(v_new, c->qkv_dtype, i) + vb;
            }
            if (c->cache_dtype == OR_I8) {
                size_t si = ((size_t)b * Hkv + h) * Lmax + L;
                oracle_quant_i8(kf, D, code, &scales[si]);
                for (int d = 0; d < D; ++d) ((int8_t*)k_cache)[cache_index(c, b, h, L, d)] = code[d];
                oracle_quant_i8(vf, D, code, &scales[plane + si]);
                for (int d = 0; d < D; ++d) ((int8_t*)v_cache)[cache_index(c, b, h, L, d)] = code[d];
            } else {
                for (int d = 0; d < D; ++d) {
                    store_elem(k_cache, c->cache_dtype, cache_index(c, b, h, L, d), kf[d]);
                    store_elem(v_cache, c->cache_dtype, cache_index(c, b, h, L, d), vf[d]);
                }
            }
        }
    }

    /* step 3: attention per (slot, token, query head) */
    const float* ks = scales;
    const float* vs = scales ? scales + plane : NULL;
    long npairs = (long)B * T * Hq;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic) num_threads(nthreads)
#endif
    for (long bh = 0; bh < npairs; ++bh) {
        int b = (int)(bh / ((long)T * Hq)), j = (int)(bh / Hq % T), h = (int)(bh % Hq), kvh = h / g;
        double* o = out + (size_t)bh * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (seq_lens[b] < 0 || seq_lens[b] > Lmax - T) continue;
        int n = seq_lens[b] + j + 1; /* token j sees positions 0 .. L + j */
        int t_lo = (c->window > 0 && n > c->window) ? n - c->window : 0;
        double qd[1024];
        for (int d = 0; d < D; ++d) {
            float qb = bias ? load_elem(bias, c->qkv_dtype, (size_t)h * D + d) : 0.0f;
            qd[d] = (double)(load_elem(q, c->qkv_dtype, (size_t)bh * D + d) + qb);
        }
        /* plain two-pass softmax over the visible positions t_lo .. L */
        double m = -INFINITY;
        for (int t = t_lo; t < n; ++t) {
            double s = 0.0;
            for (int d = 0; d < D; ++d) s += qd[d] * dequant(c, k_cache, ks, b, kvh, t, d);
            s *= scale;
            if (s > m) m = s;
        }
        double denom = 0.0;
        for (int t = t_lo; t < n; ++t) {
            double s = 0.0;
            for (int d = 0; d < D; ++d) s += qd[d] * dequant(c, k_cache, ks, b, kvh, t, d);
            s *= scale;
            double w = exp(s - m);
            denom += w;
            for (int d = 0; d < D; ++d) o[d] += w * dequant(c, v_cache, vs, b, kvh, t, d);
        }
        for (int d = 0; d < D; ++d) o[d] /= denom;
    }
    (void)nthreads;
    return overflow;
}

/* Step 5: y [n_tok][F] = x [n_tok][K] times the transpose of W [F][K], in float64. */
void oracle_out_proj(const double* x, const double* W, int n_tok, int K, int F, double* y) {
    for (int t = 0; t < n_tok; ++t)
        for (int f = 0; f < F; ++f) {
            double s = 0.0;
            for (int k = 0; k < K; ++k) s += W[(size_t)f * K + k] * x[(size_t)t * K + k];
            y[(size_t)t * F + f] = s;
        }
}
