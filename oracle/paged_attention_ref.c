/*
 * CPU fp64 oracle for ubatch-aligned paged attention (UA-PagedAttention).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the GPU path computes.  Only the test suite, the smoke
 * check and the CPU-baseline leg of the benchmark may load it.  It shares no
 * code, header, table or helper with the CUDA library; the product path never
 * calls it.
 *
 * Source of the method: "面向多并发长上下文的 llama.cpp 分页式 KV Cache 与计算加速优化"
 * (gitlink IFwnjPgFSU/mxzntdncglxtsjysx), section 作品简介: the KV cache keeps a
 * page mapping and a true length per sequence; at graph build the page table
 * and the true KV length are expanded per ubatch token, in token order, by the
 * sequence each token belongs to; the backend operator then reads only the
 * valid pages of each query's own sequence.  The result is ordinary causal,
 * sequence-restricted softmax attention -- paging only changes which cells are
 * touched -- so the oracle is that definition written out.
 *
 * Readings taken where the page is silent (each is listed in the design notes):
 *   - tok_kv_len[t] is the number of keys token t may see (its position + 1:
 *     the token's own K/V row is appended before attention);
 *   - query head h reads KV head h / (Hq / Hkv) (contiguous GQA grouping);
 *   - softmax is base e of scale * q.k, with max subtraction;
 *   - tok_kv_len[t] == 0 gives an all-zero output row;
 *   - slot_mapping[t] < 0 means "do not write" (padding token);
 *   - pool layout is [num_pages][Hkv][P][d], binary16 values.
 *
 * Parity pins (tests, not this file): brute-force unpaged attention from the
 * contiguous K/V before paging, torch SDPA in fp64 for one sequence, a
 * hand-derived closed-form fixture, and invariants (page permutation, NaN in
 * free cells, constant V, kv_len = 1, q = 0, shared prefix pages).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* IEEE 754 binary16 -> double, exact.  sign | 5-bit exponent (bias 15) | 10-bit fraction. */
double ref_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);               /* subnormal: m * 2^-14 * 2^-10 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);   /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/*
 * Per-token expansion of the page table and true KV length (作品简介: "将页表和
 * 真实 KV 长度按 token 顺序展开").  For ubatch token t of sequence s at position p:
 *   tok_page_table[t][:] = seq_page_table[s][:]
 *   tok_kv_len[t]        = p + 1
 *   slot_mapping[t]      = page * P + p % P, page = seq_page_table[s][p / P]
 * tok_seq[t] < 0 marks a padding token: row of -1, kv_len 0, slot -1.
 * A position whose page is not allocated (-1) gets slot -1.
 * Returns 0, or -1 if a sequence index or position is out of range.
 */
int ref_expand_ubatch(const int32_t *seq_page_table, int n_seq, int max_pages,
                      const int32_t *tok_seq, const int32_t *tok_pos, int T, int P,
                      int32_t *tok_page_table, int32_t *tok_kv_len, int64_t *slot_mapping)
{
    for (int t = 0; t < T; ++t) {
        int s = tok_seq[t];
        int32_t *row = tok_page_table + (size_t)t * max_pages;
        if (s < 0) {
            for (int i = 0; i < max_pages; ++i) row[i] = -1;
            tok_kv_len[t] = 0;
            slot_mapping[t] = -1;
            continue;
        }
        if (s >= n_seq) return -1;
        int p = tok_pos[t];
        if (p < 0 || p / P >= max_pages) return -1;
        const int32_t *srow = seq_page_table + (size_t)s * max_pages;
        for (int i = 0; i < max_pages; ++i) row[i] = srow[i];
        tok_kv_len[t] = p + 1;
        int page = srow[p / P];
        slot_mapping[t] = page < 0 ? -1 : (int64_t)page * P + (p % P);
    }
    return 0;
}

/*
 * reshape-and-cache (CacheFlow, 核心架构 3): write each token's new K and V rows
 * into its slot.  slot = page * P + offset; the row lands at
 * pages[page][h][offset][0:d].  Bit copy; slots < 0 are skipped.
 * Returns 0, or -1 if a slot is beyond the pool.
 */
int ref_kv_append(const uint16_t *k, const uint16_t *v, const int64_t *slot_mapping, int T,
                  uint16_t *k_pages, uint16_t *v_pages, int num_pages, int Hkv, int P, int d)
{
    for (int t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= (int64_t)num_pages * P) return -1;
        int64_t page = slot / P, off = slot % P;
        for (int h = 0; h < Hkv; ++h) {
            size_t dst = (((size_t)page * Hkv + h) * P + off) * d;
            size_t src = ((size_t)t * Hkv + h) * d;
            memcpy(k_pages + dst, k + src, (size_t)d * sizeof(uint16_t));
            memcpy(v_pages + dst, v + src, (size_t)d * sizeof(uint16_t));
        }
    }
    return 0;
}

/*
 * Page copy for a copy-on-write fork (CacheFlow page "CacheFlow：基于 llama.cpp 的
 * 多请求 LLM 推理优化引擎", section 核心架构 2 and 3: blocks shared by reference
 * count; a block-copy kernel makes a private copy before a shared, partly filled
 * block is written).  For each pair i < n: page dst[i] of both pools receives the
 * contents of page src[i] (all KV heads).  Bit copy, pairs in order.  A pair with
 * an id outside [0, num_pages) is skipped; returns the number of skipped pairs.
 */
int ref_copy_pages(const int32_t *src, const int32_t *dst, int n, uint16_t *k_pages,
                   uint16_t *v_pages, int num_pages, int Hkv, int P, int d)
{
    int skipped = 0;
    size_t page = (size_t)Hkv * P * d;
    for (int i = 0; i < n; ++i) {
        if (src[i] < 0 || src[i] >= num_pages || dst[i] < 0 || dst[i] >= num_pages) {
            ++skipped;
            continue;
        }
        memcpy(k_pages + (size_t)dst[i] * page, k_pages + (size_t)src[i] * page,
               page * sizeof(uint16_t));
        memcpy(v_pages + (size_t)dst[i] * page, v_pages + (size_t)src[i] * page,
               page * sizeof(uint16_t));
    }
    return skipped;
}

/*
 * Paged attention, by definition.  For each selected token t and query head h,
 * with L = tok_kv_len[t] and g = h / (Hq / Hkv):
 *   K_t[j] = k_pages[tok_page_table[t][j / P]][g][j % P][:]   (j < L), same for V
 *   s_j    = scale * sum_i q[t][h][i] * K_t[j][i]
 *   out[t][h][:] = sum_j softmax(s)_j * V_t[j][:]
 * all in double.  The K/V of the token are first gathered into contiguous
 * buffers, then the softmax is computed -- no blocking, no online rescaling.
 *
 * tokens == NULL selects all T tokens (out is [T][Hq][d]); otherwise the n_tok
 * listed token indices are computed and out is [n_tok][Hq][d].
 * Returns 0, or -1 on a page id outside [0, num_pages) or L beyond the row.
 */
int ref_paged_attention(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                        const int32_t *tok_page_table, int max_pages, const int32_t *tok_kv_len,
                        int T, int Hq, int Hkv, int P, int d, int num_pages, double scale,
                        const int32_t *tokens, int n_tok, double *out)
{
    int G = Hq / Hkv;
    int n = tokens ? n_tok : T;
    int bad = 0;
    long long pairs = (long long)n * Hq;
#pragma omp parallel for schedule(dynamic, 1) reduction(|: bad)
    for (long long pi = 0; pi < pairs; ++pi) {
        int ti = (int)(pi / Hq), h = (int)(pi % Hq);
        int t = tokens ? tokens[ti] : ti;
        int g = h / G;
        int L = tok_kv_len[t];
        double *o = out + ((size_t)ti * Hq + h) * d;
        for (int i = 0; i < d; ++i) o[i] = 0.0;
        if (L <= 0) continue;
        if (L > max_pages * P) { bad = 1; continue; }
        double *Kt = (double *)malloc(sizeof(double) * (size_t)L * d);
        double *Vt = (double *)malloc(sizeof(double) * (size_t)L * d);
        double *s = (double *)malloc(sizeof(double) * (size_t)L);
        const int32_t *row = tok_page_table + (size_t)t * max_pages;
        int ok = 1;
        /* gather this token's keys and values through its page-table row */
        for (int j = 0; j < L && ok; ++j) {
            int page = row[j / P];
            if (page < 0 || page >= num_pages) { ok = 0; break; }
            size_t base = (((size_t)page * Hkv + g) * P + (j % P)) * d;
            for (int i = 0; i < d; ++i) {
                Kt[(size_t)j * d + i] = ref_f16_to_f64(k_pages[base + i]);
                Vt[(size_t)j * d + i] = ref_f16_to_f64(v_pages[base + i]);
            }
        }
        if (ok) {
            const uint16_t *qh = q + ((size_t)t * Hq + h) * d;
            double m = -INFINITY;
            for (int j = 0; j < L; ++j) {
                double acc = 0.0;
                for (int i = 0; i < d; ++i) acc += ref_f16_to_f64(qh[i]) * Kt[(size_t)j * d + i];
                s[j] = scale * acc;
                if (s[j] > m) m = s[j];
            }
            double Z = 0.0;
            for (int j = 0; j < L; ++j) { s[j] = exp(s[j] - m); Z += s[j]; }
            for (int j = 0; j < L; ++j) {
                double w = s[j] / Z;
                for (int i = 0; i < d; ++i) o[i] += w * Vt[(size_t)j * d + i];
            }
        } else {
            bad = 1;
        }
        free(Kt); free(Vt); free(s);
    }
    return bad ? -1 : 0;
}

/*
 * Masked attention over a shared span of cells, the baseline that paging replaces
 * (UA-PagedAttention page, section 作品简介: the original cache is one span shared
 * by all sequences and attention reads all of it under a mask).  As
 * ref_paged_attention, except that key j (slot s = page * P + j % P of the token's
 * row) is used only if cell_seq[s] == tok_seq[t] and cell_pos[s] <= tok_pos[t];
 * the softmax runs over the kept keys; a token that keeps none gets a zero row.
 * Keys are gathered with their mask first, then the softmax is computed.
 */
int ref_masked_attention(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                         const int32_t *tok_page_table, int max_pages, const int32_t *tok_kv_len,
                         int T, int Hq, int Hkv, int P, int d, int num_pages, double scale,
                         const int32_t *cell_seq, const int32_t *cell_pos,
                         const int32_t *tok_seq, const int32_t *tok_pos,
                         const int32_t *tokens, int n_tok, double *out)
{
    int G = Hq / Hkv;
    int n = tokens ? n_tok : T;
    int bad = 0;
    long long pairs = (long long)n * Hq;
#pragma omp parallel for schedule(dynamic, 1) reduction(|: bad)
    for (long long pi = 0; pi < pairs; ++pi) {
        int ti = (int)(pi / Hq), h = (int)(pi % Hq);
        int t = tokens ? tokens[ti] : ti;
        int g = h / G;
        int L = tok_kv_len[t];
        double *o = out + ((size_t)ti * Hq + h) * d;
        for (int i = 0; i < d; ++i) o[i] = 0.0;
        if (L <= 0) continue;
        if (L > max_pages * P) { bad = 1; continue; }
        double *Kt = (double *)malloc(sizeof(double) * (size_t)L * d);
        double *Vt = (double *)malloc(sizeof(double) * (size_t)L * d);
        double *s = (double *)malloc(sizeof(double) * (size_t)L);
        const int32_t *row = tok_page_table + (size_t)t * max_pages;
        int kept = 0, ok = 1;
        /* gather the kept keys and values of this token */
        for (int j = 0; j < L && ok; ++j) {
            int page = row[j / P];
            if (page < 0 || page >= num_pages) { ok = 0; break; }
            size_t slot = (size_t)page * P + (j % P);
            if (cell_seq[slot] != tok_seq[t] || cell_pos[slot] > tok_pos[t]) continue;
            size_t base = (((size_t)page * Hkv + g) * P + (j % P)) * d;
            for (int i = 0; i < d; ++i) {
                Kt[(size_t)kept * d + i] = ref_f16_to_f64(k_pages[base + i]);
                Vt[(size_t)kept * d + i] = ref_f16_to_f64(v_pages[base + i]);
            }
            ++kept;
        }
        if (!ok) {
            bad = 1;
        } else if (kept > 0) {
            const uint16_t *qh = q + ((size_t)t * Hq + h) * d;
            double m = -INFINITY;
            for (int j = 0; j < kept; ++j) {
                double acc = 0.0;
                for (int i = 0; i < d; ++i) acc += ref_f16_to_f64(qh[i]) * Kt[(size_t)j * d + i];
                s[j] = scale * acc;
                if (s[j] > m) m = s[j];
            }
            double Z = 0.0;
            for (int j = 0; j < kept; ++j) { s[j] = exp(s[j] - m); Z += s[j]; }
            for (int j = 0; j < kept; ++j) {
                double w = s[j] / Z;
                for (int i = 0; i < d; ++i) o[i] += w * Vt[(size_t)j * d + i];
            }
        }
        free(Kt); free(Vt); free(s);
    }
    return bad ? -1 : 0;
}

/*
 * Reduced-precision KV pages (the adaptive KV quantisation named on the
 * "面向边缘智能体推理的 llama.cpp KV Cache 共享与复用优化" page; the model's KV
 * stays binary16 on the UA-PagedAttention page): FP8 E4M3 codes with one scale
 * per cached row (token, KV head).
 *
 * E4M3 ("fn" variant of the OCP 8-bit floating point formats): 1 sign bit, 4
 * exponent bits with bias 7, 3 mantissa bits; exponent 0 encodes subnormals
 * m/8 * 2^-6; the all-ones pattern (S.1111.111) is NaN; there is no infinity;
 * the largest finite magnitude is 1.75 * 2^8 = 448.
 */
double ref_e4m3_to_f64(uint8_t c)
{
    int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/*
 * Round x to the nearest E4M3 value, ties to the code with an even mantissa,
 * magnitudes past 448 to +-448 (saturating), NaN to NaN: a search over the 127
 * finite non-negative codes.
 */
uint8_t ref_f32_to_e4m3(float x)
{
    if (x != x) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7E;
    int best = 0;
    double best_err = a;  /* distance to code 0 */
    for (int c = 1; c <= 0x7E; ++c) {
        double err = fabs(ref_e4m3_to_f64((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return sign | (uint8_t)best;
}

/*
 * Quantise one binary16 row of n values: scale = amax / 448 in binary32 (1 if
 * the row is all zeros), code_i = E4M3(x_i / scale) with the division in binary32.
 */
static float quantise_row(const uint16_t *x, int n, uint8_t *codes, size_t stride)
{
    float amax = 0.f;
    for (int i = 0; i < n; ++i) {
        float v = fabsf((float)ref_f16_to_f64(x[i]));
        if (v > amax) amax = v;
    }
    float scale = amax > 0.f ? amax / 448.0f : 1.0f;
    for (int i = 0; i < n; ++i)
        codes[(size_t)i * stride] = ref_f32_to_e4m3((float)ref_f16_to_f64(x[i]) / scale);
    return scale;
}

/*
 * Quantising reshape-and-cache into FP8 pages.  For each token with slot >= 0
 * and each KV head h, the row of k (and of v) is quantised (quantise_row) and
 * written at page = slot / P, offset = slot % P:
 *   k8  [num_pages][Hkv][P][d]  codes, one row per cached token (as the f16 pool)
 *   v8t [num_pages][Hkv][d][P]  codes, transposed inside each (page, head) block
 *   k_scale, v_scale [num_pages][Hkv][P]  binary32 scale of each row
 * Returns 0, or -1 if a slot is beyond the pool.
 */
int ref_kv_append_fp8(const uint16_t *k, const uint16_t *v, const int64_t *slot_mapping, int T,
                      uint8_t *k8, uint8_t *v8t, float *k_scale, float *v_scale, int num_pages,
                      int Hkv, int P, int d)
{
    for (int t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= (int64_t)num_pages * P) return -1;
        int64_t page = slot / P, off = slot % P;
        for (int h = 0; h < Hkv; ++h) {
            size_t row = ((size_t)page * Hkv + h) * P + off;
            const uint16_t *kr = k + ((size_t)t * Hkv + h) * d;
            const uint16_t *vr = v + ((size_t)t * Hkv + h) * d;
            k_scale[row] = quantise_row(kr, d, k8 + row * d, 1);
            v_scale[row] = quantise_row(vr, d, v8t + ((size_t)page * Hkv + h) * d * P + off, P);
        }
    }
    return 0;
}

/*
 * Paged attention over FP8 pages: as ref_paged_attention, with
 *   K_t[j][i] = e4m3(k8[page][g][j % P][i]) * k_scale[page][g][j % P]
 *   V_t[j][i] = e4m3(v8t[page][g][i][j % P]) * v_scale[page][g][j % P]
 * (page = tok_page_table[t][j / P]), all in double.
 */
int ref_paged_attention_fp8(const uint16_t *q, const uint8_t *k8, const uint8_t *v8t,
                            const float *k_scale, const float *v_scale,
                            const int32_t *tok_page_table, int max_pages,
                            const int32_t *tok_kv_len, int T, int Hq, int Hkv, int P, int d,
                            int num_pages, double scale, const int32_t *tokens, int n_tok,
                            double *out)
{
    int G = Hq / Hkv;
    int n = tokens ? n_tok : T;
    int bad = 0;
    long long pairs = (long long)n * Hq;
#pragma omp parallel for schedule(dynamic, 1) reduction(|: bad)
    for (long long pi = 0; pi < pairs; ++pi) {
        int ti = (int)(pi / Hq), h = (int)(pi % Hq);
        int t = tokens ? tokens[ti] : ti;
        int g = h / G;
        int L = tok_kv_len[t];
        double *o = out + ((size_t)ti * Hq + h) * d;
        for (int i = 0; i < d; ++i) o[i] = 0.0;
        if (L <= 0) continue;
        if (L > max_pages * P) { bad = 1; continue; }
        double *Kt = (double *)malloc(sizeof(double) * (size_t)L * d);
        double *Vt = (double *)malloc(sizeof(double) * (size_t)L * d);
        double *s = (double *)malloc(sizeof(double) * (size_t)L);
        const int32_t *row = tok_page_table + (size_t)t * max_pages;
        int ok = 1;
        /* gather and dequantise this token's keys and values */
        for (int j = 0; j < L && ok; ++j) {
            int page = row[j / P];
            if (page < 0 || page >= num_pages) { ok = 0; break; }
            size_t r = ((size_t)page * Hkv + g) * P + (j % P);
            size_t vb = ((size_t)page * Hkv + g) * d * P + (j % P);
            for (int i = 0; i < d; ++i) {
                Kt[(size_t)j * d + i] = ref_e4m3_to_f64(k8[r * d + i]) * (double)k_scale[r];
                Vt[(size_t)j * d + i] = ref_e4m3_to_f64(v8t[vb + (size_t)i * P]) * (double)v_scale[r];
            }
        }
        if (ok) {
            const uint16_t *qh = q + ((size_t)t * Hq + h) * d;
            double m = -INFINITY;
            for (int j = 0; j < L; ++j) {
                double acc = 0.0;
                for (int i = 0; i < d; ++i) acc += ref_f16_to_f64(qh[i]) * Kt[(size_t)j * d + i];
                s[j] = scale * acc;
                if (s[j] > m) m = s[j];
            }
            double Z = 0.0;
            for (int j = 0; j < L; ++j) { s[j] = exp(s[j] - m); Z += s[j]; }
            for (int j = 0; j < L; ++j) {
                double w = s[j] / Z;
                for (int i = 0; i < d; ++i) o[i] += w * Vt[(size_t)j * d + i];
            }
        } else {
            bad = 1;
        }
        free(Kt); free(Vt); free(s);
    }
    return bad ? -1 : 0;
}

/* Number of threads the OpenMP runtime will use (reported beside CPU timings). */
int ref_num_threads(void)
{
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        {
#ifdef _OPENMP
            n = omp_get_num_threads();
#endif
        }
    }
    return n;
}
