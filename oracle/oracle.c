/*
 * Plain CPU oracle for paged-KV append and paged attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library: the cache layout, the FP8 code and the bf16 rounding are
 * restated here from their definitions.
 *
 * What it computes (the plain reading of the pages):
 *   - inferd README, "Paged KV" phase and the "Paged KV equivalence" result
 *     (max |dlogit| = 0): attention through a block table equals dense
 *     attention over the gathered context.  So attention here is the textbook
 *     definition softmax(q . K^T * scale) . V in fp64, over K/V gathered one
 *     token at a time through the block table.
 *   - lfm25-inference README, "Paged GQA/XQA Decode Attention": query heads are
 *     grouped over KV heads; query head h reads KV head h / (Hq / Hkv).
 *   - inferd README, speculative-decoding section: a verify step scores a short
 *     window of draft tokens causally; query i of a Q-token window sees context
 *     positions 0 .. L - Q + i (L counts the appended window).
 *   - lfm25-inference README, "--page-size 16": block size 16.
 *   - FP8 cache (no page defines it): OCP 8-bit floating point, E4M3 variant
 *     "fn" (bias 7, no infinities, S.1111.111 = NaN, max finite 448, subnormals
 *     m * 2^-9), stored value = e4m3(RNE, saturating)( (float)x / scale ), the
 *     division done once in IEEE fp32 round-to-nearest; dequantised value =
 *     code value * scale, exact in fp64.
 *
 * Cache layout (the library's ABI; the pages fix none): K and V are
 * [num_blocks][num_kv_heads][page], one page holding the 16 tokens of a block
 * for one kv-head as [16/8][D/C][8][C] with C = 16 bytes / element size
 * (C = 8 for bf16, 16 for fp8): groups of 8 tokens, then 16-byte chunks of the
 * head dimension, then the 8 tokens of the group, then the C elements of the
 * chunk.  Element (token off, dim d) of a page is at
 *   ((off / 8) * (D / C) + d / C) * 8 * C + (off % 8) * C + d % C.
 *
 * Build: gcc -O2 -std=c11 -shared -fPIC -pthread oracle.c -lm (no -ffast-math:
 * the FP8 encode relies on IEEE fp32 division and round-half-even nearbyint).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_BLOCK 16

/* ---------------------------------------------------------------- formats */

/* OCP E4M3 ("fn") code -> value.  NaN codes give NaN. */
double oracle_e4m3_decode(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);              /* subnormal: m/8 * 2^-6 */
    else
        v = ldexp((double)(8 + m), e - 10);    /* (1 + m/8) * 2^(e-7) */
    return s ? -v : v;
}

/* fp32 -> OCP E4M3 ("fn") code, round to nearest even, saturate to +-448.
 * NaN -> S.1111.111 with the input's sign; -0 -> 0x80. */
uint8_t oracle_e4m3_encode(float xf) {
    uint32_t bits;
    memcpy(&bits, &xf, 4);
    uint8_t sign = (bits >> 31) ? 0x80 : 0x00;
    if (isnan(xf)) return (uint8_t)(sign | 0x7F);
    double a = fabs((double)xf);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);      /* incl. inf: satfinite */
    if (a < ldexp(1.0, -6)) {                            /* subnormal spacing 2^-9 */
        double m = nearbyint(a * 512.0);                 /* 0..8; 8 is 2^-6 = 0x08 */
        return (uint8_t)(sign | (uint8_t)m);
    }
    int ex;
    double fr = frexp(a, &ex);                           /* a = fr * 2^ex, fr in [0.5,1) */
    int E = ex - 1;                                      /* a in [2^E, 2^(E+1)) */
    double t = nearbyint((2.0 * fr - 1.0) * 8.0);        /* mantissa in eighths; 8 carries */
    int code = ((E + 7) << 3) + (int)t;
    if (code > 0x7E) code = 0x7E;
    return (uint8_t)(sign | code);
}

/* fp64 -> bf16 bits, one rounding, to nearest even (overflow -> inf). */
uint16_t oracle_bf16_round(double x) {
    if (isnan(x)) return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80);
    int ex;
    frexp(a, &ex);
    int E = ex - 1;
    if (E < -126) E = -126;                  /* subnormal bf16: ulp 2^-133 */
    double ulp = ldexp(1.0, E - 7);          /* 8 significant bits */
    double r = nearbyint(a / ulp) * ulp;
    if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
    float f = (float)r;                      /* exact */
    uint32_t b;
    memcpy(&b, &f, 4);
    return (uint16_t)(sign | (b >> 16));
}

static double bf16_value(uint16_t h) {
    uint32_t b = (uint32_t)h << 16;
    float f;
    memcpy(&f, &b, 4);
    return (double)f;
}

/* ---------------------------------------------------------------- layout */

size_t oracle_cache_index(int64_t blk, int g, int off, int d, int num_kv_heads, int head_dim,
                          int elem_bytes) {
    int C = 16 / elem_bytes;
    size_t page = ((size_t)blk * (size_t)num_kv_heads + (size_t)g) * ORACLE_BLOCK * (size_t)head_dim;
    size_t within = ((size_t)(off / 8) * (size_t)(head_dim / C) + (size_t)(d / C)) * 8 * (size_t)C
                    + (size_t)(off % 8) * (size_t)C + (size_t)(d % C);
    return page + within;
}

/* ---------------------------------------------------------------- append */

/* kv_dtype 0 = bf16, 1 = fp8 e4m3.  k_new/v_new: [T][Hkv][D] bf16 bits.
 * Slot s >= 0 goes to block s / 16, offset s % 16; s < 0 is skipped.
 * Returns the number of slots that were out of range (skipped), or -1 on bad args. */
int64_t oracle_paged_kv_append(int kv_dtype, void* k_cache, void* v_cache, const float* k_scales,
                               const float* v_scales, int64_t num_blocks, int num_kv_heads,
                               int head_dim, const uint16_t* k_new, const uint16_t* v_new,
                               const int64_t* slots, int64_t num_tokens) {
    if (kv_dtype != 0 && kv_dtype != 1) return -1;
    int esz = kv_dtype == 1 ? 1 : 2;
    int64_t bad = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t s = slots[t];
        if (s < 0) continue;
        int64_t blk = s / ORACLE_BLOCK;
        int off = (int)(s % ORACLE_BLOCK);
        if (blk >= num_blocks) { ++bad; continue; }
        for (int g = 0; g < num_kv_heads; ++g) {
            for (int d = 0; d < head_dim; ++d) {
                size_t src = ((size_t)t * num_kv_heads + g) * head_dim + d;
                size_t dst = oracle_cache_index(blk, g, off, d, num_kv_heads, head_dim, esz);
                if (kv_dtype == 0) {
                    ((uint16_t*)k_cache)[dst] = k_new[src];
                    ((uint16_t*)v_cache)[dst] = v_new[src];
                } else {
                    float ks = k_scales[blk * num_kv_heads + g];
                    float vs = v_scales[blk * num_kv_heads + g];
                    /* one IEEE fp32 division, round to nearest (volatile keeps it fp32) */
                    volatile float kq = (float)bf16_value(k_new[src]) / ks;
                    volatile float vq = (float)bf16_value(v_new[src]) / vs;
                    ((uint8_t*)k_cache)[dst] = oracle_e4m3_encode(kq);
                    ((uint8_t*)v_cache)[dst] = oracle_e4m3_encode(vq);
                }
            }
        }
    }
    return bad;
}

/* ---------------------------------------------------------------- attention */

typedef struct {
    int kv_dtype;
    const void* k_cache;
    const void* v_cache;
    const float* k_scales;
    const float* v_scales;
    int64_t num_blocks;
    int num_kv_heads, head_dim, num_q_heads;
    const uint16_t* q;
    const int32_t* block_tables;
    int max_blocks_per_seq;
    const int32_t* context_lens;
    const int32_t* q_lens;
    const int64_t* q_offsets;
    int num_seqs;
    float scale;
    double* out;
    uint16_t* out_bf16;
    int nthreads;
    int tid;
    int status;
} attn_job;

static double kv_value(const attn_job* J, const void* cache, const float* scales, int64_t blk,
                       int g, int off, int d) {
    if (J->kv_dtype == 0) {
        size_t i = oracle_cache_index(blk, g, off, d, J->num_kv_heads, J->head_dim, 2);
        return bf16_value(((const uint16_t*)cache)[i]);
    }
    size_t i = oracle_cache_index(blk, g, off, d, J->num_kv_heads, J->head_dim, 1);
    return oracle_e4m3_decode(((const uint8_t*)cache)[i]) * (double)scales[blk * J->num_kv_heads + g];
}

/* One output row: sequence b, query index i of its window, query head h. */
static int attend_row(const attn_job* J, int b, int i, int h, double* s, double* acc) {
    int D = J->head_dim;
    int G = J->num_q_heads / J->num_kv_heads;
    int g = h / G;
    int L = J->context_lens[b], Q = J->q_lens[b];
    int lim = L - Q + i;                         /* last visible position, inclusive */
    if (lim < 0) return 2;
    const uint16_t* qrow = J->q + ((size_t)(J->q_offsets[b] + i) * J->num_q_heads + h) * D;
    double m = -INFINITY;
    for (int j = 0; j <= lim; ++j) {
        int64_t blk = J->block_tables[(size_t)b * J->max_blocks_per_seq + j / ORACLE_BLOCK];
        if (blk < 0 || blk >= J->num_blocks) return 3;
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += bf16_value(qrow[d]) * kv_value(J, J->k_cache, J->k_scales, blk, g, j % ORACLE_BLOCK, d);
        s[j] = (double)J->scale * dot;
        if (s[j] > m) m = s[j];
    }
    double den = 0.0;
    for (int d = 0; d < D; ++d) acc[d] = 0.0;
    for (int j = 0; j <= lim; ++j) {
        int64_t blk = J->block_tables[(size_t)b * J->max_blocks_per_seq + j / ORACLE_BLOCK];
        double w = exp(s[j] - m);
        den += w;
        for (int d = 0; d < D; ++d)
            acc[d] += w * kv_value(J, J->v_cache, J->v_scales, blk, g, j % ORACLE_BLOCK, d);
    }
    size_t o = ((size_t)(J->q_offsets[b] + i) * J->num_q_heads + h) * D;
    for (int d = 0; d < D; ++d) {
        double v = acc[d] / den;
        J->out[o + d] = v;
        if (J->out_bf16) J->out_bf16[o + d] = oracle_bf16_round(v);
    }
    return 0;
}

static void* attn_worker(void* arg) {
    attn_job* J = (attn_job*)arg;
    int maxL = 1;
    for (int b = 0; b < J->num_seqs; ++b)
        if (J->context_lens[b] > maxL) maxL = J->context_lens[b];
    double* s = (double*)malloc(sizeof(double) * (size_t)maxL);
    double* acc = (double*)malloc(sizeof(double) * (size_t)J->head_dim);
    if (!s || !acc) { J->status = 4; free(s); free(acc); return NULL; }
    /* work items (b, h), strided over threads */
    int64_t n_items = (int64_t)J->num_seqs * J->num_q_heads;
    for (int64_t it = J->tid; it < n_items; it += J->nthreads) {
        int b = (int)(it / J->num_q_heads), h = (int)(it % J->num_q_heads);
        for (int i = 0; i < J->q_lens[b]; ++i) {
            int st = attend_row(J, b, i, h, s, acc);
            if (st) { J->status = st; break; }
        }
        if (J->status) break;
    }
    free(s);
    free(acc);
    return NULL;
}

/* q: [sum q_lens][Hq][D] bf16 bits, packed by sequence.  out: same shape, fp64.
 * out_bf16 (optional): the bf16 rounding of out.  Returns 0, or
 * 1 bad args, 2 q_len > context_len, 3 block id out of range, 4 no memory. */
int oracle_paged_attention(int kv_dtype, const void* k_cache, const void* v_cache,
                           const float* k_scales, const float* v_scales, int64_t num_blocks,
                           int num_kv_heads, int head_dim, const uint16_t* q, int num_q_heads,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           const int32_t* context_lens, const int32_t* q_lens, int num_seqs,
                           float scale, double* out, uint16_t* out_bf16, int nthreads) {
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0) return 1;
    if (kv_dtype != 0 && kv_dtype != 1) return 1;
    if (nthreads < 1) nthreads = 1;
    int64_t* qoff = (int64_t*)malloc(sizeof(int64_t) * (size_t)(num_seqs + 1));
    if (!qoff) return 4;
    qoff[0] = 0;
    for (int b = 0; b < num_seqs; ++b) qoff[b + 1] = qoff[b] + q_lens[b];
    attn_job* jobs = (attn_job*)calloc((size_t)nthreads, sizeof(attn_job));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(qoff); free(jobs); free(th); return 4; }
    for (int t = 0; t < nthreads; ++t) {
        attn_job J = {kv_dtype, k_cache, v_cache, k_scales, v_scales, num_blocks, num_kv_heads,
                      head_dim, num_q_heads, q, block_tables, max_blocks_per_seq, context_lens,
                      q_lens, qoff, num_seqs, scale, out, out_bf16, nthreads, t, 0};
        jobs[t] = J;
    }
    for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, attn_worker, &jobs[t]);
    attn_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
    int st = 0;
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].status) st = jobs[t].status;
    free(qoff);
    free(jobs);
    free(th);
    return st;
}

/* ---------------------------------------------------------------- RoPE */

/* Rotary position embedding, rotate-half form (the lfm25-inference file list
 * names kernels/rope.cu; the pages fix no form, this is the reading): for a
 * row x of head_dim D at position p and i < D/2, with angle = p * theta^(-2i/D),
 *   y_i       = x_i * cos(angle) - x_{i+D/2} * sin(angle)
 *   y_{i+D/2} = x_{i+D/2} * cos(angle) + x_i * sin(angle)
 * evaluated in fp64 and rounded once to bf16 (nearest even).
 * x, y: [T][H][D] bf16 bits (may be the same buffer); positions: [T]. */
void oracle_rope(const uint16_t* x, uint16_t* y, const int32_t* positions, int64_t T, int H, int D,
                 double theta) {
    int half = D / 2;
    double* row = (double*)malloc(sizeof(double) * (size_t)D);
    if (!row) return;
    for (int64_t t = 0; t < T; ++t) {
        for (int h = 0; h < H; ++h) {
            const uint16_t* src = x + ((size_t)t * H + h) * D;
            uint16_t* dst = y + ((size_t)t * H + h) * D;
            for (int d = 0; d < D; ++d) row[d] = bf16_value(src[d]);
            for (int i = 0; i < half; ++i) {
                double inv_freq = pow(theta, -2.0 * (double)i / (double)D);
                double angle = (double)positions[t] * inv_freq;
                double c = cos(angle), s = sin(angle);
                double a = row[i], b = row[i + half];
                dst[i] = oracle_bf16_round(a * c - b * s);
                dst[i + half] = oracle_bf16_round(b * c + a * s);
            }
        }
    }
    free(row);
}

/* FP8 scales chosen at append time: for every (block, kv-head) whose
 * offset-0 slot this call writes (a block the call starts), the scale is the
 * largest |value| among this call's values stored in that block and head,
 * NaN ignored, divided by 448 in IEEE fp32 (1.0 if that maximum is 0); other
 * blocks keep their scale.  k_new / v_new: [T][Hkv][D] bf16 bits (K already
 * rotated when RoPE is fused); slots as for the append. */
void oracle_fp8_autoscale(const uint16_t* k_new, const uint16_t* v_new, const int64_t* slots, int64_t T,
                          int Hkv, int D, int64_t num_blocks, float* k_scales, float* v_scales) {
    for (int64_t t = 0; t < T; ++t) {
        int64_t s = slots[t];
        if (s < 0 || s / ORACLE_BLOCK >= num_blocks || s % ORACLE_BLOCK != 0) continue;
        int64_t blk = s / ORACLE_BLOCK;
        for (int g = 0; g < Hkv; ++g) {
            double mk = 0.0, mv = 0.0;
            for (int64_t u = 0; u < T; ++u) {
                if (slots[u] < 0 || slots[u] / ORACLE_BLOCK != blk) continue;
                for (int d = 0; d < D; ++d) {
                    double a = fabs(bf16_value(k_new[((size_t)u * Hkv + g) * D + d]));
                    double b = fabs(bf16_value(v_new[((size_t)u * Hkv + g) * D + d]));
                    if (a > mk) mk = a;                 /* (NaN compares false: ignored) */
                    if (b > mv) mv = b;
                }
            }
            volatile float fk = (float)mk, fv = (float)mv;   /* exact: bf16 values */
            volatile float sk = fk / 448.0f, sv = fv / 448.0f;
            k_scales[blk * Hkv + g] = fk > 0.0f ? sk : 1.0f;
            v_scales[blk * Hkv + g] = fv > 0.0f ? sv : 1.0f;
        }
    }
}
