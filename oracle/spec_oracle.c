/*
 * spec_oracle.c — plain single-threaded CPU oracle of the exact greedy verify
 * step.  TEST INFRASTRUCTURE ONLY (see spec_oracle.h): nothing in the product
 * library links or calls it.  Build with -O2 -ffp-contract=off so that every
 * fp32 product and sum below is rounded on its own, as written.
 *
 * Every function is the plain definition, scalar, in serial order.  Precision:
 *   - integer sums are exact (int32/int64);
 *   - the per-superblock combination is fp32 with each operation rounded
 *     (our reading of the integer-dot anchor's fixed combination order,
 *     [32] §32.7);
 *   - sums of many fp32 terms (GEMM outputs over superblocks) accumulate in
 *     fp64 and are rounded to fp32 once;
 *   - RMSNorm, attention and SwiGLU are computed in fp64 and stored as fp32;
 *   - the residual stream is fp32 ([32] chapter intro: F32 residual);
 *   - K/V rows are stored as bf16, round-to-nearest-even.
 */
#include "spec_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* number formats                                                            */
/* ------------------------------------------------------------------------ */

/* IEEE binary16 -> binary32, exact. */
float orc_half_to_float(uint16_t h) {
    int sign = (h >> 15) & 1;
    int exp = (h >> 10) & 0x1f;
    int man = h & 0x3ff;
    double v;
    if (exp == 0) {
        v = ldexp((double)man, -24);                 /* subnormal: man * 2^-24 */
    } else if (exp == 31) {
        v = man ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + man), exp - 25);   /* (1 + man/1024) 2^(exp-15) */
    }
    return (float)(sign ? -v : v);
}

float orc_bf16_to_float(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* binary32 -> bfloat16, round to nearest, ties to even; NaN stays NaN. */
uint16_t orc_float_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return (uint16_t)((u >> 16) | 0x40);
    uint32_t keep = u >> 16;
    uint32_t rest = u & 0xffffu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1;
    return (uint16_t)keep;
}

/* ------------------------------------------------------------------------ */
/* Q4_K superblock (canonical byte layout, spec_verify.h)                    */
/*   bytes 0..1 d, 2..3 dmin (binary16); 4..15 a 96-bit LE field with sc_j at */
/*   bits 6j..6j+5 and m_j at bits 48+6j..; 16..143 codes, element e of      */
/*   sub-block j = e/32 in byte 16+16j+(e%32)%16, low nibble if e%32 < 16.   */
/* ------------------------------------------------------------------------ */

void orc_q4k_scale_min(const uint8_t* sb, int j, int* sc, int* m) {
    const uint8_t* f = sb + 4;
    int s = 0, mm = 0;
    for (int bit = 0; bit < 6; ++bit) {
        int p = 6 * j + bit;                 /* bit index in the 96-bit field */
        s |= ((f[p / 8] >> (p % 8)) & 1) << bit;
        int r = 48 + 6 * j + bit;
        mm |= ((f[r / 8] >> (r % 8)) & 1) << bit;
    }
    *sc = s;
    *m = mm;
}

int orc_q4k_code(const uint8_t* sb, int e) {
    int j = e / 32, r = e % 32;
    uint8_t byte = sb[16 + 16 * j + (r % 16)];
    return r < 16 ? (byte & 0x0f) : (byte >> 4);
}

static uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* w_e = d * sc_j * q_e - dmin * m_j, in fp64. */
void orc_q4k_dequant_f64(const uint8_t* W, int N, int K, double* out) {
    int nb = K / 256;
    for (int n = 0; n < N; ++n) {
        for (int b = 0; b < nb; ++b) {
            const uint8_t* sb = W + ((size_t)n * nb + b) * 144;
            double d = orc_half_to_float(rd16(sb));
            double dmin = orc_half_to_float(rd16(sb + 2));
            for (int e = 0; e < 256; ++e) {
                int sc, m;
                orc_q4k_scale_min(sb, e / 32, &sc, &m);
                out[(size_t)n * K + 256 * b + e] = d * sc * orc_q4k_code(sb, e) - dmin * m;
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Q8 activation quantisation, per row and 256-block:                        */
/*   d_a = amax / 127 (fp32 division); q = clamp(rint(x / d_a), -127, 127)   */
/*   with round-half-even (the default rounding mode); all-zero block -> 0.  */
/*   A_j = sum of the 32 codes of sub-block j.                                */
/* ------------------------------------------------------------------------ */
int orc_quantize_q8(const float* x, int M, int K, int8_t* q, float* d_a, int32_t* A) {
    int status = 0;
    int nb = K / 256;
    for (int m = 0; m < M; ++m) {
        for (int b = 0; b < nb; ++b) {
            const float* xb = x + (size_t)m * K + 256 * b;
            float amax = 0.0f;
            for (int e = 0; e < 256; ++e) {
                if (!isfinite(xb[e])) status |= ORC_ST_NONFINITE;
                float a = fabsf(xb[e]);
                if (a > amax) amax = a;
            }
            float d = amax / 127.0f;
            d_a[m * nb + b] = d;
            for (int e = 0; e < 256; ++e) {
                int v = 0;
                if (d != 0.0f && isfinite(xb[e])) {
                    float r = rintf(xb[e] / d);
                    if (r > 127.0f) r = 127.0f;
                    if (r < -127.0f) r = -127.0f;
                    v = (int)r;
                }
                q[(size_t)m * K + 256 * b + e] = (int8_t)v;
            }
            for (int j = 0; j < 8; ++j) {
                int32_t s = 0;
                for (int i = 0; i < 32; ++i) s += q[(size_t)m * K + 256 * b + 32 * j + i];
                A[(size_t)m * (K / 32) + 8 * b + j] = s;
            }
        }
    }
    return status;
}

/* ------------------------------------------------------------------------ */
/* Integer-dot GEMM ([32] §32.7 integer-dot anchor):                          */
/*   S_j = sum_i q_w * q_a (exact), ISc = sum_j sc_j S_j, IMn = sum_j m_j A_j */
/*   v_b = d_a * (f32(d) * f32(ISc) - f32(dmin) * f32(IMn)), each op rounded  */
/*   y = sum_b v_b, accumulated in fp64, rounded to fp32 once.               */
/* ------------------------------------------------------------------------ */
void orc_gemm_q4k(const uint8_t* W, int N, int K, const int8_t* q, const float* d_a,
                  const int32_t* A, int M, float* y, int32_t* isc, int32_t* imn, float* vb) {
    int nb = K / 256;
    double* acc = (double*)malloc(sizeof(double) * (size_t)M);
    for (int n = 0; n < N; ++n) {
        for (int m = 0; m < M; ++m) acc[m] = 0.0;
        for (int b = 0; b < nb; ++b) {
            /* decode the superblock once: codes, sub-scales, sub-mins, d, dmin */
            const uint8_t* sb = W + ((size_t)n * nb + b) * 144;
            int code[256], sc[8], mn[8];
            for (int j = 0; j < 8; ++j) orc_q4k_scale_min(sb, j, &sc[j], &mn[j]);
            for (int e = 0; e < 256; ++e) code[e] = orc_q4k_code(sb, e);
            float d = orc_half_to_float(rd16(sb));
            float dmin = orc_half_to_float(rd16(sb + 2));
            for (int m = 0; m < M; ++m) {
                const int8_t* qa = q + (size_t)m * K + 256 * b;
                int32_t ISc = 0, IMn = 0;
                for (int j = 0; j < 8; ++j) {
                    int32_t S = 0;
                    for (int i = 0; i < 32; ++i) S += code[32 * j + i] * qa[32 * j + i];
                    ISc += sc[j] * S;
                    IMn += mn[j] * A[(size_t)m * (K / 32) + 8 * b + j];
                }
                float t1 = d * (float)ISc;
                float t2 = dmin * (float)IMn;
                float diff = t1 - t2;
                float v = d_a[m * nb + b] * diff;
                size_t o = ((size_t)m * N + n) * nb + b;
                if (isc) isc[o] = ISc;
                if (imn) imn[o] = IMn;
                if (vb) vb[o] = v;
                acc[m] += (double)v;                 /* superblock order, per (m, n) */
            }
        }
        for (int m = 0; m < M; ++m) y[(size_t)m * N + n] = (float)acc[m];
    }
    free(acc);
}

/* ------------------------------------------------------------------------ */
/* The fixed fp32 order of the sum over superblocks (reading c6 of the       */
/* integer-dot contract, "a canonical order both sides implement"):          */
/*   units u = (group g of 128 output columns, superblock b), numbered       */
/*   g-major, U = ceil(N/128) * nb of them, are cut into G contiguous ranges */
/*   [floor(iU/G), floor((i+1)U/G)), i = 0..G-1;                             */
/*   inside a range, one group's values v_b are added in b order to a         */
/*   partial that starts at +0.0f;                                            */
/*   a group's partials are then added in range order, the first partial     */
/*   being the start value.                                                  */
/* G comes from the number of processors P: the largest G <= min(P, U,        */
/* floor(6U/nb)), at least 1, for which no group meets more than 8 ranges.    */
/* With G = 1 the result is the plain left-to-right fp32 sum over b.         */
/* ------------------------------------------------------------------------ */
static int orc_range_of_unit(long long x, long long U, int G) {
    return (int)(((x + 1) * (long long)G - 1) / U);   /* largest i: floor(iU/G) <= x */
}

int orc_split_ranges(int N, int K, int processors) {
    int nb = K / 256, ngroups = (N + 127) / 128;
    long long U = (long long)ngroups * nb;
    long long G = processors;
    if (G > U) G = U;
    if (nb > 0 && G > (6 * U) / nb) G = (6 * U) / nb;
    if (G < 1) G = 1;
    for (;;) {
        int worst = 1;
        for (int g = 0; g < ngroups; ++g) {
            long long first = (long long)g * nb, last = first + nb - 1;
            int n = orc_range_of_unit(last, U, (int)G) - orc_range_of_unit(first, U, (int)G) + 1;
            if (n > worst) worst = n;
        }
        if (worst <= 8 || G == 1) break;
        --G;
    }
    return (int)G;
}

void orc_sum_split(const float* vb, int M, int N, int nb, int G, float* y) {
    int ngroups = (N + 127) / 128;
    long long U = (long long)ngroups * nb;
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            int g = n / 128;
            const float* v = vb + ((size_t)m * N + n) * nb;
            float total = 0.0f;
            int have = 0;
            /* the ranges that meet group g, in order */
            int r0 = orc_range_of_unit((long long)g * nb, U, G);
            int r1 = orc_range_of_unit((long long)g * nb + nb - 1, U, G);
            for (int r = r0; r <= r1; ++r) {
                long long lo = (long long)r * U / G, hi = (long long)(r + 1) * U / G;
                long long b0 = lo > (long long)g * nb ? lo - (long long)g * nb : 0;
                long long b1 = hi < (long long)(g + 1) * nb ? hi - (long long)g * nb : nb;
                float part = 0.0f;
                for (long long b = b0; b < b1; ++b) part = part + v[b];
                total = have ? total + part : part;
                have = 1;
            }
            y[(size_t)m * N + n] = total;
        }
}

int orc_linear(const uint8_t* W, int N, int K, const float* x, int M, float* y) {
    int8_t* q = (int8_t*)malloc((size_t)M * K);
    float* d_a = (float*)malloc(sizeof(float) * (size_t)M * (K / 256));
    int32_t* A = (int32_t*)malloc(sizeof(int32_t) * (size_t)M * (K / 32));
    int st = orc_quantize_q8(x, M, K, q, d_a, A);
    orc_gemm_q4k(W, N, K, q, d_a, A, M, y, NULL, NULL, NULL);
    free(q);
    free(d_a);
    free(A);
    return st;
}

void orc_dense_f64(const uint8_t* W, int N, int K, const double* x, int M, double* y) {
    double* w = (double*)malloc(sizeof(double) * (size_t)N * K);
    orc_q4k_dequant_f64(W, N, K, w);
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int k = 0; k < K; ++k) acc += w[(size_t)n * K + k] * x[(size_t)m * K + k];
            y[(size_t)m * N + n] = acc;
        }
    free(w);
}

/* ------------------------------------------------------------------------ */
/* RMSNorm: y = x / sqrt(mean(x^2) + eps) * gamma  (fp64, stored fp32).      */
/* ------------------------------------------------------------------------ */
void orc_rmsnorm(const float* x, const float* gamma, int M, int H, float eps, float* y) {
    for (int m = 0; m < M; ++m) {
        double ss = 0.0;
        for (int i = 0; i < H; ++i) ss += (double)x[(size_t)m * H + i] * x[(size_t)m * H + i];
        double r = 1.0 / sqrt(ss / H + (double)eps);
        for (int i = 0; i < H; ++i) {
            double g = gamma ? gamma[i] : 1.0;
            y[(size_t)m * H + i] = (float)((double)x[(size_t)m * H + i] * r * g);
        }
    }
}

/* SwiGLU: h = silu(g) * u, silu(x) = x / (1 + e^-x)  (fp64, stored fp32). */
void orc_silu_mul(const float* gate, const float* up, int n, float* h) {
    for (int i = 0; i < n; ++i) {
        double g = gate[i];
        h[i] = (float)(g / (1.0 + exp(-g)) * (double)up[i]);
    }
}

/* Per-row argmax, lowest index among equal maxima; gap = top1 - top2. */
void orc_argmax(const float* logits, int M, int V, int32_t* idx, float* gap) {
    for (int m = 0; m < M; ++m) {
        const float* r = logits + (size_t)m * V;
        int best = 0;
        for (int v = 1; v < V; ++v)
            if (r[v] > r[best]) best = v;
        float second = -INFINITY;
        for (int v = 0; v < V; ++v)
            if (v != best && r[v] > second) second = r[v];
        idx[m] = best;
        if (gap) gap[m] = r[best] - second;
    }
}

/* ------------------------------------------------------------------------ */
/* Greedy acceptance ([33] §33.2 at temperature 0).  The stochastic rule       */
/* accepts token t with probability min(p_t/q_t, 1) and on the first reject  */
/* draws from normalize(max(p - q, 0)); on all-accept it draws from the last  */
/* row.  With one-hot p (target argmax) and q (draft token):                  */
/*   draft == argmax -> p/q = 1, accepted with certainty;                     */
/*   draft != argmax -> p_t = 0, rejected; the residual is one-hot at argmax. */
/* Hence L = first i < k with draft[i] != idx[i] (else k) and next = idx[L].  */
/* Geometry guard first: a token outside [0, vocab) rejects the whole call.   */
/* ------------------------------------------------------------------------ */
int orc_accept(const int32_t* idx, const int32_t* draft, int k, int vocab,
               int32_t* accepted, int32_t* next) {
    for (int i = 0; i < k; ++i)
        if (draft[i] < 0 || draft[i] >= vocab) return ORC_ST_TOKEN_RANGE;
    int L = k;
    for (int i = 0; i < k; ++i)
        if (draft[i] != idx[i]) { L = i; break; }
    *accepted = L;
    *next = idx[L];
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Stochastic exact acceptance ([33] §33.2, the general rule of which the     */
/* greedy accept above is the one-hot case).                                 */
/* ------------------------------------------------------------------------ */

/* MT19937, from its published definition (Matsumoto & Nishimura 1998):
 * degree n = 624, middle word m = 397, twist matrix a = 0x9908B0DF, tempering
 * (u, s, b, t, c, l) = (11, 7, 0x9D2C5680, 15, 0xEFC60000, 18), seeding
 * multiplier 1812433253.  The state is 625 words: the 624 state words and
 * the index of the next word to temper (624 = twist first). */
#define ORC_MT_N 624
#define ORC_MT_M 397

void orc_mt_seed(uint32_t* st, uint32_t seed) {
    st[0] = seed;
    for (uint32_t i = 1; i < ORC_MT_N; ++i)
        st[i] = 1812433253u * (st[i - 1] ^ (st[i - 1] >> 30)) + i;
    st[ORC_MT_N] = ORC_MT_N;
}

static void orc_mt_twist(uint32_t* st) {
    for (int i = 0; i < ORC_MT_N; ++i) {
        uint32_t x = (st[i] & 0x80000000u) | (st[(i + 1) % ORC_MT_N] & 0x7fffffffu);
        uint32_t xa = x >> 1;
        if (x & 1u) xa ^= 0x9908B0DFu;
        st[i] = st[(i + ORC_MT_M) % ORC_MT_N] ^ xa;
    }
    st[ORC_MT_N] = 0;
}

uint32_t orc_mt_next(uint32_t* st) {
    if (st[ORC_MT_N] >= ORC_MT_N) orc_mt_twist(st);
    uint32_t y = st[st[ORC_MT_N]++];
    y ^= y >> 11;
    y ^= (y << 7) & 0x9D2C5680u;
    y ^= (y << 15) & 0xEFC60000u;
    y ^= y >> 18;
    return y;
}

/* uniform in [0, 1): the top 24 bits of one draw, times 2^-24 (exact in
 * binary32).  The pages name uniform_f32 without its conversion; this is the
 * plainest one that uses every bit a binary32 in [0, 1) can hold. */
float orc_uniform_f32(uint32_t* st) { return (float)(orc_mt_next(st) >> 8) * 0x1p-24f; }

/* softmax of one logit row: p_x = exp(l_x - max) / sum, computed in fp64 and
 * rounded to fp32 once (temperature 1) */
void orc_softmax_row(const float* l, int V, float* p) {
    double m = -INFINITY;
    for (int x = 0; x < V; ++x)
        if (l[x] > m) m = l[x];
    double s = 0.0;
    for (int x = 0; x < V; ++x) s += exp((double)l[x] - m);
    for (int x = 0; x < V; ++x) p[x] = (float)(exp((double)l[x] - m) / s);
}

/* The draw of [33] §33.2 (sample_distribution_mt_ordered is named there, not
 * printed): one uniform u, then the tokens of the row's order with a running
 * fp32 sum c of their probabilities w; the first token with u < c.  The order
 * is index order (our reading of the precomputed order the rule walks), restricted to
 * the tokens with w > 0 as the listing filters it; a token of weight 0 adds
 * nothing to c and can never be the first with u < c, so the walk below skips
 * nothing explicitly.  If rounding leaves c <= u after the last token, the
 * last token of the order (the last with w > 0).
 * *margin receives the distance of u from the nearest running-sum boundary
 * around the chosen token. */
int32_t orc_sample_ordered(const float* w, int V, uint32_t* mt, double* margin) {
    const float u = orc_uniform_f32(mt);
    float c = 0.f, prev = 0.f;
    int32_t last = -1;
    for (int x = 0; x < V; ++x) {
        if (!(w[x] > 0.f)) continue;
        last = x;
        prev = c;
        c += w[x];
        if (u < c) {
            double d0 = (double)u - prev, d1 = (double)c - u;
            *margin = d0 < d1 ? d0 : d1;
            return x;
        }
    }
    *margin = (double)u - c;
    return last;
}

/* The accept rule of [33] §33.2 over k drafts, step by step as printed:
 *   for i < k: x = draft[i], p = p_i(x), q = q_i(x),
 *       a = 1 if q <= 0 else min(p / q, 1); one uniform u;
 *       u <= a: accept and go on; otherwise stop and build the residual
 *       r = max(p_i - q_i, 0) (fp32, token by token), total = its fp32 sum in
 *       token order; total <= 0: r = p_i; else every r_x /= total (fp32
 *       division); the next token is drawn from r (orc_sample_ordered);
 *   all accepted: the next token is drawn from p_k.
 * logits fp32 [k+1][V] (p = softmax, temperature 1); q fp32 [k][V] (the draft's
 * distributions); mt the 625-word MT19937 state, advanced by the draws.
 * res = {accepted, next}; *margin = the smallest distance of a uniform from
 * the threshold it was compared with (for tests that skip knife-edge draws).
 * Returns ORC_ST_TOKEN_RANGE for a draft token outside [0, V), before any draw. */
int orc_sample_accept(const float* logits, const float* q, const int32_t* draft, int k, int V,
                      uint32_t* mt, int32_t* res, double* margin) {
    for (int i = 0; i < k; ++i)
        if (draft[i] < 0 || draft[i] >= V) return ORC_ST_TOKEN_RANGE;
    float* p = (float*)malloc(sizeof(float) * (size_t)V);
    float* r = (float*)malloc(sizeof(float) * (size_t)V);
    double mg = INFINITY, m1;
    int L = k;
    for (int i = 0; i < k; ++i) {
        orc_softmax_row(logits + (size_t)i * V, V, p);
        const float qx = q[(size_t)i * V + draft[i]];
        const float px = p[draft[i]];
        const float a = qx <= 0.f ? 1.f : fminf(px / qx, 1.f);
        const float u = orc_uniform_f32(mt);
        if (fabs((double)u - a) < mg) mg = fabs((double)u - a);
        if (u <= a) continue;
        L = i;
        break;
    }
    int32_t next;
    if (L < k) {
        const float* qi = q + (size_t)L * V;
        float total = 0.f;
        for (int x = 0; x < V; ++x) {
            r[x] = fmaxf(p[x] - qi[x], 0.f);
            total += r[x];
        }
        if (total <= 0.f) {
            memcpy(r, p, sizeof(float) * (size_t)V);
        } else {
            for (int x = 0; x < V; ++x) r[x] /= total;
        }
        next = orc_sample_ordered(r, V, mt, &m1);
    } else {
        orc_softmax_row(logits + (size_t)k * V, V, p);
        next = orc_sample_ordered(p, V, mt, &m1);
    }
    if (m1 < mg) mg = m1;
    free(p);
    free(r);
    res[0] = L;
    res[1] = next;
    if (margin) *margin = mg;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Paged KV metadata ([8] §8.6 item 4: checkpoint = metadata rewind).         */
/* Free pages form a LIFO stack, initialised descending so that pops yield    */
/* ids 0, 1, 2, ...; pages are mapped in ascending logical order; a rollback  */
/* pushes the unmapped ids from the highest logical page down.                */
/* ------------------------------------------------------------------------ */
#define ORC_PAGE 16

void orc_kv_reset(orc_kv* kv) {
    for (int p = 0; p < kv->max_seq_pages; ++p) kv->page_table[p] = -1;
    for (int i = 0; i < kv->num_pages; ++i) kv->free_stack[i] = kv->num_pages - 1 - i;
    *kv->free_top = kv->num_pages;
    *kv->seq_len = 0;
}

int orc_kv_reserve(orc_kv* kv, int32_t upto) {
    int32_t pages = (upto + ORC_PAGE - 1) / ORC_PAGE;
    if (pages > kv->max_seq_pages) return ORC_ST_CTX_FULL;
    int need = 0;
    for (int p = 0; p < pages; ++p)
        if (kv->page_table[p] < 0) ++need;
    if (need > *kv->free_top) return ORC_ST_POOL_EMPTY;
    for (int p = 0; p < pages; ++p)
        if (kv->page_table[p] < 0) {
            *kv->free_top -= 1;
            kv->page_table[p] = kv->free_stack[*kv->free_top];
        }
    return 0;
}

int orc_kv_extend(orc_kv* kv, int32_t n) {
    int st = orc_kv_reserve(kv, *kv->seq_len + n);
    if (st) return st;
    *kv->seq_len += n;
    return 0;
}

int orc_kv_rollback(orc_kv* kv, int32_t new_len) {
    int32_t len = *kv->seq_len;
    if (new_len < 0 || new_len > len) return ORC_ST_ROLLBACK;
    int32_t hi = (len + ORC_PAGE - 1) / ORC_PAGE;       /* mapped: p < hi      */
    int32_t lo = (new_len + ORC_PAGE - 1) / ORC_PAGE;   /* kept:   p < lo      */
    for (int p = hi - 1; p >= lo; --p) {
        if (kv->page_table[p] >= 0) {
            kv->free_stack[*kv->free_top] = kv->page_table[p];
            *kv->free_top += 1;
            kv->page_table[p] = -1;
        }
    }
    *kv->seq_len = new_len;
    return 0;
}

static size_t kv_index(const orc_cfg* c, int page, int layer, int which, int head, int slot) {
    return ((((size_t)page * c->n_layers + layer) * 2 + which) * c->n_kv_heads + head) *
               (size_t)c->page_size * c->head_dim + (size_t)slot * c->head_dim;
}

void orc_kv_write_row(const orc_cfg* c, orc_kv* kv, int layer, int pos,
                      const float* k_row, const float* v_row) {
    int page = kv->page_table[pos / c->page_size];
    int slot = pos % c->page_size;
    for (int h = 0; h < c->n_kv_heads; ++h)
        for (int d = 0; d < c->head_dim; ++d) {
            kv->pool[kv_index(c, page, layer, 0, h, slot) + d] = orc_float_to_bf16(k_row[h * c->head_dim + d]);
            kv->pool[kv_index(c, page, layer, 1, h, slot) + d] = orc_float_to_bf16(v_row[h * c->head_dim + d]);
        }
}

/* ------------------------------------------------------------------------ */
/* Verify attention: row i sits at position n_past + i and sees positions     */
/* 0..n_past+i (its own block's earlier rows included).  Query head h reads   */
/* KV head h / (n_q/n_kv).  s_t = q.k_t / sqrt(head_dim), softmax over the    */
/* visible t (max subtracted), o = sum_t softmax_t v_t.  K and V are the      */
/* stored bf16 values.  fp64 throughout, stored fp32.                          */
/* ------------------------------------------------------------------------ */
int orc_layer_window(const orc_cfg* c, int layer) {
    if (c->swa_window > 0 && c->swa_period > 0 && layer % c->swa_period == c->swa_period - 1)
        return c->swa_window;
    return 0;
}

/* Row i sees the positions 0..n_past-1 and the block rows j with bit j of
 * mask[i] set (mask NULL: the causal block, j <= i).  A token tree's mask is
 * a node's ancestors and itself (up to 64 nodes).  In a sliding-window layer of window W the
 * row at position p = n_past + i sees only the positions t > p - W of those. */
void orc_attention_tree(const orc_cfg* c, const orc_kv* kv, int layer, const float* q,
                        int M, int n_past, const uint64_t* mask, float* out) {
    int dh = c->head_dim, group = c->n_q_heads / c->n_kv_heads;
    int max_vis = n_past + M;
    int W = orc_layer_window(c, layer);
    double* s = (double*)malloc(sizeof(double) * (size_t)max_vis);
    int* vt = (int*)malloc(sizeof(int) * (size_t)max_vis);
    double scale = 1.0 / sqrt((double)dh);
    for (int i = 0; i < M; ++i) {
        int nv = 0;                                   /* the visible positions, in order */
        int lo = W > 0 ? n_past + i - W + 1 : 0;      /* the window's first position */
        for (int t = 0; t < n_past; ++t)
            if (t >= lo) vt[nv++] = t;
        for (int j = 0; j < M; ++j)
            if ((mask ? ((mask[i] >> j) & 1ull) : (j <= i)) && n_past + j >= lo) vt[nv++] = n_past + j;
        for (int h = 0; h < c->n_q_heads; ++h) {
            int g = h / group;
            const float* qh = q + ((size_t)i * c->n_q_heads + h) * dh;
            double mx = -INFINITY;
            for (int e = 0; e < nv; ++e) {
                int t = vt[e];
                int page = kv->page_table[t / c->page_size];
                const uint16_t* kr = kv->pool + kv_index(c, page, layer, 0, g, t % c->page_size);
                double dot = 0.0;
                for (int d = 0; d < dh; ++d) dot += (double)qh[d] * orc_bf16_to_float(kr[d]);
                s[e] = dot * scale;
                if (s[e] > mx) mx = s[e];
            }
            double den = 0.0;
            for (int e = 0; e < nv; ++e) {
                s[e] = exp(s[e] - mx);
                den += s[e];
            }
            for (int d = 0; d < dh; ++d) {
                double o = 0.0;
                for (int e = 0; e < nv; ++e) {
                    int t = vt[e];
                    int page = kv->page_table[t / c->page_size];
                    const uint16_t* vr = kv->pool + kv_index(c, page, layer, 1, g, t % c->page_size);
                    o += s[e] * orc_bf16_to_float(vr[d]);
                }
                out[((size_t)i * c->n_q_heads + h) * dh + d] = (float)(o / den);
            }
        }
    }
    free(s);
    free(vt);
}

void orc_attention(const orc_cfg* c, const orc_kv* kv, int layer, const float* q,
                   int M, int n_past, float* out) {
    orc_attention_tree(c, kv, layer, q, M, n_past, NULL, out);
}

/* ------------------------------------------------------------------------ */
/* QK-norm and rotary position embedding (The DFlash draft, Ch. 8 §8.2,     */
/* lists both for the draft's attention, without formulas).  Readings:       */
/*   QK-norm: each q head and each k head x (head_dim values) becomes         */
/*     x_d / sqrt(mean(x^2) + eps) * g_d, the layer's gain g shared by heads; */
/*   RoPE ("rotate half"): with h = head_dim/2 and f_i = theta^(-i/h), the    */
/*     pair (x_i, x_{i+h}) at position p rotates by the angle p * f_i:        */
/*     x_i' = x_i cos - x_{i+h} sin,  x_{i+h}' = x_{i+h} cos + x_i sin.       */
/* Computed in fp64 and stored fp32; v is not touched.                        */
/* ------------------------------------------------------------------------ */
static void orc_head_norm_rope(const orc_cfg* c, const float* gain, float* x, int pos) {
    int dh = c->head_dim, h = dh / 2;
    double y[256];
    if (gain) {
        double ss = 0.0;
        for (int d = 0; d < dh; ++d) ss += (double)x[d] * x[d];
        double r = 1.0 / sqrt(ss / dh + (double)c->rms_eps);
        for (int d = 0; d < dh; ++d) y[d] = (double)x[d] * r * gain[d];
    } else {
        for (int d = 0; d < dh; ++d) y[d] = x[d];
    }
    if (c->rope_theta > 0.f) {
        for (int i = 0; i < h; ++i) {
            double a = (double)pos * pow((double)c->rope_theta, -(double)i / h);
            double cs = cos(a), sn = sin(a);
            double u = y[i], v = y[i + h];
            y[i] = u * cs - v * sn;
            y[i + h] = v * cs + u * sn;
        }
    }
    for (int d = 0; d < dh; ++d) x[d] = (float)y[d];
}

void orc_qk_norm_rope(const orc_cfg* c, const orc_weights* w, int layer, float* qkv, int M, int n_past) {
    int dh = c->head_dim;
    int Nqkv = (c->n_q_heads + 2 * c->n_kv_heads) * dh;
    const float* gq = w->q_norm ? w->q_norm[layer] : NULL;
    const float* gk = w->k_norm ? w->k_norm[layer] : NULL;
    if (!gq && !gk && !(c->rope_theta > 0.f)) return;
    for (int i = 0; i < M; ++i) {
        float* row = qkv + (size_t)i * Nqkv;
        for (int hq = 0; hq < c->n_q_heads; ++hq) orc_head_norm_rope(c, gq, row + (size_t)hq * dh, n_past + i);
        for (int hk = 0; hk < c->n_kv_heads; ++hk)
            orc_head_norm_rope(c, gk, row + (size_t)(c->n_q_heads + hk) * dh, n_past + i);
    }
}

/* ------------------------------------------------------------------------ */
/* One transformer block over M rows at positions n_past.. :                  */
/*   xn = rmsnorm(x, attn_norm); [Q|K|V] = W_qkv q8(xn); K,V -> bf16 cache;   */
/*   x += W_o q8(attention(Q));                                               */
/*   xn = rmsnorm(x, ffn_norm); [g|u] = W_gu q8(xn); x += W_down q8(silu(g)u) */
/* ------------------------------------------------------------------------ */
static int orc_block_tree(const orc_cfg* c, const orc_weights* w, orc_kv* kv, int layer,
                          const float* x_in, int M, int n_past, const uint64_t* mask, float* x_out) {
    int H = c->hidden, dh = c->head_dim, F = c->ffn;
    int nq = c->n_q_heads * dh, nkv = c->n_kv_heads * dh;
    int Nqkv = nq + 2 * nkv;
    int st = 0;
    float* xn = (float*)malloc(sizeof(float) * (size_t)M * H);
    float* qkv = (float*)malloc(sizeof(float) * (size_t)M * Nqkv);
    float* qv = (float*)malloc(sizeof(float) * (size_t)M * nq);
    float* att = (float*)malloc(sizeof(float) * (size_t)M * nq);
    float* o = (float*)malloc(sizeof(float) * (size_t)M * H);
    float* gu = (float*)malloc(sizeof(float) * (size_t)M * 2 * F);
    float* hh = (float*)malloc(sizeof(float) * (size_t)M * F);
    float* x = (float*)malloc(sizeof(float) * (size_t)M * H);

    const float* g_attn = (w->attn_norm) ? w->attn_norm[layer] : NULL;
    const float* g_ffn = (w->ffn_norm) ? w->ffn_norm[layer] : NULL;

    orc_rmsnorm(x_in, g_attn, M, H, c->rms_eps, xn);
    st |= orc_linear(w->w_qkv[layer], Nqkv, H, xn, M, qkv);
    orc_qk_norm_rope(c, w, layer, qkv, M, n_past);
    for (int i = 0; i < M; ++i) {
        memcpy(qv + (size_t)i * nq, qkv + (size_t)i * Nqkv, sizeof(float) * nq);
        orc_kv_write_row(c, kv, layer, n_past + i, qkv + (size_t)i * Nqkv + nq,
                         qkv + (size_t)i * Nqkv + nq + nkv);
    }
    orc_attention_tree(c, kv, layer, qv, M, n_past, mask, att);
    st |= orc_linear(w->w_o[layer], H, nq, att, M, o);
    for (size_t i = 0; i < (size_t)M * H; ++i) x[i] = x_in[i] + o[i];

    orc_rmsnorm(x, g_ffn, M, H, c->rms_eps, xn);
    st |= orc_linear(w->w_gate_up[layer], 2 * F, H, xn, M, gu);
    for (int i = 0; i < M; ++i)
        orc_silu_mul(gu + (size_t)i * 2 * F, gu + (size_t)i * 2 * F + F, F, hh + (size_t)i * F);
    st |= orc_linear(w->w_down[layer], H, F, hh, M, o);
    for (size_t i = 0; i < (size_t)M * H; ++i) x_out[i] = x[i] + o[i];

    free(xn); free(qkv); free(qv); free(att); free(o); free(gu); free(hh); free(x);
    return st;
}

int orc_block(const orc_cfg* c, const orc_weights* w, orc_kv* kv, int layer,
              const float* x_in, int M, int n_past, float* x_out) {
    return orc_block_tree(c, w, kv, layer, x_in, M, n_past, NULL, x_out);
}

static int orc_forward_tree(const orc_cfg* c, const orc_weights* w, orc_kv* kv, const float* hidden,
                            int M, const uint64_t* mask, int32_t* idx, float* logits, float* resid) {
    int H = c->hidden, V = c->vocab;
    int n_past = *kv->seq_len;
    int st = orc_kv_reserve(kv, n_past + M);
    if (st) return st;
    float* x = (float*)malloc(sizeof(float) * (size_t)M * H);
    float* y = (float*)malloc(sizeof(float) * (size_t)M * H);
    float* lg = logits ? logits : (float*)malloc(sizeof(float) * (size_t)M * V);
    memcpy(x, hidden, sizeof(float) * (size_t)M * H);
    for (int l = 0; l < c->n_layers; ++l) {
        if (resid) memcpy(resid + (size_t)l * M * H, x, sizeof(float) * (size_t)M * H);
        st |= orc_block_tree(c, w, kv, l, x, M, n_past, mask, y);
        memcpy(x, y, sizeof(float) * (size_t)M * H);
    }
    if (resid) memcpy(resid + (size_t)c->n_layers * M * H, x, sizeof(float) * (size_t)M * H);
    orc_rmsnorm(x, w->final_norm, M, H, c->rms_eps, y);
    st |= orc_linear(w->w_head, V, H, y, M, lg);
    for (size_t i = 0; i < (size_t)M * V; ++i)
        if (!isfinite(lg[i])) st |= ORC_ST_NONFINITE;
    orc_argmax(lg, M, V, idx, NULL);
    *kv->seq_len = n_past + M;
    if (!logits) free(lg);
    free(x);
    free(y);
    return st;
}

int orc_forward(const orc_cfg* c, const orc_weights* w, orc_kv* kv, const float* hidden,
                int M, int32_t* idx, float* logits, float* resid) {
    return orc_forward_tree(c, w, kv, hidden, M, NULL, idx, logits, resid);
}

/* The verify step ([33] §33.2, §33.7; [8] §8.6).  Returns -2 for a verify
 * length outside {3, 7, 15} (rejected before any work, [8] §8.6 item 3).
 * res = {accepted_len, next_token, status, seq_len}.  On a device-class error
 * the KV metadata is restored to its state before the step. */
int orc_verify_step(const orc_cfg* c, const orc_weights* w, orc_kv* kv, const float* hidden,
                    const int32_t* draft, int k, int32_t* res, int32_t* idx, float* logits,
                    float* resid) {
    if (k != 3 && k != 7 && k != 15) return -2;
    int n_past = *kv->seq_len;
    res[0] = 0;
    res[1] = -1;
    res[3] = n_past;
    for (int i = 0; i < k; ++i)
        if (draft[i] < 0 || draft[i] >= c->vocab) {
            res[2] = ORC_ST_TOKEN_RANGE;
            return 0;
        }
    int st = orc_forward(c, w, kv, hidden, k + 1, idx, logits, resid);
    if (st & (ORC_ST_POOL_EMPTY | ORC_ST_CTX_FULL)) {
        res[2] = st;
        return 0;
    }
    int32_t L = 0, next = -1;
    st |= orc_accept(idx, draft, k, c->vocab, &L, &next);
    if (st) {
        orc_kv_rollback(kv, n_past);
        res[2] = st;
        return 0;
    }
    orc_kv_rollback(kv, n_past + L + 1);
    res[0] = L;
    res[1] = next;
    res[2] = 0;
    res[3] = *kv->seq_len;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Token-tree verification ([33] §33.7: a tree spends the batch on covering  */
/* near-miss branches; it names trees of 24, 32, 48 and 64 nodes).  Node 0  */
/* is the carried frontier; node i >= 1 holds the draft token tokens[i],      */
/* proposed as the continuation of parent[i] < i.  Node i's row sees the      */
/* context and its ancestors and itself.  Up to ORC_TREE_MAX = 64 nodes.      */
/* ------------------------------------------------------------------------ */

/* ancestor-or-self masks; ORC_ST_BAD_TREE for a parent list that is not a
 * tree in topological order, ORC_ST_TOKEN_RANGE for a token outside [0, V) */
int orc_tree_masks(const int32_t* tokens, const int32_t* parent, int n, int vocab, uint64_t* mask) {
    if (n < 1 || n > ORC_TREE_MAX || parent[0] != -1) return ORC_ST_BAD_TREE;
    mask[0] = 1ull;
    for (int i = 1; i < n; ++i) {
        if (parent[i] < 0 || parent[i] >= i) return ORC_ST_BAD_TREE;
        if (tokens[i] < 0 || tokens[i] >= vocab) return ORC_ST_TOKEN_RANGE;
        mask[i] = mask[parent[i]] | (1ull << i);
    }
    return 0;
}

/* The greedy rule on a tree: the root is accepted; node i is accepted when
 * its parent is and tokens[i] equals the parent's argmax.  The deepest
 * accepted node (the lowest index among equals) ends the path root -> a;
 * L = depth(a) drafts accepted, next = idx[a].  path[0..L] = the nodes. */
void orc_tree_accept(const int32_t* idx, const int32_t* tokens, const int32_t* parent, int n,
                     int32_t* L, int32_t* next, int32_t* path) {
    int acc[ORC_TREE_MAX], depth[ORC_TREE_MAX];
    int best = 0;
    acc[0] = 1;
    depth[0] = 0;
    for (int i = 1; i < n; ++i) {
        acc[i] = acc[parent[i]] && tokens[i] == idx[parent[i]];
        depth[i] = depth[parent[i]] + 1;
        if (acc[i] && depth[i] > depth[best]) best = i;
    }
    *L = depth[best];
    *next = idx[best];
    int a = best;
    for (int d = depth[best]; d >= 0; --d) {
        path[d] = a;
        a = d > 0 ? parent[a] : a;
    }
}

/* move the K/V rows of block slots path[d] to slots d (d = 1..L), every layer */
void orc_kv_compact(const orc_cfg* c, orc_kv* kv, int n_past, const int32_t* path, int L) {
    size_t row = (size_t)c->head_dim;
    uint16_t* tmp = (uint16_t*)malloc(sizeof(uint16_t) * row * ORC_TREE_MAX);
    for (int l = 0; l < c->n_layers; ++l)
        for (int which = 0; which < 2; ++which)
            for (int g = 0; g < c->n_kv_heads; ++g) {
                for (int d = 1; d <= L; ++d) {              /* read all sources first */
                    int t = n_past + path[d];
                    int page = kv->page_table[t / c->page_size];
                    memcpy(tmp + (size_t)d * row, kv->pool + kv_index(c, page, l, which, g, t % c->page_size),
                           sizeof(uint16_t) * row);
                }
                for (int d = 1; d <= L; ++d) {
                    int t = n_past + d;
                    int page = kv->page_table[t / c->page_size];
                    memcpy(kv->pool + kv_index(c, page, l, which, g, t % c->page_size), tmp + (size_t)d * row,
                           sizeof(uint16_t) * row);
                }
            }
    free(tmp);
}

/* The tree verify step: res = {accepted_len, next_token, status, seq_len},
 * path[0..L] the accepted nodes.  The forward runs the n node rows with the
 * tree mask; the accepted path's K/V rows end at positions n_past .. n_past+L
 * and the KV is rolled back to n_past + L + 1.  A bad tree or token range is
 * reported before any work. */
int orc_verify_tree(const orc_cfg* c, const orc_weights* w, orc_kv* kv, const float* hidden,
                    const int32_t* tokens, const int32_t* parent, int n, int32_t* res, int32_t* path,
                    int32_t* idx, float* logits) {
    uint64_t mask[ORC_TREE_MAX];
    int n_past = *kv->seq_len;
    /* the rotary angle of a tree node follows its depth, not its row: not
     * modelled here, so a rotary configuration is refused */
    if (c->rope_theta > 0.f) return -1;
    res[0] = 0;
    res[1] = -1;
    res[3] = n_past;
    int st = orc_tree_masks(tokens, parent, n, c->vocab, mask);
    if (st) {
        res[2] = st;
        return 0;
    }
    st = orc_forward_tree(c, w, kv, hidden, n, mask, idx, logits, NULL);
    if (st & (ORC_ST_POOL_EMPTY | ORC_ST_CTX_FULL)) {
        res[2] = st;
        return 0;
    }
    if (st) {
        orc_kv_rollback(kv, n_past);
        res[2] = st;
        return 0;
    }
    int32_t L, next;
    orc_tree_accept(idx, tokens, parent, n, &L, &next, path);
    orc_kv_compact(c, kv, n_past, path, L);
    orc_kv_rollback(kv, n_past + L + 1);
    res[0] = L;
    res[1] = next;
    res[2] = 0;
    res[3] = *kv->seq_len;
    return 0;
}

/* Serial greedy decode ([TF] temp-0 token-fidelity gate): the same k+1 rows,
 * one forward per row, each appending its KV row before the next.  Row i+1 is
 * taken as the embedding of draft token i, so tokens[0..L] of a serial run
 * must equal the accepted drafts plus the next token of the batched step. */
int orc_serial_greedy(const orc_cfg* c, const orc_weights* w, orc_kv* kv, const float* hidden,
                      int k, int32_t* tokens) {
    int st = 0;
    for (int i = 0; i <= k; ++i) {
        int32_t t;
        st |= orc_forward(c, w, kv, hidden + (size_t)i * c->hidden, 1, &t, NULL, NULL);
        tokens[i] = t;
    }
    return st;
}
