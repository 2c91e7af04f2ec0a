/*
 * csa_oracle.c -- CPU oracle for DeepSeek-V4's hybrid compressed attention.
 *
 * TEST INFRASTRUCTURE ONLY.  The CUDA library never loads, links or calls this
 * code.  Only the test-suite, the package smoke check and the benchmark's CPU
 * baseline leg use it.
 *
 * Plain and slow on purpose: every function follows the method's definition
 * step by step so that it can be checked against the sources by eye.
 * Attention is computed in fp64 from the dequantised cache.  Where floating
 * point decides a stored code (compressed entries, FP8/FP4 codes, indexer
 * scores that decide the top-k), the fp32 operation sequence is part of the
 * definition and is written out with one rounding per operation (compile
 * with -ffp-contract=off; fmaf only where written).
 *
 * Sources (page title, section):
 *  [XM]  xmsumi.com DeepSeek-V4 article -- "CSA（压缩稀疏注意力）",
 *        "HCA（重度压缩注意力）", "关键技术细节" (key technical details),
 *        and the heterogeneous KV cache paragraph under
 *        "百万Token 长上下文真实表现".
 *  [HU]  "DeepSeek-V4 — MoE nyelvmodellek milliós kontextussal"
 *        (hortopato.cc wiki) -- the CSA list (Tömörítés, Lightning Indexer,
 *        Sliding Window figyelem) and "Heavily Compressed Attention (HCA)".
 *  [ZC]  zcldvi.com DeepSeek-V4 news article -- FP4 indexer remark, the
 *        lossless FP4->FP8 remark and the sliding-window branch in both
 *        attentions.
 *  Where the pages leave a form open, the reading taken is stated at the
 *  function (the per-slot softmax with per-channel scale, power-of-two block
 *  scales, fp32 accumulation, tie order, joint softmax, RoPE position of an
 *  entry and its visibility rule).
 *  Number formats: OCP 8-bit floating point (E4M3) and OCP Microscaling
 *  (MX) v1.0 (E2M1 elements with UE8M0 block scales).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* threads                                                                   */
/* ------------------------------------------------------------------------ */
void orc_set_threads(int n) {
#ifdef _OPENMP
    omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int orc_get_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* RoPE table.  [XM] key technical details: rotary position encoding acts on  */
/* the last 64 dims of q and of the KV entries only.                          */
/* theta_i = base^(-2i/R), i < R/2; cos/sin of p*theta_i in fp64, stored as  */
/* the nearest fp32.  Pairs (2i, 2i+1) of the RoPE slice rotate by theta_i.  */
/* ------------------------------------------------------------------------ */
void orc_rope_table(int64_t P, int R, double base, float *cos_out, float *sin_out) {
    int half = R / 2;
    for (int64_t p = 0; p < P; ++p) {
        for (int i = 0; i < half; ++i) {
            double theta = pow(base, -2.0 * i / R);
            double a = (double)p * theta;
            cos_out[p * half + i] = (float)cos(a);
            sin_out[p * half + i] = (float)sin(a);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Project exponential (fp32), the step that turns compression logits into  */
/* weights.  Cody & Waite argument reduction by ln 2 split into a 16-bit     */
/* head and a tail, then the degree-7 Taylor polynomial of exp(r) in Horner  */
/* form with fma, then an exact scaling by 2^n.  Constants: log2(e) rounded  */
/* to fp32; ln 2 truncated to 16 fractional bits and its remainder rounded   */
/* to fp32; 1/k! rounded to fp32.  Returns 0 below -87 (the result would be  */
/* far below every weight that matters).  sexp(0) == 1 exactly.              */
/* ------------------------------------------------------------------------ */
static const float SX_LOG2E = 0x1.715476p+0f;
static const float SX_LN2_HI = 0x1.62e4p-1f;
static const float SX_LN2_LO = 0x1.7f7d1cp-20f;
static const float SX_C[8] = {
    0x1p+0f, 0x1p+0f, 0x1p-1f, 0x1.555556p-3f,
    0x1.555556p-5f, 0x1.111112p-7f, 0x1.6c16c2p-10f, 0x1.a01a02p-13f,
};

static float pow2i_f(int n) { /* 2^n as fp32 for n in [-126, 127] */
    uint32_t bits = (uint32_t)(n + 127) << 23;
    float f;
    memcpy(&f, &bits, 4);
    return f;
}

float orc_sexp(float x) {
    if (!(x >= -87.0f)) return 0.0f;
    if (x > 88.0f) x = 88.0f;
    float t = x * SX_LOG2E;
    float nf = nearbyintf(t);
    float r = fmaf(-nf, SX_LN2_HI, x);
    r = fmaf(-nf, SX_LN2_LO, r);
    float p = SX_C[7];
    for (int k = 6; k >= 0; --k) p = fmaf(p, r, SX_C[k]);
    return p * pow2i_f((int)nf);
}

/* ------------------------------------------------------------------------ */
/* OCP FP8 E4M3 (bias 7, no infinities, max finite 448): round to nearest,   */
/* ties to even, saturating to +-448.  The sign of the input is kept (a       */
/* negative value that rounds to zero gives 0x80).                           */
/* ------------------------------------------------------------------------ */
uint8_t orc_e4m3_encode(double x) {
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0) return sign | 0x7E;
    if (a < 0x1p-6) {                       /* subnormal binade: multiples of 2^-9 */
        double q = nearbyint(a * 512.0);    /* 0..8; 8 is the smallest normal */
        return sign | (uint8_t)q;
    }
    int E;
    frexp(a, &E);
    int ex = E - 1;                         /* a in [2^ex, 2^(ex+1)) */
    double q = nearbyint(ldexp(a, 3 - ex)); /* 8..16 */
    if (q == 16.0) { q = 8.0; ex += 1; }
    return sign | (uint8_t)(((ex + 7) << 3) | ((int)q - 8));
}

double orc_e4m3_decode(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    double v = (e == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    return s ? -v : v;
}

/* ------------------------------------------------------------------------ */
/* OCP E2M1 (FP4): magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}; nearest, ties to  */
/* the even code, saturating at 6; the sign of the input is kept.            */
/* ------------------------------------------------------------------------ */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

uint8_t orc_e2m1_encode(double x) {
    uint8_t sign = signbit(x) ? 8 : 0;
    double a = fabs(x);
    if (a >= 6.0) return sign | 7;
    int best = 0;
    double bd = a;
    for (int c = 1; c < 8; ++c) {
        double d = fabs(a - E2M1_MAG[c]);
        if (d < bd || (d == bd && (c & 1) == 0)) { best = c; bd = d; }
    }
    return sign | (uint8_t)best;
}

double orc_e2m1_decode(uint8_t c) {
    double v = E2M1_MAG[c & 7];
    return (c & 8) ? -v : v;
}

static float bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* nearest bf16, ties to even (inputs finite) */
static uint16_t f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t r = ((u >> 16) & 1u) + 0x7FFFu;
    return (uint16_t)((u + r) >> 16);
}

/* ------------------------------------------------------------------------ */
/* Block compression.  [XM] CSA: the KV entries of every m tokens are fused   */
/* into one compressed entry by a weighted sum; [HU] Tömörítés (m = 4);       */
/* [XM]/[HU] HCA: the same at m' = 128.                                      */
/* Reading taken: one learned logit per token; the weights of block j are     */
/* the softmax of its m logits, times a per-channel scale s_c (s == NULL     */
/* means s_c = 1).  fp32 sequence, per block j and channel c:                */
/*   mu = max_i z_i;  e_i = sexp(z_i - mu);  S = e_0 + e_1 + ... (in order);  */
/*   a_i = e_i / S;  acc = 0; acc = fma(a_i, x_{jm+i,c}, acc) for i = 0..m-1; */
/*   C_c = acc * s_c.                                                        */
/* Then the last R channels rotate at the block's last token position,       */
/* pos0 + jm + m - 1 (fp32, one rounding per product and per sum):           */
/*   y0 = x0*c - x1*s;  y1 = x0*s + x1*c.                                    */
/* Only complete blocks are produced: N = floor(T / m).                      */
/* x: fp32 [B, T, C]; z: [B, T]; out: fp32 [B, N, C].                         */
/* ------------------------------------------------------------------------ */
void orc_compress(const float *x, const float *z, const float *s, int64_t B, int64_t T, int C,
                  int m, int R, int64_t pos0, const float *rcos, const float *rsin,
                  int64_t rope_rows, float *out) {
    int64_t N = T / m;
    int half = R / 2;
    float *alpha = (float *)malloc(sizeof(float) * (size_t)m);
    float *e = (float *)malloc(sizeof(float) * (size_t)m);
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t j = 0; j < N; ++j) {
            const float *zb = z + b * T + j * m;
            float mu = zb[0];
            for (int i = 1; i < m; ++i) mu = fmaxf(mu, zb[i]);
            for (int i = 0; i < m; ++i) e[i] = orc_sexp(zb[i] - mu);
            float S = e[0];
            for (int i = 1; i < m; ++i) S = S + e[i];
            for (int i = 0; i < m; ++i) alpha[i] = e[i] / S;
            float *o = out + (b * N + j) * C;
            for (int c = 0; c < C; ++c) {
                float acc = 0.0f;
                for (int i = 0; i < m; ++i) acc = fmaf(alpha[i], x[(b * T + j * m + i) * C + c], acc);
                o[c] = acc * (s ? s[c] : 1.0f);
            }
            if (R > 0) {
                int64_t p = pos0 + j * m + m - 1;
                if (p < 0 || p >= rope_rows) abort();
                for (int i = 0; i < half; ++i) {
                    float cs = rcos[p * half + i], sn = rsin[p * half + i];
                    float x0 = o[C - R + 2 * i], x1 = o[C - R + 2 * i + 1];
                    float a0 = x0 * cs, a1 = x1 * sn, b0 = x0 * sn, b1 = x1 * cs;
                    o[C - R + 2 * i] = a0 - a1;
                    o[C - R + 2 * i + 1] = b0 + b1;
                }
            }
        }
    }
    free(alpha);
    free(e);
}

/* ------------------------------------------------------------------------ */
/* Block compression with per-channel logits (the other plain reading of     */
/* [XM] CSA's weighted sum: one learned logit per token and channel).  Each   */
/* channel c of block j takes its own softmax over the block's m logits       */
/* z_{jm+i, c}, with the fp32 sequence of orc_compress written per channel:   */
/*   mu_c = max_i z_{i,c};  e_i = sexp(z_{i,c} - mu_c);  S_c = e_0 + e_1 + ...*/
/*   (in order);  a_i = e_i / S_c;  acc = fma(a_i, x_{jm+i,c}, acc) over i;  */
/*   C_c = acc * s_c;  then the same RoPE of the last R channels.            */
/* With z_{t,c} equal across c this is orc_compress exactly.                 */
/* x: fp32 [B, T, C]; z: [B, T, C]; out: fp32 [B, N, C].                      */
/* ------------------------------------------------------------------------ */
void orc_compress_channel_logits(const float *x, const float *z, const float *s, int64_t B, int64_t T,
                                 int C, int m, int R, int64_t pos0, const float *rcos,
                                 const float *rsin, int64_t rope_rows, float *out) {
    int64_t N = T / m;
    int half = R / 2;
    float *e = (float *)malloc(sizeof(float) * (size_t)m);
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t j = 0; j < N; ++j) {
            float *o = out + (b * N + j) * C;
            for (int c = 0; c < C; ++c) {
                const float *zc = z + (b * T + j * m) * C + c;   /* z_{jm+i, c} = zc[i * C] */
                float mu = zc[0];
                for (int i = 1; i < m; ++i) mu = fmaxf(mu, zc[(int64_t)i * C]);
                for (int i = 0; i < m; ++i) e[i] = orc_sexp(zc[(int64_t)i * C] - mu);
                float S = e[0];
                for (int i = 1; i < m; ++i) S = S + e[i];
                float acc = 0.0f;
                for (int i = 0; i < m; ++i) acc = fmaf(e[i] / S, x[(b * T + j * m + i) * C + c], acc);
                o[c] = acc * (s ? s[c] : 1.0f);
            }
            if (R > 0) {
                int64_t p = pos0 + j * m + m - 1;
                if (p < 0 || p >= rope_rows) abort();
                for (int i = 0; i < half; ++i) {
                    float cs = rcos[p * half + i], sn = rsin[p * half + i];
                    float x0 = o[C - R + 2 * i], x1 = o[C - R + 2 * i + 1];
                    float a0 = x0 * cs, a1 = x1 * sn, b0 = x0 * sn, b1 = x1 * cs;
                    o[C - R + 2 * i] = a0 - a1;
                    o[C - R + 2 * i + 1] = b0 + b1;
                }
            }
        }
    }
    free(e);
}

/* ------------------------------------------------------------------------ */
/* Mixed FP8/BF16 cache row.  [XM] key technical details: the KV cache keeps  */
/* the RoPE dims in BF16 and the other dims in FP8, close to half the size  */
/* of a pure BF16 cache.  Row of D = 512 post-RoPE values (448 nope + 64     */
/* RoPE) -> 592 bytes:                                                       */
/*   [0, 448)   E4M3 codes of v_c * 2^-e_g, group g = c / 128 (4 groups:     */
/*              3 x 128 + 1 x 64 channels);                                  */
/*   [448, 576) 64 bf16 (little endian) of the RoPE dims, nearest-even;      */
/*   [576, 592) 4 fp32 group scales 2^e_g.                                   */
/* Reading taken: power-of-two scales, e_g = the smallest integer with        */
/* amax_g / 2^e_g <= 448 (with frexp(amax) = f 2^E: E-8 if f > 0.875 else    */
/* E-9), clamped to >= -126; amax_g == 0 gives e_g = 0.                      */
/* ------------------------------------------------------------------------ */
#define MX_D 512
#define MX_DN 448
#define MX_ROW 592

static int fp8_group_exp(float amax) {
    if (amax == 0.0f) return 0;
    int E;
    float f = frexpf(amax, &E);
    int e = (f > 0.875f) ? E - 8 : E - 9;
    return e < -126 ? -126 : e;
}

void orc_pack_mixed(const float *v, int64_t n, uint8_t *out) {
    for (int64_t r = 0; r < n; ++r) {
        const float *x = v + r * MX_D;
        uint8_t *o = out + r * MX_ROW;
        for (int g = 0; g < 4; ++g) {
            int lo = 128 * g, hi = lo + 128 < MX_DN ? lo + 128 : MX_DN;
            float amax = 0.0f;
            for (int c = lo; c < hi; ++c) amax = fmaxf(amax, fabsf(x[c]));
            int e = fp8_group_exp(amax);
            for (int c = lo; c < hi; ++c) o[c] = orc_e4m3_encode(ldexp((double)x[c], -e));
            float sc = (float)ldexp(1.0, e);
            memcpy(o + 576 + 4 * g, &sc, 4);
        }
        for (int c = MX_DN; c < MX_D; ++c) {
            uint16_t h = f32_to_bf16(x[c]);
            o[448 + 2 * (c - MX_DN)] = (uint8_t)(h & 0xFF);
            o[448 + 2 * (c - MX_DN) + 1] = (uint8_t)(h >> 8);
        }
    }
}

/* dequantised value of one mixed row, fp64 [512] */
static void unpack_mixed_row(const uint8_t *o, double *out) {
    float sc[4];
    memcpy(sc, o + 576, 16);
    for (int c = 0; c < MX_DN; ++c) out[c] = orc_e4m3_decode(o[c]) * (double)sc[c / 128];
    for (int c = MX_DN; c < MX_D; ++c) {
        uint16_t h = (uint16_t)(o[448 + 2 * (c - MX_DN)] | (o[448 + 2 * (c - MX_DN) + 1] << 8));
        out[c] = (double)bf16_to_f32(h);
    }
}

void orc_unpack_mixed(const uint8_t *rows, int64_t n, double *out) {
    for (int64_t r = 0; r < n; ++r) unpack_mixed_row(rows + r * MX_ROW, out + r * MX_D);
}

/* ------------------------------------------------------------------------ */
/* MXFP4 (OCP MX v1.0): blocks of 32 along the vector share a UE8M0 scale    */
/* X = 2^(floor(log2 amax) - 2) (emax of E2M1 is 2); byte = that exponent +  */
/* 127, clamped to >= 0; amax == 0 gives byte 127.  Elements are E2M1 of     */
/* x / X (saturating).  Two elements per byte, the even element in the low   */
/* nibble.  [XM] key technical details and [ZC]: the lightning indexer runs  */
/* its attention in FP4; the reading taken is E2M1 with power-of-two block   */
/* scales of 32, per the OCP MX format.                                      */
/* v: fp32 [n, d] -> codes [n, d/2], scales [n, d/32].                        */
/* ------------------------------------------------------------------------ */
void orc_mxfp4_quant(const float *v, int64_t n, int d, uint8_t *codes, uint8_t *scales) {
    int nb = d / 32;
    for (int64_t r = 0; r < n; ++r) {
        memset(codes + r * (d / 2), 0, (size_t)(d / 2));
        for (int b = 0; b < nb; ++b) {
            const float *x = v + r * d + 32 * b;
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
            int sx = 0;
            if (amax != 0.0f) {
                int E;
                frexpf(amax, &E);
                sx = E - 3;
                if (sx < -127) sx = -127;
            }
            scales[r * nb + b] = (uint8_t)(sx + 127);
            for (int i = 0; i < 32; ++i) {
                uint8_t c = orc_e2m1_encode(ldexp((double)x[i], -sx));
                int el = 32 * b + i;
                codes[r * (d / 2) + el / 2] |= (uint8_t)(c << (4 * (el & 1)));
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Lightning indexer scores and top-k.  [XM] CSA: a light "lightning         */
/* indexer" picks, for each query token, the top-k most relevant compressed  */
/* entries; [HU] Lightning Indexer (k = 1024 in V4-Pro); [XM] key technical  */
/* details: the indexer's internal attention runs in FP4.                    */
/* Reading taken: score(t, j) = sum over indexer heads h (ascending) of       */
/*   s = fma(w_{t,h}, relu(d_{t,h,j}), s), starting from s = +0, where       */
/*   d = the exact dot of the dequantised MXFP4 vectors, rounded once to     */
/*   fp32 (FP4 path), or d = fma(q_i, k_i, d) over i ascending from +0       */
/*   (fp32 path).  relu(d) = d > 0 ? d : +0.                                  */
/* Candidates: entry j is visible to the query at absolute position t iff    */
/* its block is complete, (j + 1) m - 1 <= t, and j < N.                     */
/* Order: score descending, then index ascending (-0 == +0).  Output the     */
/* first min(k, |visible|) indices in that order, then -1.                   */
/* ------------------------------------------------------------------------ */
typedef struct {
    float s;
    int32_t j;
} cand_t;

static int cand_cmp(const void *a, const void *b) {
    const cand_t *x = (const cand_t *)a, *y = (const cand_t *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->j > y->j) - (x->j < y->j);
}

/* exact dot of two dequantised MXFP4 vectors of length d, rounded once to fp32 */
float orc_mxfp4_dot(const uint8_t *qc, const uint8_t *qs, const uint8_t *kc, const uint8_t *ks,
                    int d) {
    long double acc = 0.0L;
    int nb = d / 32;
    int emin = 1 << 30, emax = -(1 << 30);
    for (int b = 0; b < nb; ++b) {
        long long P = 0; /* in units of 1/4: E2M1 values are multiples of 1/2 */
        for (int i = 32 * b; i < 32 * b + 32; ++i) {
            int cq = (qc[i / 2] >> (4 * (i & 1))) & 15;
            int ck = (kc[i / 2] >> (4 * (i & 1))) & 15;
            long long vq = (long long)(2.0 * orc_e2m1_decode((uint8_t)cq));
            long long vk = (long long)(2.0 * orc_e2m1_decode((uint8_t)ck));
            P += vq * vk;
        }
        int e = ((int)qs[b] - 127) + ((int)ks[b] - 127) - 2;
        if (P != 0) {
            if (e < emin) emin = e;
            if (e > emax) emax = e;
        }
        acc += ldexpl((long double)P, e);
    }
    /* |P| < 2^13; the 64-bit significand holds the sum exactly while the
     * exponents span at most 50 bits, so the cast below is the one rounding. */
    if (emax - emin > 50) abort();
    return (float)acc;
}

static void topk_emit(cand_t *c, int64_t nv, int k, int32_t *idx, float *sc) {
    qsort(c, (size_t)nv, sizeof(cand_t), cand_cmp);
    for (int r = 0; r < k; ++r) {
        idx[r] = r < nv ? c[r].j : -1;
        if (sc) sc[r] = r < nv ? c[r].s : -INFINITY;
    }
}

static int64_t n_visible(int64_t t, int m, int64_t N) {
    int64_t nv = (t + 1) / m;
    if (nv < 0) nv = 0;
    return nv < N ? nv : N;
}

/* qI: fp32 [B, Tq, HI, dI] (bf16 widened); w: [B, Tq, HI];
 * kc: [B, N, dI/2]; ks: [B, N, dI/32]; q_pos: [B, Tq];
 * idx_out: [B, Tq, k]; score_out (nullable): [B, Tq, k]. */
void orc_indexer_topk_fp4(const float *qI, const float *w, const uint8_t *kc, const uint8_t *ks,
                          const int64_t *q_pos, int64_t B, int64_t Tq, int HI, int dI, int64_t N,
                          int m, int k, int32_t *idx_out, float *score_out) {
    int nb = dI / 32;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bt = 0; bt < B * Tq; ++bt) {
        int64_t b = bt / Tq;
        int64_t t = q_pos[bt];
        int64_t nv = n_visible(t, m, N);
        uint8_t *qc = (uint8_t *)malloc((size_t)(HI * dI / 2));
        uint8_t *qs = (uint8_t *)malloc((size_t)(HI * nb));
        orc_mxfp4_quant(qI + bt * HI * dI, HI, dI, qc, qs);
        cand_t *c = (cand_t *)malloc(sizeof(cand_t) * (size_t)(nv > 0 ? nv : 1));
        for (int64_t j = 0; j < nv; ++j) {
            const uint8_t *kcj = kc + (b * N + j) * (dI / 2);
            const uint8_t *ksj = ks + (b * N + j) * nb;
            float s = 0.0f;
            for (int h = 0; h < HI; ++h) {
                float d = orc_mxfp4_dot(qc + h * (dI / 2), qs + h * nb, kcj, ksj, dI);
                float r = d > 0.0f ? d : 0.0f;
                s = fmaf(w[bt * HI + h], r, s);
            }
            c[j].s = s;
            c[j].j = (int32_t)j;
        }
        topk_emit(c, nv, k, idx_out + bt * k, score_out ? score_out + bt * k : NULL);
        free(c);
        free(qc);
        free(qs);
    }
}

/* ------------------------------------------------------------------------ */
/* FP8 indexer keys (the scope's next row: an FP4-query x FP8-key indexer).   */
/* [XM] "算力与内存效率": an FP4 x FP8 product runs at the FP8 x FP8 rate;    */
/* [ZC]: dequantising FP4 to FP8 is lossless (E4M3 holds every E2M1 value    */
/* times a power of two in its range).                                       */
/* Reading taken for the key format: E4M3 codes with one power-of-two scale  */
/* per block of 32 channels, the mixed cache's group rule -- the smallest     */
/* integer e with amax / 2^e <= 448 (no element saturates), 0 for an         */
/* all-zero block, clamped to >= -126 -- stored as a UE8M0 byte e + 127.      */
/* v: fp32 [n, d] -> codes [n, d] (one byte per element), scales [n, d/32].   */
/* ------------------------------------------------------------------------ */
void orc_fp8b32_quant(const float *v, int64_t n, int d, uint8_t *codes, uint8_t *scales) {
    int nb = d / 32;
    for (int64_t r = 0; r < n; ++r) {
        for (int b = 0; b < nb; ++b) {
            const float *x = v + r * d + 32 * b;
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
            int e = fp8_group_exp(amax);
            scales[r * nb + b] = (uint8_t)(e + 127);
            for (int i = 0; i < 32; ++i) codes[r * d + 32 * b + i] = orc_e4m3_encode(ldexp((double)x[i], -e));
        }
    }
}

/* Exact dot of a dequantised MXFP4 query head (qc, qs) with a dequantised   */
/* FP8 key (kc8: d E4M3 codes, ks8: d/32 scale bytes), rounded once to fp32. */
/* Per block b the integer P_b = sum_i (2 q_i / 2^eq) (512 k_i / 2^ek): twice */
/* an E2M1 value is an integer in [-12, 12] and 512 times an E4M3 value an   */
/* integer below 2^18, so |P_b| < 2^28 and the block's value is               */
/* P_b 2^(eq + ek - 10).  The two blocks are summed exactly in a 64-bit       */
/* significand (their exponents may differ by at most 36 here) and the cast  */
/* to fp32 is the one rounding.                                              */
float orc_fp4q_fp8k_dot(const uint8_t *qc, const uint8_t *qs, const uint8_t *kc8, const uint8_t *ks8, int d) {
    long double acc = 0.0L;
    int nb = d / 32;
    int emin = 1 << 30, emax = -(1 << 30);
    for (int b = 0; b < nb; ++b) {
        long long P = 0;
        for (int i = 32 * b; i < 32 * b + 32; ++i) {
            int cq = (qc[i / 2] >> (4 * (i & 1))) & 15;
            long long vq = (long long)(2.0 * orc_e2m1_decode((uint8_t)cq));
            long long vk = (long long)ldexp(orc_e4m3_decode(kc8[i]), 9);
            P += vq * vk;
        }
        int e = ((int)qs[b] - 127) + ((int)ks8[b] - 127) - 10;
        if (P != 0) {
            if (e < emin) emin = e;
            if (e > emax) emax = e;
        }
        acc += ldexpl((long double)P, e);
    }
    if (emax - emin > 36) abort();
    return (float)acc;
}

/* Lightning-indexer top-k with MXFP4 queries (quantised per head and 32-block */
/* exactly as orc_indexer_topk_fp4 does) and FP8 keys: the same head sum,      */
/* visibility rule and order, with d from orc_fp4q_fp8k_dot.                   */
/* kc8: [B, N, dI] codes; ks8: [B, N, dI/32] scale bytes.                      */
void orc_indexer_topk_fp4q_fp8k(const float *qI, const float *w, const uint8_t *kc8, const uint8_t *ks8,
                                const int64_t *q_pos, int64_t B, int64_t Tq, int HI, int dI, int64_t N,
                                int m, int k, int32_t *idx_out, float *score_out) {
    int nb = dI / 32;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bt = 0; bt < B * Tq; ++bt) {
        int64_t b = bt / Tq;
        int64_t nv = n_visible(q_pos[bt], m, N);
        uint8_t *qc = (uint8_t *)malloc((size_t)(HI * dI / 2));
        uint8_t *qs = (uint8_t *)malloc((size_t)(HI * nb));
        orc_mxfp4_quant(qI + bt * HI * dI, HI, dI, qc, qs);
        cand_t *c = (cand_t *)malloc(sizeof(cand_t) * (size_t)(nv > 0 ? nv : 1));
        for (int64_t j = 0; j < nv; ++j) {
            const uint8_t *kj = kc8 + (b * N + j) * dI;
            const uint8_t *sj = ks8 + (b * N + j) * nb;
            float s = 0.0f;
            for (int h = 0; h < HI; ++h) {
                float dd = orc_fp4q_fp8k_dot(qc + h * (dI / 2), qs + h * nb, kj, sj, dI);
                float r = dd > 0.0f ? dd : 0.0f;
                s = fmaf(w[bt * HI + h], r, s);
            }
            c[j].s = s;
            c[j].j = (int32_t)j;
        }
        topk_emit(c, nv, k, idx_out + bt * k, score_out ? score_out + bt * k : NULL);
        free(c);
        free(qc);
        free(qs);
    }
}

/* fp32 indexer: kI fp32 [B, N, dI] */
void orc_indexer_topk_f32(const float *qI, const float *w, const float *kI, const int64_t *q_pos,
                          int64_t B, int64_t Tq, int HI, int dI, int64_t N, int m, int k,
                          int32_t *idx_out, float *score_out) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bt = 0; bt < B * Tq; ++bt) {
        int64_t b = bt / Tq;
        int64_t nv = n_visible(q_pos[bt], m, N);
        cand_t *c = (cand_t *)malloc(sizeof(cand_t) * (size_t)(nv > 0 ? nv : 1));
        for (int64_t j = 0; j < nv; ++j) {
            const float *kj = kI + (b * N + j) * dI;
            float s = 0.0f;
            for (int h = 0; h < HI; ++h) {
                const float *qh = qI + (bt * HI + h) * dI;
                float d = 0.0f;
                for (int i = 0; i < dI; ++i) d = fmaf(qh[i], kj[i], d);
                float r = d > 0.0f ? d : 0.0f;
                s = fmaf(w[bt * HI + h], r, s);
            }
            c[j].s = s;
            c[j].j = (int32_t)j;
        }
        topk_emit(c, nv, k, idx_out + bt * k, score_out ? score_out + bt * k : NULL);
        free(c);
    }
}

/* ------------------------------------------------------------------------ */
/* Attention over compressed entries plus the sliding window.                */
/* [XM] CSA: multi-query attention over the selected entries only, with a    */
/* sliding-window branch kept for the nearest tokens; [HU] Sliding Window    */
/* figyelem (window 128); [ZC] both attentions add the window branch;        */
/* [XM]/[HU] HCA: dense attention over all compressed entries, no selection; */
/* [XM] key technical details: RoPE on the last 64 dims of q and KV, and the */
/* attention output gets the inverse rotation.                               */
/* Readings taken: all H heads share one KV (MQA) and the value is the key   */
/* entry itself (V = K, all D dims); the key set of the query at absolute    */
/* position t is {selected entries} (CSA, idx >= 0) or {visible entries}     */
/* (HCA: j < min(N, floor((t+1)/m))), together with the window tokens u,     */
/* t - W < u <= t, u >= 0, read from the window cache row u - swa_pos0[b];   */
/* one softmax over the union (an entry that also sits in the window is not  */
/* removed); logits = scale * (RoPE_t(q_h) . kappa); o_h = sum p kappa, then */
/* its last R dims rotate back by -t.  No keys: o = 0, lse = -inf.           */
/* Selected indices that are >= N or not yet visible are skipped and counted */
/* in *n_invalid, as are window rows outside the cache.                      */
/* q: fp32 [B, Tq, H, D]; cache / swa rows: fmt 0 = fp32 [.., D],            */
/* fmt 1 = mixed 592-byte rows (D = 512, R = 64); idx: [B, Tq, k] or NULL     */
/* for dense; out: fp64 [B, Tq, H, D]; lse (nullable): fp64 [B, Tq, H].      */
/* ------------------------------------------------------------------------ */
static void load_row(int fmt, const void *base, int64_t row, int D, double *out) {
    if (fmt == 0) {
        const float *r = (const float *)base + row * D;
        for (int c = 0; c < D; ++c) out[c] = (double)r[c];
    } else {
        unpack_mixed_row((const uint8_t *)base + row * MX_ROW, out);
    }
}

void orc_attention(const float *q, const int64_t *q_pos, int64_t B, int64_t Tq, int H, int D,
                   int R, int fmt, const void *cache, int64_t N, int m, const int32_t *idx, int k,
                   const void *swa, const int64_t *swa_pos0, int64_t Ts, int W, double scale,
                   const float *rcos, const float *rsin, int64_t rope_rows, double *out,
                   double *lse, int64_t *n_invalid) {
    int half = R / 2;
    int64_t bad_total = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad_total)
    for (int64_t bt = 0; bt < B * Tq; ++bt) {
        int64_t b = bt / Tq;
        int64_t t = q_pos[bt];
        if (t < 0 || t >= rope_rows) abort();
        int64_t cap = (idx ? k : n_visible(t, m, N)) + (W > 0 ? W : 0);
        double *keys = (double *)malloc(sizeof(double) * (size_t)(cap > 0 ? cap : 1) * D);
        int64_t nk = 0;
        if (idx) {
            for (int r = 0; r < k; ++r) {
                int32_t j = idx[bt * k + r];
                if (j < 0) continue;
                if (j >= N || (int64_t)(j + 1) * m - 1 > t) { bad_total++; continue; }
                load_row(fmt, cache, b * N + j, D, keys + nk * D);
                nk++;
            }
        } else {
            int64_t nv = n_visible(t, m, N);
            for (int64_t j = 0; j < nv; ++j) load_row(fmt, cache, b * N + j, D, keys + (nk++) * D);
        }
        for (int64_t u = t - W + 1; u <= t; ++u) {
            if (u < 0) continue;
            int64_t row = u - swa_pos0[b];
            if (row < 0 || row >= Ts) { bad_total++; continue; }
            load_row(fmt, swa, b * Ts + row, D, keys + (nk++) * D);
        }
        const float *cs = rcos + t * half, *sn = rsin + t * half;
        double *qr = (double *)malloc(sizeof(double) * D);
        double *lg = (double *)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
        for (int h = 0; h < H; ++h) {
            const float *qh = q + (bt * H + h) * D;
            for (int c = 0; c < D; ++c) qr[c] = (double)qh[c];
            for (int i = 0; i < half; ++i) {
                double x0 = qr[D - R + 2 * i], x1 = qr[D - R + 2 * i + 1];
                qr[D - R + 2 * i] = x0 * cs[i] - x1 * sn[i];
                qr[D - R + 2 * i + 1] = x0 * sn[i] + x1 * cs[i];
            }
            double *o = out + (bt * H + h) * D;
            for (int c = 0; c < D; ++c) o[c] = 0.0;
            if (nk == 0) {
                if (lse) lse[bt * H + h] = -INFINITY;
                continue;
            }
            double mx = -INFINITY;
            for (int64_t i = 0; i < nk; ++i) {
                double d = 0.0;
                for (int c = 0; c < D; ++c) d += qr[c] * keys[i * D + c];
                lg[i] = scale * d;
                if (lg[i] > mx) mx = lg[i];
            }
            double sum = 0.0;
            for (int64_t i = 0; i < nk; ++i) {
                double p = exp(lg[i] - mx);
                sum += p;
                for (int c = 0; c < D; ++c) o[c] += p * keys[i * D + c];
            }
            for (int c = 0; c < D; ++c) o[c] /= sum;
            for (int i = 0; i < half; ++i) {
                double x0 = o[D - R + 2 * i], x1 = o[D - R + 2 * i + 1];
                o[D - R + 2 * i] = x0 * cs[i] + x1 * sn[i];
                o[D - R + 2 * i + 1] = -x0 * sn[i] + x1 * cs[i];
            }
            if (lse) lse[bt * H + h] = mx + log(sum);
        }
        free(qr);
        free(lg);
        free(keys);
    }
    if (n_invalid) *n_invalid = bad_total;
}

/* ------------------------------------------------------------------------ */
/* array helpers for the Python wrapper                                      */
/* ------------------------------------------------------------------------ */
void orc_sexp_vec(const float *x, int64_t n, float *y) {
    for (int64_t i = 0; i < n; ++i) y[i] = orc_sexp(x[i]);
}

void orc_e4m3_encode_vec(const double *x, int64_t n, uint8_t *y) {
    for (int64_t i = 0; i < n; ++i) y[i] = orc_e4m3_encode(x[i]);
}

void orc_e2m1_encode_vec(const double *x, int64_t n, uint8_t *y) {
    for (int64_t i = 0; i < n; ++i) y[i] = orc_e2m1_encode(x[i]);
}
