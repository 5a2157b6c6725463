/*
 * CPU oracle for hybrid compressed attention (CSA + HCA): TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, scalar C in fp64.  It restates, step by step, what the method
 * computes, as described on the DeepSeek-V4 summary pages:
 *   - "CSA: 압축한 뒤, 필요한 기억만 골라서 보기" (honbul.tistory.com/221, CSA section):
 *     compress blocks of tokens, an indexer picks relevant blocks, top-k selection,
 *     a separate sliding window of recent raw tokens;
 *   - "HCA: 더 강하게 압축하고, 압축된 전체를 보기" (same page, HCA section):
 *     stronger compression, no sparse selection, attention over every compressed entry;
 *   - "4. CSA와 HCA를 결합한 하이브리드 어텐션" (pogovet.com DeepSeek-V4 article, detail 4):
 *     m=4 with softmax-gated pooling and a learned position bias, FP4 lightning indexer
 *     choosing the top-k compressed blocks per query, sliding-window branch; HCA with m=128
 *     attending densely over all compressed blocks;
 *   - "KV cache를 줄이는 방식" (honbul.tistory.com/221): compressed cache, window cache and
 *     tail state kept apart.
 * Numeric formats (OCP FP8 e4m3, OCP MX e2m1 with UE8M0 block scales) are written from their
 * public definitions.
 *
 * Only tests, the smoke check and the benchmark's CPU-baseline leg may load this library.
 * It shares no code, header or helper with the CUDA library.
 *
 * Storage dtype codes used in every signature: 0 = float32, 1 = bfloat16 (uint16 bits).
 */
#include <stdint.h>
#include <string.h>
#include <math.h>
#include <stdlib.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- scalar I/O */

static double bf16_bits_to_double(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* dtype 0 = float32, 1 = bfloat16 bits, 2 = float64 (dequantised values handed back in) */
static double load_elem(const void* p, int dtype, int64_t i) {
    if (dtype == 0) return (double)((const float*)p)[i];
    if (dtype == 2) return ((const double*)p)[i];
    return bf16_bits_to_double(((const uint16_t*)p)[i]);
}

/* Round a double to the nearest bfloat16 (ties to even), straight from the definition of
 * the format: 8 significant bits, exponent range of float32, gradual underflow below 2^-126. */
uint16_t oc_double_to_bf16(double x) {
    if (isnan(x)) return 0x7FC0;
    double a = fabs(x);
    int neg = signbit(x) ? 1 : 0;
    double y;
    if (a == 0.0) {
        y = 0.0;
    } else {
        int ex;
        frexp(a, &ex);                 /* a in [2^(ex-1), 2^ex) */
        int e_ulp = ex - 8;            /* 8 significant bits */
        if (e_ulp < -133) e_ulp = -133; /* subnormal spacing 2^-133 */
        double q = nearbyint(ldexp(a, -e_ulp));
        y = ldexp(q, e_ulp);
        if (y >= ldexp(1.0, 128)) y = INFINITY;
    }
    float f = (float)y;                /* exact: y is a bfloat16 value */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint16_t h = (uint16_t)(u >> 16);
    if (neg) h |= 0x8000;
    return h;
}

void oc_round_bf16(const double* in, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oc_double_to_bf16(in[i]);
}

void oc_round_f32(const double* in, int64_t n, float* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = (float)in[i];
}

/* ------------------------------------------------------- a1/a2: gated pooling */
/*
 * Softmax-gated pooling with a learned per-slot position bias (pogovet.com article,
 * detail 4; honbul.tistory.com/221 CSA and HCA sections).  Block j covers tokens
 * j*m .. j*m+m-1.  For slot i:  z_i = gate[j*m+i] + bias[i];  alpha = softmax(z);
 * out[j] = sum_i alpha_i * x[j*m+i].  One scalar gate per token; K and V share alpha.
 *
 * x: [n_blocks*m][d] in dtype x_dt;  out: [n_blocks][d] fp64;  alpha_out: [n_blocks][m] or NULL.
 */
void oc_pool(const void* x, int x_dt, const float* gate, const float* bias, int m,
             int64_t n_blocks, int d, double* out, double* alpha_out) {
    #pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n_blocks; ++j) {
        double z[512];
        double zmax = -INFINITY;
        for (int i = 0; i < m; ++i) {
            z[i] = (double)gate[j * m + i] + (double)bias[i];
            if (z[i] > zmax) zmax = z[i];
        }
        double zs = 0.0;
        for (int i = 0; i < m; ++i) { z[i] = exp(z[i] - zmax); zs += z[i]; }
        for (int i = 0; i < m; ++i) z[i] /= zs;
        if (alpha_out) for (int i = 0; i < m; ++i) alpha_out[j * m + i] = z[i];
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int i = 0; i < m; ++i) acc += z[i] * load_elem(x, x_dt, (j * m + i) * (int64_t)d + c);
            out[j * (int64_t)d + c] = acc;
        }
    }
}

/* ------------------------------------------------- a4: index-key quantisation */
/* OCP FP8 E4M3 (the "fn" variant): bias 7, 3 mantissa bits, max 448, no infinities,
 * S.1111.111 is NaN.  Values are rounded to nearest, ties to even, and saturate at 448. */
double oc_e4m3_decode(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 0xF, mant = c & 7;
    if (e == 0xF && mant == 7) return NAN;
    double v = (e == 0) ? ldexp((double)mant, -9) : ldexp(1.0 + mant / 8.0, e - 7);
    return s ? -v : v;
}

uint8_t oc_e4m3_encode(double y) {
    int neg = signbit(y) ? 1 : 0;
    double a = fabs(y);
    if (isnan(a) || a >= 448.0) a = 448.0;
    double q;
    if (a < ldexp(1.0, -6)) {
        q = nearbyint(ldexp(a, 9));                       /* subnormal grid, step 2^-9 */
        q = ldexp(q, -9);
    } else {
        int ex;
        frexp(a, &ex);                                    /* a in [2^(ex-1), 2^ex) */
        int e_ulp = (ex - 1) - 3;
        q = ldexp(nearbyint(ldexp(a, -e_ulp)), e_ulp);
    }
    if (q > 448.0) q = 448.0;
    uint8_t code;
    if (q == 0.0) {
        code = 0;
    } else if (q < ldexp(1.0, -6)) {
        code = (uint8_t)(int)ldexp(q, 9);                 /* exponent field 0 */
    } else {
        int ex;
        double f = frexp(q, &ex);                         /* q = f * 2^ex, f in [0.5,1) */
        int e = ex - 1;                                   /* q = (2f) * 2^e */
        int mant = (int)((2.0 * f - 1.0) * 8.0 + 0.5);
        code = (uint8_t)(((e + 7) << 3) | mant);
    }
    return (uint8_t)(code | (neg ? 0x80 : 0));
}

/* OCP MX E2M1: bias 1, 1 mantissa bit; magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}. */
double oc_e2m1_decode(uint8_t c) {
    int s = (c >> 3) & 1, e = (c >> 1) & 3, mant = c & 1;
    double v = (e == 0) ? 0.5 * mant : ldexp(1.0 + 0.5 * mant, e - 1);
    return s ? -v : v;
}

uint8_t oc_e2m1_encode(double y) {
    int neg = signbit(y) ? 1 : 0;
    double a = fabs(y);
    if (isnan(a)) a = 6.0;
    double ulp = (a < 2.0) ? 0.5 : (a < 4.0 ? 1.0 : 2.0);
    double q = nearbyint(a / ulp) * ulp;
    if (q > 6.0) q = 6.0;
    static const double mags[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    uint8_t code = 0;
    for (int i = 0; i < 8; ++i) if (mags[i] == q) code = (uint8_t)i;
    return (uint8_t)(code | (neg ? 8 : 0));
}

/* Per-row scale s = amax / 448 (float32 division; s = 1 when the row is all zero);
 * code = RNE_e4m3(x / s) with the division done in float32.  Dequantised key = s * code. */
void oc_quant_e4m3_rowscale(const void* x, int x_dt, int64_t rows, int d,
                            uint8_t* codes, float* scale) {
    for (int64_t r = 0; r < rows; ++r) {
        float amax = 0.0f;
        for (int c = 0; c < d; ++c) {
            float v = (float)load_elem(x, x_dt, r * d + c);
            if (fabsf(v) > amax) amax = fabsf(v);
        }
        float s = (amax > 0.0f) ? amax / 448.0f : 1.0f;
        scale[r] = s;
        for (int c = 0; c < d; ++c) {
            float v = (float)load_elem(x, x_dt, r * d + c);
            float yv = v / s;
            codes[r * d + c] = oc_e4m3_encode((double)yv);
        }
    }
}

/* Smallest integer e with amax <= 6 * 2^e (e = 0 for an all-zero block), clamped to the
 * UE8M0 range; stored as the biased byte e + 127. */
static int ue8m0_exponent(double amax) {
    if (!(amax > 0.0)) return 0;
    int ex;
    frexp(amax, &ex);
    int e = ex - 4;
    while (ldexp(6.0, e) < amax) ++e;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* Blocks of 32 consecutive values along the row share one UE8M0 scale 2^e;
 * code = RNE_e2m1(x * 2^-e) (exact scaling), saturating at 6.  Two codes per byte,
 * the even element in the low nibble. */
void oc_quant_e2m1_ue8m0(const void* x, int x_dt, int64_t rows, int d,
                         uint8_t* packed, uint8_t* scale_e8) {
    int nb = d / 32;
    for (int64_t r = 0; r < rows; ++r) {
        for (int b = 0; b < nb; ++b) {
            double amax = 0.0;
            for (int c = 0; c < 32; ++c) {
                double v = fabs(load_elem(x, x_dt, r * d + b * 32 + c));
                if (v > amax) amax = v;
            }
            int e = ue8m0_exponent(amax);
            scale_e8[r * nb + b] = (uint8_t)(e + 127);
            for (int c = 0; c < 32; c += 2) {
                uint8_t lo = oc_e2m1_encode(ldexp(load_elem(x, x_dt, r * d + b * 32 + c), -e));
                uint8_t hi = oc_e2m1_encode(ldexp(load_elem(x, x_dt, r * d + b * 32 + c + 1), -e));
                packed[(r * d + b * 32 + c) / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
}

/* Dequantised index keys, fp64.  fmt: 0 f32, 1 bf16, 2 e4m3 + fp32 row scale,
 * 3 e2m1 + UE8M0 per 32 values. */
void oc_dequant_keys(int fmt, const void* codes, const void* scales, int64_t rows, int d,
                     double* out) {
    for (int64_t r = 0; r < rows; ++r) {
        for (int c = 0; c < d; ++c) {
            double v;
            if (fmt == 0 || fmt == 1) {
                v = load_elem(codes, fmt, r * d + c);
            } else if (fmt == 2) {
                v = (double)((const float*)scales)[r] * oc_e4m3_decode(((const uint8_t*)codes)[r * d + c]);
            } else {
                uint8_t byte = ((const uint8_t*)codes)[(r * d + c) / 2];
                uint8_t code = (c & 1) ? (byte >> 4) : (byte & 0xF);
                int e = (int)((const uint8_t*)scales)[r * (d / 32) + c / 32] - 127;
                v = ldexp(oc_e2m1_decode(code), e);
            }
            out[r * d + c] = v;
        }
    }
}

/* ------------------------------- f2: FP8 compressed K/V with BF16 RoPE dimensions */
/*
 * "Most KV entries are stored in FP8 and only the RoPE dimensions in BF16" (pogovet.com
 * article, detail 5).  The pages fix neither the RoPE width, the FP8 variant nor the scale;
 * the reading taken: a row of d values keeps its last d_keep values (the RoPE dims of a K row;
 * none for a V row) in BF16, rounded to nearest even; every other value is OCP FP8 E4M3 with
 * one UE8M0 scale 2^e per 64 consecutive values, e = the smallest integer with
 * amax <= 448 * 2^e (e = 0 for an all-zero block, clamped to [-127, 127]), and
 * code = RNE_e4m3(x * 2^-e) -- exact scaling, so code * 2^e is the dequantised value and is
 * exactly a BF16 number.  The values are first rounded to float32, the precision the device
 * pools in, so both sides take every rounding decision on the same input.
 * x: [rows][d] fp64;  codes: [rows][d - d_keep];  scales: [rows][(d - d_keep) / 64] biased
 * bytes e + 127;  keep: [rows][d_keep] BF16 bits (unused when d_keep = 0).
 */
static int e4m3_block_exponent(double amax) {
    if (!(amax > 0.0)) return 0;
    int ex;
    frexp(amax, &ex);                                     /* amax in [2^(ex-1), 2^ex) */
    int e = ex - 10;                                      /* 448 * 2^(ex-10) < 2^(ex-1) */
    while (ldexp(448.0, e) < amax) ++e;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

void oc_quant_kv_fp8(const double* x, int64_t rows, int d, int d_keep, uint8_t* codes, uint8_t* scales,
                     uint16_t* keep) {
    const int dq = d - d_keep, nb = dq / 64;
    for (int64_t r = 0; r < rows; ++r) {
        for (int b = 0; b < nb; ++b) {
            double amax = 0.0;
            for (int c = 0; c < 64; ++c) {
                double v = fabs((double)(float)x[r * d + b * 64 + c]);
                if (v > amax) amax = v;
            }
            int e = e4m3_block_exponent(amax);
            scales[r * nb + b] = (uint8_t)(e + 127);
            for (int c = 0; c < 64; ++c)
                codes[r * dq + b * 64 + c] = oc_e4m3_encode(ldexp((double)(float)x[r * d + b * 64 + c], -e));
        }
        for (int c = 0; c < d_keep; ++c) keep[r * d_keep + c] = oc_double_to_bf16((double)(float)x[r * d + dq + c]);
    }
}

/* The dequantised rows, fp64: [rows][d]. */
void oc_dequant_kv_fp8(const uint8_t* codes, const uint8_t* scales, const uint16_t* keep, int64_t rows, int d,
                       int d_keep, double* out) {
    const int dq = d - d_keep, nb = dq / 64;
    for (int64_t r = 0; r < rows; ++r) {
        for (int c = 0; c < dq; ++c)
            out[r * d + c] = ldexp(oc_e4m3_decode(codes[r * dq + c]), (int)scales[r * nb + c / 64] - 127);
        for (int c = 0; c < d_keep; ++c) out[r * d + dq + c] = bf16_bits_to_double(keep[r * d_keep + c]);
    }
}

/* ------------------------------------------------------- a5: indexer scores */
/*
 * Lightning indexer score: I(t,s) = sum_h w[t,h] * max(0, q[t,h,:] . khat[s,:]).
 * One index key per compressed entry, shared by all indexer heads.
 * q: [T][H_I][d_I] (dtype q_dt); w: [T][H_I] fp32; khat: [N][d_I] fp64;
 * n_vis[t]: entries visible to query t (others get -inf).  S: [T][N] fp64.
 */
void oc_index_scores(const void* q, int q_dt, const float* w, int T, int H_I, int d_I,
                     const double* khat, int64_t N, const int64_t* n_vis, double* S) {
    #pragma omp parallel
    {
        double* qv = (double*)malloc(sizeof(double) * (size_t)H_I * d_I);
        #pragma omp for schedule(static)
        for (int t = 0; t < T; ++t) {
            for (int i = 0; i < H_I * d_I; ++i) qv[i] = load_elem(q, q_dt, (int64_t)t * H_I * d_I + i);
            for (int64_t s = 0; s < N; ++s) {
                if (s >= n_vis[t]) { S[(int64_t)t * N + s] = -INFINITY; continue; }
                double acc = 0.0;
                for (int h = 0; h < H_I; ++h) {
                    double dot = 0.0;
                    for (int c = 0; c < d_I; ++c) dot += qv[h * d_I + c] * khat[s * d_I + c];
                    if (dot > 0.0) acc += (double)w[(int64_t)t * H_I + h] * dot;
                }
                S[(int64_t)t * N + s] = acc;
            }
        }
        free(qv);
    }
}

/* ------------------------------------------------------------- a6: top-k */
typedef struct { double v; int64_t i; } oc_pair;

static int cmp_desc_then_index(const void* a, const void* b) {
    const oc_pair* x = (const oc_pair*)a;
    const oc_pair* y = (const oc_pair*)b;
    if (x->v > y->v) return -1;
    if (x->v < y->v) return 1;
    return (x->i < y->i) ? -1 : (x->i > y->i);
}

static int cmp_index(const void* a, const void* b) {
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

/* Top-k of the visible candidates of every row: order by score descending, equal scores
 * by lower index; output in ascending index order, padded with -1.  Scores are given in
 * fp64 (a float32 score tensor is passed through exactly). */
void oc_topk(const double* S, int64_t stride, int R, const int64_t* n_vis, int k, int32_t* idx) {
    #pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < R; ++r) {
        int64_t n = n_vis[r];
        oc_pair* p = (oc_pair*)malloc(sizeof(oc_pair) * (size_t)(n > 0 ? n : 1));
        for (int64_t s = 0; s < n; ++s) {
            double v = S[(int64_t)r * stride + s];
            p[s].v = (v == 0.0) ? 0.0 : v;    /* -0 and +0 compare equal */
            p[s].i = s;
        }
        qsort(p, (size_t)n, sizeof(oc_pair), cmp_desc_then_index);
        int take = (int)((n < k) ? n : k);
        int32_t* out = idx + (int64_t)r * k;
        for (int j = 0; j < take; ++j) out[j] = (int32_t)p[j].i;
        qsort(out, (size_t)take, sizeof(int32_t), cmp_index);
        for (int j = take; j < k; ++j) out[j] = -1;
        free(p);
    }
}

/* ------------------------------------------------------- a7/a8: attention */
/*
 * One joint softmax over the union of compressed rows and raw window rows (the window is
 * not de-duplicated against the compressed entries).  For each head h:
 *   s_i = scale * q[h,:] . key_i;   p = softmax(s);   o[h,:] = sum_i p_i value_i;
 *   lse[h] = log sum_i exp(s_i).
 * kc/vc: compressed rows [*][d] (dtype c_dt), selected by c_rows[0..n_c);
 * kw/vw: raw rows [*][d] (dtype w_dt), selected by w_rows[0..n_w).
 * q: [H][d] (q_dt).  o: [H][d] fp64; lse: [H] fp64.  An empty union gives o = 0, lse = -inf.
 */
void oc_attend(const void* q, int q_dt, int H, int d, double scale,
               const void* kc, const void* vc, int c_dt, const int64_t* c_rows, int64_t n_c,
               const void* kw, const void* vw, int w_dt, const int64_t* w_rows, int64_t n_w,
               double* o, double* lse) {
    int64_t n = n_c + n_w;
    #pragma omp parallel for schedule(static)
    for (int h = 0; h < H; ++h) {
        double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        double smax = -INFINITY;
        for (int64_t i = 0; i < n; ++i) {
            const void* kp = (i < n_c) ? kc : kw;
            int dt = (i < n_c) ? c_dt : w_dt;
            int64_t row = (i < n_c) ? c_rows[i] : w_rows[i - n_c];
            double dot = 0.0;
            for (int c = 0; c < d; ++c)
                dot += load_elem(q, q_dt, (int64_t)h * d + c) * load_elem(kp, dt, row * d + c);
            s[i] = scale * dot;
            if (s[i] > smax) smax = s[i];
        }
        double l = 0.0;
        for (int64_t i = 0; i < n; ++i) { s[i] = exp(s[i] - smax); l += s[i]; }
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int64_t i = 0; i < n; ++i) {
                const void* vp = (i < n_c) ? vc : vw;
                int dt = (i < n_c) ? c_dt : w_dt;
                int64_t row = (i < n_c) ? c_rows[i] : w_rows[i - n_c];
                acc += s[i] * load_elem(vp, dt, row * d + c);
            }
            o[(int64_t)h * d + c] = (n > 0) ? acc / l : 0.0;
        }
        lse[h] = (n > 0) ? smax + log(l) : -INFINITY;
        free(s);
    }
}

/* Exact log-sum-exp merge of S partial results (o_s normalised, lse_s), in the fixed order
 * s = 0..S-1:  lse = log sum_s exp(lse_s);  o = sum_s exp(lse_s - lse) * o_s.
 * o_parts: [S][H][d]; lse_parts: [S][H]. */
void oc_lse_merge(const double* o_parts, const double* lse_parts, int S, int H, int d,
                  double* o, double* lse) {
    for (int h = 0; h < H; ++h) {
        double mx = -INFINITY;
        for (int s = 0; s < S; ++s) if (lse_parts[s * H + h] > mx) mx = lse_parts[s * H + h];
        double tot = 0.0;
        for (int s = 0; s < S; ++s) if (lse_parts[s * H + h] > -INFINITY) tot += exp(lse_parts[s * H + h] - mx);
        double L = (tot > 0.0) ? mx + log(tot) : -INFINITY;
        lse[h] = L;
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int s = 0; s < S; ++s) {
                double ls = lse_parts[s * H + h];
                if (ls > -INFINITY) acc += exp(ls - L) * o_parts[((int64_t)s * H + h) * d + c];
            }
            o[(int64_t)h * d + c] = acc;
        }
    }
}

int oc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
