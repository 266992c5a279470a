/*
 * oracle.c -- plain, slow, single-threaded fp64 CPU oracle of the DeepSeek-V4
 * hybrid attention layer (CSA + HCA + SWA, merged with a per-head sink).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline leg may load this library.  The product path
 * (the CUDA library) shares no code, header, table or constant with it.
 *
 * Every floating-point step runs in IEEE fp64 with libm sin/cos/exp/log/pow.
 * Inputs are read as the same bf16 (uint16 storage) bytes the GPU reads,
 * widened exactly to fp64.  Loops follow the definitions literally: no
 * blocking, no fusion, no partial-select tricks.
 *
 * Sources (web pages on DeepSeek-V4, cited by title and section):
 *  [DD]  "Why DeepSeek V4 Stands Apart: A Deep Dive into Its Architecture and
 *        Performance", section "Core Architectural Innovations": SWA over the
 *        most recent 128 tokens; CSA compresses KV 4x (m=4) then keeps the
 *        top-1024 (Pro) / top-512 (Flash) entries per query; HCA compresses
 *        128:1 and attends densely to the compressed entries.
 *  [AT]  "DeepSeek-V4" (atlas spec sheet), section "Design overview": CSA
 *        compresses every 4 tokens into two overlapping streams and applies the
 *        V3.2 lightning-indexer top-k; RMSNorm on queries and on compressed KV
 *        entries; section "Spec sheet / Core block": partial RoPE, QK-norm,
 *        attention sinks; "Provenance references" items 16-18: RoPE on the last
 *        64 dims with inverse RoPE on outputs, RMSNorm on q and compressed KV,
 *        designed attention sinks; section "Inference efficiency": shared-KV MQA.
 *
 * Readings adopted where the pages are silent:
 *  - entry j of C(m,w) pools tokens u in [m(j+1)-w, m(j+1)-1], u >= 0, with
 *    weights softmax(gate_u) over the existing tokens (CSA: m=4, w=8, i.e. the
 *    8 tokens [4j-4, 4j+4));
 *  - the pooled vector is RMSNorm'd (eps, gamma) then RoPE'd at position
 *    m(j+1)-1; the indexer key is pooled with the same weights, no norm/RoPE;
 *  - entry j is visible to a query at position t iff m(j+1)-1 <= t;
 *  - indexer score I(t,j) = sum_h w[t,h] * max(0, qI[t,h] . kI[j]);
 *  - top-k keeps the min(k, visible) largest scores, ties to the smaller j;
 *  - logits s * q~ . k~ with s = 1/sqrt(D); values V = K~ (shared latent);
 *  - RoPE: interleaved pairs (d0+2i, d0+2i+1), d0 = D-r, angle p*base^(-2i/r);
 *  - merge: Z = sum_b exp(lse_b) + exp(sink_h); out = sum_b exp(lse_b) o_b / Z,
 *    then the last r dims are rotated back by the query position;
 *  - low-precision indexer path (optional): keys and query rows as E4M3 codes
 *    with one fp32 scale amax/448 per row, dequantised before the score;
 *  - MXFP4 indexer rows (optional): E2M1 codes in blocks of 32 along the
 *    head dim, each block with an E8M0 scale 2^(floor(log2 amax) - 2).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL 1
#define ORC_ENOMEM 2

/* ------------------------------------------------------------------ */
/* bf16 <-> fp64                                                       */
/* ------------------------------------------------------------------ */

/* Exact widening: a bf16 value is the upper half of an fp32 value. */
double orc_bf16_to_f64(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round an fp64 value to the nearest bf16 (ties to even), in one step (no
 * double rounding through fp32).  bf16: 8 significant bits, fp32 exponent
 * range, subnormal spacing 2^-133. */
uint16_t orc_f64_to_bf16(double x) {
    if (isnan(x)) return (uint16_t)0x7FC0;
    if (x == 0.0) return signbit(x) ? (uint16_t)0x8000 : (uint16_t)0x0000;
    double ax = fabs(x);
    int e;
    frexp(ax, &e);               /* ax = f * 2^e, f in [0.5, 1) */
    int q = e - 8;               /* spacing of 8-significant-bit numbers */
    if (q < -133) q = -133;      /* subnormal range */
    double scaled = ldexp(ax, -q);
    double r = nearbyint(scaled);    /* default mode: round half to even */
    double v = ldexp(r, q);
    /* largest finite bf16 is (2 - 2^-7) * 2^127 */
    if (v > ldexp(2.0 - ldexp(1.0, -7), 127)) v = INFINITY;
    float f = (float)(signbit(x) ? -v : v);  /* exact: v is a bf16 value */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

void orc_bf16_array_to_f64(const uint16_t* in, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_f64(in[i]);
}

void orc_f64_array_to_bf16(const double* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f64_to_bf16(in[i]);
}

/* ------------------------------------------------------------------ */
/* RMSNorm and partial RoPE  ([AT] "Design overview"; provenance 16-17) */
/* ------------------------------------------------------------------ */

/* x <- x / sqrt(mean(x^2) + eps) * gamma  over all D entries. */
void orc_rmsnorm(double* x, int D, const float* gamma, double eps) {
    double ss = 0.0;
    for (int d = 0; d < D; ++d) ss += x[d] * x[d];
    double inv = 1.0 / sqrt(ss / (double)D + eps);
    for (int d = 0; d < D; ++d) {
        double g = gamma ? (double)gamma[d] : 1.0;
        x[d] = x[d] * inv * g;
    }
}

/* Rotate the last r dims of x in interleaved pairs (d0+2i, d0+2i+1),
 * d0 = D - r, by the angle sign * p * base^(-2i/r). */
void orc_rope(double* x, int D, int r, double base, int64_t p, int sign) {
    int d0 = D - r;
    for (int i = 0; i < r / 2; ++i) {
        double theta = pow(base, -2.0 * (double)i / (double)r);
        double phi = (double)sign * (double)p * theta;
        double c = cos(phi), s = sin(phi);
        double a = x[d0 + 2 * i], b = x[d0 + 2 * i + 1];
        x[d0 + 2 * i] = a * c - b * s;
        x[d0 + 2 * i + 1] = a * s + b * c;
    }
}

/* ------------------------------------------------------------------ */
/* Compressor C(m, w)  ([DD] "Core Architectural Innovations": m=4 for  */
/* CSA, 128:1 for HCA; [AT] "Design overview": every 4 tokens into two  */
/* overlapping streams; RMSNorm on compressed KV entries)               */
/* ------------------------------------------------------------------ */

/*
 * For each sequence b and entry j in [j_begin, j_end):
 *   S_j   = { u : m(j+1)-w <= u <= m(j+1)-1, u >= 0 }
 *   a_u   = exp(g_u) / sum_{v in S_j} exp(g_v)
 *   c_j   = sum_u a_u kv_raw[u]          -> RMSNorm(gamma, eps) -> RoPE at m(j+1)-1
 *   kI_j  = sum_u a_u ik_raw[u]          (no norm, no RoPE)
 * kv_raw [B][L_cap][D], ik_raw [B][L_cap][dI] (may be NULL), gate [B][L_cap].
 * Outputs are fp64: kv_out [B][nj][D], ik_out [B][nj][dI] (may be NULL),
 * alpha_out [B][nj][w] (may be NULL; slot s holds the weight of token
 * m(j+1)-w+s, 0 for tokens that do not exist).
 */
int orc_compress(const uint16_t* kv_raw, const uint16_t* ik_raw, const uint16_t* gate,
                 const float* gamma, int B, int64_t L_cap, int D, int dI, int m, int w,
                 int r, double base, double eps, int64_t j_begin, int64_t j_end,
                 double* kv_out, double* ik_out, double* alpha_out) {
    if (B <= 0 || L_cap <= 0 || D <= 0 || m <= 0 || w <= 0 || r < 0 || r > D || (r % 2) ||
        j_begin < 0 || j_end < j_begin)
        return ORC_EINVAL;
    if ((int64_t)m * j_end > L_cap) return ORC_EINVAL; /* last token m*j_end-1 must exist */
    int64_t nj = j_end - j_begin;
    double* alpha = (double*)malloc(sizeof(double) * (size_t)w);
    double* acc = (double*)malloc(sizeof(double) * (size_t)D);
    double* acc_i = (double*)malloc(sizeof(double) * (size_t)(dI > 0 ? dI : 1));
    if (!alpha || !acc || !acc_i) {
        free(alpha); free(acc); free(acc_i);
        return ORC_ENOMEM;
    }
    for (int b = 0; b < B; ++b) {
        for (int64_t j = j_begin; j < j_end; ++j) {
            int64_t u0 = (int64_t)m * (j + 1) - w; /* first token of the window */
            /* softmax of the gate logits over the tokens that exist */
            double gmax = -INFINITY;
            for (int s = 0; s < w; ++s) {
                int64_t u = u0 + s;
                if (u < 0) continue;
                double g = orc_bf16_to_f64(gate[(int64_t)b * L_cap + u]);
                if (g > gmax) gmax = g;
            }
            double z = 0.0;
            for (int s = 0; s < w; ++s) {
                int64_t u = u0 + s;
                if (u < 0) { alpha[s] = 0.0; continue; }
                double g = orc_bf16_to_f64(gate[(int64_t)b * L_cap + u]);
                alpha[s] = exp(g - gmax);
                z += alpha[s];
            }
            for (int s = 0; s < w; ++s) alpha[s] /= z;
            /* weighted sums */
            for (int d = 0; d < D; ++d) acc[d] = 0.0;
            for (int d = 0; d < dI; ++d) acc_i[d] = 0.0;
            for (int s = 0; s < w; ++s) {
                int64_t u = u0 + s;
                if (u < 0) continue;
                const uint16_t* row = kv_raw + ((int64_t)b * L_cap + u) * D;
                for (int d = 0; d < D; ++d) acc[d] += alpha[s] * orc_bf16_to_f64(row[d]);
                if (ik_raw && dI > 0) {
                    const uint16_t* irow = ik_raw + ((int64_t)b * L_cap + u) * dI;
                    for (int d = 0; d < dI; ++d) acc_i[d] += alpha[s] * orc_bf16_to_f64(irow[d]);
                }
            }
            orc_rmsnorm(acc, D, gamma, eps);
            orc_rope(acc, D, r, base, (int64_t)m * (j + 1) - 1, +1);
            int64_t o = (int64_t)b * nj + (j - j_begin);
            memcpy(kv_out + o * D, acc, sizeof(double) * (size_t)D);
            if (ik_out && dI > 0) memcpy(ik_out + o * dI, acc_i, sizeof(double) * (size_t)dI);
            if (alpha_out) memcpy(alpha_out + o * w, alpha, sizeof(double) * (size_t)w);
        }
    }
    free(alpha); free(acc); free(acc_i);
    return ORC_OK;
}

/*
 * C(m, w) of projected hidden states ("Why DeepSeek V4 Stands Apart",
 * section "Core Architectural Innovations": the compressor that turns the
 * per-token KV into compressed entries, here fed from the hidden states).
 * Each token's KV and indexer-key row is the projection x_u . W of its
 * hidden state, in fp64 without rounding: W [dm][D + dI] bf16 holds the KV
 * columns, then the indexer-key columns.  The entries then follow
 * orc_compress: gate-softmax pooling of the window's projected rows, RMSNorm
 * and RoPE of the KV part.  x [B][L_cap][dm] bf16.
 */
int orc_compress_hidden(const uint16_t* x, const uint16_t* W, const uint16_t* gate,
                        const float* gamma, int B, int64_t L_cap, int dm, int D, int dI, int m,
                        int w, int r, double base, double eps, int64_t j_begin, int64_t j_end,
                        double* kv_out, double* ik_out) {
    if (B <= 0 || L_cap <= 0 || dm <= 0 || D <= 0 || dI < 0 || m <= 0 || w <= 0 || r < 0 ||
        r > D || (r % 2) || j_begin < 0 || j_end < j_begin)
        return ORC_EINVAL;
    if ((int64_t)m * j_end > L_cap) return ORC_EINVAL;
    const int P = D + dI;
    int64_t nj = j_end - j_begin;
    double* alpha = (double*)malloc(sizeof(double) * (size_t)w);
    double* acc = (double*)malloc(sizeof(double) * (size_t)P);
    double* proj = (double*)malloc(sizeof(double) * (size_t)P);
    double* Wd = (double*)malloc(sizeof(double) * (size_t)dm * P);
    if (!alpha || !acc || !proj || !Wd) {
        free(alpha); free(acc); free(proj); free(Wd);
        return ORC_ENOMEM;
    }
    for (int64_t i = 0; i < (int64_t)dm * P; ++i) Wd[i] = orc_bf16_to_f64(W[i]);
    for (int b = 0; b < B; ++b) {
        for (int64_t j = j_begin; j < j_end; ++j) {
            int64_t u0 = (int64_t)m * (j + 1) - w;
            double gmax = -INFINITY;
            for (int s = 0; s < w; ++s) {
                int64_t u = u0 + s;
                if (u < 0) continue;
                double g = orc_bf16_to_f64(gate[(int64_t)b * L_cap + u]);
                if (g > gmax) gmax = g;
            }
            double z = 0.0;
            for (int s = 0; s < w; ++s) {
                int64_t u = u0 + s;
                if (u < 0) { alpha[s] = 0.0; continue; }
                alpha[s] = exp(orc_bf16_to_f64(gate[(int64_t)b * L_cap + u]) - gmax);
                z += alpha[s];
            }
            for (int s = 0; s < w; ++s) alpha[s] /= z;
            for (int c = 0; c < P; ++c) acc[c] = 0.0;
            for (int s = 0; s < w; ++s) {
                int64_t u = u0 + s;
                if (u < 0) continue;
                /* the token's projected row */
                const uint16_t* xr = x + ((int64_t)b * L_cap + u) * dm;
                for (int c = 0; c < P; ++c) proj[c] = 0.0;
                for (int i = 0; i < dm; ++i) {
                    double xi = orc_bf16_to_f64(xr[i]);
                    const double* wr = Wd + (int64_t)i * P;
                    for (int c = 0; c < P; ++c) proj[c] += xi * wr[c];
                }
                for (int c = 0; c < P; ++c) acc[c] += alpha[s] * proj[c];
            }
            orc_rmsnorm(acc, D, gamma, eps);
            orc_rope(acc, D, r, base, (int64_t)m * (j + 1) - 1, +1);
            int64_t o = (int64_t)b * nj + (j - j_begin);
            memcpy(kv_out + o * D, acc, sizeof(double) * (size_t)D);
            if (ik_out && dI > 0) memcpy(ik_out + o * dI, acc + D, sizeof(double) * (size_t)dI);
        }
    }
    free(alpha); free(acc); free(proj); free(Wd);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Lightning indexer score and top-k  ([DD] "Core Architectural         */
/* Innovations": top-1024 / top-512 entries per query; [AT] "Design     */
/* overview": the V3.2 lightning-indexer sparse attention)              */
/* ------------------------------------------------------------------ */

/* Number of compressed entries visible to a query at position t. */
int64_t orc_visible(int64_t t, int m) { return t < 0 ? 0 : (t + 1) / m; }

/*
 * scores[b][t][j] = sum_h w[b][t][h] * max(0, sum_d iq[b][t][h][d] * ik[b][j][d])
 * for j < min(visible(pos[b][t]), N_cap); entries beyond are set to NaN.
 * iq [B][T][HI][dI] bf16, w [B][T][HI] fp32, ik [B][N_cap][dI] bf16, pos [B][T].
 */
int orc_indexer_scores(const uint16_t* iq, const float* w, const uint16_t* ik, const int32_t* pos,
                       int B, int T, int HI, int dI, int64_t N_cap, int m, double* scores) {
    if (B <= 0 || T <= 0 || HI <= 0 || dI <= 0 || N_cap < 0 || m <= 0) return ORC_EINVAL;
    for (int b = 0; b < B; ++b) {
        for (int t = 0; t < T; ++t) {
            int64_t bt = (int64_t)b * T + t;
            int64_t n = orc_visible(pos[bt], m);
            if (n > N_cap) n = N_cap;
            double* out = scores + bt * N_cap;
            for (int64_t j = 0; j < N_cap; ++j) out[j] = NAN;
            for (int64_t j = 0; j < n; ++j) {
                const uint16_t* kj = ik + ((int64_t)b * N_cap + j) * dI;
                double s = 0.0;
                for (int h = 0; h < HI; ++h) {
                    const uint16_t* qh = iq + (bt * HI + h) * dI;
                    double dot = 0.0;
                    for (int d = 0; d < dI; ++d) dot += orc_bf16_to_f64(qh[d]) * orc_bf16_to_f64(kj[d]);
                    s += (double)w[bt * HI + h] * (dot > 0.0 ? dot : 0.0);
                }
                out[j] = s;
            }
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* FP8 indexer keys  ("DeepSeek-V4" atlas spec sheet, section           */
/* "Inference efficiency": the indexer QK path is quantised to low      */
/* precision).  The pages do not fix the format; the reading here is    */
/* OCP FP8 E4M3 codes with one fp32 scale per 128-dim row.              */
/* ------------------------------------------------------------------ */

/* E4M3 ("fn" variant): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits;
 * no infinities, code S.1111.111 is NaN, largest finite 1.75 * 2^8 = 448,
 * subnormals m * 2^-9 for m = 1..7. */
double orc_e4m3_to_f64(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* Nearest E4M3 value to an fp32 value (ties to the even code), with values
 * beyond 448 in magnitude clamped to 448 (saturating). */
uint8_t orc_f32_to_e4m3(float x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    int e;
    frexp(a, &e);                 /* a = f * 2^e, f in [0.5, 1) */
    int q = e - 4;                /* spacing of 4-significant-bit numbers */
    if (q < -9) q = -9;           /* subnormal spacing */
    double r = nearbyint(ldexp(a, -q));   /* units of 2^q, half to even */
    /* r * 2^q is exactly representable; the code is its bit pattern */
    double v = ldexp(r, q);
    if (v == 0.0) return sign;
    int ev;
    frexp(v, &ev);
    int E = ev - 1 + 7;           /* biased exponent of v = 1.m * 2^(ev-1) */
    uint8_t code;
    if (E <= 0) code = (uint8_t)ldexp(v, 9);                 /* subnormal: m */
    else code = (uint8_t)((E << 3) | ((int)(ldexp(v, -(ev - 1)) * 8.0) - 8));
    return (uint8_t)(sign | code);
}

/* One row of n bf16 values to E4M3 codes and a scale, in fp32 arithmetic:
 * amax = max |x|; inv = 448 / amax; code_i = e4m3(x_i * inv); the row
 * decodes as code_i * scale with scale = amax / 448.  A zero row gives
 * zero codes and scale 0. */
void orc_quantize_e4m3_row(const uint16_t* x, int n, uint8_t* codes, float* scale) {
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf((float)orc_bf16_to_f64(x[i]));
        if (a > amax) amax = a;
    }
    if (!(amax > 0.0f)) {
        for (int i = 0; i < n; ++i) codes[i] = 0;
        *scale = 0.0f;
        return;
    }
    float inv = 448.0f / amax;
    for (int i = 0; i < n; ++i) codes[i] = orc_f32_to_e4m3((float)orc_bf16_to_f64(x[i]) * inv);
    *scale = amax / 448.0f;
}

void orc_quantize_e4m3_rows(const uint16_t* x, int64_t rows, int n, uint8_t* codes,
                            float* scales) {
    for (int64_t r = 0; r < rows; ++r)
        orc_quantize_e4m3_row(x + r * n, n, codes + r * n, scales + r);
}

/*
 * Indexer scores with FP8 keys: the keys arrive as codes ik8 [B][N_cap][dI]
 * with scales iks [B][N_cap]; each query row iq[b][t][h] (bf16) is quantised
 * the same way; both are dequantised to fp64 and the score is the plain
 * definition sum_h w[t,h] * max(0, q^[t,h] . k^[j]).  NaN past the visible
 * entries.
 */
int orc_indexer_scores_e4m3(const uint16_t* iq, const float* w, const uint8_t* ik8,
                            const float* iks, const int32_t* pos, int B, int T, int HI, int dI,
                            int64_t N_cap, int m, double* scores) {
    if (B <= 0 || T <= 0 || HI <= 0 || dI <= 0 || N_cap < 0 || m <= 0) return ORC_EINVAL;
    uint8_t* qc = (uint8_t*)malloc((size_t)HI * dI);
    float* qs = (float*)malloc(sizeof(float) * (size_t)HI);
    double* qd = (double*)malloc(sizeof(double) * (size_t)HI * dI);
    double* kd = (double*)malloc(sizeof(double) * (size_t)dI);
    if (!qc || !qs || !qd || !kd) { free(qc); free(qs); free(qd); free(kd); return ORC_ENOMEM; }
    for (int b = 0; b < B; ++b) {
        for (int t = 0; t < T; ++t) {
            int64_t bt = (int64_t)b * T + t;
            for (int h = 0; h < HI; ++h) {
                orc_quantize_e4m3_row(iq + (bt * HI + h) * dI, dI, qc + (size_t)h * dI, qs + h);
                for (int d = 0; d < dI; ++d)
                    qd[(size_t)h * dI + d] = orc_e4m3_to_f64(qc[(size_t)h * dI + d]) * (double)qs[h];
            }
            int64_t n = orc_visible(pos[bt], m);
            if (n > N_cap) n = N_cap;
            double* out = scores + bt * N_cap;
            for (int64_t j = 0; j < N_cap; ++j) out[j] = NAN;
            for (int64_t j = 0; j < n; ++j) {
                const uint8_t* kj = ik8 + ((int64_t)b * N_cap + j) * dI;
                double sk = (double)iks[(int64_t)b * N_cap + j];
                for (int d = 0; d < dI; ++d) kd[d] = orc_e4m3_to_f64(kj[d]) * sk;
                double s = 0.0;
                for (int h = 0; h < HI; ++h) {
                    double dot = 0.0;
                    for (int d = 0; d < dI; ++d) dot += qd[(size_t)h * dI + d] * kd[d];
                    s += (double)w[bt * HI + h] * (dot > 0.0 ? dot : 0.0);
                }
                out[j] = s;
            }
        }
    }
    free(qc); free(qs); free(qd); free(kd);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* MXFP4 indexer rows                                                  */
/* ------------------------------------------------------------------ */

/* "DeepSeek-V4" atlas spec sheet, section "Inference efficiency": the indexer
 * QK path is trained for FP4 (MXFP4); "Why DeepSeek V4 Stands Apart",
 * section "Core Architectural Innovations" (FP4 quantization-aware
 * training): the FP4 elements are E2M1.  MXFP4 is the OCP
 * Microscaling format: E2M1 elements, 32 consecutive elements sharing one
 * power-of-two scale stored as E8M0.
 *
 * E2M1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit, no Inf or NaN;
 * exponent field 0 is subnormal (m * 0.5), so the magnitudes are
 * 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double orc_e2m1_to_f64(uint8_t c) {
    int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

/* Nearest E2M1 code to y (ties to the even code), magnitudes beyond 6
 * clamped to 6; a result of zero is encoded +0 whatever the sign of y. */
uint8_t orc_f64_to_e2m1(double y) {
    double a = fabs(y);
    uint8_t code;
    if (a >= 6.0) {
        code = 7;
    } else {
        int e;
        frexp(a, &e);              /* a = f * 2^e, f in [0.5, 1) */
        int q = e - 2;             /* spacing of 2-significant-bit numbers */
        if (q < -1) q = -1;        /* subnormal spacing 0.5 */
        double v = ldexp(nearbyint(ldexp(a, -q)), q);   /* half to even */
        if (v == 0.0) return 0;
        if (v == 0.5) {
            code = 1;
        } else {
            int ev;
            frexp(v, &ev);         /* v = 1.m * 2^(ev-1), biased exponent ev */
            code = (uint8_t)((ev << 1) | (int)((ldexp(v, -(ev - 1)) - 1.0) * 2.0));
        }
    }
    return (uint8_t)((signbit(y) ? 8 : 0) | code);
}

/* E8M0 scale code c stands for 2^(c - 127); c = 255 is NaN. */
double orc_e8m0_to_f64(uint8_t c) { return c == 255 ? NAN : ldexp(1.0, (int)c - 127); }

/* The block's scale exponent: floor(log2(amax)) minus the largest E2M1
 * exponent (2), so amax / X lies in [4, 8); clamped to E8M0's range
 * [-127, 127].  An all-zero block takes the smallest scale. */
static int orc_mx_scale_exp(double amax) {
    if (!(amax > 0.0)) return -127;
    int e;
    frexp(amax, &e);               /* floor(log2(amax)) = e - 1 */
    int s = e - 1 - 2;
    return s < -127 ? -127 : (s > 127 ? 127 : s);
}

/* One row of n bf16 values (n a multiple of 32) to MXFP4: codes [n/2] bytes
 * with element 2i in the low nibble and 2i+1 in the high nibble of byte i,
 * and scales [n/32] E8M0 codes, block b covering elements [32b, 32b+32). */
void orc_quantize_mxfp4_row(const uint16_t* x, int n, uint8_t* codes, uint8_t* scales) {
    for (int b = 0; b < n / 32; ++b) {
        double amax = 0.0;
        for (int i = 32 * b; i < 32 * b + 32; ++i) {
            double a = fabs(orc_bf16_to_f64(x[i]));
            if (a > amax) amax = a;
        }
        int se = orc_mx_scale_exp(amax);
        scales[b] = (uint8_t)(se + 127);
        for (int i = 32 * b; i < 32 * b + 32; i += 2) {
            uint8_t lo = orc_f64_to_e2m1(ldexp(orc_bf16_to_f64(x[i]), -se));
            uint8_t hi = orc_f64_to_e2m1(ldexp(orc_bf16_to_f64(x[i + 1]), -se));
            codes[i / 2] = (uint8_t)(lo | (hi << 4));
        }
    }
}

void orc_quantize_mxfp4_rows(const uint16_t* x, int64_t rows, int n, uint8_t* codes,
                             uint8_t* scales) {
    for (int64_t r = 0; r < rows; ++r)
        orc_quantize_mxfp4_row(x + r * n, n, codes + r * (n / 2), scales + r * (n / 32));
}

/* Element d of an MXFP4 row. */
static double orc_mxfp4_value(const uint8_t* codes, const uint8_t* scales, int d) {
    uint8_t c = (uint8_t)((codes[d / 2] >> (4 * (d & 1))) & 15);
    return orc_e2m1_to_f64(c) * orc_e8m0_to_f64(scales[d / 32]);
}

/*
 * Indexer scores with MXFP4 keys: codes ik4 [B][N_cap][dI/2] and E8M0 scales
 * iks [B][N_cap][dI/32]; each bf16 query row iq[b][t][h] is quantised the
 * same way; both are dequantised to fp64 and the score is the plain
 * definition sum_h w[t,h] * max(0, q^[t,h] . k^[j]).  NaN past the visible
 * entries.  dI must be a multiple of 32.
 */
int orc_indexer_scores_mxfp4(const uint16_t* iq, const float* w, const uint8_t* ik4,
                             const uint8_t* iks, const int32_t* pos, int B, int T, int HI, int dI,
                             int64_t N_cap, int m, double* scores) {
    if (B <= 0 || T <= 0 || HI <= 0 || dI <= 0 || dI % 32 || N_cap < 0 || m <= 0)
        return ORC_EINVAL;
    uint8_t* qc = (uint8_t*)malloc((size_t)dI / 2);
    uint8_t* qs = (uint8_t*)malloc((size_t)dI / 32);
    double* qd = (double*)malloc(sizeof(double) * (size_t)HI * dI);
    double* kd = (double*)malloc(sizeof(double) * (size_t)dI);
    if (!qc || !qs || !qd || !kd) { free(qc); free(qs); free(qd); free(kd); return ORC_ENOMEM; }
    for (int b = 0; b < B; ++b) {
        for (int t = 0; t < T; ++t) {
            int64_t bt = (int64_t)b * T + t;
            for (int h = 0; h < HI; ++h) {
                orc_quantize_mxfp4_row(iq + (bt * HI + h) * dI, dI, qc, qs);
                for (int d = 0; d < dI; ++d) qd[(size_t)h * dI + d] = orc_mxfp4_value(qc, qs, d);
            }
            int64_t n = orc_visible(pos[bt], m);
            if (n > N_cap) n = N_cap;
            double* out = scores + bt * N_cap;
            for (int64_t j = 0; j < N_cap; ++j) out[j] = NAN;
            for (int64_t j = 0; j < n; ++j) {
                const uint8_t* kc = ik4 + ((int64_t)b * N_cap + j) * (dI / 2);
                const uint8_t* ks = iks + ((int64_t)b * N_cap + j) * (dI / 32);
                for (int d = 0; d < dI; ++d) kd[d] = orc_mxfp4_value(kc, ks, d);
                double s = 0.0;
                for (int h = 0; h < HI; ++h) {
                    double dot = 0.0;
                    for (int d = 0; d < dI; ++d) dot += qd[(size_t)h * dI + d] * kd[d];
                    s += (double)w[bt * HI + h] * (dot > 0.0 ? dot : 0.0);
                }
                out[j] = s;
            }
        }
    }
    free(qc); free(qs); free(qd); free(kd);
    return ORC_OK;
}

typedef struct { double s; int64_t j; } orc_pair;

/* score descending, then index ascending */
static int orc_pair_cmp(const void* a, const void* b) {
    const orc_pair* x = (const orc_pair*)a;
    const orc_pair* y = (const orc_pair*)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->j < y->j) ? -1 : (x->j > y->j);
}

/*
 * Top-k over the first n = min(visible(pos), N_cap) scores of each row,
 * by full sort (score descending, index ascending).  idx [B*T][k] gets the
 * k_eff = min(k, n) selected indices in that order, padded with -1.
 * scores [B*T][N_cap] (any precision representable in double).
 */
int orc_topk(const double* scores, const int32_t* pos, int rows, int64_t N_cap, int m, int k,
             int32_t* idx) {
    if (rows <= 0 || N_cap < 0 || m <= 0 || k <= 0) return ORC_EINVAL;
    orc_pair* buf = (orc_pair*)malloc(sizeof(orc_pair) * (size_t)(N_cap > 0 ? N_cap : 1));
    if (!buf) return ORC_ENOMEM;
    for (int rI = 0; rI < rows; ++rI) {
        int64_t n = orc_visible(pos[rI], m);
        if (n > N_cap) n = N_cap;
        for (int64_t j = 0; j < n; ++j) {
            buf[j].s = scores[(int64_t)rI * N_cap + j];
            buf[j].j = j;
        }
        qsort(buf, (size_t)n, sizeof(orc_pair), orc_pair_cmp);
        int64_t keff = n < k ? n : k;
        for (int64_t i = 0; i < k; ++i)
            idx[(int64_t)rI * k + i] = i < keff ? (int32_t)buf[i].j : -1;
    }
    free(buf);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Attention branches ([DD] "Core Architectural Innovations"; shared-KV */
/* MQA latent from [AT] "Inference efficiency")                         */
/* ------------------------------------------------------------------ */

/* q~ = RoPE_t(RMSNorm(q; gamma_q, eps)) over the D dims of one head. */
static void prep_query(const uint16_t* q, const float* gamma_q, int D, int r, double base,
                       double eps, int64_t t, double* out) {
    for (int d = 0; d < D; ++d) out[d] = orc_bf16_to_f64(q[d]);
    orc_rmsnorm(out, D, gamma_q, eps);
    orc_rope(out, D, r, base, t, +1);
}

/* Softmax attention of one prepared query over nk key rows (V = K).
 * Two passes: max, then exp/sum.  Empty set: o = 0, lse = -inf.
 * weights (may be NULL) receives the nk softmax probabilities. */
static void attend(const double* qt, const double* keys, int64_t nk, int D, double scale,
                   double* o, double* lse, double* logit_buf, double* weights) {
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (nk == 0) { *lse = -INFINITY; return; }
    double mx = -INFINITY;
    for (int64_t i = 0; i < nk; ++i) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qt[d] * keys[i * D + d];
        logit_buf[i] = scale * dot;
        if (logit_buf[i] > mx) mx = logit_buf[i];
    }
    double z = 0.0;
    for (int64_t i = 0; i < nk; ++i) {
        logit_buf[i] = exp(logit_buf[i] - mx);
        z += logit_buf[i];
    }
    for (int64_t i = 0; i < nk; ++i) {
        double p = logit_buf[i] / z;
        if (weights) weights[i] = p;
        for (int d = 0; d < D; ++d) o[d] += p * keys[i * D + d];
    }
    *lse = mx + log(z);
}

/*
 * One attention branch for every (b, t, h).
 *   kind 0 (CSA sparse): keys are cache[b][idx[b][t][i]] for the idx >= 0.
 *   kind 1 (HCA dense) : keys are cache[b][j] for j < min(visible(t, m), N_cap).
 *   kind 2 (SWA)       : keys are raw tokens u in [max(0, t-W+1), t], each
 *                        RMSNorm'd (gamma_kv, eps) and RoPE'd at position u.
 * q [B][T][H][D] bf16, pos [B][T], cache [B][N_cap][D] bf16 (kinds 0/1) or
 * raw [B][L_cap][D] bf16 (kind 2; N_cap is L_cap), idx [B][T][k] (kind 0).
 * Outputs o [B][T][H][D] fp64, lse [B][T][H] fp64.
 */
int orc_attention(int kind, const uint16_t* q, const float* gamma_q, const uint16_t* cache,
                  const float* gamma_kv, const int32_t* idx, const int32_t* pos, int B, int T, int H,
                  int D, int64_t N_cap, int k, int m, int W, int r, double base, double eps,
                  double scale, double* o, double* lse) {
    if (B <= 0 || T <= 0 || H <= 0 || D <= 0 || N_cap < 0 || r < 0 || r > D || (r % 2))
        return ORC_EINVAL;
    if (kind == 0 && k <= 0) return ORC_EINVAL;
    if (kind == 1 && m <= 0) return ORC_EINVAL;
    if (kind == 2 && W <= 0) return ORC_EINVAL;
    if (kind < 0 || kind > 2) return ORC_EINVAL;
    int64_t maxk = kind == 0 ? k : (kind == 1 ? N_cap : W);
    double* keys = (double*)malloc(sizeof(double) * (size_t)((maxk > 0 ? maxk : 1) * D));
    double* lbuf = (double*)malloc(sizeof(double) * (size_t)(maxk > 0 ? maxk : 1));
    double* qt = (double*)malloc(sizeof(double) * (size_t)D);
    if (!keys || !lbuf || !qt) {
        free(keys); free(lbuf); free(qt);
        return ORC_ENOMEM;
    }
    for (int b = 0; b < B; ++b) {
        for (int t = 0; t < T; ++t) {
            int64_t bt = (int64_t)b * T + t;
            int64_t tp = pos[bt];
            int64_t nk = 0;
            if (kind == 0) {
                for (int i = 0; i < k; ++i) {
                    int32_t j = idx[bt * k + i];
                    if (j < 0) continue;
                    if (j >= N_cap) { free(keys); free(lbuf); free(qt); return ORC_EINVAL; }
                    const uint16_t* row = cache + ((int64_t)b * N_cap + j) * D;
                    for (int d = 0; d < D; ++d) keys[nk * D + d] = orc_bf16_to_f64(row[d]);
                    ++nk;
                }
            } else if (kind == 1) {
                int64_t n = orc_visible(tp, m);
                if (n > N_cap) n = N_cap;
                for (int64_t j = 0; j < n; ++j) {
                    const uint16_t* row = cache + ((int64_t)b * N_cap + j) * D;
                    for (int d = 0; d < D; ++d) keys[nk * D + d] = orc_bf16_to_f64(row[d]);
                    ++nk;
                }
            } else {
                int64_t lo = tp - W + 1;
                if (lo < 0) lo = 0;
                for (int64_t u = lo; u <= tp && u < N_cap; ++u) {
                    const uint16_t* row = cache + ((int64_t)b * N_cap + u) * D;
                    double* kr = keys + nk * D;
                    for (int d = 0; d < D; ++d) kr[d] = orc_bf16_to_f64(row[d]);
                    orc_rmsnorm(kr, D, gamma_kv, eps);
                    orc_rope(kr, D, r, base, u, +1);
                    ++nk;
                }
            }
            for (int h = 0; h < H; ++h) {
                prep_query(q + (bt * H + h) * D, gamma_q, D, r, base, eps, tp, qt);
                attend(qt, keys, nk, D, scale, o + (bt * H + h) * D, lse + bt * H + h, lbuf, NULL);
            }
        }
    }
    free(keys); free(lbuf); free(qt);
    return ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Sink-augmented log-sum-exp merge and inverse RoPE on the output      */
/* ([AT] "Spec sheet": attention sinks yes; provenance 16: "-i RoPE on  */
/* outputs")                                                            */
/* ------------------------------------------------------------------ */

/*
 * For every (b, t, h):
 *   Z   = sum_i exp(lse_i) + exp(sink[h])        (nb branches, nb >= 0)
 *   out = RoPE_{-pos}( sum_i exp(lse_i) * o_i / Z )   over the last r dims
 *   lse_out = log Z
 * o_i [B][T][H][D] fp64, lse_i [B][T][H] fp64, sink [H] fp32 (NULL: no sink).
 */
int orc_merge(const double* const* o_list, const double* const* lse_list, int nb,
              const float* sink, const int32_t* pos, int B, int T, int H, int D, int r,
              double base, double* out, double* lse_out) {
    if (nb < 0 || B <= 0 || T <= 0 || H <= 0 || D <= 0 || r < 0 || r > D || (r % 2))
        return ORC_EINVAL;
    for (int64_t bt = 0; bt < (int64_t)B * T; ++bt) {
        for (int h = 0; h < H; ++h) {
            int64_t row = bt * H + h;
            double mx = sink ? (double)sink[h] : -INFINITY;
            for (int i = 0; i < nb; ++i)
                if (lse_list[i][row] > mx) mx = lse_list[i][row];
            double* y = out + row * D;
            for (int d = 0; d < D; ++d) y[d] = 0.0;
            if (mx == -INFINITY) { /* nothing to attend and no sink */
                lse_out[row] = -INFINITY;
                continue;
            }
            double z = sink ? exp((double)sink[h] - mx) : 0.0;
            for (int i = 0; i < nb; ++i) z += exp(lse_list[i][row] - mx);
            double lz = mx + log(z);
            for (int i = 0; i < nb; ++i) {
                double c = exp(lse_list[i][row] - lz);
                if (c == 0.0) continue;
                const double* oi = o_list[i] + row * D;
                for (int d = 0; d < D; ++d) y[d] += c * oi[d];
            }
            orc_rope(y, D, r, base, pos[bt], -1);
            lse_out[row] = lz;
        }
    }
    return ORC_OK;
}

/* Softmax weights of one head over a key list plus the sink, for the
 * invariant "weights + sink = 1".  keys fp64 [nk][D] already prepared;
 * q fp64 [D] already prepared.  w_out [nk], returns the sink weight. */
double orc_weights_with_sink(const double* qt, const double* keys, int64_t nk, int D,
                             double scale, double sink, double* w_out) {
    double mx = sink;
    for (int64_t i = 0; i < nk; ++i) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qt[d] * keys[i * D + d];
        w_out[i] = scale * dot;
        if (w_out[i] > mx) mx = w_out[i];
    }
    double z = exp(sink - mx);
    for (int64_t i = 0; i < nk; ++i) {
        w_out[i] = exp(w_out[i] - mx);
        z += w_out[i];
    }
    for (int64_t i = 0; i < nk; ++i) w_out[i] /= z;
    return exp(sink - mx) / z;
}
