/*
 * spark_oracle.c -- plain fp64 CPU oracle of the Spark-X2.5 attention core.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file.  Only the test suite, the smoke check of the package entry
 * file and the CPU-baseline leg of the benchmark use it.  It shares no code,
 * header, table or constant with the CUDA library.
 *
 * What it computes, and where each step comes from:
 *
 *  - Spark-X2.5 architecture (4B / 1.7B), §3 "head-wise output gate", Eq. 1:
 *      o = ( softmax(Q K^T / sqrt(d_head)) V ) (.) sigmoid(W_g x)
 *    one gate scalar per head, broadcast over the head's 256 dims.  The fused
 *    q_k_v_proj output is Q || K || V with width H*256 + 2*Hkv*256 (same §3).
 *  - Same page, §4 "layered RoPE" table: full_attention layers use theta=5e6
 *    and rotate the first 64 of 256 dims; sliding_attention layers use
 *    theta=1e4 and rotate all 256 dims.  The 192 other dims are left as they
 *    are (the page calls them NoPE).  Partial RoPE, as the MiniMax-M2 chapter
 *    §13.3 of the translated LLM-architecture notes defines it, rotates the
 *    first rotary_dim channels of every head and leaves the rest unchanged.
 *  - Same page, §2 "hybrid attention": full layers use a causal mask, sliding
 *    layers a sliding-window causal mask of window 512.
 *    The gate activation is sigmoid; the page notes the code also supports
 *    silu (gate_attn_act_mode), which multiplies by x * sigmoid(x) instead.
 *  - Spark-X2.5-4B hybrid-attention explainer (lshu.cn), section on the
 *    sliding layer's KV cache: a sliding layer keeps only the latest 512
 *    tokens; older ones are dropped.  Full layers keep every token.
 *
 * Readings taken where the pages are silent (each one is listed with its
 * reason in the design notes of the repository):
 *  - window: key j is visible from query i iff 0 <= i-j < W (self included);
 *  - rotation pairs dims (k, k + r/2) inside the first r dims (rotate_half),
 *    with inverse frequency theta^(-2k/r), k = 0 .. r/2-1;
 *  - query head h reads KV head floor(h / (H/Hkv));
 *  - scale is exactly 1/sqrt(256) = 1/16, no soft-cap;
 *  - everything is exact fp64: the bf16 inputs are widened exactly, angles
 *    are pos * inv_freq in fp64, no intermediate is rounded to bf16.
 *  - decode: a contiguous cache stores token j at slot j; a ring of `cap`
 *    slots stores token j at slot j mod cap.  Cached keys are post-RoPE.
 *    The new token is written first, then attended (write-then-attend).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_HEAD_DIM 256

enum { ORACLE_FULL = 0, ORACLE_SLIDING = 1 };

enum {
    ORACLE_OK = 0,
    ORACLE_ERR_ARG = 1,
    ORACLE_ERR_NOMEM = 2
};

/* Exact widening of a bf16 bit pattern: bf16 is the top half of an fp32. */
static double bf16_bits_to_f64(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/*
 * Gate activation (Spark-X2.5 architecture, §3): the released checkpoints use
 * sigmoid; the code also supports silu, x * sigmoid(x).
 */
enum { ORACLE_GATE_SIGMOID = 0, ORACLE_GATE_SILU = 1 };

static double gate_act(double x, int mode)
{
    return mode == ORACLE_GATE_SILU ? x * sigmoid(x) : sigmoid(x);
}

/*
 * RoPE on one head vector x[0..255] at position pos, written to y.
 * Layered RoPE (§4 of the Spark-X2.5 architecture page): for k < r/2
 *   a     = pos * theta^(-2k/r)
 *   y_k       = x_k cos a - x_{k+r/2} sin a
 *   y_{k+r/2} = x_{k+r/2} cos a + x_k sin a
 * and y_i = x_i for i >= r (partial RoPE, MiniMax-M2 chapter §13.3).
 */
static void rope_head(const double *x, double pos, int rot_dim, double theta, double *y)
{
    int half = rot_dim / 2;
    for (int i = 0; i < ORACLE_HEAD_DIM; ++i)
        y[i] = x[i];
    for (int k = 0; k < half; ++k) {
        double inv_freq = pow(theta, -2.0 * (double)k / (double)rot_dim);
        double a = pos * inv_freq;
        double c = cos(a), s = sin(a);
        double x1 = x[k], x2 = x[k + half];
        y[k] = x1 * c - x2 * s;
        y[k + half] = x2 * c + x1 * s;
    }
}

/* Public RoPE entry: n head vectors (fp64, [n,256]) with positions pos[n]. */
int oracle_rope(const double *x, const int32_t *pos, int64_t n, int rot_dim,
                double theta, double *y)
{
    if (!x || !pos || !y || n < 0 || rot_dim < 0 || rot_dim > ORACLE_HEAD_DIM ||
        (rot_dim & 1))
        return ORACLE_ERR_ARG;
    for (int64_t i = 0; i < n; ++i)
        rope_head(x + i * ORACLE_HEAD_DIM, (double)pos[i], rot_dim, theta,
                  y + i * ORACLE_HEAD_DIM);
    return ORACLE_OK;
}

/*
 * Softmax-weighted average over a list of visible keys, for one query head:
 *   s_j = q . k_j / 16,  p = softmax(s),  o = sum_j p_j v_j,
 *   out = o * sigmoid(g).
 * keys/vals are arrays of pointers to 256-dim fp64 vectors.
 */
static void attend_one(const double *q, const double *const *keys,
                       const double *const *vals, int64_t nvis, double gate_logit,
                       int gate_mode, double *s_scratch, double *out)
{
    const double scale = 1.0 / sqrt((double)ORACLE_HEAD_DIM);
    double m = -INFINITY;
    for (int64_t j = 0; j < nvis; ++j) {
        double dot = 0.0;
        for (int d = 0; d < ORACLE_HEAD_DIM; ++d)
            dot += q[d] * keys[j][d];
        s_scratch[j] = dot * scale;
        if (s_scratch[j] > m)
            m = s_scratch[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < nvis; ++j) {
        s_scratch[j] = exp(s_scratch[j] - m);
        l += s_scratch[j];
    }
    for (int d = 0; d < ORACLE_HEAD_DIM; ++d)
        out[d] = 0.0;
    for (int64_t j = 0; j < nvis; ++j) {
        double p = s_scratch[j] / l;
        for (int d = 0; d < ORACLE_HEAD_DIM; ++d)
            out[d] += p * vals[j][d];
    }
    double gsig = gate_act(gate_logit, gate_mode);
    for (int d = 0; d < ORACLE_HEAD_DIM; ++d)
        out[d] *= gsig;
}

/* First visible key index for query token i (mask of §2, window reading). */
static int64_t first_visible(int kind, int window, int64_t i)
{
    if (kind == ORACLE_SLIDING) {
        int64_t lo = i - (int64_t)window + 1;
        return lo > 0 ? lo : 0;
    }
    return 0;
}

/*
 * Prefill.  qkv: bf16 bits [B, T, (H+2Hkv)*256]; gate: fp32 [B, T, H];
 * pos: [B, T] RoPE positions; rows: list of flat row ids (b*T + t) to compute
 * (NULL = every row, in order); out: fp64 [nrows, H*256].
 * The mask is on the token index inside the sequence; RoPE uses pos.
 */
int oracle_prefill(const uint16_t *qkv, const float *gate, const int32_t *pos,
                   int kind, int window, double theta, int rot_dim, int gate_mode, int B,
                   int T, int H, int Hkv, const int64_t *rows, int64_t nrows, double *out)
{
    if (!qkv || !gate || !pos || !out || B <= 0 || T <= 0 || H <= 0 || Hkv <= 0 ||
        H % Hkv != 0 || rot_dim < 0 || rot_dim > ORACLE_HEAD_DIM || (rot_dim & 1) ||
        (kind != ORACLE_FULL && kind != ORACLE_SLIDING) ||
        (kind == ORACLE_SLIDING && window < 1) ||
        (gate_mode != ORACLE_GATE_SIGMOID && gate_mode != ORACLE_GATE_SILU))
        return ORACLE_ERR_ARG;
    if (!rows)
        nrows = (int64_t)B * T;
    const int D = ORACLE_HEAD_DIM;
    const int G = H / Hkv;
    const int64_t width = (int64_t)(H + 2 * Hkv) * D;

    /* Rotated keys and widened values of every token: [B*T, Hkv, 256]. */
    int64_t ntok = (int64_t)B * T;
    double *krot = (double *)malloc(sizeof(double) * ntok * Hkv * D);
    double *vf = (double *)malloc(sizeof(double) * ntok * Hkv * D);
    if (!krot || !vf) {
        free(krot);
        free(vf);
        return ORACLE_ERR_NOMEM;
    }
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < ntok; ++r) {
        double kx[ORACLE_HEAD_DIM];
        for (int g = 0; g < Hkv; ++g) {
            const uint16_t *ks = qkv + r * width + (int64_t)(H + g) * D;
            const uint16_t *vs = qkv + r * width + (int64_t)(H + Hkv + g) * D;
            for (int d = 0; d < D; ++d) {
                kx[d] = bf16_bits_to_f64(ks[d]);
                vf[(r * Hkv + g) * D + d] = bf16_bits_to_f64(vs[d]);
            }
            rope_head(kx, (double)pos[r], rot_dim, theta, krot + (r * Hkv + g) * D);
        }
    }

    int status = ORACLE_OK;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)T);
        const double **kp = (const double **)malloc(sizeof(double *) * (size_t)T);
        const double **vp = (const double **)malloc(sizeof(double *) * (size_t)T);
        if (!s || !kp || !vp) {
#pragma omp atomic write
            status = ORACLE_ERR_NOMEM;
        } else {
#pragma omp for schedule(dynamic, 1) collapse(2)
            for (int64_t ri = 0; ri < nrows; ++ri) {
                for (int h = 0; h < H; ++h) {
                    int64_t row = rows ? rows[ri] : ri;
                    int64_t b = row / T, i = row % T;
                    int g = h / G;
                    double qx[ORACLE_HEAD_DIM], q[ORACLE_HEAD_DIM];
                    const uint16_t *qs = qkv + row * width + (int64_t)h * D;
                    for (int d = 0; d < D; ++d)
                        qx[d] = bf16_bits_to_f64(qs[d]);
                    rope_head(qx, (double)pos[row], rot_dim, theta, q);
                    int64_t lo = first_visible(kind, window, i);
                    int64_t nvis = i - lo + 1;
                    for (int64_t j = 0; j < nvis; ++j) {
                        int64_t tok = b * T + lo + j;
                        kp[j] = krot + (tok * Hkv + g) * D;
                        vp[j] = vf + (tok * Hkv + g) * D;
                    }
                    attend_one(q, kp, vp, nvis, (double)gate[row * H + h], gate_mode, s,
                               out + ri * (int64_t)H * D + (int64_t)h * D);
                }
            }
        }
        free(s);
        free(kp);
        free(vp);
    }
    free(krot);
    free(vf);
    return status;
}

/*
 * Decode: one new token per sequence.
 *   qkv     bf16 bits [B, (H+2Hkv)*256]  (the new token's fused projection)
 *   gate    fp32 [B, H]
 *   pos     [B]: position of the new token == number of tokens already cached
 *   k_cache, v_cache  bf16 bits [B, Hkv, cap, 256], contents BEFORE the call,
 *           post-RoPE keys.  FULL: token j at slot j (needs cap >= pos+1).
 *           SLIDING: a ring, token j at slot j mod cap (needs cap >= window).
 *   out     fp64 [B, H*256]
 *   k_new, v_new  fp64 [B, Hkv, 256]: the rotated key and the value that the
 *           update writes into slot(pos) (may be NULL).
 * The visible tokens are [0, pos] (FULL) or [max(0, pos-W+1), pos] (SLIDING);
 * token pos is the new one, the others are read from their slots.
 */
int oracle_decode(const uint16_t *qkv, const float *gate, const int32_t *pos,
                  const uint16_t *k_cache, const uint16_t *v_cache, int64_t cap,
                  int kind, int window, double theta, int rot_dim, int gate_mode, int B,
                  int H, int Hkv, double *out, double *k_new, double *v_new)
{
    if (!qkv || !gate || !pos || !k_cache || !v_cache || !out || B <= 0 || H <= 0 ||
        Hkv <= 0 || H % Hkv != 0 || rot_dim < 0 || rot_dim > ORACLE_HEAD_DIM ||
        (rot_dim & 1) || cap <= 0 || (kind != ORACLE_FULL && kind != ORACLE_SLIDING) ||
        (kind == ORACLE_SLIDING && (window < 1 || cap < window)) ||
        (gate_mode != ORACLE_GATE_SIGMOID && gate_mode != ORACLE_GATE_SILU))
        return ORACLE_ERR_ARG;
    for (int b = 0; b < B; ++b)
        if (pos[b] < 0 || (kind == ORACLE_FULL && (int64_t)pos[b] + 1 > cap))
            return ORACLE_ERR_ARG;
    const int D = ORACLE_HEAD_DIM;
    const int G = H / Hkv;
    const int64_t width = (int64_t)(H + 2 * Hkv) * D;
    const double scale = 1.0 / sqrt((double)D);

    /* the new token's rotated key and value, per (b, g) */
    double *kn = (double *)malloc(sizeof(double) * (size_t)B * Hkv * D);
    double *vn = (double *)malloc(sizeof(double) * (size_t)B * Hkv * D);
    if (!kn || !vn) {
        free(kn);
        free(vn);
        return ORACLE_ERR_NOMEM;
    }
    for (int b = 0; b < B; ++b)
        for (int g = 0; g < Hkv; ++g) {
            double kx[ORACLE_HEAD_DIM];
            const uint16_t *ks = qkv + b * width + (int64_t)(H + g) * D;
            const uint16_t *vs = qkv + b * width + (int64_t)(H + Hkv + g) * D;
            double *vd = vn + ((int64_t)b * Hkv + g) * D;
            for (int d = 0; d < D; ++d) {
                kx[d] = bf16_bits_to_f64(ks[d]);
                vd[d] = bf16_bits_to_f64(vs[d]);
            }
            rope_head(kx, (double)pos[b], rot_dim, theta, kn + ((int64_t)b * Hkv + g) * D);
        }
    if (k_new)
        memcpy(k_new, kn, sizeof(double) * (size_t)B * Hkv * D);
    if (v_new)
        memcpy(v_new, vn, sizeof(double) * (size_t)B * Hkv * D);

    int status = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            int64_t p = pos[b];
            int g = h / G;
            int64_t lo = first_visible(kind, window, p);
            int64_t nvis = p - lo + 1;
            double *s = (double *)malloc(sizeof(double) * (size_t)nvis);
            if (!s) {
#pragma omp atomic write
                status = ORACLE_ERR_NOMEM;
                continue;
            }
            double qx[ORACLE_HEAD_DIM], q[ORACLE_HEAD_DIM];
            const uint16_t *qs = qkv + b * width + (int64_t)h * D;
            for (int d = 0; d < D; ++d)
                qx[d] = bf16_bits_to_f64(qs[d]);
            rope_head(qx, (double)p, rot_dim, theta, q);
            const uint16_t *kc = k_cache + ((int64_t)b * Hkv + g) * cap * D;
            const uint16_t *vc = v_cache + ((int64_t)b * Hkv + g) * cap * D;
            const double *knew = kn + ((int64_t)b * Hkv + g) * D;
            const double *vnew = vn + ((int64_t)b * Hkv + g) * D;
            /* scores s_j = q . k_j / 16 over the visible tokens */
            double m = -INFINITY;
            for (int64_t j = 0; j < nvis; ++j) {
                int64_t tok = lo + j;
                double dot = 0.0;
                if (tok == p) {
                    for (int d = 0; d < D; ++d)
                        dot += q[d] * knew[d];
                } else {
                    int64_t slot = (kind == ORACLE_SLIDING) ? tok % cap : tok;
                    for (int d = 0; d < D; ++d)
                        dot += q[d] * bf16_bits_to_f64(kc[slot * D + d]);
                }
                s[j] = dot * scale;
                if (s[j] > m)
                    m = s[j];
            }
            /* softmax weights, then the weighted sum of values */
            double l = 0.0;
            for (int64_t j = 0; j < nvis; ++j) {
                s[j] = exp(s[j] - m);
                l += s[j];
            }
            double o[ORACLE_HEAD_DIM];
            for (int d = 0; d < D; ++d)
                o[d] = 0.0;
            for (int64_t j = 0; j < nvis; ++j) {
                int64_t tok = lo + j;
                double pj = s[j] / l;
                if (tok == p) {
                    for (int d = 0; d < D; ++d)
                        o[d] += pj * vnew[d];
                } else {
                    int64_t slot = (kind == ORACLE_SLIDING) ? tok % cap : tok;
                    for (int d = 0; d < D; ++d)
                        o[d] += pj * bf16_bits_to_f64(vc[slot * D + d]);
                }
            }
            double gsig = gate_act((double)gate[(int64_t)b * H + h], gate_mode);
            double *dst = out + (int64_t)b * H * D + (int64_t)h * D;
            for (int d = 0; d < D; ++d)
                dst[d] = o[d] * gsig;
            free(s);
        }
    }
    free(kn);
    free(vn);
    return status;
}
