/*
 * Routed MoE layer -- plain, slow fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or constant with the CUDA
 * library: it reads the Q8_0 weight bytes in the pages' own 34-byte block
 * format and decodes them itself.
 *
 * What it computes (the definition, written out, in fp64):
 *   1. router logits  l[t][e] = sum_j x[t][j] * Wr[e][j]  (+ bias[e])
 *        -- "LinearGate" routing (amalgafy.com/evidence, "Layer-qualified
 *           experts"); "GPU router/top-k" (amalgafy.com/technical-overview,
 *           "Not complete today").
 *   2. top-k selection by logit, ties broken towards the lower expert id,
 *      output in descending-logit order ("Learned top-8 selection",
 *      amalgafy.com/evidence, "Historical baseline environment").
 *   3. renormalised softmax weights over the selected experts:
 *        w_i = exp(l_i - l_max) / sum_sel exp(l_j - l_max)
 *      (equal to a softmax over all E followed by renormalisation over the
 *      selection, since the common denominator cancels).
 *   4. per (token, slot): Q8_0 SwiGLU expert
 *        g = Wg x, u = Wu x, h = silu(g) * u, silu(z) = z / (1 + exp(-z)),
 *        y = Wd h,  with every weight dequantised as w = q * d
 *      (Q8_0 weights: amalgafy.com/evidence "Historical baseline
 *      environment" checkpoint and amalgafy.com/technical-overview
 *      "Validated GPU foundation"; down projection K=768 -> 2048 rows:
 *      expxa.com reuse-ordering-qualification, "What changed from the first
 *      experiment").
 *   5. weighted combine out[t] = (residual ? x[t] : 0) + sum_slot w * y
 *      ("GPU routing, Q4 expert execution, weighted combine",
 *      amalgafy.com/technical-overview, "Execution architecture").
 *   6. compact expert grouping (bucketing) of (token, slot) pairs by expert,
 *      stable in (token, slot) order (expxa.com, "What changed from the first
 *      experiment": "compact expert grouping").
 *
 * Q8_0 block (34 bytes, little endian): fp16 scale d, then 32 int8 values q
 * along K.  A Q8_0 matrix of rows x K is rows * (K/32) blocks, row-major.
 *
 * Q4_0 block (18 bytes): fp16 scale d, then 16 bytes holding 32 unsigned
 * 4-bit values n along K: byte j carries element j in its low nibble and
 * element j + 16 in its high nibble; w = (n - 8) * d.  ("Q4 expert
 * execution", amalgafy.com/technical-overview, "Execution architecture"; the
 * pages give no block layout, so this is the plain 4-bit sibling of Q8_0:
 * same 32-wide blocks and fp16 scale, values offset by 8.)
 *
 * Parallelism: tokens are independent, so the token loops may run under
 * OpenMP; that changes no arithmetic and no summation order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_Q8_BLOCK_ELEMS 32
#define ORACLE_Q8_BLOCK_BYTES 34

int oracle_q8_block_bytes(void) { return ORACLE_Q8_BLOCK_BYTES; }
int oracle_q8_block_elems(void) { return ORACLE_Q8_BLOCK_ELEMS; }

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* IEEE 754 binary16 -> double (exact). */
double oracle_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int mant = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)mant, -24);              /* zero or subnormal */
    } else if (expo == 31) {
        v = mant ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + mant), expo - 25); /* (1.m) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* Dequantise one Q8_0 row of K weights: w[j] = q[j] * d[block(j)]. */
static void dequant_row(const uint8_t* row_blocks, int K, double* w) {
    int nb = K / ORACLE_Q8_BLOCK_ELEMS;
    for (int b = 0; b < nb; ++b) {
        const uint8_t* blk = row_blocks + (size_t)b * ORACLE_Q8_BLOCK_BYTES;
        uint16_t dbits = (uint16_t)(blk[0] | (blk[1] << 8));
        double d = oracle_half_to_double(dbits);
        for (int j = 0; j < ORACLE_Q8_BLOCK_ELEMS; ++j) {
            int q = (int)(int8_t)blk[2 + j];
            w[b * ORACLE_Q8_BLOCK_ELEMS + j] = (double)q * d;
        }
    }
}

#define ORACLE_Q4_BLOCK_BYTES 18

/* Dequantise one Q4_0 row of K weights: w = (n - 8) * d. */
static void dequant_row_q4(const uint8_t* row_blocks, int K, double* w) {
    int nb = K / ORACLE_Q8_BLOCK_ELEMS;
    for (int b = 0; b < nb; ++b) {
        const uint8_t* q4b = row_blocks + (size_t)b * ORACLE_Q4_BLOCK_BYTES;
        double d4 = oracle_half_to_double((uint16_t)(q4b[0] | (q4b[1] << 8)));
        for (int j = 0; j < 16; ++j) {
            int lo = q4b[2 + j] & 0x0F, hi = q4b[2 + j] >> 4;
            w[b * ORACLE_Q8_BLOCK_ELEMS + j] = (double)(lo - 8) * d4;
            w[b * ORACLE_Q8_BLOCK_ELEMS + 16 + j] = (double)(hi - 8) * d4;
        }
    }
}

/* Block format: 0 = Q8_0, 1 = Q4_0. */
static size_t row_bytes_of(int K, int fmt) {
    return (size_t)(K / ORACLE_Q8_BLOCK_ELEMS) * (fmt == 1 ? ORACLE_Q4_BLOCK_BYTES : ORACLE_Q8_BLOCK_BYTES);
}

static void dequant_row_fmt(const uint8_t* row_blocks, int K, int fmt, double* w) {
    if (fmt == 1)
        dequant_row_q4(row_blocks, K, w);
    else
        dequant_row(row_blocks, K, w);
}

/* Dequantise a whole rows x K matrix (format fmt) into out[rows][K]. */
void oracle_dequant(const uint8_t* blocks, int rows, int K, int fmt, double* out) {
    size_t row_bytes = row_bytes_of(K, fmt);
    for (int r = 0; r < rows; ++r) dequant_row_fmt(blocks + (size_t)r * row_bytes, K, fmt, out + (size_t)r * K);
}

/* Dequantise a whole rows x K Q8_0 matrix into out[rows][K]. */
void oracle_dequant_q8(const uint8_t* blocks, int rows, int K, double* out) { oracle_dequant(blocks, rows, K, 0, out); }

/* y[r] = sum_j W[r][j] * v[j], W given as rows x K blocks of format fmt, j ascending. */
static void q_matvec(const uint8_t* blocks, int rows, int K, int fmt, const double* v, double* y, double* wrow) {
    size_t row_bytes = row_bytes_of(K, fmt);
    for (int r = 0; r < rows; ++r) {
        dequant_row_fmt(blocks + (size_t)r * row_bytes, K, fmt, wrow);
        double acc = 0.0;
        for (int j = 0; j < K; ++j) acc += wrow[j] * v[j];
        y[r] = acc;
    }
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

/*
 * One SwiGLU expert on one token vector.
 *   gate, up: [f][dm] (K = dm); down: [dm][f] (K = f); blocks of format fmt.
 *   x[dm] -> y[dm].
 */
int oracle_expert_swiglu_fmt(const uint8_t* gate, const uint8_t* up, const uint8_t* down, int dm, int f, int fmt,
                             const double* x, double* y) {
    int kmax = dm > f ? dm : f;
    double* g = (double*)malloc(sizeof(double) * (size_t)f);
    double* u = (double*)malloc(sizeof(double) * (size_t)f);
    double* h = (double*)malloc(sizeof(double) * (size_t)f);
    double* wrow = (double*)malloc(sizeof(double) * (size_t)kmax);
    int ok = g && u && h && wrow;
    if (ok) {
        q_matvec(gate, f, dm, fmt, x, g, wrow);
        q_matvec(up, f, dm, fmt, x, u, wrow);
        for (int r = 0; r < f; ++r) h[r] = silu(g[r]) * u[r];
        q_matvec(down, dm, f, fmt, h, y, wrow);
    }
    free(g); free(u); free(h); free(wrow);
    return ok ? 0 : -1;
}

/* Returns 0, or -1 when scratch memory could not be allocated. */
int oracle_expert_swiglu(const uint8_t* gate, const uint8_t* up, const uint8_t* down, int dm, int f,
                         const double* x, double* y) {
    return oracle_expert_swiglu_fmt(gate, up, down, dm, f, 0, x, y);
}

/*
 * Router for one token: logits (fp64), then the k largest, ties to the lower
 * id, in descending-logit order; then renormalised softmax weights.
 * If forced != NULL the selection is taken from it instead (the weights are
 * still computed from the fp64 logits of the forced experts).
 * Returns 0, or -1 when scratch memory could not be allocated.
 */
static int route_token(const double* xt, int dm, int E, int k, const float* Wr, const float* bias,
                       const int32_t* forced, int32_t* idx, double* w, double* logits) {
    for (int e = 0; e < E; ++e) {
        double acc = 0.0;
        const float* wr = Wr + (size_t)e * dm;
        for (int j = 0; j < dm; ++j) acc += xt[j] * (double)wr[j];
        if (bias) acc += (double)bias[e];
        logits[e] = acc;
    }
    if (forced) {
        for (int s = 0; s < k; ++s) idx[s] = forced[s];
    } else {
        unsigned char* taken = (unsigned char*)calloc((size_t)E, 1);
        if (!taken) return -1;
        for (int s = 0; s < k; ++s) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || logits[e] > logits[best]) best = e; /* strict >: lower id wins ties */
            }
            taken[best] = 1;
            idx[s] = best;
        }
        free(taken);
    }
    double lmax = logits[idx[0]];
    for (int s = 1; s < k; ++s) if (logits[idx[s]] > lmax) lmax = logits[idx[s]];
    double den = 0.0;
    for (int s = 0; s < k; ++s) den += exp(logits[idx[s]] - lmax);
    for (int s = 0; s < k; ++s) w[s] = exp(logits[idx[s]] - lmax) / den;
    return 0;
}

/* Round a double to fp32 (RNE) and then to bf16 (RNE): the cast the tensor-core
 * path applies to its expert inputs.  Finite inputs only. */
static double to_bf16_via_f32(double v) {
    float f = (float)v;
    uint32_t bits;
    memcpy(&bits, &f, 4);
    uint32_t lsb = (bits >> 16) & 1u;
    bits = (bits + 0x7fffu + lsb) & 0xffff0000u;
    memcpy(&f, &bits, 4);
    return (double)f;
}

/*
 * Routing only, for all tokens.  logits [T][E] may be NULL.
 * Returns 0, -1 on invalid arguments, -3 when scratch memory could not be
 * allocated.
 */
int oracle_route(int T, int dm, int E, int k, const double* x, const float* Wr, const float* bias,
                 int32_t* idx, double* w, double* logits) {
    if (T < 0 || dm <= 0 || E <= 0 || k <= 0 || k > E || !Wr || !idx || !w || (T > 0 && !x)) return -1;
    int nomem = 0;
    int t;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : nomem)
    for (t = 0; t < T; ++t) {
        double* lg = (double*)malloc(sizeof(double) * (size_t)E);
        if (!lg) { nomem = 1; continue; }
        if (route_token(x + (size_t)t * dm, dm, E, k, Wr, bias, NULL, idx + (size_t)t * k, w + (size_t)t * k, lg))
            nomem = 1;
        else if (logits)
            memcpy(logits + (size_t)t * E, lg, sizeof(double) * (size_t)E);
        free(lg);
    }
    return nomem ? -3 : 0;
}

/*
 * One MoE layer.
 *   x [T][dm] (fp64 values; the router reads them as given)
 *   Wr [E][dm] fp32, bias [E] fp32 or NULL
 *   gate, up: E experts of [f][dm]; down: E experts of [dm][f]; blocks of
 *       format fmt (0 = Q8_0, 1 = Q4_0)
 *   residual: add x[t] to the combined output
 *   expert_input_bf16: feed the experts bf16(fp32(x)) instead of x (the
 *       tensor-core path's cast; the router still reads x)
 *   forced_idx [T][k] or NULL: use this selection instead of the top-k
 *   out [T][dm]; idx [T][k]; w [T][k]; logits [T][E] or NULL
 * Returns 0; -1 on invalid arguments; -2 when a selected expert id is out of
 * range; -3 when scratch memory could not be allocated.
 */
int oracle_moe_layer_fmt(int T, int dm, int f, int E, int k, const double* x, const float* Wr, const float* bias,
                         const uint8_t* gate, const uint8_t* up, const uint8_t* down, int fmt, int residual,
                         int expert_input_bf16, const int32_t* forced_idx, double* out, int32_t* idx, double* w,
                         double* logits) {
    if (T < 0 || dm <= 0 || f <= 0 || E <= 0 || k <= 0 || k > E) return -1;
    if (dm % ORACLE_Q8_BLOCK_ELEMS || f % ORACLE_Q8_BLOCK_ELEMS) return -1;
    if (T == 0) return 0;
    if (!x || !Wr || !gate || !up || !down || !out || !idx || !w) return -1;
    if (fmt != 0 && fmt != 1) return -1;
    size_t gu_bytes = (size_t)f * row_bytes_of(dm, fmt);
    size_t dn_bytes = (size_t)dm * row_bytes_of(f, fmt);
    int bad = 0, nomem = 0;
    int t;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad, nomem)
    for (t = 0; t < T; ++t) {
        const double* xt = x + (size_t)t * dm;
        double* lg = (double*)malloc(sizeof(double) * (size_t)E);
        double* xin = (double*)malloc(sizeof(double) * (size_t)dm);
        double* y = (double*)malloc(sizeof(double) * (size_t)dm);
        double* acc = (double*)calloc((size_t)dm, sizeof(double));
        int32_t* it = idx + (size_t)t * k;
        double* wt = w + (size_t)t * k;
        if (!lg || !xin || !y || !acc ||
            route_token(xt, dm, E, k, Wr, bias, forced_idx ? forced_idx + (size_t)t * k : NULL, it, wt, lg)) {
            nomem = 1;
            free(lg); free(xin); free(y); free(acc);
            continue;
        }
        if (logits) memcpy(logits + (size_t)t * E, lg, sizeof(double) * (size_t)E);
        for (int j = 0; j < dm; ++j) xin[j] = expert_input_bf16 ? to_bf16_via_f32(xt[j]) : xt[j];
        for (int s = 0; s < k; ++s) {
            int e = it[s];
            if (e < 0 || e >= E) { bad = 1; continue; }
            if (oracle_expert_swiglu_fmt(gate + (size_t)e * gu_bytes, up + (size_t)e * gu_bytes,
                                         down + (size_t)e * dn_bytes, dm, f, fmt, xin, y)) {
                nomem = 1;
                continue;
            }
            for (int o = 0; o < dm; ++o) acc[o] += wt[s] * y[o];
        }
        double* ot = out + (size_t)t * dm;
        for (int o = 0; o < dm; ++o) ot[o] = residual ? xt[o] + acc[o] : acc[o];
        free(lg); free(xin); free(y); free(acc);
    }
    return nomem ? -3 : bad ? -2 : 0;
}

/* The layer with Q8_0 experts. */
int oracle_moe_layer(int T, int dm, int f, int E, int k, const double* x, const float* Wr, const float* bias,
                     const uint8_t* gate, const uint8_t* up, const uint8_t* down, int residual,
                     int expert_input_bf16, const int32_t* forced_idx, double* out, int32_t* idx, double* w,
                     double* logits) {
    return oracle_moe_layer_fmt(T, dm, f, E, k, x, Wr, bias, gate, up, down, 0, residual, expert_input_bf16,
                                forced_idx, out, idx, w, logits);
}

/*
 * Compact expert grouping: a stable counting sort of the T*k (token, slot)
 * pairs by expert id.
 *   off [E+1]: off[e] = number of pairs with expert < e (off[E] = T*k)
 *   pair_tok, pair_slot [T*k]: the pairs in bucket order; within one expert,
 *       ascending (token, slot)
 *   pos [T*k]: pos[t*k + s] = bucket position of pair (t, s)
 * Returns 0, -1 if an id is out of range (outputs then undefined), or -3 when
 * scratch memory could not be allocated.
 */
int oracle_bucket(const int32_t* idx, int T, int k, int E, int32_t* off, int32_t* pair_tok, int32_t* pair_slot,
                  int32_t* pos) {
    if (T < 0 || k <= 0 || E <= 0) return -1;
    int32_t* cnt = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    if (!cnt) return -3;
    for (long p = 0; p < (long)T * k; ++p) {
        int e = idx[p];
        if (e < 0 || e >= E) { free(cnt); return -1; }
        cnt[e]++;
    }
    off[0] = 0;
    for (int e = 0; e < E; ++e) off[e + 1] = off[e] + cnt[e];
    memset(cnt, 0, sizeof(int32_t) * (size_t)E);
    for (int t = 0; t < T; ++t) {
        for (int s = 0; s < k; ++s) {
            int e = idx[(size_t)t * k + s];
            int p = off[e] + cnt[e]++;
            pair_tok[p] = t;
            pair_slot[p] = s;
            pos[(size_t)t * k + s] = p;
        }
    }
    free(cnt);
    return 0;
}
