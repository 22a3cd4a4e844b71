/*
 * oracle.c -- plain, slow, single-threaded CPU oracle for the fused operator chains.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call this
 * file: only the tests, the package's smoke check and the benchmark's CPU-baseline leg
 * use it.  It shares no code, header, table or constant with the CUDA path.
 *
 * What it computes is the *unfused* chain, one operator after another, exactly as the
 * pages define the operators; the fused GPU kernels must reproduce it.
 *
 *   BOLT notes, "Persistent kernel (GEMM/Conv) fusion" and "Threadblock residence":
 *       GEMM0 -> epilogue -> GEMM1 (-> epilogue), the second GEMM reading the first
 *       one's output tile.
 *   BOLT notes, "Prerequisite: Epilogue fusion": element-wise operator, dtype
 *       conversion, column-broadcast vector (the bias).
 *   BOLT notes, "Graph Level": Conv2D + BiasAdd + Hardswish as one operator.
 *   Welder notes, "Operator-tile and Tile-graph" and "Tile-graph Scheduling"
 *       (Figure 5): Conv computes a 1x1xC output from a 3x3xC input tile; ReLU; MaxPool
 *       reduces a 2x2xF reuse tile to 1x1xF.
 *   Interview notes, "Conv optimisation", item 5: a 1x1 conv is a GEMM.
 *   Welder notes, "Operator-tile and Tile-graph", tile propagation: a strided conv reads
 *       a strided (non-contiguous) input region.
 *   Interview notes, TVM Relay vs. TIR scheduling primitives, SimplifyInference: batch
 *       normalisation becomes a scale and a bias at inference, which folded into the
 *       preceding conv's weights and bias is the chain's bias epilogue.
 *
 * Arithmetic:
 *   - every stored tensor is fp16 or bf16 (bit patterns in uint16_t);
 *   - products and sums are formed in double precision, summed in ascending reduction
 *     index starting from 0.0; the bias is added after the full sum;
 *   - the activation is applied in double precision;
 *   - the result is rounded once, to nearest with ties to even, to the storage type;
 *   - the chain's intermediate is stored in the storage type (that rounding is part
 *     of what the fused kernel computes: it writes an fp16/bf16 tile on chip).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - conv is cross-correlation, dilation 1, zero padding `pad`, stride `stride` in both
 *     spatial dimensions (1 unless given);
 *   - weight layouts: GEMM W[K][N] row-major; conv W[Cout][R][S][Cin];
 *   - hardswish(x) = x * min(max(x + 3, 0), 6) / 6;
 *   - max-pool 2x2, stride 2, floor mode (odd trailing row/column dropped).
 *
 * Build:  gcc -O2 -ffp-contract=off -fPIC -shared oracle.c -o liboracle.so -lm
 * (-ffp-contract=off keeps a*b+c as two roundings on every host, x86 or Arm.)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_F16 = 0, OR_BF16 = 1 };
enum { OR_ACT_NONE = 0, OR_ACT_RELU = 1, OR_ACT_HARDSWISH = 2 };
enum { OR_OK = 0, OR_BAD_ARG = 1, OR_NO_MEM = 2 };

/* ------------------------------------------------------------------------------------ */
/* Storage formats.                                                                      */
/*   fp16 (IEEE binary16): 1 sign, 5 exponent (bias 15), 10 fraction bits.              */
/*   bf16: 1 sign, 8 exponent (bias 127), 7 fraction bits.                              */
/* ------------------------------------------------------------------------------------ */

typedef struct {
    int frac_bits;   /* stored fraction bits */
    int exp_bits;    /* exponent field width */
    int bias;        /* exponent bias */
} or_format;

static or_format fmt_of(int dt)
{
    or_format f;
    if (dt == OR_BF16) { f.frac_bits = 7; f.exp_bits = 8; f.bias = 127; }
    else               { f.frac_bits = 10; f.exp_bits = 5; f.bias = 15; }
    return f;
}

/* Exact value of a stored bit pattern. */
double oracle_decode(int dt, uint16_t bits)
{
    or_format f = fmt_of(dt);
    int sign = (bits >> 15) & 1;
    int emax_field = (1 << f.exp_bits) - 1;
    int e = (bits >> f.frac_bits) & emax_field;
    uint32_t frac = bits & ((1u << f.frac_bits) - 1u);
    double v;
    if (e == emax_field) {
        v = frac ? NAN : INFINITY;
    } else if (e == 0) {
        /* subnormal: frac * 2^(1 - bias - frac_bits) */
        v = ldexp((double)frac, 1 - f.bias - f.frac_bits);
    } else {
        v = ldexp((double)((1u << f.frac_bits) | frac), e - f.bias - f.frac_bits);
    }
    return sign ? -v : v;
}

/* Round a double to the storage format: nearest, ties to even; overflow to infinity. */
uint16_t oracle_encode(int dt, double v)
{
    or_format f = fmt_of(dt);
    const int p = f.frac_bits + 1;                 /* significand precision */
    const int emin = 1 - f.bias;                   /* smallest normal exponent */
    const int emax = f.bias;                       /* largest finite exponent */
    const uint16_t inf_bits = (uint16_t)(((1u << f.exp_bits) - 1u) << f.frac_bits);
    uint16_t sign_bit = 0;
    double a, n, fl, diff, r;
    int e;

    if (isnan(v)) return (uint16_t)(inf_bits | (1u << (f.frac_bits - 1)));
    if (signbit(v)) { sign_bit = 0x8000; a = -v; } else { a = v; }
    if (a == 0.0) return sign_bit;
    if (isinf(a)) return (uint16_t)(sign_bit | inf_bits);

    /* a = m * 2^ex with m in [0.5, 1): the leading bit has weight 2^(ex-1). */
    (void)frexp(a, &e);
    e -= 1;
    if (e < emin) e = emin;                        /* subnormal range: fixed quantum */
    if (e > emax + 1) return (uint16_t)(sign_bit | inf_bits);

    /* n = a / quantum, where quantum = 2^(e - (p-1)); scaling by a power of two is exact. */
    n = ldexp(a, (p - 1) - e);
    fl = floor(n);
    diff = n - fl;                                 /* exact: n < 2^p here */
    if (diff > 0.5) r = fl + 1.0;
    else if (diff < 0.5) r = fl;
    else r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;

    if (r >= ldexp(1.0, p)) {                      /* carried into the next binade */
        r = ldexp(1.0, p - 1);
        e += 1;
    }
    if (r >= ldexp(1.0, p - 1)) {                  /* normal */
        if (e > emax) return (uint16_t)(sign_bit | inf_bits);
        {
            uint32_t field = (uint32_t)(e + f.bias);
            uint32_t frac = (uint32_t)(r - ldexp(1.0, p - 1));
            return (uint16_t)(sign_bit | (field << f.frac_bits) | frac);
        }
    }
    /* subnormal (or rounded to zero) */
    return (uint16_t)(sign_bit | (uint32_t)r);
}

void oracle_decode_array(int dt, int64_t n, const uint16_t* in, double* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_decode(dt, in[i]);
}

void oracle_encode_array(int dt, int64_t n, const double* in, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_encode(dt, in[i]);
}

/* ------------------------------------------------------------------------------------ */
/* Epilogue element-wise operators (BOLT notes, "Graph Level" and "Epilogue fusion").     */
/* ------------------------------------------------------------------------------------ */

double oracle_activation(int act, double x)
{
    switch (act) {
    case OR_ACT_RELU:
        return x > 0.0 ? x : 0.0;
    case OR_ACT_HARDSWISH: {
        double t = x + 3.0;
        if (t < 0.0) t = 0.0;
        if (t > 6.0) t = 6.0;
        return x * t / 6.0;
    }
    default:
        return x;
    }
}

static double* decode_alloc(int dt, int64_t n, const uint16_t* in)
{
    double* out = (double*)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    if (out) oracle_decode_array(dt, n, in, out);
    return out;
}

/* ------------------------------------------------------------------------------------ */
/* One GEMM stage with its epilogue:                                                      */
/*   out[m][n] = rnd( act( b[n] + sum_{k=0}^{K-1} A[m][k] * W[k][n] ) )                   */
/* A [M][K], W [K][N] row-major; b [N] or NULL (no bias); out [M][N].                     */
/* ------------------------------------------------------------------------------------ */
int oracle_gemm_bias_act(int dt, int64_t M, int64_t K, int64_t N,
                         const uint16_t* A, const uint16_t* W, const uint16_t* b,
                         int act, uint16_t* out)
{
    double *w, *arow, *acc;
    if (M < 0 || K < 0 || N < 0 || !A || !W || !out) return OR_BAD_ARG;
    w = decode_alloc(dt, K * N, W);
    arow = (double*)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
    acc = (double*)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    if (!w || !arow || !acc) { free(w); free(arow); free(acc); return OR_NO_MEM; }

    for (int64_t m = 0; m < M; ++m) {
        oracle_decode_array(dt, K, A + m * K, arow);
        for (int64_t n = 0; n < N; ++n) acc[n] = 0.0;
        /* For each output element the terms are added in ascending k. */
        for (int64_t k = 0; k < K; ++k) {
            const double a = arow[k];
            const double* wk = w + k * N;
            for (int64_t n = 0; n < N; ++n) acc[n] += a * wk[n];
        }
        for (int64_t n = 0; n < N; ++n) {
            double z = acc[n] + (b ? oracle_decode(dt, b[n]) : 0.0);
            out[m * N + n] = oracle_encode(dt, oracle_activation(act, z));
        }
    }
    free(w); free(arow); free(acc);
    return OR_OK;
}

/* GEMM0 -> epilogue0 -> (intermediate stored in the storage type) -> GEMM1 -> epilogue1.
 * A [M][K0], W0 [K0][N0], W1 [N0][N1], out [M][N1].  Rows are independent, so the
 * intermediate is formed one block of rows at a time to bound memory. */
int oracle_b2b_gemm(int dt, int64_t M, int64_t K0, int64_t N0, int64_t N1,
                    const uint16_t* A, const uint16_t* W0, const uint16_t* b0, int act0,
                    const uint16_t* W1, const uint16_t* b1, int act1, uint16_t* out)
{
    const int64_t block = 4096;
    uint16_t* h;
    if (M < 0 || K0 < 0 || N0 < 0 || N1 < 0 || !A || !W0 || !W1 || !out) return OR_BAD_ARG;
    h = (uint16_t*)malloc((size_t)((block * N0) > 0 ? block * N0 : 1) * sizeof(uint16_t));
    if (!h) return OR_NO_MEM;
    for (int64_t m0 = 0; m0 < M; m0 += block) {
        int64_t rows = (M - m0 < block) ? (M - m0) : block;
        int rc = oracle_gemm_bias_act(dt, rows, K0, N0, A + m0 * K0, W0, b0, act0, h);
        if (rc == OR_OK) rc = oracle_gemm_bias_act(dt, rows, N0, N1, h, W1, b1, act1, out + m0 * N1);
        if (rc != OR_OK) { free(h); return rc; }
    }
    free(h);
    return OR_OK;
}

/* ------------------------------------------------------------------------------------ */
/* Direct 2-D convolution, NHWC, stride st, zero padding `pad`, cross-correlation:        */
/*   z[n][h][w][co] = b[co] + sum_{r<R} sum_{s<S} sum_{ci<C}                              */
/*                      x[n][st*h+r-pad][st*w+s-pad][ci] * Wt[co][r][s][ci]                */
/* with x taken as 0 outside [0,H) x [0,W).  The sum runs r, then s, then ci.             */
/* Output spatial size Ho = (H + 2*pad - R) / st + 1, Wo = (W + 2*pad - S) / st + 1       */
/* (floor; no output if H + 2*pad < R or W + 2*pad < S).                                  */
/* out[n][h][w][co] = rnd(act(z)).                                                        */
/* ------------------------------------------------------------------------------------ */
static int64_t conv_out_size(int64_t in, int64_t pad, int64_t k, int64_t st)
{
    return in + 2 * pad < k ? 0 : (in + 2 * pad - k) / st + 1;
}

int oracle_conv2d_nhwc_strided(int dt, int64_t N, int64_t H, int64_t W, int64_t C,
                               const uint16_t* x, int64_t Co, int64_t R, int64_t S, int64_t pad,
                               int64_t st, const uint16_t* Wt, const uint16_t* b, int act,
                               uint16_t* out)
{
    const int64_t Ho = conv_out_size(H, pad, R, st), Wo = conv_out_size(W, pad, S, st);
    double *wt, *img, *acc;
    if (N < 0 || H < 0 || W < 0 || C < 0 || Co < 0 || R < 1 || S < 1 || pad < 0 || st < 1)
        return OR_BAD_ARG;
    if (!x || !Wt || !out) return OR_BAD_ARG;
    if (Ho <= 0 || Wo <= 0) return OR_OK;
    wt = decode_alloc(dt, Co * R * S * C, Wt);
    img = (double*)malloc((size_t)((H * W * C) > 0 ? H * W * C : 1) * sizeof(double));
    acc = (double*)malloc((size_t)(Co > 0 ? Co : 1) * sizeof(double));
    if (!wt || !img || !acc) { free(wt); free(img); free(acc); return OR_NO_MEM; }

    for (int64_t n = 0; n < N; ++n) {
        oracle_decode_array(dt, H * W * C, x + n * H * W * C, img);
        for (int64_t ho = 0; ho < Ho; ++ho) {
            for (int64_t wo = 0; wo < Wo; ++wo) {
                for (int64_t co = 0; co < Co; ++co) {
                    double s_acc = 0.0;
                    for (int64_t r = 0; r < R; ++r) {
                        const int64_t hi = st * ho + r - pad;
                        if (hi < 0 || hi >= H) continue;      /* zero padding row */
                        for (int64_t s = 0; s < S; ++s) {
                            const int64_t wi = st * wo + s - pad;
                            const double* xp;
                            const double* wp;
                            if (wi < 0 || wi >= W) continue;  /* zero padding column */
                            xp = img + (hi * W + wi) * C;
                            wp = wt + ((co * R + r) * S + s) * C;
                            for (int64_t ci = 0; ci < C; ++ci) s_acc += xp[ci] * wp[ci];
                        }
                    }
                    acc[co] = s_acc;
                }
                for (int64_t co = 0; co < Co; ++co) {
                    double z = acc[co] + (b ? oracle_decode(dt, b[co]) : 0.0);
                    out[((n * Ho + ho) * Wo + wo) * Co + co] = oracle_encode(dt, oracle_activation(act, z));
                }
            }
        }
    }
    free(wt); free(img); free(acc);
    return OR_OK;
}

int oracle_conv2d_nhwc(int dt, int64_t N, int64_t H, int64_t W, int64_t C,
                       const uint16_t* x, int64_t Co, int64_t R, int64_t S, int64_t pad,
                       const uint16_t* Wt, const uint16_t* b, int act, uint16_t* out)
{
    return oracle_conv2d_nhwc_strided(dt, N, H, W, C, x, Co, R, S, pad, 1, Wt, b, act, out);
}

/* Max-pool 2x2, stride 2, floor mode, NHWC: out [N][H/2][W/2][C].  The maximum of
 * four stored values is one of them, so the result is copied, never re-rounded. */
int oracle_maxpool2x2_nhwc(int dt, int64_t N, int64_t H, int64_t W, int64_t C,
                           const uint16_t* x, uint16_t* out)
{
    const int64_t Hp = H / 2, Wp = W / 2;
    if (N < 0 || H < 0 || W < 0 || C < 0 || !x || !out) return OR_BAD_ARG;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t i = 0; i < Hp; ++i)
            for (int64_t j = 0; j < Wp; ++j)
                for (int64_t c = 0; c < C; ++c) {
                    uint16_t best = x[((n * H + 2 * i) * W + 2 * j) * C + c];
                    double bv = oracle_decode(dt, best);
                    for (int64_t dy = 0; dy < 2; ++dy)
                        for (int64_t dx = 0; dx < 2; ++dx) {
                            uint16_t cand = x[((n * H + 2 * i + dy) * W + 2 * j + dx) * C + c];
                            double cv = oracle_decode(dt, cand);
                            if (cv > bv) { bv = cv; best = cand; }
                        }
                    out[((n * Hp + i) * Wp + j) * C + c] = best;
                }
    return OR_OK;
}

/* conv(R x S, pad, stride st) + bias + act0 -> intermediate (storage type) -> 1x1 conv
 * (stride 1) + bias + act1.  x [N][H][W][C], W0 [C0][R][S][C], W1 [C1][C0],
 * out [N][Ho][Wo][C1].  Images are independent, so the intermediate is formed one image
 * at a time. */
int oracle_b2b_conv_nhwc_strided(int dt, int64_t N, int64_t H, int64_t W, int64_t C,
                                 const uint16_t* x, const uint16_t* W0, int64_t C0, int64_t R,
                                 int64_t S, int64_t pad, int64_t st, const uint16_t* b0, int act0,
                                 const uint16_t* W1, int64_t C1, const uint16_t* b1, int act1,
                                 uint16_t* out)
{
    const int64_t Ho = st >= 1 ? conv_out_size(H, pad, R, st) : 0;
    const int64_t Wo = st >= 1 ? conv_out_size(W, pad, S, st) : 0;
    uint16_t* h;
    if (N < 0 || st < 1 || !x || !W0 || !W1 || !out) return OR_BAD_ARG;
    if (Ho <= 0 || Wo <= 0) return OR_OK;
    h = (uint16_t*)malloc((size_t)((Ho * Wo * C0) > 0 ? Ho * Wo * C0 : 1) * sizeof(uint16_t));
    if (!h) return OR_NO_MEM;
    for (int64_t n = 0; n < N; ++n) {
        int rc = oracle_conv2d_nhwc_strided(dt, 1, H, W, C, x + n * H * W * C, C0, R, S, pad, st,
                                            W0, b0, act0, h);
        if (rc == OR_OK)
            rc = oracle_conv2d_nhwc(dt, 1, Ho, Wo, C0, h, C1, 1, 1, 0, W1, b1, act1,
                                    out + n * Ho * Wo * C1);
        if (rc != OR_OK) { free(h); return rc; }
    }
    free(h);
    return OR_OK;
}

int oracle_b2b_conv_nhwc(int dt, int64_t N, int64_t H, int64_t W, int64_t C,
                         const uint16_t* x, const uint16_t* W0, int64_t C0, int64_t R, int64_t S,
                         int64_t pad, const uint16_t* b0, int act0,
                         const uint16_t* W1, int64_t C1, const uint16_t* b1, int act1,
                         uint16_t* out)
{
    return oracle_b2b_conv_nhwc_strided(dt, N, H, W, C, x, W0, C0, R, S, pad, 1, b0, act0, W1, C1,
                                        b1, act1, out);
}

/* Batch normalisation folded into the weights and bias of the operator before it
 * (interview notes, SimplifyInference: BN becomes scale and bias at inference):
 *   y = gamma * (z - mean) / sqrt(var + eps) + beta,   z = sum_k W[co][k] x[k] + b[co]
 *     = sum_k (W[co][k] * s[co]) x[k] + ((b[co] - mean[co]) * s[co] + beta[co]),
 *   s[co] = gamma[co] / sqrt(var[co] + eps).
 * W is [Co][K] (out_inner = 0: conv filters [Co][R][S][Cin], K = R*S*Cin) or [K][Co]
 * (out_inner = 1: row-major GEMM weights); gamma, beta, mean, var are fp32 (float), b
 * may be NULL (0).  Each folded value is formed in double and rounded once to the
 * storage type. */
int oracle_fold_batchnorm(int dt, int64_t Co, int64_t K, int out_inner, const uint16_t* Wt,
                          const uint16_t* b, const float* gamma, const float* beta,
                          const float* mean, const float* var, double eps, uint16_t* W_out,
                          uint16_t* b_out)
{
    if (Co < 0 || K < 0 || !Wt || !gamma || !beta || !mean || !var || !W_out || !b_out)
        return OR_BAD_ARG;
    for (int64_t co = 0; co < Co; ++co) {
        const double s = (double)gamma[co] / sqrt((double)var[co] + eps);
        const double bias = b ? oracle_decode(dt, b[co]) : 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const int64_t i = out_inner ? k * Co + co : co * K + k;
            W_out[i] = oracle_encode(dt, oracle_decode(dt, Wt[i]) * s);
        }
        b_out[co] = oracle_encode(dt, (bias - (double)mean[co]) * s + (double)beta[co]);
    }
    return OR_OK;
}

/* conv3x3 (pad 1, stride 1) + bias + ReLU -> intermediate (storage type) -> max-pool 2x2/2.
 * x [N][H][W][Cin], Wt [Cout][3][3][Cin], out [N][H/2][W/2][Cout]. */
int oracle_conv_relu_maxpool(int dt, int64_t N, int64_t H, int64_t W, int64_t Cin,
                             const uint16_t* x, const uint16_t* Wt, const uint16_t* b, int64_t Cout,
                             uint16_t* out)
{
    const int64_t Hp = H / 2, Wp = W / 2;
    uint16_t* c;
    if (N < 0 || !x || !Wt || !out) return OR_BAD_ARG;
    c = (uint16_t*)malloc((size_t)((H * W * Cout) > 0 ? H * W * Cout : 1) * sizeof(uint16_t));
    if (!c) return OR_NO_MEM;
    for (int64_t n = 0; n < N; ++n) {
        int rc = oracle_conv2d_nhwc(dt, 1, H, W, Cin, x + n * H * W * Cin, Cout, 3, 3, 1, Wt, b,
                                    OR_ACT_RELU, c);
        if (rc == OR_OK) rc = oracle_maxpool2x2_nhwc(dt, 1, H, W, Cout, c, out + n * Hp * Wp * Cout);
        if (rc != OR_OK) { free(c); return rc; }
    }
    free(c);
    return OR_OK;
}
