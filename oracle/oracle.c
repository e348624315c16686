/*
 * oracle.c -- fp64 host oracle for the tensor-parallel sharded linear layer
 * and the Megatron-style MLP block built from it.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
 * and the bench's CPU-baseline / reference arm load this library.  It shares
 * no code, header, table or helper with the CUDA path.
 *
 * Every routine is the plain definition written out: naive loops, double
 * accumulation, no blocking, no fusion, no reordering beyond what the
 * definition states.  The only liberty taken is running independent output
 * rows on several host threads (OpenMP), which does not change any sum.
 *
 * Sources (web pages on tensor parallelism; see the Python wrapper for the
 * list of readings taken where the pages are silent):
 *   [TP-topic]  chipfoundryservices.com, "Tensor Parallelism" topic page:
 *               "Tensor Parallelism Fundamentals", "Column-Wise Parallelism",
 *               "Row-Wise Parallelism", "Megatron-LM Tensor Parallelism",
 *               and the SVG figure's "Attention Head Parallelism" panel.
 *   [Glossary]  aiforbusinessandlife.com glossary "Tensor Parallelism":
 *               "How it works" and "Worked example".
 *
 * All matrices are row-major.  Y = X W with X [M,K], W [K,N], Y [M,N].
 */
#define _GNU_SOURCE
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* The unsharded linear map.                                                */
/* ------------------------------------------------------------------------ */

/* Y[M,N] = X[M,K] . W[K,N]  ([TP-topic] Fundamentals, "Y = XW").
 * y[i][j] = sum over k = 0..K-1, in ascending k, of x[i][k] * w[k][j]. */
void orc_matmul(const double *X, const double *W, double *Y,
                int64_t M, int64_t K, int64_t N)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) {
        double *y = Y + i * N;
        for (int64_t j = 0; j < N; ++j)
            y[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double x = X[i * K + k];
            const double *w = W + k * N;
            for (int64_t j = 0; j < N; ++j)
                y[j] += x * w[j];
        }
    }
}

/* Exact GeLU: x * Phi(x), Phi the standard normal CDF.  The pages only say
 * an activation is applied to each shard with no exchange ([TP-topic]
 * Megatron-LM, "MLP Layer Splitting"); the exact (erf) GeLU is the reading
 * taken for every MLP block.  Phi(x) = (1 + erf(x/sqrt 2))/2 is evaluated as
 * erfc(-x/sqrt 2)/2 (the same function; host libm erfc), which keeps full
 * relative precision in the negative tail where 1 + erf cancels. */
double orc_gelu(double x)
{
    return x * (0.5 * erfc(-x / sqrt(2.0)));
}

void orc_gelu_inplace(double *v, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        v[i] = orc_gelu(v[i]);
}

/* ------------------------------------------------------------------------ */
/* bf16 <-> double, written from the format's definition:                   */
/* 1 sign bit, 8 exponent bits (bias 127, same range as IEEE binary32),     */
/* 7 stored significand bits; rounding to nearest, ties to even.            */
/* ------------------------------------------------------------------------ */

double orc_bf16_to_double(uint16_t b)
{
    const int sign = (b >> 15) & 1;
    const int e = (b >> 7) & 0xFF;
    const int m = b & 0x7F;
    double v;
    if (e == 0xFF)
        v = m ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)m, -126 - 7);           /* subnormal: m * 2^-133 */
    else
        v = ldexp((double)(128 + m), e - 127 - 7); /* 1.m * 2^(e-127) */
    return sign ? -v : v;
}

uint16_t orc_bf16_from_double(double x)
{
    const uint16_t s = signbit(x) ? 0x8000 : 0;
    if (isnan(x))
        return (uint16_t)(s | 0x7FC0);
    double a = fabs(x);
    /* The midpoint between the largest finite value (2-2^-7)*2^127 and 2^128
     * rounds to the even neighbour, 2^128, which is out of range. */
    const double overflow_mid = ldexp(2.0 - ldexp(1.0, -8), 127);
    if (a >= overflow_mid)
        return (uint16_t)(s | 0x7F80);
    if (a == 0.0)
        return s;
    int e2;
    frexp(a, &e2);              /* a = f * 2^e2, f in [0.5, 1) */
    int E = e2 - 1;             /* a = 1.xxx * 2^E */
    if (E < -126)
        E = -126;               /* subnormal range shares the quantum 2^-133 */
    const double q = ldexp(1.0, E - 7);
    const double r = nearbyint(a / q); /* a/q is exact; default mode = ties to even */
    /* r in [0, 256].  For normals r in [128, 256]; r == 256 carries into the
     * exponent.  For subnormals r in [0, 128]; r == 128 is the smallest normal.
     * Both cases are covered by adding r to the biased exponent field. */
    uint32_t bits = (uint32_t)((E + 127 - 1) << 7) + (uint32_t)r;
    if (bits >= 0x7F80)
        return (uint16_t)(s | 0x7F80);
    return (uint16_t)(s | bits);
}

void orc_bf16_to_double_array(const uint16_t *src, double *dst, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = orc_bf16_to_double(src[i]);
}

void orc_double_to_bf16_array(const double *src, uint16_t *dst, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = orc_bf16_from_double(src[i]);
}

/* ------------------------------------------------------------------------ */
/* Column-parallel linear ([TP-topic] "Column-Wise Parallelism"; [Glossary]  */
/* "How it works": splitting W by output columns gives different columns    */
/* of Y, which are concatenated).                                            */
/*                                                                           */
/* W = [W_0, ..., W_{n-1}]; shard i computes Y_i = X . W_i; Y = concat(Y_i). */
/*                                                                           */
/* With col_groups G > 1 the output columns form G equal blocks (for an      */
/* attention QKV projection: Q | K | V) and shard i owns the i-th slice of   */
/* every block -- the head-group split of the SVG figure's "Attention Head   */
/* Parallelism" panel, where each device owns a subset of heads.  With       */
/* gw = N/G and sw = gw/n, shard i owns columns {b*gw + i*sw + j}, b < G,    */
/* j < sw, and its local output is [M, G*sw] ordered block by block.         */
/* ------------------------------------------------------------------------ */
void orc_column_linear(const double *X, const double *W, const double *bias, double *Y,
                       double *Ys, int64_t M, int64_t K, int64_t N, int64_t n_shards,
                       int64_t col_groups, int act_gelu)
{
    const int64_t gw = N / col_groups;
    const int64_t sw = gw / n_shards;
    const int64_t nl = col_groups * sw;
    double *Wi = (double *)malloc(sizeof(double) * (size_t)(K * nl > 0 ? K * nl : 1));
    double *Yi = (double *)malloc(sizeof(double) * (size_t)(M * nl > 0 ? M * nl : 1));
    for (int64_t i = 0; i < n_shards; ++i) {
        /* the shard's weight block, copied out as a separate matrix */
        for (int64_t k = 0; k < K; ++k)
            for (int64_t b = 0; b < col_groups; ++b)
                for (int64_t j = 0; j < sw; ++j)
                    Wi[k * nl + b * sw + j] = W[k * N + b * gw + i * sw + j];
        orc_matmul(X, Wi, Yi, M, K, nl);
        if (bias)   /* the shard's slice of the bias, before the activation */
            for (int64_t r = 0; r < M; ++r)
                for (int64_t b = 0; b < col_groups; ++b)
                    for (int64_t j = 0; j < sw; ++j)
                        Yi[r * nl + b * sw + j] += bias[b * gw + i * sw + j];
        if (act_gelu)
            orc_gelu_inplace(Yi, M * nl);       /* per shard, no exchange */
        /* all-gather: place the shard's columns into the full output */
        if (Y)
            for (int64_t r = 0; r < M; ++r)
                for (int64_t b = 0; b < col_groups; ++b)
                    for (int64_t j = 0; j < sw; ++j)
                        Y[r * N + b * gw + i * sw + j] = Yi[r * nl + b * sw + j];
        if (Ys)
            memcpy(Ys + i * M * nl, Yi, sizeof(double) * (size_t)(M * nl));
    }
    free(Wi);
    free(Yi);
}

/* ------------------------------------------------------------------------ */
/* QKV projection with grouped-query attention heads ([TP-topic] SVG figure, */
/* "Attention Head Parallelism": Q heads split evenly across devices, the    */
/* shared KV heads replicated).  Wqkv = [Wq | Wk | Wv] with hq, hkv, hkv     */
/* heads of hd columns each.  Shard i owns Q heads [i*hq/n, (i+1)*hq/n);     */
/* its KV heads are [i*hkv/n, (i+1)*hkv/n) when n divides hkv (split) and    */
/* the single head floor(i*hkv/n) when hkv divides n (each KV head held by   */
/* n/hkv shards).  Shard i's local output is [M, (hq/n + 2*kvs)*hd] ordered  */
/* Q | K | V (kvs = KV heads per shard); Y is the full projection X.Wqkv in  */
/* Wqkv's column order (the replicated heads appear once).                   */
/* ------------------------------------------------------------------------ */
void orc_qkv_linear(const double *X, const double *W, double *Y, double *Ys, int64_t M,
                    int64_t K, int64_t hq, int64_t hkv, int64_t hd, int64_t n_shards)
{
    const int64_t N = (hq + 2 * hkv) * hd;
    const int64_t qs = hq / n_shards;
    const int64_t kvs = hkv >= n_shards ? hkv / n_shards : 1;
    const int64_t nl = (qs + 2 * kvs) * hd;
    int64_t *cols = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nl > 0 ? nl : 1));
    double *Wi = (double *)malloc(sizeof(double) * (size_t)(K * nl > 0 ? K * nl : 1));
    orc_matmul(X, W, Y, M, K, N);
    for (int64_t i = 0; i < n_shards; ++i) {
        const int64_t kv0 = hkv >= n_shards ? i * kvs : (i * hkv) / n_shards;
        int64_t c = 0;
        for (int64_t h = i * qs; h < (i + 1) * qs; ++h)            /* Q heads */
            for (int64_t j = 0; j < hd; ++j) cols[c++] = h * hd + j;
        for (int64_t h = kv0; h < kv0 + kvs; ++h)                  /* K heads */
            for (int64_t j = 0; j < hd; ++j) cols[c++] = hq * hd + h * hd + j;
        for (int64_t h = kv0; h < kv0 + kvs; ++h)                  /* V heads */
            for (int64_t j = 0; j < hd; ++j) cols[c++] = (hq + hkv) * hd + h * hd + j;
        /* the shard's weight columns, copied out; its output X . W_i */
        for (int64_t k = 0; k < K; ++k)
            for (int64_t j = 0; j < nl; ++j)
                Wi[k * nl + j] = W[k * N + cols[j]];
        orc_matmul(X, Wi, Ys + i * M * nl, M, K, nl);
    }
    free(cols);
    free(Wi);
}

/* ------------------------------------------------------------------------ */
/* Row-parallel linear ([TP-topic] "Row-Wise Parallelism": W stacked         */
/* vertically [W_0; ...; W_{n-1}], X split to match, Y_i = X_i . W_i,       */
/* Y = sum_i Y_i; [Glossary] "Worked example": splitting the contracted      */
/* dimension gives partial contributions that are added).                    */
/*                                                                           */
/* Shard i owns rows [i*K/n, (i+1)*K/n) of W and the same columns of X.     */
/* The partials are summed in ascending shard order.  P, if given, receives */
/* the partials as [n, M, N].                                                */
/* ------------------------------------------------------------------------ */
void orc_row_linear(const double *X, const double *W, const double *bias, double *Y,
                    double *P, int64_t M, int64_t K, int64_t N, int64_t n_shards)
{
    const int64_t ks = K / n_shards;
    double *Xi = (double *)malloc(sizeof(double) * (size_t)(M * ks > 0 ? M * ks : 1));
    double *Pi = (double *)malloc(sizeof(double) * (size_t)(M * N > 0 ? M * N : 1));
    for (int64_t t = 0; t < M * N; ++t)
        Y[t] = 0.0;
    for (int64_t i = 0; i < n_shards; ++i) {
        for (int64_t r = 0; r < M; ++r)
            for (int64_t k = 0; k < ks; ++k)
                Xi[r * ks + k] = X[r * K + i * ks + k];
        /* W_i is a contiguous block of rows of W: rows i*ks .. i*ks+ks-1 */
        orc_matmul(Xi, W + i * ks * N, Pi, M, ks, N);
        /* all-reduce: add this shard's partial */
        for (int64_t t = 0; t < M * N; ++t)
            Y[t] += Pi[t];
        if (P)
            memcpy(P + i * M * N, Pi, sizeof(double) * (size_t)(M * N));
    }
    if (bias)   /* added once, after the sum of the shards (not per shard) */
        for (int64_t r = 0; r < M; ++r)
            for (int64_t j = 0; j < N; ++j)
                Y[r * N + j] += bias[j];
    free(Xi);
    free(Pi);
}

/* ------------------------------------------------------------------------ */
/* Megatron-style MLP block ([TP-topic] Megatron-LM, "MLP Layer Splitting":  */
/* first linear split by columns, activation applied independently per      */
/* shard, second linear split by rows, one sum at the end; [TP-topic]        */
/* "Row-Wise Parallelism": the row-split input is already split by the      */
/* preceding column-split layer).                                            */
/*                                                                           */
/* X [M,d], W1 [d,f], W2 [f,d].  Shard i: H_i = GeLU(X . W1_i) [M, f/n];     */
/* P_i = H_i . W2_i with W2_i = rows [i*f/n, (i+1)*f/n) of W2;               */
/* Y = sum_i P_i (ascending i).  Biases (optional): b1 [f] split with W1's  */
/* columns and added per shard before the GeLU; b2 [d] added once after the */
/* sum (a bias per shard would be counted n times).                          */
/* If mirror_h_bf16 != 0, H_i is rounded to bf16 before the second product  */
/* (a diagnostic that separates rounding of the hidden activation from       */
/* other differences; it is not the reference result).                       */
/* ------------------------------------------------------------------------ */
void orc_mlp_block(const double *X, const double *W1, const double *b1, const double *W2,
                   const double *b2, double *Y, int64_t M, int64_t d, int64_t f,
                   int64_t n_shards, int mirror_h_bf16)
{
    const int64_t fs = f / n_shards;
    double *W1i = (double *)malloc(sizeof(double) * (size_t)(d * fs > 0 ? d * fs : 1));
    double *Hi = (double *)malloc(sizeof(double) * (size_t)(M * fs > 0 ? M * fs : 1));
    double *Pi = (double *)malloc(sizeof(double) * (size_t)(M * d > 0 ? M * d : 1));
    for (int64_t t = 0; t < M * d; ++t)
        Y[t] = 0.0;
    for (int64_t i = 0; i < n_shards; ++i) {
        for (int64_t k = 0; k < d; ++k)
            for (int64_t j = 0; j < fs; ++j)
                W1i[k * fs + j] = W1[k * f + i * fs + j];
        orc_matmul(X, W1i, Hi, M, d, fs);
        if (b1)   /* the shard's slice of the first bias, before the activation */
            for (int64_t r = 0; r < M; ++r)
                for (int64_t j = 0; j < fs; ++j)
                    Hi[r * fs + j] += b1[i * fs + j];
        orc_gelu_inplace(Hi, M * fs);
        if (mirror_h_bf16)
            for (int64_t t = 0; t < M * fs; ++t)
                Hi[t] = orc_bf16_to_double(orc_bf16_from_double(Hi[t]));
        orc_matmul(Hi, W2 + i * fs * d, Pi, M, fs, d);
        for (int64_t t = 0; t < M * d; ++t)
            Y[t] += Pi[t];
    }
    if (b2)   /* the second bias once, after the sum */
        for (int64_t r = 0; r < M; ++r)
            for (int64_t j = 0; j < d; ++j)
                Y[r * d + j] += b2[j];
    free(W1i);
    free(Hi);
    free(Pi);
}

/* ------------------------------------------------------------------------ */
/* Backward pass.  The pages give no formulas, only the structure: the       */
/* identity operator that feeds every shard the same input in the forward  */
/* pass becomes an all-reduce (a sum over shards) in the backward pass, and */
/* the forward all-reduce becomes an identity (every shard receives the     */
/* full output gradient) ([TP-topic] Megatron-LM, "Identity Operators");    */
/* each shard computes the gradients of its own 1/N of the weights          */
/* ([TP-topic] "Memory Distribution", gradient memory).  The gradients      */
/* themselves are the chain rule for L = sum(Y * dY) written out shard by   */
/* shard with the transposes copied out as matrices.                        */
/* ------------------------------------------------------------------------ */

/* GeLU'(x) = Phi(x) + x * phi(x), phi the standard normal density. */
double orc_gelu_grad(double x)
{
    return 0.5 * erfc(-x / sqrt(2.0)) + x * exp(-0.5 * x * x) / sqrt(2.0 * M_PI);
}

/* T[c][r] = A[r][c] for A [R, C]. */
static void transpose(const double *A, double *T, int64_t R, int64_t C)
{
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c)
            T[c * R + r] = A[r * C + c];
}

static double *alloc_d(int64_t n)
{
    return (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
}

/* Column-parallel linear Y_i = X . W_i (columns [i*N/n, (i+1)*N/n) of W).
 * Shard i receives its output columns dY_i of dY and computes
 *   dW_i = X^T . dY_i      (its own weight block: columns of dW)
 *   dX_i = dY_i . W_i^T    (a partial of the input gradient)
 * and dX = sum_i dX_i in ascending i (the backward all-reduce). */
void orc_column_linear_backward(const double *X, const double *W, const double *dY,
                                double *dX, double *dW, int64_t M, int64_t K, int64_t N,
                                int64_t n_shards)
{
    const int64_t ns = N / n_shards;
    double *Xt = alloc_d(K * M), *Wi = alloc_d(K * ns), *Wit = alloc_d(ns * K);
    double *dYi = alloc_d(M * ns), *dWi = alloc_d(K * ns), *dXi = alloc_d(M * K);
    transpose(X, Xt, M, K);
    for (int64_t t = 0; t < M * K; ++t)
        dX[t] = 0.0;
    for (int64_t i = 0; i < n_shards; ++i) {
        for (int64_t k = 0; k < K; ++k)
            for (int64_t j = 0; j < ns; ++j)
                Wi[k * ns + j] = W[k * N + i * ns + j];
        for (int64_t r = 0; r < M; ++r)
            for (int64_t j = 0; j < ns; ++j)
                dYi[r * ns + j] = dY[r * N + i * ns + j];
        orc_matmul(Xt, dYi, dWi, K, M, ns);
        for (int64_t k = 0; k < K; ++k)
            for (int64_t j = 0; j < ns; ++j)
                dW[k * N + i * ns + j] = dWi[k * ns + j];
        transpose(Wi, Wit, K, ns);
        orc_matmul(dYi, Wit, dXi, M, ns, K);
        for (int64_t t = 0; t < M * K; ++t)
            dX[t] += dXi[t];
    }
    free(Xt); free(Wi); free(Wit); free(dYi); free(dWi); free(dXi);
}

/* Row-parallel linear Y = sum_i X_i . W_i (rows [i*K/n, (i+1)*K/n) of W and
 * the same columns of X).  Every shard receives the full dY and computes
 *   dW_i = X_i^T . dY      (its own weight block: rows of dW)
 *   dX_i = dY . W_i^T      (its own columns of dX; no exchange). */
void orc_row_linear_backward(const double *X, const double *W, const double *dY,
                             double *dX, double *dW, int64_t M, int64_t K, int64_t N,
                             int64_t n_shards)
{
    const int64_t ks = K / n_shards;
    double *Xi = alloc_d(M * ks), *Xit = alloc_d(ks * M), *Wit = alloc_d(N * ks);
    double *dWi = alloc_d(ks * N), *dXi = alloc_d(M * ks);
    for (int64_t i = 0; i < n_shards; ++i) {
        for (int64_t r = 0; r < M; ++r)
            for (int64_t k = 0; k < ks; ++k)
                Xi[r * ks + k] = X[r * K + i * ks + k];
        transpose(Xi, Xit, M, ks);
        orc_matmul(Xit, dY, dWi, ks, M, N);
        memcpy(dW + i * ks * N, dWi, sizeof(double) * (size_t)(ks * N));
        transpose(W + i * ks * N, Wit, ks, N);
        orc_matmul(dY, Wit, dXi, M, N, ks);
        for (int64_t r = 0; r < M; ++r)
            for (int64_t k = 0; k < ks; ++k)
                dX[r * K + i * ks + k] = dXi[r * ks + k];
    }
    free(Xi); free(Xit); free(Wit); free(dWi); free(dXi);
}

/* MLP block Y = sum_i GeLU(X . W1_i) . W2_i.  Shard i recomputes
 * Z_i = X . W1_i and H_i = GeLU(Z_i), receives the full dY, and computes
 *   dW2_i = H_i^T . dY                 (rows i of dW2)
 *   dZ_i  = (dY . W2_i^T) * GeLU'(Z_i) (elementwise; no exchange)
 *   dW1_i = X^T . dZ_i                 (columns i of dW1)
 *   dX    = sum_i dZ_i . W1_i^T        (ascending i: the backward all-reduce) */
void orc_mlp_block_backward(const double *X, const double *W1, const double *W2,
                            const double *dY, double *dX, double *dW1, double *dW2,
                            int64_t M, int64_t d, int64_t f, int64_t n_shards)
{
    const int64_t fs = f / n_shards;
    double *Xt = alloc_d(d * M), *W1i = alloc_d(d * fs), *W1it = alloc_d(fs * d);
    double *W2it = alloc_d(d * fs), *Zi = alloc_d(M * fs), *Hit = alloc_d(fs * M);
    double *dHi = alloc_d(M * fs), *dWi = alloc_d((d > fs ? d : fs) * (d > fs ? fs : d));
    double *dXi = alloc_d(M * d);
    transpose(X, Xt, M, d);
    for (int64_t t = 0; t < M * d; ++t)
        dX[t] = 0.0;
    for (int64_t i = 0; i < n_shards; ++i) {
        for (int64_t k = 0; k < d; ++k)
            for (int64_t j = 0; j < fs; ++j)
                W1i[k * fs + j] = W1[k * f + i * fs + j];
        orc_matmul(X, W1i, Zi, M, d, fs);
        for (int64_t r = 0; r < M; ++r)
            for (int64_t j = 0; j < fs; ++j)
                Hit[j * M + r] = orc_gelu(Zi[r * fs + j]);
        orc_matmul(Hit, dY, dWi, fs, M, d);                  /* dW2_i [fs, d] */
        memcpy(dW2 + i * fs * d, dWi, sizeof(double) * (size_t)(fs * d));
        transpose(W2 + i * fs * d, W2it, fs, d);
        orc_matmul(dY, W2it, dHi, M, d, fs);                 /* dH_i [M, fs] */
        for (int64_t t = 0; t < M * fs; ++t)
            dHi[t] *= orc_gelu_grad(Zi[t]);                  /* dZ_i */
        orc_matmul(Xt, dHi, dWi, d, M, fs);                  /* dW1_i [d, fs] */
        for (int64_t k = 0; k < d; ++k)
            for (int64_t j = 0; j < fs; ++j)
                dW1[k * f + i * fs + j] = dWi[k * fs + j];
        transpose(W1i, W1it, d, fs);
        orc_matmul(dHi, W1it, dXi, M, fs, d);                /* dX_i [M, d] */
        for (int64_t t = 0; t < M * d; ++t)
            dX[t] += dXi[t];
    }
    free(Xt); free(W1i); free(W1it); free(W2it); free(Zi); free(Hit); free(dHi); free(dWi);
    free(dXi);
}

/* ------------------------------------------------------------------------ */
/* The two combine steps on their own.                                       */
/* ------------------------------------------------------------------------ */

/* All-reduce as an on-device sum: Y[r,c] = sum_i P[i,r,c] over ascending i,
 * in double, from fp32 partials laid out [n, rows, cols]. */
void orc_shard_reduce(const float *P, double *Y, int64_t rows, int64_t cols, int64_t n_shards)
{
    const int64_t total = rows * cols;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < total; ++t) {
        double acc = 0.0;
        for (int64_t i = 0; i < n_shards; ++i)
            acc += (double)P[i * total + t];
        Y[t] = acc;
    }
}

/* All-gather as an on-device concat: n shard outputs [n][rows, G*sw] placed
 * into Y [rows, G*n*sw] with the same column ownership as orc_column_linear. */
void orc_shard_concat(const double *Ys, double *Y, int64_t rows, int64_t shard_cols,
                      int64_t n_shards, int64_t col_groups)
{
    const int64_t sw = shard_cols / col_groups;
    const int64_t N = shard_cols * n_shards;
    const int64_t gw = N / col_groups;
    for (int64_t i = 0; i < n_shards; ++i)
        for (int64_t r = 0; r < rows; ++r)
            for (int64_t b = 0; b < col_groups; ++b)
                for (int64_t j = 0; j < sw; ++j)
                    Y[r * N + b * gw + i * sw + j] = Ys[(i * rows + r) * shard_cols + b * sw + j];
}

/* ------------------------------------------------------------------------ */
/* Sequence parallelism ([TP-topic] "Sequence Parallelism Extension"):       */
/* outside the tensor-parallel block the token (sequence) dimension is split */
/* across the shards, each holding a contiguous subset of the token rows;    */
/* before the block the token subsets are all-gathered (every shard needs    */
/* every token), and after it the shards' partial outputs are all-reduced.  */
/* Reading: after the all-reduce each shard keeps only its own token subset */
/* for the sequence-split part that follows, so the combine is "sum over    */
/* shards, then split by token rows" (a reduce-scatter over token rows).    */
/* Shard i owns token rows [i*Mb, (i+1)*Mb), Mb = M / n.                    */
/* ------------------------------------------------------------------------ */

/* All-gather of token blocks: Xs [n][Mb][cols] -> X [n*Mb][cols]. */
void orc_allgather_rows(const double *Xs, double *X, int64_t n_shards, int64_t rows_per_shard,
                        int64_t cols)
{
    for (int64_t i = 0; i < n_shards; ++i)
        for (int64_t r = 0; r < rows_per_shard; ++r)
            for (int64_t c = 0; c < cols; ++c)
                X[(i * rows_per_shard + r) * cols + c] = Xs[(i * rows_per_shard + r) * cols + c];
}

/* Reduce-scatter over token rows: P [n][M][cols] (shard j's partial output  */
/* for every token) -> Ys [n][M/n][cols], Ys[i] = token rows of shard i of  */
/* sum_j P_j, the sum over ascending j (the all-reduce), then the split.    */
void orc_reduce_scatter_rows(const double *P, double *Ys, int64_t n_shards, int64_t M,
                             int64_t cols)
{
    const int64_t Mb = M / n_shards;
    double *S = (double *)malloc(sizeof(double) * (size_t)(M * cols > 0 ? M * cols : 1));
    for (int64_t t = 0; t < M * cols; ++t) {            /* all-reduce */
        double acc = 0.0;
        for (int64_t j = 0; j < n_shards; ++j)
            acc += P[j * M * cols + t];
        S[t] = acc;
    }
    for (int64_t i = 0; i < n_shards; ++i)             /* keep own token rows */
        for (int64_t r = 0; r < Mb; ++r)
            for (int64_t c = 0; c < cols; ++c)
                Ys[(i * Mb + r) * cols + c] = S[(i * Mb + r) * cols + c];
    free(S);
}

/* MLP block between two sequence-split regions: token blocks Xs [n][Mb][d] */
/* -> all-gather -> per shard i: P_i = GeLU(X . W1_i) . W2_i for every token */
/* -> reduce-scatter over token rows -> Ys [n][Mb][d].                       */
void orc_seq_parallel_mlp_block(const double *Xs, const double *W1, const double *W2,
                                double *Ys, int64_t n_shards, int64_t rows_per_shard, int64_t d,
                                int64_t f)
{
    const int64_t M = n_shards * rows_per_shard, fs = f / n_shards;
    double *X = (double *)malloc(sizeof(double) * (size_t)(M * d > 0 ? M * d : 1));
    double *W1i = (double *)malloc(sizeof(double) * (size_t)(d * fs > 0 ? d * fs : 1));
    double *Hi = (double *)malloc(sizeof(double) * (size_t)(M * fs > 0 ? M * fs : 1));
    double *P = (double *)malloc(sizeof(double) * (size_t)(n_shards * M * d > 0 ? n_shards * M * d : 1));
    orc_allgather_rows(Xs, X, n_shards, rows_per_shard, d);
    for (int64_t i = 0; i < n_shards; ++i) {
        for (int64_t k = 0; k < d; ++k)
            for (int64_t j = 0; j < fs; ++j)
                W1i[k * fs + j] = W1[k * f + i * fs + j];
        orc_matmul(X, W1i, Hi, M, d, fs);
        orc_gelu_inplace(Hi, M * fs);
        orc_matmul(Hi, W2 + i * fs * d, P + i * M * d, M, fs, d);
    }
    orc_reduce_scatter_rows(P, Ys, n_shards, M, d);
    free(X); free(W1i); free(Hi); free(P);
}

/* ------------------------------------------------------------------------ */
/* The MLP block's backward on sampled outputs, for checks at sizes whose   */
/* full fp64 backward is too slow: rows `rx` of dX, columns `c1` of dW1 and */
/* rows `r2` of dW2.  Each sampled value is the same chain rule as          */
/* orc_mlp_block_backward, written per value (no matrix copies):             */
/*   Z[r, j] = sum_k X[r, k] W1[k, j],  H = GeLU(Z),                         */
/*   dZ[r, j] = GeLU'(Z[r, j]) * sum_c dY[r, c] W2[j, c],                    */
/*   dW2[j, c] = sum_r H[r, j] dY[r, c],  dW1[k, j] = sum_r X[r, k] dZ[r, j], */
/*   dX[r, k] = sum over shards i (ascending) of sum_{j in shard i}          */
/*              dZ[r, j] W1[k, j].                                           */
/* ------------------------------------------------------------------------ */
static double z_at(const double *X, const double *W1, int64_t r, int64_t j, int64_t d,
                   int64_t f)
{
    double acc = 0.0;
    for (int64_t k = 0; k < d; ++k)
        acc += X[r * d + k] * W1[k * f + j];
    return acc;
}

static double dz_at(const double *X, const double *W1, const double *W2, const double *dY,
                    int64_t r, int64_t j, int64_t d, int64_t f)
{
    double dh = 0.0;
    for (int64_t c = 0; c < d; ++c)
        dh += dY[r * d + c] * W2[j * d + c];
    return dh * orc_gelu_grad(z_at(X, W1, r, j, d, f));
}

void orc_mlp_block_backward_sampled(const double *X, const double *W1, const double *W2,
                                    const double *dY, int64_t M, int64_t d, int64_t f,
                                    int64_t n_shards, const int64_t *rx, int64_t nrx,
                                    const int64_t *c1, int64_t nc1, const int64_t *r2,
                                    int64_t nr2, double *dXs, double *dW1s, double *dW2s)
{
    const int64_t fs = f / n_shards;
#pragma omp parallel for schedule(dynamic)
    for (int64_t s = 0; s < nrx; ++s) {           /* dX rows */
        const int64_t r = rx[s];
        double *dz = (double *)malloc(sizeof(double) * (size_t)(f > 0 ? f : 1));
        /* Z[r, :] with k outer (rows of W1 read in order; each Z[r, j] is   */
        /* still summed over k ascending), then dZ[r, j]                     */
        for (int64_t j = 0; j < f; ++j)
            dz[j] = 0.0;
        for (int64_t k = 0; k < d; ++k) {
            const double xk = X[r * d + k];
            for (int64_t j = 0; j < f; ++j)
                dz[j] += xk * W1[k * f + j];
        }
        for (int64_t j = 0; j < f; ++j) {
            double dh = 0.0;
            for (int64_t c = 0; c < d; ++c)
                dh += dY[r * d + c] * W2[j * d + c];
            dz[j] = dh * orc_gelu_grad(dz[j]);
        }
        for (int64_t k = 0; k < d; ++k) {
            double tot = 0.0;
            for (int64_t i = 0; i < n_shards; ++i) {
                double part = 0.0;
                for (int64_t j = i * fs; j < (i + 1) * fs; ++j)
                    part += dz[j] * W1[k * f + j];
                tot += part;
            }
            dXs[s * d + k] = tot;
        }
        free(dz);
    }
#pragma omp parallel for schedule(dynamic)
    for (int64_t s = 0; s < nc1; ++s) {           /* dW1 columns */
        const int64_t j = c1[s];
        double *dz = (double *)malloc(sizeof(double) * (size_t)(M > 0 ? M : 1));
        for (int64_t r = 0; r < M; ++r)
            dz[r] = dz_at(X, W1, W2, dY, r, j, d, f);
        for (int64_t k = 0; k < d; ++k) {
            double acc = 0.0;
            for (int64_t r = 0; r < M; ++r)
                acc += X[r * d + k] * dz[r];
            dW1s[k * nc1 + s] = acc;
        }
        free(dz);
    }
#pragma omp parallel for schedule(dynamic)
    for (int64_t s = 0; s < nr2; ++s) {           /* dW2 rows */
        const int64_t j = r2[s];
        double *h = (double *)malloc(sizeof(double) * (size_t)(M > 0 ? M : 1));
        for (int64_t r = 0; r < M; ++r)
            h[r] = orc_gelu(z_at(X, W1, r, j, d, f));
        for (int64_t c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int64_t r = 0; r < M; ++r)
                acc += h[r] * dY[r * d + c];
            dW2s[s * d + c] = acc;
        }
        free(h);
    }
}
