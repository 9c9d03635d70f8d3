/*
 * gemm_oracle.c -- plain CPU oracle for the half-precision GEMM with a fused
 * ReLU epilogue, C = ReLU(A @ B).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; it is used by the tests, by the smoke check and by the
 * bench's CPU-baseline leg.  It shares no code, header, table or constant
 * with the CUDA path.
 *
 * What it computes (written out from the definition, nothing reordered):
 *
 *   C[i,j] = f16_rne( R( sum_{k=0..K-1} (double)A[i,k] * (double)B[k,j] ) )
 *
 *   A (M,K), B (K,N), C (M,N): dense row-major IEEE binary16, leading
 *   dimensions K, N and N.  R(x) = (x > 0) ? x : +0 when relu is set, else x.
 *
 * Sources, all on "Writing High-Performance Kernels in TileLang, from GEMM to
 * MLA" (atlascloud.ai), section "Let's write a GEMM": the kernel computes
 * C = ReLU(A @ B) with A (M,K), B (K,N) and C (M,N) in float16; the
 * accumulator fragment is declared in float (fp32); ReLU is applied to the
 * accumulator (max with 0) and the accumulator is then copied out to the
 * float16 C, i.e. one cast at write-back.  The TileLang-MUSA lesson
 * (7yue.com, section 3, "first TileLang kernel: GEMM") has the same
 * contraction without ReLU and checks it against A.float() @ B.float().
 *
 * Readings where the pages leave a step open:
 *   - accumulation: widened here to fp64 (every fp16 x fp16 product is exact
 *     in fp64; the sum's own rounding is far below one fp16 ulp), summed in
 *     ascending k for every output element;
 *   - ReLU: applied to the accumulator before the cast; every x <= 0, -0 and
 *     NaN give +0 (the "(x > 0) ? x : 0" reading of max(x, 0));
 *   - cast: IEEE-754 round-to-nearest-even, overflow to +-inf, subnormals
 *     kept (the rounding of the fp32 -> fp16 copy is not stated on the pages);
 *   - K == 0: the empty sum is +0, so C = R(+0) = +0.
 *
 * Loop order: rows i in parallel (OpenMP), then k, then j with one fp64
 * accumulator per output column of the row.  Each C[i,j] is still the sum
 * over k in ascending order, exactly as the i-j-k loop would form it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <omp.h>

/* IEEE binary16 -> binary64 (exact).  Layout: 1 sign bit, 5 exponent bits
 * (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int e = (h >> 10) & 0x1f;
    const int m = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24);              /* zero or subnormal: m * 2^-24 */
    } else if (e == 31) {
        v = (m == 0) ? INFINITY : NAN;          /* infinity or NaN */
    } else {
        v = ldexp((double)(m + 1024), e - 25);  /* (1 + m/2^10) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* IEEE binary64 -> binary16, round to nearest, ties to even.  Relies on the
 * default floating-point environment (FE_TONEAREST) for nearbyint(). */
uint16_t oracle_f64_to_f16(double x)
{
    const uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | 0x7e00u);
    const double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | 0x7c00u);
    if (a < ldexp(1.0, -14)) {
        /* Subnormal range: the representable values are q * 2^-24 for
         * integer q.  Scaling by 2^24 is exact; q == 1024 is the smallest
         * normal number and its encoding is the same integer. */
        const double q = nearbyint(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)q);
    }
    int e2;
    (void)frexp(a, &e2);           /* a in [2^(e2-1), 2^e2) */
    int E = e2 - 1;                /* unbiased exponent, E >= -14 here */
    double q = nearbyint(ldexp(a, 10 - E));   /* significand * 2^10, in [1024, 2048] */
    if (q == 2048.0) {             /* rounded up into the next binade */
        q = 1024.0;
        E += 1;
    }
    if (E > 15) return (uint16_t)(sign | 0x7c00u);   /* overflow -> infinity */
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(q - 1024.0));
}

/* Decoded value of every binary16 bit pattern, filled from
 * oracle_f16_to_f64 before any row is computed. */
static double g_f16_value[65536];
static int g_f16_value_ready = 0;

static void fill_f16_values(void)
{
    if (g_f16_value_ready) return;
    for (int h = 0; h < 65536; ++h) g_f16_value[h] = oracle_f16_to_f64((uint16_t)h);
    g_f16_value_ready = 1;
}

/*
 * Computes the requested output rows.  rows[r] (0 <= rows[r] < M) names an
 * output row; its N values are written to C_out[r*N .. r*N+N-1].  Passing
 * rows = NULL means every row 0..M-1 in order (n_rows must then be M).
 * Returns 0 on success, -1 on bad arguments or allocation failure.
 */
int oracle_gemm_f16_rows(const uint16_t *A, const uint16_t *B, uint16_t *C_out,
                         int64_t M, int64_t N, int64_t K, int relu,
                         const int64_t *rows, int64_t n_rows)
{
    if (M < 0 || N < 0 || K < 0 || n_rows < 0) return -1;
    if (rows == NULL && n_rows != M) return -1;
    for (int64_t r = 0; rows != NULL && r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= M) return -1;
    if (n_rows == 0 || N == 0) return 0;
    fill_f16_values();

    int failed = 0;
#pragma omp parallel
    {
        double *acc = (double *)malloc((size_t)N * sizeof(double));
        if (acc == NULL) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n_rows; ++r) {
            if (acc == NULL) continue;
            const int64_t i = rows ? rows[r] : r;
            for (int64_t j = 0; j < N; ++j) acc[j] = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double a = g_f16_value[A[i * K + k]];
                const uint16_t *b_row = B + k * N;
                for (int64_t j = 0; j < N; ++j) acc[j] += a * g_f16_value[b_row[j]];
            }
            uint16_t *c_row = C_out + r * N;
            for (int64_t j = 0; j < N; ++j) {
                double x = acc[j];
                if (relu) x = (x > 0.0) ? x : 0.0;
                c_row[j] = oracle_f64_to_f16(x);
            }
        }
        free(acc);
    }
    return failed ? -1 : 0;
}

/* Whole matrix: C (M,N) row-major. */
int oracle_gemm_f16(const uint16_t *A, const uint16_t *B, uint16_t *C,
                    int64_t M, int64_t N, int64_t K, int relu)
{
    return oracle_gemm_f16_rows(A, B, C, M, N, K, relu, NULL, M);
}

/* Number of threads an OpenMP parallel region of this library uses. */
int oracle_num_threads(void)
{
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        n = omp_get_num_threads();
    }
    return n;
}

/*
 * Gradient through the ReLU epilogue, for the backward pass of C = ReLU(A @ B):
 * dZ[i] = dC[i] where C[i] > 0, else +0.  C is the stored forward output (its
 * value decides the sign of the pre-activation, which is not kept); +inf > 0,
 * NaN is not > 0.  The autograd wrapper of the TileLang-MUSA lesson (7yue.com,
 * section 6) then forms dA = dZ @ B^T and dB = A^T @ dZ.
 */
void oracle_relu_backward(const uint16_t *dC, const uint16_t *C, uint16_t *dZ, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        const double c = oracle_f16_to_f64(C[i]);
        dZ[i] = (c > 0.0) ? dC[i] : (uint16_t)0x0000u;
    }
}

/* ======================================================================
 * FP8 block-scaled GEMM (TEST INFRASTRUCTURE ONLY, like everything above).
 *
 * The TileLang-MUSA lesson (7yue.com, section 8.2, "reusing TileKernels")
 * calls a linear layer on an FP8 weight with per-block scales,
 * fp8_block_scaled_linear(x, w_fp8, scale_w, block=128), and the nxmr.cn
 * TileLang article (section 7) names CUTLASS-style per-block scaling as the
 * way FP8 GEMMs are scaled.  Neither page writes out the arithmetic; the
 * plainest reading, which this function follows, is:
 *
 *   C[i,j] = f16_rne( R( sum_b  SA[i,b] * SW[j/block, b] * P_b[i,j] ) ),
 *   P_b[i,j] = sum_{k in block b, k < K} A[i,k] * W[j,k]
 *
 *   A (M,K) and W (N,K): row-major OCP FP8 E4M3 (the weight is stored
 *   out-features x in-features, as a linear layer keeps it, so C = A @ W^T);
 *   SA (M, KB): one fp32 scale per row of A per block of `block` K elements;
 *   SW (NB, KB): one fp32 scale per `block` x `block` block of W;
 *   KB = ceil(K/block), NB = ceil(N/block); a partial last block keeps its
 *   own scale.  Everything is formed in fp64 (FP8 and fp32 values are exact
 *   there); each block's P_b is summed in ascending k, multiplied by the
 *   product of its two scales, and the blocks are added in ascending b.
 *   R and the final binary16 rounding are those of oracle_gemm_f16_rows.
 * ====================================================================== */

/* OCP FP8 E4M3 (the "fn" variant: finite, no infinities) -> binary64,
 * exact.  1 sign bit, 4 exponent bits (bias 7), 3 fraction bits; exponent
 * field 0 holds zero and the subnormals m * 2^-9; exponent field 15 with
 * fraction 7 (0x7F, 0xFF) is NaN; the largest finite magnitude is 448. */
double oracle_e4m3_to_f64(uint8_t x)
{
    const int sign = (x >> 7) & 1;
    const int e = (x >> 3) & 0xf;
    const int m = x & 0x7;
    double v;
    if (e == 15 && m == 7) {
        v = NAN;
    } else if (e == 0) {
        v = ldexp((double)m, -9);               /* m/8 * 2^(1-7) */
    } else {
        v = ldexp((double)(m + 8), e - 10);     /* (1 + m/8) * 2^(e-7) */
    }
    return sign ? -v : v;
}

int oracle_gemm_fp8_block_scaled_rows(const uint8_t *A, const float *SA, const uint8_t *W, const float *SW,
                                      uint16_t *C_out, int64_t M, int64_t N, int64_t K, int64_t block, int relu,
                                      const int64_t *rows, int64_t n_rows)
{
    if (M < 0 || N < 0 || K < 0 || n_rows < 0 || block <= 0) return -1;
    if (rows == NULL && n_rows != M) return -1;
    for (int64_t r = 0; rows != NULL && r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= M) return -1;
    if (n_rows == 0 || N == 0) return 0;
    const int64_t KB = (K + block - 1) / block;

    double e4m3[256];
    for (int v = 0; v < 256; ++v) e4m3[v] = oracle_e4m3_to_f64((uint8_t)v);

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
        const int64_t i = rows ? rows[r] : r;
        const uint8_t *a_row = A + i * K;
        uint16_t *c_row = C_out + r * N;
        for (int64_t j = 0; j < N; ++j) {
            const uint8_t *w_row = W + j * K;
            double acc = 0.0;
            for (int64_t b = 0; b < KB; ++b) {
                const int64_t k_end = (b + 1) * block < K ? (b + 1) * block : K;
                double p = 0.0;
                for (int64_t k = b * block; k < k_end; ++k) p += e4m3[a_row[k]] * e4m3[w_row[k]];
                const double s = (double)SA[i * KB + b] * (double)SW[(j / block) * KB + b];
                acc += s * p;
            }
            if (relu) acc = (acc > 0.0) ? acc : 0.0;
            c_row[j] = oracle_f64_to_f16(acc);
        }
    }
    return 0;
}

/* ======================================================================
 * Attention forward (TEST INFRASTRUCTURE ONLY, like everything above).
 *
 * The TileLang-MUSA lesson (7yue.com, section 5, "FlashAttention skeleton")
 * and "Writing High-Performance Kernels in TileLang, from GEMM to MLA"
 * (section "A real one: MLA decode", the FlashAttention loop) describe the
 * FlashAttention forward: Q, K, V, O of shape (batch, heads, seq, dim) in
 * float16; per query row the scores against every key, a softmax over them
 * (computed blockwise with a running max and sum), and the probability-
 * weighted sum of the value rows.  The blockwise online form is an
 * implementation of the plain definition, which this function writes out:
 *
 *   s_j   = sm_scale * sum_d Q[b,h,i,d] * K[b,h,j,d]     for keys j allowed
 *   O[b,h,i,d] = f16_rne( sum_j exp(s_j - max_j s_j) * V[b,h,j,d]
 *                          / sum_j exp(s_j - max_j s_j) )
 *
 * Keys allowed: all j < seq; with `causal`, only j <= i.  The skeletons do
 * not show the softmax temperature; sm_scale is a parameter (callers pass
 * 1/sqrt(dim), the usual choice).  Everything is fp64 (fp16 inputs are exact
 * there, exp from libm); the only rounding that matters is the final cast.
 * ====================================================================== */

int oracle_attention_fwd_rows(const uint16_t *Q, const uint16_t *K, const uint16_t *V, uint16_t *O_out,
                              int64_t batch, int64_t heads, int64_t seq, int64_t dim, double sm_scale, int causal,
                              const int64_t *rows, int64_t n_rows)
{
    if (batch < 0 || heads < 0 || seq < 0 || dim < 0 || n_rows < 0) return -1;
    const int64_t total = batch * heads * seq;
    if (rows == NULL && n_rows != total) return -1;
    for (int64_t r = 0; rows != NULL && r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= total) return -1;
    if (n_rows == 0 || dim == 0) return 0;
    fill_f16_values();

    int failed = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc((size_t)(seq > 0 ? seq : 1) * sizeof(double));
        double *o = (double *)malloc((size_t)dim * sizeof(double));
        if (s == NULL || o == NULL) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n_rows; ++r) {
            if (s == NULL || o == NULL) continue;
            const int64_t flat = rows ? rows[r] : r;     /* (b*heads + h)*seq + i */
            const int64_t bh = flat / seq, i = flat % seq;
            const uint16_t *q = Q + flat * dim;
            const uint16_t *kbase = K + bh * seq * dim;
            const uint16_t *vbase = V + bh * seq * dim;
            const int64_t n_keys = causal ? i + 1 : seq;
            double m = -INFINITY;
            for (int64_t j = 0; j < n_keys; ++j) {
                double dot = 0.0;
                for (int64_t d = 0; d < dim; ++d) dot += g_f16_value[q[d]] * g_f16_value[kbase[j * dim + d]];
                s[j] = sm_scale * dot;
                if (s[j] > m) m = s[j];
            }
            double l = 0.0;
            for (int64_t d = 0; d < dim; ++d) o[d] = 0.0;
            for (int64_t j = 0; j < n_keys; ++j) {
                const double p = exp(s[j] - m);
                l += p;
                for (int64_t d = 0; d < dim; ++d) o[d] += p * g_f16_value[vbase[j * dim + d]];
            }
            uint16_t *out = O_out + r * dim;
            for (int64_t d = 0; d < dim; ++d) out[d] = oracle_f64_to_f16(o[d] / l);
        }
        free(s);
        free(o);
    }
    return failed ? -1 : 0;
}
