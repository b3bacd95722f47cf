/*
 * Plain CPU oracle for the fp16 TN GEMM  D = A * B^T.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the bench's CPU
 * baseline leg use it.  It shares no code, header or table with the CUDA
 * library; both sides only receive the same seeded fp16 bit patterns.
 *
 * What it computes (the plain definition, written out):
 *
 *   D[i][j] = fp16_rne( sum_{k<K} double(A[i][k]) * double(B[j][k]) )
 *
 * with A M x K row-major (leading dimension K), B N x K row-major
 * (leading dimension K) and D M x N row-major (leading dimension N).  This is
 * the operation of "cute(9) multistage_gemm" (kernel signature and the
 * global-tensor definitions in its code listing, section 11 "性能测试": A(M,K),
 * B(N,K), D(M,N), all row-major, D = A @ B^T).  The page accumulates in fp16;
 * this oracle accumulates in double and rounds once at the end, so it is the
 * exact product rounded to fp16 (every fp16 x fp16 product is exact in
 * double; only the K-1 additions round, at 2^-53 relative).
 *
 * The stage-count helper follows "第 6 课：Shared Memory 布局与异步流水",
 * section 4 (性能与工程取舍), S_min = ceil(T_copy / T_compute) + 1, for
 * positive integer arguments as the lesson's exercise states.
 *
 * Converters are written from the IEEE 754 binary16 definition (1 sign bit,
 * 5 exponent bits with bias 15, 10 fraction bits; exponent 0 = subnormal,
 * exponent 31 = inf/NaN), not from any library routine.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>

/* ---- binary16 -> double (exact) ---------------------------------------- */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);              /* subnormal or zero */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + frac), expo - 25); /* 1.frac * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* ---- double -> binary16, round to nearest, ties to even ----------------- */
static uint16_t encode_exact_half(double v, uint16_t sign)
{
    /* v >= 0 is exactly representable as a binary16 value here. */
    if (v == 0.0) return sign;
    if (v < ldexp(1.0, -14)) {                     /* subnormal: v = m * 2^-24 */
        return (uint16_t)(sign | (uint16_t)ldexp(v, 24));
    }
    int e2;
    frexp(v, &e2);                                 /* v = f * 2^e2, f in [0.5,1) */
    int e_unb = e2 - 1;                            /* v = (2f) * 2^e_unb */
    if (e_unb > 15) return (uint16_t)(sign | 0x7c00);
    int mant = (int)ldexp(v, 10 - e_unb) - 1024;   /* 10 fraction bits */
    return (uint16_t)(sign | ((e_unb + 15) << 10) | mant);
}

uint16_t oracle_double_to_half(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return (uint16_t)(sign | 0x7e00);
    double a = fabs(x);
    /* 65504 is the largest finite value; halfway to the next binade step
     * (65536) is 65520, and the tie goes to the even neighbour 65536 = inf. */
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00);
    if (a == 0.0) return sign;
    int e2;
    frexp(a, &e2);
    int e_unb = e2 - 1;
    /* spacing of binary16 values near a: 2^(max(e,-14) - 10) */
    int q_exp = (e_unb < -14 ? -14 : e_unb) - 10;
    double n = ldexp(a, -q_exp);                   /* a in units of the spacing */
    double r = floor(n);
    double rem = n - r;                            /* exact: n < 2^11 */
    if (rem > 0.5 || (rem == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
    return encode_exact_half(ldexp(r, q_exp), sign);
}

/* ---- the GEMM itself ---------------------------------------------------- */
static double dot_row_row(const uint16_t* a_row, const uint16_t* b_row, int64_t K)
{
    double s = 0.0;
    for (int64_t k = 0; k < K; ++k)
        s += oracle_half_to_double(a_row[k]) * oracle_half_to_double(b_row[k]);
    return s;
}

typedef struct {
    const uint16_t* A; const uint16_t* B; uint16_t* D;
    int64_t M, N, K, row_begin, row_end;
} rows_job;

static void* run_rows(void* p)
{
    rows_job* j = (rows_job*)p;
    for (int64_t i = j->row_begin; i < j->row_end; ++i)
        for (int64_t n = 0; n < j->N; ++n)
            j->D[i * j->N + n] = oracle_double_to_half(
                dot_row_row(j->A + i * j->K, j->B + n * j->K, j->K));
    return NULL;
}

/* Full D (M x N).  Rows are split over `threads` POSIX threads; each output
 * element is still one sequential k-loop, so the result does not depend on
 * the thread count.  Returns 0, or -1 on bad arguments. */
int oracle_gemm_tn(const uint16_t* A, const uint16_t* B, uint16_t* D,
                   int64_t M, int64_t N, int64_t K, int threads)
{
    enum { MAX_THREADS = 256 };
    if (M < 0 || N < 0 || K < 0 || (M * N > 0 && (!A || !B || !D))) return -1;
    if (M == 0 || N == 0) return 0;
    if (threads < 1) threads = 1;
    if (threads > MAX_THREADS) threads = MAX_THREADS;
    if (threads > M) threads = (int)M;
    pthread_t tid[MAX_THREADS];
    int joined[MAX_THREADS];
    rows_job job[MAX_THREADS];
    int64_t per = (M + threads - 1) / threads;
    for (int t = 0; t < threads; ++t) {
        int64_t b = t * per, e = (t + 1) * per;
        if (b > M) b = M;
        if (e > M) e = M;
        job[t] = (rows_job){A, B, D, M, N, K, b, e};
        joined[t] = 0;
    }
    /* thread 0's rows run on the calling thread; a failed create falls back
     * to running that chunk inline as well */
    for (int t = 1; t < threads; ++t) {
        if (job[t].row_begin >= job[t].row_end) continue;
        if (pthread_create(&tid[t], NULL, run_rows, &job[t]) == 0) joined[t] = 1;
        else run_rows(&job[t]);
    }
    run_rows(&job[0]);
    for (int t = 1; t < threads; ++t)
        if (joined[t]) pthread_join(tid[t], NULL);
    return 0;
}

/* ---- the scaled form: D = alpha * A op(B) + beta * C ---------------------
 *
 * "CUDA 算子笔记 2", section "General Matrix Multiplication（GEMM）", states the
 * problem as C = alpha * A * B + beta * C with A M x K and B K x N row-major
 * (the NN layout), fp16 matrices and fp32 alpha, beta (its "C is M x K" is a
 * slip: C has the product's shape, M x N).  Written out:
 *
 *   D[i][j] = fp16_rne( alpha * sum_k A[i][k] * B(k, j) + beta * C[i][j] )
 *
 * with B(k, j) = B[k*N + j] when b_kn != 0 (B is K x N) and B[j*K + k] when
 * b_kn == 0 (B is N x K, the TN case above).  alpha and beta are fp32 values,
 * exact in double; the sum is the same double sum as oracle_gemm_tn; the
 * combination alpha*s + beta*c is formed in double and rounded once to fp16.
 * When beta == 0, C is not read (it may be NULL), as in BLAS.  D may be C. */
typedef struct {
    const uint16_t* A; const uint16_t* B; const uint16_t* C; uint16_t* D;
    int64_t M, N, K, row_begin, row_end;
    double alpha, beta;
    int b_kn;
} scaled_job;

static void* run_scaled_rows(void* p)
{
    scaled_job* j = (scaled_job*)p;
    for (int64_t i = j->row_begin; i < j->row_end; ++i) {
        for (int64_t n = 0; n < j->N; ++n) {
            double s = 0.0;
            for (int64_t k = 0; k < j->K; ++k) {
                const uint16_t b = j->b_kn ? j->B[k * j->N + n] : j->B[n * j->K + k];
                s += oracle_half_to_double(j->A[i * j->K + k]) * oracle_half_to_double(b);
            }
            double v = j->alpha * s;
            if (j->beta != 0.0) v += j->beta * oracle_half_to_double(j->C[i * j->N + n]);
            j->D[i * j->N + n] = oracle_double_to_half(v);
        }
    }
    return NULL;
}

int oracle_gemm_scaled(const uint16_t* A, const uint16_t* B, const uint16_t* C, uint16_t* D,
                       int64_t M, int64_t N, int64_t K, float alpha, float beta, int b_kn,
                       int threads)
{
    enum { MAX_THREADS = 256 };
    if (M < 0 || N < 0 || K < 0) return -1;
    if (M == 0 || N == 0) return 0;
    if (!D || (K > 0 && (!A || !B)) || (beta != 0.0f && !C)) return -1;
    if (threads < 1) threads = 1;
    if (threads > MAX_THREADS) threads = MAX_THREADS;
    if (threads > M) threads = (int)M;
    /* D may be C: each element of C is read once, by the thread that then
     * writes that element, before it writes it. */
    pthread_t tid[MAX_THREADS];
    int joined[MAX_THREADS];
    scaled_job job[MAX_THREADS];
    int64_t per = (M + threads - 1) / threads;
    for (int t = 0; t < threads; ++t) {
        int64_t b = t * per, e = (t + 1) * per;
        if (b > M) b = M;
        if (e > M) e = M;
        job[t] = (scaled_job){A, B, C, D, M, N, K, b, e, (double)alpha, (double)beta, b_kn};
        joined[t] = 0;
    }
    for (int t = 1; t < threads; ++t) {
        if (job[t].row_begin >= job[t].row_end) continue;
        if (pthread_create(&tid[t], NULL, run_scaled_rows, &job[t]) == 0) joined[t] = 1;
        else run_scaled_rows(&job[t]);
    }
    run_scaled_rows(&job[0]);
    for (int t = 1; t < threads; ++t)
        if (joined[t]) pthread_join(tid[t], NULL);
    return 0;
}

/* ---- fp16 accumulation ---------------------------------------------------
 *
 * "cute(9) multistage_gemm" builds its kernel on an MMA atom whose
 * accumulator is fp16 (SM80_16x8x16_F16F16F16F16_TN in its config listing):
 * every instruction adds a 16-deep slice of the K sum to an fp16
 * accumulator and rounds the result to fp16.  Written out with the slice's
 * products summed exactly:
 *
 *   acc = 0;  for each slice c of 16 consecutive k:
 *       acc = fp16_rne( acc + sum_{k in c} double(A[i][k]) * double(B[j][k]) )
 *   D[i][j] = acc
 *
 * (TN layout as oracle_gemm_tn; a last slice shorter than 16 when K is not
 * a multiple of 16.) */
static void* run_f16acc_rows(void* p)
{
    rows_job* j = (rows_job*)p;
    for (int64_t i = j->row_begin; i < j->row_end; ++i) {
        for (int64_t n = 0; n < j->N; ++n) {
            const uint16_t* a_row = j->A + i * j->K;
            const uint16_t* b_row = j->B + n * j->K;
            double acc = 0.0;
            for (int64_t k0 = 0; k0 < j->K; k0 += 16) {
                double s = acc;
                for (int64_t k = k0; k < k0 + 16 && k < j->K; ++k)
                    s += oracle_half_to_double(a_row[k]) * oracle_half_to_double(b_row[k]);
                acc = oracle_half_to_double(oracle_double_to_half(s));
            }
            j->D[i * j->N + n] = oracle_double_to_half(acc);
        }
    }
    return NULL;
}

int oracle_gemm_tn_f16acc(const uint16_t* A, const uint16_t* B, uint16_t* D,
                          int64_t M, int64_t N, int64_t K, int threads)
{
    enum { MAX_THREADS = 256 };
    if (M < 0 || N < 0 || K < 0 || (M * N > 0 && (!A || !B || !D))) return -1;
    if (M == 0 || N == 0) return 0;
    if (threads < 1) threads = 1;
    if (threads > MAX_THREADS) threads = MAX_THREADS;
    if (threads > M) threads = (int)M;
    pthread_t tid[MAX_THREADS];
    int joined[MAX_THREADS];
    rows_job job[MAX_THREADS];
    int64_t per = (M + threads - 1) / threads;
    for (int t = 0; t < threads; ++t) {
        int64_t b = t * per, e = (t + 1) * per;
        if (b > M) b = M;
        if (e > M) e = M;
        job[t] = (rows_job){A, B, D, M, N, K, b, e};
        joined[t] = 0;
    }
    for (int t = 1; t < threads; ++t) {
        if (job[t].row_begin >= job[t].row_end) continue;
        if (pthread_create(&tid[t], NULL, run_f16acc_rows, &job[t]) == 0) joined[t] = 1;
        else run_f16acc_rows(&job[t]);
    }
    run_f16acc_rows(&job[0]);
    for (int t = 1; t < threads; ++t)
        if (joined[t]) pthread_join(tid[t], NULL);
    return 0;
}

/* Selected elements only: out[s] = D[rows[s]][cols[s]].  Used where the full
 * product is too large for the CPU (the 8192^3 case). */
int oracle_gemm_tn_sampled(const uint16_t* A, const uint16_t* B,
                           int64_t M, int64_t N, int64_t K,
                           const int64_t* rows, const int64_t* cols,
                           int64_t count, uint16_t* out)
{
    if (M < 0 || N < 0 || K < 0 || count < 0) return -1;
    for (int64_t s = 0; s < count; ++s) {
        if (rows[s] < 0 || rows[s] >= M || cols[s] < 0 || cols[s] >= N) return -1;
        out[s] = oracle_double_to_half(dot_row_row(A + rows[s] * K, B + cols[s] * K, K));
    }
    return 0;
}

/* S_min = ceil(copy / compute) + 1 for positive integers; -1 otherwise. */
int64_t oracle_minimum_stages(int64_t copy_cycles, int64_t compute_cycles)
{
    if (copy_cycles <= 0 || compute_cycles <= 0) return -1;
    int64_t in_flight = copy_cycles / compute_cycles
                      + (copy_cycles % compute_cycles != 0);
    return in_flight + 1;
}
