/*
 * conv3d_fp8_oracle.c -- plain CPU oracle for the FP8 (e4m3) 3D convolution with a BF16 output.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check of the package entry file and the
 * CPU-baseline leg of the benchmark may load this code. The product path never calls it, and it
 * shares no code, header, table or constant with the CUDA library.
 *
 * What it computes (the plain definition, no blocking or fusion):
 *
 *   S[n,k,do,ho,wo] = sum_{c<C} sum_{t<T} sum_{r<R} sum_{s<S}
 *                       X[n, c, do*sd + t - pd, ho*sh + r - ph, wo*sw + s - pw] * Wt[k, c, t, r, s]
 *   y64  = (double)sx * (double)sw * S
 *   ybf16 = round-to-nearest-even of y64 to bfloat16
 *
 * with X and Wt the exactly decoded e4m3 bytes, and X = 0 outside [0,D) x [0,H) x [0,W).
 *
 * Passages followed ("[Fix] conv3d fp8: guard padded M rows in the epilogue store", ROCm/FlyDSL
 * pull request 969):
 *   - "Problem": the kernel is checked against an fp8-cast reference for the case
 *     [N-C-D-H-W-K-stride-pad] = [1-96-4-8-9-96-1-1]; inputs are e4m3 bytes and the output is BF16.
 *   - "Root cause": the output is NCDHW (the store offset is off_ncdhw, col*dhw + row for n == 1),
 *     and filter taps that fall outside the input are zero (the im2col mask zeroes A).
 * The GEMM view (M = N*Do*Ho*Wo rows, N_gemm = K, K_gemm = C*T*R*S) does not change the sum; the
 * oracle evaluates the sum directly. Zero padding, dilation 1 and one group are the plain
 * convolution reading where the page is silent.
 *
 * Exactness. Every e4m3 value is an integer multiple of 2^-9 with magnitude <= 448, so every
 * product is an integer multiple of 2^-18 below 2^18 in magnitude. A sum of fewer than 2^35 such
 * terms is an integer multiple of 2^-18 below 2^53 * 2^-18, which fp64 holds exactly in any order.
 * The only rounding before the final BF16 rounding is the one fp64 multiply by sx*sw (the fp32 x
 * fp32 product itself is exact in fp64).
 *
 * The BF16-input twin (the same page, "Notes": the BF16 implicit-GEMM conv3d kernel that
 * already guards its padded rows) computes the same sum with X and Wt bfloat16 values and no
 * scales: y64 = S, ybf16 = round-to-nearest-even of S. Its products are exact in fp64 (two 8-bit
 * significands); the fp64 sum in the loop order below differs from the exact sum by at most
 * (n - 1) * 2^-53 * sum|terms| (recursive summation, n terms), far below one BF16 ulp for the
 * workloads here.
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC (OpenMP optional; without it the loops run serially).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------------------------------------
 * e4m3 ("float8_e4m3fn", OCP FP8 E4M3): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
 * bits, no infinities, S.1111.111 is NaN. Exponent field 0 is subnormal: m/8 * 2^-6.
 * Normal: (1 + m/8) * 2^(e-7) = (8 + m) * 2^(e-10). Subnormal: m * 2^-9.
 * ------------------------------------------------------------------------------------------- */
double o_e4m3_decode(unsigned char b)
{
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xF;
    int m = b & 0x7;
    double mag;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);
    else
        mag = ldexp((double)(8 + m), e - 10);
    return sign ? -mag : mag;
}

/* ---------------------------------------------------------------------------------------------
 * bfloat16: 1 sign bit, 8 exponent bits with bias 127, 7 mantissa bits. Exponent field 0 is
 * subnormal: m * 2^-133; field 255 is infinity (m == 0) or NaN. Normal: (128 + m) * 2^(e-134).
 * ------------------------------------------------------------------------------------------- */
double o_bf16_decode(unsigned short b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xFF;
    int m = b & 0x7F;
    double mag;
    if (e == 0xFF)
        return m ? NAN : (sign ? -INFINITY : INFINITY);
    if (e == 0)
        mag = ldexp((double)m, -133);
    else
        mag = ldexp((double)(128 + m), e - 134);
    return sign ? -mag : mag;
}

/* ---------------------------------------------------------------------------------------------
 * Round a double to bfloat16 (1 sign, 8 exponent bits with bias 127, 7 mantissa bits) with
 * round-to-nearest, ties to even, in ONE step from the double (no intermediate fp32 rounding).
 * Returns the 16-bit pattern.
 * ------------------------------------------------------------------------------------------- */
unsigned short o_bf16_rne(double v)
{
    unsigned short sign;
    double a, scaled, fl, fr, r;
    int e, q;
    float f;
    uint32_t bits;

    if (v != v)
        return 0x7FC0;
    sign = signbit(v) ? 0x8000 : 0;
    a = fabs(v);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (unsigned short)(sign | 0x7F80);
    (void)frexp(a, &e);  /* a in [2^(e-1), 2^e) */
    q = e - 8;           /* spacing of bf16 values in that binade: 2^(e-1-7) */
    if (q < -133)
        q = -133;        /* bf16 subnormal spacing */
    scaled = ldexp(a, -q); /* exact: a power-of-two rescale */
    fl = floor(scaled);
    fr = scaled - fl;
    if (fr > 0.5 || (fr == 0.5 && fmod(fl, 2.0) == 1.0))
        fl += 1.0;
    r = ldexp(fl, q);
    if (r > 0x1.fep127) /* largest finite bf16 is (2 - 2^-7) * 2^127 */
        return (unsigned short)(sign | 0x7F80);
    f = (float)r;        /* exact: r has at most 8 significant bits */
    memcpy(&bits, &f, sizeof bits);
    return (unsigned short)(sign | (bits >> 16));
}

/* Output extent of a zero-padded, undilated convolution: floor((in + 2*pad - k) / stride) + 1. */
int o_out_dim(int in, int k, int stride, int pad)
{
    int span = in + 2 * pad - k;
    if (stride <= 0 || span < 0)
        return 0;
    return span / stride + 1;
}

int o_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

typedef struct {
    int N, C, D, H, W, K, T, R, S;
    int sd, sh, sw, pd, ph, pw;
    int Do, Ho, Wo;
} o_shape;

static int o_make_shape(o_shape *sh, int N, int C, int D, int H, int W, int K, int T, int R, int S,
                        int sd, int shh, int sww, int pd, int ph, int pw)
{
    sh->N = N; sh->C = C; sh->D = D; sh->H = H; sh->W = W; sh->K = K;
    sh->T = T; sh->R = R; sh->S = S;
    sh->sd = sd; sh->sh = shh; sh->sw = sww; sh->pd = pd; sh->ph = ph; sh->pw = pw;
    if (N <= 0 || C <= 0 || D <= 0 || H <= 0 || W <= 0 || K <= 0 || T <= 0 || R <= 0 || S <= 0)
        return -1;
    if (sd <= 0 || shh <= 0 || sww <= 0 || pd < 0 || ph < 0 || pw < 0)
        return -1;
    sh->Do = o_out_dim(D, T, sd, pd);
    sh->Ho = o_out_dim(H, R, shh, ph);
    sh->Wo = o_out_dim(W, S, sww, pw);
    if (sh->Do <= 0 || sh->Ho <= 0 || sh->Wo <= 0)
        return -1;
    return 0;
}

/* The unscaled sum S for one output element, straight from the definition. */
static double o_point_sum(const o_shape *p, const unsigned char *x, const unsigned char *w,
                          const double *tab, int n, int k, int od, int oh, int ow)
{
    double acc = 0.0;
    int c, t, r, s;
    for (c = 0; c < p->C; ++c) {
        for (t = 0; t < p->T; ++t) {
            int id = od * p->sd + t - p->pd;
            if (id < 0 || id >= p->D)
                continue; /* zero padding: the tap contributes 0 */
            for (r = 0; r < p->R; ++r) {
                int ih = oh * p->sh + r - p->ph;
                if (ih < 0 || ih >= p->H)
                    continue;
                for (s = 0; s < p->S; ++s) {
                    int iw = ow * p->sw + s - p->pw;
                    size_t xi, wi;
                    if (iw < 0 || iw >= p->W)
                        continue;
                    xi = ((((size_t)n * p->C + c) * p->D + id) * p->H + ih) * p->W + iw;
                    wi = ((((size_t)k * p->C + c) * p->T + t) * p->R + r) * p->S + s;
                    acc += tab[x[xi]] * tab[w[wi]];
                }
            }
        }
    }
    return acc;
}

static int o_check_bytes(const unsigned char *b, size_t n)
{
    size_t i;
    for (i = 0; i < n; ++i)
        if ((b[i] & 0x7F) == 0x7F)
            return -2; /* NaN byte: not a valid input for the oracle */
    return 0;
}

/*
 * Full output. x: N*C*D*H*W e4m3 bytes (NCDHW), w: K*C*T*R*S e4m3 bytes (KCTRS).
 * Outputs (each may be NULL): ysum = unscaled exact sums, y64 = scaled fp64, ybf16 = BF16 bits,
 * all N*K*Do*Ho*Wo in NCDHW order. Returns 0, -1 on a bad shape, -2 on a NaN input byte.
 */
int o_conv3d_fp8(const unsigned char *x, const unsigned char *w, float sx, float sw,
                 int N, int C, int D, int H, int W, int K, int T, int R, int S,
                 int sd, int sh, int sww, int pd, int ph, int pw,
                 double *ysum, double *y64, unsigned short *ybf16)
{
    o_shape p;
    double tab[256];
    double scale = (double)sx * (double)sw;
    long long nk;
    int i;

    if (o_make_shape(&p, N, C, D, H, W, K, T, R, S, sd, sh, sww, pd, ph, pw) != 0)
        return -1;
    if (o_check_bytes(x, (size_t)N * C * D * H * W) != 0 ||
        o_check_bytes(w, (size_t)K * C * T * R * S) != 0)
        return -2;
    for (i = 0; i < 256; ++i)
        tab[i] = o_e4m3_decode((unsigned char)i);

    nk = (long long)N * K;
#pragma omp parallel for schedule(dynamic, 1)
    for (long long job = 0; job < nk; ++job) {
        int n = (int)(job / K), k = (int)(job % K);
        int od, oh, ow;
        for (od = 0; od < p.Do; ++od)
            for (oh = 0; oh < p.Ho; ++oh)
                for (ow = 0; ow < p.Wo; ++ow) {
                    size_t yi = ((((size_t)n * K + k) * p.Do + od) * p.Ho + oh) * p.Wo + ow;
                    double sum = o_point_sum(&p, x, w, tab, n, k, od, oh, ow);
                    double v = scale * sum;
                    if (ysum)
                        ysum[yi] = sum;
                    if (y64)
                        y64[yi] = v;
                    if (ybf16)
                        ybf16[yi] = o_bf16_rne(v);
                }
    }
    return 0;
}

/*
 * Selected outputs only. idx[i] is a flat NCDHW index into the N*K*Do*Ho*Wo output.
 * Same outputs and return codes as o_conv3d_fp8, one entry per index; -3 on an index out of range.
 */
int o_conv3d_fp8_points(const unsigned char *x, const unsigned char *w, float sx, float sw,
                        int N, int C, int D, int H, int W, int K, int T, int R, int S,
                        int sd, int sh, int sww, int pd, int ph, int pw,
                        const long long *idx, long long npts,
                        double *ysum, double *y64, unsigned short *ybf16)
{
    o_shape p;
    double tab[256];
    double scale = (double)sx * (double)sw;
    long long total;
    int i, bad = 0;

    if (o_make_shape(&p, N, C, D, H, W, K, T, R, S, sd, sh, sww, pd, ph, pw) != 0)
        return -1;
    if (o_check_bytes(x, (size_t)N * C * D * H * W) != 0 ||
        o_check_bytes(w, (size_t)K * C * T * R * S) != 0)
        return -2;
    total = (long long)N * K * p.Do * p.Ho * p.Wo;
    for (long long j = 0; j < npts; ++j)
        if (idx[j] < 0 || idx[j] >= total)
            bad = 1;
    if (bad)
        return -3;
    for (i = 0; i < 256; ++i)
        tab[i] = o_e4m3_decode((unsigned char)i);

#pragma omp parallel for schedule(dynamic, 64)
    for (long long j = 0; j < npts; ++j) {
        long long f = idx[j];
        int ow = (int)(f % p.Wo);
        int oh = (int)((f / p.Wo) % p.Ho);
        int od = (int)((f / ((long long)p.Wo * p.Ho)) % p.Do);
        int k = (int)((f / ((long long)p.Wo * p.Ho * p.Do)) % K);
        int n = (int)(f / ((long long)p.Wo * p.Ho * p.Do * K));
        double sum = o_point_sum(&p, x, w, tab, n, k, od, oh, ow);
        double v = scale * sum;
        if (ysum)
            ysum[j] = sum;
        if (y64)
            y64[j] = v;
        if (ybf16)
            ybf16[j] = o_bf16_rne(v);
    }
    return 0;
}

/* ============================================================================================
 * BF16-input twin: x and w are bfloat16 bit patterns, no scales.
 * ========================================================================================== */

/* The sum S for one output element, straight from the definition (bfloat16 inputs). */
static double o_point_sum_bf16(const o_shape *p, const unsigned short *x, const unsigned short *w,
                               int n, int k, int od, int oh, int ow)
{
    double acc = 0.0;
    int c, t, r, s;
    for (c = 0; c < p->C; ++c) {
        for (t = 0; t < p->T; ++t) {
            int id = od * p->sd + t - p->pd;
            if (id < 0 || id >= p->D)
                continue;
            for (r = 0; r < p->R; ++r) {
                int ih = oh * p->sh + r - p->ph;
                if (ih < 0 || ih >= p->H)
                    continue;
                for (s = 0; s < p->S; ++s) {
                    int iw = ow * p->sw + s - p->pw;
                    size_t xi, wi;
                    if (iw < 0 || iw >= p->W)
                        continue;
                    xi = ((((size_t)n * p->C + c) * p->D + id) * p->H + ih) * p->W + iw;
                    wi = ((((size_t)k * p->C + c) * p->T + t) * p->R + r) * p->S + s;
                    acc += o_bf16_decode(x[xi]) * o_bf16_decode(w[wi]);
                }
            }
        }
    }
    return acc;
}

static int o_check_bf16(const unsigned short *b, size_t n)
{
    size_t i;
    for (i = 0; i < n; ++i)
        if ((b[i] & 0x7F80) == 0x7F80)
            return -2; /* infinity or NaN: not a valid input for the oracle */
    return 0;
}

/*
 * Full output of the BF16 twin. x: N*C*D*H*W bfloat16 (NCDHW), w: K*C*T*R*S bfloat16 (KCTRS).
 * Outputs (each may be NULL): y64 = fp64 sums, ybf16 = their BF16 rounding, N*K*Do*Ho*Wo NCDHW.
 * Returns 0, -1 on a bad shape, -2 on an infinite or NaN input.
 */
int o_conv3d_bf16(const unsigned short *x, const unsigned short *w,
                  int N, int C, int D, int H, int W, int K, int T, int R, int S,
                  int sd, int sh, int sww, int pd, int ph, int pw,
                  double *y64, unsigned short *ybf16)
{
    o_shape p;
    long long nk;

    if (o_make_shape(&p, N, C, D, H, W, K, T, R, S, sd, sh, sww, pd, ph, pw) != 0)
        return -1;
    if (o_check_bf16(x, (size_t)N * C * D * H * W) != 0 ||
        o_check_bf16(w, (size_t)K * C * T * R * S) != 0)
        return -2;
    nk = (long long)N * K;
#pragma omp parallel for schedule(dynamic, 1)
    for (long long job = 0; job < nk; ++job) {
        int n = (int)(job / K), k = (int)(job % K);
        int od, oh, ow;
        for (od = 0; od < p.Do; ++od)
            for (oh = 0; oh < p.Ho; ++oh)
                for (ow = 0; ow < p.Wo; ++ow) {
                    size_t yi = ((((size_t)n * K + k) * p.Do + od) * p.Ho + oh) * p.Wo + ow;
                    double v = o_point_sum_bf16(&p, x, w, n, k, od, oh, ow);
                    if (y64)
                        y64[yi] = v;
                    if (ybf16)
                        ybf16[yi] = o_bf16_rne(v);
                }
    }
    return 0;
}

/* Selected outputs of the BF16 twin; idx[i] is a flat NCDHW output index. -3: index out of range. */
int o_conv3d_bf16_points(const unsigned short *x, const unsigned short *w,
                         int N, int C, int D, int H, int W, int K, int T, int R, int S,
                         int sd, int sh, int sww, int pd, int ph, int pw,
                         const long long *idx, long long npts,
                         double *y64, unsigned short *ybf16)
{
    o_shape p;
    long long total;
    int bad = 0;

    if (o_make_shape(&p, N, C, D, H, W, K, T, R, S, sd, sh, sww, pd, ph, pw) != 0)
        return -1;
    if (o_check_bf16(x, (size_t)N * C * D * H * W) != 0 ||
        o_check_bf16(w, (size_t)K * C * T * R * S) != 0)
        return -2;
    total = (long long)N * K * p.Do * p.Ho * p.Wo;
    for (long long j = 0; j < npts; ++j)
        if (idx[j] < 0 || idx[j] >= total)
            bad = 1;
    if (bad)
        return -3;
#pragma omp parallel for schedule(dynamic, 64)
    for (long long j = 0; j < npts; ++j) {
        long long f = idx[j];
        int ow = (int)(f % p.Wo);
        int oh = (int)((f / p.Wo) % p.Ho);
        int od = (int)((f / ((long long)p.Wo * p.Ho)) % p.Do);
        int k = (int)((f / ((long long)p.Wo * p.Ho * p.Do)) % K);
        int n = (int)(f / ((long long)p.Wo * p.Ho * p.Do * K));
        double v = o_point_sum_bf16(&p, x, w, n, k, od, oh, ow);
        if (y64)
            y64[j] = v;
        if (ybf16)
            ybf16[j] = o_bf16_rne(v);
    }
    return 0;
}
