/*
 * Plain CPU oracle for the ZeRO-DP partitioned mixed-precision AdamW step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  It shares no code,
 * header, table or constant generator with the CUDA path of the package.
 *
 * Every routine here is a literal loop over elements, written so that a reader
 * can check it against the definition by eye.  There is no blocking, fusion or
 * reordering of arithmetic beyond what the definition states.  OpenMP only
 * splits independent elements (or independent fixed chunks) across threads;
 * it never changes an element's order of operations.
 *
 * Build flags (see oracle/build.py): -O2 -ffp-contract=off -fno-fast-math,
 * so every float operation below is one IEEE-754 binary32 operation rounded
 * to nearest even, and no multiply-add is ever fused.
 *
 * Formats: 16-bit values travel as uint16_t bit patterns; fmt 0 = bfloat16,
 * fmt 1 = IEEE binary16 ("fp16").
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* 16-bit decode, exact (every 16-bit value is representable in binary32).    */
/* ------------------------------------------------------------------------ */

/* bfloat16 is the upper half of a binary32 bit pattern. */
static float orc_bf16_to_f32(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static float orc_f16_to_f32(uint16_t h) {
    uint32_t sign = (uint32_t)(h >> 15) & 1u;
    uint32_t e = (uint32_t)(h >> 10) & 0x1Fu;
    uint32_t f = (uint32_t)h & 0x3FFu;
    float mag;
    if (e == 0u) {
        mag = ldexpf((float)f, -24);             /* subnormal: f * 2^-24 */
    } else if (e == 31u) {
        mag = (f != 0u) ? NAN : INFINITY;
    } else {
        mag = ldexpf((float)(f + 1024u), (int)e - 25); /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -mag : mag;
}

static float orc_decode(uint16_t h, int32_t fmt) {
    return fmt == 0 ? orc_bf16_to_f32(h) : orc_f16_to_f32(h);
}

/* ------------------------------------------------------------------------ */
/* 16-bit encode: round to nearest, ties to even (IEEE-754 default rounding).  */
/* ------------------------------------------------------------------------ */

/* Round a non-negative double that holds an exact value to the nearest
 * integer, ties to even. */
static double orc_rne_integer(double q) {
    double fl = floor(q);
    double d = q - fl; /* exact: q and fl share an exponent range */
    if (d > 0.5) return fl + 1.0;
    if (d < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* binary32 -> bfloat16: keep the upper 16 bits, rounding the dropped 16 bits
 * to nearest, ties to the even kept pattern.  A carry out of the fraction
 * correctly bumps the exponent (and overflows the largest finite to inf). */
uint16_t orc_f32_to_bf16(float x) {
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u); /* NaN stays NaN (quiet) */
    uint32_t keep = u >> 16;
    uint32_t rest = u & 0xFFFFu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u) != 0u)) keep += 1u;
    return (uint16_t)keep;
}

/* binary32 -> binary16 from the definition: find the representable
 * neighbours on the binary16 grid for the magnitude and round to nearest,
 * ties to even.  Subnormals use the fixed 2^-24 grid.  Magnitudes at or above
 * 65520 (half-way between 65504 and 2^16, where the tie goes to the even
 * pattern, i.e. 2^16) become infinity. */
uint16_t orc_f32_to_f16(float x) {
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | 0x7E00u);
    double a = fabs((double)x);
    if (a >= 65520.0) return (uint16_t)(sign | 0x7C00u);
    if (a < 0x1p-14) {
        double n = orc_rne_integer(a * 0x1p24); /* exact scaling by 2^24 */
        return (uint16_t)(sign | (uint16_t)n);  /* n == 1024 encodes 2^-14 */
    }
    int e;
    double fr = frexp(a, &e);          /* a = fr * 2^e, fr in [0.5, 1) */
    double n = orc_rne_integer(ldexp(fr, 11)); /* significand in [1024, 2048] */
    if (n == 2048.0) { n = 1024.0; e += 1; }
    int biased = (e - 1) + 15;         /* value = (n / 1024) * 2^(e-1) */
    if (biased >= 31) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (uint16_t)(biased << 10) | (uint16_t)((int)n - 1024));
}

void orc_decode_array(int64_t n, const uint16_t* h, int32_t fmt, float* out) {
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < n; ++i) out[i] = orc_decode(h[i], fmt);
}

/* Cast of the fp32 master to the 16-bit parameter format. */
void orc_cast_array(int64_t n, const float* x, int32_t fmt, uint16_t* out) {
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < n; ++i) out[i] = fmt == 0 ? orc_f32_to_bf16(x[i]) : orc_f32_to_f16(x[i]);
}

/* ------------------------------------------------------------------------ */
/* Gradient reduction (the arithmetic of the reduce-scatter / all-reduce).    */
/* ------------------------------------------------------------------------ */

/* For i in [0, n): s = x_0 + x_1 + ... + x_{nd-1} in rank order, each add
 * rounded to binary32 (x_r = decode(rep[r][i])); g[i] = s / D.
 * D is N_d * loss_scale.  *nonfinite is set to 1 if any s is inf or NaN
 * (it is never cleared here). */
void orc_reduce(int32_t nd, const uint16_t* const* rep, int32_t fmt, int64_t n,
                float D, float* g, int32_t* nonfinite) {
    int32_t bad = 0;
    int64_t i;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (i = 0; i < n; ++i) {
        float s = orc_decode(rep[0][i], fmt);
        for (int32_t r = 1; r < nd; ++r) s = s + orc_decode(rep[r][i], fmt);
        if (!isfinite(s)) bad = 1;
        g[i] = s / D;
    }
    if (bad) *nonfinite = 1;
}

/* ------------------------------------------------------------------------ */
/* Gradient accumulation over micro-batches.                                 */
/* ------------------------------------------------------------------------ */

/* ZeRO-1 local accumulation (no communication): for one rank's 16-bit
 * micro-batch gradient x, acc[i] = x[i] on the first micro-batch, else
 * acc[i] = acc[i] + x[i] (binary32). */
void orc_accumulate(int64_t n, const uint16_t* x, int32_t fmt, float* acc, int32_t first) {
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < n; ++i) {
        float xi = orc_decode(x[i], fmt);
        acc[i] = first ? xi : acc[i] + xi;
    }
}

/* Reduce of fp32 accumulators (ZeRO-1 after the last micro-batch):
 * s = a_0 + a_1 + ... in rank order, g = s / D. */
void orc_reduce_f32(int32_t nd, const float* const* acc, int64_t n, float D, float* g, int32_t* nonfinite) {
    int32_t bad = 0;
    int64_t i;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (i = 0; i < n; ++i) {
        float s = acc[0][i];
        for (int32_t r = 1; r < nd; ++r) s = s + acc[r][i];
        if (!isfinite(s)) bad = 1;
        g[i] = s / D;
    }
    if (bad) *nonfinite = 1;
}

/* ZeRO-2/3 per-micro-batch reduce-scatter into the fp32 shard accumulator:
 * s = x_0 + ... + x_{nd-1} in rank order, then
 *   mode 1 (first):  acc = s
 *   mode 2 (middle): acc = acc + s
 *   mode 3 (last):   acc = (acc + s) / D   (the averaged gradient)  */
void orc_reduce_accumulate(int32_t nd, const uint16_t* const* rep, int32_t fmt, int64_t n, float* acc,
                           int32_t mode, float D, int32_t* nonfinite) {
    int32_t bad = 0;
    int64_t i;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (i = 0; i < n; ++i) {
        float s = orc_decode(rep[0][i], fmt);
        for (int32_t r = 1; r < nd; ++r) s = s + orc_decode(rep[r][i], fmt);
        if (mode == 1) {
            acc[i] = s;
        } else if (mode == 2) {
            acc[i] = acc[i] + s;
        } else {
            float t = acc[i] + s;
            if (!isfinite(t)) bad = 1;
            acc[i] = t / D;
        }
    }
    if (bad) *nonfinite = 1;
}

/* ------------------------------------------------------------------------ */
/* Global gradient norm pieces.                                              */
/* ------------------------------------------------------------------------ */

/* Chunk sums of squares: out[k] = sum over the 128 elements of chunk k, in
 * index order, of (double)g * (double)g.  A binary32 square is exact in
 * binary64, so only the additions round.  n must be a multiple of 128. */
void orc_sumsq_chunks128(const float* g, int64_t n, double* out) {
    int64_t nk = n / 128, k;
#pragma omp parallel for schedule(static)
    for (k = 0; k < nk; ++k) {
        double s = 0.0;
        for (int64_t j = 0; j < 128; ++j) {
            double x = (double)g[k * 128 + j];
            s = s + x * x;
        }
        out[k] = s;
    }
}

/* Plain left-to-right binary64 sum. */
double orc_sum_sequential(const double* x, int64_t n) {
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i) s = s + x[i];
    return s;
}

/* ------------------------------------------------------------------------ */
/* AdamW with decoupled weight decay, one binary32 rounding per operation.    */
/* ------------------------------------------------------------------------ */

typedef struct {
    float decay;      /* 1 - lr * weight_decay          */
    float beta1;      /* beta1                           */
    float beta2;      /* beta2                           */
    float omb1;       /* 1 - beta1                       */
    float omb2;       /* 1 - beta2                       */
    float eps;        /* epsilon                         */
    float step_size;  /* lr / (1 - beta1^t)              */
    float sqrt_bc2;   /* sqrt(1 - beta2^t)               */
    float clip;       /* global clip coefficient (1: none) */
} orc_adamw_consts;

/* For every element:
 *   g'  = g * clip
 *   p1  = p * decay
 *   m   = beta1 * m + (1 - beta1) * g'
 *   v   = beta2 * v + (1 - beta2) * (g' * g')
 *   den = sqrt(v) / sqrt(1 - beta2^t) + eps
 *   p   = p1 - (lr / (1 - beta1^t)) * (m / den)                            */
void orc_adamw(int64_t n, float* p, float* m, float* v, const float* g,
               const orc_adamw_consts* k) {
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < n; ++i) {
        float gi = g[i] * k->clip;
        float p1 = p[i] * k->decay;
        float mi = k->beta1 * m[i] + k->omb1 * gi;
        float vi = k->beta2 * v[i] + k->omb2 * (gi * gi);
        float den = sqrtf(vi) / k->sqrt_bc2 + k->eps;
        p[i] = p1 - k->step_size * (mi / den);
        m[i] = mi;
        v[i] = vi;
    }
}

int32_t orc_num_threads(void) {
#ifdef _OPENMP
    return (int32_t)omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int32_t n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads((int)n);
#else
    (void)n;
#endif
}
