/*
 * CPU oracle for tile-elementwise streaming.  TEST INFRASTRUCTURE ONLY: the
 * tests, the smoke check and the benchmark's CPU-baseline leg call it; the
 * library never does.  It shares no code, header or table with the CUDA path.
 *
 * What it computes.  Staging a tile through shared memory, splitting it into
 * TMA boxes and pipelining the stages must not change a single value, so the
 * result of the whole path is the plain elementwise definition applied to
 * every element of the [rows, cols] tensor:
 *
 *   copy  out = a, bit for bit    (TVM "copy_async -> tma", Demonstration
 *                                  program: the tile read back equals A)
 *   sqrt  out = RN_t(sqrt(a))     (TVM "elementwise -> smem", Generated CUDA:
 *                                  the tile equals sqrt(A))
 *   exp   out ~ exp(a)            (same page, "How inputs change the
 *                                  algorithm": unary ops per component)
 *   add   out = RN_t(a + b)       (same table: binary ops combine two inputs)
 *   mul   out = RN_t(a * b)
 *   fma   out = RN_t(a * b + c)   (same table: fma is a * b + c), one rounding
 *
 * RN_t is round-to-nearest, ties-to-even, into the element type t (fp16,
 * bf16 or fp32) with gradual underflow and overflow to infinity.  The pages
 * fix no precision, so every operation is evaluated in fp64 and rounded once
 * into t; the roundings that are not obviously single are argued where they
 * happen.
 *
 * Build: gcc -O2 -ffp-contract=off (never -ffast-math): the error-free sum
 * below relies on strict IEEE binary64 evaluation.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

enum { O_F16 = 0, O_BF16 = 1, O_F32 = 2 };
enum { O_COPY = 0, O_SQRT = 1, O_EXP = 2, O_ADD = 3, O_MUL = 4, O_FMA = 5 };

/* Format parameters: p significand bits (hidden bit included), exponent bits. */
static int fmt_p(int dt) { return dt == O_F16 ? 11 : dt == O_BF16 ? 8 : 24; }
static int fmt_ebits(int dt) { return dt == O_F16 ? 5 : 8; }
static int fmt_size(int dt) { return dt == O_F32 ? 4 : 2; }

/* ------------------------------------------------------------------------
 * Decoding: the exact value of a bit pattern, from the IEEE 754 definition
 * (sign, biased exponent, fraction; exponent field 0 = subnormal).
 * ---------------------------------------------------------------------- */
double tsxo_value(uint32_t bits, int dt)
{
    const int p = fmt_p(dt), eb = fmt_ebits(dt);
    const int bias = (1 << (eb - 1)) - 1;
    const uint32_t frac = bits & ((1u << (p - 1)) - 1);
    const uint32_t expf_ = (bits >> (p - 1)) & ((1u << eb) - 1);
    const int neg = (bits >> (p - 1 + eb)) & 1;
    double v;
    if (expf_ == (1u << eb) - 1)
        v = frac ? NAN : INFINITY;
    else if (expf_ == 0)
        v = ldexp((double)frac, 1 - bias - (p - 1));
    else
        v = ldexp((double)(frac | (1u << (p - 1))), (int)expf_ - bias - (p - 1));
    return neg ? -v : v;
}

/* ------------------------------------------------------------------------
 * Encoding: RN_t(x).  x is written as m * 2^q with q the quantum (unit in
 * the last place) of the binade of |x|, clamped at the subnormal quantum;
 * the integer part of |x| / 2^q is kept and the remainder decides the
 * rounding, ties going to the even integer.  A carry out of the significand
 * moves to the next binade; a result above the largest finite exponent is
 * infinity.  NaN becomes the positive canonical quiet NaN.
 * ---------------------------------------------------------------------- */
uint32_t tsxo_round(double x, int dt)
{
    const int p = fmt_p(dt), eb = fmt_ebits(dt);
    const int bias = (1 << (eb - 1)) - 1;
    const int emin = 1 - bias, emax = bias;
    const uint32_t exp_ones = (1u << eb) - 1;
    const uint32_t sign = signbit(x) ? (1u << (p - 1 + eb)) : 0u;

    if (isnan(x))
        return (exp_ones << (p - 1)) | (1u << (p - 2));
    if (isinf(x))
        return sign | (exp_ones << (p - 1));
    const double ax = fabs(x);
    if (ax == 0.0)
        return sign;

    int e2;
    (void)frexp(ax, &e2);          /* ax = f * 2^e2, f in [0.5, 1)          */
    int e = e2 - 1;                /* so 2^e <= ax < 2^(e+1)                */
    if (e < emin)
        e = emin;                  /* subnormals share the quantum of emin  */
    int q = e - (p - 1);

    const double scaled = ldexp(ax, -q);   /* exact: a power-of-two scaling */
    const double whole = floor(scaled);
    const double rem = scaled - whole;     /* exact: scaled < 2^p <= 2^24   */
    uint64_t m = (uint64_t)whole;
    if (rem > 0.5 || (rem == 0.5 && (m & 1u)))
        m += 1;
    if (m == (1ull << p)) {        /* carry into the next binade            */
        m >>= 1;
        q += 1;
    }
    if (m < (1ull << (p - 1)))     /* subnormal (or zero after rounding)    */
        return sign | (uint32_t)m;
    const int E = q + (p - 1);
    if (E > emax)
        return sign | (exp_ones << (p - 1));
    return sign | ((uint32_t)(E + bias) << (p - 1)) | (uint32_t)(m - (1ull << (p - 1)));
}

/* ------------------------------------------------------------------------
 * x + y in binary64 rounded to odd: the exactly rounded sum is kept if it is
 * exact, otherwise the neighbour with an odd last bit.  Rounding a
 * round-to-odd result of precision p' >= p + 2 to nearest in precision p
 * gives the correctly rounded result (S. Boldo and G. Melquiond, "Emulation
 * of FMA and correctly rounded sums: proved algorithms using rounding to
 * odd", IEEE Trans. Computers 57(4), 2008).  The rounding error of the sum
 * is recovered exactly by Knuth's TwoSum.
 * ---------------------------------------------------------------------- */
double tsxo_add_round_odd(double x, double y)
{
    double s = x + y;
    if (!isfinite(s))
        return s;
    const double yv = s - x;
    const double err = (x - (s - yv)) + (y - yv);
    if (err != 0.0) {
        uint64_t b;
        memcpy(&b, &s, sizeof b);
        if ((b & 1u) == 0)
            s = nextafter(s, err > 0.0 ? INFINITY : -INFINITY);
    }
    return s;
}

/* One element of one op, on exact fp64 values of the operands. */
static uint32_t apply(int op, int dt, double a, double b, double c)
{
    switch (op) {
    case O_SQRT:
        /* binary64 sqrt is correctly rounded; a second rounding into a
         * format of p <= 24 bits is innocuous for sqrt because 53 >= 2p + 2
         * (S. A. Figueroa, "When is double rounding innocuous?", SIGNUM
         * Newsletter 30(3), 1995). */
        return tsxo_round(sqrt(a), dt);
    case O_EXP:
        return tsxo_round(exp(a), dt);
    case O_ADD:
        return tsxo_round(tsxo_add_round_odd(a, b), dt);
    case O_MUL:
        /* a * b of two p-bit significands needs at most 2p <= 48 bits: the
         * binary64 product is exact, so this is the only rounding. */
        return tsxo_round(a * b, dt);
    case O_FMA:
        /* a * b is exact (as above); the sum is rounded to odd, then once
         * into t: a single rounding of the exact a * b + c. */
        return tsxo_round(tsxo_add_round_odd(a * b, c), dt);
    default:
        return 0;
    }
}

static uint32_t load_bits(const void *p, int64_t i, int dt)
{
    if (fmt_size(dt) == 4) {
        uint32_t v;
        memcpy(&v, (const char *)p + 4 * i, 4);
        return v;
    }
    uint16_t v;
    memcpy(&v, (const char *)p + 2 * i, 2);
    return v;
}

static void store_bits(void *p, int64_t i, int dt, uint32_t v)
{
    if (fmt_size(dt) == 4) {
        memcpy((char *)p + 4 * i, &v, 4);
    } else {
        const uint16_t h = (uint16_t)v;
        memcpy((char *)p + 2 * i, &h, 2);
    }
}

/* out[i] = op(a[i], b[i], c[i]) for i < n; element bits in and out.
 * Returns 0, or -1 for an unknown dtype / op or a missing operand. */
int tsxo_ewise(int dt, int op, int64_t n, const void *a, const void *b, const void *c, void *out)
{
    if (dt < O_F16 || dt > O_F32 || op < O_COPY || op > O_FMA || !a || !out)
        return -1;
    if ((op == O_ADD || op == O_MUL || op == O_FMA) && !b)
        return -1;
    if (op == O_FMA && !c)
        return -1;
    for (int64_t i = 0; i < n; ++i) {
        if (op == O_COPY) {
            store_bits(out, i, dt, load_bits(a, i, dt));
            continue;
        }
        const double av = tsxo_value(load_bits(a, i, dt), dt);
        const double bv = b ? tsxo_value(load_bits(b, i, dt), dt) : 0.0;
        const double cv = c ? tsxo_value(load_bits(c, i, dt), dt) : 0.0;
        store_bits(out, i, dt, apply(op, dt, av, bv, cv));
    }
    return 0;
}

/* dst[i] = the exact value of element i (bits of type dt), i < n. */
int tsxo_decode(int dt, int64_t n, const void *src, double *dst)
{
    if (dt < O_F16 || dt > O_F32 || !src || !dst)
        return -1;
    for (int64_t i = 0; i < n; ++i)
        dst[i] = tsxo_value(load_bits(src, i, dt), dt);
    return 0;
}
