/*
 * oracle.c -- plain, slow, obviously correct CPU oracle for the logical-rank
 * all-reduce and allgather.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the bench's CPU-baseline / reference arm may load this code.  It shares no
 * code, header, table or helper with the CUDA library in
 * tensor_decode_all_gb300/csrc, and it includes nothing from there.
 *
 * What it computes (the plain definition; the method reaches it exactly):
 *
 *   all-reduce: for inputs x_0 .. x_{R-1}, each n elements of format D
 *   (IEEE binary16 or bfloat16), every rank r receives
 *
 *       out_r[i] = RNE_D( (..((f32(x_0[i]) + f32(x_1[i])) + f32(x_2[i])) ..)
 *                         + f32(x_{R-1}[i]) )
 *
 *   with IEEE binary32 additions (round to nearest, ties to even), taken in
 *   rank order, and one final rounding to D.  Sources:
 *     - "[Kernel] Two-rank FP16 all-reduce through pinned host memory for GPUs
 *       without P2P", section "Purpose": each block adds
 *       the peer's chunk; the sum has a single FP16 rounding, is commutative and
 *       gives both ranks the same bits.
 *     - "[SM120] Add optional FlashInfer PCIe-IPC all-reduce for switch-free
 *       hosts", section "Accuracy": with eight ranks the
 *       accumulation order moves results by one bf16 step, so the order must be
 *       fixed; this oracle fixes it as rank order 0..R-1 on every rank.
 *   Readings where the pages are silent: the accumulator starts at f32(x_0)
 *   (not at +0.0, which would turn an all-(-0) sum into +0); no fused
 *   multiply-add or reassociation; overflow rounds to +-inf; subnormal results
 *   are kept; a NaN anywhere gives a NaN (its payload is not specified).
 *
 *   allgather: every rank receives x_0 || x_1 || .. || x_{R-1}, the flat
 *   rank-major concatenation of the shards ("fix(group): run each rank on a
 *   non-blocking stream", sections "What" and
 *   "Why": DeviceGroup.allgather of the complex64 S_j and core uploads).
 *
 * The conversions between the 16-bit formats and binary32 are written here from
 * the IEEE 754 bit layouts (sign | biased exponent | fraction):
 *   binary16: 1 | 5 (bias 15)  | 10      bfloat16: 1 | 8 (bias 127) | 7
 *   binary32: 1 | 8 (bias 127) | 23
 * Build flags must keep binary32 arithmetic exact-IEEE: no -ffast-math, and
 * -ffp-contract=off (there are only additions here, but the flag documents it).
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F16 1
#define ORACLE_BF16 2

static uint32_t f32_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

static float bits_f32(uint32_t u) {
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Widen binary16 -> binary32.  Exact: every binary16 value is a binary32 value. */
static float widen_f16(uint16_t h) {
    uint32_t sign = (uint32_t)(h >> 15) << 31;
    uint32_t e = (h >> 10) & 0x1fu;
    uint32_t m = h & 0x3ffu;
    if (e == 0x1fu) {                       /* inf (m == 0) or NaN (m != 0) */
        return bits_f32(sign | 0x7f800000u | (m << 13));
    }
    if (e == 0) {
        if (m == 0) return bits_f32(sign);  /* +-0 */
        /* subnormal: value m * 2^-24; normalise so the leading 1 sits at bit 10 */
        int k = 0;
        while ((m & 0x400u) == 0) { m <<= 1; k++; }
        /* value = 1.f * 2^(-14 - k) */
        uint32_t e32 = (uint32_t)(127 - 14 - k);
        return bits_f32(sign | (e32 << 23) | ((m & 0x3ffu) << 13));
    }
    /* normal: value 1.m * 2^(e - 15) */
    return bits_f32(sign | ((e - 15u + 127u) << 23) | (m << 13));
}

/* Widen bfloat16 -> binary32.  bfloat16 is the top half of a binary32. */
static float widen_bf16(uint16_t b) {
    return bits_f32((uint32_t)b << 16);
}

/*
 * Round a binary32 value to a narrower IEEE-style format with `frac` fraction
 * bits, minimum normal exponent `emin` and maximum finite exponent `emax`,
 * round to nearest, ties to even.  Returns the 16-bit encoding, whose exponent
 * field has bias `bias`.
 *
 * Method: write |x| = sig * 2^(ex - 23) with sig an integer (24 bits for a
 * normal binary32).  In the target, values of exponent E >= emin are spaced by
 * 2^(E - frac); below emin (subnormals) by 2^(emin - frac).  So the target
 * quantum exponent is q = max(E, emin) - frac.  Drop the low (q - (ex - 23))
 * bits of sig with round-half-even; the kept integer k gives |result| = k * 2^q.
 */
static uint16_t narrow_f32(float x, int frac, int emin, int emax, int bias) {
    uint32_t u = f32_bits(x);
    uint16_t sign = (uint16_t)((u >> 31) << 15);
    uint32_t e = (u >> 23) & 0xffu;
    uint32_t m = u & 0x7fffffu;
    uint16_t exp_all_ones = (uint16_t)(((1u << (15 - frac)) - 1u) << frac);

    if (e == 0xffu) {
        if (m != 0) return (uint16_t)(sign | exp_all_ones | (1u << (frac - 1))); /* quiet NaN */
        return (uint16_t)(sign | exp_all_ones);                                  /* inf */
    }
    if (e == 0 && m == 0) return sign;                                           /* +-0 */

    int ex;          /* unbiased exponent of the leading bit */
    uint32_t sig;    /* integer significand, |x| = sig * 2^(ex - 23) */
    if (e == 0) {    /* binary32 subnormal: |x| = m * 2^-149 = m * 2^(-126 - 23) */
        ex = -126;
        sig = m;
    } else {
        ex = (int)e - 127;
        sig = m | 0x800000u;
    }

    int q = (ex > emin ? ex : emin) - frac;  /* quantum exponent in the target */
    int shift = q - (ex - 23);               /* low bits of sig to drop (>= 0 here) */
    uint64_t k;
    if (shift <= 0) {
        k = (uint64_t)sig << (-shift);       /* cannot happen for frac < 23, kept for clarity */
    } else if (shift > 25) {
        k = 0;                               /* |x| < 2^(q-1): below half a quantum */
    } else {
        uint64_t s = sig;
        k = s >> shift;
        uint64_t rem = s & ((1ull << shift) - 1ull);
        uint64_t half = 1ull << (shift - 1);
        if (rem > half || (rem == half && (k & 1ull))) k++;
    }
    /* |result| = k * 2^q.  Encode. */
    if (q == emin - frac) {
        /* subnormal range (or rounded up into the smallest normal: k == 2^frac,
           which the encoding below handles, since field = k for k <= 2^frac) */
        if (k < (1ull << frac)) return (uint16_t)(sign | (uint16_t)k);
        /* k in [2^frac, 2^(frac+1)]: normal with exponent emin (or emin+1 if k hit 2^(frac+1)) */
    }
    int E = q + frac;                        /* exponent of the leading bit if k in [2^frac, 2^(frac+1)) */
    if (k == (1ull << (frac + 1))) {         /* rounding carried into the next binade */
        k >>= 1;
        E += 1;
    }
    if (E > emax) return (uint16_t)(sign | exp_all_ones);      /* overflow: |x| rounds to >= 2^(emax+1) */
    uint32_t field = (uint32_t)(E + bias);
    return (uint16_t)(sign | (field << frac) | (uint32_t)(k - (1ull << frac)));
}

static uint16_t narrow_f16(float x) { return narrow_f32(x, 10, -14, 15, 15); }
static uint16_t narrow_bf16(float x) { return narrow_f32(x, 7, -126, 127, 127); }

static float widen(int fmt, uint16_t v) {
    return fmt == ORACLE_F16 ? widen_f16(v) : widen_bf16(v);
}

static uint16_t narrow(int fmt, float x) {
    return fmt == ORACLE_F16 ? narrow_f16(x) : narrow_bf16(x);
}

/* ---- exported, so tests can pin each piece ---- */

float oracle_widen(int fmt, uint16_t v) { return widen(fmt, v); }

uint16_t oracle_narrow(int fmt, float x) { return narrow(fmt, x); }

/*
 * All-reduce oracle.  ins[p] points to rank p's n input elements (16-bit
 * patterns of format fmt); outs[r] receives rank r's n output elements.  Each
 * rank's output is computed from the definition on its own, as the method does
 * on every rank.  nthreads > 1 spreads the element loop over OpenMP threads
 * (the arithmetic per element is unchanged).  Returns 0, or -1 on a bad
 * argument.
 */
int oracle_allreduce(int R, int fmt, const uint16_t *const *ins, uint16_t *const *outs,
                     size_t n, int nthreads) {
    if (R < 1 || (fmt != ORACLE_F16 && fmt != ORACLE_BF16) || !ins || !outs) return -1;
    for (int r = 0; r < R; r++) {
        uint16_t *out = outs[r];
        if (!out) continue;
        long long nn = (long long)n;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nthreads > 0 ? nthreads : 1) if (nthreads > 1)
#endif
        for (long long i = 0; i < nn; i++) {
            float acc = widen(fmt, ins[0][i]);
            for (int p = 1; p < R; p++) {
                acc = acc + widen(fmt, ins[p][i]);
            }
            out[i] = narrow(fmt, acc);
        }
    }
    (void)nthreads;
    return 0;
}

/*
 * Allgather oracle.  ins[p] points to rank p's shard of `bytes` bytes; outs[r]
 * receives R * bytes bytes: shard 0, then shard 1, ..., then shard R-1.
 */
int oracle_allgather(int R, const void *const *ins, void *const *outs, size_t bytes) {
    if (R < 1 || !ins || !outs) return -1;
    for (int r = 0; r < R; r++) {
        unsigned char *out = (unsigned char *)outs[r];
        if (!out) continue;
        for (int p = 0; p < R; p++) {
            memcpy(out + (size_t)p * bytes, ins[p], bytes);
        }
    }
    return 0;
}

/* Element-wise forms of the two conversions, for pinning them on their own. */
void oracle_widen_array(int fmt, const uint16_t *in, float *out, size_t n) {
    for (size_t i = 0; i < n; i++) out[i] = widen(fmt, in[i]);
}

void oracle_narrow_array(int fmt, const float *in, uint16_t *out, size_t n) {
    for (size_t i = 0; i < n; i++) out[i] = narrow(fmt, in[i]);
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
