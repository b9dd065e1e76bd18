/* quotient_check.c -- exhaustive CPU check of the NVFP4 quantizer's division-free
 * element coding.  Test infrastructure: neither the oracle nor the CUDA library;
 * it restates, in scalar C, the arithmetic identity the quantizer kernel relies on.
 *
 * "Composer 2 Technical Report", section 6.1, asks for IEEE division in the NVFP4
 * quantizer: the code of x is E2M1(fl32(x / e)), e = fl32(dec(sb) S) with S =
 * fl32(amax / 2688) the per-token scale and sb the block's E4M3 scale code.  The
 * kernel never divides for e >= 2^-76; it forms
 *     n = fl32(x * (-r)),  rho = fl32(n * e + x),  t = fl32(rho * (-r) + n)
 * (r an approximate reciprocal of e, the two last steps fused multiply-adds) and
 * codes -t.  This program checks, with the C library's correctly rounded fmaf and
 * IEEE binary32 division:
 *   A. every positive finite bf16 amax, every sb in 1..126 with e >= 2^-76, every r
 *      within K ulps of fl32(1/e), every bf16 x > 0 with fl32(x / e) in
 *      [2^-4, 8], and x = +0 and -0: -t equals fl32(x / e) bit for bit;
 *   B. every STRIDE-th amax, all such sb and r, every finite bf16 x of either sign
 *      with |x / e| below 2^-4: |t| < 0.25 and t has the sign opposite to x's,
 *      so -t and fl32(x / e) have the same E2M1 code, a zero of x's sign; and
 *      for |x / e| in [2^-4, 8], negative x: -t equals fl32(x / e) bit for bit.
 * Larger quotients cannot occur (x is at most the block amax, and e is at least
 * the block amax / 6 up to the E4M3 rounding of the block scale).
 *
 * Usage: quotient_check K STRIDE.  Prints "checked=N mismatches=M".
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float from_bits(uint32_t b) {
  float f;
  memcpy(&f, &b, 4);
  return f;
}

static uint32_t to_bits(float f) {
  uint32_t b;
  memcpy(&b, &f, 4);
  return b;
}

/* Value of a positive E4M3 code (1..126): 4 exponent bits (bias 7), 3 mantissa bits. */
static float e4m3_decode(int code) {
  const int ex = (code >> 3) & 15, man = code & 7;
  return ex ? ldexpf(1.0f + (float)man / 8.0f, ex - 7) : ldexpf((float)man / 8.0f, -6);
}

/* The kernel's sequence; returns t (the kernel codes -t). */
static float negated_step(float x, float e, float nr) {
  const float n = x * nr;
  const float rho = fmaf(n, e, x);
  return fmaf(rho, nr, n);
}

int main(int argc, char **argv) {
  const int K = argc > 1 ? atoi(argv[1]) : 4;
  const int stride = argc > 2 ? atoi(argv[2]) : 997;
  const float min_scale = 0x1p-76f;
  long long checked = 0, mismatches = 0;
#pragma omp parallel for schedule(dynamic, 64) reduction(+ : checked, mismatches)
  for (uint32_t ab = 1; ab < 0x7F80u; ++ab) {
    const float amax = from_bits(ab << 16);
    const float S = amax / 2688.0f;
    const int sampled = (ab % (uint32_t)stride) == 0;
    for (int sb = 1; sb <= 126; ++sb) {
      const float e = e4m3_decode(sb) * S;
      if (!(e >= min_scale)) continue;
      const float rn = 1.0f / e;
      /* reciprocals rn - K ulps .. rn + K ulps */
      float r = rn;
      for (int k = 0; k < K; ++k) r = nextafterf(r, 0.0f);
      for (int k = -K; k <= K; ++k, r = nextafterf(r, INFINITY)) {
        const float nr = -r;
        /* A: zeros */
        for (int s = 0; s < 2; ++s) {
          const float x = s ? -0.0f : 0.0f;
          ++checked;
          if (to_bits(-negated_step(x, e, nr)) != to_bits(x / e)) ++mismatches;
        }
        /* A: positive x with quotient in [2^-4, 8] */
        uint32_t lo = to_bits(e * 0x1p-4f) >> 16, hi = (to_bits(e * 8.0f) >> 16) + 1;
        if (hi > 0x7F7Fu) hi = 0x7F7Fu;
        for (uint32_t xb = lo; xb <= hi; ++xb) {
          const float x = from_bits(xb << 16);
          const float want = x / e;
          if (!(want >= 0x1p-4f && want <= 8.0f)) continue;
          ++checked;
          if (to_bits(-negated_step(x, e, nr)) != to_bits(want)) ++mismatches;
          if (sampled) {
            ++checked;
            if (to_bits(-negated_step(-x, e, nr)) != to_bits(-want)) ++mismatches;
          }
        }
        if (!sampled) continue;
        /* B: every finite nonzero bf16 x, both signs, with |x / e| below 2^-4 */
        for (uint32_t xb = 1; xb < 0x7F80u; ++xb) {
          const float x = from_bits(xb << 16);
          if (!(x / e < 0x1p-4f)) break;
          for (int s = 0; s < 2; ++s) {
            const float xs = s ? -x : x;
            const float t = negated_step(xs, e, nr);
            ++checked;
            if (!(fabsf(t) < 0.25f) || signbit(t) == signbit(xs)) ++mismatches;
          }
        }
      }
    }
  }
  printf("checked=%lld mismatches=%lld\n", checked, mismatches);
  return mismatches != 0;
}
