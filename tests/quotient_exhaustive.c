/* Exhaustive check, run by tests/test_quotient_exhaustive.py (CPU only).
 *
 * The indexer-K store's rule is code = e4m3(RN32(k / scale)) with
 * scale = RN32(amax / 448).  Its kernel computes the quotient without a
 * division instruction:
 *     y  = RN(1 / scale)                 (once per token)
 *     q0 = RN(k * y)
 *     r  = RN(k - q0 * scale)            (one fused multiply-add)
 *     q1 = RN(q0 + r * y)                (one fused multiply-add)
 * and then ORs the sign bit of k into the code (q1 of k = -0 is +0).  This program enumerates
 * every pair (amax, k) of one input type -- bf16 or fp16, every finite
 * amax > 0 with amax / 448 >= 2^-90 (smaller scales take IEEE divisions),
 * every k with |k| <= amax, both signs -- and counts the pairs where q1
 * differs from the IEEE quotient k / scale in a way the e4m3 code can see:
 * either the two differ as fp32 values while one of them exceeds 2^-10 in
 * magnitude (below that, round-to-nearest-even gives the zero code), or
 * their sign bits differ after the sign fix.  C's float arithmetic is IEEE
 * single precision with round to nearest even and no flush to zero, and
 * fmaf() is the IEEE fused multiply-add, so each line is one of the
 * kernel's instructions.  Prints "<type> <pairs> <mismatches>".
 *
 * Usage: quotient_exhaustive {bf16|fp16} [threads] [uncorrected]
 * ("uncorrected" checks q0 itself, which must show mismatches: a check
 * that the enumeration can fail.)
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static int g_fp16;
static int g_threads;
static int g_uncorrected; /* check q0 instead of q1 (must fail) */

static float from_bits(uint32_t b) {
  float f;
  memcpy(&f, &b, 4);
  return f;
}

static uint32_t to_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}

/* The value of a 16-bit input pattern (sign bit 15). */
static float input_value(uint32_t h) {
  if (!g_fp16) return from_bits(h << 16);
  {
    const uint32_t e = (h >> 10) & 31u, m = h & 1023u;
    const float v = e == 0 ? ldexpf((float)m, -24)
                           : ldexpf((float)(m | 1024u), (int)e - 25);
    return (h & 0x8000u) ? -v : v;
  }
}

typedef struct {
  int index;
  long long pairs, bad;
} Work;

static void* run(void* arg) {
  Work* w = (Work*)arg;
  const uint32_t top = g_fp16 ? 0x7BFFu : 0x7F7Fu; /* largest finite */
  const float tiny = 0x1p-10f;
  for (uint32_t a = 1u + (uint32_t)w->index; a <= top;
       a += (uint32_t)g_threads) {
    const float amax = input_value(a);
    const float scale = amax / 448.0f;
    if (!(scale >= 0x1p-90f)) continue;
    const float y = 1.0f / scale;
    for (uint32_t kb = 0; kb <= a; ++kb) {
      for (int neg = 0; neg < 2; ++neg) {
        const float k = input_value(kb | (neg ? 0x8000u : 0u));
        const float ieee = k / scale;
        const float q0 = k * y;
        const float r = fmaf(-q0, scale, k);
        float q1 = g_uncorrected ? q0 : fmaf(r, y, q0);
        /* the kernel ORs k's sign bit into the code; the conversion is
           symmetric in the sign, so OR-ing it into q1 is the same */
        q1 = from_bits(to_bits(q1) | (to_bits(k) & 0x80000000u));
        const int big = fabsf(ieee) > tiny || fabsf(q1) > tiny;
        const int differ = big ? to_bits(q1) != to_bits(ieee)
                               : (to_bits(q1) >> 31) != (to_bits(ieee) >> 31);
        w->pairs += 1;
        w->bad += differ;
      }
    }
  }
  return NULL;
}

int main(int argc, char** argv) {
  if (argc < 2) return 2;
  g_fp16 = strcmp(argv[1], "fp16") == 0;
  g_threads = argc > 2 ? atoi(argv[2]) : 1;
  g_uncorrected = argc > 3 && strcmp(argv[3], "uncorrected") == 0;
  if (g_threads < 1) g_threads = 1;
  if (g_threads > 64) g_threads = 64;
  pthread_t tid[64];
  Work work[64];
  for (int i = 0; i < g_threads; ++i) {
    work[i].index = i;
    work[i].pairs = work[i].bad = 0;
    pthread_create(&tid[i], NULL, run, &work[i]);
  }
  long long pairs = 0, bad = 0;
  for (int i = 0; i < g_threads; ++i) {
    pthread_join(tid[i], NULL);
    pairs += work[i].pairs;
    bad += work[i].bad;
  }
  printf("%s %lld %lld\n", g_fp16 ? "fp16" : "bf16", pairs, bad);
  return 0;
}
