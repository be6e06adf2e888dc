/*
 * Brute-force reference encoders used to pin the oracle's E2M1 / E4M3
 * rounding.  Deliberately a different algorithm from the oracle: the value
 * grid is enumerated from the bit-field definition and the nearest grid point
 * is found by comparing distances (ties go to the even code), instead of the
 * oracle's threshold ladder (E2M1) and binade-quantum rounding (E4M3).
 *
 * E2M1: 1 sign, 2 exponent, 1 mantissa bit ("SOAR Weekly Champion Notes 05",
 * section 02; "The Core of the Ledger").  E4M3: the OCP 8-bit "fn" format used
 * for the block scales ("The Core of the Ledger": FP8 (E4M3) block scale).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static double grid2[8];
static double grid4[127];
static int ready = 0;

static void init(void) {
  int c;
  if (ready) return;
  for (c = 0; c < 8; ++c) {
    int e = c >> 1, m = c & 1;
    /* subnormal when the exponent field is 0: 0.m * 2^(1-bias), bias 1 */
    grid2[c] = e ? pow(2.0, e - 1) * (1.0 + m / 2.0) : (m / 2.0);
  }
  for (c = 0; c < 127; ++c) {
    int e = c >> 3, m = c & 7;
    /* bias 7; exponent field 0 is subnormal 0.m * 2^(1-7) */
    grid4[c] = e ? pow(2.0, e - 7) * (1.0 + m / 8.0) : pow(2.0, -6) * (m / 8.0);
  }
  ready = 1;
}

static int nearest(const double *grid, int n, double a) {
  /* grid is increasing; binary search for the first point >= a */
  int lo = 0, hi = n - 1, best;
  if (a >= grid[n - 1]) return n - 1; /* saturate */
  while (lo < hi) {
    int mid = (lo + hi) / 2;
    if (grid[mid] >= a) hi = mid; else lo = mid + 1;
  }
  if (lo == 0) return 0;
  {
    double dlo = a - grid[lo - 1], dhi = grid[lo] - a;
    if (dlo < dhi) best = lo - 1;
    else if (dhi < dlo) best = lo;
    else best = ((lo - 1) % 2 == 0) ? lo - 1 : lo;
  }
  return best;
}

uint8_t bf_e2m1(float y) {
  init();
  return (uint8_t)((signbit(y) ? 8 : 0) | nearest(grid2, 8, fabs((double)y)));
}

uint8_t bf_e4m3(float y) {
  init();
  return (uint8_t)((signbit(y) ? 0x80 : 0) | nearest(grid4, 127, fabs((double)y)));
}

/* Compare against a buffer produced by the oracle for bit patterns
 * [start, start+count).  NaN patterns are skipped (undefined).  Returns the
 * number of mismatches and stores the first mismatching pattern. */
int64_t bf_compare(int which, uint32_t start, uint32_t count, const uint8_t *got, uint32_t *first_bad) {
  int64_t bad = 0;
  uint32_t i;
  init();
  for (i = 0; i < count; ++i) {
    uint32_t u = start + i;
    float f;
    uint8_t want;
    memcpy(&f, &u, 4);
    if (isnan(f)) continue;
    want = which == 2 ? bf_e2m1(f) : bf_e4m3(f);
    if (want != got[i]) {
      if (bad == 0) *first_bad = u;
      ++bad;
    }
  }
  return bad;
}
