/*
 * nvfp4kv oracle: a plain, scalar, single-threaded CPU statement of what the
 * NVFP4 / FP8 paged KV-cache hot path computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library and includes nothing from it.
 *
 * Sources (page title, section):
 *   [P1] "SOAR Weekly Champion Notes 05 | Zhisuan Team One: NVFP4 KV Cache and
 *        Mixed-Precision Practice", sections 02 (NVFP4 KV Cache) and
 *        03 (Mixed-precision KV Cache).
 *   [P2] "SGLang x Qwen x NVIDIA Collaboration: NVFP4 KV Cache Breaks
 *        Long-Context and Agentic Inference Bottlenecks", sections
 *        "The Core of the Ledger: 4-bit Does Not Equal 2x" and
 *        "Three Paths: Putting the Quantization Cost on the Compute-Bound Side".
 *
 * The pages fix the structure (E2M1 = 1 sign + 2 exponent + 1 mantissa bits,
 * two codes per byte, one E4M3 scale per 16 values, one FP32 global scale per
 * tensor, 9 bytes per 16 values) but give no formula.  The formulas below are
 * the plainest reading, stated once here and followed literally:
 *
 *   global g      = amax|x over the tensor| / (6 * 448)        (FP32 divide)
 *   per 16-block  : amax_b; d = 6*g; sf = amax_b / d; sbyte = E4M3_RNE_sat(sf)
 *                   S = E4M3 value of sbyte (exact); den = S*g
 *   per element   : code = E2M1_RNE_sat(x / den); byte j = code[2j] | code[2j+1]<<4
 *   zero cases    : g == 0 or den == 0  ->  scale byte 0x00 (g == 0) and codes 0x0
 *   FP8 layers    : s8 = amax / 448; byte = E4M3_RNE_sat(x / s8); s8 == 0 -> 0x00
 *
 * Cache layout (the pages give none): one contiguous block per (page, KV
 * head), pages then heads.  Inside a block the page's slots form groups of
 * R rows, R = 8 when the page size is a multiple of 8 (else R = page size):
 * slot off is row r = off % R of group off / R.  A group holds, in this
 * order, NVFP4: K codes (R*D/2 bytes), K scales (R*D/16), V codes (R*D/2),
 * V scales (R*D/16); FP8: K (R*D), V (R*D).  K bytes of a group are stored in
 * chunks of w = min(16, row bytes) bytes, chunk-major: byte j of row r sits at
 * (j/w)*R*w + r*w + j%w; K scales are row-major (R*D/16: row r, block b at
 * r*D/16 + b).  In a group of R = 8 rows, V is stored by row pairs (2c, 2c+1),
 * c = r/2, e = r%2, value d in block b = d/16 at j = d%16:
 *   NVFP4 codes : byte b*64 + c*16 + j holds value d of row 2c in its low
 *                 nibble and of row 2c+1 in its high nibble (e = nibble);
 *   NVFP4 scales: byte b*8 + r (block-major);
 *   FP8 bytes   : byte (j/8)*(D*4) + b*64 + c*16 + (j%8)*2 + e.
 * Groups of R != 8 rows (page sizes below 8) keep V row-major: byte d/2 of
 * row r at r*D/2 (nibble d%2), scales at r*D/16 + b, FP8 at r*D + d.
 * Only the positions differ from a plain row layout: every value's content is
 * the definition below.
 *
 * Every FP32 step is one IEEE-754 binary32 operation with round-to-nearest-even
 * and no fused multiply-add (build with -ffp-contract=off).  Attention runs in
 * FP64 over values dequantized exactly.
 *
 * Parity pins (tests, not here): the E2M1 code table, brute-force nearest-value
 * rounding over every FP32 bit pattern, the 9-byte ledger, exact round trips,
 * brute-force dense attention and the split / log-sum-exp merge identity; for
 * the chunked extend, a dense causal brute force, closed forms, causality and
 * the decode attention over an FP8 cache holding the same bytes.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* E2M1 ([P1] 02, [P2] Core of the Ledger: 1 sign + 2 exponent + 1 mantissa). */
/* Exponent bias 1; exponent field 0 is subnormal (0 or 0.5).                 */
/* ------------------------------------------------------------------------ */

double orc_e2m1_value(uint8_t code) {
  int e = (code >> 1) & 3, m = code & 1;
  double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return (code & 8) ? -mag : mag;
}

/* Round to nearest E2M1 value, ties to the even code, saturating at 6.
 * Magnitude grid 0, .5, 1, 1.5, 2, 3, 4, 6; the decision points are the
 * midpoints between neighbours, and at a midpoint the even code wins. */
uint8_t orc_e2m1_encode(float y) {
  uint8_t sign = signbit(y) ? 8 : 0;
  double a = fabs((double)y);
  uint8_t mag;
  if (isnan(y)) return 0; /* undefined; inputs are finite */
  if (a <= 0.25) mag = 0;
  else if (a < 0.75) mag = 1;
  else if (a <= 1.25) mag = 2;
  else if (a < 1.75) mag = 3;
  else if (a <= 2.5) mag = 4;
  else if (a < 3.5) mag = 5;
  else if (a <= 5.0) mag = 6;
  else mag = 7;
  return sign | mag;
}

/* ------------------------------------------------------------------------ */
/* E4M3, the OCP 8-bit "fn" variant ([P2] Core of the Ledger: the per-16   */
/* value block scale is E4M3; [P1] 01: FP8 KV cache): bias 7, 3 mantissa bits, */
/* subnormals m*2^-9, no infinities, 0x7F/0xFF = NaN, largest finite 448.     */
/* ------------------------------------------------------------------------ */

double orc_e4m3_value(uint8_t b) {
  int e = (b >> 3) & 15, m = b & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  v = (e == 0) ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 10);
  return (b & 0x80) ? -v : v;
}

/* Round to nearest E4M3 value, ties to even mantissa; finite values above
 * 448 and infinity saturate to 448 (sign kept). */
uint8_t orc_e4m3_encode(float y) {
  uint8_t sign = signbit(y) ? 0x80 : 0;
  double a, quantum, n, v;
  int ex, e, m;
  if (isnan(y)) return sign | 0x7F;
  a = fabs((double)y);
  if (a > 448.0) return sign | 0x7E;
  if (a < ldexp(1.0, -6)) {
    quantum = ldexp(1.0, -9); /* subnormal spacing */
  } else {
    frexp(a, &ex);                   /* a in [2^(ex-1), 2^ex) */
    quantum = ldexp(1.0, ex - 1 - 3); /* 3 mantissa bits */
  }
  n = nearbyint(a / quantum); /* exact quotient; default mode = ties-to-even */
  v = n * quantum;
  if (v == 0.0) return sign;
  if (v < ldexp(1.0, -6)) return sign | (uint8_t)n;
  frexp(v, &ex);
  e = ex - 1 + 7;
  m = (int)(v / ldexp(1.0, ex - 1) * 8.0) - 8;
  return sign | (uint8_t)(e << 3) | (uint8_t)m;
}

/* Bulk forms over raw FP32 bit patterns, for exhaustive sweeps. */
void orc_e2m1_encode_bits(uint32_t start, uint32_t count, uint8_t *out) {
  uint32_t i;
  for (i = 0; i < count; ++i) {
    uint32_t u = start + i;
    float f;
    memcpy(&f, &u, 4);
    out[i] = orc_e2m1_encode(f);
  }
}

void orc_e4m3_encode_bits(uint32_t start, uint32_t count, uint8_t *out) {
  uint32_t i;
  for (i = 0; i < count; ++i) {
    uint32_t u = start + i;
    float f;
    memcpy(&f, &u, 4);
    out[i] = orc_e4m3_encode(f);
  }
}

/* ------------------------------------------------------------------------ */
/* Global scale ([P2] Core of the Ledger: one FP32 scale per tensor).        */
/* g = amax / divisor, divisor 2688 = 6*448 for NVFP4 and                     */
/* 448 for the FP8 per-tensor scale.                                          */
/* ------------------------------------------------------------------------ */

float orc_global_scale(const float *x, int64_t n, float divisor) {
  float amax = 0.0f;
  int64_t i;
  for (i = 0; i < n; ++i) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  return amax / divisor;
}

/* ------------------------------------------------------------------------ */
/* Quantizers                                                                 */
/* ------------------------------------------------------------------------ */

/* One head vector x[D] -> D/2 code bytes and D/16 E4M3 scale bytes. */
static void nvfp4_quantize_vector(const float *x, int D, float g, uint8_t *codes, uint8_t *scales) {
  int b, i;
  for (b = 0; b < D / 16; ++b) {
    const float *blk = x + 16 * b;
    uint8_t q[16];
    float amax = 0.0f, d, sf, S, den;
    uint8_t sbyte;
    for (i = 0; i < 16; ++i) {
      float a = fabsf(blk[i]);
      if (a > amax) amax = a;
    }
    if (g == 0.0f) {
      sbyte = 0;
      den = 0.0f;
    } else {
      d = 6.0f * g;
      sf = amax / d;
      sbyte = orc_e4m3_encode(sf);
      S = (float)orc_e4m3_value(sbyte);
      den = S * g;
    }
    for (i = 0; i < 16; ++i) q[i] = (den == 0.0f) ? 0 : orc_e2m1_encode(blk[i] / den);
    for (i = 0; i < 8; ++i) codes[8 * b + i] = (uint8_t)(q[2 * i] | (q[2 * i + 1] << 4));
    scales[b] = sbyte;
  }
}

static void fp8_quantize_vector(const float *x, int D, float s8, uint8_t *out) {
  int i;
  for (i = 0; i < D; ++i) out[i] = (s8 == 0.0f) ? 0 : orc_e4m3_encode(x[i] / s8);
}

/* Byte positions inside the cache (layout in the header comment). */
static int64_t nv_block_bytes(int P, int D) { return (int64_t)P * 2 * (D / 2 + D / 16); }
static int64_t fp8_block_bytes(int P, int D) { return (int64_t)P * 2 * D; }

/* Rows per group. */
static int group_rows(int P) { return P % 8 == 0 ? 8 : P; }

/* K byte j of row r inside a group of R rows of `rowbytes` bytes: chunks of
 * w bytes, chunk-major. */
static int64_t k_chunked(int R, int rowbytes, int r, int j) {
  const int w = rowbytes < 16 ? rowbytes : 16;
  return (int64_t)(j / w) * R * w + (int64_t)r * w + j % w;
}

/* NVFP4: byte holding code d of slot `off` (kind 0 = K, 1 = V); *shift = its
 * nibble's bit offset (0 or 4). */
static int64_t nv_code_at(int64_t page, int Hkv, int h, int P, int D, int kind, int off, int d, int *shift) {
  const int R = group_rows(P), r = off % R;
  const int64_t half = (int64_t)R * (D / 2 + D / 16);  /* K (or V) part of a group */
  const int64_t base = (page * Hkv + h) * nv_block_bytes(P, D) + (int64_t)(off / R) * 2 * half + kind * half;
  if (kind == 0 || R != 8) {
    *shift = 4 * (d & 1);
    return base + (kind == 0 ? k_chunked(R, D / 2, r, d / 2) : (int64_t)r * (D / 2) + d / 2);
  }
  *shift = 4 * (r % 2);
  return base + (int64_t)(d / 16) * 64 + (r / 2) * 16 + d % 16;
}

/* NVFP4: byte holding the E4M3 scale of 16-value block b of slot `off`. */
static int64_t nv_scale_at(int64_t page, int Hkv, int h, int P, int D, int kind, int off, int b) {
  const int R = group_rows(P), r = off % R;
  const int64_t half = (int64_t)R * (D / 2 + D / 16);
  const int64_t base = (page * Hkv + h) * nv_block_bytes(P, D) + (int64_t)(off / R) * 2 * half + kind * half +
                       (int64_t)R * (D / 2);
  if (kind == 0 || R != 8) return base + (int64_t)r * (D / 16) + b;
  return base + (int64_t)b * 8 + r;
}

/* FP8 byte of value d (< D) of slot `off`. */
static int64_t fp8_at(int64_t page, int Hkv, int h, int P, int D, int kind, int off, int d) {
  const int R = group_rows(P), r = off % R;
  const int64_t base = (page * Hkv + h) * fp8_block_bytes(P, D) + (int64_t)(off / R) * 2 * R * D;
  if (kind == 0) return base + k_chunked(R, D, r, d);
  if (R != 8) return base + (int64_t)R * D + (int64_t)r * D + d;
  return base + (int64_t)R * D + (int64_t)((d % 16) / 8) * D * 4 + (int64_t)(d / 16) * 64 + (r / 2) * 16 +
         (d % 8) * 2 + r % 2;
}

/* Positions of the bytes of slot `off` inside its (page, KV head) block, in
 * the order K codes (D/2), K scales (D/16), V codes, V scales (D/16) (FP8: K
 * bytes, V bytes, value order).  V codes: the bytes holding values 0..D-1 in
 * value order, D bytes when V rows are paired (each byte holds one nibble of
 * the slot), else D/2.  out holds up to 2*D + D/8 entries; returns how many
 * were written, or -1. */
int orc_slot_bytes(int prec, int P, int D, int off, int64_t *out) {
  int kind, j, n = 0, sh;
  if (off < 0 || off >= P) return -1;
  for (kind = 0; kind < 2; ++kind) {
    if (prec == 0) {
      const int paired = kind == 1 && group_rows(P) == 8;
      for (j = 0; j < (paired ? D : D / 2); ++j) out[n++] = nv_code_at(0, 1, 0, P, D, kind, off, paired ? j : 2 * j, &sh);
      for (j = 0; j < D / 16; ++j) out[n++] = nv_scale_at(0, 1, 0, P, D, kind, off, j);
    } else {
      for (j = 0; j < D; ++j) out[n++] = fp8_at(0, 1, 0, P, D, kind, off, j);
    }
  }
  return n;
}

/* NVFP4 V: for slot `off` and value d, the byte (inside a block) and nibble
 * bit offset of its code; pos and shift hold D entries. */
int orc_v_code_layout(int P, int D, int off, int64_t *pos, int32_t *shift) {
  int d, sh;
  if (off < 0 || off >= P) return -1;
  for (d = 0; d < D; ++d) {
    pos[d] = nv_code_at(0, 1, 0, P, D, 1, off, d, &sh);
    shift[d] = sh;
  }
  return 0;
}

/* Quantized write into paged slots ([P1] 02, the quantized write; [P2] Three
 * Paths: new KV goes into the NVFP4 cache quantized).
 * k, v: [T][Hkv][D] FP32.  slot = page*P + offset; slot < 0 skips the token.
 * g[0], g[1] = global scales of K and V.  Returns 0, or -1 on a bad slot. */
int orc_nvfp4_quantize_write(const float *k, const float *v, int64_t T, int Hkv, int D,
                             const int64_t *slot_mapping, const float *g, int P, int64_t num_pages,
                             uint8_t *cache) {
  int64_t t;
  int h, kind;
  for (t = 0; t < T; ++t) {
    int64_t slot = slot_mapping[t], page;
    int off;
    if (slot < 0) continue;
    if (slot >= num_pages * P) return -1;
    page = slot / P;
    off = (int)(slot % P);
    for (h = 0; h < Hkv; ++h)
      for (kind = 0; kind < 2; ++kind) {
        const float *src = (kind ? v : k) + (t * Hkv + h) * D;
        uint8_t codes[512], scales[64];
        int j;
        if (D > 1024) return -1;
        nvfp4_quantize_vector(src, D, g[kind], codes, scales);
        for (j = 0; j < D; ++j) {  /* each code into its nibble, the other nibble kept */
          int sh;
          const int64_t at = nv_code_at(page, Hkv, h, P, D, kind, off, j, &sh);
          const uint8_t code = (uint8_t)((codes[j / 2] >> (4 * (j & 1))) & 15);
          cache[at] = (uint8_t)((cache[at] & ~(15 << sh)) | (code << sh));
        }
        for (j = 0; j < D / 16; ++j) cache[nv_scale_at(page, Hkv, h, P, D, kind, off, j)] = scales[j];
      }
  }
  return 0;
}

/* FP8 E4M3 write for the FP8 layers ([P1] 03: sensitive layers keep FP8);
 * s8[0], s8[1] = per-tensor scales of K, V. */
int orc_fp8_quantize_write(const float *k, const float *v, int64_t T, int Hkv, int D,
                           const int64_t *slot_mapping, const float *s8, int P, int64_t num_pages,
                           uint8_t *cache) {
  int64_t t;
  int h, kind;
  for (t = 0; t < T; ++t) {
    int64_t slot = slot_mapping[t], page;
    int off;
    if (slot < 0) continue;
    if (slot >= num_pages * P) return -1;
    page = slot / P;
    off = (int)(slot % P);
    for (h = 0; h < Hkv; ++h)
      for (kind = 0; kind < 2; ++kind) {
        uint8_t row[1024];
        int j;
        if (D > 1024) return -1;
        fp8_quantize_vector((kind ? v : k) + (t * Hkv + h) * D, D, s8[kind], row);
        for (j = 0; j < D; ++j) cache[fp8_at(page, Hkv, h, P, D, kind, off, j)] = row[j];
      }
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Dequantization of one cached head vector to FP64 (exact).                 */
/* prec 0 = NVFP4: x = e2m1(code) * E4M3(scale) * g                           */
/* prec 1 = FP8:   x = E4M3(byte) * s8                                        */
/* ------------------------------------------------------------------------ */

static void dequant_row(int prec, const uint8_t *cache, int64_t page, int Hkv, int h, int P, int D, int kind,
                        int off, float g, double *out) {
  int d;
  if (prec == 0) {
    for (d = 0; d < D; ++d) {
      int sh;
      const uint8_t code = (uint8_t)((cache[nv_code_at(page, Hkv, h, P, D, kind, off, d, &sh)] >> sh) & 15);
      const uint8_t sc = cache[nv_scale_at(page, Hkv, h, P, D, kind, off, d / 16)];
      out[d] = orc_e2m1_value(code) * orc_e4m3_value(sc) * (double)g;
    }
  } else {
    for (d = 0; d < D; ++d) out[d] = orc_e4m3_value(cache[fp8_at(page, Hkv, h, P, D, kind, off, d)]) * (double)g;
  }
}

/* Dequantize K (kind 0) or V (kind 1) of tokens [0, L) of one (sequence, KV
 * head) into dense [L][D]. */
int orc_gather_dequant(int prec, const uint8_t *cache, int kind, float g, const int32_t *block_row, int L, int Hkv,
                       int h, int D, int P, int64_t num_pages, double *out) {
  int t;
  for (t = 0; t < L; ++t) {
    int64_t page = block_row[t / P];
    if (page < 0 || page >= num_pages) return -1;
    dequant_row(prec, cache, page, Hkv, h, P, D, kind, t % P, g, out + (int64_t)t * D);
  }
  return 0;
}

static double bf16_bits_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* ------------------------------------------------------------------------ */
/* Paged GQA decode attention ([P2] Three Paths: decode reads the NVFP4 cache */
/* directly).  Plain dense softmax in FP64 over the gathered tokens of each   */
/* sequence; query head h reads KV head h / (Hq/Hkv); every token in [0, L)   */
/* is visible; L == 0 gives zeros.                                            */
/*   q   [B][Hq][D] BF16 bits;  out [B][Hq][D] FP64.                          */
/*   num_splits <= 1: one softmax over all L tokens.  num_splits > 1: the L   */
/*   tokens are cut into num_splits equal contiguous ranges (the last ones    */
/*   may be empty), each range gives (o_k = sum p v, m_k, l_k) and the ranges */
/*   are merged with the log-sum-exp rule M = max m_k,                        */
/*   out = sum e^(m_k - M) o_k / sum e^(m_k - M) l_k.                         */
/* ------------------------------------------------------------------------ */
int orc_paged_decode_attention(const uint16_t *q, int B, int Hq, int Hkv, int D, int P, int prec,
                               const uint8_t *cache, const float *g, const int32_t *block_table,
                               int max_pages, const int32_t *seq_lens, int64_t num_pages, double sm_scale,
                               int num_splits, double *out) {
  int b, h, G = Hq / Hkv;
  int rc = 0;
  for (b = 0; b < B && rc == 0; ++b) {
    int L = seq_lens[b];
    for (h = 0; h < Hkv && rc == 0; ++h) {
      double *K, *V, *s;
      int j;
      if (L <= 0) {
        for (j = 0; j < G; ++j) memset(out + ((int64_t)b * Hq + h * G + j) * D, 0, sizeof(double) * D);
        continue;
      }
      if ((L + P - 1) / P > max_pages) return -1;
      K = (double *)malloc(sizeof(double) * (size_t)L * D);
      V = (double *)malloc(sizeof(double) * (size_t)L * D);
      s = (double *)malloc(sizeof(double) * (size_t)L);
      rc |= orc_gather_dequant(prec, cache, 0, g[0], block_table + (int64_t)b * max_pages, L, Hkv, h, D, P,
                               num_pages, K);
      rc |= orc_gather_dequant(prec, cache, 1, g[1], block_table + (int64_t)b * max_pages, L, Hkv, h, D, P,
                               num_pages, V);
      for (j = 0; j < G && rc == 0; ++j) {
        int qh = h * G + j, t, d, nsp = num_splits > 1 ? num_splits : 1, sp;
        const uint16_t *qv = q + ((int64_t)b * Hq + qh) * D;
        double *o = out + ((int64_t)b * Hq + qh) * D;
        double M = -INFINITY, lsum = 0.0;
        double *ms = (double *)malloc(sizeof(double) * nsp), *ls = (double *)malloc(sizeof(double) * nsp);
        double *os = (double *)calloc((size_t)nsp * D, sizeof(double));
        for (t = 0; t < L; ++t) {
          double acc = 0.0;
          for (d = 0; d < D; ++d) acc += bf16_bits_to_double(qv[d]) * K[(int64_t)t * D + d];
          s[t] = acc * sm_scale;
        }
        for (sp = 0; sp < nsp; ++sp) {
          int chunk = (L + nsp - 1) / nsp, t0 = sp * chunk, t1 = t0 + chunk < L ? t0 + chunk : L;
          double m = -INFINITY, l = 0.0;
          for (t = t0; t < t1; ++t)
            if (s[t] > m) m = s[t];
          for (t = t0; t < t1; ++t) {
            double p = exp(s[t] - m);
            l += p;
            for (d = 0; d < D; ++d) os[(int64_t)sp * D + d] += p * V[(int64_t)t * D + d];
          }
          ms[sp] = m;
          ls[sp] = l;
          if (m > M) M = m;
        }
        for (d = 0; d < D; ++d) o[d] = 0.0;
        for (sp = 0; sp < nsp; ++sp) {
          double w;
          if (ls[sp] == 0.0) continue; /* empty range */
          w = exp(ms[sp] - M);
          lsum += w * ls[sp];
          for (d = 0; d < D; ++d) o[d] += w * os[(int64_t)sp * D + d];
        }
        for (d = 0; d < D; ++d) o[d] /= lsum;
        free(ms);
        free(ls);
        free(os);
      }
      free(K);
      free(V);
      free(s);
    }
  }
  return rc;
}

/* ------------------------------------------------------------------------ */
/* Chunked-extend dequant into the shared FP8 workspace ([P2] Three Paths:    */
/* for chunked extend the cached prefix is gathered and dequantized into an   */
/* FP8 workspace shared by all layers).  For sequence seq_ids[i], tokens [0, prefix_lens[i]) */
/* go to workspace rows cu_prefix[i] + t, layout [rows][Hkv][D] E4M3:          */
/*   w = e2m1(code) * S       (exact in FP32)                                 */
/*   r = g / ws_scale         (FP32 divide, once per K and V)                  */
/*   byte = E4M3_RNE_sat(w * r)                                               */
/* ------------------------------------------------------------------------ */
int orc_dequant_to_fp8_workspace(const int32_t *block_table, int max_pages, const int32_t *seq_ids,
                                 const int32_t *prefix_lens, const int64_t *cu_prefix, int n, int Hkv, int D,
                                 int P, int64_t num_pages, const uint8_t *cache, const float *g,
                                 const float *ws_scale, uint8_t *ws_k, uint8_t *ws_v) {
  int i, pass;
  for (pass = 0; pass < 2; ++pass) {
    uint8_t *ws = pass ? ws_v : ws_k;
    float r;
    if (!(ws_scale[pass] > 0.0f)) return -1;
    r = g[pass] / ws_scale[pass];
    for (i = 0; i < n; ++i) {
      const int32_t *brow = block_table + (int64_t)seq_ids[i] * max_pages;
      int t, h, d;
      for (t = 0; t < prefix_lens[i]; ++t) {
        int64_t page = brow[t / P];
        if (page < 0 || page >= num_pages) return -1;
        for (h = 0; h < Hkv; ++h) {
          uint8_t *dst = ws + ((cu_prefix[i] + t) * Hkv + h) * D;
          for (d = 0; d < D; ++d) {
            int sh;
            const uint8_t code = (uint8_t)((cache[nv_code_at(page, Hkv, h, P, D, pass, t % P, d, &sh)] >> sh) & 15);
            const uint8_t sc = cache[nv_scale_at(page, Hkv, h, P, D, pass, t % P, d / 16)];
            float w = (float)(orc_e2m1_value(code) * orc_e4m3_value(sc));
            dst[d] = orc_e4m3_encode(w * r);
          }
        }
      }
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* The current chunk joins the FP8 workspace ([P2] Three Paths: the chunk's  */
/* KV is appended to the dequantized prefix in the FP8 workspace and FP8      */
/* attention runs over both).  The pages give no rule for the chunk's FP8 bytes; the    */
/* plainest reading is the per-tensor FP8 quantizer of the FP8 layers with    */
/* the workspace scale: byte = E4M3_RNE_sat(x / ws_scale) (FP32 divide).      */
/* Token t of k / v ([T][Hkv][D] FP32) goes to workspace row rows[t]          */
/* (negative: skipped; >= ws_rows: error).                                    */
/* ------------------------------------------------------------------------ */
int orc_fp8_workspace_append(const float *k, const float *v, int64_t T, int Hkv, int D, const int64_t *rows,
                             const float *ws_scale, int64_t ws_rows, uint8_t *ws_k, uint8_t *ws_v) {
  int64_t t;
  int kind;
  if (!(ws_scale[0] > 0.0f) || !(ws_scale[1] > 0.0f)) return -1;
  for (t = 0; t < T; ++t) {
    int64_t r = rows[t];
    if (r < 0) continue;
    if (r >= ws_rows) return -1;
    for (kind = 0; kind < 2; ++kind)
      fp8_quantize_vector((kind ? v : k) + t * Hkv * D, Hkv * D, ws_scale[kind], (kind ? ws_v : ws_k) + r * Hkv * D);
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Chunked-extend attention over the FP8 workspace ([P2] Three Paths: the     */
/* chunk's queries attend, in FP8 attention, to the dequantized prefix        */
/* concatenated with the chunk's own KV).  Sequence i owns workspace rows     */
/* [cu_kv[i], cu_kv[i] + kv_lens[i]): positions 0 .. kv_lens[i]-1, prefix     */
/* first, then the chunk.  Its nq = cu_q[i+1] - cu_q[i] queries are the last  */
/* nq positions: query j sits at position kv_lens[i] - nq + j and sees the    */
/* positions up to and including its own (causal inside the chunk).  Query   */
/* head qh reads KV head qh / (Hq / Hkv).  K = E4M3(byte) * ws_scale[0],      */
/* V = E4M3(byte) * ws_scale[1] (exact in FP64); plain softmax in FP64.      */
/*   q [Tq][Hq][D] BF16 bits, out [Tq][Hq][D] FP64.                           */
/* ------------------------------------------------------------------------ */
int orc_fp8_extend_attention(const uint16_t *q, const int64_t *cu_q, const uint8_t *ws_k, const uint8_t *ws_v,
                             const int64_t *cu_kv, const int32_t *kv_lens, int n, int Hq, int Hkv, int D,
                             const float *ws_scale, double sm_scale, double *out) {
  int i, G;
  if (Hkv <= 0 || Hq % Hkv != 0) return -1;
  G = Hq / Hkv;
  for (i = 0; i < n; ++i) {
    const int64_t nq = cu_q[i + 1] - cu_q[i];
    const int L = kv_lens[i];
    int64_t j;
    int qh;
    double *s;
    if (nq < 0 || nq > L) return -1;
    s = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    for (j = 0; j < nq; ++j) {
      const int64_t pos = L - nq + j; /* this query's position; it sees [0, pos] */
      for (qh = 0; qh < Hq; ++qh) {
        const int h = qh / G;
        const uint16_t *qv = q + ((cu_q[i] + j) * Hq + qh) * D;
        double *o = out + ((cu_q[i] + j) * Hq + qh) * D;
        double m = -INFINITY, l = 0.0;
        int64_t t;
        int d;
        for (t = 0; t <= pos; ++t) {
          const uint8_t *kr = ws_k + ((cu_kv[i] + t) * Hkv + h) * D;
          double acc = 0.0;
          for (d = 0; d < D; ++d) acc += bf16_bits_to_double(qv[d]) * (orc_e4m3_value(kr[d]) * (double)ws_scale[0]);
          s[t] = acc * sm_scale;
          if (s[t] > m) m = s[t];
        }
        for (d = 0; d < D; ++d) o[d] = 0.0;
        for (t = 0; t <= pos; ++t) {
          const uint8_t *vr = ws_v + ((cu_kv[i] + t) * Hkv + h) * D;
          const double p = exp(s[t] - m);
          l += p;
          for (d = 0; d < D; ++d) o[d] += p * (orc_e4m3_value(vr[d]) * (double)ws_scale[1]);
        }
        for (d = 0; d < D; ++d) o[d] /= l;
      }
    }
    free(s);
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Initial-prefill write from FP8 ([P2] Three Paths: in the initial prefill  */
/* the attention runs on FP8 K/V and the KV is requantized from FP8 into the */
/* NVFP4 cache).  The FP8 input is decoded with its per-tensor scale, one   */
/* FP32 multiply per value, x = E4M3(byte) * s8[kind] (exact E4M3 value,    */
/* rounded once), then written by the NVFP4 quantized write above with the  */
/* NVFP4 global scales g.  k8, v8: [T][Hkv][D] E4M3 bytes.                  */
/* ------------------------------------------------------------------------ */
int orc_nvfp4_requantize_write_fp8(const uint8_t *k8, const uint8_t *v8, const float *s8, int64_t T, int Hkv,
                                   int D, const int64_t *slot_mapping, const float *g, int P, int64_t num_pages,
                                   uint8_t *cache) {
  const int64_t n = T * Hkv * D;
  float *k = (float *)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
  float *v = (float *)malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
  int64_t i;
  int rc;
  for (i = 0; i < n; ++i) {
    k[i] = (float)orc_e4m3_value(k8[i]) * s8[0];
    v[i] = (float)orc_e4m3_value(v8[i]) * s8[1];
  }
  rc = orc_nvfp4_quantize_write(k, v, T, Hkv, D, slot_mapping, g, P, num_pages, cache);
  free(k);
  free(v);
  return rc;
}
