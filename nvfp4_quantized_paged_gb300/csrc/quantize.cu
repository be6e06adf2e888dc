// Write-side kernels of the NVFP4 / FP8 paged KV cache:
//   * global scale (one FP32 per tensor, "SGLang x Qwen x NVIDIA ...", The
//     Core of the Ledger),
//   * NVFP4 quantized write into paged slots ("SOAR Weekly Champion Notes
//     05", 02: quantized write path; Three Paths: the new chunk is quantized
//     into the NVFP4 cache),
//   * FP8 E4M3 write for the FP8 layers (Notes 05, 03),
//   * chunked-extend prefix dequant into the shared FP8 workspace (Three Paths),
//   * element encoders.
//
// All are HBM-bound streaming kernels: one thread owns one 16-value block
// (one E4M3 scale), loads it with 128-bit loads, and stores its codes with one
// 64-bit (NVFP4) or 128-bit (FP8) store.  FP32 steps use the IEEE-rounded
// intrinsics (__fdiv_rn, __fmul_rn) so that no multiply-add is contracted and
// the bytes equal the quantizer stated in include/nvfp4kv.h.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <mutex>

#include "nvkv_device.cuh"
#include "nvkv_host.h"

namespace nvkv {
namespace {

constexpr int kD = 128;
constexpr int kBlocksPerRow = kD / 16;  // E4M3 scales per head vector

// ---------------------------------------------------------------------------
// Loading one 16-value block as FP32 (BF16 widens exactly).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void load16(const float *src, float (&x)[16]) {
  const float4 *p = reinterpret_cast<const float4 *>(src);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float4 v = __ldg(p + i);
    x[4 * i + 0] = v.x;
    x[4 * i + 1] = v.y;
    x[4 * i + 2] = v.z;
    x[4 * i + 3] = v.w;
  }
}

__device__ __forceinline__ void load16(const __nv_bfloat16 *src, float (&x)[16]) {
  const uint4 *p = reinterpret_cast<const uint4 *>(src);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint4 v = __ldg(p + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[8 * i + 2 * j + 0] = __uint_as_float(w[j] << 16);
      x[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
  }
}

// E4M3 input with its per-tensor scale (the prefill's FP8 K/V): each value
// decoded exactly, then one FP32 multiply, x = E4M3(byte) * s8.
__device__ __forceinline__ void load16(const uint8_t *src, float s8, float (&x)[16]) {
  const uint4 v = __ldg(reinterpret_cast<const uint4 *>(src));
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t lo = f16x2_from_e4m3x2<0>(w[j]), hi = f16x2_from_e4m3x2<1>(w[j]);
    x[4 * j + 0] = __fmul_rn(f32_lo(lo), s8);
    x[4 * j + 1] = __fmul_rn(f32_hi(lo), s8);
    x[4 * j + 2] = __fmul_rn(f32_lo(hi), s8);
    x[4 * j + 3] = __fmul_rn(f32_hi(hi), s8);
  }
}

// ---------------------------------------------------------------------------
// Global scale: amax over the tensor (atomic max on the bit pattern of a
// non-negative float), then one FP32 divide.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) amax_kernel(const T *__restrict__ x, int64_t n, bool vec,
                                                   uint32_t *out_bits) {
  float m = 0.0f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t n16 = vec ? n / 16 : 0;  // 128-bit loads need a 16-byte aligned base
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride) {
    float v[16];
    load16(x + 16 * i, v);
#pragma unroll
    for (int j = 0; j < 16; ++j) m = fmaxf(m, fabsf(v[j]));
  }
  for (int64_t i = 16 * n16 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    float v;
    if constexpr (sizeof(T) == 4) v = x[i];
    else v = __bfloat162float(x[i]);
    m = fmaxf(m, fabsf(v));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) m = fmaxf(m, red[w]);
    atomicMax(out_bits, __float_as_uint(m));  // non-negative floats order like their bits
  }
}

__global__ void divide_kernel(float *out, float divisor) {
  const float amax = __uint_as_float(*reinterpret_cast<uint32_t *>(out));
  out[0] = __fdiv_rn(amax, divisor);
}

// One 16-value block: its E4M3 scale byte and 16 E2M1 codes, two per byte
// (value 2j in the low nibble of byte j): lo = values 0..7, hi = 8..15.
__device__ __forceinline__ void quant16(const float (&x)[16], float g, uint32_t &sbyte, uint32_t &lo, uint32_t &hi) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  sbyte = 0;
  float den = 0.0f;
  if (g != 0.0f) {
    const float d = __fmul_rn(6.0f, g);
    const float sf = __fdiv_rn(amax, d);
    sbyte = e4m3x2_from_f32(sf, 0.0f) & 0xFFu;
    den = __fmul_rn(f32_from_e4m3(sbyte), g);
  }
  lo = hi = 0;
  if (den != 0.0f) {
    const float r = __frcp_rn(den);
    if (quot_fast_ok(r)) {  // codes of fl(x / den) from one reciprocal (exact, see e2m1x2_quot)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        lo |= e2m1x2_quot(x[2 * j], x[2 * j + 1], den, r) << (8 * j);
        hi |= e2m1x2_quot(x[8 + 2 * j], x[8 + 2 * j + 1], den, r) << (8 * j);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        lo |= e2m1x2_from_f32(__fdiv_rn(x[2 * j], den), __fdiv_rn(x[2 * j + 1], den)) << (8 * j);
        hi |= e2m1x2_from_f32(__fdiv_rn(x[8 + 2 * j], den), __fdiv_rn(x[8 + 2 * j + 1], den)) << (8 * j);
      }
    }
  }
}

// Four 4-bit codes (bits 15:0) -> the low nibbles of four bytes.
__device__ __forceinline__ uint32_t spread4(uint32_t four) {
  return (four & 0xFu) | ((four & 0xF0u) << 4) | ((four & 0xF00u) << 8) | ((four & 0xF000u) << 12);
}

// ---------------------------------------------------------------------------
// NVFP4 quantized write of one item = (kind K|V, token t, KV head h, 16-block).
// T = uint8_t: E4M3 input decoded with in_scale[kind] (initial prefill).
// V: value 16 blk + j goes to byte j of the pair's 16 bytes, nibble off % 2.
// When the neighbouring token (t ^ 1) holds the partner slot (tokens written
// in slot order, as prefill and decode do), the even token's item writes both
// slots' bytes with plain stores and the odd one has nothing to do;
// otherwise this slot's nibbles are cleared and set with atomics (the partner
// slot may be written by another thread of the same launch).
// ---------------------------------------------------------------------------
template <typename T>
__device__ void nvfp4_write_item(const T *__restrict__ k, const T *__restrict__ v, int64_t num_tokens,
                                 const int64_t *__restrict__ slot_mapping, const float *__restrict__ gs,
                                 const CacheDev &c, const float *__restrict__ in_scale, int kind, int64_t t, int h,
                                 int blk) {
  const int64_t th = t * c.Hkv + h;
  const int64_t tp = t ^ 1;
  const int64_t slot = slot_mapping[t];
  const int64_t slot_p = (kind == 1 && tp < num_tokens) ? slot_mapping[tp] : -1;  // loaded together
  if (slot < 0) return;
  if (slot >= static_cast<int64_t>(c.num_pages) * c.P) {
    if (kind == 0 && h == 0 && blk == 0) set_err(c.err, NVKV_DEVERR_SLOT);
    return;
  }
  const int64_t page = slot >> (__ffs(c.P) - 1);  // page sizes are powers of two (16, 32, 64)
  const int off = static_cast<int>(slot & (c.P - 1));
  const bool paired = slot_p == (slot ^ 1);
  if (paired && (t & 1)) return;
  float x[16];
  if constexpr (sizeof(T) == 1)
    load16((kind == 0 ? k : v) + th * kD + 16 * blk, in_scale[kind], x);
  else
    load16((kind == 0 ? k : v) + th * kD + 16 * blk, x);
  uint32_t sbyte, lo, hi;
  quant16(x, gs[kind], sbyte, lo, hi);
  if (kind == 0) {
    *reinterpret_cast<uint2 *>(c.data + c.nv_kcodes(page, h, off, blk)) = make_uint2(lo, hi);
    c.data[c.nv_scale(page, h, kind, off, blk)] = static_cast<uint8_t>(sbyte);
    return;
  }
  uint32_t *dst = reinterpret_cast<uint32_t *>(c.data + c.nv_vcodes(page, h, off, blk));
  if (paired) {
    float y[16];
    if constexpr (sizeof(T) == 1)
      load16(v + (tp * c.Hkv + h) * kD + 16 * blk, in_scale[kind], y);
    else
      load16(v + (tp * c.Hkv + h) * kD + 16 * blk, y);
    uint32_t sb2, lo2, hi2;
    quant16(y, gs[kind], sb2, lo2, hi2);
    const bool mine_even = (off & 1) == 0;
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t a = spread4(((q < 2 ? lo : hi) >> (16 * (q & 1))) & 0xFFFFu);
      const uint32_t b = spread4(((q < 2 ? lo2 : hi2) >> (16 * (q & 1))) & 0xFFFFu);
      w[q] = mine_even ? (a | (b << 4)) : (b | (a << 4));
    }
    *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    c.data[c.nv_scale(page, h, kind, off, blk)] = static_cast<uint8_t>(sbyte);
    c.data[c.nv_scale(page, h, kind, off ^ 1, blk)] = static_cast<uint8_t>(sb2);
    return;
  }
  const int sh = 4 * (off & 1);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t spread = spread4(((q < 2 ? lo : hi) >> (16 * (q & 1))) & 0xFFFFu);  // codes 4q .. 4q+3
    atomicAnd(dst + q, ~(0x0F0F0F0Fu << sh));
    atomicOr(dst + q, spread << sh);
  }
  c.data[c.nv_scale(page, h, kind, off, blk)] = static_cast<uint8_t>(sbyte);
}

// ---------------------------------------------------------------------------
// NVFP4 quantized write, one warp per (8 consecutive input tokens, KV head).
// When the 8 tokens go to the 8 slots of one 8-slot group in order (as a
// prefill or a chunk fills its pages), the warp builds the group's whole
// 1152-byte image in shared memory and stores it with 16-byte coalesced
// stores: lane = (token lane / 4, K blocks 2 (lane % 4), + 1) for K and
// (slot pair lane / 8, block lane % 8) for V, whose two tokens' codes share
// bytes.  Any other pattern (decode steps, skipped or scattered slots, a
// ragged last group) takes the item path above, 4 items per lane.
// ---------------------------------------------------------------------------
constexpr int kWriteWarps = 8;

template <typename T>
__global__ void __launch_bounds__(kWriteWarps * 32)
    nvfp4_write_kernel(const T *__restrict__ k, const T *__restrict__ v, int64_t num_tokens,
                       const int64_t *__restrict__ slot_mapping, const float *__restrict__ gs, CacheDev c,
                       const float *__restrict__ in_scale) {
  __shared__ __align__(16) uint8_t img[kWriteWarps][kNvGroup];
  // programmatic dependent of the previous kernel: wait for it before any
  // global access, then let the next kernel start its set-up
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t wid = static_cast<int64_t>(blockIdx.x) * kWriteWarps + warp;
  const int64_t ngroups = (num_tokens + 7) / 8;
  if (wid >= ngroups * c.Hkv) return;
  int h;
  int64_t t0;
  if ((c.Hkv & (c.Hkv - 1)) == 0) {  // shifts for power-of-two head counts
    h = static_cast<int>(wid & (c.Hkv - 1));
    t0 = (wid >> (__ffs(c.Hkv) - 1)) * 8;
  } else {
    h = static_cast<int>(wid % c.Hkv);
    t0 = (wid / c.Hkv) * 8;
  }
  const int64_t sl = t0 + (lane & 7) < num_tokens ? slot_mapping[t0 + (lane & 7)] : -1;
  const int64_t s0 = __shfl_sync(0xffffffffu, sl, 0);
  const bool whole = __all_sync(0xffffffffu, s0 >= 0 && (s0 & 7) == 0 && sl == s0 + (lane & 7) &&
                                                 s0 + 7 < static_cast<int64_t>(c.num_pages) * c.P);
  if (!whole) {
    for (int it = lane; it < 2 * 8 * kBlocksPerRow; it += 32) {
      const int kind = it / (8 * kBlocksPerRow), tt = (it / kBlocksPerRow) % 8, blk = it % kBlocksPerRow;
      if (t0 + tt < num_tokens) nvfp4_write_item<T>(k, v, num_tokens, slot_mapping, gs, c, in_scale, kind, t0 + tt, h, blk);
    }
    return;
  }
  uint8_t *im = img[warp];
  {  // K: token tk, blocks 2 (lane % 4) and 2 (lane % 4) + 1
    const int tk = lane >> 2;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int blk = 2 * (lane & 3) + j;
      float x[16];
      const int64_t e = ((t0 + tk) * c.Hkv + h) * kD + 16 * blk;
      if constexpr (sizeof(T) == 1)
        load16(k + e, in_scale[0], x);
      else
        load16(k + e, x);
      uint32_t sb, lo, hi;
      quant16(x, gs[0], sb, lo, hi);
      *reinterpret_cast<uint2 *>(im + (blk >> 1) * 128 + tk * 16 + (blk & 1) * 8) = make_uint2(lo, hi);
      im[kNvKScales + tk * 8 + blk] = static_cast<uint8_t>(sb);
    }
  }
  {  // V: slots 2p and 2p + 1, block blk (value 16 blk + j at byte j, slot 2p in the low nibble)
    const int p = lane >> 3, blk = lane & 7;
    uint32_t sb[2], lo[2], hi[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float x[16];
      const int64_t e = ((t0 + 2 * p + u) * c.Hkv + h) * kD + 16 * blk;
      if constexpr (sizeof(T) == 1)
        load16(v + e, in_scale[1], x);
      else
        load16(v + e, x);
      quant16(x, gs[1], sb[u], lo[u], hi[u]);
    }
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      w[q] = spread4(((q < 2 ? lo[0] : hi[0]) >> (16 * (q & 1))) & 0xFFFFu) |
             (spread4(((q < 2 ? lo[1] : hi[1]) >> (16 * (q & 1))) & 0xFFFFu) << 4);
    *reinterpret_cast<uint4 *>(im + kNvVCodes + blk * 64 + p * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    im[kNvVScales + blk * 8 + 2 * p] = static_cast<uint8_t>(sb[0]);
    im[kNvVScales + blk * 8 + 2 * p + 1] = static_cast<uint8_t>(sb[1]);
  }
  __syncwarp();
  const int64_t page = s0 >> (__ffs(c.P) - 1);  // page sizes are powers of two (16, 32, 64)
  const int off = static_cast<int>(s0 & (c.P - 1));
  uint4 *dst = reinterpret_cast<uint4 *>(c.data + c.block(page, h, kNvTokBytes) + static_cast<int64_t>(off >> 3) * kNvGroup);
  const uint4 *src = reinterpret_cast<const uint4 *>(im);
  for (int i = lane; i < kNvGroup / 16; i += 32) dst[i] = src[i];
}

// ---------------------------------------------------------------------------
// Initial-prefill write from FP8 K/V ([P2] Three Paths: the prefill's FP8 KV is
// requantized into the NVFP4 cache) by thresholds instead of per-value
// arithmetic.  Every value is x = fl(E4M3(byte) s8) and every block's divisor
// is den = fl(E4M3(sbyte) g), so a code depends only on (sbyte, byte):
// code = E2M1_RNE(fl(x_byte / den_sbyte)).  For s8 > 0 (finite) x grows with
// the byte's magnitude e = byte & 0x7F and is +-|x_e| with the byte's sign,
// and fl(. / den) and E2M1_RNE are monotone and odd, so the code is the
// byte's sign over a magnitude code that steps up at seven magnitudes:
// T_k(sbyte) = the least e whose magnitude code is >= k (k = 1..7; 128 when
// none).  These are found once per CTA by bisection with the write rule's
// own IEEE operations; a value's magnitude code is then #{k : e >= T_k}.  A
// block's amax is x of its largest magnitude and its scale byte is
// sb[e_max] = E4M3_RNE(fl(x_emax / fl(6 g))).  A block whose den is 0
// (g = 0, or the scale byte 0) writes code 0 everywhere, as the rule does.
// An input scale that is not a positive finite number, or a global scale that
// is negative or not finite, sends every item through the per-value path.
// NaN input bytes are outside the rule (undefined), as for every write.
// One warp per (8 tokens, KV head) as in nvfp4_write_kernel (whole 8-slot
// groups assembled in shared memory, other patterns through the item path),
// in a persistent grid of one CTA of 32 warps per SM.
// ---------------------------------------------------------------------------
constexpr int kRqWarps = 32;
constexpr int kRqScales = 127;                      // scale bytes 0 .. 0x7E (sf <= 448)
constexpr int kRqOffX = kRqWarps * kNvGroup;        // after the group images: [2][128] f32 x of each magnitude
constexpr int kRqOffDen = kRqOffX + 2 * 128 * 4;    // [2][127] f32 den of each scale byte (padded to 128)
constexpr int kRqOffThr = kRqOffDen + 2 * 128 * 4;  // [2][128] u8x8 T_1..T_7 of each scale byte (byte 7 unused)
constexpr int kRqOffSb = kRqOffThr + 2 * 128 * 8;   // [2][128] u8 scale byte of a block's largest magnitude
constexpr int kRqOffTab = kRqOffSb + 2 * 128;       // [2][128] of 32 B: the block entry of each largest magnitude
constexpr int kRqSmem = kRqOffTab + 2 * 128 * 32;

// A block's entry, indexed by its largest magnitude m: the seven thresholds
// of its scale byte sb[m], each repeated in the four bytes of a word, then
// sb[m] in byte 0 and the sign mask (0x80, or 0 when den is 0: every code 0)
// in byte 1 of the last word.  When den is 0 the thresholds are all 128.
struct RqEntry {
  uint4 a, b;  // a = T1..T4, b = T5, T6, T7, meta
};

// Codes of one 16-byte E4M3 block: the scale byte, and X[q] = the codes of
// values 4q..4q+3 in the low nibbles of bytes 0..3.  Four values at a time:
// with a = byte | 0x80 in each byte lane, a - T_k (T_k <= 0x80, so no lane
// borrows from the next) has bit 7 set exactly when e >= T_k.  The seven
// flags are monotone in k, so the magnitude code's bits are f4 (bit 2),
// f2 ^ f4 ^ f6 (bit 1) and f1 ^ ... ^ f7 (bit 0).  The largest magnitude is
// the byte maximum of the four a words (bit 7 set in all of them).
__device__ __forceinline__ void requant_codes(const uint4 w, const RqEntry *tab, uint32_t &sbyte, uint32_t X[4]) {
  const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
  uint32_t a[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) a[q] = ww[q] | 0x80808080u;
  uint32_t mx = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t ev = ww[q] & 0x007F007Fu, od = (ww[q] >> 8) & 0x007F007Fu, t;
    asm("max.u16x2 %0, %1, %2;" : "=r"(t) : "r"(ev), "r"(od));
    asm("max.u16x2 %0, %1, %2;" : "=r"(mx) : "r"(mx), "r"(t));
  }
  const uint32_t m4 = max(mx & 0xFFFFu, mx >> 16);
  const RqEntry e = tab[m4];
  sbyte = e.b.w & 0xFFu;
  const uint32_t smask = __byte_perm(e.b.w, 0, 0x1111);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t f1 = a[q] - e.a.x, f2 = a[q] - e.a.y, f3 = a[q] - e.a.z, f4 = a[q] - e.a.w, f5 = a[q] - e.b.x,
                   f6 = a[q] - e.b.y, f7 = a[q] - e.b.z;
    const uint32_t b0 = f1 ^ f2 ^ f3 ^ f4 ^ f5 ^ f6 ^ f7, b1 = f2 ^ f4 ^ f6;
    X[q] = ((ww[q] & smask) >> 4) | ((f4 >> 5) & 0x04040404u) | ((b1 >> 6) & 0x02020202u) | ((b0 >> 7) & 0x01010101u);
  }
}

// Four codes in the low nibbles of bytes 0..3 of x and y -> the 8 nibbles of
// one word (x's codes first, code i in nibble i).
__device__ __forceinline__ uint32_t pack8(uint32_t x, uint32_t y) {
  return __byte_perm(x | (x >> 4), y | (y >> 4), 0x6420);
}

__global__ void __launch_bounds__(kRqWarps * 32, 1)
    nvfp4_requant_kernel(const uint8_t *__restrict__ k8, const uint8_t *__restrict__ v8, int64_t num_tokens,
                         const int64_t *__restrict__ slot_mapping, const float *__restrict__ gs, CacheDev c,
                         const float *__restrict__ in_scale) {
  extern __shared__ __align__(16) uint8_t sm[];
  float *xs = reinterpret_cast<float *>(sm + kRqOffX);
  float *dens = reinterpret_cast<float *>(sm + kRqOffDen);
  uint8_t *thr = sm + kRqOffThr;
  uint8_t *sbl = sm + kRqOffSb;
  RqEntry *tab = reinterpret_cast<RqEntry *>(sm + kRqOffTab);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the thresholds hold for a positive finite input scale and a finite global
  // scale >= 0 (each comparison is false for NaN)
  const bool by_thr = in_scale[0] > 0.0f && in_scale[1] > 0.0f && in_scale[0] <= FLT_MAX && in_scale[1] <= FLT_MAX &&
                      gs[0] >= 0.0f && gs[1] >= 0.0f && gs[0] <= FLT_MAX && gs[1] <= FLT_MAX;
  // the tables of K (kind 0) and V (kind 1)
  for (int i = tid; i < 2 * 128; i += blockDim.x) {
    const int kind = i >> 7, e = i & 127;
    xs[i] = __fmul_rn(f32_from_e4m3(static_cast<uint32_t>(e)), in_scale[kind]);
    dens[i] = e < kRqScales ? __fmul_rn(f32_from_e4m3(static_cast<uint32_t>(e)), gs[kind]) : 0.0f;
  }
  __syncthreads();
  for (int i = tid; i < 2 * 128; i += blockDim.x) {
    const int kind = i >> 7;
    const float g = gs[kind];
    uint32_t sb = 0;
    if (g != 0.0f) sb = e4m3x2_from_f32(__fdiv_rn(xs[i], __fmul_rn(6.0f, g)), 0.0f) & 0xFFu;
    sbl[i] = static_cast<uint8_t>(sb);
  }
  // T_k of (kind, scale byte): the least e in [0, 127) whose magnitude code
  // is >= k, by bisection (127: none below the NaN byte, stored as 128)
  for (int i = tid; i < 2 * 128 * 8; i += blockDim.x) {
    const int kind = i >> 10, sb = (i >> 3) & 127, k = (i & 7) + 1;
    const float den = dens[kind * 128 + sb];
    int lo_e = 0, hi_e = 127;
    if (k <= 7 && den != 0.0f) {
      while (lo_e < hi_e) {
        const int mid = (lo_e + hi_e) >> 1;
        const uint32_t mag = e2m1x2_from_f32(__fdiv_rn(xs[kind * 128 + mid], den), 0.0f) & 0x7u;
        if (mag >= static_cast<uint32_t>(k)) hi_e = mid;
        else lo_e = mid + 1;
      }
    }
    thr[i] = static_cast<uint8_t>(lo_e == 127 ? 128 : lo_e);
  }
  __syncthreads();
  for (int i = tid; i < 2 * 128; i += blockDim.x) {  // the entry of each largest magnitude
    const int kind = i >> 7;
    const uint32_t sb = sbl[i];
    const bool zero = !(sb < static_cast<uint32_t>(kRqScales)) || dens[kind * 128 + sb] == 0.0f;
    uint32_t t[8];
#pragma unroll
    for (int k = 0; k < 7; ++k) t[k] = zero ? 0x80808080u : thr[(kind * 128 + sb) * 8 + k] * 0x01010101u;
    t[7] = (sb & 0xFFu) | (zero ? 0u : 0x8000u);
    tab[i].a = make_uint4(t[0], t[1], t[2], t[3]);
    tab[i].b = make_uint4(t[4], t[5], t[6], t[7]);
  }
  __syncthreads();
  const int64_t ngroups = (num_tokens + 7) / 8;
  const int64_t items = ngroups * c.Hkv;
  const int lgP = __ffs(c.P) - 1;  // page sizes are powers of two (16, 32, 64)
  const bool hk_pow2 = (c.Hkv & (c.Hkv - 1)) == 0;
  const int lgH = __ffs(c.Hkv) - 1;
  for (int64_t wid = static_cast<int64_t>(blockIdx.x) * kRqWarps + warp; wid < items;
       wid += static_cast<int64_t>(gridDim.x) * kRqWarps) {
    int h;
    int64_t t0;
    if (hk_pow2) {
      h = static_cast<int>(wid & (c.Hkv - 1));
      t0 = (wid >> lgH) * 8;
    } else if (items <= 0x7fffffff) {  // 32-bit index arithmetic when it fits
      const uint32_t w32 = static_cast<uint32_t>(wid), hk = static_cast<uint32_t>(c.Hkv);
      h = static_cast<int>(w32 % hk);
      t0 = static_cast<int64_t>(w32 / hk) * 8;
    } else {
      h = static_cast<int>(wid % c.Hkv);
      t0 = (wid / c.Hkv) * 8;
    }
    // this lane's K and V blocks, loaded before the slots are known (tokens past
    // the end are not read: such an item takes the per-value path)
    const int tk = lane >> 2, p = lane >> 3, vb = lane & 7;
    uint4 kw[2], vw[2];
    const bool full8 = t0 + 8 <= num_tokens;
    if (full8) {
#pragma unroll
      for (int j = 0; j < 2; ++j)
        kw[j] = __ldg(reinterpret_cast<const uint4 *>(k8 + ((t0 + tk) * c.Hkv + h) * kD + 16 * (2 * (lane & 3) + j)));
#pragma unroll
      for (int u = 0; u < 2; ++u)
        vw[u] = __ldg(reinterpret_cast<const uint4 *>(v8 + ((t0 + 2 * p + u) * c.Hkv + h) * kD + 16 * vb));
    }
    const int64_t sl = t0 + (lane & 7) < num_tokens ? slot_mapping[t0 + (lane & 7)] : -1;
    const int64_t s0 = __shfl_sync(0xffffffffu, sl, 0);
    const bool whole = __all_sync(0xffffffffu, full8 && s0 >= 0 && (s0 & 7) == 0 && sl == s0 + (lane & 7) &&
                                                   s0 + 7 < static_cast<int64_t>(c.num_pages) * c.P);
    if (!whole || !by_thr) {
      for (int it = lane; it < 2 * 8 * kBlocksPerRow; it += 32) {
        const int kind = it / (8 * kBlocksPerRow), tt = (it / kBlocksPerRow) % 8, blk = it % kBlocksPerRow;
        if (t0 + tt < num_tokens)
          nvfp4_write_item<uint8_t>(k8, v8, num_tokens, slot_mapping, gs, c, in_scale, kind, t0 + tt, h, blk);
      }
      continue;
    }
    uint8_t *im = sm + warp * kNvGroup;
    {  // K: token tk, blocks 2 (lane % 4) and 2 (lane % 4) + 1
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int blk = 2 * (lane & 3) + j;
        uint32_t sb, X[4];
        requant_codes(kw[j], tab, sb, X);
        *reinterpret_cast<uint2 *>(im + (blk >> 1) * 128 + tk * 16 + (blk & 1) * 8) =
            make_uint2(pack8(X[0], X[1]), pack8(X[2], X[3]));
        im[kNvKScales + tk * 8 + blk] = static_cast<uint8_t>(sb);
      }
    }
    {  // V: slots 2p and 2p + 1, block vb (slot 2p in the low nibble)
      uint32_t sb[2], X0[4], X1[4];
      requant_codes(vw[0], tab + 128, sb[0], X0);
      requant_codes(vw[1], tab + 128, sb[1], X1);
      *reinterpret_cast<uint4 *>(im + kNvVCodes + vb * 64 + p * 16) =
          make_uint4(X0[0] | (X1[0] << 4), X0[1] | (X1[1] << 4), X0[2] | (X1[2] << 4), X0[3] | (X1[3] << 4));
      im[kNvVScales + vb * 8 + 2 * p] = static_cast<uint8_t>(sb[0]);
      im[kNvVScales + vb * 8 + 2 * p + 1] = static_cast<uint8_t>(sb[1]);
    }
    __syncwarp();
    const int64_t page = s0 >> lgP;
    const int off = static_cast<int>(s0 & (c.P - 1));
    uint4 *dst =
        reinterpret_cast<uint4 *>(c.data + c.block(page, h, kNvTokBytes) + static_cast<int64_t>(off >> 3) * kNvGroup);
    const uint4 *src = reinterpret_cast<const uint4 *>(im);
    for (int i = lane; i < kNvGroup / 16; i += 32) dst[i] = src[i];
    __syncwarp();  // the image is rewritten by the warp's next item
  }
}

// ---------------------------------------------------------------------------
// FP8 E4M3 write: byte = E4M3(x / s8).
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256)
    fp8_write_kernel(const T *__restrict__ k, const T *__restrict__ v, int64_t num_tokens,
                     const int64_t *__restrict__ slot_mapping, const float *__restrict__ gs, CacheDev c) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // as in nvfp4_write_kernel
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t items = num_tokens * c.Hkv * kBlocksPerRow;
  if (gid >= items) return;
  const int kind = blockIdx.y;
  const int blk = static_cast<int>(gid % kBlocksPerRow);
  const int64_t th = gid / kBlocksPerRow;
  int h;
  int64_t t;
  if ((c.Hkv & (c.Hkv - 1)) == 0) {  // shifts for power-of-two head counts
    h = static_cast<int>(th & (c.Hkv - 1));
    t = th >> (__ffs(c.Hkv) - 1);
  } else {
    h = static_cast<int>(th % c.Hkv);
    t = th / c.Hkv;
  }
  const int64_t slot = slot_mapping[t];
  if (slot < 0) return;
  if (slot >= static_cast<int64_t>(c.num_pages) * c.P) {
    if (kind == 0 && h == 0 && blk == 0) set_err(c.err, NVKV_DEVERR_SLOT);
    return;
  }
  const int64_t page = slot >> (__ffs(c.P) - 1);
  const int off = static_cast<int>(slot & (c.P - 1));
  float x[16];
  load16((kind == 0 ? k : v) + th * kD + 16 * blk, x);
  const float s8 = gs[kind];
  uint32_t w[4] = {0, 0, 0, 0};
  if (s8 != 0.0f) {
    const float r = __frcp_rn(s8);
    const bool fast = quot_fast_ok(fabsf(r));  // bytes of fl(x / s8) from one reciprocal (exact)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (fast)
        w[j] = e4m3x2_quot(x[4 * j], x[4 * j + 1], s8, r) | (e4m3x2_quot(x[4 * j + 2], x[4 * j + 3], s8, r) << 16);
      else
        w[j] = e4m3x2_from_f32(__fdiv_rn(x[4 * j], s8), __fdiv_rn(x[4 * j + 1], s8)) |
               (e4m3x2_from_f32(__fdiv_rn(x[4 * j + 2], s8), __fdiv_rn(x[4 * j + 3], s8)) << 16);
    }
  }
  if (kind == 0) {
    *reinterpret_cast<uint4 *>(c.data + c.f8_kblock(page, h, off, blk)) = make_uint4(w[0], w[1], w[2], w[3]);
  } else {  // V: value 16 blk + 8 half + j' at byte 2 j' + off % 2 of its chunk (the partner owns the others)
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint8_t *dst = c.data + c.f8_vchunk(page, h, off, blk, half) + (off & 1);
#pragma unroll
      for (int j = 0; j < 8; ++j) dst[2 * j] = static_cast<uint8_t>(w[2 * half + (j >> 2)] >> (8 * (j & 3)));
    }
  }
}

// ---------------------------------------------------------------------------
// Element encoders (one byte per value).
// ---------------------------------------------------------------------------
__global__ void encode_e2m1_kernel(const float *__restrict__ x, int64_t n, uint8_t *__restrict__ out) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = static_cast<uint8_t>(e2m1x2_from_f32(x[i], 0.0f) & 0xFu);
}

__global__ void encode_e4m3_kernel(const float *__restrict__ x, int64_t n, uint8_t *__restrict__ out) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    out[i] = static_cast<uint8_t>(e4m3x2_from_f32(x[i], 0.0f) & 0xFFu);
}

// ---------------------------------------------------------------------------
// Chunked-extend prefix dequant: NVFP4 cache -> FP8 E4M3 workspace rows.
// Thread = (workspace row, KV head, 16-block); gridDim.y = K|V.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
    dequant_ws_kernel(const int32_t *__restrict__ block_table, int32_t max_pages,
                      const int32_t *__restrict__ seq_ids, const int32_t *__restrict__ prefix_lens,
                      const int64_t *__restrict__ cu_prefix, int32_t n, CacheDev c,
                      const float *__restrict__ ws_scale, uint8_t *__restrict__ ws_k, uint8_t *__restrict__ ws_v,
                      int64_t ws_rows) {
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= ws_rows * c.Hkv * kBlocksPerRow) return;
  const int kind = blockIdx.y;
  const int blk = static_cast<int>(gid % kBlocksPerRow);
  const int64_t rh = gid / kBlocksPerRow;
  int h;
  int64_t r;
  if ((c.Hkv & (c.Hkv - 1)) == 0) {  // shifts for power-of-two head counts (a 64-bit division is a long subroutine)
    h = static_cast<int>(rh & (c.Hkv - 1));
    r = rh >> (__ffs(c.Hkv) - 1);
  } else {
    h = static_cast<int>(rh % c.Hkv);
    r = rh / c.Hkv;
  }
  const int64_t total = cu_prefix[n];
  if (r == 0 && h == 0 && blk == 0 && kind == 0 && total > ws_rows) set_err(c.err, NVKV_DEVERR_WS_ROWS);
  if (r >= total) return;
  int lo = 0, hi = n - 1;  // sequence owning row r: the last i with cu_prefix[i] <= r
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu_prefix[mid] <= r) lo = mid;
    else hi = mid - 1;
  }
  const int64_t t = r - cu_prefix[lo];
  if (t >= prefix_lens[lo]) return;
  const int lgP = __ffs(c.P) - 1;  // page sizes are powers of two (16, 32, 64)
  if ((t >> lgP) >= max_pages) {  // prefix longer than its block-table row
    set_err(c.err, NVKV_DEVERR_SEQLEN);
    return;
  }
  const int64_t page = block_table[static_cast<int64_t>(seq_ids[lo]) * max_pages + (t >> lgP)];
  if (page < 0 || page >= c.num_pages) {
    set_err(c.err, NVKV_DEVERR_PAGE);
    return;
  }
  const int off = static_cast<int>(t & (c.P - 1));
  uint2 cw;
  if (kind == 0) {
    cw = *reinterpret_cast<const uint2 *>(c.data + c.nv_kcodes(page, h, off, blk));
  } else {  // V: this slot's nibbles of the pair's 16 bytes, back to two codes per byte
    const uint4 pw = *reinterpret_cast<const uint4 *>(c.data + c.nv_vcodes(page, h, off, blk));
    const uint32_t ww[4] = {pw.x, pw.y, pw.z, pw.w};
    uint32_t packed[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t n = (ww[q] >> (4 * (off & 1))) & 0x0F0F0F0Fu;  // code 4q + i in byte i
      packed[q] = (n & 0xFu) | ((n >> 4) & 0xF0u) | ((n >> 8) & 0xF00u) | ((n >> 12) & 0xF000u);
    }
    cw = make_uint2(packed[0] | (packed[1] << 16), packed[2] | (packed[3] << 16));
  }
  const float S = f32_from_e4m3(c.data[c.nv_scale(page, h, kind, off, blk)]);
  const float ratio = __fdiv_rn(c.scale[kind], ws_scale[kind]);
  const uint32_t words[2] = {cw.x, cw.y};
  uint32_t out[4];
#pragma unroll
  for (int wi = 0; wi < 2; ++wi) {
    // bytes 0,1 -> values d..d+3; bytes 2,3 -> d+4..d+7
    const uint32_t h0 = f16x2_from_e2m1x2<0>(words[wi]), h1 = f16x2_from_e2m1x2<1>(words[wi]);
    const uint32_t h2 = f16x2_from_e2m1x2<2>(words[wi]), h3 = f16x2_from_e2m1x2<3>(words[wi]);
    const float e[8] = {f32_lo(h0), f32_hi(h0), f32_lo(h1), f32_hi(h1), f32_lo(h2), f32_hi(h2), f32_lo(h3), f32_hi(h3)};
    float y[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) y[q] = __fmul_rn(__fmul_rn(e[q], S), ratio);
    out[2 * wi] = e4m3x2_from_f32(y[0], y[1]) | (e4m3x2_from_f32(y[2], y[3]) << 16);
    out[2 * wi + 1] = e4m3x2_from_f32(y[4], y[5]) | (e4m3x2_from_f32(y[6], y[7]) << 16);
  }
  uint8_t *dst = (kind == 0 ? ws_k : ws_v) + (r * c.Hkv + h) * kD + 16 * blk;
  *reinterpret_cast<uint4 *>(dst) = make_uint4(out[0], out[1], out[2], out[3]);
}

// Launch with programmatic dependent launch (the kernel starts with
// griddepcontrol.wait); an ordinary launch where that is refused.
template <typename... KArgs, typename... Args>
void launch_pdl(void (*kernel)(KArgs...), dim3 grid, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...) != cudaSuccess) {
    cudaGetLastError();
    kernel<<<grid, 256, 0, s>>>(static_cast<KArgs>(args)...);
  }
}

// As launch_pdl, with a block size and dynamic shared memory of the caller's.
template <typename... KArgs, typename... Args>
void launch_pdl_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...) != cudaSuccess) {
    cudaGetLastError();
    kernel<<<grid, block, smem, s>>>(static_cast<KArgs>(args)...);
  }
}

inline int grid_for(int64_t items, int threads) {
  const int64_t b = (items + threads - 1) / threads;
  return static_cast<int>(b < 1 ? 1 : b);
}

int amax_grid(int64_t n) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 1;
  const int64_t want = (n / 16 + 255) / 256;
  return static_cast<int>(want < 1 ? 1 : (want > 4L * sms ? 4L * sms : want));
}

nvkv_status launch_amax(const void *x, nvkv_dtype dtype, int64_t n, float *acc, cudaStream_t s) {
  const int grid = amax_grid(n);
  const bool vec = aligned16(x);
  if (dtype == NVKV_DTYPE_F32)
    amax_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float *>(x), n, vec,
                                             reinterpret_cast<uint32_t *>(acc));
  else
    amax_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(x), n, vec,
                                                     reinterpret_cast<uint32_t *>(acc));
  return launch_status();
}

nvkv_status write_common(const void *k, const void *v, nvkv_dtype dtype, int64_t num_tokens,
                         const int64_t *slot_mapping, const float *global_scale, const nvkv_cache *cache,
                         void *stream, int prec) {
  nvkv_status st = check_cache(cache, prec);
  if (st != NVKV_OK) return st;
  if (num_tokens < 0) return NVKV_ERR_INVALID_ARG;
  if (dtype != NVKV_DTYPE_F32 && dtype != NVKV_DTYPE_BF16) return NVKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return NVKV_OK;
  if (!k || !v || !slot_mapping) return NVKV_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v)) return NVKV_ERR_UNSUPPORTED;
  const float *gs = global_scale ? global_scale : cache->kv_scale;
  CacheDev c = to_dev(cache);
  const int64_t items = num_tokens * cache->num_kv_heads * kBlocksPerRow;
  dim3 grid(grid_for(items, 256), 2);
  // NVFP4: one warp per (8 tokens, KV head)
  const dim3 ngrid(grid_for((num_tokens + 7) / 8 * cache->num_kv_heads, kWriteWarps));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (prec == NVKV_PREC_NVFP4) {
    if (dtype == NVKV_DTYPE_F32)
      launch_pdl(nvfp4_write_kernel<float>, ngrid, s, static_cast<const float *>(k), static_cast<const float *>(v),
                 num_tokens, slot_mapping, gs, c, static_cast<const float *>(nullptr));
    else
      launch_pdl(nvfp4_write_kernel<__nv_bfloat16>, ngrid, s, static_cast<const __nv_bfloat16 *>(k),
                 static_cast<const __nv_bfloat16 *>(v), num_tokens, slot_mapping, gs, c,
                 static_cast<const float *>(nullptr));
  } else {
    if (dtype == NVKV_DTYPE_F32)
      launch_pdl(fp8_write_kernel<float>, grid, s, static_cast<const float *>(k), static_cast<const float *>(v),
                 num_tokens, slot_mapping, gs, c);
    else
      launch_pdl(fp8_write_kernel<__nv_bfloat16>, grid, s, static_cast<const __nv_bfloat16 *>(k),
                 static_cast<const __nv_bfloat16 *>(v), num_tokens, slot_mapping, gs, c);
  }
  return launch_status();
}

}  // namespace
}  // namespace nvkv

using namespace nvkv;

extern "C" {

const char *nvkv_status_string(nvkv_status s) {
  switch (s) {
    case NVKV_OK: return "ok";
    case NVKV_ERR_INVALID_ARG: return "invalid argument";
    case NVKV_ERR_UNSUPPORTED: return "unsupported configuration";
    case NVKV_ERR_CUDA: return "CUDA launch error";
    case NVKV_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
  }
  return "unknown status";
}

nvkv_status nvkv_global_scale(const void *x, nvkv_dtype dtype, int64_t n, float divisor, float *out,
                              void *stream) {
  NVKV_ABI_RANGE();
  if (!out || n < 0 || (n > 0 && !x) || !(divisor > 0.0f)) return NVKV_ERR_INVALID_ARG;
  if (dtype != NVKV_DTYPE_F32 && dtype != NVKV_DTYPE_BF16) return NVKV_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(out, 0, sizeof(float), s) != cudaSuccess) return NVKV_ERR_CUDA;
  if (n > 0) {
    nvkv_status st = launch_amax(x, dtype, n, out, s);
    if (st != NVKV_OK) return st;
  }
  divide_kernel<<<1, 1, 0, s>>>(out, divisor);
  return launch_status();
}

nvkv_status nvkv_amax_update(const void *x, nvkv_dtype dtype, int64_t n, float *amax, void *stream) {
  NVKV_ABI_RANGE();
  if (!amax || n < 0 || (n > 0 && !x)) return NVKV_ERR_INVALID_ARG;
  if (dtype != NVKV_DTYPE_F32 && dtype != NVKV_DTYPE_BF16) return NVKV_ERR_INVALID_ARG;
  if (n == 0) return NVKV_OK;
  return launch_amax(x, dtype, n, amax, static_cast<cudaStream_t>(stream));
}

nvkv_status nvfp4_kv_quantize_write(const void *k, const void *v, nvkv_dtype dtype, int64_t num_tokens,
                                    const int64_t *slot_mapping, const float *global_scale,
                                    const nvkv_cache *cache, void *stream) {
  NVKV_ABI_RANGE();
  return write_common(k, v, dtype, num_tokens, slot_mapping, global_scale, cache, stream, NVKV_PREC_NVFP4);
}

nvkv_status fp8_kv_quantize_write(const void *k, const void *v, nvkv_dtype dtype, int64_t num_tokens,
                                  const int64_t *slot_mapping, const float *global_scale, const nvkv_cache *cache,
                                  void *stream) {
  NVKV_ABI_RANGE();
  return write_common(k, v, dtype, num_tokens, slot_mapping, global_scale, cache, stream, NVKV_PREC_FP8_E4M3);
}

nvkv_status nvfp4_kv_requantize_write_fp8(const uint8_t *k8, const uint8_t *v8, const float *in_scale,
                                          int64_t num_tokens, const int64_t *slot_mapping, const float *global_scale,
                                          const nvkv_cache *cache, void *stream) {
  NVKV_ABI_RANGE();
  nvkv_status st = check_cache(cache, NVKV_PREC_NVFP4);
  if (st != NVKV_OK) return st;
  if (num_tokens < 0) return NVKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return NVKV_OK;
  if (!k8 || !v8 || !in_scale || !slot_mapping) return NVKV_ERR_INVALID_ARG;
  if (!aligned16(k8) || !aligned16(v8)) return NVKV_ERR_UNSUPPORTED;
  const float *gs = global_scale ? global_scale : cache->kv_scale;
  // a persistent grid of one 32-warp CTA per SM (each builds the tables once), at most one warp per item
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 1;
  static std::once_flag attr_once;
  std::call_once(attr_once, [] {
    cudaFuncSetAttribute(nvfp4_requant_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRqSmem);
  });
  const int64_t items = (num_tokens + 7) / 8 * cache->num_kv_heads;
  const int64_t ctas = (items + kRqWarps - 1) / kRqWarps;
  const dim3 grid(static_cast<unsigned>(ctas < sms ? ctas : sms));
  launch_pdl_ex(nvfp4_requant_kernel, grid, dim3(kRqWarps * 32), kRqSmem, static_cast<cudaStream_t>(stream), k8, v8,
                num_tokens, slot_mapping, gs, to_dev(cache), in_scale);
  return launch_status();
}

nvkv_status nvkv_encode_e2m1(const float *x, int64_t n, uint8_t *out, void *stream) {
  NVKV_ABI_RANGE();
  if (n < 0 || (n > 0 && (!x || !out))) return NVKV_ERR_INVALID_ARG;
  if (n == 0) return NVKV_OK;
  const int64_t b = (n + 255) / 256;
  encode_e2m1_kernel<<<static_cast<int>(b > 65536 ? 65536 : b), 256, 0, static_cast<cudaStream_t>(stream)>>>(x, n,
                                                                                                          out);
  return launch_status();
}

nvkv_status nvkv_encode_e4m3(const float *x, int64_t n, uint8_t *out, void *stream) {
  NVKV_ABI_RANGE();
  if (n < 0 || (n > 0 && (!x || !out))) return NVKV_ERR_INVALID_ARG;
  if (n == 0) return NVKV_OK;
  const int64_t b = (n + 255) / 256;
  encode_e4m3_kernel<<<static_cast<int>(b > 65536 ? 65536 : b), 256, 0, static_cast<cudaStream_t>(stream)>>>(x, n,
                                                                                                          out);
  return launch_status();
}

nvkv_status nvfp4_kv_dequant_to_fp8_workspace(const int32_t *block_table, int32_t max_pages,
                                              const int32_t *seq_ids, const int32_t *prefix_lens,
                                              const int64_t *cu_prefix, int32_t n, const nvkv_cache *cache,
                                              const float *ws_scale, uint8_t *ws_k, uint8_t *ws_v,
                                              int64_t ws_rows, void *stream) {
  NVKV_ABI_RANGE();
  nvkv_status st = check_cache(cache, NVKV_PREC_NVFP4);
  if (st != NVKV_OK) return st;
  if (n < 0 || ws_rows < 0 || max_pages <= 0) return NVKV_ERR_INVALID_ARG;
  if (n == 0 || ws_rows == 0) return NVKV_OK;
  if (!block_table || !seq_ids || !prefix_lens || !cu_prefix || !ws_scale || !ws_k || !ws_v)
    return NVKV_ERR_INVALID_ARG;
  if (!aligned16(ws_k) || !aligned16(ws_v)) return NVKV_ERR_UNSUPPORTED;
  CacheDev c = to_dev(cache);
  const int64_t items = ws_rows * cache->num_kv_heads * kBlocksPerRow;
  dim3 grid(grid_for(items, 256), 2);
  dequant_ws_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      block_table, max_pages, seq_ids, prefix_lens, cu_prefix, n, c, ws_scale, ws_k, ws_v, ws_rows);
  return launch_status();
}

}  // extern "C"
