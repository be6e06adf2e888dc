// Paged GQA decode attention reading the NVFP4 (or FP8 E4M3) cache straight
// from HBM ("SGLang x Qwen x NVIDIA ...", Three Paths: decode is memory-bound,
// so the kernel reads NVFP4 directly and dequantizes on the fly; it must read
// exactly as much as it computes).  The per-layer FP8 variant serves the
// sensitive layers ("SOAR Weekly Champion Notes 05", 03).
//
// Design (sm_103a, one GPU):
//   * Work unit = one 64-token tile of one (sequence, KV head).  The units of
//     the whole batch are laid end to end and cut into equal contiguous shares,
//     one per CTA of a persistent grid (about SMs x resident CTAs), so every
//     CTA streams the same number of bytes whatever the sequence lengths.  A
//     (sequence, KV head) cut between CTAs yields split-KV partials that the
//     last-arriving CTA merges with the log-sum-exp rule (no second kernel,
//     no spin: an atomic arrival counter).
//   * One producer warp streams tiles into a shared-memory ring with 1-D bulk
//     copies (cp.async.bulk + mbarrier transaction counts).  The cache keeps
//     each (page, KV head) as one contiguous block, so a 64-token tile is one
//     9216-byte copy at page size 64 (NVFP4; 16 KB for FP8), or 64/P copies of
//     whole page blocks.  Block-table entries are fetched 32 at a time, one
//     window ahead.  An L2 evict-first hint marks the stream.
//   * Four consumer warps share every tile: warp w takes tokens [16w, 16w+16),
//     copies its slice into registers and releases the stage at once, so the
//     ring stays almost entirely in flight while the warps compute.
//   * E2M1 pairs become f16x2 with one cvt.rn.f16x2.e2m1x2 and are scaled by
//     their E4M3 block scale with one f16x2 multiply; code * scale has at most
//     6 significant bits and lies in [2^-10, 2688], so it is exact in FP16.
//     Scores and P.V run on the tensor cores as m16n8k16 FP16 MMAs with FP32
//     accumulation: tokens form M, the GQA query group (<= 8 heads) forms N.
//     g_K, sm_scale, log2(e) and a per-head power of two that brings the BF16
//     query into FP16 range form one FP32 factor per score; g_V is applied
//     once to the output.  Online softmax in FP32 with exp2 and a lazily raised
//     running max (rescale only when the max grows by more than 2^8).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "nvkv_device.cuh"
#include "nvkv_host.h"

namespace nvkv {
namespace {

constexpr int kD = 128;
constexpr int kTile = 64;          // tokens per work unit / ring stage
constexpr int kSub = 16;           // tokens per consumer warp per stage
constexpr int kConsumerWarps = kTile / kSub;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxBatch = 1024;    // sequences per call (prefix sums live in shared memory)
constexpr int kMaxGroup = 8;       // query heads per KV head (MMA N)
constexpr int kSlotFloats = kMaxGroup * kD + 2 * kMaxGroup;  // one partial (o, m, l)
constexpr float kRescaleThreshold = 8.0f;                   // log2 units

template <int PREC>
struct Layout;
template <>
struct Layout<NVKV_PREC_NVFP4> {
  static constexpr int kTokBytes = kNvTokBytes;                // 144
  static constexpr int kStageBytes = kTile * kTokBytes;        // 9216
  static constexpr int kStages = 6;
  static constexpr int kMinBlocks = 3;
};
template <>
struct Layout<NVKV_PREC_FP8_E4M3> {
  static constexpr int kTokBytes = kF8TokBytes;                // 256
  static constexpr int kStageBytes = kTile * kTokBytes;        // 16384
  static constexpr int kStages = 6;
  static constexpr int kMinBlocks = 2;
};

struct DecodeArgs {
  const __nv_bfloat16 *q;
  CacheDev c;
  const int32_t *block_table;
  const int32_t *seq_lens;
  int32_t max_pages;
  int32_t B, Hq, G;
  float sm_scale;
  int32_t num_ctas;
  int32_t *meta;      // written by CTA 0: cum[0..B] (tiles before each sequence), then NC
  float *partials;    // [num_ctas][2][kSlotFloats]
  __nv_bfloat16 *out;
};

template <int PREC>
constexpr int smem_bytes_for(int G) {
  return Layout<PREC>::kStages * Layout<PREC>::kStageBytes  // ring
         + 2 * Layout<PREC>::kStages * 8                       // full/empty barriers
         + (kMaxBatch + 1) * 4                                 // tile prefix sums
         + kConsumerWarps * G * kD * 4                         // warp merge: o
         + kConsumerWarps * kMaxGroup * 2 * 4                  // warp merge: m, l
         + 4 * (1 + Layout<PREC>::kStages);                    // abort, fills
}

// Segment = run of consecutive units of one (sequence, KV head).
struct Seg {
  int b, h, t0, t1;  // tiles [t0, t1) of (b, h)
};

// cum[b] = tiles of sequences before b; units before sequence b = Hkv * cum[b].
__device__ __forceinline__ Seg seg_at(int64_t u, int64_t u_end, const int32_t *cum, int B, int Hkv) {
  int lo = 0, hi = B - 1;  // last b with Hkv*cum[b] <= u (sequences without tiles are skipped)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(cum[mid]) * Hkv <= u) lo = mid;
    else hi = mid - 1;
  }
  const int nb = cum[lo + 1] - cum[lo];
  const int64_t r = u - static_cast<int64_t>(cum[lo]) * Hkv;
  Seg s;
  s.b = lo;
  s.h = static_cast<int>(r / nb);
  s.t0 = static_cast<int>(r % nb);
  const int64_t left = u_end - u;
  s.t1 = static_cast<int>(left < nb - s.t0 ? s.t0 + left : nb);
  return s;
}

// Shares: CTA c owns units [floor(c W / NC), floor((c+1) W / NC)); with W >= NC
// every share is non-empty.  owner_of(u) = the CTA whose share holds unit u.
__device__ __forceinline__ int64_t share_begin(int64_t c, int64_t W, int64_t NC) { return c * W / NC; }
__device__ __forceinline__ int64_t owner_of(int64_t u, int64_t W, int64_t NC) {
  return ((u + 1) * NC + W - 1) / W - 1;
}

__device__ __forceinline__ int clamped_len(const DecodeArgs &a, int b) {
  const int64_t cap = static_cast<int64_t>(a.max_pages) * a.c.P;
  const int64_t L = a.seq_lens[b];
  return static_cast<int>(L < 0 ? 0 : (L > cap ? cap : L));
}

// ---------------------------------------------------------------------------
// Producer warp: one bulk copy per page block of each tile of this CTA's
// share (a tile spans 64 / P whole page blocks).  Lane j copies block j.
// ---------------------------------------------------------------------------
template <int PREC>
__device__ void producer(const DecodeArgs &a, uint8_t *ring, uint64_t *full, uint64_t *empty, const int32_t *cum,
                         int64_t u0, int64_t u1, volatile int *abort, int *fills) {
  using Lay = Layout<PREC>;
  const int lane = threadIdx.x & 31;
  const int Hkv = a.c.Hkv, P = a.c.P;
  const uint64_t policy = policy_evict_first();
  const uint32_t block_bytes = static_cast<uint32_t>(P) * Lay::kTokBytes;
  int64_t i = 0;  // stage counter
  for (int64_t u = u0; u < u1;) {
    const Seg s = seg_at(u, u1, cum, a.B, Hkv);
    const int len = clamped_len(a, s.b);
    const int32_t *brow = a.block_table + static_cast<int64_t>(s.b) * a.max_pages;
    // Block-table window: lane l holds the entry of page index wbase + l; the
    // next window is requested when the current one comes into use.
    int wbase = (s.t0 * kTile) / P;
    int32_t pg = wbase + lane < a.max_pages ? brow[wbase + lane] : 0;
    int32_t pg_next = wbase + 32 + lane < a.max_pages ? brow[wbase + 32 + lane] : 0;
    for (int t = s.t0; t < s.t1; ++t, ++i) {
      const int slot = static_cast<int>(i % Lay::kStages);
      const uint32_t fill = static_cast<uint32_t>(i / Lay::kStages);
      if (__any_sync(0xffffffffu, *abort)) return;
      if (lane == 0 && fill > 0) mbar_wait_bounded(&empty[slot], (fill - 1) & 1u, abort);
      if (__any_sync(0xffffffffu, *abort)) return;  // warp-uniform exit
      const int tok0 = t * kTile;
      const int ntok = min(kTile, len - tok0);
      const int nblk = (ntok + P - 1) / P;  // page blocks holding the tile's tokens
      if ((tok0 + ntok - 1) / P >= wbase + 32) {  // the tile leaves the window (warp-uniform)
        wbase += 32;
        pg = pg_next;
        pg_next = wbase + 32 + lane < a.max_pages ? brow[wbase + 32 + lane] : 0;
      }
      if (lane == 0) mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(nblk) * block_bytes);
      const int pidx = lane < nblk ? tok0 / P + lane - wbase : 0;
      const int64_t page_w = __shfl_sync(0xffffffffu, pg, pidx & 31);
      if (lane < nblk) {
        int64_t page = page_w;
        if (page < 0 || page >= a.c.num_pages) {
          set_err(a.c.err, NVKV_DEVERR_PAGE);
          page = 0;  // a valid address; the output of this sequence is then undefined
        }
        bulk_g2s(ring + static_cast<size_t>(slot) * Lay::kStageBytes + static_cast<size_t>(lane) * block_bytes,
                 a.c.data + a.c.block(page, s.h, Lay::kTokBytes), block_bytes, &full[slot], policy);
      }
      if (lane == 0) fills[slot] = static_cast<int>(fill) + 1;
    }
    u += s.t1 - s.t0;
  }
}

// ---------------------------------------------------------------------------
// Consumer warps.  Lane = 4r + c.  Warp w owns tokens [16w, 16w+16) of every
// stage.  Scores: MMA rows = tokens r, r + 8 of the slice; head_dim order
// inside one MMA k-step s is permuted so that a thread reads 16 contiguous code
// bytes (d in [32c, 32c+32), step s covers d = 32c + 4s + {0,1,2,3}); the
// query fragment uses the same order.  P.V: MMA rows = head_dim (thread r owns
// d in [16r, 16r+16)), k = tokens 2c, 2c+1, 2c+8, 2c+9, n = query head.  O for
// heads 2c, 2c+1 of the group and d in [16r, 16r+16) lives in 32 registers.
//
// The warp runs its slices as a two-deep software pipeline: while the P.V
// MMAs of slice i issue, the score MMAs of slice i+1 issue between them (the
// two chains are independent), and the softmax of slice i+1 follows.  K of a
// slice is read from shared memory when its scores start, V when its P.V
// starts; the stage is released after both.
// ---------------------------------------------------------------------------
struct WarpState {
  float o[8][4];
  float m[2];
  float l[2];
};

// Offsets of a warp's slice inside a stage (block layout of the header).
template <int PREC>
struct SliceOffsets {
  int kc, ks, vc, vs;  // row 0 of K codes, K scales, V codes, V scales (NVFP4); kc, vc for FP8
  __device__ SliceOffsets(int warp, int P) {
    const int blk = (kSub * warp) / P, row0 = (kSub * warp) % P;
    const int base = blk * P * Layout<PREC>::kTokBytes;
    if constexpr (PREC == NVKV_PREC_NVFP4) {
      kc = base + row0 * kNvCodeRow;
      ks = base + P * kNvCodeRow + row0 * kNvScaleRow;
      vc = base + P * (kNvCodeRow + kNvScaleRow) + row0 * kNvCodeRow;
      vs = base + P * (2 * kNvCodeRow + kNvScaleRow) + row0 * kNvScaleRow;
    } else {
      kc = base + row0 * kF8Row;
      vc = base + P * kF8Row + row0 * kF8Row;
      ks = vs = 0;
    }
  }
};

// K operand of a slice: code words of rows r, r + 8 and (NVFP4) their block
// scales as f16x2 pairs {S, S} for d blocks 2c (lo) and 2c + 1 (hi).
template <int PREC>
struct KOps {
  uint32_t k0[PREC == NVKV_PREC_NVFP4 ? 4 : 8], k1[PREC == NVKV_PREC_NVFP4 ? 4 : 8];
  uint32_t lo0, hi0, lo1, hi1;
};

// V operand of a slice.  NVFP4: per 8-byte half w, the e2m1 pairs of tokens
// (2c, 2c+1) at d and d + 1 (x, y) and of tokens (2c+8, 2c+9) (z, t), and the
// f16x2 block scales of those token pairs; masked tokens carry scale 0.  FP8:
// the raw code words of tokens 2c, 2c+1, 2c+8, 2c+9, masked tokens zeroed.
template <int PREC>
struct VOps {
  uint32_t w[PREC == NVKV_PREC_NVFP4 ? 2 : 4][4];
  uint32_t sAB, sCD;
};

template <int PREC>
__device__ __forceinline__ void load_k(const uint8_t *stage, const SliceOffsets<PREC> &o, int r, int c,
                                       KOps<PREC> &x) {
  if constexpr (PREC == NVKV_PREC_NVFP4) {
    const uint4 a = *reinterpret_cast<const uint4 *>(stage + o.kc + r * kNvCodeRow + 16 * c);
    const uint4 b = *reinterpret_cast<const uint4 *>(stage + o.kc + (r + 8) * kNvCodeRow + 16 * c);
    x.k0[0] = a.x; x.k0[1] = a.y; x.k0[2] = a.z; x.k0[3] = a.w;
    x.k1[0] = b.x; x.k1[1] = b.y; x.k1[2] = b.z; x.k1[3] = b.w;
    const uint32_t s0 = *reinterpret_cast<const uint16_t *>(stage + o.ks + r * kNvScaleRow + 2 * c);
    const uint32_t s1 = *reinterpret_cast<const uint16_t *>(stage + o.ks + (r + 8) * kNvScaleRow + 2 * c);
    const uint32_t h0 = f16x2_from_e4m3x2<0>(s0), h1 = f16x2_from_e4m3x2<0>(s1);
    x.lo0 = prmt(h0, 0, 0x1010);  // {S_2c, S_2c}
    x.hi0 = prmt(h0, 0, 0x3232);  // {S_2c+1, S_2c+1}
    x.lo1 = prmt(h1, 0, 0x1010);
    x.hi1 = prmt(h1, 0, 0x3232);
  } else {
    const uint4 *p0 = reinterpret_cast<const uint4 *>(stage + o.kc + r * kF8Row + 32 * c);
    const uint4 *p1 = reinterpret_cast<const uint4 *>(stage + o.kc + (r + 8) * kF8Row + 32 * c);
    const uint4 a0 = p0[0], a1 = p0[1], b0 = p1[0], b1 = p1[1];
    x.k0[0] = a0.x; x.k0[1] = a0.y; x.k0[2] = a0.z; x.k0[3] = a0.w;
    x.k0[4] = a1.x; x.k0[5] = a1.y; x.k0[6] = a1.z; x.k0[7] = a1.w;
    x.k1[0] = b0.x; x.k1[1] = b0.y; x.k1[2] = b0.z; x.k1[3] = b0.w;
    x.k1[4] = b1.x; x.k1[5] = b1.y; x.k1[6] = b1.z; x.k1[7] = b1.w;
    x.lo0 = x.hi0 = x.lo1 = x.hi1 = 0;
  }
}

// nvalid = valid tokens of the slice (0..16): tokens past it are masked.
template <int PREC>
__device__ __forceinline__ void load_v(const uint8_t *stage, const SliceOffsets<PREC> &o, int r, int c, int nvalid,
                                       VOps<PREC> &x) {
  const int tA = 2 * c;
  if constexpr (PREC == NVKV_PREC_NVFP4) {
    const uint2 A = *reinterpret_cast<const uint2 *>(stage + o.vc + tA * kNvCodeRow + 8 * r);
    const uint2 B = *reinterpret_cast<const uint2 *>(stage + o.vc + (tA + 1) * kNvCodeRow + 8 * r);
    const uint2 C = *reinterpret_cast<const uint2 *>(stage + o.vc + (tA + 8) * kNvCodeRow + 8 * r);
    const uint2 D = *reinterpret_cast<const uint2 *>(stage + o.vc + (tA + 9) * kNvCodeRow + 8 * r);
    const uint8_t *vs = stage + o.vs + r;
    uint32_t sv = static_cast<uint32_t>(vs[tA * kNvScaleRow]) | (static_cast<uint32_t>(vs[(tA + 1) * kNvScaleRow]) << 8) |
                  (static_cast<uint32_t>(vs[(tA + 8) * kNvScaleRow]) << 16) |
                  (static_cast<uint32_t>(vs[(tA + 9) * kNvScaleRow]) << 24);
    if (nvalid < kSub) {  // masked tokens get scale 0 -> value 0 (codes are finite)
      if (tA >= nvalid) sv &= 0xFFFFFF00u;
      if (tA + 1 >= nvalid) sv &= 0xFFFF00FFu;
      if (tA + 8 >= nvalid) sv &= 0xFF00FFFFu;
      if (tA + 9 >= nvalid) sv &= 0x00FFFFFFu;
    }
    x.sAB = f16x2_from_e4m3x2<0>(sv);
    x.sCD = f16x2_from_e4m3x2<1>(sv);
    const uint32_t a[2] = {A.x, A.y}, b[2] = {B.x, B.y}, cc[2] = {C.x, C.y}, dd[2] = {D.x, D.y};
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      // byte j: the token pair's low nibbles (d = 16r + 2j') or high nibbles (d + 1)
      x.w[w][0] = (a[w] & 0x0F0F0F0Fu) | ((b[w] & 0x0F0F0F0Fu) << 4);
      x.w[w][1] = ((a[w] >> 4) & 0x0F0F0F0Fu) | (b[w] & 0xF0F0F0F0u);
      x.w[w][2] = (cc[w] & 0x0F0F0F0Fu) | ((dd[w] & 0x0F0F0F0Fu) << 4);
      x.w[w][3] = ((cc[w] >> 4) & 0x0F0F0F0Fu) | (dd[w] & 0xF0F0F0F0u);
    }
  } else {
    const uint4 A = *reinterpret_cast<const uint4 *>(stage + o.vc + tA * kF8Row + 16 * r);
    const uint4 B = *reinterpret_cast<const uint4 *>(stage + o.vc + (tA + 1) * kF8Row + 16 * r);
    const uint4 C = *reinterpret_cast<const uint4 *>(stage + o.vc + (tA + 8) * kF8Row + 16 * r);
    const uint4 D = *reinterpret_cast<const uint4 *>(stage + o.vc + (tA + 9) * kF8Row + 16 * r);
    x.w[0][0] = A.x; x.w[1][0] = A.y; x.w[2][0] = A.z; x.w[3][0] = A.w;
    x.w[0][1] = B.x; x.w[1][1] = B.y; x.w[2][1] = B.z; x.w[3][1] = B.w;
    x.w[0][2] = C.x; x.w[1][2] = C.y; x.w[2][2] = C.z; x.w[3][2] = C.w;
    x.w[0][3] = D.x; x.w[1][3] = D.y; x.w[2][3] = D.z; x.w[3][3] = D.w;
    if (nvalid < kSub) {  // masked tokens -> E4M3 zero (stale bytes could be NaN)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (tA >= nvalid) x.w[q][0] = 0;
        if (tA + 1 >= nvalid) x.w[q][1] = 0;
        if (tA + 8 >= nvalid) x.w[q][2] = 0;
        if (tA + 9 >= nvalid) x.w[q][3] = 0;
      }
    }
    x.sAB = x.sCD = 0;
  }
}

// Score MMA k-step S (even steps accumulate into e, odd into od).
template <int PREC, int S>
__device__ __forceinline__ void qk_step(const KOps<PREC> &x, const uint32_t (&qf)[8][2], float (&e)[4],
                                        float (&od)[4]) {
  float(&acc)[4] = (S & 1) ? od : e;
  if constexpr (PREC == NVKV_PREC_NVFP4) {
    const uint32_t m0 = S < 4 ? x.lo0 : x.hi0, m1 = S < 4 ? x.lo1 : x.hi1;
    constexpr int B0 = (S & 1) ? 2 : 0, B1 = B0 + 1;
    const uint32_t a0 = hmul2_u32(f16x2_from_e2m1x2<B0>(x.k0[S >> 1]), m0);
    const uint32_t a2 = hmul2_u32(f16x2_from_e2m1x2<B1>(x.k0[S >> 1]), m0);
    const uint32_t a1 = hmul2_u32(f16x2_from_e2m1x2<B0>(x.k1[S >> 1]), m1);
    const uint32_t a3 = hmul2_u32(f16x2_from_e2m1x2<B1>(x.k1[S >> 1]), m1);
    mma_f16_16816(acc, a0, a1, a2, a3, qf[S][0], qf[S][1]);
  } else {
    mma_f16_16816(acc, f16x2_from_e4m3x2<0>(x.k0[S]), f16x2_from_e4m3x2<0>(x.k1[S]), f16x2_from_e4m3x2<1>(x.k0[S]),
                  f16x2_from_e4m3x2<1>(x.k1[S]), qf[S][0], qf[S][1]);
  }
}

// P.V MMA for output tile J (NVFP4: half w = J / 4, byte J % 4 of each pair
// word; FP8: token-pair word J / 2, byte pair J % 2).
template <int PREC, int J>
__device__ __forceinline__ void pv_tile(const VOps<PREC> &x, uint32_t b0, uint32_t b1, WarpState &st) {
  if constexpr (PREC == NVKV_PREC_NVFP4) {
    constexpr int w = J >> 2, I = J & 3;
    mma_f16_16816(st.o[J], hmul2_u32(f16x2_from_e2m1x2<I>(x.w[w][0]), x.sAB),
                  hmul2_u32(f16x2_from_e2m1x2<I>(x.w[w][1]), x.sAB), hmul2_u32(f16x2_from_e2m1x2<I>(x.w[w][2]), x.sCD),
                  hmul2_u32(f16x2_from_e2m1x2<I>(x.w[w][3]), x.sCD), b0, b1);
  } else {
    constexpr int qd = J >> 1;
    constexpr uint32_t sel = (J & 1) ? 0x7362u : 0x5140u;
    const uint32_t ab = prmt(x.w[qd][0], x.w[qd][1], sel), cd = prmt(x.w[qd][2], x.w[qd][3], sel);
    mma_f16_16816(st.o[J], f16x2_from_e4m3x2<0>(ab), f16x2_from_e4m3x2<1>(ab), f16x2_from_e4m3x2<0>(cd),
                  f16x2_from_e4m3x2<1>(cd), b0, b1);
  }
}

// Step J of the pipeline: score k-step J of the next slice and P.V tile J of
// the current one, each only when asked for.
template <int PREC, int J, bool QK, bool PV>
__device__ __forceinline__ void pipe_step(const KOps<PREC> &kx, const uint32_t (&qf)[8][2], float (&e)[4],
                                          float (&od)[4], const VOps<PREC> &vx, uint32_t b0, uint32_t b1,
                                          WarpState &st) {
  if constexpr (QK) qk_step<PREC, J>(kx, qf, e, od);
  if constexpr (PV) pv_tile<PREC, J>(vx, b0, b1, st);
}

template <int PREC, bool QK, bool PV>
__device__ __forceinline__ void pipe_all(const KOps<PREC> &kx, const uint32_t (&qf)[8][2], float (&e)[4],
                                         float (&od)[4], const VOps<PREC> &vx, uint32_t b0, uint32_t b1,
                                         WarpState &st) {
  pipe_step<PREC, 0, QK, PV>(kx, qf, e, od, vx, b0, b1, st);
  pipe_step<PREC, 1, QK, PV>(kx, qf, e, od, vx, b0, b1, st);
  pipe_step<PREC, 2, QK, PV>(kx, qf, e, od, vx, b0, b1, st);
  pipe_step<PREC, 3, QK, PV>(kx, qf, e, od, vx, b0, b1, st);
  pipe_step<PREC, 4, QK, PV>(kx, qf, e, od, vx, b0, b1, st);
  pipe_step<PREC, 5, QK, PV>(kx, qf, e, od, vx, b0, b1, st);
  pipe_step<PREC, 6, QK, PV>(kx, qf, e, od, vx, b0, b1, st);
  pipe_step<PREC, 7, QK, PV>(kx, qf, e, od, vx, b0, b1, st);
}

// Online softmax of one slice's scores (e + od, rows r / r + 8, heads 2c,
// 2c+1, scaled by cs into log2 units; rows at or past nvalid masked): raises
// the running max only when a score exceeds it by more than the threshold
// (then O and l are rescaled), and returns P as the two f16x2 B fragments of
// the P.V MMA (zero for a slice without valid tokens): b0 = P[tok 2c, 2c+1][head r], b1 = P[tok 2c+8, 2c+9][head r].
__device__ __forceinline__ void softmax_slice(const float (&e)[4], const float (&od)[4], int nvalid, int r,
                                              const float (&cs)[2], WarpState &st, uint32_t &b0, uint32_t &b1) {
  if (nvalid <= 0) {  // warp-uniform: a slice past the end of the sequence adds nothing
    b0 = b1 = 0;
    return;
  }
  const bool v0 = r < nvalid, v1 = r + 8 < nvalid;
  const float s0 = v0 ? (e[0] + od[0]) * cs[0] : -INFINITY;
  const float s1 = v0 ? (e[1] + od[1]) * cs[1] : -INFINITY;
  const float s2 = v1 ? (e[2] + od[2]) * cs[0] : -INFINITY;
  const float s3 = v1 ? (e[3] + od[3]) * cs[1] : -INFINITY;
  const bool need = (s0 > st.m[0] + kRescaleThreshold) | (s2 > st.m[0] + kRescaleThreshold) |
                    (s1 > st.m[1] + kRescaleThreshold) | (s3 > st.m[1] + kRescaleThreshold);
  if (__any_sync(0xffffffffu, need)) {
    float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    const float n0 = fmaxf(st.m[0], mx0), n1 = fmaxf(st.m[1], mx1);
    const float al0 = ex2(st.m[0] - n0), al1 = ex2(st.m[1] - n1);
    st.m[0] = n0;
    st.m[1] = n1;
    st.l[0] *= al0;
    st.l[1] *= al1;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      st.o[j][0] *= al0;
      st.o[j][1] *= al1;
      st.o[j][2] *= al0;
      st.o[j][3] *= al1;
    }
  }
  const float p0 = ex2(s0 - st.m[0]), p1 = ex2(s1 - st.m[1]);
  const float p2 = ex2(s2 - st.m[0]), p3 = ex2(s3 - st.m[1]);
  st.l[0] += p0 + p2;
  st.l[1] += p1 + p3;
  b0 = movmatrix_trans(pack_f16x2(p0, p1));
  b1 = movmatrix_trans(pack_f16x2(p2, p3));
}

// Ring position of the next stage a consumer warp reads.
struct RingPos {
  int slot = 0;
  uint32_t phase = 0;
  template <int PREC>
  __device__ __forceinline__ void advance() {
    if (++slot == Layout<PREC>::kStages) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// Wait for the stage at `p`; false (warp-uniform) after a timeout.
__device__ __forceinline__ bool wait_stage(uint64_t *full, const RingPos &p, volatile int *abort) {
  const bool ready = mbar_wait_bounded(&full[p.slot], p.phase, abort);
  return __all_sync(0xffffffffu, ready);
}

__device__ __forceinline__ int slice_valid(int64_t rem) {
  return rem < kSub ? (rem > 0 ? static_cast<int>(rem) : 0) : kSub;
}

template <int PREC>
__global__ void __launch_bounds__(kThreads, Layout<PREC>::kMinBlocks) decode_kernel(const DecodeArgs a) {
  using Lay = Layout<PREC>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *ring = smem;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + Lay::kStages * Lay::kStageBytes);
  uint64_t *empty = full + Lay::kStages;
  int32_t *cum = reinterpret_cast<int32_t *>(empty + Lay::kStages);
  float *mrg_o = reinterpret_cast<float *>(cum + kMaxBatch + 1);
  float *mrg_ml = mrg_o + kConsumerWarps * a.G * kD;
  int *flags = reinterpret_cast<int *>(mrg_ml + kConsumerWarps * kMaxGroup * 2);
  volatile int *abort = flags;              // flags[0]
  int *fills = flags + 1;                   // flags[1 .. kStages]: fills issued per slot

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hkv = a.c.Hkv, B = a.B, G = a.G;
  const int64_t cap = static_cast<int64_t>(a.max_pages) * a.c.P;

  // ---- prologue: tiles per sequence -> prefix sums (warp 0), barriers ----
  if (tid == 0) {
    flags[0] = 0;
    for (int s = 0; s < Lay::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);  // every consumer warp reads every stage
      fills[s] = 0;
    }
    fence_mbar_init();
  }
  if (warp == 0) {
    int carry = 0;
    if (lane == 0) cum[0] = 0;
    for (int base = 0; base < B; base += 32) {
      const int b = base + lane;
      int n = 0;
      if (b < B) {
        int64_t Lb = a.seq_lens[b];
        if (Lb < 0 || Lb > cap) {
          if (blockIdx.x == 0) set_err(a.c.err, NVKV_DEVERR_SEQLEN);
          Lb = Lb < 0 ? 0 : cap;
        }
        n = static_cast<int>((Lb + kTile - 1) / kTile);
      }
      int incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (b < B) cum[b + 1] = carry + incl;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();

  const int64_t W = static_cast<int64_t>(cum[B]) * Hkv;
  // never more shares than units: every active CTA owns at least one unit,
  // which the contributor count of the merge relies on
  const int64_t NC = W < a.num_ctas ? (W > 0 ? W : 1) : a.num_ctas;
  const bool active = blockIdx.x < NC;
  const int64_t u0 = active ? share_begin(blockIdx.x, W, NC) : 0;
  const int64_t u1 = active ? share_begin(blockIdx.x + 1, W, NC) : 0;

  // the combine kernel needs the same schedule: CTA 0 publishes it
  if (blockIdx.x == 0) {
    for (int b = tid; b <= B; b += kThreads) a.meta[b] = cum[b];
    if (tid == 0) a.meta[B + 1] = static_cast<int32_t>(NC);
  }

  // zero rows of empty sequences (spread over CTAs)
  for (int b = blockIdx.x; b < B; b += a.num_ctas) {
    if (cum[b + 1] == cum[b]) {
      uint4 *o = reinterpret_cast<uint4 *>(a.out + static_cast<int64_t>(b) * a.Hq * kD);
      for (int i = tid; i < a.Hq * kD / 8; i += kThreads) o[i] = make_uint4(0, 0, 0, 0);
    }
  }

  if (warp == kConsumerWarps) {
    producer<PREC>(a, ring, full, empty, cum, u0, u1, abort, fills);
  } else {
    const int r = lane >> 2, c = lane & 3;
    const SliceOffsets<PREC> so(warp, a.c.P);
    const float kscale = __fmul_rn(a.c.scale[0], a.sm_scale * 1.4426950408889634f);
    const float vscale = a.c.scale[1];
    RingPos pos;  // ring position and parity of the next stage this warp reads
    for (int64_t u = u0; u < u1;) {
      const Seg s = seg_at(u, u1, cum, B, Hkv);
      const int64_t Lb = clamped_len(a, s.b);
      // query of head j = r of the group, d in [32c, 32c+32), scaled by 2^-e_j into FP16
      uint32_t qf[8][2];
      float cs[2];
      {
        float qv[32];
        if (r < G) {
          const uint4 *qp =
              reinterpret_cast<const uint4 *>(a.q + (static_cast<int64_t>(s.b) * a.Hq + s.h * G + r) * kD + 32 * c);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            const uint4 w = __ldg(qp + v4);
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              qv[8 * v4 + 2 * e] = __uint_as_float(ww[e] << 16);
              qv[8 * v4 + 2 * e + 1] = __uint_as_float(ww[e] & 0xFFFF0000u);
            }
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) qv[e] = 0.0f;
        }
        float am = 0.0f;
#pragma unroll
        for (int e = 0; e < 32; ++e) am = fmaxf(am, fabsf(qv[e]));
        am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
        am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
        // ex = exponent of the head's max minus 14: the scaled max lies in [2^14, 2^15)
        int ex = 0;
        if (am > 0.0f) ex = static_cast<int>((__float_as_uint(am) >> 23) & 0xFF) - 127 - 14;
        ex = max(-110, min(110, ex));
        const float down = __uint_as_float(static_cast<uint32_t>(127 - ex) << 23);
#pragma unroll
        for (int s2 = 0; s2 < 8; ++s2) {
          qf[s2][0] = pack_f16x2(qv[4 * s2] * down, qv[4 * s2 + 1] * down);
          qf[s2][1] = pack_f16x2(qv[4 * s2 + 2] * down, qv[4 * s2 + 3] * down);
        }
        const int e0 = __shfl_sync(0xffffffffu, ex, 8 * c);
        const int e1 = __shfl_sync(0xffffffffu, ex, 8 * c + 4);
        cs[0] = __fmul_rn(kscale, __uint_as_float(static_cast<uint32_t>(127 + e0) << 23));
        cs[1] = __fmul_rn(kscale, __uint_as_float(static_cast<uint32_t>(127 + e1) << 23));
      }
      WarpState st;
#pragma unroll
      for (int j = 0; j < 8; ++j) st.o[j][0] = st.o[j][1] = st.o[j][2] = st.o[j][3] = 0.0f;
      st.m[0] = st.m[1] = -INFINITY;
      st.l[0] = st.l[1] = 0.0f;

      // two-deep pipeline over the segment's slices (see the consumer notes)
      const int ntiles = s.t1 - s.t0;
      const int64_t rem0 = Lb - static_cast<int64_t>(s.t0) * kTile - kSub * warp;
      bool ok = wait_stage(full, pos, abort);
      RingPos cur = pos;
      int nv_cur = slice_valid(rem0);
      uint32_t b0 = 0, b1 = 0;
      {
        KOps<PREC> kx;
        VOps<PREC> vx;
        float e[4] = {0.f, 0.f, 0.f, 0.f}, od[4] = {0.f, 0.f, 0.f, 0.f};
        load_k<PREC>(ring + static_cast<size_t>(cur.slot) * Lay::kStageBytes, so, r, c, kx);
        pipe_all<PREC, true, false>(kx, qf, e, od, vx, 0, 0, st);
        softmax_slice(e, od, nv_cur, r, cs, st, b0, b1);
      }
      pos.template advance<PREC>();
      for (int k = 0; k < ntiles && ok; ++k) {
        const uint8_t *stage_cur = ring + static_cast<size_t>(cur.slot) * Lay::kStageBytes;
        VOps<PREC> vx;
        load_v<PREC>(stage_cur, so, r, c, nv_cur, vx);
        if (k + 1 < ntiles) {
          ok = wait_stage(full, pos, abort);
          const int nv_next = slice_valid(rem0 - static_cast<int64_t>(k + 1) * kTile);
          KOps<PREC> kx;
          load_k<PREC>(ring + static_cast<size_t>(pos.slot) * Lay::kStageBytes, so, r, c, kx);
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[cur.slot]);
          float e[4] = {0.f, 0.f, 0.f, 0.f}, od[4] = {0.f, 0.f, 0.f, 0.f};
          pipe_all<PREC, true, true>(kx, qf, e, od, vx, b0, b1, st);
          softmax_slice(e, od, nv_next, r, cs, st, b0, b1);
          cur = pos;
          nv_cur = nv_next;
          pos.template advance<PREC>();
        } else {
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[cur.slot]);
          KOps<PREC> kx;
          float e[4], od[4];
          pipe_all<PREC, false, true>(kx, qf, e, od, vx, b0, b1, st);
        }
      }

      // ---- merge the four warps: (m, l) per head, O per (head, d) ----
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        st.l[0] += __shfl_xor_sync(0xffffffffu, st.l[0], o);
        st.l[1] += __shfl_xor_sync(0xffffffffu, st.l[1], o);
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int hd = 2 * c + e;
        if (hd < G) {
          float *dst = mrg_o + (warp * G + hd) * kD + 16 * r;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            dst[2 * j] = st.o[j][e];
            dst[2 * j + 1] = st.o[j][2 + e];
          }
          if (r == 0) {
            mrg_ml[(warp * kMaxGroup + hd) * 2 + 0] = st.m[e];
            mrg_ml[(warp * kMaxGroup + hd) * 2 + 1] = st.l[e];
          }
        }
      }
      named_bar_sync(1, kConsumerWarps * 32);

      const int nb = cum[s.b + 1] - cum[s.b];
      const bool complete = (s.t0 == 0) && (s.t1 == nb);
      const int slot_id = (u == u0) ? 0 : 1;
      float *part = a.partials + (static_cast<int64_t>(blockIdx.x) * 2 + slot_id) * kSlotFloats;
      for (int e = tid; e < G * kD; e += kConsumerWarps * 32) {
        const int hd = e / kD, d = e % kD;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mrg_ml[(w * kMaxGroup + hd) * 2]);
        float o = 0.0f, l = 0.0f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float mw = mrg_ml[(w * kMaxGroup + hd) * 2];
          const float f = (mw == -INFINITY) ? 0.0f : ex2(mw - M);
          o += f * mrg_o[(w * G + hd) * kD + d];
          l += f * mrg_ml[(w * kMaxGroup + hd) * 2 + 1];
        }
        if (complete) {
          a.out[(static_cast<int64_t>(s.b) * a.Hq + s.h * G + hd) * kD + d] = __float2bfloat16_rn(o * (vscale / l));
        } else {
          part[hd * kD + d] = o;
          if (d == 0) {
            part[kMaxGroup * kD + hd] = M;
            part[kMaxGroup * kD + kMaxGroup + hd] = l;
          }
        }
      }
      named_bar_sync(1, kConsumerWarps * 32);
      u += ntiles;
    }
  }

  // this CTA's partials are written: the combine grid may start launching
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __syncthreads();
  // after a timeout, wait (bounded) for copies still in flight before the CTA exits
  if (*abort) {
    if (tid == 0) set_err(a.c.err, NVKV_DEVERR_TIMEOUT);
    if (tid == kConsumerWarps * 32) {
      volatile int never = 0;
      for (int s = 0; s < Lay::kStages; ++s)
        if (fills[s] > 0) mbar_wait_bounded(&full[s], static_cast<uint32_t>(fills[s] - 1) & 1u, &never);
    }
  }
}


// ---------------------------------------------------------------------------
// Split-KV merge (log-sum-exp rule), one CTA per (sequence, KV head, query
// head of the group), thread = head_dim element.  Runs after the decode grid
// (programmatic dependent launch: griddepcontrol.wait returns once the decode
// grid has completed and its writes are visible).  Contributor k of a
// (sequence, KV head) left (o_k, m_k, l_k) in log2 units; out = sum_k
// 2^(m_k - M) o_k / sum_k 2^(m_k - M) l_k * g_V, M = max_k m_k.  (Sequence,
// head) pairs that one CTA covered entirely were written by the decode grid.
// ---------------------------------------------------------------------------
struct CombineArgs {
  const int32_t *meta;
  const float *partials;
  const float *scale;
  int32_t B, Hkv, Hq, G;
  __nv_bfloat16 *out;
};

constexpr int kCombineThreads = kD;
constexpr int kCombineBatch = 16;  // contributors whose loads are in flight together

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineArgs a) {
  const int tid = threadIdx.x;
  const int hd = blockIdx.x % a.G, bh = blockIdx.x / a.G, h = bh % a.Hkv, b = bh / a.Hkv;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int32_t c0 = a.meta[b], c1 = a.meta[b + 1];
  const int nb = c1 - c0;
  if (nb == 0) return;
  const int64_t W = static_cast<int64_t>(a.meta[a.B]) * a.Hkv, NC = a.meta[a.B + 1];
  const int64_t ubh0 = static_cast<int64_t>(c0) * a.Hkv + static_cast<int64_t>(h) * nb;
  const int64_t c_first = owner_of(ubh0, W, NC);
  const int n = static_cast<int>(owner_of(ubh0 + nb - 1, W, NC) - c_first + 1);
  if (n == 1) return;  // written directly by the decode grid
  // Every thread (one head_dim element) loads the statistics and its element
  // of a batch of contributors at once and folds them into a running
  // (max, sum, acc) triple: one round trip per batch, no block reductions.
  float M = -INFINITY, L = 0.0f, acc = 0.0f;
  for (int k0 = 0; k0 < n; k0 += kCombineBatch) {
    float m[kCombineBatch], l[kCombineBatch], o[kCombineBatch];
#pragma unroll
    for (int q = 0; q < kCombineBatch; ++q) {
      if (k0 + q < n) {
        const int64_t cc = c_first + k0 + q;
        const float *st = a.partials + (cc * 2 + (share_begin(cc, W, NC) >= ubh0 ? 0 : 1)) * kSlotFloats;
        m[q] = st[kMaxGroup * kD + hd];
        l[q] = st[kMaxGroup * kD + kMaxGroup + hd];
        o[q] = st[hd * kD + tid];
      } else {
        m[q] = -INFINITY;
        l[q] = 0.0f;
        o[q] = 0.0f;
      }
    }
    float mb = M;
#pragma unroll
    for (int q = 0; q < kCombineBatch; ++q) mb = fmaxf(mb, m[q]);
    const float r = M == -INFINITY ? 0.0f : ex2(M - mb);
    L *= r;
    acc *= r;
#pragma unroll
    for (int q = 0; q < kCombineBatch; ++q) {
      const float w = m[q] == -INFINITY ? 0.0f : ex2(m[q] - mb);
      L += w * l[q];
      acc += w * o[q];
    }
    M = mb;
  }
  a.out[(static_cast<int64_t>(b) * a.Hq + h * a.G + hd) * kD + tid] = __float2bfloat16_rn(acc * (a.scale[1] / L));
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
struct DevInfo {
  int sms = 0;
  int occ[2][kMaxGroup + 1] = {};
};

DevInfo g_info[64];
std::once_flag g_once[64];

template <int PREC>
int occupancy_for(int G) {
  const int smem = smem_bytes_for<PREC>(G);
  if (cudaFuncSetAttribute(decode_kernel<PREC>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<PREC>, kThreads, smem) != cudaSuccess) return 0;
  return n;
}

const DevInfo *dev_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::call_once(g_once[dev], [dev] {
    DevInfo &d = g_info[dev];
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    for (int G = 1; G <= kMaxGroup; ++G) {
      d.occ[0][G] = occupancy_for<NVKV_PREC_NVFP4>(G);
      d.occ[1][G] = occupancy_for<NVKV_PREC_FP8_E4M3>(G);
    }
  });
  return g_info[dev].sms > 0 ? &g_info[dev] : nullptr;
}

// CTAs of the persistent grid.  num_splits > 0: batch * Hkv * num_splits, so
// equal-length sequences are cut into exactly num_splits shares each.
int64_t num_ctas_for(int prec, int32_t batch, int32_t Hkv, int32_t G, int64_t max_units, int32_t num_splits) {
  int64_t n;
  if (num_splits > 0) {
    n = static_cast<int64_t>(batch) * Hkv * num_splits;
  } else {
    const DevInfo *d = dev_info();
    if (!d) return -1;
    const int occ = d->occ[prec][G] > 0 ? d->occ[prec][G] : 1;
    n = static_cast<int64_t>(d->sms) * occ;
  }
  if (n > max_units) n = max_units;
  return n < 1 ? 1 : n;
}

// Workspace = schedule (cum[0..B], NC) + two partial slots per CTA.
size_t meta_bytes(int32_t batch) { return (static_cast<size_t>(batch + 2) * 4 + 255) / 256 * 256; }

size_t workspace_bytes_for(int32_t batch, int32_t Hkv, int64_t nctas) {
  (void)Hkv;
  return meta_bytes(batch) + static_cast<size_t>(nctas) * 2 * kSlotFloats * sizeof(float);
}

nvkv_status decode_common(const void *q, const nvkv_cache *cache, const int32_t *block_table, int32_t max_pages,
                          const int32_t *seq_lens, int32_t batch, int32_t num_q_heads, int32_t prec, float sm_scale,
                          int32_t num_splits, void *workspace, size_t workspace_bytes, void *out, void *stream) {
  nvkv_status st = check_cache(cache, prec);
  if (st != NVKV_OK) return st;
  if (batch < 0 || num_q_heads <= 0 || max_pages <= 0 || num_splits < 0) return NVKV_ERR_INVALID_ARG;
  if (batch == 0) return NVKV_OK;
  if (batch > kMaxBatch) return NVKV_ERR_UNSUPPORTED;
  const int Hkv = cache->num_kv_heads;
  if (num_q_heads % Hkv != 0) return NVKV_ERR_INVALID_ARG;
  const int G = num_q_heads / Hkv;
  if (G > kMaxGroup) return NVKV_ERR_UNSUPPORTED;
  if (!q || !block_table || !seq_lens || !out || !workspace) return NVKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out) || !aligned16(workspace)) return NVKV_ERR_UNSUPPORTED;
  if (!(sm_scale >= 0.0f)) return NVKV_ERR_INVALID_ARG;
  const int64_t max_units = static_cast<int64_t>(batch) * Hkv *
                            ((static_cast<int64_t>(max_pages) * cache->page_size + kTile - 1) / kTile);
  const int64_t nctas = num_ctas_for(prec, batch, Hkv, G, max_units, num_splits);
  if (nctas < 0) return NVKV_ERR_CUDA;
  if (nctas > 0x7fffffff) return NVKV_ERR_UNSUPPORTED;
  if (workspace_bytes < workspace_bytes_for(batch, Hkv, nctas)) return NVKV_ERR_WORKSPACE_TOO_SMALL;
  if (!dev_info()) return NVKV_ERR_CUDA;

  DecodeArgs a;
  a.q = static_cast<const __nv_bfloat16 *>(q);
  a.c = to_dev(cache);
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.max_pages = max_pages;
  a.B = batch;
  a.Hq = num_q_heads;
  a.G = G;
  a.sm_scale = sm_scale > 0.0f ? sm_scale : 1.0f / sqrtf(static_cast<float>(cache->head_dim));
  a.num_ctas = static_cast<int32_t>(nctas);
  a.meta = static_cast<int32_t *>(workspace);
  a.partials = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + meta_bytes(batch));
  a.out = static_cast<__nv_bfloat16 *>(out);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (prec == NVKV_PREC_NVFP4)
    decode_kernel<NVKV_PREC_NVFP4><<<static_cast<int>(nctas), kThreads, smem_bytes_for<NVKV_PREC_NVFP4>(G), s>>>(a);
  else
    decode_kernel<NVKV_PREC_FP8_E4M3>
        <<<static_cast<int>(nctas), kThreads, smem_bytes_for<NVKV_PREC_FP8_E4M3>(G), s>>>(a);
  st = launch_status();
  if (st != NVKV_OK) return st;
  // split-KV merge, launched as a programmatic dependent of the decode grid
  CombineArgs ca;
  ca.meta = a.meta;
  ca.partials = a.partials;
  ca.scale = a.c.scale;
  ca.B = batch;
  ca.Hkv = Hkv;
  ca.Hq = num_q_heads;
  ca.G = G;
  ca.out = a.out;
  const int64_t cgrid = static_cast<int64_t>(batch) * Hkv * G;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cgrid));
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, combine_kernel, ca) != cudaSuccess) {
    cudaGetLastError();  // clear, then fall back to an ordinary stream-ordered launch
    combine_kernel<<<static_cast<unsigned>(cgrid), kCombineThreads, 0, s>>>(ca);
  }
  return launch_status();
}

}  // namespace
}  // namespace nvkv

// Scratch of nvfp4_paged_decode_attention_noalloc: a fixed device array for
// callers that cannot allocate (see the header).  Host code must not pass the
// symbol itself to a kernel (it is a host-side stand-in); the device address
// comes from cudaGetSymbolAddress, looked up once per device.
static __device__ __align__(256) uint8_t nvkv_noalloc_scratch[NVKV_NOALLOC_SCRATCH_BYTES];

namespace nvkv {
namespace {

struct NoAllocScratch {
  void *ptr = nullptr;
  cudaError_t err = cudaSuccess;
};
NoAllocScratch g_noalloc[64];
std::once_flag g_noalloc_once[64];

// Device address of the scratch array on the current device (nullptr on failure).
void *noalloc_scratch_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::call_once(g_noalloc_once[dev], [dev] {
    g_noalloc[dev].err = cudaGetSymbolAddress(&g_noalloc[dev].ptr, nvkv_noalloc_scratch);
    if (g_noalloc[dev].err != cudaSuccess) g_noalloc[dev].ptr = nullptr;
  });
  return g_noalloc[dev].ptr;
}

}  // namespace
}  // namespace nvkv

using namespace nvkv;

extern "C" {

nvkv_status nvfp4_paged_decode_attention_noalloc(const void *q, const nvkv_cache *cache,
                                                 const int32_t *block_table, int32_t max_pages,
                                                 const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                                                 int32_t layer_precision, float sm_scale, int32_t num_splits,
                                                 void *out, void *stream) {
  if (!cache || layer_precision != cache->prec) return NVKV_ERR_INVALID_ARG;
  if (layer_precision != NVKV_PREC_NVFP4 && layer_precision != NVKV_PREC_FP8_E4M3) return NVKV_ERR_INVALID_ARG;
  nvkv_status st = check_cache(cache, layer_precision);
  if (st != NVKV_OK) return st;
  if (batch < 0 || batch > kMaxBatch) return batch < 0 ? NVKV_ERR_INVALID_ARG : NVKV_ERR_UNSUPPORTED;
  if (batch == 0) return NVKV_OK;
  void *scratch = noalloc_scratch_ptr();
  if (!scratch) return NVKV_ERR_CUDA;
  // every call rewrites the scratch it later reads (schedule and partials): nothing needs clearing
  return decode_common(q, cache, block_table, max_pages, seq_lens, batch, num_q_heads, layer_precision, sm_scale,
                       num_splits, scratch, NVKV_NOALLOC_SCRATCH_BYTES, out, stream);
}

size_t nvkv_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t num_splits) {
  if (batch <= 0 || batch > kMaxBatch || num_kv_heads <= 0 || num_q_heads <= 0 || head_dim != kD ||
      num_splits < 0)
    return 0;
  if (num_q_heads % num_kv_heads != 0) return 0;
  const int G = num_q_heads / num_kv_heads;
  if (G > kMaxGroup) return 0;
  int64_t nctas;
  if (num_splits > 0) {
    nctas = static_cast<int64_t>(batch) * num_kv_heads * num_splits;
  } else {
    const DevInfo *d = dev_info();
    if (!d) return 0;
    int occ = 1;
    for (int p = 0; p < 2; ++p) occ = d->occ[p][G] > occ ? d->occ[p][G] : occ;
    nctas = static_cast<int64_t>(d->sms) * occ;
  }
  return workspace_bytes_for(batch, num_kv_heads, nctas);
}

nvkv_status nvkv_decode_workspace_init(void *workspace, size_t bytes, void *stream) {
  if (!workspace && bytes) return NVKV_ERR_INVALID_ARG;
  if (bytes == 0) return NVKV_OK;
  return cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream)) == cudaSuccess ? NVKV_OK
                                                                                               : NVKV_ERR_CUDA;
}

nvkv_status nvfp4_paged_decode_attention(const void *q, const nvkv_cache *cache, const int32_t *block_table,
                                         int32_t max_pages, const int32_t *seq_lens, int32_t batch,
                                         int32_t num_q_heads, int32_t layer_precision, float sm_scale,
                                         int32_t num_splits, void *workspace, size_t workspace_bytes, void *out,
                                         void *stream) {
  if (!cache || layer_precision != cache->prec) return NVKV_ERR_INVALID_ARG;
  if (layer_precision != NVKV_PREC_NVFP4 && layer_precision != NVKV_PREC_FP8_E4M3) return NVKV_ERR_INVALID_ARG;
  return decode_common(q, cache, block_table, max_pages, seq_lens, batch, num_q_heads, layer_precision, sm_scale,
                       num_splits, workspace, workspace_bytes, out, stream);
}

nvkv_status fp8_paged_decode_attention(const void *q, const nvkv_cache *cache, const int32_t *block_table,
                                       int32_t max_pages, const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                                       float sm_scale, int32_t num_splits, void *workspace, size_t workspace_bytes,
                                       void *out, void *stream) {
  return decode_common(q, cache, block_table, max_pages, seq_lens, batch, num_q_heads, NVKV_PREC_FP8_E4M3, sm_scale,
                       num_splits, workspace, workspace_bytes, out, stream);
}

}  // extern "C"
