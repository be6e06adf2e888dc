// Paged GQA decode attention reading the NVFP4 (or FP8 E4M3) cache straight
// from HBM ("SGLang x Qwen x NVIDIA ...", Three Paths: decode is memory-bound,
// so the kernel reads the NVFP4 cache itself and dequantizes inside; it must read
// exactly as much as it computes).  The per-layer FP8 variant serves the
// sensitive layers ("SOAR Weekly Champion Notes 05", 03).
//
// Design (sm_103a, one GPU):
//   * Work unit = one 128-token tile of one (sequence, KV head).  The units of
//     the whole batch are laid end to end and cut into equal contiguous shares,
//     one per CTA of a persistent grid (SMs x resident CTAs), so every CTA
//     streams the same number of bytes whatever the sequence lengths.  A
//     (sequence, KV head) cut between CTAs leaves split-KV partials; each
//     contributor counts itself on the pair's arrival counter and the CTA
//     that arrives last merges the parts with the log-sum-exp rule at its
//     end (one launch per call, no merge kernel).
//   * Warp roles: a producer warp per consumer group streams the group's tiles
//     into its shared-memory ring with 1-D bulk copies (one per page block,
//     mbarrier transaction counts); a query warp prepares each segment's query
//     operand; twelve consumer warps
//     in three groups of four (one warp per TMEM lane quadrant, 32 tokens each)
//     take the tiles round-robin: each warp arms its group's next tile (its
//     rows' scale factors, a count on the group's arming counter) as soon as
//     it has read its rows of the current scores, the fourth warp to arm
//     issues the score MMAs, and every warp then runs the softmax and P.V.
//     In the decode step (nvfp4_paged_decode_step) the producer that copies a
//     sequence's last tile first quantizes the step's new token into it.
//   * Scores S = K Q^T straight from the packed cache: the K codes of a staged
//     tile are the A operand of one block-scaled MMA (kind::mxf4nvf4, M = 128
//     tokens, K = 64 per instruction) and the E4M3 block scales of K are its
//     scale factors, so K is never dequantized by a thread.  The BF16 query
//     enters as the B operand in the same format: each query head is written
//     as a sum of NVFP4 terms (E2M1 codes, one E4M3 scale per 16 values; eight
//     terms at four heads per KV head, six at eight), stacked along N, and the
//     score is the sum of the head's columns.  The FP8 variant does the same
//     with kind::f8f6f4 and four E4M3 terms.  Scores land in TMEM (one buffer
//     per consumer group) and are read with tcgen05.ld, one token per consumer
//     thread.
//   * P.V on warp MMAs (m16n8k16 FP16 -> FP32; tokens = K, GQA heads = N):
//     E2M1 pairs -> f16x2 by cvt.rn.f16x2.e2m1x2, times the E4M3 block scale
//     (f16x2 multiply; code * scale has at most 6 significant bits in
//     [2^-10, 2688], exact in FP16).  P goes to the MMA operand layout through
//     a small per-warp shared-memory transpose.
//   * g_K, sm_scale, log2(e) and the power of two that scales each query head
//     before its decomposition form one FP32 factor per head; g_V is applied to
//     the output.  Online softmax in FP32 with exp2 and a lazily raised running
//     max (rescale only when the max grows by more than 2^8).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "nvkv_device.cuh"
#include "nvkv_host.h"

namespace nvkv {
namespace {

constexpr int kD = 128;
constexpr int kTile = 128;         // tokens per work unit / ring stage (the MMA M)
constexpr int kGroups = 3;         // consumer groups: group g takes the tiles i = g (mod 3) of the CTA
constexpr int kGroupWarps = 4;     // warp w of a group owns tokens [32w, 32w+32) of a tile = TMEM lane quadrant w
constexpr int kConsumerWarps = kGroups * kGroupWarps;
constexpr int kProducerWarp = kConsumerWarps;       // producer warps kProducerWarp + g, one per group
constexpr int kQueryWarp = kConsumerWarps + kGroups;
constexpr int kThreads = (kConsumerWarps + kGroups + 1) * 32;
constexpr int kMaxBatch = 1024;    // sequences per call (prefix sums live in shared memory)
constexpr int kMaxShares = 184;    // CTAs per launch (weighted shares keep every share's start in shared memory)
constexpr int kMaxGroup = 8;       // query heads per KV head
constexpr int kQBufs = 4;          // query images in flight: a group issues a tile at most three
                                   // segments ahead of the one all warps are in (segments of one tile)
constexpr int kSlotFloats = kMaxGroup * kD + 2 * kMaxGroup;  // one partial (o, m, l)
constexpr float kRescaleThreshold = 8.0f;                   // log2 units
constexpr float kNoMax = -1e30f;  // running max before any score: finite, so exp2(-inf - m) = 0

// Per-precision tile geometry (groups of 8 tokens, see nvkv_host.h).
template <int PREC>
struct Prec;
template <>
struct Prec<NVKV_PREC_NVFP4> {
  static constexpr int kTokBytes = kNvTokBytes;       // 144
  static constexpr int kGroup = kNvGroup;             // 1152
  static constexpr int kKRow = 64;                    // K bytes per token
  static constexpr int kMmas = 2;                     // K = 64 values per instruction
  static constexpr int kRing = 3;                     // stages per consumer group
};
template <>
struct Prec<NVKV_PREC_FP8_E4M3> {
  static constexpr int kTokBytes = kF8TokBytes;       // 256
  static constexpr int kGroup = kF8Group;             // 2048
  static constexpr int kKRow = 128;
  static constexpr int kMmas = 4;                     // K = 32 values per instruction
  static constexpr int kRing = 2;
};

// NH = heads per group slot set (4 or 8), N = NH * kTerms columns of the score
// MMA.  Query terms per head: E4M3 terms keep ~4 more bits each, so four
// reach FP32-like precision; E2M1 terms keep ~2.6 bits each relative to the
// residual of their 16-value block, so a block holding one outlier needs more
// (eight at four heads; six at eight heads, where TMEM columns run short).
template <int PREC, int NH>
struct Cfg {
  using P = Prec<PREC>;
  static constexpr bool kNv = PREC == NVKV_PREC_NVFP4;
  static constexpr int kTerms = !kNv ? 4 : (NH == 4 ? 8 : 6);
  // The head's largest |q| is scaled into [2^kHeadExp, 2^(kHeadExp+1)) before
  // the decomposition: E4M3 terms up to 448 (so [128, 256)); E2M1 terms carry
  // an E4M3 scale, so the top of the range is 6 x 448 = 2688 and [1024, 2048)
  // leaves the most room above the smallest scale (2^-9) for later terms.
  static constexpr int kHeadExp = kNv ? 10 : 7;
  static constexpr int N = NH * kTerms;
  static constexpr int kStageBytes = kTile / kGroupRows * P::kGroup;     // 18432 / 32768
  // Each consumer group has its own ring of kStagesG stages, filled by its own
  // producer warp: tile i (group i % 3, ordinal i / 3 within the group) sits
  // in slot slot_of(i) of the flat stage array, fill fill_of(i).
  static constexpr int kStagesG = P::kRing;
  static constexpr int kStages = kGroups * kStagesG;
  __host__ __device__ static constexpr int slot_of(int64_t i) {
    return static_cast<int>(i % kGroups) * kStagesG + static_cast<int>((i / kGroups) % kStagesG);
  }
  __host__ __device__ static constexpr uint32_t fill_of(int64_t i) {
    return static_cast<uint32_t>(i / kGroups / kStagesG);
  }
  static constexpr int kMH = kNv ? 4 : (NH == 8 ? 1 : 2);  // heads per pass of the segment merge
  // NVFP4 at four heads: the consumers leave a segment's (m, l, O) in shared
  // memory and go on; the query warp merges it (one pass holds every head)
  static constexpr bool kAsyncMerge = kNv && NH == 4;
  static constexpr int kQRow = P::kKRow;                                 // B row bytes
  static constexpr int kQImg = N * kQRow;                                // one query image
  static constexpr int kQSbo = 8 * kQRow;                                // 8-row group stride of B
  // TMEM columns: scores (one buffer of N per consumer group) from 0; NVFP4
  // scale factors at 16-column boundaries: A (K scales of the group's next
  // tile) at kSfaBase + 32 * group + 16 * mma (kSfaBase >= 3 N), B at 256 +
  // 32 * query image + 16 * mma.  One CTA per SM holds all 512.
  static constexpr uint32_t kTmemCols = kNv ? 512 : 128;
  static constexpr uint32_t kSfaBase = 3 * N <= 128 ? 128 : (3 * N + 15) / 16 * 16;
  static_assert(!kNv || kSfaBase + 32 * 2 + 16 + 4 <= 256, "A scale factors overlap B's");
  static_assert(kNv || 3 * N <= 128, "score buffers exceed the TMEM allocation");
  __host__ __device__ static constexpr uint32_t sfa_col(int buf, int k) { return kSfaBase + 32 * buf + 16 * k; }
  __host__ __device__ static constexpr uint32_t sfb_col(int qb, int k) { return 256 + 32 * qb + 16 * k; }
  // shared memory (bytes)
  static constexpr int oRing = 0;
  static constexpr int oQImg = oRing + kStages * kStageBytes;
  static constexpr int oSfb = oQImg + kQBufs * kQImg;                       // [4][2][32][16] (NVFP4)
  static constexpr int oPt = oSfb + (kNv ? kQBufs * 2 * 512 : 0);          // [12 warps][NH][32] f16
  static constexpr int oCs = oPt + kConsumerWarps * NH * 32 * 2;           // [4][8] f32
  static constexpr int oMrgO = oCs + kQBufs * 8 * 4;                       // [12 warps][kMH][128] f32
  static constexpr int oMrgMl = oMrgO + kConsumerWarps * kMH * kD * 4;     // [12 warps][8][2] f32
  static constexpr int oMrgHd = oMrgMl + kConsumerWarps * kMaxGroup * 2 * 4;  // [8][M, l] f32 per head
  static constexpr int oCum = oMrgHd + kMaxGroup * 2 * 4;                     // [kMaxBatch + 1] i32
  static constexpr int oLast = oCum + (kMaxBatch + 1) * 4;                // [kMaxBatch] u8
  static constexpr int oBars = (oLast + kMaxBatch + 15) / 16 * 16;
  static constexpr int kBars = 2 * kStages + kGroups + 2 * kQBufs + 1;  // full, empty, sready, qready, qfree, mdone
  static constexpr int oFlags = oBars + kBars * 8;  // tmem holder, abort, fills[kStages], W, NC, u0, u1, npend
  static constexpr int oPend = oFlags + 4 * (7 + kStages);  // [2][4] i32: split pairs this CTA merges at its end
  static constexpr int oArm = oPend + 4 * 8;  // [kGroups] i32 arming counters, [kGroups] i32 last tile armed
  static constexpr int kSmem = oArm + 4 * 2 * kGroups;
  // weighted shares (see tile_at): every share's first unit, after the rest
  static constexpr int oStarts = kSmem;  // [kMaxShares + 1] i32
  static constexpr int kSmemW = oStarts + 4 * (kMaxShares + 1);
  static_assert(kSmemW <= 232448, "shared memory exceeds the per-block limit");
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
  uint32_t *counters;  // [B][Hkv] arrivals of split (sequence, KV head) pairs; 0 between calls
  float *partials;     // [num_ctas][2][kSlotFloats]
  __nv_bfloat16 *out;
  const void *k_new, *v_new;  // decode step: [B][Hkv][128] newest token of each sequence (null: none)
  int32_t new_dtype;          // NVKV_DTYPE_F32 or NVKV_DTYPE_BF16
};

// Segment = run of consecutive units of one (sequence, KV head).
struct Seg {
  int b, h, t0, t1;  // tiles [t0, t1) of (b, h)
};

// cum[b] = tiles of sequences before b; units before sequence b = Hkv * cum[b].
// Unit indices fit in 32 bits (the host refuses larger problems).
__device__ __forceinline__ Seg seg_at(int64_t u64, int64_t u_end, const int32_t *cum, int B, int Hkv) {
  const int u = static_cast<int>(u64);
  int lo = 0, hi = B - 1;  // last b with Hkv*cum[b] <= u (sequences without tiles are skipped)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cum[mid] * Hkv <= u) lo = mid;
    else hi = mid - 1;
  }
  const int nb = cum[lo + 1] - cum[lo];
  const int r = u - cum[lo] * Hkv;
  Seg s;
  s.b = lo;
  s.h = r / nb;
  s.t0 = r - s.h * nb;
  const int left = static_cast<int>(u_end - u64);
  s.t1 = left < nb - s.t0 ? s.t0 + left : nb;
  return s;
}

// The segment after s, which ended at the end of its (b, h), starting at unit
// u (< u_end): the next KV head, or the next sequence that has tiles.
__device__ __forceinline__ Seg seg_next(const Seg &s, int64_t u, int64_t u_end, const int32_t *cum, int Hkv) {
  Seg n;
  n.b = s.b;
  n.h = s.h + 1;
  if (n.h == Hkv) {
    n.h = 0;
    do ++n.b; while (cum[n.b + 1] == cum[n.b]);
  }
  const int nb = cum[n.b + 1] - cum[n.b];
  const int64_t left = u_end - u;
  n.t0 = 0;
  n.t1 = left < nb ? static_cast<int>(left) : nb;
  return n;
}

// Shares: CTA c owns units [floor(c W / NC), floor((c+1) W / NC)); with W >= NC
// every share is non-empty.  owner_of(u) = the CTA whose share holds unit u.
__device__ __forceinline__ int64_t share_begin(int64_t c, int64_t W, int64_t NC) { return c * W / NC; }
__device__ __forceinline__ int64_t owner_of(int64_t u, int64_t W, int64_t NC) {
  return ((u + 1) * NC + W - 1) / W - 1;
}

// Shares weighted by pairs, for batches of many (sequence, KV head) pairs
// per CTA.  A pair costs a CTA more than its tiles: its query image, the
// merge of its partial results and the restart of the tile pipeline
// (measured ~1.2 us per pair a share holds on a batch of many short
// sequences, ~3 tiles' worth).  So the tiles are laid on a "virtual" line on
// which tile u of pair q = b Hkv + h starts at kVTile u + vk (q + 1): every
// pair (empty sequences' pairs included, which hold no tile) is preceded by
// vk units.  The line's length is V = kVTile W + vk B Hkv, CTA c's range is
// [floor(c V / NC), floor((c+1) V / NC)) and it owns the tiles whose start
// lies in it; a share is still a contiguous run of tiles.  With NC <= W a
// range is at least one tile long, so inside a pair (no gaps between its
// tiles) every CTA between the pair's first and last owner owns some of its
// tiles (the merge's contributor count relies on it); a range that falls
// between two pairs may hold no tile: that CTA has nothing to do.  vk =
// kVPair when the batch has at least kVPairMin pairs with tiles per CTA,
// else 0 (the equal split floor(c W / NC)).  The kernel that weighs shares
// is launched when batch x Hkv reaches kVPairMin per CTA; with fewer pairs
// per share the weight measured slower.
constexpr int64_t kVTile = 8, kVPair = 24, kVPairMin = 4;

__device__ __forceinline__ int64_t vpos(int64_t u, int b, int h, int Hkv, int64_t vk) {
  return kVTile * u + vk * (static_cast<int64_t>(b) * Hkv + h + 1);
}

// floor(n / d) for 0 <= n < 2^52 and 0 < d < 2^11, by two 32-bit divisions:
// n = hi 2^20 + lo, floor(n / d) = floor(hi / d) 2^20 +
// floor(((hi mod d) 2^20 + lo) / d), the second numerator < 2^31.
__device__ __forceinline__ int64_t div_small(int64_t n, uint32_t d) {
  const uint32_t hi = static_cast<uint32_t>(n >> 20), lo = static_cast<uint32_t>(n) & 0xFFFFFu;
  const uint32_t qh = hi / d;
  const uint32_t ql = (((hi - qh * d) << 20) | lo) / d;
  return (static_cast<int64_t>(qh) << 20) + ql;
}

// floor(n / d) for 0 <= n, 0 < d, when the quotient is known to be < 2^16:
// a single-precision estimate (relative error < 2^-20, so within one of the
// quotient) corrected by exact integer comparisons.
__device__ __forceinline__ int64_t div_est(int64_t n, int64_t d) {
  int64_t q = static_cast<int64_t>(__fdividef(static_cast<float>(n), static_cast<float>(d)));
  if (q < 0) q = 0;
  while (q > 0 && q * d > n) --q;
  while ((q + 1) * d <= n) ++q;
  return q;
}

// The first tile whose virtual start is >= vt (W when none is).  Sequence b's
// pairs start at base_b + h (kVTile nb + vk), base_b = vpos(Hkv cum[b], b,
// 0): a search over sequences, then the head by a short division.
__device__ __forceinline__ int64_t tile_at(int64_t vt, const int32_t *cum, int B, int Hkv, int64_t vk) {
  int lo = 0, hi = B - 1;  // the last sequence whose first position is <= vt
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (vpos(static_cast<int64_t>(cum[mid]) * Hkv, mid, 0, Hkv, vk) <= vt) lo = mid;
    else hi = mid - 1;
  }
  const int nb = cum[lo + 1] - cum[lo];
  const int64_t u_b = static_cast<int64_t>(cum[lo]) * Hkv;
  const int64_t base = vpos(u_b, lo, 0, Hkv, vk);
  if (base >= vt) return u_b;
  const int64_t step = kVTile * nb + vk;  // from one pair's first position to the next's
  if (step == 0) return u_b;            // (an empty sequence without weights: no tile here)
  int64_t h = div_est(vt - base, step);
  if (h > Hkv - 1) h = Hkv - 1;
  const int64_t p0 = base + h * step, u = u_b + h * nb;
  const int64_t t = (vt - p0 + kVTile - 1) / kVTile;
  return t < nb ? u + t : u + nb;  // past the pair: the next pair's first tile
}

// Weighted shares: the CTA whose share holds unit u (0 <= u < W), the last
// share starting at or before u (shares without tiles start where the next
// one does).
__device__ __forceinline__ int64_t owner_in(int64_t u, const int *starts, int64_t NC) {
  int lo = 0, hi = static_cast<int>(NC) - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (starts[mid] <= u) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Split-KV arrival, by one thread once this CTA's partial of segment s is
// written and fenced.  The contributors of (b, h) are the CTAs owning its
// first through last unit: contributor 0 left its part in slot 0 of its CTA
// if the pair opens that CTA's share, else in slot 1; contributor k > 0 in
// slot 0 of CTA c_first + k (the pair opens its share).  The contributor
// that arrives last resets the counter for the next call and records the
// pair {b, h, n, 2 c_first + slot} in the CTA's pending list (at most two:
// a share cuts at most its first and its last pair).
template <bool WT>
__device__ __forceinline__ void split_arrive(const DecodeArgs &a, const int32_t *cum, const Seg &s, int64_t W,
                                             int64_t NC, const int *starts, int *npend, int *pend) {
  const int Hkv = a.c.Hkv;
  const int nb = cum[s.b + 1] - cum[s.b];
  const int64_t ubh0 = static_cast<int64_t>(cum[s.b]) * Hkv + static_cast<int64_t>(s.h) * nb;
  const int64_t c_first = WT ? owner_in(ubh0, starts, NC) : owner_of(ubh0, W, NC);
  const int n = static_cast<int>((WT ? owner_in(ubh0 + nb - 1, starts, NC) : owner_of(ubh0 + nb - 1, W, NC)) -
                                 c_first + 1);
  uint32_t *cnt = a.counters + static_cast<int64_t>(s.b) * Hkv + s.h;
  const uint32_t before = atomicAdd(cnt, 1u);
  if (before == static_cast<uint32_t>(n - 1)) {  // every other part is in place
    atomicExch(cnt, 0u);
    const int r = atomicAdd(npend, 1);
    if (r < 2) {
      pend[4 * r + 0] = s.b;
      pend[4 * r + 1] = s.h;
      pend[4 * r + 2] = n;
      const int64_t first = WT ? starts[c_first] : share_begin(c_first, W, NC);
      pend[4 * r + 3] = static_cast<int>(c_first) * 2 + (first == ubh0 ? 0 : 1);
    }
  }
}

// Visible tokens of sequence b, from the set-up's shared-memory copies: its
// tile count and the tokens in its last tile (the clamped seq_lens[b]).
__device__ __forceinline__ int seq_len_of(const int32_t *cum, int b) {
  const int nb = cum[b + 1] - cum[b];
  return nb > 0 ? (nb - 1) * kTile + reinterpret_cast<const uint8_t *>(cum + kMaxBatch + 1)[b] : 0;
}

// Wait for `parity` of `bar`; false (warp-uniform) after a timeout or abort.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
  const bool ok = mbar_wait_bounded(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

// ---------------------------------------------------------------------------
// The decode step's new token (nvfp4_paged_decode_step): the token at
// position len - 1 of (b, h), read from k_new / v_new ([batch][Hkv][128]), is
// quantized into its cache slot by the producer warp of the tile that holds
// it, right before that tile is copied, with the layer's write rule and the
// cache descriptor's global scales g:
//   NVFP4: per 16-value block, scale byte = E4M3(amax / (6 g)), codes =
//          E2M1(x / (E4M3 scale x g)); K codes two per byte (value 2j in the
//          low nibble of byte j), V codes in this slot's nibble of the slot
//          pair's bytes, the partner slot's nibble kept;
//   FP8:   E4M3(x / g) per value.
// Lane = (block blk = lane / 4, values 4 (lane % 4) .. + 3 of it).  No other
// thread of the launch writes these bytes, so the shared V bytes are read,
// modified and written with plain accesses.
// ---------------------------------------------------------------------------
template <int PREC>
__device__ void append_token(const DecodeArgs &a, int b, int h, int64_t page, int off) {
  const int lane = threadIdx.x & 31, blk = lane >> 2, q = lane & 3;
  const CacheDev &c = a.c;
  const int64_t e = (static_cast<int64_t>(b) * c.Hkv + h) * kD + 16 * blk + 4 * q;  // first of the lane's values
#pragma unroll
  for (int kind = 0; kind < 2; ++kind) {
    const void *src = kind == 0 ? a.k_new : a.v_new;
    float x[4];
    if (a.new_dtype == NVKV_DTYPE_F32) {
      const float4 v = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(src) + e));
      x[0] = v.x;
      x[1] = v.y;
      x[2] = v.z;
      x[3] = v.w;
    } else {
      const uint2 v = __ldg(reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(src) + e));
      x[0] = __uint_as_float(v.x << 16);
      x[1] = __uint_as_float(v.x & 0xFFFF0000u);
      x[2] = __uint_as_float(v.y << 16);
      x[3] = __uint_as_float(v.y & 0xFFFF0000u);
    }
    const float g = c.scale[kind];
    if constexpr (PREC == NVKV_PREC_NVFP4) {
      float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));  // the block's four lanes
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      uint32_t sbyte = 0;
      float den = 0.0f;
      if (g != 0.0f) {
        sbyte = e4m3x2_from_f32(__fdiv_rn(amax, __fmul_rn(6.0f, g)), 0.0f) & 0xFFu;
        den = __fmul_rn(f32_from_e4m3(sbyte), g);
      }
      uint32_t codes = 0;  // values 4q .. 4q+3, one nibble each from bit 0
      if (den != 0.0f) {
        const float r = __frcp_rn(den);
        if (quot_fast_ok(r))  // codes of fl(x / den) from one reciprocal (exact, see e2m1x2_quot)
          codes = e2m1x2_quot(x[0], x[1], den, r) | (e2m1x2_quot(x[2], x[3], den, r) << 8);
        else
          codes = e2m1x2_from_f32(__fdiv_rn(x[0], den), __fdiv_rn(x[1], den)) |
                  (e2m1x2_from_f32(__fdiv_rn(x[2], den), __fdiv_rn(x[3], den)) << 8);
      }
      if (kind == 0) {
        *reinterpret_cast<uint16_t *>(c.data + c.nv_kcodes(page, h, off, blk) + 2 * q) = static_cast<uint16_t>(codes);
      } else {  // value 16 blk + j: byte j of the pair's 16 bytes, nibble off % 2
        uint32_t *dst = reinterpret_cast<uint32_t *>(c.data + c.nv_vcodes(page, h, off, blk) + 4 * q);
        const int sh = 4 * (off & 1);
        const uint32_t spread =
            (codes & 0xFu) | ((codes & 0xF0u) << 4) | ((codes & 0xF00u) << 8) | ((codes & 0xF000u) << 12);
        *dst = (*dst & ~(0x0F0F0F0Fu << sh)) | (spread << sh);
      }
      if (q == 0) c.data[c.nv_scale(page, h, kind, off, blk)] = static_cast<uint8_t>(sbyte);
    } else {
      uint32_t w = 0;
      if (g != 0.0f) {
        const float r = __frcp_rn(g);
        if (quot_fast_ok(fabsf(r)))  // bytes of fl(x / g) from one reciprocal (exact, see e4m3x2_quot)
          w = e4m3x2_quot(x[0], x[1], g, r) | (e4m3x2_quot(x[2], x[3], g, r) << 16);
        else
          w = e4m3x2_from_f32(__fdiv_rn(x[0], g), __fdiv_rn(x[1], g)) |
              (e4m3x2_from_f32(__fdiv_rn(x[2], g), __fdiv_rn(x[3], g)) << 16);
      }
      if (kind == 0) {
        *reinterpret_cast<uint32_t *>(c.data + c.f8_kblock(page, h, off, blk) + 4 * q) = w;
      } else {  // value 16 blk + 8 half + j: byte 2 j + off % 2 of chunk `half`
        uint8_t *dst = c.data + c.f8_vchunk(page, h, off, blk, q >> 1) + (off & 1) + 8 * (q & 1);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[2 * i] = static_cast<uint8_t>(w >> (8 * i));
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Producer warps, one per consumer group: producer g streams the tiles
// i = g (mod 3) of this CTA's share into group g's ring, one bulk copy per
// page block (a tile spans 128 / P whole page blocks, placed back to back, so
// the stage is 16 groups of 8 tokens at a uniform stride).  Lane j copies
// block j.
// ---------------------------------------------------------------------------
template <int PREC, int NH>
__device__ void producer(const DecodeArgs &a, uint8_t *ring, uint64_t *full, uint64_t *empty, const int32_t *cum,
                         int64_t u0, int64_t u1, int grp, volatile int *abort, int *fills) {
  using C = Cfg<PREC, NH>;
  const int lane = threadIdx.x & 31;
  const int Hkv = a.c.Hkv, P = a.c.P;
  const int lgP = __ffs(P) - 1;  // page sizes are powers of two (16, 32, 64)
  const uint64_t policy = policy_evict_first();
  const uint32_t block_bytes = static_cast<uint32_t>(P) * C::P::kTokBytes;
  int slot_l = 0;     // ring position of the group's next tile
  uint32_t fill = 0;  // fills of that slot so far
  int ibase = 0;      // CTA-local index of the segment's first tile
  Seg s = u0 < u1 ? seg_at(u0, u1, cum, a.B, Hkv) : Seg{0, 0, 0, 0};
  for (int64_t u = u0; u < u1; s = u < u1 ? seg_next(s, u, u1, cum, Hkv) : s) {
    const int ntiles = s.t1 - s.t0;
    const int kfirst = (grp - ibase % kGroups + kGroups) % kGroups;  // this group's first tile here
    if (kfirst < ntiles) {
      const int len = seq_len_of(cum, s.b);
      const int32_t *brow = a.block_table + static_cast<int64_t>(s.b) * a.max_pages;
      const uint8_t *src_h = a.c.data + a.c.block(0, s.h, C::P::kTokBytes);  // page 0 of head h
      const int64_t page_stride = a.c.block(1, 0, C::P::kTokBytes) - a.c.block(0, 0, C::P::kTokBytes);
      // Block-table window: lane l holds the entry of page index wbase + l; the
      // next window is requested when the current one comes into use.  Window
      // edges fall on tile edges (32 pages hold whole tiles at P = 16, 32, 64).
      int wbase = ((s.t0 + kfirst) * kTile) >> lgP;
      int32_t pg = wbase + lane < a.max_pages ? brow[wbase + lane] : 0;
      int32_t pg_next = wbase + 32 + lane < a.max_pages ? brow[wbase + 32 + lane] : 0;
      // The step's new token (position len - 1) lies in the pair's last tile:
      // if this group copies that tile, the warp writes the token while it
      // would otherwise wait for a free stage, at the latest just before the
      // tile's own copy (never before the ring's first fills go out).
      bool pend = a.k_new != nullptr && s.t1 == cum[s.b + 1] - cum[s.b] && (ntiles - 1 - kfirst) % kGroups == 0;
      for (int k = kfirst; k < ntiles; k += kGroups) {
        const int slot = grp * C::kStagesG + slot_l;
        const int tok0 = (s.t0 + k) * kTile;
        const int ntok = min(kTile, len - tok0);
        if (pend && (fill > 0 || tok0 + ntok == len)) {
          const int pos = len - 1;
          const int32_t pw = __ldg(brow + (pos >> lgP));
          if (pw >= 0 && pw < a.c.num_pages) append_token<PREC>(a, s.b, s.h, pw, pos & (P - 1));
          asm volatile("fence.proxy.async.global;" ::: "memory");  // the written bytes, before the copy reads them
          __syncwarp();
          pend = false;
        }
        if (lane == 0 && fill > 0) mbar_wait_bounded(&empty[slot], (fill - 1) & 1u, abort);
        if (__any_sync(0xffffffffu, *abort)) return;  // warp-uniform exit
        const int nblk = (ntok + P - 1) >> lgP;  // page blocks holding the tile's tokens
        while (((tok0 + ntok - 1) >> lgP) >= wbase + 32) {  // the tile leaves the window (warp-uniform)
          wbase += 32;
          pg = pg_next;
          pg_next = wbase + 32 + lane < a.max_pages ? brow[wbase + 32 + lane] : 0;
        }
        if (lane == 0) mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(nblk) * block_bytes);
        const int page = __shfl_sync(0xffffffffu, pg, ((tok0 >> lgP) + lane - wbase) & 31);
        if (lane < nblk) {
          int64_t pgc = page;
          if (page < 0 || page >= a.c.num_pages) {
            set_err(a.c.err, NVKV_DEVERR_PAGE);
            pgc = 0;  // a valid address; the output of this sequence is then undefined
          }
          bulk_g2s(ring + slot * C::kStageBytes + lane * block_bytes, src_h + pgc * page_stride, block_bytes,
                   &full[slot], policy);
        }
        if (lane == 0) fills[slot] = static_cast<int>(fill) + 1;
        if (++slot_l == C::kStagesG) {
          slot_l = 0;
          ++fill;
        }
      }
    }
    ibase += ntiles;
    u += ntiles;
  }
}

// ---------------------------------------------------------------------------
// Query images.  Lane (j, kb) of the query warp takes head j of the group and
// values [16 kb, 16 kb + 16); the head is scaled by 2^-e (its max lands in
// [2^kHeadExp, 2^(kHeadExp+1))) and written as kTerms terms, each the residual
// of the previous ones rounded to the operand format:
//   NVFP4: term = E2M1 codes x one E4M3 scale per 16 values (scale = residual
//          max / 6, rounded to E4M3); the codes fill B row n = kTerms j + term
//          in the MMA's K-major core-matrix order, the scale goes to the
//          scale-factor atom of MMA kb / 4, row n % 32, byte 4 (n / 32) + kb % 4.
//   FP8:   term = E4M3(residual), 16 bytes per lane and term.
// cs[j] = g_K * sm_scale * log2(e) * 2^e turns a score column sum into log2
// units.  Heads j >= G get zero terms and cs = 0.
// ---------------------------------------------------------------------------
template <int PREC, int NH>
__device__ void prepare_query(const DecodeArgs &a, const Seg &s, uint8_t *img, uint8_t *sfb, float *cs,
                              float kscale) {
  using C = Cfg<PREC, NH>;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int pass = 0; pass < NH / 4; ++pass) {
    const int j = (lane >> 3) + 4 * pass, kb = lane & 7;
    float v[16];
    if (j < a.G) {
      const uint4 *qp = reinterpret_cast<const uint4 *>(a.q + (static_cast<int64_t>(s.b) * a.Hq + s.h * a.G + j) * kD +
                                                        16 * kb);
#pragma unroll
      for (int v4 = 0; v4 < 2; ++v4) {
        const uint4 w = __ldg(qp + v4);
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v[8 * v4 + 2 * e] = __uint_as_float(ww[e] << 16);
          v[8 * v4 + 2 * e + 1] = __uint_as_float(ww[e] & 0xFFFF0000u);
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] = 0.0f;
    }
    float am = 0.0f;
#pragma unroll
    for (int e = 0; e < 16; ++e) am = fmaxf(am, fabsf(v[e]));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 4));
    int ex = 0;
    if (am > 0.0f) ex = static_cast<int>((__float_as_uint(am) >> 23) & 0xFF) - 127 - C::kHeadExp;
    ex = max(-100, min(100, ex));
    const float down = __uint_as_float(static_cast<uint32_t>(127 - ex) << 23);
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] *= down;  // exact (power of two)
#pragma unroll
    for (int t = 0; t < C::kTerms; ++t) {
      const int n = C::kTerms * j + t;
      if constexpr (C::kNv) {
        float m = 0.0f;
#pragma unroll
        for (int e = 0; e < 16; ++e) m = fmaxf(m, fabsf(v[e]));
        const uint32_t sb = e4m3x2_from_f32(m * (1.0f / 6.0f), 0.0f) & 0xFFu;
        const float sv = f32_from_e4m3(sb);
        uint32_t w[2] = {0u, 0u};
        if (sv > 0.0f) {
          const float inv = 1.0f / sv;
#pragma unroll
          for (int p = 0; p < 8; ++p) {
            const uint32_t byte = e2m1x2_from_f32(v[2 * p] * inv, v[2 * p + 1] * inv);
            w[p >> 2] |= byte << (8 * (p & 3));
            const uint32_t h2 = f16x2_from_e2m1x2<0>(byte);
            v[2 * p] -= f32_lo(h2) * sv;  // exact: at most 6 significant bits
            v[2 * p + 1] -= f32_hi(h2) * sv;
          }
        }
        *reinterpret_cast<uint2 *>(img + (n >> 3) * C::kQSbo + (kb >> 1) * 128 + (n & 7) * 16 + (kb & 1) * 8) =
            make_uint2(w[0], w[1]);
        // row n's four scale bytes of MMA kb / 4: word n / 32 of atom row n % 32
        sfb[(kb >> 2) * 512 + (n & 31) * 16 + (n >> 5) * 4 + (kb & 3)] = static_cast<uint8_t>(sb);
      } else {
        uint32_t w[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const uint32_t lo = e4m3x2_from_f32(v[4 * p], v[4 * p + 1]);
          const uint32_t hi = e4m3x2_from_f32(v[4 * p + 2], v[4 * p + 3]);
          w[p] = lo | (hi << 16);
          const uint32_t h0 = f16x2_from_e4m3x2<0>(w[p]), h1 = f16x2_from_e4m3x2<1>(w[p]);
          v[4 * p] -= f32_lo(h0);
          v[4 * p + 1] -= f32_hi(h0);
          v[4 * p + 2] -= f32_lo(h1);
          v[4 * p + 3] -= f32_hi(h1);
        }
        *reinterpret_cast<uint4 *>(img + (n >> 3) * C::kQSbo + kb * 128 + (n & 7) * 16) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    if (kb == 0) cs[j] = j < a.G ? __fmul_rn(kscale, __uint_as_float(static_cast<uint32_t>(127 + ex) << 23)) : 0.0f;
  }
  fence_proxy_async_smem();  // the images are read by the tensor cores (async proxy)
  __syncwarp();
}

// ---------------------------------------------------------------------------
// Query warp: the query images of the CTA's segments, in order, into a ring of
// four.  Image s overwrites image s - 4 once all consumer warps have merged
// segment s - 4 (qfree), which means every MMA that read it has completed.  A
// group issues a tile at most three tiles (so three segments) ahead of the
// segment it is in, and every warp has finished the segment before that one:
// the image it waits for never waits for the group itself.
// qready[q] completes when the image, its scale factors in TMEM (NVFP4: two
// tcgen05.cp copies, tracked by a commit) and its score factors are in place.
// ---------------------------------------------------------------------------
// Merge of one segment by the query warp (async merge): the twelve consumer
// warps left their (m, l) in mrg_ml and O of every head in mrg_o.  Per head:
// M = max_w m_w, factors f_w = 2^(m_w - M) (over m_w in place), l = sum f_w
// l_w; then O = sum_w f_w O_w goes to the output (the CTA held all of (b, h))
// or to the CTA's partial slot for the merge kernel.
template <int PREC, int NH, bool WT>
__device__ void merge_segment(const DecodeArgs &a, uint8_t *smem, const int32_t *cum, const Seg &s, int slot_id,
                              int64_t W, int64_t NC, int *npend) {
  using C = Cfg<PREC, NH>;
  const int lane = threadIdx.x & 31;
  const int G = a.G;
  const float *mrg_o = reinterpret_cast<const float *>(smem + C::oMrgO);
  float *mrg_ml = reinterpret_cast<float *>(smem + C::oMrgMl);
  float *mrg_hd = reinterpret_cast<float *>(smem + C::oMrgHd);
  const int nb = cum[s.b + 1] - cum[s.b];
  const bool complete = (s.t0 == 0) && (s.t1 == nb);
  if (lane < G) {
    const int hd = lane;
    float M = kNoMax;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mrg_ml[(w * kMaxGroup + hd) * 2]);
    float lsum = 0.0f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float f = ex2(mrg_ml[(w * kMaxGroup + hd) * 2] - M);  // warps without tokens: 0
      lsum += f * mrg_ml[(w * kMaxGroup + hd) * 2 + 1];
      mrg_ml[(w * kMaxGroup + hd) * 2] = f;
    }
    mrg_hd[2 * hd] = M;
    mrg_hd[2 * hd + 1] = lsum;
  }
  __syncwarp();
  const float vscale = a.c.scale[1];
  float *part = a.partials + (static_cast<int64_t>(blockIdx.x) * 2 + slot_id) * kSlotFloats;
  static_assert(kD == 4 * 32, "one head per pass: four values per lane");
  for (int hd = 0; hd < G; ++hd) {  // lane: values 4 lane .. 4 lane + 3 of head hd
    float4 o = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float f = mrg_ml[(w * kMaxGroup + hd) * 2];
      const float4 x = reinterpret_cast<const float4 *>(mrg_o + (w * C::kMH + hd) * kD)[lane];
      o.x += f * x.x;
      o.y += f * x.y;
      o.z += f * x.z;
      o.w += f * x.w;
    }
    const float lsum = mrg_hd[2 * hd + 1];
    if (complete) {
      const float sc = vscale / lsum;
      const __nv_bfloat162 lo = __floats2bfloat162_rn(o.x * sc, o.y * sc), hi = __floats2bfloat162_rn(o.z * sc, o.w * sc);
      uint2 pk;
      pk.x = *reinterpret_cast<const uint32_t *>(&lo);
      pk.y = *reinterpret_cast<const uint32_t *>(&hi);
      reinterpret_cast<uint2 *>(a.out + (static_cast<int64_t>(s.b) * a.Hq + s.h * G + hd) * kD)[lane] = pk;
    } else {
      reinterpret_cast<float4 *>(part + hd * kD)[lane] = o;
      if (lane == 0) {
        part[kMaxGroup * kD + hd] = mrg_hd[2 * hd];
        part[kMaxGroup * kD + kMaxGroup + hd] = lsum;
      }
    }
  }
  if (!complete) {
    __threadfence();  // this lane's part of the partial, visible before the arrival
    __syncwarp();
    if (lane == 0)
      split_arrive<WT>(a, cum, s, W, NC, reinterpret_cast<const int *>(smem + C::oStarts), npend, npend + 1);
  }
  __syncwarp();
}

// The query warp: prepares each segment's query image (at most kQBufs
// segments ahead of the consumers) and, with the async merge, merges each
// segment the consumers have finished, in order, but the share's last.
template <int PREC, int NH, bool WT>
__device__ int query_role(const DecodeArgs &a, uint8_t *smem, uint32_t tmem, uint64_t *qready, uint64_t *qfree,
                          uint64_t *mdone, const int32_t *cum, int64_t u0, int64_t u1, int64_t W, int64_t NC,
                          volatile int *abort, float kscale, int *npend) {
  using C = Cfg<PREC, NH>;
  const int lane = threadIdx.x & 31;
  uint8_t *qimg = smem + C::oQImg;
  uint8_t *sfb = smem + C::oSfb;
  float *cs = reinterpret_cast<float *>(smem + C::oCs);
  if (u0 >= u1) return 0;
  int sp = 0, sm = 0;  // images prepared, segments merged
  Seg s_p = seg_at(u0, u1, cum, a.B, a.c.Hkv), s_m = s_p;
  int64_t u_p = u0, u_m = u0;
  for (;;) {
    if (u_p < u1 && (!C::kAsyncMerge || sp < sm + kQBufs)) {
      const int q = sp % kQBufs;
      if (sp >= kQBufs && !warp_wait(&qfree[q], static_cast<uint32_t>(sp / kQBufs - 1) & 1u, abort)) return sp;
      prepare_query<PREC, NH>(a, s_p, qimg + q * C::kQImg, sfb + q * 1024, cs + q * 8, kscale);
      if (lane == 0) {
        if constexpr (C::kNv) {
          tc_fence_after();
          tmem_cp_32x128b_x4(tmem + C::sfb_col(q, 0), umma_desc(smem_u32(sfb + q * 1024), 128, 128));
          tmem_cp_32x128b_x4(tmem + C::sfb_col(q, 1), umma_desc(smem_u32(sfb + q * 1024 + 512), 128, 128));
          umma_commit(&qready[q]);  // arrives when the copies are done
        } else {
          mbar_arrive(&qready[q]);
        }
        mbar_arrive(&qready[q]);    // the image and score factors (release)
      }
      __syncwarp();
      u_p += s_p.t1 - s_p.t0;
      ++sp;
      if (u_p < u1) s_p = seg_next(s_p, u_p, u1, cum, a.c.Hkv);
    } else if (C::kAsyncMerge && u_m + (s_m.t1 - s_m.t0) < u1) {  // the last segment: merged by the consumers
      const int q = sm % kQBufs;
      if (!warp_wait(&qfree[q], static_cast<uint32_t>(sm / kQBufs) & 1u, abort)) return sp;  // segment sm done
      merge_segment<PREC, NH, WT>(a, smem, cum, s_m, u_m == u0 ? 0 : 1, W, NC, npend);
      if (lane == 0) mbar_arrive(mdone);  // its buffers may be rewritten
      __syncwarp();
      u_m += s_m.t1 - s_m.t0;
      ++sm;
      if (u_m < u1) s_m = seg_next(s_m, u_m, u1, cum, a.c.Hkv);
    } else {
      break;
    }
  }
  return sp;  // images prepared
}

// ---------------------------------------------------------------------------
// Consumer warps: P.V of a 16-token slice.  Lane = 4r + c.  MMA rows = head_dim
// (thread r owns d in [16r, 16r+16): tile J covers d = 16r + 2J, +1), k =
// tokens 2c, 2c+1, 2c+8, 2c+9 of the slice, n = query head.  O for heads
// 2c, 2c+1 of the group and d in [16r, 16r+16) lives in 32 registers.
// ---------------------------------------------------------------------------
struct WarpO {
  float o[8][4];
};

// V operand of a slice, straight from the pair-interleaved V layout: a[q] /
// b[q] hold the 16 bytes of token pairs (2c, 2c+1) / (2c+8, 2c+9) for values
// 16r .. 16r+15 (NVFP4: byte j = both tokens' codes of value 16r + j; FP8:
// two 8-value chunks, 16-bit half j' = both tokens' bytes of value 16r + 8h +
// j').  NVFP4 also carries the f16x2 block scales of both pairs; masked
// tokens get scale 0 (NVFP4) or a zero byte (FP8).
template <int PREC>
struct VOps {
  uint32_t a[PREC == NVKV_PREC_NVFP4 ? 4 : 8], b[PREC == NVKV_PREC_NVFP4 ? 4 : 8];
  uint32_t sAB, sCD;
};

// g0 = the slice's first group (two groups of 8 tokens); nvalid = valid tokens (1..16).
template <int PREC>
__device__ __forceinline__ void load_v(const uint8_t *g0, int r, int c, int nvalid, VOps<PREC> &x) {
  const int tA = 2 * c;
  if constexpr (PREC == NVKV_PREC_NVFP4) {
    const uint8_t *g1 = g0 + kNvGroup;
    const uint4 A = *reinterpret_cast<const uint4 *>(g0 + kNvVCodes + r * 64 + c * 16);
    const uint4 B = *reinterpret_cast<const uint4 *>(g1 + kNvVCodes + r * 64 + c * 16);
    uint32_t sv = static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(g0 + kNvVScales + r * 8 + tA)) |
                  (static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(g1 + kNvVScales + r * 8 + tA)) << 16);
    if (nvalid < 16) {  // masked tokens get scale 0 -> value 0 (codes are finite)
      if (tA >= nvalid) sv &= 0xFFFFFF00u;
      if (tA + 1 >= nvalid) sv &= 0xFFFF00FFu;
      if (tA + 8 >= nvalid) sv &= 0xFF00FFFFu;
      if (tA + 9 >= nvalid) sv &= 0x00FFFFFFu;
    }
    x.sAB = f16x2_from_e4m3x2<0>(sv);
    x.sCD = f16x2_from_e4m3x2<1>(sv);
    x.a[0] = A.x; x.a[1] = A.y; x.a[2] = A.z; x.a[3] = A.w;
    x.b[0] = B.x; x.b[1] = B.y; x.b[2] = B.z; x.b[3] = B.w;
  } else {
    const uint8_t *g1 = g0 + kF8Group;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const uint4 A = *reinterpret_cast<const uint4 *>(g0 + kF8V + hh * 512 + r * 64 + c * 16);
      const uint4 B = *reinterpret_cast<const uint4 *>(g1 + kF8V + hh * 512 + r * 64 + c * 16);
      x.a[4 * hh + 0] = A.x; x.a[4 * hh + 1] = A.y; x.a[4 * hh + 2] = A.z; x.a[4 * hh + 3] = A.w;
      x.b[4 * hh + 0] = B.x; x.b[4 * hh + 1] = B.y; x.b[4 * hh + 2] = B.z; x.b[4 * hh + 3] = B.w;
    }
    if (nvalid < 16) {  // masked tokens -> E4M3 zero (stale bytes could be NaN)
      const uint32_t ma = (tA >= nvalid ? 0u : 0x00FF00FFu) | (tA + 1 >= nvalid ? 0u : 0xFF00FF00u);
      const uint32_t mb = (tA + 8 >= nvalid ? 0u : 0x00FF00FFu) | (tA + 9 >= nvalid ? 0u : 0xFF00FF00u);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        x.a[q] &= ma;
        x.b[q] &= mb;
      }
    }
    x.sAB = x.sCD = 0;
  }
}

// P.V MMA for output tile J (values d = 16r + 2J, 16r + 2J + 1).  NVFP4: bytes
// 2J, 2J + 1 of each pair, i.e. bytes 2(J%2), 2(J%2)+1 of word J/2.  FP8:
// chunk J/4, word J%4, halves 0 (d) and 1 (d + 1).
template <int PREC, int J>
__device__ __forceinline__ void pv_tile(const VOps<PREC> &x, uint32_t b0, uint32_t b1, WarpO &st) {
  if constexpr (PREC == NVKV_PREC_NVFP4) {
    constexpr int w = J >> 1, I = 2 * (J & 1);
    mma_f16_16816(st.o[J], hmul2_u32(f16x2_from_e2m1x2<I>(x.a[w]), x.sAB),
                  hmul2_u32(f16x2_from_e2m1x2<I + 1>(x.a[w]), x.sAB), hmul2_u32(f16x2_from_e2m1x2<I>(x.b[w]), x.sCD),
                  hmul2_u32(f16x2_from_e2m1x2<I + 1>(x.b[w]), x.sCD), b0, b1);
  } else {
    constexpr int q = 4 * (J >> 2) + (J & 3);
    mma_f16_16816(st.o[J], f16x2_from_e4m3x2<0>(x.a[q]), f16x2_from_e4m3x2<1>(x.a[q]), f16x2_from_e4m3x2<0>(x.b[q]),
                  f16x2_from_e4m3x2<1>(x.b[q]), b0, b1);
  }
}

// Two slices: MMA J of slice 1 follows MMA J of slice 0 (same accumulator),
// the eight accumulator chains run side by side.
template <int PREC>
__device__ __forceinline__ void pv_pair(const VOps<PREC> &x, uint32_t b0, uint32_t b1, const VOps<PREC> &y, uint32_t c0,
                                        uint32_t c1, WarpO &st) {
  pv_tile<PREC, 0>(x, b0, b1, st);
  pv_tile<PREC, 1>(x, b0, b1, st);
  pv_tile<PREC, 2>(x, b0, b1, st);
  pv_tile<PREC, 3>(x, b0, b1, st);
  pv_tile<PREC, 0>(y, c0, c1, st);
  pv_tile<PREC, 1>(y, c0, c1, st);
  pv_tile<PREC, 2>(y, c0, c1, st);
  pv_tile<PREC, 3>(y, c0, c1, st);
  pv_tile<PREC, 4>(x, b0, b1, st);
  pv_tile<PREC, 5>(x, b0, b1, st);
  pv_tile<PREC, 6>(x, b0, b1, st);
  pv_tile<PREC, 7>(x, b0, b1, st);
  pv_tile<PREC, 4>(y, c0, c1, st);
  pv_tile<PREC, 5>(y, c0, c1, st);
  pv_tile<PREC, 6>(y, c0, c1, st);
  pv_tile<PREC, 7>(y, c0, c1, st);
}

template <int PREC>
__device__ __forceinline__ void pv_slice(const VOps<PREC> &x, uint32_t b0, uint32_t b1, WarpO &st) {
  pv_tile<PREC, 0>(x, b0, b1, st);
  pv_tile<PREC, 1>(x, b0, b1, st);
  pv_tile<PREC, 2>(x, b0, b1, st);
  pv_tile<PREC, 3>(x, b0, b1, st);
  pv_tile<PREC, 4>(x, b0, b1, st);
  pv_tile<PREC, 5>(x, b0, b1, st);
  pv_tile<PREC, 6>(x, b0, b1, st);
  pv_tile<PREC, 7>(x, b0, b1, st);
}

// ---------------------------------------------------------------------------
// Consumer warps, three groups of four.  Group g takes the tiles i = g (mod 3)
// of the CTA's share; per tile each warp reads its 32 rows of the group's
// score buffer (one token per lane, kTerms columns per head), runs the online
// softmax per head with the running max shared by the warp, writes P to a
// per-warp [head][token] FP16 tile in shared memory, then P.V for its two
// 16-token slices with V straight from the stage.  At the end of a segment
// the twelve warps merge (m, l, O).
// ---------------------------------------------------------------------------
// Index of the segment holding CTA-local tile x, walking forward from the
// segment that starts at unit u (index sidx, ntiles tiles).
__device__ __forceinline__ int seg_index_of(int64_t x, int64_t u, int sidx, int ntiles, int64_t u0, int64_t u1,
                                            const int32_t *cum, int B, int Hkv) {
  while (x >= (u - u0) + ntiles) {
    u += ntiles;
    ++sidx;
    const Seg ns = seg_at(u, u1, cum, B, Hkv);
    ntiles = ns.t1 - ns.t0;
  }
  return sidx;
}

// Score MMAs of one tile of consumer group grp (stage = ring slot `slot`,
// query image qb with parity qpar), armed by the group's four warps without
// a barrier.  Each warp calls this once the stage has landed and it has read
// its rows of the group's previous scores (so the score buffer and the scale
// columns are free for its rows): NVFP4 writes the K block scales of its 32
// rows into the group's TMEM scale-factor columns (row m = 32 qd + lane is
// read by the MMA from lane m, column sfa_col(grp, mma) + qd), then the warp
// counts itself on the group's arming counter in shared memory.  The warp
// that arrives fourth waits for the query image and issues the MMAs into the
// group's score buffer, committing them to sready[grp].  The counter only
// grows: the four arrivals of one tile all come before any arrival for the
// group's next tile (which needs these MMAs' scores), so the fourth arrival
// of a tile is the one that finds count = 3 (mod 4).  Returns true (lane 0)
// when this warp issued the MMAs.
template <int PREC, int NH>
__device__ __forceinline__ bool arm_tile(uint8_t *smem, uint32_t tmem, uint32_t tq, uint64_t *sready, uint64_t *qready,
                                         int *arm_cnt, int slot, int qb, uint32_t qpar, int grp, int qd, int lane,
                                         volatile int *abort) {
  using C = Cfg<PREC, NH>;
  const uint8_t *stage = smem + C::oRing + slot * C::kStageBytes;
  if constexpr (C::kNv) {
    const int t = 32 * qd + lane;
    const uint2 sc = *reinterpret_cast<const uint2 *>(stage + (t >> 3) * kNvGroup + kNvKScales + (t & 7) * 8);
    tmem_st1(tq + C::sfa_col(grp, 0) + qd, sc.x);  // blocks 0..3 (MMA 0)
    tmem_st1(tq + C::sfa_col(grp, 1) + qd, sc.y);  // blocks 4..7 (MMA 1)
    tmem_st_wait();
  }
  tc_fence_before();
  __syncwarp();
  bool issued = false;
  if (lane == 0) {
    __threadfence_block();  // this warp's scale columns and score reads, before its arrival
    if ((atomicAdd(&arm_cnt[grp], 1) & (kGroupWarps - 1)) == kGroupWarps - 1 && mbar_wait_bounded(&qready[qb], qpar, abort)) {
      __threadfence_block();
      tc_fence_after();
      const uint32_t d = tmem + static_cast<uint32_t>(grp * C::N);
      const uint32_t a0 = smem_u32(stage), b0 = smem_u32(smem + C::oQImg + qb * C::kQImg);
      if constexpr (C::kNv) {
#pragma unroll
        for (int kk = 0; kk < C::P::kMmas; ++kk)
          umma_nvfp4(d, umma_desc(a0 + kk * 256, 128, kNvGroup), umma_desc(b0 + kk * 256, 128, C::kQSbo),
                     idesc_nvfp4(C::N), tmem + C::sfa_col(grp, kk), tmem + C::sfb_col(qb, kk), kk > 0 ? 1u : 0u);
      } else {
#pragma unroll
        for (int kk = 0; kk < C::P::kMmas; ++kk)
          umma_e4m3(d, umma_desc(a0 + kk * 256, 128, kF8Group), umma_desc(b0 + kk * 256, 128, C::kQSbo),
                    idesc_e4m3(C::N), kk > 0 ? 1u : 0u);
      }
      umma_commit(&sready[grp]);
      issued = true;
    }
  }
  __syncwarp();
  return issued;
}

template <int NH>
__device__ __forceinline__ float pick(const float (&v)[NH], int i) {  // v[i] for a runtime i < NH
  float r = v[0];
#pragma unroll
  for (int k = 1; k < NH; ++k) r = i == k ? v[k] : r;
  return r;
}

template <int PREC, int NH, bool WT>
__device__ void consumer_role(const DecodeArgs &a, uint8_t *smem, uint32_t tmem, uint64_t *full, uint64_t *empty,
                              uint64_t *sready, uint64_t *qready, uint64_t *qfree, uint64_t *mdone, const int32_t *cum,
                              int64_t u0, int64_t u1, int64_t W, int64_t NC, volatile int *abort,
                              int *arm_cnt, int *last_iss, int *npend) {
  using C = Cfg<PREC, NH>;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int grp = warp / kGroupWarps, qd = warp % kGroupWarps;  // consumer group, TMEM lane quadrant
  const int r = lane >> 2, c = lane & 3;
  const int Hkv = a.c.Hkv, G = a.G;
  uint8_t *ring = smem + C::oRing;
  const float *csb = reinterpret_cast<const float *>(smem + C::oCs);
  __half *pt = reinterpret_cast<__half *>(smem + C::oPt) + warp * NH * 32;
  float *mrg_o = reinterpret_cast<float *>(smem + C::oMrgO);
  float *mrg_ml = reinterpret_cast<float *>(smem + C::oMrgMl);
  float *mrg_hd = reinterpret_cast<float *>(smem + C::oMrgHd);
  const float vscale = a.c.scale[1];
  const uint32_t tq = tmem + (static_cast<uint32_t>(32 * qd) << 16);  // this warp's lane quadrant
  // The group's tiles are i = grp, grp + 3, ... (CTA-local); its n-th tile
  // uses ring slot kStagesG * grp + n % kStagesG with fill parity
  // (n / kStagesG) & 1, and score buffer phase n & 1.  Counters advance
  // per tile instead of being divided out.
  const int ntotal = static_cast<int>(u1 - u0);  // tiles of the share
  int slot_l = 0;          // ring position of the group's current tile
  uint32_t fpar = 0;       // its fill parity
  uint32_t spar = 0;       // score buffer phase of the current tile
  int ibase = 0;           // CTA-local index of the segment's first tile
  int sidx = 0;
  bool ok = true;
  // The group's first tile is armed before anything else.
  if (grp < ntotal) {
    const Seg s0 = seg_at(u0, u1, cum, a.B, Hkv);
    const int sx = seg_index_of(grp, u0, 0, s0.t1 - s0.t0, u0, u1, cum, a.B, Hkv);
    ok = warp_wait(&full[grp * C::kStagesG], 0u, abort);
    if (ok && arm_tile<PREC, NH>(smem, tmem, tq, sready, qready, arm_cnt, grp * C::kStagesG, sx % kQBufs,
                                 static_cast<uint32_t>(sx / kQBufs) & 1u, grp, qd, lane, abort))
      last_iss[grp] = grp;
  }
  // After a timeout (ok false) the warps skip all work but keep walking the
  // same segments, so every named barrier of the merge still meets.
  Seg s = u0 < u1 ? seg_at(u0, u1, cum, a.B, Hkv) : Seg{0, 0, 0, 0};
  for (int64_t u = u0; u < u1; ++sidx) {
    // the segment after this one (its length places the group's next tile
    // when that crosses the boundary)
    const int ntiles = s.t1 - s.t0;
    const Seg s_nx = u + ntiles < u1 ? seg_next(s, u + ntiles, u1, cum, Hkv) : s;
    const int Lb = seq_len_of(cum, s.b);
    const int qb = sidx % kQBufs;
    ok = ok && warp_wait(&qready[qb], static_cast<uint32_t>(sidx / kQBufs) & 1u, abort);
    float cs[NH], m[NH], mt[NH], l[NH];  // mt = m + the rescale threshold
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      cs[h] = csb[qb * 8 + h];
      m[h] = mt[h] = kNoMax;
      l[h] = 0.0f;
    }
    WarpO st;
#pragma unroll
    for (int j = 0; j < 8; ++j) st.o[j][0] = st.o[j][1] = st.o[j][2] = st.o[j][3] = 0.0f;
    for (int k = (grp - ibase % kGroups + kGroups) % kGroups; k < ntiles; k += kGroups) {
      const int i = ibase + k;
      const int slot = grp * C::kStagesG + slot_l;
      const int nslot_l = slot_l + 1 == C::kStagesG ? 0 : slot_l + 1;  // the group's next tile
      const uint32_t nfpar = nslot_l == 0 ? fpar ^ 1u : fpar;
      ok = ok && warp_wait(&sready[grp], spar, abort);
      float ssum[NH];  // per head: the sum of its kTerms score columns
      float sp[NH][2];  // per head: partial sums of its even and odd columns
#pragma unroll
      for (int h = 0; h < NH; ++h) ssum[h] = sp[h][0] = sp[h][1] = 0.0f;
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int ch = 0; ch < C::N / 16; ++ch) {
          float x[16];
          tmem_ld16(tq + static_cast<uint32_t>(grp * C::N + 16 * ch), x);
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            if constexpr (C::kTerms % 2 == 0) {  // adjacent columns of one head: packed pairs, folded at the end
              add_f32x2(sp[(16 * ch + e) / C::kTerms][0], sp[(16 * ch + e) / C::kTerms][1], x[e], x[e + 1]);
            } else {
              ssum[(16 * ch + e) / C::kTerms] += x[e];
              ssum[(16 * ch + e + 1) / C::kTerms] += x[e + 1];
            }
          }
        }
        if constexpr (C::kTerms % 2 == 0) {
#pragma unroll
          for (int h = 0; h < NH; ++h) ssum[h] = sp[h][0] + sp[h][1];
        }
      }
      // This warp's rows of the group's score buffer are read: it arms the
      // group's next tile now if that tile's stage has landed, else after
      // this tile's P.V, so it never waits for data it does not need yet.
      const bool has_next = i + kGroups < ntotal;
      int nqb = qb;
      uint32_t nqpar = static_cast<uint32_t>(sidx / kQBufs) & 1u;
      bool armed = false;
      if (has_next) {
        if (k + kGroups >= ntiles) {  // the next tile lies in a later segment
          int sx = sidx + 1;
          if (k + kGroups - ntiles >= s_nx.t1 - s_nx.t0)  // beyond the next segment too (short segments)
            sx = seg_index_of(i + kGroups, u, sidx, ntiles, u0, u1, cum, a.B, Hkv);
          nqb = sx % kQBufs;
          nqpar = static_cast<uint32_t>(sx / kQBufs) & 1u;
        }
        if (ok && mbar_test(&full[grp * C::kStagesG + nslot_l], nfpar)) {
          if (arm_tile<PREC, NH>(smem, tmem, tq, sready, qready, arm_cnt, grp * C::kStagesG + nslot_l, nqb, nqpar,
                                 grp, qd, lane, abort))
            last_iss[grp] = i + kGroups;  // its MMAs went out
          armed = true;
        }
      }
      slot_l = nslot_l;
      fpar = nfpar;
      spar ^= 1u;
      if (!ok) continue;

      // scores of this lane's token, log2 units; masked past the sequence end
      const int t = s.t0 + k;
      const bool valid = t * kTile + 32 * qd + lane < Lb;
      // heads >= G have cs = 0: finite dummy scores, never written out
      float sc[NH];
      bool need = false;
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        sc[h] = valid ? ssum[h] * cs[h] : -INFINITY;
        need |= sc[h] > mt[h];
      }
      if (__any_sync(0xffffffffu, need)) {  // raise the running max (warp-uniform)
        float al[NH];
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          float mx = sc[h];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          const float nm = fmaxf(m[h], mx);
          al[h] = ex2(m[h] - nm);
          m[h] = nm;
          mt[h] = nm + kRescaleThreshold;
          l[h] *= al[h];
        }
        const float alo = 2 * c < NH ? pick<NH>(al, 2 * c) : 1.0f;
        const float ahi = 2 * c + 1 < NH ? pick<NH>(al, 2 * c + 1) : 1.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          st.o[j][0] *= alo;
          st.o[j][2] *= alo;
          st.o[j][1] *= ahi;
          st.o[j][3] *= ahi;
        }
      }
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        const float p = ex2(sc[h] - m[h]);  // masked tokens: exp2(-inf) = 0
        l[h] += p;
        pt[h * 32 + lane] = __float2half_rn(p);
      }
      __syncwarp();

      // P.V over the warp's two 16-token slices, their MMA chains interleaved
      const uint8_t *stage = ring + slot * C::kStageBytes;
      const int rem = Lb - (t * kTile + 32 * qd);  // warp-uniform
      if (rem > 0) {
        uint32_t b[4] = {0u, 0u, 0u, 0u};
        if (r < NH) {
#pragma unroll
          for (int q = 0; q < 4; ++q) b[q] = *reinterpret_cast<const uint32_t *>(pt + r * 32 + 8 * q + 2 * c);
        }
        VOps<PREC> v0;
        load_v<PREC>(stage + (4 * qd) * C::P::kGroup, r, c, rem < 16 ? rem : 16, v0);
        if (rem > 16) {
          VOps<PREC> v1;
          load_v<PREC>(stage + (4 * qd + 2) * C::P::kGroup, r, c, rem < 32 ? rem - 16 : 16, v1);
          pv_pair<PREC>(v0, b[0], b[1], v1, b[2], b[3], st);
        } else {
          pv_slice<PREC>(v0, b[0], b[1], st);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      if (has_next && !armed) {
        ok = warp_wait(&full[grp * C::kStagesG + slot_l], fpar, abort);
        if (ok && arm_tile<PREC, NH>(smem, tmem, tq, sready, qready, arm_cnt, grp * C::kStagesG + slot_l, nqb, nqpar,
                                     grp, qd, lane, abort))
          last_iss[grp] = i + kGroups;  // its MMAs went out
      }
    }
    ibase += ntiles;

    // the query warp may still be merging the previous segment out of the
    // merge buffers
    if (C::kAsyncMerge && sidx > 0) ok = warp_wait(mdone, static_cast<uint32_t>(sidx - 1) & 1u, abort) && ok;
    if (C::kAsyncMerge && u + ntiles < u1) {
      // not the share's last segment: leave (m, l, O) for the query warp and
      // go on (the last segment is merged by all twelve warps, below)
#pragma unroll
      for (int h = 0; h < NH; ++h)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l[h] += __shfl_xor_sync(0xffffffffu, l[h], o);
      if (lane == 0) {
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          mrg_ml[(warp * kMaxGroup + h) * 2 + 0] = m[h];
          mrg_ml[(warp * kMaxGroup + h) * 2 + 1] = l[h];
        }
      }
#pragma unroll
      for (int hd = 0; hd < NH; ++hd) {  // the lanes with c = hd / 2 hold head hd in column hd % 2
        if (hd < G && (hd >> 1) == c) {
          float2 *dst = reinterpret_cast<float2 *>(mrg_o + (warp * C::kMH + hd) * kD + 16 * r);
#pragma unroll
          for (int j = 0; j < 8; ++j) dst[j] = make_float2(st.o[j][hd & 1], st.o[j][2 + (hd & 1)]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&qfree[qb]);  // scores read, merge data written
      u += ntiles;
      s = s_nx;
      continue;
    }
    // ---- merge the four warps: (m, l) per head, O per (head, d) ----
#pragma unroll
    for (int h = 0; h < NH; ++h)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) l[h] += __shfl_xor_sync(0xffffffffu, l[h], o);
    if (lane == 0) {
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        mrg_ml[(warp * kMaxGroup + h) * 2 + 0] = m[h];
        mrg_ml[(warp * kMaxGroup + h) * 2 + 1] = l[h];
      }
    }
    const int nb = cum[s.b + 1] - cum[s.b];
    const bool complete = (s.t0 == 0) && (s.t1 == nb);
    const int slot_id = (u == u0) ? 0 : 1;
    float *part = a.partials + (static_cast<int64_t>(blockIdx.x) * 2 + slot_id) * kSlotFloats;
    for (int hp = 0; hp < G; hp += C::kMH) {  // kMH heads per pass
#pragma unroll
      for (int e = 0; e < C::kMH; ++e) {
        const int hd = hp + e;  // held by the lanes with c = hd / 2, accumulator column hd % 2
        if (hd < G && (hd >> 1) == c) {
          float2 *dst = reinterpret_cast<float2 *>(mrg_o + (warp * C::kMH + e) * kD + 16 * r);
#pragma unroll
          for (int j = 0; j < 8; ++j) dst[j] = make_float2(st.o[j][hd & 1], st.o[j][2 + (hd & 1)]);
        }
      }
      named_bar_sync(1, kConsumerWarps * 32);
      if (tid < C::kMH && hp + tid < G) {  // per head: M, the warps' factors 2^(m_w - M) (over m_w), l
        const int hd = hp + tid;
        float M = kNoMax;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mrg_ml[(w * kMaxGroup + hd) * 2]);
        float lsum = 0.0f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float f = ex2(mrg_ml[(w * kMaxGroup + hd) * 2] - M);  // warps without tokens: 0
          lsum += f * mrg_ml[(w * kMaxGroup + hd) * 2 + 1];
          mrg_ml[(w * kMaxGroup + hd) * 2] = f;
        }
        mrg_hd[2 * hd] = M;
        mrg_hd[2 * hd + 1] = lsum;
      }
      named_bar_sync(1, kConsumerWarps * 32);
      for (int e2 = tid; e2 < C::kMH * kD; e2 += kConsumerWarps * 32) {
        const int e = e2 / kD, d = e2 % kD, hd = hp + e;
        if (hd < G) {
          float o = 0.0f;
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) o += mrg_ml[(w * kMaxGroup + hd) * 2] * mrg_o[(w * C::kMH + e) * kD + d];
          const float lsum = mrg_hd[2 * hd + 1];
          if (complete) {
            a.out[(static_cast<int64_t>(s.b) * a.Hq + s.h * G + hd) * kD + d] = __float2bfloat16_rn(o * (vscale / lsum));
          } else {
            part[hd * kD + d] = o;
            if (d == 0) {
              part[kMaxGroup * kD + hd] = mrg_hd[2 * hd];
              part[kMaxGroup * kD + kMaxGroup + hd] = lsum;
            }
          }
        }
      }
      if (!complete) __threadfence();  // this thread's part of the partial, visible before the arrival
      named_bar_sync(1, kConsumerWarps * 32);
    }
    if (!complete && tid == 0)
      split_arrive<WT>(a, cum, s, W, NC, reinterpret_cast<const int *>(smem + C::oStarts), npend, npend + 1);
    if (lane == 0) mbar_arrive(&qfree[qb]);  // every score of this segment was read: its image may be reused
    u += ntiles;
    s = s_nx;
  }
}

// ---------------------------------------------------------------------------
// Split-KV merge (log-sum-exp rule) of one (sequence, KV head) whose parts
// have all arrived, by every thread of the CTA that arrived last.
// Contributor k left (o_k, m_k, l_k) in log2 units; out = sum_k 2^(m_k - M)
// o_k / sum_k 2^(m_k - M) l_k * g_V, M = max_k m_k.  A thread takes one
// output element (head, value) and folds the parts in contributor order,
// loading a batch of contributors at once (one round trip per batch); the
// result does not depend on which CTA arrived last.
// ---------------------------------------------------------------------------
constexpr int kMergeBatch = 8;  // contributors whose loads are in flight together

__device__ void final_merge(const DecodeArgs &a, const int *rec) {
  const int b = rec[0], h = rec[1], n = rec[2], c_first = rec[3] >> 1, slot0 = rec[3] & 1;
  const float vscale = a.c.scale[1];
  __threadfence();  // the other contributors' parts were published before their arrivals
  for (int e = threadIdx.x; e < a.G * kD; e += kThreads) {
    const int hd = e / kD, d = e % kD;
    float M = -INFINITY, L = 0.0f, acc = 0.0f;
    for (int k0 = 0; k0 < n; k0 += kMergeBatch) {
      float m[kMergeBatch], l[kMergeBatch], o[kMergeBatch];
#pragma unroll
      for (int q = 0; q < kMergeBatch; ++q) {
        const int k = k0 + q;
        if (k < n) {
          const float *st = a.partials + (static_cast<int64_t>(c_first + k) * 2 + (k == 0 ? slot0 : 0)) * kSlotFloats;
          m[q] = __ldcg(st + kMaxGroup * kD + hd);
          l[q] = __ldcg(st + kMaxGroup * kD + kMaxGroup + hd);
          o[q] = __ldcg(st + hd * kD + d);
        } else {
          m[q] = -INFINITY;
          l[q] = 0.0f;
          o[q] = 0.0f;
        }
      }
      float mb = M;
#pragma unroll
      for (int q = 0; q < kMergeBatch; ++q) mb = fmaxf(mb, m[q]);
      const float r = M == -INFINITY ? 0.0f : ex2(M - mb);
      L *= r;
      acc *= r;
#pragma unroll
      for (int q = 0; q < kMergeBatch; ++q) {
        const float w = m[q] == -INFINITY ? 0.0f : ex2(m[q] - mb);
        L += w * l[q];
        acc += w * o[q];
      }
      M = mb;
    }
    a.out[(static_cast<int64_t>(b) * a.Hq + h * a.G + hd) * kD + d] = __float2bfloat16_rn(acc * (vscale / L));
  }
}

// ---------------------------------------------------------------------------
// The decode kernel: set-up, role dispatch, split-KV merges, teardown.
// ---------------------------------------------------------------------------
template <int PREC, int NH, bool WT>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const DecodeArgs a) {
  using C = Cfg<PREC, NH>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::oBars);
  uint64_t *empty = full + C::kStages;
  uint64_t *sready = empty + C::kStages;  // score buffer g holds a finished tile
  uint64_t *qready = sready + kGroups;    // query image q, its scale factors and score factors ready
  uint64_t *qfree = qready + kQBufs;      // every consumer warp finished the segment of image q
  uint64_t *mdone = qfree + kQBufs;       // the query warp merged a segment (async merge)
  int32_t *cum = reinterpret_cast<int32_t *>(smem + C::oCum);
  int *flags = reinterpret_cast<int *>(smem + C::oFlags);
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(flags);
  volatile int *abort = flags + 1;
  int *fills = flags + 2;  // fills issued per ring slot
  int *npend = flags + 6 + C::kStages;  // split pairs to merge at the end, then their records (oPend)
  int *arm_cnt = reinterpret_cast<int *>(smem + C::oArm);  // per group: warps that armed its tiles so far
  int *last_iss = arm_cnt + kGroups;                       // per group: the last tile whose MMAs went out

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hkv = a.c.Hkv, B = a.B;
  const int64_t cap = static_cast<int64_t>(a.max_pages) * a.c.P;

  // ---- set-up: barriers, TMEM, tiles per sequence -> prefix sums ----
  if (tid == 0) {
    flags[1] = 0;
    *npend = 0;
    for (int g = 0; g < kGroups; ++g) {
      arm_cnt[g] = 0;
      last_iss[g] = -1;
    }
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kGroupWarps);  // the four warps of the tile's group read it
      fills[s] = 0;
    }
    for (int b = 0; b < kGroups; ++b) {
      mbar_init(&sready[b], 1);
    }
    for (int q = 0; q < kQBufs; ++q) {
      mbar_init(&qready[q], 2);  // TMEM copies done + image written
      mbar_init(&qfree[q], kConsumerWarps);
    }
    {
      mbar_init(mdone, 1);
    }
    fence_mbar_init();
  }
  if (warp == kQueryWarp) tmem_alloc(tmem_holder, C::kTmemCols);
  // Launched as a programmatic dependent of the previous kernel on the
  // stream: everything above touches only this CTA's shared memory and TMEM;
  // every global access below waits for that kernel to complete.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // every sequence length in flight at once (one load per thread), then the
  // prefix sums by warp 0 from shared memory
  for (int b = tid; b < B; b += kThreads) cum[b + 1] = a.seq_lens[b];
  __syncthreads();
  if constexpr (WT) {
    // Prefix sums, kThreads sequences per pass: a scan within each warp, then
    // over the warps' totals (in the merge scratch, which only the set-up
    // uses at this point).  Then thread c finds the start of share c on the
    // virtual line (thread NC: W).
    int *wsum = reinterpret_cast<int *>(smem + C::oMrgO);
    if (tid == 0) cum[0] = 0;
    int carry = 0, nonempty = 0;  // tiles and sequences with tiles so far
    for (int base = 0; base < B; base += kThreads) {
      const int b = base + tid;
      int n = 0;
      if (b < B) {
        int64_t Lb = cum[b + 1];
        if (Lb < 0 || Lb > cap) {
          if (blockIdx.x == 0) set_err(a.c.err, NVKV_DEVERR_SEQLEN);
          Lb = Lb < 0 ? 0 : cap;
        }
        n = static_cast<int>((Lb + kTile - 1) / kTile);
        reinterpret_cast<uint8_t *>(cum + kMaxBatch + 1)[b] = static_cast<uint8_t>(Lb - (n > 0 ? (n - 1) * kTile : 0));
      }
      int incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) wsum[warp] = incl;
      nonempty += __syncthreads_count(n > 0);
      int wv = lane < kThreads / 32 ? wsum[lane] : 0;  // the warps' totals, scanned
#pragma unroll
      for (int o = 1; o < kThreads / 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, wv, o);
        if (lane >= o) wv += y;
      }
      const int before = warp > 0 ? __shfl_sync(0xffffffffu, wv, warp - 1) : 0;
      if (b < B) cum[b + 1] = carry + before + incl;
      carry += __shfl_sync(0xffffffffu, wv, kThreads / 32 - 1);
      __syncthreads();  // the totals are read before the next pass writes them
    }
    // never more shares than units, so a share is at least one tile long on
    // the virtual line (see tile_at)
    const int64_t W = static_cast<int64_t>(carry) * Hkv;
    const int NC = static_cast<int>(W < a.num_ctas ? (W > 0 ? W : 1) : a.num_ctas);
    const int64_t vk = static_cast<int64_t>(nonempty) * Hkv >= kVPairMin * NC ? kVPair : 0;
    int *starts = reinterpret_cast<int *>(smem + C::oStarts);
    if (tid <= NC) {
      int64_t st = 0;
      if (W > 0 && tid == NC) st = W;
      else if (W > 0 && vk == 0) st = div_small(tid * W, NC);
      else if (W > 0) st = tile_at(div_small(tid * (kVTile * W + vk * static_cast<int64_t>(B) * Hkv), NC), cum, B, Hkv, vk);
      starts[tid] = static_cast<int>(st);
    }
    __syncthreads();
    if (tid == 0) {
      const bool active = static_cast<int>(blockIdx.x) < NC;
      int *sh = flags + 2 + C::kStages;
      sh[0] = static_cast<int>(W);
      sh[1] = NC;
      sh[2] = active ? starts[blockIdx.x] : 0;
      sh[3] = active ? starts[blockIdx.x + 1] : 0;
    }
  } else {
    if (warp == 0) {
      int carry = 0;
      if (lane == 0) cum[0] = 0;
      for (int base = 0; base < B; base += 32) {
        const int b = base + lane;
        int n = 0;
        if (b < B) {
          int64_t Lb = cum[b + 1];
          if (Lb < 0 || Lb > cap) {
            if (blockIdx.x == 0) set_err(a.c.err, NVKV_DEVERR_SEQLEN);
            Lb = Lb < 0 ? 0 : cap;
          }
          n = static_cast<int>((Lb + kTile - 1) / kTile);
          reinterpret_cast<uint8_t *>(cum + kMaxBatch + 1)[b] = static_cast<uint8_t>(Lb - (n > 0 ? (n - 1) * kTile : 0));
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
      if (lane == 0) {  // this CTA's share of the units, computed once
        // never more shares than units: every active CTA owns at least one unit,
        // which the contributor count of the merge relies on
        const int64_t W = static_cast<int64_t>(carry) * Hkv;
        const int64_t NC = W < a.num_ctas ? (W > 0 ? W : 1) : a.num_ctas;
        const bool active = blockIdx.x < NC;
        int *sh = flags + 2 + C::kStages;
        sh[0] = static_cast<int>(W);
        sh[1] = static_cast<int>(NC);
        sh[2] = active ? static_cast<int>(share_begin(blockIdx.x, W, NC)) : 0;
        sh[3] = active ? static_cast<int>(share_begin(blockIdx.x + 1, W, NC)) : 0;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  const int *sh = flags + 2 + C::kStages;
  const int64_t W = sh[0], NC = sh[1], u0 = sh[2], u1 = sh[3];

  // zero rows of empty sequences (spread over CTAs)
  for (int b = blockIdx.x; b < B; b += a.num_ctas) {
    if (cum[b + 1] == cum[b]) {
      uint4 *o = reinterpret_cast<uint4 *>(a.out + static_cast<int64_t>(b) * a.Hq * kD);
      for (int i = tid; i < a.Hq * kD / 8; i += kThreads) o[i] = make_uint4(0, 0, 0, 0);
    }
  }

  int64_t last_issued = -1;  // query warp: the images it prepared
  if (warp >= kProducerWarp && warp < kProducerWarp + kGroups) {
    producer<PREC, NH>(a, smem + C::oRing, full, empty, cum, u0, u1, warp - kProducerWarp, abort, fills);
  } else if (warp == kQueryWarp) {
    const float kscale = __fmul_rn(a.c.scale[0], a.sm_scale * 1.4426950408889634f);
    last_issued = query_role<PREC, NH, WT>(a, smem, tmem, qready, qfree, mdone, cum, u0, u1, W, NC, abort, kscale, npend);
  } else {
    consumer_role<PREC, NH, WT>(a, smem, tmem, full, empty, sready, qready, qfree, mdone, cum, u0, u1, W, NC, abort,
                            arm_cnt, last_iss, npend);
  }

  // the next kernel on the stream may start its set-up
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  if (!*abort) {  // split pairs whose last part arrived from this CTA
    const int np = min(*npend, 2);
    for (int r = 0; r < np; ++r) final_merge(a, npend + 1 + 4 * r);
  } else {  // after a timeout, wait (bounded) for copies and MMAs still in flight
    if (tid == 0) set_err(a.c.err, NVKV_DEVERR_TIMEOUT);
    volatile int never = 0;
    if (tid == kProducerWarp * 32) {
      for (int s = 0; s < C::kStages; ++s)
        if (fills[s] > 0) mbar_wait_bounded(&full[s], static_cast<uint32_t>(fills[s] - 1) & 1u, &never);
    }
    if (warp < kConsumerWarps && warp % kGroupWarps == 0 && lane == 0) {  // the group's last score MMAs
      const int li = last_iss[warp / kGroupWarps];
      if (li >= 0) mbar_wait_bounded(&sready[warp / kGroupWarps], static_cast<uint32_t>(li / kGroups) & 1u, &never);
    }
    if (tid == kQueryWarp * 32 && last_issued > 0) {  // the query warp's last image (its TMEM copies)
      const int q = static_cast<int>((last_issued - 1) % kQBufs);
      mbar_wait_bounded(&qready[q], static_cast<uint32_t>((last_issued - 1) / kQBufs) & 1u, &never);
    }
  }
  if (warp == kQueryWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
struct DevInfo {
  int sms = 0;
  int occ[2][2] = {};  // [precision][heads per group slot set: 4, 8]
};

DevInfo g_info[64];
std::once_flag g_once[64];

// Resident CTAs per SM, from the kernel's shared memory, registers and TMEM
// columns.  (The runtime's occupancy query reports one CTA per SM for every
// kernel that allocates TMEM, whatever its resources; two of these CTAs do
// fit and run side by side.)
template <int PREC, int NH>
int occupancy_for(int dev) {
  const int smem = Cfg<PREC, NH>::kSmem;
  if (cudaFuncSetAttribute(decode_kernel<PREC, NH, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
          cudaSuccess ||
      cudaFuncSetAttribute(decode_kernel<PREC, NH, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Cfg<PREC, NH>::kSmemW) != cudaSuccess)
    return 0;
  // two CTAs of ~110 KB per SM need the largest shared-memory carveout
  if (cudaFuncSetAttribute(decode_kernel<PREC, NH, false>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
      cudaFuncSetAttribute(decode_kernel<PREC, NH, true>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared) != cudaSuccess)
    return 0;
  // (the weighted-share kernel holds kSmemW - kSmem bytes more: one CTA per SM either way)
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, decode_kernel<PREC, NH, false>) != cudaSuccess) return 0;
  int sm_smem = 0, reserved = 0, sm_regs = 0, sm_threads = 0;
  cudaDeviceGetAttribute(&sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
  cudaDeviceGetAttribute(&sm_regs, cudaDevAttrMaxRegistersPerMultiprocessor, dev);
  cudaDeviceGetAttribute(&sm_threads, cudaDevAttrMaxThreadsPerMultiProcessor, dev);
  const int by_smem = sm_smem / (smem + static_cast<int>(fa.sharedSizeBytes) + reserved);
  const int warp_regs = (fa.numRegs * 32 + 255) / 256 * 256;  // allocation unit: 256 registers per warp
  const int by_regs = warp_regs > 0 ? sm_regs / (warp_regs * (kThreads / 32)) : 0;
  const int by_threads = sm_threads / kThreads;
  const int by_tmem = static_cast<int>(512 / Cfg<PREC, NH>::kTmemCols);  // TMEM columns per SM
  int n = by_smem;
  n = by_regs < n ? by_regs : n;
  n = by_threads < n ? by_threads : n;
  n = by_tmem < n ? by_tmem : n;
  return n;
}

const DevInfo *dev_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::call_once(g_once[dev], [dev] {
    DevInfo &d = g_info[dev];
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    d.occ[0][0] = occupancy_for<NVKV_PREC_NVFP4, 4>(dev);
    d.occ[0][1] = occupancy_for<NVKV_PREC_NVFP4, 8>(dev);
    d.occ[1][0] = occupancy_for<NVKV_PREC_FP8_E4M3, 4>(dev);
    d.occ[1][1] = occupancy_for<NVKV_PREC_FP8_E4M3, 8>(dev);
  });
  return g_info[dev].sms > 0 ? &g_info[dev] : nullptr;
}

// CTAs of the persistent grid, one share each: as many as are resident at
// once on the device, and with num_splits > 0 at most batch * Hkv *
// num_splits (equal-length sequences are then cut into exactly num_splits
// shares each while that fits in one wave; more shares than resident CTAs
// would only add waves of set-up and merging, so the request is capped there).
int64_t num_ctas_for(int prec, int32_t batch, int32_t Hkv, int32_t G, int64_t max_units, int32_t num_splits) {
  const DevInfo *d = dev_info();
  int64_t n;
  if (num_splits > 0) {
    n = static_cast<int64_t>(batch) * Hkv * num_splits;
    if (d) {
      const int o = d->occ[prec][G > 4 ? 1 : 0];
      const int64_t wave = static_cast<int64_t>(d->sms) * (o > 0 ? o : 1);
      if (wave < n) n = wave;
    }
  } else {
    if (!d) return -1;
    const int o = d->occ[prec][G > 4 ? 1 : 0];
    n = static_cast<int64_t>(d->sms) * (o > 0 ? o : 1);
  }
  if (n > max_units) n = max_units;
  if (n > kMaxShares) n = kMaxShares;
  return n < 1 ? 1 : n;
}

// Workspace = an arrival counter per (sequence, KV head) + two partial slots per CTA.
size_t counter_bytes(int32_t batch, int32_t Hkv) { return (static_cast<size_t>(batch) * Hkv * 4 + 255) / 256 * 256; }

size_t workspace_bytes_for(int32_t batch, int32_t Hkv, int64_t nctas) {
  return counter_bytes(batch, Hkv) + static_cast<size_t>(nctas) * 2 * kSlotFloats * sizeof(float);
}

// Programmatic dependent launch: the grid may start while the previous kernel
// on the stream finishes (its set-up overlaps that kernel's tail); the kernel
// waits for it before touching global memory.
template <int PREC, int NH, bool WT>
void launch_decode(const DecodeArgs &a, cudaStream_t s) {
  constexpr int smem = WT ? Cfg<PREC, NH>::kSmemW : Cfg<PREC, NH>::kSmem;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.num_ctas));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, decode_kernel<PREC, NH, WT>, a) != cudaSuccess) {
    cudaGetLastError();  // clear, then an ordinary stream-ordered launch
    decode_kernel<PREC, NH, WT><<<static_cast<unsigned>(a.num_ctas), kThreads, smem, s>>>(a);
  }
}

nvkv_status decode_common(const void *q, const nvkv_cache *cache, const int32_t *block_table, int32_t max_pages,
                          const int32_t *seq_lens, int32_t batch, int32_t num_q_heads, int32_t prec, float sm_scale,
                          int32_t num_splits, void *workspace, size_t workspace_bytes, void *out, void *stream,
                          const void *k_new = nullptr, const void *v_new = nullptr,
                          nvkv_dtype new_dtype = NVKV_DTYPE_F32) {
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
  if (max_units > 0x7fffffff) return NVKV_ERR_UNSUPPORTED;  // unit indices are 32-bit in the kernel
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
  a.counters = static_cast<uint32_t *>(workspace);
  a.partials = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + counter_bytes(batch, Hkv));
  a.out = static_cast<__nv_bfloat16 *>(out);
  a.k_new = k_new;
  a.v_new = v_new;
  a.new_dtype = new_dtype;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // shares weighted by pairs when the batch has many pairs per CTA
  const bool wt = static_cast<int64_t>(batch) * Hkv >= kVPairMin * nctas;
  if (prec == NVKV_PREC_NVFP4) {
    if (G <= 4) wt ? launch_decode<NVKV_PREC_NVFP4, 4, true>(a, s) : launch_decode<NVKV_PREC_NVFP4, 4, false>(a, s);
    else wt ? launch_decode<NVKV_PREC_NVFP4, 8, true>(a, s) : launch_decode<NVKV_PREC_NVFP4, 8, false>(a, s);
  } else {
    if (G <= 4) wt ? launch_decode<NVKV_PREC_FP8_E4M3, 4, true>(a, s) : launch_decode<NVKV_PREC_FP8_E4M3, 4, false>(a, s);
    else wt ? launch_decode<NVKV_PREC_FP8_E4M3, 8, true>(a, s) : launch_decode<NVKV_PREC_FP8_E4M3, 8, false>(a, s);
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
  NVKV_ABI_RANGE();
  if (!cache || layer_precision != cache->prec) return NVKV_ERR_INVALID_ARG;
  if (layer_precision != NVKV_PREC_NVFP4 && layer_precision != NVKV_PREC_FP8_E4M3) return NVKV_ERR_INVALID_ARG;
  nvkv_status st = check_cache(cache, layer_precision);
  if (st != NVKV_OK) return st;
  if (batch < 0 || batch > kMaxBatch) return batch < 0 ? NVKV_ERR_INVALID_ARG : NVKV_ERR_UNSUPPORTED;
  if (batch == 0) return NVKV_OK;
  if (num_q_heads <= 0 || num_q_heads % cache->num_kv_heads != 0) return NVKV_ERR_INVALID_ARG;
  // counters plus at least one CTA's two partial slots (refused before any CUDA call)
  const size_t cb = counter_bytes(batch, cache->num_kv_heads);
  if (cb + 2 * kSlotFloats * sizeof(float) > NVKV_NOALLOC_SCRATCH_BYTES) return NVKV_ERR_WORKSPACE_TOO_SMALL;
  void *scratch = noalloc_scratch_ptr();
  if (!scratch) return NVKV_ERR_CUDA;
  // The arrival counters must start at zero.  A call cut short by a device
  // error can leave them otherwise, so every call clears them first (one
  // memset on the stream, no allocation); the partial slots need nothing.
  if (cudaMemsetAsync(scratch, 0, cb, static_cast<cudaStream_t>(stream)) != cudaSuccess) return NVKV_ERR_CUDA;
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
    for (int p = 0; p < 2; ++p) occ = d->occ[p][G > 4 ? 1 : 0] > occ ? d->occ[p][G > 4 ? 1 : 0] : occ;
    nctas = static_cast<int64_t>(d->sms) * occ;
  }
  return workspace_bytes_for(batch, num_kv_heads, nctas);
}

nvkv_status nvkv_decode_workspace_init(void *workspace, size_t bytes, void *stream) {
  NVKV_ABI_RANGE();
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
  NVKV_ABI_RANGE();
  if (!cache || layer_precision != cache->prec) return NVKV_ERR_INVALID_ARG;
  if (layer_precision != NVKV_PREC_NVFP4 && layer_precision != NVKV_PREC_FP8_E4M3) return NVKV_ERR_INVALID_ARG;
  return decode_common(q, cache, block_table, max_pages, seq_lens, batch, num_q_heads, layer_precision, sm_scale,
                       num_splits, workspace, workspace_bytes, out, stream);
}

nvkv_status nvfp4_paged_decode_step(const void *q, const void *k_new, const void *v_new, nvkv_dtype dtype,
                                    const nvkv_cache *cache, const int32_t *block_table, int32_t max_pages,
                                    const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                                    int32_t layer_precision, float sm_scale, int32_t num_splits, void *workspace,
                                    size_t workspace_bytes, void *out, void *stream) {
  NVKV_ABI_RANGE();
  if (!cache || layer_precision != cache->prec) return NVKV_ERR_INVALID_ARG;
  if (layer_precision != NVKV_PREC_NVFP4 && layer_precision != NVKV_PREC_FP8_E4M3) return NVKV_ERR_INVALID_ARG;
  if (dtype != NVKV_DTYPE_F32 && dtype != NVKV_DTYPE_BF16) return NVKV_ERR_INVALID_ARG;
  if (batch > 0 && (!k_new || !v_new)) return NVKV_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new)) return NVKV_ERR_UNSUPPORTED;
  return decode_common(q, cache, block_table, max_pages, seq_lens, batch, num_q_heads, layer_precision, sm_scale,
                       num_splits, workspace, workspace_bytes, out, stream, k_new, v_new, dtype);
}

nvkv_status fp8_paged_decode_attention(const void *q, const nvkv_cache *cache, const int32_t *block_table,
                                       int32_t max_pages, const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                                       float sm_scale, int32_t num_splits, void *workspace, size_t workspace_bytes,
                                       void *out, void *stream) {
  NVKV_ABI_RANGE();
  return decode_common(q, cache, block_table, max_pages, seq_lens, batch, num_q_heads, NVKV_PREC_FP8_E4M3, sm_scale,
                       num_splits, workspace, workspace_bytes, out, stream);
}

}  // extern "C"
