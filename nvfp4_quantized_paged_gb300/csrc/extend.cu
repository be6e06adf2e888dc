// Chunked-extend attention over the shared FP8 workspace, and the append of
// the current chunk's K/V into that workspace (sm_103a).
//
// "SGLang x Qwen x NVIDIA Collaboration: NVFP4 KV Cache Breaks Long-Context
// and Agentic Inference Bottlenecks", section "Three Paths": for chunked
// prefill / extend the cached prefix is dequantized into an FP8 workspace that
// all layers share, the current chunk's KV is appended to it, and the chunk's
// queries run FP8 attention over both (causal inside the chunk).
//
// Two kernels per call.  extend_tiles_kernel expands the E4M3 workspace once
// into FP16 operand tiles in the tensor cores' K-major layout (K by 8-row
// groups, V transposed so that keys run along K); E4M3 -> FP16 is exact.
// Every M-tile of a (sequence, KV head) then reads the same tiles from L2
// instead of converting them again.
//
// extend_attention_kernel, work item (sequence, KV head, M-tile of 128 query
// rows): row r of an M-tile is query token r / G of the tile with query head
// h G + r % G, so the G query heads that share a KV head share every K/V
// tile.  Per tile of 128 keys, QK^T and P.V run on the tensor cores
// (tcgen05.mma kind::f16, M = N = 128, K = 16 per instruction, FP32
// accumulators in TMEM: scores in two ping-pong buffers, the output in a
// third); the softmax runs in the registers of the thread that owns the row's
// TMEM lane.  Roles (192 threads, one CTA per SM):
//   warps 0-3  the Q tile (BF16 -> FP16) once; then the softmax: thread r owns
//              query row r; base-2 online softmax with a lazily raised running
//              max, P to shared memory as FP16, the output rescaled in TMEM
//              when the max rises, the epilogue.
//   warp 4     producer: bulk copies of each tile's K (one 32 KB copy) and V^T
//              (sixteen 2 KB copies) into a double-buffered stage.
//   warp 5     one thread issues the MMAs.
// BF16 queries convert to FP16 exactly inside the FP16 normal range
// [2^-14, 65504].
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "nvfp4kv.h"
#include "nvkv_device.cuh"
#include "nvkv_host.h"

namespace nvkv {
namespace {

constexpr int kXD = 128;                 // head_dim
constexpr int kXRows = 128;              // query rows per half, keys per KV tile
constexpr int kXThreads = 352;           // 11 warps
constexpr int kXKProducerWarp = 8, kXVProducerWarp = 9, kXIssuerWarp = 10;
constexpr uint32_t kXTmemCols = 512;     // scores of half X at 128 X, its output at 256 + 128 X
constexpr int kXTile = kXRows * kXD * 2; // one FP16 operand tile (32 KB)
constexpr int kXSbo = 2048;              // bytes between 8-row groups of a tile
constexpr int kXGroupBytes = 8 * kXD * 2;  // one 8-row group of an FP16 operand tile (2 KB)
// Shared memory: Q[2 halves] | K | V^T[2 stages] | P[2 halves] | barriers | TMEM holder, abort flag, pick.
constexpr int oXQ = 0, oXK = 2 * kXTile, oXV = 3 * kXTile, oXP = 5 * kXTile, oXBar = 7 * kXTile;
// barriers: k_full k_free v_full[2] v_free[2] s_full[2] s_free[2] p_full[2] pv_done[2] fin q_full
constexpr int bKFull = 0, bKFree = 1, bVFull = 2, bVFree = 4, bSFull = 6, bSFree = 8, bPFull = 10, bPvDone = 12,
              bFin = 14, bQFull = 15, kXBars = 16;
constexpr int oXFlags = oXBar + 8 * kXBars;
constexpr int kXSmem = oXFlags + 16;
constexpr float kXNoMax = -1e30f;        // running max before any score (finite: exp2(-inf - m) = 0)
constexpr float kXRescale = 8.0f;        // raise the running max only when it grows by more than 2^8

struct ExtendArgs {
  const __nv_bfloat16 *q;
  const int64_t *cu_q;
  const uint8_t *ws_k, *ws_v;
  const int64_t *cu_kv;
  const int32_t *kv_lens;
  const float *ws_scale;
  __nv_bfloat16 *out;
  int32_t *err;
  const uint8_t *tiles;  // expanded FP16 operand tiles
  int64_t ngroups;       // 8-row groups per head in `tiles`
  int64_t ws_rows;
  int Hq, Hkv, G, lgG, Tm;
  float sm_scale;
};

// Byte offset of 16-byte chunk `chunk` (8 FP16 along K) of row `row` in a
// K-major operand tile without swizzle: 8-row x 16-byte core matrices, 128
// bytes apart along K, 2048 bytes between 8-row groups.
__device__ __forceinline__ uint32_t kmaj(int row, int chunk) {
  return static_cast<uint32_t>((row >> 3) * kXSbo + chunk * 128 + (row & 7) * 16);
}

__device__ __forceinline__ uint32_t f16x2_from_bf16x2(uint32_t w) {
  return pack_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ bool warp_wait_x(uint64_t *bar, uint32_t parity, volatile int *abort) {
  const bool ok = mbar_wait_bounded(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

struct Tile {            // the CTA's work item, uniform over the CTA
  int h;                 // KV head
  int64_t q0;            // first query row of the sequence in q / out
  int tok0;              // first chunk token of the CTA (half 0); half 1 starts Tm tokens later
  int ntok[2];           // valid tokens of each half (half 1 may have none)
  int L;                 // keys of the sequence (prefix + chunk)
  int p;                 // prefix length: chunk token t sits at position p + t
  int64_t kv_base;       // workspace row of position 0 (a multiple of 8)
  int ntiles;            // KV tiles that some row of the CTA sees
};

// ---------------------------------------------------------------------------
// The Q tile of half X, by that half's softmax warps before their loop.
// Thread r = (rb, dc): 8-row block rb, 16-element column chunk dc; rows
// 8 rb + (s + dc) % 8, so the eight threads of a store phase (dc = 0..7)
// write eight different rows of their core matrices: no bank conflicts.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void x_load_q(const ExtendArgs &a, const Tile &t, uint8_t *smem, int X) {
  const int ct = static_cast<int>(threadIdx.x) & 127;
  const int rb = ct >> 3, dc = ct & 7;
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  const int tbase = t.tok0 + X * a.Tm;
  const int ntok = X ? t.ntok[1] : t.ntok[0];
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int r = 8 * rb + ((s + dc) & 7);
    const int tok = r >> a.lgG, g = r & (a.G - 1);
    uint4 lo = zero, hi = zero;
    if (tok < ntok) {
      const uint4 *src = reinterpret_cast<const uint4 *>(
          a.q + ((t.q0 + tbase + tok) * a.Hq + static_cast<int64_t>(t.h) * a.G + g) * kXD + 16 * dc);
      lo = src[0];
      hi = src[1];
    }
    uint8_t *dst = smem + oXQ + X * kXTile + kmaj(r, 2 * dc);
    *reinterpret_cast<uint4 *>(dst) = make_uint4(f16x2_from_bf16x2(lo.x), f16x2_from_bf16x2(lo.y),
                                                 f16x2_from_bf16x2(lo.z), f16x2_from_bf16x2(lo.w));
    *reinterpret_cast<uint4 *>(dst + 128) = make_uint4(f16x2_from_bf16x2(hi.x), f16x2_from_bf16x2(hi.y),
                                                       f16x2_from_bf16x2(hi.z), f16x2_from_bf16x2(hi.w));
  }
}

// ---------------------------------------------------------------------------
// Producers.  Tile j = keys [128 j, 128 j + 128) of the sequence = row groups
// g0 .. g0 + 15, g0 = (cu_kv + 128 j) / 8, of the expanded tiles.
//   warp 8: K as one 32 KB copy into the single K buffer, once both halves'
//           QK^T of tile j - 1 are done (its latency hides behind the
//           softmax of tile j - 1);
//   warp 9: V^T as one 2 KB copy per 8-value group d (lane d) into stage
//           j % 2, once both halves' P.V of tile j - 2 are done (v_free), so
//           the P.V of tile j never waits for its copy.
// Each returns the number of tiles whose copies it issued.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int x_produce_k(const ExtendArgs &a, const Tile &t, uint8_t *smem, uint64_t *bars,
                                           volatile int *abort) {
  const int lane = static_cast<int>(threadIdx.x) & 31;
  const uint64_t policy = policy_evict_last();
  const uint8_t *kt = a.tiles + static_cast<int64_t>(t.h) * a.ngroups * kXGroupBytes;
  int issued = 0;
  for (int j = 0; j < t.ntiles; ++j) {
    if (j >= 1 && !warp_wait_x(&bars[bKFree], static_cast<uint32_t>(j - 1) & 1u, abort)) break;
    const int64_t g0 = (t.kv_base + static_cast<int64_t>(j) * kXRows) >> 3;
    if (lane == 0) {
      mbar_arrive_expect_tx(&bars[bKFull], kXTile);
      bulk_g2s(smem + oXK, kt + g0 * kXGroupBytes, kXTile, &bars[bKFull], policy);
    }
    __syncwarp();
    ++issued;
  }
  return issued;
}

__device__ __forceinline__ int x_produce_v(const ExtendArgs &a, const Tile &t, uint8_t *smem, uint64_t *bars,
                                           volatile int *abort) {
  const int lane = static_cast<int>(threadIdx.x) & 31;
  const uint64_t policy = policy_evict_last();
  const uint8_t *vt = a.tiles + (static_cast<int64_t>(a.Hkv) + t.h) * a.ngroups * kXGroupBytes;
  int issued = 0;
  for (int j = 0; j < t.ntiles; ++j) {
    const int b = j & 1;
    if (j >= 2 && !warp_wait_x(&bars[bVFree + b], static_cast<uint32_t>((j - 2) >> 1) & 1u, abort)) break;
    const int64_t g0 = (t.kv_base + static_cast<int64_t>(j) * kXRows) >> 3;
    if (lane == 0) mbar_arrive_expect_tx(&bars[bVFull + b], kXTile);
    __syncwarp();
    if (lane < 16)
      bulk_g2s(smem + oXV + b * kXTile + lane * kXGroupBytes, vt + (lane * a.ngroups + g0) * 128, kXGroupBytes,
               &bars[bVFull + b], policy);
    ++issued;
  }
  return issued;
}

// ---------------------------------------------------------------------------
// Expanded tiles: tiles = [K: Hkv][ngroups][2048 B] [V: Hkv][16][ngroups][128 B].
// K group (h, g): 16-byte chunk c (values 8c .. 8c + 7) of row r (key 8g + r)
// at c * 128 + r * 16.  V run (h, d, g): value row e (value 8d + e), keys 8g ..
// 8g + 7 at e * 16 + 2 r.  Rows at or past ws_rows are zero; an E4M3 NaN byte
// (never written by this library) becomes -448 so that masked keys stay finite.
// One thread per (g, h, d): an 8 x 8 byte block of the workspace.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t f16x2_finite(uint32_t h2) {
  return __hmax2_as_u32(h2, 0xDF00DF00u);  // max(x, -448): NaN -> -448, every E4M3 value unchanged
}

__global__ void __launch_bounds__(256) extend_tiles_kernel(const uint8_t *__restrict__ ws_k,
                                                           const uint8_t *__restrict__ ws_v, int64_t ws_rows,
                                                           int Hkv, int64_t ngroups, uint8_t *__restrict__ tiles) {
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= ngroups * Hkv * 16) return;
  const int d = static_cast<int>(gid & 15);
  const int h = static_cast<int>((gid >> 4) % Hkv);
  const int64_t g = (gid >> 4) / Hkv;
  uint32_t kw[8][2], vw[8][2];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int64_t row = 8 * g + r;
    uint2 x = make_uint2(0u, 0u), y = x;
    if (row < ws_rows) {
      x = *reinterpret_cast<const uint2 *>(ws_k + (row * Hkv + h) * kXD + 8 * d);
      y = *reinterpret_cast<const uint2 *>(ws_v + (row * Hkv + h) * kXD + 8 * d);
    }
    kw[r][0] = x.x;
    kw[r][1] = x.y;
    vw[r][0] = y.x;
    vw[r][1] = y.y;
  }
  uint8_t *kdst = tiles + (static_cast<int64_t>(h) * ngroups + g) * kXGroupBytes + d * 128;
#pragma unroll
  for (int r = 0; r < 8; ++r)
    *reinterpret_cast<uint4 *>(kdst + r * 16) =
        make_uint4(f16x2_finite(f16x2_from_e4m3x2<0>(kw[r][0])), f16x2_finite(f16x2_from_e4m3x2<1>(kw[r][0])),
                   f16x2_finite(f16x2_from_e4m3x2<0>(kw[r][1])), f16x2_finite(f16x2_from_e4m3x2<1>(kw[r][1])));
  uint8_t *vdst = tiles + ((static_cast<int64_t>(Hkv) + h) * ngroups * kXGroupBytes) +
                  (static_cast<int64_t>(d) * ngroups + g) * 128;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const uint32_t sel = static_cast<uint32_t>(e & 3) | (static_cast<uint32_t>(4 + (e & 3)) << 4);
    uint32_t o[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      o[u] = f16x2_finite(f16x2_from_e4m3x2<0>(prmt(vw[2 * u][e >> 2], vw[2 * u + 1][e >> 2], sel)));
    *reinterpret_cast<uint4 *>(vdst + e * 16) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// ---------------------------------------------------------------------------
// Softmax of half X (warps 4X .. 4X + 3): thread r owns TMEM lane r = row r
// of the half.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void x_softmax(const ExtendArgs &a, const Tile &t, uint8_t *smem, uint32_t tmem,
                                          uint64_t *bars, int X, volatile int *abort) {
  const int r = static_cast<int>(threadIdx.x) & 127, quad = r >> 5;
  const int tok = r >> a.lgG, g = r & (a.G - 1);
  const int tbase = t.tok0 + X * a.Tm;
  const int ntok = X ? t.ntok[1] : t.ntok[0];
  const int nt = ntok > 0 ? ntok : 1;
  const int qpos = t.p + tbase + (tok < nt ? tok : nt - 1);  // sees positions [0, qpos]
  const float c2 = a.ws_scale[0] * a.sm_scale * 1.4426950408889634f;  // score -> log2 units
  const uint32_t lanes = tmem + (static_cast<uint32_t>(32 * quad) << 16);
  const uint32_t scol = static_cast<uint32_t>(X * 128), ocol = static_cast<uint32_t>(256 + X * 128);
  const int first_partial = t.p + tbase;  // the smallest position of the half
  uint64_t *s_full = &bars[bSFull + X], *s_free = &bars[bSFree + X], *p_full = &bars[bPFull + X];
  uint64_t *pv_done = &bars[bPvDone + X];
  uint8_t *ps = smem + oXP + X * kXTile;
  float m = kXNoMax, mt = kXNoMax, l = 0.0f;
  bool ok = true;
  for (int j = 0; j < t.ntiles; ++j) {
    const int kv0 = j * kXRows;
    ok = warp_wait_x(s_full, static_cast<uint32_t>(j) & 1u, abort);
    if (!ok) break;
    tc_fence_after();
    // the row's 128 scores: eight loads in flight, one wait
    uint32_t v[8][16];
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) tmem_ld16_async(lanes + scol + 16 * ch, v[ch]);
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int ch = 0; ch < 8; ++ch)
#pragma unroll
      for (int e = 0; e < 16; ++e) asm volatile("" : "+r"(v[ch][e]));
    tc_fence_before();
    mbar_arrive(s_free);  // this half's score buffer may take the next tile
    if (kv0 + kXRows - 1 > first_partial) {  // a diagonal tile (uniform): mask columns past the row's position
      const int lim = qpos - kv0;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch)
#pragma unroll
        for (int e = 0; e < 16; ++e)
          if (16 * ch + e > lim) v[ch][e] = __float_as_uint(-INFINITY);
    }
    float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int ch = 0; ch < 8; ++ch)
#pragma unroll
      for (int e = 0; e < 16; ++e) mq[e & 3] = fmaxf(mq[e & 3], __uint_as_float(v[ch][e]));
    const float mx2 = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * c2;
    float alpha = 1.0f;
    const bool need = mx2 > mt;
    if (need) {
      alpha = ex2(m - mx2);
      m = mx2;
      mt = mx2 + kXRescale;
      l *= alpha;
    }
    // P and the output of this half are free once its previous P.V is done
    if (j >= 1) {
      ok = warp_wait_x(pv_done, static_cast<uint32_t>(j - 1) & 1u, abort);
      if (!ok) break;
      tc_fence_after();
      if (__any_sync(0xffffffffu, need)) {  // rescale the output rows whose max rose (warp-uniform)
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          float o[16];
          tmem_ld16(lanes + ocol + 16 * ch, o);
#pragma unroll
          for (int e = 0; e < 16; ++e) o[e] *= alpha;
          tmem_st16(lanes + ocol + 16 * ch, o);
        }
        tmem_st_wait();
      }
    }
    const float nm = -m;
    float la[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
      uint32_t pk[8];
#pragma unroll
      for (int e = 0; e < 16; e += 2) {
        float a0, a1;
        fma_f32x2(a0, a1, __uint_as_float(v[ch][e]), __uint_as_float(v[ch][e + 1]), c2, c2, nm, nm);
        const float p0 = ex2(a0), p1 = ex2(a1);  // masked: exp2(-inf) = 0
        add_f32x2(la[(e >> 1) & 2], la[((e >> 1) & 2) + 1], p0, p1);
        pk[e / 2] = pack_f16x2(p0, p1);
      }
      *reinterpret_cast<uint4 *>(ps + kmaj(r, 2 * ch)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      *reinterpret_cast<uint4 *>(ps + kmaj(r, 2 * ch + 1)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
    }
    l += (la[0] + la[1]) + (la[2] + la[3]);
    fence_proxy_async_smem();
    tc_fence_before();
    mbar_arrive(p_full);
  }
  if (ok) ok = warp_wait_x(pv_done, static_cast<uint32_t>(t.ntiles - 1) & 1u, abort);
  if (!ok) return;
  tc_fence_after();
  const float inv = a.ws_scale[1] / l;
  const bool write = tok < ntok;
  __nv_bfloat16 *dst = a.out + ((t.q0 + tbase + tok) * a.Hq + static_cast<int64_t>(t.h) * a.G + g) * kXD;
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    float o[16];
    tmem_ld16(lanes + ocol + 16 * ch, o);
    uint32_t w[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const __nv_bfloat162 v2 = __floats2bfloat162_rn(o[2 * e] * inv, o[2 * e + 1] * inv);
      w[e] = *reinterpret_cast<const uint32_t *>(&v2);
    }
    if (write) {
      *reinterpret_cast<uint4 *>(dst + 16 * ch) = make_uint4(w[0], w[1], w[2], w[3]);
      *reinterpret_cast<uint4 *>(dst + 16 * ch + 8) = make_uint4(w[4], w[5], w[6], w[7]);
    }
  }
}

// ---------------------------------------------------------------------------
// MMA issuer (one thread of warp 10), polling four in-order streams:
//   QK_0(j), QK_1(j): S_X = Q_X K_j^T once K_j landed and half X's softmax has
//                     read S_X of tile j - 1 (QK_0(j) before QK_1(j); the
//                     commit after QK_1(j) frees the K buffer);
//   PV_0(j), PV_1(j): O_X += P_X V_j once P_X is written and V_j landed
//                     (PV_0(j) before PV_1(j); the commit after PV_1(j) frees
//                     V^T stage j % 2).
// The tensor cores so run one half's MMAs while the other half's softmax runs.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void x_issuer(uint8_t *smem, uint32_t tmem, int ntiles, uint64_t *bars,
                                         volatile int *abort) {
  const uint32_t qs = smem_u32(smem + oXQ), ps = smem_u32(smem + oXP), vts = smem_u32(smem + oXV);
  constexpr uint32_t id = idesc_f16(kXRows);
  int nqk[2] = {0, 0}, npv[2] = {0, 0};  // next tile whose QK^T / P.V of half X goes out
  uint64_t t_last = global_timer_ns();
  while (npv[1] < ntiles) {
    bool did = false;
#pragma unroll
    for (int X = 0; X < 2; ++X) {
      const int j = nqk[X];
      if (j < ntiles && (X == 0 || j < nqk[0]) && mbar_test(&bars[bKFull], static_cast<uint32_t>(j) & 1u) &&
          (j == 0 || mbar_test(&bars[bSFree + X], static_cast<uint32_t>(j - 1) & 1u))) {
        tc_fence_after();
        const uint32_t ks = smem_u32(smem + oXK);
#pragma unroll
        for (int kk = 0; kk < kXD / 16; ++kk)
          umma_f16(tmem + static_cast<uint32_t>(X * 128), umma_desc(qs + X * kXTile + kk * 256, 128, kXSbo),
                   umma_desc(ks + kk * 256, 128, kXSbo), id, kk > 0 ? 1u : 0u);
        umma_commit(&bars[bSFull + X]);
        if (X == 1) umma_commit(&bars[bKFree]);
        ++nqk[X];
        did = true;
      }
    }
#pragma unroll
    for (int X = 0; X < 2; ++X) {
      const int j = npv[X];
      if (j < nqk[X] && (X == 0 || j < npv[0]) && mbar_test(&bars[bPFull + X], static_cast<uint32_t>(j) & 1u) &&
          mbar_test(&bars[bVFull + (j & 1)], static_cast<uint32_t>(j >> 1) & 1u)) {
        tc_fence_after();
        const uint32_t vt = vts + static_cast<uint32_t>((j & 1) * kXTile);
#pragma unroll
        for (int kk = 0; kk < kXRows / 16; ++kk)
          umma_f16(tmem + static_cast<uint32_t>(256 + X * 128), umma_desc(ps + X * kXTile + kk * 256, 128, kXSbo),
                   umma_desc(vt + kk * 256, 128, kXSbo), id, (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&bars[bPvDone + X]);
        if (X == 1) umma_commit(&bars[bVFree + (j & 1)]);
        ++npv[X];
        did = true;
      }
    }
    if (did) {
      t_last = global_timer_ns();
    } else {
      if (*abort) return;
      if (global_timer_ns() - t_last > 2000000000ull) {  // no progress for 2 s
        *abort = 1;
        return;
      }
      __nanosleep(20);
    }
  }
}

__global__ void __launch_bounds__(kXThreads, 1) extend_attention_kernel(const ExtendArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = static_cast<int>(threadIdx.x), warp = tid >> 5;
  // Heaviest sequences first (the longest CTAs start in the first waves, the
  // tail holds short ones): with at most 64 sequences CTA row z takes the
  // sequence of rank z by length (ties by index); above that, index order.
  int i = static_cast<int>(blockIdx.z);
  const int n = static_cast<int>(gridDim.z);
  if (n > 1 && n <= 64) {
    int *pick = reinterpret_cast<int *>(smem + oXFlags + 8);
    if (warp == 0) {
      const int lane = tid & 31;
      int found = -1;
      for (int c = lane; c < n; c += 32) {
        const int Lc = a.kv_lens[c];
        int rank = 0;
        for (int j = 0; j < n; ++j) {
          const int Lj = a.kv_lens[j];
          rank += (Lj > Lc || (Lj == Lc && j < c)) ? 1 : 0;
        }
        if (rank == static_cast<int>(blockIdx.z)) found = c;
      }
      const unsigned m = __ballot_sync(0xffffffffu, found >= 0);
      const int src = m ? __ffs(m) - 1 : 0;
      const int v = __shfl_sync(0xffffffffu, found, src);
      if (lane == 0) *pick = m ? v : static_cast<int>(blockIdx.z);
    }
    __syncthreads();
    i = *pick;
  }
  Tile t;
  t.h = static_cast<int>(blockIdx.y);
  t.q0 = a.cu_q[i];
  const int64_t nq = a.cu_q[i + 1] - t.q0;
  t.L = a.kv_lens[i];
  t.kv_base = a.cu_kv[i];
  if (nq < 0 || nq > t.L || t.kv_base < 0 || t.kv_base + t.L > a.ws_rows || (t.kv_base & 7) != 0) {
    if (tid == 0 && blockIdx.x == 0 && t.h == 0)
      set_err(a.err, (nq < 0 || nq > t.L) ? NVKV_DEVERR_SEQLEN
                                          : ((t.kv_base & 7) != 0 ? NVKV_DEVERR_ALIGN : NVKV_DEVERR_WS_ROWS));
    return;
  }
  if (tid == 0 && blockIdx.x == 0 && t.h == 0 && nq > static_cast<int64_t>(gridDim.x) * 2 * a.Tm)
    set_err(a.err, NVKV_DEVERR_SEQLEN);  // more queries than max_q_len: the rest are not computed
  const int cta = static_cast<int>(gridDim.x - 1 - blockIdx.x);  // longest work items launch first
  t.tok0 = 2 * cta * a.Tm;
  if (t.tok0 >= nq) return;  // uniform: before any barrier or TMEM allocation
  const int rest = static_cast<int>(nq - t.tok0);
  t.ntok[0] = rest < a.Tm ? rest : a.Tm;
  t.ntok[1] = rest - t.ntok[0] < a.Tm ? rest - t.ntok[0] : a.Tm;
  t.p = t.L - static_cast<int>(nq);
  t.ntiles = (t.p + t.tok0 + t.ntok[0] + t.ntok[1] + kXRows - 1) / kXRows;

  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + oXBar);
  uint32_t *holder = reinterpret_cast<uint32_t *>(smem + oXFlags);
  volatile int *abort = reinterpret_cast<volatile int *>(smem + oXFlags + 4);
  if (tid == 0) {
    for (int b = 0; b < kXBars; ++b) {
      const uint32_t count = (b == bSFree || b == bSFree + 1 || b == bPFull || b == bPFull + 1) ? 128u
                             : (b == bQFull)                                                  ? 256u
                                                                                              : 1u;
      mbar_init(&bars[b], count);  // count 1: an expect_tx arrive or a tcgen05.commit
    }
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == kXIssuerWarp) tmem_alloc(holder, kXTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *holder;

  int issued = 0;  // producers: tiles whose copies went out
  if (warp < 8) {
    const int X = warp >> 2;
    x_load_q(a, t, smem, X);
    fence_proxy_async_smem();  // generic-proxy stores -> visible to the MMAs
    mbar_arrive(&bars[bQFull]);
    x_softmax(a, t, smem, tmem, bars, X, abort);
  } else if (warp == kXKProducerWarp) {
    issued = x_produce_k(a, t, smem, bars, abort);
  } else if (warp == kXVProducerWarp) {
    issued = x_produce_v(a, t, smem, bars, abort);
  } else if (tid == kXIssuerWarp * 32) {
    if (mbar_wait_bounded(&bars[bQFull], 0u, abort)) x_issuer(smem, tmem, t.ntiles, bars, abort);
    umma_commit(&bars[bFin]);  // every MMA issued is complete before TMEM is freed
    volatile int never = 0;
    mbar_wait_bounded(&bars[bFin], 0u, &never);
  }
  tc_fence_before();
  __syncthreads();
  if (*abort) {  // after a timeout: the last copies in flight land before the CTA exits
    if (tid == 0) set_err(a.err, NVKV_DEVERR_TIMEOUT);
    if ((warp == kXKProducerWarp || warp == kXVProducerWarp) && (tid & 31) == 0) {
      volatile int never = 0;
      for (int j = issued > 2 ? issued - 2 : 0; j < issued; ++j) {
        if (warp == kXKProducerWarp)
          mbar_wait_bounded(&bars[bKFull], static_cast<uint32_t>(j) & 1u, &never);
        else
          mbar_wait_bounded(&bars[bVFull + (j & 1)], static_cast<uint32_t>(j >> 1) & 1u, &never);
      }
    }
    __syncthreads();
  }
  if (warp == kXIssuerWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kXTmemCols);
  }
}

// ---------------------------------------------------------------------------
// The chunk's K/V into workspace rows: byte = E4M3_RNE_sat(x / ws_scale).
// One thread per 16 values; blockIdx.y = 0 (K) or 1 (V).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void x_load16(const float *src, float (&x)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 v = reinterpret_cast<const float4 *>(src)[i];
    x[4 * i] = v.x;
    x[4 * i + 1] = v.y;
    x[4 * i + 2] = v.z;
    x[4 * i + 3] = v.w;
  }
}

__device__ __forceinline__ void x_load16(const __nv_bfloat16 *src, float (&x)[16]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint4 v = reinterpret_cast<const uint4 *>(src)[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[8 * i + 2 * k] = __uint_as_float(w[k] << 16);
      x[8 * i + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256)
    ws_append_kernel(const T *__restrict__ k, const T *__restrict__ v, int64_t num_tokens, int Hkv, int D,
                     const int64_t *__restrict__ rows, const float *__restrict__ ws_scale, uint8_t *__restrict__ ws_k,
                     uint8_t *__restrict__ ws_v, int64_t ws_rows, int32_t *err) {
  const int kind = static_cast<int>(blockIdx.y);
  const int bpr = D / 16;  // 16-value blocks per row
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (gid >= num_tokens * Hkv * bpr) return;
  const int64_t tok = gid / (static_cast<int64_t>(Hkv) * bpr);
  const int64_t within = gid - tok * Hkv * bpr;  // h * bpr + blk
  const int64_t row = rows[tok];
  if (row < 0) return;
  if (row >= ws_rows) {
    if (within == 0 && kind == 0) set_err(err, NVKV_DEVERR_WS_ROWS);
    return;
  }
  float x[16];
  x_load16((kind == 0 ? k : v) + tok * Hkv * D + within * 16, x);
  const float s = ws_scale[kind];
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    w[j] = e4m3x2_from_f32(__fdiv_rn(x[4 * j], s), __fdiv_rn(x[4 * j + 1], s)) |
           (e4m3x2_from_f32(__fdiv_rn(x[4 * j + 2], s), __fdiv_rn(x[4 * j + 3], s)) << 16);
  *reinterpret_cast<uint4 *>((kind == 0 ? ws_k : ws_v) + row * Hkv * D + within * 16) =
      make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace
}  // namespace nvkv

using namespace nvkv;

extern "C" {

nvkv_status fp8_workspace_append_chunk(const void *k, const void *v, nvkv_dtype dtype, int64_t num_tokens,
                                       const int64_t *rows, int32_t num_kv_heads, int32_t head_dim,
                                       const float *ws_scale, uint8_t *ws_k, uint8_t *ws_v, int64_t ws_rows,
                                       int32_t *err_flag, void *stream) {
  NVKV_ABI_RANGE();
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || ws_rows < 0) return NVKV_ERR_INVALID_ARG;
  if (dtype != NVKV_DTYPE_F32 && dtype != NVKV_DTYPE_BF16) return NVKV_ERR_INVALID_ARG;
  if (head_dim % 16 != 0) return NVKV_ERR_UNSUPPORTED;
  if (num_tokens == 0) return NVKV_OK;
  if (!k || !v || !rows || !ws_scale || !ws_k || !ws_v) return NVKV_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(ws_k) || !aligned16(ws_v)) return NVKV_ERR_UNSUPPORTED;
  const int64_t items = num_tokens * num_kv_heads * (head_dim / 16);
  const int64_t blocks = (items + 255) / 256;
  if (blocks > 0x7fffffff) return NVKV_ERR_UNSUPPORTED;
  dim3 grid(static_cast<unsigned>(blocks), 2);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == NVKV_DTYPE_F32)
    ws_append_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float *>(k), static_cast<const float *>(v),
                                                 num_tokens, num_kv_heads, head_dim, rows, ws_scale, ws_k, ws_v,
                                                 ws_rows, err_flag);
  else
    ws_append_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
        static_cast<const __nv_bfloat16 *>(k), static_cast<const __nv_bfloat16 *>(v), num_tokens, num_kv_heads,
        head_dim, rows, ws_scale, ws_k, ws_v, ws_rows, err_flag);
  return launch_status();
}

size_t fp8_extend_scratch_size(int64_t ws_rows, int32_t num_kv_heads, int32_t head_dim) {
  if (ws_rows < 0 || num_kv_heads <= 0 || head_dim != kXD) return 0;
  const int64_t ngroups = (ws_rows + 7) / 8 + kXRows / 8;  // + one tile of zero rows past the end
  return static_cast<size_t>(2 * static_cast<int64_t>(num_kv_heads) * ngroups * kXGroupBytes);
}

nvkv_status fp8_chunked_extend_attention(const void *q, const int64_t *cu_q, int32_t n, int32_t max_q_len,
                                         int32_t num_q_heads, const uint8_t *ws_k, const uint8_t *ws_v,
                                         const int64_t *cu_kv, const int32_t *kv_lens, int32_t num_kv_heads,
                                         int32_t head_dim, int64_t ws_rows, const float *ws_scale, float sm_scale,
                                         void *scratch, size_t scratch_bytes, void *out, int32_t *err_flag,
                                         void *stream) {
  NVKV_ABI_RANGE();
  if (n < 0 || max_q_len < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || ws_rows < 0) return NVKV_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads != 0) return NVKV_ERR_INVALID_ARG;
  if (head_dim != kXD) return NVKV_ERR_UNSUPPORTED;
  const int G = num_q_heads / num_kv_heads;
  if (G > kXRows || (G & (G - 1)) != 0) return NVKV_ERR_UNSUPPORTED;
  if (n == 0 || max_q_len == 0) return NVKV_OK;
  if (!q || !cu_q || !ws_k || !ws_v || !cu_kv || !kv_lens || !ws_scale || !out || !scratch)
    return NVKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(ws_k) || !aligned16(ws_v) || !aligned16(out) || !aligned16(scratch))
    return NVKV_ERR_UNSUPPORTED;
  if (scratch_bytes < fp8_extend_scratch_size(ws_rows, num_kv_heads, head_dim)) return NVKV_ERR_WORKSPACE_TOO_SMALL;
  if (n > 65535 || num_kv_heads > 65535) return NVKV_ERR_UNSUPPORTED;
  ExtendArgs a;
  a.q = static_cast<const __nv_bfloat16 *>(q);
  a.cu_q = cu_q;
  a.ws_k = ws_k;
  a.ws_v = ws_v;
  a.cu_kv = cu_kv;
  a.kv_lens = kv_lens;
  a.ws_scale = ws_scale;
  a.out = static_cast<__nv_bfloat16 *>(out);
  a.err = err_flag;
  a.tiles = static_cast<const uint8_t *>(scratch);
  a.ngroups = (ws_rows + 7) / 8 + kXRows / 8;
  a.ws_rows = ws_rows;
  a.Hq = num_q_heads;
  a.Hkv = num_kv_heads;
  a.G = G;
  a.lgG = __builtin_ctz(static_cast<unsigned>(G));
  a.Tm = kXRows / G;
  a.sm_scale = sm_scale > 0.0f ? sm_scale : 1.0f / sqrtf(static_cast<float>(head_dim));
  const dim3 grid(static_cast<unsigned>((max_q_len + 2 * a.Tm - 1) / (2 * a.Tm)), static_cast<unsigned>(num_kv_heads),
                  static_cast<unsigned>(n));
  if (cudaFuncSetAttribute(extend_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kXSmem) !=
      cudaSuccess)
    return NVKV_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t items = a.ngroups * num_kv_heads * 16;
  if ((items + 255) / 256 > 0x7fffffff) return NVKV_ERR_UNSUPPORTED;
  extend_tiles_kernel<<<static_cast<unsigned>((items + 255) / 256), 256, 0, s>>>(
      ws_k, ws_v, ws_rows, num_kv_heads, a.ngroups, static_cast<uint8_t *>(scratch));
  extend_attention_kernel<<<grid, kXThreads, kXSmem, s>>>(a);
  return launch_status();
}

}  // extern "C"
