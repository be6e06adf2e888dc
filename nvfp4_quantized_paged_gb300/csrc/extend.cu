// Chunked-extend attention over the shared FP8 workspace, and the append of
// the current chunk's K/V into that workspace (sm_103a).
//
// "SGLang x Qwen x NVIDIA Collaboration: NVFP4 KV Cache Breaks Long-Context
// and Agentic Inference Bottlenecks", section "Three Paths": in chunked
// prefill / extend the cached prefix is dequantized into a cross-layer shared
// FP8 workspace, concatenated with the current chunk's KV, and the chunk's
// queries run FP8 attention over the concatenation (causal inside the chunk).
//
// Work item: (sequence, KV head, M-tile of 128 query rows).  Row r of an
// M-tile is query token r / G of the tile with query head h G + r % G, so the
// G query heads that share a KV head share every converted K/V tile.  Per
// tile of 128 keys, QK^T and P.V run on the tensor cores (tcgen05.mma
// kind::f16, M = N = 128, K = 16 per instruction, FP32 accumulators in TMEM:
// scores in two ping-pong buffers, the output in a third); the softmax runs
// in the registers of the thread that owns the row's TMEM lane.
//
// Roles (288 threads, one CTA per SM):
//   warps 0-3  softmax: thread r owns query row r; base-2 online softmax with
//              a lazily raised running max, P to shared memory as FP16, the
//              output rescaled in TMEM when the max rises, the epilogue.
//   warps 4-7  converters: the Q tile (BF16 -> FP16) once, then per KV tile
//              the E4M3 K rows into an FP16 K-major tile and the E4M3 V rows
//              into an FP16 V^T tile (keys along K), double-buffered.
//   warp 8     one thread issues the MMAs.
// E4M3 -> FP16 is exact; BF16 queries convert to FP16 exactly inside the FP16
// normal range [2^-14, 65504].
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "nvfp4kv.h"
#include "nvkv_device.cuh"
#include "nvkv_host.h"

namespace nvkv {
namespace {

constexpr int kXD = 128;                 // head_dim
constexpr int kXRows = 128;              // query rows per M-tile, keys per KV tile
constexpr int kXThreads = 288;
constexpr int kXIssuerWarp = 8;
constexpr uint32_t kXTmemCols = 512;     // scores 0..127 and 128..255, output 256..383
constexpr uint32_t kXColO = 256;
constexpr int kXTile = kXRows * kXD * 2; // one FP16 operand tile (32 KB)
constexpr int kXSbo = 2048;              // bytes between 8-row groups of a tile
// Shared memory: Q | K[2] | V^T[2] | P | barriers | TMEM holder, abort flag.
constexpr int oXQ = 0, oXK = kXTile, oXV = 3 * kXTile, oXP = 5 * kXTile, oXBar = 6 * kXTile;
constexpr int kXBars = 10;               // kv_full[2] s_full[2] s_free[2] p_full pv_done[2] fin
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

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int k) {
  return k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
}

__device__ __forceinline__ bool warp_wait_x(uint64_t *bar, uint32_t parity, volatile int *abort) {
  const bool ok = mbar_wait_bounded(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

struct Tile {            // the CTA's work item, uniform over the CTA
  int h;                 // KV head
  int64_t q0;            // first query row of the sequence in q / out
  int tok0, ntok;        // first chunk token of the M-tile, valid tokens in it
  int L;                 // keys of the sequence (prefix + chunk)
  int p;                 // prefix length: chunk token t sits at position p + t
  int64_t kv_base;       // workspace row of position 0
  int ntiles;            // KV tiles that some row of the M-tile sees
};

// ---------------------------------------------------------------------------
// Converters (warps 4-7).  Thread ct = (rb, dc): 8-row block rb, 16-element
// column chunk dc.  Stores are rotated so that the eight threads of a store
// phase (dc = 0..7, one rb) write eight different rows of their core
// matrices: no shared-memory bank conflicts.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void x_converter(const ExtendArgs &a, const Tile &t, uint8_t *smem, uint64_t *kv_full,
                            uint64_t *pv_done, volatile int *abort) {
  const int ct = static_cast<int>(threadIdx.x) - 128;
  const int rb = ct >> 3, dc = ct & 7;
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  // Q rows 8 rb + (s + dc) % 8, elements 16 dc .. 16 dc + 15 -> chunks 2 dc, 2 dc + 1
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int r = 8 * rb + ((s + dc) & 7);
    const int tok = r >> a.lgG, g = r & (a.G - 1);
    uint4 lo = zero, hi = zero;
    if (tok < t.ntok) {
      const uint4 *src = reinterpret_cast<const uint4 *>(
          a.q + ((t.q0 + t.tok0 + tok) * a.Hq + static_cast<int64_t>(t.h) * a.G + g) * kXD + 16 * dc);
      lo = src[0];
      hi = src[1];
    }
    uint8_t *dst = smem + oXQ + kmaj(r, 2 * dc);
    *reinterpret_cast<uint4 *>(dst) = make_uint4(f16x2_from_bf16x2(lo.x), f16x2_from_bf16x2(lo.y),
                                                 f16x2_from_bf16x2(lo.z), f16x2_from_bf16x2(lo.w));
    *reinterpret_cast<uint4 *>(dst + 128) = make_uint4(f16x2_from_bf16x2(hi.x), f16x2_from_bf16x2(hi.y),
                                                       f16x2_from_bf16x2(hi.z), f16x2_from_bf16x2(hi.w));
  }
  const int rho = dc >> 2, tau = dc & 3;
  for (int j = 0; j < t.ntiles; ++j) {
    const int b = j & 1, kv0 = j * kXRows;
    // loads first (their latency overlaps the wait for the buffer); keys past
    // the sequence read as zero (never NaN: P is 0 there and 0 * NaN = NaN)
    uint4 kr[8], vr[8];
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const int key = kv0 + 8 * rb + ((s + dc) & 7);
      kr[s] = key < t.L ? *reinterpret_cast<const uint4 *>(
                              a.ws_k + ((t.kv_base + key) * a.Hkv + t.h) * kXD + 16 * dc)
                        : zero;
    }
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const int key = kv0 + 8 * rb + s;
      vr[s] = key < t.L ? *reinterpret_cast<const uint4 *>(
                              a.ws_v + ((t.kv_base + key) * a.Hkv + t.h) * kXD + 16 * dc)
                        : zero;
    }
    // the buffer was last read by the MMAs of tile j - 2
    if (j >= 2 && !warp_wait_x(&pv_done[b], static_cast<uint32_t>((j - 2) >> 1) & 1u, abort)) return;
    uint8_t *ks = smem + oXK + b * kXTile;
    uint8_t *vt = smem + oXV + b * kXTile;
    // K: row 8 rb + (s + dc) % 8 (the key), chunks 2 dc and 2 dc + 1
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      uint8_t *dst = ks + kmaj(8 * rb + ((s + dc) & 7), 2 * dc);
      const uint4 w = kr[s];
      *reinterpret_cast<uint4 *>(dst) = make_uint4(f16x2_from_e4m3x2<0>(w.x), f16x2_from_e4m3x2<1>(w.x),
                                                   f16x2_from_e4m3x2<0>(w.y), f16x2_from_e4m3x2<1>(w.y));
      *reinterpret_cast<uint4 *>(dst + 128) = make_uint4(f16x2_from_e4m3x2<0>(w.z), f16x2_from_e4m3x2<1>(w.z),
                                                         f16x2_from_e4m3x2<0>(w.w), f16x2_from_e4m3x2<1>(w.w));
    }
    // V^T: row = value 16 dc + e, chunk rb = keys 8 rb .. 8 rb + 7.  Word w
    // of vr[s] holds values 16 dc + 4 w .. + 3 of key 8 rb + s.  Step (sg, bt)
    // handles e = 4 ((sg + rho) % 4) + (bt + tau) % 4: e % 8 differs across
    // the eight threads of a store phase.
    uint32_t wv[8][4];
#pragma unroll
    for (int s = 0; s < 8; ++s)
#pragma unroll
      for (int k = 0; k < 4; ++k) wv[s][k] = rho ? word_of(vr[s], (k + 1) & 3) : word_of(vr[s], k);
#pragma unroll
    for (int bt = 0; bt < 4; ++bt) {
      const uint32_t bb = static_cast<uint32_t>((bt + tau) & 3);
      const uint32_t sel = bb | ((bb + 4u) << 4);  // byte bb of the first word, byte bb of the second
#pragma unroll
      for (int sg = 0; sg < 4; ++sg) {
        const int e = 4 * ((sg + rho) & 3) + static_cast<int>(bb);
        uint32_t o[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) o[u] = f16x2_from_e4m3x2<0>(prmt(wv[2 * u][sg], wv[2 * u + 1][sg], sel));
        *reinterpret_cast<uint4 *>(vt + (2 * dc + (e >> 3)) * kXSbo + rb * 128 + (e & 7) * 16) =
            make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    fence_proxy_async_smem();  // generic-proxy stores -> visible to the MMAs
    mbar_arrive(&kv_full[b]);
  }
}

// ---------------------------------------------------------------------------
// Softmax (warps 0-3): thread r owns TMEM lane r = query row r.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void x_softmax(const ExtendArgs &a, const Tile &t, uint8_t *smem, uint32_t tmem, uint64_t *s_full,
                          uint64_t *s_free, uint64_t *p_full, uint64_t *pv_done, volatile int *abort) {
  const int r = static_cast<int>(threadIdx.x), warp = r >> 5;
  const int tok = r >> a.lgG, g = r & (a.G - 1);
  const int qpos = t.p + t.tok0 + (tok < t.ntok ? tok : t.ntok - 1);  // sees positions [0, qpos]
  const float c2 = a.ws_scale[0] * a.sm_scale * 1.4426950408889634f;  // score -> log2 units
  const uint32_t lanes = tmem + (static_cast<uint32_t>(32 * warp) << 16);
  const int first_partial = t.p + t.tok0;  // the smallest qpos of the M-tile
  float m = kXNoMax, mt = kXNoMax, l = 0.0f;
  bool ok = true;
  for (int j = 0; j < t.ntiles; ++j) {
    const int b = j & 1, kv0 = j * kXRows;
    ok = warp_wait_x(&s_full[b], static_cast<uint32_t>(j >> 1) & 1u, abort);
    if (!ok) break;
    tc_fence_after();
    // the row's 128 scores: eight loads in flight, one wait
    const uint32_t sadr = lanes + static_cast<uint32_t>(b * 128);
    uint32_t v[8][16];
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) tmem_ld16_async(sadr + 16 * ch, v[ch]);
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int ch = 0; ch < 8; ++ch)
#pragma unroll
      for (int e = 0; e < 16; ++e) asm volatile("" : "+r"(v[ch][e]));
    tc_fence_before();
    mbar_arrive(&s_free[b]);  // the score buffer may take the next-but-one tile
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
    const float nm = -m;
    float la[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    uint32_t pk[64];
#pragma unroll
    for (int ch = 0; ch < 8; ++ch)
#pragma unroll
      for (int e = 0; e < 16; e += 2) {
        float a0, a1;
        fma_f32x2(a0, a1, __uint_as_float(v[ch][e]), __uint_as_float(v[ch][e + 1]), c2, c2, nm, nm);
        const float p0 = ex2(a0), p1 = ex2(a1);  // masked: exp2(-inf) = 0
        add_f32x2(la[(e >> 1) & 2], la[((e >> 1) & 2) + 1], p0, p1);
        pk[8 * ch + e / 2] = pack_f16x2(p0, p1);
      }
    l += (la[0] + la[1]) + (la[2] + la[3]);
    // P and the output are free once the previous tile's P.V is done
    if (j >= 1) {
      ok = warp_wait_x(&pv_done[(j - 1) & 1], static_cast<uint32_t>((j - 1) >> 1) & 1u, abort);
      if (!ok) break;
      tc_fence_after();
      if (__any_sync(0xffffffffu, need)) {  // rescale the output rows whose max rose (warp-uniform)
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          float o[16];
          tmem_ld16(lanes + kXColO + 16 * ch, o);
#pragma unroll
          for (int e = 0; e < 16; ++e) o[e] *= alpha;
          tmem_st16(lanes + kXColO + 16 * ch, o);
        }
        tmem_st_wait();
      }
    }
    uint8_t *ps = smem + oXP;
#pragma unroll
    for (int c = 0; c < 16; ++c)
      *reinterpret_cast<uint4 *>(ps + kmaj(r, c)) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
    fence_proxy_async_smem();
    tc_fence_before();
    mbar_arrive(p_full);
  }
  if (ok) {
    const int jl = t.ntiles - 1;
    ok = warp_wait_x(&pv_done[jl & 1], static_cast<uint32_t>(jl >> 1) & 1u, abort);
  }
  if (!ok) return;
  tc_fence_after();
  const float inv = a.ws_scale[1] / l;
  const bool write = tok < t.ntok;
  __nv_bfloat16 *dst = a.out + ((t.q0 + t.tok0 + tok) * a.Hq + static_cast<int64_t>(t.h) * a.G + g) * kXD;
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    float o[16];
    tmem_ld16(lanes + kXColO + 16 * ch, o);
    uint32_t w[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const __nv_bfloat162 v = __floats2bfloat162_rn(o[2 * e] * inv, o[2 * e + 1] * inv);
      w[e] = *reinterpret_cast<const uint32_t *>(&v);
    }
    if (write) {
      *reinterpret_cast<uint4 *>(dst + 16 * ch) = make_uint4(w[0], w[1], w[2], w[3]);
      *reinterpret_cast<uint4 *>(dst + 16 * ch + 8) = make_uint4(w[4], w[5], w[6], w[7]);
    }
  }
}

// ---------------------------------------------------------------------------
// MMA issuer (one thread of warp 8), polling: S_b = Q K_b^T as soon as K_b is
// staged and S_b's previous scores are read (at most one tile ahead of P.V,
// so the next tile's scores are computed during this tile's softmax);
// O += P V_b as soon as P is written.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void x_issuer(uint8_t *smem, uint32_t tmem, int ntiles, uint64_t *kv_full, uint64_t *s_full,
                         uint64_t *s_free, uint64_t *p_full, uint64_t *pv_done, volatile int *abort) {
  const uint32_t qs = smem_u32(smem + oXQ), ps = smem_u32(smem + oXP);
  constexpr uint32_t id = idesc_f16(kXRows);
  int nqk = 0, npv = 0;  // next tile whose QK^T / P.V goes out
  uint64_t t_last = global_timer_ns();
  while (npv < ntiles) {
    bool did = false;
    // QK^T of tile nqk: K staged, and its score buffer read by the softmax of tile nqk - 2
    if (nqk < ntiles && nqk <= npv + 1) {
      const int b = nqk & 1;
      if (mbar_test(&kv_full[b], static_cast<uint32_t>(nqk >> 1) & 1u) &&
          (nqk < 2 || mbar_test(&s_free[b], static_cast<uint32_t>((nqk - 2) >> 1) & 1u))) {
        tc_fence_after();
        const uint32_t ks = smem_u32(smem + oXK + b * kXTile);
#pragma unroll
        for (int kk = 0; kk < kXD / 16; ++kk)
          umma_f16(tmem + static_cast<uint32_t>(b * 128), umma_desc(qs + kk * 256, 128, kXSbo),
                   umma_desc(ks + kk * 256, 128, kXSbo), id, kk > 0 ? 1u : 0u);
        umma_commit(&s_full[b]);
        ++nqk;
        did = true;
      }
    }
    // P.V of tile npv once its P is written
    if (npv < nqk && mbar_test(p_full, static_cast<uint32_t>(npv) & 1u)) {
      tc_fence_after();
      const uint32_t vt = smem_u32(smem + oXV + (npv & 1) * kXTile);
#pragma unroll
      for (int kk = 0; kk < kXRows / 16; ++kk)
        umma_f16(tmem + kXColO, umma_desc(ps + kk * 256, 128, kXSbo), umma_desc(vt + kk * 256, 128, kXSbo), id,
                 (npv > 0 || kk > 0) ? 1u : 0u);
      umma_commit(&pv_done[npv & 1]);
      ++npv;
      did = true;
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
  const int i = static_cast<int>(blockIdx.z);
  Tile t;
  t.h = static_cast<int>(blockIdx.y);
  t.q0 = a.cu_q[i];
  const int64_t nq = a.cu_q[i + 1] - t.q0;
  t.L = a.kv_lens[i];
  t.kv_base = a.cu_kv[i];
  if (nq < 0 || nq > t.L || t.kv_base < 0 || t.kv_base + t.L > a.ws_rows) {
    if (tid == 0 && blockIdx.x == 0 && t.h == 0)
      set_err(a.err, (nq < 0 || nq > t.L) ? NVKV_DEVERR_SEQLEN : NVKV_DEVERR_WS_ROWS);
    return;
  }
  if (tid == 0 && blockIdx.x == 0 && t.h == 0 && nq > static_cast<int64_t>(gridDim.x) * a.Tm)
    set_err(a.err, NVKV_DEVERR_SEQLEN);  // more queries than max_q_len: the rest are not computed
  const int mtile = static_cast<int>(gridDim.x - 1 - blockIdx.x);  // longest M-tiles launch first
  t.tok0 = mtile * a.Tm;
  if (t.tok0 >= nq) return;  // uniform: before any barrier or TMEM allocation
  t.ntok = static_cast<int>(nq - t.tok0 < a.Tm ? nq - t.tok0 : a.Tm);
  t.p = t.L - static_cast<int>(nq);
  t.ntiles = (t.p + t.tok0 + t.ntok + kXRows - 1) / kXRows;

  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + oXBar);
  uint64_t *kv_full = bars, *s_full = bars + 2, *s_free = bars + 4, *p_full = bars + 6, *pv_done = bars + 7;
  uint64_t *fin = bars + 9;
  uint32_t *holder = reinterpret_cast<uint32_t *>(smem + oXFlags);
  volatile int *abort = reinterpret_cast<volatile int *>(smem + oXFlags + 4);
  if (tid == 0) {
    mbar_init(&kv_full[0], 128);
    mbar_init(&kv_full[1], 128);
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(&s_free[0], 128);
    mbar_init(&s_free[1], 128);
    mbar_init(p_full, 128);
    mbar_init(&pv_done[0], 1);
    mbar_init(&pv_done[1], 1);
    mbar_init(fin, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == kXIssuerWarp) tmem_alloc(holder, kXTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *holder;

  if (warp < 4) {
    x_softmax(a, t, smem, tmem, s_full, s_free, p_full, pv_done, abort);
  } else if (warp < 8) {
    x_converter(a, t, smem, kv_full, pv_done, abort);
  } else if (tid == kXIssuerWarp * 32) {
    x_issuer(smem, tmem, t.ntiles, kv_full, s_full, s_free, p_full, pv_done, abort);
    umma_commit(fin);  // every MMA issued is complete before TMEM is freed
    volatile int never = 0;
    mbar_wait_bounded(fin, 0u, &never);
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort) set_err(a.err, NVKV_DEVERR_TIMEOUT);
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

nvkv_status fp8_chunked_extend_attention(const void *q, const int64_t *cu_q, int32_t n, int32_t max_q_len,
                                         int32_t num_q_heads, const uint8_t *ws_k, const uint8_t *ws_v,
                                         const int64_t *cu_kv, const int32_t *kv_lens, int32_t num_kv_heads,
                                         int32_t head_dim, int64_t ws_rows, const float *ws_scale, float sm_scale,
                                         void *out, int32_t *err_flag, void *stream) {
  if (n < 0 || max_q_len < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || ws_rows < 0) return NVKV_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads != 0) return NVKV_ERR_INVALID_ARG;
  if (head_dim != kXD) return NVKV_ERR_UNSUPPORTED;
  const int G = num_q_heads / num_kv_heads;
  if (G > kXRows || (G & (G - 1)) != 0) return NVKV_ERR_UNSUPPORTED;
  if (n == 0 || max_q_len == 0) return NVKV_OK;
  if (!q || !cu_q || !ws_k || !ws_v || !cu_kv || !kv_lens || !ws_scale || !out) return NVKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(ws_k) || !aligned16(ws_v) || !aligned16(out)) return NVKV_ERR_UNSUPPORTED;
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
  a.ws_rows = ws_rows;
  a.Hq = num_q_heads;
  a.Hkv = num_kv_heads;
  a.G = G;
  a.lgG = __builtin_ctz(static_cast<unsigned>(G));
  a.Tm = kXRows / G;
  a.sm_scale = sm_scale > 0.0f ? sm_scale : 1.0f / sqrtf(static_cast<float>(head_dim));
  const dim3 grid(static_cast<unsigned>((max_q_len + a.Tm - 1) / a.Tm), static_cast<unsigned>(num_kv_heads),
                  static_cast<unsigned>(n));
  if (cudaFuncSetAttribute(extend_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kXSmem) !=
      cudaSuccess)
    return NVKV_ERR_CUDA;
  extend_attention_kernel<<<grid, kXThreads, kXSmem, static_cast<cudaStream_t>(stream)>>>(a);
  return launch_status();
}

}  // extern "C"
