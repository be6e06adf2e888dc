// Host-side helpers shared by the nvfp4kv translation units: argument checks
// and error mapping.  Part of the C-ABI implementation (include/nvfp4kv.h).
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "../../include/nvfp4kv.h"

namespace nvkv {

// NVTX range around one C-ABI call that launches device work, named after the
// call, so a profiler's timeline and kernel filters can attribute launches to
// it.  With no tool attached the push and pop return at once.
struct AbiRange {
  explicit AbiRange(const char *name) { nvtxRangePushA(name); }
  ~AbiRange() { nvtxRangePop(); }
  AbiRange(const AbiRange &) = delete;
  AbiRange &operator=(const AbiRange &) = delete;
};
#define NVKV_ABI_RANGE() ::nvkv::AbiRange nvkv_abi_range_(__func__)

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape and pointer checks of a cache descriptor against the precision the
// caller expects (want_prec < 0: either).  Returns NVKV_OK or the status.
inline nvkv_status check_cache(const nvkv_cache *c, int32_t want_prec) {
  if (!c) return NVKV_ERR_INVALID_ARG;
  if (c->prec != NVKV_PREC_NVFP4 && c->prec != NVKV_PREC_FP8_E4M3) return NVKV_ERR_INVALID_ARG;
  if (want_prec >= 0 && c->prec != want_prec) return NVKV_ERR_INVALID_ARG;
  if (c->num_pages <= 0 || c->num_kv_heads <= 0 || c->page_size <= 0 || c->head_dim <= 0)
    return NVKV_ERR_INVALID_ARG;
  if (c->head_dim != 128) return NVKV_ERR_UNSUPPORTED;
  if (c->page_size != 16 && c->page_size != 32 && c->page_size != 64) return NVKV_ERR_UNSUPPORTED;  // multiples of 8
  if (!c->data || !c->kv_scale) return NVKV_ERR_INVALID_ARG;
  if (!aligned16(c->data)) return NVKV_ERR_UNSUPPORTED;
  return NVKV_OK;
}

inline nvkv_status launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? NVKV_OK : NVKV_ERR_CUDA;
}

// Device-side view of a cache descriptor (passed by value to kernels).
// Byte layout of one (page, KV head) block at head_dim 128 (see the header):
// groups of 8 slots; an NVFP4 group is [K codes 512 | K scales 64 | V codes
// 512 | V scales 64] = 1152 bytes, an FP8 group [K 1024 | V 1024]; K bytes in
// 16-byte chunks, chunk-major (the tensor-core operand order).  V is stored by
// slot pairs (2c, 2c+1), the layout of a P.V operand register (two tokens of
// one value): NVFP4 code of value 16b + j of slot r at byte b*64 + (r/2)*16 + j
// of the V codes, nibble r % 2; V scales block-major (b*8 + r); FP8 byte of
// value 16b + j at (j/8)*512 + b*64 + (r/2)*16 + (j%8)*2 + r%2 of V.
constexpr int kNvTokBytes = 144, kF8TokBytes = 256;  // per token, K + V
constexpr int kGroupRows = 8;
constexpr int kNvGroup = kGroupRows * kNvTokBytes;    // 1152
constexpr int kF8Group = kGroupRows * kF8TokBytes;    // 2048
constexpr int kNvKScales = 512, kNvVCodes = 576, kNvVScales = 1088;  // offsets inside an NVFP4 group
constexpr int kF8V = 1024;                                          // offset of V inside an FP8 group


struct CacheDev {
  uint8_t *data;
  const float *scale;
  int32_t *err;
  int32_t num_pages, P, Hkv;
  __host__ __device__ int64_t block(int64_t page, int h, int tok_bytes) const {
    return (page * Hkv + h) * static_cast<int64_t>(P) * tok_bytes;
  }
  // NVFP4 K: the 8 code bytes of 16-value block `blk` of slot `off`
  __host__ __device__ int64_t nv_kcodes(int64_t page, int h, int off, int blk) const {
    return block(page, h, kNvTokBytes) + static_cast<int64_t>(off >> 3) * kNvGroup + (blk >> 1) * 128 +
           (off & 7) * 16 + (blk & 1) * 8;
  }
  // NVFP4 V: the 16 bytes holding block `blk` of slot `off` and of its pair
  // partner (value 16 blk + j at byte j; this slot's nibble is off % 2)
  __host__ __device__ int64_t nv_vcodes(int64_t page, int h, int off, int blk) const {
    return block(page, h, kNvTokBytes) + static_cast<int64_t>(off >> 3) * kNvGroup + kNvVCodes + blk * 64 +
           ((off & 7) >> 1) * 16;
  }
  // NVFP4: the E4M3 scale byte of block `blk` of slot `off` (kind 0 = K, 1 = V)
  __host__ __device__ int64_t nv_scale(int64_t page, int h, int kind, int off, int blk) const {
    return block(page, h, kNvTokBytes) + static_cast<int64_t>(off >> 3) * kNvGroup +
           (kind == 0 ? kNvKScales + (off & 7) * 8 + blk : kNvVScales + blk * 8 + (off & 7));
  }
  // FP8 K: the 16 bytes of 16-value block `blk` of slot `off`
  __host__ __device__ int64_t f8_kblock(int64_t page, int h, int off, int blk) const {
    return block(page, h, kF8TokBytes) + static_cast<int64_t>(off >> 3) * kF8Group + blk * 128 + (off & 7) * 16;
  }
  // FP8 V: the 16 bytes holding values 16 blk + 8 half + j' (j' < 8) of slot
  // `off` and its partner (this slot's byte of value j' is 2 j' + off % 2)
  __host__ __device__ int64_t f8_vchunk(int64_t page, int h, int off, int blk, int half) const {
    return block(page, h, kF8TokBytes) + static_cast<int64_t>(off >> 3) * kF8Group + kF8V + half * 512 + blk * 64 +
           ((off & 7) >> 1) * 16;
  }
};

inline CacheDev to_dev(const nvkv_cache *c) {
  CacheDev d;
  d.data = c->data;
  d.scale = c->kv_scale;
  d.err = c->err_flag;
  d.num_pages = c->num_pages;
  d.P = c->page_size;
  d.Hkv = c->num_kv_heads;
  return d;
}

}  // namespace nvkv
