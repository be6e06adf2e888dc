// Host-side helpers shared by the nvfp4kv translation units: argument checks
// and error mapping.  Part of the C-ABI implementation (include/nvfp4kv.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/nvfp4kv.h"

namespace nvkv {

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
  if (c->page_size != 16 && c->page_size != 32 && c->page_size != 64) return NVKV_ERR_UNSUPPORTED;
  if (!c->data || !c->kv_scale) return NVKV_ERR_INVALID_ARG;
  if (!aligned16(c->data)) return NVKV_ERR_UNSUPPORTED;
  return NVKV_OK;
}

inline nvkv_status launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? NVKV_OK : NVKV_ERR_CUDA;
}

// Device-side view of a cache descriptor (passed by value to kernels).
// Byte layout of one (page, KV head) block at head_dim 128 (see the header).
constexpr int kNvCodeRow = 64, kNvScaleRow = 8, kNvTokBytes = 144;  // NVFP4: per token, K+V
constexpr int kF8Row = 128, kF8TokBytes = 256;                      // FP8

struct CacheDev {
  uint8_t *data;
  const float *scale;
  int32_t *err;
  int32_t num_pages, P, Hkv;
  // NVFP4 plane offsets inside a block: kind 0 = K, 1 = V
  __host__ __device__ int64_t block(int64_t page, int h, int tok_bytes) const {
    return (page * Hkv + h) * static_cast<int64_t>(P) * tok_bytes;
  }
  __host__ __device__ int64_t nv_codes(int64_t page, int h, int kind, int off) const {
    return block(page, h, kNvTokBytes) + static_cast<int64_t>(kind) * P * (kNvCodeRow + kNvScaleRow) +
           static_cast<int64_t>(off) * kNvCodeRow;
  }
  __host__ __device__ int64_t nv_scales(int64_t page, int h, int kind, int off) const {
    return block(page, h, kNvTokBytes) + static_cast<int64_t>(kind) * P * (kNvCodeRow + kNvScaleRow) +
           static_cast<int64_t>(P) * kNvCodeRow + static_cast<int64_t>(off) * kNvScaleRow;
  }
  __host__ __device__ int64_t f8_row(int64_t page, int h, int kind, int off) const {
    return block(page, h, kF8TokBytes) + static_cast<int64_t>(kind) * P * kF8Row + static_cast<int64_t>(off) * kF8Row;
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
