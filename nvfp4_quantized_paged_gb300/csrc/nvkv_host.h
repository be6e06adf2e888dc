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
  if (c->page_size != 16 && c->page_size != 32 && c->page_size != 64 && c->page_size != 128)
    return NVKV_ERR_UNSUPPORTED;
  if (!c->k_data || !c->v_data || !c->kv_scale) return NVKV_ERR_INVALID_ARG;
  if (!aligned16(c->k_data) || !aligned16(c->v_data)) return NVKV_ERR_UNSUPPORTED;
  if (c->prec == NVKV_PREC_NVFP4) {
    if (!c->k_scale || !c->v_scale) return NVKV_ERR_INVALID_ARG;
    if (!aligned16(c->k_scale) || !aligned16(c->v_scale)) return NVKV_ERR_UNSUPPORTED;
  }
  return NVKV_OK;
}

inline nvkv_status launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? NVKV_OK : NVKV_ERR_CUDA;
}

// Device-side view of a cache descriptor (passed by value to kernels).
struct CacheDev {
  uint8_t *kd, *vd, *ks, *vs;
  const float *scale;
  int32_t *err;
  int32_t num_pages, P, Hkv;
};

inline CacheDev to_dev(const nvkv_cache *c) {
  CacheDev d;
  d.kd = c->k_data;
  d.vd = c->v_data;
  d.ks = c->k_scale;
  d.vs = c->v_scale;
  d.scale = c->kv_scale;
  d.err = c->err_flag;
  d.num_pages = c->num_pages;
  d.P = c->page_size;
  d.Hkv = c->num_kv_heads;
  return d;
}

}  // namespace nvkv
