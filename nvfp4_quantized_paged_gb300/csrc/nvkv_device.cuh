// Device-side building blocks of the nvfp4kv CUDA library (sm_103a):
// number-format conversions, mbarrier / bulk-copy staging, warp MMA.
//
// Formats ("SOAR Weekly Champion Notes 05", 02: E2M1 = 1 sign + 2 exponent +
// 1 mantissa bit, two values per byte; "SGLang x Qwen x NVIDIA ...", The Core
// of the Ledger: one E4M3 scale per 16 values, one FP32 global scale).
// Every conversion below is a hardware cvt instruction; the rounding mode is
// round-to-nearest-even with satfinite saturation, which the exhaustive
// encoder tests check bit for bit against the quantizer definition.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace nvkv {

// ---------------------------------------------------------------------------
// Conversions
// ---------------------------------------------------------------------------

// Two FP32 values -> one byte of two E2M1 codes: `lo` in bits 3:0, `hi` in 7:4.
__device__ __forceinline__ uint32_t e2m1x2_from_f32(float lo, float hi) {
  uint32_t r;
  asm("{ .reg .b8 q; .reg .b16 w;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q, %1, %2;\n\t"
      "cvt.u16.u8 w, q;\n\t"
      "cvt.u32.u16 %0, w; }"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r & 0xFFu;
}

// Two FP32 values -> two E4M3 bytes: `lo` in bits 7:0, `hi` in 15:8.
__device__ __forceinline__ uint32_t e4m3x2_from_f32(float lo, float hi) {
  uint32_t r;
  asm("{ .reg .b16 w;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 w, %1, %2;\n\t"
      "cvt.u32.u16 %0, w; }"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r & 0xFFFFu;
}

// Byte I (0..3) of a word holding pairs of E2M1 codes -> half2 {low nibble, high nibble}.
template <int I>
__device__ __forceinline__ uint32_t f16x2_from_e2m1x2(uint32_t w) {
  uint32_t r;
  asm("{ .reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b%2;\n\t"
      "}"
      : "=r"(r)
      : "r"(w), "n"(I));
  return r;
}

// Low (H=0) or high (H=1) 16 bits of a word holding two E4M3 bytes -> half2.
template <int H>
__device__ __forceinline__ uint32_t f16x2_from_e4m3x2(uint32_t w) {
  uint32_t r;
  if (H == 0) {
    asm("{ .reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %1;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo; }"
        : "=r"(r)
        : "r"(w));
  } else {
    asm("{ .reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %1;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, hi; }"
        : "=r"(r)
        : "r"(w));
  }
  return r;
}

// Exact FP32 value of an E4M3 byte (never NaN for bytes this library writes).
__device__ __forceinline__ float f32_from_e4m3(uint32_t b) {
  const uint32_t h2 = f16x2_from_e4m3x2<0>(b & 0xFFu);
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

__device__ __forceinline__ float f32_lo(uint32_t h2) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

__device__ __forceinline__ float f32_hi(uint32_t h2) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16)));
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// ---------------------------------------------------------------------------
// Warp MMA m16n8k16, FP16 inputs, FP32 accumulate (C += A * B)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_f16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 8x8 b16 transpose across the warp: thread (r, c) holding row r, cols 2c..2c+1
// gets row r, cols 2c..2c+1 of the transposed matrix.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

// Hardware base-2 exponential (MUFU.EX2).
__device__ __forceinline__ float ex2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// ---------------------------------------------------------------------------
// Shared-memory addresses, mbarriers and bulk copies
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait: true once the phase with `parity` completed; false if *abort
// became nonzero or the wait exceeded ~2 s (then *abort is raised).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, volatile int *abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if ((it & 255u) == 0 && global_timer_ns() - t0 > 2000000000ull) {
      *abort = 1;
      return false;
    }
  }
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void set_err(int32_t *err, int32_t code) {
  if (err) atomicCAS(err, 0, code);
}

}  // namespace nvkv
