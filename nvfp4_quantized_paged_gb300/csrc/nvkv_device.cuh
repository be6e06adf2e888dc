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
// Exact codes of correctly rounded quotients without a division per value.
// The write rule takes code = RNE(fl(x / den)) (E2M1 or E4M3, saturating).
// With r = fl(1 / den) and q = fl(x r): q = (x / den)(1 + d1)(1 + d2) and
// fl(x / den) = (x / den)(1 + d3), |di| <= 2^-24, so fl(x / den) lies within
// 3 2^-24 |q| of q.  The bracket ends fl(q (1 - 2^-21)) and fl(q (1 + 2^-21))
// (2^-21 = 8 2^-24, each end rounded once more) lie outside that interval on
// either side, and rounding to the code grid is monotone in the magnitude, so
// when both ends give the same code it is the code of fl(x / den).  When a
// rounding boundary falls inside the bracket (a fraction of about 2^-20 of
// the values) the quotient is taken exactly.  Requires r normal and finite
// (den neither tiny nor huge); callers divide otherwise.  Quotients below the
// normal range give code 0 at both ends whatever their rounding error.
constexpr float kBracketLo = 1.0f - 0x1p-21f, kBracketHi = 1.0f + 0x1p-21f;

__device__ __forceinline__ bool quot_fast_ok(float r) { return r >= 0x1p-126f && r <= 0x1p127f; }

__device__ __forceinline__ uint32_t e2m1x2_quot(float x0, float x1, float den, float r);
__device__ __forceinline__ uint32_t e4m3x2_quot(float x0, float x1, float den, float r);

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

// (a0 + b0, a1 + b1) as one packed FP32x2 add (round to nearest even each).
__device__ __forceinline__ void add_f32x2(float &a0, float &a1, float b0, float b1) {
  asm("{ .reg .b64 p, q;\n\t"
      "mov.b64 p, {%0, %1};\n\t"
      "mov.b64 q, {%2, %3};\n\t"
      "add.rn.f32x2 p, p, q;\n\t"
      "mov.b64 {%0, %1}, p; }"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1));
}

// Elementwise max of two half2 (an input that is NaN yields the other).
__device__ __forceinline__ uint32_t __hmax2_as_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
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

// try_wait that suspends the thread in hardware until the phase completes or
// about `hint_ns` nanoseconds pass, so a waiting warp takes no issue slots.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Bounded wait: true once the phase with `parity` completed; false if *abort
// became nonzero or the wait exceeded ~2 s (then *abort is raised).  Between
// tries the warp sleeps (32 ns, doubling up to 256 ns), so a long wait costs
// few issue slots; the sleep bounds the added wake-up latency.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, volatile int *abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  uint32_t ns = 32;
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > 2000000000ull) {
      *abort = 1;
      return false;
    }
    __nanosleep(ns);
    if (ns < 256) ns <<= 1;
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

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also ANDs a predicate over its nthreads threads.
__device__ __forceinline__ bool named_bar_and(int id, int nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q; }"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// Non-blocking test: true if the phase with `parity` has completed.
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p; }"
      : "=r"(r)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void set_err(int32_t *err, int32_t code) {
  if (err) atomicCAS(err, 0, code);
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// 5th-generation tensor cores (tcgen05): TMEM, descriptors, MMA
// ---------------------------------------------------------------------------

// Shared-memory matrix descriptor, no swizzle: 8-row x 16-byte core matrices;
// lbo = byte distance between core matrices along K, sbo = between 8-row
// groups along M (or N).  Addresses and offsets are multiples of 16.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (static_cast<uint64_t>(1) << 46);
}

// Instruction descriptors, M = 128, FP32 accumulator, both operands K-major.
// kind::mxf4nvf4 (E2M1 x E2M1, E4M3 block scales per 16 values):
__host__ __device__ constexpr uint32_t idesc_nvfp4(int n) {
  return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);
}
// kind::f8f6f4 with E4M3 x E4M3:
__host__ __device__ constexpr uint32_t idesc_e4m3(int n) {
  return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);
}

__device__ __forceinline__ void tmem_alloc(uint32_t *holder_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(holder_smem)),
               "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[128 x n] (+)= A * B with E2M1 operands and E4M3 scale factors in TMEM.
__device__ __forceinline__ void umma_nvfp4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                           uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p;\n\t setp.ne.u32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p; }" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

// D[128 x n] (+)= A * B with E4M3 operands.
__device__ __forceinline__ void umma_e4m3(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p;\n\t setp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p; }" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// kind::f16 with FP16 x FP16 operands, FP32 accumulator, M = 128, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16(int n) {
  return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);
}

// D[128 x n] (+)= A * B with FP16 operands (K = 16 per instruction).
__device__ __forceinline__ void umma_f16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p;\n\t setp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 32 rows x 16 bytes of shared memory -> 4 TMEM columns of lanes 32q + row, for
// every lane quadrant q (scale-factor copies).
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// One 32-bit column of this warp's 32 TMEM lanes (one value per lane), and the
// wait that makes this thread's TMEM stores complete.
__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 16 consecutive FP32 columns of this warp's 32 TMEM lanes (one row per lane);
// the load and its completion wait form one statement, so no use of the
// registers can be scheduled before the data is there.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&x)[16]) {
  uint32_t v[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) x[i] = __uint_as_float(v[i]);
}

// 16 consecutive FP32 columns of this warp's 32 TMEM lanes without waiting:
// the registers may be read only after tmem_ld_wait() on the same values.
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}

// Wait for this thread's TMEM loads, then pass each loaded register through
// an empty statement ordered after the wait, so no use of it can be
// scheduled before the data is there.
template <int N>
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&v)[N]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(v[i]));
}

// (a0, a1) * (b0, b1) + (c0, c1) as one packed FP32x2 fused multiply-add.
__device__ __forceinline__ void fma_f32x2(float &d0, float &d1, float a0, float a1, float b0, float b1, float c0,
                                          float c1) {
  asm("{ .reg .b64 a, b, c;\n\t"
      "mov.b64 a, {%2, %3};\n\t"
      "mov.b64 b, {%4, %5};\n\t"
      "mov.b64 c, {%6, %7};\n\t"
      "fma.rn.f32x2 a, a, b, c;\n\t"
      "mov.b64 {%0, %1}, a; }"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// 16 consecutive 32-bit columns of this warp's 32 TMEM lanes (one row per
// lane); the caller waits with tmem_st_wait() before the columns are read.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&x)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(__float_as_uint(x[0])), "r"(__float_as_uint(x[1])), "r"(__float_as_uint(x[2])), "r"(__float_as_uint(x[3])),
      "r"(__float_as_uint(x[4])), "r"(__float_as_uint(x[5])), "r"(__float_as_uint(x[6])), "r"(__float_as_uint(x[7])),
      "r"(__float_as_uint(x[8])), "r"(__float_as_uint(x[9])), "r"(__float_as_uint(x[10])), "r"(__float_as_uint(x[11])),
      "r"(__float_as_uint(x[12])), "r"(__float_as_uint(x[13])), "r"(__float_as_uint(x[14])), "r"(__float_as_uint(x[15]))
      : "memory");
}

// E2M1 codes of fl(x0 / den) (low nibble) and fl(x1 / den), r = fl(1 / den).
__device__ __forceinline__ uint32_t e2m1x2_quot(float x0, float x1, float den, float r) {
  const float q0 = __fmul_rn(x0, r), q1 = __fmul_rn(x1, r);
  const uint32_t lo = e2m1x2_from_f32(__fmul_rn(q0, kBracketLo), __fmul_rn(q1, kBracketLo));
  const uint32_t hi = e2m1x2_from_f32(__fmul_rn(q0, kBracketHi), __fmul_rn(q1, kBracketHi));
  if (lo == hi) return lo;
  return e2m1x2_from_f32(__fdiv_rn(x0, den), __fdiv_rn(x1, den));
}

// E4M3 bytes of fl(x0 / den) (low byte) and fl(x1 / den), r = fl(1 / den).
__device__ __forceinline__ uint32_t e4m3x2_quot(float x0, float x1, float den, float r) {
  const float q0 = __fmul_rn(x0, r), q1 = __fmul_rn(x1, r);
  const uint32_t lo = e4m3x2_from_f32(__fmul_rn(q0, kBracketLo), __fmul_rn(q1, kBracketLo));
  const uint32_t hi = e4m3x2_from_f32(__fmul_rn(q0, kBracketHi), __fmul_rn(q1, kBracketHi));
  if (lo == hi) return lo;
  return e4m3x2_from_f32(__fdiv_rn(x0, den), __fdiv_rn(x1, den));
}

}  // namespace nvkv
