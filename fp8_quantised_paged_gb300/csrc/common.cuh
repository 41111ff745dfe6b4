// common.cuh -- device helpers shared by the library's kernels (sm_103a).
// Inline PTX for the async-copy engine (TMA tensor and bulk copies with
// mbarrier completion), FP8 <-> f16/f32 conversions, the legacy warp MMA used
// for the tiny grouped-query contraction, and the device error word.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fp8pa.h"

namespace fp8pa {

// ---------------------------------------------------------------- errors
__device__ __forceinline__ void raise_error(uint32_t* err, uint32_t bit) {
  if (err) atomicOr(err, bit);
}

// ---------------------------------------------------------------- smem / mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Make initialised barriers visible to the async proxy (the copy engine).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Whether phase `parity` of `bar` has completed, without waiting.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` for at most ~`limit_cycles` SM cycles.
// Returns false if the wait ran out (the caller records an error and stops).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  long long limit_cycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit_cycles) return false;
  }
  return true;
}

// ---------------------------------------------------------------- async copies
// 2-D tiled tensor copy global -> shared, completing on `bar` (tx bytes).
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- shared loads
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// ---------------------------------------------------------------- code conversions
// INT8 codes -> f16, exactly.  A code is stored as its integer b + 128
// (excess-128, b in [-127, 127]), so the byte itself becomes the low
// mantissa byte of the f16 1024 (giving 1024 + b + 128) and 1152 is
// subtracted: one byte permute and one f16 subtract per pair.  `sel` picks
// the two bytes of `four_codes`.
__device__ __forceinline__ uint32_t int8x2_to_f16x2(uint32_t four_codes, uint32_t sel) {
  const uint32_t biased = __byte_perm(four_codes, 0x64646464u, sel);
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&biased),
                            __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480)));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// Two codes (low byte = element 0) -> f16x2, exact for every format.
template <int FMT>
__device__ __forceinline__ uint32_t codes2_to_f16x2(uint32_t two_codes) {
  if constexpr (FMT == FP8PA_INT8) return int8x2_to_f16x2(two_codes, 0x5140u);
  uint32_t r;
  const uint16_t v = static_cast<uint16_t>(two_codes & 0xFFFFu);
  if constexpr (FMT == FP8PA_E4M3) {
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  } else {
    asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(r) : "h"(v));
  }
  return r;
}

// Four codes (byte i = element i) -> two f16x2: lo = elements 0,1 and
// hi = elements 2,3; the two halves of the word are converted in place.
template <int FMT>
__device__ __forceinline__ void codes4_to_f16x2x2(uint32_t four_codes, uint32_t& lo, uint32_t& hi) {
  if constexpr (FMT == FP8PA_INT8) {
    lo = int8x2_to_f16x2(four_codes, 0x5140u);
    hi = int8x2_to_f16x2(four_codes, 0x5342u);
  } else if constexpr (FMT == FP8PA_E4M3) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(four_codes));
  } else {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e5m2x2 %0, l;\n\tcvt.rn.f16x2.e5m2x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(four_codes));
  }
}

// Two fp32 values -> two codes (lo -> low byte), round to nearest even.
// FP8: finite overflow saturated to +-max, NaN to NaN.  INT8: clamped to
// [-127, 127] (infinities too), NaN to 0, stored + 128.
template <int FMT>
__device__ __forceinline__ uint32_t f32x2_to_codes2(float lo, float hi) {
  if constexpr (FMT == FP8PA_INT8) {
    const int a = min(127, max(-127, __float2int_rn(lo))) + 128;
    const int b = min(127, max(-127, __float2int_rn(hi))) + 128;
    return static_cast<uint32_t>(a) | (static_cast<uint32_t>(b) << 8);
  }
  uint16_t r;
  if constexpr (FMT == FP8PA_E4M3) {
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  } else {
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  }
  return static_cast<uint32_t>(r);
}

// Largest code magnitude: FMAX of the absmax / FMAX scale.
template <int FMT>
__host__ __device__ constexpr float code_max() {
  return FMT == FP8PA_E4M3 ? 448.0f : (FMT == FP8PA_E5M2 ? 57344.0f : 127.0f);
}

// ---------------------------------------------------------------- math
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// (x0, x1) as two f16x2 planes: hi = f16(x), lo = f16(x - hi); hi + lo carries
// about 22 significant bits.
__device__ __forceinline__ void split_pack(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(x0, x1);
  const float2 hf = __half22float2(h);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = pack_half2(x0 - hf.x, x1 - hf.y);
}

// 2^e as a float for integer e (0 below the normal range).
__device__ __forceinline__ float exp2i(int e) {
  if (e < -126) return 0.0f;
  if (e > 127) e = 127;
  return __int_as_float((e + 127) << 23);
}

// The smallest E with |x| < 2^E for finite x > 0 (x = 0 gives -127).
__device__ __forceinline__ int exp_above(float x) {
  const int b = (__float_as_int(x) >> 23) & 0xFF;
  return b == 0 ? -127 : b - 126;
}

// D (16x8 f32) += A (16x16 f16, row) * B (16x8 f16, col).
__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start before its predecessor finishes; it must call
// griddep_wait() before touching anything the predecessor writes.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Visible length of virtual request v in a causal chunk of `qlen` queries per
// request: query i of request b (v = b * qlen + i) sees the first
// seq_lens[b] - (qlen - 1 - i) cached tokens; qlen = 1 is plain decode.
// `bad` reports a length outside [0, cap], or shorter than the chunk.
__device__ __forceinline__ int visible_len(const int32_t* seq_lens, int v, int qlen, int cap,
                                           bool* bad) {
  const int L = seq_lens[v / qlen];
  *bad = L < 0 || L > cap || (qlen > 1 && L < qlen);
  const int vis = min(L, cap) - (qlen - 1 - v % qlen);
  return vis < 0 ? 0 : vis;
}

// Cycles a bounded wait may spin (about two seconds at GB300 clocks).
constexpr long long kWaitLimitCycles = 4000000000ll;

}  // namespace fp8pa
