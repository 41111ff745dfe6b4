// append.cu -- the append step: absmax scale, FP8 (or INT8) rounding and the
// slot scatter into the paged cache; and the static per-channel scale
// calibration.
//
// Method: scale = absmax / 448 (E4M3) or / 57344 (E5M2), clamped below at
// 1e-12, code = fp8(x / scale) ("Llama 3 70B FP8 deployment",
// dpshk.com/news/5605006, sec. 3.1; "FP8混合精度推理全链路部署实战",
// ybb.press/ai-applications/14145.html, sec. 1.1 and 2.3).  One scale per
// (token, kv head), per (token, latent group) ("DeepSeek V4 950",
// 2kiu.com/news/4508674, sec. 2.2 / 2.4) or a static one per channel
// ("DeepSeek-V4.1 512K", hotelren.com/news/5711065, sec. 3.3).  Codes land in
// block slot / block_size at offset slot % block_size (same page, sec. 3.3).
// MX block mode: a power-of-two scale per block of 16 or 32 dims (E8M0).
// The symmetric INT8 codec takes 127 as the maximum and rounds x / scale to
// the nearest integer, ties to even, clamped to [-127, 127].
//
// One warp per (token, kv head, K-or-V) row.  Each lane owns 8 contiguous
// values (one 16-byte load, one 8-byte code store).  The divisions are IEEE
// fp32 round-to-nearest (__fdiv_rn) and the FP8 cast is the hardware
// cvt.rn.satfinite (INT8: cvt.rni), so codes and scales are bit-exact with
// the definition.
#include "common.cuh"
#include "internal.h"
#include "plan.cuh"

namespace fp8pa {

namespace {

constexpr int kAppendWarps = 8;

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// One (token, kv head, K-or-V) row per warp.
template <int FMT, int MODE, int R>
__device__ __forceinline__ void append_row(const AppendArgs& a, long row, int lane) {
  const int per_tok = a.hkv * a.ntens;
  if (row >= static_cast<long>(a.num_tokens) * per_tok) return;
  const int t = static_cast<int>(row / per_tok);
  const int rem = static_cast<int>(row % per_tok);
  const int which = rem / a.hkv;
  const int h = rem % a.hkv;
  const int slot = __ldg(a.slot_mapping + t);
  if (slot < 0) return;  // padding token
  const long blk = slot / a.bs;
  const int off = slot % a.bs;
  if (blk >= a.num_blocks) {
    if (lane == 0) raise_error(a.err, FP8PA_DEVERR_SLOT_RANGE);
    return;
  }
  const uint16_t* x = a.src[which] + (static_cast<long>(t) * a.hkv + h) * a.d;
  const long crow = (blk * a.hkv + h) * a.bs + off;
  uint8_t* dst = a.cache[which] + crow * a.d;
  const int nch = a.d / 8;

  float v[R][8];
  float cmax[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int ci = lane + 32 * r;
    cmax[r] = 0.0f;
    if (ci < nch) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(x + ci * 8));
      bf16x8_to_f32(u, v[r]);
#pragma unroll
      for (int e = 0; e < 8; ++e) cmax[r] = fmaxf(cmax[r], fabsf(v[r][e]));
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) v[r][e] = 0.0f;
    }
  }

  constexpr float kFmax = code_max<FMT>();
  constexpr int kEmax = FMT == FP8PA_E4M3 ? 8 : 15;  // exponent of the largest normal
  float s[R];
  if constexpr (MODE == FP8PA_SCALE_TOKEN_HEAD) {
    float m = 0.0f;
#pragma unroll
    for (int r = 0; r < R; ++r) m = fmaxf(m, cmax[r]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float sc = fmaxf(__fdiv_rn(m, kFmax), 1e-12f);
#pragma unroll
    for (int r = 0; r < R; ++r) s[r] = sc;
    if (lane == 0) a.scale[which][crow] = sc;
  } else if constexpr (MODE == FP8PA_SCALE_TOKEN_GROUP) {
    const int lpg = a.gs / 8;  // lanes per group: a power of two <= 32
    const int ngroups = a.d / a.gs;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float m = cmax[r];
      for (int o = 1; o < lpg; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      s[r] = fmaxf(__fdiv_rn(m, kFmax), 1e-12f);
      const int ci = lane + 32 * r;
      if (ci < nch && (lane & (lpg - 1)) == 0)
        a.scale[which][crow * ngroups + (ci * 8) / a.gs] = s[r];
    }
  } else if constexpr (MODE == FP8PA_SCALE_MX_BLOCK) {
    // s = 2^e with e = floor(log2(block absmax)) - emax, read off the fp32
    // exponent field (a zero or subnormal absmax gives the floor, -127); the
    // codes below multiply by 2^-e, which is exact.
    const int lpg = a.gs / 8;
    const int ngroups = a.d / a.gs;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float m = cmax[r];
      for (int o = 1; o < lpg; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      const int ef = (__float_as_int(m) >> 23) & 0xFF;
      const int e = ef == 0 ? -127 : min(127, max(-127, ef - 127 - kEmax));
      s[r] = exp2i(-e);  // the multiplier 2^-e (e <= 119 for bf16 inputs)
      const int ci = lane + 32 * r;
      if (ci < nch && (lane & (lpg - 1)) == 0)
        reinterpret_cast<uint8_t*>(a.scale[which])[crow * ngroups + (ci * 8) / a.gs] =
            static_cast<uint8_t>(e + 127);
    }
  }

#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int ci = lane + 32 * r;
    if (ci >= nch) continue;
    float q[8];
    if constexpr (MODE == FP8PA_SCALE_CHANNEL_STATIC) {
      const float4* sp = reinterpret_cast<const float4*>(a.scale[which] + h * a.d + ci * 8);
      const float4 s0 = __ldg(sp), s1 = __ldg(sp + 1);
      const float sc[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) q[e] = __fdiv_rn(v[r][e], sc[e]);
    } else if constexpr (MODE == FP8PA_SCALE_MX_BLOCK) {
#pragma unroll
      for (int e = 0; e < 8; ++e) q[e] = v[r][e] * s[r];
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) q[e] = __fdiv_rn(v[r][e], s[r]);
    }
    uint2 packed;
    packed.x = f32x2_to_codes2<FMT>(q[0], q[1]) | (f32x2_to_codes2<FMT>(q[2], q[3]) << 16);
    packed.y = f32x2_to_codes2<FMT>(q[4], q[5]) | (f32x2_to_codes2<FMT>(q[6], q[7]) << 16);
    *reinterpret_cast<uint2*>(dst + ci * 8) = packed;
  }
}

template <int FMT, int MODE, int R>
__global__ void __launch_bounds__(kAppendWarps * 32) append_kernel(AppendArgs a) {
  griddep_wait();  // launched early (programmatic serialisation): inputs may be in flight
  griddep_launch_dependents();
  append_row<FMT, MODE, R>(a, static_cast<long>(blockIdx.x) * kAppendWarps + (threadIdx.x >> 5),
                           threadIdx.x & 31);
}

// A decode step's prologue in one launch: CTA 0's first warp plans the
// split of the attention that follows, the other CTAs append the new rows.
template <int FMT, int MODE, int R>
__global__ void __launch_bounds__(kAppendWarps * 32) append_plan_kernel(AppendArgs a, PlanArgs pl) {
  griddep_wait();
  griddep_launch_dependents();
  if (blockIdx.x == 0) {
    if (threadIdx.x < 32)
      plan_warp(pl.seq_lens, pl.batch, pl.qlen, pl.qw, 1, pl.bs, pl.max_blocks, pl.workers,
                pl.plan, pl.err);
    return;
  }
  append_row<FMT, MODE, R>(a,
                           static_cast<long>(blockIdx.x - 1) * kAppendWarps + (threadIdx.x >> 5),
                           threadIdx.x & 31);
}

// pl == nullptr: the append alone; else the fused append + plan prologue.
template <int FMT, int MODE>
cudaError_t launch_append_r(const AppendArgs& a, const PlanArgs* pl, cudaStream_t stream) {
  const long rows = static_cast<long>(a.num_tokens) * a.hkv * a.ntens;
  if (rows == 0 && !pl) return cudaSuccess;
  const dim3 grid(
      static_cast<unsigned>((rows + kAppendWarps - 1) / kAppendWarps + (pl ? 1 : 0)));
  const int nch = a.d / 8;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kAppendWarps * 32);
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  if (pl) {
    if (nch <= 32) return cudaLaunchKernelEx(&cfg, append_plan_kernel<FMT, MODE, 1>, a, *pl);
    if (nch <= 64) return cudaLaunchKernelEx(&cfg, append_plan_kernel<FMT, MODE, 2>, a, *pl);
    return cudaLaunchKernelEx(&cfg, append_plan_kernel<FMT, MODE, 3>, a, *pl);
  }
  if (nch <= 32) return cudaLaunchKernelEx(&cfg, append_kernel<FMT, MODE, 1>, a);
  if (nch <= 64) return cudaLaunchKernelEx(&cfg, append_kernel<FMT, MODE, 2>, a);
  return cudaLaunchKernelEx(&cfg, append_kernel<FMT, MODE, 3>, a);
}

template <int FMT>
cudaError_t launch_append_m(const AppendArgs& a, int mode, const PlanArgs* pl,
                            cudaStream_t stream) {
  switch (mode) {
    case FP8PA_SCALE_TOKEN_HEAD:
      return launch_append_r<FMT, FP8PA_SCALE_TOKEN_HEAD>(a, pl, stream);
    case FP8PA_SCALE_CHANNEL_STATIC:
      return launch_append_r<FMT, FP8PA_SCALE_CHANNEL_STATIC>(a, pl, stream);
    case FP8PA_SCALE_MX_BLOCK:  // FP8 only (rejected for INT8 by the caller)
      if constexpr (FMT != FP8PA_INT8) return launch_append_r<FMT, FP8PA_SCALE_MX_BLOCK>(a, pl, stream);
      return cudaErrorInvalidValue;
    default:
      return launch_append_r<FMT, FP8PA_SCALE_TOKEN_GROUP>(a, pl, stream);
  }
}

// ---------------------------------------------------------------- calibration
constexpr int kCalTokens = 256;  // tokens per CTA row of the grid

// Running per-channel absmax: each thread owns 8 channels over kCalTokens
// tokens and folds its maximum into `amax_bits` (non-negative floats order
// like their bit patterns, so an unsigned atomicMax is a float max).
__global__ void __launch_bounds__(256) chanmax_kernel(const uint16_t* x, int n, int hd,
                                                      uint32_t* amax_bits) {
  const int ci = blockIdx.x * blockDim.x + threadIdx.x;
  if (ci * 8 >= hd) return;
  const int t0 = blockIdx.y * kCalTokens;
  const int t1 = min(n, t0 + kCalTokens);
  float m[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int t = t0; t < t1; ++t) {
    float f[8];
    bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(x + static_cast<long>(t) * hd + ci * 8)),
                  f);
#pragma unroll
    for (int e = 0; e < 8; ++e) m[e] = fmaxf(m[e], fabsf(f[e]));
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) atomicMax(amax_bits + ci * 8 + e, __float_as_uint(m[e]));
}

template <int FMT>
__global__ void chanscale_finalize_kernel(const float* amax, float* s, int hd) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= hd) return;
  s[i] = fmaxf(__fdiv_rn(amax[i], code_max<FMT>()), 1e-12f);
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, int fmt, int mode, cudaStream_t stream) {
  switch (fmt) {
    case FP8PA_E4M3: return launch_append_m<FP8PA_E4M3>(a, mode, nullptr, stream);
    case FP8PA_E5M2: return launch_append_m<FP8PA_E5M2>(a, mode, nullptr, stream);
    default: return launch_append_m<FP8PA_INT8>(a, mode, nullptr, stream);
  }
}

cudaError_t launch_append_plan(const AppendArgs& a, int fmt, int mode, const PlanArgs& pl,
                               cudaStream_t stream) {
  switch (fmt) {
    case FP8PA_E4M3: return launch_append_m<FP8PA_E4M3>(a, mode, &pl, stream);
    case FP8PA_E5M2: return launch_append_m<FP8PA_E5M2>(a, mode, &pl, stream);
    default: return launch_append_m<FP8PA_INT8>(a, mode, &pl, stream);
  }
}

cudaError_t launch_channel_absmax(const uint16_t* x, int num_tokens, int hd, float* amax,
                                  cudaStream_t stream) {
  if (num_tokens > 0) {
    const dim3 grid((hd / 8 + 255) / 256, (num_tokens + kCalTokens - 1) / kCalTokens);
    chanmax_kernel<<<grid, 256, 0, stream>>>(x, num_tokens, hd, reinterpret_cast<uint32_t*>(amax));
  }
  return cudaGetLastError();
}

cudaError_t launch_scales_from_absmax(const float* amax, int n, int fmt, float* out,
                                      cudaStream_t stream) {
  const int blocks = (n + 255) / 256;
  if (fmt == FP8PA_E4M3)
    chanscale_finalize_kernel<FP8PA_E4M3><<<blocks, 256, 0, stream>>>(amax, out, n);
  else if (fmt == FP8PA_E5M2)
    chanscale_finalize_kernel<FP8PA_E5M2><<<blocks, 256, 0, stream>>>(amax, out, n);
  else
    chanscale_finalize_kernel<FP8PA_INT8><<<blocks, 256, 0, stream>>>(amax, out, n);
  return cudaGetLastError();
}

cudaError_t launch_channel_scales(const uint16_t* x, int num_tokens, int hd, int fmt, float* out,
                                  cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(out, 0, sizeof(float) * static_cast<size_t>(hd), stream);
  if (e != cudaSuccess) return e;
  e = launch_channel_absmax(x, num_tokens, hd, out, stream);
  if (e != cudaSuccess) return e;
  return launch_scales_from_absmax(out, hd, fmt, out, stream);
}

}  // namespace fp8pa
