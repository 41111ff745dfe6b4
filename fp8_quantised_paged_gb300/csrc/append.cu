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
// A group of lanes per (token, kv head, K-or-V) row, several rows per warp.
// Each lane owns 8 contiguous values per 16-byte chunk (one 16-byte load and
// 8 bytes of codes; a lane with consecutive chunks stores two chunks' codes
// at once).  Every quotient is the IEEE fp32 round-to-nearest one
// (__fdiv_rn for the scales and static channel scales; for per-token and
// per-group scales a reciprocal per scale and a corrected product, see
// quot_rn) and the FP8 cast is the hardware cvt.rn.satfinite (INT8:
// cvt.rni), so codes and scales are bit-exact with the definition.
#include <float.h>

#include "common.cuh"
#include "internal.h"
#include "plan.cuh"

namespace fp8pa {

namespace {

constexpr int kAppendWarps = 8;

// x / s rounded to nearest even, given r = rn(1 / s): y = rn(x r) lies within
// two units in the last place of x / s, the residual y s - x is exact in one
// fma, and one more fma adds its correction (the final correction step of
// Markstein's division, "Computation of elementary functions on the IBM
// RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990).  Checked
// exhaustively against IEEE x / s for the scales this file forms,
// s = max(rn(m / FMAX), 1e-12) with m a bf16 absmax and FMAX 448, 57344 or
// 127, over every bf16 m and every bf16 x with |x| <= m: equal bit for bit,
// except where x is an fp32 subnormal and the residual underflows; both
// quotients are then below 2^-73, so every FP8 and INT8 code is zero (of
// x's sign) either way.  Signed zeros come out as x / s gives them.  An
// infinite scale (an infinite input) takes __fdiv_rn instead.
__device__ __forceinline__ float quot_rn(float x, float s, float r) {
  const float y = __fmul_rn(x, r);
  const float e = fmaf(y, s, -x);
  return fmaf(-e, r, y);
}

// The absmax scale max(rn(m / FMAX), 1e-12) of a row or group whose bf16
// absmax is m, by the same corrected product with the constant rn(1 / FMAX)
// (equal to IEEE m / FMAX for every finite bf16 m, checked exhaustively);
// an infinite m gives an infinite scale, as the division does.
template <int FMT>
__device__ __forceinline__ float scale_of(float m) {
  constexpr float kFmax = code_max<FMT>();
  constexpr float kRcp = 1.0f / kFmax;
  return m <= FLT_MAX ? fmaxf(quot_rn(m, kFmax, kRcp), 1e-12f) : m;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Lanes per row: a sub-group of LPR lanes (a power of two, at most 32)
// appends one row; a lane owns R of the row's 16-byte chunks -- chunks sl,
// sl + LPR, ... (strided, CONSEC false), or R consecutive chunks sl * R ..
// sl * R + R - 1 (CONSEC true: the bulk kernel's per-token and static-channel
// modes, where fewer lanes per row spread each row's bookkeeping over more
// values) -- so a warp covers 32 / LPR rows per step.
template <int LPR, int R, bool CONSEC>
__device__ __forceinline__ int chunk_of(int sl, int r) {
  return CONSEC ? sl * R + r : sl + LPR * r;
}

// Row `row` of the call: its (K-or-V, head) index `rem` (-1 past the end), its
// slot, and its bf16 words (zeros where the lane has no chunk), left packed
// so that nothing waits on the loads until the row is stored.
template <int LPR, int R, bool CONSEC = false>
__device__ __forceinline__ void load_row(const AppendArgs& a, long row, int sl, uint4 (&w)[R],
                                         int& rem, int& slot) {
  const int per_tok = a.hkv * a.ntens;
  const bool in = row < static_cast<long>(a.num_tokens) * per_tok;
  const uint32_t r32 = in ? static_cast<uint32_t>(row) : 0u;
  const uint32_t t = fast_div(r32, a.div_tok);
  const int rw = static_cast<int>(r32 - t * static_cast<uint32_t>(per_tok));
  rem = in ? rw : -1;
  slot = in ? __ldg(a.slot_mapping + t) : -1;
  const bool second = rw >= a.hkv;  // the V row
  const uint16_t* x =
      (second ? a.src[1] : a.src[0]) +
      (static_cast<long>(t) * a.hkv + (second ? rw - a.hkv : rw)) * a.d;
  const int nch = a.d / 8;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int ci = chunk_of<LPR, R, CONSEC>(sl, r);
    w[r] = (in && ci < nch) ? __ldg(reinterpret_cast<const uint4*>(x + ci * 8))
                            : make_uint4(0u, 0u, 0u, 0u);
  }
}

// Scale, round and scatter one loaded row (the whole sub-group joins the
// shuffles, also for rows that are skipped: past the end, a negative slot,
// or a slot past the pool).
template <int FMT, int MODE, int LPR, int R, bool CONSEC = false>
__device__ __forceinline__ void store_row(const AppendArgs& a, const uint4 (&w)[R], int rem,
                                          int slot, int sl) {
  // per-group modes need the chunks of a group on consecutive lanes
  static_assert(!CONSEC || MODE == FP8PA_SCALE_TOKEN_HEAD || MODE == FP8PA_SCALE_CHANNEL_STATIC,
                "consecutive chunks serve the per-token and static-channel modes only");
  constexpr float kFmax = code_max<FMT>();
  constexpr int kEmax = FMT == FP8PA_E4M3 ? 8 : 15;  // exponent of the largest normal
  const int nch = a.d / 8;
  const int which = rem >= a.hkv ? 1 : 0;
  const int h = rem - which * a.hkv;
  const uint32_t bq = slot < 0 ? 0u : fast_div(static_cast<uint32_t>(slot), a.div_bs);
  const long blk = slot < 0 ? -1 : static_cast<long>(bq);
  const int off = slot < 0 ? 0 : slot - static_cast<int>(bq) * a.bs;
  const bool live = rem >= 0 && slot >= 0 && blk < a.num_blocks;
  if (rem >= 0 && blk >= a.num_blocks && sl == 0) raise_error(a.err, FP8PA_DEVERR_SLOT_RANGE);
  const long crow = live ? (blk * a.hkv + h) * a.bs + off : 0;
  uint8_t* dst = live ? (which ? a.cache[1] : a.cache[0]) + crow * a.d : nullptr;
  float* scl = which ? a.scale[1] : a.scale[0];

  float v[R][8];
#pragma unroll
  for (int r = 0; r < R; ++r) bf16x8_to_f32(w[r], v[r]);
  float cmax[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    cmax[r] = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) cmax[r] = fmaxf(cmax[r], fabsf(v[r][e]));
  }
  float s[R], rs[R];  // scales and (per-token and per-group modes) their reciprocals
  if constexpr (MODE == FP8PA_SCALE_TOKEN_HEAD) {
    float m = 0.0f;
#pragma unroll
    for (int r = 0; r < R; ++r) m = fmaxf(m, cmax[r]);
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float sc = scale_of<FMT>(m);
    const float rc = __frcp_rn(sc);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      s[r] = sc;
      rs[r] = rc;
    }
    if (live && sl == 0) scl[crow] = sc;
  } else if constexpr (MODE == FP8PA_SCALE_TOKEN_GROUP) {
    const int lpg = a.gs / 8;  // lanes per group: a power of two <= LPR
    const int ngroups = a.d / a.gs;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float m = cmax[r];
      for (int o = 1; o < lpg; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      s[r] = scale_of<FMT>(m);
      rs[r] = __frcp_rn(s[r]);
      const int ci = sl + LPR * r;
      if (live && ci < nch && (sl & (lpg - 1)) == 0)
        scl[crow * ngroups + (ci * 8) / a.gs] = s[r];
    }
  } else if constexpr (MODE == FP8PA_SCALE_MX_BLOCK) {
    // s = 2^e with e = floor(log2(block absmax)) - emax, read off the fp32
    // exponent field (a zero or subnormal absmax gives the floor, -127);
    // the codes below multiply by 2^-e, which is exact.
    const int lpg = a.gs / 8;
    const int ngroups = a.d / a.gs;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float m = cmax[r];
      for (int o = 1; o < lpg; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      const int ef = (__float_as_int(m) >> 23) & 0xFF;
      const int e = ef == 0 ? -127 : min(127, max(-127, ef - 127 - kEmax));
      s[r] = exp2i(-e);  // the multiplier 2^-e (e <= 119 for bf16 inputs)
      const int ci = sl + LPR * r;
      if (live && ci < nch && (sl & (lpg - 1)) == 0)
        reinterpret_cast<uint8_t*>(scl)[crow * ngroups + (ci * 8) / a.gs] =
            static_cast<uint8_t>(e + 127);
    }
  }
  if (!live) return;

  uint2 pk[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int ci = chunk_of<LPR, R, CONSEC>(sl, r);
    float q[8];
    if constexpr (MODE == FP8PA_SCALE_CHANNEL_STATIC) {
      // a lane past the row's last chunk reads chunk 0's scales (unused)
      const float4* sp = reinterpret_cast<const float4*>(scl + h * a.d + (ci < nch ? ci : 0) * 8);
      const float4 s0 = __ldg(sp), s1 = __ldg(sp + 1);
      const float sc[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) q[e] = __fdiv_rn(v[r][e], sc[e]);
    } else if constexpr (MODE == FP8PA_SCALE_MX_BLOCK) {
#pragma unroll
      for (int e = 0; e < 8; ++e) q[e] = v[r][e] * s[r];
    } else if (s[r] <= FLT_MAX) {
#pragma unroll
      for (int e = 0; e < 8; ++e) q[e] = quot_rn(v[r][e], s[r], rs[r]);
    } else {  // an infinite input made the scale infinite
#pragma unroll
      for (int e = 0; e < 8; ++e) q[e] = __fdiv_rn(v[r][e], s[r]);
    }
    pk[r].x = f32x2_to_codes2<FMT>(q[0], q[1]) | (f32x2_to_codes2<FMT>(q[2], q[3]) << 16);
    pk[r].y = f32x2_to_codes2<FMT>(q[4], q[5]) | (f32x2_to_codes2<FMT>(q[6], q[7]) << 16);
  }
  if constexpr (CONSEC && R % 2 == 0) {
    // Two chunks per 16-byte store: ci is even, head_dim a multiple of 16
    // and the cache 16-byte aligned, so the store is aligned and, with ci
    // inside the row, so is ci + 1.
#pragma unroll
    for (int r = 0; r < R; r += 2) {
      const int ci = chunk_of<LPR, R, CONSEC>(sl, r);
      if (ci + 1 < nch)
        *reinterpret_cast<uint4*>(dst + ci * 8) =
            make_uint4(pk[r].x, pk[r].y, pk[r + 1].x, pk[r + 1].y);
    }
  } else {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int ci = chunk_of<LPR, R, CONSEC>(sl, r);
      if (ci < nch) *reinterpret_cast<uint2*>(dst + ci * 8) = pk[r];
    }
  }
}

// Few rows (a decode step): one step of 32 / LPR rows per warp, so the
// launch (and the attention waiting on it) ends one load latency after it
// starts.
template <int FMT, int MODE, int LPR, int R>
__device__ __forceinline__ void append_step(const AppendArgs& a, long warp, int lane) {
  constexpr int SG = 32 / LPR;
  const int sg = lane / LPR, sl = lane % LPR;
  uint4 w[R];
  int rem, slot;
  load_row<LPR, R>(a, warp * SG + sg, sl, w, rem, slot);
  store_row<FMT, MODE, LPR, R>(a, w, rem, slot, sl);
}

template <int FMT, int MODE, int LPR, int R>
__global__ void __launch_bounds__(kAppendWarps * 32) append_kernel(AppendArgs a) {
  griddep_wait();  // launched early (programmatic serialisation): inputs may be in flight
  griddep_launch_dependents();
  append_step<FMT, MODE, LPR, R>(a, static_cast<long>(blockIdx.x) * kAppendWarps + (threadIdx.x >> 5),
                                 threadIdx.x & 31);
}

// Many rows (a prefill): a persistent grid whose warps stride over the
// steps of rows with a ring of kStreamDepth steps in registers -- a step's
// loads are issued kStreamDepth - 1 steps before the warp works on it, and
// its words stay packed until then, so loads stay in flight while the warp
// scales and rounds.  Rows are spread over few lanes, each with several
// consecutive 16-byte chunks (stored as 16-byte code words), to share every
// row's index arithmetic.
constexpr int kStreamDepth = 3;

template <int FMT, int MODE, int LPR, int R, bool CONSEC>
__global__ void __launch_bounds__(kAppendWarps * 32) append_stream_kernel(AppendArgs a) {
  griddep_wait();
  griddep_launch_dependents();
  constexpr int SG = 32 / LPR, P = kStreamDepth;
  const int lane = threadIdx.x & 31, sg = lane / LPR, sl = lane % LPR;
  const long nsteps = (static_cast<long>(a.num_tokens) * a.hkv * a.ntens + SG - 1) / SG;
  const long stride = static_cast<long>(gridDim.x) * kAppendWarps;
  const long first = static_cast<long>(blockIdx.x) * kAppendWarps + (threadIdx.x >> 5);
  uint4 v[P][R];
  int rem[P], slot[P];
#pragma unroll
  for (int p = 0; p < P; ++p)
    load_row<LPR, R, CONSEC>(a, (first + p * stride) * SG + sg, sl, v[p], rem[p], slot[p]);
  for (long s0 = first; s0 < nsteps; s0 += P * stride) {
#pragma unroll
    for (int p = 0; p < P; ++p) {
      const long st = s0 + p * stride;
      if (st >= nsteps) break;  // warp-uniform
      store_row<FMT, MODE, LPR, R, CONSEC>(a, v[p], rem[p], slot[p], sl);
      load_row<LPR, R, CONSEC>(a, (st + P * stride) * SG + sg, sl, v[p], rem[p], slot[p]);
    }
  }
}

// A decode step's prologue in one launch: CTA 0's first warp plans the
// split of the attention that follows, the other CTAs append the new rows.
template <int FMT, int MODE, int LPR, int R>
__global__ void __launch_bounds__(kAppendWarps * 32) append_plan_kernel(AppendArgs a, PlanArgs pl) {
  griddep_wait();
  griddep_launch_dependents();
  if (blockIdx.x == 0) {
    if (threadIdx.x < 32)
      plan_warp(pl.seq_lens, pl.batch, pl.qlen, pl.qw, 1, pl.bs, pl.max_blocks, pl.workers,
                pl.plan, pl.err, pl.upages);
    return;
  }
  append_step<FMT, MODE, LPR, R>(
      a, static_cast<long>(blockIdx.x - 1) * kAppendWarps + (threadIdx.x >> 5), threadIdx.x & 31);
}

// Calls of at least this many rows stream through the persistent kernel.
constexpr long kBulkRows = 16384;

template <int FMT, int MODE, int LPR, int R, int SLPR, int SR, bool SCONSEC>
cudaError_t launch_append_shape(const AppendArgs& a, const PlanArgs* pl, cudaStream_t stream) {
  const long rows = static_cast<long>(a.num_tokens) * a.hkv * a.ntens;
  if (rows == 0 && !pl) return cudaSuccess;
  constexpr long kRowsPerCta = static_cast<long>(kAppendWarps) * (32 / LPR);
  const long ctas = (rows + kRowsPerCta - 1) / kRowsPerCta;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kAppendWarps * 32);
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  if (pl) {
    cfg.gridDim = dim3(static_cast<unsigned>(ctas + 1));
    return cudaLaunchKernelEx(&cfg, append_plan_kernel<FMT, MODE, LPR, R>, a, *pl);
  }
  if (rows >= kBulkRows) {
    const auto fn = append_stream_kernel<FMT, MODE, SLPR, SR, SCONSEC>;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    constexpr long kStreamRowsPerCta = static_cast<long>(kAppendWarps) * (32 / SLPR);
    const long sctas = (rows + kStreamRowsPerCta - 1) / kStreamRowsPerCta;
    const long resident = static_cast<long>(sm_count(dev)) *
                          ctas_per_sm(reinterpret_cast<const void*>(fn), kAppendWarps * 32, 0);
    cfg.gridDim = dim3(static_cast<unsigned>(sctas < resident ? sctas : resident));
    return cudaLaunchKernelEx(&cfg, fn, a);
  }
  cfg.gridDim = dim3(static_cast<unsigned>(ctas));
  return cudaLaunchKernelEx(&cfg, append_kernel<FMT, MODE, LPR, R>, a);
}

// pl == nullptr: the append alone; else the fused append + plan prologue.
// Lanes per row follow the row's 16-byte chunks (head_dim / 8): 8 lanes up
// to head_dim 64, 16 at 128, 32 (with 2 or 3 chunks each) beyond 256.  The
// bulk kernel gives a lane 4 consecutive chunks in the per-token and
// static-channel modes (4 lanes per row at head_dim 128).
template <int FMT, int MODE>
cudaError_t launch_append_r(const AppendArgs& a, const PlanArgs* pl, cudaStream_t stream) {
  const int nch = a.d / 8;
  if constexpr (MODE == FP8PA_SCALE_TOKEN_HEAD || MODE == FP8PA_SCALE_CHANNEL_STATIC) {
    if (nch <= 8) return launch_append_shape<FMT, MODE, 8, 1, 2, 4, true>(a, pl, stream);
    if (nch <= 16) return launch_append_shape<FMT, MODE, 16, 1, 4, 4, true>(a, pl, stream);
    if (nch <= 32) return launch_append_shape<FMT, MODE, 32, 1, 8, 4, true>(a, pl, stream);
    if (nch <= 64) return launch_append_shape<FMT, MODE, 32, 2, 16, 4, true>(a, pl, stream);
  } else {
    if (nch <= 8) return launch_append_shape<FMT, MODE, 8, 1, 8, 1, false>(a, pl, stream);
    if (nch <= 16) return launch_append_shape<FMT, MODE, 16, 1, 16, 1, false>(a, pl, stream);
    if (nch <= 32) return launch_append_shape<FMT, MODE, 32, 1, 32, 1, false>(a, pl, stream);
    if (nch <= 64) return launch_append_shape<FMT, MODE, 32, 2, 32, 2, false>(a, pl, stream);
  }
  return launch_append_shape<FMT, MODE, 32, 3, 32, 3, false>(a, pl, stream);
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
