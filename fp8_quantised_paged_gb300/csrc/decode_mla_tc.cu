// decode_mla_tc.cu -- split-K paged decode attention for the shared-latent
// (MLA) layout on the fifth-generation tensor cores (tcgen05 + TMEM), for
// FP8 codes.
//
// Method ("DeepSeek V4 950: whole-network FP8 dataflow", 2kiu.com/news/4508674,
// sec. 2.2: one cached latent per token, one scale per latent group; sec. 2.3:
// softmax and accumulation in FP32):
//   z[h,t] = sm_scale * q[h,:576] . c^[t,:576],  o[h,:] = sum_t softmax(z)[h,t] c^[t,:512]
//   c^[t,d] = decode(code[t,d]) * s[t, d / 64]   (9 groups of 64 dims)
//
// GB300 design.  A CTA serves 64 query heads of one page range (two CTAs per
// range cover 128 heads); its steps are page pairs (128 tokens).
//  * QK^T on FP8 tensor cores: S^T[t,h] = sum_g s[t,g] sum_{d in g} code[t,d] q[h,d].
//    The pair's codes arrive by TMA as 64-byte-swizzled tiles, one per 64-dim
//    group, and are the A operand (M = 128 tokens) as they are; q is held as
//    two E4M3 terms hi + lo (B operand, N = 64 heads), exact to about 2^-8 of
//    each element and far below that against the largest.  Each group's
//    product accumulates in its own TMEM buffer; the score warps (one token
//    per thread) read it back, scale it by the token's group scale in FP32
//    and add: the scores are products of codes and q, scaled exactly.
//  * FP32 online softmax in the log2 domain: per-head running maxima across
//    the 128 token lanes (warp butterflies, then shared memory); when a
//    head's maximum rises its column of O is rescaled in TMEM.
//  * P.V on bf16 tensor cores: O^T[dv,h] (M = 128 dv per tile, four tiles,
//    N = 64 heads, K = tokens) += V^T P.  A = V^ = code * scale split as
//    bf16 hi + lo, built per 16-token K step into a four-slot ring by the
//    builder warps; B = P as bf16 hi + lo; three MMAs per step (hi.hi, hi.lo,
//    lo.hi) keep ~16 significant bits on both sides with the full FP32 range.
//  * Roles: warps 0-3 score, softmax and write the partials; warps 4-7 build
//    V^; lane 0 of warp 8 issues the MMAs; warp 9 issues a pair's copies (a
//    lane per latent group and page) as soon as the stage is free, with the
//    block ids read beforehand.  Handshakes are mbarriers; every wait is
//    bounded.  Pieces are merged by merge.cu.
#include <float.h>

#include "common.cuh"
#include "internal.h"
#include "plan.cuh"
#include "tc.cuh"

namespace fp8pa {

namespace {

constexpr int kDk = 576, kDv = 512, kBs = 64, kGroups = 9;
constexpr int kH = 64;              // query heads per CTA: N of every MMA
constexpr int kT = 128;             // tokens per step (a page pair)
constexpr int kThreads = 10 * 32;   // 4 score warps, 4 builder warps, 1 issuing warp, 1 copying warp
constexpr int kNB = 3;              // score buffers in TMEM (64 columns each)
constexpr int kVS = 4;              // V^ ring slots (16 tokens each), handed over in pairs
constexpr int kVD = kVS / 2;        // double slots
constexpr int kTile = kT * 64;      // one 64-dim group of a pair: 128 rows x 64 B
constexpr int kPageScales = kBs * kGroups * 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 256;     // score buffers: columns 256 + 64 b
constexpr uint32_t kColSum = 448;   // per-token partial sums of p: 64 columns
// The running maximum of a head moves only when a score passes it by more
// than kTau (log2 units): p stays below 2^kTau, and most steps skip the
// cross-token reduction.  Any choice is exact: O, the sums and the maximum
// written with the piece always agree.
constexpr float kTau = 8.f;
constexpr float kNegBig = -1e30f;   // running maximum before the first token

struct Smem {
  static constexpr int kCodes = 0;                              // 9 tiles of 8 KB (SW64)
  static constexpr int kScales = kCodes + kGroups * kTile;      // 2 pages of scales
  static constexpr int kQ = kScales + 2 * kPageScales;          // 2 terms x 9 x 4 KB (SW64)
  static constexpr int kP = kQ + 2 * kGroups * kH * 64;         // 2 terms x 16 KB
  static constexpr int kV = kP + 2 * kT * kH * 2;               // 4 slots x 2 terms x 4 KB
  static constexpr int kRed = kV + kVS * 2 * 4096;              // f32 [4][64] maxima / sums
  static constexpr int kM = kRed + 4 * kH * 4;                  // f32 [64] running maxima
  static constexpr int kAlpha = kM + kH * 4;                    // f32 [64] rescale factors
  static constexpr int kMisc = kAlpha + kH * 4;                 // f32 [16]: flags
  static constexpr int kTmem = kMisc + 64;                      // u32 TMEM base
  static constexpr int kBars = kTmem + 16;                      // mbarriers
  static constexpr int kNumBars = 1 + 2 * kNB + 1 + 1 + 2 * kVD + 1 + 1;
  static constexpr int kBytes = kBars + kNumBars * 8 + 1024;    // + alignment slack
};
static_assert(Smem::kScales % 16 == 0 && Smem::kQ % 512 == 0 && Smem::kP % 16 == 0 &&
                  Smem::kV % 16 == 0 && Smem::kM % 16 == 0 && Smem::kBars % 8 == 0,
              "operand alignment");

struct TcParams {
  const uint16_t* q;
  const uint8_t* cache;
  const float* scale;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int* plan;
  float* part_ml;
  float* part_o;
  uint32_t* err;
  int B, hq, H, max_blocks, num_blocks, qlen;
  uint32_t idesc_qk;
  float qk_scale_log2;
};

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t x) {
  return *reinterpret_cast<const __nv_bfloat162*>(&x);
}
__device__ __forceinline__ uint32_t bf2_bits(__nv_bfloat162 x) {
  return *reinterpret_cast<const uint32_t*>(&x);
}

// Byte offset of byte `d` (0..63) of row `r` in a 64-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw64(int r, int d) {
  return static_cast<uint32_t>(r * 64 + ((((d >> 4) ^ (r >> 1)) & 3) << 4) + (d & 15));
}

// Two FP8 codes (bytes `sel` picks from `w`) as a bf16 pair of the same
// values, exactly: the code's sign, exponent and mantissa bits moved into a
// bf16 pattern give value * 2^-120 (E4M3) or 2^-112 (E5M2) -- subnormal
// codes land on bf16 subnormals -- and one bf16 multiply by the power of two
// restores the value.
template <int FMT>
__device__ __forceinline__ __nv_bfloat162 codes2_to_bf16x2(uint32_t w, uint32_t sel) {
  constexpr uint32_t kShift = FMT == FP8PA_E4M3 ? 4 : 5;
  constexpr uint32_t kMask = FMT == FP8PA_E4M3 ? 0x87F087F0u : 0x8FE08FE0u;
  constexpr uint32_t kUnit = FMT == FP8PA_E4M3 ? 0x7B807B80u : 0x77807780u;  // 2^120 | 2^112
  const uint32_t b = (prmt_sign(w, sel) << kShift) & kMask;
  return __hmul2_rn(as_bf2(b), as_bf2(kUnit));
}

// Eight dequantised values c * s as bf16 hi + lo.  s = sh + sl (bf16 each,
// s's leading 16 bits); hi = rn(c * sh), the product's remainder
// c * sh - hi is exact in bf16 (c has 4 significant bits, sh 8), and
// lo = rn(c * sl + remainder): hi + lo holds c * s to about 2^-16.
template <int FMT>
__device__ __forceinline__ void dequant8(uint2 c8, __nv_bfloat162 sh, __nv_bfloat162 sl,
                                         uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 c =
        codes2_to_bf16x2<FMT>(i < 2 ? c8.x : c8.y, (i & 1) ? 0xB3A2u : 0x9180u);
    const __nv_bfloat162 ph = __hmul2_rn(c, sh);
    const __nv_bfloat162 rem = __hfma2(c, sh, __hneg2(ph));
    h[i] = bf2_bits(ph);
    l[i] = bf2_bits(__hfma2(c, sl, rem));
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

template <int FMT, int SEG>
__global__ void __launch_bounds__(kThreads, 1)
    mla_tc_kernel(const __grid_constant__ CUtensorMap tm_lat, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* codes = sm + Smem::kCodes;
  float* scl = reinterpret_cast<float*>(sm + Smem::kScales);
  uint8_t* qs = sm + Smem::kQ;
  uint8_t* ps = sm + Smem::kP;
  uint8_t* vs = sm + Smem::kV;
  float* red = reinterpret_cast<float*>(sm + Smem::kRed);
  float* msm = reinterpret_cast<float*>(sm + Smem::kM);
  float* asm_ = reinterpret_cast<float*>(sm + Smem::kAlpha);
  float* misc = reinterpret_cast<float*>(sm + Smem::kMisc);
  int* abort_flag = reinterpret_cast<int*>(misc + 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + Smem::kTmem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Smem::kBars);
  uint64_t* bar_full = bars;
  uint64_t* bar_qk = bars + 1;
  uint64_t* bar_sfree = bars + 1 + kNB;
  uint64_t* bar_stage = bars + 1 + 2 * kNB;
  uint64_t* bar_pready = bar_stage + 1;
  uint64_t* bar_vfull = bar_pready + 1;
  uint64_t* bar_vfree = bar_vfull + kVD;
  uint64_t* bar_pv = bar_vfree + kVD;
  uint64_t* bar_drain = bar_pv + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float NEG_INF = __int_as_float(0xff800000);
  constexpr uint32_t kVTerm = 4096, kPTerm = kT * kH * 2;
  const uint32_t idesc_pv = tc_idesc(1, 1, 1, 1, 128, kH);  // bf16, both MN-major

  if (tid == 0) {
    mbar_init(bar_full, 1);
    for (int b = 0; b < kNB; ++b) {
      mbar_init(bar_qk + b, 1);
      mbar_init(bar_sfree + b, 4);    // one arrival per score warp
    }
    mbar_init(bar_stage, 1 + 4 + 4);  // tensor core, score warps, builder warps
    mbar_init(bar_pready, 4);
    for (int v = 0; v < kVD; ++v) {
      mbar_init(bar_vfull + v, 8);    // one arrival per builder and score warp
      mbar_init(bar_vfree + v, 1);
    }
    mbar_init(bar_pv, 1);
    mbar_init(bar_drain, 1);
    misc[0] = misc[1] = 0.f;
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tm_lat);
  }
  __syncthreads();
  griddep_wait();
  griddep_launch_dependents();

  const int* uprefix = p.plan + kPlanHeader;
  const int* segbase = uprefix + p.B + 1;
  const int U = *reinterpret_cast<const volatile int*>(p.plan);
  const int upw = *reinterpret_cast<const volatile int*>(p.plan + 1);
  const int hg = blockIdx.x % p.H;    // this CTA's group of 64 heads
  const long wid = blockIdx.x / p.H;  // its range of page pairs
  const long u0 = wid * upw;
  if (u0 >= U) return;  // before any TMEM is held
  const int n_units = static_cast<int>(min(static_cast<long>(upw), U - u0));

  if (warp == 8) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto locate = [&](long u, int& b) {
    int lo = 0, hi = p.B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (uprefix[mid] <= u) lo = mid; else hi = mid;
    }
    b = lo;
  };
  // bounded wait; on expiry the whole CTA gives up (flag, then drains)
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    return tc_wait(bar, parity, abort_flag, p.err);
  };
  // the same, with one answer for the whole warp (tcgen05.ld/st and the
  // warp-level arrivals need every lane to take the same path)
  auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, wait(bar, parity));
  };

  // Barrier phases: every role walks the same units, so each keeps its own
  // copy of the counters.
  int pc = 0;                        // pairs done by this CTA
  int quse[kNB] = {0, 0, 0};         // completions of each score buffer
  int vd = 0;                        // issuer: V^ double slots consumed
  int fills_b = 0, fills_s = 0;      // V^ double slots filled by builders / score warps

  long u = u0;
  const long uend = u0 + n_units;
  while (u < uend) {
    // ---- one segment: the units of request b inside the range
    int b;
    locate(u, b);
    const int first_u = uprefix[b];
    const long seg_end = min(uend, static_cast<long>(uprefix[b + 1]));
    bool bad;
    const int Lb = visible_len(p.seq_lens, b, p.qlen, p.max_blocks * kBs, &bad);
    const int npages = (Lb + kBs - 1) / kBs;
    const long brow = static_cast<long>(b / p.qlen) * p.max_blocks;

    // q of the 64 heads -> two E4M3 terms with a power-of-two normaliser
    // (the largest |q| below 2^8), written as 64-byte-swizzled tiles
    __syncthreads();
    const uint16_t* qsrc = p.q + (static_cast<long>(b) * p.hq + hg * kH) * kDk;
    float amax = 0.f;
    for (int c = tid; c < kH * kDk / 8; c += kThreads) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(qsrc) + c);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int k = 0; k < 4; ++k)
        amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(ww[k] << 16)),
                                 fabsf(__uint_as_float(ww[k] & 0xFFFF0000u))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    amax = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) amax = fmaxf(amax, red[w]);
    const int eq = amax > 0.f ? exp_above(amax) : 0;
    const float fq = exp2i(8 - eq);
    const float zs = p.qk_scale_log2 * exp2i(eq - 8);
    for (int c = tid; c < kH * kDk / 8; c += kThreads) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(qsrc) + c);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
      float x[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        x[2 * k] = __uint_as_float(ww[k] << 16) * fq;
        x[2 * k + 1] = __uint_as_float(ww[k] & 0xFFFF0000u) * fq;
      }
      uint32_t hw[2], lw[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const uint32_t h01 = f32x2_to_codes2<FP8PA_E4M3>(x[4 * k], x[4 * k + 1]);
        const uint32_t h23 = f32x2_to_codes2<FP8PA_E4M3>(x[4 * k + 2], x[4 * k + 3]);
        uint32_t d01, d23;  // the hi codes back as f16 (exact)
        codes4_to_f16x2x2<FP8PA_E4M3>(h01 | (h23 << 16), d01, d23);
        const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&d01));
        const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&d23));
        const uint32_t l01 = f32x2_to_codes2<FP8PA_E4M3>(x[4 * k] - f01.x, x[4 * k + 1] - f01.y);
        const uint32_t l23 =
            f32x2_to_codes2<FP8PA_E4M3>(x[4 * k + 2] - f23.x, x[4 * k + 3] - f23.y);
        hw[k] = h01 | (h23 << 16);
        lw[k] = l01 | (l23 << 16);
      }
      const int h = c / (kDk / 8), col = (c % (kDk / 8)) * 8;
      const int g = col >> 6, d = col & 63;
      const uint32_t off = g * (kH * 64) + sw64(h, d);
      *reinterpret_cast<uint2*>(qs + off) = make_uint2(hw[0], hw[1]);
      *reinterpret_cast<uint2*>(qs + kGroups * kH * 64 + off) = make_uint2(lw[0], lw[1]);
    }
    fence_proxy_async();
    if (tid < kH) msm[tid] = kNegBig;
    __syncthreads();

    const long seg_begin = u;
    // tokens of each page of pair j that hold data (0 for a missing or
    // rejected block)
    auto pair_tokens = [&](int j, int (&ntok)[2]) {
#pragma unroll
      for (int pg = 0; pg < 2; ++pg) {
        const int pi = 2 * j + pg;
        int n = pi < npages ? min(kBs, Lb - pi * kBs) : 0;
        if (n > 0) {
          const int bk = __ldg(p.block_tables + brow + pi);
          if (bk < 0 || bk >= p.num_blocks) n = 0;
        }
        ntok[pg] = n;
      }
    };
    // One half (`part`: 256 of the 512 items of 8 dims) of V^ double slot n
    // (k-steps 2n, 2n + 1: 32 tokens of one 128-dv tile) by 128 threads
    // (index bt), into ring half n & 1 once that half's previous MMAs have
    // completed (`fills` counts this group's fills of the double slots).
    // False if the wait ran out; warp-uniform.
    auto build_double = [&](int n, int part, int bt, const int (&ntok)[2], int& fills) -> bool {
      uint4 vh[2], vl[2];
      uint32_t off[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int s = 2 * n + k, tile = s >> 3, ks = s & 7, slot = s & 3;
        {
          const int item = bt + 128 * part;
          const int tl = item & 15, mg = item >> 4;
          const int t = ks * 16 + tl, pg = t >> 6, row = t & 63;
          const int dv0 = tile * 128 + mg * 8, g = dv0 >> 6, dd = dv0 & 63;
          if (row < ntok[pg]) {
            const uint2 c8 = *reinterpret_cast<const uint2*>(codes + g * kTile + pg * (kTile / 2) +
                                                             sw64(row, dd));
            const float sv = SEG ? scl[pg * 4] : scl[(pg * kBs + row) * kGroups + g];
            const __nv_bfloat16 sh = __float2bfloat16_rn(sv);
            const __nv_bfloat16 sl = __float2bfloat16_rn(sv - __bfloat162float(sh));
            dequant8<FMT>(c8, __bfloat162bfloat162(sh), __bfloat162bfloat162(sl), vh[k], vl[k]);
          } else {
            vh[k] = vl[k] = make_uint4(0u, 0u, 0u, 0u);
          }
          off[k] = slot * 2 * kVTerm + (tl >> 3) * 2048 + mg * 128 + (tl & 7) * 16;
        }
      }
      const int ds = n & 1;
      if (fills >= kVD && !wait_warp(bar_vfree + ds, ((fills >> 1) - 1) & 1)) return false;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        *reinterpret_cast<uint4*>(vs + off[k]) = vh[k];
        *reinterpret_cast<uint4*>(vs + off[k] + kVTerm) = vl[k];
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_vfull + ds);
      ++fills;
      return true;
    };
    if (warp == 8) {
      // =================================================== issuing thread
      if (lane == 0) {
        const uint32_t codes_a = smem_u32(codes), q_a = smem_u32(qs), p_a = smem_u32(ps),
                       v_a = smem_u32(vs);
        // P.V operand descriptors: V^ slot (hi, lo) and P k-step (hi, lo)
        uint64_t dvh[kVS], dvl[kVS], dph[8], dpl[8];
#pragma unroll
        for (int v = 0; v < kVS; ++v) {
          dvh[v] = tc_desc(v_a + v * 2 * kVTerm, 2048, 128, 0);
          dvl[v] = tc_desc(v_a + v * 2 * kVTerm + kVTerm, 2048, 128, 0);
        }
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          dph[ks] = tc_desc(p_a + ks * 2048, 1024, 128, 0);
          dpl[ks] = tc_desc(p_a + kPTerm + ks * 2048, 1024, 128, 0);
        }
        for (long uu = seg_begin; uu < seg_end; ++uu) {
          if (!wait(bar_full, pc & 1)) break;
          tc_fence_after();
          // ---- QK^T: group g into score buffer g % kNB
          bool qok = true;
#pragma unroll
          for (int g = 0; g < kGroups; ++g) {
            const int bf = g % kNB;
            if (!qok || (quse[bf] > 0 && !wait(bar_sfree + bf, (quse[bf] - 1) & 1))) {
              qok = false;
              continue;
            }
            tc_fence_after();
            for (int ks = 0; ks < 2; ++ks)
              for (int term = 0; term < 2; ++term) {
                const uint64_t ad = tc_desc(codes_a + g * kTile + ks * 32, 16, 512, 4);
                const uint64_t bd =
                    tc_desc(q_a + (term * kGroups + g) * (kH * 64) + ks * 32, 16, 512, 4);
                tc_mma_f8(tmem + kColS + bf * 64, ad, bd, p.idesc_qk, (ks | term) != 0);
              }
            tc_commit(bar_qk + bf);
            ++quse[bf];
          }
          tc_commit(bar_stage);  // the tensor core is done reading the stage
          if (*reinterpret_cast<volatile int*>(abort_flag)) break;
          // ---- P.V: O^T[tile] += V^[slot]^T P[k-step], hi.hi + hi.lo + lo.hi
          if (!wait(bar_pready, pc & 1)) break;
          tc_fence_after();
          bool vok = true;
#pragma unroll 1
          for (int tile = 0; tile < 4 && vok; ++tile) {
            const uint32_t d = tmem + tile * 64;
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2) {  // double slot: k-steps 2 k2, 2 k2 + 1
              const int ds = k2 & 1;
              if (!wait(bar_vfull + ds, (vd >> 1) & 1)) {
                vok = false;
                break;
              }
              tc_fence_after();
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int ks = 2 * k2 + h, slot = ks & 3;
                const bool first = (uu == seg_begin) && ks == 0;  // each tile starts its sum
                tc_mma_f16(d, dvh[slot], dph[ks], idesc_pv, !first);
                tc_mma_f16(d, dvh[slot], dpl[ks], idesc_pv, true);
                tc_mma_f16(d, dvl[slot], dph[ks], idesc_pv, true);
              }
              tc_commit(bar_vfree + ds);
              ++vd;
            }
          }
          if (!vok) break;
          tc_commit(bar_pv);
          ++pc;
          if (*reinterpret_cast<volatile int*>(abort_flag)) break;
        }
      }
    } else if (warp == 9) {
      // =================================================== copying warp
      // Pair j of the segment into the stage once the tensor core, the score
      // warps and the builders are done with the previous pair: lane l < 18
      // copies group l % 9 of page l / 9, lanes 18 and 19 the two pages'
      // scales; lanes 20 and 21 prefetch the next pair's pages into L2.  The
      // block ids are read before the wait (block tables are inputs).
      const int pg = lane < 18 ? lane / 9 : (lane < 22 ? (lane - 18) & 1 : -1);
      int last = -1;  // the last pair whose copy went out
      for (long uu = seg_begin; uu < seg_end; ++uu) {
        const int j = static_cast<int>(uu - first_u);
        int blk = -1;
        if (lane < 20) {
          const int pi = 2 * j + pg;
          if (pi < npages) {
            blk = __ldg(p.block_tables + brow + pi);
            if (blk < 0 || blk >= p.num_blocks) {
              if (lane == 0 || lane == 9) raise_error(p.err, FP8PA_DEVERR_BLOCK_RANGE);
              blk = -1;
            }
          }
        }
        uint32_t bytes = 0;
#pragma unroll
        for (int q = 0; q < 2; ++q)
          if (__shfl_sync(0xffffffffu, blk, 9 * q) >= 0)
            bytes += kGroups * (kTile / 2) + (SEG ? 16 : kPageScales);
        if (pc > 0 && !wait_warp(bar_stage, (pc - 1) & 1)) break;
        if (lane == 0) mbar_arrive_expect_tx(bar_full, bytes);
        __syncwarp();
        if (blk >= 0) {
          if (lane < 18) {
            const int g = lane % 9;
            tma_load_2d(codes + g * kTile + pg * (kTile / 2), &tm_lat, g * 64, blk * kBs, bar_full);
          } else if (SEG) {
            bulk_load(reinterpret_cast<uint8_t*>(scl) + pg * 16,
                      p.scale + static_cast<long>(blk) * 4, 16, bar_full);
          } else {
            bulk_load(reinterpret_cast<uint8_t*>(scl) + pg * kPageScales,
                      p.scale + static_cast<long>(blk) * kBs * kGroups, kPageScales, bar_full);
          }
        }
        last = pc;
        if (lane >= 20 && lane < 22 && uu + 1 < seg_end) {
          const int pi = 2 * (j + 1) + pg;
          if (pi < npages) {
            const int nb = __ldg(p.block_tables + brow + pi);
            if (nb >= 0 && nb < p.num_blocks)
              prefetch_l2(p.cache + static_cast<long>(nb) * kBs * kDk, kBs * kDk);
          }
        }
        ++pc;
      }
      // the last copy lands before anything is freed (it normally has: the
      // pair was consumed; a waited phase reads as complete)
      if (last >= 0) (void)mbar_wait_bounded(bar_full, last & 1, kWaitLimitCycles);
    } else if (warp < 4) {
      // =================================================== score warps
      const int t = tid;  // token of the pair, TMEM lane
      const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
      const uint32_t t_sum = tmem + lane_base + kColSum;
      bool dead = false;
      // The score warps meet at named barriers, so none of them may leave the
      // loop alone: after a failed wait a warp stays `dead`, skipping its
      // work and waits but passing the same barriers and arrivals.
      for (long uu = seg_begin; uu < seg_end; ++uu) {
        const int j = static_cast<int>(uu - first_u);
        const bool first = uu == seg_begin;
        if (!dead && !wait_warp(bar_full, pc & 1)) dead = true;
        const int pg = t >> 6, row = t & 63, pi = 2 * j + pg;
        bool valid = pi < npages && j * kT + t < Lb;
        if (valid) {
          const int bk = __ldg(p.block_tables + brow + pi);
          valid = bk >= 0 && bk < p.num_blocks;
        }
        // the token's group scales, with the log2-domain score factor
        float sk[kGroups];
#pragma unroll
        for (int g = 0; g < kGroups; ++g)
          sk[g] = !valid ? 0.f
                         : zs * (SEG ? scl[pg * 4] : scl[(pg * kBs + row) * kGroups + g]);
        float z[kH];
#pragma unroll
        for (int h = 0; h < kH; ++h) z[h] = 0.f;
#pragma unroll
        for (int g = 0; g < kGroups; ++g) {
          const int bf = g % kNB;
          if (!dead && !wait_warp(bar_qk + bf, quse[bf] & 1)) dead = true;
          if (!dead) {
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              uint32_t r[32];
              tmem_ld32(tmem + lane_base + kColS + bf * 64 + c * 32, r);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i)
                z[c * 32 + i] = fmaf(__uint_as_float(r[i]), sk[g], z[c * 32 + i]);
            }
            tc_fence_before();
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_sfree + bf);
          ++quse[bf];
        }
        if (!valid) {
#pragma unroll
          for (int h = 0; h < kH; ++h) z[h] = NEG_INF;
        }
        // ---- running maxima: reduced over the tokens only when some score
        // passes its head's maximum by more than kTau
        const int fk = pc & 1;
        bool up = false;
#pragma unroll
        for (int h4 = 0; h4 < kH / 4; ++h4) {
          const float4 m4 = reinterpret_cast<const float4*>(msm)[h4];
          up |= (z[4 * h4] > m4.x + kTau) | (z[4 * h4 + 1] > m4.y + kTau) |
                (z[4 * h4 + 2] > m4.z + kTau) | (z[4 * h4 + 3] > m4.w + kTau);
        }
        if (__any_sync(0xffffffffu, up) && lane == 0) misc[fk] = 1.f;
        named_sync(1, 128);
        const bool rescale = misc[fk] != 0.f;
        if (t == 0) misc[fk ^ 1] = 0.f;  // everyone has read the previous pair's flag
        if (rescale) {
#pragma unroll
          for (int h = 0; h < kH; ++h) {
            const float m = warp_max_f32(z[h]);
            if (lane == (h & 31)) red[warp * kH + h] = m;
          }
          named_sync(1, 128);
          if (t < kH) {
            const float mo = msm[t];
            const float mn = fmaxf(mo, fmaxf(fmaxf(red[t], red[kH + t]),
                                             fmaxf(red[2 * kH + t], red[3 * kH + t])));
            asm_[t] = ex2(mo - mn);  // 0 before the first token, 1 if unchanged
            msm[t] = mn;
          }
          named_sync(1, 128);
        }
        // p = 2^(z - m), at most 2^kTau; 0 for masked tokens
#pragma unroll
        for (int h4 = 0; h4 < kH / 4; ++h4) {
          const float4 m4 = reinterpret_cast<const float4*>(msm)[h4];
          z[4 * h4] = ex2(z[4 * h4] - m4.x);
          z[4 * h4 + 1] = ex2(z[4 * h4 + 1] - m4.y);
          z[4 * h4 + 2] = ex2(z[4 * h4 + 2] - m4.z);
          z[4 * h4 + 3] = ex2(z[4 * h4 + 3] - m4.w);
        }
        // this token's running partial sums of p, in TMEM
        if (!dead) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t r[16];
            if (!first) {
              tmem_ld16(t_sum + c * 16, r);
              tmem_ld_wait();
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float acc = first ? 0.f : __uint_as_float(r[i]);
              if (rescale) acc *= asm_[c * 16 + i];
              r[i] = __float_as_uint(acc + z[c * 16 + i]);
            }
            tmem_st16(t_sum + c * 16, r);
          }
        }
        // the previous pair's P.V must be done before P is rewritten and O
        // rescaled
        if (!first && !dead && !wait_warp(bar_pv, (pc - 1) & 1)) dead = true;
        if (!dead) {
          tc_fence_after();
          // P as bf16 hi + lo, MN-major: core (token / 8, head / 8), token
          // row t % 8.  hi keeps p's leading 16 bits (exact), lo = rn(p - hi).
#pragma unroll
          for (int ng = 0; ng < kH / 8; ++ng) {
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t a = __float_as_uint(z[ng * 8 + 2 * i]);
              const uint32_t c = __float_as_uint(z[ng * 8 + 2 * i + 1]);
              hw[i] = __byte_perm(a, c, 0x7632);
              lw[i] = bf16x2_bits(__uint_as_float(a) - __uint_as_float(a & 0xFFFF0000u),
                                  __uint_as_float(c) - __uint_as_float(c & 0xFFFF0000u));
            }
            const uint32_t off = (t >> 3) * 1024 + ng * 128 + (t & 7) * 16;
            *reinterpret_cast<uint4*>(ps + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(ps + kPTerm + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
          if (!first && rescale) {
#pragma unroll 1
            for (int tile = 0; tile < 4; ++tile)
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                uint32_t r[16];
                const uint32_t ta = tmem + lane_base + tile * 64 + c * 16;
                tmem_ld16(ta, r);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                  r[i] = __float_as_uint(__uint_as_float(r[i]) * asm_[c * 16 + i]);
                tmem_st16(ta, r);
              }
          }
          tmem_st_wait();
        }
        fence_proxy_async();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_pready);
        // the second half of every V^ double slot of this pair (the builder
        // warps make the first); then the stage is no longer read by this warp
        if (!dead) {
          int ntok[2];
          pair_tokens(j, ntok);
          // unrolled by 4: the double slot's index arithmetic folds into
          // constants (by 8 or fully, the larger loop body costs more than
          // that saves)
#pragma unroll 4
          for (int n = 0; n < 16; ++n)
            if (!dead && !build_double(n, 1, t, ntok, fills_s)) dead = true;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_stage);
        ++pc;
      }
      // ---- segment end: this CTA's piece of (request b, head group hg)
      const bool ok = !dead && wait_warp(bar_pv, (pc - 1) & 1);
      tc_fence_after();
      // head sums over the 128 tokens (every score warp takes part: named
      // barriers)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t r[32];
        tmem_ld32(t_sum + c * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float l = __uint_as_float(r[i]);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
          if (lane == i) red[warp * kH + c * 32 + i] = l;
        }
      }
      named_sync(1, 128);
      const long seg = (segbase[b] + (wid - first_u / upw)) * p.H + hg;
      if (ok && t < kH) {
        const float l = (red[t] + red[kH + t]) + (red[2 * kH + t] + red[3 * kH + t]);
        p.part_ml[(seg * kH + t) * 2] = l > 0.f ? msm[t] : NEG_INF;
        p.part_ml[(seg * kH + t) * 2 + 1] = l;
      }
      if (ok) {
#pragma unroll 1
        for (int tile = 0; tile < 4; ++tile)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_base + tile * 64 + c * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              p.part_o[(seg * kH + c * 32 + i) * kDv + tile * 128 + t] = __uint_as_float(r[i]);
          }
      }
      tc_fence_before();
    } else {
      // =================================================== V^ builders
      const int bt = tid - 128;
      for (long uu = seg_begin; uu < seg_end; ++uu) {
        const int j = static_cast<int>(uu - first_u);
        int ntok[2];
        pair_tokens(j, ntok);
        if (!wait_warp(bar_full, pc & 1)) break;
        bool ok = true;
#pragma unroll 4
        for (int n = 0; n < 16; ++n)
          if (ok) ok = build_double(n, 0, bt, ntok, fills_b);
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_stage);
        ++pc;
      }
    }
    u = seg_end;
    // every role has finished the segment, so the flag is read by all
    // threads after its last write: the decision is uniform
    __syncthreads();
    if (*reinterpret_cast<volatile int*>(abort_flag)) break;
  }

  // ---- drain and free: no copy or MMA may still be in flight
  if (warp == 8 && lane == 0) {
    tc_commit(bar_drain);  // arrives once every MMA issued so far has completed
    (void)mbar_wait_bounded(bar_drain, 0, kWaitLimitCycles);
  }
  __syncthreads();
  tc_fence_after();
  if (warp == 8) tmem_dealloc(tmem, kTmemCols);
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

// The tensor-core kernel for FP8 latents with 64-head groups (the planner
// counts page pairs); workspace as the warp-MMA kernel's, with head groups
// of 64.
cudaError_t launch_decode_mla_tc(const DecodeShape& s, const DecodeArgs& a, cudaStream_t stream) {
  const int H = s.hq / kH;
  const int ranges = s.workers / H;
  const bool seg = a.mode == FP8PA_SCALE_SEGMENT;
  auto kfn = a.fmt == FP8PA_E4M3
                 ? (seg ? mla_tc_kernel<FP8PA_E4M3, 1> : mla_tc_kernel<FP8PA_E4M3, 0>)
                 : (seg ? mla_tc_kernel<FP8PA_E5M2, 1> : mla_tc_kernel<FP8PA_E5M2, 0>);
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kfn), Smem::kBytes);
  if (e != cudaSuccess) return e;
  CUtensorMap tm;
  if (!encode_tensor_map_2d_u8(&tm, a.k_cache, kDk, static_cast<uint64_t>(a.num_blocks) * kBs, 64,
                               kBs, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  char* ws = static_cast<char*>(a.workspace);
  int* plan = reinterpret_cast<int*>(ws);
  const size_t plan_bytes = align256(sizeof(int) * (kPlanHeader + 2 * (s.batch + 1)));
  const size_t rows = (static_cast<size_t>(ranges) + s.batch) * H * kH;
  float* part_ml = reinterpret_cast<float*>(ws + plan_bytes);
  float* part_o = reinterpret_cast<float*>(ws + plan_bytes + align256(rows * 2 * sizeof(float)));
  if (!a.plan_ready) {
    e = launch_plan(a.seq_lens, s.batch, s.qlen, 1, 1, kBs, s.max_blocks, ranges, plan, a.err,
                    stream, 2);
    if (e != cudaSuccess) return e;
  }
  TcParams p;
  p.q = a.q;
  p.cache = a.k_cache;
  p.scale = a.k_scale;
  p.block_tables = a.block_tables;
  p.seq_lens = a.seq_lens;
  p.plan = plan;
  p.part_ml = part_ml;
  p.part_o = part_o;
  p.err = a.err;
  p.B = s.batch;
  p.hq = s.hq;
  p.H = H;
  p.max_blocks = s.max_blocks;
  p.num_blocks = a.num_blocks;
  p.qlen = s.qlen;
  p.idesc_qk = tc_idesc(a.fmt == FP8PA_E5M2 ? 1 : 0, 0, 0, 0, 128, kH);
  p.qk_scale_log2 = a.sm_scale * 1.4426950408889634f;

  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(s.workers);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Smem::kBytes;
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  if (g_split_ev_start) cudaEventRecord(g_split_ev_start, stream);
  e = cudaLaunchKernelEx(&cfg, kfn, tm, p);
  if (e != cudaSuccess) return e;
  if (g_split_ev_stop) cudaEventRecord(g_split_ev_stop, stream);
  return launch_merge(plan, part_ml, part_o, a.out, s.batch, 1, s.hq, H, kH, kDv, a.out_dtype,
                      stream);
}

}  // namespace fp8pa
