// decode_gqa_tc.cu -- a causal chunk of queries over the grouped-query
// layout on the fifth-generation tensor cores (tcgen05 + TMEM), for FP8 codes
// with one scale per (token, KV head) and head_dim 128.
//
// Method ("Llama 3 70B FP8 deployment", dpshk.com, sec. 3.3: chunked prefill
// attends a chunk of new queries to the cached tokens; sec. 3.1: one absmax
// scale per token and KV head; softmax and accumulation in FP32):
//   z[q,h,t] = sm_scale * q[q,h,:] . k^[t,:],  k^[t,d] = decode(code) * sk[t]
//   o[q,h,:] = sum_{t visible to q} softmax(z)[q,h,t] v^[t,:],  v^ likewise
//
// GB300 design.  A CTA serves one KV head of a range of 128-token steps; the
// chunk's G heads x q_len queries form the N = 16 or 32 columns of every MMA,
// so each page is read, and its values converted, once for all of them.
//  * QK^T on FP8 tensor cores: S^T[t, hq] = sum_d code[t,d] q[hq,d], A = the
//    step's K codes as TMA landed them (M = 128 tokens, 128-byte rows,
//    128-byte swizzle, one copy per page), B = q as two E4M3 terms hi + lo
//    (64-byte-swizzled halves of 64 dims); the token's K scale
//    is applied in fp32 when the score warps read the accumulator.
//  * FP32 online softmax in the log2 domain with a lazy running maximum per
//    column (reduced over the tokens only when a score passes it by 2^8);
//    masks per query: query i of a chunk of n sees its request's first
//    L - (n - 1 - i) tokens.
//  * P.V on f16 tensor cores: O^T[dv, hq] += V^T P'.  The V codes become
//    f16 exactly by moving bits (a byte permute, and for E4M3 a shift and a
//    mask, per pair; E4M3 comes out scaled by 2^-8, which the output takes
//    back); each token's V scale goes into P' = p * sv[t] * 2^-e, e a running
//    power-of-two bound of the scales seen, carried as f16 hi + lo (about 22
//    bits): two MMAs per 16-token step.
//  * Two stages of K codes with both scales in shared memory, refilled as
//    soon as QK^T and the score warps have read them, and one or two stages
//    of V codes (as many as fit at two CTAs per SM), refilled once the codes
//    sit in the converting warps' registers.  Two P' buffers: a step's
//    scores and P' are made while the previous step's P.V runs; only an O
//    rescale waits for it.  Roles: warps 0-3 score one token each, warps 4-7
//    convert V, lane 0 of warp 8 issues the MMAs, warp 9 the copies (a lane
//    per page); mbarrier hand-overs, every wait bounded.  Pieces are merged
//    by merge.cu.
#include <float.h>

#include "common.cuh"
#include "internal.h"
#include "plan.cuh"
#include "tc.cuh"

namespace fp8pa {

namespace {

constexpr int kD = 128;             // head_dim (K and V)
constexpr int kT = 128;             // tokens per step: M of QK^T, K of P.V
constexpr int kThreads = 10 * 32;   // 4 score, 4 converting, 1 MMA-issuing, 1 copying warp
constexpr int kVS = 4;              // V^ ring slots (16 tokens x 128 dims f16)
constexpr int kVP = kVS / 2;        // ... handed over in pairs
constexpr int kTile = kT * kD;      // a step's K or V codes: 128 rows x 128 B, 128-byte swizzled
// QK^T takes q hi and lo in one MMA of 2N columns (scores from hi and from
// lo side by side, added when read) where that fits the score warps'
// registers, N = 16; with N = 32 the two terms accumulate in the same N
// columns by two MMAs.
template <int N>
constexpr bool kQJoin = N == 16;
// With N = 16 the issuing thread sets the step: it polls each barrier ahead
// of use (a poll costs ~170 cycles of latency even on a completed phase),
// its P.V pairs are unrolled, and the copy warp gathers the scale rows of 4
// pages per copy, so the next step's K codes land sooner.  Measured on the
// 32-column kernel, whose step the score warps set, the same changes were
// slower, so it keeps the plain forms.
template <int N>
constexpr bool kFastIssue = N == 16;
// TMEM columns: two score buffers (2N or N wide), then O^T as 2N (from P'
// hi, from P' lo)
template <int N>
constexpr int kSW = kQJoin<N> ? 2 * N : N;
template <int N>
constexpr uint32_t kTmemCols = 2 * kSW<N> + 2 * N <= 128 ? 128 : 256;
constexpr float kTau = 8.f;
constexpr float kNegBig = -1e30f;

template <int N>
struct Smem {
  // two K stages (K halves, K scales, V scales); V stages (V halves): two
  // where they fit beside the rest at two CTAs per SM, else one
  static constexpr int kVSt = N <= 16 ? 2 : 1;
  static constexpr int kKStage = kTile + 2 * kT * 4;
  static constexpr int kKSt = 0;
  static constexpr int kVStg = kKSt + 2 * kKStage;
  static constexpr int kQ = kVStg + kVSt * kTile;               // 2 terms x 2 halves x N x 64 B
  static constexpr int kPBuf = 2 * kT * N * 2;                   // 2 terms x 128 x N f16
  static constexpr int kP = kQ + 4 * N * 64;                     // two P' buffers
  static constexpr int kV = kP + 2 * kPBuf;                      // ring of V^ slots
  static constexpr int kRed = kV + kVS * 4096;                   // f32 [4][N]
  static constexpr int kM = kRed + 4 * N * 4;                    // f32 [N] running maxima
  static constexpr int kMT = kM + N * 4;                         // f32 [N] maxima + kTau
  static constexpr int kAlpha = kMT + N * 4;                     // f32 [N] rescale factors
  static constexpr int kMisc = kAlpha + N * 4;                   // flags, exponents
  static constexpr int kBlk = kMisc + 128;  // int [K, V][stage][8]: a step's block ids
  static constexpr int kTmem = kBlk + 128;
  static constexpr int kBars = kTmem + 16;
  static constexpr int kNumBars = 4 * 2 + 2 + 2 + 2 + 2 * kVP + 2 + 1;
  static constexpr int kBytes = kBars + kNumBars * 8 + 1024;
};

struct GtcParams {
  const uint16_t* q;
  const float* k_scale;
  const float* v_scale;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int* plan;
  float* part_ml;
  float* part_o;
  uint32_t* err;
  int B, hq, hkv, G, qlen, qw, bs, max_blocks, num_blocks;  // qw queries per planned request
  uint32_t idesc_qk;
  float qk_scale_log2;
};

// Byte offsets of (row r, byte d) in 64- and 128-byte swizzled tiles: the
// 16-byte chunk index is XORed with the row's position in its 512 / 1024
// byte swizzle span.
__device__ __forceinline__ uint32_t sw128(int r, int d) {
  return static_cast<uint32_t>(r * 128 + ((((d >> 4) ^ r) & 7) << 4) + (d & 15));
}
__device__ __forceinline__ uint32_t sw64(int r, int d) {
  return static_cast<uint32_t>(r * 64 + ((((d >> 4) ^ (r >> 1)) & 3) << 4) + (d & 15));
}

// hi = f16(x), lo = f16(x - hi), two values each.
__device__ __forceinline__ void split_f16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 f = __half22float2(h);
  const __half2 l = __floats2half2_rn(a - f.x, b - f.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Eight codes -> four f16x2 words with exact values.  E5M2 is the top byte
// of an f16; `keep` false gives zeros instead (the byte permute selects the
// zero operand), for bytes that may hold infinities or NaNs.  E4M3 moves
// its exponent and mantissa bits under the f16 ones (the sign-replicating
// byte permute puts the sign at bit 15 after the shift): that f16 holds the
// code's value times 2^-8 for normal and subnormal codes alike, a factor the
// output takes back.  Every E4M3 word is finite whatever the byte (the NaN
// code reads as 1.875 * 2^-8, outside the inputs the append step writes),
// so `keep` is not needed there: a finite value times a zero P' adds zero.
template <int FMT>
__device__ __forceinline__ uint4 codes8_to_f16(uint2 c, bool keep) {
  uint32_t w[4];
  const uint32_t s0 = keep ? 0x1404u : 0x4444u, s1 = keep ? 0x3424u : 0x4444u;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t x = i < 2 ? c.x : c.y;
    if constexpr (FMT == FP8PA_E4M3) {
      w[i] = (prmt_sign(x, (i & 1) ? 0xB3A2u : 0x9180u) << 7) & 0xBF80BF80u;
    } else {
      w[i] = prmt_sign(x, (i & 1) ? s1 : s0);
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
// log2 of the factor codes8_to_f16 leaves out
template <int FMT>
constexpr int kVExp = FMT == FP8PA_E4M3 ? 8 : 0;


// Both N-column halves of O^T (from P' hi and from P' lo) in this thread's
// TMEM lane times beta * (alpha[c] if `rescale`), out of line: it runs only
// when a running maximum or the V-scale exponent moves.
template <int N>
__device__ __noinline__ void gtc_rescale_o(uint32_t ta, const float* alpha, float beta,
                                           bool rescale) {
#pragma unroll 1
  for (int c0 = 0; c0 < 2 * N; c0 += 16) {
    uint32_t r[16];
    tmem_ld16(ta + c0, r);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i)
      r[i] = __float_as_uint(__uint_as_float(r[i]) * beta *
                             (rescale ? alpha[(c0 + i) % N] : 1.f));
    tmem_st16(ta + c0, r);
  }
  tmem_st_wait();
}

template <int FMT, int N>
__global__ void __launch_bounds__(kThreads, 2)
    gqa_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_ks, const __grid_constant__ CUtensorMap tm_vs,
                  const GtcParams p) {
  using SM = Smem<N>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  constexpr int kVSt = SM::kVSt;
  uint8_t* kstages = sm + SM::kKSt;   // K stage s: [K h0][K h1][K scales][V scales]
  uint8_t* vstages = sm + SM::kVStg;  // V stage s: [V h0][V h1]
  uint8_t* qs = sm + SM::kQ;
  uint8_t* ps = sm + SM::kP;
  uint8_t* vs = sm + SM::kV;
  float* red = reinterpret_cast<float*>(sm + SM::kRed);
  float* msm = reinterpret_cast<float*>(sm + SM::kM);
  float* asm_ = reinterpret_cast<float*>(sm + SM::kAlpha);
  float* mthr = reinterpret_cast<float*>(sm + SM::kMT);  // a score above it moves the maximum
  float* misc = reinterpret_cast<float*>(sm + SM::kMisc);
  int* eexp = reinterpret_cast<int*>(misc + 4);     // [2]: running V-scale exponent, by step parity
  int* abort_flag = reinterpret_cast<int*>(misc + 8);
  float* svred = misc + 16;                          // [2][4]: per-warp maxima of the V scales
  // [stage][page]: block id, -1 if none; one copy for the K half of a stage,
  // one for the V half, since the two are refilled at different times
  int* kblk = reinterpret_cast<int*>(sm + SM::kBlk);
  int* vblk = kblk + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + SM::kTmem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + SM::kBars);
  uint64_t* bar_kfull = bars;           // [2] a stage's K codes and scales landed
  uint64_t* bar_kfree = bars + 2;       // [2] ... read by the tensor core and the score warps
  uint64_t* bar_vland = bars + 4;       // [2] a stage's V codes landed
  uint64_t* bar_vsfree = bars + 6;      // [2] ... converted
  uint64_t* bar_qk = bars + 8;          // [2] scores of a step in TMEM
  uint64_t* bar_sfree = bars + 10;      // [2] a score buffer read
  uint64_t* bar_pready = bars + 12;     // [2] P' buffer written (and O rescaled)
  uint64_t* bar_vfull = bars + 14;      // [kVP] a pair of V^ slots written
  uint64_t* bar_vfree = bar_vfull + kVP;  // [kVP] ... read by the tensor core
  uint64_t* bar_pv = bar_vfree + kVP;   // [2] P.V of a step done, by step parity
  uint64_t* bar_drain = bar_pv + 2;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float NEG_INF = __int_as_float(0xff800000);
  // P' as 2N columns, hi then lo: one MMA per 16 tokens reads V^ once and
  // accumulates O^T from hi and from lo side by side
  constexpr uint32_t kPLbo = (2 * N / 8) * 128;  // 8 tokens of P' (K direction)
  const uint32_t idesc_pv = tc_idesc(0, 0, 1, 1, 128, 2 * N);  // f16, both MN-major
  const int up = kT / p.bs;                   // pages per step
  const int lgbs = __ffs(p.bs) - 1, lgG = __ffs(p.G) - 1;  // both powers of two

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_kfull + s, 1);
      mbar_init(bar_kfree + s, 1 + 4);  // tensor core, score warps
      mbar_init(bar_vland + s, 1);
      mbar_init(bar_vsfree + s, 4);     // converting warps
      mbar_init(bar_qk + s, 1);
      mbar_init(bar_sfree + s, 4);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_pready + s, 4);
      mbar_init(bar_pv + s, 1);
    }
    for (int v = 0; v < kVP; ++v) {
      mbar_init(bar_vfull + v, 4);
      mbar_init(bar_vfree + v, 1);
    }
    mbar_init(bar_drain, 1);
    misc[0] = misc[1] = 0.f;
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    if (kFastIssue<N>) {
      prefetch_tensormap(&tm_ks);
      prefetch_tensormap(&tm_vs);
    }
  }
  __syncthreads();
  griddep_wait();
  griddep_launch_dependents();

  const int* uprefix = p.plan + kPlanHeader;
  const int* segbase = uprefix + p.B + 1;
  const int U = *reinterpret_cast<const volatile int*>(p.plan);
  const int upw = *reinterpret_cast<const volatile int*>(p.plan + 1);
  const int kvh = blockIdx.x % p.hkv;
  const long wid = blockIdx.x / p.hkv;  // range of steps
  const long u0 = wid * upw;
  if (u0 >= U) return;  // before any TMEM is held
  const int n_units = static_cast<int>(min(static_cast<long>(upw), U - u0));

  if (warp == 8) {
    tmem_alloc(tmem_slot, kTmemCols<N>);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;  // two score buffers, then O^T

  auto locate = [&](long u, int& b) {
    int lo = 0, hi = p.B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (uprefix[mid] <= u) lo = mid; else hi = mid;
    }
    b = lo;
  };
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    return tc_wait(bar, parity, abort_flag, p.err);
  };
  auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, tc_wait(bar, parity, abort_flag, p.err));
  };

  int sc = 0;  // steps done by this CTA (every role keeps its own count)

  long u = u0;
  const long uend = u0 + n_units;
  while (u < uend) {
    // ---- one segment: the steps of request b inside the range
    int b;
    locate(u, b);
    const int first_u = uprefix[b];
    const long seg_end = min(uend, static_cast<long>(uprefix[b + 1]));
    const int nsteps = static_cast<int>(seg_end - u);
    const int cap = p.max_blocks * p.bs;
    bool bad;
    // the chunk's last query sees the most tokens; query i sees Lc - (n - 1 - i)
    // planned request b: queries q0 .. q0 + qw - 1 of the chunk of request
    // breal; its last query sees the most tokens
    const int breal = (b * p.qw) / p.qlen, q0 = (b * p.qw) % p.qlen;
    const int Lmax = visible_len(p.seq_lens, b * p.qw + p.qw - 1, p.qlen, cap, &bad);
    const int npages = (Lmax + p.bs - 1) / p.bs;
    const long brow = static_cast<long>(breal) * p.max_blocks;  // the request's block table

    // q of the N (query, head) columns -> two E4M3 terms after a power-of-two
    // normaliser (the largest |q| just below 2^8), 64-byte-swizzled halves
    __syncthreads();
    float amax = 0.f;
    for (int c = tid; c < N * kD / 8; c += kThreads) {
      const int hq = c / (kD / 8), qi = hq / p.G, h = hq % p.G;
      const uint16_t* src =
          p.q + ((static_cast<long>(b) * p.qw + qi) * p.hq + kvh * p.G + h) * kD;
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(src) + c % (kD / 8));
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
    for (int c = tid; c < N * kD / 8; c += kThreads) {
      const int hq = c / (kD / 8), qi = hq / p.G, h = hq % p.G;
      const uint16_t* src =
          p.q + ((static_cast<long>(b) * p.qw + qi) * p.hq + kvh * p.G + h) * kD;
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(src) + c % (kD / 8));
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
        uint32_t d01, d23;
        codes4_to_f16x2x2<FP8PA_E4M3>(h01 | (h23 << 16), d01, d23);
        const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&d01));
        const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&d23));
        const uint32_t l01 = f32x2_to_codes2<FP8PA_E4M3>(x[4 * k] - f01.x, x[4 * k + 1] - f01.y);
        const uint32_t l23 =
            f32x2_to_codes2<FP8PA_E4M3>(x[4 * k + 2] - f23.x, x[4 * k + 3] - f23.y);
        hw[k] = h01 | (h23 << 16);
        lw[k] = l01 | (l23 << 16);
      }
      // per 64-dim half: the N rows of the hi term, then the N of the lo
      // term, so that one MMA of 2N columns takes both
      const int col = (c % (kD / 8)) * 8, half = col >> 6, d = col & 63;
      const uint32_t off = half * (2 * N * 64) + sw64(hq, d);
      *reinterpret_cast<uint2*>(qs + off) = make_uint2(hw[0], hw[1]);
      *reinterpret_cast<uint2*>(qs + N * 64 + off) = make_uint2(lw[0], lw[1]);
    }
    fence_proxy_async();
    if (tid < N) msm[tid] = mthr[tid] = kNegBig;
    if (tid == 0) eexp[0] = eexp[1] = -1000;  // before the first V scale
    __syncthreads();

    const long seg_begin = u;
    if (warp == 8) {
      // =================================================== issuing thread
      if (lane == 0) {
        // descriptors of the first K half, q term, V^ slot and P' k-step; a
        // later tile's start address (bits 0-13: byte address / 16) is the
        // first one's plus its byte offset / 16
        const uint64_t dk0 = tc_desc(smem_u32(kstages), 16, 1024, 2);  // 128-byte swizzle
        const uint64_t dq0 = tc_desc(smem_u32(qs), 16, 512, 4);
        const uint64_t dv0 = tc_desc(smem_u32(vs), 2048, 128, 0);
        const uint64_t dp0 = tc_desc(smem_u32(ps), kPLbo, 128, 0);
        const int sc0 = sc, nend = sc + nsteps;  // global steps of the segment
        bool ok = true;
        int qk_next = sc0;  // next step whose QK^T is to be issued
        for (int n = sc0; n < nend && ok; ++n) {
          // QK^T of this step (if not issued yet), and of the next one too if
          // its K codes have landed, into score buffer step & 1; P.V of this
          // step does not wait for the next step's copies
          while (qk_next < nend && qk_next <= n + 1) {
            const int m = qk_next, st = m & 1;
            if constexpr (kFastIssue<N>) {
              // both polls go out before either answer is used; a phase seen
              // complete is not waited on again
              const bool kr = mbar_test_wait(bar_kfull + st, (m >> 1) & 1);
              const bool sr = m < 2 || mbar_test_wait(bar_sfree + st, ((m >> 1) - 1) & 1);
              if (m > n && !(kr && sr)) break;
              if ((!kr && !wait(bar_kfull + st, (m >> 1) & 1)) ||
                  (!sr && !wait(bar_sfree + st, ((m >> 1) - 1) & 1))) {
                ok = false;
                break;
              }
            } else {
              if (m > n && !mbar_test_wait(bar_kfull + st, (m >> 1) & 1)) break;
              if (!wait(bar_kfull + st, (m >> 1) & 1) ||
                  (m >= 2 && !wait(bar_sfree + st, ((m >> 1) - 1) & 1))) {
                ok = false;
                break;
              }
            }
            tc_fence_after();
            const uint64_t dk = dk0 + ((st * SM::kKStage) >> 4);
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int ks = 0; ks < 2; ++ks)
#pragma unroll
                for (int term = 0; term < (kQJoin<N> ? 1 : 2); ++term)
                  tc_mma_f8(tmem + st * kSW<N>, dk + ((h * 64 + ks * 32) >> 4),
                            dq0 + ((h * (2 * N * 64) + term * (N * 64) + ks * 32) >> 4),
                            p.idesc_qk, (h | ks | term) != 0);
            tc_commit(bar_qk + st);
            tc_commit(bar_kfree + st);  // the tensor core is done with the K codes
            ++qk_next;
          }
          if (!ok) break;
          // ---- P.V: O^T[:, hi | lo] += V^[slot]^T P'[k-step, hi | lo], a
          // pair of 16-token slots per hand-over.  A step uses the ring's two
          // pairs twice, so pair pp % 2 is in phase pp / 2.
          // (with kFastIssue: the pairs unrolled, pair pp + 1's hand-over polled
          // before pair pp's MMAs go out)
          bool nx = kFastIssue<N> && mbar_test_wait(bar_vfull, 0);  // pair 0
          if (!wait(bar_pready + (n & 1), (n >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
          uint64_t dp = dp0 + (((n & 1) * SM::kPBuf) >> 4);  // P' buffer of the step
#pragma unroll(kFastIssue<N> ? kT / 32 : 1)
          for (int pp = 0; pp < kT / 32; ++pp) {
            const int rp = pp & (kVP - 1);
            if (!nx && !wait(bar_vfull + rp, (pp / kVP) & 1)) { ok = false; break; }
            if (kFastIssue<N> && pp + 1 < kT / 32)
              nx = mbar_test_wait(bar_vfull + ((pp + 1) & (kVP - 1)), ((pp + 1) / kVP) & 1);
            tc_fence_after();
            const uint64_t av = dv0 + static_cast<uint32_t>(rp * (8192 >> 4));
            tc_mma_f16(tmem + 2 * kSW<N>, av, dp, idesc_pv, n > sc0 || pp > 0);
            tc_mma_f16(tmem + 2 * kSW<N>, av + (4096 >> 4), dp + ((2 * kPLbo) >> 4), idesc_pv,
                       true);
            tc_commit(bar_vfree + rp);
            dp += (4 * kPLbo) >> 4;
          }
          if (!ok) break;
          tc_commit(bar_pv + (n & 1));
          if (*reinterpret_cast<volatile int*>(abort_flag)) { ok = false; break; }
        }
        sc = sc0 + nsteps;
      }
    }
    else if (warp == 9) {
      // =================================================== copying warp
      // step k of the segment (global step n) into stage n & 1, in two
      // halves: K codes with both scales once the tensor core and the score
      // warps are done with step n - 2's, V codes once the converting warps
      // are; lane pg < pages per step copies page pg
      int lastk = -1, lastv = -1;  // last step whose K / V half was copied
      for (int k = 0; k < nsteps; ++k) {
        const int n = sc + k, st = n & 1;
        const int j = static_cast<int>(seg_begin + k - first_u);
        int blk = -1;  // read before the wait: block tables are inputs
        if (lane < up) {
          const int pi = j * up + lane;
          if (pi < npages) {
            blk = __ldg(p.block_tables + brow + pi);
            if (blk < 0 || blk >= p.num_blocks) {
              raise_error(p.err, FP8PA_DEVERR_BLOCK_RANGE);
              blk = -1;
            }
          }
        }
        const uint32_t pages = __popc(__ballot_sync(0xffffffffu, blk >= 0));
        uint8_t* dst = kstages + st * SM::kKStage;
        const int row = (blk * p.hkv + kvh) * p.bs;
        if (n >= 2 && !wait_warp(bar_kfree + st, ((n >> 1) - 1) & 1)) break;
        if (lane < 8) kblk[st * 8 + lane] = blk;  // for the score warps
        __syncwarp();
        // scales: with kFastIssue and block 16 or 32, the rows (bs floats)
        // of 4 pages per copy, every page slot of the step (a missing page
        // reads row 0, unused); otherwise each page's row
        const bool gather = kFastIssue<N> && p.bs <= 32;
        const uint32_t sbytes = gather ? 2 * kT * 4 : pages * 2 * p.bs * 4;
        if (lane == 0) mbar_arrive_expect_tx(bar_kfull + st, pages * p.bs * kD + sbytes);
        __syncwarp();
        if (blk >= 0) tma_load_2d(dst + lane * p.bs * kD, &tm_k, 0, row, bar_kfull + st);
        if (gather) {
          const int srow = blk >= 0 ? blk * p.hkv + kvh : 0;  // the page's row of the scale maps
          int r4[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) r4[i] = __shfl_sync(0xffffffffu, srow, ((lane >> 1) & 7) * 4 + i);
          if (lane < 2 * (up / 4)) {  // lane 2g: K scales of pages 4g..4g+3, lane 2g+1: V
            uint8_t* sd = dst + kTile + (lane & 1) * kT * 4 + (lane >> 1) * 4 * p.bs * 4;
            tma_gather4_2d(sd, (lane & 1) ? &tm_vs : &tm_ks, 0, r4[0], r4[1], r4[2], r4[3],
                           bar_kfull + st);
          }
        } else if (blk >= 0) {
          bulk_load(dst + kTile + lane * p.bs * 4, p.k_scale + row, p.bs * 4, bar_kfull + st);
          bulk_load(dst + kTile + kT * 4 + lane * p.bs * 4, p.v_scale + row, p.bs * 4,
                    bar_kfull + st);
        }
        lastk = n;
        const int vi = n % kVSt;
        if (n >= kVSt && !wait_warp(bar_vsfree + vi, ((n / kVSt) - 1) & 1)) break;
        if (lane < 8) vblk[vi * 8 + lane] = blk;  // for the converting warps
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(bar_vland + vi, pages * (p.bs * kD));
        __syncwarp();
        if (blk >= 0)
          tma_load_2d(vstages + vi * kTile + lane * p.bs * kD, &tm_v, 0, row, bar_vland + vi);
        lastv = n;
      }
      // the copies issued land before anything is freed (they normally have:
      // every step was consumed; a waited phase reads as complete)
      for (int i = 0; i < 2; ++i) {
        const int nk = lastk - i, nv = lastv - i;  // the last copy into each stage
        if (nk >= sc) (void)mbar_wait_bounded(bar_kfull + (nk & 1), (nk >> 1) & 1, kWaitLimitCycles);
        if (i < kVSt && nv >= sc)
          (void)mbar_wait_bounded(bar_vland + nv % kVSt, (nv / kVSt) & 1, kWaitLimitCycles);
      }
      sc += nsteps;
    }
    else if (warp < 4) {
      // =================================================== score warps
      const int t = tid;  // token of the step, TMEM lane; also the dv row of O^T
      const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
      const int Lc = min(p.seq_lens[breal], cap);
      float lt[N];  // this token's running sums of p per column
#pragma unroll
      for (int c = 0; c < N; ++c) lt[c] = 0.f;
      bool dead = false;
      // A poll of an mbarrier costs ~170 cycles of latency even on a phase
      // already complete, so each of the step's three is issued ahead of its
      // use (the next step's K copy at the end of this step), and a phase seen
      // complete by every lane is not waited on.
      bool kr = mbar_test_wait(bar_kfull + (sc & 1), (sc >> 1) & 1);
      for (int k = 0; k < nsteps; ++k) {
        const int n = sc, st = n & 1;
        const int j = static_cast<int>(seg_begin + k - first_u);
        const bool qr = mbar_test_wait(bar_qk + st, (n >> 1) & 1);
        const bool pr = k < 2 || mbar_test_wait(bar_pv + (n & 1), ((n >> 1) - 1) & 1);
        if (!dead && !__all_sync(0xffffffffu, kr) && !wait_warp(bar_kfull + st, (n >> 1) & 1))
          dead = true;
        const int pos = j * kT + t;
        const bool vpage = kblk[st * 8 + (t >> lgbs)] >= 0;
        const float* scl = reinterpret_cast<const float*>(kstages + st * SM::kKStage + kTile);
        const float sk = vpage ? scl[t] : 0.f;
        const float sv = vpage && pos < Lmax ? scl[kT + t] : 0.f;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_kfree + st);
        if (!dead && !__all_sync(0xffffffffu, qr) && !wait_warp(bar_qk + st, (n >> 1) & 1))
          dead = true;
        tc_fence_after();
        const float f = zs * sk;
        // query q0 + qi sees pos < Lc - (qlen - 1 - q0 - qi), i.e. qi >= d0:
        // column c = qi * G + h is visible from c = d0 * G on (none once dead)
        const int d0 = vpage && !dead ? pos - (Lc - p.qlen + 1) + 1 - q0 : N;
        const int cmin = max(min(d0, N), 0) << lgG;
        // every column of every token of the warp visible: the usual case
        // (only a request's last step masks), and then no compare per column
        const bool open = __all_sync(0xffffffffu, cmin == 0);
        const uint32_t sa = tmem + lane_base + st * kSW<N>;  // this step's scores
        // N = 32 scores are read from TMEM 16 columns at a time, up to three
        // times a step, rather than held (they would not fit beside the
        // running sums); N = 16 are read once and kept
        float zk[16];
        auto scores16 = [&](int c0, float (&z)[16]) {
          if (N == 16 && c0 < 0) {  // a later pass over the kept scores
#pragma unroll
            for (int i = 0; i < 16; ++i) z[i] = zk[i];
            return;
          }
          c0 = c0 < 0 ? 0 : c0;
          if constexpr (kQJoin<N>) {
            uint32_t rh[16], rl[16];  // from q hi, from q lo
            tmem_ld16(sa + c0, rh);
            tmem_ld16(sa + N + c0, rl);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i)
              z[i] = (__uint_as_float(rh[i]) + __uint_as_float(rl[i])) * f;
            if (!open) {
#pragma unroll
              for (int i = 0; i < 16; ++i) z[i] = c0 + i >= cmin ? z[i] : NEG_INF;
            }
          } else {
            uint32_t r[16];
            tmem_ld16(sa + c0, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) z[i] = __uint_as_float(r[i]) * f;
            if (!open) {
#pragma unroll
              for (int i = 0; i < 16; ++i) z[i] = c0 + i >= cmin ? z[i] : NEG_INF;
            }
          }
          if (N == 16) {
#pragma unroll
            for (int i = 0; i < 16; ++i) zk[i] = z[i];
          }
        };
        const int again = N == 16 ? -1 : 0;  // passes after the first: c0 + again
        // ---- running maxima (lazy) and the V-scale exponent
        const int fk = n & 1;
        bool upf = false;
#pragma unroll
        for (int c0 = 0; c0 < N; c0 += 16) {
          float z[16];
          scores16(c0, z);
#pragma unroll
          for (int i = 0; i < 16; i += 4) {
            const float4 m4 = *reinterpret_cast<const float4*>(mthr + c0 + i);
            upf |= (z[i] > m4.x) | (z[i + 1] > m4.y) | (z[i + 2] > m4.z) | (z[i + 3] > m4.w);
          }
        }
        if (__any_sync(0xffffffffu, upf) && lane == 0) misc[fk] = 1.f;
        const float svw = warp_max_f32(sv);
        if (lane == 0) svred[fk * 4 + warp] = svw;  // by step parity: read below, rewritten two steps on
        named_sync(1, 128);
        const bool rescale = misc[fk] != 0.f;
        const float* svr = svred + fk * 4;
        const float svmax = fmaxf(fmaxf(svr[0], svr[1]), fmaxf(svr[2], svr[3]));
        const int eold = eexp[fk ^ 1];
        const int et = svmax > 0.f ? exp_above(svmax) : eold;
        const int enew = max(eold, et);
        // O's factor for the new exponent (0 before the first V scale)
        const float beta = eold == enew ? 1.f : (eold < -900 ? 0.f : exp2i(eold - enew));
        if (t == 0) {
          misc[fk ^ 1] = 0.f;  // everyone has read the previous step's flag
          eexp[fk] = enew;
        }
        if (rescale) {
#pragma unroll 1
          for (int c0 = 0; c0 < N; c0 += 16) {
            float z[16];
            scores16(c0 + again, z);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float m = warp_max_f32(z[i]);
              if (lane == ((c0 + i) & 31)) red[warp * N + c0 + i] = m;
            }
          }
          named_sync(1, 128);
          if (t < N) {
            const float mo = msm[t];
            const float mn = fmaxf(mo, fmaxf(fmaxf(red[t], red[N + t]),
                                             fmaxf(red[2 * N + t], red[3 * N + t])));
            asm_[t] = ex2(mo - mn);
            msm[t] = mn;
            mthr[t] = mn + kTau;
          }
          named_sync(1, 128);
#pragma unroll
          for (int c = 0; c < N; c += 4) {
            const float4 a4 = *reinterpret_cast<const float4*>(asm_ + c);
            lt[c] *= a4.x;
            lt[c + 1] *= a4.y;
            lt[c + 2] *= a4.z;
            lt[c + 3] *= a4.w;
          }
        }
        // P' buffer n & 1 was last read by P.V(n - 2); O is rescaled between
        // P.V(n - 1) and P.V(n), so only then does this step wait for the
        // previous one (a step's P.V overlaps the next step's scores)
        const bool resc = k > 0 && (rescale || beta != 1.f);
        if (k > 1 && !dead && !__all_sync(0xffffffffu, pr) &&
            !wait_warp(bar_pv + (n & 1), ((n >> 1) - 1) & 1))
          dead = true;
        if (resc && !dead && !wait_warp(bar_pv + ((n - 1) & 1), ((n - 1) >> 1) & 1)) dead = true;
        if (!dead) {
          tc_fence_after();
          // p (at most 2^kTau), its running sums, and P' = p * sv * 2^-enew
          // as f16 hi + lo, MN-major: core (token / 8, column / 8), row t % 8
          const float pf = enew < -900 ? 0.f : sv * exp2i(-enew);  // nothing valid yet: sv = 0
          uint8_t* pb = ps + (n & 1) * SM::kPBuf;
#pragma unroll
          for (int c0 = 0; c0 < N; c0 += 16) {
            float z[16];
            if constexpr (kQJoin<N>) {
              scores16(c0 + again, z);  // the kept scores
#pragma unroll
              for (int i = 0; i < 16; i += 4) {
                const float4 m4 = *reinterpret_cast<const float4*>(msm + c0 + i);
                z[i] -= m4.x;
                z[i + 1] -= m4.y;
                z[i + 2] -= m4.z;
                z[i + 3] -= m4.w;
              }
            } else {
              // read again: the score times its scale less the maximum, one FMA
              uint32_t r[16];
              tmem_ld16(sa + c0, r);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 16; i += 4) {
                const float4 m4 = *reinterpret_cast<const float4*>(msm + c0 + i);
                z[i] = fmaf(__uint_as_float(r[i]), f, -m4.x);
                z[i + 1] = fmaf(__uint_as_float(r[i + 1]), f, -m4.y);
                z[i + 2] = fmaf(__uint_as_float(r[i + 2]), f, -m4.z);
                z[i + 3] = fmaf(__uint_as_float(r[i + 3]), f, -m4.w);
              }
              if (!open) {
#pragma unroll
                for (int i = 0; i < 16; ++i) z[i] = c0 + i >= cmin ? z[i] : NEG_INF;
              }
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float pv = ex2(z[i]);
              lt[c0 + i] += pv;
              z[i] = pv * pf;
            }
#pragma unroll
            for (int g = 0; g < 2; ++g) {
              uint32_t hw[4], lw[4];
#pragma unroll
              for (int i = 0; i < 4; ++i)
                split_f16x2(z[g * 8 + 2 * i], z[g * 8 + 2 * i + 1], hw[i], lw[i]);
              const uint32_t off = (t >> 3) * kPLbo + ((c0 >> 3) + g) * 128 + (t & 7) * 16;
              *reinterpret_cast<uint4*>(pb + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
              *reinterpret_cast<uint4*>(pb + off + (N / 8) * 128) =
                  make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
          }
          if (resc) gtc_rescale_o<N>(tmem + lane_base + 2 * kSW<N>, asm_, beta, rescale);
        }
        // the score buffer is read for the last time
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_sfree + st);
        fence_proxy_async();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_pready + (n & 1));
        if (k + 1 < nsteps) kr = mbar_test_wait(bar_kfull + ((n + 1) & 1), ((n + 1) >> 1) & 1);
        ++sc;
      }
      // ---- segment end: the piece of (request b, KV head kvh)
      const bool ok = !dead && wait_warp(bar_pv + ((sc - 1) & 1), ((sc - 1) >> 1) & 1);
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < N; ++c) {
        float l = lt[c];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == (c & 31)) red[warp * N + c] = l;
      }
      named_sync(1, 128);
      const int efin = eexp[(sc - 1) & 1];  // written by thread 0 before the barrier
      const long seg = segbase[b] + (wid - first_u / upw);
      // piece rows: (piece, KV head, query, head): column c = query * G + head
      const long row0 = (seg * p.hkv + kvh) * N;
      if (ok && t < N) {
        const float l = (red[t] + red[N + t]) + (red[2 * N + t] + red[3 * N + t]);
        p.part_ml[(row0 + t) * 2] = l > 0.f ? msm[t] : NEG_INF;
        p.part_ml[(row0 + t) * 2 + 1] = l;
      }
      if (ok) {
        const float fo = efin < -900 ? 0.f : exp2i(efin + kVExp<FMT>);
#pragma unroll
        for (int c0 = 0; c0 < N; c0 += 16) {
          uint32_t rh[16], rl[16];  // O^T from P' hi and from P' lo
          tmem_ld16(tmem + lane_base + 2 * kSW<N> + c0, rh);
          tmem_ld16(tmem + lane_base + 2 * kSW<N> + N + c0, rl);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i)
            p.part_o[(row0 + c0 + i) * kD + t] =
                (__uint_as_float(rh[i]) + __uint_as_float(rl[i])) * fo;
        }
      }
      tc_fence_before();
    }
    else {
      // =================================================== V^ converting warps
      // thread bt owns token tl = bt & 15 of every 16-token slot and dims
      // 8 mg .. 8 mg + 7 of both 64-dim halves (mg = bt >> 4): a step's 16
      // code words are read at once, the stage's V half released, and the
      // eight slots filled as the tensor core frees them
      const int bt = tid - 128, tl = bt & 15, mg = bt >> 4;
      // dims 8 mg .. 8 mg + 7 of the first half; the second half's chunk
      // index differs in bit 2 (64 bytes on); + 2048 per slot (16 rows)
      const uint32_t src = sw128(tl, mg * 8), src1 = src ^ 64u;
      const uint32_t dst = (tl >> 3) * 2048 + mg * 128 + (tl & 7) * 16;  // + 1024 per half
      bool ok = true;
      for (int k = 0; k < nsteps && ok; ++k) {
        const int n = sc, vi = n % kVSt;
        const int j = static_cast<int>(seg_begin + k - first_u);
        if (!wait_warp(bar_vland + vi, (n / kVSt) & 1)) { ok = false; break; }
        const uint8_t* vt = vstages + vi * kTile;
        uint2 c[kT / 16][2];
#pragma unroll
        for (int s = 0; s < kT / 16; ++s)
#pragma unroll
          for (int h = 0; h < 2; ++h)
            c[s][h] = *reinterpret_cast<const uint2*>(vt + (h ? src1 : src) + s * 2048);
        // bit s: token s * 16 + tl is cached and visible.  Other tokens have
        // a zero P'; only E5M2 bytes can convert to an infinity or a NaN,
        // which would turn that zero into a NaN, so only E5M2 zeroes them.
        uint32_t vm = 0xFFu;
        if constexpr (FMT == FP8PA_E5M2) {
          vm = 0;
#pragma unroll
          for (int s = 0; s < kT / 16; ++s) {
            const int t = s * 16 + tl;
            if (j * kT + t < Lmax && vblk[vi * 8 + (t >> lgbs)] >= 0) vm |= 1u << s;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_vsfree + vi);  // the codes are in registers
#pragma unroll
        for (int s = 0; s < kT / 16; ++s) {
          uint4 o[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) o[h] = codes8_to_f16<FMT>(c[s][h], (vm >> s) & 1);
          // slots in pairs, the ring's two pairs twice per step: pair
          // position rp was last freed in phase (s / 4) ^ 1 (the previous
          // step's second use for s < 4)
          const int slot = s % kVS, rp = (s >> 1) % kVP;
          if ((s & 1) == 0 && (n > 0 || s >= kVS) &&
              !wait_warp(bar_vfree + rp, ((s / kVS) + 1) & 1)) {
            ok = false;
            break;
          }
          *reinterpret_cast<uint4*>(vs + slot * 4096 + dst) = o[0];
          *reinterpret_cast<uint4*>(vs + slot * 4096 + 1024 + dst) = o[1];
          if (s & 1) {
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_vfull + rp);
          }
        }
        if (!ok) break;
        ++sc;
      }
    }
    u = seg_end;
    // every role has finished the segment, so the flag is read by all
    // threads after its last write: the decision is uniform
    __syncthreads();
    if (*reinterpret_cast<volatile int*>(abort_flag)) break;
  }

  // ---- drain and free: no MMA may still be in flight
  if (warp == 8 && lane == 0) {
    tc_commit(bar_drain);  // arrives once every MMA issued so far has completed
    (void)mbar_wait_bounded(bar_drain, 0, kWaitLimitCycles);
  }
  __syncthreads();
  tc_fence_after();
  if (warp == 8) tmem_dealloc(tmem, kTmemCols<N>);
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

template <int N>
void* pick_gtc(int fmt) {
  return fmt == FP8PA_E4M3 ? reinterpret_cast<void*>(gqa_tc_kernel<FP8PA_E4M3, N>)
                           : reinterpret_cast<void*>(gqa_tc_kernel<FP8PA_E5M2, N>);
}

}  // namespace

// Queries per planned request: the largest divisor qw of q_len with
// G x qw = 16 or 32 columns (a chunk longer than that runs as several
// planned requests of qw queries), 0 if there is none.
int gqa_tc_qw(int G, int qlen) {
  for (int qw = qlen; qw >= 1; --qw)
    if (qlen % qw == 0 && (G * qw == 16 || G * qw == 32)) return qw;
  return 0;
}

bool gqa_tc_eligible(int fmt, int mode, int d, int dv, int bs, int hq, int hkv, int qlen) {
  return (fmt == FP8PA_E4M3 || fmt == FP8PA_E5M2) && mode == FP8PA_SCALE_TOKEN_HEAD && d == kD &&
         dv == kD && (bs == 16 || bs == 32 || bs == 64) && qlen >= 2 && qlen <= 8 &&
         hq % hkv == 0 && gqa_tc_qw(hq / hkv, qlen) > 0;
}

// Ranges of 128-token steps: two CTAs per SM, one per KV head of a range.
int gqa_tc_workers(const DecodeShape& s, int device) {
  const int ranges = 2 * sm_count(device) / s.hkv;
  return ranges < 1 ? 1 : ranges;
}

cudaError_t launch_decode_gqa_tc(const DecodeShape& s, const DecodeArgs& a, cudaStream_t stream) {
  const int G = s.hq / s.hkv, qw = gqa_tc_qw(G, s.qlen), N = G * qw, bp = s.batch / qw;
  void* kfn = N == 32 ? pick_gtc<32>(a.fmt) : pick_gtc<16>(a.fmt);
  const int smem = N == 32 ? Smem<32>::kBytes : Smem<16>::kBytes;
  cudaError_t e = ensure_smem_attr(kfn, smem);
  if (e != cudaSuccess) return e;
  // room for two CTAs per SM
  e = cudaFuncSetAttribute(kfn, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  CUtensorMap tmk, tmv, tmks, tmvs;
  const uint64_t rows = static_cast<uint64_t>(a.num_blocks) * s.hkv * s.bs;
  // a page's rows of one KV head, whole (128 bytes), 128-byte swizzled; the
  // scales as rows of one page of one KV head (bs floats), gathered 4 at a
  // time by the N = 16 kernel
  if (!encode_tensor_map_2d_u8(&tmk, a.k_cache, kD, rows, kD, s.bs, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tensor_map_2d_u8(&tmv, a.v_cache, kD, rows, kD, s.bs, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tensor_map_2d_f32(&tmks, a.k_scale, s.bs, rows / s.bs, s.bs, 1) ||
      !encode_tensor_map_2d_f32(&tmvs, a.v_scale, s.bs, rows / s.bs, s.bs, 1))
    return cudaErrorInvalidValue;
  char* ws = static_cast<char*>(a.workspace);
  int* plan = reinterpret_cast<int*>(ws);
  const size_t plan_bytes = align256(sizeof(int) * (kPlanHeader + 2 * (bp + 1)));
  const size_t prow = (static_cast<size_t>(s.workers) + bp) * s.hkv * qw * G;
  float* part_ml = reinterpret_cast<float*>(ws + plan_bytes);
  float* part_o = reinterpret_cast<float*>(ws + plan_bytes + align256(prow * 2 * sizeof(float)));
  if (!a.plan_ready) {
    e = launch_plan(a.seq_lens, bp, s.qlen, qw, 1, s.bs, s.max_blocks, s.workers, plan, a.err,
                    stream, kT / s.bs);
    if (e != cudaSuccess) return e;
  }
  GtcParams p;
  p.q = a.q;
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  p.block_tables = a.block_tables;
  p.seq_lens = a.seq_lens;
  p.plan = plan;
  p.part_ml = part_ml;
  p.part_o = part_o;
  p.err = a.err;
  p.B = bp;
  p.hq = s.hq;
  p.hkv = s.hkv;
  p.G = G;
  p.qlen = s.qlen;
  p.qw = qw;
  p.bs = s.bs;
  p.max_blocks = s.max_blocks;
  p.num_blocks = a.num_blocks;
  // q hi | lo as 2N columns where the kernel joins them (N = 16)
  p.idesc_qk = tc_idesc(a.fmt == FP8PA_E5M2 ? 1 : 0, 0, 0, 0, 128, N == 16 ? 2 * N : N);
  p.qk_scale_log2 = a.sm_scale * 1.4426950408889634f;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(s.workers) * s.hkv);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  if (g_split_ev_start) cudaEventRecord(g_split_ev_start, stream);
  void* args[] = {&tmk, &tmv, &tmks, &tmvs, &p};
  e = cudaLaunchKernelExC(&cfg, kfn, args);
  if (e != cudaSuccess) return e;
  if (g_split_ev_stop) cudaEventRecord(g_split_ev_stop, stream);
  return launch_merge(plan, part_ml, part_o, a.out, bp, qw, s.hq, s.hkv, G, s.dv, a.out_dtype,
                      stream);
}

}  // namespace fp8pa
