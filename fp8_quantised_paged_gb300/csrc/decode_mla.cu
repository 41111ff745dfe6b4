// decode_mla.cu -- split-K paged decode attention for the shared-latent (MLA)
// layout: every query head attends to one cached latent per token.
//
// Method ("DeepSeek V4 950: whole-network FP8 dataflow", 2kiu.com/news/4508674,
// sec. 2.2: the cache holds one compressed latent per token, quantised with
// one scale per latent group; sec. 2.3: softmax and accumulation in FP32):
//   z[h,t] = sm_scale * q[h,:576] . c^[t,:576],  o[h,:] = sum_t softmax(z)[h,t] c^[t,:512]
//   c^[t,d] = decode(code[t,d]) * s[t, d / 64]   (9 groups of 64 dims)
// The 576-dim latent is 512 latent dims plus the 64-dim rope part; V is the
// first 512 dims of the same dequantised latent.
//
// GB300 design.  128 heads x 576 dims against one latent per token is a real
// dense contraction (~455 flop per cached byte), so the kernel is built around
// the tensor cores:
//  * Work = (request, 64-token page); the planner cuts the flat page list into
//    contiguous ranges, and each range is processed by H = Hq / 32 CTAs with
//    adjacent block indices, one per group of 32 heads.  They run together, so
//    a page comes from DRAM once and from L2 for the other head groups.  The
//    merge kernel folds the partial pieces, as for the GQA layout.
//  * A page (36,864 code bytes + 2,304 scale bytes) arrives by 1-D bulk copy
//    into a two-stage ring; all 256 threads convert its codes once to exact f16
//    in a padded shared tile read by every warp through ldmatrix.
//  * QK^T runs per 64-dim group on warp MMA (m16n8k16, f16 in, f32 out) and
//    each group's partial is scaled by its per-token group scale in FP32, so
//    the scores are exact products of codes and q.
//  * P.V folds the V group scale (and a running power-of-two normaliser) into
//    P, carried as f16 hi + lo so P keeps ~22 significant bits.
//  * FP32 online softmax in the log2 domain; the page maximum is combined
//    across the four token-quarter warps through shared memory.
#include <float.h>

#include "common.cuh"
#include "internal.h"
#include "plan.cuh"

namespace fp8pa {

namespace {

constexpr int kDk = 576, kDv = 512, kBs = 64, kGroups = 9, kGs = 64;
constexpr int kHeads = 32;                       // heads per CTA
constexpr int kThreads = 256;                    // 8 warps
constexpr int kStride = kDk + 8;                 // padded f16 row (1168 B)
constexpr int kPStride = 68;                     // padded fp32 P row
constexpr int kCodeBytes = kBs * kDk;            // 36,864
constexpr int kScaleBytes = kBs * kGroups * 4;   // 2,304
constexpr int kStageBytes = kCodeBytes + kScaleBytes;

struct MlaSmem {
  static constexpr int kStages = 0;                                     // 2 x stage
  static constexpr int kCs = kStages + 2 * kStageBytes;                 // f16 [64][584]
  static constexpr int kQs = kCs + kBs * kStride * 2;                   // f16 [32][584]
  static constexpr int kPs = kQs + kHeads * kStride * 2;                // f32 [32][68]
  static constexpr int kSs = kPs + kHeads * kPStride * 4;               // f32 [64][9]
  static constexpr int kRed = kSs + kBs * kGroups * 4;                  // f32 [4][32]
  static constexpr int kMisc = kRed + 4 * kHeads * 4;                   // scratch
  static constexpr int kBars = kMisc + 64;                              // 2 mbarriers
  static constexpr int kOk = kBars + 16;
  static constexpr int kBytes = kOk + 16 + 128;
};

struct MlaParams {
  const uint16_t* q;
  const uint8_t* cache;
  const float* scale;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int* plan;
  float* part_ml;
  float* part_o;
  uint32_t* err;
  int B, hq, ngroups_h, max_blocks, num_blocks;
  int qlen;  // queries per request: B counts (request, query) pairs
  float qk_scale_log2;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// SEG: one scale per page (the segment mode: block-wise cumulative
// rescaling) in place of one per (token, 64-dim group).
template <int FMT, bool SEG>
__global__ void __launch_bounds__(kThreads, 1) mla_split_kernel(const MlaParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stages = smem + MlaSmem::kStages;
  __half* Cs = reinterpret_cast<__half*>(smem + MlaSmem::kCs);
  __half* Qs = reinterpret_cast<__half*>(smem + MlaSmem::kQs);
  float* Ps = reinterpret_cast<float*>(smem + MlaSmem::kPs);
  float* Ss = reinterpret_cast<float*>(smem + MlaSmem::kSs);
  float* red = reinterpret_cast<float*>(smem + MlaSmem::kRed);
  float* misc = reinterpret_cast<float*>(smem + MlaSmem::kMisc);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + MlaSmem::kBars);
  int* okf = reinterpret_cast<int*>(smem + MlaSmem::kOk);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 2, c = lane & 3;
  const int ht = warp & 1;        // head tile (16 heads) in both phases
  const int tq = warp >> 1;       // token quarter (QK) / dv quarter (PV)

  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_barrier_init();
  }
  __syncthreads();
  griddep_wait();
  griddep_launch_dependents();

  const int* uprefix = p.plan + kPlanHeader;
  const int* segbase = uprefix + p.B + 1;
  const int U = *reinterpret_cast<const volatile int*>(p.plan);
  const int upw = *reinterpret_cast<const volatile int*>(p.plan + 1);
  const int H = p.ngroups_h;              // head groups per request
  const int hg = blockIdx.x % H;          // this CTA's group of 32 heads
  const long wid = blockIdx.x / H;        // its page range
  const long u0 = wid * upw;
  if (u0 >= U) return;
  const int n_units = static_cast<int>(min(static_cast<long>(upw), U - u0));

  // unit -> (request b, page j)
  struct Cur {
    int b, hg, j, nb;
    long brow;  // offset of request b's block-table row (b / qlen)
  };
  auto locate = [&](long u) {
    int lo = 0, hi = p.B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (uprefix[mid] <= u) lo = mid; else hi = mid;
    }
    Cur cu;
    cu.b = lo;
    cu.nb = uprefix[lo + 1] - uprefix[lo];
    cu.hg = hg;
    cu.j = static_cast<int>(u - uprefix[lo]);
    cu.brow = static_cast<long>(lo / p.qlen) * p.max_blocks;
    return cu;
  };
  auto advance = [&](Cur& cu) {
    if (++cu.j < cu.nb) return;
    cu.j = 0;
    do {
      ++cu.b;
    } while (cu.b < p.B && uprefix[cu.b + 1] == uprefix[cu.b]);
    if (cu.b < p.B) {
      cu.nb = uprefix[cu.b + 1] - uprefix[cu.b];
      cu.brow = static_cast<long>(cu.b / p.qlen) * p.max_blocks;
    }
  };
  auto issue = [&](const Cur& cu, int s) {  // thread 0 only
    const int blk = __ldg(p.block_tables + cu.brow + cu.j);
    const bool ok = blk >= 0 && blk < p.num_blocks;
    okf[s] = ok ? 1 : 0;
    if (ok) {
      mbar_arrive_expect_tx(&bars[s], kCodeBytes + (SEG ? 16 : kScaleBytes));
      bulk_load(stages + s * kStageBytes, p.cache + static_cast<long>(blk) * kCodeBytes,
                kCodeBytes, &bars[s]);
      if constexpr (SEG)  // the page's row of 4 scales (one KV head, padded to 16 bytes)
        bulk_load(stages + s * kStageBytes + kCodeBytes, p.scale + static_cast<long>(blk) * 4, 16,
                  &bars[s]);
      else
        bulk_load(stages + s * kStageBytes + kCodeBytes,
                  p.scale + static_cast<long>(blk) * kBs * kGroups, kScaleBytes, &bars[s]);
    } else {
      raise_error(p.err, FP8PA_DEVERR_BLOCK_RANGE);
      mbar_arrive(&bars[s]);
    }
  };

  Cur cc = locate(u0);
  Cur pc = cc;
  int ip = 0;
  for (; ip < 2 && ip < n_units; ++ip) {
    if (tid == 0) issue(pc, ip);
    advance(pc);
  }

  const float NEG_INF = __int_as_float(0xff800000);
  float O[16][4];                 // 16 heads x 128 dv: 16 n-tiles of 8 dv
  float m_h[2], l_h[2];           // heads 16ht+g8 and 16ht+g8+8
  float zs = 0.f;
  int erun = -127, Lb = 0;
  const uint32_t cs_base = smem_u32(Cs), qs_base = smem_u32(Qs);
  bool abandoned = false;
  int i = 0;

  for (; i < n_units; ++i) {
    const int s = i & 1;
    const uint32_t par = static_cast<uint32_t>((i >> 1) & 1);
    if (i == 0 || cc.j == 0) {
      // ---- new segment: q of the 32 heads -> f16 (power-of-two normalised)
      __syncthreads();
      bool bad;
      Lb = visible_len(p.seq_lens, cc.b, p.qlen, p.max_blocks * kBs, &bad);
      const uint16_t* qsrc = p.q + (static_cast<long>(cc.b) * p.hq + cc.hg * kHeads) * kDk;
      float amax = 0.f;
      for (int e = tid; e < kHeads * kDk / 8; e += kThreads) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(qsrc) + e);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
          amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[k] << 16)),
                                   fabsf(__uint_as_float(w[k] & 0xFFFF0000u))));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      if (lane == 0) misc[warp] = amax;
      __syncthreads();
      amax = 0.f;
#pragma unroll
      for (int w = 0; w < kThreads / 32; ++w) amax = fmaxf(amax, misc[w]);
      const int eq = amax > 0.f ? exp_above(amax) : 0;
      const float fq = exp2i(14 - eq);
      for (int e = tid; e < kHeads * kDk / 8; e += kThreads) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(qsrc) + e);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
        const int h = e / (kDk / 8), col = (e % (kDk / 8)) * 8;
        uint4 o;
        uint32_t* op = &o.x;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          op[k] = pack_half2(__uint_as_float(w[k] << 16) * fq,
                             __uint_as_float(w[k] & 0xFFFF0000u) * fq);
        *reinterpret_cast<uint4*>(Qs + h * kStride + col) = o;
      }
      zs = p.qk_scale_log2 * exp2i(eq - 14);
      m_h[0] = m_h[1] = NEG_INF;
      l_h[0] = l_h[1] = 0.f;
      erun = -127;
#pragma unroll
      for (int n = 0; n < 16; ++n) O[n][0] = O[n][1] = O[n][2] = O[n][3] = 0.f;
    }

    // ---- wait for the page, dequantise it once into Cs, stage its scales
    const bool landed = mbar_wait_bounded(&bars[s], par, kWaitLimitCycles);
    if (__syncthreads_or(!landed)) {
      if (tid == 0) raise_error(p.err, FP8PA_DEVERR_TIMEOUT);
      abandoned = true;
      break;
    }
    const int valid = okf[s] ? min(kBs, Lb - cc.j * kBs) : 0;
    const uint8_t* codes = stages + s * kStageBytes;
    const float* sc = reinterpret_cast<const float*>(codes + kCodeBytes);
    for (int e = tid; e < kBs * kDk / 16; e += kThreads) {
      const int t = e / (kDk / 16), col = (e % (kDk / 16)) * 16;
      uint4 lo4, hi4;
      if (t < valid) {
        const uint4 u = *reinterpret_cast<const uint4*>(codes + t * kDk + col);
        lo4.x = codes2_to_f16x2<FMT>(u.x);
        lo4.y = codes2_to_f16x2<FMT>(u.x >> 16);
        lo4.z = codes2_to_f16x2<FMT>(u.y);
        lo4.w = codes2_to_f16x2<FMT>(u.y >> 16);
        hi4.x = codes2_to_f16x2<FMT>(u.z);
        hi4.y = codes2_to_f16x2<FMT>(u.z >> 16);
        hi4.z = codes2_to_f16x2<FMT>(u.w);
        hi4.w = codes2_to_f16x2<FMT>(u.w >> 16);
      } else {
        lo4 = make_uint4(0, 0, 0, 0);
        hi4 = lo4;
      }
      *reinterpret_cast<uint4*>(Cs + t * kStride + col) = lo4;
      *reinterpret_cast<uint4*>(Cs + t * kStride + col + 8) = hi4;
    }
    for (int e = tid; e < kBs * kGroups; e += kThreads)
      Ss[e] = (e / kGroups) < valid ? sc[SEG ? 0 : e] : 0.f;
    __syncthreads();
    // the stage is consumed: refill it with the page two ahead
    if (ip < n_units) {
      if (tid == 0) issue(pc, s);
      ++ip;
      advance(pc);
    }

    // ---- S = Q . C^T for 16 heads (ht) x 16 tokens (tq), exact per group
    float S[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n) S[n][0] = S[n][1] = S[n][2] = S[n][3] = 0.f;
    {
      const int arow = 16 * ht + (lane & 7) + 8 * ((lane >> 3) & 1);
      const int acol = 8 * (lane >> 4);
      const int brow = 16 * tq + (lane & 7) + 8 * (lane >> 4);
      const int bcol = 8 * ((lane >> 3) & 1);
      const uint32_t aaddr = qs_base + (arow * kStride + acol) * 2;
      const uint32_t baddr = cs_base + (brow * kStride + bcol) * 2;
#pragma unroll 9
      for (int gi = 0; gi < kGroups; ++gi) {
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int k0 = gi * kGs + kk * 16;
          uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
          ldsm_x4(aaddr + k0 * 2, a0, a1, a2, a3);
          ldsm_x4(baddr + k0 * 2, b0, b1, b2, b3);
          mma_16816(acc[0], a0, a1, a2, a3, b0, b1);
          mma_16816(acc[1], a0, a1, a2, a3, b2, b3);
        }
#pragma unroll
        for (int n = 0; n < 2; ++n) {
          const int t0 = 16 * tq + 8 * n + 2 * c;
          const float s0 = Ss[t0 * kGroups + gi], s1 = Ss[(t0 + 1) * kGroups + gi];
          S[n][0] += acc[n][0] * s0;
          S[n][1] += acc[n][1] * s1;
          S[n][2] += acc[n][2] * s0;
          S[n][3] += acc[n][3] * s1;
        }
      }
    }
    // scores in the log2 domain, invalid tokens masked
    float mx[2] = {NEG_INF, NEG_INF};
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      const int t0 = 16 * tq + 8 * n + 2 * c;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int t = t0 + (e & 1);
        S[n][e] = t < valid ? S[n][e] * zs : NEG_INF;
        mx[e >> 1] = fmaxf(mx[e >> 1], S[n][e]);
      }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
    }
    if (c == 0) {
      red[tq * kHeads + 16 * ht + g8] = mx[0];
      red[tq * kHeads + 16 * ht + g8 + 8] = mx[1];
    }
    __syncthreads();
    float alpha[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int h = 16 * ht + g8 + 8 * r;
      float pm = fmaxf(fmaxf(red[h], red[kHeads + h]), fmaxf(red[2 * kHeads + h], red[3 * kHeads + h]));
      const float mn = fmaxf(m_h[r], pm);
      alpha[r] = mn == NEG_INF ? 1.f : ex2(m_h[r] - mn);
      m_h[r] = mn;
    }
    float lsum[2] = {0.f, 0.f};
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      const int t0 = 16 * tq + 8 * n + 2 * c;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float pa = m_h[r] == NEG_INF ? 0.f : ex2(S[n][2 * r] - m_h[r]);
        const float pb = m_h[r] == NEG_INF ? 0.f : ex2(S[n][2 * r + 1] - m_h[r]);
        lsum[r] += pa + pb;
        *reinterpret_cast<float2*>(Ps + (16 * ht + g8 + 8 * r) * kPStride + t0) = make_float2(pa, pb);
      }
    }
    l_h[0] = l_h[0] * alpha[0] + lsum[0];
    l_h[1] = l_h[1] * alpha[1] + lsum[1];
    __syncthreads();

    // ---- O[16 heads x 128 dv] += (P * s_v) . C[:, dv]   (warp: ht, dv quarter tq)
    {
      // running power-of-two normaliser of the V group scales this warp uses
      float svm = 0.f;
      for (int e = lane; e < kBs * 2; e += 32) {
        const int t = e >> 1, gv = 2 * tq + (e & 1);
        svm = fmaxf(svm, Ss[t * kGroups + gv]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) svm = fmaxf(svm, __shfl_xor_sync(0xffffffffu, svm, o));
      float rs = 1.f;
      if (svm > 0.f) {
        const int et = exp_above(svm);
        if (et > erun) {
          rs = exp2i(erun - et);
          erun = et;
        }
      }
      const float f0 = alpha[0] * rs, f1 = alpha[1] * rs;
      if (__any_sync(0xffffffffu, f0 != 1.f || f1 != 1.f)) {
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          O[n][0] *= f0;
          O[n][1] *= f0;
          O[n][2] *= f1;
          O[n][3] *= f1;
        }
      }
      const float pf = exp2i(15 - erun);
      const int vrow = (lane & 7) + 8 * ((lane >> 3) & 1);
      const int vcol = 8 * (lane >> 4);
#pragma unroll
      for (int gg = 0; gg < 2; ++gg) {
        const int gv = 2 * tq + gg;
#pragma unroll 4
        for (int kk = 0; kk < 4; ++kk) {
          const int t0 = 16 * kk + 2 * c;
          const float sa = Ss[t0 * kGroups + gv] * pf, sb = Ss[(t0 + 1) * kGroups + gv] * pf;
          const float sc8 = Ss[(t0 + 8) * kGroups + gv] * pf,
                      sd = Ss[(t0 + 9) * kGroups + gv] * pf;
          const float* pr0 = Ps + (16 * ht + g8) * kPStride;
          const float* pr1 = pr0 + 8 * kPStride;
          const float2 p00 = *reinterpret_cast<const float2*>(pr0 + t0);
          const float2 p10 = *reinterpret_cast<const float2*>(pr1 + t0);
          const float2 p01 = *reinterpret_cast<const float2*>(pr0 + t0 + 8);
          const float2 p11 = *reinterpret_cast<const float2*>(pr1 + t0 + 8);
          uint32_t ah[4], al[4];
          split_pack(p00.x * sa, p00.y * sb, ah[0], al[0]);
          split_pack(p10.x * sa, p10.y * sb, ah[1], al[1]);
          split_pack(p01.x * sc8, p01.y * sd, ah[2], al[2]);
          split_pack(p11.x * sc8, p11.y * sd, ah[3], al[3]);
          const uint32_t vaddr =
              cs_base + ((16 * kk + vrow) * kStride + 128 * tq + 64 * gg + vcol) * 2;
#pragma unroll
          for (int np = 0; np < 4; ++np) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(vaddr + np * 16 * 2, b0, b1, b2, b3);
            const int n0 = 8 * gg + 2 * np;
            mma_16816(O[n0], ah[0], ah[1], ah[2], ah[3], b0, b1);
            mma_16816(O[n0], al[0], al[1], al[2], al[3], b0, b1);
            mma_16816(O[n0 + 1], ah[0], ah[1], ah[2], ah[3], b2, b3);
            mma_16816(O[n0 + 1], al[0], al[1], al[2], al[3], b2, b3);
          }
        }
      }
    }

    // ---- segment end: write this CTA's piece of (b, head group)
    if (i == n_units - 1 || cc.j == cc.nb - 1) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        l_h[r] += __shfl_xor_sync(0xffffffffu, l_h[r], 1);
        l_h[r] += __shfl_xor_sync(0xffffffffu, l_h[r], 2);
      }
      __syncthreads();  // red[] is free again
      if (c == 0) {
        red[tq * kHeads + 16 * ht + g8] = l_h[0];
        red[tq * kHeads + 16 * ht + g8 + 8] = l_h[1];
      }
      __syncthreads();
      // piece rows: (piece of request b) x head group x head
      const int fu = uprefix[cc.b];
      const long seg = (segbase[cc.b] + (wid - fu / upw)) * H + cc.hg;
      const float fin = exp2i(erun - 15);
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int h = 16 * ht + g8 + 8 * r;
        float* po = p.part_o + (seg * kHeads + h) * kDv + 128 * tq;
#pragma unroll
        for (int n = 0; n < 16; ++n)
          *reinterpret_cast<float2*>(po + 8 * n + 2 * c) =
              make_float2(O[n][2 * r] * fin, O[n][2 * r + 1] * fin);
      }
      if (tq == 0 && c == 0) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int h = 16 * ht + g8 + 8 * r;
          p.part_ml[(seg * kHeads + h) * 2] = m_h[r];
          p.part_ml[(seg * kHeads + h) * 2 + 1] =
              red[h] + red[kHeads + h] + red[2 * kHeads + h] + red[3 * kHeads + h];
        }
      }
    }
    __syncthreads();  // Cs, Ps, red are rewritten by the next page
    advance(cc);
  }

  if (abandoned) {
    for (int k = i; k < ip; ++k)
      (void)mbar_wait_bounded(&bars[k & 1], static_cast<uint32_t>((k >> 1) & 1), kWaitLimitCycles);
  }
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

// Workspace for the shared-latent layout: same shape as the GQA one with the
// head groups of 32 in the role of KV heads.
cudaError_t launch_decode_mla(const DecodeShape& s, const DecodeArgs& a, cudaStream_t stream) {
  if (s.mla_tc) return launch_decode_mla_tc(s, a, stream);
  const int H = s.hq / kHeads;
  const int ranges = s.workers / H;
  const int smem = MlaSmem::kBytes;
  const bool seg = a.mode == FP8PA_SCALE_SEGMENT;
  auto kfn = a.fmt == FP8PA_E4M3
                 ? (seg ? mla_split_kernel<FP8PA_E4M3, true> : mla_split_kernel<FP8PA_E4M3, false>)
             : a.fmt == FP8PA_E5M2
                 ? (seg ? mla_split_kernel<FP8PA_E5M2, true> : mla_split_kernel<FP8PA_E5M2, false>)
                 : (seg ? mla_split_kernel<FP8PA_INT8, true> : mla_split_kernel<FP8PA_INT8, false>);
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kfn), smem);
  if (e != cudaSuccess) return e;
  char* ws = static_cast<char*>(a.workspace);
  int* plan = reinterpret_cast<int*>(ws);
  const size_t plan_bytes = align256(sizeof(int) * (kPlanHeader + 2 * (s.batch + 1)));
  const size_t rows = (static_cast<size_t>(ranges) + s.batch) * H * kHeads;
  float* part_ml = reinterpret_cast<float*>(ws + plan_bytes);
  float* part_o = reinterpret_cast<float*>(ws + plan_bytes + align256(rows * 2 * sizeof(float)));

  if (!a.plan_ready) {
    e = launch_plan(a.seq_lens, s.batch, s.qlen, 1, 1, kBs, s.max_blocks, ranges, plan, a.err,
                    stream);
    if (e != cudaSuccess) return e;
  }
  MlaParams p;
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
  p.ngroups_h = H;
  p.max_blocks = s.max_blocks;
  p.num_blocks = a.num_blocks;
  p.qlen = s.qlen;
  p.qk_scale_log2 = a.sm_scale * 1.4426950408889634f;

  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(s.workers);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  if (g_split_ev_start) cudaEventRecord(g_split_ev_start, stream);
  e = cudaLaunchKernelEx(&cfg, kfn, p);
  if (e != cudaSuccess) return e;
  if (g_split_ev_stop) cudaEventRecord(g_split_ev_stop, stream);
  return launch_merge(plan, part_ml, part_o, a.out, s.batch, 1, s.hq, H, kHeads, kDv,
                      a.out_dtype, stream);
}

}  // namespace fp8pa
