// decode_gqa.cu -- split-K paged decode attention for grouped-query heads.
//
// Method ("Llama 3 70B FP8 deployment", dpshk.com/news/5605006, sec. 1.2:
// GQA; "DeepSeek V4 950", 2kiu.com/news/4508674, sec. 2.3: softmax and
// accumulation in FP32; "DeepSeek-V4.1 512K", hotelren.com/news/5711065,
// sec. 2.2: blockwise attention with an online softmax, sec. 3.3: paged
// blocks through a per-request block table):
//   out[b][h] = sum_t softmax_t(sm_scale * q[b][h] . k^_t) v^_t,
//   k^ = decode(code) * scale, query head h reading KV head h / G.
//
// GB300 design.
//  * Work is the flat list of units (request b, page j).  The planner
//    (plan.cuh) cuts it into equal contiguous ranges, one per resident CTA.
//    A CTA's warps are the KV heads of one head set and walk the range's
//    pages together, so they read each block's adjacent per-head slices.  A
//    range that crosses a request boundary yields one partial per request;
//    the merge (merge.cu) folds the partials of each output row with the
//    log-sum-exp rule.  Balance is exact for ragged batches and a
//    128K-token request spreads over the whole GPU.
//  * Each warp streams its pages, as 16-token slices, through a private
//    ring of shared-memory stages filled by the tensor-copy engine (TMA,
//    2-D boxes of 16 x head_dim bytes with the 128/64-byte swizzle) plus 1-D
//    bulk copies of the per-token scales, completion tracked by mbarriers.
//    One lane issues; no thread waits on another CTA.  Every wait is
//    bounded.
//  * The G <= 8 heads sharing a KV head form a tiny dense contraction
//    (16 tokens x 8 heads x head_dim per tile).  GB300's FP32 pipe cannot
//    keep up with HBM on it (about 8 FMA per cached byte), so QK^T and PV
//    run on warp MMA (m16n8k16, f16 in, f32 accumulate) over codes (FP8 or
//    INT8) converted exactly to f16 in registers.  Scales stay outside the
//    contraction: the per-token K scale multiplies the score, the per-token
//    V scale folds into P, per-channel K scales fold into q (as an f16 high
//    and low part; with G <= 4 both parts share one MMA's head columns),
//    per-channel V scales multiply the output; MX block exponents scale the
//    f16 fragments by exact powers of two.  Power-of-two normalisers keep q
//    and P inside f16's range.
//  * Softmax runs in FP32 in the log2 domain with warp-shuffle maxima.
#include <float.h>

#include "common.cuh"
#include "internal.h"
#include "plan.cuh"

namespace fp8pa {

namespace {

constexpr int kMaxWarps = 8;  // warps per CTA: one per KV head of the CTA's head set
// Internal kernel mode: static channel scales with at most 4 query heads per
// KV head.  The high and low f16 parts of q then share one MMA: the high
// parts in head columns 0..G-1, the low parts in columns G..2G-1.
constexpr int kModeStaticPacked = 16;
// MX block mode with blocks of 32 dims (FP8PA_SCALE_MX_BLOCK itself runs the
// kernel for blocks of 16): the block size is a compile-time constant.
constexpr int kModeMx32 = 17;

__device__ __forceinline__ int ld_i32(const int* p) { return *reinterpret_cast<const volatile int*>(p); }

// ---------------------------------------------------------------- planner
// One warp; lets the split kernel launch at once (it waits for the plan).
__global__ void __launch_bounds__(32) plan_kernel(const int32_t* seq_lens, int B, int qlen,
                                                  int qw, int groups, int bs, int max_blocks,
                                                  int workers, int* ws, uint32_t* err,
                                                  int upages) {
  griddep_wait();  // inputs may come from the kernel before us in the stream
  griddep_launch_dependents();
  plan_warp(seq_lens, B, qlen, qw, groups, bs, max_blocks, workers, ws, err, upages);
}

// ---------------------------------------------------------------- split kernel
struct GqaParams {
  const uint16_t* q;
  const float* k_scale;
  const float* v_scale;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int* plan;
  float* part_ml;
  float* part_o;
  uint32_t* err;
  int B, hq, hkv, G, max_blocks, num_blocks;
  int qlen;  // queries per request of a causal chunk
  int qw;    // query warps per KV head: B planned requests of qw queries each
  int gs;    // dims per block exponent (MX block mode)
  int hp;    // segment mode: page scales per block (KV heads rounded up to 4)
  float qk_scale_log2;
};

// MX block mode helpers.  2^k for an integer k <= 0 as an f16 bit pattern in
// both halves: the fp32 power of two rounded to f16 (exact down to the
// subnormal 2^-24; 2^-25 and below round to 0).
__device__ __forceinline__ uint32_t h2_pow2(int k) {
  const float f = __int_as_float((max(k, -126) + 127) << 23);
  const __half2 h = __floats2half2_rn(f, f);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
  const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a),
                            *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}
// Shared-memory layout for `w` warps (each with its own NST-stage ring of
// 16-token slices of K and V); SCB = scale bytes per token per tensor in the
// ring (4 for one fp32 scale, D/16 for the largest count of E8M0 block
// exponents, 0 for static scales); XTW = words of the per-warp MX factor
// table (0 outside MX block mode).
template <int D, int NST, int SCB, int XTW>
struct GqaSmem {
  static constexpr int kPage = 16 * D;  // one slice of one tensor
  __host__ __device__ static constexpr int pages(int w) { return w * NST * 2 * kPage; }
  __host__ __device__ static constexpr int scales(int w) { return w * NST * 2 * 16 * SCB; }
  __host__ __device__ static constexpr int ps(int w) { return w * 512; }
  __host__ __device__ static constexpr int bars(int w) { return w * NST * 8; }
  __host__ __device__ static constexpr int oks(int w) { return w * NST * 4; }
  __host__ __device__ static constexpr int xt(int w) { return w * XTW * 4; }
  __host__ __device__ static constexpr int bytes(int w) {
    return pages(w) + scales(w) + ps(w) + bars(w) + oks(w) + xt(w) + 1024;
  }
};

// MX factor table of one 16-token tile: row r < 16 is K token r, row 16 + r
// is V token r; word k < D/16 of a row holds 2^(e_k - e_max) of block k as
// an f16 pair, word D/16 the token's scale 2^(e_max - 127) as an fp32.  Rows
// have an odd stride so that the column reads of a tile spread over banks.
template <int D>
struct MxTable {
  static constexpr int kStride = D / 16 + 1;
  static constexpr int kWords = 32 * kStride;
};

// Byte offset of 16-byte chunk `ch` of row `r` in a TMA box written with the
// 128-byte (128-byte rows) or 64-byte (64-byte rows) swizzle.
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int ch) {
  if constexpr (D == 128) {
    return static_cast<uint32_t>(r * 128 + ((ch ^ (r & 7)) << 4));
  } else {
    return static_cast<uint32_t>(r * 64 + ((ch ^ ((r >> 1) & 3)) << 4));
  }
}

struct Cursor {
  int b, j, nb;
  long brow;  // offset of the block-table row of planned request b (b * qw / qlen)
};

template <int D, int BS, int FMT, int MODE, int NST>
__global__ void __launch_bounds__(kMaxWarps * 32)
    gqa_split_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                     const GqaParams p) {
  constexpr bool SEG = (MODE == FP8PA_SCALE_SEGMENT);  // one scale per (page, KV head)
  constexpr bool TOKSC = (MODE == FP8PA_SCALE_TOKEN_HEAD) || SEG;
  constexpr bool PK = (MODE == kModeStaticPacked);
  constexpr bool MX = (MODE == FP8PA_SCALE_MX_BLOCK) || (MODE == kModeMx32);
  constexpr int GS = MODE == kModeMx32 ? 32 : 16;  // MX: dims per block exponent
  constexpr bool DYN = TOKSC || MX;  // per-token scales: q stays exact in f16
  constexpr int SCB = SEG ? 1 : (TOKSC ? 4 : (MX ? D / 16 : 0));
  constexpr int XS = MxTable<D>::kStride;
  // A stage holds one 16-token slice of a page (SUB slices per page), so
  // large pages do not make a warp's ring large.
  constexpr int SUB = BS / 16;
  using SM = GqaSmem<D, NST, SCB, MX ? MxTable<D>::kWords : 0>;
  constexpr int PAGE = SM::kPage;  // bytes of one slice of one tensor
  constexpr int KW = D / 16;   // K words per row per thread = k-steps
  constexpr int KCH = D / 64;  // 16-byte K chunks per row per thread
  constexpr int VW = D / 32;   // V words per token per thread
  constexpr int MT = D / 16;   // dv tiles of 16
  constexpr int nbx = MX ? D / GS : 0;  // exponent bytes per token (MX)
  const uint32_t TX = 2 * PAGE + (SEG ? 2 * 16 : (TOKSC ? 2 * 16 * 4 : (MX ? 2 * 16 * nbx : 0)));

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const int W = blockDim.x >> 5;  // warps in this CTA
  uint8_t* pages = smem + warp * (NST * 2 * PAGE);
  uint8_t* sclb = smem + SM::pages(W) + warp * (NST * 2 * 16 * SCB);
  float* scl = reinterpret_cast<float*>(sclb);
  // P^T for the PV MMA as two f16 planes (hi + lo carry ~22 significant bits)
  uint16_t* ps = reinterpret_cast<uint16_t*>(smem + SM::pages(W) + SM::scales(W)) + warp * 256;
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(smem + SM::pages(W) + SM::scales(W) + SM::ps(W)) + warp * NST;
  int* okf = reinterpret_cast<int*>(smem + SM::pages(W) + SM::scales(W) + SM::ps(W) +
                                    SM::bars(W)) + warp * NST;
  uint32_t* xt = reinterpret_cast<uint32_t*>(smem + SM::pages(W) + SM::scales(W) + SM::ps(W) +
                                             SM::bars(W) + SM::oks(W)) +
                 warp * (MX ? MxTable<D>::kWords : 0);

  if (lane == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
  }
  __syncwarp();
  // Everything above overlaps the planner; the plan is read only after it.
  griddep_wait();
  griddep_launch_dependents();
  const int* uprefix = p.plan + kPlanHeader;
  const int* segbase = uprefix + p.B + 1;
  const int U = ld_i32(p.plan), upw = ld_i32(p.plan + 1);
  // CTA = (page range, set of W KV heads); warp = one KV head.  All warps of
  // a CTA walk the same pages, so together they read a block's adjacent
  // per-head slices.
  // A CTA's warps are (KV head, query) pairs: hpc KV heads x qw queries of
  // the same planned request, all walking the same pages (the qw warps of a
  // KV head ask for each page together: one DRAM read, the rest from L2).
  const int hpc = W / p.qw;
  const int hsets = p.hkv / hpc;
  const long wid = blockIdx.x / hsets;                            // page range
  const int kvh = (blockIdx.x % hsets) * hpc + warp / p.qw;       // this warp's KV head
  const int qi = warp % p.qw;                                     // and query
  const long u0 = wid * upw;
  if (u0 >= U) return;
  const int n_units = static_cast<int>(min(static_cast<long>(upw), U - u0));

  // ---- unit cursor: (request, page) of a flat page index.  The request
  // holding unit u is the count of request starts <= u, less one (the
  // prefix is nondecreasing and uprefix[B] = U > u); the whole warp tests
  // 32 starts per load, so for up to 31 requests this is one load latency.
  auto locate = [&](long u) {
    int cnt = 0;
    for (int base = 0; base <= p.B; base += 32) {
      const int k = base + lane;
      const unsigned le = __ballot_sync(0xffffffffu, k <= p.B && uprefix[k] <= u);
      cnt += __popc(le);
      if (le != 0xffffffffu) break;
    }
    const int lo = cnt - 1;
    Cursor cu;
    cu.b = lo;
    cu.nb = uprefix[lo + 1] - uprefix[lo];
    cu.j = static_cast<int>(u - uprefix[lo]);
    cu.brow = static_cast<long>(lo) * p.qw / p.qlen * p.max_blocks;
    return cu;
  };
  auto advance = [&](Cursor& cu) {
    if (++cu.j < cu.nb) return;
    cu.j = 0;
    do {
      ++cu.b;
    } while (cu.b < p.B && uprefix[cu.b + 1] == uprefix[cu.b]);
    if (cu.b < p.B) {
      cu.nb = uprefix[cu.b + 1] - uprefix[cu.b];
      cu.brow = static_cast<long>(cu.b) * p.qw / p.qlen * p.max_blocks;
    }
  };
  auto block_of = [&](const Cursor& cu) { return __ldg(p.block_tables + cu.brow + cu.j); };
  // Issue the copies of slice `sub` of one page into stage s (lane 0 only
  // acts).
  auto issue = [&](int blk, int s, int sub) {
    if (lane == 0) {
      const bool ok = blk >= 0 && blk < p.num_blocks;
      okf[s] = ok ? 1 : 0;
      if (ok) {
        const int row = (blk * p.hkv + kvh) * BS + 16 * sub;
        mbar_arrive_expect_tx(&bars[s], TX);
        tma_load_2d(pages + s * 2 * PAGE, &tmk, 0, row, &bars[s]);
        tma_load_2d(pages + s * 2 * PAGE + PAGE, &tmv, 0, row, &bars[s]);
        if constexpr (SEG) {
          // the 16-byte quad of page scales holding this KV head's
          const long quad = static_cast<long>(blk) * p.hp + (kvh & ~3);
          bulk_load(sclb + s * 2 * 16, p.k_scale + quad, 16, &bars[s]);
          bulk_load(sclb + s * 2 * 16 + 16, p.v_scale + quad, 16, &bars[s]);
        } else if constexpr (TOKSC) {
          bulk_load(scl + s * 2 * 16, p.k_scale + row, 16 * 4, &bars[s]);
          bulk_load(scl + s * 2 * 16 + 16, p.v_scale + row, 16 * 4, &bars[s]);
        } else if constexpr (MX) {
          const uint8_t* ke = reinterpret_cast<const uint8_t*>(p.k_scale);
          const uint8_t* ve = reinterpret_cast<const uint8_t*>(p.v_scale);
          bulk_load(sclb + s * 2 * 16 * SCB, ke + static_cast<long>(row) * nbx, 16 * nbx,
                    &bars[s]);
          bulk_load(sclb + s * 2 * 16 * SCB + 16 * SCB, ve + static_cast<long>(row) * nbx,
                    16 * nbx, &bars[s]);
        }
      } else {
        raise_error(p.err, FP8PA_DEVERR_BLOCK_RANGE);
        mbar_arrive(&bars[s]);
      }
    }
  };

  // Per-thread byte offsets inside a slice: the swizzle phase of every row a
  // thread touches depends only on its lane, so they are fixed for the
  // whole kernel.
  uint32_t koff[2][KCH], voff[4];
#pragma unroll
  for (int rr = 0; rr < 2; ++rr)
#pragma unroll
    for (int qq = 0; qq < KCH; ++qq) koff[rr][qq] = swz<D>(g + 8 * rr, c * KCH + qq);
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int tau = 4 * c + ((u + c) & 3);
    voff[u] = D == 128 ? swz<D>(tau, g) : swz<D>(tau, g >> 1) + 8 * (g & 1);
  }

  const int n_sub = n_units * SUB;  // slices of the range, in page order
  Cursor cc = locate(u0);
  Cursor pc = cc;
  int ip = 0;  // slices issued
  int pblk = block_of(pc);
  {
    const int npro = min(NST, n_sub);
    for (; ip < npro; ++ip) {
      issue(pblk, ip, ip % SUB);
      if (ip % SUB == SUB - 1) {
        advance(pc);
        if (ip + 1 < n_sub) pblk = block_of(pc);
      }
    }
  }
  // ---- per-segment state.  Q enters the MMA as f16; with static channel
  // scales folded in it is no longer exact in f16, so it is split into a
  // high and a low f16 part and the contraction runs twice (or, packed, on
  // two sets of head columns of one MMA).
  constexpr int QP = (DYN || PK) ? 1 : 2;
  uint32_t qb[QP][KW][2];
  float O[MT][4];
  float m0 = -FLT_MAX, m1 = -FLT_MAX, l0 = 0.f, l1 = 0.f, zs = 0.f;
  int erun = -127, Lb = 0;
  const float NEG_INF = __int_as_float(0xff800000);
  bool abandoned = false;
  int i = 0;

  for (; i < n_sub; ++i) {
    const int s = i % NST;
    const uint32_t par = static_cast<uint32_t>((i / NST) & 1);
    const int sub = i % SUB;  // slice of page cc.j
    if (sub == 0 && (i == 0 || cc.j == 0)) {
      // ---- new segment: load q for the G heads of (b, kv head)
      bool bad;
      const int v = cc.b * p.qw + qi;  // this warp's query: row of q and of out
      Lb = visible_len(p.seq_lens, v, p.qlen, p.max_blocks * BS, &bad);
      // packed: column g >= G carries the low part of head g - G
      const int hc = (PK && g >= p.G) ? g - p.G : g;
      const int h = kvh * p.G + hc;
      float qv[D / 4];
      if (g < (PK ? 2 * p.G : p.G)) {
        const uint4* src = reinterpret_cast<const uint4*>(
            p.q + (static_cast<long>(v) * p.hq + h) * D + c * (D / 4));
#pragma unroll
        for (int x = 0; x < D / 32; ++x) {
          const uint4 u = __ldg(src + x);
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            qv[8 * x + 2 * e] = __uint_as_float(w[e] << 16);
            qv[8 * x + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
          }
        }
        if constexpr (!DYN) {  // static channel scales fold into q
          const float* ksc = p.k_scale + kvh * D + c * (D / 4);
#pragma unroll
          for (int e = 0; e < D / 4; ++e) qv[e] *= __ldg(ksc + e);
        }
      } else {
#pragma unroll
        for (int e = 0; e < D / 4; ++e) qv[e] = 0.f;
      }
      float amax = 0.f;
#pragma unroll
      for (int e = 0; e < D / 4; ++e) amax = fmaxf(amax, fabsf(qv[e]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const int eq = amax > 0.f ? exp_above(amax) : 0;
      const float fq = exp2i(14 - eq);
#pragma unroll
      for (int e = 0; e < D / 4; ++e) qv[e] *= fq;
#pragma unroll
      for (int j = 0; j < KW; ++j) {
        qb[0][j][0] = pack_half2(qv[4 * j], qv[4 * j + 1]);
        qb[0][j][1] = pack_half2(qv[4 * j + 2], qv[4 * j + 3]);
        if constexpr (QP == 2) {
          float r[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            r[e] = qv[4 * j + e] - __half2float(__float2half_rn(qv[4 * j + e]));
          qb[QP - 1][j][0] = pack_half2(r[0], r[1]);
          qb[QP - 1][j][1] = pack_half2(r[2], r[3]);
        }
        if constexpr (PK) {
          if (g >= p.G) {
            float r[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              r[e] = qv[4 * j + e] - __half2float(__float2half_rn(qv[4 * j + e]));
            qb[0][j][0] = pack_half2(r[0], r[1]);
            qb[0][j][1] = pack_half2(r[2], r[3]);
          }
        }
      }
      zs = p.qk_scale_log2 * exp2i(eq - 14);
      m0 = m1 = NEG_INF;
      l0 = l1 = 0.f;
      erun = DYN ? -127 : 1;
#pragma unroll
      for (int t = 0; t < MT; ++t) O[t][0] = O[t][1] = O[t][2] = O[t][3] = 0.f;
    }

    const bool landed = mbar_wait_bounded(&bars[s], par, kWaitLimitCycles);
    if (!__all_sync(0xffffffffu, landed)) {
      if (lane == 0) raise_error(p.err, FP8PA_DEVERR_TIMEOUT);
      abandoned = true;
      break;
    }
    const int valid = okf[s] ? min(16, Lb - cc.j * BS - 16 * sub) : 0;
    const uint32_t kbase = smem_u32(pages + s * 2 * PAGE);
    const uint32_t vbase = kbase + PAGE;
    const float* sks = scl + s * 2 * 16;
    const float* svs = sks + 16;
    const uint8_t* kex = sclb + s * 2 * 16 * SCB;  // MX: exponent bytes of K, V
    const uint8_t* vex = kex + 16 * SCB;

    if (valid > 0) {  // the slice holds tokens of the request (one 16-token tile)
      constexpr int r0 = 0;
      const int tv = valid - r0;
      const bool full = tv >= 16;  // warp-uniform
      // ---- S^T = K . Q^T : rows = tokens (g, g+8), cols = heads (2c, 2c+1)
      uint32_t kw[2][KW];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
#pragma unroll
        for (int qq = 0; qq < KCH; ++qq) {
          const uint4 x = lds128(kbase + r0 * D + koff[rr][qq]);
          kw[rr][4 * qq] = x.x;
          kw[rr][4 * qq + 1] = x.y;
          kw[rr][4 * qq + 2] = x.z;
          kw[rr][4 * qq + 3] = x.w;
        }
      }
      const bool v0 = full || g < tv, v1 = full || g + 8 < tv;
      float sk0 = 1.f, sk1 = 1.f, sv0 = 1.f, sv1 = 1.f;
      // MX: each K row's f16 codes are multiplied by 2^(e_block - e_max of
      // the token) (exact), and 2^e_max becomes the row's scale; this lane's
      // K words cover block kb0 (words with 4j < gs) and kb1.
      uint32_t fk0a = 0u, fk0b = 0u, fk1a = 0u, fk1b = 0u;
      if constexpr (SEG) {
        const float* quad = reinterpret_cast<const float*>(sclb + s * 2 * 16);
        sk0 = sk1 = quad[kvh & 3];
        sv0 = v0 ? quad[4 + (kvh & 3)] : 0.f;
        sv1 = v1 ? quad[4 + (kvh & 3)] : 0.f;
      } else if constexpr (TOKSC) {
        sk0 = sks[r0 + g];
        sk1 = sks[r0 + g + 8];
        sv0 = v0 ? svs[r0 + g] : 0.f;
        sv1 = v1 ? svs[r0 + g + 8] : 0.f;
      } else if constexpr (MX) {
        // Each lane builds one row of the tile's factor table (lane < 16: K
        // token lane, else V token lane - 16), then every lane reads the
        // words its fragments need.
        __syncwarp();  // the previous tile's reads are done
        {
          const uint8_t* eb = (lane < 16 ? kex : vex) + (r0 + (lane & 15)) * nbx;
          uint32_t w[2];
          if constexpr (nbx == 8) {
            const uint2 x = *reinterpret_cast<const uint2*>(eb);
            w[0] = x.x;
            w[1] = x.y;
          } else if constexpr (nbx == 4) {
            w[0] = *reinterpret_cast<const uint32_t*>(eb);
            w[1] = 0u;
          } else {
            w[0] = *reinterpret_cast<const uint16_t*>(eb);
            w[1] = 0u;
          }
          auto ebyte = [&](int k) {
            return static_cast<int>(__byte_perm(w[k >> 2], 0u, 0x4440u | (k & 3)));
          };
          int em = 0;
#pragma unroll
          for (int k = 0; k < nbx; ++k) em = max(em, ebyte(k));
          uint32_t* row = xt + lane * XS;
#pragma unroll
          for (int k = 0; k < nbx; ++k) row[k] = h2_pow2(ebyte(k) - em);
          row[D / 16] = __float_as_uint(exp2i(em - 127));
        }
        __syncwarp();
        constexpr int kbs = D / 4;  // dims of a lane's K words (c * kbs ..)
        const int kb0 = (c * kbs) / GS, kb1 = (c * kbs + kbs - 1) / GS;
        fk0a = xt[g * XS + kb0];
        fk0b = xt[g * XS + kb1];
        fk1a = xt[(g + 8) * XS + kb0];
        fk1b = xt[(g + 8) * XS + kb1];
        sk0 = __uint_as_float(xt[g * XS + D / 16]);
        sk1 = __uint_as_float(xt[(g + 8) * XS + D / 16]);
        sv0 = v0 ? __uint_as_float(xt[(16 + g) * XS + D / 16]) : 0.f;
        sv1 = v1 ? __uint_as_float(xt[(24 + g) * XS + D / 16]) : 0.f;
      }
      // two independent accumulator chains (even / odd k-steps)
      float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < KW; ++j) {
        uint32_t a0, a1, a2, a3;
        codes4_to_f16x2x2<FMT>(kw[0][j], a0, a2);
        codes4_to_f16x2x2<FMT>(kw[1][j], a1, a3);
        if constexpr (MX) {
          const bool hb = 4 * j >= GS;
          const uint32_t f0 = hb ? fk0b : fk0a, f1 = hb ? fk1b : fk1a;
          a0 = hmul2_bits(a0, f0);
          a2 = hmul2_bits(a2, f0);
          a1 = hmul2_bits(a1, f1);
          a3 = hmul2_bits(a3, f1);
        }
#pragma unroll
        for (int qp = 0; qp < QP; ++qp)
          mma_16816((j & 1) ? acc2 : acc, a0, a1, a2, a3, qb[qp][j][0], qb[qp][j][1]);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[e] += acc2[e];
      if constexpr (PK) {
        // add each head's low-part column (G columns to the right) into its
        // high-part column; the columns from G on are then unused
        if (p.G == 1) {
          acc[0] += acc[1];
          acc[2] += acc[3];
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], p.G >> 1);
        }
      }
      const float z00 = v0 ? acc[0] * (zs * sk0) : NEG_INF;
      const float z01 = v0 ? acc[1] * (zs * sk0) : NEG_INF;
      const float z10 = v1 ? acc[2] * (zs * sk1) : NEG_INF;
      const float z11 = v1 ? acc[3] * (zs * sk1) : NEG_INF;
      float mx0 = fmaxf(z00, z10), mx1 = fmaxf(z01, z11);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const bool live0 = mn0 != NEG_INF, live1 = mn1 != NEG_INF;
      const float al0 = live0 ? ex2(m0 - mn0) : 1.f;
      const float al1 = live1 ? ex2(m1 - mn1) : 1.f;
      const float p00 = live0 ? ex2(z00 - mn0) : 0.f;
      const float p10 = live0 ? ex2(z10 - mn0) : 0.f;
      const float p01 = live1 ? ex2(z01 - mn1) : 0.f;
      const float p11 = live1 ? ex2(z11 - mn1) : 0.f;
      l0 = l0 * al0 + p00 + p10;
      l1 = l1 * al1 + p01 + p11;
      m0 = mn0;
      m1 = mn1;
      // ---- fold the V scale into P, normalised by a running power of two
      float rs = 1.f, q00, q01, q10, q11;
      if constexpr (DYN) {
        float svm = fmaxf(sv0, sv1);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) svm = fmaxf(svm, __shfl_xor_sync(0xffffffffu, svm, o));
        const int et = svm > 0.f ? exp_above(svm) : erun;
        if (et > erun) {
          rs = exp2i(erun - et);
          erun = et;
        }
        const float pf = exp2i(15 - erun);
        q00 = p00 * sv0 * pf;
        q01 = p01 * sv0 * pf;
        q10 = p10 * sv1 * pf;
        q11 = p11 * sv1 * pf;
      } else {
        q00 = p00 * 16384.f;
        q01 = p01 * 16384.f;
        q10 = p10 * 16384.f;
        q11 = p11 * 16384.f;
      }
      const float f0 = al0 * rs, f1 = al1 * rs;
      // Once the running maxima settle the factors are exactly 1: skip.
      if (__any_sync(0xffffffffu, f0 != 1.f || f1 != 1.f)) {
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          O[t][0] *= f0;
          O[t][2] *= f0;
          O[t][1] *= f1;
          O[t][3] *= f1;
        }
      }
      // ---- P^T through shared memory into the B layout of the PV MMA.
      // Position 4c'+u of a head row holds token 4c' + ((u + c') & 3).
      __syncwarp();
      {
        const int pos0 = 4 * (g >> 2) + (((g & 3) - (g >> 2)) & 3);
        const int t1 = g + 8;
        const int pos1 = 4 * (t1 >> 2) + (((t1 & 3) - (t1 >> 2)) & 3);
        const int idx[4] = {(2 * c) * 16 + pos0, (2 * c + 1) * 16 + pos0, (2 * c) * 16 + pos1,
                            (2 * c + 1) * 16 + pos1};
        // hi = f16(x), lo = f16(x - hi), two values per conversion
        const __half2 h01 = __floats2half2_rn(q00, q01), h23 = __floats2half2_rn(q10, q11);
        const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
        const __half2 l01 = __floats2half2_rn(q00 - f01.x, q01 - f01.y);
        const __half2 l23 = __floats2half2_rn(q10 - f23.x, q11 - f23.y);
        ps[idx[0]] = __half_as_ushort(__low2half(h01));
        ps[idx[1]] = __half_as_ushort(__high2half(h01));
        ps[idx[2]] = __half_as_ushort(__low2half(h23));
        ps[idx[3]] = __half_as_ushort(__high2half(h23));
        ps[128 + idx[0]] = __half_as_ushort(__low2half(l01));
        ps[128 + idx[1]] = __half_as_ushort(__high2half(l01));
        ps[128 + idx[2]] = __half_as_ushort(__low2half(l23));
        ps[128 + idx[3]] = __half_as_ushort(__high2half(l23));
      }
      __syncwarp();
      const uint2 pb = lds64(smem_u32(ps + g * 16 + 4 * c));
      const uint2 pl = lds64(smem_u32(ps + 128 + g * 16 + 4 * c));
      // ---- O^T += V^T . P^T : rows = dv, cols = heads (V token order
      // rotated per lane for conflict-free reads)
      uint32_t vw[4][VW];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int tau = 4 * c + ((u + c) & 3);
        if constexpr (D == 128) {
          const uint4 x = lds128(vbase + r0 * D + voff[u]);
          vw[u][0] = x.x;
          vw[u][1] = x.y;
          vw[u][2] = x.z;
          vw[u][3] = x.w;
        } else {
          const uint2 x = lds64(vbase + r0 * D + voff[u]);
          vw[u][0] = x.x;
          vw[u][1] = x.y;
        }
        if (!full && tau >= tv) {
#pragma unroll
          for (int e = 0; e < VW; ++e) vw[u][e] = 0u;
        }
      }
      // MX: the V codes of token tau_u, in this lane's block vb, times
      // 2^(e_block - e_max of the token); 2^e_max went into P above.
      uint32_t fv01 = 0u, fv23 = 0u;
      if constexpr (MX) {
        const int vb = ((D == 128 ? 16 : 8) * g) / GS;
        uint32_t f[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) f[u] = xt[(16 + 4 * c + ((u + c) & 3)) * XS + vb];
        fv01 = (f[0] & 0xFFFFu) | (f[1] & 0xFFFF0000u);
        fv23 = (f[2] & 0xFFFFu) | (f[3] & 0xFFFF0000u);
      }
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        const uint32_t sel = (t & 1) ? 0x7362u : 0x5140u;
        const uint32_t x01 = prmt(vw[0][t >> 1], vw[1][t >> 1], sel);
        const uint32_t x23 = prmt(vw[2][t >> 1], vw[3][t >> 1], sel);
        uint32_t a0, a1, a2, a3;
        codes4_to_f16x2x2<FMT>(x01, a0, a1);
        codes4_to_f16x2x2<FMT>(x23, a2, a3);
        if constexpr (MX) {
          a0 = hmul2_bits(a0, fv01);
          a1 = hmul2_bits(a1, fv01);
          a2 = hmul2_bits(a2, fv23);
          a3 = hmul2_bits(a3, fv23);
        }
        mma_16816(O[t], a0, a1, a2, a3, pb.x, pb.y);
        mma_16816(O[t], a0, a1, a2, a3, pl.x, pl.y);
      }
    }
    __syncwarp();

    // ---- refill this stage with the next slice of the range
    if (ip < n_sub) {
      issue(pblk, ip % NST, ip % SUB);
      const bool page_done = ip % SUB == SUB - 1;
      ++ip;
      if (page_done) {
        advance(pc);
        if (ip < n_sub) pblk = block_of(pc);
      }
    }

    // ---- segment end: write the partial (m, l, o) of this warp's piece
    if (sub == SUB - 1 && (i == n_sub - 1 || cc.j == cc.nb - 1)) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, o);
        l1 += __shfl_xor_sync(0xffffffffu, l1, o);
      }
      // piece rows: (piece of request b) x KV head x query head of the group
      const long seg =
          ((segbase[cc.b] + (wid - uprefix[cc.b] / upw)) * p.hkv + kvh) * p.qw + qi;
      const float fin = DYN ? exp2i(erun - 15) : (1.0f / 16384.f);
#pragma unroll
      for (int hsel = 0; hsel < 2; ++hsel) {
        const int hh = 2 * c + hsel;
        if (hh >= p.G) continue;
        float vals[D / 8];
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          vals[2 * t] = O[t][hsel] * fin;
          vals[2 * t + 1] = O[t][2 + hsel] * fin;
        }
        const int dv0 = (D / 8) * g;
        if constexpr (!DYN) {
          const float* vsc = p.v_scale + kvh * D + dv0;
#pragma unroll
          for (int e = 0; e < D / 8; ++e) vals[e] *= __ldg(vsc + e);
        }
        float4* po = reinterpret_cast<float4*>(p.part_o + (seg * p.G + hh) * D + dv0);
#pragma unroll
        for (int e = 0; e < D / 32; ++e)
          po[e] = make_float4(vals[4 * e], vals[4 * e + 1], vals[4 * e + 2], vals[4 * e + 3]);
        if (g == 0) {
          p.part_ml[(seg * p.G + hh) * 2] = hsel ? m1 : m0;
          p.part_ml[(seg * p.G + hh) * 2 + 1] = hsel ? l1 : l0;
        }
      }
    }
    if (sub == SUB - 1) advance(cc);
  }

  if (abandoned) {
    // Drain the copies still in flight into this warp's stages before the
    // CTA may exit (bounded again).
    for (int k = i; k < ip; ++k)
      (void)mbar_wait_bounded(&bars[k % NST], static_cast<uint32_t>((k / NST) & 1),
                              kWaitLimitCycles);
  }
}

// ---------------------------------------------------------------- host side
// Stages of one warp's ring: 8 KB of K+V slices (2 stages at head_dim 128).
// A stage is one 16-token slice whatever the block size, so a warp's ring
// (and the warps resident per SM) does not shrink with larger blocks.
// Registers hold 16 warps per SM; one slice in flight per warp while it
// computes on the other already covers the memory latency (a third stage
// measured 1 % slower, and 24 warps with 2 stages spill registers).
template <int D>
constexpr int stages_for() {
  constexpr int stage = 2 * 16 * D;  // one 16-token slice of K and of V
  constexpr int n = 8192 / stage;
  return n < 2 ? 2 : (n > 8 ? 8 : n);
}

using SplitFn = void (*)(const CUtensorMap, const CUtensorMap, const GqaParams);

struct SplitKernel {
  SplitFn fn;
  int per_warp;  // shared-memory bytes per warp (the CTA adds 1024 for alignment)
  int smem(int w) const { return w * per_warp + 1024; }
};

template <int D, int BS, int FMT, int MODE>
SplitKernel pick4() {
  constexpr int NST = stages_for<D>();
  constexpr bool MX = MODE == FP8PA_SCALE_MX_BLOCK || MODE == kModeMx32;
  constexpr int SCB = MODE == FP8PA_SCALE_SEGMENT
                          ? 1
                          : (MODE == FP8PA_SCALE_TOKEN_HEAD ? 4 : (MX ? D / 16 : 0));
  using SM = GqaSmem<D, NST, SCB, MX ? MxTable<D>::kWords : 0>;
  return {gqa_split_kernel<D, BS, FMT, MODE, NST>, SM::bytes(1) - 1024};
}

template <int D, int BS, int FMT>
SplitKernel pick3(int mode) {
  switch (mode) {
    case FP8PA_SCALE_TOKEN_HEAD: return pick4<D, BS, FMT, FP8PA_SCALE_TOKEN_HEAD>();
    case FP8PA_SCALE_MX_BLOCK:  // FP8 codes only (rejected for INT8 before launch)
      if constexpr (FMT != FP8PA_INT8) return pick4<D, BS, FMT, FP8PA_SCALE_MX_BLOCK>();
      return pick4<D, BS, FMT, FP8PA_SCALE_TOKEN_HEAD>();
    case kModeMx32:
      if constexpr (FMT != FP8PA_INT8) return pick4<D, BS, FMT, kModeMx32>();
      return pick4<D, BS, FMT, FP8PA_SCALE_TOKEN_HEAD>();
    case kModeStaticPacked: return pick4<D, BS, FMT, kModeStaticPacked>();
    case FP8PA_SCALE_SEGMENT: return pick4<D, BS, FMT, FP8PA_SCALE_SEGMENT>();
    default: return pick4<D, BS, FMT, FP8PA_SCALE_CHANNEL_STATIC>();
  }
}

template <int D, int BS>
SplitKernel pick2(int fmt, int mode) {
  switch (fmt) {
    case FP8PA_E4M3: return pick3<D, BS, FP8PA_E4M3>(mode);
    case FP8PA_E5M2: return pick3<D, BS, FP8PA_E5M2>(mode);
    default: return pick3<D, BS, FP8PA_INT8>(mode);
  }
}

template <int D>
SplitKernel pick1(int bs, int fmt, int mode) {
  switch (bs) {
    case 16: return pick2<D, 16>(fmt, mode);
    case 32: return pick2<D, 32>(fmt, mode);
    default: return pick2<D, 64>(fmt, mode);
  }
}

SplitKernel pick(int d, int bs, int fmt, int mode) {
  return d == 128 ? pick1<128>(bs, fmt, mode) : pick1<64>(bs, fmt, mode);
}

// Kernel mode of a scale mode for G query heads per KV head (gs: dims per
// MX block).
int kernel_mode(int mode, int G, int gs) {
  const bool pack = mode == FP8PA_SCALE_CHANNEL_STATIC && (G == 1 || G == 2 || G == 4);
  if (mode == FP8PA_SCALE_MX_BLOCK && gs == 32) return kModeMx32;
  return pack ? kModeStaticPacked : mode;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Warps per CTA: qw query warps for each KV head of the CTA's head set, the
// head set being the divisor of Hkv (with at most 8 warps in all) that keeps
// the most warps resident per SM -- large pages make a warp's ring big
// enough that 8 warps would not fit in one CTA's shared memory, or would
// leave one CTA per SM.  Among equals, a layout with at least two CTAs per
// SM wins (an SM holding one CTA works one page range alone, and ranges of
// ragged requests differ in cost), then the larger head set (its warps share
// each page's block-table entry and DRAM rows).
constexpr int kMaxCtaSmem = 227 * 1024;
int gqa_wpc(int hkv, int qw, const SplitKernel& k) {
  int best = qw, best_warps = 0, best_two = 0;
  for (int h = 1; h * qw <= kMaxWarps; ++h) {
    const int w = h * qw;
    if (hkv % h != 0 || k.smem(w) > kMaxCtaSmem) continue;
    const int ctas = ctas_per_sm(reinterpret_cast<const void*>(k.fn), w * 32, k.smem(w));
    const int warps = w * ctas, two = ctas >= 2 ? 1 : 0;
    if (warps > best_warps || (warps == best_warps && two >= best_two)) {
      best = w;
      best_warps = warps;
      best_two = two;
    }
  }
  return best;
}

}  // namespace

int g_decode_workers_override = 0;
cudaEvent_t g_split_ev_start = nullptr, g_split_ev_stop = nullptr;

// Number of page ranges the planner cuts (GQA: one per resident CTA over the
// head sets; MLA: one per SM over the head groups, times the head groups).
int decode_workers(const DecodeShape& s, int fmt, int mode, int device) {
  const int sms = sm_count(device);
  if (s.mla) {
    // one CTA per SM (202 or 221 KB of shared memory); a whole number of
    // head-group sets (H = Hq / 32, or Hq / 64 on tensor cores)
    const int H = s.hq / mla_group_heads(s);
    int ranges = (g_decode_workers_override > 0 ? g_decode_workers_override : sms) / H;
    return (ranges < 1 ? 1 : ranges) * H;
  }
  if (g_decode_workers_override > 0) return g_decode_workers_override;
  if (s.gqa_tc) return gqa_tc_workers(s, device);
  const SplitKernel k = pick(s.d, s.bs, fmt, kernel_mode(mode, s.hq / s.hkv, s.gs));
  const int qw = gqa_qw(s);
  const int wpc = gqa_wpc(s.hkv, qw, k), hsets = s.hkv / (wpc / qw);
  const int per_sm = ctas_per_sm(reinterpret_cast<const void*>(k.fn), wpc * 32, k.smem(wpc));
  const int ranges = sms * per_sm / hsets;
  return ranges < 1 ? 1 : ranges;
}

// Pieces are numbered per request (the planner runs over pages only) and
// each piece holds one row per head group (KV head for GQA, 32-head group for
// MLA) and query head of the group.
size_t decode_workspace_bytes(const DecodeShape& s) {
  const int groups = s.mla ? s.hq / mla_group_heads(s) : s.hkv;
  const int G = s.hq / groups;
  const int qw = s.mla ? 1 : gqa_qw(s);
  const size_t bp = s.batch / qw;  // planned requests
  const size_t ranges = s.mla ? static_cast<size_t>(s.workers / groups) : s.workers;
  const size_t plan = align256(sizeof(int) * (kPlanHeader + 2 * (bp + 1)));
  const size_t rows = (ranges + bp) * groups * qw * G;
  const size_t ml = align256(rows * 2 * sizeof(float));
  const size_t o = align256(rows * static_cast<size_t>(s.dv) * sizeof(float));
  return plan + ml + o;
}

cudaError_t launch_decode_gqa(const DecodeShape& s, const DecodeArgs& a, cudaStream_t stream) {
  if (s.gqa_tc) return launch_decode_gqa_tc(s, a, stream);
  const int G = s.hq / s.hkv;
  const SplitKernel k = pick(s.d, s.bs, a.fmt, kernel_mode(a.mode, G, a.gs));
  const int qw = gqa_qw(s);
  const int bp = s.batch / qw;  // planned requests
  const int wpc = gqa_wpc(s.hkv, qw, k), hsets = s.hkv / (wpc / qw);
  const int smem = k.smem(wpc);
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(k.fn), smem);
  if (e != cudaSuccess) return e;

  CUtensorMap tmk, tmv;
  const uint64_t rows = static_cast<uint64_t>(a.num_blocks) * s.hkv * s.bs;
  const CUtensorMapSwizzle swz =
      s.d == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  if (!encode_tensor_map_2d_u8(&tmk, a.k_cache, s.d, rows, s.d, 16, swz) ||
      !encode_tensor_map_2d_u8(&tmv, a.v_cache, s.d, rows, s.d, 16, swz))
    return cudaErrorInvalidValue;

  char* ws = static_cast<char*>(a.workspace);
  int* plan = reinterpret_cast<int*>(ws);
  const size_t plan_bytes = align256(sizeof(int) * (kPlanHeader + 2 * (bp + 1)));
  const size_t prow = (static_cast<size_t>(s.workers) + bp) * s.hkv * qw * G;
  float* part_ml = reinterpret_cast<float*>(ws + plan_bytes);
  float* part_o = reinterpret_cast<float*>(ws + plan_bytes + align256(prow * 2 * sizeof(float)));

  if (!a.plan_ready) {
    e = launch_plan(a.seq_lens, bp, s.qlen, qw, 1, s.bs, s.max_blocks, s.workers, plan, a.err,
                    stream);
    if (e != cudaSuccess) return e;
  }
  // Every kernel of the decode is launched with programmatic stream
  // serialisation: it may start while its predecessor drains, and waits
  // (griddepcontrol.wait) before reading anything that predecessor wrote.
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  GqaParams p;
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
  p.max_blocks = s.max_blocks;
  p.num_blocks = a.num_blocks;
  p.qlen = s.qlen;
  p.qw = qw;
  p.gs = a.gs;
  p.hp = segment_scale_heads(s.hkv);
  p.qk_scale_log2 = a.sm_scale * 1.4426950408889634f;
  cfg.gridDim = dim3(static_cast<unsigned>(s.workers) * hsets);
  cfg.blockDim = dim3(wpc * 32);
  cfg.dynamicSmemBytes = smem;
  if (g_split_ev_start) cudaEventRecord(g_split_ev_start, stream);
  e = cudaLaunchKernelEx(&cfg, k.fn, tmk, tmv, p);
  if (e != cudaSuccess) return e;
  if (g_split_ev_stop) cudaEventRecord(g_split_ev_stop, stream);

  return launch_merge(plan, part_ml, part_o, a.out, bp, qw, s.hq, s.hkv, G, s.dv, a.out_dtype,
                      stream);
}

cudaError_t launch_plan(const int32_t* seq_lens, int batch, int qlen, int qw, int groups, int bs,
                        int max_blocks, int workers, int* plan, uint32_t* err,
                        cudaStream_t stream, int upages) {
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(32);
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, plan_kernel, seq_lens, batch, qlen, qw, groups, bs, max_blocks,
                            workers, plan, err, upages);
}

}  // namespace fp8pa
