// merge.cu -- the second pass of the split-K decode: every output row folds
// the partial (running max m, sum l, unnormalised o) of each piece of its
// request with the log-sum-exp rule,
//   M = max_i m_i,  out = sum_i 2^(m_i - M) o_i / sum_i 2^(m_i - M) l_i
// (m in the log2 domain), and writes bf16 or f32.  Method: the online
// softmax of blockwise attention carried across blocks ("DeepSeek-V4.1
// 512K", hotelren.com/news/5711065, sec. 2.2), in FP32 ("DeepSeek V4 950",
// 2kiu.com/news/4508674, sec. 2.3).
#include "common.cuh"
#include "internal.h"
#include "plan.cuh"

namespace fp8pa {

namespace {

// ---------------------------------------------------------------- merge
struct MergeParams {
  const int* plan;
  const float* part_ml;
  const float* part_o;
  void* out;
  int B, hq, hkv, G, dv, out_f32;  // hkv: head groups (KV heads, or 32-head groups)
  int qw;  // queries per planned request: B planned requests, B * qw output rows of heads
};

// One CTA of kMergeWarps warps per output row (b, h): the warps share the
// row's pieces round-robin, then combine through shared memory.
constexpr int kMergeWarps = 4;

template <int DV>
__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(const MergeParams p) {
  constexpr int PER = DV / 32;
  __shared__ float s_acc[kMergeWarps][DV];
  __shared__ float s_ml[kMergeWarps][2];
  griddep_wait();
  griddep_launch_dependents();
  const int row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int v = row / p.hq, h = row % p.hq;  // output row (virtual request v, head h)
  const int b = v / p.qw, qi = v % p.qw;     // planned request and its query
  const int kvh = h / p.G, hh = h % p.G;
  const int* segbase = p.plan + kPlanHeader + p.B + 1;
  // pieces of planned request b: [segbase[b], segbase[b + 1]); piece s holds
  // one row per (head group, query, head of the group)
  const int sb = segbase[b], se = segbase[b + 1];
  // row of piece s for this head
  auto prow = [&](int s) -> long {
    return ((static_cast<long>(s) * p.hkv + kvh) * p.qw + qi) * p.G + hh;
  };
  const float NEG_INF = __int_as_float(0xff800000);
  // Each warp folds its pieces (s = sb + warp, + kMergeWarps, ...) in chunks
  // of C: every load of a chunk (the pieces' (m, l) and this lane's slice of
  // their o) is issued before any is used, so a chunk costs one round trip;
  // a running maximum carries between chunks.
  constexpr int C = PER <= 4 ? 8 : (PER <= 8 ? 4 : 2);
  float M = NEG_INF, L = 0.f;
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  for (int s0 = sb + warp; s0 < se; s0 += C * kMergeWarps) {
    float2 ml[C];
    float2 v[C][PER / 2];
#pragma unroll
    for (int k = 0; k < C; ++k) {
      const int s = s0 + k * kMergeWarps;
      if (s < se) {
        const long r = prow(s);
        ml[k] = *reinterpret_cast<const float2*>(p.part_ml + r * 2);
        const float2* po = reinterpret_cast<const float2*>(p.part_o + r * DV + lane * PER);
#pragma unroll
        for (int e = 0; e < PER / 2; ++e) v[k][e] = po[e];
      } else {
        ml[k] = make_float2(NEG_INF, 0.f);
#pragma unroll
        for (int e = 0; e < PER / 2; ++e) v[k][e] = make_float2(0.f, 0.f);
      }
    }
    float mn = M;
#pragma unroll
    for (int k = 0; k < C; ++k) mn = fmaxf(mn, ml[k].x);
    if (mn == NEG_INF) continue;  // no piece so far saw a token
    const float a = ex2(M - mn);  // ex2(-inf) = 0
    L *= a;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] *= a;
#pragma unroll
    for (int k = 0; k < C; ++k) {
      const float wgt = ex2(ml[k].x - mn);  // 0 for a piece that saw no token
      L += wgt * ml[k].y;
#pragma unroll
      for (int e = 0; e < PER / 2; ++e) {
        acc[2 * e] += wgt * v[k][e].x;
        acc[2 * e + 1] += wgt * v[k][e].y;
      }
    }
    M = mn;
  }
#pragma unroll
  for (int e = 0; e < PER; ++e) s_acc[warp][lane * PER + e] = acc[e];
  if (lane == 0) {
    s_ml[warp][0] = M;
    s_ml[warp][1] = L;
  }
  __syncthreads();
  if (warp != 0) return;
  float Mt = NEG_INF;
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) Mt = fmaxf(Mt, s_ml[w][0]);
  float f[kMergeWarps], Lt = 0.f;
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) {
    f[w] = Mt == NEG_INF ? 0.f : ex2(s_ml[w][0] - Mt);
    Lt += f[w] * s_ml[w][1];
  }
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) v += f[w] * s_acc[w][lane * PER + e];
    acc[e] = v;
  }
  const float inv = Lt > 0.f ? 1.0f / Lt : 0.f;
  const long ob = (static_cast<long>(v) * p.hq + h) * DV + lane * PER;
  if (p.out_f32) {
    float* o = reinterpret_cast<float*>(p.out) + ob;
#pragma unroll
    for (int e = 0; e < PER; ++e) o[e] = acc[e] * inv;
  } else {
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + ob;
#pragma unroll
    for (int e = 0; e < PER; e += 2)
      *reinterpret_cast<__nv_bfloat162*>(o + e) =
          __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
  }
}

}  // namespace

cudaError_t launch_merge(const int* plan, const float* part_ml, const float* part_o, void* out,
                         int batch, int qw, int hq, int groups, int G, int dv, int out_dtype,
                         cudaStream_t stream) {
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(batch * qw * hq);
  cfg.blockDim = dim3(kMergeWarps * 32);
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  MergeParams mp{plan, part_ml, part_o, out, batch, hq, groups, G, dv, out_dtype, qw};
  cudaError_t e;
  if (dv == 128)
    e = cudaLaunchKernelEx(&cfg, merge_kernel<128>, mp);
  else if (dv == 64)
    e = cudaLaunchKernelEx(&cfg, merge_kernel<64>, mp);
  else
    e = cudaLaunchKernelEx(&cfg, merge_kernel<512>, mp);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace fp8pa
