// segment.cu -- the append step with block-wise cumulative rescaling (the
// segment scale mode): one scale per (page, KV head), frozen for each
// 1024-token segment from a running absmax.
#include "common.cuh"
#include "internal.h"

namespace fp8pa {

namespace {

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Block-wise cumulative rescaling ("DeepSeek V4 950", 2kiu.com/news/4508674,
// sec. 4.3: the cache is cut into length blocks, each keeps a cumulative
// scale, refreshed every 1024 tokens).  Per (sequence, K or V, KV head) a
// running absmax R covers every appended token; the token at a position that
// is a multiple of 1024 opens a segment whose scale is frozen as
// max(R / FMAX, 1e-12) with R including that token; every token of the
// segment is coded as x / S and the page stores S once per KV head.
//
// One CTA per (sequence, K or V, KV head) of the call walks the call's rows
// in windows of kSegWindow segments: (1) every row's absmax is folded into
// its segment's maximum in shared memory, and the opening row's absmax is
// kept; (2) one thread runs the segments in order, carrying R, and fixes
// each segment's scale; (3) the rows are read again, coded and scattered.
// Maxima of non-negative floats are exact and order-free, so the scales are
// bit-exact with the token-by-token definition.
constexpr int kSegWarps = 8;
constexpr int kSegWindow = 32;

template <int FMT, int LPR, int R>
__global__ void __launch_bounds__(kSegWarps * 32) segment_append_kernel(SegmentArgs a) {
  griddep_wait();
  griddep_launch_dependents();
  constexpr int SG = 32 / LPR;
  constexpr float kFmax = code_max<FMT>();
  __shared__ unsigned segmax[kSegWindow];  // float bits of each segment's maximum
  __shared__ float aopen[kSegWindow];      // absmax of the segment's opening row, or -1
  __shared__ float sscale[kSegWindow];
  __shared__ float carry[2];               // R and S between windows
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sg = lane / LPR, sl = lane % LPR;
  const int r = blockIdx.x / (a.ntens * a.hkv);
  const int which = (blockIdx.x / a.hkv) % a.ntens;
  const int h = blockIdx.x % a.hkv;
  const int t0 = a.seq_offsets[r];
  const int n = a.seq_offsets[r + 1] - t0;
  if (n <= 0) return;
  const long p0 = a.seq_start[r];
  float* st = a.state + ((static_cast<long>(r) * 2 + which) * a.hkv + h) * 2;
  if (tid == 0) {
    carry[0] = p0 == 0 ? 0.0f : st[0];  // position 0 starts a new sequence
    carry[1] = st[1];
  }
  const uint16_t* src = which ? a.src[1] : a.src[0];
  uint8_t* cache = which ? a.cache[1] : a.cache[0];
  float* scl = which ? a.scale[1] : a.scale[0];
  const int nch = a.d / 8;
  const long seg_last = (p0 + n - 1) / kSegmentTokens;

  // Row i of the sequence (position p0 + i): its values, absmax, block and
  // offset; live = a slot inside the pool.
  auto load_row = [&](int i, float (&v)[R][8], long& blk, int& off) -> bool {
    const int slot = __ldg(a.slot_mapping + t0 + i);
    blk = slot < 0 ? -1 : slot / a.bs;
    off = slot < 0 ? 0 : slot % a.bs;
    const bool live = slot >= 0 && blk < a.num_blocks;
    if (slot >= 0 && blk >= a.num_blocks && sl == 0) raise_error(a.err, FP8PA_DEVERR_SLOT_RANGE);
    const uint16_t* x = src + (static_cast<long>(t0 + i) * a.hkv + h) * a.d;
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
      const int ci = sl + LPR * rr;
      if (live && ci < nch) {
        bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(x + ci * 8)), v[rr]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[rr][e] = 0.0f;
      }
    }
    return live;
  };

  for (long w0 = p0 / kSegmentTokens; w0 <= seg_last; w0 += kSegWindow) {
    const long pa = max(p0, w0 * kSegmentTokens);
    const long pb = min(p0 + n, (w0 + kSegWindow) * kSegmentTokens);
    const int ia = static_cast<int>(pa - p0), ib = static_cast<int>(pb - p0);
    if (tid < kSegWindow) {
      segmax[tid] = 0u;
      aopen[tid] = -1.0f;
    }
    __syncthreads();
    // (1) segment maxima and opening rows
    for (int i0 = ia + warp * SG; i0 < ib; i0 += kSegWarps * SG) {
      const int i = i0 + sg;
      float v[R][8];
      long blk;
      int off;
      const bool live = i < ib && load_row(i, v, blk, off);
      float m = 0.0f;
#pragma unroll
      for (int rr = 0; rr < R; ++rr)
#pragma unroll
        for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(v[rr][e]));
#pragma unroll
      for (int o = LPR / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (live && sl == 0) {
        const long p = p0 + i;
        const int j = static_cast<int>(p / kSegmentTokens - w0);
        atomicMax(&segmax[j], __float_as_uint(m));
        if (p % kSegmentTokens == 0) aopen[j] = m;
      }
    }
    __syncthreads();
    // (2) the segments in order
    if (tid == 0) {
      float Rr = carry[0], S = carry[1];
      for (int j = 0; j < kSegWindow && w0 + j <= seg_last; ++j) {
        if (aopen[j] >= 0.0f) S = fmaxf(__fdiv_rn(fmaxf(Rr, aopen[j]), kFmax), 1e-12f);
        Rr = fmaxf(Rr, __uint_as_float(segmax[j]));
        sscale[j] = S;
      }
      carry[0] = Rr;
      carry[1] = S;
    }
    __syncthreads();
    // (3) code and scatter
    for (int i0 = ia + warp * SG; i0 < ib; i0 += kSegWarps * SG) {
      const int i = i0 + sg;
      float v[R][8];
      long blk;
      int off;
      const bool live = i < ib && load_row(i, v, blk, off);
      if (!live) continue;
      const float S = sscale[static_cast<int>((p0 + i) / kSegmentTokens - w0)];
      uint8_t* dst = cache + ((blk * a.hkv + h) * a.bs + off) * a.d;
#pragma unroll
      for (int rr = 0; rr < R; ++rr) {
        const int ci = sl + LPR * rr;
        if (ci >= nch) continue;
        float q[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) q[e] = __fdiv_rn(v[rr][e], S);
        uint2 packed;
        packed.x = f32x2_to_codes2<FMT>(q[0], q[1]) | (f32x2_to_codes2<FMT>(q[2], q[3]) << 16);
        packed.y = f32x2_to_codes2<FMT>(q[4], q[5]) | (f32x2_to_codes2<FMT>(q[6], q[7]) << 16);
        *reinterpret_cast<uint2*>(dst + ci * 8) = packed;
      }
      if (sl == 0) scl[blk * a.hp + h] = S;
    }
    __syncthreads();  // the window's shared arrays are rewritten next
  }
  if (tid == 0) {
    st[0] = carry[0];
    st[1] = carry[1];
  }
}

template <int FMT>
cudaError_t launch_segment_f(const SegmentArgs& a, cudaStream_t stream) {
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.num_seqs * a.ntens * a.hkv));
  cfg.blockDim = dim3(kSegWarps * 32);
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  const int nch = a.d / 8;
  if (nch <= 8) return cudaLaunchKernelEx(&cfg, segment_append_kernel<FMT, 8, 1>, a);
  if (nch <= 16) return cudaLaunchKernelEx(&cfg, segment_append_kernel<FMT, 16, 1>, a);
  if (nch <= 32) return cudaLaunchKernelEx(&cfg, segment_append_kernel<FMT, 32, 1>, a);
  if (nch <= 64) return cudaLaunchKernelEx(&cfg, segment_append_kernel<FMT, 32, 2>, a);
  return cudaLaunchKernelEx(&cfg, segment_append_kernel<FMT, 32, 3>, a);
}

}  // namespace

cudaError_t launch_append_segment(const SegmentArgs& a, int fmt, cudaStream_t stream) {
  if (a.num_seqs == 0) return cudaSuccess;
  switch (fmt) {
    case FP8PA_E4M3: return launch_segment_f<FP8PA_E4M3>(a, stream);
    case FP8PA_E5M2: return launch_segment_f<FP8PA_E5M2>(a, stream);
    default: return launch_segment_f<FP8PA_INT8>(a, stream);
  }
}

}  // namespace fp8pa
