// plan.cuh -- the split-K planner as a one-warp device routine, shared by
// the planner kernel and the fused append + plan prologue.
//
// Work is the flat list of units (virtual request b, page j), b counting the
// (request, query) pairs of a causal chunk.  The planner writes, into the
// head of the decode workspace:
//   [0] U = total units, [1] units per worker (range length),
//   [kPlanHeader ..] unit prefix per request (B + 1 ints),
//   then the base index of each request's partial pieces (B + 1 ints).
// A range of consecutive units that crosses a request boundary yields one
// partial piece per request it touches.
#pragma once

#include "common.cuh"

namespace fp8pa {

constexpr int kPlanHeader = 4;

__device__ __forceinline__ int warp_incl_scan(int x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += t;
  }
  return x;
}

// Run by one whole warp.  `groups` multiplies the units of a request (1: the
// split kernels cover every head group of a page in one unit).  A planned
// request b holds the qw queries b*qw .. b*qw + qw - 1 of a causal chunk of
// qlen (qw = 1: one virtual request per query; qw = qlen: one per real
// request); its pages are those its last query sees.
// A unit is `upages` blocks of `bs` tokens (the latent tensor-core kernel
// works on page pairs).
__device__ __forceinline__ void plan_warp(const int32_t* seq_lens, int B, int qlen, int qw,
                                          int groups, int bs, int max_blocks, int workers,
                                          int* ws, uint32_t* err, int upages = 1) {
  const int lane = threadIdx.x & 31;
  const int cap = max_blocks * bs;
  const int ut = bs * upages;  // tokens per unit
  int* uprefix = ws + kPlanHeader;
  int* segbase = uprefix + B + 1;
  int carry = 0;
  for (int base = 0; base < B; base += 32) {
    const int b = base + lane;
    int n = 0;
    if (b < B) {
      bool bad;
      const int L = visible_len(seq_lens, b * qw + qw - 1, qlen, cap, &bad);
      if (bad) raise_error(err, FP8PA_DEVERR_SEQ_LEN);
      n = (L + ut - 1) / ut;
    }
    const int incl = warp_incl_scan(n);
    if (b < B) uprefix[b] = (carry + incl - n) * groups;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  const int U = carry * groups;
  const int upw = max(1, (U + workers - 1) / workers);
  if (lane == 0) {
    uprefix[B] = U;
    ws[0] = U;
    ws[1] = upw;
  }
  __syncwarp();
  carry = 0;
  const int E = B * groups;
  for (int base = 0; base < E; base += 32) {
    const int e = base + lane;
    int segs = 0;
    if (e < E) {
      const int b = e / groups, g = e % groups;
      const int nb = (uprefix[b + 1] - uprefix[b]) / groups;
      if (nb > 0) {
        const int fu = uprefix[b] + g * nb;
        segs = (fu + nb - 1) / upw - fu / upw + 1;
      }
    }
    const int incl = warp_incl_scan(segs);
    if (e < E) segbase[e] = carry + incl - segs;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) segbase[E] = carry;
}

}  // namespace fp8pa
