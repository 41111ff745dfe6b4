// internal.h -- host-side declarations shared by the library's translation
// units (not part of the public ABI; the ABI is include/fp8pa.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace fp8pa {

constexpr int kMaxDevices = 64;

// Device address of a __device__ variable (`symbol`, its host-side name) on
// the current device: looked up again on every call made outside stream
// capture; during a capture, the address the last uncaptured call on this
// device recorded in cache[device] (kMaxDevices entries) is used.  NULL on
// failure.
void* symbol_device_address(const void* symbol, void** cache, cudaStream_t stream,
                            int* dev_out);

// Division of a non-negative 32-bit integer by a divisor d >= 1 fixed for a
// launch, as a multiply-high and two shifts (Granlund and Montgomery,
// "Division by invariant integers using multiplication", PLDI 1994, the
// N = 32 case of their unsigned algorithm); the magic number is made once
// on the host by make_fast_div.
struct FastDiv {
  uint32_t m;  // multiplier
  uint32_t s;  // ceil(log2 d)
};
inline FastDiv make_fast_div(uint32_t d) {
  uint32_t s = 0;
  while ((1ull << s) < d) ++s;
  const uint64_t m = ((1ull << 32) * ((1ull << s) - d)) / d + 1;
  return FastDiv{static_cast<uint32_t>(m), s};
}
__device__ __forceinline__ uint32_t fast_div(uint32_t n, FastDiv f) {
  if (f.s == 0) return n;
  const uint32_t t = __umulhi(f.m, n);
  return (t + ((n - t) >> 1)) >> (f.s - 1);
}

struct AppendArgs {
  const uint16_t* src[2];   // k, v rows (bf16 bits), [num_tokens][hkv][d]
  uint8_t* cache[2];        // k, v codes
  float* scale[2];          // k, v scales (written, or read in CHANNEL_STATIC)
  const int32_t* slot_mapping;
  int num_tokens, hkv, d, ntens, gs, num_blocks, bs;
  FastDiv div_tok;          // by hkv * ntens (rows of a token)
  FastDiv div_bs;           // by bs
  uint32_t* err;
};

cudaError_t launch_append(const AppendArgs& a, int fmt, int mode, cudaStream_t stream);

// The segment-scale append (block-wise cumulative rescaling): tokens per
// segment, and the arguments of one call (sequence r owns rows
// seq_offsets[r] .. seq_offsets[r+1]-1 at positions seq_start[r] + 0, 1, ...).
constexpr int kSegmentTokens = 1024;
inline int segment_scale_heads(int hkv) { return (hkv + 3) / 4 * 4; }
struct SegmentArgs {
  const uint16_t* src[2];  // k, v rows (bf16 bits), [num_tokens][hkv][d]
  uint8_t* cache[2];       // k, v codes
  float* scale[2];         // k, v page scales [num_blocks][segment_scale_heads(hkv)]
  const int32_t* slot_mapping;
  const int32_t* seq_offsets;
  const int32_t* seq_start;
  float* state;            // [num_seqs][2][hkv][2]: running absmax, segment scale
  int num_seqs, hkv, hp, d, ntens, num_blocks, bs;
  uint32_t* err;
};
cudaError_t launch_append_segment(const SegmentArgs& a, int fmt, cudaStream_t stream);

// The planner's inputs (see plan.cuh); `plan` is the head of the workspace.
struct PlanArgs {
  const int32_t* seq_lens;
  int batch, qlen, bs, max_blocks, workers;
  int qw;  // queries per planned request (batch = planned requests)
  int* plan;
  uint32_t* err;
  int upages;  // blocks per planned unit
};

// Append and plan in one launch (the prologue of fp8pa_decode_step).
cudaError_t launch_append_plan(const AppendArgs& a, int fmt, int mode, const PlanArgs& pl,
                               cudaStream_t stream);
cudaError_t launch_channel_scales(const uint16_t* x, int num_tokens, int hd, int fmt, float* out,
                                  cudaStream_t stream);
cudaError_t launch_channel_absmax(const uint16_t* x, int num_tokens, int hd, float* amax,
                                  cudaStream_t stream);
cudaError_t launch_scales_from_absmax(const float* amax, int n, int fmt, float* out,
                                      cudaStream_t stream);

// Workspace layout of the split-K decode, shared by planner, split and merge.
struct DecodeShape {
  int batch, hq, hkv, d, dv, bs, max_blocks;
  int workers;        // split workers (warps or CTAs, per kernel family)
  int mla;            // 1 for the shared-latent layout
  int mla_tc;         // 1 when the latent tensor-core kernel serves it (FP8, 64-head groups)
  int qlen;           // queries per request (batch counts request x query)
  int gqa_tc;         // 1 when a grouped-query chunk runs the tensor-core kernel
  int gs;             // dims per scale group or MX block
};

// Query warps per KV head in the grouped-query split kernel: a causal chunk of
// up to 8 queries has its queries' warps walk the same pages in one CTA (one
// DRAM read per page); longer chunks run one virtual request per query.
int gqa_tc_qw(int G, int qlen);
inline int gqa_qw(const DecodeShape& s) {
  if (s.gqa_tc) return gqa_tc_qw(s.hq / s.hkv, s.qlen);
  return (!s.mla && s.qlen > 1 && s.qlen <= 8) ? s.qlen : 1;
}

size_t decode_workspace_bytes(const DecodeShape& s);

struct DecodeArgs {
  const uint16_t* q;
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const float* k_scale;
  const float* v_scale;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  int num_blocks, fmt, mode, gs, out_dtype;
  float sm_scale;
  void* out;
  void* workspace;
  uint32_t* err;
  bool plan_ready;  // the workspace already holds this call's plan
};

// Page ranges the planner cuts for this shape (its `workers`), and the
// block size of the pages it counts.
// Query heads per CTA of the latent kernels (64 on tensor cores, 32 on warp MMA).
inline int mla_group_heads(const DecodeShape& s) { return s.mla_tc ? 64 : 32; }
inline int plan_workers(const DecodeShape& s) {
  return s.mla ? s.workers / (s.hq / mla_group_heads(s)) : s.workers;
}
inline int plan_block_size(const DecodeShape& s) { return s.mla ? 64 : s.bs; }
inline int plan_unit_pages(const DecodeShape& s) {
  return s.mla_tc ? 2 : (s.gqa_tc ? 128 / s.bs : 1);
}

int decode_workers(const DecodeShape& s, int fmt, int mode, int device);

// Shared by both kernel families: the planner (flat (request, group, page)
// list cut into equal ranges) and the log-sum-exp merge of the pieces.
// `groups` is the number of head groups per request (KV heads for GQA, groups
// of 32 query heads for MLA) and G the query heads per group.  `batch`
// counts virtual requests (request x query of a causal chunk of `qlen`).
cudaError_t launch_plan(const int32_t* seq_lens, int batch, int qlen, int qw, int groups, int bs,
                        int max_blocks, int workers, int* plan, uint32_t* err,
                        cudaStream_t stream, int upages = 1);
cudaError_t launch_merge(const int* plan, const float* part_ml, const float* part_o, void* out,
                         int batch, int qw, int hq, int groups, int G, int dv, int out_dtype,
                         cudaStream_t stream);
cudaError_t launch_decode_gqa(const DecodeShape& s, const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_decode_mla(const DecodeShape& s, const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_decode_mla_tc(const DecodeShape& s, const DecodeArgs& a, cudaStream_t stream);
// The tensor-core kernel for a causal chunk over the grouped-query layout:
// FP8 codes, per-token scales, head_dim 128, G x q_len = 16 or 32 columns.
bool gqa_tc_eligible(int fmt, int mode, int d, int dv, int bs, int hq, int hkv, int qlen);
int gqa_tc_workers(const DecodeShape& s, int device);
cudaError_t launch_decode_gqa_tc(const DecodeShape& s, const DecodeArgs& a, cudaStream_t stream);

// Cached launch set-up (per device): SM count, the dynamic shared-memory
// opt-in of a kernel (made once), and a kernel's resident CTAs per SM.
int sm_count(int device);
cudaError_t ensure_smem_attr(const void* fn, int smem);
int ctas_per_sm(const void* fn, int threads, int smem);

// Tensor-map encoder from the driver (resolved once through the runtime).
bool encode_tensor_map_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype,
                          uint32_t esize, uint64_t inner, uint64_t rows, uint32_t box_inner,
                          uint32_t box_rows, CUtensorMapSwizzle swz);
bool encode_tensor_map_2d_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                             uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swz);
bool encode_tensor_map_2d_f32(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                              uint32_t box_inner, uint32_t box_rows);

extern int g_decode_workers_override;
extern cudaEvent_t g_split_ev_start, g_split_ev_stop;

}  // namespace fp8pa
