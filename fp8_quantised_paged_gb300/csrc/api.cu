// api.cu -- the extern "C" boundary declared in include/fp8pa.h: argument
// validation, dispatch to the kernels, tensor-map encoding, the per-device
// error word and status strings.  No call allocates device memory.
#include <cudaTypedefs.h>

#include <mutex>
#include <utility>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace fp8pa {

// The device error word (one per device that loads the library).
__device__ uint32_t g_device_error;

namespace {

void* g_err_ptr[kMaxDevices] = {nullptr};

uint32_t* device_error_ptr(cudaStream_t stream, int* dev_out) {
  return static_cast<uint32_t*>(
      symbol_device_address(reinterpret_cast<const void*>(&g_device_error), g_err_ptr, stream,
                            dev_out));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? FP8PA_OK : FP8PA_ERR_CUDA; }

std::mutex g_sym_mu;

}  // namespace

// Device address of a __device__ variable on the current device.  It is
// looked up again on every call made outside stream capture, so nothing
// stale survives a cudaDeviceReset (which reloads the module) or a switch
// of context; during a capture (where a first-time module load must not
// happen) the address recorded by the last uncaptured call on this device
// is used.  `cache` has kMaxDevices entries.
void* symbol_device_address(const void* symbol, void** cache, cudaStream_t stream,
                            int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  if (dev_out) *dev_out = dev;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lock(g_sym_mu);
  if (cs == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess || !p) return nullptr;
    cache[dev] = p;
  }
  return cache[dev];
}

// Per-device host caches of the launch set-up that does not change between
// calls: the SM count, the dynamic shared-memory opt-in of each kernel, and
// each kernel's resident CTAs per SM.
namespace {
struct FnKey {
  int dev;
  const void* fn;
  int threads, smem;
};
std::mutex g_cache_mu;
int g_sms[kMaxDevices] = {0};
std::vector<std::pair<FnKey, int>> g_occ;  // (key, CTAs per SM)
std::vector<FnKey> g_attr;                 // smem opt-ins already made
}  // namespace

int sm_count(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return 1;
  std::lock_guard<std::mutex> lock(g_cache_mu);
  if (g_sms[dev] <= 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return 1;
    g_sms[dev] = n;
  }
  return g_sms[dev];
}

cudaError_t ensure_smem_attr(const void* fn, int smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_cache_mu);
  for (const FnKey& k : g_attr)
    if (k.dev == dev && k.fn == fn && k.smem >= smem) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) g_attr.push_back(FnKey{dev, fn, 0, smem});
  return e;
}

int ctas_per_sm(const void* fn, int threads, int smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  {
    std::lock_guard<std::mutex> lock(g_cache_mu);
    for (const auto& kv : g_occ)
      if (kv.first.dev == dev && kv.first.fn == fn && kv.first.threads == threads &&
          kv.first.smem == smem)
        return kv.second;
  }
  if (ensure_smem_attr(fn, smem) != cudaSuccess) return 1;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem) != cudaSuccess ||
      per_sm <= 0)
    return 1;
  std::lock_guard<std::mutex> lock(g_cache_mu);
  g_occ.push_back({FnKey{dev, fn, threads, smem}, per_sm});
  return per_sm;
}

namespace {

// One warp waits on a barrier that no copy or thread completes; the bounded
// wait gives up after `limit` cycles and records the timeout.
__global__ void __launch_bounds__(32) bounded_wait_selftest_kernel(long long limit,
                                                                  uint32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncwarp();
  const bool landed = mbar_wait_bounded(&bar, 0, limit);
  if (!__all_sync(0xffffffffu, landed) && threadIdx.x == 0)
    raise_error(err, FP8PA_DEVERR_TIMEOUT);
}

}  // namespace

bool encode_tensor_map_2d_f32(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                              uint32_t box_inner, uint32_t box_rows) {
  return encode_tensor_map_2d(map, base, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, inner, rows,
                              box_inner, box_rows, CU_TENSOR_MAP_SWIZZLE_NONE);
}

bool encode_tensor_map_2d_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                             uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swz) {
  return encode_tensor_map_2d(map, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, inner, rows, box_inner,
                              box_rows, swz);
}

// A row-major 2-D tensor of `rows` rows of `inner` elements of `esize` bytes.
bool encode_tensor_map_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype,
                          uint32_t esize, uint64_t inner, uint64_t rows, uint32_t box_inner,
                          uint32_t box_rows, CUtensorMapSwizzle swz) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return false;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * esize};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, dtype, 2, const_cast<void*>(base), dims,
                            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace fp8pa

using namespace fp8pa;

namespace {

struct DecodePath {
  DecodeShape shape;
  int status;
};

// Validate the decode shapes of `batch` virtual requests (requests x q_len
// queries; pointers are checked by the caller) and choose the kernel family.
DecodePath decode_path(int batch, int q_len, int hq, int hkv, int d, int dv, int bs,
                       int max_blocks, int fmt, int mode, int gs, int num_blocks,
                       int out_dtype) {
  DecodePath r{};
  r.status = FP8PA_OK;
  DecodeShape& s = r.shape;
  s.batch = batch;
  s.hq = hq;
  s.hkv = hkv;
  s.d = d;
  s.dv = dv;
  s.bs = bs;
  s.max_blocks = max_blocks;
  s.mla = 0;
  s.qlen = q_len;
  s.gqa_tc = 0;
  s.gs = gs;
  if ((fmt != FP8PA_E4M3 && fmt != FP8PA_E5M2 && fmt != FP8PA_INT8) ||
      (mode != FP8PA_SCALE_TOKEN_HEAD && mode != FP8PA_SCALE_CHANNEL_STATIC &&
       mode != FP8PA_SCALE_TOKEN_GROUP && mode != FP8PA_SCALE_MX_BLOCK &&
       mode != FP8PA_SCALE_SEGMENT) ||
      (out_dtype != FP8PA_OUT_BF16 && out_dtype != FP8PA_OUT_F32)) {
    r.status = FP8PA_ERR_BAD_ENUM;
    return r;
  }
  if (batch < 0 || hq <= 0 || hkv <= 0 || hq % hkv != 0 || bs <= 0 || max_blocks <= 0 ||
      num_blocks <= 0 || d <= 0 || dv <= 0) {
    r.status = FP8PA_ERR_BAD_SHAPE;
    return r;
  }
  // chunks with G x qw = 16 or 32 (query, head) columns run on the tensor cores
  s.gqa_tc = gqa_tc_eligible(fmt, mode, d, dv, bs, hq, hkv, q_len) ? 1 : 0;
  if (static_cast<long long>(num_blocks) * hkv * bs >= (1ll << 31) ||
      static_cast<long long>(max_blocks) * bs >= (1ll << 31) ||
      static_cast<long long>(batch) * max_blocks * bs * hkv >= (1ll << 31)) {
    r.status = FP8PA_ERR_UNSUPPORTED;
    return r;
  }
  if (d == 576) {
    s.mla = 1;
    if (hkv != 1 || dv != 512 || bs != 64 || hq % 32 != 0 ||
        !((mode == FP8PA_SCALE_TOKEN_GROUP && gs == 64) || mode == FP8PA_SCALE_SEGMENT))
      r.status = FP8PA_ERR_UNSUPPORTED;
    // FP8 latents with whole groups of 64 heads run on the tensor cores
    s.mla_tc = (fmt != FP8PA_INT8 && hq % 64 == 0) ? 1 : 0;
    return r;
  }
  if ((d != 64 && d != 128) || dv != d || (bs != 16 && bs != 32 && bs != 64) ||
      (hq / hkv > 8 && !s.gqa_tc) ||
      mode == FP8PA_SCALE_TOKEN_GROUP ||
      (mode == FP8PA_SCALE_MX_BLOCK && ((gs != 16 && gs != 32) || fmt == FP8PA_INT8)))
    r.status = FP8PA_ERR_UNSUPPORTED;
  return r;
}

// Validate the attention arguments of `batch` requests with `q_len` queries
// each (a causal chunk; q_len = 1 is plain decode) and fill the launch
// description.  The kernels see batch * q_len virtual requests; q and out
// rows are (request, query) in that order.  Returns FP8PA_OK with
// path->shape.batch == 0 when there is nothing to launch.
int attention_prepare(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                      const float* k_scale, const float* v_scale, const int32_t* block_tables,
                      int max_blocks_per_seq, const int32_t* seq_lens, int batch, int q_len,
                      int block_size, int n_q_heads, int n_kv_heads, int head_dim,
                      int head_dim_v, int fmt, int scale_mode, int group_size, float sm_scale,
                      int num_blocks, void* out, int out_dtype, void* workspace,
                      size_t workspace_bytes, cudaStream_t stream, DecodePath* path,
                      DecodeArgs* a) {
  if (q_len <= 0 || batch < 0) return FP8PA_ERR_BAD_SHAPE;
  if (static_cast<long long>(batch) * q_len >= (1ll << 31)) return FP8PA_ERR_UNSUPPORTED;
  *path = decode_path(batch * q_len, q_len, n_q_heads, n_kv_heads, head_dim, head_dim_v,
                      block_size, max_blocks_per_seq, fmt, scale_mode, group_size, num_blocks,
                      out_dtype);
  if (path->status != FP8PA_OK) return path->status;
  if (batch == 0) return FP8PA_OK;
  if (!q || !k_cache || !k_scale || !block_tables || !seq_lens || !out || !workspace)
    return FP8PA_ERR_NULL_POINTER;
  if (path->shape.mla) {
    if (v_cache != k_cache || v_scale != k_scale) return FP8PA_ERR_UNSUPPORTED;
  } else if (!v_cache || !v_scale) {
    return FP8PA_ERR_NULL_POINTER;
  }
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_scale) ||
      !aligned16(v_scale) || !aligned16(workspace) || !aligned16(out))
    return FP8PA_ERR_ALIGNMENT;
  int dev = 0;
  uint32_t* err = device_error_ptr(stream, &dev);
  if (!err) return FP8PA_ERR_CUDA;
  path->shape.workers = decode_workers(path->shape, fmt, scale_mode, dev);
  if (workspace_bytes < decode_workspace_bytes(path->shape)) return FP8PA_ERR_WORKSPACE;
  *a = DecodeArgs{};
  a->q = static_cast<const uint16_t*>(q);
  a->k_cache = k_cache;
  a->v_cache = v_cache;
  a->k_scale = k_scale;
  a->v_scale = v_scale;
  a->block_tables = block_tables;
  a->seq_lens = seq_lens;
  a->num_blocks = num_blocks;
  a->fmt = fmt;
  a->mode = scale_mode;
  a->gs = group_size;
  a->out_dtype = out_dtype;
  a->sm_scale = sm_scale;
  a->out = out;
  a->workspace = workspace;
  a->err = err;
  a->plan_ready = false;
  return FP8PA_OK;
}

cudaError_t launch_decode(const DecodePath& path, const DecodeArgs& a, cudaStream_t st) {
  return path.shape.mla ? launch_decode_mla(path.shape, a, st)
                         : launch_decode_gqa(path.shape, a, st);
}

int attention_impl(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                   const float* k_scale, const float* v_scale, const int32_t* block_tables,
                   int max_blocks_per_seq, const int32_t* seq_lens, int batch, int q_len,
                   int block_size, int n_q_heads, int n_kv_heads, int head_dim, int head_dim_v,
                   int fmt, int scale_mode, int group_size, float sm_scale, int num_blocks,
                   void* out, int out_dtype, void* workspace, size_t workspace_bytes,
                   void* stream) {
  DecodePath path;
  DecodeArgs a;
  const int st = attention_prepare(q, k_cache, v_cache, k_scale, v_scale, block_tables,
                                   max_blocks_per_seq, seq_lens, batch, q_len, block_size,
                                   n_q_heads, n_kv_heads, head_dim, head_dim_v, fmt, scale_mode,
                                   group_size, sm_scale, num_blocks, out, out_dtype, workspace,
                                   workspace_bytes, static_cast<cudaStream_t>(stream), &path, &a);
  if (st != FP8PA_OK || batch == 0) return st;
  return cuda_status(launch_decode(path, a, static_cast<cudaStream_t>(stream)));
}

// Validate the append arguments and fill `a` (its error word excluded).
int append_prepare(const void* k, const void* v, const int32_t* slot_mapping, int num_tokens,
                   int n_kv_heads, int head_dim, int fmt, int scale_mode, int group_size,
                   uint8_t* k_cache, uint8_t* v_cache, float* k_scale, float* v_scale,
                   int num_blocks, int block_size, AppendArgs* a) {
  if (num_tokens < 0 || n_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0 || block_size <= 0)
    return FP8PA_ERR_BAD_SHAPE;
  if ((fmt != FP8PA_E4M3 && fmt != FP8PA_E5M2 && fmt != FP8PA_INT8) ||
      (scale_mode != FP8PA_SCALE_TOKEN_HEAD && scale_mode != FP8PA_SCALE_CHANNEL_STATIC &&
       scale_mode != FP8PA_SCALE_TOKEN_GROUP && scale_mode != FP8PA_SCALE_MX_BLOCK &&
       scale_mode != FP8PA_SCALE_SEGMENT))
    return FP8PA_ERR_BAD_ENUM;
  if (head_dim % 16 != 0 || head_dim > 768) return FP8PA_ERR_UNSUPPORTED;
  if (scale_mode == FP8PA_SCALE_TOKEN_GROUP &&
      (!pow2(group_size) || group_size < 16 || group_size > 256 || head_dim % group_size != 0))
    return FP8PA_ERR_UNSUPPORTED;
  if (scale_mode == FP8PA_SCALE_MX_BLOCK &&
      ((group_size != 16 && group_size != 32) || head_dim % group_size != 0 || fmt == FP8PA_INT8))
    return FP8PA_ERR_UNSUPPORTED;
  // the segment mode needs token positions: fp8pa_kv_append_quant_segment
  if (scale_mode == FP8PA_SCALE_SEGMENT) return FP8PA_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_blocks) * block_size >= (1ll << 31) ||
      static_cast<long long>(num_tokens) * n_kv_heads * 2 >= (1ll << 31))
    return FP8PA_ERR_UNSUPPORTED;
  *a = AppendArgs{};
  a->num_tokens = num_tokens;
  if (num_tokens == 0) return FP8PA_OK;
  if (!k || !slot_mapping || !k_cache || !k_scale) return FP8PA_ERR_NULL_POINTER;
  if (v && (!v_cache || !v_scale)) return FP8PA_ERR_NULL_POINTER;
  if (!aligned16(k) || !aligned16(k_cache) || (v && (!aligned16(v) || !aligned16(v_cache))) ||
      !aligned16(k_scale) || (v && !aligned16(v_scale)))
    return FP8PA_ERR_ALIGNMENT;
  a->src[0] = static_cast<const uint16_t*>(k);
  a->src[1] = static_cast<const uint16_t*>(v);
  a->cache[0] = k_cache;
  a->cache[1] = v_cache;
  a->scale[0] = k_scale;
  a->scale[1] = v_scale;
  a->slot_mapping = slot_mapping;
  a->hkv = n_kv_heads;
  a->d = head_dim;
  a->ntens = v ? 2 : 1;
  a->gs = (scale_mode == FP8PA_SCALE_TOKEN_GROUP || scale_mode == FP8PA_SCALE_MX_BLOCK)
              ? group_size
              : head_dim;
  a->num_blocks = num_blocks;
  a->bs = block_size;
  a->div_tok = make_fast_div(static_cast<uint32_t>(n_kv_heads * a->ntens));
  a->div_bs = make_fast_div(static_cast<uint32_t>(block_size));
  return FP8PA_OK;
}

}  // namespace

extern "C" {

int fp8pa_version(void) { return (1 << 16) | 0; }

const char* fp8pa_error_string(int code) {
  switch (code) {
    case FP8PA_OK: return "ok";
    case FP8PA_ERR_NULL_POINTER: return "a required pointer is NULL";
    case FP8PA_ERR_BAD_ENUM: return "unknown fmt, scale_mode or out_dtype";
    case FP8PA_ERR_BAD_SHAPE: return "inconsistent or non-positive sizes";
    case FP8PA_ERR_UNSUPPORTED: return "shape or mode combination not supported";
    case FP8PA_ERR_WORKSPACE: return "workspace missing or too small";
    case FP8PA_ERR_ALIGNMENT: return "a pointer is not 16-byte aligned";
    case FP8PA_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown status";
  }
}

int fp8pa_set_decode_workers(int workers) {
  if (workers < 0) return FP8PA_ERR_BAD_SHAPE;
  g_decode_workers_override = workers;
  return FP8PA_OK;
}

int fp8pa_set_split_events(void* start, void* stop) {
  if ((start == nullptr) != (stop == nullptr)) return FP8PA_ERR_NULL_POINTER;
  g_split_ev_start = static_cast<cudaEvent_t>(start);
  g_split_ev_stop = static_cast<cudaEvent_t>(stop);
  return FP8PA_OK;
}

int fp8pa_kv_append_quant(const void* k, const void* v, const int32_t* slot_mapping,
                          int num_tokens, int n_kv_heads, int head_dim, int fmt, int scale_mode,
                          int group_size, uint8_t* k_cache, uint8_t* v_cache, float* k_scale,
                          float* v_scale, int num_blocks, int block_size, void* stream) {
  AppendArgs a;
  const int st = append_prepare(k, v, slot_mapping, num_tokens, n_kv_heads, head_dim, fmt,
                                scale_mode, group_size, k_cache, v_cache, k_scale, v_scale,
                                num_blocks, block_size, &a);
  if (st != FP8PA_OK || num_tokens == 0) return st;
  a.err = device_error_ptr(static_cast<cudaStream_t>(stream), nullptr);
  if (!a.err) return FP8PA_ERR_CUDA;
  return cuda_status(launch_append(a, fmt, scale_mode, static_cast<cudaStream_t>(stream)));
}

int fp8pa_kv_append_quant_segment(const void* k, const void* v, const int32_t* slot_mapping,
                                  const int32_t* seq_offsets, const int32_t* seq_start_pos,
                                  int num_seqs, int n_kv_heads, int head_dim, int fmt,
                                  float* seg_state, uint8_t* k_cache, uint8_t* v_cache,
                                  float* k_scale, float* v_scale, int num_blocks, int block_size,
                                  void* stream) {
  if (num_seqs < 0 || n_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0 || block_size <= 0)
    return FP8PA_ERR_BAD_SHAPE;
  if (fmt != FP8PA_E4M3 && fmt != FP8PA_E5M2 && fmt != FP8PA_INT8) return FP8PA_ERR_BAD_ENUM;
  if (head_dim % 16 != 0 || head_dim > 768 || kSegmentTokens % block_size != 0)
    return FP8PA_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_blocks) * block_size >= (1ll << 31) ||
      static_cast<long long>(num_seqs) * 2 * n_kv_heads >= (1ll << 31))
    return FP8PA_ERR_UNSUPPORTED;
  if (num_seqs == 0) return FP8PA_OK;
  if (!k || !slot_mapping || !seq_offsets || !seq_start_pos || !seg_state || !k_cache ||
      !k_scale)
    return FP8PA_ERR_NULL_POINTER;
  if (v && (!v_cache || !v_scale)) return FP8PA_ERR_NULL_POINTER;
  if (!aligned16(k) || !aligned16(k_cache) || !aligned16(k_scale) ||
      (v && (!aligned16(v) || !aligned16(v_cache) || !aligned16(v_scale))))
    return FP8PA_ERR_ALIGNMENT;
  SegmentArgs a{};
  a.src[0] = static_cast<const uint16_t*>(k);
  a.src[1] = static_cast<const uint16_t*>(v);
  a.cache[0] = k_cache;
  a.cache[1] = v_cache;
  a.scale[0] = k_scale;
  a.scale[1] = v_scale;
  a.slot_mapping = slot_mapping;
  a.seq_offsets = seq_offsets;
  a.seq_start = seq_start_pos;
  a.state = seg_state;
  a.num_seqs = num_seqs;
  a.hkv = n_kv_heads;
  a.hp = segment_scale_heads(n_kv_heads);
  a.d = head_dim;
  a.ntens = v ? 2 : 1;
  a.num_blocks = num_blocks;
  a.bs = block_size;
  a.err = device_error_ptr(static_cast<cudaStream_t>(stream), nullptr);
  if (!a.err) return FP8PA_ERR_CUDA;
  return cuda_status(launch_append_segment(a, fmt, static_cast<cudaStream_t>(stream)));
}

int fp8pa_kv_channel_scales(const void* x, int num_tokens, int n_kv_heads, int head_dim, int fmt,
                            float* scale_out, void* stream) {
  if (num_tokens < 0 || n_kv_heads <= 0 || head_dim <= 0) return FP8PA_ERR_BAD_SHAPE;
  if (fmt != FP8PA_E4M3 && fmt != FP8PA_E5M2 && fmt != FP8PA_INT8) return FP8PA_ERR_BAD_ENUM;
  if (head_dim % 16 != 0) return FP8PA_ERR_UNSUPPORTED;
  if (!scale_out || (num_tokens > 0 && !x)) return FP8PA_ERR_NULL_POINTER;
  if ((num_tokens > 0 && !aligned16(x)) || !aligned16(scale_out)) return FP8PA_ERR_ALIGNMENT;
  return cuda_status(launch_channel_scales(static_cast<const uint16_t*>(x), num_tokens,
                                           n_kv_heads * head_dim, fmt, scale_out,
                                           static_cast<cudaStream_t>(stream)));
}

int fp8pa_kv_channel_absmax_update(const void* x, int num_tokens, int n_kv_heads, int head_dim,
                                   float* running_absmax, void* stream) {
  if (num_tokens < 0 || n_kv_heads <= 0 || head_dim <= 0) return FP8PA_ERR_BAD_SHAPE;
  if (head_dim % 16 != 0) return FP8PA_ERR_UNSUPPORTED;
  if (!running_absmax || (num_tokens > 0 && !x)) return FP8PA_ERR_NULL_POINTER;
  if ((num_tokens > 0 && !aligned16(x)) || !aligned16(running_absmax)) return FP8PA_ERR_ALIGNMENT;
  return cuda_status(launch_channel_absmax(static_cast<const uint16_t*>(x), num_tokens,
                                           n_kv_heads * head_dim, running_absmax,
                                           static_cast<cudaStream_t>(stream)));
}

int fp8pa_kv_scales_from_absmax(const float* absmax, int n, int fmt, float* scale_out,
                                void* stream) {
  if (n <= 0) return FP8PA_ERR_BAD_SHAPE;
  if (fmt != FP8PA_E4M3 && fmt != FP8PA_E5M2 && fmt != FP8PA_INT8) return FP8PA_ERR_BAD_ENUM;
  if (!absmax || !scale_out) return FP8PA_ERR_NULL_POINTER;
  return cuda_status(
      launch_scales_from_absmax(absmax, n, fmt, scale_out, static_cast<cudaStream_t>(stream)));
}

size_t fp8pa_multiquery_workspace_bytes(int batch, int q_len, int n_q_heads, int n_kv_heads,
                                        int head_dim, int head_dim_v, int block_size,
                                        int max_blocks_per_seq) {
  if (q_len <= 0 || batch < 0 || static_cast<long long>(batch) * q_len >= (1ll << 31)) return 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  // The largest need over the scale modes and formats of this layout (the
  // split count follows each kernel's occupancy; MX blocks of 16 and of 32
  // dims run different kernels).
  const bool mla = head_dim == 576;
  const int modes[5] = {mla ? FP8PA_SCALE_TOKEN_GROUP : FP8PA_SCALE_TOKEN_HEAD,
                        mla ? FP8PA_SCALE_SEGMENT : FP8PA_SCALE_CHANNEL_STATIC,
                        FP8PA_SCALE_MX_BLOCK, FP8PA_SCALE_MX_BLOCK, FP8PA_SCALE_SEGMENT};
  const int sizes[5] = {mla ? 64 : 16, mla ? 64 : 16, 16, 32, 16};
  size_t need = 0;
  for (int m = 0; m < (mla ? 2 : 5); ++m)
    for (int fmt = FP8PA_E4M3; fmt <= FP8PA_INT8; ++fmt) {
      DecodePath path = decode_path(batch * q_len, q_len, n_q_heads, n_kv_heads, head_dim,
                                    head_dim_v, block_size, max_blocks_per_seq, fmt, modes[m],
                                    sizes[m], 1, FP8PA_OUT_BF16);
      if (path.status != FP8PA_OK) continue;
      path.shape.workers = decode_workers(path.shape, fmt, modes[m], dev);
      const size_t n = decode_workspace_bytes(path.shape);
      need = n > need ? n : need;
    }
  return need;
}

size_t fp8pa_decode_workspace_bytes(int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                    int head_dim_v, int block_size, int max_blocks_per_seq) {
  return fp8pa_multiquery_workspace_bytes(batch, 1, n_q_heads, n_kv_heads, head_dim, head_dim_v,
                                          block_size, max_blocks_per_seq);
}

int fp8pa_paged_decode_attention(const void* q, const uint8_t* k_cache, const uint8_t* v_cache,
                                 const float* k_scale, const float* v_scale,
                                 const int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* seq_lens, int batch, int block_size,
                                 int n_q_heads, int n_kv_heads, int head_dim, int head_dim_v,
                                 int fmt, int scale_mode, int group_size, float sm_scale,
                                 int num_blocks, void* out, int out_dtype, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  return attention_impl(q, k_cache, v_cache, k_scale, v_scale, block_tables, max_blocks_per_seq,
                        seq_lens, batch, 1, block_size, n_q_heads, n_kv_heads, head_dim,
                        head_dim_v, fmt, scale_mode, group_size, sm_scale, num_blocks, out,
                        out_dtype, workspace, workspace_bytes, stream);
}

int fp8pa_paged_multiquery_attention(const void* q, const uint8_t* k_cache,
                                     const uint8_t* v_cache, const float* k_scale,
                                     const float* v_scale, const int32_t* block_tables,
                                     int max_blocks_per_seq, const int32_t* seq_lens, int batch,
                                     int q_len, int block_size, int n_q_heads, int n_kv_heads,
                                     int head_dim, int head_dim_v, int fmt, int scale_mode,
                                     int group_size, float sm_scale, int num_blocks, void* out,
                                     int out_dtype, void* workspace, size_t workspace_bytes,
                                     void* stream) {
  return attention_impl(q, k_cache, v_cache, k_scale, v_scale, block_tables, max_blocks_per_seq,
                        seq_lens, batch, q_len, block_size, n_q_heads, n_kv_heads, head_dim,
                        head_dim_v, fmt, scale_mode, group_size, sm_scale, num_blocks, out,
                        out_dtype, workspace, workspace_bytes, stream);
}

int fp8pa_decode_step(const void* k_new, const void* v_new, const int32_t* slot_mapping,
                      int num_new_tokens, const void* q, uint8_t* k_cache, uint8_t* v_cache,
                      float* k_scale, float* v_scale, const int32_t* block_tables,
                      int max_blocks_per_seq, const int32_t* seq_lens, int batch, int q_len,
                      int block_size, int n_q_heads, int n_kv_heads, int head_dim,
                      int head_dim_v, int fmt, int scale_mode, int group_size, float sm_scale,
                      int num_blocks, void* out, int out_dtype, void* workspace,
                      size_t workspace_bytes, void* stream) {
  AppendArgs ap;
  int st = append_prepare(k_new, v_new, slot_mapping, num_new_tokens, n_kv_heads, head_dim, fmt,
                          scale_mode, group_size, k_cache, v_cache, k_scale, v_scale, num_blocks,
                          block_size, &ap);
  if (st != FP8PA_OK) return st;
  DecodePath path;
  DecodeArgs a;
  st = attention_prepare(q, k_cache, v_cache, k_scale, v_scale, block_tables, max_blocks_per_seq,
                         seq_lens, batch, q_len, block_size, n_q_heads, n_kv_heads, head_dim,
                         head_dim_v, fmt, scale_mode, group_size, sm_scale, num_blocks, out,
                         out_dtype, workspace, workspace_bytes, static_cast<cudaStream_t>(stream),
                         &path, &a);
  if (st != FP8PA_OK) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  ap.err = a.err ? a.err : device_error_ptr(cs, nullptr);
  if (!ap.err) return FP8PA_ERR_CUDA;
  if (batch == 0)
    return num_new_tokens == 0 ? FP8PA_OK : cuda_status(launch_append(ap, fmt, scale_mode, cs));
  PlanArgs pl;
  pl.seq_lens = seq_lens;
  pl.qw = path.shape.mla ? 1 : gqa_qw(path.shape);
  pl.batch = path.shape.batch / pl.qw;  // planned requests
  pl.qlen = q_len;
  pl.bs = plan_block_size(path.shape);
  pl.max_blocks = max_blocks_per_seq;
  pl.workers = plan_workers(path.shape);
  pl.upages = plan_unit_pages(path.shape);
  pl.plan = static_cast<int*>(workspace);
  pl.err = a.err;
  cudaError_t e = launch_append_plan(ap, fmt, scale_mode, pl, cs);
  if (e != cudaSuccess) return FP8PA_ERR_CUDA;
  a.plan_ready = true;
  return cuda_status(launch_decode(path, a, cs));
}

int fp8pa_selftest_bounded_wait(long long limit_cycles, void* stream) {
  const long long limit =
      limit_cycles < 1000 ? 1000 : (limit_cycles > kWaitLimitCycles ? kWaitLimitCycles : limit_cycles);
  uint32_t* err = device_error_ptr(static_cast<cudaStream_t>(stream), nullptr);
  if (!err) return FP8PA_ERR_CUDA;
  bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit, err);
  return cuda_status(cudaGetLastError());
}

int fp8pa_get_device_error(void* stream, uint32_t* flags) {
  if (!flags) return FP8PA_ERR_NULL_POINTER;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FP8PA_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof v) != cudaSuccess) return FP8PA_ERR_CUDA;
  const uint32_t zero = 0;
  if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero) != cudaSuccess) return FP8PA_ERR_CUDA;
  *flags = v;
  return FP8PA_OK;
}

}  // extern "C"
