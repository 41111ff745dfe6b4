// decode_noalloc.cu -- fp8pa_paged_decode_attention_static_ws: the decode
// for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc or any allocator: a
// host framework that hands its plugins only the input and output buffers
// and keeps the device allocator to itself, or a serving process that fixes
// its memory footprint at start-up and forbids allocations afterwards.  The
// regular decode needs a caller-provided workspace for its split partials,
// which such callers have no way to obtain.  This entry point gives them the
// same computation with the scratch taken from a fixed array compiled into
// the library.
//
// The array is a file-scope static __device__ buffer of
// FP8PA_STATIC_WORKSPACE_BYTES.  Its device address is looked up once per
// device (cudaGetSymbolAddress, with that device current) on the first call
// made on that device; make that first call before any stream capture.  All
// calls on a device share the one array and it keeps whatever the last call
// left there: nothing in it has to start at zero, because every byte the
// decode reads from its workspace is written earlier in the same call.  Two
// calls whose kernels overlap on the GPU (different streams, no ordering
// between them) race on the array and give undefined results.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace fp8pa {
namespace {

static __device__ __align__(256) unsigned char g_static_workspace[FP8PA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevs = 64;
void* g_static_ws_addr[kMaxDevs] = {nullptr};
std::mutex g_static_ws_mu;

// Device address of the array on the current device (set up on first use).
int static_workspace(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevs) return FP8PA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_static_ws_mu);
  if (!g_static_ws_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return FP8PA_ERR_CUDA;
    g_static_ws_addr[dev] = p;
  }
  *out = g_static_ws_addr[dev];
  return FP8PA_OK;
}

}  // namespace
}  // namespace fp8pa

extern "C" int fp8pa_paged_decode_attention_static_ws(
    const void* q, const uint8_t* k_cache, const uint8_t* v_cache, const float* k_scale,
    const float* v_scale, const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* seq_lens, int batch, int block_size, int n_q_heads, int n_kv_heads,
    int head_dim, int head_dim_v, int fmt, int scale_mode, int group_size, float sm_scale,
    int num_blocks, void* out, int out_dtype, void* stream) {
  void* ws = nullptr;
  const int st = fp8pa::static_workspace(&ws);
  if (st != FP8PA_OK) return st;
  // The size the regular decode needs for these shapes on this device (0
  // when the shapes are rejected; the call below then returns the reason).
  const size_t need = fp8pa_decode_workspace_bytes(batch, n_q_heads, n_kv_heads, head_dim,
                                                   head_dim_v, block_size, max_blocks_per_seq);
  if (need > FP8PA_STATIC_WORKSPACE_BYTES) return FP8PA_ERR_WORKSPACE;
  return fp8pa_paged_decode_attention(q, k_cache, v_cache, k_scale, v_scale, block_tables,
                                      max_blocks_per_seq, seq_lens, batch, block_size, n_q_heads,
                                      n_kv_heads, head_dim, head_dim_v, fmt, scale_mode,
                                      group_size, sm_scale, num_blocks, out, out_dtype, ws,
                                      FP8PA_STATIC_WORKSPACE_BYTES, stream);
}
