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
// FP8PA_STATIC_WORKSPACE_BYTES.  In host code its name is only a host-side
// stand-in, so its device address is looked up (cudaGetSymbolAddress, with
// the device current) on every call made outside stream capture; a call
// made during a capture uses the address the last uncaptured call on that
// device found, so make the first call on each device before any capture.
// Looking it up again each time keeps the call correct after a
// cudaDeviceReset, which reloads the library's module at a new address.
// All calls on a device share the one array and it keeps whatever the last
// call left there: nothing in it has to start at zero, because every byte
// the decode reads from its workspace is written earlier in the same call.
// Two calls whose kernels overlap on the GPU (different streams, no ordering
// between them) race on the array and give undefined results.
#include "common.cuh"
#include "internal.h"

namespace fp8pa {
namespace {

static __device__ __align__(256) unsigned char g_static_workspace[FP8PA_STATIC_WORKSPACE_BYTES];

void* g_static_ws_addr[kMaxDevices] = {nullptr};

}  // namespace
}  // namespace fp8pa

extern "C" int fp8pa_paged_decode_attention_static_ws(
    const void* q, const uint8_t* k_cache, const uint8_t* v_cache, const float* k_scale,
    const float* v_scale, const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* seq_lens, int batch, int block_size, int n_q_heads, int n_kv_heads,
    int head_dim, int head_dim_v, int fmt, int scale_mode, int group_size, float sm_scale,
    int num_blocks, void* out, int out_dtype, void* stream) {
  void* ws = fp8pa::symbol_device_address(
      reinterpret_cast<const void*>(&fp8pa::g_static_workspace), fp8pa::g_static_ws_addr,
      static_cast<cudaStream_t>(stream), nullptr);
  if (!ws) return FP8PA_ERR_CUDA;
  // The regular decode checks this call's own need (its format, scale mode
  // and split) against the array's size and returns FP8PA_ERR_WORKSPACE,
  // launching nothing, when it does not fit.
  return fp8pa_paged_decode_attention(q, k_cache, v_cache, k_scale, v_scale, block_tables,
                                      max_blocks_per_seq, seq_lens, batch, block_size, n_q_heads,
                                      n_kv_heads, head_dim, head_dim_v, fmt, scale_mode,
                                      group_size, sm_scale, num_blocks, out, out_dtype, ws,
                                      FP8PA_STATIC_WORKSPACE_BYTES, stream);
}
