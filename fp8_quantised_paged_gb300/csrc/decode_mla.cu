// decode_mla.cu -- placeholder until the shared-latent kernel lands.
#include "common.cuh"
#include "internal.h"

namespace fp8pa {

cudaError_t launch_decode_mla(const DecodeShape&, const DecodeArgs&, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace fp8pa
