// Tensor-core tiles for the multi-token (chunked-prefill) rows of a varlen batch.
#include "pa_common.cuh"

namespace pa {

int prefill_tile_tokens(int group) {
  int g8 = 1;
  while (g8 < group && g8 < 8) g8 <<= 1;
  return 128 / g8;
}

bool prefill_mma_supported(int, int, int, int, int) { return false; }

cudaError_t launch_prefill_mma(const AttnParams&, int, int, int, const CUtensorMap*,
                               const CUtensorMap*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace pa
