// fd_split_mma.cu -- split kernel on tensor cores (placeholder until written).
#include "fd_common.cuh"

namespace fd {

bool mma_supports(int, int, int, int, int, int, int) { return false; }

void mma_config(int, int, int, int, int sms, int* hc, int* tile, int* grid) {
  *hc = 1;
  *tile = 16;
  *grid = sms;
}

cudaError_t launch_split_mma(const Params&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace fd
