// fd_split_mma_i8.cu -- the tensor-core split kernel's variants for INT8 caches
// (see fd_split_mma.cuh); one translation unit per cache format so that the
// variants compile in parallel.
#include "fd_split_mma.cuh"

namespace fd {
namespace mma {

cudaError_t launch_i8(const Params& p, const Shape& sh, const Maps& m, cudaStream_t st) {
  return p.head_dim == 128 ? launch_8bit<FD_I8, 128>(p, sh, m, st)
                           : launch_8bit<FD_I8, 64>(p, sh, m, st);
}

}  // namespace mma
}  // namespace fd
