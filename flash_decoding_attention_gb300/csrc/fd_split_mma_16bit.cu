// fd_split_mma_16bit.cu -- the tensor-core split kernel's variants for fp16 and bf16 caches
// (see fd_split_mma.cuh); one translation unit per cache format so that the
// variants compile in parallel.
#include "fd_split_mma.cuh"

namespace fd {
namespace mma {

cudaError_t launch_16bit(const Params& p, const Shape& sh, const Maps& m, cudaStream_t st) {
  if (p.kv_dtype == FD_F16)
    return p.head_dim == 128 ? launch_plain<FD_F16, __half, 128>(p, sh, m, st)
                             : launch_plain<FD_F16, __half, 64>(p, sh, m, st);
  return p.head_dim == 128 ? launch_plain<FD_BF16, __nv_bfloat16, 128>(p, sh, m, st)
                           : launch_plain<FD_BF16, __nv_bfloat16, 64>(p, sh, m, st);
}

}  // namespace mma
}  // namespace fd
