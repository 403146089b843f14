// fd_split_mma_e4m3.cu -- the tensor-core split kernel's variants for FP8-e4m3 caches
// (see fd_split_mma.cuh); one translation unit per cache format so that the
// variants compile in parallel.
#include "fd_split_mma.cuh"

namespace fd {
namespace mma {

cudaError_t launch_e4m3(const Params& p, const Shape& sh, const Maps& m, cudaStream_t st) {
  return p.head_dim == 128 ? launch_8bit<FD_E4M3, 128>(p, sh, m, st)
                           : launch_8bit<FD_E4M3, 64>(p, sh, m, st);
}

#ifdef FD_STAMPS
cudaError_t read_stamps_e4m3(unsigned long long* host, int n) {
  if (n > kStampCtas * kStampSlots) n = kStampCtas * kStampSlots;
  return cudaMemcpyFromSymbol(host, g_split_stamps, sizeof(unsigned long long) * n);
}
#endif

}  // namespace mma
}  // namespace fd
