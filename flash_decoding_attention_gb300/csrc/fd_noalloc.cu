// fd_noalloc.cu -- decode attention for callers that cannot allocate device
// memory themselves.
//
// Some hosts of this library have no way to obtain extra device memory: code
// that runs inside a framework whose allocator is not exposed to plugins,
// tools that only receive pointers to existing tensors, or callers that must
// not add allocations to a pre-planned memory budget.  For them,
// fd_decode_attention_noalloc runs the same kernels as fd_decode_attention
// but takes its scratch memory from a fixed array compiled into this library
// instead of a caller-provided workspace.
//
// The array is a file-scope __device__ object, so every GPU that loads the
// library holds kStaticScratchBytes of it until the process exits.  Host code
// cannot use the array's name as a device address; the device address is
// looked up once per device with cudaGetSymbolAddress (while that device is
// current) on the first call made on that device, and cached for the life of
// the process (the entry point is not for use after cudaDeviceReset).
#include <mutex>

#include "fd_common.cuh"

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;   // 16 MiB per device
constexpr int kMaxDevices = 64;

__device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the static scratch array on the current device, or
// nullptr if it cannot be obtained.
void* scratch_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess) return nullptr;
    g_scratch_addr[dev] = ptr;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" fd_status fd_decode_attention_noalloc(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* kv_start_idx,
    const int32_t* block_table, int block_table_stride, const int32_t* seq_len, int64_t kv_rows,
    int batch, int num_q_heads, int num_kv_heads, int head_dim, int page_size,
    float softmax_scale, float k_scale, float v_scale, fd_dtype q_dtype, fd_dtype kv_dtype,
    void* out, float* lse, fd_stream_t stream) {
  // the argument checks of fd_decode_attention first, so that both entry
  // points give bad arguments the same status (the array stands in for the
  // workspace, which is only checked for presence here)
  const fd_status chk = fd::check_decode_args(
      q, k_cache, v_cache, kv_start_idx, block_table, block_table_stride, seq_len, kv_rows, batch,
      num_q_heads, num_kv_heads, head_dim, page_size, softmax_scale, k_scale, v_scale,
      FD_SCALE_TENSOR, nullptr, nullptr, q_dtype, kv_dtype, out, lse, g_static_scratch, 1);
  if (chk != FD_OK) return chk;
  const size_t need = fd_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim);
  if (need == 0) return FD_ERR_CUDA;   // valid sizes: only the device query can fail
  if (need > kStaticScratchBytes) return FD_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = scratch_for_current_device();
  if (scratch == nullptr) return FD_ERR_CUDA;
  // The array keeps the previous call's contents; only the header's device
  // error word must start at zero (every other byte is written before it is
  // read within a call).
  if (cudaMemsetAsync(scratch, 0, sizeof(fd::WsHeader), reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return FD_ERR_CUDA;
  return fd_decode_attention(q, k_cache, v_cache, kv_start_idx, block_table, block_table_stride,
                             seq_len, kv_rows, batch, num_q_heads, num_kv_heads, head_dim,
                             page_size, softmax_scale, k_scale, v_scale, q_dtype, kv_dtype, out,
                             lse, scratch, kStaticScratchBytes, stream);
}
