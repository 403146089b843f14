// fd_split_mma.cu -- host side of the tensor-core split kernel: tensor maps
// (cached), shapes, dispatch to the per-format translation units.
#include <cstring>
#include <mutex>

#include "fd_split_mma.cuh"

namespace fd {

// the tcgen05 split kernel (fd_split_tc.cu)
cudaError_t launch_split_tc(const Params& p, const CUtensorMap& mk, const CUtensorMap& mv,
                            cudaStream_t stream);

namespace mma {
namespace {

// ---------------------------------------------------------------------------
// Host side: tensor maps (cached), launch
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

struct MapKey {
  const void* ptr;
  long long rows;
  int kvh, d, dtype, box_rows, row_bytes, heads;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && rows == o.rows && kvh == o.kvh && d == o.d && dtype == o.dtype &&
           box_rows == o.box_rows && row_bytes == o.row_bytes && heads == o.heads;
  }
};

constexpr int kMapCache = 32;
std::mutex g_map_mu;
MapKey g_keys[kMapCache];
CUtensorMap g_maps[kMapCache];
int g_map_used = 0, g_map_next = 0;

// 3-D view of a cache.  heads == 0: dims {head_dim, kv_heads, rows}, box
// {row_bytes/elem, 1, box_rows} (one head per box).  heads > 0: dims
// {head_dim, rows, kv_heads}, box {row_bytes/elem, box_rows, heads}, so that
// one box lands in shared memory as [heads][box_rows][row_bytes].
bool get_map(const void* ptr, long long rows, int kvh, int d, int dtype, int box_rows,
             int row_bytes, int heads, CUtensorMap* out) {
  MapKey key{ptr, rows, kvh, d, dtype, box_rows, row_bytes, heads};
  std::lock_guard<std::mutex> lk(g_map_mu);
  for (int i = 0; i < g_map_used; ++i)
    if (g_keys[i] == key) {
      *out = g_maps[i];
      return true;
    }
  auto fn = encode_fn();
  if (!fn) return false;
  const int elem = kv_elem_bytes(dtype);
  CUtensorMapDataType dt = elem == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                     : CU_TENSOR_MAP_DATA_TYPE_UINT16;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)kvh, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)d * elem, (cuuint64_t)d * elem * kvh};
  cuuint32_t box[3] = {(cuuint32_t)(row_bytes / elem), 1u, (cuuint32_t)box_rows};
  if (heads > 0) {
    dims[1] = (cuuint64_t)rows;
    dims[2] = (cuuint64_t)kvh;
    strides[0] = (cuuint64_t)d * elem * kvh;
    strides[1] = (cuuint64_t)d * elem;
    box[1] = (cuuint32_t)box_rows;
    box[2] = (cuuint32_t)heads;
  }
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUtensorMap m;
  CUresult res = fn(&m, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                    row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (res != CUDA_SUCCESS) return false;
  int slot = g_map_used < kMapCache ? g_map_used++ : (g_map_next++ % kMapCache);
  g_keys[slot] = key;
  g_maps[slot] = m;
  *out = m;
  return true;
}

// 2-D view of a per-token scale array [rows][kvh] fp32: box {heads, box_rows},
// landing as [box_rows][heads].  Needs 16-byte rows and a 16-byte box width.
constexpr int kScaleMapTag = 99;   // MapKey dtype of scale maps

bool get_scale_map(const float* ptr, long long rows, int kvh, int heads, int box_rows,
                   CUtensorMap* out) {
  if ((kvh * 4) % 16 != 0 || (heads * 4) % 16 != 0 ||
      reinterpret_cast<uintptr_t>(ptr) % 16 != 0)
    return false;
  MapKey key{ptr, rows, kvh, 0, kScaleMapTag, box_rows, 0, heads};
  std::lock_guard<std::mutex> lk(g_map_mu);
  for (int i = 0; i < g_map_used; ++i)
    if (g_keys[i] == key) {
      *out = g_maps[i];
      return true;
    }
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kvh, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kvh * 4};
  cuuint32_t box[2] = {(cuuint32_t)heads, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  CUtensorMap m;
  CUresult res = fn(&m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(ptr), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (res != CUDA_SUCCESS) return false;
  int slot = g_map_used < kMapCache ? g_map_used++ : (g_map_next++ % kMapCache);
  g_keys[slot] = key;
  g_maps[slot] = m;
  *out = m;
  return true;
}

}  // namespace
}  // namespace mma

using namespace mma;

#ifdef FD_STAMPS
// the FP8-e4m3 kernels' stamps (the workloads the stamps are taken on)
cudaError_t read_split_stamps(unsigned long long* host, int n) { return read_stamps_e4m3(host, n); }

__global__ void empty_kernel(int) {}
struct BigParams { unsigned char b[1024]; };
__global__ void empty_kernel_big(const __grid_constant__ BigParams) {}

// An empty kernel of the given launch shape (launch-cost floor); smem < 0:
// 1 KB of parameters; threads < 0: cooperative launch.
cudaError_t launch_empty(int grid, int threads, int smem, cudaStream_t st) {
  cudaFuncSetAttribute(empty_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
  if (smem < 0) {
    BigParams bp;
    memset(&bp, 0, sizeof(bp));
    empty_kernel_big<<<grid, threads, 0, st>>>(bp);
    return cudaGetLastError();
  }
  if (threads < 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(-threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, empty_kernel, 0);
  }
  empty_kernel<<<grid, threads, smem, st>>>(0);
  return cudaGetLastError();
}
#endif

bool mma_supports(int group, int num_kv_heads, int head_dim, int q_dtype, int kv_dtype, int paged,
                  int page_size) {
  (void)q_dtype;
  (void)kv_dtype;
  if (head_dim != 64 && head_dim != 128) return false;
  if (group < 1 || group > 128 || num_kv_heads < 1) return false;
  if (paged && (page_size < 1 || page_size > 256)) return false;
  // (pages too small for a TMA box to start on a 1024-byte swizzle atom of
  // shared memory are gathered by the producer warp instead)
  if (!encode_fn()) return false;
  return true;
}

// A segment start costs the consumers a Q reload and the producer a row-data
// load, each a DRAM round trip under full load: about what streaming
// 128 KB takes per SM.  The plan charges it in tiles of this shape.
void mma_config(int group, int num_kv_heads, int head_dim, int kv_dtype, int sms, int* hc,
                int* tile, int* grid, int* seg_units) {
  const Shape s = make_shape(group, num_kv_heads, head_dim, kv_dtype, 0, false);
  *hc = s.hc;
  *tile = s.tile;
  *grid = sms;
  const int stage = 2 * s.kv_bytes;
  // when the warps of a head tile merge at every segment end (wph > 1), a
  // segment start also waits for that merge and for a refill of the
  // pipeline behind it: twice the cost
  *seg_units = (s.wph > 1 ? 2 : 1) * ((131072 + stage - 1) / stage);
}

bool fma_supports(int group, int num_kv_heads, int head_dim, int kv_dtype, int paged,
                  int page_size, bool token_scales) {
  if (kv_dtype != FD_E4M3 || head_dim != 128 || group < 1 || group > 8 || token_scales)
    return false;
  if (paged && (page_size < 1 || page_size > 256)) return false;
  Shape s;
  if (!fma_shape(group, num_kv_heads, paged ? page_size : 0, &s)) return false;
  return encode_fn() != nullptr;
}

cudaError_t launch_split_mma(const Params& p, cudaStream_t stream) {
  if (p.kv_rows >= (1ll << 31)) return cudaErrorInvalidValue;
  if (p.kernel == FD_KERNEL_FMA) {
    Shape sh;
    if (!fma_shape(p.group, p.num_kv_heads, p.block_table ? p.page_size : 0, &sh) ||
        sh.tile != p.tile || sh.hc != p.hc)
      return cudaErrorInvalidValue;
    Maps maps;
    std::memset(&maps, 0, sizeof(maps));
    if (sh.box_rows == sh.tile &&
        get_map(p.k, p.kv_rows, p.num_kv_heads, p.head_dim, p.kv_dtype, sh.box_rows, sh.row_bytes,
                sh.hc, &maps.k) &&
        get_map(p.v, p.kv_rows, p.num_kv_heads, p.head_dim, p.kv_dtype, sh.box_rows, sh.row_bytes,
                sh.hc, &maps.v)) {
      sh.heads_box = 1;
    } else if (!get_map(p.k, p.kv_rows, p.num_kv_heads, p.head_dim, p.kv_dtype, sh.box_rows,
                        sh.row_bytes, 0, &maps.k) ||
               !get_map(p.v, p.kv_rows, p.num_kv_heads, p.head_dim, p.kv_dtype, sh.box_rows,
                        sh.row_bytes, 0, &maps.v)) {
      return cudaErrorInvalidValue;
    }
    return launch_fma(p, sh, maps, stream);
  }
  if (p.kernel == FD_KERNEL_TC) {
    // one KV head per box, 64-token tiles (or the page's rows)
    const int box_rows = p.block_table && p.page_size < p.tile ? p.page_size : p.tile;
    CUtensorMap mk, mv;
    if (!get_map(p.k, p.kv_rows, p.num_kv_heads, p.head_dim, p.kv_dtype, box_rows, 128, 0, &mk) ||
        !get_map(p.v, p.kv_rows, p.num_kv_heads, p.head_dim, p.kv_dtype, box_rows, 128, 0, &mv))
      return cudaErrorInvalidValue;
    return launch_split_tc(p, mk, mv, stream);
  }
  Shape sh = make_shape(p.group, p.num_kv_heads, p.head_dim, p.kv_dtype,
                        p.block_table ? p.page_size : 0, p.scale_kind == FD_SCALE_TOKEN);
  if (sh.stages < 2 || sh.tile != p.tile || sh.hc != p.hc) return cudaErrorInvalidValue;
  Maps maps;
  std::memset(&maps, 0, sizeof(maps));
  CUtensorMap& mk = maps.k;
  CUtensorMap& mv = maps.v;
  // Prefer one box per tile covering all hc heads (fewer, larger TMA copies);
  // fall back to one box per head when the tile spans several pages or the
  // driver refuses the head-minor view.  Gathered rows need no tensor map.
  if (sh.gather) {
    // no maps
  } else if (sh.hc > 1 && sh.box_rows == sh.tile &&
      get_map(p.k, p.kv_rows, p.num_kv_heads, p.head_dim, p.kv_dtype, sh.box_rows, sh.row_bytes,
              sh.hc, &mk) &&
      get_map(p.v, p.kv_rows, p.num_kv_heads, p.head_dim, p.kv_dtype, sh.box_rows, sh.row_bytes,
              sh.hc, &mv)) {
    sh.heads_box = 1;
  } else if (!get_map(p.k, p.kv_rows, p.num_kv_heads, p.head_dim, p.kv_dtype, sh.box_rows,
                      sh.row_bytes, 0, &mk) ||
             !get_map(p.v, p.kv_rows, p.num_kv_heads, p.head_dim, p.kv_dtype, sh.box_rows,
                      sh.row_bytes, 0, &mv)) {
    return cudaErrorInvalidValue;
  }
  if (p.scale_kind == FD_SCALE_TOKEN && !sh.gather &&
      get_scale_map(p.k_scales, p.kv_rows, p.num_kv_heads, sh.hc, sh.box_rows, &maps.ks) &&
      get_scale_map(p.v_scales, p.kv_rows, p.num_kv_heads, sh.hc, sh.box_rows, &maps.vs))
    sh.scale_tma = 1;
  if (p.kv_dtype == FD_E4M3) return launch_e4m3(p, sh, maps, stream);
  if (p.kv_dtype == FD_I8) return launch_i8(p, sh, maps, stream);
  return launch_16bit(p, sh, maps, stream);
}

}  // namespace fd
