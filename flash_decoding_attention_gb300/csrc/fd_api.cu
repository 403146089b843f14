// fd_api.cu -- the C ABI: argument validation, kernel choice, workspace
// sizing, launches and the test/debug hooks declared in fd_attention.h.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "fd_common.cuh"

// Optional NVTX ranges around the host-side launch of each phase (append,
// split, combine), for timeline tools; built with -DFD_NVTX (FD_NVTX=1 in
// the build environment), absent otherwise.
#ifdef FD_NVTX
#include <nvtx3/nvToolsExt.h>
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};
#define FD_RANGE(name) NvtxRange fd_nvtx_range_(name)
#else
#define FD_RANGE(name) ((void)0)
#endif

namespace fd {

// Tensor-core kernel entry points (fd_split_mma.cu).
bool mma_supports(int group, int num_kv_heads, int head_dim, int q_dtype, int kv_dtype,
                  int paged, int page_size);
void mma_config(int group, int num_kv_heads, int head_dim, int kv_dtype, int sms, int* hc,
                int* tile, int* grid, int* seg_units);
// CUDA-core form of the mma.sync kernel (fd_split_fma.cu, fd_split_mma.cu)
bool fma_supports(int group, int num_kv_heads, int head_dim, int kv_dtype, int paged,
                  int page_size, bool token_scales);
// tcgen05 kernel (fd_split_tc.cu)
bool tc_supports(int group, int head_dim, int q_dtype, int kv_dtype, int paged, int page_size,
                 bool token_scales);
void tc_config(int group, int sms, int* hc, int* tile, int* grid, int* seg_units);

namespace {

std::atomic<int> g_kernel{FD_KERNEL_AUTO};
// fd_debug_set_wait_limit: bound of the split kernel's pipeline waits (ns,
// 0 = one second) and the switch that starves its consumers
constexpr unsigned long long kDefaultWaitNs = 1000000000ull;
std::atomic<long long> g_wait_ns{0};
std::atomic<int> g_starve{0};
thread_local cudaEvent_t t_ev_before = nullptr;
thread_local cudaEvent_t t_ev_after = nullptr;

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
int g_dev_sms[kMaxDevices] = {0};

int current_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_dev_sms[dev] == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_dev_sms[dev] = sms;
  }
  return g_dev_sms[dev];
}

struct Config {
  int kernel;   // FD_KERNEL_SIMT or FD_KERNEL_MMA
  int hc, hg, hq, tile, grid;
  int seg_units;   // plan cost of a segment start, in tiles
};

constexpr int kSimtTile = 32;

bool dtypes_ok(int q_dtype, int kv_dtype) {
  if (q_dtype != FD_F16 && q_dtype != FD_BF16) return false;
  if (kv_dtype == FD_E4M3 || kv_dtype == FD_I8) return true;
  return kv_dtype == q_dtype;
}

// Chooses the split kernel and its plan shape; false if unsupported.
bool choose(int pref, int num_q_heads, int num_kv_heads, int head_dim, int q_dtype, int kv_dtype,
            int paged, int page_size, int sms, Config* c, bool token_scales = false) {
  if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return false;
  const int group = num_q_heads / num_kv_heads;
  if (!dtypes_ok(q_dtype, kv_dtype) || (head_dim != 64 && head_dim != 128)) return false;
  const bool tc_ok = tc_supports(group, head_dim, q_dtype, kv_dtype, paged, page_size, token_scales);
  // Automatic choice of the tcgen05 kernel where it measured faster than the
  // mma.sync one: a single KV head with at least 64 query rows (the
  // long-context MQA workload with 4 and 8 query tokens).  With several KV
  // heads the mma.sync kernel carries two to eight of them per stream and
  // stays ahead.
  const bool tc_auto = tc_ok && num_kv_heads == 1 && group >= 64;
  if (pref == FD_KERNEL_TC || (pref == FD_KERNEL_AUTO && tc_auto)) {
    if (!tc_ok) return false;
    c->kernel = FD_KERNEL_TC;
    tc_config(group, sms, &c->hc, &c->tile, &c->grid, &c->seg_units);
    c->hg = num_kv_heads;
    c->hq = group;
    return true;
  }
  if (pref == FD_KERNEL_FMA) {
    // the mma.sync kernel's plan shape, CUDA-core arithmetic
    if (!fma_supports(group, num_kv_heads, head_dim, kv_dtype, paged, page_size, token_scales))
      return false;
    c->kernel = FD_KERNEL_FMA;
    mma_config(group, num_kv_heads, head_dim, kv_dtype, sms, &c->hc, &c->tile, &c->grid,
               &c->seg_units);
    c->hg = num_kv_heads / c->hc;
    c->hq = c->hc * group;
    return true;
  }
  const bool mma_ok = mma_supports(group, num_kv_heads, head_dim, q_dtype, kv_dtype, paged, page_size);
  if (pref == FD_KERNEL_MMA || (pref == FD_KERNEL_AUTO && mma_ok)) {
    if (!mma_ok) return false;
    c->kernel = FD_KERNEL_MMA;
    mma_config(group, num_kv_heads, head_dim, kv_dtype, sms, &c->hc, &c->tile, &c->grid,
               &c->seg_units);
    c->hg = num_kv_heads / c->hc;
    c->hq = c->hc * group;
    return true;
  }
  if (!simt_supports(group, head_dim)) return false;
  c->kernel = FD_KERNEL_SIMT;
  c->hc = 1;
  c->hq = simt_heads_per_stream(group);
  c->hg = num_q_heads / c->hq;
  c->tile = kSimtTile;
  c->grid = sms * simt_ctas_per_sm();
  c->seg_units = 0;
  return true;
}

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

int log2i(int x) {
  int r = 0;
  while ((1 << r) < x) ++r;
  return r;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The new token's rows and where they go (KV append).
struct AppendArgs {
  const void* k_new;
  const void* v_new;
  const int32_t* positions;
  void* k_cache;
  void* v_cache;
  float* k_scales;   // written with per-token scales
  float* v_scales;
};

// Checks of the append's own arguments; the cache, layout and scale-kind
// arguments are checked by the caller.  8-bit codes divide by the scales.
fd_status check_append(const AppendArgs& a, int kv_dtype, float k_scale, float v_scale) {
  if (!a.k_new || !a.v_new || !a.positions || !a.k_cache || !a.v_cache) return FD_ERR_INVALID_ARG;
  if (!aligned(a.k_new, 16) || !aligned(a.v_new, 16) || !aligned(a.positions, 4))
    return FD_ERR_INVALID_ARG;
  if (kv_elem_bytes(kv_dtype) == 1 && !(k_scale > 0.f && v_scale > 0.f)) return FD_ERR_INVALID_ARG;
  return FD_OK;
}

void set_append(Params& p, const AppendArgs& a, int n_new, float k_scale, float v_scale) {
  p.n_new = n_new;
  p.k_new = a.k_new;
  p.v_new = a.v_new;
  p.positions = a.positions;
  p.k_dst = a.k_cache;
  p.v_dst = a.v_cache;
  p.k_scales_dst = p.scale_kind == FD_SCALE_TOKEN ? a.k_scales : nullptr;
  p.v_scales_dst = p.scale_kind == FD_SCALE_TOKEN ? a.v_scales : nullptr;
  p.k_scale_raw = k_scale;
  p.v_scale_raw = v_scale;
}

// Gather of the stored K or V slice of every token, with the kernels'
// addressing (test hook).  CTA b copies sequence b; its destination offset
// is the sum of the earlier sequences' lengths.
__global__ void gather_kernel(const Params p, uint8_t* dst, int row_bytes) {
  const int b = blockIdx.x;
  long long off = 0;
  for (int i = 0; i < b; ++i) {
    int t = __ldg(p.seq_len + i);
    off += t > 0 ? t : 0;
  }
  int T = __ldg(p.seq_len + b);
  if (T < 0) T = 0;
  const uint8_t* src = static_cast<const uint8_t*>(p.k);
  for (int t = 0; t < T; ++t) {
    const long long row = cache_row(p, b, t);
    uint8_t* d = dst + (off + t) * row_bytes;
    for (int x = threadIdx.x; x < row_bytes; x += blockDim.x)
      d[x] = row >= 0 ? src[row * row_bytes + x] : 0;
  }
}

// The segments every CTA of the split kernel takes (test hook): the plan and
// the segment walk of the split kernels, run by a grid of the same size.
// Row c of dst: the number of segments, then per segment (stream, t_begin,
// t_end, complete, slot), at most `cap` of them.
__global__ void plan_segments_kernel(const Params p, int32_t* dst, int cap) {
  __shared__ long long red[35];
  const PlanResult plan = compute_plan(p, red, blockDim.x, 0);
  if (threadIdx.x != 0) return;
  SegmentIter it;
  it.init(p, plan);
  Segment seg;
  int32_t* d = dst + (size_t)blockIdx.x * (1 + 5 * (size_t)cap);
  int k = 0;
  while (it.next(p, seg)) {
    if (k < cap) {
      int32_t* e = d + 1 + 5 * k;
      e[0] = seg.s;
      e[1] = seg.t_begin;
      e[2] = seg.t_end;
      e[3] = seg.complete ? 1 : 0;
      e[4] = seg.slot;
    }
    ++k;
  }
  d[0] = k;
}

}  // namespace
}  // namespace fd

namespace fd {
// Host-side checks of a decode call's arguments, in the order every entry
// point applies them; `workspace` is only checked for presence and alignment
// (the no-allocation entry point passes its own array).
fd_status check_decode_args(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* kv_start_idx, const int32_t* block_table,
                            int block_table_stride, const int32_t* seq_len, int64_t kv_rows,
                            int batch, int num_q_heads, int num_kv_heads, int head_dim,
                            int page_size, float softmax_scale, float k_scale, float v_scale,
                            fd_scale_kind scale_kind, const float* k_scales,
                            const float* v_scales, fd_dtype q_dtype, fd_dtype kv_dtype,
                            const void* out, const float* lse, const void* workspace, int q_len) {
  // q_len query tokens per sequence run as q_len virtual query heads per head
  if (q_len < 1 || q_len > 16) return FD_ERR_INVALID_ARG;
  if (num_q_heads > 0 && num_kv_heads > 0 && num_q_heads % num_kv_heads == 0 &&
      (num_q_heads / num_kv_heads) * q_len > 128)
    return FD_ERR_UNSUPPORTED;
  if (scale_kind != FD_SCALE_TENSOR && scale_kind != FD_SCALE_HEAD &&
      scale_kind != FD_SCALE_TOKEN)
    return FD_ERR_INVALID_ARG;
  if (scale_kind != FD_SCALE_TENSOR) {
    if (!k_scales || !v_scales || !aligned(k_scales, 4) || !aligned(v_scales, 4))
      return FD_ERR_INVALID_ARG;
    if (kv_elem_bytes(kv_dtype) != 1) return FD_ERR_UNSUPPORTED;
  }
  if (!q || !k_cache || !v_cache || !seq_len || !out || !workspace) return FD_ERR_INVALID_ARG;
  if ((kv_start_idx == nullptr) == (block_table == nullptr)) return FD_ERR_INVALID_ARG;
  if (batch <= 0 || batch > (1 << 24)) return FD_ERR_INVALID_ARG;
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
    return FD_ERR_INVALID_ARG;
  if (num_q_heads / num_kv_heads > 128 || num_q_heads > 4096) return FD_ERR_UNSUPPORTED;
  if (kv_rows <= 0 || kv_rows > (int64_t(1) << 40)) return FD_ERR_INVALID_ARG;
  const int paged = block_table != nullptr;
  if (paged) {
    if (!is_pow2(page_size) || page_size > 256) return FD_ERR_UNSUPPORTED;
    if (block_table_stride <= 0 || kv_rows % page_size != 0) return FD_ERR_INVALID_ARG;
  }
  if (!std::isfinite(softmax_scale) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
    return FD_ERR_INVALID_ARG;
  if (q_dtype != FD_F16 && q_dtype != FD_BF16) return FD_ERR_INVALID_ARG;
  if (kv_dtype != FD_F16 && kv_dtype != FD_BF16 && kv_dtype != FD_E4M3 && kv_dtype != FD_I8)
    return FD_ERR_INVALID_ARG;
  if (!dtypes_ok(q_dtype, kv_dtype)) return FD_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return FD_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(workspace, 256) || (lse && !aligned(lse, 4)))
    return FD_ERR_INVALID_ARG;
  return FD_OK;
}
}  // namespace fd

using namespace fd;

extern "C" {

const char* fd_status_string(fd_status status) {
  switch (status) {
    case FD_OK: return "ok";
    case FD_ERR_INVALID_ARG: return "invalid argument";
    case FD_ERR_UNSUPPORTED: return "unsupported configuration";
    case FD_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case FD_ERR_CUDA: return "CUDA error";
    case FD_ERR_DEVICE_BOUNDS: return "device: cache row or page id out of range";
    case FD_ERR_DEVICE_TIMEOUT: return "device: bounded wait expired";
  }
  return "unknown status";
}

fd_status fd_set_kernel(fd_kernel kernel) {
  if (kernel != FD_KERNEL_AUTO && kernel != FD_KERNEL_SIMT && kernel != FD_KERNEL_MMA &&
      kernel != FD_KERNEL_TC && kernel != FD_KERNEL_FMA)
    return FD_ERR_INVALID_ARG;
  g_kernel.store(kernel);
  return FD_OK;
}

int fd_selected_kernel(int num_q_heads, int num_kv_heads, int head_dim, fd_dtype q_dtype,
                       fd_dtype kv_dtype, int paged, int page_size) {
  return fd_selected_kernel_scaled(num_q_heads, num_kv_heads, head_dim, q_dtype, kv_dtype, paged,
                                   page_size, FD_SCALE_TENSOR);
}

int fd_selected_kernel_scaled(int num_q_heads, int num_kv_heads, int head_dim, fd_dtype q_dtype,
                              fd_dtype kv_dtype, int paged, int page_size,
                              fd_scale_kind scale_kind) {
  Config c;
  const int sms = current_sms();
  if (sms <= 0) return -1;
  if (!choose(g_kernel.load(), num_q_heads, num_kv_heads, head_dim, q_dtype, kv_dtype, paged,
              page_size, sms, &c, scale_kind == FD_SCALE_TOKEN))
    return -1;
  return c.kernel;
}

fd_status fd_set_split_events(fd_event_t before, fd_event_t after) {
  if ((before == nullptr) != (after == nullptr)) return FD_ERR_INVALID_ARG;
  t_ev_before = reinterpret_cast<cudaEvent_t>(before);
  t_ev_after = reinterpret_cast<cudaEvent_t>(after);
  return FD_OK;
}

size_t fd_workspace_bytes(int batch, int num_q_heads, int num_kv_heads, int head_dim) {
  if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads)
    return 0;
  if (head_dim != 64 && head_dim != 128) return 0;
  const int sms = current_sms();
  if (sms <= 0) return 0;
  size_t need = 0;
  // Largest layout over every kernel and dtype choice for these sizes.
  const int dts[6][2] = {{FD_F16, FD_F16}, {FD_BF16, FD_BF16}, {FD_F16, FD_E4M3},
                         {FD_BF16, FD_E4M3}, {FD_F16, FD_I8}, {FD_BF16, FD_I8}};
  for (int pref : {FD_KERNEL_SIMT, FD_KERNEL_MMA, FD_KERNEL_TC, FD_KERNEL_FMA}) {
    for (auto& dt : dts) {
      for (int paged : {0, 1}) {
        Config c;
        if (!choose(pref, num_q_heads, num_kv_heads, head_dim, dt[0], dt[1], paged, 64, sms, &c))
          continue;
        WsLayout L = ws_layout(batch * c.hg, c.grid, c.hq, head_dim);
        if (L.total > need) need = L.total;
      }
    }
  }
  return need;
}

fd_status fd_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* kv_start_idx, const int32_t* block_table,
                              int block_table_stride, const int32_t* seq_len, int64_t kv_rows,
                              int batch, int num_q_heads, int num_kv_heads, int head_dim,
                              int page_size, float softmax_scale, float k_scale, float v_scale,
                              fd_dtype q_dtype, fd_dtype kv_dtype, void* out, float* lse,
                              void* workspace, size_t workspace_bytes, fd_stream_t stream) {
  return fd_decode_attention_scaled(q, k_cache, v_cache, kv_start_idx, block_table,
                                    block_table_stride, seq_len, kv_rows, batch, num_q_heads,
                                    num_kv_heads, head_dim, page_size, softmax_scale, k_scale,
                                    v_scale, FD_SCALE_TENSOR, nullptr, nullptr, q_dtype, kv_dtype,
                                    out, lse, workspace, workspace_bytes, stream);
}


// The attention of one decode step, optionally preceded by the KV append of
// the step's new token (then the split kernel runs as a programmatic
// dependent of the append and waits for it before reading the caches).
static fd_status decode_impl(const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* kv_start_idx, const int32_t* block_table,
                             int block_table_stride, const int32_t* seq_len, int64_t kv_rows,
                             int batch, int num_q_heads, int num_kv_heads, int head_dim,
                             int page_size, float softmax_scale, float k_scale, float v_scale,
                             fd_scale_kind scale_kind, const float* k_scales,
                             const float* v_scales, fd_dtype q_dtype, fd_dtype kv_dtype, void* out,
                             float* lse, void* workspace, size_t workspace_bytes,
                             fd_stream_t stream, const AppendArgs* app, int q_len = 1) {
  const fd_status chk = check_decode_args(
      q, k_cache, v_cache, kv_start_idx, block_table, block_table_stride, seq_len, kv_rows, batch,
      num_q_heads, num_kv_heads, head_dim, page_size, softmax_scale, k_scale, v_scale, scale_kind,
      k_scales, v_scales, q_dtype, kv_dtype, out, lse, workspace, q_len);
  if (chk != FD_OK) return chk;
  const int virt_heads = num_q_heads * q_len;
  const int paged = block_table != nullptr;
  if (app) {
    const fd_status st = check_append(*app, kv_dtype, k_scale, v_scale);
    if (st != FD_OK) return st;
  }

  const int sms = current_sms();
  if (sms <= 0) return FD_ERR_CUDA;
  Config c;
  if (!choose(g_kernel.load(), virt_heads, num_kv_heads, head_dim, q_dtype, kv_dtype, paged,
              page_size, sms, &c, scale_kind == FD_SCALE_TOKEN))
    return FD_ERR_UNSUPPORTED;
  const WsLayout L = ws_layout(batch * c.hg, c.grid, c.hq, head_dim);
  if (workspace_bytes < L.total) return FD_ERR_WORKSPACE_TOO_SMALL;

  Params p;
  std::memset(&p, 0, sizeof(p));
  p.q = q;
  p.k = k_cache;
  p.v = v_cache;
  p.kv_start = kv_start_idx;
  p.block_table = block_table;
  p.seq_len = seq_len;
  p.out = out;
  p.lse = lse;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.ws = reinterpret_cast<WsHeader*>(ws);
  p.prefix = reinterpret_cast<int32_t*>(ws + L.prefix_off);
  p.part_ml = reinterpret_cast<float2*>(ws + L.ml_off);
  p.part_acc = reinterpret_cast<float*>(ws + L.acc_off);
  p.kv_rows = kv_rows;
  p.bt_stride = paged ? block_table_stride : 0;
  p.batch = batch;
  p.num_q_heads = virt_heads;
  p.num_kv_heads = num_kv_heads;
  p.head_dim = head_dim;
  p.page_size = paged ? page_size : 1;
  p.page_shift = paged ? log2i(page_size) : 0;
  p.group = virt_heads / num_kv_heads;
  p.q_len = q_len;
  p.hc = c.hc;
  p.hg = c.hg;
  p.hq = c.hq;
  p.tile = c.tile;
  p.seg_units = c.seg_units;
  p.grid = c.grid;
  p.kernel = c.kernel;
  p.q_dtype = q_dtype;
  p.kv_dtype = kv_dtype;
  p.score_scale = softmax_scale * k_scale * kLog2e;
  p.v_scale = v_scale;
  p.scale_kind = scale_kind;
  p.k_scales = scale_kind == FD_SCALE_TENSOR ? nullptr : k_scales;
  p.v_scales = scale_kind == FD_SCALE_TENSOR ? nullptr : v_scales;
  const long long wns = g_wait_ns.load();
  p.wait_ns = wns > 0 ? (unsigned long long)wns : kDefaultWaitNs;
  p.starve = g_starve.load();

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  FD_RANGE("fd_decode_attention");
  if (app) {
    FD_RANGE("fd.append");
    set_append(p, *app, q_len, k_scale, v_scale);
    if (launch_append(p, st) != cudaSuccess) return FD_ERR_CUDA;
    p.pdl = 1;
  }
  const bool timed = t_ev_before != nullptr;
  if (timed && cudaEventRecord(t_ev_before, st) != cudaSuccess) return FD_ERR_CUDA;
  {
    FD_RANGE("fd.split");
    cudaError_t e = c.kernel == FD_KERNEL_SIMT ? launch_split_simt(p, st) : launch_split_mma(p, st);
    if (e != cudaSuccess) return FD_ERR_CUDA;
  }
  if (timed && cudaEventRecord(t_ev_after, st) != cudaSuccess) return FD_ERR_CUDA;
  {
    FD_RANGE("fd.combine");
    if (launch_combine(p, st) != cudaSuccess) return FD_ERR_CUDA;
  }
  return FD_OK;
}

fd_status fd_decode_attention_scaled(const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* kv_start_idx, const int32_t* block_table,
                                     int block_table_stride, const int32_t* seq_len,
                                     int64_t kv_rows, int batch, int num_q_heads,
                                     int num_kv_heads, int head_dim, int page_size,
                                     float softmax_scale, float k_scale, float v_scale,
                                     fd_scale_kind scale_kind, const float* k_scales,
                                     const float* v_scales, fd_dtype q_dtype, fd_dtype kv_dtype,
                                     void* out, float* lse, void* workspace,
                                     size_t workspace_bytes, fd_stream_t stream) {
  return decode_impl(q, k_cache, v_cache, kv_start_idx, block_table, block_table_stride, seq_len,
                     kv_rows, batch, num_q_heads, num_kv_heads, head_dim, page_size,
                     softmax_scale, k_scale, v_scale, scale_kind, k_scales, v_scales, q_dtype,
                     kv_dtype, out, lse, workspace, workspace_bytes, stream, nullptr);
}

fd_status fd_decode_attention_multi(const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* kv_start_idx, const int32_t* block_table,
                                    int block_table_stride, const int32_t* seq_len,
                                    int64_t kv_rows, int batch, int q_len, int num_q_heads,
                                    int num_kv_heads, int head_dim, int page_size,
                                    float softmax_scale, float k_scale, float v_scale,
                                    fd_scale_kind scale_kind, const float* k_scales,
                                    const float* v_scales, fd_dtype q_dtype, fd_dtype kv_dtype,
                                    void* out, float* lse, void* workspace,
                                    size_t workspace_bytes, fd_stream_t stream) {
  return decode_impl(q, k_cache, v_cache, kv_start_idx, block_table, block_table_stride, seq_len,
                     kv_rows, batch, num_q_heads, num_kv_heads, head_dim, page_size,
                     softmax_scale, k_scale, v_scale, scale_kind, k_scales, v_scales, q_dtype,
                     kv_dtype, out, lse, workspace, workspace_bytes, stream, nullptr, q_len);
}

fd_status fd_decode_attention_append(const void* q, const void* k_new, const void* v_new,
                                     void* k_cache, void* v_cache, const int32_t* kv_start_idx,
                                     const int32_t* block_table, int block_table_stride,
                                     const int32_t* positions, const int32_t* seq_len,
                                     int64_t kv_rows, int batch, int q_len, int num_q_heads,
                                     int num_kv_heads, int head_dim, int page_size,
                                     float softmax_scale, float k_scale, float v_scale,
                                     fd_scale_kind scale_kind, float* k_scales, float* v_scales,
                                     fd_dtype q_dtype, fd_dtype kv_dtype, void* out, float* lse,
                                     void* workspace, size_t workspace_bytes, fd_stream_t stream) {
  const AppendArgs app{k_new, v_new, positions, k_cache, v_cache, k_scales, v_scales};
  return decode_impl(q, k_cache, v_cache, kv_start_idx, block_table, block_table_stride, seq_len,
                     kv_rows, batch, num_q_heads, num_kv_heads, head_dim, page_size,
                     softmax_scale, k_scale, v_scale, scale_kind, k_scales, v_scales, q_dtype,
                     kv_dtype, out, lse, workspace, workspace_bytes, stream, &app, q_len);
}

fd_status fd_append_kv(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                       const int32_t* kv_start_idx, const int32_t* block_table,
                       int block_table_stride, const int32_t* positions, int64_t kv_rows,
                       int batch, int n_new, int num_kv_heads, int head_dim, int page_size,
                       float k_scale, float v_scale, fd_scale_kind scale_kind, float* k_scales,
                       float* v_scales,
                       fd_dtype new_dtype, fd_dtype kv_dtype, void* workspace,
                       size_t workspace_bytes, fd_stream_t stream) {
  if (scale_kind != FD_SCALE_TENSOR && scale_kind != FD_SCALE_HEAD &&
      scale_kind != FD_SCALE_TOKEN)
    return FD_ERR_INVALID_ARG;
  if (scale_kind != FD_SCALE_TENSOR) {
    if (!k_scales || !v_scales || !aligned(k_scales, 4) || !aligned(v_scales, 4))
      return FD_ERR_INVALID_ARG;
    if (kv_elem_bytes(kv_dtype) != 1) return FD_ERR_UNSUPPORTED;
  }
  const AppendArgs app{k_new, v_new, positions, k_cache, v_cache, k_scales, v_scales};
  if (!workspace || !aligned(workspace, 256)) return FD_ERR_INVALID_ARG;
  if ((kv_start_idx == nullptr) == (block_table == nullptr)) return FD_ERR_INVALID_ARG;
  if (batch <= 0 || batch > (1 << 24) || num_kv_heads <= 0 || num_kv_heads > 4096)
    return FD_ERR_INVALID_ARG;
  if (n_new < 1 || n_new > 16) return FD_ERR_INVALID_ARG;
  if (kv_rows <= 0 || kv_rows > (int64_t(1) << 40)) return FD_ERR_INVALID_ARG;
  const int paged = block_table != nullptr;
  if (paged) {
    if (!is_pow2(page_size) || page_size > 256) return FD_ERR_UNSUPPORTED;
    if (block_table_stride <= 0 || kv_rows % page_size != 0) return FD_ERR_INVALID_ARG;
  }
  if (!std::isfinite(k_scale) || !std::isfinite(v_scale)) return FD_ERR_INVALID_ARG;
  if (new_dtype != FD_F16 && new_dtype != FD_BF16) return FD_ERR_INVALID_ARG;
  if (kv_dtype != FD_F16 && kv_dtype != FD_BF16 && kv_dtype != FD_E4M3 && kv_dtype != FD_I8)
    return FD_ERR_INVALID_ARG;
  if (!dtypes_ok(new_dtype, kv_dtype)) return FD_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return FD_ERR_UNSUPPORTED;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16)) return FD_ERR_INVALID_ARG;
  const fd_status cs = check_append(app, kv_dtype, k_scale, v_scale);
  if (cs != FD_OK) return cs;
  if (workspace_bytes < sizeof(WsHeader)) return FD_ERR_WORKSPACE_TOO_SMALL;

  Params p;
  std::memset(&p, 0, sizeof(p));
  p.k = k_cache;
  p.v = v_cache;
  p.kv_start = kv_start_idx;
  p.block_table = block_table;
  p.bt_stride = paged ? block_table_stride : 0;
  p.ws = static_cast<WsHeader*>(workspace);
  p.kv_rows = kv_rows;
  p.batch = batch;
  p.num_kv_heads = num_kv_heads;
  p.head_dim = head_dim;
  p.page_size = paged ? page_size : 1;
  p.page_shift = paged ? log2i(page_size) : 0;
  p.q_dtype = new_dtype;
  p.kv_dtype = kv_dtype;
  p.scale_kind = scale_kind;
  p.k_scales = scale_kind == FD_SCALE_TENSOR ? nullptr : k_scales;
  p.v_scales = scale_kind == FD_SCALE_TENSOR ? nullptr : v_scales;
  set_append(p, app, n_new, k_scale, v_scale);
  return launch_append(p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? FD_OK
                                                                                : FD_ERR_CUDA;
}

fd_status fd_check_device_error(void* workspace, fd_stream_t stream, int64_t* info) {
  if (!workspace) return FD_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  WsHeader h;
  if (cudaMemcpyAsync(&h, workspace, 16, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return FD_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return FD_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, 16, st) != cudaSuccess) return FD_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return FD_ERR_CUDA;
  if (info) *info = h.error_info ? (int64_t)(h.error_info - 1) : 0;
  if (h.error_bits & (kErrTimeout | kErrDrain)) return FD_ERR_DEVICE_TIMEOUT;
  if (h.error_bits & (kErrBounds | kErrPlan)) return FD_ERR_DEVICE_BOUNDS;
  return FD_OK;
}

fd_status fd_debug_read_plan(const void* workspace, fd_stream_t stream, int32_t* plan,
                             int capacity) {
  if (!workspace || !plan || capacity < 8) return FD_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  WsHeader h;
  if (cudaMemcpyAsync(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return FD_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return FD_ERR_CUDA;
  std::memcpy(plan, h.plan, sizeof(h.plan));
  const int S = h.plan[0];
  if (S < 0 || 8 + S + 1 > capacity) return FD_ERR_INVALID_ARG;
  if (cudaMemcpyAsync(plan + 8, static_cast<const uint8_t*>(workspace) + sizeof(WsHeader),
                      sizeof(int32_t) * (S + 1), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return FD_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return FD_ERR_CUDA;
  return FD_OK;
}

fd_status fd_debug_set_wait_limit(int64_t wait_ns, int starve_first_stage) {
  if (wait_ns < 0 || wait_ns > (int64_t)10000000000LL) return FD_ERR_INVALID_ARG;
  g_wait_ns.store((long long)wait_ns);
  g_starve.store(starve_first_stage ? 1 : 0);
  return FD_OK;
}

fd_status fd_debug_plan_segments(const int32_t* seq_len, const int32_t* kv_start_idx, int batch,
                                 int q_len, int num_q_heads,
                                 int num_kv_heads, int head_dim, int paged, int page_size,
                                 fd_dtype q_dtype, fd_dtype kv_dtype, int32_t* dst,
                                 int64_t dst_len, int capacity_per_cta, int* grid_out,
                                 void* workspace,
                                 size_t workspace_bytes, fd_stream_t stream) {
  if (!seq_len || !dst || !workspace || !grid_out || capacity_per_cta < 1 || batch <= 0 ||
      q_len < 1 || q_len > 16 || !aligned(workspace, 256))
    return FD_ERR_INVALID_ARG;
  if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0)
    return FD_ERR_INVALID_ARG;
  const int sms = current_sms();
  if (sms <= 0) return FD_ERR_CUDA;
  Config c;
  if (!choose(g_kernel.load(), num_q_heads * q_len, num_kv_heads, head_dim, q_dtype, kv_dtype,
              paged ? 1 : 0, paged ? page_size : 0, sms, &c))
    return FD_ERR_UNSUPPORTED;
  const WsLayout L = ws_layout(batch * c.hg, c.grid, c.hq, head_dim);
  if (workspace_bytes < L.total) return FD_ERR_WORKSPACE_TOO_SMALL;
  *grid_out = c.grid;
  if (dst_len < (int64_t)c.grid * (1 + 5 * (int64_t)capacity_per_cta)) return FD_ERR_INVALID_ARG;
  Params p;
  std::memset(&p, 0, sizeof(p));
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.ws = reinterpret_cast<WsHeader*>(ws);
  p.prefix = reinterpret_cast<int32_t*>(ws + L.prefix_off);
  p.seq_len = seq_len;
  p.kv_start = kv_start_idx;
  p.batch = batch;
  p.hg = c.hg;
  p.hq = c.hq;
  p.tile = c.tile;
  p.seg_units = c.seg_units;
  p.grid = c.grid;
  p.kernel = c.kernel;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  plan_segments_kernel<<<c.grid, 256, 0, st>>>(p, dst, capacity_per_cta);
  return cudaGetLastError() == cudaSuccess ? FD_OK : FD_ERR_CUDA;
}

fd_status fd_debug_gather_kv(const void* cache, const int32_t* kv_start_idx,
                             const int32_t* block_table, int block_table_stride,
                             const int32_t* seq_len, int64_t kv_rows, int batch,
                             int num_kv_heads, int head_dim, int page_size, fd_dtype kv_dtype,
                             void* dst, void* workspace, fd_stream_t stream) {
  if (!cache || !seq_len || !dst || !workspace || batch <= 0 || num_kv_heads <= 0 ||
      head_dim <= 0 || kv_rows <= 0)
    return FD_ERR_INVALID_ARG;
  if ((kv_start_idx == nullptr) == (block_table == nullptr)) return FD_ERR_INVALID_ARG;
  if (block_table && (!is_pow2(page_size) || page_size > 256 || block_table_stride <= 0))
    return FD_ERR_INVALID_ARG;
  if (kv_dtype != FD_F16 && kv_dtype != FD_BF16 && kv_dtype != FD_E4M3 && kv_dtype != FD_I8)
    return FD_ERR_INVALID_ARG;
  Params p;
  std::memset(&p, 0, sizeof(p));
  p.k = cache;
  p.kv_start = kv_start_idx;
  p.block_table = block_table;
  p.bt_stride = block_table ? block_table_stride : 0;
  p.seq_len = seq_len;
  p.kv_rows = kv_rows;
  p.page_size = block_table ? page_size : 1;
  p.page_shift = block_table ? log2i(page_size) : 0;
  p.ws = static_cast<WsHeader*>(workspace);
  const int row_bytes = num_kv_heads * head_dim * kv_elem_bytes(kv_dtype);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  gather_kernel<<<batch, 128, 0, st>>>(p, static_cast<uint8_t*>(dst), row_bytes);
  return cudaGetLastError() == cudaSuccess ? FD_OK : FD_ERR_CUDA;
}

#ifdef FD_STAMPS
// Instrumented builds only (not in the public header): copies the phase
// stamps of the last split (which = 0) or combine (which = 1) launch,
// 8 per CTA, into host memory; synchronises the device.
int fd_debug_empty_launch(int grid, int threads, int smem, fd_stream_t stream) {
  return launch_empty(grid, threads, smem, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FD_OK
             : FD_ERR_CUDA;
}

int fd_debug_read_stamps(int which, unsigned long long* host, int n) {
  if (!host || n <= 0) return FD_ERR_INVALID_ARG;
  const cudaError_t e = which == 0   ? read_split_stamps(host, n)
                        : which == 1 ? read_combine_stamps(host, n)
                                     : read_tc_stamps(host, n);
  return e == cudaSuccess ? FD_OK : FD_ERR_CUDA;
}
#endif

}  // extern "C"
