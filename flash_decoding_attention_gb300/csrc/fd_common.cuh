// fd_common.cuh -- pieces shared by the split and combine kernels: workspace
// layout, the device-side split plan, cache addressing, device error flags.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include <atomic>

#include "fd_attention.h"

namespace fd {

// ---------------------------------------------------------------------------
// Device error word (sticky, in the workspace header)
// ---------------------------------------------------------------------------
enum : uint32_t {
  kErrBounds = 1u,   // cache row or page id outside the cache
  kErrTimeout = 2u,  // a bounded wait expired
  kErrPlan = 4u,     // plan does not fit the workspace (more tiles than int32)
  kErrDrain = 8u,    // copies still in flight when a CTA gave up waiting for them
};

struct WsHeader {
  uint32_t error_bits;
  uint32_t pad0;
  unsigned long long error_info;   // first offending value (+1, so 0 = none)
  int32_t plan[8];                 // see fd_debug_read_plan
  uint8_t pad[256 - 16 - 32];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Bytes of one K/V element: 1 for the 8-bit codes (e4m3, int8), else 2.
__host__ __device__ constexpr int kv_elem_bytes(int kv_dtype) {
  return kv_dtype == FD_E4M3 || kv_dtype == FD_I8 ? 1 : 2;
}

// Workspace = header | prefix int32[num_streams + 1] | ml float2[2*grid][hq] |
// acc float[2*grid][hq][head_dim].  Every partial slot belongs to one CTA:
// slot 2c holds the CTA's first segment when that segment continues a stream
// begun by an earlier CTA, slot 2c+1 its last segment when a later CTA
// continues it.
struct WsLayout {
  size_t prefix_off, ml_off, acc_off, total;
};

__host__ __device__ inline WsLayout ws_layout(int num_streams, int grid, int hq, int head_dim) {
  WsLayout L;
  L.prefix_off = sizeof(WsHeader);
  L.ml_off = align_up(L.prefix_off + sizeof(int32_t) * (size_t)(num_streams + 1), 256);
  L.acc_off = align_up(L.ml_off + sizeof(float2) * 2 * (size_t)grid * hq, 256);
  L.total = align_up(L.acc_off + sizeof(float) * 2 * (size_t)grid * hq * head_dim, 256);
  return L;
}

__device__ inline void raise_error(WsHeader* h, uint32_t bit, long long info) {
  atomicOr(&h->error_bits, bit);
  atomicCAS(&h->error_info, 0ull, (unsigned long long)(info + 1));
}

// ---------------------------------------------------------------------------
// Parameters of one decode call (same struct for every kernel)
// ---------------------------------------------------------------------------
struct Params {
  const void* q;
  const void* k;
  const void* v;
  const int32_t* kv_start;
  const int32_t* block_table;
  const int32_t* seq_len;
  void* out;
  float* lse;
  WsHeader* ws;
  int32_t* prefix;
  float2* part_ml;
  float* part_acc;
  long long kv_rows;
  int bt_stride;
  int batch, num_q_heads, num_kv_heads, head_dim, page_size, page_shift;
  int group;        // query heads per KV head
  int hc;           // KV heads per work stream (tensor-core kernel; 1 otherwise)
  int hg;           // work streams per sequence
  int hq;           // query heads per work stream; stream j of a sequence
                    // serves query heads [j * hq, (j + 1) * hq)
  int tile;         // tokens per plan tile
  int seg_units;    // plan cost of starting a segment, in tiles (see compute_plan)
  int grid;         // CTAs of the split kernel
  int kernel;       // fd_kernel of the split kernel
  int q_dtype, kv_dtype;   // fd_dtype
  float score_scale;   // softmax_scale * k_scale * log2(e)  (scores in log2 units)
  float v_scale;
  int scale_kind;            // fd_scale_kind: finer K/V scales on top of the two above
  const float* k_scales;     // FD_SCALE_HEAD: [KVH]; FD_SCALE_TOKEN: [kv_rows][KVH]
  const float* v_scales;
  int pdl;                   // split kernel launched as a programmatic dependent (of the append)
  // Query tokens per sequence.  With q_len > 1 the kernels see q_len virtual
  // query heads per query head (num_q_heads and group above already count
  // them): virtual head v = qh * q_len + j is token j of query head qh, and
  // it attends to the first T - (q_len - 1 - j) keys of its sequence.
  int q_len;
  // KV append (fd_append.cu); q_dtype is the dtype of k_new / v_new
  const void* k_new;         // [batch][n_new][KVH][D]
  const void* v_new;
  const int32_t* positions;  // [batch] token index of the first new token, < 0: none
  int n_new;                 // new tokens per sequence
  void* k_dst;               // the caches, written
  void* v_dst;
  float* k_scales_dst;       // FD_SCALE_TOKEN: per-token scales, written
  float* v_scales_dst;
  float k_scale_raw, v_scale_raw;   // the per-tensor scales as given
  // Bound of every pipeline wait of the tensor-core split kernel, in ns
  // (one second unless a test shortens it), and a test switch under which
  // its producer issues no copy at all, so that the consumers' first wait
  // runs out with nothing in flight (fd_debug_set_wait_limit).
  unsigned long long wait_ns;
  int starve;
};

// Optional phase timestamps (built with -DFD_STAMPS, a separate library):
// slot i of CTA c in a kernel's stamp array holds %globaltimer (ns) when the
// CTA passed phase i; fd_debug_read_stamps copies them out.
#ifdef FD_STAMPS
constexpr int kStampCtas = 4096, kStampSlots = 24;
#define FD_STAMP_ARRAY(name) __device__ unsigned long long name[kStampCtas * kStampSlots]
#define FD_STAMP(arr, i, v)                                                        \
  do {                                                                             \
    if (blockIdx.x < kStampCtas) arr[blockIdx.x * kStampSlots + (i)] = (v);        \
  } while (0)
__device__ __forceinline__ unsigned long long stamp_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
cudaError_t read_split_stamps(unsigned long long* host, int n);
cudaError_t read_combine_stamps(unsigned long long* host, int n);
cudaError_t read_tc_stamps(unsigned long long* host, int n);
cudaError_t launch_empty(int grid, int threads, int smem, cudaStream_t st);
#else
#define FD_STAMP(arr, i, v) ((void)0)
#endif

// ---------------------------------------------------------------------------
// Split plan ("stream-K", balanced on cost).  A work stream is (sequence b,
// a run of hq consecutive query heads and the KV heads they read); stream
// s = b * hg + j.  Stream s has n_s = ceil(T_b / tile) tiles and, when
// n_s > 0, costs u_s = A + n_s plan units: A units for starting a segment
// (reloading Q and the row data; A = seg_units) followed by one unit per
// tile.  The streams' units are concatenated in stream order and CTA c takes
// units [c * L, min(U, (c + 1) * L)) with U = sum u_s and L = ceil(U / grid),
// so a CTA that starts more segments gets fewer tiles.  The tiles of stream
// s inside one CTA's range form a segment; a range that holds only some of
// a stream's A leading units holds no segment of it.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int stream_tokens(const Params& p, int s) {
  int t = __ldg(p.seq_len + s / p.hg);
  return t > 0 ? t : 0;
}

__device__ __forceinline__ int stream_tiles(const Params& p, int s) {
  return (stream_tokens(p, s) + p.tile - 1) / p.tile;
}

__device__ __forceinline__ int stream_units(const Params& p, int s) {
  const int n = stream_tiles(p, s);
  return n > 0 ? n + p.seg_units : 0;
}

struct PlanResult {
  long long total;      // U
  long long per_cta;    // L
  int s_first;          // stream holding this CTA's first unit (or num_streams)
  long long p_first;    // prefix (in units) of s_first
  long long first_start;   // kv_start of s_first's sequence (contiguous caches), or -1
};

__device__ inline void write_plan_words(const Params& p, long long total, long long per_cta) {
  p.ws->plan[0] = p.batch * p.hg;
  p.ws->plan[1] = p.hg;
  p.ws->plan[2] = p.tile;
  p.ws->plan[3] = p.grid;
  p.ws->plan[4] = (int32_t)total;
  p.ws->plan[5] = (int32_t)per_cta;
  p.ws->plan[6] = p.kernel;
  p.ws->plan[7] = p.seg_units;
  if (total > 0x7fffffffLL) raise_error(p.ws, kErrPlan, total);
}

// Barrier `id` over the first `nthreads` threads of the CTA (id 0 with
// every thread is __syncthreads).
__device__ __forceinline__ void plan_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// The plan over threads [0, nthreads) of the CTA (barrier `bar`); every one
// of them gets the same result.  CTA 0 also writes the prefix array and the
// plan words of the header.  `red` is >= 35 long longs of shared memory.
// With at most one stream per thread it is one pass (one read of seq_len,
// and of kv_start alongside it); else two.
__device__ inline PlanResult compute_plan(const Params& p, long long* red, int nthreads, int bar,
                                          unsigned long long* stamp = nullptr) {
  const int S = p.batch * p.hg;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = nthreads >> 5;
  if (S <= nthreads) {
    const long long v = tid < S ? stream_units(p, tid) : 0;
    const long long kvs = tid < S && p.kv_start ? (long long)__ldg(p.kv_start + tid / p.hg) : -1;
    long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) red[warp] = x;
    if (tid == 0) red[32] = S;
    plan_sync(bar, nthreads);
    long long woff = 0, total = 0;
    for (int w = 0; w < nwarps; ++w) {
      if (w < warp) woff += red[w];
      total += red[w];
    }
#ifdef FD_STAMPS
    if (stamp && tid == 0) *stamp = stamp_ns();
#else
    (void)stamp;
#endif
    PlanResult r;
    r.total = total;
    r.per_cta = total > 0 ? (total + p.grid - 1) / p.grid : 0;
    const long long target = (long long)blockIdx.x * r.per_cta;
    const bool has_work = target < total;
    const long long excl = woff + x - v;
    if (tid < S) {
      if (blockIdx.x == 0) p.prefix[tid] = (int32_t)excl;
      if (has_work && v > 0 && excl <= target && target < excl + v) {
        red[32] = tid;
        red[33] = excl;
        red[34] = kvs;
      }
    }
    if (blockIdx.x == 0 && tid == 0) {
      p.prefix[S] = (int32_t)total;
      write_plan_words(p, total, r.per_cta);
    }
    plan_sync(bar, nthreads);
    r.s_first = has_work ? (int)red[32] : S;
    r.p_first = has_work ? red[33] : total;
    r.first_start = has_work ? red[34] : -1;
    plan_sync(bar, nthreads);
    return r;
  }
  // pass 1: total units
  long long acc = 0;
  for (int s = tid; s < S; s += nthreads) acc += stream_units(p, s);
  for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) red[warp] = acc;
  plan_sync(bar, nthreads);
  long long total = 0;
  for (int w = 0; w < nwarps; ++w) total += red[w];
  plan_sync(bar, nthreads);
#ifdef FD_STAMPS
  if (stamp && tid == 0) *stamp = stamp_ns();
#else
  (void)stamp;
#endif
  PlanResult r;
  r.total = total;
  r.per_cta = total > 0 ? (total + p.grid - 1) / p.grid : 0;
  const long long target = (long long)blockIdx.x * r.per_cta;
  const bool has_work = target < total;
  // pass 2: exclusive prefix, position of this CTA's first tile
  if (tid == 0) { red[32] = S; }
  long long carry = 0;
  for (int base = 0; base < S; base += nthreads) {
    int s = base + tid;
    long long v = s < S ? stream_units(p, s) : 0;
    long long x = v;
    for (int o = 1; o < 32; o <<= 1) {
      long long y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) red[warp] = x;
    plan_sync(bar, nthreads);
    long long woff = 0, ctot = 0;
    for (int w = 0; w < nwarps; ++w) {
      if (w < warp) woff += red[w];
      ctot += red[w];
    }
    long long excl = carry + woff + x - v;
    if (s < S) {
      if (blockIdx.x == 0) p.prefix[s] = (int32_t)excl;
      if (has_work && v > 0 && excl <= target && target < excl + v) {
        red[32] = s;
        red[33] = excl;
      }
    }
    carry += ctot;
    plan_sync(bar, nthreads);
  }
  if (blockIdx.x == 0 && tid == 0) {
    p.prefix[S] = (int32_t)total;
    write_plan_words(p, total, r.per_cta);
  }
  r.s_first = has_work ? (int)red[32] : S;
  r.p_first = has_work ? red[33] : total;
  r.first_start = -1;
  plan_sync(bar, nthreads);
  return r;
}

// One segment: stream s, tokens [t_begin, t_end).
struct Segment {
  int s;
  int t_begin, t_end;
  int T;                // stream length
  bool complete;        // the whole stream is inside this CTA
  int slot;             // partial slot if !complete
};

// Iterates the segments of one CTA; every thread of a warp (or block) that
// uses it sees the same sequence.
struct SegmentIter {
  long long g, g_end;   // next unit, end of this CTA's range
  int s;                // stream holding unit g
  long long ps;         // prefix (units) of s
  int S;

  __device__ void init(const Params& p, const PlanResult& r) {
    S = p.batch * p.hg;
    g = (long long)blockIdx.x * r.per_cta;
    g_end = g + r.per_cta;
    if (g_end > r.total) g_end = r.total;
    s = r.s_first;
    ps = r.p_first;
  }
  // Returns false when the CTA has no more segments.
  __device__ bool next(const Params& p, Segment& seg) {
    for (;;) {
      if (g >= g_end || s >= S) return false;
      int nu = stream_units(p, s);
      while (g >= ps + nu) {   // skip empty / finished streams
        ps += nu;
        ++s;
        if (s >= S) return false;
        nu = stream_units(p, s);
      }
      const long long a = g, e = ps + nu < g_end ? ps + nu : g_end;
      const long long tb = ps + p.seg_units;   // unit of tile 0
      g = e;
      if (e <= tb) continue;                   // only leading units of s: no segment
      seg.s = s;
      seg.T = stream_tokens(p, s);
      const long long first = a > tb ? a - tb : 0;
      seg.t_begin = (int)(first * p.tile);
      const long long te = (e - tb) * p.tile;
      seg.t_end = te < seg.T ? (int)te : seg.T;
      const bool starts_mid = a > tb;
      const bool ends_mid = e < ps + nu;
      seg.complete = !starts_mid && !ends_mid;
      seg.slot = 2 * (int)blockIdx.x + (starts_mid ? 0 : 1);
      return true;
    }
  }
};

// ---------------------------------------------------------------------------
// Cache addressing (the one place the library maps tokens to rows)
// ---------------------------------------------------------------------------
// Row of token t of sequence b, or -1 (recorded as a device error) when the
// row or page id lies outside the cache.
__device__ __forceinline__ long long cache_row(const Params& p, int b, int t) {
  long long row;
  if (p.block_table) {
    int page = __ldg(p.block_table + (long long)b * p.bt_stride + (t >> p.page_shift));
    row = ((long long)page << p.page_shift) + (t & (p.page_size - 1));
    if (page < 0 || row >= p.kv_rows) {
      raise_error(p.ws, kErrBounds, page);
      return -1;
    }
  } else {
    row = (long long)__ldg(p.kv_start + b) + t;
    if (row < 0 || row >= p.kv_rows) {
      raise_error(p.ws, kErrBounds, row);
      return -1;
    }
  }
  return row;
}

// Lets the dependent (combine) grid be scheduled while this grid still runs;
// the dependent grid waits for this grid's completion before it reads.
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Waits until the grid this one depends on programmatically (the KV append,
// when the split kernel is launched after it with programmatic stream
// serialisation) has completed and its writes are visible.  Returns at once
// for a grid launched in plain stream order.
__device__ __forceinline__ void wait_prior_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Small math helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Signed 8-bit code (the low byte of `bits`, two's complement) -> its value
// as fp32, exactly, by the exponent-bias construction of IEEE-754 binary32:
// the biased byte u = code + 128 placed in the low mantissa bits of 2^23 reads
// as 2^23 + u, and subtracting 2^23 + 128 leaves the code.
__device__ __forceinline__ float i8_to_f32(uint32_t bits) {
  return __uint_as_float(0x4B000000u | ((bits ^ 0x80u) & 0xFFu)) - 8388736.0f;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <typename T> struct QType;
template <> struct QType<__half> {
  static __device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
  static __device__ __forceinline__ __half from_f32(float x) { return __float2half_rn(x); }
};
template <> struct QType<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from_f32(float x) { return __float2bfloat16_rn(x); }
};

// Launches a split kernel, as a programmatic dependent of the previous
// kernel in the stream when p.pdl (the kernel calls wait_prior_grid before
// it reads the caches).
template <typename Kernel, typename... Args>
inline cudaError_t launch_split(const Params& p, Kernel kern, dim3 grid, dim3 block, size_t smem,
                                cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per device: the limit belongs to the function on each device,
// so a process driving several GPUs sets it on each.  `done` holds one bit per
// device ordinal below 64 (higher ordinals set the limit on every call).
template <typename Kernel>
inline cudaError_t ensure_smem_limit(Kernel kern, int bytes,
                                     std::atomic<unsigned long long>* done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
  if (bit && (done->load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done->fetch_or(bit, std::memory_order_release);
  return e;
}

// Host-side argument checks shared by the decode entry points (fd_api.cu).
fd_status check_decode_args(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* kv_start_idx, const int32_t* block_table,
                            int block_table_stride, const int32_t* seq_len, int64_t kv_rows,
                            int batch, int num_q_heads, int num_kv_heads, int head_dim,
                            int page_size, float softmax_scale, float k_scale, float v_scale,
                            fd_scale_kind scale_kind, const float* k_scales,
                            const float* v_scales, fd_dtype q_dtype, fd_dtype kv_dtype,
                            const void* out, const float* lse, const void* workspace, int q_len);

// Launchers (defined in their .cu files).
cudaError_t launch_split_simt(const Params& p, cudaStream_t stream);
// the tensor-core kernels: mma.sync, or tcgen05 when p.kernel is FD_KERNEL_TC
cudaError_t launch_split_mma(const Params& p, cudaStream_t stream);
cudaError_t launch_combine(const Params& p, cudaStream_t stream);
cudaError_t launch_append(const Params& p, cudaStream_t stream);
int simt_ctas_per_sm();
bool simt_supports(int group, int head_dim);
int simt_heads_per_stream(int group);

}  // namespace fd
