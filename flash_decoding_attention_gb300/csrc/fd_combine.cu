// fd_combine.cu -- log-sum-exp merge of the partial states of split streams.
//
// A stream that the split plan cut across CTAs c0 .. c1 (the CTAs holding its
// first and last tile units) left one partial state (m_i in log2 units, l_i,
// acc_i[D]) per CTA: slot 2*c0+1 for the CTA that holds its first tile, slot
// 2*c for every later CTA.  Merging is the
// rescale step of the online softmax ("SGLang Prefill optimisation:
// dissecting FlashAttention kernel bottlenecks with GPU Trace", section 2.2)
// applied to whole partial states:
//   M = max_i m_i,  L = sum_i l_i 2^(m_i - M),  A = sum_i acc_i 2^(m_i - M),
//   out = v_scale * A / L,  lse = (M + log2 L) * ln 2.
// Streams held by a single CTA were finalised by the split kernel; streams
// with no token get out = 0 and lse = -inf here.
#include <type_traits>

#include "fd_common.cuh"

namespace fd {
namespace {

constexpr int kCombineWarps = 8;
constexpr int kCombineThreads = kCombineWarps * 32;
constexpr int kPrefixMax = 1024;   // streams up to which every CTA rebuilds the prefix itself

#ifdef FD_STAMPS
// 0 past griddepcontrol.wait, 1 merge done (warp 0), 2 stored (warp 0)
FD_STAMP_ARRAY(g_combine_stamps);
#endif

// Segment k of a stream whose first tile is in CTA c0 -> its partial slot:
// the first CTA's "last" slot, then each later CTA's "first" slot.
__device__ __forceinline__ int seg_slot(int c0, int k) { return k == 0 ? 2 * c0 + 1 : 2 * (c0 + k); }

// Exclusive prefix of the streams' plan units (the split plan's own count,
// from seq_len alone) into sp[0..S], S <= kPrefixMax; every thread of the
// CTA takes part.  seq_len is an input of the call, not written by the split
// kernel, so this runs before griddepcontrol.wait, while the split kernel
// still streams.
__device__ void stream_prefix(const Params& p, int S, int32_t* sp, int32_t* wsum) {
  constexpr int PER = kPrefixMax / kCombineThreads;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int32_t u[PER];
  int32_t mine = 0;
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int st = tid * PER + k;
    u[k] = st < S ? (int32_t)stream_units(p, st) : 0;
    mine += u[k];
  }
  int32_t x = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  int32_t woff = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kCombineWarps; ++w) {
    if (w < warp) woff += wsum[w];
    total += wsum[w];
  }
  int32_t e = woff + x - mine;
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    const int st = tid * PER + k;
    if (st < S) sp[st] = e;
    e += u[k];
  }
  if (tid == 0) sp[S] = total;
  __syncthreads();
}

template <typename QT>
__device__ __forceinline__ void store_row4(QT* dst, float a, float b, float c, float d) {
  uint2 w;
  if constexpr (std::is_same<QT, __half>::value) {
    __half2 h0 = __floats2half2_rn(a, b), h1 = __floats2half2_rn(c, d);
    w.x = *reinterpret_cast<uint32_t*>(&h0);
    w.y = *reinterpret_cast<uint32_t*>(&h1);
  } else {
    __nv_bfloat162 b0 = __floats2bfloat162_rn(a, b), b1 = __floats2bfloat162_rn(c, d);
    w.x = *reinterpret_cast<uint32_t*>(&b0);
    w.y = *reinterpret_cast<uint32_t*>(&b1);
  }
  *reinterpret_cast<uint2*>(dst) = w;
}

// One item = one (stream, query head).  A stream cut across CTAs c0..c1 has
// nseg = c1 - c0 + 1 partial states; nseg = 0 marks a stream the split
// kernel finalised itself and -1 a stream with no token.
struct Item {
  int s, i, c0, nseg;
};

__device__ __forceinline__ Item describe(const Params& p, int item, bool own, const int32_t* sp,
                                        int per_cta) {
  Item it;
  it.s = item / p.hq;
  it.i = item - it.s * p.hq;
  const int P0 = own ? sp[it.s] : p.prefix[it.s];
  const int P1 = own ? sp[it.s + 1] : p.prefix[it.s + 1];
  it.c0 = 0;
  if (P1 == P0) {
    it.nseg = -1;
  } else {
    it.c0 = (P0 + p.seg_units) / per_cta;   // CTA holding tile 0
    const int c1 = (P1 - 1) / per_cta;        // CTA holding the last tile
    it.nseg = it.c0 == c1 ? 0 : c1 - it.c0 + 1;
  }
  return it;
}

// One item per WPI warps; a CTA of 8 warps takes 8 / WPI items.  The WPI
// warps of an item split its partial states (state k goes to part k mod
// WPI), so that few long streams still spread their loads over many warps,
// while many short ones run one warp per item in a single wave.  With at
// most kPrefixMax streams every CTA rebuilds the streams' plan prefix from
// seq_len before griddepcontrol.wait (the CTAs resident beside the split
// kernel do it while it still streams); else it reads the split kernel's
// prefix after the wait.  Then the m/l pairs (one state per lane) and the
// first BATCH accumulator rows travel together: one round trip to memory
// for a stream with up to BATCH * WPI states.  Every lane owns D / 32 dims.
template <typename QT, int D, int WPI>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const Params p) {
  constexpr int DPL = D / 32;
  constexpr int IPC = kCombineWarps / WPI;   // items per CTA
  constexpr int BATCH = 6;                   // accumulator rows loaded with the m/l pairs
  using VecT = typename std::conditional<DPL == 4, float4, float2>::type;
  __shared__ int32_t sp[kPrefixMax + 1];
  __shared__ int32_t wsum[kCombineWarps];
  __shared__ float red_m[kCombineWarps];
  __shared__ float red_l[kCombineWarps];
  __shared__ float red_a[WPI > 1 ? kCombineWarps : 1][D];
  const int S = p.batch * p.hg;
  const bool own = S <= kPrefixMax;
  if (own) stream_prefix(p, S, sp, wsum);
  // wait for the split kernel (programmatic dependent launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) FD_STAMP(g_combine_stamps, 0, stamp_ns());
  const int total = own ? sp[S] : p.prefix[S];
  const int per_cta = total > 0 ? (total + p.grid - 1) / p.grid : 1;
  const long long items = (long long)S * p.hq;
  const int part = warp % WPI, slot_in_cta = warp / WPI;
  const long long item = (long long)blockIdx.x * IPC + slot_in_cta;
  Item it{0, 0, 0, 0};
  if (item < items) it = describe(p, (int)item, own, sp, per_cta);

  auto acc_row = [&](int k) -> const VecT* {
    const long long slot = seg_slot(it.c0, k);
    return reinterpret_cast<const VecT*>(p.part_acc + (slot * p.hq + it.i) * D + lane * DPL);
  };
  auto ml_of = [&](int k) -> float2 {
    return p.part_ml[(long long)seg_slot(it.c0, k) * p.hq + it.i];
  };
  float a[DPL];
#pragma unroll
  for (int k = 0; k < DPL; ++k) a[k] = 0.f;
  auto fma_row = [&](const VecT& x, float w) {
    if constexpr (DPL == 4) {
      a[0] = fmaf(x.x, w, a[0]);
      a[1] = fmaf(x.y, w, a[1]);
      a[2] = fmaf(x.z, w, a[2]);
      a[3] = fmaf(x.w, w, a[3]);
    } else {
      a[0] = fmaf(x.x, w, a[0]);
      a[1] = fmaf(x.y, w, a[1]);
    }
  };
  // this part's states: k_u = part + WPI * u, u < nu
  const int nu = it.nseg > part ? (it.nseg - part + WPI - 1) / WPI : 0;
  const float2 ml0 = lane < nu ? ml_of(part + WPI * lane) : make_float2(-INFINITY, 0.f);
  VecT v[BATCH];
#pragma unroll
  for (int u = 0; u < BATCH; ++u) v[u] = u < nu ? *acc_row(part + WPI * u) : VecT{};
  // max over this part's states (beyond 32 states: extra passes)
  float M = ml0.x;
  for (int u = 32 + lane; u < nu; u += 32) M = fmaxf(M, ml_of(part + WPI * u).x);
#pragma unroll
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if constexpr (WPI > 1) {
    if (lane == 0) red_m[warp] = M;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < WPI; ++w) M = fmaxf(M, red_m[slot_in_cta * WPI + w]);
  }
  // weighted sums; lane u holds the weight of state u of the current chunk
  float f = ml0.x == -INFINITY ? 0.f : fast_exp2(ml0.x - M);
  float L = ml0.y * f;
#pragma unroll
  for (int u = 0; u < BATCH; ++u) fma_row(v[u], __shfl_sync(0xffffffffu, f, u));
  for (int c = 0; c < nu; c += 32) {
    if (c > 0) {   // next chunk of 32 states: its m/l and weights
      const float2 ml = c + lane < nu ? ml_of(part + WPI * (c + lane)) : make_float2(-INFINITY, 0.f);
      f = ml.x == -INFINITY ? 0.f : fast_exp2(ml.x - M);
      L = fmaf(ml.y, f, L);
    }
    const int cnt = min(32, nu - c);
    for (int u0 = c == 0 ? BATCH : 0; u0 < cnt; u0 += BATCH) {
#pragma unroll
      for (int u = 0; u < BATCH; ++u)
        v[u] = u0 + u < cnt ? *acc_row(part + WPI * (c + u0 + u)) : VecT{};
#pragma unroll
      for (int u = 0; u < BATCH; ++u) fma_row(v[u], __shfl_sync(0xffffffffu, f, (u0 + u) & 31));
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  if constexpr (WPI > 1) {
    if (lane == 0) red_l[warp] = L;
#pragma unroll
    for (int k = 0; k < DPL; ++k) red_a[warp][lane * DPL + k] = a[k];
    __syncthreads();
    if (part != 0) return;
    L = 0.f;
#pragma unroll
    for (int w = 0; w < WPI; ++w) L += red_l[slot_in_cta * WPI + w];
#pragma unroll
    for (int k = 0; k < DPL; ++k) {
      float x = 0.f;
#pragma unroll
      for (int w = 0; w < WPI; ++w) x += red_a[slot_in_cta * WPI + w][lane * DPL + k];
      a[k] = x;
    }
  }
  if (threadIdx.x == 0) FD_STAMP(g_combine_stamps, 1, stamp_ns());
  if (item >= items || it.nseg == 0) return;
  const int b = it.s / p.hg, j = it.s - b * p.hg;
  const int qh = j * p.hq + it.i;
  QT* out = static_cast<QT*>(p.out) + ((long long)b * p.num_q_heads + qh) * D + lane * DPL;
  float* lse = p.lse ? p.lse + (long long)b * p.num_q_heads + qh : nullptr;
  if (it.nseg < 0) {   // no token: out = 0, lse = -inf
#pragma unroll
    for (int k = 0; k < DPL; ++k) out[k] = QType<QT>::from_f32(0.f);
    if (lse && lane == 0) *lse = -INFINITY;
    return;
  }
  // per-KV-head V scales apply here; per-token ones are inside the partials
  float vsc = p.v_scale;
  if (p.scale_kind == FD_SCALE_HEAD) vsc *= __ldg(p.v_scales + qh / p.group);
  const float r = L > 0.f ? vsc / L : 0.f;
  if constexpr (DPL == 4) {
    store_row4<QT>(out, a[0] * r, a[1] * r, a[2] * r, a[3] * r);
  } else {
#pragma unroll
    for (int k = 0; k < DPL; ++k) out[k] = QType<QT>::from_f32(a[k] * r);
  }
  if (lse && lane == 0) *lse = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
  if (threadIdx.x == 0) FD_STAMP(g_combine_stamps, 2, stamp_ns());
}

// Launched as a programmatic dependent of the split kernel: its CTAs may be
// scheduled while the split kernel drains, and wait (griddepcontrol.wait)
// until the split kernel has completed and its writes are visible.
template <typename QT, int D, int WPI>
cudaError_t launch_w(const Params& p, cudaStream_t stream) {
  const long long items = (long long)p.batch * p.hg * p.hq;
  const long long blocks = (items + kCombineWarps / WPI - 1) / (kCombineWarps / WPI);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel<QT, D, WPI>, p);
}

// Warps per item: enough to give every SM about 8 warps of merging work.
template <typename QT, int D>
cudaError_t launch_t(const Params& p, cudaStream_t stream) {
  const long long items = (long long)p.batch * p.hg * p.hq;
  const long long target = (long long)p.grid * kCombineWarps;
  if (items * 4 <= target) return launch_w<QT, D, 8>(p, stream);
  if (items * 2 <= target) return launch_w<QT, D, 4>(p, stream);
  if (items <= target) return launch_w<QT, D, 2>(p, stream);
  return launch_w<QT, D, 1>(p, stream);
}

}  // namespace

#ifdef FD_STAMPS
cudaError_t read_combine_stamps(unsigned long long* host, int n) {
  if (n > kStampCtas * kStampSlots) n = kStampCtas * kStampSlots;
  return cudaMemcpyFromSymbol(host, g_combine_stamps, sizeof(unsigned long long) * n);
}
#endif

cudaError_t launch_combine(const Params& p, cudaStream_t stream) {
  if (p.q_dtype == FD_F16)
    return p.head_dim == 128 ? launch_t<__half, 128>(p, stream) : launch_t<__half, 64>(p, stream);
  return p.head_dim == 128 ? launch_t<__nv_bfloat16, 128>(p, stream)
                           : launch_t<__nv_bfloat16, 64>(p, stream);
}

}  // namespace fd
