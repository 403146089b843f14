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

#ifdef FD_STAMPS
// 0 past griddepcontrol.wait, 1 merge done (warp 0), 2 stored (warp 0)
FD_STAMP_ARRAY(g_combine_stamps);
#endif

// Segment k of a stream whose first tile is in CTA c0 -> its partial slot:
// the first CTA's "last" slot, then each later CTA's "first" slot.
__device__ __forceinline__ int seg_slot(int c0, int k) { return k == 0 ? 2 * c0 + 1 : 2 * (c0 + k); }

// One item = one (stream, query head).  A CTA of 8 warps takes 8 / WPI items;
// the WPI warps of an item split its segments (segment k goes to part
// k mod WPI), so that few long streams still spread their loads over many
// warps, while many short ones run one warp per item in a single wave.
// Every load that does not depend on another is issued before the first use:
// after the plan words, the m/l pairs (one segment per lane) and the first
// batch of accumulator rows travel together, so a stream with up to 8 * WPI
// segments costs two dependent round trips to memory.
template <typename QT, int D, int WPI>
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const Params p) {
  constexpr int DPL = D / 32;
  constexpr int IPC = kCombineWarps / WPI;          // items per CTA
  constexpr int BATCH = 8;                          // accumulator rows in flight per lane
  using VecT = typename std::conditional<DPL == 4, float4, float2>::type;
  __shared__ float red_m[kCombineWarps];
  __shared__ float red_l[kCombineWarps];
  __shared__ float red_a[kCombineWarps][D];
  // wait for the split kernel (programmatic dependent launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) FD_STAMP(g_combine_stamps, 0, stamp_ns());
  const int part = warp % WPI, slot_in_cta = warp / WPI;
  const int S = p.batch * p.hg;
  const long long item = (long long)blockIdx.x * IPC + slot_in_cta;
  const bool live = item < (long long)S * p.hq;
  int s = 0, i = 0, nseg = 0, c0 = 0;
  QT* out = nullptr;
  float* lse = nullptr;
  if (live) {
    s = (int)(item / p.hq);
    i = (int)(item - (long long)s * p.hq);
    const int b = s / p.hg, j = s - b * p.hg;
    const int qh = j * p.hq + i;
    out = static_cast<QT*>(p.out) + ((long long)b * p.num_q_heads + qh) * D;
    lse = p.lse ? p.lse + (long long)b * p.num_q_heads + qh : nullptr;
    const long long P0 = p.prefix[s], P1 = p.prefix[s + 1], total = p.prefix[S];
    if (P1 == P0) {
      if (part == 0) {
#pragma unroll
        for (int k = 0; k < DPL; ++k) out[lane * DPL + k] = QType<QT>::from_f32(0.f);
        if (lse && lane == 0) *lse = -INFINITY;
      }
    } else {
      const long long per_cta = (total + p.grid - 1) / p.grid;
      c0 = (int)((P0 + p.seg_units) / per_cta);   // CTA holding tile 0
      const int c1 = (int)((P1 - 1) / per_cta);     // CTA holding the last tile
      nseg = c0 == c1 ? 0 : c1 - c0 + 1;   // 0: the split kernel wrote the output
    }
  }
  // this part's segments: k_u = part + WPI * u, u < nu
  const int nu = nseg > part ? (nseg - part + WPI - 1) / WPI : 0;
  auto acc_row = [&](int u) -> const VecT* {
    const long long slot = seg_slot(c0, part + WPI * u);
    return reinterpret_cast<const VecT*>(p.part_acc + (slot * p.hq + i) * D + lane * DPL);
  };
  auto ml_of = [&](int u) -> float2 {
    return p.part_ml[(long long)seg_slot(c0, part + WPI * u) * p.hq + i];
  };
  // round trip 1: m/l of the first 32 segments (lane u) + first accumulator batch
  const float2 ml0 = lane < nu ? ml_of(lane) : make_float2(-INFINITY, 0.f);
  VecT v[BATCH];
#pragma unroll
  for (int u = 0; u < BATCH; ++u) {
    if (u < nu) v[u] = *acc_row(u);
    else v[u] = VecT{};
  }
  // max over this part's segments (beyond 32 segments: extra passes)
  float M = ml0.x;
  for (int u = 32 + lane; u < nu; u += 32) M = fmaxf(M, ml_of(u).x);
#pragma unroll
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if constexpr (WPI > 1) {
    if (lane == 0) red_m[warp] = M;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < WPI; ++w) M = fmaxf(M, red_m[slot_in_cta * WPI + w]);
  }
  // weighted sums; lane u holds the weight of segment u of the current chunk
  float f = ml0.x == -INFINITY ? 0.f : fast_exp2(ml0.x - M);
  float L = ml0.y * f;
  float acc[DPL];
#pragma unroll
  for (int k = 0; k < DPL; ++k) acc[k] = 0.f;
  auto accumulate = [&](const VecT& x, float w) {
    if constexpr (DPL == 4) {
      acc[0] = fmaf(x.x, w, acc[0]);
      acc[1] = fmaf(x.y, w, acc[1]);
      acc[2] = fmaf(x.z, w, acc[2]);
      acc[3] = fmaf(x.w, w, acc[3]);
    } else {
      acc[0] = fmaf(x.x, w, acc[0]);
      acc[1] = fmaf(x.y, w, acc[1]);
    }
  };
#pragma unroll
  for (int u = 0; u < BATCH; ++u) accumulate(v[u], __shfl_sync(0xffffffffu, f, u));
  for (int c = 0; c < nu; c += 32) {
    if (c > 0) {   // next chunk of 32 segments: its m/l and weights
      const float2 ml = c + lane < nu ? ml_of(c + lane) : make_float2(-INFINITY, 0.f);
      f = ml.x == -INFINITY ? 0.f : fast_exp2(ml.x - M);
      L = fmaf(ml.y, f, L);
    }
    const int cnt = min(32, nu - c);
    for (int u0 = c == 0 ? BATCH : 0; u0 < cnt; u0 += BATCH) {
#pragma unroll
      for (int u = 0; u < BATCH; ++u) {
        if (u0 + u < cnt) v[u] = *acc_row(c + u0 + u);
        else v[u] = VecT{};
      }
#pragma unroll
      for (int u = 0; u < BATCH; ++u) accumulate(v[u], __shfl_sync(0xffffffffu, f, (u0 + u) & 31));
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  if constexpr (WPI > 1) {
    if (lane == 0) red_l[warp] = L;
#pragma unroll
    for (int k = 0; k < DPL; ++k) red_a[warp][lane * DPL + k] = acc[k];
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
      acc[k] = x;
    }
  }
  if (threadIdx.x == 0) FD_STAMP(g_combine_stamps, 1, stamp_ns());
  if (nseg == 0) return;
  // per-KV-head V scales apply here; per-token ones are inside the partials
  float vsc = p.v_scale;
  if (p.scale_kind == FD_SCALE_HEAD) {
    const int qh = (s - (s / p.hg) * p.hg) * p.hq + i;   // query head of the item
    vsc *= __ldg(p.v_scales + qh / p.group);
  }
  const float r = L > 0.f ? vsc / L : 0.f;
  if constexpr (DPL == 4) {
    uint2 w;
    __half2 h0, h1;
    if constexpr (std::is_same<QT, __half>::value) {
      h0 = __floats2half2_rn(acc[0] * r, acc[1] * r);
      h1 = __floats2half2_rn(acc[2] * r, acc[3] * r);
      w.x = *reinterpret_cast<uint32_t*>(&h0);
      w.y = *reinterpret_cast<uint32_t*>(&h1);
    } else {
      __nv_bfloat162 b0 = __floats2bfloat162_rn(acc[0] * r, acc[1] * r);
      __nv_bfloat162 b1 = __floats2bfloat162_rn(acc[2] * r, acc[3] * r);
      w.x = *reinterpret_cast<uint32_t*>(&b0);
      w.y = *reinterpret_cast<uint32_t*>(&b1);
    }
    *reinterpret_cast<uint2*>(out + lane * DPL) = w;
  } else {
#pragma unroll
    for (int k = 0; k < DPL; ++k) out[lane * DPL + k] = QType<QT>::from_f32(acc[k] * r);
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
  cfg.blockDim = dim3(kCombineWarps * 32);
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
