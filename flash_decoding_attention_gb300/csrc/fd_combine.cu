// fd_combine.cu -- log-sum-exp merge of the partial states of split streams.
//
// A stream that the split plan cut across CTAs c0 .. c1 left one partial
// state (m_i in log2 units, l_i, acc_i[D]) per CTA: slot 2*c0+1 for the CTA
// that holds its first tile, slot 2*c for every later CTA.  Merging is the
// rescale step of the online softmax ("SGLang Prefill optimisation:
// dissecting FlashAttention kernel bottlenecks with GPU Trace", section 2.2)
// applied to whole partial states:
//   M = max_i m_i,  L = sum_i l_i 2^(m_i - M),  A = sum_i acc_i 2^(m_i - M),
//   out = v_scale * A / L,  lse = (M + log2 L) * ln 2.
// Streams held by a single CTA were finalised by the split kernel; streams
// with no token get out = 0 and lse = -inf here.
//
// One warp merges one (stream, query head): its lanes first read the
// segments' (m, l) in parallel, then sweep the accumulators with several
// segment loads in flight per lane.
#include "fd_common.cuh"

namespace fd {
namespace {

constexpr int kCombineWarps = 4;
constexpr int kMaxSegments = 1024;   // per stream; more are merged in chunks

// Segment k of a stream whose first tile is in CTA c0 -> its partial slot:
// the first CTA's "last" slot, then each later CTA's "first" slot.
__device__ __forceinline__ int seg_slot(int c0, int k) { return k == 0 ? 2 * c0 + 1 : 2 * (c0 + k); }

template <typename QT, int D>
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const Params p) {
  constexpr int DPL = D / 32;
  __shared__ float wts[kCombineWarps][kMaxSegments];
  // wait for the split kernel (programmatic dependent launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.batch * p.hg;
  const long long gw = (long long)blockIdx.x * kCombineWarps + warp;
  if (gw >= (long long)S * p.hq) return;
  const int s = (int)(gw / p.hq), i = (int)(gw - (long long)s * p.hq);
  const int b = s / p.hg, j = s - b * p.hg;
  const int qh = j * p.hq + i;
  QT* out = static_cast<QT*>(p.out) + ((long long)b * p.num_q_heads + qh) * D + lane * DPL;
  float* lse = p.lse ? p.lse + (long long)b * p.num_q_heads + qh : nullptr;

  const long long P0 = p.prefix[s], P1 = p.prefix[s + 1], total = p.prefix[S];
  if (P1 == P0) {
#pragma unroll
    for (int k = 0; k < DPL; ++k) out[k] = QType<QT>::from_f32(0.f);
    if (lse && lane == 0) *lse = -INFINITY;
    return;
  }
  const long long per_cta = (total + p.grid - 1) / p.grid;
  const int c0 = (int)(P0 / per_cta), c1 = (int)((P1 - 1) / per_cta);
  if (c0 == c1) return;
  const int nseg = c1 - c0 + 1;

  float M = -INFINITY;
  for (int k = lane; k < nseg; k += 32) M = fmaxf(M, p.part_ml[(long long)seg_slot(c0, k) * p.hq + i].x);
#pragma unroll
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));

  float L = 0.f, acc[DPL];
#pragma unroll
  for (int k = 0; k < DPL; ++k) acc[k] = 0.f;
  for (int k0 = 0; k0 < nseg; k0 += kMaxSegments) {
    const int kn = min(kMaxSegments, nseg - k0);
    for (int k = lane; k < kn; k += 32) {
      const float2 ml = p.part_ml[(long long)seg_slot(c0, k0 + k) * p.hq + i];
      const float f = ml.x == -INFINITY ? 0.f : fast_exp2(ml.x - M);
      wts[warp][k] = f;
      L = fmaf(ml.y, f, L);
    }
    __syncwarp();
#pragma unroll 8
    for (int k = 0; k < kn; ++k) {
      const float f = wts[warp][k];
      const float* a = p.part_acc + ((long long)seg_slot(c0, k0 + k) * p.hq + i) * D + lane * DPL;
      if constexpr (DPL == 4) {
        const float4 v = *reinterpret_cast<const float4*>(a);
        acc[0] = fmaf(v.x, f, acc[0]);
        acc[1] = fmaf(v.y, f, acc[1]);
        acc[2] = fmaf(v.z, f, acc[2]);
        acc[3] = fmaf(v.w, f, acc[3]);
      } else {
        const float2 v = *reinterpret_cast<const float2*>(a);
        acc[0] = fmaf(v.x, f, acc[0]);
        acc[1] = fmaf(v.y, f, acc[1]);
      }
    }
    __syncwarp();
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  const float r = L > 0.f ? p.v_scale / L : 0.f;
#pragma unroll
  for (int k = 0; k < DPL; ++k) out[k] = QType<QT>::from_f32(acc[k] * r);
  if (lse && lane == 0) *lse = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
}

// Launched as a programmatic dependent of the split kernel: its CTAs may be
// scheduled while the split kernel drains, and wait (griddepcontrol.wait)
// until the split kernel has completed and its writes are visible.
template <typename QT, int D>
cudaError_t launch_t(const Params& p, cudaStream_t stream) {
  const long long warps = (long long)p.batch * p.hg * p.hq;
  const long long blocks = (warps + kCombineWarps - 1) / kCombineWarps;
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
  return cudaLaunchKernelEx(&cfg, combine_kernel<QT, D>, p);
}

}  // namespace

cudaError_t launch_combine(const Params& p, cudaStream_t stream) {
  if (p.q_dtype == FD_F16)
    return p.head_dim == 128 ? launch_t<__half, 128>(p, stream) : launch_t<__half, 64>(p, stream);
  return p.head_dim == 128 ? launch_t<__nv_bfloat16, 128>(p, stream)
                           : launch_t<__nv_bfloat16, 64>(p, stream);
}

}  // namespace fd
