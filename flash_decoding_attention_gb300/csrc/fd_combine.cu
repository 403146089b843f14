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
#include "fd_common.cuh"

namespace fd {
namespace {

constexpr int kCombineWarps = 4;

template <typename QT, int D>
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const Params p) {
  constexpr int DPL = D / 32;
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

  float M = -INFINITY;
  for (int c = c0; c <= c1; ++c) {
    const int slot = c == c0 ? 2 * c0 + 1 : 2 * c;
    M = fmaxf(M, p.part_ml[(long long)slot * p.hq + i].x);
  }
  float L = 0.f, acc[DPL];
#pragma unroll
  for (int k = 0; k < DPL; ++k) acc[k] = 0.f;
  for (int c = c0; c <= c1; ++c) {
    const int slot = c == c0 ? 2 * c0 + 1 : 2 * c;
    const float2 ml = p.part_ml[(long long)slot * p.hq + i];
    const float f = ml.x == -INFINITY ? 0.f : fast_exp2(ml.x - M);
    L = fmaf(ml.y, f, L);
    const float* a = p.part_acc + ((long long)slot * p.hq + i) * D + lane * DPL;
#pragma unroll
    for (int k = 0; k < DPL; ++k) acc[k] = fmaf(a[k], f, acc[k]);
  }
  const float r = L > 0.f ? p.v_scale / L : 0.f;
#pragma unroll
  for (int k = 0; k < DPL; ++k) out[k] = QType<QT>::from_f32(acc[k] * r);
  if (lse && lane == 0) *lse = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
}

template <typename QT, int D>
cudaError_t launch_t(const Params& p, cudaStream_t stream) {
  const long long warps = (long long)p.batch * p.hg * p.hq;
  const long long blocks = (warps + kCombineWarps - 1) / kCombineWarps;
  combine_kernel<QT, D><<<(unsigned)blocks, kCombineWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_combine(const Params& p, cudaStream_t stream) {
  if (p.q_dtype == FD_F16)
    return p.head_dim == 128 ? launch_t<__half, 128>(p, stream) : launch_t<__half, 64>(p, stream);
  return p.head_dim == 128 ? launch_t<__nv_bfloat16, 128>(p, stream)
                           : launch_t<__nv_bfloat16, 64>(p, stream);
}

}  // namespace fd
