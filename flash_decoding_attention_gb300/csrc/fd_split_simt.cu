// fd_split_simt.cu -- split (partial attention) kernel on CUDA-core FMAs.
//
// Computes, for every segment of the stream-K split plan, the online softmax
// state of each query head of the segment's KV head: running max m (log2
// units), running sum l and the rescaled V accumulator acc, following the
// online softmax loop of "SGLang Prefill optimisation: dissecting
// FlashAttention kernel bottlenecks with GPU Trace", section 2.2, with one
// query row per head as in decode.  One work stream is one KV head of one
// sequence; its `group` query heads are served by the same K/V reads
// ("Learn CUDA from scratch, chapter 15", section 15.12).  FP8 K/V are
// converted to fp32 right after the load ("From SGLang kernel source to GPU
// trace: DeepSeek V4.1 Flash-Decode", section 2.2).
//
// A work stream is one KV head of one sequence and up to 16 of its query
// heads (groups larger than 16 are cut into runs of 16).
//
// Mapping: 8 warps per CTA; warp w takes tokens t = t_begin + w, + 8, ...;
// lane l holds dims [l * D/32, (l + 1) * D/32) of q, k, v and acc; each score
// is a warp all-reduce.  At the end of a segment the 8 warps' states are
// merged in shared memory; a segment that holds a whole stream writes the
// final output, any other segment writes its partial state to its slot.
#include "fd_common.cuh"

namespace fd {
namespace {

constexpr int kSimtThreads = 256;
constexpr int kSimtWarps = kSimtThreads / 32;
constexpr int kSimtMaxGroup = 16;

template <int KVT, int DPL> struct KvRow;

template <int DPL> struct KvRow<FD_F16, DPL> {
  static __device__ __forceinline__ void load(const void* base, long long off, float* f) {
    const __half* p = static_cast<const __half*>(base) + off;
    if constexpr (DPL == 4) {
      uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
      float2 a = __half22float2(*reinterpret_cast<__half2*>(&u.x));
      float2 b = __half22float2(*reinterpret_cast<__half2*>(&u.y));
      f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    } else {
      uint32_t u = __ldg(reinterpret_cast<const unsigned int*>(p));
      float2 a = __half22float2(*reinterpret_cast<__half2*>(&u));
      f[0] = a.x; f[1] = a.y;
    }
  }
};

template <int DPL> struct KvRow<FD_BF16, DPL> {
  static __device__ __forceinline__ void load(const void* base, long long off, float* f) {
    const __nv_bfloat16* p = static_cast<const __nv_bfloat16*>(base) + off;
    if constexpr (DPL == 4) {
      uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
      float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u.x));
      float2 b = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u.y));
      f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    } else {
      uint32_t u = __ldg(reinterpret_cast<const unsigned int*>(p));
      float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u));
      f[0] = a.x; f[1] = a.y;
    }
  }
};

__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t pair) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(pair), __NV_E4M3);
  return __half22float2(*reinterpret_cast<__half2*>(&h));
}

template <int DPL> struct KvRow<FD_E4M3, DPL> {
  static __device__ __forceinline__ void load(const void* base, long long off, float* f) {
    const uint8_t* p = static_cast<const uint8_t*>(base) + off;
    if constexpr (DPL == 4) {
      uint32_t u = __ldg(reinterpret_cast<const unsigned int*>(p));
      float2 a = e4m3x2_to_float2(static_cast<uint16_t>(u & 0xffffu));
      float2 b = e4m3x2_to_float2(static_cast<uint16_t>(u >> 16));
      f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    } else {
      uint16_t u = __ldg(reinterpret_cast<const unsigned short*>(p));
      float2 a = e4m3x2_to_float2(u);
      f[0] = a.x; f[1] = a.y;
    }
  }
};

template <int DPL> struct KvRow<FD_I8, DPL> {
  static __device__ __forceinline__ void load(const void* base, long long off, float* f) {
    const uint8_t* p = static_cast<const uint8_t*>(base) + off;
    uint32_t u;
    if constexpr (DPL == 4) u = __ldg(reinterpret_cast<const unsigned int*>(p));
    else u = __ldg(reinterpret_cast<const unsigned short*>(p));
#pragma unroll
    for (int k = 0; k < DPL; ++k) f[k] = i8_to_f32(u >> (8 * k));
  }
};

template <int KVT, typename QT, int D>
__global__ void __launch_bounds__(kSimtThreads) simt_split_kernel(const Params p) {
  constexpr int DPL = D / 32;
  extern __shared__ float sm[];
  __shared__ long long red[35];

  const PlanResult plan = compute_plan(p, red, blockDim.x, 0);
  allow_dependent_launch();
  wait_prior_grid();   // a KV append launched just before may still be writing rows
  SegmentIter it;
  it.init(p, plan);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.hq;   // query heads of this stream (<= 16)
  float* sm_m = sm;
  float* sm_l = sm + kSimtWarps * G;
  float* sm_acc = sm + 2 * kSimtWarps * G;
  const QT* q = static_cast<const QT*>(p.q);

  Segment seg;
  while (it.next(p, seg)) {
    const int b = seg.s / p.hg;
    const int qh0 = (seg.s - b * p.hg) * G;
    const int kvh = qh0 / p.group;
    // finer scales: per KV head fold into q and the output, per token into
    // each score and each V row below
    float ksc = 1.f, vsc = 1.f;
    if (p.scale_kind == FD_SCALE_HEAD) {
      ksc = __ldg(p.k_scales + kvh);
      vsc = __ldg(p.v_scales + kvh);
    }

    float qv[kSimtMaxGroup][DPL];
    float m[kSimtMaxGroup], l[kSimtMaxGroup], acc[kSimtMaxGroup][DPL];
    // keys each (virtual) head attends to: all T, or for multi-token queries
    // up to its token's own position
    int lim[kSimtMaxGroup];
#pragma unroll
    for (int i = 0; i < kSimtMaxGroup; ++i) lim[i] = seg.T - (p.q_len - 1 - (qh0 + i) % p.q_len);
#pragma unroll
    for (int i = 0; i < kSimtMaxGroup; ++i) {
      m[i] = -INFINITY;
      l[i] = 0.f;
#pragma unroll
      for (int j = 0; j < DPL; ++j) {
        acc[i][j] = 0.f;
        qv[i][j] = i < G ? QType<QT>::to_f32(q[((long long)b * p.num_q_heads + qh0 + i) * D +
                                               lane * DPL + j]) * (p.score_scale * ksc)
                         : 0.f;
      }
    }

    for (int t = seg.t_begin + warp; t < seg.t_end; t += kSimtWarps) {
      const long long row = cache_row(p, b, t);
      if (row < 0) continue;
      const long long off = (row * p.num_kv_heads + kvh) * D + lane * DPL;
      float kf[DPL], vf[DPL];
      KvRow<KVT, DPL>::load(p.k, off, kf);
      KvRow<KVT, DPL>::load(p.v, off, vf);
      float tks = 1.f, tvs = 1.f;   // per-token scales of this row
      if (p.scale_kind == FD_SCALE_TOKEN) {
        tks = __ldg(p.k_scales + row * p.num_kv_heads + kvh);
        tvs = __ldg(p.v_scales + row * p.num_kv_heads + kvh);
      }
#pragma unroll
      for (int i = 0; i < kSimtMaxGroup; ++i) {
        if (i < G && t < lim[i]) {
          float s = 0.f;
#pragma unroll
          for (int j = 0; j < DPL; ++j) s = fmaf(qv[i][j], kf[j], s);
#pragma unroll
          for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
          s *= tks;
          const float mn = fmaxf(m[i], s);
          const float alpha = fast_exp2(m[i] - mn);
          const float pr = fast_exp2(s - mn);
          l[i] = fmaf(l[i], alpha, pr);
#pragma unroll
          for (int j = 0; j < DPL; ++j) acc[i][j] = fmaf(acc[i][j], alpha, (pr * tvs) * vf[j]);
          m[i] = mn;
        }
      }
    }

    // merge the warps' states
#pragma unroll
    for (int i = 0; i < kSimtMaxGroup; ++i) {
      if (i < G) {
        if (lane == 0) {
          sm_m[warp * G + i] = m[i];
          sm_l[warp * G + i] = l[i];
        }
#pragma unroll
        for (int j = 0; j < DPL; ++j) sm_acc[(warp * G + i) * D + lane * DPL + j] = acc[i][j];
      }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * D; idx += kSimtThreads) {
      const int i = idx / D, d = idx - (idx / D) * D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kSimtWarps; ++w) M = fmaxf(M, sm_m[w * G + i]);
      float L = 0.f, A = 0.f;
#pragma unroll
      for (int w = 0; w < kSimtWarps; ++w) {
        const float mw = sm_m[w * G + i];
        const float f = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
        L = fmaf(sm_l[w * G + i], f, L);
        A = fmaf(sm_acc[(w * G + i) * D + d], f, A);
      }
      if (seg.complete) {
        const float o = L > 0.f ? A * (p.v_scale * vsc / L) : 0.f;
        static_cast<QT*>(p.out)[((long long)b * p.num_q_heads + qh0 + i) * D + d] =
            QType<QT>::from_f32(o);
        if (d == 0 && p.lse)
          p.lse[(long long)b * p.num_q_heads + qh0 + i] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
      } else {
        p.part_acc[((long long)seg.slot * p.hq + i) * D + d] = A;
        if (d == 0) p.part_ml[(long long)seg.slot * p.hq + i] = make_float2(M, L);
      }
    }
    __syncthreads();
  }
}

template <int KVT, typename QT, int D>
cudaError_t launch_t(const Params& p, cudaStream_t stream) {
  auto kern = simt_split_kernel<KVT, QT, D>;
  const size_t smem = sizeof(float) * (2 * kSimtWarps * p.hq + kSimtWarps * p.hq * D);
  static std::atomic<unsigned long long> limit_set{0};
  cudaError_t e = ensure_smem_limit(
      kern, (int)(sizeof(float) * (2 * kSimtWarps * kSimtMaxGroup + kSimtWarps * kSimtMaxGroup * D)),
      &limit_set);
  if (e != cudaSuccess) return e;
  return launch_split(p, kern, dim3(p.grid), dim3(kSimtThreads), smem, stream, p);
}

template <int D>
cudaError_t launch_d(const Params& p, cudaStream_t stream) {
  if (p.kv_dtype == FD_F16) return launch_t<FD_F16, __half, D>(p, stream);
  if (p.kv_dtype == FD_BF16) return launch_t<FD_BF16, __nv_bfloat16, D>(p, stream);
  if (p.kv_dtype == FD_I8)
    return p.q_dtype == FD_F16 ? launch_t<FD_I8, __half, D>(p, stream)
                               : launch_t<FD_I8, __nv_bfloat16, D>(p, stream);
  if (p.q_dtype == FD_F16) return launch_t<FD_E4M3, __half, D>(p, stream);
  return launch_t<FD_E4M3, __nv_bfloat16, D>(p, stream);
}

}  // namespace

int simt_ctas_per_sm() { return 1; }

bool simt_supports(int group, int head_dim) {
  if (head_dim != 64 && head_dim != 128) return false;
  return group >= 1 && group <= 128 && (group <= kSimtMaxGroup || group % kSimtMaxGroup == 0);
}

int simt_heads_per_stream(int group) { return group <= kSimtMaxGroup ? group : kSimtMaxGroup; }

cudaError_t launch_split_simt(const Params& p, cudaStream_t stream) {
  if (p.head_dim == 128) return launch_d<128>(p, stream);
  return launch_d<64>(p, stream);
}

}  // namespace fd
