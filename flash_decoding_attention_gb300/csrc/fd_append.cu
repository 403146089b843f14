// fd_append.cu -- KV-cache append of one new token per sequence.
//
// A decode step first writes the new token's K and V rows (the projection's
// output, in the query dtype) into the cache, then attends over the cache
// including them ("Learn CUDA from scratch, chapter 15", section 15.9: cache
// write layouts, contiguous and paged, and its single-token decode append);
// a speculative verify step (section 15.21) writes its n_new drafted tokens,
// token i of sequence b at position positions[b] + i.
// For 8-bit caches the rows are quantised on the way in, with the scales of
// section 15.11 of the same chapter:
//   s = k_scale                          per tensor
//     = k_scale * k_scales[h]            per KV head
//     = k_scale * ks, ks = amax / (QMAX * k_scale), written to
//       k_scales[row * KVH + h]          per token (amax over the row's head dims)
//   code = enc(x / s)    e4m3: nearest, ties to even, saturating at +-448;
//                        int8: nearest integer, ties to even, clamped to +-127.
// Every product and quotient that decides a code is a single IEEE fp32
// operation (explicit round-to-nearest intrinsics, so no contraction), which
// makes the codes reproducible off the device.
//
// One warp per (sequence, new token, KV head): each lane holds head_dim / 32 elements,
// so a row is one coalesced 256- or 128-byte load per tensor and the row's
// amax one warp reduction.
#include <type_traits>

#include "fd_common.cuh"

namespace fd {
namespace {

constexpr int kAppendWarps = 8;

template <typename XT, int DPL>
__device__ __forceinline__ void load_row(const XT* src, float* x, uint2& raw) {
  if constexpr (DPL == 4) {
    raw = __ldg(reinterpret_cast<const uint2*>(src));
    float2 a, b;
    if constexpr (std::is_same<XT, __half>::value) {
      a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
      b = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
    } else {
      a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
      b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
    }
    x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
  } else {
    raw.x = __ldg(reinterpret_cast<const unsigned int*>(src));
    raw.y = 0;
    float2 a;
    if constexpr (std::is_same<XT, __half>::value)
      a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
    else
      a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
    x[0] = a.x; x[1] = a.y;
  }
}

// Two fp32 quotients -> two 8-bit codes (low byte first).
template <int KVT>
__device__ __forceinline__ uint32_t encode2(float a, float b) {
  if constexpr (KVT == FD_E4M3) {
    return static_cast<uint32_t>(
        __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
  } else {
    const int ia = min(max(__float2int_rn(a), -127), 127);
    const int ib = min(max(__float2int_rn(b), -127), 127);
    return (static_cast<uint32_t>(ia) & 0xffu) | ((static_cast<uint32_t>(ib) & 0xffu) << 8);
  }
}

// One row (one KV head of one token) of K or V.
template <typename XT, int KVT, int DPL>
__device__ __forceinline__ void append_row(const XT* src, void* cache, long long dst, float scale,
                                           int kind, const float* head_scales, float* tok_scales,
                                           long long srow, int h, int lane) {
  float x[DPL];
  uint2 raw;
  load_row<XT, DPL>(src, x, raw);
  if constexpr (KVT == FD_F16 || KVT == FD_BF16) {
    XT* d = static_cast<XT*>(cache) + dst;
    if constexpr (DPL == 4) *reinterpret_cast<uint2*>(d) = raw;
    else *reinterpret_cast<unsigned int*>(d) = raw.x;
  } else {
    float s = scale;
    if (kind == FD_SCALE_HEAD) {
      s = __fmul_rn(scale, __ldg(head_scales + h));
    } else if (kind == FD_SCALE_TOKEN) {
      float amax = 0.f;
#pragma unroll
      for (int k = 0; k < DPL; ++k) amax = fmaxf(amax, fabsf(x[k]));
#pragma unroll
      for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const float qmax = KVT == FD_I8 ? 127.f : 448.f;
      const float ks = amax > 0.f ? __fdiv_rn(amax, __fmul_rn(qmax, scale)) : 1.f;
      if (lane == 0) tok_scales[srow] = ks;
      s = __fmul_rn(scale, ks);
    }
    uint32_t codes = 0;
#pragma unroll
    for (int k = 0; k < DPL; k += 2)
      codes |= encode2<KVT>(__fdiv_rn(x[k], s), __fdiv_rn(x[k + 1], s)) << (8 * k);
    uint8_t* d = static_cast<uint8_t*>(cache) + dst;
    if constexpr (DPL == 4) *reinterpret_cast<uint32_t*>(d) = codes;
    else *reinterpret_cast<uint16_t*>(d) = static_cast<uint16_t>(codes);
  }
}

template <typename XT, int KVT, int D>
__global__ void __launch_bounds__(kAppendWarps * 32) append_kernel(const Params p) {
  // The attention's split kernel, launched as a programmatic dependent, may
  // run its plan now; it waits for this grid before it reads K/V.
  allow_dependent_launch();
  constexpr int DPL = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long item = (long long)blockIdx.x * kAppendWarps + warp;
  if (item >= (long long)p.batch * p.n_new * p.num_kv_heads) return;
  const long long bi = item / p.num_kv_heads;            // b * n_new + i
  const int h = (int)(item - bi * p.num_kv_heads);
  const int b = (int)(bi / p.n_new), i = (int)(bi - (long long)b * p.n_new);
  const int t0 = __ldg(p.positions + b);
  if (t0 < 0) return;
  const long long row = cache_row(p, b, t0 + i);   // records out-of-range rows itself
  if (row < 0) return;
  const long long src = (bi * p.num_kv_heads + h) * D + lane * DPL;
  const long long dst = (row * p.num_kv_heads + h) * D + lane * DPL;
  const long long srow = row * p.num_kv_heads + h;
  append_row<XT, KVT, DPL>(static_cast<const XT*>(p.k_new) + src, p.k_dst, dst, p.k_scale_raw,
                           p.scale_kind, p.k_scales, p.k_scales_dst, srow, h, lane);
  append_row<XT, KVT, DPL>(static_cast<const XT*>(p.v_new) + src, p.v_dst, dst, p.v_scale_raw,
                           p.scale_kind, p.v_scales, p.v_scales_dst, srow, h, lane);
}

template <typename XT, int KVT>
cudaError_t launch_t(const Params& p, cudaStream_t stream) {
  const long long items = (long long)p.batch * p.n_new * p.num_kv_heads;
  const unsigned blocks = (unsigned)((items + kAppendWarps - 1) / kAppendWarps);
  if (p.head_dim == 128)
    append_kernel<XT, KVT, 128><<<blocks, kAppendWarps * 32, 0, stream>>>(p);
  else
    append_kernel<XT, KVT, 64><<<blocks, kAppendWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

template <typename XT>
cudaError_t launch_x(const Params& p, cudaStream_t stream) {
  if (p.kv_dtype == FD_E4M3) return launch_t<XT, FD_E4M3>(p, stream);
  if (p.kv_dtype == FD_I8) return launch_t<XT, FD_I8>(p, stream);
  // 16-bit caches hold the new rows' own dtype
  if constexpr (std::is_same<XT, __half>::value) return launch_t<XT, FD_F16>(p, stream);
  else return launch_t<XT, FD_BF16>(p, stream);
}

}  // namespace

cudaError_t launch_append(const Params& p, cudaStream_t stream) {
  return p.q_dtype == FD_F16 ? launch_x<__half>(p, stream) : launch_x<__nv_bfloat16>(p, stream);
}

}  // namespace fd
