// fd_split_fma.cu -- the split kernel with its arithmetic on CUDA-core FMAs
// instead of tensor cores, on the same TMA pipeline, plan, stage shapes and
// partial-state format as the mma.sync kernel (fd_split_mma.cuh), so that the
// two differ only in how S = Q K^T and O += P V are computed.  FP8-e4m3
// caches, head_dim 128, at most 8 query heads per KV head, KV heads a
// multiple of 8 (one consumer warp per KV head), no per-token scales.
//
// The online softmax loop is that of "SGLang Prefill optimisation:
// dissecting FlashAttention kernel bottlenecks with GPU Trace", section 2.2;
// one pass over a KV tile serves every query head of its KV head ("Learn CUDA
// from scratch, chapter 15", section 15.12); FP8 K/V are widened right after
// the shared-memory load ("From SGLang kernel source to GPU trace: DeepSeek
// V4.1 Flash-Decode", section 2.2).
//
// Per consumer warp (one KV head, G <= 8 query heads), per 32 tokens:
//  - scores: lane t takes token t; its K row (eight 16-byte chunks under the
//    128-byte swizzle) is widened to fp32 16 dims at a time and multiplied
//    with the G query rows, held in shared memory as fp32 and read as
//    broadcast 16-byte vectors: G x 128 FMAs per lane;
//  - softmax: per head a warp max, the exponentials and a warp sum;
//  - O += P V: lane l takes head dims 4l .. 4l + 3 of all G heads; for each
//    token it widens its 4 V bytes and takes the token's G probabilities by
//    shuffles: 4 G FMAs per lane and token.
#include "fd_split_mma.cuh"

namespace fd {
namespace mma {
namespace {

constexpr int kFmaHeads = 8;   // query heads per KV head, at most

// e4m3 code -> the fp32 value code * 2^-120, on the integer ALUs: the code's
// sign to bit 31, its exponent and mantissa bits to bits 26..20 (an fp32
// exponent field of e means 2^(e - 127), i.e. 2^-120 times the e4m3 scale
// 2^(e - 7); codes with e = 0 land on fp32 subnormals with the same factor).
// The factor 2^120 is folded into the score scale and the output.  The two
// NaN codes (S.1111.111) read as +-480 * 2^-120.
constexpr float kFmaUnscale = 1.329227995784916e36f;   // 2^120

__device__ __forceinline__ float e4m3_byte_scaled(uint32_t w, int byte) {
  const int t = (int)(w << (24 - 8 * byte));   // the byte in bits 31..24
  return __int_as_float((t >> 4) & (int)0x87F00000);
}

__device__ __forceinline__ void widen16(uint4 w, float (&f)[16]) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int k = 0; k < 4; ++k) f[4 * i + k] = e4m3_byte_scaled(ws[i], k);
  }
}

__device__ __forceinline__ float4 lds_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

template <typename QT>
__global__ void __launch_bounds__(kThreads, 1)
    fma_split_kernel(const Params p, const Shape sh, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv) {
  constexpr int D = 128;
  constexpr bool BF16 = std::is_same<QT, __nv_bfloat16>::value;
  extern __shared__ uint8_t dyn_smem[];
  __shared__ Shared sm;
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  const uint32_t stage0 = smem_u32(base);
  // fp32 query rows: [consumer warp][head][D]
  const uint32_t qs0 = stage0 + sh.stages * 2 * sh.kv_bytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  uint64_t kv_policy;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(kv_policy));
  if (threadIdx.x == 0) {
    for (int i = 0; i < sh.stages; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], kConsumerWarps);
    }
    sm.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (threadIdx.x == kConsumerWarps * 32) {
    prefetch_map(&tmk);
    prefetch_map(&tmv);
  }
  prefetch_index_arrays(p);
  const PlanResult plan = compute_plan(p, sm.red, kThreads, 0);
  allow_dependent_launch();
  wait_prior_grid();   // a KV append launched just before may still be writing rows

  const int S = sh.stages;
  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    // (the mma.sync kernel's producer, without the gather and per-token
    // scale paths)
    SegmentIter it;
    it.init(p, plan);
    Segment seg;
    int n = 0;
    bool stop = p.starve != 0;
    while (!stop && it.next(p, seg)) {
      const int b = seg.s / p.hg;
      const int kvh0 = (seg.s - b * p.hg) * sh.hc;
      const long long start = p.block_table ? 0
                              : n == 0 && seg.s == plan.s_first && plan.first_start >= 0
                                  ? plan.first_start
                                  : (long long)__ldg(p.kv_start + b);
      int win_lo = 0, win_hi = 0;
      for (int t0 = seg.t_begin; t0 < seg.t_end; t0 += sh.tile, ++n) {
        const int valid = min(sh.tile, seg.t_end - t0);
        if (p.block_table) {
          const int pg_lo = t0 >> p.page_shift;
          const int pg_hi = ((t0 + valid - 1) >> p.page_shift) + 1;
          if (pg_lo < win_lo || pg_hi > win_hi) {
            const int last = ((seg.t_end - 1) >> p.page_shift) + 1;
            win_lo = pg_lo;
            win_hi = min(pg_lo + kPageWindow, last);
            __syncwarp();
            for (int k = lane; k < win_hi - win_lo; k += 32)
              sm.pages[k] = __ldg(p.block_table + (long long)b * p.bt_stride + win_lo + k);
            __syncwarp();
          }
        }
        if (lane == 0) {
          const int stg = (int)(n % S);
          const uint32_t ph = (uint32_t)((n / S) & 1);
          const bool waited = !*(volatile int*)&sm.abort_flag &&
                              mbar_wait(&sm.empty[stg], ph ^ 1u, p.wait_ns);
          if (!waited) {
            if (!*(volatile int*)&sm.abort_flag) {
              raise_error(p.ws, kErrTimeout, 1);
              *(volatile int*)&sm.abort_flag = 1;
            }
            stop = true;
          } else {
            const int nbox = sh.tile / sh.box_rows;
            uint8_t* kst = base + (size_t)stg * 2 * sh.kv_bytes;
            uint8_t* vst = kst + sh.kv_bytes;
            int bad = 0;
            uint32_t bytes = 0;
            for (int pass = 0; pass < 2; ++pass) {
              if (pass == 1) {
                sm.bad[stg] = bad;
                mbar_arrive_tx(&sm.full[stg], bytes);
              }
#pragma unroll 1
              for (int i = 0; i < nbox; ++i) {
                const int t = t0 + i * sh.box_rows;
                if (t - t0 >= valid) break;
                const int nval = min(sh.box_rows, valid - (t - t0));
                long long row;
                bool ok;
                if (p.block_table) {
                  const int page = sm.pages[(t >> p.page_shift) - win_lo];
                  row = ((long long)page << p.page_shift) + (t & (p.page_size - 1));
                  ok = page >= 0 && row + nval <= p.kv_rows;
                  if (!ok && pass == 0) raise_error(p.ws, kErrBounds, page);
                } else {
                  row = start + t;
                  ok = row >= 0 && row + nval <= p.kv_rows;
                  if (!ok && pass == 0) raise_error(p.ws, kErrBounds, row < 0 ? row : row + nval - 1);
                }
                if (pass == 0) {
                  if (ok) bytes += 2u * sh.hc * sh.nx * sh.box_rows * sh.row_bytes;
                  else bad = 1;
                  continue;
                }
                if (!ok) continue;
                if (sh.heads_box) {
                  tma_load_3d_hint(kst, &tmk, 0, (int)row, kvh0, &sm.full[stg], kv_policy);
                  tma_load_3d_hint(vst, &tmv, 0, (int)row, kvh0, &sm.full[stg], kv_policy);
                  continue;
                }
                for (int h = 0; h < sh.hc; ++h) {
                  const size_t off = (size_t)h * sh.region_bytes + (size_t)i * sh.box_rows * sh.row_bytes;
                  tma_load_3d_hint(kst + off, &tmk, 0, kvh0 + h, (int)row, &sm.full[stg], kv_policy);
                  tma_load_3d_hint(vst + off, &tmv, 0, kvh0 + h, (int)row, &sm.full[stg], kv_policy);
                }
              }
            }
          }
        }
        stop = __shfl_sync(0xffffffffu, stop, 0);
        if (stop) break;
      }
    }
    if (lane == 0 && stop) {
      for (int i = n - S < 0 ? 0 : n - S; i < n; ++i)
        if (!mbar_wait(&sm.full[i % S], (uint32_t)((i / S) & 1), kDrainNs))
          raise_error(p.ws, kErrDrain, 3);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int kvl = warp;   // one KV head per warp (hc = 8, one head tile each)
    const int G = p.group;
    const QT* qg = static_cast<const QT*>(p.q);
    const uint32_t qw = qs0 + (uint32_t)warp * kFmaHeads * D * 4u;
    const uint32_t pw = qs0 + (uint32_t)kConsumerWarps * kFmaHeads * D * 4u +
                        (uint32_t)warp * 32u * kFmaHeads * 4u;   // [32 tokens][8 heads] fp32
    SegmentIter it;
    it.init(p, plan);
    Segment seg;
    int n = 0;
    while (it.next(p, seg)) {
      const int b = seg.s / p.hg;
      const int j = seg.s - b * p.hg;
      const long long qrow0 = (long long)b * p.num_q_heads + (long long)j * p.hq + kvl * G;
      float sc = p.score_scale, vsc = p.v_scale;
      if (p.scale_kind == FD_SCALE_HEAD) {
        const int kvh = j * sh.hc + kvl;
        sc *= __ldg(p.k_scales + kvh);
        vsc *= __ldg(p.v_scales + kvh);
      }
      sc *= kFmaUnscale;   // K read as code * 2^-120
      // the segment's query rows, fp32, [head][D]
      __syncwarp();
      for (int h = 0; h < G; ++h) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(qg + (qrow0 + h) * D + 4 * lane));
        float2 a, c;
        if constexpr (BF16) {
          a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
          c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
        } else {
          a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
          c = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
        }
        asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(qw + (uint32_t)(h * D + 4 * lane) * 4u),
                     "f"(a.x), "f"(a.y), "f"(c.x), "f"(c.y)
                     : "memory");
      }
      __syncwarp();
      // causal limit of each head row (multi-token queries)
      int cut[kFmaHeads];
#pragma unroll
      for (int h = 0; h < kFmaHeads; ++h) cut[h] = p.q_len - 1 - (kvl * G + h) % p.q_len;
      float o[kFmaHeads][4], m[kFmaHeads], l[kFmaHeads];
#pragma unroll
      for (int h = 0; h < kFmaHeads; ++h) {
        o[h][0] = o[h][1] = o[h][2] = o[h][3] = 0.f;
        m[h] = -INFINITY;
        l[h] = 0.f;
      }
      for (int t0 = seg.t_begin; t0 < seg.t_end; t0 += sh.tile, ++n) {
        const int stg = (int)(n % S);
        const uint32_t ph = (uint32_t)((n / S) & 1);
        bool ok = !*(volatile int*)&sm.abort_flag;
        if (ok && !mbar_wait(&sm.full[stg], ph, p.wait_ns)) {
          raise_error(p.ws, kErrTimeout, 2);
          *(volatile int*)&sm.abort_flag = 1;
          ok = false;
        }
        if (ok && !sm.bad[stg]) {
          const uint32_t kreg = stage0 + stg * 2 * sh.kv_bytes + kvl * sh.region_bytes;
          const uint32_t vreg = kreg + sh.kv_bytes;
#pragma unroll 1
          for (int sub = 0; sub < sh.tile; sub += 32) {
            const int left = seg.t_end - (t0 + sub);   // valid tokens from the sub-tile start
            if (left <= 0) break;
            const int tk = sub + lane;                 // this lane's token in the tile
            // ---- scores of this lane's token for the G heads
            float s[kFmaHeads];
#pragma unroll
            for (int h = 0; h < kFmaHeads; ++h) s[h] = 0.f;
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
              float kf[16];
              widen16(lds128(chunk_addr(kreg, tk, c, 128)), kf);
#pragma unroll
              for (int h = 0; h < kFmaHeads; ++h) {
                if (h < G) {
#pragma unroll
                  for (int e = 0; e < 16; e += 4) {
                    const float4 q4 = lds_f32x4(qw + (uint32_t)(h * D + 16 * c + e) * 4u);
                    s[h] = fmaf(q4.x, kf[e], s[h]);
                    s[h] = fmaf(q4.y, kf[e + 1], s[h]);
                    s[h] = fmaf(q4.z, kf[e + 2], s[h]);
                    s[h] = fmaf(q4.w, kf[e + 3], s[h]);
                  }
                }
              }
            }
            // ---- online softmax per head (warp reductions over the tokens)
            float pr[kFmaHeads];
#pragma unroll
            for (int h = 0; h < kFmaHeads; ++h) {
              if (h >= G) {
                pr[h] = 0.f;
                continue;
              }
              const int lim = min(left, seg.T - cut[h] - (t0 + sub));
              const float x = lane < lim ? s[h] * sc : -INFINITY;
              float mx = x;
#pragma unroll
              for (int off = 16; off; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
              const float mn = fmaxf(m[h], mx);
              const float bse = mn == -INFINITY ? 0.f : mn;
              const float a = fast_exp2(m[h] - bse);
              const float pv = fast_exp2(x - bse);
              float sum = pv;
#pragma unroll
              for (int off = 16; off; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
              l[h] = fmaf(l[h], a, sum);
              m[h] = mn;
              o[h][0] *= a;
              o[h][1] *= a;
              o[h][2] *= a;
              o[h][3] *= a;
              pr[h] = pv;
            }
            // ---- O += P V over the valid tokens: lane owns dims 4 lane .. + 3;
            //      the probabilities go through shared memory, [token][head]
            asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(pw + lane * 32u),
                         "f"(pr[0]), "f"(pr[1]), "f"(pr[2]), "f"(pr[3])
                         : "memory");
            asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(pw + lane * 32u + 16u),
                         "f"(pr[4]), "f"(pr[5]), "f"(pr[6]), "f"(pr[7])
                         : "memory");
            __syncwarp();
            const int nt = min(32, left);
#pragma unroll 4
            for (int t = 0; t < nt; ++t) {
              const int row = sub + t;
              const uint32_t vw =
                  lds_u32(vreg + row * 128 + ((((lane >> 2) ^ (row & 7))) << 4) + (lane & 3) * 4);
              float vf[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) vf[k] = e4m3_byte_scaled(vw, k);
              const float4 p0 = lds_f32x4(pw + t * 32u), p1 = lds_f32x4(pw + t * 32u + 16u);
              const float pt[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
              for (int h = 0; h < kFmaHeads; ++h) {
                if (h < G) {
                  o[h][0] = fmaf(pt[h], vf[0], o[h][0]);
                  o[h][1] = fmaf(pt[h], vf[1], o[h][1]);
                  o[h][2] = fmaf(pt[h], vf[2], o[h][2]);
                  o[h][3] = fmaf(pt[h], vf[3], o[h][3]);
                }
              }
            }
            __syncwarp();
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[stg]);
      }
      // ---- segment end: this lane's 4 dims of every head (V was read as
      //      code * 2^-120)
#pragma unroll
      for (int h = 0; h < kFmaHeads; ++h) {
        o[h][0] *= kFmaUnscale;
        o[h][1] *= kFmaUnscale;
        o[h][2] *= kFmaUnscale;
        o[h][3] *= kFmaUnscale;
      }
      QT* outp = static_cast<QT*>(p.out);
      float* part = p.part_acc + ((long long)seg.slot * p.hq + kvl * G) * D;
      float2* pml = p.part_ml + (long long)seg.slot * p.hq + kvl * G;
#pragma unroll
      for (int h = 0; h < kFmaHeads; ++h) {
        if (h >= G) continue;
        if (seg.complete) {
          const float rs = l[h] > 0.f ? vsc / l[h] : 0.f;
          uint2 w;
          w.x = pack_f32x2(o[h][0] * rs, o[h][1] * rs, BF16);
          w.y = pack_f32x2(o[h][2] * rs, o[h][3] * rs, BF16);
          *reinterpret_cast<uint2*>(outp + (qrow0 + h) * D + 4 * lane) = w;
          if (lane == 0 && p.lse)
            p.lse[qrow0 + h] = l[h] > 0.f ? (m[h] + log2f(l[h])) * kLn2 : -INFINITY;
        } else {
          *reinterpret_cast<float4*>(part + h * D + 4 * lane) =
              make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
          if (lane == 0) pml[h] = make_float2(m[h], l[h]);
        }
      }
    }
  }
  __syncthreads();
}

template <typename QT>
cudaError_t launch_q(const Params& p, const Shape& sh, const Maps& m, cudaStream_t stream) {
  auto kern = fma_split_kernel<QT>;
  const int smem = sh.smem_bytes;
  static std::atomic<unsigned long long> limit_set{0};
  cudaError_t e = ensure_smem_limit(kern, kSmemBudget, &limit_set);
  if (e != cudaSuccess) return e;
  return launch_split(p, kern, dim3(p.grid), dim3(kThreads), smem, stream, p, sh, m.k, m.v);
}

}  // namespace

// Shape of the FMA form: the mma.sync kernel's shape for the group, with the
// Q fragment area replaced by fp32 query rows (8 warps x 8 heads x 128 dims).
bool fma_shape(int group, int num_kv_heads, int page_size, Shape* out) {
  Shape s = make_shape(group, num_kv_heads, 128, FD_E4M3, page_size, false);
  if (s.mt != 1 || s.hc != kConsumerWarps || s.wph != 1 || s.gather) return false;
  const int qbytes = kConsumerWarps * kFmaHeads * 128 * 4 + kConsumerWarps * 32 * kFmaHeads * 4;
  int st = (kSmemBudget - 1024 - qbytes) / (2 * s.kv_bytes);
  if (st > kMaxStages) st = kMaxStages;
  if (st < 2) return false;
  s.stages = st;
  s.merge_in_stage = 0;
  s.merge_bytes = 0;
  s.qfrag_bytes = qbytes;
  s.smem_bytes = 1024 + st * 2 * s.kv_bytes + qbytes;
  *out = s;
  return true;
}

cudaError_t launch_fma(const Params& p, const Shape& sh, const Maps& m, cudaStream_t st) {
  return p.q_dtype == FD_F16 ? launch_q<__half>(p, sh, m, st) : launch_q<__nv_bfloat16>(p, sh, m, st);
}

}  // namespace mma
}  // namespace fd
