// fd_split_tc.cu -- the split kernel on the fifth-generation tensor cores
// (tcgen05.mma, accumulators in tensor memory) for query groups of 17..128
// rows per KV head: the q_len query tokens of a speculative verify step
// ("Learn CUDA from scratch, chapter 15", section 15.21) run as q_len rows of
// each query head, and large GQA/MQA groups (section 15.12) the same way.
// FP8-e4m3 caches (the first page's FP8 KV, section 2.2), fp16 queries,
// head_dim 128, per-tensor or per-KV-head scales.
//
// Per tile of one (sequence, KV head) stream (128 tokens when the group has
// at most 64 rows, else 64):
//   producer warp:   K and V tiles (e4m3) HBM -> shared memory by TMA;
//   converter warps: e4m3 -> f16 once per tile into the operand layouts of
//                    the tensor core (K: K-major, V: MN-major, 128-byte
//                    swizzle), rows past the sequence's end zeroed in V;
//   MMA warp:        S = Q K^T (M = 64 or 128 query rows, N = the tile,
//                    K = 128 dims) into one of two S buffers in tensor memory
//                    and O += P V (N = 128 dims, K = the tile) into tensor
//                    memory, whichever of the two is ready first;
//   softmax warps:   the online-softmax update of each row ("SGLang Prefill
//                    optimisation: dissecting FlashAttention kernel
//                    bottlenecks with GPU Trace", section 2.2), 64 scores per
//                    thread (M = 64: a row's two halves on lanes l and l + 16),
//                    P in f16 into shared memory for the P V product.
// One tcgen05.mma costs the issuing thread about 68 cycles on this GB300
// whatever its shape up to N = 128, so the tiles are sized to need few of
// them: 8 for S and tile / 16 for P V.
// The running maximum used for the exponentials is moved only when a tile's
// maximum exceeds it by more than 2^8, so that O in tensor memory is rescaled
// rarely; P then stays below 256, and O, l and the reference maximum m are
// kept consistent, which is all the LSE merge needs.  Segment ends write the
// same partial states (m in log2 units, l, unnormalised O) or final outputs
// as the mma.sync split kernel, so the plan and the combine are shared.
#include <cstring>

#include "fd_split_mma.cuh"

namespace fd {
namespace tc {
namespace {

using mma::mbar_arrive;
using mma::mbar_arrive_tx;
using mma::mbar_init;
using mma::mbar_try_wait;
using mma::mbar_wait;
using mma::smem_u32;

constexpr int kWarpsTC = 10;                      // 4 softmax, 4 converter, producer, MMA
constexpr int kThreadsTC = kWarpsTC * 32;
constexpr int kConvWarp0 = 4, kProducerWarp = 8, kMmaWarp = 9;
constexpr uint32_t kRowBytes = 128;               // one e4m3 row of 128 dims
constexpr int kCols = 64;                         // scores per softmax thread per tile

// Shape of the kernel for M query rows per MMA.
template <int M>
struct TcShape {
  static constexpr int kTile = M == 64 ? 128 : 64;               // tokens per tile
  static constexpr int kStages = M == 64 ? 2 : 6;                // e4m3 stages
  static constexpr uint32_t kStageBytes = 2u * kTile * kRowBytes;    // K then V
  static constexpr uint32_t kF16Bytes = (uint32_t)kTile * 256u;      // one f16 tile
  // one f16 K buffer (read only by the S product of its tile), two V buffers
  static constexpr uint32_t kOffK16 = kStages * kStageBytes;
  static constexpr uint32_t kOffV16 = kOffK16 + kF16Bytes;
  static constexpr uint32_t kOffQ = kOffV16 + 2u * kF16Bytes;
  static constexpr uint32_t kQBytes = (uint32_t)M * 256u;
  static constexpr uint32_t kOffP = kOffQ + kQBytes;
  static constexpr uint32_t kPBytes = (uint32_t)M * kTile * 2u;
  static constexpr uint32_t kSmem = 1024u + kOffP + 2u * kPBytes;   // two P buffers
  static constexpr int kTmemCols = M == 64 ? 512 : 256;         // S: 2 x tile, O: 128
};
static_assert(TcShape<64>::kSmem <= (uint32_t)mma::kSmemBudget, "shared memory");
static_assert(TcShape<128>::kSmem <= (uint32_t)mma::kSmemBudget, "shared memory");

// Shared-memory matrix descriptor: 128-byte swizzle, start address, leading
// and stride byte offsets (bytes, multiples of 16), descriptor version 1.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor, kind::f16: f16 A and B, f32 accumulator, A K-major,
// B K-major (b_mn = 0) or MN-major (b_mn = 1), M x N.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int b_mn) {
  return (1u << 4) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, int acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// Arrives on `bar` once every tcgen05.mma this thread issued so far is done.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// generic-proxy shared-memory writes -> visible to the tensor core
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Non-blocking test of a barrier phase.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

#define TC_REGS32(r, o)                                                                    \
  "=r"(r[o + 0]), "=r"(r[o + 1]), "=r"(r[o + 2]), "=r"(r[o + 3]), "=r"(r[o + 4]),          \
      "=r"(r[o + 5]), "=r"(r[o + 6]), "=r"(r[o + 7]), "=r"(r[o + 8]), "=r"(r[o + 9]),      \
      "=r"(r[o + 10]), "=r"(r[o + 11]), "=r"(r[o + 12]), "=r"(r[o + 13]), "=r"(r[o + 14]), \
      "=r"(r[o + 15]), "=r"(r[o + 16]), "=r"(r[o + 17]), "=r"(r[o + 18]), "=r"(r[o + 19]), \
      "=r"(r[o + 20]), "=r"(r[o + 21]), "=r"(r[o + 22]), "=r"(r[o + 23]), "=r"(r[o + 24]), \
      "=r"(r[o + 25]), "=r"(r[o + 26]), "=r"(r[o + 27]), "=r"(r[o + 28]), "=r"(r[o + 29]), \
      "=r"(r[o + 30]), "=r"(r[o + 31])
#define TC_FREGS32(v, o)                                                                  \
  "f"(v[o + 0]), "f"(v[o + 1]), "f"(v[o + 2]), "f"(v[o + 3]), "f"(v[o + 4]), "f"(v[o + 5]), \
      "f"(v[o + 6]), "f"(v[o + 7]), "f"(v[o + 8]), "f"(v[o + 9]), "f"(v[o + 10]),           \
      "f"(v[o + 11]), "f"(v[o + 12]), "f"(v[o + 13]), "f"(v[o + 14]), "f"(v[o + 15]),       \
      "f"(v[o + 16]), "f"(v[o + 17]), "f"(v[o + 18]), "f"(v[o + 19]), "f"(v[o + 20]),       \
      "f"(v[o + 21]), "f"(v[o + 22]), "f"(v[o + 23]), "f"(v[o + 24]), "f"(v[o + 25]),       \
      "f"(v[o + 26]), "f"(v[o + 27]), "f"(v[o + 28]), "f"(v[o + 29]), "f"(v[o + 30]),       \
      "f"(v[o + 31])
#define TC_LIST32                                                                        \
  "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23," \
  "%24,%25,%26,%27,%28,%29,%30,%31}"
#define TC_LIST32_1                                                                        \
  "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24," \
  "%25,%26,%27,%28,%29,%30,%31,%32}"

// 32 columns of this thread's accumulator row.  M = 128: lane l of the warp's
// lane quarter, columns [c, c + 32).  M = 64 (rows in lanes 0..15 of each
// quarter): lanes 0..15 read columns [c, c + 32) of rows 0..15 and lanes
// 16..31 columns [c + 64, c + 96) of the same rows.
template <int M>
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  if constexpr (M == 128) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 " TC_LIST32 ", [%32];"
                 : TC_REGS32(r, 0)
                 : "r"(taddr));
  } else {
    asm volatile("tcgen05.ld.sync.aligned.16x32bx2.x32.b32 " TC_LIST32 ", [%32], 64;"
                 : TC_REGS32(r, 0)
                 : "r"(taddr));
  }
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

template <int M>
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  if constexpr (M == 128) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], " TC_LIST32_1 ";" ::"r"(taddr),
                 TC_FREGS32(v, 0)
                 : "memory");
  } else {
    asm volatile("tcgen05.st.sync.aligned.16x32bx2.x32.b32 [%0], 64, " TC_LIST32_1 ";" ::"r"(taddr),
                 TC_FREGS32(v, 0)
                 : "memory");
  }
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Operand layouts (byte offsets inside a buffer), 128-byte swizzle: the
// 16-byte chunk index inside a 128-byte row is XORed with the row index mod 8.
//   K-major [rows][K] f16: blocks of 64 K-elements, each rows x 128 bytes.
__device__ __forceinline__ uint32_t kmajor_chunk(uint32_t rows, int r, int c16) {
  return (uint32_t)(c16 >> 3) * rows * 128u + (uint32_t)r * 128u +
         ((uint32_t)((c16 & 7) ^ (r & 7)) << 4);
}
//   MN-major V [tile tokens][128 dims] f16: dims in two 64-dim atoms of
//   tile x 128 bytes, tokens in groups of 8 rows of 128 bytes, 1 KB apart.
__device__ __forceinline__ uint32_t vmn_chunk(uint32_t tile, int t, int c16) {
  return (uint32_t)(c16 >> 3) * tile * 128u + (uint32_t)(t >> 3) * 1024u +
         (uint32_t)(t & 7) * 128u + ((uint32_t)((c16 & 7) ^ (t & 7)) << 4);
}

constexpr int kMaxStagesTC = 6;

struct SharedTC {
  uint64_t e_full[kMaxStagesTC], e_empty[kMaxStagesTC];
  uint64_t k_full[2], v_full[2], s_full[2], s_free[2], done[2];
  uint64_t p_full[2], o_free, fin;
  int bad[kMaxStagesTC];   // stage held a row outside the cache (producer)
  // tile j came from such a stage (converters, slot j mod 4: the converters
  // run at most three tiles ahead of the softmax warps that read it)
  int fbad[4];
  int tfirst[4];   // tile j (slot j mod 4) starts a segment (converters -> MMA thread)
  int abort_flag;
  uint32_t tmem_base;
  long long red[35];
  int pages[mma::kPageWindow];
};

#ifdef FD_STAMPS
// per-tile phase stamps of tiles 4..5 of each CTA (slot 2 * event + tile - 4)
FD_STAMP_ARRAY(g_tc_stamps);
#define TC_STAMP(ev, jt)                                                                   \
  do {                                                                                     \
    if ((jt) >= 4 && (jt) < 6) FD_STAMP(g_tc_stamps, 2 * (ev) + (jt) - 4, stamp_ns());   \
  } while (0)
#else
#define TC_STAMP(ev, jt) ((void)0)
#endif

// The CTA's tiles in order, segment by segment.
struct TileSeq {
  SegmentIter it;
  Segment seg;
  int t0;
  bool have;
  __device__ void init(const Params& p, const PlanResult& plan) {
    it.init(p, plan);
    have = it.next(p, seg);
    t0 = have ? seg.t_begin : 0;
  }
  __device__ bool first() const { return t0 == seg.t_begin; }
  __device__ bool last(int tile) const { return t0 + tile >= seg.t_end; }
  __device__ __noinline__ void next(const Params& p, int tile) {
    t0 += tile;
    if (t0 >= seg.t_end) {
      have = it.next(p, seg);
      t0 = have ? seg.t_begin : 0;
    }
  }
};

__device__ __forceinline__ bool aborted(const SharedTC& sm) {
  return *(volatile const int*)&sm.abort_flag != 0;
}

__device__ __noinline__ void record_abort(SharedTC& sm, const Params& p, int role) {
  if (!aborted(sm)) {
    raise_error(p.ws, kErrTimeout, role);
    *(volatile int*)&sm.abort_flag = 1;
  }
}

// A bounded wait; on expiry records the timeout (with the waiting role) and
// raises the CTA's abort flag.
__device__ __forceinline__ bool wait_or_abort(SharedTC& sm, const Params& p, uint64_t* bar,
                                              uint32_t parity, int role) {
  if (mbar_try_wait(bar, parity)) return true;
  if (aborted(sm)) return false;
  if (mbar_wait(bar, parity, p.wait_ns)) return true;
  record_abort(sm, p, role);
  return false;
}

// M: query rows per MMA (64 or 128, at least the group's rows);
// CAUSAL: q_len > 1, row r (token r mod q_len of its head) stops
// q_len - 1 - r mod q_len keys before its sequence's end.
template <int M, bool CAUSAL>
__global__ void __launch_bounds__(kThreadsTC, 1)
    tc_split_kernel(const Params p, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv) {
  using SH = TcShape<M>;
  constexpr int TILE = SH::kTile;
  constexpr int NS = SH::kStages;
  extern __shared__ uint8_t dyn_smem[];
  __shared__ SharedTC sm;
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(base);
  const uint32_t sK16 = sbase + SH::kOffK16;
  const uint32_t sV16 = sbase + SH::kOffV16;
  const uint32_t sQ = sbase + SH::kOffQ;
  const uint32_t sP = sbase + SH::kOffP;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  uint64_t kv_policy;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(kv_policy));
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&sm.e_full[i], 1);
      mbar_init(&sm.e_empty[i], 4);   // the converter warps
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.k_full[i], 4);    // the converter warps (K of a tile in f16)
      mbar_init(&sm.v_full[i], 4);    // the converter warps (V of a tile in f16)
      mbar_init(&sm.s_full[i], 1);    // MMA commit after Q K^T
      mbar_init(&sm.s_free[i], 4);    // the softmax warps
      mbar_init(&sm.done[i], 1);      // MMA commit after P V
    }
    mbar_init(&sm.p_full[0], 4);      // the softmax warps
    mbar_init(&sm.p_full[1], 4);
    mbar_init(&sm.o_free, 4);
    mbar_init(&sm.fin, 1);
    sm.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&sm.tmem_base)),
                 "r"(SH::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x == kProducerWarp * 32) {
    mma::prefetch_map(&tmk);
    mma::prefetch_map(&tmv);
  }
  mma::prefetch_index_arrays(p);
  tc_fence_before();
  const PlanResult plan = compute_plan(p, sm.red, kThreadsTC, 0);   // (barriers: all threads)
  tc_fence_after();
  const uint32_t tbase = sm.tmem_base;
  allow_dependent_launch();
  wait_prior_grid();   // a KV append launched just before may still be writing rows

  const int R = p.hq;   // query rows of the stream (one KV head)
  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    SegmentIter it;
    it.init(p, plan);
    Segment seg;
    int n = 0;
    bool stop = p.starve != 0;   // test switch: issue nothing
    const int box_rows = p.block_table && p.page_size < TILE ? p.page_size : TILE;
    while (!stop && it.next(p, seg)) {
      const int b = seg.s / p.hg;
      const int kvh = seg.s - b * p.hg;
      const long long start = p.block_table ? 0
                              : n == 0 && seg.s == plan.s_first && plan.first_start >= 0
                                  ? plan.first_start
                                  : (long long)__ldg(p.kv_start + b);
      int win_lo = 0, win_hi = 0;
      for (int t0 = seg.t_begin; t0 < seg.t_end; t0 += TILE, ++n) {
        const int valid = min(TILE, seg.t_end - t0);
        if (p.block_table) {
          const int pg_lo = t0 >> p.page_shift;
          const int pg_hi = ((t0 + valid - 1) >> p.page_shift) + 1;
          if (pg_lo < win_lo || pg_hi > win_hi) {
            const int last = ((seg.t_end - 1) >> p.page_shift) + 1;
            win_lo = pg_lo;
            win_hi = min(pg_lo + mma::kPageWindow, last);
            __syncwarp();
            for (int k = lane; k < win_hi - win_lo; k += 32)
              sm.pages[k] = __ldg(p.block_table + (long long)b * p.bt_stride + win_lo + k);
            __syncwarp();
          }
        }
        if (lane == 0) {
          const int stg = n % NS;
          const uint32_t ph = (uint32_t)((n / NS) & 1);
          if (!wait_or_abort(sm, p, &sm.e_empty[stg], ph ^ 1u, 1)) {
            stop = true;
          } else {
            uint8_t* kst = base + (size_t)stg * SH::kStageBytes;
            uint8_t* vst = kst + TILE * kRowBytes;
            const int nbox = (valid + box_rows - 1) / box_rows;
            int bad = 0;
            uint32_t bytes = 0;
            for (int pass = 0; pass < 2; ++pass) {
              if (pass == 1) {
                sm.bad[stg] = bad;
                mbar_arrive_tx(&sm.e_full[stg], bytes);
              }
              for (int i = 0; i < nbox; ++i) {
                const int t = t0 + i * box_rows;
                const int nval = min(box_rows, valid - i * box_rows);
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
                  if (ok) bytes += 2u * (uint32_t)box_rows * kRowBytes;
                  else bad = 1;
                  continue;
                }
                if (!ok) continue;
                const uint32_t off = (uint32_t)i * box_rows * kRowBytes;
                mma::tma_load_3d_hint(kst + off, &tmk, 0, kvh, (int)row, &sm.e_full[stg], kv_policy);
                mma::tma_load_3d_hint(vst + off, &tmv, 0, kvh, (int)row, &sm.e_full[stg], kv_policy);
              }
            }
          }
        }
        stop = __shfl_sync(0xffffffffu, stop, 0);
        if (stop) break;
      }
    }
    if (lane == 0 && stop) {
      // copies of the last issued stages must land before the CTA exits
      for (int i = n - NS < 0 ? 0 : n - NS; i < n; ++i)
        if (!mbar_wait(&sm.e_full[i % NS], (uint32_t)((i / NS) & 1), mma::kDrainNs))
          raise_error(p.ws, kErrDrain, 3);
    }
  } else if (warp >= kConvWarp0 && warp < kProducerWarp) {
    // ------------------------------------------------------------ converters
    const int ct = threadIdx.x - kConvWarp0 * 32;   // 0..127
    const __half* qg = static_cast<const __half*>(p.q);
    TileSeq ts;
    ts.init(p, plan);
    int j = 0;
    while (ts.have) {
      const int bi = j & 1;
      if (ts.first()) {
        // the segment's Q rows into the Q buffer, K-major, once every
        // product of the previous tile (the last S with the old rows) is done
        if (j > 0 && !wait_or_abort(sm, p, &sm.s_full[(j - 1) & 1], (uint32_t)(((j - 1) >> 1) & 1), 5))
          break;
        const int b = ts.seg.s / p.hg;
        const long long qrow0 = (long long)b * p.num_q_heads + (long long)(ts.seg.s - b * p.hg) * R;
        for (int idx = ct; idx < R * 16; idx += 128) {
          const int r = idx >> 4, c = idx & 15;
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(qg + (qrow0 + r) * 128 + c * 8));
          sts128(sQ + kmajor_chunk(M, r, c), v);
        }
      }
      const int stg = j % NS;
      if (!wait_or_abort(sm, p, &sm.e_full[stg], (uint32_t)((j / NS) & 1), 6)) break;
      if (ct == 0) TC_STAMP(11, j);
      const int valid = min(TILE, ts.seg.t_end - ts.t0);
      const int bad = sm.bad[stg];
      const uint32_t k8 = sbase + (uint32_t)stg * SH::kStageBytes, v8 = k8 + TILE * kRowBytes;
      const uint32_t k16 = sK16, v16 = sV16 + (uint32_t)bi * SH::kF16Bytes;
      // K of tile j into f16 once S of tile j - 1 (the last reader of the
      // buffer) is done; V once P V of tile j - 2 is done
      if (j >= 1 && !ts.first() &&
          !wait_or_abort(sm, p, &sm.s_full[(j - 1) & 1], (uint32_t)(((j - 1) >> 1) & 1), 4))
        break;
#pragma unroll 2
      for (int u = 0; u < TILE / 16; ++u) {
        const int qi = ct + 128 * u;
        const int t = qi % TILE, c = qi / TILE;   // token, 16-byte chunk of its e4m3 row
        const uint4 kw = lds128(k8 + (uint32_t)t * kRowBytes + ((uint32_t)(c ^ (t & 7)) << 4));
        const uint2 k0 = mma::widen8x4<FD_E4M3, false>(kw.x), k1 = mma::widen8x4<FD_E4M3, false>(kw.y);
        const uint2 k2 = mma::widen8x4<FD_E4M3, false>(kw.z), k3 = mma::widen8x4<FD_E4M3, false>(kw.w);
        sts128(k16 + kmajor_chunk(TILE, t, 2 * c), make_uint4(k0.x, k0.y, k1.x, k1.y));
        sts128(k16 + kmajor_chunk(TILE, t, 2 * c + 1), make_uint4(k2.x, k2.y, k3.x, k3.y));
      }
      if (ct == 0) {
        sm.fbad[j & 3] = bad;
        sm.tfirst[j & 3] = ts.first() ? 1 : 0;
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.k_full[bi]);
      if (!wait_or_abort(sm, p, &sm.done[bi], (uint32_t)(((j >> 1) & 1) ^ 1), 4)) break;
      TC_STAMP(10, j - 2);
#pragma unroll 2
      for (int u = 0; u < TILE / 16; ++u) {
        const int qi = ct + 128 * u;
        const int t = qi % TILE, c = qi / TILE;
        uint4 va = make_uint4(0, 0, 0, 0), vb = make_uint4(0, 0, 0, 0);
        if (!bad && t < valid) {
          const uint4 vw = lds128(v8 + (uint32_t)t * kRowBytes + ((uint32_t)(c ^ (t & 7)) << 4));
          const uint2 v0 = mma::widen8x4<FD_E4M3, false>(vw.x), v1 = mma::widen8x4<FD_E4M3, false>(vw.y);
          const uint2 v2 = mma::widen8x4<FD_E4M3, false>(vw.z), v3 = mma::widen8x4<FD_E4M3, false>(vw.w);
          va = make_uint4(v0.x, v0.y, v1.x, v1.y);
          vb = make_uint4(v2.x, v2.y, v3.x, v3.y);
        }
        sts128(v16 + vmn_chunk(TILE, t, 2 * c), va);
        sts128(v16 + vmn_chunk(TILE, t, 2 * c + 1), vb);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sm.e_empty[stg]);
        mbar_arrive(&sm.v_full[bi]);
      }
      if (ct == 0) TC_STAMP(0, j);
      ts.next(p, TILE);
      ++j;
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    // One thread issues S and P V products as their inputs become ready,
    // polling the barriers without blocking (S runs at most two tiles ahead,
    // bounded by the two S buffers and the two f16 buffers).
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_f16(M, TILE, 0);
      constexpr uint32_t id_o = idesc_f16(M, 128, 1);
      const uint32_t tS = tbase, tO = tbase + 2 * TILE;
      // the CTA's tile count; whether a tile starts a segment comes from the
      // converters (slot j mod 4, written before the tile's K is released)
      int ntiles = 0;
      {
        SegmentIter it;
        it.init(p, plan);
        Segment sg;
        while (it.next(p, sg)) ntiles += (sg.t_end - sg.t_begin + TILE - 1) / TILE;
      }
      // descriptors: one Q and one K buffer for S; P and V by tile parity.
      // A descriptor's low field is the address / 16, so an operand offset
      // inside shared memory (below 256 KB) is added as offset / 16.
      const uint64_t dq = sdesc(sQ, 0, 1024), dk = sdesc(sK16, 0, 1024);
      const uint64_t dp = sdesc(sP, 0, 1024), dv = sdesc(sV16, TILE * 128u, 1024);
      int js = 0, jp = 0, kb = -1;
      unsigned long long t_prog = 0;
      uint32_t spins = 0;
      while (jp < ntiles) {
        bool prog = false;
        if (js < ntiles && mbar_test(&sm.k_full[js & 1], (uint32_t)((js >> 1) & 1)) &&
            mbar_test(&sm.s_free[js & 1], (uint32_t)(((js >> 1) & 1) ^ 1))) {
          TC_STAMP(1, js);
          tc_fence_after();
          const uint32_t ds = tS + (uint32_t)(js & 1) * TILE;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            umma(ds, dq + (((ks >> 2) * M * 128 + (ks & 3) * 32) >> 4),
                 dk + (((ks >> 2) * TILE * 128 + (ks & 3) * 32) >> 4), id_s, ks > 0);
          umma_commit(&sm.s_full[js & 1]);
          TC_STAMP(2, js);
          ++js;
          prog = true;
        }
        if (jp < js) {
          const bool first = *(volatile int*)&sm.tfirst[jp & 3] != 0;
          if ((!first || kb < 0 || mbar_test(&sm.o_free, (uint32_t)(kb & 1))) &&
              mbar_test(&sm.p_full[jp & 1], (uint32_t)((jp >> 1) & 1)) &&
              mbar_test(&sm.v_full[jp & 1], (uint32_t)((jp >> 1) & 1))) {
            if (first) ++kb;
            TC_STAMP(8, jp);
            tc_fence_after();
            const uint64_t dpj = dp + (((jp & 1) * SH::kPBytes) >> 4);
            const uint64_t dvj = dv + (((jp & 1) * SH::kF16Bytes) >> 4);
#pragma unroll
            for (int ks = 0; ks < TILE / 16; ++ks)
              umma(tO, dpj + (((ks >> 2) * M * 128 + (ks & 3) * 32) >> 4), dvj + ((ks * 2048) >> 4),
                   id_o, !(first && ks == 0));
            umma_commit(&sm.done[jp & 1]);
            TC_STAMP(9, jp);
            ++jp;
            prog = true;
          }
        }
        if (prog) {
          spins = 0;
        } else if ((++spins & 1023u) == 0) {
          // no progress for a while: bounded like every other wait
          const unsigned long long now = mma::global_ns();
          if (spins == 1024) t_prog = now;
          if (aborted(sm)) break;
          if (now - t_prog > p.wait_ns) {
            record_abort(sm, p, 7);
            break;
          }
        }
      }
      // every issued product done before the tensor memory is freed
      umma_commit(&sm.fin);
      if (!mbar_wait(&sm.fin, 0, mma::kDrainNs)) raise_error(p.ws, kErrDrain, 10);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    // M = 128: thread = one row (tensor-memory lane); M = 64: lanes l and
    // l + 16 hold the two halves of row l of the warp's 16 rows.
    const int row = M == 128 ? 32 * warp + lane : 16 * warp + (lane & 15);
    const int half = M == 128 ? 0 : lane >> 4;
    const int colbase = half * kCols;            // first token of this thread's scores
    const bool vrow = row < R;
    const bool warp_rows = (M == 128 ? 32 * warp : 16 * warp) < R;
    const uint32_t tl = tbase + ((uint32_t)(32 * warp) << 16);
    const uint32_t tS = tl, tO = tl + 2 * TILE;
    int cut = 0;
    if constexpr (CAUSAL) cut = p.q_len - 1 - row % p.q_len;
    TileSeq ts;
    ts.init(p, plan);
    int j = 0;
    float m_ref = -INFINITY, l = 0.f, sc = 0.f, vsc = 0.f;
    while (ts.have) {
      const Segment& seg = ts.seg;
      const bool first = ts.first(), last = ts.last(TILE);
      if (first) {
        const int bq = seg.s / p.hg;
        const int kvh = seg.s - bq * p.hg;
        sc = p.score_scale;
        vsc = p.v_scale;
        if (p.scale_kind == FD_SCALE_HEAD) {
          sc *= __ldg(p.k_scales + kvh);
          vsc *= __ldg(p.v_scales + kvh);
        }
        m_ref = -INFINITY;
        l = 0.f;
      }
      const int sb = j & 1;
      if (!wait_or_abort(sm, p, &sm.s_full[sb], (uint32_t)((j >> 1) & 1), 11)) break;
      if (warp == 0 && lane == 0) TC_STAMP(3, j);
      tc_fence_after();
      float s[kCols];
      if (warp_rows) {
        float x0[32], x1[32];
        tmem_ld32<M>(tS + (uint32_t)sb * TILE, x0);
        tmem_ld32<M>(tS + (uint32_t)sb * TILE + 32, x1);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          s[i] = x0[i];
          s[32 + i] = x1[i];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.s_free[sb]);
      if (warp == 0 && lane == 0) TC_STAMP(4, j);
      // valid keys of this row among the tile's tokens, in this thread's columns
      int lim = *(volatile int*)&sm.fbad[j & 3] ? 0 : min(TILE, seg.t_end - ts.t0);
      if constexpr (CAUSAL) lim = min(lim, seg.T - cut - ts.t0);
      lim -= colbase;
      // row maximum of sc * s over the valid keys (sc may be negative: then
      // the minimum of s)
      float mt;
      {
        const float sg = sc >= 0.f ? 1.f : -1.f;
        float mx[2] = {-INFINITY, -INFINITY};
        if (lim >= kCols) {
#pragma unroll
          for (int i = 0; i < kCols; ++i) mx[i & 1] = fmaxf(mx[i & 1], sg * s[i]);
        } else {
#pragma unroll
          for (int i = 0; i < kCols; ++i) mx[i & 1] = fmaxf(mx[i & 1], i < lim ? sg * s[i] : -INFINITY);
        }
        const float smax = fmaxf(mx[0], mx[1]);
        mt = smax == -INFINITY ? -INFINITY : smax * fabsf(sc);
      }
      if constexpr (M == 64) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
      float fac = 1.f;
      bool resc = false;
      if (first) {
        m_ref = mt;
      } else if (mt > m_ref + 8.f) {
        if (m_ref == -INFINITY) {
          m_ref = mt;   // nothing accumulated yet: O holds zeros
        } else {
          fac = exp2f(m_ref - mt);
          m_ref = mt;
          l *= fac;
          resc = true;
        }
      }
      if (!vrow) resc = false;
      // P = 2^(sc s - m_ref) in f16 (at most 2^8), and the row sum
      uint32_t pk[kCols / 2];
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
      const bool live = m_ref != -INFINITY;
      const float nm = live ? -m_ref : 0.f;
      if (live && lim >= kCols) {
#pragma unroll
        for (int i = 0; i < kCols; i += 2) {
          const float p0 = fast_exp2(fmaf(s[i], sc, nm)), p1 = fast_exp2(fmaf(s[i + 1], sc, nm));
          ps[(i >> 1) & 3] += p0 + p1;
          pk[i / 2] = pack_half2(p0, p1);
        }
      } else {
#pragma unroll
        for (int i = 0; i < kCols; i += 2) {
          float p0 = fast_exp2(fmaf(s[i], sc, nm)), p1 = fast_exp2(fmaf(s[i + 1], sc, nm));
          if (!live || i >= lim) p0 = 0.f;
          if (!live || i + 1 >= lim) p1 = 0.f;
          ps[(i >> 1) & 3] += p0 + p1;
          pk[i / 2] = pack_half2(p0, p1);
        }
      }
      float psum = (ps[0] + ps[1]) + (ps[2] + ps[3]);
      if constexpr (M == 64) psum += __shfl_xor_sync(0xffffffffu, psum, 16);
      l += psum;
      if (warp == 0 && lane == 0) TC_STAMP(5, j);
      // this P buffer is free once P V of tile j - 2 is done
      if (j > 1 && !wait_or_abort(sm, p, &sm.done[j & 1], (uint32_t)(((j >> 1) & 1) ^ 1), 13))
        break;
      if (__any_sync(0xffffffffu, resc)) {
        // O holds P V of tile j - 1 before it is rescaled
        if (!wait_or_abort(sm, p, &sm.done[(j - 1) & 1], (uint32_t)(((j - 1) >> 1) & 1), 14))
          break;
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < (M == 128 ? 128 : 64); c0 += 32) {
          float o[32];
          tmem_ld32<M>(tO + (uint32_t)c0, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= fac;
          tmem_st32<M>(tO + (uint32_t)c0, o);
        }
        tmem_wait_st();
      }
      // this thread's scores are the K-block `half` of row `row` of P
#pragma unroll
      for (int c = 0; c < 8; ++c)
        sts128(sP + (uint32_t)(j & 1) * SH::kPBytes + kmajor_chunk(M, row, 8 * half + c),
               make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]));
      if (warp == 0 && lane == 0) TC_STAMP(6, j);
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.p_full[j & 1]);
      if (warp == 0 && lane == 0) TC_STAMP(7, j);
      if (last) {
        // the segment's output: O after P V of this tile
        if (!wait_or_abort(sm, p, &sm.done[j & 1], (uint32_t)((j >> 1) & 1), 15)) break;
        tc_fence_after();
        const int bq = seg.s / p.hg;
        const long long qrow0 = (long long)bq * p.num_q_heads + (long long)(seg.s - bq * p.hg) * R;
        const float rs = l > 0.f ? vsc / l : 0.f;
        // M = 128: columns [c0, c0 + 32); M = 64: [64 half + c0, + 32)
#pragma unroll 1
        for (int c0 = 0; c0 < (M == 128 ? 128 : 64); c0 += 32) {
          float o[32];
          if (warp_rows) {
            tmem_ld32<M>(tO + (uint32_t)c0, o);
            tmem_wait_ld();
          }
          if (!vrow) continue;
          const int d0 = (M == 128 ? 0 : 64 * half) + c0;
          if (seg.complete) {
            __half* op = static_cast<__half*>(p.out) + (qrow0 + row) * 128 + d0;
#pragma unroll
            for (int i = 0; i < 32; i += 8)
              *reinterpret_cast<uint4*>(op + i) =
                  make_uint4(pack_half2(o[i] * rs, o[i + 1] * rs), pack_half2(o[i + 2] * rs, o[i + 3] * rs),
                             pack_half2(o[i + 4] * rs, o[i + 5] * rs), pack_half2(o[i + 6] * rs, o[i + 7] * rs));
          } else {
            float* pa = p.part_acc + ((long long)seg.slot * p.hq + row) * 128 + d0;
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4*>(pa + i) = make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.o_free);
        if (vrow && half == 0) {
          if (seg.complete) {
            if (p.lse) p.lse[qrow0 + row] = l > 0.f ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
          } else {
            p.part_ml[(long long)seg.slot * p.hq + row] = make_float2(m_ref, l);
          }
        }
      }
      ts.next(p, TILE);
      ++j;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase),
                 "r"(SH::kTmemCols)
                 : "memory");
  }
}

template <int M, bool CAUSAL>
cudaError_t launch_m(const Params& p, const CUtensorMap& mk, const CUtensorMap& mv,
                     cudaStream_t stream) {
  constexpr uint32_t smem = TcShape<M>::kSmem;
  static std::atomic<unsigned long long> limit_set{0};
  cudaError_t e = ensure_smem_limit(tc_split_kernel<M, CAUSAL>, (int)smem, &limit_set);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.grid);
  cfg.blockDim = dim3(kThreadsTC);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, tc_split_kernel<M, CAUSAL>, p, mk, mv);
}

}  // namespace
}  // namespace tc

#ifdef FD_STAMPS
cudaError_t read_tc_stamps(unsigned long long* host, int n) {
  if (n > kStampCtas * kStampSlots) n = kStampCtas * kStampSlots;
  return cudaMemcpyFromSymbol(host, tc::g_tc_stamps, sizeof(unsigned long long) * n);
}
#endif

bool tc_supports(int group, int head_dim, int q_dtype, int kv_dtype, int paged, int page_size,
                 bool token_scales) {
  if (q_dtype != FD_F16 || kv_dtype != FD_E4M3 || head_dim != 128 || token_scales) return false;
  if (group <= 16 || group > 128) return false;
  // a TMA box of page rows must fill whole 1024-byte swizzle atoms
  if (paged && (page_size < 8 || page_size > 256)) return false;
  return true;
}

// Plan shape: one KV head per stream; 128-token tiles for groups of up to 64
// rows (M = 64), else 64; a segment start costs about what streaming 128 KB
// takes per SM.
void tc_config(int group, int sms, int* hc, int* tile, int* grid, int* seg_units) {
  const int t = group <= 64 ? tc::TcShape<64>::kTile : tc::TcShape<128>::kTile;
  const int stage = 2 * t * (int)tc::kRowBytes;
  *hc = 1;
  *tile = t;
  *grid = sms;
  *seg_units = (131072 + stage - 1) / stage;
}

cudaError_t launch_split_tc(const Params& p, const CUtensorMap& mk, const CUtensorMap& mv,
                            cudaStream_t stream) {
  if (p.hc != 1 || p.hq > 128 || p.hq <= 16) return cudaErrorInvalidValue;
  if (p.hq <= 64) {
    if (p.tile != tc::TcShape<64>::kTile) return cudaErrorInvalidValue;
    return p.q_len > 1 ? tc::launch_m<64, true>(p, mk, mv, stream)
                       : tc::launch_m<64, false>(p, mk, mv, stream);
  }
  if (p.tile != tc::TcShape<128>::kTile) return cudaErrorInvalidValue;
  return p.q_len > 1 ? tc::launch_m<128, true>(p, mk, mv, stream)
                     : tc::launch_m<128, false>(p, mk, mv, stream);
}

}  // namespace fd
