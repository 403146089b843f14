// fd_split_mma.cuh -- split (partial attention) kernel on tensor cores, fed by
// TMA through a multi-stage shared-memory pipeline; included by one
// translation unit per cache format (fd_split_mma_*.cu), which instantiate
// its variants, and by fd_split_mma.cu (shapes, tensor maps, dispatch).
//
// What it computes is the same online softmax state as the CUDA-core kernel
// (running max m in log2 units, running sum l, rescaled V accumulator) for
// each segment of the stream-K split plan: the online softmax loop of
// "SGLang Prefill optimisation: dissecting FlashAttention kernel bottlenecks
// with GPU Trace", section 2.2, with one query row per head.  One pass over
// a KV tile serves all query heads of its group ("Learn CUDA from scratch,
// chapter 15", section 15.12), and FP8 K/V are converted inside the load
// path ("From SGLang kernel source to GPU trace: DeepSeek V4.1
// Flash-Decode", section 2.2).
//
// Work split inside a CTA (one persistent CTA per SM, 9 warps):
//  - warp 8 is the producer: it walks the CTA's tiles, stages the current
//    sequence's block-table entries in shared memory (one parallel load per
//    window of 256 pages), and its lane 0 issues, per stage, TMA tensor loads
//    of the K and V rows of `tile` tokens for the stream's hc KV heads into
//    shared memory (128-byte swizzle, or 64-byte for 64-byte rows),
//    completing on the stage's "full" mbarrier, as soon as all consumer warps
//    have released the stage on its "empty" mbarrier;
//  - consumer warp w (0..7) owns head tile w / wph (16 query heads of one KV
//    head) and the w % wph-th run of 16 * r tokens of every stage.  The head
//    tile's Q fragments sit in shared memory for the whole segment (nine
//    warps leave at most 168 registers per thread).
//    Per 16-token sub-tile it computes S = Q K^T with m16n8k16 MMAs (query
//    heads are the M rows, tokens the N columns, head dims the K depth),
//    the online softmax update in registers, and O += P V with P taken
//    straight from the S accumulators (tokens become the K depth), then
//    releases the stage on its "empty" mbarrier.
// 8-bit codes (FP8 e4m3, or INT8 as in the KV quantisation of "Learn CUDA
// from scratch, chapter 15", section 15.11) are widened exactly to f16 (or
// bf16) pairs in registers right before the MMAs.  The head-dim order inside each MMA is permuted consistently on Q and
// K (a dot product does not depend on it), and the token and head-dim orders
// of the V operand are chosen so that every shared-memory load is a 16-byte,
// bank-conflict-free access under the TMA swizzle.
//
// Every wait is bounded (about one second); on expiry the kernel records
// kErrTimeout, stops issuing copies, drains the copies it issued and exits.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <type_traits>

#include "fd_common.cuh"

namespace fd {
namespace mma {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;   // + one producer warp
constexpr int kPageWindow = 256;   // block-table entries staged per window
constexpr int kMaxStages = 8;
constexpr int kSmemBudget = 225 * 1024;
// Bound of the exit drain (waits for copies already issued); unlike the
// pipeline waits it is never shortened.
constexpr unsigned long long kDrainNs = 1000000000ull;

struct Shape {
  int mt;            // 16-row head tiles per KV head (power of two)
  int hc;            // KV heads per stream
  int wph;           // consumer warps per head tile
  int r;             // consumer sub-tiles (32 tokens for FP8, 16 for 16-bit KV) per warp per stage
  int tile;          // tokens per stage = sub-tile tokens * wph * r
  int box_rows;      // rows per TMA box
  int row_bytes;     // bytes of one swizzled row of a box (128 or 64)
  int nx;            // boxes across head_dim (head_dim * elem / row_bytes)
  int region_bytes;  // tile * row_bytes; a stage holds K then V, each as
                     // [nx][hc][tile][row_bytes] regions
  int kv_bytes;      // K (or V) bytes of one stage = hc * nx * region_bytes
  int heads_box;     // 1: one TMA box covers all hc heads of a tile
  int scale_tma;     // 1: per-token scales come by TMA (else by 4-byte cp.async)
  int gather;        // 1: K/V rows gathered by the producer warp with 16-byte cp.async
                     // (pages too small for a TMA box to start on a swizzle atom)
  int flip;          // 1: the kernel's FLIP form (tokens as the MMA's M) serves
                     // one-token queries of this shape
  int stages;
  int merge_in_stage;   // 1: the warps of a head tile merge in the stage of the segment's last tile
  int merge_bytes;      // a dedicated merge area (wph > 1 and no stage is large enough)
  int qfrag_bytes;
  int qrows;         // Q rows kept per head tile: 16, or 8 when no tile has more (see make_shape)
  int scale_bytes;   // per stage with per-token scales: K then V scales, each [tile][hc] fp32
  int smem_bytes;
};

__host__ __device__ inline int next_pow2(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

inline Shape make_shape(int group, int num_kv_heads, int head_dim, int kv_dtype, int page_size,
                        bool token_scales) {
  Shape s;
  const int elem = kv_elem_bytes(kv_dtype);
  s.mt = next_pow2((group + 15) / 16);
  int hc = kConsumerWarps / s.mt;
  while (hc > 1 && num_kv_heads % hc != 0) hc >>= 1;
  s.hc = hc;
  s.wph = kConsumerWarps / (s.mt * s.hc);
  const int row_elems_bytes = head_dim * elem;
  s.row_bytes = row_elems_bytes >= 128 ? 128 : 64;
  s.nx = row_elems_bytes / s.row_bytes;
  const int sub = elem == 1 ? 32 : 16;   // tokens per consumer sub-tile (matches the kernel)
  const int per_subtile = sub * s.wph * s.hc * row_elems_bytes * 2;   // K+V bytes per r step
  s.r = 65536 / per_subtile;
  if (s.r < 1) s.r = 1;
  if (s.r > 4) s.r = 4;
  while (s.r > 1 && sub * s.wph * s.r > 256) s.r >>= 1;   // TMA box height <= 256
  s.tile = sub * s.wph * s.r;
  s.box_rows = page_size > 0 && page_size < s.tile ? page_size : s.tile;
  s.region_bytes = s.tile * s.row_bytes;
  // a TMA box must land on a whole swizzle atom (1024 bytes) of shared memory
  s.gather = page_size > 0 && (s.box_rows * s.row_bytes) % 1024 != 0 ? 1 : 0;
  s.heads_box = 0;   // decided at launch (needs a tensor map over {dims, rows, heads})
  s.scale_tma = 0;   // decided at launch (needs a tensor map over the scale arrays)
  s.kv_bytes = s.hc * s.nx * s.region_bytes;
  // the segment-end merge of a head tile's warps stages 16 rows of every
  // consumer warp's output state: in the stage holding the segment's last
  // tile when it is large enough (its release is held until the merge is
  // done), else in an area of its own
  const int merge_need = kConsumerWarps * 16 * head_dim * 4;
  s.merge_in_stage = s.wph > 1 && 2 * s.kv_bytes >= merge_need ? 1 : 0;
  s.merge_bytes = s.wph > 1 && !s.merge_in_stage ? merge_need : 0;
  // One Q fragment set per head tile.  With at most 8 query heads per KV
  // head, rows 8..15 of every tile are zero: only rows 0..7 are kept (a
  // third stage beside the per-token scale areas; room for the combine's
  // CTA beside the split kernel's on the 64/8-head shape).
  (void)token_scales;
  s.qrows = group <= 8 ? 8 : 16;
  s.flip = head_dim == 128 && group <= 8 && s.wph == 1 ? 1 : 0;
  s.qfrag_bytes = s.mt * s.hc * (head_dim / 16) * (s.qrows == 8 ? 256 : 512);
  s.scale_bytes = token_scales ? 2 * s.hc * s.tile * 4 : 0;
  int st = (kSmemBudget - 1024 - s.merge_bytes - s.qfrag_bytes) / (2 * s.kv_bytes + s.scale_bytes);
  if (st > kMaxStages) st = kMaxStages;
  s.stages = st;
  s.smem_bytes = 1024 + st * (2 * s.kv_bytes + s.scale_bytes) + s.merge_bytes + s.qfrag_bytes;
  return s;
}

// ---------------------------------------------------------------------------
// PTX wrappers: mbarrier, TMA, MMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait on a barrier phase bounded by limit_ns; false on expiry.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 255u) == 0 && global_ns() - t0 > limit_ns) return false;
  }
}

// TMA 3-D tile load into shared memory, completing on an mbarrier, with an
// L2 cache policy (createpolicy) for the copied lines.
__device__ __forceinline__ void tma_load_3d_hint(void* dst, const CUtensorMap* map, int c0, int c1,
                                                 int c2, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)),
      "l"(policy)
      : "memory");
}

// TMA 2-D tile load into shared memory, completing on an mbarrier.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// 16-byte asynchronous global -> shared copy, cached in L2 only.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}

// 4-byte asynchronous global -> shared copy; src_bytes 0 writes zero.
__device__ __forceinline__ void cp_async4(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* a) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
}

__device__ __forceinline__ void prefetch_l2_keep(const void* a) {
  asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(a));
}

// Start-up, before the plan: pulls the index array the producer reads right
// after the plan (the block table, or kv_start) into L2, a slice per CTA.
// Tables above 4 MB are left to the producer's own loads.
__device__ __forceinline__ void prefetch_index_arrays(const Params& p) {
  const char* a = p.block_table ? reinterpret_cast<const char*>(p.block_table)
                                : reinterpret_cast<const char*>(p.kv_start);
  const size_t bytes = p.block_table ? (size_t)p.batch * (size_t)p.bt_stride * 4u
                                     : (size_t)p.batch * 4u;
  if (bytes > ((size_t)4 << 20)) return;
  const size_t lines = (bytes + 127) / 128;
  for (size_t l = (size_t)blockIdx.x * blockDim.x + threadIdx.x; l < lines;
       l += (size_t)gridDim.x * blockDim.x)
    prefetch_l2(a + l * 128);
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

template <bool BF16>
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (BF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7},"
        " {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7},"
        " {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// A fragment of k-step kk of this lane's head tile: rows r and r + 8 (QROWS
// 16), or row r with zeros for the absent rows 8..15 (QROWS 8).
template <int QROWS>
__device__ __forceinline__ uint4 load_qfrag(uint32_t qf, int kk) {
  if constexpr (QROWS == 16) {
    return lds128(qf + kk * 512);
  } else {
    const uint2 h = lds64(qf + kk * 256);
    return make_uint4(h.x, 0u, h.y, 0u);
  }
}

// Two e4m3 codes (low byte first) -> two f16 (or bf16) in one register, exact.
template <bool BF16>
__device__ __forceinline__ uint32_t widen_e4m3x2(uint32_t pair16) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(pair16 & 0xffffu),
                                              __NV_E4M3);
  if constexpr (BF16) {
    float2 f = __half22float2(*reinterpret_cast<__half2*>(&h));
    __nv_bfloat162 b = __float22bfloat162_rn(f);
    return *reinterpret_cast<uint32_t*>(&b);
  } else {
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// Two int8 codes (low byte first) -> two f16 (or bf16) in one register, exact.
// f16: each biased byte u = code + 128 becomes the low mantissa byte of 1024.0
// (exponent-bias construction: the half reads 1024 + u), then one packed
// subtraction of 1152 leaves the codes.  bf16 has too few mantissa bits for
// that; it goes through exact fp32 values.
template <bool BF16>
__device__ __forceinline__ uint32_t widen_i8x2(uint32_t pair16) {
  if constexpr (BF16) {
    __nv_bfloat162 b = __floats2bfloat162_rn(i8_to_f32(pair16), i8_to_f32(pair16 >> 8));
    return *reinterpret_cast<uint32_t*>(&b);
  } else {
    const uint32_t biased = __byte_perm(pair16 ^ 0x8080u, 0x64u, 0x4140);
    __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&biased), __half2half2(__ushort_as_half(0x6480)));
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// Four 8-bit codes of the cache format KVT (one word, low byte first) -> two
// registers of f16 (or bf16) pairs: bytes 0, 1 in .x and bytes 2, 3 in .y,
// exact.  For int8 with f16 the sign flip of all four bytes is one XOR and
// each pair is one byte permutation into 1024.0 patterns plus one packed
// subtraction (see widen_i8x2).
template <int KVT, bool BF16>
__device__ __forceinline__ uint2 widen8x4(uint32_t w) {
  if constexpr (KVT == FD_I8 && !BF16) {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t lo = __byte_perm(u, 0x64u, 0x4140), hi = __byte_perm(u, 0x64u, 0x4342);
    const __half2 bias = __half2half2(__ushort_as_half(0x6480));
    __half2 a = __hsub2(*reinterpret_cast<const __half2*>(&lo), bias);
    __half2 b = __hsub2(*reinterpret_cast<const __half2*>(&hi), bias);
    return make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
  } else if constexpr (KVT == FD_I8) {
    return make_uint2(widen_i8x2<BF16>(w), widen_i8x2<BF16>(w >> 16));
  } else {
    return make_uint2(widen_e4m3x2<BF16>(w), widen_e4m3x2<BF16>(w >> 16));
  }
}

// Four int8 codes -> two registers of f16 pairs holding code + 1152 (the
// sign flip and byte permutation of widen8x4 without its subtraction).  The
// FLIP form with f16 queries feeds K and V this way: a second product per
// 16-dim k-step takes K's bias back out of the scores, and 1152 times the
// sub-tile's probability sums leave the O^T accumulator after its products.
__device__ __forceinline__ uint2 widen_i8x4_biased(uint32_t w) {
  const uint32_t u = w ^ 0x80808080u;
  return make_uint2(__byte_perm(u, 0x64u, 0x4140), __byte_perm(u, 0x64u, 0x4342));
}

// FLIP form, head_dim 128: head dim of row r of the O^T accumulator's
// m-tile j (row r + 8 is the next dim).  8-bit caches: 16 r + 2 j (a lane's
// V bytes are one 16-byte chunk); 16-bit caches: 64 (j / 4) + 8 r + 2 (j % 4)
// (one 16-byte chunk of each 128-byte region).
template <int ELEM>
__device__ __forceinline__ int flip_dim(int j, int r) {
  return ELEM == 1 ? 16 * r + 2 * j : 64 * (j >> 2) + 8 * r + 2 * (j & 3);
}

// Transpose of an 8x8 matrix of 16-bit values held one row pair per lane
// (lane l: row l / 4, columns 2 (l % 4) and 2 (l % 4) + 1) into the same
// fragment layout.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_f32x2(float lo, float hi, bool bf16) {
  if (bf16) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&b);
  }
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ---------------------------------------------------------------------------
// Operand layouts (per D and element size)
// ---------------------------------------------------------------------------
// K operand: k-step kk of lane quad position q covers the 4 head dims
// kdim(kk, q) .. +3 (pairs {0,1} -> b0, {2,3} -> b1; Q uses the same dims).
template <int D, int ELEM>
__device__ __forceinline__ int kdim(int kk, int q) {
  if constexpr (D == 128 && ELEM == 1) return 32 * q + 4 * kk;
  else if constexpr (D == 128 && ELEM == 2) return (kk >> 2) * 64 + 16 * q + 4 * (kk & 3);
  else return 16 * q + 4 * kk;
}

// V operand / O accumulator: n-tile j, column n <-> head dim vdim(j, n).
template <int D, int ELEM>
__device__ __forceinline__ int vdim(int j, int n) {
  if constexpr (D == 128 && ELEM == 1) return 16 * n + j;
  else if constexpr (D == 128 && ELEM == 2) return j < 8 ? 8 * n + j : 64 + 8 * n + (j - 8);
  else return 8 * n + j;
}

// Byte address of 16-byte chunk c of row tt in a swizzled box region.
__device__ __forceinline__ uint32_t chunk_addr(uint32_t region, int tt, int c, int row_bytes) {
  const int swz = row_bytes == 128 ? (tt & 7) : ((tt >> 1) & 3);
  return region + tt * row_bytes + ((c ^ swz) << 4);
}

// V rows of tokens past a segment's end are whatever the stage held (a
// skipped box, a page tail, a gap between sequences): they may hold NaN or
// Inf bit patterns, and 0 * NaN would poison the accumulator, so their words
// are zeroed before the P V product.  w0..w3 are the rows of sub-tile tokens
// tk, tk + 1, tk + 8, tk + 9; `left` tokens of the sub-tile are valid.
template <typename W>
__device__ __forceinline__ void zero_rows_past_end(W& w0, W& w1, W& w2, W& w3, int tk, int left) {
  if (tk >= left) w0 = W{};
  if (tk + 1 >= left) w1 = W{};
  if (tk + 8 >= left) w2 = W{};
  if (tk + 9 >= left) w3 = W{};
}

#ifdef FD_STAMPS
// (one array per translation unit that instantiates kernels)
// 0 entry, 1 plan done, 2 first copy issued, 3 first stage landed (warp 0),
// 4 last stage released (warp 0), 5 last segment stored (warp 0), 6 exit,
// 7 stages consumed by warp 0, 8 plan total known, 9 producer has its first
// segment, 10 producer has the segment's row data, 11 before the plan,
// 13-15 segment-end merge of a head tile's warps (stage read, states
// staged, merged), 20 the SM's id
namespace {
FD_STAMP_ARRAY(g_split_stamps);
}
#endif

// Float4 chunk c of row x of a warp's area in the segment-end merge: an XOR
// swizzle within each group of 8 chunks, so that the 8 lanes of a quarter
// warp storing their fragments (rows r, r + 1; chunks 8q + const) and a warp
// reading one row both hit 8 different 16-byte bank groups.
__device__ __forceinline__ uint32_t merge_chunk(int x, int c) {
  return (uint32_t)(c ^ (((x & 1) << 2) | ((c >> 3) & 3)));
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------

struct Shared {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  int bad[kMaxStages];
  int abort_flag;
  long long red[35];
  int pages[kPageWindow];   // producer's window of the current sequence's block table
};

// TOK: per-token K/V scales (fd_scale_kind FD_SCALE_TOKEN).  The producer
// brings each tile's scales into the stage's scale area, [tile][hc] fp32 for K
// then for V: by TMA next to the K/V boxes when the scale arrays allow it
// (counted on the stage's "full" barrier like them), else by 4-byte cp.async
// completing on the same barrier (one more arrival per producer lane).  A
// consumer multiplies each score by its token's K scale and each probability
// by its token's V scale before the P V product (the softmax sum keeps the
// unscaled probabilities).
// FLIP: at most 8 query heads per KV head, one warp per head tile
// (head_dim 128, one query token): the MMAs take tokens as M and the heads
// as N (see the FLIP branch of the sub-tile loop).
template <int KVT, typename QT, int D, bool TOK, int QROWS, bool CAUSAL, bool FLIP = false>
__global__ void __launch_bounds__(kThreads, 1)
    mma_split_kernel(const Params p, const Shape sh, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv,
                     const __grid_constant__ CUtensorMap tmks,
                     const __grid_constant__ CUtensorMap tmvs) {
  constexpr int ELEM = kv_elem_bytes(KVT);
  constexpr bool BF16 = std::is_same<QT, __nv_bfloat16>::value;
  constexpr int KSTEPS = D / 16;
  constexpr int NT = D / 8;     // n-tiles of the PV product
  constexpr int SUB = ELEM == 1 ? 32 : 16;   // tokens per sub-tile (one softmax step)
  constexpr int NJ = SUB / 8;                // n-tiles of the QK product
  extern __shared__ uint8_t dyn_smem[];
  __shared__ Shared sm;

  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  const uint32_t stage0 = smem_u32(base);
  const uint32_t qfrag0 = stage0 + sh.stages * 2 * sh.kv_bytes + sh.merge_bytes;
  float* scl = reinterpret_cast<float*>(base + sh.stages * 2 * sh.kv_bytes + sh.merge_bytes +
                                        sh.qfrag_bytes);   // per-token scales (TOK)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // K/V lines are read once: they leave L2 first (policy made before the plan)
  uint64_t kv_policy;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(kv_policy));
  if (threadIdx.x == 0) FD_STAMP(g_split_stamps, 0, stamp_ns());
#ifdef FD_STAMPS
  if (threadIdx.x == 0) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    FD_STAMP(g_split_stamps, 20, (unsigned long long)smid);
  }
#endif
  if (threadIdx.x == 0) {
    for (int i = 0; i < sh.stages; ++i) {
      // producer lane 0, plus every producer lane when it copies with cp.async
      mbar_init(&sm.full[i], sh.gather || (TOK && !sh.scale_tma) ? 1 + 32 : 1);
      mbar_init(&sm.empty[i], kConsumerWarps);
    }
    sm.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // work that does not need the plan: the tensor-map descriptors and the
  // index array the producer reads first
  if (threadIdx.x == kConsumerWarps * 32 && !sh.gather) {
    prefetch_map(&tmk);
    prefetch_map(&tmv);
  }
  prefetch_index_arrays(p);
  if (threadIdx.x == 0) FD_STAMP(g_split_stamps, 11, stamp_ns());
#ifdef FD_STAMPS
  const PlanResult plan = compute_plan(
      p, sm.red, kThreads, 0,
      blockIdx.x < kStampCtas ? &g_split_stamps[blockIdx.x * kStampSlots + 8] : nullptr);
#else
  const PlanResult plan = compute_plan(p, sm.red, kThreads, 0);
#endif
  if (threadIdx.x == 0) FD_STAMP(g_split_stamps, 1, stamp_ns());
  allow_dependent_launch();
  if (threadIdx.x == kConsumerWarps * 32) FD_STAMP(g_split_stamps, 21, stamp_ns());
  wait_prior_grid();   // a KV append launched just before may still be writing rows
  if (threadIdx.x == kConsumerWarps * 32) FD_STAMP(g_split_stamps, 22, stamp_ns());

  const int S = sh.stages;
  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    // The whole warp walks the CTA's tiles; it stages block-table entries in
    // shared memory with one parallel load per window, and lane 0 issues the
    // TMA copies of each tile as soon as its stage is free.
    // K/V lines are read once: they leave L2 first, before Q rows, index
    // data and partial states

    SegmentIter it;
    it.init(p, plan);
    Segment seg;
    int n = 0;
    bool stop = p.starve != 0;   // test switch: issue nothing, the consumers' waits run out
    long long next_start = -1;   // kv_start of the next segment's sequence, read ahead
    while (!stop && it.next(p, seg)) {
      if (n == 0 && lane == 0) FD_STAMP(g_split_stamps, 9, stamp_ns());
      const int b = seg.s / p.hg;
      const int kvh0 = (seg.s - b * p.hg) * sh.hc;
      // the plan already read the first segment's kv_start, and each
      // segment reads the next one's once its own copies fill the pipeline
      const long long start = p.block_table ? 0
                              : n == 0 && seg.s == plan.s_first && plan.first_start >= 0
                                  ? plan.first_start
                              : next_start >= 0 ? next_start
                                                : (long long)__ldg(p.kv_start + b);
      next_start = -1;
      const int n_seg0 = n;
#ifdef FD_STAMPS
      if (n == 0 && lane == 0 && start >= 0) FD_STAMP(g_split_stamps, 10, stamp_ns());
#endif
      int win_lo = 0, win_hi = 0;   // logical pages [win_lo, win_hi) held in sm.pages
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
          const bool waited = !*(volatile int*)&sm.abort_flag && mbar_wait(&sm.empty[stg], ph ^ 1u, p.wait_ns);
          if (n == 0) FD_STAMP(g_split_stamps, 23, stamp_ns());
          if (!waited) {
            if (!*(volatile int*)&sm.abort_flag) {
              raise_error(p.ws, kErrTimeout, 1);
              *(volatile int*)&sm.abort_flag = 1;
            }
            stop = true;
          } else if (!sh.gather) {
            const int nbox = sh.tile / sh.box_rows;
            uint8_t* kst = base + (size_t)stg * 2 * sh.kv_bytes;
            uint8_t* vst = kst + sh.kv_bytes;
            int bad = 0;
            uint32_t bytes = 0;
            // pass 1: validate rows, count bytes; pass 2: issue
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
                  if (ok && TOK && sh.scale_tma) bytes += 2u * sh.hc * sh.box_rows * 4u;
                  if (!ok) bad = 1;
                  continue;
                }
                if (!ok) continue;
                if (n == 0 && i == 0) FD_STAMP(g_split_stamps, 2, stamp_ns());
                if constexpr (TOK) {
                  if (sh.scale_tma) {   // the box rows' scales of the hc heads
                    float* sk = scl + (size_t)stg * (sh.scale_bytes / 4) +
                                (size_t)i * sh.box_rows * sh.hc;
                    tma_load_2d(sk, &tmks, kvh0, (int)row, &sm.full[stg]);
                    tma_load_2d(sk + sh.hc * sh.tile, &tmvs, kvh0, (int)row, &sm.full[stg]);
                  }
                }
                if (sh.heads_box) {
                  // one box per head-dim slice: all hc heads of the tile's rows
                  for (int x = 0; x < sh.nx; ++x) {
                    const size_t off = (size_t)x * sh.hc * sh.region_bytes;
                    const int xc = x * (sh.row_bytes / ELEM);
                    tma_load_3d_hint(kst + off, &tmk, xc, (int)row, kvh0, &sm.full[stg], kv_policy);
                    tma_load_3d_hint(vst + off, &tmv, xc, (int)row, kvh0, &sm.full[stg], kv_policy);
                  }
                  continue;
                }
                for (int h = 0; h < sh.hc; ++h) {
                  for (int x = 0; x < sh.nx; ++x) {
                    const size_t off = (size_t)(x * sh.hc + h) * sh.region_bytes +
                                       (size_t)i * sh.box_rows * sh.row_bytes;
                    const int xc = x * (sh.row_bytes / ELEM);
                    tma_load_3d_hint(kst + off, &tmk, xc, kvh0 + h, (int)row, &sm.full[stg],
                                     kv_policy);
                    tma_load_3d_hint(vst + off, &tmv, xc, kvh0 + h, (int)row, &sm.full[stg],
                                     kv_policy);
                  }
                }
              }
            }
          }
        }
        stop = __shfl_sync(0xffffffffu, stop, 0);
        if (stop) break;
        if (sh.gather) {
          // every lane copies 16-byte chunks of the tile's rows into the
          // layout the TMA boxes would have written (regions [nx][hc], rows
          // of row_bytes, chunks swizzled); rows outside the cache are
          // recorded and leave the stage marked bad
          const int stg = (int)(n % S);
          uint8_t* kst = base + (size_t)stg * 2 * sh.kv_bytes;
          uint8_t* vst = kst + sh.kv_bytes;
          const int cpr = sh.row_bytes >> 4;              // chunks per row of a region
          const int per_row = sh.hc * sh.nx * cpr;         // chunks of one token, one tensor
          const int lpr = per_row < 32 ? per_row : 32;     // lanes per token
          const int rstep = 32 / lpr;
          const size_t row_stride = (size_t)p.num_kv_heads * D * ELEM;
          bool badrow = false;
          for (int j = lane % lpr; j < per_row; j += lpr) {
            const int c = j % cpr, hx = j / cpr, x = hx % sh.nx, h = hx / sh.nx;
            const size_t col = ((size_t)(kvh0 + h) * D) * ELEM + (size_t)x * sh.row_bytes + (c << 4);
            const size_t dcol = (size_t)(x * sh.hc + h) * sh.region_bytes;
            for (int tt = lane / lpr; tt < valid; tt += rstep) {
              const int t = t0 + tt;
              long long row;
              if (p.block_table) {
                const int page = sm.pages[(t >> p.page_shift) - win_lo];
                row = ((long long)page << p.page_shift) + (t & (p.page_size - 1));
                if (page < 0 || row >= p.kv_rows) {
                  if (!badrow) raise_error(p.ws, kErrBounds, page);
                  badrow = true;
                  continue;
                }
              } else {
                row = start + t;
                if (row < 0 || row >= p.kv_rows) {
                  if (!badrow) raise_error(p.ws, kErrBounds, row);
                  badrow = true;
                  continue;
                }
              }
              const uint32_t swz = sh.row_bytes == 128 ? (tt & 7) : ((tt >> 1) & 3);
              const size_t src = (size_t)row * row_stride + col;
              const size_t dst = dcol + (size_t)tt * sh.row_bytes + ((c ^ swz) << 4);
              const uint8_t* ks = static_cast<const uint8_t*>(p.k) + src;
              const uint8_t* vs = static_cast<const uint8_t*>(p.v) + src;
              // (self-check: 16-byte aligned, inside the stage and the cache)
              if (((reinterpret_cast<uintptr_t>(ks) | reinterpret_cast<uintptr_t>(vs) |
                    reinterpret_cast<uintptr_t>(kst + dst)) & 15u) != 0 ||
                  dst + 16 > (size_t)sh.kv_bytes || src + 16 > (size_t)p.kv_rows * row_stride) {
                if (!badrow) raise_error(p.ws, kErrBounds, (long long)dst);
                badrow = true;
                continue;
              }
              cp_async16(kst + dst, ks);
              cp_async16(vst + dst, vs);
            }
          }
          const bool anybad = __any_sync(0xffffffffu, badrow);
          if (lane == 0) {
            sm.bad[stg] = anybad ? 1 : 0;
            mbar_arrive(&sm.full[stg]);
          }
        }
        if (n == n_seg0 + S - 1) {   // the next copy waits for a released stage anyway
          // the next segment's row data ahead: its kv_start into a register,
          // or its first window of block-table entries into L2
          SegmentIter ahead = it;
          Segment sn;
          if (ahead.next(p, sn)) {
            const int bn = sn.s / p.hg;
            if (!p.block_table) {
              next_start = __ldg(p.kv_start + bn);
            } else {
              const int pg0 = sn.t_begin >> p.page_shift, pg1 = (sn.t_end - 1) >> p.page_shift;
              if (lane < kPageWindow / 32 && pg0 + 32 * lane <= pg1)
                prefetch_l2(p.block_table + (long long)bn * p.bt_stride + pg0 + 32 * lane);
            }
          }
        }
        if (sh.gather || (TOK && !sh.scale_tma)) {
          // the tile's per-token scales of its hc heads, element by element
          // (rows past the end, or outside the cache, read as zero); then
          // every lane's copies complete on the stage's "full" barrier
          const int stg = (int)(n % S);
          float* dk = scl + (size_t)stg * (sh.scale_bytes / 4);
          float* dv = dk + sh.hc * sh.tile;
          for (int idx = lane; TOK && !sh.scale_tma && idx < sh.hc * sh.tile; idx += 32) {
            const int tt = idx / sh.hc, h = idx - tt * sh.hc;
            const int t = t0 + tt;
            long long row = -1;
            if (tt < valid) {
              row = p.block_table
                        ? ((long long)sm.pages[(t >> p.page_shift) - win_lo] << p.page_shift) +
                              (t & (p.page_size - 1))
                        : start + t;
              if (row < 0 || row >= p.kv_rows) row = -1;
            }
            const long long e = row >= 0 ? row * p.num_kv_heads + kvh0 + h : 0;
            cp_async4(dk + idx, p.k_scales + e, row >= 0 ? 4 : 0);
            cp_async4(dv + idx, p.v_scales + e, row >= 0 ? 4 : 0);
          }
          asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(
                           smem_u32(&sm.full[stg]))
                       : "memory");
        }
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (lane == 0 && stop) {
      // drain: copies of the last S issued tiles must land before the CTA
      // exits; a drain that gives up is recorded on its own
      for (int i = n - S < 0 ? 0 : n - S; i < n; ++i)
        if (!mbar_wait(&sm.full[i % S], (uint32_t)((i / S) & 1), kDrainNs))
          raise_error(p.ws, kErrDrain, 3);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int ht = warp / sh.wph, ts = warp - ht * sh.wph;
    const int kvl = ht / sh.mt, mtile = ht - kvl * sh.mt;
    const int r = lane >> 2, q = lane & 3;
    const int G = p.group;
    const QT* qg = static_cast<const QT*>(p.q);
    // local query heads (within the stream) of rows r and r + 8
    const int h0 = mtile * 16 + r, h1 = h0 + 8;
    const bool v0 = h0 < G, v1 = h1 < G;
    // multi-token kernels: rows r and r + 8 (token j of their head) stop
    // q_len - 1 - j keys before the sequence's end
    int cut0 = 0, cut1 = 0;
    if constexpr (CAUSAL) {
      cut0 = p.q_len - 1 - h0 % p.q_len;
      cut1 = p.q_len - 1 - h1 % p.q_len;
    }
    const int li0 = kvl * G + h0, li1 = kvl * G + h1;   // slot rows
    // this head tile's Q fragments in shared memory: [kk][lane] x 16 bytes
    const uint32_t qf = qfrag0 + (uint32_t)ht * KSTEPS * (QROWS * 32) + lane * (QROWS);

    SegmentIter it;
    it.init(p, plan);
    {
      // the Q rows of this head tile for the CTA's later segments, into L2
      // (kept there): a segment start then waits for L2, not for DRAM
      SegmentIter ahead = it;
      Segment sa;
      const int row = lane >> 1, lh = mtile * 16 + row;
      for (int k = 0; k < 8 && ahead.next(p, sa); ++k) {
        if (k == 0 || lh >= G) continue;   // the first segment's Q is loaded next
        const int bs = sa.s / p.hg;
        const long long qr = (long long)bs * p.num_q_heads + (long long)(sa.s - bs * p.hg) * p.hq +
                             kvl * G + lh;
        prefetch_l2_keep(qg + qr * D + (lane & 1) * (D / 2));
      }
    }
    Segment seg;
    int n = 0;
    while (it.next(p, seg)) {
      const int b = seg.s / p.hg;
      const int j = seg.s - b * p.hg;
      const long long qrow0 = (long long)b * p.num_q_heads + j * p.hq;   // first head of stream
      // score and output factors of this warp's KV head (per-KV-head scales)
      float sc = p.score_scale, vsc = p.v_scale;
      if (ELEM == 1 && p.scale_kind == FD_SCALE_HEAD) {   // finer scales: 8-bit caches only
        const int kvh = j * sh.hc + kvl;
        sc *= __ldg(p.k_scales + kvh);
        vsc *= __ldg(p.v_scales + kvh);
      }
      // Q fragments (A operand), head dims permuted as kdim(); every warp of
      // the head tile writes the same values
#pragma unroll
      for (int kk = 0; kk < KSTEPS; ++kk) {
        const int dd = kdim<D, ELEM>(kk, q);   // same dims as the K operand
        uint2 x0 = make_uint2(0, 0), x1 = make_uint2(0, 0);
        if (v0) x0 = __ldg(reinterpret_cast<const uint2*>(qg + (qrow0 + li0) * D + dd));
        if (v1) x1 = __ldg(reinterpret_cast<const uint2*>(qg + (qrow0 + li1) * D + dd));
        if constexpr (QROWS == 8)
          asm volatile("st.shared.v2.u32 [%0], {%1,%2};" ::"r"(qf + kk * 256), "r"(x0.x), "r"(x0.y)
                       : "memory");
        else
          asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(qf + kk * 512), "r"(x0.x),
                       "r"(x1.x), "r"(x0.y), "r"(x1.y)
                       : "memory");
      }
      __syncwarp();
      float o[NT][4];
#pragma unroll
      for (int t = 0; t < NT; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
      float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
      int last_stg = 0;

      for (int t0 = seg.t_begin; t0 < seg.t_end; t0 += sh.tile, ++n) {
        const int stg = (int)(n % S);
        const uint32_t ph = (uint32_t)((n / S) & 1);
        bool ok = !*(volatile int*)&sm.abort_flag;
        if (ok && !mbar_wait(&sm.full[stg], ph, p.wait_ns)) {
          raise_error(p.ws, kErrTimeout, 2);
          *(volatile int*)&sm.abort_flag = 1;
          ok = false;
        }
        if (n == 0 && warp == 0 && lane == 0) FD_STAMP(g_split_stamps, 3, stamp_ns());
        if (ok && !sm.bad[stg]) {
          const uint32_t kreg = stage0 + stg * 2 * sh.kv_bytes + kvl * sh.region_bytes;
          const uint32_t xstride = sh.hc * sh.region_bytes;   // next head-dim slice
          const uint32_t vreg = kreg + sh.kv_bytes;
#pragma unroll 1
          for (int rr = 0; rr < sh.r; ++rr) {
            const int sub = ts * SUB * sh.r + SUB * rr;   // first token of the sub-tile in the tile
            const int left = seg.t_end - (t0 + sub);      // valid tokens from the sub-tile start
            if (left <= 0) break;
            int left0 = left, left1 = left;   // valid keys of rows r and r + 8 (see below)
            if (TOK && p.q_len > 1) {
              const int tail = seg.T - (t0 + sub);
              left0 = min(left, tail - (p.q_len - 1 - h0 % p.q_len));
              left1 = min(left, tail - (p.q_len - 1 - h1 % p.q_len));
            }
            const bool edge = min(left0, left1) < SUB;
            if constexpr (FLIP) {
              // ---- S^T = K Q^T: MT m-tiles of 16 tokens (8-bit: this lane's
              //      tokens r, r + 8, r + 16, r + 24 of the sub-tile; 16-bit:
              //      r, r + 8) by the 8 heads (this lane: heads 2q, 2q + 1).
              //      K is the A operand, from the same row slices as in the
              //      unflipped form (the same head-dim order, kdim); Q of
              //      head r is the B operand (the 8-row fragment store).
              constexpr int MT = SUB / 16;
              float st[MT][4];
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) st[mt][0] = st[mt][1] = st[mt][2] = st[mt][3] = 0.f;
              if constexpr (ELEM == 1) {
                uint32_t w[4][8];
#pragma unroll
                for (int jn = 0; jn < 4; ++jn) {
                  const int tk = sub + 8 * jn + r;
                  const uint4 a0 = lds128(chunk_addr(kreg, tk, 2 * q, sh.row_bytes));
                  const uint4 a1 = lds128(chunk_addr(kreg, tk, 2 * q + 1, sh.row_bytes));
                  w[jn][0] = a0.x; w[jn][1] = a0.y; w[jn][2] = a0.z; w[jn][3] = a0.w;
                  w[jn][4] = a1.x; w[jn][5] = a1.y; w[jn][6] = a1.z; w[jn][7] = a1.w;
                }
                // INT8 cache, f16 queries: K enters as code + 1152, and after
                // each 16-dim k-step a second product with A = -1152 takes
                // that k-step's bias (1152 times the head's Q sum over those
                // dims) back out, so the accumulator never holds more than
                // one k-step's bias
                constexpr bool KFOLD = KVT == FD_I8 && !BF16;
                constexpr uint32_t kNeg1152 = 0xE480E480u;   // f16 pair (-1152, -1152)
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                  const uint2 qb = lds64(qf + kk * 256);
#pragma unroll
                  for (int mt = 0; mt < MT; ++mt) {
                    if constexpr (KFOLD) {
                      const uint2 ka = widen_i8x4_biased(w[2 * mt][kk]);       // token r
                      const uint2 kb = widen_i8x4_biased(w[2 * mt + 1][kk]);   // token r + 8
                      mma16816<false>(st[mt], ka.x, kb.x, ka.y, kb.y, qb.x, qb.y);
                      mma16816<false>(st[mt], kNeg1152, kNeg1152, kNeg1152, kNeg1152, qb.x, qb.y);
                    } else {
                      const uint2 ka = widen8x4<KVT, BF16>(w[2 * mt][kk]);       // token r
                      const uint2 kb = widen8x4<KVT, BF16>(w[2 * mt + 1][kk]);   // token r + 8
                      mma16816<BF16>(st[mt], ka.x, kb.x, ka.y, kb.y, qb.x, qb.y);
                    }
                  }
                }
              } else {   // 16-bit: chunk pairs (2q, 2q + 1) of each 128-byte region
#pragma unroll
                for (int x2 = 0; x2 < D / 64; ++x2) {
                  const uint32_t reg = kreg + x2 * xstride;
                  const uint4 c00 = lds128(chunk_addr(reg, sub + r, 2 * q, sh.row_bytes));
                  const uint4 c01 = lds128(chunk_addr(reg, sub + r, 2 * q + 1, sh.row_bytes));
                  const uint4 c10 = lds128(chunk_addr(reg, sub + r + 8, 2 * q, sh.row_bytes));
                  const uint4 c11 = lds128(chunk_addr(reg, sub + r + 8, 2 * q + 1, sh.row_bytes));
#pragma unroll
                  for (int k4 = 0; k4 < 4; ++k4) {
                    const uint2 qb = lds64(qf + (x2 * 4 + k4) * 256);
                    const uint4 t0 = k4 < 2 ? c00 : c01, t1 = k4 < 2 ? c10 : c11;
                    const uint32_t a0 = (k4 & 1) ? t0.z : t0.x, a2 = (k4 & 1) ? t0.w : t0.y;
                    const uint32_t a1 = (k4 & 1) ? t1.z : t1.x, a3 = (k4 & 1) ? t1.w : t1.y;
                    mma16816<BF16>(st[0], a0, a1, a2, a3, qb.x, qb.y);
                  }
                }
              }
              // ---- online softmax per head: st[mt][e] is token 16 mt + r
              //      (+ 8 for e >= 2) of head 2q + (e & 1); the 8 lanes of a
              //      head (r = 0..7) hold its tokens
              const uint32_t tsk =
                  smem_u32(scl) + 4u * (uint32_t)(stg * (sh.scale_bytes / 4) + sub * sh.hc + kvl);
              const uint32_t tsv = tsk + 4u * (uint32_t)(sh.hc * sh.tile);
              float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                  const int tok = 16 * mt + r + 8 * hf;
                  float ksc = sc;
                  if constexpr (TOK) ksc *= lds_f32(tsk + 4u * (uint32_t)(tok * sh.hc));
                  float va = st[mt][2 * hf] * ksc, vb = st[mt][2 * hf + 1] * ksc;
                  if (edge && tok >= left) va = vb = -INFINITY;
                  st[mt][2 * hf] = va;
                  st[mt][2 * hf + 1] = vb;
                  mx0 = fmaxf(mx0, va);
                  mx1 = fmaxf(mx1, vb);
                }
              }
#pragma unroll
              for (int o2 = 4; o2 < 32; o2 <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o2));
              }
              const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
              const float base0 = mn0 == -INFINITY ? 0.f : mn0;
              const float base1 = mn1 == -INFINITY ? 0.f : mn1;
              const float a0 = fast_exp2(m0 - base0), a1 = fast_exp2(m1 - base1);
              m0 = mn0;
              m1 = mn1;
              float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                  st[mt][2 * hf] = fast_exp2(st[mt][2 * hf] - base0);
                  st[mt][2 * hf + 1] = fast_exp2(st[mt][2 * hf + 1] - base1);
                  ps0 += st[mt][2 * hf];
                  ps1 += st[mt][2 * hf + 1];
                }
              }
              l0 = fmaf(l0, a0, ps0);   // this lane's tokens; the head's 8 lanes add up at the end
              l1 = fmaf(l1, a1, ps1);
              if constexpr (TOK) {   // V scales weight the probabilities, not their sum
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
                  for (int hf = 0; hf < 2; ++hf) {
                    const int tok = 16 * mt + r + 8 * hf;
                    const float vs = tok < left ? lds_f32(tsv + 4u * (uint32_t)(tok * sh.hc)) : 0.f;
                    st[mt][2 * hf] *= vs;
                    st[mt][2 * hf + 1] *= vs;
                  }
                }
              }
              if (!__all_sync(0xffffffffu, a0 == 1.f && a1 == 1.f)) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  o[j][0] *= a0;
                  o[j][1] *= a1;
                  o[j][2] *= a0;
                  o[j][3] *= a1;
                }
              }
              // ---- O^T += V^T P^T, one k-step of 16 tokens (one S^T m-tile)
              //      at a time.  P^T (B operand): the probabilities packed per
              //      token row and transposed by movmatrix, so that this
              //      lane holds tokens 2q, 2q + 1 (+ 8) of head r.  V^T (A
              //      operand): rows r and r + 8 of m-tile j are head dims
              //      flip_dim(j, r) and flip_dim(j, r) + 1, so this lane's V
              //      values are one 16-byte chunk of each of its four token
              //      rows (per 128-byte region).
              // INT8 cache, f16 queries: V enters the products as code + 1152
              // (no subtraction per element); an all-ones row of A sums the
              // packed probabilities of the sub-tile per head in lanes 0..3,
              // and 1152 times that sum leaves O^T after the sub-tile.
              constexpr bool VFOLD = KVT == FD_I8 && !BF16 && ELEM == 1;
              float psum[4] = {0.f, 0.f, 0.f, 0.f};
              const uint32_t ones = r == 0 ? 0x3C003C00u : 0u;   // row 0 of A: 1.0
#pragma unroll
              for (int kt = 0; kt < MT; ++kt) {
                const uint32_t pb0 =
                    movmatrix_trans(pack_f32x2(st[kt][0], st[kt][1], BF16));   // token r
                const uint32_t pb1 =
                    movmatrix_trans(pack_f32x2(st[kt][2], st[kt][3], BF16));   // token r + 8
                if constexpr (VFOLD) mma16816<false>(psum, ones, 0u, ones, 0u, pb0, pb1);
                const int u0 = sub + 16 * kt + 2 * q, u1 = u0 + 1, u2 = u0 + 8, u3 = u0 + 9;
#pragma unroll
                for (int x2 = 0; x2 < (ELEM == 1 ? 1 : D / 64); ++x2) {
                  const uint32_t reg = vreg + x2 * xstride;
                  uint4 w0 = lds128(chunk_addr(reg, u0, r, sh.row_bytes));
                  uint4 w1 = lds128(chunk_addr(reg, u1, r, sh.row_bytes));
                  uint4 w2 = lds128(chunk_addr(reg, u2, r, sh.row_bytes));
                  uint4 w3 = lds128(chunk_addr(reg, u3, r, sh.row_bytes));
                  if (left < SUB) zero_rows_past_end(w0, w1, w2, w3, 16 * kt + 2 * q, left);
                  const uint32_t A[4] = {w0.x, w0.y, w0.z, w0.w}, B[4] = {w1.x, w1.y, w1.z, w1.w};
                  const uint32_t C[4] = {w2.x, w2.y, w2.z, w2.w}, E[4] = {w3.x, w3.y, w3.z, w3.w};
#pragma unroll
                  for (int wd = 0; wd < 4; ++wd) {
                    if constexpr (ELEM == 1) {
                      const uint32_t lo01 = __byte_perm(A[wd], B[wd], 0x5140);
                      const uint32_t hi01 = __byte_perm(A[wd], B[wd], 0x7362);
                      const uint32_t lo89 = __byte_perm(C[wd], E[wd], 0x5140);
                      const uint32_t hi89 = __byte_perm(C[wd], E[wd], 0x7362);
                      uint2 l01, l89, h01, h89;
                      if constexpr (VFOLD) {
                        l01 = widen_i8x4_biased(lo01);
                        l89 = widen_i8x4_biased(lo89);
                        h01 = widen_i8x4_biased(hi01);
                        h89 = widen_i8x4_biased(hi89);
                      } else {
                        l01 = widen8x4<KVT, BF16>(lo01);
                        l89 = widen8x4<KVT, BF16>(lo89);
                        h01 = widen8x4<KVT, BF16>(hi01);
                        h89 = widen8x4<KVT, BF16>(hi89);
                      }
                      mma16816<BF16>(o[2 * wd], l01.x, l01.y, l89.x, l89.y, pb0, pb1);
                      mma16816<BF16>(o[2 * wd + 1], h01.x, h01.y, h89.x, h89.y, pb0, pb1);
                    } else {   // two head dims per word
                      mma16816<BF16>(o[4 * x2 + wd], __byte_perm(A[wd], B[wd], 0x5410),
                                     __byte_perm(A[wd], B[wd], 0x7632),
                                     __byte_perm(C[wd], E[wd], 0x5410),
                                     __byte_perm(C[wd], E[wd], 0x7632), pb0, pb1);
                    }
                  }
                }
              }
              if constexpr (VFOLD) {
                // heads 2q and 2q + 1: row 0 of the sums, held by lane q
                const float s0 = __shfl_sync(0xffffffffu, psum[0], q);
                const float s1 = __shfl_sync(0xffffffffu, psum[1], q);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  o[j][0] = fmaf(-1152.f, s0, o[j][0]);
                  o[j][1] = fmaf(-1152.f, s1, o[j][1]);
                  o[j][2] = fmaf(-1152.f, s0, o[j][2]);
                  o[j][3] = fmaf(-1152.f, s1, o[j][3]);
                }
              }
            } else {
            // ---- S = Q K^T over NJ n-tiles of 8 tokens.  Each Q fragment is
            //      read from shared memory once and used for every n-tile.
            float s[NJ][4];
#pragma unroll
            for (int jn = 0; jn < NJ; ++jn) s[jn][0] = s[jn][1] = s[jn][2] = s[jn][3] = 0.f;
            if constexpr (ELEM == 1 && D == 128) {
              uint32_t w[NJ][8];
#pragma unroll
              for (int jn = 0; jn < NJ; ++jn) {
                const int tk = sub + 8 * jn + r;
                const uint4 a0 = lds128(chunk_addr(kreg, tk, 2 * q, sh.row_bytes));
                const uint4 a1 = lds128(chunk_addr(kreg, tk, 2 * q + 1, sh.row_bytes));
                w[jn][0] = a0.x; w[jn][1] = a0.y; w[jn][2] = a0.z; w[jn][3] = a0.w;
                w[jn][4] = a1.x; w[jn][5] = a1.y; w[jn][6] = a1.z; w[jn][7] = a1.w;
              }
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                const uint4 a = load_qfrag<QROWS>(qf, kk);
#pragma unroll
                for (int jn = 0; jn < NJ; ++jn) {
                  const uint2 kb = widen8x4<KVT, BF16>(w[jn][kk]);
                  mma16816<BF16>(s[jn], a.x, a.y, a.z, a.w, kb.x, kb.y);
                }
              }
            } else if constexpr (ELEM == 1) {   // D == 64, 64-byte rows
              uint32_t w[NJ][4];
#pragma unroll
              for (int jn = 0; jn < NJ; ++jn) {
                const uint4 a0 = lds128(chunk_addr(kreg, sub + 8 * jn + r, q, sh.row_bytes));
                w[jn][0] = a0.x; w[jn][1] = a0.y; w[jn][2] = a0.z; w[jn][3] = a0.w;
              }
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint4 a = load_qfrag<QROWS>(qf, kk);
#pragma unroll
                for (int jn = 0; jn < NJ; ++jn) {
                  const uint2 kb = widen8x4<KVT, BF16>(w[jn][kk]);
                  mma16816<BF16>(s[jn], a.x, a.y, a.z, a.w, kb.x, kb.y);
                }
              }
            } else {   // 16-bit: chunk pairs (2q, 2q+1) of each 128-byte region
#pragma unroll
              for (int x2 = 0; x2 < D / 64; ++x2) {
                const uint32_t reg = kreg + x2 * xstride;
                uint4 c[NJ][2];
#pragma unroll
                for (int jn = 0; jn < NJ; ++jn) {
                  c[jn][0] = lds128(chunk_addr(reg, sub + 8 * jn + r, 2 * q, sh.row_bytes));
                  c[jn][1] = lds128(chunk_addr(reg, sub + 8 * jn + r, 2 * q + 1, sh.row_bytes));
                }
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                  const uint4 a = load_qfrag<QROWS>(qf, x2 * 4 + k4);
#pragma unroll
                  for (int jn = 0; jn < NJ; ++jn) {
                    const uint4 pp = c[jn][k4 >> 1];
                    mma16816<BF16>(s[jn], a.x, a.y, a.z, a.w, (k4 & 1) ? pp.z : pp.x,
                                   (k4 & 1) ? pp.w : pp.y);
                  }
                }
              }
            }
            // ---- online softmax (rows r and r + 8; this lane holds tokens
            //      8*jn + 2q + {0,1} of the sub-tile).  Keys past the segment
            //      end are masked; with multi-token queries rows r and r + 8
            //      (token j of their head) also stop q_len - 1 - j keys before
            //      the sequence's end: folded into the same test in the
            //      per-token-scale kernels, a separate pass near the end in
            //      the others (either way fewer registers).
            float pr[NJ][4];
            float mx0 = -INFINITY, mx1 = -INFINITY;
            // per-token scales of this warp's KV head in the stage (TOK):
            // token tt of the tile at [tt * hc + kvl]
            // (32-bit shared-memory addresses: fewer registers than pointers)
            const uint32_t tsk =
                smem_u32(scl) + 4u * (uint32_t)(stg * (sh.scale_bytes / 4) + sub * sh.hc + kvl);
            const uint32_t tsv = tsk + 4u * (uint32_t)(sh.hc * sh.tile);
#pragma unroll
            for (int jn = 0; jn < NJ; ++jn) {
              float2 kk2 = make_float2(1.f, 1.f);
              if constexpr (TOK) {
                kk2.x = lds_f32(tsk + 4u * (uint32_t)((8 * jn + 2 * q) * sh.hc));
                kk2.y = lds_f32(tsk + 4u * (uint32_t)((8 * jn + 2 * q + 1) * sh.hc));
              }
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int tok = 8 * jn + 2 * q + (e & 1);
                float v = s[jn][e] * sc;
                if constexpr (TOK) v *= (e & 1) ? kk2.y : kk2.x;
                if (edge && tok >= ((e & 2) ? left1 : left0)) v = -INFINITY;
                pr[jn][e] = v;
              }
              mx0 = fmaxf(mx0, fmaxf(pr[jn][0], pr[jn][1]));
              mx1 = fmaxf(mx1, fmaxf(pr[jn][2], pr[jn][3]));
            }
            if (CAUSAL && !TOK) {
              const int tail = seg.T - (t0 + sub);
              const int lim0 = tail - cut0, lim1 = tail - cut1;
              if (min(lim0, lim1) < SUB) {
                mx0 = mx1 = -INFINITY;
#pragma unroll
                for (int jn = 0; jn < NJ; ++jn) {
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    const int tok = 8 * jn + 2 * q + (e & 1);
                    if (tok >= ((e & 2) ? lim1 : lim0)) pr[jn][e] = -INFINITY;
                  }
                  mx0 = fmaxf(mx0, fmaxf(pr[jn][0], pr[jn][1]));
                  mx1 = fmaxf(mx1, fmaxf(pr[jn][2], pr[jn][3]));
                }
              }
            }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float base0 = mn0 == -INFINITY ? 0.f : mn0;
            const float base1 = mn1 == -INFINITY ? 0.f : mn1;
            const float a0 = fast_exp2(m0 - base0), a1 = fast_exp2(m1 - base1);
            m0 = mn0;
            m1 = mn1;
            float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
            for (int jn = 0; jn < NJ; ++jn) {
              pr[jn][0] = fast_exp2(pr[jn][0] - base0);
              pr[jn][1] = fast_exp2(pr[jn][1] - base0);
              pr[jn][2] = fast_exp2(pr[jn][2] - base1);
              pr[jn][3] = fast_exp2(pr[jn][3] - base1);
              ps0 += pr[jn][0] + pr[jn][1];
              ps1 += pr[jn][2] + pr[jn][3];
            }
            l0 = fmaf(l0, a0, ps0);
            l1 = fmaf(l1, a1, ps1);
            if constexpr (TOK) {   // V scales weight the probabilities, not their sum
#pragma unroll
              for (int jn = 0; jn < NJ; ++jn) {
                // tokens past the end: their scale slot may hold anything
                const int tk = 8 * jn + 2 * q;
                const float vx = tk < left ? lds_f32(tsv + 4u * (uint32_t)(tk * sh.hc)) : 0.f;
                const float vy = tk + 1 < left ? lds_f32(tsv + 4u * (uint32_t)((tk + 1) * sh.hc)) : 0.f;
                pr[jn][0] *= vx;
                pr[jn][1] *= vy;
                pr[jn][2] *= vx;
                pr[jn][3] *= vy;
              }
            }
            if (!__all_sync(0xffffffffu, a0 == 1.f && a1 == 1.f)) {
#pragma unroll
              for (int t = 0; t < NT; ++t) {
                o[t][0] *= a0;
                o[t][1] *= a0;
                o[t][2] *= a1;
                o[t][3] *= a1;
              }
            }
            // ---- O += P V, one k-step of 16 tokens at a time.  This lane's B
            //      fragments: tokens 2q, 2q+1 (b0) and 2q+8, 2q+9 (b1) of the
            //      k-step, head dims vdim(j, r).
#pragma unroll
            for (int kt = 0; kt < SUB / 16; ++kt) {
              const uint32_t pa0 = pack_f32x2(pr[2 * kt][0], pr[2 * kt][1], BF16);
              const uint32_t pa1 = pack_f32x2(pr[2 * kt][2], pr[2 * kt][3], BF16);
              const uint32_t pa2 = pack_f32x2(pr[2 * kt + 1][0], pr[2 * kt + 1][1], BF16);
              const uint32_t pa3 = pack_f32x2(pr[2 * kt + 1][2], pr[2 * kt + 1][3], BF16);
              const int u0 = sub + 16 * kt + 2 * q, u1 = u0 + 1, u2 = u0 + 8, u3 = u0 + 9;
              if constexpr (ELEM == 1 && D == 128) {
                uint4 w0 = lds128(chunk_addr(vreg, u0, r, sh.row_bytes));
                uint4 w1 = lds128(chunk_addr(vreg, u1, r, sh.row_bytes));
                uint4 w2 = lds128(chunk_addr(vreg, u2, r, sh.row_bytes));
                uint4 w3 = lds128(chunk_addr(vreg, u3, r, sh.row_bytes));
                if (left < SUB) zero_rows_past_end(w0, w1, w2, w3, 16 * kt + 2 * q, left);
                const uint32_t A[4] = {w0.x, w0.y, w0.z, w0.w}, B[4] = {w1.x, w1.y, w1.z, w1.w};
                const uint32_t C[4] = {w2.x, w2.y, w2.z, w2.w}, E[4] = {w3.x, w3.y, w3.z, w3.w};
#pragma unroll
                for (int wd = 0; wd < 4; ++wd) {
                  const uint32_t lo01 = __byte_perm(A[wd], B[wd], 0x5140);
                  const uint32_t hi01 = __byte_perm(A[wd], B[wd], 0x7362);
                  const uint32_t lo89 = __byte_perm(C[wd], E[wd], 0x5140);
                  const uint32_t hi89 = __byte_perm(C[wd], E[wd], 0x7362);
                  const uint2 l01 = widen8x4<KVT, BF16>(lo01), l89 = widen8x4<KVT, BF16>(lo89);
                  const uint2 h01 = widen8x4<KVT, BF16>(hi01), h89 = widen8x4<KVT, BF16>(hi89);
                  mma16816<BF16>(o[4 * wd + 0], pa0, pa1, pa2, pa3, l01.x, l89.x);
                  mma16816<BF16>(o[4 * wd + 1], pa0, pa1, pa2, pa3, l01.y, l89.y);
                  mma16816<BF16>(o[4 * wd + 2], pa0, pa1, pa2, pa3, h01.x, h89.x);
                  mma16816<BF16>(o[4 * wd + 3], pa0, pa1, pa2, pa3, h01.y, h89.y);
                }
              } else if constexpr (ELEM == 1) {   // D == 64: 8 bytes per token
                const int c = r >> 1, half = (r & 1) * 8;
                uint2 w0 = lds64(chunk_addr(vreg, u0, c, sh.row_bytes) + half);
                uint2 w1 = lds64(chunk_addr(vreg, u1, c, sh.row_bytes) + half);
                uint2 w2 = lds64(chunk_addr(vreg, u2, c, sh.row_bytes) + half);
                uint2 w3 = lds64(chunk_addr(vreg, u3, c, sh.row_bytes) + half);
                if (left < SUB) zero_rows_past_end(w0, w1, w2, w3, 16 * kt + 2 * q, left);
                const uint32_t A[2] = {w0.x, w0.y}, B[2] = {w1.x, w1.y};
                const uint32_t C[2] = {w2.x, w2.y}, E[2] = {w3.x, w3.y};
#pragma unroll
                for (int wd = 0; wd < 2; ++wd) {
                  const uint32_t lo01 = __byte_perm(A[wd], B[wd], 0x5140);
                  const uint32_t hi01 = __byte_perm(A[wd], B[wd], 0x7362);
                  const uint32_t lo89 = __byte_perm(C[wd], E[wd], 0x5140);
                  const uint32_t hi89 = __byte_perm(C[wd], E[wd], 0x7362);
                  const uint2 l01 = widen8x4<KVT, BF16>(lo01), l89 = widen8x4<KVT, BF16>(lo89);
                  const uint2 h01 = widen8x4<KVT, BF16>(hi01), h89 = widen8x4<KVT, BF16>(hi89);
                  mma16816<BF16>(o[4 * wd + 0], pa0, pa1, pa2, pa3, l01.x, l89.x);
                  mma16816<BF16>(o[4 * wd + 1], pa0, pa1, pa2, pa3, l01.y, l89.y);
                  mma16816<BF16>(o[4 * wd + 2], pa0, pa1, pa2, pa3, h01.x, h89.x);
                  mma16816<BF16>(o[4 * wd + 3], pa0, pa1, pa2, pa3, h01.y, h89.y);
                }
              } else {   // 16-bit: chunk r of each 128-byte region holds 8 dims
#pragma unroll
                for (int x2 = 0; x2 < D / 64; ++x2) {
                  const uint32_t reg = vreg + x2 * xstride;
                  uint4 w0 = lds128(chunk_addr(reg, u0, r, sh.row_bytes));
                  uint4 w1 = lds128(chunk_addr(reg, u1, r, sh.row_bytes));
                  uint4 w2 = lds128(chunk_addr(reg, u2, r, sh.row_bytes));
                  uint4 w3 = lds128(chunk_addr(reg, u3, r, sh.row_bytes));
                  if (left < SUB) zero_rows_past_end(w0, w1, w2, w3, 16 * kt + 2 * q, left);
                  const uint32_t A[4] = {w0.x, w0.y, w0.z, w0.w}, B[4] = {w1.x, w1.y, w1.z, w1.w};
                  const uint32_t C[4] = {w2.x, w2.y, w2.z, w2.w}, E[4] = {w3.x, w3.y, w3.z, w3.w};
#pragma unroll
                  for (int wd = 0; wd < 4; ++wd) {
                    const int jt = x2 * 8 + 2 * wd;
                    mma16816<BF16>(o[jt], pa0, pa1, pa2, pa3, __byte_perm(A[wd], B[wd], 0x5410),
                                   __byte_perm(C[wd], E[wd], 0x5410));
                    mma16816<BF16>(o[jt + 1], pa0, pa1, pa2, pa3, __byte_perm(A[wd], B[wd], 0x7632),
                                   __byte_perm(C[wd], E[wd], 0x7632));
                  }
                }
              }
            }
            }   // FLIP
          }
        }
        __syncwarp();
        // the segment's last stage stays held when the head tile's warps
        // merge in it (released after the merge)
        last_stg = stg;
        if (lane == 0 && !(sh.merge_in_stage && t0 + sh.tile >= seg.t_end))
          mbar_arrive(&sm.empty[stg]);
        if (warp == 0 && lane == 0) {
          FD_STAMP(g_split_stamps, 4, stamp_ns());
          FD_STAMP(g_split_stamps, 7, (unsigned long long)(n + 1));
        }
      }

      float* part = p.part_acc + (long long)seg.slot * p.hq * D;
      float2* pml = p.part_ml + (long long)seg.slot * p.hq;
      QT* outp = static_cast<QT*>(p.out) + qrow0 * D;
      float* lsep = p.lse ? p.lse + qrow0 : nullptr;
      if constexpr (FLIP) {
        // ---- end of segment: a head's sum over its 8 lanes; head 2q + hh
        //      holds head dims flip_dim(j, r) (o[j][hh]) and flip_dim(j, r) + 1
        //      (o[j][2 + hh]); m-tiles j, j + 1 (j even) are 4 consecutive dims
#pragma unroll
        for (int o2 = 4; o2 < 32; o2 <<= 1) {
          l0 += __shfl_xor_sync(0xffffffffu, l0, o2);
          l1 += __shfl_xor_sync(0xffffffffu, l1, o2);
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int h = 2 * q + hh;
          if (h >= G) continue;
          const long long li = (long long)kvl * G + h;
          const float L = hh ? l1 : l0, M = hh ? m1 : m0;
          if (seg.complete) {
            const float rs = L > 0.f ? vsc / L : 0.f;
#pragma unroll
            for (int j = 0; j < 8; j += 2)
              *reinterpret_cast<uint2*>(outp + li * D + flip_dim<ELEM>(j, r)) =
                  make_uint2(pack_f32x2(o[j][hh] * rs, o[j][2 + hh] * rs, BF16),
                             pack_f32x2(o[j + 1][hh] * rs, o[j + 1][2 + hh] * rs, BF16));
            if (lsep && r == 0) lsep[li] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
          } else {
#pragma unroll
            for (int j = 0; j < 8; j += 2)
              *reinterpret_cast<float4*>(part + li * D + flip_dim<ELEM>(j, r)) =
                  make_float4(o[j][hh], o[j][2 + hh], o[j + 1][hh], o[j + 1][2 + hh]);
            if (r == 0) pml[li] = make_float2(M, L);
          }
        }
      } else {
      // ---- end of segment: full row sums, merge the warps of a head tile
      l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
      l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
      if (sh.wph == 1) {
        // This warp alone holds the head tile's state.  Its head dims form
        // runs of consecutive dims (vdim), written 4 at a time.
        const float r0 = l0 > 0.f ? vsc / l0 : 0.f;
        const float r1 = l1 > 0.f ? vsc / l1 : 0.f;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const bool vh = hh ? v1 : v0;
          const long long li = hh ? li1 : li0;
          const float rs = hh ? r1 : r0;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
#pragma unroll
            for (int t4 = 0; t4 < NT / 4; ++t4) {
              const int d = vdim<D, ELEM>(4 * t4, 2 * q + e);
              const float a0 = o[4 * t4][2 * hh + e], a1 = o[4 * t4 + 1][2 * hh + e];
              const float a2 = o[4 * t4 + 2][2 * hh + e], a3 = o[4 * t4 + 3][2 * hh + e];
              if (!vh) continue;
              if (seg.complete) {
                uint2 w;
                w.x = pack_f32x2(a0 * rs, a1 * rs, BF16);
                w.y = pack_f32x2(a2 * rs, a3 * rs, BF16);
                *reinterpret_cast<uint2*>(outp + li * D + d) = w;
              } else {
                *reinterpret_cast<float4*>(part + li * D + d) = make_float4(a0, a1, a2, a3);
              }
            }
          }
        }
        if (q == 0) {
          if (seg.complete) {
            if (lsep && v0) lsep[li0] = l0 > 0.f ? (m0 + log2f(l0)) * kLn2 : -INFINITY;
            if (lsep && v1) lsep[li1] = l1 > 0.f ? (m1 + log2f(l1)) * kLn2 : -INFINITY;
          } else {
            if (v0) pml[li0] = make_float2(m0, l0);
            if (v1) pml[li1] = make_float2(m1, l1);
          }
        }
      } else {
        // Stage every warp's state in shared memory, then the wph warps of a
        // head tile merge its 16 x D outputs together.  The area is the
        // stage of the segment's last tile (held back from the producer) or
        // a dedicated one: warp w's 16 rows of D floats at w * 16 * D,
        // float4 chunk c of row x at chunk swz(x, c) (see merge_chunk), its
        // row maxima and sums in the Q-fragment area (free at a segment end).
        const uint32_t marea =
            sh.merge_in_stage ? stage0 + (uint32_t)last_stg * 2u * sh.kv_bytes
                              : stage0 + (uint32_t)(sh.stages * 2 * sh.kv_bytes);
        asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");   // stage read
        if (warp == 0 && lane == 0) FD_STAMP(g_split_stamps, 13, stamp_ns());
        const uint32_t mine = marea + (uint32_t)warp * (16u * D * 4u);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
#pragma unroll
            for (int t4 = 0; t4 < NT / 4; ++t4) {
              const int d = vdim<D, ELEM>(4 * t4, 2 * q + e);
              const int row = r + 8 * hh;
              asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(
                               mine + (uint32_t)row * (D * 4) + merge_chunk(row, d >> 2) * 16u),
                           "f"(o[4 * t4][2 * hh + e]), "f"(o[4 * t4 + 1][2 * hh + e]),
                           "f"(o[4 * t4 + 2][2 * hh + e]), "f"(o[4 * t4 + 3][2 * hh + e])
                           : "memory");
            }
          }
        }
        float* mstat = reinterpret_cast<float*>(base + (size_t)(qfrag0 - stage0));   // [warp][m 16 | l 16]
        if (q == 0) {
          mstat[warp * 32 + r] = m0;
          mstat[warp * 32 + r + 8] = m1;
          mstat[warp * 32 + 16 + r] = l0;
          mstat[warp * 32 + 16 + r + 8] = l1;
        }
        asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
        if (warp == 0 && lane == 0) FD_STAMP(g_split_stamps, 14, stamp_ns());
        // each warp of the head tile merges whole rows, a lane 4 dims of one
        // row; the row's weights come from broadcast reads of m and l
        const uint32_t grp = marea + (uint32_t)(ht * sh.wph) * (16u * D * 4u);
        const float* gstat = mstat + ht * sh.wph * 32;
        for (int idx = ts * 32 + lane; idx < 16 * (D / 4); idx += sh.wph * 32) {
          const int row = idx / (D / 4), c = idx - row * (D / 4), d = 4 * c;
          const int lh = mtile * 16 + row;
          if (lh >= G) continue;
          // (at most 8 warps per head tile: a fixed bound, predicated, so
          // that all loads issue before the first use)
          float mw[kConsumerWarps], lw[kConsumerWarps];
          uint4 vb[kConsumerWarps];
          const uint32_t cofs = (uint32_t)row * (D * 4) + merge_chunk(row, c) * 16u;
#pragma unroll
          for (int w2 = 0; w2 < kConsumerWarps; ++w2) {
            if (w2 < sh.wph) {
              mw[w2] = gstat[w2 * 32 + row];
              lw[w2] = gstat[w2 * 32 + 16 + row];
              vb[w2] = lds128(grp + (uint32_t)w2 * (16u * D * 4u) + cofs);
            } else {
              mw[w2] = -INFINITY;
              lw[w2] = 0.f;
              vb[w2] = make_uint4(0u, 0u, 0u, 0u);
            }
          }
          float M = -INFINITY;
#pragma unroll
          for (int w2 = 0; w2 < kConsumerWarps; ++w2) M = fmaxf(M, mw[w2]);
          float L = 0.f;
          float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int w2 = 0; w2 < kConsumerWarps; ++w2) {
            const float f = mw[w2] == -INFINITY ? 0.f : fast_exp2(mw[w2] - M);
            L = fmaf(lw[w2], f, L);
            A.x = fmaf(__uint_as_float(vb[w2].x), f, A.x);
            A.y = fmaf(__uint_as_float(vb[w2].y), f, A.y);
            A.z = fmaf(__uint_as_float(vb[w2].z), f, A.z);
            A.w = fmaf(__uint_as_float(vb[w2].w), f, A.w);
          }
          const int li = kvl * G + lh;
          if (seg.complete) {
            const float rs = L > 0.f ? vsc / L : 0.f;
            uint2 w;
            w.x = pack_f32x2(A.x * rs, A.y * rs, BF16);
            w.y = pack_f32x2(A.z * rs, A.w * rs, BF16);
            *reinterpret_cast<uint2*>(outp + (long long)li * D + d) = w;
            if (d == 0 && lsep) lsep[li] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
          } else {
            *reinterpret_cast<float4*>(part + (long long)li * D + d) = A;
            if (d == 0) pml[li] = make_float2(M, L);
          }
        }
        asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
        if (warp == 0 && lane == 0) FD_STAMP(g_split_stamps, 15, stamp_ns());
        if (sh.merge_in_stage && lane == 0) mbar_arrive(&sm.empty[last_stg]);
      }
      }
      if (warp == 0 && lane == 0) FD_STAMP(g_split_stamps, 5, stamp_ns());
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) FD_STAMP(g_split_stamps, 6, stamp_ns());
}


struct Maps {
  CUtensorMap k, v, ks, vs;   // caches; per-token scale arrays (when sh.scale_tma)
};

// CAUSAL: multi-token queries (q_len > 1) without per-token scales; the
// per-token-scale kernels fold the causal limit into their ragged-end test.
template <int KVT, typename QT, int D, bool TOK, int QROWS = 16, bool CAUSAL = false,
          bool FLIP = false>
cudaError_t launch_t(const Params& p, const Shape& sh, const Maps& m, cudaStream_t stream) {
  auto kern = mma_split_kernel<KVT, QT, D, TOK, QROWS, CAUSAL, FLIP>;
  static std::atomic<unsigned long long> limit_set{0};
  cudaError_t e = ensure_smem_limit(kern, kSmemBudget, &limit_set);
  if (e != cudaSuccess) return e;
  return launch_split(p, kern, dim3(p.grid), dim3(kThreads), sh.smem_bytes, stream, p, sh, m.k,
                      m.v, m.ks, m.vs);
}

// Without per-token scales: one query token per sequence, or several; all
// 16 Q rows, or 8.
template <int KVT, typename QT, int D>
cudaError_t launch_plain(const Params& p, const Shape& sh, const Maps& m, cudaStream_t st) {
  if constexpr (D == 128)
    if (sh.flip && p.q_len == 1) return launch_t<KVT, QT, D, false, 8, false, true>(p, sh, m, st);
  if (sh.qrows == 8)
    return p.q_len > 1 ? launch_t<KVT, QT, D, false, 8, true>(p, sh, m, st)
                       : launch_t<KVT, QT, D, false, 8, false>(p, sh, m, st);
  return p.q_len > 1 ? launch_t<KVT, QT, D, false, 16, true>(p, sh, m, st)
                     : launch_t<KVT, QT, D, false, 16, false>(p, sh, m, st);
}

// 8-bit caches with per-token scales: all 16 Q rows, or 8.
template <int KVT, typename QT, int D>
cudaError_t launch_tok(const Params& p, const Shape& sh, const Maps& m, cudaStream_t st) {
  if constexpr (D == 128)
    if (sh.flip && p.q_len == 1) return launch_t<KVT, QT, D, true, 8, false, true>(p, sh, m, st);
  return sh.qrows == 8 ? launch_t<KVT, QT, D, true, 8>(p, sh, m, st)
                       : launch_t<KVT, QT, D, true, 16>(p, sh, m, st);
}

// 8-bit caches: q dtype x per-token scales or not.
template <int KVT, int D>
cudaError_t launch_8bit(const Params& p, const Shape& sh, const Maps& m, cudaStream_t st) {
  const bool tok = p.scale_kind == FD_SCALE_TOKEN;
  if (p.q_dtype == FD_F16)
    return tok ? launch_tok<KVT, __half, D>(p, sh, m, st)
               : launch_plain<KVT, __half, D>(p, sh, m, st);
  return tok ? launch_tok<KVT, __nv_bfloat16, D>(p, sh, m, st)
             : launch_plain<KVT, __nv_bfloat16, D>(p, sh, m, st);
}



// Per cache format (one translation unit each): launches the split kernel
// variant for p's query dtype, head_dim, scale kind and q_len.
cudaError_t launch_e4m3(const Params& p, const Shape& sh, const Maps& m, cudaStream_t st);
cudaError_t launch_i8(const Params& p, const Shape& sh, const Maps& m, cudaStream_t st);
cudaError_t launch_16bit(const Params& p, const Shape& sh, const Maps& m, cudaStream_t st);
// The CUDA-core form (fd_split_fma.cu): its shape for a group, and its launch.
bool fma_shape(int group, int num_kv_heads, int page_size, Shape* out);
cudaError_t launch_fma(const Params& p, const Shape& sh, const Maps& m, cudaStream_t st);
#ifdef FD_STAMPS
cudaError_t read_stamps_e4m3(unsigned long long* host, int n);
#endif

}  // namespace mma
}  // namespace fd
