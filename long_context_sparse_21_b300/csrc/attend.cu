// Steps 4 and 5 of the hot path: core attention of CSA (selected compressed
// entries + sliding window) and HCA (every visible compressed entry + window).
//
// DeepSeek-V4 report (cnblogs translation) §2.3.1 "shared key-value MQA":
// every compressed entry is both key and value for all query heads; §2.3.2:
// HCA attends densely to all compressed entries; §2.3.3: a sliding-window
// branch adds n_win uncompressed entries per query, and learnable sink logits
// may take part of the attention mass.  HF blog "DeepSeek-V4" (translation),
// Fig. 3 / Fig. 4: the compressed branch and the window branch feed one MQA.
//
// One softmax runs over the union of the two sets, merged by online softmax
// (running max and rescaled sums, in the log2 domain).  Decode splits a
// query's item list across CTAs (flash-decoding); a combine kernel merges
// the partial (max, sum, unnormalized output) triples with log-sum-exp
// weights in a fixed split order, so results do not depend on timing.
//
// Kernels:
//  * attend_f32_kernel   float32 path on CUDA cores (dense f32 entries).
//  * attend_tc_kernel    BF16 queries, FP8-e4m3 + BF16-RoPE pooled entries and
//                        BF16 window tokens: tcgen05 MMAs with TMEM
//                        accumulators, 64 heads x 576 dims, 32-item tiles:
//                        entries staged by bulk async copies and dequantized
//                        by converter warps, window rows loaded by TMA.
//  * combine_kernel      log-sum-exp merge of split partials.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "host.hpp"
#include "tc.cuh"

namespace csa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ int n_visible(int t, int m) { return t < 0 ? 0 : (t + 1) / m; }

struct AttArgs {
  const void* q;
  const int32_t* pos;
  const int32_t* seq;
  const int32_t* idx;  // NULL -> dense (HCA)
  const int32_t* cnt;
  int top_k, m, window, T, H, D, splits, items_per_split;
  int kv_cap;          // entries the store holds per sequence (clamps visibility)
  Store kv;
  const void* win;
  int win_ring;
  float scale_log2;    // scale * log2(e)
  const float* sink;   // natural-log logits, or NULL
  void* out;
  int out_bf16;
  float* lse;
  // split partials (splits > 1)
  float* part_o;       // [T][splits][H][D]
  float* part_ml;      // [T][splits][H][2]: running max (log2 domain), sum
  int* status;
};

// Item list of query r: [0, n_sel) compressed entries, then the window.
struct Items {
  int b, t, n_sel, nvis, n_win, L;
};

__device__ __forceinline__ Items query_items(const AttArgs& a, int r) {
  Items it;
  it.b = a.seq ? a.seq[r] : r;
  it.t = a.pos[r];
  it.nvis = min(n_visible(it.t, a.m), a.kv_cap);
  it.n_sel = a.idx ? min(max(a.cnt[r], 0), a.top_k) : it.nvis;
  it.n_win = it.t < 0 ? 0 : min(a.window, it.t + 1);
  it.L = it.n_sel + it.n_win;
  return it;
}

// Compressed entry of item i (< n_sel), or -1 if its index is invalid.
__device__ __forceinline__ int item_entry(const AttArgs& a, const Items& it, int r, int i) {
  const int e = a.idx ? a.idx[(size_t)r * a.top_k + i] : i;
  if (e < 0 || e >= it.nvis) {
    set_status(a.status, CSA_ERR_INVALID_ARG);
    return -1;
  }
  return e;
}

__device__ __forceinline__ size_t win_row(const AttArgs& a, const Items& it, int i) {
  const int p = it.t - it.n_win + 1 + (i - it.n_sel);
  return ((size_t)it.b * a.win_ring + (size_t)(p % a.win_ring)) * a.D;
}

// Final normalization of one (query, head) row held as (m2, l) with output
// accumulators; writes lse when requested.  Returns 1/den (0 for an empty set).
__device__ __forceinline__ float finalize_row(const AttArgs& a, int r, int h, float m2, float l) {
  float mx = m2;
  float s2 = -INFINITY;
  if (a.sink) {
    s2 = a.sink[h] * kLog2e;
    mx = fmaxf(mx, s2);
  }
  float den = (l > 0.f ? l * exp2f(m2 - mx) : 0.f) + (a.sink ? exp2f(s2 - mx) : 0.f);
  if (a.lse) a.lse[(size_t)r * a.H + h] = den > 0.f ? (mx + log2f(den)) * kLn2 : -INFINITY;
  // output = sum p x / den, where the accumulators hold sum 2^(s - m2) x
  return (l > 0.f && den > 0.f) ? exp2f(m2 - mx) / den : 0.f;
}

// ================================================================== float32 path

constexpr int kF32Threads = 256;
constexpr int kF32Tile = 32;
constexpr int kF32MaxPer = 32;  // H * D <= 256 * 32

__global__ void __launch_bounds__(kF32Threads) attend_f32_kernel(AttArgs a) {
  extern __shared__ float sm[];
  const int H = a.H, D = a.D, DP = D + 1;
  float* qs = sm;                       // [H][D+1]
  float* xs = qs + H * DP;              // [kF32Tile][D+1]
  float* ps = xs + kF32Tile * DP;       // [H][kF32Tile]
  float* mrow = ps + H * kF32Tile;      // [H]
  float* lrow = mrow + H;               // [H]
  float* crow = lrow + H;               // [H] rescale factors of the current tile
  const int r = blockIdx.x, split = blockIdx.y, tid = threadIdx.x;
  const Items it = query_items(a, r);
  const int i0 = split * a.items_per_split;
  const int i1 = min(it.L, i0 + a.items_per_split);
  const float* q = static_cast<const float*>(a.q) + (size_t)r * H * D;
  for (int i = tid; i < H * D; i += kF32Threads) qs[(i / D) * DP + i % D] = q[i];
  for (int h = tid; h < H; h += kF32Threads) {
    mrow[h] = -INFINITY;
    lrow[h] = 0.f;
  }
  float o[kF32MaxPer];
#pragma unroll
  for (int i = 0; i < kF32MaxPer; ++i) o[i] = 0.f;
  __syncthreads();

  for (int base = i0; base < i1; base += kF32Tile) {
    const int nt = min(kF32Tile, i1 - base);
    for (int u = tid; u < kF32Tile * D; u += kF32Threads) {
      const int e = u / D, d = u % D, i = base + e;
      float v = 0.f;
      if (e < nt) {
        if (i < it.n_sel) {
          const int ent = item_entry(a, it, r, i);
          if (ent >= 0) v = reinterpret_cast<const float*>(a.kv.base)[((size_t)it.b * a.kv.capacity + ent) * D + d];
        } else {
          v = static_cast<const float*>(a.win)[win_row(a, it, i) + d];
        }
      }
      xs[e * DP + d] = v;
    }
    __syncthreads();
    for (int pr = tid; pr < H * kF32Tile; pr += kF32Threads) {
      const int h = pr / kF32Tile, e = pr % kF32Tile;
      float s = -INFINITY;
      if (e < nt) {
        float acc = 0.f;
        for (int d = 0; d < D; ++d) acc = fmaf(qs[h * DP + d], xs[e * DP + d], acc);
        s = acc * a.scale_log2;
      }
      ps[h * kF32Tile + e] = s;
    }
    __syncthreads();
    for (int h = tid; h < H; h += kF32Threads) {
      float mt = -INFINITY;
      for (int e = 0; e < nt; ++e) mt = fmaxf(mt, ps[h * kF32Tile + e]);
      const float mn = fmaxf(mrow[h], mt);
      const float c = exp2f(mrow[h] - mn);  // 0 when the old max was -inf
      float l = lrow[h] * c;
      for (int e = 0; e < kF32Tile; ++e) {
        const float p = e < nt ? exp2f(ps[h * kF32Tile + e] - mn) : 0.f;
        ps[h * kF32Tile + e] = p;
        l += p;
      }
      mrow[h] = mn;
      lrow[h] = l;
      crow[h] = c;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kF32MaxPer; ++k) {
      const int el = tid + k * kF32Threads;
      if (el < H * D) {
        const int h = el / D, d = el % D;
        float acc = o[k] * crow[h];
        for (int e = 0; e < nt; ++e) acc = fmaf(ps[h * kF32Tile + e], xs[e * DP + d], acc);
        o[k] = acc;
      }
    }
    __syncthreads();
  }

  if (a.splits == 1) {
    for (int h = tid; h < H; h += kF32Threads) crow[h] = finalize_row(a, r, h, mrow[h], lrow[h]);
    __syncthreads();
    float* out = static_cast<float*>(a.out) + (size_t)r * H * D;
#pragma unroll
    for (int k = 0; k < kF32MaxPer; ++k) {
      const int el = tid + k * kF32Threads;
      if (el < H * D) out[el] = o[k] * crow[el / D];
    }
  } else {
    float* po = a.part_o + ((size_t)r * a.splits + split) * H * D;
#pragma unroll
    for (int k = 0; k < kF32MaxPer; ++k) {
      const int el = tid + k * kF32Threads;
      if (el < H * D) po[el] = o[k];
    }
    for (int h = tid; h < H; h += kF32Threads) {
      float* ml = a.part_ml + (((size_t)r * a.splits + split) * H + h) * 2;
      ml[0] = mrow[h];
      ml[1] = lrow[h];
    }
  }
}

// ================================================================== shared constants / helpers

constexpr int kHeads = 64;
constexpr int kDim = kKvDim;            // 576


// ================================================================== tcgen05 path (bf16 / fp8)
//
// One CTA = one (query, split).  The split's item list is cut into tiles of
// 32 items; the compressed entries come first, padded to a whole tile, then
// the window rows.  Warp roles:
//   MMA warp:  S[64 heads x 32 items] = Q . X^T      (tcgen05 M=64, N=32, K=576)
//              O[576 dims x 64 heads] += X^T . P^T   (M=128 per 128-dim chunk,
//              X read MN-major from the same tile, N=64, K=32)
//   producer warp: gathers the items of a compressed tile (FP8 content row,
//              BF16 RoPE row, the 16-byte block holding the scale) into one of
//              three staging slots with 16-byte cp.async copies.
//   converter warps (4): staging -> X tile (FP8 x scale -> BF16), 128-byte
//              swizzled K-major, double buffered; a window tile (BF16 rows)
//              is loaded by TMA straight into the swizzled X tile.
//   softmax warps (4): one thread per head holds the head's 32 scores (M=64
//              accumulator rows r live in TMEM lane 32 (r / 16) + r % 16),
//              keeps a running reference max per head and writes P = 2^(s - m)
//              as BF16.
// The reference max only moves when a tile's max exceeds it by more than 2^8;
// then O's column of that head is rescaled in TMEM before the tile's PV runs.
// The 576 output dims are covered by five 128-row chunks, the last at dims
// [448, 576) (its first 64 rows repeat chunk 3 and are not written out).
constexpr int kTI = 32;                       // items per tile
constexpr int kTcWarps = 1 + 1 + 4 + 4;       // MMA, producer, softmax x4, converters x4
constexpr int kTcThreads2 = kTcWarps * 32;
constexpr int kTcKBlocks = kDim / 64;         // 9
constexpr int kTcTileBytes = kTcKBlocks * kTI * 128;   // 36864
constexpr int kTcQBytes = kTcKBlocks * kHeads * 128;   // 73728
constexpr int kTcPBytes = kHeads * 128;                // 8192 (32 of 64 columns used)
constexpr int kRawContent = kKvContent + 16;           // padded rows: conflict-free converter reads
constexpr int kRawRope = 2 * kKvRope + 16;
constexpr int kRawStage = kTI * (kRawContent + kRawRope + 16);  // 22016
constexpr int kRawStages = 3;
constexpr int kTcSmemBytes = kTcQBytes + 2 * kTcTileBytes + 2 * kTcPBytes + kRawStages * kRawStage;
constexpr uint32_t kTcSCol = 0;      // S buffers: columns [0, 128): per buffer S_content, S_rope
constexpr uint32_t kTcOCol = 128;    // O: columns [128, 448)
constexpr float kTcRescale = 8.0f;   // log2 headroom before the reference max moves

struct TcCtl {
  uint64_t x_full[2], x_empty[2], s_full[2], s_empty[2], win_full[2], p_full[2], p_empty[2], done;
  uint64_t raw_full[kRawStages], raw_empty[kRawStages];
  uint32_t tmem_base;
  int abort;
  int8_t meta[kRawStages][kTI];  // per staged item: -1 invalid, else slot % 4 (scale word)
  alignas(16) float scl[2][kTI]; // per X-tile item: its entry scale (1 for window rows)
  float corr[2][kHeads];
  float m_ref[kHeads];
  float l_sum[kHeads];
  float fin[kHeads];
};

// Byte offset of 16-byte chunk c8 (dims 8 c8 .. 8 c8 + 7) of row `row` in a
// K-major swizzled operand made of 64-dim blocks of `rows` rows.
__device__ __forceinline__ uint32_t tc_chunk_off(int row, int c8, int rows) {
  return (uint32_t)(c8 >> 3) * (uint32_t)(rows * 128) + (uint32_t)(row >> 3) * 1024u + (uint32_t)(row & 7) * 128u +
         ((uint32_t)((c8 & 7) ^ (row & 7)) << 4);
}

// 8 e4m3 codes (half of a 16-byte load) -> 8 FP16 values, exactly.
__device__ __forceinline__ uint4 fp8x8_to_f16x8(uint4 raw, bool hi) {
  const uint32_t w0 = hi ? raw.z : raw.x, w1 = hi ? raw.w : raw.y;
  uint4 v;
  __half2_raw h;
  h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w0 & 0xFFFF), __NV_E4M3);
  v.x = (uint32_t)h.x | ((uint32_t)h.y << 16);
  h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w0 >> 16), __NV_E4M3);
  v.y = (uint32_t)h.x | ((uint32_t)h.y << 16);
  h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w1 & 0xFFFF), __NV_E4M3);
  v.z = (uint32_t)h.x | ((uint32_t)h.y << 16);
  h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w1 >> 16), __NV_E4M3);
  v.w = (uint32_t)h.x | ((uint32_t)h.y << 16);
  return v;
}
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  const __half2 h = __floats2half2_rn(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  return *reinterpret_cast<const uint32_t*>(&h);
}
// 8 BF16 values -> 8 FP16 values (exact inside FP16's normal range).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
  return make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Bits j (0..31) with lo <= g0 + j < hi, without branches.
__device__ __forceinline__ uint32_t range_bits(int g0, int lo, int hi) {
  const int a = min(max(lo - g0, 0), 32), b = min(max(hi - g0, 0), 32);
  return (uint32_t)(((1ull << b) - 1ull) & ~((1ull << a) - 1ull));
}

// Barrier over the `count` threads of named barrier `id`, returning the AND
// (resp. OR) of every participant's predicate.
__device__ __forceinline__ bool bar_red_and(int id, int count, bool v) {
  uint32_t out;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n barrier.cta.red.and.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(out)
      : "r"((uint32_t)v), "r"(id), "r"(count)
      : "memory");
  return out != 0;
}
__device__ __forceinline__ bool bar_red_or(int id, int count, bool v) {
  uint32_t out;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n barrier.cta.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(out)
      : "r"((uint32_t)v), "r"(id), "r"(count)
      : "memory");
  return out != 0;
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
          "r"(tc::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(tc::smem_u32(bar))
      : "memory");
}

__global__ void __launch_bounds__(kTcThreads2, 1)
    attend_tc_kernel(AttArgs a, const __grid_constant__ CUtensorMap win_map, int win_dense) {
  extern __shared__ __align__(1024) uint8_t tc_smem[];
  __shared__ TcCtl C;
  uint8_t* Qs = tc_smem;
  uint8_t* Xs = tc_smem + kTcQBytes;  // two tiles
  uint8_t* Ps = Xs + 2 * kTcTileBytes;  // two P buffers
  uint8_t* Rs = Ps + 2 * kTcPBytes;     // staging slots
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = blockIdx.x, split = blockIdx.y;
  const Items it = query_items(a, r);
  const int sel_pad = (it.n_sel + kTI - 1) / kTI * kTI;
  const int Lp = sel_pad + it.n_win;          // padded item count
  const int i0 = split * a.items_per_split;
  const int i1 = min(Lp, i0 + a.items_per_split);
  const int ntiles = i1 > i0 ? (i1 - i0 + kTI - 1) / kTI : 0;
  const int ncomp = i1 > i0 ? max(0, min(ntiles, (sel_pad - i0 + kTI - 1) / kTI)) : 0;  // compressed tiles first

  if ((tc::smem_u32(tc_smem) & 1023u) != 0) {  // the swizzled operands need 1 KiB alignment
    if (tid == 0) set_status(a.status, CSA_ERR_ALIGN);
    return;
  }
  if (ntiles == 0) {  // empty split: an empty partial (or an empty output row set)
    if (a.splits == 1) {
      for (int h = tid; h < kHeads; h += blockDim.x) finalize_row(a, r, h, -INFINITY, 0.f);
      for (int u = tid; u < kHeads * kDim; u += blockDim.x) {
        const size_t off = (size_t)r * kHeads * kDim + u;
        if (a.out_bf16) static_cast<uint16_t*>(a.out)[off] = 0;
        else static_cast<float*>(a.out)[off] = 0.f;
      }
    } else {
      float* po = a.part_o + ((size_t)r * a.splits + split) * kHeads * kDim;
      for (int u = tid; u < kHeads * kDim; u += blockDim.x) po[u] = 0.f;
      for (int h = tid; h < kHeads; h += blockDim.x) {
        float* ml = a.part_ml + (((size_t)r * a.splits + split) * kHeads + h) * 2;
        ml[0] = -INFINITY;
        ml[1] = 0.f;
      }
    }
    return;
  }

  // ---- query -> shared memory (K-major swizzled, 64 rows)
  const uint16_t* q = static_cast<const uint16_t*>(a.q) + (size_t)r * kHeads * kDim;
  for (int u = tid; u < kHeads * (kDim / 8); u += kTcThreads2) {
    const int h = u / (kDim / 8), c8 = u % (kDim / 8);
    *reinterpret_cast<uint4*>(Qs + tc_chunk_off(h, c8, kHeads)) =
        bf16x8_to_f16x8(*reinterpret_cast<const uint4*>(q + h * kDim + c8 * 8));
  }
  tc::fence_proxy_async_smem();
  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&C.x_full[b], 128);   // the converter threads
      tc::mbar_init(&C.x_empty[b], 1);
      tc::mbar_init(&C.s_full[b], 1);
      tc::mbar_init(&C.s_empty[b], 128);
      tc::mbar_init(&C.win_full[b], 1);
      tc::mbar_init(&C.p_full[b], 128);
      tc::mbar_init(&C.p_empty[b], 1);
    }
    for (int s = 0; s < kRawStages; ++s) {
      tc::mbar_init(&C.raw_full[s], 64);  // per producer lane: its metadata store, then its copies
      tc::mbar_init(&C.raw_empty[s], 128);
    }
    tc::mbar_init(&C.done, 1);
    C.abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0) tc::tmem_alloc(&C.tmem_base, 512);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = C.tmem_base;
  volatile int* abort = &C.abort;

  if (warp == 0) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop converged: descriptors are warp-uniform
    // and one elected lane issues (tc::mma_elect).  Offsets within a tile are
    // compile-time constants added to a base descriptor (the start address
    // field is the low 14 bits, byte address / 16; shared addresses stay
    // below 256 KiB so the sum cannot carry out of it).
    constexpr uint32_t id_qk = tc::idesc_f16_f32_a(64, kTI, 0);
    constexpr uint32_t id_pv = tc::idesc_f16_f32_a(128, kHeads, 1);
    const uint64_t dq = tc::desc_sw128_lbo(tc::smem_u32(Qs), 16, 1024);
    const uint32_t xa = tc::smem_u32(Xs), pa = tc::smem_u32(Ps);
    auto qk = [&](int n) {
      const int b = n & 1;
      tc::tc_fence_after();
      const uint64_t dx = tc::desc_sw128_lbo(xa + b * kTcTileBytes, 16, 1024);
      const uint32_t d0 = tmem + kTcSCol + b * 2 * kTI;
      // content dims (k-blocks 0-7) -> S_c, RoPE dims (k-block 8) -> S_r
#pragma unroll
      for (int kb = 0; kb < kTcKBlocks; ++kb)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc::mma_elect(d0 + (kb == kTcKBlocks - 1 ? kTI : 0), dq + ((kb * (kHeads * 128) + ks * 32) >> 4),
                        dx + ((kb * (kTI * 128) + ks * 32) >> 4), id_qk,
                        (kb == kTcKBlocks - 1 ? ks : (kb | ks)) != 0);
      tc::mma_commit_elect(&C.s_full[b]);
    };
    auto pv = [&](int n) {
      tc::tc_fence_after();
      const uint64_t dx = tc::desc_sw128_lbo(xa + (n & 1) * kTcTileBytes, kTI * 128, 1024);
      const uint64_t dp = tc::desc_sw128_lbo(pa + (n & 1) * kTcPBytes, 16, 1024);
      // chunks 0-3: content dims [128 c, 128 c + 128) with P' = p x scale;
      // chunk 4: the 64 RoPE dims with P (its other 64 rows are not used)
#pragma unroll
      for (int c = 0; c < 5; ++c) {
        const int blk = c < 4 ? 2 * c : kTcKBlocks - 1;
#pragma unroll
        for (int ks = 0; ks < kTI / 16; ++ks)
          tc::mma_elect(tmem + kTcOCol + c * kHeads, dx + ((blk * (kTI * 128) + ks * 2048) >> 4),
                        dp + (((c < 4 ? 0 : 64) + ks * 32) >> 4), id_pv, (n | ks) != 0);
      }
      tc::mma_commit_elect(&C.x_empty[n & 1]);
      tc::mma_commit_elect(&C.p_empty[n & 1]);
    };
    // QK(n + 1) and PV(n) are issued in whichever order their inputs become
    // ready, so neither waits behind the other.  Lane 0 polls and the warp
    // follows its decision; every lane then observes the completed phases
    // itself before the elected lane issues.
    int next_qk = 0, next_pv = 0;
    long long t0 = clock64();
    while (next_pv < ntiles) {
      int st = 0;  // bit 0: QK(next_qk) ready, bit 1: PV(next_pv) ready, bit 2: stop
      if (lane == 0) {
        if (next_qk < ntiles && next_qk <= next_pv + 1 && tc::mbar_test(&C.x_full[next_qk & 1], (next_qk >> 1) & 1) &&
            tc::mbar_test(&C.s_empty[next_qk & 1], ((next_qk >> 1) & 1) ^ 1))
          st |= 1;
        if (next_pv < next_qk && tc::mbar_test(&C.p_full[next_pv & 1], (next_pv >> 1) & 1)) st |= 2;
        if (st) {
          t0 = clock64();
        } else if (*abort) {
          st = 4;
        } else if (clock64() - t0 > tc::kWaitCycles) {
          *abort = 1;
          set_status(a.status, CSA_ERR_TIMEOUT);
          st = 4;
        }
      }
      st = __shfl_sync(0xffffffffu, st, 0);
      if (st & 4) break;
      if (st & 1) {  // these phases cannot move on before this warp's next commit
        tc::mbar_test(&C.x_full[next_qk & 1], (next_qk >> 1) & 1);
        tc::mbar_test(&C.s_empty[next_qk & 1], ((next_qk >> 1) & 1) ^ 1);
        qk(next_qk++);
      }
      if (st & 2) {
        tc::mbar_test(&C.p_full[next_pv & 1], (next_pv >> 1) & 1);
        pv(next_pv++);
      }
    }
    // every MMA this warp issued has completed before TMEM can be freed
    tc::mma_commit_elect(&C.done);
    tc::mbar_wait_warp(&C.done, 0, abort, a.status, false);
  } else if (warp == 1) {
    // ------------------------------------------------------------ producer
    // Compressed tiles only.  Lane j owns item j of every tile: its address
    // takes two dependent lookups (selected index, then page id), run as a
    // software pipeline (index of tile n + 2, page of tile n + 1, copies of
    // tile n).  The copies are 16-byte cp.async operations: one warp
    // instruction moves one item's 512-byte content row (lanes = 16-byte
    // pieces), so the gather stays coalesced; each lane's completion arrives
    // on the stage's barrier.
    const int P = a.kv.page_entries;
    const size_t page_bytes_kv = (size_t)kKvEntryBytes * P;
    auto entry_of = [&](int tile) -> int {  // selected entry of this lane's item, -1 if none
      const int i = i0 + tile * kTI + lane;
      if (tile >= ncomp || i >= it.n_sel) return -1;
      return item_entry(a, it, r, i);
    };
    auto page_base = [&](int e) -> const uint8_t* {
      if (e < 0) return nullptr;
      return a.kv.base + (size_t)a.kv.page_table[(size_t)it.b * a.kv.max_pages + e / P] * page_bytes_kv;
    };
    int e1 = entry_of(0), e2 = entry_of(1);
    const uint8_t* pg1 = page_base(e1);
    for (int n = 0; n < ncomp; ++n) {
      const int e_n = e1;
      const uint8_t* pg_n = pg1;
      e1 = e2;
      pg1 = page_base(e1);
      e2 = entry_of(n + 2);
      const int s = n % kRawStages;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&C.raw_empty[s], ((n / kRawStages) & 1) ^ 1, abort, a.status)))
        break;
      uint8_t* st = Rs + s * kRawStage;
      const int sl = e_n >= 0 ? e_n % P : 0;
      const uint8_t* content = pg_n ? pg_n + (size_t)sl * kKvContent : nullptr;
      const uint8_t* rope = pg_n ? pg_n + (size_t)kKvContent * P + (size_t)sl * (2 * kKvRope) : nullptr;
      const uint8_t* scale = pg_n ? pg_n + (size_t)(kKvContent + 2 * kKvRope) * P + (size_t)sl * 4 : nullptr;
      const uintptr_t sb = reinterpret_cast<uintptr_t>(scale) & ~uintptr_t(15);
      C.meta[s][lane] = pg_n ? (int8_t)((reinterpret_cast<uintptr_t>(scale) - sb) >> 2) : (int8_t)-1;
      tc::mbar_arrive(&C.raw_full[s]);  // releases the metadata store
      // content: item k's row per instruction, lane = 16-byte piece
#pragma unroll 4
      for (int k = 0; k < kTI; ++k) {
        const uint8_t* src = reinterpret_cast<const uint8_t*>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(content), k));
        if (src) tc::cp_async16(st + k * kRawContent + lane * 16, src + lane * 16);
      }
      // RoPE: four items per instruction, 8 pieces each
#pragma unroll
      for (int k4 = 0; k4 < kTI / 4; ++k4) {
        const int k = 4 * k4 + (lane >> 3), piece = lane & 7;
        const uint8_t* src = reinterpret_cast<const uint8_t*>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(rope), k));
        if (src) tc::cp_async16(st + kTI * kRawContent + k * kRawRope + piece * 16, src + piece * 16);
      }
      // the 16-byte block holding the lane's own scale
      if (scale) tc::cp_async16(st + kTI * (kRawContent + kRawRope) + lane * 16, reinterpret_cast<const void*>(sb));
      tc::cp_async_arrive(&C.raw_full[s]);
    }
    // every copy this warp started has landed before the CTA can exit
    for (int n = max(0, ncomp - kRawStages); n < ncomp; ++n)
      if (!tc::mbar_wait(&C.raw_full[n % kRawStages], (n / kRawStages) & 1, abort, a.status, false)) break;
  } else if (warp < 6) {
    // ------------------------------------------------------------ softmax warpgroup
    const int quad = warp & 3;                 // TMEM lanes [32 quad, 32 quad + 32)
    const int h = 16 * quad + lane;            // head of this thread (lane < 16)
    const bool head = lane < 16;
    const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int n = 0; n < ntiles; ++n) {
      const int b = n & 1;
      const int g0 = i0 + n * kTI;
      // the tile's entry scales were written before its x_full arrival
      const bool got = __all_sync(0xffffffffu, tc::mbar_wait(&C.x_full[b], (n >> 1) & 1, abort, a.status) &&
                                                   tc::mbar_wait(&C.s_full[b], (n >> 1) & 1, abort, a.status));
      uint32_t v[32], vr[32];
      if (got) {  // warp-uniform
        tc::tc_fence_after();
        tc::tmem_ld32(tmem + lane_base + kTcSCol + b * 2 * kTI, v);
        tc::tmem_ld32(tmem + lane_base + kTcSCol + b * 2 * kTI + kTI, vr);
        tc::tmem_wait_ld();
        tc::tc_fence_before();
        tc::mbar_arrive(&C.s_empty[b]);
      }
      // real items of the tile: [0, n_sel) and [sel_pad, sel_pad + n_win), both cut at i1
      const uint32_t vmask = range_bits(g0, 0, min(it.n_sel, i1)) | range_bits(g0, sel_pad, min(sel_pad + it.n_win, i1));
      float sc[kTI];  // entry scales, eight 16-byte broadcast loads
#pragma unroll
      for (int q4 = 0; q4 < kTI / 4; ++q4) {
        const float4 f = reinterpret_cast<const float4*>(C.scl[b])[q4];
        sc[4 * q4] = f.x;
        sc[4 * q4 + 1] = f.y;
        sc[4 * q4 + 2] = f.z;
        sc[4 * q4 + 3] = f.w;
      }
      float tmax = -INFINITY;
#pragma unroll
      for (int j = 0; j < kTI; ++j) {
        // logit = scale * (entry scale * q . codes + q_rope . rope)
        const float x = fmaf(__uint_as_float(v[j]), sc[j], __uint_as_float(vr[j])) * a.scale_log2;
        const float y = (vmask >> j) & 1u ? x : -INFINITY;
        v[j] = __float_as_uint(y);
        tmax = fmaxf(tmax, y);
      }
      float corr = 1.f;
      if (head) {
        if (m_ref == -INFINITY) {
          m_ref = tmax;  // the first tile with a valid item
        } else if (tmax > m_ref + kTcRescale) {
          corr = exp2f(m_ref - tmax);
          m_ref = tmax;
        }
        C.corr[b][h] = corr;
      }
      // this tile's P buffer is free once the PV two tiles back has completed
      const bool freed = n < 2 || tc::mbar_wait(&C.p_empty[b], ((n >> 1) & 1) ^ 1, abort, a.status);
      ok = bar_red_and(1, 128, got && freed);
      const bool need = bar_red_or(1, 128, corr != 1.f);
      if (!ok) break;  // uniform over the softmax warpgroup
      // a rescale needs O stable: the previous tile's PV has completed
      if (need && n > 0) ok = bar_red_and(1, 128, tc::mbar_wait(&C.p_empty[b ^ 1], ((n - 1) >> 1) & 1, abort, a.status));
      if (!ok) break;
      tc::tc_fence_after();
      if (need) {
        // O[d][h] *= corr[h] for every head column, all five chunks (this warp's 32 lanes)
#pragma unroll 1
        for (int c = 0; c < 5; ++c)
#pragma unroll 1
          for (int half = 0; half < 2; ++half) {
            uint32_t o[32];
            const uint32_t ta = tmem + lane_base + kTcOCol + c * kHeads + half * 32;
            tc::tmem_ld32(ta, o);
            tc::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * C.corr[b][half * 32 + j]);
            tc::tmem_st32(ta, o);
          }
        tc::tmem_wait_st();
      }
      if (head) {
        // row h of the P buffer: chunks 0-3 hold P' = p x entry scale (content
        // dims), chunks 4-7 hold p (RoPE dims), both FP16
        // an item with logit -inf gives p = 0 (a head with no finite logit yet has m_ref = -inf: use 0)
        const float mr = m_ref == -INFINITY ? 0.f : m_ref;
        float psum = 0.f;
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
          float p[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            p[e] = exp2f(__uint_as_float(v[c8 * 8 + e]) - mr);
            psum += p[e];
          }
          uint4 w, ws;
          w.x = pack_f16x2(p[0], p[1]);
          w.y = pack_f16x2(p[2], p[3]);
          w.z = pack_f16x2(p[4], p[5]);
          w.w = pack_f16x2(p[6], p[7]);
          const float* scc = &sc[c8 * 8];
          ws.x = pack_f16x2(p[0] * scc[0], p[1] * scc[1]);
          ws.y = pack_f16x2(p[2] * scc[2], p[3] * scc[3]);
          ws.z = pack_f16x2(p[4] * scc[4], p[5] * scc[5]);
          ws.w = pack_f16x2(p[6] * scc[6], p[7] * scc[7]);
          *reinterpret_cast<uint4*>(Ps + b * kTcPBytes + tc_chunk_off(h, c8, kHeads)) = ws;
          *reinterpret_cast<uint4*>(Ps + b * kTcPBytes + tc_chunk_off(h, 4 + c8, kHeads)) = w;
        }
        l = l * corr + psum;
      }
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      tc::mbar_arrive(&C.p_full[b]);
    }
    // ---- epilogue: wait for the last PV, then O (lanes = dims) -> output
    const bool last = ok && tc::mbar_wait(&C.p_empty[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1, abort, a.status, false);
    if (head) {
      C.m_ref[h] = m_ref;
      C.l_sum[h] = l;
    }
    ok = bar_red_and(1, 128, last);
    const int hh0 = tid - 64;  // 0..127 over the softmax warpgroup
    if (ok && a.splits == 1 && hh0 < kHeads) C.fin[hh0] = finalize_row(a, r, hh0, C.m_ref[hh0], C.l_sum[hh0]);
    bar_red_and(1, 128, true);
    tc::tc_fence_after();
    if (ok) {
#pragma unroll 1
      for (int c = 0; c < 5; ++c) {
        const int d = (c < 4 ? 128 * c : kKvContent) + 32 * quad + lane;
        const bool write = c < 4 || quad < 2;  // chunk 4: RoPE dims in lanes 0..63
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          uint32_t o[32];
          tc::tmem_ld32(tmem + lane_base + kTcOCol + c * kHeads + half * 32, o);
          tc::tmem_wait_ld();
          if (!write) continue;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int hh = half * 32 + j;
            const float x = __uint_as_float(o[j]);
            if (a.splits == 1) {
              const size_t off = ((size_t)r * kHeads + hh) * kDim + d;
              const float y = x * C.fin[hh];
              if (a.out_bf16) static_cast<uint16_t*>(a.out)[off] = float_to_bf16_bits(y);
              else static_cast<float*>(a.out)[off] = y;
            } else {
              a.part_o[(((size_t)r * a.splits + split) * kHeads + hh) * kDim + d] = x;
            }
          }
        }
      }
      if (a.splits > 1 && hh0 < kHeads) {
        float* ml = a.part_ml + (((size_t)r * a.splits + split) * kHeads + hh0) * 2;
        ml[0] = C.m_ref[hh0];
        ml[1] = C.l_sum[hh0];
      }
    }
  } else {
    // ------------------------------------------------------------ converters
    const int t = tid - 6 * 32;   // 0..127
    const int j = t >> 2, qq = t & 3;  // item row of the tile, quarter
    for (int n = 0; n < ntiles; ++n) {
      const int b = n & 1;
      if (n < ncomp) {
        const int s = n % kRawStages;
        if (!tc::mbar_wait(&C.raw_full[s], (n / kRawStages) & 1, abort, a.status)) break;
        if (!tc::mbar_wait(&C.x_empty[b], ((n >> 1) & 1) ^ 1, abort, a.status)) break;
        const uint8_t* st = Rs + s * kRawStage;
        uint8_t* xt = Xs + b * kTcTileBytes;
        const int mw = C.meta[s][j];
        if (mw >= 0) {
          // content: the e4m3 codes as FP16 (exact; the entry scale is applied
          // to the logit and to P); RoPE dims BF16 -> FP16
          if (qq == 0) C.scl[b][j] = reinterpret_cast<const float*>(st + kTI * (kRawContent + kRawRope) + j * 16)[mw];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int c16 = 4 * u + qq;  // 16 content bytes = dims 16 c16 .. 16 c16 + 15
            const uint4 raw = *reinterpret_cast<const uint4*>(st + j * kRawContent + c16 * 16);
            *reinterpret_cast<uint4*>(xt + tc_chunk_off(j, 2 * c16, kTI)) = fp8x8_to_f16x8(raw, false);
            *reinterpret_cast<uint4*>(xt + tc_chunk_off(j, 2 * c16 + 1, kTI)) = fp8x8_to_f16x8(raw, true);
          }
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int c16 = 4 * u + qq;
            *reinterpret_cast<uint4*>(xt + tc_chunk_off(j, 64 + c16, kTI)) =
                bf16x8_to_f16x8(*reinterpret_cast<const uint4*>(st + kTI * kRawContent + j * kRawRope + c16 * 16));
          }
        } else {
          if (qq == 0) C.scl[b][j] = 0.f;
          const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int u = 0; u < 18; ++u) *reinterpret_cast<uint4*>(xt + tc_chunk_off(j, 4 * u + qq, kTI)) = z;
        }
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(&C.raw_empty[s]);
        tc::mbar_arrive(&C.x_full[b]);
      } else {
        // window tile: BF16 rows by TMA straight into the swizzled X tile
        const int wi = n - ncomp;
        if (!tc::mbar_wait(&C.x_empty[b], ((n >> 1) & 1) ^ 1, abort, a.status)) break;
        if (t == 0) {
          const int w = (i0 + n * kTI - sel_pad) / kTI;
          const int row0 = win_dense ? it.t - it.n_win + 1 + kTI * w : kTI * w;
          uint8_t* xt = Xs + b * kTcTileBytes;
          tc::mbar_arrive_expect_tx(&C.win_full[b], kTcTileBytes);
          for (int kb = 0; kb < kTcKBlocks; ++kb)
            tma_load_3d(xt + kb * (kTI * 128), &win_map, 64 * kb, row0, it.b, &C.win_full[b]);
        }
        if (!tc::mbar_wait(&C.win_full[b], (wi >> 1) & 1, abort, a.status, t == 0 ? false : true)) break;
        // the window rows arrive as BF16: convert the tile to FP16 in place
        uint8_t* xt = Xs + b * kTcTileBytes;
#pragma unroll 2
        for (int c = t; c < kTcTileBytes / 16; c += 128) {
          uint4* pc = reinterpret_cast<uint4*>(xt + c * 16);
          *pc = bf16x8_to_f16x8(*pc);
        }
        if (t < kTI) C.scl[b][t] = 1.f;
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(&C.x_full[b]);
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

// ================================================================== split combine

constexpr int kMaxSplits = 64;

__global__ void __launch_bounds__(128) combine_kernel(AttArgs a) {
  const int r = blockIdx.x, h = blockIdx.y, S = a.splits, D = a.D, H = a.H;
  __shared__ float ms_s[kMaxSplits], ls_s[kMaxSplits], wgt[kMaxSplits];
  __shared__ float inv_s;
  // every split's (running max, sum), loaded in parallel
  for (int s = threadIdx.x; s < S; s += blockDim.x) {
    const float* ml = a.part_ml + (((size_t)r * S + s) * H + h) * 2;
    ms_s[s] = ml[0];
    ls_s[s] = ml[1];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) M = fmaxf(M, ms_s[s]);
    float l = 0.f;
    for (int s = 0; s < S; ++s) {
      const float w = (ls_s[s] > 0.f) ? exp2f(ms_s[s] - M) : 0.f;
      wgt[s] = w;
      l += w * ls_s[s];
    }
    inv_s = finalize_row(a, r, h, M, l);
  }
  __syncthreads();
  const float inv = inv_s;
  const float* po = a.part_o + ((size_t)r * S * H + h) * D;  // split s at + s * H * D
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float acc = 0.f;
#pragma unroll 8
    for (int s = 0; s < S; ++s) acc = fmaf(wgt[s], po[(size_t)s * H * D + d], acc);
    const float v = acc * inv;
    const size_t off = ((size_t)r * H + h) * D + d;
    if (a.out_bf16) static_cast<uint16_t*>(a.out)[off] = float_to_bf16_bits(v);
    else static_cast<float*>(a.out)[off] = v;
  }
}

// ------------------------------------------------------------------ host


// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      ptr = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }();
  return fn;
}

struct Plan {
  int splits, items_per_split, tile;
  bool mma;
};

int plan(const csa_attend_params* p, bool sparse, Plan* pl) {
  CSA_CHECK(p != nullptr && p->struct_size >= sizeof(csa_attend_params), CSA_ERR_INVALID_ARG);
  CSA_CHECK(p->num_queries >= 0 && p->batch >= 1 && p->m >= 1 && p->window >= 0 && p->max_pos >= 0,
            CSA_ERR_SHAPE);
  CSA_CHECK(p->heads >= 1 && p->dim >= 1, CSA_ERR_SHAPE);
  CSA_CHECK(p->win_ring >= 1, CSA_ERR_SHAPE);
  const int64_t nmax = (int64_t)(p->max_pos + 1) / p->m;
  int64_t Lmax = (sparse ? std::min<int64_t>(p->top_k, nmax) : nmax) + std::min<int64_t>(p->window, p->max_pos + 1);
  if (p->kv.format == CSA_FMT_KV_POOL_FP8)  // compressed items padded to a whole tile, then the window
    Lmax = ((sparse ? std::min<int64_t>(p->top_k, nmax) : nmax) + kTI - 1) / kTI * kTI +
           std::min<int64_t>(p->window, p->max_pos + 1);
  if (p->kv.format == CSA_FMT_DENSE_F32) {
    CSA_CHECK(p->q_dtype == CSA_F32 && p->win_dtype == CSA_F32 && p->out_dtype == CSA_F32, CSA_ERR_UNSUPPORTED);
    CSA_CHECK(p->kv.dim == p->dim && p->heads * p->dim <= kF32Threads * kF32MaxPer, CSA_ERR_UNSUPPORTED);
    pl->mma = false;
    pl->tile = kF32Tile;
  } else if (p->kv.format == CSA_FMT_KV_POOL_FP8) {
    CSA_CHECK(p->q_dtype == CSA_BF16 && p->win_dtype == CSA_BF16, CSA_ERR_UNSUPPORTED);
    CSA_CHECK(p->out_dtype == CSA_BF16 || p->out_dtype == CSA_F32, CSA_ERR_UNSUPPORTED);
    CSA_CHECK(p->heads == kHeads && p->dim == kDim, CSA_ERR_UNSUPPORTED);
    // window source: an exact ring of W rows, or a raw sequence covering every position
    CSA_CHECK(p->win_ring == p->window || p->win_ring >= p->max_pos + 1, CSA_ERR_UNSUPPORTED);
    pl->mma = true;
    pl->tile = kTI;
  } else {
    return CSA_ERR_UNSUPPORTED;
  }
  // split-K: enough CTAs to cover the SMs, each split at least 4 tiles
  const int T = std::max(p->num_queries, 1);
  const int64_t tiles = std::max<int64_t>(1, (Lmax + pl->tile - 1) / pl->tile);
  int splits = (int)std::max<int64_t>(1, std::min<int64_t>({(int64_t)sm_count() / T, (tiles + 3) / 4, kMaxSplits}));
  int64_t ips = (tiles + splits - 1) / splits * pl->tile;
  splits = (int)((Lmax + ips - 1) / ips);
  pl->splits = std::max(1, splits);
  pl->items_per_split = (int)ips;
  return CSA_OK;
}

int check_attend(const csa_attend_params* p, bool sparse, Plan* pl) {
  int st = plan(p, sparse, pl);
  if (st != CSA_OK) return st;
  if (p->num_queries == 0) return CSA_OK;
  CSA_CHECK(p->q && p->pos && p->out && p->win, CSA_ERR_INVALID_ARG);
  if (sparse) CSA_CHECK(p->idx && p->cnt && p->top_k >= 0, CSA_ERR_INVALID_ARG);
  CSA_CHECK(aligned(p->q, 16) && aligned(p->out, 16) && aligned(p->win, 16) && aligned(p->pos, 4) &&
                (!p->seq || aligned(p->seq, 4)) && (!p->lse || aligned(p->lse, 4)) &&
                (!p->sink || aligned(p->sink, 4)) && (!sparse || (aligned(p->idx, 4) && aligned(p->cnt, 4))),
            CSA_ERR_ALIGN);
  const int64_t nmax = (int64_t)(p->max_pos + 1) / p->m;
  return check_store(p->kv, p->batch, nmax);
}

size_t workspace_bytes(const csa_attend_params* p, const Plan& pl) {
  if (pl.splits <= 1) return kWsHeader;
  const size_t T = p->num_queries, S = pl.splits, H = p->heads, D = p->dim;
  return kWsHeader + T * S * H * D * sizeof(float) + T * S * H * 2 * sizeof(float);
}

int run(const csa_attend_params* p, bool sparse, void* ws, size_t ws_bytes, cudaStream_t s) {
  Plan pl;
  int st = check_attend(p, sparse, &pl);
  if (st != CSA_OK) return st;
  if (p->num_queries == 0) return CSA_OK;
  CSA_CHECK(ws != nullptr && aligned(ws, 1024), ws ? CSA_ERR_ALIGN : CSA_ERR_WORKSPACE);
  CSA_CHECK(ws_bytes >= workspace_bytes(p, pl), CSA_ERR_WORKSPACE);
  AttArgs a{};
  a.q = p->q;
  a.pos = p->pos;
  a.seq = p->seq;
  a.idx = sparse ? p->idx : nullptr;
  a.cnt = sparse ? p->cnt : nullptr;
  a.top_k = sparse ? p->top_k : 0;
  a.m = p->m;
  a.window = p->window;
  a.T = p->num_queries;
  a.H = p->heads;
  a.D = p->dim;
  a.splits = pl.splits;
  a.items_per_split = pl.items_per_split;
  a.kv = to_device(p->kv);
  a.kv_cap = p->kv.format == CSA_FMT_DENSE_F32 ? p->kv.capacity : p->kv.max_pages * p->kv.page_entries;
  a.win = p->win;
  a.win_ring = p->win_ring;
  a.scale_log2 = p->scale * kLog2e;
  a.sink = p->sink;
  a.out = p->out;
  a.out_bf16 = p->out_dtype == CSA_BF16;
  a.lse = p->lse;
  a.status = static_cast<int*>(ws);
  uint8_t* w8 = static_cast<uint8_t*>(ws) + kWsHeader;
  a.part_o = reinterpret_cast<float*>(w8);
  a.part_ml = reinterpret_cast<float*>(w8 + (size_t)p->num_queries * pl.splits * p->heads * p->dim * sizeof(float));
  CSA_CHECK(p->num_queries <= 2147483647 && pl.splits <= 65535, CSA_ERR_SHAPE);
  const dim3 grid(p->num_queries, pl.splits);
  if (pl.mma) {
    // TMA descriptor of the window source: [batch][win_ring][576] BF16, boxes
    // of 64 dims x 32 rows, 128-byte swizzle (the layout of an X tile block)
    CUtensorMap win_map;
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    CSA_CHECK(encode != nullptr, CSA_ERR_CUDA);
    const cuuint64_t dims[3] = {(cuuint64_t)kDim, (cuuint64_t)p->win_ring, (cuuint64_t)p->batch};
    const cuuint64_t strides[2] = {(cuuint64_t)kDim * 2, (cuuint64_t)p->win_ring * kDim * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)kTI, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CSA_CHECK(encode(&win_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p->win), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS,
              CSA_ERR_INVALID_ARG);
    const int win_dense = p->win_ring >= p->max_pos + 1 ? 1 : 0;
    cudaFuncSetAttribute(attend_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemBytes);
    attend_tc_kernel<<<grid, kTcThreads2, kTcSmemBytes, s>>>(a, win_map, win_dense);
  } else {
    const size_t smem = ((size_t)p->heads * (p->dim + 1) + kF32Tile * (p->dim + 1) + p->heads * kF32Tile + 3 * p->heads) *
                        sizeof(float);
    CSA_CHECK(smem <= 200 * 1024, CSA_ERR_UNSUPPORTED);
    cudaFuncSetAttribute(attend_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    attend_f32_kernel<<<grid, kF32Threads, smem, s>>>(a);
  }
  st = launch_status();
  if (st != CSA_OK || pl.splits == 1) return st;
  combine_kernel<<<dim3(p->num_queries, p->heads), 128, 0, s>>>(a);
  return launch_status();
}

}  // namespace
}  // namespace csa

using namespace csa;

extern "C" size_t csa_attend_workspace_size(const csa_attend_params* p) {
  Plan pl;
  if (check_attend(p, true, &pl) != CSA_OK) return 0;
  return workspace_bytes(p, pl);
}

extern "C" size_t hca_attend_workspace_size(const csa_attend_params* p) {
  Plan pl;
  if (check_attend(p, false, &pl) != CSA_OK) return 0;
  return workspace_bytes(p, pl);
}

extern "C" int csa_attend(const csa_attend_params* p, void* ws, size_t ws_bytes, csa_stream_t stream) {
  return run(p, true, ws, ws_bytes, (cudaStream_t)stream);
}

extern "C" int hca_attend(const csa_attend_params* p, void* ws, size_t ws_bytes, csa_stream_t stream) {
  return run(p, false, ws, ws_bytes, (cudaStream_t)stream);
}
