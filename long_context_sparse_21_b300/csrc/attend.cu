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
//                        entries gathered into registers by converter warps
//                        and written as FP16 tiles (exact e4m3 codes), window
//                        rows loaded by TMA.
//  * combine_kernel      log-sum-exp merge of split partials.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>

#include <cooperative_groups.h>

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
  int top_k, m, window, T, H, D, splits, items_per_split, batch;
  int invariant;       // split boundaries from each query's own item count (batch-invariant results)
  int merge;           // kMergeDirect, kMergeCluster or kMergeGlobal
  int window_only;     // no compressed branch (kv_cap is 0 and no store is read)
  const float* q_norm;   // RMSNorm gain of the query heads, or NULL
  const float* win_norm; // RMSNorm gain of the window rows, or NULL
  float norm_eps;
  int rope;              // RoPE: query at t, window rows at their positions, output back by t
  RopeFreq freq;
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

// How the splits of a query are merged: a single split writes its output
// directly; the splits of a query launched as one thread-block cluster merge
// their partials (kept in L2) after one cluster barrier, each CTA writing a
// slice of the output; otherwise partials go to the workspace and
// combine_kernel merges them.
constexpr int kMergeDirect = 0, kMergeCluster = 1, kMergeGlobal = 2;
constexpr int kMaxClusterSplits = 8;      // a portable cluster
constexpr int kInvTilesPerSplit = 5;      // batch-invariant plan: about 5 tiles of 32 items per split

// Item list of query r: [0, n_sel) compressed entries, then the window.
struct Items {
  int b, t, n_sel, nvis, n_win, L;
};

// A sequence index outside [0, batch) makes the query's item list empty (its
// output row is zero) and records CSA_ERR_INVALID_ARG.
__device__ __forceinline__ Items query_items(const AttArgs& a, int r) {
  Items it;
  it.b = a.seq ? a.seq[r] : r;
  it.t = a.pos[r];
  if ((unsigned)it.b >= (unsigned)a.batch) {
    if (threadIdx.x == 0) set_status(a.status, CSA_ERR_INVALID_ARG);
    it.b = 0;
    it.t = -1;
  }
  it.nvis = min(n_visible(it.t, a.m), a.kv_cap);
  it.n_sel = a.idx ? min(max(a.cnt[r], 0), a.top_k) : it.nvis;
  if (it.t < 0 || a.window_only) it.n_sel = 0;
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

// Items [i0, i1) of split `split` in a query's (padded) item list of Lp
// items.  Batch-invariant plan: the query's own tile count fixes the number
// of splits, min(splits of the launch, ceil(tiles / kInvTilesPerSplit)), and
// their boundaries, so the same query gives the same splits (and the same
// bits) in any batch; splits past its own count are empty.  Otherwise every
// query uses the launch's items_per_split.
__device__ __forceinline__ void split_range(const AttArgs& a, int Lp, int split, int* i0, int* i1) {
  int ips = a.items_per_split;
  if (a.invariant) {
    const int tiles = (Lp + 31) / 32;
    const int ns = min(a.splits, max(1, (tiles + kInvTilesPerSplit - 1) / kInvTilesPerSplit));
    ips = (tiles + ns - 1) / ns * 32;
  }
  *i0 = split * ips;
  *i1 = min(Lp, *i0 + ips);
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
  tc::pdl_wait();
  tc::pdl_trigger();
  const Items it = query_items(a, r);
  int i0, i1;
  split_range(a, it.L, split, &i0, &i1);
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
// the window rows.  Three FP16 X tiles are in flight.  Warp roles:
//   MMA warp (converged; one elected lane issues):
//              S[64 heads x 32 items] = Q . X^T      (tcgen05 M=64, N=32, K=576;
//              content dims -> S_c, RoPE dims -> S_r, two TMEM buffers)
//              O[576 dims x 64 heads] += X^T . P^T   (M=128 per 128-dim chunk,
//              X read MN-major from the same tile, N=64, K=32)
//              in the fixed order QK(0), QK(1), then PV(n), QK(n + 2).
//   producer warp: resolves each item of a compressed tile (selected index,
//              page id) into (page, slot) in an address ring.
//   converter warps (4): load each item's FP8 content, RoPE row and scale
//              into registers two tiles ahead, and write the X tile (e4m3
//              codes as FP16, exactly; RoPE BF16 -> FP16), 128-byte swizzled
//              K-major, plus the tile's entry scales; a window tile (BF16
//              rows) comes by TMA and is converted to FP16 in place.
//   softmax warps (4): 16x256b TMEM loads give each thread two heads x 8
//              items; logit = scale_log2 (entry scale x S_c + S_r); a
//              running reference max per head; P (RoPE dims) and P x entry
//              scale (content dims) written as FP16 pairs.
// The reference max only moves when a tile's max exceeds it by more than 2^8;
// then O's column of that head is rescaled in TMEM before the tile's PV runs.
// The 576 output dims are covered by five 128-row chunks; the fifth holds
// the 64 RoPE dims in its first 64 rows (its other rows are not used).
constexpr int kTI = 32;                       // items per tile
constexpr int kTcWarps = 1 + 1 + 4 + 4;       // MMA, producer, softmax x4, converters x4
constexpr int kTcThreads2 = kTcWarps * 32;
constexpr int kTcKBlocks = kDim / 64;         // 9
constexpr int kTcTileBytes = kTcKBlocks * kTI * 128;   // 36864
constexpr int kTcQBytes = kTcKBlocks * kHeads * 128;   // 73728
constexpr int kTcPBytes = kHeads * 128;                // 8192 (32 of 64 columns used)
constexpr int kXBufs = 3;                              // X tiles in flight
constexpr int kMetaStages = 4;                         // producer -> converter address ring
constexpr int kTcSmemBytes = kTcQBytes + kXBufs * kTcTileBytes + 2 * kTcPBytes;
constexpr uint32_t kTcSCol = 0;      // S buffers: columns [0, 128): per buffer S_content, S_rope
constexpr uint32_t kTcOCol = 128;    // O: columns [128, 448)
constexpr float kTcRescale = 8.0f;   // log2 headroom before the reference max moves
constexpr int kPtCache = 256;        // page ids of a sequence kept in shared memory

struct TcCtl {
  uint64_t x_full[kXBufs], x_empty[kXBufs], win_full[kXBufs];
  uint64_t s_full[2], s_empty[2], p_full[2], p_empty[2], done;
  uint64_t q_full, q_ready;
  uint64_t meta_full[kMetaStages], meta_empty[kMetaStages];
  uint32_t tmem_base;
  int abort;
  const uint8_t* page[kMetaStages][kTI];  // per item of a compressed tile: its KV page (nullptr: none)
  int slot[kMetaStages][kTI];             // and its slot in the page
  alignas(16) float scl[kXBufs][kTI];     // per X-tile item: its entry scale (1 for window rows)
  float corr[2][kHeads];
  float m_ref[kHeads];
  float l_sum[kHeads];
  float fin[kHeads];
  float2 rope_t[kRopePairs];  // (cos, sin) of t f_i for the query position t
  int tiles_ok;                          // cluster merge: this CTA's O, m_ref and l_sum are complete
  float wgt[kMaxClusterSplits][kHeads];  // and the weight of every split
  int pt[kPtCache];                      // the first page ids of the query's sequence
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

// 8 BF16 values -> floats; the sum of their squares.
__device__ __forceinline__ void bf16x8_unpack(uint4 v, float (&x)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ float bf16x8_sumsq(uint4 v) {
  float x[8];
  bf16x8_unpack(v, x);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) s = fmaf(x[i], x[i], s);
  return s;
}
// 1 / sqrt(mean of squares + eps) over the 576 dims, 0 for an all-zero row
// without eps (a padding row of a tile).
__device__ __forceinline__ float rms_inv(float ss, float eps) {
  return (ss > 0.f || eps > 0.f) ? 1.0f / sqrtf(ss / (float)kDim + eps) : 0.f;
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
    attend_tc_kernel(AttArgs a, const __grid_constant__ CUtensorMap win_map, const __grid_constant__ CUtensorMap q_map,
                     int win_dense) {
  extern __shared__ __align__(1024) uint8_t tc_smem[];
  __shared__ TcCtl C;
  uint8_t* Qs = tc_smem;
  uint8_t* Xs = tc_smem + kTcQBytes;        // kXBufs tiles
  uint8_t* Ps = Xs + kXBufs * kTcTileBytes;  // two P buffers
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = blockIdx.x, split = blockIdx.y;

  if ((tc::smem_u32(tc_smem) & 1023u) != 0) {  // the swizzled operands need 1 KiB alignment (uniform over the launch)
    tc::pdl_wait();
    if (tid == 0) set_status(a.status, CSA_ERR_ALIGN);
    return;
  }
  // ---- prologue that reads nothing an earlier kernel of the stream may still
  // be writing: barriers, TMEM, and the query (an input of the step), which
  // one thread fetches by TMA (9 boxes of 64 dims x 64 heads, 128-byte
  // swizzled: the K-major operand layout); the softmax warps convert it to
  // FP16 in place once it has landed.
  if (tid == 0) {
    for (int b = 0; b < kXBufs; ++b) {
      tc::mbar_init(&C.x_full[b], 128);   // the converter threads
      tc::mbar_init(&C.x_empty[b], 1);
      tc::mbar_init(&C.win_full[b], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&C.s_full[b], 1);
      tc::mbar_init(&C.s_empty[b], 128);
      tc::mbar_init(&C.p_full[b], 128);
      tc::mbar_init(&C.p_empty[b], 1);
    }
    for (int s = 0; s < kMetaStages; ++s) {
      tc::mbar_init(&C.meta_full[s], 1);   // producer lane 0, after the warp's stores
      tc::mbar_init(&C.meta_empty[s], 4);  // one arrival per converter warp
    }
    tc::mbar_init(&C.done, 1);
    tc::mbar_init(&C.q_full, 1);
    tc::mbar_init(&C.q_ready, 128);        // the softmax threads, after the conversion
    C.abort = 0;
    C.tiles_ok = 0;
    tc::fence_mbar_init();
    tc::mbar_arrive_expect_tx(&C.q_full, kTcQBytes);
    for (int kb = 0; kb < kTcKBlocks; ++kb)
      tc::tma_load_2d(Qs + kb * (kHeads * 128), &q_map, 64 * kb, r * kHeads, &C.q_full);
  }
  if (warp == 0) tc::tmem_alloc(&C.tmem_base, 512);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = C.tmem_base;
  volatile int* abort = &C.abort;
  // from here on the kernel reads the outputs of earlier kernels (selection,
  // cache pages, window ring)
  tc::pdl_wait();
  tc::pdl_trigger();

  const Items it = query_items(a, r);
  const int sel_pad = (it.n_sel + kTI - 1) / kTI * kTI;
  const int Lp = sel_pad + it.n_win;          // padded item count
  int i0, i1;
  split_range(a, Lp, split, &i0, &i1);
  const int ntiles = i1 > i0 ? (i1 - i0 + kTI - 1) / kTI : 0;
  const int ncomp = i1 > i0 ? max(0, min(ntiles, (sel_pad - i0 + kTI - 1) / kTI)) : 0;  // compressed tiles first
  if (a.rope) {  // uniform over the launch
    if (tid < kRopePairs) C.rope_t[tid] = rope_cs(a.freq.f[tid], it.t);
    __syncthreads();
  }

  if (ntiles == 0) {
    // empty split: no item; the query's TMA must land before the CTA exits
    tc::mbar_wait(&C.q_full, 0, abort, a.status, false);
    if (a.merge != kMergeCluster) {
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
    } else if (tid < kHeads) {
      C.m_ref[tid] = -INFINITY;
      C.l_sum[tid] = 0.f;
    }
  } else if (warp == 0) {
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
      const uint64_t dx = tc::desc_sw128_lbo(xa + (n % kXBufs) * kTcTileBytes, 16, 1024);
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
      const uint64_t dx = tc::desc_sw128_lbo(xa + (n % kXBufs) * kTcTileBytes, kTI * 128, 1024);
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
      tc::mma_commit_elect(&C.x_empty[n % kXBufs]);
      tc::mma_commit_elect(&C.p_empty[n & 1]);
    };
    // Fixed order QK(0), QK(1), then PV(n), QK(n + 2) for n = 0, 1, ...:
    // PV(n) waits for the softmax of tile n, which has by then released S
    // buffer n % 2 for QK(n + 2); every wait is on one barrier, spun by the
    // whole warp (every lane observes the phase before the elected lane
    // issues).
    auto qk_ready = [&](int m) {
      return tc::mbar_wait_warp(&C.x_full[m % kXBufs], (m / kXBufs) & 1, abort, a.status) &&
             tc::mbar_wait_warp(&C.s_empty[m & 1], ((m >> 1) & 1) ^ 1, abort, a.status);
    };
    // the query must be in FP16 before the first QK
    bool ok = tc::mbar_wait_warp(&C.q_ready, 0, abort, a.status);
    for (int m = 0; ok && m < min(2, ntiles); ++m) {
      ok = qk_ready(m);
      if (ok) qk(m);
    }
    for (int n = 0; ok && n < ntiles; ++n) {
      ok = tc::mbar_wait_warp(&C.p_full[n & 1], (n >> 1) & 1, abort, a.status);
      if (!ok) break;
      pv(n);
      if (n + 2 < ntiles) {
        ok = qk_ready(n + 2);
        if (ok) qk(n + 2);
      }
    }
    // every MMA this warp issued has completed before TMEM can be freed
    tc::mma_commit_elect(&C.done);
    tc::mbar_wait_warp(&C.done, 0, abort, a.status, false);
  } else if (warp == 1) {
    // ------------------------------------------------------------ producer
    // Addresses of the compressed tiles only.  Lane j resolves item j of each
    // tile (selected index, then page id: two dependent loads, run as a
    // software pipeline: index of tile n + 2, page of tile n + 1) and
    // publishes (page, slot) to the address ring, up to kMetaStages tiles
    // ahead of the converters.
    const int P = a.kv.page_entries;
    const size_t page_bytes_kv = (size_t)kKvEntryBytes * P;
    auto entry_of = [&](int tile) -> int {  // selected entry of this lane's item, -1 if none
      const int i = i0 + tile * kTI + lane;
      if (tile >= ncomp || i >= it.n_sel) return -1;
      return item_entry(a, it, r, i);
    };
    auto page_base = [&](int e) -> const uint8_t* {
      if (e < 0) return nullptr;
      const int pgi = e / P;
      const int pg = pgi < kPtCache ? C.pt[pgi] : a.kv.page_table[(size_t)it.b * a.kv.max_pages + pgi];
      if ((unsigned)pg >= (unsigned)a.kv.num_pages) {  // outside the pool: the item reads as zeros
        set_status(a.status, CSA_ERR_INVALID_ARG);
        return nullptr;
      }
      return a.kv.base + (size_t)pg * page_bytes_kv;
    };
    // the page-table row of the sequence goes to shared memory, loaded
    // together with the first selected indices
    int pv[kPtCache / 32];
#pragma unroll
    for (int u = 0; u < kPtCache / 32; ++u) {
      const int i = lane + 32 * u;
      pv[u] = ncomp > 0 && i < a.kv.max_pages ? a.kv.page_table[(size_t)it.b * a.kv.max_pages + i] : 0;
    }
    int e1 = entry_of(0), e2 = entry_of(1);
#pragma unroll
    for (int u = 0; u < kPtCache / 32; ++u) C.pt[lane + 32 * u] = pv[u];
    __syncwarp();
    const uint8_t* pg1 = page_base(e1);
    for (int n = 0; n < ncomp; ++n) {
      const int e_n = e1;
      const uint8_t* pg_n = pg1;
      e1 = e2;
      pg1 = page_base(e1);
      e2 = entry_of(n + 2);
      const int s = n % kMetaStages;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&C.meta_empty[s], ((n / kMetaStages) & 1) ^ 1, abort, a.status)))
        break;
      C.page[s][lane] = pg_n;
      C.slot[s][lane] = e_n >= 0 ? e_n % P : 0;
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&C.meta_full[s]);  // releases the warp's stores
    }
  } else if (warp < 6) {
    // ------------------------------------------------------------ softmax warpgroup
    // S (M=64 heads) sits in TMEM lanes 32 quad .. 32 quad + 15 of this
    // warp's quadrant (rows 16 quad ..).  A 16x256b load gives thread t the
    // heads hA = 16 quad + t / 4 and hB = hA + 8, and for each of them the
    // item pairs (8 g + 2 c, 8 g + 2 c + 1), c = t % 4, g = 0..3: every lane
    // works, a head's 32 items are spread over 4 adjacent threads, and the
    // pairs pack straight into the FP16 P rows.
    const int quad = warp & 3;
    const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
    const int c = lane & 3;
    const int hA = 16 * quad + (lane >> 2), hB = hA + 8;
    float m_ref[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    // the query has landed as BF16 (the TMA keeps each 16-byte chunk in its
    // swizzled place): convert it to FP16 in place, then release the MMA warp
    bool ok = bar_red_and(1, 128, tc::mbar_wait(&C.q_full, 0, abort, a.status));
    if (ok && (a.q_norm || a.rope)) {
      // two threads per head, 36 of its 72 chunks each: RMSNorm over the
      // 576 dims, then RoPE of the last 64 at t, in float32
      const int u = tid - 64, h = u >> 1, c_lo = (u & 1) * 36;
      float ss = 0.f;
      for (int c8 = c_lo; c8 < c_lo + 36; ++c8) {
        const uint4 v = *reinterpret_cast<const uint4*>(Qs + tc_chunk_off(h, c8, kHeads));
        ss += bf16x8_sumsq(v);
      }
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      const float inv = a.q_norm ? rms_inv(ss, a.norm_eps) : 1.f;
      for (int c8 = c_lo; c8 < c_lo + 36; ++c8) {
        uint4* pc = reinterpret_cast<uint4*>(Qs + tc_chunk_off(h, c8, kHeads));
        float x[8];
        bf16x8_unpack(*pc, x);
        if (a.q_norm)
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] *= inv * a.q_norm[8 * c8 + e];
        if (a.rope && c8 >= kKvContent / 8)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 v = rotate_pair(x[2 * e], x[2 * e + 1], C.rope_t[4 * (c8 - kKvContent / 8) + e]);
            x[2 * e] = v.x;
            x[2 * e + 1] = v.y;
          }
        *pc = make_uint4(pack_f16x2(x[0], x[1]), pack_f16x2(x[2], x[3]), pack_f16x2(x[4], x[5]),
                         pack_f16x2(x[6], x[7]));
      }
      tc::fence_proxy_async_smem();
    } else if (ok) {
      for (int c = tid - 64; c < kTcQBytes / 16; c += 128) {
        uint4* pc = reinterpret_cast<uint4*>(Qs + c * 16);
        *pc = bf16x8_to_f16x8(*pc);
      }
      tc::fence_proxy_async_smem();
    }
    tc::mbar_arrive(&C.q_ready);
    for (int n = 0; ok && n < ntiles; ++n) {
      const int b = n & 1, xb = n % kXBufs;
      const int g0 = i0 + n * kTI;
      // the tile's entry scales were written before its x_full arrival
      const bool got = __all_sync(0xffffffffu, tc::mbar_wait(&C.x_full[xb], (n / kXBufs) & 1, abort, a.status) &&
                                                   tc::mbar_wait(&C.s_full[b], (n >> 1) & 1, abort, a.status));
      uint32_t v[16], vr[16];  // [4 g + 2 head + e]: item 8 g + 2 c + e of head (hA, hB)
      if (got) {  // warp-uniform
        tc::tc_fence_after();
        tc::tmem_ld16x256(tmem + lane_base + kTcSCol + b * 2 * kTI, v);
        tc::tmem_ld16x256(tmem + lane_base + kTcSCol + b * 2 * kTI + kTI, vr);
        tc::tmem_wait_ld();
        tc::tc_fence_before();
        tc::mbar_arrive(&C.s_empty[b]);
      }
      // real items of the tile: [0, n_sel) and [sel_pad, sel_pad + n_win), both cut at i1
      const uint32_t vmask = range_bits(g0, 0, min(it.n_sel, i1)) | range_bits(g0, sel_pad, min(sel_pad + it.n_win, i1));
      float sc[8];  // entry scales of items 8 g + 2 c + e
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const float2 f = *reinterpret_cast<const float2*>(&C.scl[xb][8 * g + 2 * c]);
        sc[2 * g] = f.x;
        sc[2 * g + 1] = f.y;
      }
      float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int g = 0; g < 4; ++g)
#pragma unroll
        for (int hd = 0; hd < 2; ++hd)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int k = 4 * g + 2 * hd + e, item = 8 * g + 2 * c + e;
            // logit = scale * (entry scale * q . codes + q_rope . rope)
            const float x = fmaf(__uint_as_float(v[k]), sc[2 * g + e], __uint_as_float(vr[k])) * a.scale_log2;
            const float y = (vmask >> item) & 1u ? x : -INFINITY;
            v[k] = __float_as_uint(y);
            tmax[hd] = fmaxf(tmax[hd], y);
          }
      float corr[2] = {1.f, 1.f};
#pragma unroll
      for (int hd = 0; hd < 2; ++hd) {
        tmax[hd] = fmaxf(tmax[hd], __shfl_xor_sync(0xffffffffu, tmax[hd], 1));
        tmax[hd] = fmaxf(tmax[hd], __shfl_xor_sync(0xffffffffu, tmax[hd], 2));
        if (m_ref[hd] == -INFINITY) {
          m_ref[hd] = tmax[hd];  // the first tile with a valid item
        } else if (tmax[hd] > m_ref[hd] + kTcRescale) {
          corr[hd] = exp2f(m_ref[hd] - tmax[hd]);
          m_ref[hd] = tmax[hd];
        }
      }
      if (c == 0) {
        C.corr[b][hA] = corr[0];
        C.corr[b][hB] = corr[1];
      }
      // this tile's P buffer is free once the PV two tiles back has completed
      const bool freed = n < 2 || tc::mbar_wait(&C.p_empty[b], ((n >> 1) & 1) ^ 1, abort, a.status);
      ok = bar_red_and(1, 128, got && freed);
      const bool need = bar_red_or(1, 128, corr[0] != 1.f || corr[1] != 1.f);
      if (!ok) break;  // uniform over the softmax warpgroup
      // a rescale needs O stable: the previous tile's PV has completed
      if (need && n > 0) ok = bar_red_and(1, 128, tc::mbar_wait(&C.p_empty[b ^ 1], ((n - 1) >> 1) & 1, abort, a.status));
      if (!ok) break;
      tc::tc_fence_after();
      if (need) {
        // O[d][h] *= corr[h] for every head column, all five chunks (this warp's 32 lanes)
#pragma unroll 1
        for (int ch = 0; ch < 5; ++ch)
#pragma unroll 1
          for (int half = 0; half < 2; ++half) {
            uint32_t o[32];
            const uint32_t ta = tmem + lane_base + kTcOCol + ch * kHeads + half * 32;
            tc::tmem_ld32(ta, o);
            tc::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * C.corr[b][half * 32 + j]);
            tc::tmem_st32(ta, o);
          }
        tc::tmem_wait_st();
      }
      // P rows: chunk g (items 8 g .. 8 g + 7) of row h holds P' = p x entry
      // scale (content dims), chunk 4 + g holds p (RoPE dims), both FP16; this
      // thread writes 4 bytes (items 8 g + 2 c, + 1) of each
#pragma unroll
      for (int hd = 0; hd < 2; ++hd) {
        const int h = hd ? hB : hA;
        // an item with logit -inf gives p = 0 (a head with no finite logit yet has m_ref = -inf: use 0)
        const float mr = m_ref[hd] == -INFINITY ? 0.f : m_ref[hd];
        float psum = 0.f;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const float p0 = exp2f(__uint_as_float(v[4 * g + 2 * hd]) - mr);
          const float p1 = exp2f(__uint_as_float(v[4 * g + 2 * hd + 1]) - mr);
          psum += p0 + p1;
          uint8_t* row = Ps + b * kTcPBytes + 4 * c;
          *reinterpret_cast<uint32_t*>(row + tc_chunk_off(h, g, kHeads)) = pack_f16x2(p0 * sc[2 * g], p1 * sc[2 * g + 1]);
          *reinterpret_cast<uint32_t*>(row + tc_chunk_off(h, 4 + g, kHeads)) = pack_f16x2(p0, p1);
        }
        l[hd] = l[hd] * corr[hd] + psum;
      }
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      tc::mbar_arrive(&C.p_full[b]);
    }
    // ---- epilogue: wait for the last PV, then O (lanes = dims) -> output
    const bool last = ok && tc::mbar_wait(&C.p_empty[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1, abort, a.status, false);
#pragma unroll
    for (int hd = 0; hd < 2; ++hd) {  // a head's sum over its 4 threads
      l[hd] += __shfl_xor_sync(0xffffffffu, l[hd], 1);
      l[hd] += __shfl_xor_sync(0xffffffffu, l[hd], 2);
    }
    if (c == 0) {
      C.m_ref[hA] = m_ref[0];
      C.l_sum[hA] = l[0];
      C.m_ref[hB] = m_ref[1];
      C.l_sum[hB] = l[1];
    }
    ok = bar_red_and(1, 128, last);
    if (tid == 64) C.tiles_ok = ok ? 1 : 0;
    const int hh0 = tid - 64;  // 0..127 over the softmax warpgroup
    if (ok && a.splits == 1 && hh0 < kHeads) C.fin[hh0] = finalize_row(a, r, hh0, C.m_ref[hh0], C.l_sum[hh0]);
    bar_red_and(1, 128, true);
    tc::tc_fence_after();
    if (ok && a.merge != kMergeCluster) {  // (the cluster merge reads O after the CTA barrier below)
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
              float y = x * C.fin[hh];
              if (a.rope && c == 4) {  // turn the RoPE dims back by t; the pair partner is the next / previous lane
                const float yp = __shfl_xor_sync(0xffffffffu, y, 1);
                const float2 cs = C.rope_t[(d - kKvContent) >> 1];
                y = (lane & 1) == 0 ? y * cs.x + yp * cs.y : y * cs.x - yp * cs.y;
              }
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
    // Thread t handles quarter qq of item j of every tile.  The FP8 content,
    // RoPE and scale of compressed tiles are loaded straight into registers
    // (read-only path), kPre tiles ahead of the conversion, so an X tile is
    // held only from its conversion to its PV.  Loads of a warp instruction:
    // 8 items x 64 contiguous bytes.
    const int t = tid - 6 * 32;   // 0..127
    const int j = t >> 2, qq = t & 3;
    const int P = a.kv.page_entries;
    constexpr int kPre = 2;                    // prefetch distance, tiles
    uint4 rc[kPre + 1][8], rr[kPre + 1][2];    // register ring, slot = tile % (kPre + 1)
    float rs[kPre + 1];
    bool rv[kPre + 1];
    auto load = [&](int n, auto slot_c) -> bool {
      constexpr int k = decltype(slot_c)::value;
      const int s = n % kMetaStages;
      if (!tc::mbar_wait(&C.meta_full[s], (n / kMetaStages) & 1, abort, a.status)) return false;
      const uint8_t* pg = C.page[s][j];
      const int sl = C.slot[s][j];
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&C.meta_empty[s]);
      rv[k] = pg != nullptr;
      if (pg) {
        const uint4* content = reinterpret_cast<const uint4*>(pg + (size_t)sl * kKvContent);
#pragma unroll
        for (int u = 0; u < 8; ++u) rc[k][u] = __ldg(content + 4 * u + qq);
        const uint4* rope = reinterpret_cast<const uint4*>(pg + (size_t)kKvContent * P + (size_t)sl * (2 * kKvRope));
        rr[k][0] = __ldg(rope + qq);
        rr[k][1] = __ldg(rope + 4 + qq);
        rs[k] = qq == 0 ? __ldg(reinterpret_cast<const float*>(pg + (size_t)(kKvContent + 2 * kKvRope) * P) + sl) : 0.f;
      }
      return true;
    };
    // one X tile: wait until its buffer is free, fill it, publish it
    auto x_tile = [&](int n, auto fill) -> bool {
      const int b = n % kXBufs;
      if (!tc::mbar_wait(&C.x_empty[b], ((n / kXBufs) & 1) ^ 1, abort, a.status)) return false;
      uint8_t* xt = Xs + b * kTcTileBytes;
      if (!fill(b, xt)) return false;
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&C.x_full[b]);
      return true;
    };
    // compressed tile n from register slot k into an X tile
    auto convert_tile = [&](int n, auto slot_c) -> bool {
      constexpr int k = decltype(slot_c)::value;
      return x_tile(n, [&](int b, uint8_t* xt) -> bool {
        if (rv[k]) {
          // content: the e4m3 codes as FP16 (exact; the entry scale is applied
          // to the logit and to P); RoPE dims BF16 -> FP16
          if (qq == 0) C.scl[b][j] = rs[k];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int c16 = 4 * u + qq;  // 16 content bytes = dims 16 c16 .. 16 c16 + 15
            *reinterpret_cast<uint4*>(xt + tc_chunk_off(j, 2 * c16, kTI)) = fp8x8_to_f16x8(rc[k][u], false);
            *reinterpret_cast<uint4*>(xt + tc_chunk_off(j, 2 * c16 + 1, kTI)) = fp8x8_to_f16x8(rc[k][u], true);
          }
#pragma unroll
          for (int u = 0; u < 2; ++u)
            *reinterpret_cast<uint4*>(xt + tc_chunk_off(j, 64 + 4 * u + qq, kTI)) = bf16x8_to_f16x8(rr[k][u]);
        } else {
          if (qq == 0) C.scl[b][j] = 0.f;
          const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int u = 0; u < 18; ++u) *reinterpret_cast<uint4*>(xt + tc_chunk_off(j, 4 * u + qq, kTI)) = z;
        }
        return true;
      });
    };
    // compressed tile n, with the load of tile n + kPre
    auto comp_step = [&](int n, auto slot_c) -> bool {
      constexpr int k = decltype(slot_c)::value;
      // the load of tile n + kPre goes into the slot of tile n - 1 (already
      // converted); it is issued first, except for tile 0, whose conversion
      // should not wait for the producer to resolve tile kPre
      if (n > 0 && n + kPre < ncomp && !load(n + kPre, std::integral_constant<int, (k + kPre) % (kPre + 1)>{}))
        return false;
      if (n == 0 && !convert_tile(n, slot_c)) return false;
      if (n == 0) return kPre >= ncomp || load(kPre, std::integral_constant<int, kPre % (kPre + 1)>{});
      return convert_tile(n, slot_c);
    };
    // window tile n (after every compressed tile: the register ring is dead here)
    auto win_step = [&](int n) -> bool {
      return x_tile(n, [&](int b, uint8_t* xt) -> bool {
        // window tile: BF16 rows by TMA straight into the swizzled X tile
        const int wi = n - ncomp;
        if (t == 0) {
          const int w = (i0 + n * kTI - sel_pad) / kTI;
          const int row0 = win_dense ? it.t - it.n_win + 1 + kTI * w : kTI * w;
          tc::mbar_arrive_expect_tx(&C.win_full[b], kTcTileBytes);
          for (int kb = 0; kb < kTcKBlocks; ++kb)
            tma_load_3d(xt + kb * (kTI * 128), &win_map, 64 * kb, row0, it.b, &C.win_full[b]);
        }
        if (!tc::mbar_wait(&C.win_full[b], (wi / kXBufs) & 1, abort, a.status, t == 0 ? false : true)) return false;
        // the window rows arrive as BF16: convert the tile to FP16 in place
        if (a.win_norm || a.rope) {
          // thread t: row j, chunks qq, qq + 4, ..; RMSNorm over the row's
          // 576 dims (4 threads per row), RoPE of its last 64 at its position
          const int w = (i0 + n * kTI - sel_pad) / kTI;
          int off;  // position of the row minus t
          if (win_dense) {
            off = kTI * w + j - (it.n_win - 1);
          } else {  // ring slot s holds the window position p with p = s (mod ring)
            const int sl = kTI * w + j;
            off = -(((it.t - sl) % a.win_ring + a.win_ring) % a.win_ring);
          }
          float ss = 0.f;
#pragma unroll 6
          for (int u = 0; u < 18; ++u)
            ss += bf16x8_sumsq(*reinterpret_cast<const uint4*>(xt + tc_chunk_off(j, 4 * u + qq, kTI)));
          ss += __shfl_xor_sync(0xffffffffu, ss, 1);
          ss += __shfl_xor_sync(0xffffffffu, ss, 2);
          const float inv = a.win_norm ? rms_inv(ss, a.norm_eps) : 1.f;
#pragma unroll 2
          for (int u = 0; u < 18; ++u) {
            const int c8 = 4 * u + qq;
            uint4* pc = reinterpret_cast<uint4*>(xt + tc_chunk_off(j, c8, kTI));
            float x[8];
            bf16x8_unpack(*pc, x);
            if (a.win_norm)
#pragma unroll
              for (int e = 0; e < 8; ++e) x[e] *= inv * a.win_norm[8 * c8 + e];
            if (a.rope && c8 >= kKvContent / 8)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                // R(p) = R(t) R(p - t): the query's angle (reduced in double) times a small one
                const int i = 4 * (c8 - kKvContent / 8) + e;
                const float2 cs = small_angle_cs((float)off * (float)a.freq.f[i]);
                const float2 ct = C.rope_t[i];
                const float2 v = rotate_pair(x[2 * e], x[2 * e + 1],
                                             make_float2(ct.x * cs.x - ct.y * cs.y, ct.y * cs.x + ct.x * cs.y));
                x[2 * e] = v.x;
                x[2 * e + 1] = v.y;
              }
            *pc = make_uint4(pack_f16x2(x[0], x[1]), pack_f16x2(x[2], x[3]), pack_f16x2(x[4], x[5]),
                             pack_f16x2(x[6], x[7]));
          }
        } else {
#pragma unroll 2
          for (int c = t; c < kTcTileBytes / 16; c += 128) {
            uint4* pc = reinterpret_cast<uint4*>(xt + c * 16);
            *pc = bf16x8_to_f16x8(*pc);
          }
        }
        if (t < kTI) C.scl[b][t] = 1.f;
        return true;
      });
    };
    bool ok = true;
    if (0 < ncomp) ok = load(0, std::integral_constant<int, 0>{});
    if (ok && 1 < ncomp) ok = load(1, std::integral_constant<int, 1>{});
    for (int n0 = 0; ok && n0 < ncomp; n0 += kPre + 1) {
      ok = comp_step(n0, std::integral_constant<int, 0>{});
      if (ok && n0 + 1 < ncomp) ok = comp_step(n0 + 1, std::integral_constant<int, 1>{});
      if (ok && n0 + 2 < ncomp) ok = comp_step(n0 + 2, std::integral_constant<int, 2>{});
    }
    for (int n = ncomp; ok && n < ntiles; ++n) ok = win_step(n);
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (a.merge == kMergeCluster) {
    // ------------------------------------------------------------ split merge inside the cluster
    // The CTAs of one query's splits form a thread-block cluster (rank =
    // split).  The [head][dim] output range is cut into S slices, slice q
    // owned by rank q.
    //  (1) each CTA writes its unnormalized O and its (m, l) per head to the
    //      workspace (they stay in L2);
    //  (2) one cluster barrier (release / acquire at cluster scope) makes both
    //      visible; each CTA derives every split's weight 2^(m_q - M) / den
    //      per head (the sink in den) from the S (m, l) pairs.  (Stores of
    //      (m, l) into the peers' shared memory, measured, took longer: about
    //      3 us more per merge than the round trip through L2);
    //  (3) each CTA sums its slice over the splits' partials in split order
    //      0 .. S-1 and writes those output elements.
    // The order is fixed, so the bits depend only on the split boundaries.
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    const int S = (int)cluster.num_blocks();
    const int me = (int)cluster.block_rank();
    float2* part_ml = reinterpret_cast<float2*>(a.part_ml) + (size_t)r * S * kHeads;  // [split][head]
    if (tid < kHeads) part_ml[me * kHeads + tid] = make_float2(C.m_ref[tid], C.l_sum[tid]);
    // the 8 warps 2..9 write O: warp w reads TMEM lanes of quadrant w % 4
    // (its dims), warps 2-5 heads 0-31, warps 6-9 heads 32-63
    float* po = a.part_o + ((size_t)r * S + me) * kHeads * kDim;
    if (warp >= 2) {
      const int quad = warp & 3, half = warp < 6 ? 0 : 1;
      const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
      const bool have = C.tiles_ok != 0;
#pragma unroll 1
      for (int c = 0; c < 5; ++c) {
        const int d = (c < 4 ? 128 * c : kKvContent) + 32 * quad + lane;
        const bool write = c < 4 || quad < 2;  // chunk 4: RoPE dims in lanes 0..63
        uint32_t o[32];
        if (have) {
          tc::tmem_ld32(tmem + lane_base + kTcOCol + c * kHeads + half * 32, o);
          tc::tmem_wait_ld();
        }
        if (!write) continue;
#pragma unroll
        for (int j = 0; j < 32; ++j) po[(half * 32 + j) * kDim + d] = have ? __uint_as_float(o[j]) : 0.f;
      }
    }
    cluster.sync();  // every split's partial and (m, l) visible to the cluster
    if (tid < kHeads) {
      const int h = tid;
      float2 ml[kMaxClusterSplits];
#pragma unroll
      for (int q = 0; q < kMaxClusterSplits; ++q)
        ml[q] = q < S ? __ldcg(part_ml + q * kHeads + h) : make_float2(-INFINITY, 0.f);
      float M = -INFINITY;
#pragma unroll
      for (int q = 0; q < kMaxClusterSplits; ++q)
        if (ml[q].y > 0.f) M = fmaxf(M, ml[q].x);
      float mx = M, s2 = -INFINITY;
      if (a.sink) {
        s2 = a.sink[h] * kLog2e;
        mx = fmaxf(mx, s2);
      }
      float den = 0.f;
#pragma unroll
      for (int q = 0; q < kMaxClusterSplits; ++q)
        if (ml[q].y > 0.f) den += ml[q].y * exp2f(ml[q].x - mx);
      if (a.sink) den += exp2f(s2 - mx);
#pragma unroll
      for (int q = 0; q < kMaxClusterSplits; ++q)
        if (q < S) C.wgt[q][h] = (ml[q].y > 0.f && den > 0.f) ? exp2f(ml[q].x - mx) / den : 0.f;
      if (me == 0 && a.lse) a.lse[(size_t)r * kHeads + h] = den > 0.f ? (mx + log2f(den)) * kLn2 : -INFINITY;
    }
    __syncthreads();
    constexpr int kTotal4 = kHeads * kDim / 4;
    const int per4 = (kTotal4 + S - 1) / S;
    const int f0 = me * per4, f1 = min(kTotal4, f0 + per4);
    const float4* src = reinterpret_cast<const float4*>(a.part_o + (size_t)r * S * kHeads * kDim);
    auto merge_one = [&](int f, const float4 (&v)[kMaxClusterSplits]) {
      const int h = (4 * f) / kDim;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int q = 0; q < kMaxClusterSplits; ++q)
        if (q < S) {
          const float w = C.wgt[q][h];
          acc.x = fmaf(w, v[q].x, acc.x);
          acc.y = fmaf(w, v[q].y, acc.y);
          acc.z = fmaf(w, v[q].z, acc.z);
          acc.w = fmaf(w, v[q].w, acc.w);
        }
      const size_t off = (size_t)r * kHeads * kDim + (size_t)f * 4;  // (head, dim) of element 4 f
      const int d0 = (4 * f) % kDim;
      if (a.rope && d0 >= kKvContent) {  // turn the RoPE dims back by t
        const float2 c0 = C.rope_t[(d0 - kKvContent) >> 1], c1 = C.rope_t[((d0 - kKvContent) >> 1) + 1];
        acc = make_float4(acc.x * c0.x + acc.y * c0.y, acc.y * c0.x - acc.x * c0.y, acc.z * c1.x + acc.w * c1.y,
                          acc.w * c1.x - acc.z * c1.y);
      }
      if (a.out_bf16) {
        uint2 o;
        o.x = (uint32_t)float_to_bf16_bits(acc.x) | ((uint32_t)float_to_bf16_bits(acc.y) << 16);
        o.y = (uint32_t)float_to_bf16_bits(acc.z) | ((uint32_t)float_to_bf16_bits(acc.w) << 16);
        *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + off) = o;
      } else {
        *reinterpret_cast<float4*>(static_cast<float*>(a.out) + off) = acc;
      }
    };
    // two output positions per iteration: every split's partial of both is
    // loaded (from L2) before either sum
    for (int f = f0 + tid; f < f1; f += 2 * kTcThreads2) {
      const int g = f + kTcThreads2;
      float4 v[kMaxClusterSplits], u[kMaxClusterSplits];
#pragma unroll
      for (int q = 0; q < kMaxClusterSplits; ++q) {
        if (q < S) v[q] = __ldcg(src + (size_t)q * kTotal4 + f);
        if (q < S && g < f1) u[q] = __ldcg(src + (size_t)q * kTotal4 + g);
      }
      merge_one(f, v);
      if (g < f1) merge_one(g, u);
    }
    // no barrier before exit: after the cluster barrier no CTA touches a peer's shared memory
  }
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

// ================================================================== split combine

constexpr int kMaxSplits = 64;

// One CTA per (query, head).  Warp 0 derives every split's weight (two
// splits per lane); meanwhile, with rows of D = 4 D4 floats, two threads per
// 16-byte column (sg = 0, 1) load the partials of splits sg, sg + 2, ...
// eight at a time, so that a split count of 30-40 costs a few round trips to
// L2; the two halves are added in a fixed order (even splits, then odd), so
// a launch shape always gives the same bits.
constexpr int kCombineMaxD4 = 512;

__device__ __forceinline__ bool combine_vec(int D) { return (D & 3) == 0 && D / 4 <= kCombineMaxD4; }

__global__ void __launch_bounds__(1024) combine_kernel(AttArgs a) {
  tc::pdl_wait();  // the partials of the attention kernel
  const int r = blockIdx.x, h = blockIdx.y, S = a.splits, D = a.D, H = a.H, tid = threadIdx.x;
  __shared__ float wgt[kMaxSplits];
  __shared__ float inv_s;
  __shared__ float4 half_acc[kCombineMaxD4];
  const bool vec = combine_vec(D);
  const int D4 = vec ? D / 4 : 0;
  const float4* po = reinterpret_cast<const float4*>(a.part_o + ((size_t)r * S * H + h) * D);  // split s at + s H D / 4
  const size_t split_stride = (size_t)H * D / 4;
  const int d4 = vec ? tid % D4 : 0, sg = vec ? tid / D4 : 2;
  const bool act = vec && sg < 2;
  constexpr int kB = 8;
  float4 buf[kB];
#pragma unroll
  for (int u = 0; u < kB; ++u) {
    const int sp = sg + 2 * u;
    buf[u] = (act && sp < S) ? __ldcg(po + sp * split_stride + d4) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (tid < 32) {  // every split's (running max, sum) -> weights
    float m[2], l[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int sp = tid + 32 * i;
      m[i] = -INFINITY;
      l[i] = 0.f;
      if (sp < S) {
        const float2 ml = *reinterpret_cast<const float2*>(a.part_ml + (((size_t)r * S + sp) * H + h) * 2);
        m[i] = ml.x;
        l[i] = ml.y;
      }
    }
    float M = fmaxf(m[0], m[1]);
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int sp = tid + 32 * i;
      const float w = (sp < S && l[i] > 0.f) ? exp2f(m[i] - M) : 0.f;
      if (sp < S) wgt[sp] = w;
      tot = fmaf(w, l[i], tot);
    }
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    if (tid == 0) inv_s = finalize_row(a, r, h, M, tot);
  }
  __syncthreads();
  const float inv = inv_s;
  if (!vec) {  // scalar rows
    const float* pf = a.part_o + ((size_t)r * S * H + h) * D;
    for (int d = tid; d < D; d += blockDim.x) {
      float acc = 0.f;
      for (int sp = 0; sp < S; ++sp) acc = fmaf(wgt[sp], pf[(size_t)sp * H * D + d], acc);
      const size_t off = ((size_t)r * H + h) * D + d;
      if (a.out_bf16) static_cast<uint16_t*>(a.out)[off] = float_to_bf16_bits(acc * inv);
      else static_cast<float*>(a.out)[off] = acc * inv;
    }
    return;
  }
  auto add = [&](float4& acc, float w, float4 x) {
    acc.x = fmaf(w, x.x, acc.x);
    acc.y = fmaf(w, x.y, acc.y);
    acc.z = fmaf(w, x.z, acc.z);
    acc.w = fmaf(w, x.w, acc.w);
  };
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (act) {
    for (int i0 = 0;; i0 += kB) {  // this thread's splits sg + 2 i, in order
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        const int sp = sg + 2 * (i0 + u);
        if (sp < S) add(acc, wgt[sp], buf[u]);
      }
      if (sg + 2 * (i0 + kB) >= S) break;
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        const int sp = sg + 2 * (i0 + kB + u);
        buf[u] = sp < S ? __ldcg(po + sp * split_stride + d4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }
  if (act && sg == 1) half_acc[d4] = acc;
  __syncthreads();
  if (!act || sg != 0) return;
  const float4 o1 = half_acc[d4];
  acc = make_float4(acc.x + o1.x, acc.y + o1.y, acc.z + o1.z, acc.w + o1.w);
  const size_t off = ((size_t)r * H + h) * D + 4 * d4;
  const int d0 = 4 * d4;
  if (a.rope && d0 >= D - kRopeDims) {  // turn the RoPE dims back by the query position
    const int i = (d0 - (D - kRopeDims)) >> 1;
    const int t = a.pos[r];
    const float2 c0 = rope_cs(a.freq.f[i], t), c1 = rope_cs(a.freq.f[i + 1], t);
    acc = make_float4(acc.x * c0.x + acc.y * c0.y, acc.y * c0.x - acc.x * c0.y, acc.z * c1.x + acc.w * c1.y,
                      acc.w * c1.x - acc.z * c1.y);
  }
  if (a.out_bf16) {
    uint2 o;
    o.x = (uint32_t)float_to_bf16_bits(acc.x * inv) | ((uint32_t)float_to_bf16_bits(acc.y * inv) << 16);
    o.y = (uint32_t)float_to_bf16_bits(acc.z * inv) | ((uint32_t)float_to_bf16_bits(acc.w * inv) << 16);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + off) = o;
  } else {
    *reinterpret_cast<float4*>(static_cast<float*>(a.out) + off) =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
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

// How many clusters of `cs` attention CTAs the current device holds at once
// (cudaOccupancyMaxActiveClusters for this kernel's block size and shared
// memory).  A property of the device and the kernel, so it is looked up once
// per device and cluster size and kept.
int max_resident_clusters(int cs) {
  constexpr int kDevs = 64;
  static std::atomic<int> cache[kDevs][kMaxClusterSplits + 1];
  static std::once_flag init;
  std::call_once(init, [] {
    for (auto& row : cache)
      for (auto& v : row) v.store(-1);
  });
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs || cs < 1 || cs > kMaxClusterSplits) return 0;
  int n = cache[dev][cs].load();
  if (n >= 0) return n;
  cudaFuncSetAttribute(attend_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemBytes);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, cs);
  cfg.blockDim = dim3(kTcThreads2);
  cfg.dynamicSmemBytes = kTcSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = cs;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaOccupancyMaxActiveClusters(&n, attend_tc_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  cache[dev][cs].store(n);
  return n;
}

struct Plan {
  int splits, items_per_split, tile;
  bool mma;
  int merge;      // kMergeDirect / kMergeCluster / kMergeGlobal
  int invariant;  // batch-invariant split boundaries
  bool overlap;   // may start before the previous kernel of the stream finishes
  bool window_only;  // no compressed branch: the window alone
};

// Flags of a call; a struct of the size before the flags field existed
// counts as flags = 0.
int attend_flags(const csa_attend_params* p) {
  return p->struct_size >= offsetof(csa_attend_params, flags) + sizeof(p->flags) ? p->flags : 0;
}

// Query / window normalization and RoPE of a call (none for a struct that
// ends before those fields).
struct Prep {
  const float* q_norm;
  const float* win_norm;
  float eps, base;
};
Prep attend_prep(const csa_attend_params* p) {
  if (p->struct_size < offsetof(csa_attend_params, rope_base) + sizeof(float)) return Prep{nullptr, nullptr, 0.f, 0.f};
  return Prep{p->q_norm, p->win_norm, p->norm_eps, p->rope_base};
}

int plan(const csa_attend_params* p, bool sparse, Plan* pl) {
  CSA_CHECK(p != nullptr && p->struct_size >= offsetof(csa_attend_params, flags), CSA_ERR_INVALID_ARG);
  const int flags = attend_flags(p);
  const Prep prep = attend_prep(p);
  CSA_CHECK(prep.eps >= 0.f && prep.base >= 0.f, CSA_ERR_INVALID_ARG);
  CSA_CHECK((!prep.q_norm || aligned(prep.q_norm, 4)) && (!prep.win_norm || aligned(prep.win_norm, 4)), CSA_ERR_ALIGN);
  const bool wants_prep = prep.q_norm || prep.win_norm || prep.base > 0.f;
  CSA_CHECK((flags & ~(CSA_ATTEND_BATCH_INVARIANT | CSA_ATTEND_WINDOW_ONLY | CSA_FLAG_OVERLAP_PREVIOUS)) == 0,
            CSA_ERR_INVALID_ARG);
  pl->overlap = (flags & CSA_FLAG_OVERLAP_PREVIOUS) != 0;
  pl->window_only = (flags & CSA_ATTEND_WINDOW_ONLY) != 0;
  CSA_CHECK(p->num_queries >= 0 && p->batch >= 1 && p->m >= 1 && p->window >= 0 && p->max_pos >= 0,
            CSA_ERR_SHAPE);
  CSA_CHECK(p->heads >= 1 && p->dim >= 1, CSA_ERR_SHAPE);
  CSA_CHECK(p->win_ring >= 1, CSA_ERR_SHAPE);
  // window-only (no compressed branch): no compressed entry is visible
  const int64_t nmax = pl->window_only ? 0 : (int64_t)(p->max_pos + 1) / p->m;
  int64_t Lmax = (sparse ? std::min<int64_t>(p->top_k, nmax) : nmax) + std::min<int64_t>(p->window, p->max_pos + 1);
  // the path: the store's format, or (window-only, no store read) the query's dtype
  const int fmt = pl->window_only ? (p->q_dtype == CSA_F32 ? CSA_FMT_DENSE_F32 : CSA_FMT_KV_POOL_FP8) : p->kv.format;
  if (fmt == CSA_FMT_KV_POOL_FP8)  // compressed items padded to a whole tile, then the window
    Lmax = ((sparse ? std::min<int64_t>(p->top_k, nmax) : nmax) + kTI - 1) / kTI * kTI +
           std::min<int64_t>(p->window, p->max_pos + 1);
  if (fmt == CSA_FMT_DENSE_F32) {
    CSA_CHECK(p->q_dtype == CSA_F32 && p->win_dtype == CSA_F32 && p->out_dtype == CSA_F32, CSA_ERR_UNSUPPORTED);
    CSA_CHECK(!wants_prep, CSA_ERR_UNSUPPORTED);  // normalization / RoPE: tensor-core path only
    CSA_CHECK((pl->window_only || p->kv.dim == p->dim) && p->heads * p->dim <= kF32Threads * kF32MaxPer,
              CSA_ERR_UNSUPPORTED);
    pl->mma = false;
    pl->tile = kF32Tile;
  } else if (fmt == CSA_FMT_KV_POOL_FP8) {
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
  const int64_t tiles = std::max<int64_t>(1, (Lmax + pl->tile - 1) / pl->tile);
  pl->invariant = (flags & CSA_ATTEND_BATCH_INVARIANT) ? 1 : 0;
  int splits;
  int64_t ips;
  if (pl->invariant) {
    // the largest split count any query of the launch can have; each query
    // derives its own count and boundaries from its item count on the device
    splits = (int)std::min<int64_t>(kMaxClusterSplits, (tiles + kInvTilesPerSplit - 1) / kInvTilesPerSplit);
    splits = std::max(1, splits);
    ips = (tiles + splits - 1) / splits * pl->tile;
  } else {
    // split-K: enough CTAs to cover the SMs, each split at least 4 tiles
    const int T = std::max(p->num_queries, 1);
    splits = (int)std::max<int64_t>(1, std::min<int64_t>({(int64_t)sm_count() / T, (tiles + 3) / 4, kMaxSplits}));
    // a few splits more than a cluster holds: fewer splits, merged in the
    // cluster, when every cluster of the launch can be resident at once
    if (pl->mma && splits > kMaxClusterSplits && splits <= kMaxClusterSplits + 2 &&
        p->num_queries <= max_resident_clusters(kMaxClusterSplits))
      splits = kMaxClusterSplits;
    ips = (tiles + splits - 1) / splits * pl->tile;
    splits = (int)((Lmax + ips - 1) / ips);
  }
  pl->splits = std::max(1, splits);
  pl->items_per_split = (int)ips;
  if (pl->splits == 1) {
    pl->merge = kMergeDirect;
  } else if (pl->mma && pl->splits <= kMaxClusterSplits &&
             (pl->invariant || p->num_queries <= max_resident_clusters(pl->splits))) {
    // every cluster of the launch resident at once (a cluster of S CTAs needs
    // S SMs of one GPC); a batch-invariant launch always merges in clusters
    pl->merge = kMergeCluster;
  } else {
    pl->merge = kMergeGlobal;
  }
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
  if (pl->window_only) return CSA_OK;  // the store is not read
  const int64_t nmax = (int64_t)(p->max_pos + 1) / p->m;
  return check_store(p->kv, p->batch, nmax);
}

size_t workspace_bytes(const csa_attend_params* p, const Plan& pl) {
  if (pl.merge == kMergeDirect) return kWsHeader;
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
  a.invariant = pl.invariant;
  a.merge = pl.merge;
  a.window_only = pl.window_only ? 1 : 0;
  {
    const Prep prep = attend_prep(p);
    a.q_norm = prep.q_norm;
    a.win_norm = prep.win_norm;
    a.norm_eps = prep.eps;
    a.rope = prep.base > 0.f;
    a.freq = rope_freq(prep.base);
  }
  a.kv = to_device(p->kv);
  a.batch = p->batch;
  a.kv_cap = pl.window_only ? 0
             : p->kv.format == CSA_FMT_DENSE_F32 ? p->kv.capacity : p->kv.max_pages * p->kv.page_entries;
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
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    CSA_CHECK(encode != nullptr, CSA_ERR_CUDA);
    const cuuint32_t estr[3] = {1, 1, 1};
    // TMA descriptor of the window source: [batch][win_ring][576] BF16, boxes
    // of 64 dims x 32 rows, 128-byte swizzle (the layout of an X tile block)
    CUtensorMap win_map;
    {
      const cuuint64_t dims[3] = {(cuuint64_t)kDim, (cuuint64_t)p->win_ring, (cuuint64_t)p->batch};
      const cuuint64_t strides[2] = {(cuuint64_t)kDim * 2, (cuuint64_t)p->win_ring * kDim * 2};
      const cuuint32_t box[3] = {64, (cuuint32_t)kTI, 1};
      CSA_CHECK(encode(&win_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p->win), dims, strides, box,
                       estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS,
                CSA_ERR_INVALID_ARG);
    }
    // TMA descriptor of the queries: [T * 64 heads][576] BF16, boxes of 64
    // dims x 64 heads, 128-byte swizzle (the layout of the Q operand)
    CUtensorMap q_map;
    {
      const cuuint64_t dims[2] = {(cuuint64_t)kDim, (cuuint64_t)p->num_queries * kHeads};
      const cuuint64_t strides[1] = {(cuuint64_t)kDim * 2};
      const cuuint32_t box[2] = {64, (cuuint32_t)kHeads};
      CSA_CHECK(encode(&q_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p->q), dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS,
                CSA_ERR_INVALID_ARG);
    }
    const int win_dense = p->win_ring >= p->max_pos + 1 ? 1 : 0;
    cudaFuncSetAttribute(attend_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemBytes);
    const int cy = pl.merge == kMergeCluster ? pl.splits : 1;
    st = launch_ex(attend_tc_kernel, grid, dim3(kTcThreads2), kTcSmemBytes, s, pl.overlap, 1, cy, a, win_map, q_map,
                   win_dense);
  } else {
    const size_t smem = ((size_t)p->heads * (p->dim + 1) + kF32Tile * (p->dim + 1) + p->heads * kF32Tile + 3 * p->heads) *
                        sizeof(float);
    CSA_CHECK(smem <= 200 * 1024, CSA_ERR_UNSUPPORTED);
    cudaFuncSetAttribute(attend_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    st = launch_ex(attend_f32_kernel, grid, dim3(kF32Threads), smem, s, pl.overlap, 1, 1, a);
  }
  if (st != CSA_OK || pl.merge != kMergeGlobal) return st;
  // the combine reads nothing before it waits for the attention kernel: it may always start early
  // two threads per 16-byte column of a row (rows of D = 4 D4 floats), else 128 over scalar columns
  const int cthreads = (p->dim % 4 == 0 && p->dim / 4 <= kCombineMaxD4) ? (2 * (p->dim / 4) + 31) / 32 * 32 : 128;
  return launch_ex(combine_kernel, dim3(p->num_queries, p->heads), dim3(cthreads), 0, s, true, 1, 1, a);
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

extern "C" int csa_attend_plan(const csa_attend_params* p, int32_t sparse, int32_t* splits, int32_t* merge) {
  CSA_CHECK(splits != nullptr && merge != nullptr, CSA_ERR_INVALID_ARG);
  Plan pl;
  const int st = check_attend(p, sparse != 0, &pl);
  if (st != CSA_OK) return st;
  *splits = pl.splits;
  *merge = pl.merge;
  return CSA_OK;
}

extern "C" int csa_attend(const csa_attend_params* p, void* ws, size_t ws_bytes, csa_stream_t stream) {
  return run(p, true, ws, ws_bytes, (cudaStream_t)stream);
}

extern "C" int hca_attend(const csa_attend_params* p, void* ws, size_t ws_bytes, csa_stream_t stream) {
  return run(p, false, ws, ws_bytes, (cudaStream_t)stream);
}
