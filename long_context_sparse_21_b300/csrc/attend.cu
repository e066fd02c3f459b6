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
//  * attend_mma_kernel   BF16 queries, FP8-e4m3 + BF16-RoPE pooled entries and
//                        BF16 window tokens, tensor-core mma.sync (m16n8k16,
//                        f32 accumulate), 64 heads x 576 dims, 32-item tiles.
//  * combine_kernel      log-sum-exp merge of split partials.
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "host.hpp"

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

// ================================================================== tensor-core path (bf16 / fp8)

constexpr int kHeads = 64;
constexpr int kDim = kKvDim;            // 576
constexpr int kMmaThreads = 256;        // 8 warps: (head group of 16) x (half)
constexpr int kItems = 32;              // items per tile
constexpr int kQStride = kDim + 8;      // bf16 elements per smem row (1168 B: conflict-free ldmatrix)
constexpr int kPStride = kItems + 8;    // 80 B rows

struct MmaSmem {
  uint16_t q[kHeads * kQStride];
  uint16_t x[kItems * kQStride];
  uint16_t p[kHeads * kPStride];
  float red[4][2][16];
  const uint8_t* src[kItems];  // per item of the tile: page base (entry) or row (window)
  int slot[kItems];            // page slot; -1 window row; -2 masked
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t saddr(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__global__ void __launch_bounds__(kMmaThreads, 1) attend_mma_kernel(AttArgs a) {
  extern __shared__ uint8_t smem_raw[];
  MmaSmem& S = *reinterpret_cast<MmaSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const int r = blockIdx.x, split = blockIdx.y, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int hg = warp >> 1, half = warp & 1;
  const int g = lane >> 2, c4 = lane & 3;
  const Items it = query_items(a, r);
  const int i0 = split * a.items_per_split;
  const int i1 = min(it.L, i0 + a.items_per_split);

  // queries -> smem
  const uint16_t* q = static_cast<const uint16_t*>(a.q) + (size_t)r * kHeads * kDim;
  for (int u = tid; u < kHeads * (kDim / 8); u += kMmaThreads) {
    const int h = u / (kDim / 8), c = u % (kDim / 8);
    *reinterpret_cast<uint4*>(&S.q[h * kQStride + c * 8]) = *reinterpret_cast<const uint4*>(q + h * kDim + c * 8);
  }

  float o[36][4];
#pragma unroll
  for (int n = 0; n < 36; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};  // rows g and g + 8 of this warp's head group
  float l_run[2] = {0.f, 0.f};               // partial sums over this warp's item half

  const int P = a.kv.page_entries;
  for (int base = i0; base < i1; base += kItems) {
    const int nt = min(kItems, i1 - base);
    __syncthreads();  // previous tile fully consumed
    if (tid < kItems) {
      const int i = base + tid;
      int sl = -2;
      const uint8_t* src = nullptr;
      if (tid < nt) {
        if (i < it.n_sel) {
          const int ent = item_entry(a, it, r, i);
          if (ent >= 0) src = page_of(a.kv, it.b, ent, &sl);
        } else {
          sl = -1;
          src = reinterpret_cast<const uint8_t*>(static_cast<const uint16_t*>(a.win) + win_row(a, it, i));
        }
      }
      S.src[tid] = src;
      S.slot[tid] = sl;
    }
    __syncthreads();
    // ---- load + dequantize the item tile (72 chunks of 8 dims per item)
    for (int u = tid; u < kItems * 72; u += kMmaThreads) {
      const int e = u / 72, c = u % 72;
      uint4 v = make_uint4(0, 0, 0, 0);
      const int sl = S.slot[e];
      if (sl != -2) {
        if (sl >= 0) {
          {
            const int slot = sl;
            const uint8_t* page = S.src[e];
            if (c < 64) {
              const float sc = reinterpret_cast<const float*>(page + (size_t)(kKvContent + 2 * kKvRope) * P)[slot];
              const uint2 raw = *reinterpret_cast<const uint2*>(page + (size_t)slot * kKvContent + c * 8);
              const float2 f0 = e4m3x2_to_float2((uint16_t)(raw.x & 0xFFFF));
              const float2 f1 = e4m3x2_to_float2((uint16_t)(raw.x >> 16));
              const float2 f2 = e4m3x2_to_float2((uint16_t)(raw.y & 0xFFFF));
              const float2 f3 = e4m3x2_to_float2((uint16_t)(raw.y >> 16));
              v.x = pack_bf16x2(f0.x * sc, f0.y * sc);
              v.y = pack_bf16x2(f1.x * sc, f1.y * sc);
              v.z = pack_bf16x2(f2.x * sc, f2.y * sc);
              v.w = pack_bf16x2(f3.x * sc, f3.y * sc);
            } else {
              v = *reinterpret_cast<const uint4*>(page + (size_t)kKvContent * P + (size_t)slot * kKvRope * 2 +
                                                  (c - 64) * 16);
            }
          }
        } else {
          v = *reinterpret_cast<const uint4*>(S.src[e] + c * 16);
        }
      }
      *reinterpret_cast<uint4*>(&S.x[e * kQStride + c * 8]) = v;
    }
    __syncthreads();

    // ---- S = Q X^T for heads [16 hg, +16) x items [16 half, +16)
    float sacc[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
    const uint32_t qa = saddr(&S.q[(hg * 16 + (lane & 15)) * kQStride + (lane >> 4) * 8]);
    const uint32_t xb = saddr(&S.x[(half * 16 + (lane & 7) + (lane >> 4) * 8) * kQStride + ((lane >> 3) & 1) * 8]);
#pragma unroll 4
    for (int k0 = 0; k0 < kDim; k0 += 16) {
      uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
      ldsm_x4(qa + k0 * 2, a0, a1, a2, a3);
      ldsm_x4(xb + k0 * 2, b0, b1, b2, b3);
      mma16816(sacc[0], a0, a1, a2, a3, b0, b1);
      mma16816(sacc[1], a0, a1, a2, a3, b2, b3);
    }
    // ---- online softmax (log2 domain); rows g and g+8, cols 2 c4 + {0,1} of each n-tile
    float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int item = half * 16 + n * 8 + c4 * 2 + (j & 1);
        float s = sacc[n][j] * a.scale_log2;
        if (item >= nt) s = -INFINITY;
        sacc[n][j] = s;
        tmax[j >> 1] = fmaxf(tmax[j >> 1], s);
      }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      tmax[rr] = fmaxf(tmax[rr], __shfl_xor_sync(0xffffffffu, tmax[rr], 1));
      tmax[rr] = fmaxf(tmax[rr], __shfl_xor_sync(0xffffffffu, tmax[rr], 2));
    }
    if (c4 == 0) {
      S.red[hg][half][g] = tmax[0];
      S.red[hg][half][g + 8] = tmax[1];
    }
    __syncthreads();
    float corr[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int row = g + rr * 8;
      const float mt = fmaxf(S.red[hg][0][row], S.red[hg][1][row]);
      const float mn = fmaxf(m_run[rr], mt);
      corr[rr] = exp2f(m_run[rr] - mn);
      m_run[rr] = mn;
      l_run[rr] *= corr[rr];
    }
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      float p[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        p[j] = exp2f(sacc[n][j] - m_run[j >> 1]);
        l_run[j >> 1] += p[j];
      }
      const int col = half * 16 + n * 8 + c4 * 2;
      *reinterpret_cast<uint32_t*>(&S.p[(hg * 16 + g) * kPStride + col]) = pack_bf16x2(p[0], p[1]);
      *reinterpret_cast<uint32_t*>(&S.p[(hg * 16 + g + 8) * kPStride + col]) = pack_bf16x2(p[2], p[3]);
    }
#pragma unroll
    for (int n = 0; n < 36; ++n) {
      o[n][0] *= corr[0];
      o[n][1] *= corr[0];
      o[n][2] *= corr[1];
      o[n][3] *= corr[1];
    }
    __syncthreads();
    // ---- O[16 heads x dims [288 half, +288)] += P[16 x 32] X[32 x 288]
    const uint32_t pa = saddr(&S.p[(hg * 16 + (lane & 15)) * kPStride + (lane >> 4) * 8]);
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(pa + ks * 32, a0, a1, a2, a3);
      const uint32_t xv = saddr(&S.x[(ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * kQStride + half * 288 +
                                     (lane >> 4) * 8]);
#pragma unroll
      for (int n2 = 0; n2 < 18; ++n2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(xv + n2 * 32, b0, b1, b2, b3);
        mma16816(o[2 * n2], a0, a1, a2, a3, b0, b1);
        mma16816(o[2 * n2 + 1], a0, a1, a2, a3, b2, b3);
      }
    }
  }

  // ---- full row sums: quad reduce, then add the partner half
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    l_run[rr] += __shfl_xor_sync(0xffffffffu, l_run[rr], 1);
    l_run[rr] += __shfl_xor_sync(0xffffffffu, l_run[rr], 2);
  }
  __syncthreads();
  if (c4 == 0) {
    S.red[hg][half][g] = l_run[0];
    S.red[hg][half][g + 8] = l_run[1];
  }
  __syncthreads();
  float l_tot[2];
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) l_tot[rr] = S.red[hg][0][g + rr * 8] + S.red[hg][1][g + rr * 8];

  if (a.splits == 1) {
    float f[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int h = hg * 16 + g + rr * 8;
      AttArgs na = a;
      if (!(half == 0 && c4 == 0)) na.lse = nullptr;  // one writer per head
      f[rr] = finalize_row(na, r, h, m_run[rr], l_tot[rr]);
    }
#pragma unroll
    for (int n = 0; n < 36; ++n) {
      const int d = half * 288 + n * 8 + c4 * 2;
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int h = hg * 16 + g + rr * 8;
        const float x0 = o[n][rr * 2] * f[rr], x1 = o[n][rr * 2 + 1] * f[rr];
        const size_t off = ((size_t)r * kHeads + h) * kDim + d;
        if (a.out_bf16) *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(a.out) + off) = pack_bf16x2(x0, x1);
        else *reinterpret_cast<float2*>(static_cast<float*>(a.out) + off) = make_float2(x0, x1);
      }
    }
  } else {
    float* po = a.part_o + ((size_t)r * a.splits + split) * kHeads * kDim;
#pragma unroll
    for (int n = 0; n < 36; ++n) {
      const int d = half * 288 + n * 8 + c4 * 2;
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int h = hg * 16 + g + rr * 8;
        *reinterpret_cast<float2*>(po + (size_t)h * kDim + d) = make_float2(o[n][rr * 2], o[n][rr * 2 + 1]);
      }
    }
    if (half == 0 && c4 == 0) {
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int h = hg * 16 + g + rr * 8;
        float* ml = a.part_ml + (((size_t)r * a.splits + split) * kHeads + h) * 2;
        ml[0] = m_run[rr];
        ml[1] = l_tot[rr];
      }
    }
  }
}

// ================================================================== split combine

__global__ void __launch_bounds__(128) combine_kernel(AttArgs a) {
  const int r = blockIdx.x, h = blockIdx.y, S = a.splits, D = a.D, H = a.H;
  __shared__ float wgt[64];
  __shared__ float inv_s;
  const float* ml = a.part_ml + ((size_t)r * S * H + h) * 2;  // split s at + s*H*2
  if (threadIdx.x == 0) {
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) M = fmaxf(M, ml[(size_t)s * H * 2]);
    float l = 0.f;
    for (int s = 0; s < S; ++s) {
      const float ms = ml[(size_t)s * H * 2], ls = ml[(size_t)s * H * 2 + 1];
      const float w = (ls > 0.f) ? exp2f(ms - M) : 0.f;
      wgt[s] = w;
      l += w * ls;
    }
    inv_s = finalize_row(a, r, h, M, l);
  }
  __syncthreads();
  const float inv = inv_s;
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float acc = 0.f;
    for (int s = 0; s < S; ++s) acc = fmaf(wgt[s], a.part_o[(((size_t)r * S + s) * H + h) * D + d], acc);
    const float v = acc * inv;
    const size_t off = ((size_t)r * H + h) * D + d;
    if (a.out_bf16) static_cast<uint16_t*>(a.out)[off] = float_to_bf16_bits(v);
    else static_cast<float*>(a.out)[off] = v;
  }
}

// ------------------------------------------------------------------ host

constexpr int kMaxSplits = 64;

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
  const int64_t Lmax = (sparse ? std::min<int64_t>(p->top_k, nmax) : nmax) + std::min<int64_t>(p->window, p->max_pos + 1);
  if (p->kv.format == CSA_FMT_DENSE_F32) {
    CSA_CHECK(p->q_dtype == CSA_F32 && p->win_dtype == CSA_F32 && p->out_dtype == CSA_F32, CSA_ERR_UNSUPPORTED);
    CSA_CHECK(p->kv.dim == p->dim && p->heads * p->dim <= kF32Threads * kF32MaxPer, CSA_ERR_UNSUPPORTED);
    pl->mma = false;
    pl->tile = kF32Tile;
  } else if (p->kv.format == CSA_FMT_KV_POOL_FP8) {
    CSA_CHECK(p->q_dtype == CSA_BF16 && p->win_dtype == CSA_BF16, CSA_ERR_UNSUPPORTED);
    CSA_CHECK(p->out_dtype == CSA_BF16 || p->out_dtype == CSA_F32, CSA_ERR_UNSUPPORTED);
    CSA_CHECK(p->heads == kHeads && p->dim == kDim, CSA_ERR_UNSUPPORTED);
    pl->mma = true;
    pl->tile = kItems;
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
    const size_t smem = sizeof(MmaSmem) + 128;
    cudaFuncSetAttribute(attend_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    attend_mma_kernel<<<grid, kMmaThreads, smem, s>>>(a);
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
