// Step 1 of the hot path: the softmax-gated KV compressor, and the quantizing
// writer of the paged cache.
//
// DeepSeek-V4 report (cnblogs translation) §2.3.1: every m KV entries are
// folded into one using compression weights and a learnable position bias;
// §2.3.2: HCA does the same with m' = 128 and no overlap; HF blog "DeepSeek-V4"
// (translation), "Hybrid attention": softmax-gated pooling with a learnable
// position bias.  Per channel d of block j:
//     c_j[d] = sum_i softmax_i(g_i[d] + b[i - j m][d]) * k_i[d]
// §2.3.4: content dims stored FP8, RoPE dims BF16; §5.2.1: indexer keys FP4.
// §3.5.1: decode appends to a state cache (window ring + uncompressed tail)
// and writes a compressed entry whenever the tail completes a block.
//
// This is HBM-streaming elementwise work: one CTA per output entry, threads
// over channels (coalesced), the m-position softmax in registers, and the
// quantize-on-write fused in so the float32 entry never goes to HBM.
#include <cooperative_groups.h>

#include "common.cuh"
#include "host.hpp"

namespace csa {
namespace {

constexpr int kThreads = 192;
constexpr int kMaxPer = 4;  // dims per thread -> dim <= 768

__device__ __forceinline__ float load_as_float(const void* p, int dtype, size_t i) {
  if (dtype == CSA_BF16) return bf16_bits_to_float(static_cast<const uint16_t*>(p)[i]);
  return static_cast<const float*>(p)[i];
}

// Maximum over the CTA of a value held by every thread.
__device__ float block_max(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float r = red[0];
  for (int i = 1; i < kThreads / 32; ++i) r = fmaxf(r, red[i]);
  return r;
}

// Sum over the CTA of a value held by every thread.
__device__ float block_sum(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float r = red[0];
  for (int i = 1; i < kThreads / 32; ++i) r += red[i];
  return r;
}

// What the compressor does to a pooled entry before storing it ([report]
// §2.3.3): RMSNorm with gain `norm` (nullptr: none), then RoPE on the last 64
// dims at the raw position j * m (rope != 0).
struct Prep {
  const float* norm;
  float eps;
  int rope;
  RopeFreq freq;
};

// RMSNorm + RoPE of one entry held as vals[i] = value of dim threadIdx.x +
// i * kThreads.  Every thread of the CTA calls it (it synchronizes).
__device__ void prep_entry(float (&vals)[kMaxPer], int dim, long long pos, const Prep& pp, float* red) {
  const int tid = threadIdx.x;
  if (pp.norm) {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxPer; ++i)
      if (tid + i * kThreads < dim) ss = fmaf(vals[i], vals[i], ss);
    ss = block_sum(ss, red);
    const float inv = 1.0f / sqrtf(ss / (float)dim + pp.eps);
#pragma unroll
    for (int i = 0; i < kMaxPer; ++i) {
      const int d = tid + i * kThreads;
      if (d < dim) vals[i] *= inv * pp.norm[d];
    }
  }
  if (pp.rope) {
    // the pair partner of dim d is dim d ^ 1, held by thread tid ^ 1 (kThreads is even)
    const int r0 = dim - kRopeDims;
#pragma unroll
    for (int i = 0; i < kMaxPer; ++i) {
      const int d = tid + i * kThreads;
      const float partner = __shfl_xor_sync(0xffffffffu, vals[i], 1);
      if (d >= r0 && d < dim) {
        const float2 cs = rope_cs(pp.freq.f[(d - r0) >> 1], pos);
        vals[i] = (d & 1) == 0 ? rotate_pair(vals[i], partner, cs).x : rotate_pair(partner, vals[i], cs).y;
      }
    }
  }
}

// Cluster-wide combination of one float per CTA (v[0] of every CTA; after a
// cluster barrier that published them): warp 0 reads them, lane q from rank
// q, and combines them in rank order (sum) or by maximum; the result goes to
// v[1] of this CTA, visible after the caller's next CTA-wide barrier.
__device__ __forceinline__ void cluster_combine(float* v, bool take_max, cooperative_groups::cluster_group& cluster) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x, n = (int)cluster.num_blocks();
    const float mine = lane < n ? *cluster.map_shared_rank(v, lane) : 0.f;
    float r = 0.f;  // the identity of both (the values are sums of squares or magnitudes: >= 0)
    for (int cq = 0; cq < n; ++cq) {  // rank order, the same in every CTA
      const float x = __shfl_sync(0xffffffffu, mine, cq);
      r = take_max ? fmaxf(r, x) : r + x;
    }
    if (lane == 0) v[1] = r;
  }
}

// The same for channels [c0, c1) of an entry held as vals[d - c0] by one CTA
// of a cluster whose CTAs own consecutive slices (c0 even); the sum of
// squares is added up over the cluster through distributed shared memory, in
// rank order.  Every CTA of the cluster calls it.
__device__ void prep_slice(float* vals, int c0, int c1, int dim, long long pos, const Prep& pp,
                           cooperative_groups::cluster_group& cluster, float* ss_s) {
  const int tid = threadIdx.x, nt = blockDim.x;
  if (pp.norm) {
    if (tid < 32) {
      float a = 0.f;
      for (int d = c0 + tid; d < c1; d += 32) a = fmaf(vals[d - c0], vals[d - c0], a);
      for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
      if (tid == 0) *ss_s = a;
    }
    cluster.sync();
    cluster_combine(ss_s, false, cluster);
    cluster.sync();  // remote reads done before any CTA moves on (and ss_s[1] visible)
    const float inv = 1.0f / sqrtf(ss_s[1] / (float)dim + pp.eps);
    for (int d = c0 + tid; d < c1; d += nt) vals[d - c0] *= inv * pp.norm[d];
    __syncthreads();
  }
  if (pp.rope) {
    const int r0 = dim - kRopeDims;
    for (int d = max(c0, r0) + 2 * tid; d + 1 < c1; d += 2 * nt) {
      const float2 v = rotate_pair(vals[d - c0], vals[d + 1 - c0], rope_cs(pp.freq.f[(d - r0) >> 1], pos));
      vals[d - c0] = v.x;
      vals[d + 1 - c0] = v.y;
    }
    __syncthreads();
  }
}

// Writes one entry held as vals[i] = value of dim threadIdx.x + i * kThreads.
// Must be called by every thread of the CTA (it synchronizes).  A page id
// outside the pool drops the write and records CSA_ERR_INVALID_ARG in
// *status (when given).
__device__ void store_entry(const Store& s, int b, int e, const float (&vals)[kMaxPer], float* red, int* status) {
  const int tid = threadIdx.x;
  // an entry beyond the store (a sequence length past its capacity) is not written
  const bool dense = s.format == CSA_FMT_DENSE_F32 || s.format == CSA_FMT_DENSE_BF16;
  if (e < 0 || (dense ? e >= s.capacity : e / s.page_entries >= s.max_pages)) return;  // uniform over the CTA
  switch (s.format) {
    case CSA_FMT_DENSE_F32: {
      float* out = reinterpret_cast<float*>(s.base) + ((size_t)b * s.capacity + e) * s.dim;
#pragma unroll
      for (int i = 0; i < kMaxPer; ++i) {
        const int d = tid + i * kThreads;
        if (d < s.dim) out[d] = vals[i];
      }
      break;
    }
    case CSA_FMT_DENSE_BF16: {
      uint16_t* out = reinterpret_cast<uint16_t*>(s.base) + ((size_t)b * s.capacity + e) * s.dim;
#pragma unroll
      for (int i = 0; i < kMaxPer; ++i) {
        const int d = tid + i * kThreads;
        if (d < s.dim) out[d] = float_to_bf16_bits(vals[i]);
      }
      break;
    }
    case CSA_FMT_KV_POOL_FP8: {
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < kMaxPer; ++i) {
        const int d = tid + i * kThreads;
        if (d < kKvContent) amax = fmaxf(amax, fabsf(vals[i]));
      }
      amax = block_max(amax, red);
      float scale = __fdiv_rn(amax, 448.0f);
      if (scale == 0.f) scale = 1.f;
      int slot;
      uint8_t* page = page_of(s, b, e, &slot);
      if (page == nullptr) {  // uniform over the CTA
        if (tid == 0) set_status(status, CSA_ERR_INVALID_ARG);
        break;
      }
      const int P = s.page_entries;
      uint8_t* content = page + (size_t)slot * kKvContent;
      uint16_t* rope = reinterpret_cast<uint16_t*>(page + (size_t)kKvContent * P) + (size_t)slot * kKvRope;
#pragma unroll
      for (int i = 0; i < kMaxPer; ++i) {
        const int d = tid + i * kThreads;
        if (d < kKvContent) content[d] = float_to_e4m3(__fdiv_rn(vals[i], scale));
        else if (d < kKvDim) rope[d - kKvContent] = float_to_bf16_bits(vals[i]);
      }
      if (tid == 0) reinterpret_cast<float*>(page + (size_t)(kKvContent + 2 * kKvRope) * P)[slot] = scale;
      break;
    }
    case CSA_FMT_INDEX_POOL_BF16: {
      int slot;
      uint8_t* page = page_of(s, b, e, &slot);
      if (page == nullptr) {
        if (tid == 0) set_status(status, CSA_ERR_INVALID_ARG);
        break;
      }
#pragma unroll
      for (int i = 0; i < kMaxPer; ++i) {
        const int d = tid + i * kThreads;
        if (d < kIdxDim) *reinterpret_cast<uint16_t*>(page + idx_bf16_offset(slot, d)) = float_to_bf16_bits(vals[i]);
      }
      break;
    }
    case CSA_FMT_INDEX_POOL_E2M1: {
      int slot;
      uint8_t* page = page_of(s, b, e, &slot);
      if (page == nullptr) {
        if (tid == 0) set_status(status, CSA_ERR_INVALID_ARG);
        break;
      }
      const int P = s.page_entries;
      uint8_t* codes = page + (size_t)slot * (kIdxDim / 2);
      uint8_t* scales = page + (size_t)(kIdxDim / 2) * P + (size_t)slot * (kIdxDim / kFp4Block);
#pragma unroll
      for (int i = 0; i < kMaxPer; ++i) {
        const int d = tid + i * kThreads;  // 16 consecutive lanes hold one 16-element block
        const bool live = d < kIdxDim;
        float a = live ? fabsf(vals[i]) : 0.f;
        for (int o = 1; o < kFp4Block; o <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        const uint8_t scode = float_to_e4m3(__fdiv_rn(a, 6.0f));
        const float sdec = e4m3_to_float(scode);
        const float qv = (sdec == 0.f) ? 0.f : __fdiv_rn(vals[i], sdec);
        const float partner = __shfl_xor_sync(0xffffffffu, qv, 1);
        if (live && (d & 1) == 0) codes[d >> 1] = (sdec == 0.f) ? (uint8_t)0 : float2_to_e2m1x2(qv, partner);
        if (live && (d % kFp4Block) == 0) scales[d / kFp4Block] = scode;
      }
      break;
    }
    default:
      break;
  }
}

// Writes channels [c0, c1) of entry e of sequence b from vals[d - c0], one
// slice per CTA of a cluster (all CTAs of the cluster call it; the FP8 entry
// scale needs the maximum over every content channel, exchanged through
// distributed shared memory).  Formats and rounding as store_entry.
__device__ void store_slice(const Store& s, int b, int e, const float* vals, int c0, int c1,
                            cooperative_groups::cluster_group& cluster, float* amax_s, int* status) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const bool dense = s.format == CSA_FMT_DENSE_F32 || s.format == CSA_FMT_DENSE_BF16;
  const bool skip = e < 0 || (dense ? e >= s.capacity : e / s.page_entries >= s.max_pages);
  if (s.format == CSA_FMT_KV_POOL_FP8) {
    // local max of |content| over this slice, then the cluster's maximum
    if (tid < 32) {
      float a = 0.f;
      for (int d = c0 + tid; d < min(c1, kKvContent); d += 32) a = fmaxf(a, fabsf(vals[d - c0]));
      for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
      if (tid == 0) *amax_s = a;
    }
    cluster.sync();
    cluster_combine(amax_s, true, cluster);
    cluster.sync();  // remote reads done before any CTA of the cluster moves on (and amax_s[1] visible)
    const float amax = amax_s[1];
    if (skip) return;
    float scale = __fdiv_rn(amax, 448.0f);
    if (scale == 0.f) scale = 1.f;
    int slot;
    uint8_t* page = page_of(s, b, e, &slot);
    if (page == nullptr) {
      if (tid == 0) set_status(status, CSA_ERR_INVALID_ARG);
      return;
    }
    const int P = s.page_entries;
    uint8_t* content = page + (size_t)slot * kKvContent;
    uint16_t* rope = reinterpret_cast<uint16_t*>(page + (size_t)kKvContent * P) + (size_t)slot * kKvRope;
    for (int d = c0 + tid; d < c1; d += nt) {
      if (d < kKvContent) content[d] = float_to_e4m3(__fdiv_rn(vals[d - c0], scale));
      else if (d < kKvDim) rope[d - kKvContent] = float_to_bf16_bits(vals[d - c0]);
    }
    if (c0 == 0 && tid == 0) reinterpret_cast<float*>(page + (size_t)(kKvContent + 2 * kKvRope) * P)[slot] = scale;
    return;
  }
  if (skip) return;
  switch (s.format) {
    case CSA_FMT_DENSE_F32: {
      float* out = reinterpret_cast<float*>(s.base) + ((size_t)b * s.capacity + e) * s.dim;
      for (int d = c0 + tid; d < c1; d += nt) out[d] = vals[d - c0];
      break;
    }
    case CSA_FMT_DENSE_BF16: {
      uint16_t* out = reinterpret_cast<uint16_t*>(s.base) + ((size_t)b * s.capacity + e) * s.dim;
      for (int d = c0 + tid; d < c1; d += nt) out[d] = float_to_bf16_bits(vals[d - c0]);
      break;
    }
    case CSA_FMT_INDEX_POOL_BF16: {
      int slot;
      uint8_t* page = page_of(s, b, e, &slot);
      if (page == nullptr) {
        if (tid == 0) set_status(status, CSA_ERR_INVALID_ARG);
        break;
      }
      for (int d = c0 + tid; d < c1; d += nt)
        *reinterpret_cast<uint16_t*>(page + idx_bf16_offset(slot, d)) = float_to_bf16_bits(vals[d - c0]);
      break;
    }
    case CSA_FMT_INDEX_POOL_E2M1: {
      // one thread per element pair; the slice holds whole 16-element blocks
      int slot;
      uint8_t* page = page_of(s, b, e, &slot);
      if (page == nullptr) {
        if (tid == 0) set_status(status, CSA_ERR_INVALID_ARG);
        break;
      }
      const int P = s.page_entries;
      uint8_t* codes = page + (size_t)slot * (kIdxDim / 2);
      uint8_t* scales = page + (size_t)(kIdxDim / 2) * P + (size_t)slot * (kIdxDim / kFp4Block);
      for (int d = c0 + 2 * tid; d < c1; d += 2 * nt) {
        const int blk0 = d - (d - c0) % kFp4Block;
        float a = 0.f;
        for (int i = 0; i < kFp4Block; ++i) a = fmaxf(a, fabsf(vals[blk0 - c0 + i]));
        const uint8_t scode = float_to_e4m3(__fdiv_rn(a, 6.0f));
        const float sdec = e4m3_to_float(scode);
        const float x0 = sdec == 0.f ? 0.f : __fdiv_rn(vals[d - c0], sdec);
        const float x1 = sdec == 0.f ? 0.f : __fdiv_rn(vals[d + 1 - c0], sdec);
        codes[d >> 1] = sdec == 0.f ? (uint8_t)0 : float2_to_e2m1x2(x0, x1);
        if (d % kFp4Block == 0) scales[d / kFp4Block] = scode;
      }
      break;
    }
    default:
      break;
  }
}

// Softmax-gated pooling of one channel over the m positions of a block.
template <typename KF, typename GF>
__device__ __forceinline__ float pool_channel(int m, const float* bias, int d, int dim, KF kf, GF gf) {
  float mx = -INFINITY;
  for (int i = 0; i < m; ++i) mx = fmaxf(mx, gf(i) + bias[(size_t)i * dim + d]);
  float se = 0.f, acc = 0.f;
  for (int i = 0; i < m; ++i) {
    const float e = expf(gf(i) + bias[(size_t)i * dim + d] - mx);
    se += e;
    acc = fmaf(e, kf(i), acc);
  }
  return acc / se;
}

// The b stream of overlapping compression: entry j also pools it over the
// previous block j - 1, under one softmax with the a stream's m logits.
struct BStream {
  const void* k;         // dense: [B][n][dim], the a stream's k dtype
  const void* g;         // dense: [B][n][dim], the a stream's g dtype
  const float* bias;     // [m][dim]
  const uint16_t* k_new; // append: bf16 [B][dim]
  const float* g_new;    // append: f32 [B][dim]
  uint16_t* keys;        // append: bf16 [B][2m][dim], slot p % 2m
  float* gates;          // append: f32 [B][2m][dim], slot p % 2m
};

// Softmax-gated pooling of one channel over block j of the a stream and block
// j - 1 of the b stream (ka/ga: position i of block j; kb/gb: position i of
// block j - 1).
template <typename KA, typename GA, typename KB, typename GB>
__device__ __forceinline__ float pool_channel_ab(int m, const float* bias, const float* bias_b, int d, int dim,
                                                 bool prev, KA ka, GA ga, KB kb, GB gb) {
  float mx = -INFINITY;
  for (int i = 0; i < m; ++i) mx = fmaxf(mx, ga(i) + bias[(size_t)i * dim + d]);
  if (prev)
    for (int i = 0; i < m; ++i) mx = fmaxf(mx, gb(i) + bias_b[(size_t)i * dim + d]);
  float se = 0.f, acc = 0.f;
  for (int i = 0; i < m; ++i) {
    const float e = expf(ga(i) + bias[(size_t)i * dim + d] - mx);
    se += e;
    acc = fmaf(e, ka(i), acc);
  }
  if (prev)
    for (int i = 0; i < m; ++i) {
      const float e = expf(gb(i) + bias_b[(size_t)i * dim + d] - mx);
      se += e;
      acc = fmaf(e, kb(i), acc);
    }
  return acc / se;
}

template <bool AB>
__global__ void __launch_bounds__(kThreads) compress_dense_kernel(
    const void* __restrict__ k, int k_dtype, const void* __restrict__ g, int g_dtype,
    const float* __restrict__ bias, int n, int m, int dim, Store dst, int* status, Prep prep, BStream bs) {
  __shared__ float red[kThreads / 32];
  const int j = blockIdx.x, b = blockIdx.y;
  float vals[kMaxPer];
#pragma unroll
  for (int i = 0; i < kMaxPer; ++i) {
    const int d = threadIdx.x + i * kThreads;
    vals[i] = 0.f;
    if (d < dim) {
      const size_t row0 = (size_t)b * n + (size_t)j * m;
      auto ka = [&](int t) { return load_as_float(k, k_dtype, (row0 + t) * dim + d); };
      auto ga = [&](int t) { return load_as_float(g, g_dtype, (row0 + t) * dim + d); };
      if constexpr (AB) {
        // block j - 1 of the b stream (j > 0 only: row0 - m is then in range)
        vals[i] = pool_channel_ab(
            m, bias, bs.bias, d, dim, j > 0, ka, ga,
            [&](int t) { return load_as_float(bs.k, k_dtype, (row0 - m + t) * dim + d); },
            [&](int t) { return load_as_float(bs.g, g_dtype, (row0 - m + t) * dim + d); });
      } else {
        vals[i] = pool_channel(m, bias, d, dim, ka, ga);
      }
    }
  }
  if (prep.norm || prep.rope) prep_entry(vals, dim, (long long)j * m, prep, red);
  store_entry(dst, b, j, vals, red, status);
}

// Decode append.  One thread-block cluster of kCs CTAs per sequence; CTA q
// owns channels [q cpc, (q + 1) cpc) (cpc a multiple of 16, so an FP4 block
// never straddles two CTAs).  Every CTA appends its slice of the new token to
// the state cache; when the token completes a block, it pools its slice over
// the block's m positions (threads = quad of channels x position group,
// vector loads for up to kPosBatchV positions issued together, an online
// softmax per channel, then a merge of the groups), the cluster agrees on the
// FP8 entry scale through distributed shared memory, and each CTA writes its
// own slice of the entry.  dim must be a multiple of 8.
constexpr int kCs = 8;           // CTAs per sequence (one portable cluster)
constexpr int kAppThreads = 512;
constexpr int kMaxCpc = 80;      // channels per CTA: ceil(dim / 8) rounded up to 16, dim <= 640
constexpr int kPosBatchV = 6;  // positions per thread and batch (25 position groups x 6 >= 128)

__device__ void append_body(const int32_t* __restrict__ seq_len, const uint16_t* __restrict__ k_new,
                            const float* __restrict__ g_new, uint16_t* __restrict__ ring, int ring_size,
                            float* __restrict__ tail_gate, const float* __restrict__ bias, int m, int dim, int cpc,
                            const Store& dst, int* status, const Prep& prep);

// When launched with programmatic serialization (CSA_FLAG_OVERLAP_PREVIOUS)
// the append runs alongside the kernel before it, which touches none of its
// buffers, and waits for that kernel only before it exits, so that its own
// completion still implies its predecessor's.
__global__ void __launch_bounds__(kAppThreads) compress_append_kernel(
    const int32_t* __restrict__ seq_len, const uint16_t* __restrict__ k_new,
    const float* __restrict__ g_new, uint16_t* __restrict__ ring, int ring_size,
    float* __restrict__ tail_gate, const float* __restrict__ bias, int m, int dim, int cpc, Store dst,
    int* status, Prep prep) {
  // a kernel launched after this one with programmatic serialization (the
  // indexer, or the other stream's append) may start now; it waits for this
  // kernel's writes before reading them
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  append_body(seq_len, k_new, g_new, ring, ring_size, tail_gate, bias, m, dim, cpc, dst, status, prep);
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ void append_body(const int32_t* __restrict__ seq_len, const uint16_t* __restrict__ k_new,
                            const float* __restrict__ g_new, uint16_t* __restrict__ ring, int ring_size,
                            float* __restrict__ tail_gate, const float* __restrict__ bias, int m, int dim, int cpc,
                            const Store& dst, int* status, const Prep& prep) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ float part[3][4 * kAppThreads];  // [position group][channel of the slice]
  __shared__ float pooled[kMaxCpc];
  __shared__ float amax_s[2], ss_s[2];  // [0]: this CTA's part, [1]: the cluster's
  const int b = blockIdx.x / kCs, q = (int)cluster.block_rank();
  const int tid = threadIdx.x;
  const int cl = tid % cpc, grp = tid / cpc, groups = kAppThreads / cpc;
  const int c = q * cpc + cl;  // channel of this thread
  const bool live = grp < groups && c < dim;
  const int L = seq_len[b];
  if (L < 0) return;  // uniform over the cluster
  if (grp == 0 && live) {
    ring[((size_t)b * ring_size + L % ring_size) * dim + c] = k_new[(size_t)b * dim + c];
    tail_gate[((size_t)b * m + L % m) * dim + c] = g_new[(size_t)b * dim + c];
  }
  if ((L + 1) % m != 0) return;  // uniform over the cluster
  const int p0 = L + 1 - m;  // a multiple of m: position p0 + i sits in tail slot i
  const int r0 = p0 % ring_size;  // ring slot of p0 (slot of p0 + i: r0 + i, wrapped once)
  // Pooling: thread t owns the quad of adjacent channels qd = t mod nq
  // (loaded 8 bytes of BF16 / 16 bytes of float32 at a time) and the
  // positions i = pg, pg + pgroups, ..., pg = t / nq, with an online softmax
  // per channel.  (One channel per thread issued four times the load
  // instructions, and the SM's loads in flight bounded this step.)
  const int nq = cpc / 4, qd = tid % nq, pg = tid / nq, pgroups = kAppThreads / nq;
  const int c4 = q * cpc + 4 * qd;  // first channel of the quad (dim is a multiple of 8)
  float mx[4], se[4], acc[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    mx[e] = -INFINITY;
    se[e] = acc[e] = 0.f;
  }
  if (pg < pgroups && c4 < dim) {
    const uint2 knq = *reinterpret_cast<const uint2*>(k_new + (size_t)b * dim + c4);
    const float4 gnq = *reinterpret_cast<const float4*>(g_new + (size_t)b * dim + c4);
    const float knv[4] = {bf16_bits_to_float((uint16_t)(knq.x & 0xFFFFu)), bf16_bits_to_float((uint16_t)(knq.x >> 16)),
                          bf16_bits_to_float((uint16_t)(knq.y & 0xFFFFu)), bf16_bits_to_float((uint16_t)(knq.y >> 16))};
    const float gnv[4] = {gnq.x, gnq.y, gnq.z, gnq.w};
    const uint16_t* ring_b = ring + (size_t)b * ring_size * dim + c4;
    const float* tail_b = tail_gate + (size_t)b * m * dim + c4;
    for (int base = pg; base < m; base += pgroups * kPosBatchV) {
      // every load of the batch is issued before any is used: positions past
      // the block read the last position's (valid) address and are masked
      // afterwards, so no load sits behind a branch
      uint2 rk[kPosBatchV];
      float4 rg[kPosBatchV], rb[kPosBatchV];
#pragma unroll
      for (int u = 0; u < kPosBatchV; ++u) {
        const int ic = min(base + u * pgroups, m - 1);
        int slot = r0 + ic;
        if (slot >= ring_size) slot -= ring_size;
        rk[u] = *reinterpret_cast<const uint2*>(ring_b + (size_t)slot * dim);
        rg[u] = *reinterpret_cast<const float4*>(tail_b + (size_t)ic * dim);
        rb[u] = *reinterpret_cast<const float4*>(bias + (size_t)ic * dim + c4);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        // logits in the log2 domain (exp(x) = 2^(x log2 e)); the block's last
        // position is the new token (its ring / tail slots are being written
        // by this kernel: the registers are used instead)
        float lg[kPosBatchV];
#pragma unroll
        for (int u = 0; u < kPosBatchV; ++u) {
          const int i = base + u * pgroups;
          const float g = e == 0 ? rg[u].x : e == 1 ? rg[u].y : e == 2 ? rg[u].z : rg[u].w;
          const float bb = e == 0 ? rb[u].x : e == 1 ? rb[u].y : e == 2 ? rb[u].z : rb[u].w;
          lg[u] = i < m ? ((i == m - 1 ? gnv[e] : g) + bb) * 1.44269504088896341f : -INFINITY;
        }
        float bm = lg[0];
#pragma unroll
        for (int u = 1; u < kPosBatchV; ++u) bm = fmaxf(bm, lg[u]);
        if (bm > mx[e]) {  // bm is finite: position `base` is in range
          const float r = exp2f(mx[e] - bm);  // 0 on the first batch
          se[e] *= r;
          acc[e] *= r;
          mx[e] = bm;
        }
#pragma unroll
        for (int u = 0; u < kPosBatchV; ++u) {
          const float w = exp2f(lg[u] - mx[e]);  // 0 for positions past the block
          const uint32_t pair = (e < 2) ? rk[u].x : rk[u].y;
          const float kv = bf16_bits_to_float((uint16_t)((e & 1) ? pair >> 16 : pair & 0xFFFFu));
          se[e] += w;
          acc[e] = fmaf(w, base + u * pgroups == m - 1 ? knv[e] : kv, acc[e]);
        }
      }
    }
  }
  if (pg < pgroups) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int ch = pg * cpc + 4 * qd + e;
      part[0][ch] = mx[e];
      part[1][ch] = se[e];
      part[2][ch] = acc[e];
    }
  }
  __syncthreads();
  if (tid < 4 * cpc) {
    // merge the position groups: four adjacent lanes per channel of the
    // slice, each over groups sub, sub + 4, ..., then across the four lanes
    const int ch = tid >> 2, sub = tid & 3;
    float M = -INFINITY;
    for (int g = sub; g < pgroups; g += 4) M = fmaxf(M, part[0][g * cpc + ch]);
    M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 1));
    M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 2));
    float S = 0.f, A = 0.f;
    for (int g = sub; g < pgroups; g += 4) {
      const float sv = part[1][g * cpc + ch];
      if (sv > 0.f) {
        const float r = exp2f(part[0][g * cpc + ch] - M);  // maxima are in the log2 domain
        S = fmaf(sv, r, S);
        A = fmaf(part[2][g * cpc + ch], r, A);
      }
    }
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      S += __shfl_xor_sync(0xffffffffu, S, o);
      A += __shfl_xor_sync(0xffffffffu, A, o);
    }
    if (sub == 0) pooled[ch] = q * cpc + ch < dim ? A / S : 0.f;
  }
  __syncthreads();
  const int e = (L + 1) / m - 1;
  if (prep.norm || prep.rope)
    prep_slice(pooled, q * cpc, min(dim, (q + 1) * cpc), dim, (long long)e * m, prep, cluster, ss_s);
  store_slice(dst, b, e, pooled, q * cpc, min(dim, (q + 1) * cpc), cluster, amax_s, status);
}

// Decode append for small m (m <= kSmallM): one CTA per sequence, thread i
// owning channels i, i + kThreads, ...  It appends the new token's channels,
// and when the token completes a block it pools each channel over the
// block's m positions (every load issued before use) and stores the entry
// (the FP8 scale by a CTA reduction).  No cluster: a batch of sequences is one
// wave of small CTAs.
// With AB (overlapping compression) it also appends the b stream's key and
// gate to slot L % 2m of their two-block tails and pools the previous block
// of that stream into the same softmax.  MAXM (4, 8 or 16) bounds m: the
// number of loads issued per pooled array.
constexpr int kSmallM = 16;

template <bool AB, int MAXM>
__global__ void __launch_bounds__(kThreads) compress_append_small_kernel(
    const int32_t* __restrict__ seq_len, const uint16_t* __restrict__ k_new, const float* __restrict__ g_new,
    uint16_t* __restrict__ ring, int ring_size, float* __restrict__ tail_gate, const float* __restrict__ bias, int m,
    int dim, Store dst, int* status, Prep prep, BStream bs) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ float red[kThreads / 32];
  const int b = blockIdx.x, tid = threadIdx.x;
  const int L = seq_len[b];
  const bool complete = L >= 0 && (L + 1) % m == 0;  // uniform over the CTA
  float vals[kMaxPer];
  if (L >= 0) {
    const int p0 = L + 1 - m;  // a multiple of m when the block completes
    const uint16_t* ring_b = ring + (size_t)b * ring_size * dim;
    const float* tail_b = tail_gate + (size_t)b * m * dim;
#pragma unroll
    for (int i = 0; i < kMaxPer; ++i) {
      const int c = tid + i * kThreads;
      vals[i] = 0.f;
      if (c >= dim) continue;
      const uint16_t kb = k_new[(size_t)b * dim + c];
      const float gn = g_new[(size_t)b * dim + c];
      if (complete) {
        // positions p0 .. L - 1 from the ring and the tail gates, L from the registers
        uint16_t rk[MAXM];
        float rg[MAXM], rb[MAXM];
#pragma unroll
        for (int u = 0; u < MAXM; ++u) {
          const int ic = min(u, m - 1);
          rk[u] = ring_b[(size_t)((p0 + ic) % ring_size) * dim + c];
          rg[u] = tail_b[(size_t)ic * dim + c];
          rb[u] = bias[(size_t)ic * dim + c];
        }
        // the b stream's previous block (block e - 1 sits in tail half (e - 1) & 1)
        const int ent = (L + 1) / m - 1;
        uint16_t rkb[AB ? MAXM : 1];
        float rgb[AB ? MAXM : 1];
        if constexpr (AB) {
          const size_t h0 = (size_t)b * 2 * m + (size_t)((ent - 1) & 1) * m;
#pragma unroll
          for (int u = 0; u < MAXM; ++u) {
            const int ic = min(u, m - 1);
            rkb[u] = bs.keys[(h0 + ic) * dim + c];
            rgb[u] = bs.gates[(h0 + ic) * dim + c] + bs.bias[(size_t)ic * dim + c];
          }
        }
        float mx = -INFINITY;
#pragma unroll
        for (int u = 0; u < MAXM; ++u) {
          rg[u] = u < m ? ((u == m - 1 ? gn : rg[u]) + rb[u]) * 1.44269504088896341f : -INFINITY;
          mx = fmaxf(mx, rg[u]);
        }
        if constexpr (AB) {
#pragma unroll
          for (int u = 0; u < MAXM; ++u) {
            rgb[u] = u < m && ent > 0 ? rgb[u] * 1.44269504088896341f : -INFINITY;
            mx = fmaxf(mx, rgb[u]);
          }
        }
        float se = 0.f, acc = 0.f;
#pragma unroll
        for (int u = 0; u < MAXM; ++u) {
          const float e = exp2f(rg[u] - mx);  // 0 past the block
          se += e;
          acc = fmaf(e, u == m - 1 ? bf16_bits_to_float(kb) : bf16_bits_to_float(rk[u]), acc);
        }
        if constexpr (AB) {
#pragma unroll
          for (int u = 0; u < MAXM; ++u) {
            // 0 past the block, and for entry 0 (whose tail half was never
            // written: its keys are replaced, so that no stale NaN leaks in)
            const float e = exp2f(rgb[u] - mx);
            se += e;
            acc = fmaf(e, ent > 0 ? bf16_bits_to_float(rkb[u]) : 0.f, acc);
          }
        }
        vals[i] = acc / se;
      }
      ring[((size_t)b * ring_size + L % ring_size) * dim + c] = kb;
      tail_gate[((size_t)b * m + L % m) * dim + c] = gn;
      if constexpr (AB) {
        // the current block's half of the b tails (never the half read above)
        const size_t slot = (size_t)b * 2 * m + L % (2 * m);
        bs.keys[slot * dim + c] = bs.k_new[(size_t)b * dim + c];
        bs.gates[slot * dim + c] = bs.g_new[(size_t)b * dim + c];
      }
    }
  }
  if (complete) {
    const int e = (L + 1) / m - 1;
    if (prep.norm || prep.rope) prep_entry(vals, dim, (long long)e * m, prep, red);
    store_entry(dst, b, e, vals, red, status);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Window-only append (layers with no compressed branch: pure sliding-window
// attention, [report] §4.2.1): the new token goes to ring slot L % ring_size.
__global__ void __launch_bounds__(kThreads) window_append_kernel(const int32_t* __restrict__ seq_len,
                                                                 const uint16_t* __restrict__ k_new,
                                                                 uint16_t* __restrict__ ring, int ring_size, int dim) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int b = blockIdx.x;
  const int L = seq_len[b];
  if (L >= 0)
    for (int c = threadIdx.x; c < dim; c += kThreads)
      ring[((size_t)b * ring_size + L % ring_size) * dim + c] = k_new[(size_t)b * dim + c];
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__global__ void __launch_bounds__(kThreads) cache_write_kernel(const float* __restrict__ src, int n,
                                                               int first, Store dst, int* status) {
  __shared__ float red[kThreads / 32];
  const int i_row = blockIdx.x, b = blockIdx.y;
  float vals[kMaxPer];
#pragma unroll
  for (int i = 0; i < kMaxPer; ++i) {
    const int d = threadIdx.x + i * kThreads;
    vals[i] = d < dst.dim ? src[((size_t)b * n + i_row) * dst.dim + d] : 0.f;
  }
  store_entry(dst, b, first + i_row, vals, red, status);
}

}  // namespace
}  // namespace csa

using namespace csa;

extern "C" size_t csa_page_bytes(int32_t format, int32_t page_entries) {
  if (page_entries <= 0 || page_entries % kTile != 0) return 0;
  return page_bytes(format, page_entries);
}

extern "C" size_t csa_compress_workspace_size(const csa_compress_params* p) {
  (void)p;
  return 0;  // no mode needs scratch: the decode append pools within one cluster per sequence
}

extern "C" int csa_cache_write(const csa_cache_write_params* p, csa_stream_t stream) {
  CSA_CHECK(p != nullptr && p->struct_size >= sizeof(csa_cache_write_params), CSA_ERR_INVALID_ARG);
  CSA_CHECK(p->batch >= 0 && p->n >= 0 && p->first >= 0, CSA_ERR_SHAPE);
  if (p->batch == 0 || p->n == 0) return CSA_OK;
  CSA_CHECK(p->src != nullptr, CSA_ERR_INVALID_ARG);
  CSA_CHECK(aligned(p->src, 16), CSA_ERR_ALIGN);
  CSA_CHECK(p->dst.dim > 0 && p->dst.dim <= kThreads * kMaxPer, CSA_ERR_SHAPE);
  int st = check_store(p->dst, p->batch, (int64_t)p->first + p->n);
  if (st != CSA_OK) return st;
  CSA_CHECK(p->batch <= 65535, CSA_ERR_SHAPE);
  CSA_CHECK(p->status == nullptr || aligned(p->status, 4), CSA_ERR_ALIGN);
  return launch_ex(cache_write_kernel, dim3(p->n, p->batch), dim3(kThreads), 0, (cudaStream_t)stream, false, 1, 1,
                   p->src, p->n, p->first, to_device(p->dst), p->status);
}

extern "C" int csa_compress(const csa_compress_params* p, csa_stream_t stream) {
  CSA_CHECK(p != nullptr && p->struct_size >= offsetof(csa_compress_params, norm), CSA_ERR_INVALID_ARG);
  CSA_CHECK(p->batch >= 0 && p->m >= 1 && p->dim >= 1, CSA_ERR_SHAPE);
  CSA_CHECK(p->dim <= kThreads * kMaxPer && (p->mode == CSA_COMPRESS_WINDOW || p->dim == p->dst.dim), CSA_ERR_SHAPE);
  CSA_CHECK(p->batch <= 65535, CSA_ERR_SHAPE);
  CSA_CHECK(p->bias != nullptr && aligned(p->bias, 16), p->bias ? CSA_ERR_ALIGN : CSA_ERR_INVALID_ARG);
  if (p->batch == 0) return CSA_OK;
  cudaStream_t s = (cudaStream_t)stream;
  // the optional workspace only carries the run-time status word
  CSA_CHECK(p->workspace == nullptr || (p->workspace_bytes >= sizeof(int32_t) && aligned(p->workspace, 4)),
            CSA_ERR_WORKSPACE);
  int* status = static_cast<int*>(p->workspace);
  // flags: a field present only in structs that reach it
  const int flags = p->struct_size >= offsetof(csa_compress_params, flags) + sizeof(p->flags) ? p->flags : 0;
  CSA_CHECK((flags & ~CSA_FLAG_OVERLAP_PREVIOUS) == 0, CSA_ERR_INVALID_ARG);
  // RMSNorm / RoPE of the pooled entries: fields present only in structs that reach them
  Prep prep{};
  if (p->struct_size >= offsetof(csa_compress_params, rope_base) + sizeof(float)) {
    CSA_CHECK(p->norm == nullptr || aligned(p->norm, 4), CSA_ERR_ALIGN);
    CSA_CHECK(p->norm_eps >= 0.f && p->rope_base >= 0.f, CSA_ERR_INVALID_ARG);
    CSA_CHECK(p->rope_base == 0.f || (p->dim >= kRopeDims && p->dim % 2 == 0), CSA_ERR_SHAPE);
    prep.norm = p->norm;
    prep.eps = p->norm_eps;
    prep.rope = p->rope_base > 0.f;
    prep.freq = rope_freq(p->rope_base);
  }
  // the b stream of overlapping compression: fields present only in structs that reach them
  const bool ab = p->mode == CSA_COMPRESS_DENSE_AB || p->mode == CSA_COMPRESS_APPEND_AB;
  BStream bs{};
  if (ab) {
    CSA_CHECK(p->struct_size >= offsetof(csa_compress_params, tail_gate_b) + sizeof(p->tail_gate_b),
              CSA_ERR_INVALID_ARG);
    CSA_CHECK(p->bias_b != nullptr, CSA_ERR_INVALID_ARG);
    CSA_CHECK(aligned(p->bias_b, 16), CSA_ERR_ALIGN);
    bs.bias = p->bias_b;
    bs.k = p->k_b;
    bs.g = p->g_b;
    bs.k_new = p->k_new_b;
    bs.g_new = p->g_new_b;
    bs.keys = p->tail_b;
    bs.gates = p->tail_gate_b;
  }
  if (p->mode == CSA_COMPRESS_DENSE || p->mode == CSA_COMPRESS_DENSE_AB) {
    CSA_CHECK(p->n_tokens >= 0, CSA_ERR_SHAPE);
    const int nb = p->n_tokens / p->m;
    if (nb == 0) return CSA_OK;
    CSA_CHECK(p->k && p->g, CSA_ERR_INVALID_ARG);
    CSA_CHECK(aligned(p->k, 16) && aligned(p->g, 16), CSA_ERR_ALIGN);
    CSA_CHECK((p->k_dtype == CSA_F32 || p->k_dtype == CSA_BF16) &&
                  (p->g_dtype == CSA_F32 || p->g_dtype == CSA_BF16),
              CSA_ERR_UNSUPPORTED);
    int st = check_store(p->dst, p->batch, nb);
    if (st != CSA_OK) return st;
    if (ab) {
      CSA_CHECK(p->k_b && p->g_b, CSA_ERR_INVALID_ARG);
      CSA_CHECK(aligned(p->k_b, 16) && aligned(p->g_b, 16), CSA_ERR_ALIGN);
      return launch_ex(compress_dense_kernel<true>, dim3(nb, p->batch), dim3(kThreads), 0, s, false, 1, 1, p->k,
                       p->k_dtype, p->g, p->g_dtype, p->bias, p->n_tokens, p->m, p->dim, to_device(p->dst), status,
                       prep, bs);
    }
    return launch_ex(compress_dense_kernel<false>, dim3(nb, p->batch), dim3(kThreads), 0, s, false, 1, 1, p->k,
                     p->k_dtype, p->g, p->g_dtype, p->bias, p->n_tokens, p->m, p->dim, to_device(p->dst), status,
                     prep, bs);
  }
  if (p->mode == CSA_COMPRESS_WINDOW) {  // no compressed entries: the ring only
    CSA_CHECK(p->seq_len && p->k_new && p->ring, CSA_ERR_INVALID_ARG);
    CSA_CHECK(aligned(p->seq_len, 4) && aligned(p->k_new, 16) && aligned(p->ring, 16), CSA_ERR_ALIGN);
    CSA_CHECK(p->ring_size >= 1, CSA_ERR_SHAPE);
    return launch_ex(window_append_kernel, dim3((unsigned)p->batch), dim3(kThreads), 0, s,
                     (flags & CSA_FLAG_OVERLAP_PREVIOUS) != 0, 1, 1, p->seq_len, p->k_new, p->ring, p->ring_size,
                     p->dim);
  }
  if (p->mode == CSA_COMPRESS_APPEND_AB) {
    CSA_CHECK(p->m <= kSmallM, CSA_ERR_UNSUPPORTED);
    CSA_CHECK(p->k_new_b && p->g_new_b && p->tail_b && p->tail_gate_b, CSA_ERR_INVALID_ARG);
    CSA_CHECK(aligned(p->k_new_b, 16) && aligned(p->g_new_b, 16) && aligned(p->tail_b, 16) &&
                  aligned(p->tail_gate_b, 16),
              CSA_ERR_ALIGN);
  }
  if (p->mode == CSA_COMPRESS_APPEND || p->mode == CSA_COMPRESS_APPEND_AB) {
    CSA_CHECK(p->seq_len && p->k_new && p->g_new && p->ring && p->tail_gate, CSA_ERR_INVALID_ARG);
    CSA_CHECK(aligned(p->seq_len, 4) && aligned(p->k_new, 16) && aligned(p->g_new, 16) &&
                  aligned(p->ring, 16) && aligned(p->tail_gate, 16),
              CSA_ERR_ALIGN);
    CSA_CHECK(p->ring_size >= p->m, CSA_ERR_SHAPE);
    // the entry index depends on device-side lengths; the store is checked for
    // layout here and the kernel trusts seq_len to stay within it
    int st = check_store(p->dst, p->batch, 0);
    if (st != CSA_OK) return st;
    CSA_CHECK(p->dim <= kCs * kMaxCpc, CSA_ERR_SHAPE);
    CSA_CHECK(p->m <= kSmallM || p->dim % 8 == 0, CSA_ERR_SHAPE);  // quads of channels for large blocks
    int cpc = (p->dim + kCs - 1) / kCs;
    cpc = (cpc + kFp4Block - 1) / kFp4Block * kFp4Block;
    if (p->m <= kSmallM) {  // a small block: one CTA per sequence
      const bool pdl = (flags & CSA_FLAG_OVERLAP_PREVIOUS) != 0;
      auto go = [&](auto kernel) {
        return launch_ex(kernel, dim3((unsigned)p->batch), dim3(kThreads), 0, s, pdl, 1, 1, p->seq_len, p->k_new,
                         p->g_new, p->ring, p->ring_size, p->tail_gate, p->bias, p->m, p->dim, to_device(p->dst),
                         status, prep, bs);
      };
      if (p->m <= 4) return ab ? go(compress_append_small_kernel<true, 4>) : go(compress_append_small_kernel<false, 4>);
      if (p->m <= 8) return ab ? go(compress_append_small_kernel<true, 8>) : go(compress_append_small_kernel<false, 8>);
      return ab ? go(compress_append_small_kernel<true, 16>) : go(compress_append_small_kernel<false, 16>);
    }
    return launch_ex(compress_append_kernel, dim3((unsigned)(p->batch * kCs)), dim3(kAppThreads), 0, s,
                     (flags & CSA_FLAG_OVERLAP_PREVIOUS) != 0, kCs, 1, p->seq_len, p->k_new, p->g_new, p->ring,
                     p->ring_size, p->tail_gate, p->bias, p->m, p->dim, cpc, to_device(p->dst), status, prep);
  }
  return CSA_ERR_INVALID_ARG;
}
