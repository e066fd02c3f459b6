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

// Writes one entry held as vals[i] = value of dim threadIdx.x + i * kThreads.
// Must be called by every thread of the CTA (it synchronizes).
__device__ void store_entry(const Store& s, int b, int e, const float (&vals)[kMaxPer], float* red) {
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

__global__ void __launch_bounds__(kThreads) compress_dense_kernel(
    const void* __restrict__ k, int k_dtype, const void* __restrict__ g, int g_dtype,
    const float* __restrict__ bias, int n, int m, int dim, Store dst) {
  __shared__ float red[kThreads / 32];
  const int j = blockIdx.x, b = blockIdx.y;
  float vals[kMaxPer];
#pragma unroll
  for (int i = 0; i < kMaxPer; ++i) {
    const int d = threadIdx.x + i * kThreads;
    vals[i] = 0.f;
    if (d < dim) {
      const size_t row0 = (size_t)b * n + (size_t)j * m;
      vals[i] = pool_channel(
          m, bias, d, dim, [&](int t) { return load_as_float(k, k_dtype, (row0 + t) * dim + d); },
          [&](int t) { return load_as_float(g, g_dtype, (row0 + t) * dim + d); });
    }
  }
  store_entry(dst, b, j, vals, red);
}

// Decode append.  Grid (B, channel groups of 32); every CTA appends its
// channel slice of the new token to the state cache and, when the token
// completes a block, pools that slice over the m positions of the block
// (warps split the positions, an online softmax per channel, then a merge of
// the warps).  The pooled slice goes to the workspace; the CTA that finishes
// last for a sequence (an atomic counter, no waiting) quantizes the whole
// entry and writes it to the store, then resets the counter.
constexpr int kGroup = 32;
constexpr int kWarps = kThreads / 32;

__global__ void __launch_bounds__(kThreads) compress_append_kernel(
    const int32_t* __restrict__ seq_len, const uint16_t* __restrict__ k_new,
    const float* __restrict__ g_new, uint16_t* __restrict__ ring, int ring_size,
    float* __restrict__ tail_gate, const float* __restrict__ bias, int m, int dim, Store dst,
    int* __restrict__ counters, float* __restrict__ pooled) {
  __shared__ float red[kThreads / 32];
  __shared__ float part[3][kWarps][kGroup];
  __shared__ int last;
  const int b = blockIdx.x, grp = blockIdx.y, groups = gridDim.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = grp * kGroup + lane;
  const bool live = c < dim;
  const int L = seq_len[b];
  if (L < 0) return;  // uniform over the CTA
  const float kn = live ? bf16_bits_to_float(k_new[(size_t)b * dim + c]) : 0.f;
  const float gn = live ? g_new[(size_t)b * dim + c] : 0.f;
  if (warp == 0 && live) {
    ring[((size_t)b * ring_size + L % ring_size) * dim + c] = k_new[(size_t)b * dim + c];
    tail_gate[((size_t)b * m + L % m) * dim + c] = gn;
  }
  if ((L + 1) % m != 0) return;  // uniform
  const int p0 = L + 1 - m;
  // online softmax over this warp's positions i = warp, warp + kWarps, ...;
  // the loads of up to kBatch positions are issued together before any use
  float mx = -INFINITY, se = 0.f, acc = 0.f;
  if (live) {
    constexpr int kBatch = 11;  // 6 warps x 11 positions cover a 64-token block per pass
    for (int base = warp; base < m; base += kWarps * kBatch) {
      float kv[kBatch], a[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int i = base + u * kWarps;
        kv[u] = 0.f;
        a[u] = -INFINITY;
        if (i < m) {
          const int p = p0 + i;
          kv[u] = i == m - 1 ? kn : bf16_bits_to_float(ring[((size_t)b * ring_size + p % ring_size) * dim + c]);
          a[u] = (i == m - 1 ? gn : tail_gate[((size_t)b * m + p % m) * dim + c]) + bias[(size_t)i * dim + c];
        }
      }
      float bm = a[0];
#pragma unroll
      for (int u = 1; u < kBatch; ++u) bm = fmaxf(bm, a[u]);
      if (bm > mx) {  // bm is finite: position `base` is in range
        const float r = expf(mx - bm);  // 0 on the first batch
        se *= r;
        acc *= r;
        mx = bm;
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const float e = expf(a[u] - mx);  // 0 for positions past the block
        se += e;
        acc = fmaf(e, kv[u], acc);
      }
    }
  }
  part[0][warp][lane] = mx;
  part[1][warp][lane] = se;
  part[2][warp][lane] = acc;
  __syncthreads();
  if (warp == 0 && live) {
    float M = -INFINITY;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, part[0][w][lane]);
    float S = 0.f, A = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      const float s = part[1][w][lane];
      if (s > 0.f) {
        const float r = expf(part[0][w][lane] - M);
        S = fmaf(s, r, S);
        A = fmaf(part[2][w][lane], r, A);
      }
    }
    pooled[(size_t)b * dim + c] = A / S;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(&counters[b], 1) == groups - 1;
  __syncthreads();
  if (!last) return;  // uniform
  __threadfence();
  float vals[kMaxPer];
#pragma unroll
  for (int i = 0; i < kMaxPer; ++i) {
    const int d = threadIdx.x + i * kThreads;
    vals[i] = d < dim ? __ldcg(&pooled[(size_t)b * dim + d]) : 0.f;
  }
  store_entry(dst, b, (L + 1) / m - 1, vals, red);
  if (threadIdx.x == 0) counters[b] = 0;
}

__global__ void __launch_bounds__(kThreads) cache_write_kernel(const float* __restrict__ src, int n,
                                                               int first, Store dst) {
  __shared__ float red[kThreads / 32];
  const int i_row = blockIdx.x, b = blockIdx.y;
  float vals[kMaxPer];
#pragma unroll
  for (int i = 0; i < kMaxPer; ++i) {
    const int d = threadIdx.x + i * kThreads;
    vals[i] = d < dst.dim ? src[((size_t)b * n + i_row) * dst.dim + d] : 0.f;
  }
  store_entry(dst, b, first + i_row, vals, red);
}

}  // namespace
}  // namespace csa

using namespace csa;

extern "C" size_t csa_page_bytes(int32_t format, int32_t page_entries) {
  if (page_entries <= 0 || page_entries % kTile != 0) return 0;
  return page_bytes(format, page_entries);
}

namespace {
size_t append_counter_bytes(int batch) { return ((size_t)batch * sizeof(int) + 255) / 256 * 256; }
}  // namespace

extern "C" size_t csa_compress_workspace_size(const csa_compress_params* p) {
  if (p == nullptr || p->struct_size < sizeof(csa_compress_params) || p->batch < 0 || p->dim < 1) return 0;
  if (p->mode != CSA_COMPRESS_APPEND) return 0;
  return kWsHeader + append_counter_bytes(p->batch) + (size_t)p->batch * p->dim * sizeof(float);
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
  cache_write_kernel<<<dim3(p->n, p->batch), kThreads, 0, (cudaStream_t)stream>>>(p->src, p->n, p->first,
                                                                                  to_device(p->dst));
  return launch_status();
}

extern "C" int csa_compress(const csa_compress_params* p, csa_stream_t stream) {
  CSA_CHECK(p != nullptr && p->struct_size >= sizeof(csa_compress_params), CSA_ERR_INVALID_ARG);
  CSA_CHECK(p->batch >= 0 && p->m >= 1 && p->dim >= 1, CSA_ERR_SHAPE);
  CSA_CHECK(p->dim <= kThreads * kMaxPer && p->dim == p->dst.dim, CSA_ERR_SHAPE);
  CSA_CHECK(p->batch <= 65535, CSA_ERR_SHAPE);
  CSA_CHECK(p->bias != nullptr && aligned(p->bias, 16), p->bias ? CSA_ERR_ALIGN : CSA_ERR_INVALID_ARG);
  if (p->batch == 0) return CSA_OK;
  cudaStream_t s = (cudaStream_t)stream;
  if (p->mode == CSA_COMPRESS_DENSE) {
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
    compress_dense_kernel<<<dim3(nb, p->batch), kThreads, 0, s>>>(p->k, p->k_dtype, p->g, p->g_dtype, p->bias,
                                                                 p->n_tokens, p->m, p->dim, to_device(p->dst));
    return launch_status();
  }
  if (p->mode == CSA_COMPRESS_APPEND) {
    CSA_CHECK(p->seq_len && p->k_new && p->g_new && p->ring && p->tail_gate, CSA_ERR_INVALID_ARG);
    CSA_CHECK(aligned(p->seq_len, 4) && aligned(p->k_new, 16) && aligned(p->g_new, 16) &&
                  aligned(p->ring, 16) && aligned(p->tail_gate, 16),
              CSA_ERR_ALIGN);
    CSA_CHECK(p->ring_size >= p->m, CSA_ERR_SHAPE);
    CSA_CHECK(p->workspace != nullptr, CSA_ERR_WORKSPACE);
    CSA_CHECK(aligned(p->workspace, 1024), CSA_ERR_ALIGN);
    CSA_CHECK(p->workspace_bytes >= csa_compress_workspace_size(p), CSA_ERR_WORKSPACE);
    // the entry index depends on device-side lengths; the store is checked for
    // layout here and the kernel trusts seq_len to stay within it
    int st = check_store(p->dst, p->batch, 0);
    if (st != CSA_OK) return st;
    uint8_t* ws = static_cast<uint8_t*>(p->workspace);
    int* counters = reinterpret_cast<int*>(ws + kWsHeader);
    float* pooled = reinterpret_cast<float*>(ws + kWsHeader + append_counter_bytes(p->batch));
    const dim3 grid(p->batch, (p->dim + kGroup - 1) / kGroup);
    compress_append_kernel<<<grid, kThreads, 0, s>>>(p->seq_len, p->k_new, p->g_new, p->ring, p->ring_size,
                                                     p->tail_gate, p->bias, p->m, p->dim, to_device(p->dst),
                                                     counters, pooled);
    return launch_status();
  }
  return CSA_ERR_INVALID_ARG;
}
