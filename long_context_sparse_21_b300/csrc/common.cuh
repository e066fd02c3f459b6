// Shared device helpers of libcsa: number formats, cache addressing, status.
//
// Storage formats follow the DeepSeek-V4 report (cnblogs translation) §2.3.4
// (FP8 content dims, BF16 RoPE dims) and §5.2.1 (FP4 indexer QK path, BF16
// index scores); the page layout follows §3.5.1 (paged classical cache plus a
// state cache for the window and the uncompressed tail).  The exact byte
// layouts are specified in include/csa.h.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/csa.h"

namespace csa {

constexpr int kKvContent = 512;   // FP8 content dims of a KV entry
constexpr int kKvRope = 64;       // BF16 RoPE dims of a KV entry
constexpr int kKvDim = kKvContent + kKvRope;
constexpr int kKvEntryBytes = kKvContent + 2 * kKvRope + 4;  // 644
constexpr int kIdxDim = 128;      // indexer head dim
constexpr int kTile = 128;        // entries per swizzled indexer tile
constexpr int kFp4Block = 16;     // elements per FP4 scale

// Status word at the head of every workspace.
constexpr size_t kWsHeader = 1024;

__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicCAS(status, CSA_OK, code);
}

// ----------------------------------------------------------------- formats

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
__device__ __forceinline__ uint16_t float_to_bf16_bits(float x) {
  __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&h);
}
__device__ __forceinline__ uint8_t float_to_e4m3(float x) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ float e4m3_to_float(uint8_t c) {
  __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(c), __NV_E4M3);
  return __half2float(__half(h));
}
// Two floats -> one byte of two e2m1 codes (x in the low nibble).
__device__ __forceinline__ uint8_t float2_to_e2m1x2(float x, float y) {
  return static_cast<uint8_t>(__nv_cvt_float2_to_fp4x2(make_float2(x, y), __NV_E2M1, cudaRoundNearest));
}

// ----------------------------------------------------------------- cache addressing

struct Store {
  int32_t format, dim;
  uint8_t* base;
  int32_t capacity, page_entries;
  const int32_t* page_table;
  int32_t max_pages, num_pages;
};

__host__ __device__ inline size_t page_bytes(int format, int P) {
  switch (format) {
    case CSA_FMT_KV_POOL_FP8: return (size_t)kKvEntryBytes * P;
    case CSA_FMT_INDEX_POOL_BF16: return (size_t)2 * kIdxDim * P;
    case CSA_FMT_INDEX_POOL_E2M1: return (size_t)(kIdxDim / 2 + kIdxDim / kFp4Block) * P;
    default: return 0;
  }
}

// Page base and slot of entry e of sequence b (pool formats only; b and e
// within the page table).  nullptr when the page id read from the table lies
// outside [0, num_pages): the caller skips the access and records
// CSA_ERR_INVALID_ARG.
__device__ __forceinline__ uint8_t* page_of(const Store& s, int b, int e, int* slot) {
  const int pg = s.page_table[(size_t)b * s.max_pages + e / s.page_entries];
  *slot = e % s.page_entries;
  if ((unsigned)pg >= (unsigned)s.num_pages) return nullptr;
  return s.base + (size_t)pg * page_bytes(s.format, s.page_entries);
}

// Byte offset of (slot, dim d) inside a BF16 indexer page (128-byte swizzle).
__host__ __device__ __forceinline__ uint32_t idx_bf16_offset(int slot, int d) {
  const int r = slot & 127;
  return (uint32_t)(slot >> 7) * 32768u + (uint32_t)(d >> 6) * 16384u + (uint32_t)r * 128u +
         (uint32_t)((((d & 63) >> 3) ^ (r & 7)) << 4) + (uint32_t)(d & 7) * 2u;
}

// ----------------------------------------------------------------- partial RoPE
// report §2.3.3: RoPE on the last 64 dims of the query and KV vectors.  The
// rotary pairs are (x_2i, x_2i+1) of those dims, turned by pos * f_i with
// f_i = base^(-2i / 64) (computed on the host in double precision).
constexpr int kRopeDims = 64;
constexpr int kRopePairs = kRopeDims / 2;
struct RopeFreq {
  double f[kRopePairs];
};

// (cos, sin) of pos * f for a raw position up to 2^31.  The product and its
// reduction into [-pi, pi] are done in double precision (a float product
// at pos ~ 1e6 would be off by ~0.06 rad); the reduced angle then goes to
// sincosf.
__device__ __forceinline__ float2 rope_cs(double f, long long pos) {
  const double a = (double)pos * f;
  const double two_pi = 6.283185307179586476925286766559;
  const double k = rint(a / two_pi);
  const float r = (float)fma(-k, two_pi, a);
  float s, c;
  __sincosf(r, &s, &c);  // |r| <= pi: the fast path is accurate to ~1e-6 there
  return make_float2(c, s);
}

// (cos, sin) of a float angle of at most a few hundred radians (a position
// offset times a frequency), reduced into [-pi, pi] in float first.
__device__ __forceinline__ float2 small_angle_cs(float a) {
  const float two_pi = 6.28318530717958647692f;
  const float r = fmaf(-rintf(a / two_pi), two_pi, a);
  float s, c;
  __sincosf(r, &s, &c);
  return make_float2(c, s);
}

// (x0, x1) turned by the angle whose (cos, sin) is cs.
__device__ __forceinline__ float2 rotate_pair(float x0, float x1, float2 cs) {
  return make_float2(x0 * cs.x - x1 * cs.y, x0 * cs.y + x1 * cs.x);
}

// Order-preserving map float -> uint32 (larger float -> larger key); -0 -> +0.
__device__ __forceinline__ uint32_t float_to_ordered(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace csa
