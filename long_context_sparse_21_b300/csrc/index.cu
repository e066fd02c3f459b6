// Steps 2 and 3 of the hot path: the lightning indexer and the top-k selector.
//
// DeepSeek-V4 report (cnblogs translation) §2.3.1 "lightning indexer": index
// queries are produced in low rank, scored against every compressed key, and a
// top-k selector keeps a subset of compressed entries for the core attention;
// §5.2.1: the indexer QK path runs in FP4 and the index scores are quantized
// FP32 -> BF16 before selection.  HF blog "DeepSeek-V4" (translation),
// "Hybrid attention": the indexer is a ReLU-scored multi-head dot product.
//     s_j = sum_h w_h * ReLU(q_h . kI_j),  j < N_c(t) = floor((t + 1) / m)
//
// Kernels:
//  * score_f32_kernel     canonical-order float32 scoring on CUDA cores (the
//                         bit-reproducible path).
//  * score_tc_kernel      tcgen05 MMA with TMEM accumulators: a 128-key tile
//                         (M) against the 64 heads of QPC queries (N = 64 QPC),
//                         K = 128, fed by bulk async copies of pre-swizzled
//                         pool tiles through a 2-stage mbarrier pipeline; the
//                         epilogue (one thread per key) applies ReLU and the
//                         head weights straight out of TMEM.  HBM-bound in
//                         decode (64 FLOP per key byte).  BF16 pools.
//  * score_fp4_kernel     FP4 pools: block-scaled tcgen05 MMA
//                         (kind::mxf4nvf4) straight on the pool's E2M1 codes
//                         and per-16 UE4M3 scales (72 B per key), against the
//                         query quantized to the same format; same epilogue.
//  * topk_kernel          radix select (11/11/10-bit digits for float32 keys,
//                         8/8 for bf16 keys; a histogram per warp for 8-bit
//                         digits, warp-aggregated updates of shared copies
//                         otherwise), then an order-preserving compaction in
//                         which each thread owns a contiguous run of blocks
//                         and one scan places them: kept blocks ascending,
//                         ties to the lower index.  A row is shared by a
//                         cluster of up to 16 CTAs that read each other's
//                         histograms through distributed shared memory.
#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include <cooperative_groups.h>

#include "common.cuh"
#include "host.hpp"
#include "tc.cuh"

namespace csa {
namespace {

__device__ __forceinline__ int query_seq(const int32_t* seq, int r) { return seq ? seq[r] : r; }
__device__ __forceinline__ int n_visible(int t, int m) { return t < 0 ? 0 : (t + 1) / m; }

__device__ __forceinline__ void store_score(void* scores, int bf16, size_t off, float s) {
  if (bf16) static_cast<uint16_t*>(scores)[off] = float_to_bf16_bits(s);
  else static_cast<float*>(scores)[off] = s;
}

// ================================================================== float32, canonical order

__global__ void __launch_bounds__(128) score_f32_kernel(const float* __restrict__ q, const float* __restrict__ w,
                                                        int w_shared, const int32_t* __restrict__ pos,
                                                        const int32_t* __restrict__ seq, int batch, int m,
                                                        const float* __restrict__ keys, int cap, int H, int dI,
                                                        void* scores, int stride, int bf16, int* status) {
  extern __shared__ float sm[];
  float* qs = sm;            // [H][dI]
  float* ws = sm + H * dI;   // [H]
  tc::pdl_wait();  // the keys may come from the kernel before
  tc::pdl_trigger();
  const int r = blockIdx.x;
  const int n = min(min(n_visible(pos[r], m), cap), stride);  // positions beyond max_pos are clamped
  const int j = blockIdx.y * 128 + threadIdx.x;
  if ((int)(blockIdx.y * 128) >= n) return;
  const int b = query_seq(seq, r);
  if ((unsigned)b >= (unsigned)batch) {  // a sequence index outside the batch: nothing is read
    if (threadIdx.x == 0) set_status(status, CSA_ERR_INVALID_ARG);
    return;
  }
  for (int i = threadIdx.x; i < H * dI; i += 128) qs[i] = q[(size_t)r * H * dI + i];
  for (int i = threadIdx.x; i < H; i += 128) ws[i] = w[(w_shared ? 0 : (size_t)r * H) + i];
  __syncthreads();
  if (j >= n) return;
  const float* kj = keys + ((size_t)b * cap + j) * dI;
  float s = 0.f;
  for (int h = 0; h < H; ++h) {
    float acc = 0.f;
    for (int d = 0; d < dI; ++d) acc = __fmaf_rn(qs[h * dI + d], kj[d], acc);
    const float rl = acc > 0.f ? acc : 0.f;
    s = __fmaf_rn(ws[h], rl, s);
  }
  store_score(scores, bf16, (size_t)r * stride + j, s);
}

// ================================================================== bf16, tcgen05

constexpr int kStages = 2;  // 2 CTAs per SM keep 4 tiles in flight per SM
constexpr int kTileBytes = kTile * kIdxDim * 2;  // 32 KiB of BF16 keys
constexpr int kTcThreads = 192;  // warp 0 copies, warp 1 MMA, warps 2-5 epilogue

template <int QPC>
struct __align__(1024) TcSmem {
  uint8_t keys[kStages][kTileBytes];
  uint8_t q[2][QPC * 64 * 128];  // K halves: dims [0,64) and [64,128), rows = QPC*64 heads
  alignas(16) float w[QPC][64];
  uint64_t full[kStages], empty[kStages], tfull[2], tempty[2], mma_done;
  uint32_t tmem_base;
  int abort;
};

struct TcArgs {
  const void* q;  // [T][64][128]: bf16 (BF16 pool) or float32 (FP4 pool, quantized in the kernel)
  const float* w;
  int w_shared;
  const int32_t* pos;
  const int32_t* seq;
  int m, T, splits, batch;
  int after_append;  // the previous kernel writes at most each query's last visible key
  Store keys;
  void* scores;
  int stride, bf16;
  int* status;
};

template <int QPC>
__global__ void __launch_bounds__(kTcThreads) score_tc_kernel(TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  TcSmem<QPC>& S = *reinterpret_cast<TcSmem<QPC>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int N = QPC * 64;
  constexpr uint32_t kCols = 2 * N;  // two accumulators
  constexpr int kThreads = kTcThreads;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int row0 = blockIdx.x * QPC;
  const int nq = min(QPC, a.T - row0);
  const int b = query_seq(a.seq, row0);  // the QPC rows of a CTA share a sequence (host-checked batch 1 for QPC > 1)
  if ((unsigned)b >= (unsigned)a.batch) {  // uniform: nothing allocated yet
    tc::pdl_wait();
    if (threadIdx.x == 0) set_status(a.status, CSA_ERR_INVALID_ARG);
    return;
  }
  int nvis[QPC];
  int n_all = 0;
#pragma unroll
  for (int i = 0; i < QPC; ++i) {
    nvis[i] = i < nq ? min(n_visible(a.pos[row0 + i], a.m), a.stride) : 0;
    n_all = max(n_all, nvis[i]);
  }
  const int n_tiles = (n_all + kTile - 1) / kTile;
  const int tps = (n_tiles + a.splits - 1) / a.splits;
  const int t_begin = blockIdx.y * tps;
  const int t_end = min(t_begin + tps, n_tiles);
  if (t_begin >= t_end) {  // uniform: nothing allocated yet
    tc::pdl_wait();
    return;
  }
  const int my_tiles = t_end - t_begin;

  // queries -> shared memory in the swizzled K-major layout, head weights
  {
    const uint16_t* q = static_cast<const uint16_t*>(a.q);
    for (int c = tid; c < N * 16; c += kThreads) {
      const int row = c >> 4, ch = c & 15, half = ch >> 3, cc = ch & 7;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (row / 64 < nq) v = *reinterpret_cast<const uint4*>(q + ((size_t)(row0 + row / 64) * 64 + row % 64) * 128 + ch * 8);
      *reinterpret_cast<uint4*>(&S.q[half][row * 128 + ((cc ^ (row & 7)) << 4)]) = v;
    }
  }
  for (int i = tid; i < N; i += kThreads) {
    const int qi = i / 64, h = i % 64;
    S.w[qi][h] = qi < nq ? a.w[(a.w_shared ? 0 : (size_t)(row0 + qi) * 64) + h] : 0.f;
  }
  tc::fence_proxy_async_smem();
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&S.full[s], 1);
      tc::mbar_init(&S.empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&S.tfull[s], 1);
      tc::mbar_init(&S.tempty[s], 128);
    }
    tc::mbar_init(&S.mma_done, 1);
    S.abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) tc::tmem_alloc(&S.tmem_base, kCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  volatile int* abort = &S.abort;
  // the queries and head weights (inputs of the step) are staged; the key
  // pool may have been written by the kernel before (the compressor's append).
  // After a decode append only the query's last visible key can have been
  // written: the producer waits before it copies that key's tile, and streams
  // every older tile meanwhile.
  const bool late_wait = a.after_append && QPC == 1;
  if (!late_wait) tc::pdl_wait();
  tc::pdl_trigger();
  const int t_new = (n_all - 1) / kTile;  // tile of the last visible key

  if (warp == 0) {
    if (lane == 0) {
      int issued = 0;
      int slot_next;
      const uint8_t* page_next = page_of(a.keys, b, t_begin * kTile, &slot_next);
      for (int it = 0; it < my_tiles; ++it) {
        const int s = it % kStages;
        const int slot = slot_next;
        const uint8_t* page = page_next;
        if (it + 1 < my_tiles) page_next = page_of(a.keys, b, (t_begin + it + 1) * kTile, &slot_next);
        if (!tc::mbar_wait(&S.empty[s], ((it / kStages) & 1) ^ 1, abort, a.status)) break;
        if (late_wait && t_begin + it == t_new) tc::pdl_wait();
        if (page == nullptr) {  // a page id outside the pool: no copy, the stage completes empty
          set_status(a.status, CSA_ERR_INVALID_ARG);
          tc::mbar_arrive(&S.full[s]);
        } else {
          tc::mbar_arrive_expect_tx(&S.full[s], kTileBytes);
          tc::bulk_g2s(S.keys[s], page + (size_t)slot * 256, kTileBytes, &S.full[s]);
        }
        issued = it + 1;
      }
      // every copy this thread started has landed before the CTA can exit
      for (int it = max(0, issued - kStages); it < issued; ++it)
        if (!tc::mbar_wait(&S.full[it % kStages], (it / kStages) & 1, abort, a.status, false)) break;
    }
  } else if (warp == 1) {
    // MMA issuer: the whole warp, converged; one elected lane issues
    // (tc::mma_elect).  The 8 K-steps of a tile are constant offsets from the
    // tile's base descriptors (address field = byte address / 16, low 14 bits,
    // no carry below 256 KiB of shared memory).
    constexpr uint32_t idesc = tc::idesc_bf16_f32(128, N);
    const uint64_t dq0 = tc::desc_sw128(tc::smem_u32(S.q[0])), dq1 = tc::desc_sw128(tc::smem_u32(S.q[1]));
    for (int it = 0; it < my_tiles; ++it) {
      const int s = it % kStages, acc = it & 1;
      if (!tc::mbar_wait_warp(&S.full[s], (it / kStages) & 1, abort, a.status)) break;
      if (!tc::mbar_wait_warp(&S.tempty[acc], ((it >> 1) & 1) ^ 1, abort, a.status)) break;
      tc::tc_fence_after();
      const uint64_t dk = tc::desc_sw128(tc::smem_u32(S.keys[s]));
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        tc::mma_elect(tmem + acc * N, dk + (((ks >> 2) * 16384 + (ks & 3) * 32) >> 4),
                      (ks >> 2 ? dq1 : dq0) + (((ks & 3) * 32) >> 4), idesc, ks > 0);
      tc::mma_commit_elect(&S.empty[s]);
      tc::mma_commit_elect(&S.tfull[acc]);
    }
    tc::mma_commit_elect(&S.mma_done);
    tc::mbar_wait_warp(&S.mma_done, 0, abort, a.status, false);
  } else if (warp < 6) {
    const int quad = warp & 3;  // TMEM lanes [32 quad, 32 quad + 32) belong to this warp
    for (int it = 0; it < my_tiles; ++it) {
      const int acc = it & 1;
      if (!tc::mbar_wait(&S.tfull[acc], (it >> 1) & 1, abort, a.status)) break;
      tc::tc_fence_after();
      const int key = (t_begin + it) * kTile + quad * 32 + lane;
#pragma unroll
      for (int qi = 0; qi < QPC; ++qi) {
        uint32_t v0[32], v1[32];
        const uint32_t ta = tmem + ((uint32_t)(quad * 32) << 16) + acc * N + qi * 64;
        tc::tmem_ld32(ta, v0);
        tc::tmem_ld32(ta + 32, v1);
        tc::tmem_wait_ld();
        float s = 0.f;
        const float4* w4 = reinterpret_cast<const float4*>(S.w[qi]);  // 16-byte broadcast loads
#pragma unroll
        for (int h4 = 0; h4 < 8; ++h4) {
          const float4 w = w4[h4];
          s = fmaf(w.x, fmaxf(__uint_as_float(v0[4 * h4]), 0.f), s);
          s = fmaf(w.y, fmaxf(__uint_as_float(v0[4 * h4 + 1]), 0.f), s);
          s = fmaf(w.z, fmaxf(__uint_as_float(v0[4 * h4 + 2]), 0.f), s);
          s = fmaf(w.w, fmaxf(__uint_as_float(v0[4 * h4 + 3]), 0.f), s);
        }
#pragma unroll
        for (int h4 = 0; h4 < 8; ++h4) {
          const float4 w = w4[8 + h4];
          s = fmaf(w.x, fmaxf(__uint_as_float(v1[4 * h4]), 0.f), s);
          s = fmaf(w.y, fmaxf(__uint_as_float(v1[4 * h4 + 1]), 0.f), s);
          s = fmaf(w.z, fmaxf(__uint_as_float(v1[4 * h4 + 2]), 0.f), s);
          s = fmaf(w.w, fmaxf(__uint_as_float(v1[4 * h4 + 3]), 0.f), s);
        }
        if (key < nvis[qi]) store_score(a.scores, a.bf16, (size_t)(row0 + qi) * a.stride + key, s);
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&S.tempty[acc]);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, kCols);
  tc::pdl_wait();  // (returns at once if it already returned) completion implies the predecessor's
}

// ================================================================== FP4, block-scaled tcgen05
//
// The FP4 pool's codes go to the tensor core as they are: one
// tcgen05.mma kind::mxf4nvf4 (E2M1 operands, one UE4M3 scale per 16 elements
// along K) per 64 dims, M = 128 keys x N = 64 heads, F32 accumulator, so a
// 128-dim score tile takes two MMAs.  The query is quantized to the same
// format in the prologue (the pool writer's rounding), so the MMA multiplies
// exactly the decoded values c_q s_q and c_k s_k of the FP4 definition
// (report §5.2.1); only the order of the F32 accumulation differs from a
// plain dot product.
//
// Per key tile the copy warp moves 8 KiB of codes by one TMA load of a 3-D
// tensor map over the pool (64 code bytes x P slots x pages), which writes
// them in the canonical 64-byte swizzled K-major layout the MMA reads, and
// 1 KiB of block scales by one bulk async copy.  Four pack warps put the
// scales into the scale-factor layout of a 32 x 128-bit tcgen05.cp (byte
// 16 (k % 32) + 4 (k / 32) + block for key k, one 512-byte block per 64-dim
// half).  The MMA warp copies the tile's scales into TMEM and issues the two
// MMAs; the epilogue warps apply ReLU and the head weights as in the BF16
// kernel.
constexpr int kF4Stages = 10;  // 9 KiB tiles: ~92 KiB of copies in flight per CTA, two CTAs per SM
constexpr int kF4Accs = 3;  // accumulators in flight between the MMA warp and the epilogue
constexpr int kF4CodeBytes = kTile * (kIdxDim / 2);           // 8 KiB
constexpr int kF4ScaleBytes = kTile * (kIdxDim / kFp4Block);  // 1 KiB
constexpr int kF4PackThreads = 128;
// copy warp, MMA warp, two epilogue warpgroups (alternate tiles), 4 pack warps
constexpr int kF4Threads = 64 + 256 + kF4PackThreads;
// TMEM columns: accumulators [0, 64 kF4Accs), then the key scales (two
// halves x 4 columns per accumulator), then the query scales (8)
constexpr uint32_t kF4SfaCol = 64 * kF4Accs, kF4SfbCol = kF4SfaCol + 8 * kF4Accs;
constexpr uint32_t kF4Cols = 256;  // two CTAs per SM
static_assert(kF4SfbCol + 8 <= kF4Cols, "TMEM columns");

struct __align__(1024) F4Smem {
  uint8_t codes[kF4Stages][kF4CodeBytes];
  uint8_t q[64 * (kIdxDim / 2)];                // query codes, 64 heads, 64-byte swizzled
  uint8_t sfa[kF4Stages][2][512];               // key scales in the tcgen05.cp layout, per 64-dim half
  uint8_t sfb[2][512];                          // query scales, same layout (rows 64-127 zero)
  uint8_t raw_sc[kF4Stages][kF4ScaleBytes];     // key scales as copied: [key][block]
  alignas(16) float w[64];
  uint64_t full[kF4Stages], packed[kF4Stages], empty[kF4Stages], tfull[kF4Accs], tempty[kF4Accs], mma_done;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// two CTAs of 448 threads per SM: at most 72 registers a thread
__global__ void __launch_bounds__(kF4Threads, 2) score_fp4_kernel(TcArgs a, const __grid_constant__ CUtensorMap codes_map) {
  extern __shared__ uint8_t smem_raw[];
  F4Smem& S = *reinterpret_cast<F4Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int r = blockIdx.x;
  const int b = query_seq(a.seq, r);
  if ((unsigned)b >= (unsigned)a.batch) {  // uniform: nothing allocated yet
    tc::pdl_wait();
    if (threadIdx.x == 0) set_status(a.status, CSA_ERR_INVALID_ARG);
    return;
  }
  const int nvis = min(n_visible(a.pos[r], a.m), a.stride);
  const int n_tiles = (nvis + kTile - 1) / kTile;
  const int tps = (n_tiles + a.splits - 1) / a.splits;
  const int t_begin = blockIdx.y * tps;
  const int t_end = min(t_begin + tps, n_tiles);
  if (t_begin >= t_end) {  // uniform: nothing allocated yet
    tc::pdl_wait();
    return;
  }
  const int my_tiles = t_end - t_begin;

  if (tid == 0) {
    for (int s = 0; s < kF4Stages; ++s) {
      tc::mbar_init(&S.full[s], 1);
      tc::mbar_init(&S.packed[s], kF4PackThreads);
      tc::mbar_init(&S.empty[s], 1);
    }
    for (int s = 0; s < kF4Accs; ++s) {
      tc::mbar_init(&S.tfull[s], 1);
      tc::mbar_init(&S.tempty[s], 128);
    }
    tc::mbar_init(&S.mma_done, 1);
    S.abort = 0;
    tc::fence_mbar_init();
  }
  for (int i = tid; i < (int)sizeof(S.sfb) / 16; i += kF4Threads) reinterpret_cast<uint4*>(&S.sfb[0][0])[i] = make_uint4(0, 0, 0, 0);
  if (warp == 1) tc::tmem_alloc(&S.tmem_base, kF4Cols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  volatile int* abort = &S.abort;
  // as in the BF16 kernel: after a decode append only the last visible key
  // can have been written, and the copy warp waits just before its tile
  const bool late_wait = a.after_append != 0;
  const int t_new = (nvis - 1) / kTile;

  if (warp == 0) {
    // copy warp: starts streaming key tiles at once; the other warps quantize
    // the query meanwhile.  Lane j looks up the page of tile base + j for 32
    // tiles at a time (one parallel round trip), and lane 0 issues the copies
    // from those registers, so no dependent page-table load sits between two
    // copies.
    if (!late_wait) tc::pdl_wait();
    tc::pdl_trigger();
    const int P = a.keys.page_entries;
    const size_t page_bytes_fp4 = (size_t)(kIdxDim / 2 + kIdxDim / kFp4Block) * P;
    int issued = 0;
    bool ok = true;
    for (int base = 0; ok && base < my_tiles; base += 32) {
      int pg_j = -1, slot_j = 0;
      if (base + lane < my_tiles) {
        const int e = (t_begin + base + lane) * kTile;
        pg_j = a.keys.page_table[(size_t)b * a.keys.max_pages + e / P];
        slot_j = e % P;
      }
      const int n = min(32, my_tiles - base);
      for (int j = 0; j < n; ++j) {
        const int it = base + j, s = it % kF4Stages;
        const int pg = __shfl_sync(0xffffffffu, pg_j, j);
        const int slot = __shfl_sync(0xffffffffu, slot_j, j);
        ok = tc::mbar_wait_warp(&S.empty[s], ((it / kF4Stages) & 1) ^ 1, abort, a.status);
        if (!ok) break;
        if (late_wait && t_begin + it == t_new) tc::pdl_wait();
        if (lane == 0) {
          if ((unsigned)pg >= (unsigned)a.keys.num_pages) {  // outside the pool: no copy, the stage completes empty
            set_status(a.status, CSA_ERR_INVALID_ARG);
            tc::mbar_arrive(&S.full[s]);
          } else {
            // codes of slots [slot, slot + 128) of page pg (swizzled by the
            // copy), then their scales [P][8] from the same page
            tc::mbar_arrive_expect_tx(&S.full[s], kF4CodeBytes + kF4ScaleBytes);
            tc::tma_load_3d(S.codes[s], &codes_map, 0, slot, pg, &S.full[s]);
            tc::bulk_g2s(S.raw_sc[s],
                         a.keys.base + (size_t)pg * page_bytes_fp4 + (size_t)(kIdxDim / 2) * P +
                             (size_t)slot * (kIdxDim / kFp4Block),
                         kF4ScaleBytes, &S.full[s]);
          }
        }
        issued = it + 1;
      }
    }
    // every copy this warp started has landed before the CTA can exit
    if (lane == 0)
      for (int it = max(0, issued - kF4Stages); it < issued; ++it)
        if (!tc::mbar_wait(&S.full[it % kF4Stages], (it / kF4Stages) & 1, abort, a.status, false)) break;
  } else {
    // warps 1-13: the query (an input of the step) -> FP4 codes (64-byte
    // swizzled rows) and scales (tcgen05.cp layout), and the head weights
    constexpr int kQThreads = kF4Threads - 32;
    const int u = tid - 32;
    for (int blk = u; blk < 64 * (kIdxDim / kFp4Block); blk += kQThreads) {
      const int h = blk / (kIdxDim / kFp4Block), bi = blk % (kIdxDim / kFp4Block);
      const float4* src =
          reinterpret_cast<const float4*>(static_cast<const float*>(a.q) + ((size_t)r * 64 + h) * kIdxDim + bi * kFp4Block);
      float x[kFp4Block];
#pragma unroll
      for (int i = 0; i < kFp4Block / 4; ++i) {
        const float4 v = src[i];
        x[4 * i] = v.x;
        x[4 * i + 1] = v.y;
        x[4 * i + 2] = v.z;
        x[4 * i + 3] = v.w;
      }
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < kFp4Block; ++i) amax = fmaxf(amax, fabsf(x[i]));
      const uint8_t sb = float_to_e4m3(__fdiv_rn(amax, 6.0f));
      const float sc = e4m3_to_float(sb);
      uint32_t cw[2] = {0u, 0u};
      if (sc != 0.f)
#pragma unroll
        for (int i = 0; i < kFp4Block / 2; ++i)
          cw[i >> 2] |= (uint32_t)float2_to_e2m1x2(__fdiv_rn(x[2 * i], sc), __fdiv_rn(x[2 * i + 1], sc)) << (8 * (i & 3));
      // elements 16 bi .. 16 bi + 15 = bytes 8 bi .. 8 bi + 7 of the row: half of chunk bi / 2
      *reinterpret_cast<uint2*>(&S.q[h * 64 + (((bi >> 1) ^ ((h >> 1) & 3)) << 4) + 8 * (bi & 1)]) = make_uint2(cw[0], cw[1]);
      S.sfb[bi >> 2][16 * (h & 31) + 4 * (h >> 5) + (bi & 3)] = sb;
    }
    for (int h = u; h < 64; h += kQThreads) S.w[h] = a.w[(a.w_shared ? 0 : (size_t)r * 64) + h];
    tc::fence_proxy_async_smem();
    named_bar_sync(1, kQThreads);
    if (warp == 1) {
      // MMA issuer: the whole warp, converged; one elected lane issues the
      // scale copies and the MMAs, which the tensor core runs in that order
      constexpr uint32_t idesc = tc::idesc_mxf4nvf4(128, 64);
      const uint64_t dq = tc::desc_sw64(tc::smem_u32(S.q));
      tc::sf_copy_elect(tmem + kF4SfbCol, tc::desc_rows16(tc::smem_u32(S.sfb[0])));
      tc::sf_copy_elect(tmem + kF4SfbCol + 4, tc::desc_rows16(tc::smem_u32(S.sfb[1])));
      for (int it = 0; it < my_tiles; ++it) {
        const int s = it % kF4Stages, acc = it % kF4Accs;
        if (!tc::mbar_wait_warp(&S.packed[s], (it / kF4Stages) & 1, abort, a.status)) break;
        // accumulator acc (and its scale columns) free: the epilogue has read tile it - kF4Accs
        if (!tc::mbar_wait_warp(&S.tempty[acc], ((it / kF4Accs) & 1) ^ 1, abort, a.status)) break;
        tc::tc_fence_after();
        const uint32_t sfa = tmem + kF4SfaCol + 8 * acc;
        tc::sf_copy_elect(sfa, tc::desc_rows16(tc::smem_u32(S.sfa[s][0])));
        tc::sf_copy_elect(sfa + 4, tc::desc_rows16(tc::smem_u32(S.sfa[s][1])));
        const uint64_t dk = tc::desc_sw64(tc::smem_u32(S.codes[s]));
        tc::mma_fp4_elect(tmem + acc * 64, dk, dq, idesc, sfa, tmem + kF4SfbCol, 0);
        tc::mma_fp4_elect(tmem + acc * 64, dk + (32 >> 4), dq + (32 >> 4), idesc, sfa + 4, tmem + kF4SfbCol + 4, 1);
        tc::mma_commit_elect(&S.empty[s]);
        tc::mma_commit_elect(&S.tfull[acc]);
      }
      tc::mma_commit_elect(&S.mma_done);
      tc::mbar_wait_warp(&S.mma_done, 0, abort, a.status, false);
    } else if (warp < 10) {
      // epilogue: warpgroup g (warps 2-5, 6-9) takes tiles it = g (mod 2);
      // warp w reads TMEM lanes [32 (w % 4), + 32), one key per thread, the
      // 64 heads in two loads of 32 columns
      const int quad = warp & 3, g = (warp - 2) >> 2;
      for (int it = g; it < my_tiles; it += 2) {
        const int acc = it % kF4Accs;
        if (!tc::mbar_wait(&S.tfull[acc], (it / kF4Accs) & 1, abort, a.status)) break;
        tc::tc_fence_after();
        const int key = (t_begin + it) * kTile + quad * 32 + lane;
        const uint32_t ta = tmem + ((uint32_t)(quad * 32) << 16) + acc * 64;
        const float4* w4 = reinterpret_cast<const float4*>(S.w);  // 16-byte broadcast loads
        // four partial sums over heads h = j (mod 4), so the FMA chains are 16 deep
        float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t v[32];
          tc::tmem_ld32(ta + 32 * half, v);
          tc::tmem_wait_ld();
#pragma unroll
          for (int h4 = 0; h4 < 8; ++h4) {
            const float4 w = w4[8 * half + h4];
            p0 = fmaf(w.x, fmaxf(__uint_as_float(v[4 * h4]), 0.f), p0);
            p1 = fmaf(w.y, fmaxf(__uint_as_float(v[4 * h4 + 1]), 0.f), p1);
            p2 = fmaf(w.z, fmaxf(__uint_as_float(v[4 * h4 + 2]), 0.f), p2);
            p3 = fmaf(w.w, fmaxf(__uint_as_float(v[4 * h4 + 3]), 0.f), p3);
          }
        }
        tc::tc_fence_before();
        tc::mbar_arrive(&S.tempty[acc]);
        const float sc = (p0 + p1) + (p2 + p3);
        if (key < nvis) store_score(a.scores, a.bf16, (size_t)r * a.stride + key, sc);
      }
    } else {
      // pack warps: thread k owns key k of every tile
      const int k = tid - 320;  // 0..127
      for (int it = 0; it < my_tiles; ++it) {
        const int s = it % kF4Stages;
        if (!tc::mbar_wait(&S.full[s], (it / kF4Stages) & 1, abort, a.status)) break;
        // scales: blocks 0-3 (dims 0-63) and 4-7 (dims 64-127) of key k
        const uint2 sc = *reinterpret_cast<const uint2*>(S.raw_sc[s] + 8 * k);
        *reinterpret_cast<uint32_t*>(&S.sfa[s][0][16 * (k & 31) + 4 * (k >> 5)]) = sc.x;
        *reinterpret_cast<uint32_t*>(&S.sfa[s][1][16 * (k & 31) + 4 * (k >> 5)]) = sc.y;
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(&S.packed[s]);
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, kF4Cols);
  tc::pdl_wait();  // (returns at once if it already returned) completion implies the predecessor's
}

// ================================================================== top-k

constexpr int kTopkThreads = 1024;
constexpr int kMaxTopkCluster = 16;  // CTAs per row at most (non-portable beyond 8: used only when they fit)
constexpr int kHistBuf = 32 * 256;  // words of one pass's histogram copies (one 256-bin copy per warp for
                                     // bf16 keys); two buffers alternate by pass, in dynamic shared memory
constexpr int kTopkMaxSmemKeys = 40960;  // keys of a CTA's chunk staged in shared memory at most: 160 KiB,
                                         // beside the two 32 KiB histogram buffers (224 KiB of dynamic shared
                                         // memory); covers rows of 655,360 scores over 16 CTAs

__device__ __forceinline__ uint32_t score_key(const void* scores, int bf16, size_t off) {
  if (bf16) {
    // bf16 order key: same construction as float32, on the 16-bit pattern
    uint32_t u = static_cast<const uint16_t*>(scores)[off];
    if (u == 0x8000u) u = 0;
    return (u & 0x8000u) ? (~u & 0xFFFFu) : (u | 0x8000u);
  }
  return float_to_ordered(static_cast<const float*>(scores)[off]);
}

// The two halves of a cluster barrier: arrive (release: this thread's earlier
// stores into peers' shared memory are visible to them after their wait) and
// wait for every thread of the cluster to have arrived (acquire).
__device__ __forceinline__ void cluster_arrive_release() { asm volatile("barrier.cluster.arrive.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait_all() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

// Exclusive prefix sum over the CTA (kTopkThreads threads); returns the total.
__device__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* excl, uint32_t* warp_tot) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t x = v;
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[wid] = x;
  __syncthreads();
  if (wid == 0) {
    uint32_t t = warp_tot[lane];
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    warp_tot[lane] = t;  // inclusive over warps
  }
  __syncthreads();
  const uint32_t before = (wid ? warp_tot[wid - 1] : 0u) + x - v;
  const uint32_t total = warp_tot[31];
  __syncthreads();
  *excl = before;
  return total;
}

// One query row per thread-block cluster of CS CTAs (CS = cluster size at
// launch, 1..8).  CTA q of the cluster owns scores [q c, (q + 1) c) of the
// row, c = ceil(stride / CS) (cut at the row's visible count n), so its loads
// go out together with the load of the query's position.  Each radix pass
// builds a histogram per CTA; every CTA reads the cluster's histograms
// through distributed shared memory and derives the same digit, and from the
// same reads it also counts, for every CTA of the cluster, its keys above the
// digit (and, after the last pass, equal to the threshold).  The compaction
// starts each CTA's output after the counts of the CTAs before it, so the
// output stays ascending, with no further exchange.  Passes alternate between
// two histogram buffers: the only cluster barrier of a pass is the one that
// publishes its histograms.  cluster.sync() is a hardware barrier: nothing
// here spins.
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const void* __restrict__ scores, int bf16, int stride,
                                                            const int32_t* __restrict__ pos, int m, int k,
                                                            int32_t* __restrict__ idx, int32_t* __restrict__ cnt,
                                                            float* __restrict__ scores_out, int scores_out_cap,
                                                            int smem_keys, int* status) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ uint32_t dyn_s[];
  uint32_t* hist = dyn_s;                   // two histogram buffers
  uint32_t* keys_s = dyn_s + 2 * kHistBuf;  // this CTA's chunk as order keys (when it fits)
  __shared__ uint32_t warp_tot[32];
  __shared__ uint32_t sh_digit, sh_krem;
  __shared__ uint32_t cq_gt[kMaxTopkCluster], cq_eq[kMaxTopkCluster];  // per CTA of the cluster: keys above /
                                                                     // equal to the threshold
  __shared__ uint32_t own_gt, own_eq;                                 // this CTA's
  tc::pdl_wait();  // the scores of the kernel before
  tc::pdl_trigger();
  const int CS = (int)cluster.num_blocks();
  const int q = (int)cluster.block_rank();
  const int r = blockIdx.x / CS, tid = threadIdx.x;
  const int32_t pos_r = pos[r];  // used only after the score loads below are issued
  const size_t base = (size_t)r * stride;
  int32_t* out = idx + (size_t)r * k;
  const int chunk = (stride + CS - 1) / CS;
  const int j_lo = q * chunk, j_hi = min(stride, j_lo + chunk);  // inside the row's stride: always readable
  const bool in_smem = chunk <= smem_keys;  // uniform over the cluster
  int n = -1, c0 = 0, c1 = 0;  // the visible scores, and this CTA's part [c0, c1) of them
  auto bounds = [&]() {
    n = min(n_visible(pos_r, m), stride);
    c0 = min(n, j_lo);
    c1 = min(n, j_hi);
  };

  // the chunk's keys, read once with sixteen loads in flight per thread, into
  // shared memory (later passes read them from there); NaN check on the way
  bool nan_seen = false;
  for (int i = tid; i < kHistBuf; i += kTopkThreads) hist[i] = 0;  // the first pass's buffer
  if (in_smem) {
    // four keys per load (8 bytes of BF16, 16 of float32: the chunk starts on
    // a multiple of 16 keys) and per shared-memory store (lane l writes
    // words 4 l .. 4 l + 3: no bank conflict), eight loads in flight per thread
    const int nvec = (j_hi - j_lo) / 4;
    for (int v0 = 0; v0 < nvec; v0 += 8 * kTopkThreads) {
      uint4 raw[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int v = v0 + u * kTopkThreads + tid;
        raw[u] = make_uint4(0u, 0u, 0u, 0u);
        if (v < nvec) {
          const size_t j = base + (size_t)j_lo + 4 * (size_t)v;
          if (bf16) {
            const uint2 x = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(scores) + j);
            raw[u].x = x.x;
            raw[u].y = x.y;
          } else {
            raw[u] = *reinterpret_cast<const uint4*>(static_cast<const float*>(scores) + j);
          }
        }
      }
      if (n < 0) bounds();
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int v = v0 + u * kTopkThreads + tid;
        const int jb = j_lo + 4 * v;
        if (v < nvec && jb >= c0 && jb < c1) {
          // float32 bit patterns of the four keys (a BF16 key in the high half)
          const uint32_t rw[4] = {bf16 ? raw[u].x << 16 : raw[u].x, bf16 ? raw[u].x & 0xFFFF0000u : raw[u].y,
                                  bf16 ? raw[u].y << 16 : raw[u].z, bf16 ? raw[u].y & 0xFFFF0000u : raw[u].w};
          uint32_t kk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (jb + e < c1) nan_seen |= (rw[e] & 0x7FFFFFFFu) > 0x7F800000u;
            kk[e] = bf16 ? (float_to_ordered(__uint_as_float(rw[e])) >> 16) : float_to_ordered(__uint_as_float(rw[e]));
          }
          *reinterpret_cast<uint4*>(keys_s + (jb - c0)) = make_uint4(kk[0], kk[1], kk[2], kk[3]);
        }
      }
    }
  }
  __syncthreads();  // staged keys and the cleared first buffer
  if (n < 0) bounds();

  if (scores_out) {
    for (int j = c0 + tid; j < c1 && j < scores_out_cap; j += kTopkThreads) {
      const size_t o = base + j;
      scores_out[(size_t)r * scores_out_cap + j] =
          bf16 ? bf16_bits_to_float(static_cast<const uint16_t*>(scores)[o]) : static_cast<const float*>(scores)[o];
    }
  }
  if (n <= k) {  // uniform over the cluster
    if (q == 0) {
      for (int j = tid; j < k; j += kTopkThreads) out[j] = j < n ? j : -1;
      if (tid == 0) cnt[r] = max(n, 0);
    }
    return;
  }

  auto key_at = [&](int j) -> uint32_t { return in_smem ? keys_s[j - c0] : score_key(scores, bf16, base + j); };

  // radix select of the k-th largest key, most significant digit first
  const int key_bits = bf16 ? 16 : 32;
  const int npass = bf16 ? 2 : 3;
  uint32_t prefix = 0, prefix_mask = 0, krem = (uint32_t)k;
  int shift = key_bits;
  if (tid == 0) own_gt = own_eq = 0u;  // (first used after the barriers of pass 0)
  for (int pass = 0; pass < npass; ++pass) {
    const int width = bf16 ? 8 : (pass < 2 ? 11 : 10);
    shift -= width;
    const uint32_t nb = 1u << width;
    // nsub copies of this pass's histogram in buffer pass % 2, warp w counting
    // into copy w % nsub.  With a copy per warp (8-bit digits) each lane adds
    // plainly (collisions stay inside the warp); with shared copies, lanes of
    // equal digit are first grouped (one atomic per distinct digit of the
    // warp).  (Grouping, or counting runs of equal digits per thread, measured
    // slower than plain adds into a warp's own copy: with 32 warps per CTA
    // these loops are bound by instructions issued per key.)
    const int nsub = kHistBuf / (int)nb;
    const bool own_copy = nsub >= kTopkThreads / 32;
    uint32_t* hb = hist + (size_t)(pass & 1) * kHistBuf;
    uint32_t* my_hist = hb + (size_t)((tid >> 5) % nsub) * nb;  // (cleared before this pass)
    for (int j0 = c0; j0 < c1; j0 += kTopkThreads) {
      const int j = j0 + tid;
      bool live = false;
      uint32_t digit = 0;
      if (j < c1) {
        const uint32_t key = key_at(j);
        if (!in_smem && pass == 0) {  // first pass: NaN check on the raw bits
          const uint32_t raw = bf16 ? (uint32_t)static_cast<const uint16_t*>(scores)[base + j] << 16
                                    : __float_as_uint(static_cast<const float*>(scores)[base + j]);
          nan_seen |= (raw & 0x7FFFFFFFu) > 0x7F800000u;
        }
        live = (key & prefix_mask) == prefix;
        digit = (key >> shift) & (nb - 1);
      }
      if (own_copy) {
        if (live) atomicAdd(&my_hist[digit], 1u);
      } else {
        const uint32_t active = __ballot_sync(0xffffffffu, live);
        if (live) {
          const uint32_t peers = __match_any_sync(active, digit);
          if ((__ffs(peers) - 1) == (tid & 31)) atomicAdd(&my_hist[digit], __popc(peers));
        }
      }
    }
    if (nsub > 1) {
      __syncthreads();
      for (int i = tid; i < (int)nb; i += kTopkThreads) {
        uint32_t v = hb[i];
        for (int c = 1; c < nsub; ++c) v += hb[(size_t)c * nb + i];
        hb[i] = v;
      }
    }
    // every CTA's histogram of this pass is complete, and every CTA has
    // finished reading the previous pass's histograms: their buffer is
    // cleared now for the next pass (ordered before it by the CTA barrier
    // below)
    cluster.sync();
    if (pass + 1 < npass) {
      uint32_t* nxt = hist + (size_t)((pass + 1) & 1) * kHistBuf;
      for (int i = tid; i < kHistBuf; i += kTopkThreads) nxt[i] = 0;
    }
    // this thread's two bins (from the high end), summed over the cluster
    const int hi_bin = (int)nb - 1 - 2 * tid;
    uint32_t h1 = 0, h0 = 0;
    if (hi_bin >= 0) {
      for (int cq = 0; cq < CS; ++cq) {
        const uint32_t* hq = cluster.map_shared_rank(hb, cq);
        h1 += hq[hi_bin];
        if (hi_bin >= 1) h0 += hq[hi_bin - 1];
      }
    }
    const uint32_t mine = h1 + h0;
    uint32_t above;
    block_exclusive_scan(mine, &above, warp_tot);  // keys in bins above hi_bin
    if (hi_bin >= 0) {
      if (above < krem && krem <= above + h1) {
        sh_digit = (uint32_t)hi_bin;
        sh_krem = krem - above;
      } else if (hi_bin >= 1 && above + h1 < krem && krem <= above + mine) {
        sh_digit = (uint32_t)(hi_bin - 1);
        sh_krem = krem - above - h1;
      }
    }
    __syncthreads();
    const int dg = (int)sh_digit;
    // this CTA's own keys of this prefix in bins above the digit (all of them
    // exceed the threshold) and, after the last pass, in the digit's bin
    // (equal to it), from its own histogram
    {
      uint32_t a = 0u;
      if (hi_bin >= 0) {
        if (hi_bin > dg) a += hb[hi_bin];
        if (hi_bin >= 1 && hi_bin - 1 > dg) a += hb[hi_bin - 1];
        if (pass == npass - 1) {
          if (hi_bin == dg) own_eq = hb[hi_bin];
          else if (hi_bin >= 1 && hi_bin - 1 == dg) own_eq = hb[hi_bin - 1];
        }
      }
      for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
      if ((tid & 31) == 0 && a) atomicAdd(&own_gt, a);
    }
    prefix |= (uint32_t)dg << shift;
    prefix_mask |= (nb - 1) << shift;
    krem = sh_krem;
  }
  // every CTA's counts into every CTA's slots (slot cq written by CTA cq
  // only); the arrive releases them and ends this CTA's reads of the peers'
  // shared memory, so after the wait nothing touches another CTA's shared
  // memory and any CTA may exit
  __syncthreads();
  if (tid < CS) {
    cluster.map_shared_rank(cq_gt, tid)[q] = own_gt;
    cluster.map_shared_rank(cq_eq, tid)[q] = own_eq;
  }
  cluster_arrive_release();
  cluster_wait_all();
  if (__syncthreads_or(nan_seen) && tid == 0) set_status(status, CSA_ERR_INVALID_ARG);
  const uint32_t thr = prefix;  // exact key of the k-th largest; take krem of its ties

  // ---- order-preserving compaction.  Thread t owns the run [c0 + t R, c0 +
  // (t + 1) R) of the chunk: it marks its keys above / equal to the
  // threshold (visiting them in a per-thread rotated order, so the warp's
  // shared-memory reads fall in different banks), one scan over the
  // per-thread counts gives its offsets, and it writes its kept blocks in
  // ascending order.  Position of a kept block = #greater before it +
  // min(#equal before it, krem).
  const int R = (c1 - c0 + kTopkThreads - 1) / kTopkThreads;
  const int r0 = c0 + tid * R, r1 = min(c1, r0 + R);
  uint64_t gtm = 0, eqm = 0;  // bit i: block r0 + i (runs of up to 64 blocks)
  uint32_t gt_loc = 0, eq_loc = 0;
  {
    int ii = R > 0 ? tid % R : 0;
    for (int i = 0; i < R; ++i, ++ii) {
      if (ii >= R) ii -= R;
      const int j = r0 + ii;
      if (j < r1) {
        const uint32_t key = key_at(j);
        const uint64_t g = key > thr, e = key == thr;
        gt_loc += (uint32_t)g;
        eq_loc += (uint32_t)e;
        if (ii < 64) {
          gtm |= g << ii;
          eqm |= e << ii;
        }
      }
    }
  }
  uint32_t gt_before, eq_before;
  block_exclusive_scan(gt_loc, &gt_before, warp_tot);
  block_exclusive_scan(eq_loc, &eq_before, warp_tot);
  for (int cq = 0; cq < q; ++cq) {  // the CTAs before this one in the row (counted from the histograms)
    gt_before += cq_gt[cq];
    eq_before += cq_eq[cq];
  }
  for (int s0 = 0; s0 < R; s0 += 64) {
    if (R > 64) {  // long runs (chunks beyond the shared-memory stage): mark this segment again, in order
      gtm = eqm = 0;
      for (int i = 0; i < 64 && r0 + s0 + i < r1; ++i) {
        const uint32_t key = key_at(r0 + s0 + i);
        gtm |= (uint64_t)(key > thr) << i;
        eqm |= (uint64_t)(key == thr) << i;
      }
    }
    uint64_t sel = gtm | eqm;
    while (sel) {
      const int i = __ffsll((long long)sel) - 1;
      sel &= sel - 1;
      const int j = r0 + s0 + i;
      if ((gtm >> i) & 1) {
        const uint32_t at = gt_before + min(eq_before, krem);
        if (at < (uint32_t)k) out[at] = j;
        ++gt_before;
      } else {
        if (eq_before < krem && gt_before + eq_before < (uint32_t)k) out[gt_before + eq_before] = j;
        ++eq_before;
      }
    }
  }
  if (q == 0 && tid == 0) cnt[r] = k;
}

}  // namespace
}  // namespace csa

using namespace csa;

namespace {

int index_stride(const csa_index_params* p) {
  const int64_t nmax = (int64_t)(p->max_pos + 1) / p->m;
  return (int)std::max<int64_t>(kTile, (nmax + kTile - 1) / kTile * kTile);
}

// Flags of a call (0 for a struct that ends before the field).
int index_flags(const csa_index_params* p) {
  return p->struct_size >= offsetof(csa_index_params, flags) + sizeof(p->flags) ? p->flags : 0;
}

int check_index(const csa_index_params* p) {
  CSA_CHECK(p != nullptr && p->struct_size >= offsetof(csa_index_params, flags), CSA_ERR_INVALID_ARG);
  CSA_CHECK((index_flags(p) & ~(CSA_FLAG_OVERLAP_PREVIOUS | CSA_FLAG_AFTER_APPEND)) == 0, CSA_ERR_INVALID_ARG);
  CSA_CHECK(p->num_queries >= 0 && p->batch >= 1 && p->m >= 1 && p->top_k >= 0 && p->max_pos >= 0,
            CSA_ERR_SHAPE);
  CSA_CHECK(p->heads >= 1 && p->dim >= 1, CSA_ERR_SHAPE);
  CSA_CHECK(p->score_dtype == CSA_F32 || p->score_dtype == CSA_BF16, CSA_ERR_INVALID_ARG);
  if (p->num_queries == 0) return CSA_OK;
  CSA_CHECK(p->q && p->w && p->pos && p->idx && p->cnt, CSA_ERR_INVALID_ARG);
  CSA_CHECK(aligned(p->q, 16) && aligned(p->w, 16) && aligned(p->pos, 4) && aligned(p->idx, 4) &&
                aligned(p->cnt, 4) && (!p->seq || aligned(p->seq, 4)),
            CSA_ERR_ALIGN);
  const int64_t nmax = (int64_t)(p->max_pos + 1) / p->m;
  CSA_CHECK(nmax <= 65535LL * kTile, CSA_ERR_SHAPE);  // key chunks on grid.y
  const int f = p->keys.format;
  if (f == CSA_FMT_DENSE_F32) {
    CSA_CHECK(p->q_dtype == CSA_F32, CSA_ERR_UNSUPPORTED);
    CSA_CHECK(p->keys.dim == p->dim && p->heads * p->dim <= 16384, CSA_ERR_SHAPE);
  } else if (f == CSA_FMT_INDEX_POOL_BF16) {
    CSA_CHECK(p->q_dtype == CSA_BF16, CSA_ERR_UNSUPPORTED);
    CSA_CHECK(p->heads == 64 && p->dim == kIdxDim, CSA_ERR_UNSUPPORTED);
  } else if (f == CSA_FMT_INDEX_POOL_E2M1) {
    CSA_CHECK(p->q_dtype == CSA_F32, CSA_ERR_UNSUPPORTED);
    CSA_CHECK(p->heads == 64 && p->dim == kIdxDim, CSA_ERR_UNSUPPORTED);
  } else {
    return CSA_ERR_UNSUPPORTED;
  }
  CSA_CHECK(p->scores_out == nullptr || (aligned(p->scores_out, 4) && p->score_capacity >= 0), CSA_ERR_ALIGN);
  return check_store(p->keys, p->batch, nmax);
}

}  // namespace

extern "C" size_t csa_index_topk_workspace_size(const csa_index_params* p) {
  if (check_index(p) != CSA_OK) return 0;
  const size_t bytes = p->score_dtype == CSA_BF16 ? 2 : 4;
  return kWsHeader + (size_t)p->num_queries * index_stride(p) * bytes;
}

namespace {

int prepare(const csa_index_params* p, void* ws, size_t ws_bytes) {
  int st = check_index(p);
  if (st != CSA_OK) return st;
  if (p->num_queries == 0) return CSA_OK;
  CSA_CHECK(ws != nullptr && aligned(ws, 1024), ws ? CSA_ERR_ALIGN : CSA_ERR_WORKSPACE);
  CSA_CHECK(ws_bytes >= csa_index_topk_workspace_size(p), CSA_ERR_WORKSPACE);
  return CSA_OK;
}

int launch_score(const csa_index_params* p, void* ws, cudaStream_t s) {
  const bool overlap = (index_flags(p) & (CSA_FLAG_OVERLAP_PREVIOUS | CSA_FLAG_AFTER_APPEND)) != 0;
  int* status = static_cast<int*>(ws);
  void* scores = static_cast<uint8_t*>(ws) + kWsHeader;
  const int stride = index_stride(p);
  const int bf16 = p->score_dtype == CSA_BF16;
  const int T = p->num_queries;
  const int nmax = (p->max_pos + 1) / p->m;
  if (nmax == 0) return CSA_OK;
  const Store keys = to_device(p->keys);
  const int f = p->keys.format;
  if (f == CSA_FMT_DENSE_F32) {
    const size_t smem = (size_t)(p->heads * p->dim + p->heads) * sizeof(float);
    if (smem > 48 * 1024) cudaFuncSetAttribute(score_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    return launch_ex(score_f32_kernel, dim3(T, (nmax + 127) / 128), dim3(128), smem, s, overlap, 1, 1,
                     static_cast<const float*>(p->q), p->w, p->w_shared, p->pos, p->seq, p->batch, p->m,
                     static_cast<const float*>(p->keys.base), p->keys.capacity, p->heads, p->dim, scores, stride,
                     bf16, status);
  } else {
    TcArgs a;
    a.q = p->q;
    a.w = p->w;
    a.w_shared = p->w_shared;
    a.pos = p->pos;
    a.seq = p->seq;
    a.batch = p->batch;
    a.after_append = (index_flags(p) & CSA_FLAG_AFTER_APPEND) != 0;
    a.m = p->m;
    a.T = T;
    a.keys = keys;
    a.scores = scores;
    a.stride = stride;
    a.bf16 = bf16;
    a.status = status;
    const int n_tiles = (nmax + kTile - 1) / kTile;
    if (f == CSA_FMT_INDEX_POOL_BF16 && p->batch == 1 && T >= 4 * sm_count()) {
      // one sequence, many queries (prefill): four queries per CTA share every
      // key tile (N = 256 per MMA)
      a.splits = 1;
      const size_t smem = sizeof(TcSmem<4>) + 1024;
      cudaFuncSetAttribute(score_tc_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      return launch_ex(score_tc_kernel<4>, dim3((T + 3) / 4, 1), dim3(kTcThreads), smem, s, overlap,
                       1, 1, a);
    }
    a.splits = std::max(1, std::min(n_tiles, (2 * sm_count()) / std::max(T, 1)));
    if (f == CSA_FMT_INDEX_POOL_BF16) {
      const size_t smem = sizeof(TcSmem<1>) + 1024;
      cudaFuncSetAttribute(score_tc_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      return launch_ex(score_tc_kernel<1>, dim3(T, a.splits), dim3(kTcThreads), smem, s, overlap, 1,
                       1, a);
    } else {
      // TMA descriptor of the pool's codes: [pages][P slots][64 bytes] with the
      // page stride of the whole page (codes + scales), boxes of 128 slots x 64
      // bytes, 64-byte swizzle (the layout of the MMA's A operand)
      const PFN_cuTensorMapEncodeTiled_v12000 encode = tiled_map_encoder();
      CSA_CHECK(encode != nullptr, CSA_ERR_CUDA);
      CUtensorMap codes_map;
      const int P = p->keys.page_entries;
      const cuuint64_t dims[3] = {(cuuint64_t)(kIdxDim / 2), (cuuint64_t)P, (cuuint64_t)p->keys.num_pages};
      const cuuint64_t strides[2] = {(cuuint64_t)(kIdxDim / 2), (cuuint64_t)page_bytes(f, P)};
      const cuuint32_t box[3] = {kIdxDim / 2, kTile, 1};
      const cuuint32_t estr[3] = {1, 1, 1};
      CSA_CHECK(encode(&codes_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, p->keys.base, dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS,
                CSA_ERR_INVALID_ARG);
      const size_t smem = sizeof(F4Smem) + 1024;
      cudaFuncSetAttribute(score_fp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      return launch_ex(score_fp4_kernel, dim3(T, a.splits), dim3(kF4Threads), smem, s, overlap, 1, 1, a, codes_map);
    }
  }
  return launch_status();
}

// Clusters of cs top-k CTAs (smem bytes of dynamic shared memory each) that
// can be resident on the current device at once (cached per device and
// shape).  A cluster of more than 8 CTAs is non-portable: it is used only
// when every cluster of the launch fits at once.
int topk_resident_clusters(int cs, size_t smem) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, size_t>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_tuple(dev, cs, smem);
  const auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) == cudaSuccess &&
      (cs <= 8 || cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess)) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cs);
    cfg.blockDim = dim3(kTopkThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, topk_kernel, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();  // a refused query is not the launch's error
  cache[key] = n;
  return n;
}

int launch_select(const csa_index_params* p, void* ws, cudaStream_t s) {
  int* status = static_cast<int*>(ws);
  void* scores = static_cast<uint8_t*>(ws) + kWsHeader;
  // CTAs per row: enough to cover the SMs when rows are few (at least 4096
  // scores per CTA), and enough that a row's chunk fits in shared memory;
  // at most kMaxTopkCluster (16 only when those clusters all fit at once)
  const int T = p->num_queries, stride = index_stride(p);
  int cs = 1;
  while (cs < kMaxTopkCluster && (((int64_t)cs * T < sm_count() && (int64_t)cs * 2 * 4096 <= stride) ||
                                  (stride + cs - 1) / cs > kTopkMaxSmemKeys))
    cs *= 2;
  // the two histogram buffers, then the chunk's keys when they fit
  auto smem_keys_for = [&](int c) {
    const int chunk_max = (stride + c - 1) / c;
    return chunk_max <= kTopkMaxSmemKeys ? chunk_max : 0;
  };
  int smem_keys = smem_keys_for(cs);
  size_t smem = (size_t)(2 * kHistBuf + smem_keys) * sizeof(uint32_t);
  if (cs > 8 && topk_resident_clusters(cs, smem) < T) {
    cs = 8;
    smem_keys = smem_keys_for(cs);
    smem = (size_t)(2 * kHistBuf + smem_keys) * sizeof(uint32_t);
  }
  if (cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return CSA_ERR_CUDA;
  // the selector reads nothing before it waits for the previous kernel: it may always start early
  return launch_ex(topk_kernel, dim3((unsigned)(T * cs)), dim3(kTopkThreads), smem, s, true, cs, 1,
                   static_cast<const void*>(scores), (int)(p->score_dtype == CSA_BF16), stride, p->pos, p->m, p->top_k,
                   p->idx, p->cnt, p->scores_out, p->score_capacity, smem_keys, status);
}

}  // namespace

extern "C" int csa_index_score(const csa_index_params* p, void* ws, size_t ws_bytes, csa_stream_t stream) {
  int st = prepare(p, ws, ws_bytes);
  if (st != CSA_OK || p->num_queries == 0) return st;
  return launch_score(p, ws, (cudaStream_t)stream);
}

extern "C" int csa_index_select(const csa_index_params* p, void* ws, size_t ws_bytes, csa_stream_t stream) {
  int st = prepare(p, ws, ws_bytes);
  if (st != CSA_OK || p->num_queries == 0) return st;
  return launch_select(p, ws, (cudaStream_t)stream);
}

extern "C" int csa_index_topk(const csa_index_params* p, void* ws, size_t ws_bytes, csa_stream_t stream) {
  int st = prepare(p, ws, ws_bytes);
  if (st != CSA_OK || p->num_queries == 0) return st;
  st = launch_score(p, ws, (cudaStream_t)stream);
  if (st != CSA_OK) return st;
  return launch_select(p, ws, (cudaStream_t)stream);
}

extern "C" int csa_workspace_status(const void* ws, int32_t* out, csa_stream_t stream) {
  CSA_CHECK(ws != nullptr && out != nullptr, CSA_ERR_INVALID_ARG);
  if (cudaMemcpyAsync(out, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, (cudaStream_t)stream) != cudaSuccess)
    return CSA_ERR_CUDA;
  return cudaStreamSynchronize((cudaStream_t)stream) == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}

extern "C" int csa_workspace_clear_status(void* ws, csa_stream_t stream) {
  CSA_CHECK(ws != nullptr, CSA_ERR_INVALID_ARG);
  return cudaMemsetAsync(ws, 0, sizeof(int32_t), (cudaStream_t)stream) == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}

// ================================================================== no-allocation variant
//
// csa_index_topk_noalloc: the same indexer + top-k as csa_index_topk, with
// its scratch (status word + per-query scores) in a fixed array that lives in
// this library's device memory instead of a caller-provided workspace.  It is
// for callers that are handed their input and output buffers by a host
// framework that owns every device allocation and gives them no way to
// allocate scratch of their own.

#include <mutex>

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB on every device that loads the library
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) uint8_t g_index_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kNoAllocMaxDevices] = {};

// Device address of g_index_scratch on the current device.  Outside a stream
// capture it is looked up on every call (with the device current), so it
// follows a reload of the module after a device reset; during a capture the
// address of the device's last uncaptured call is used (no lookup inside a
// capture).
int scratch_address(cudaStream_t s, void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return CSA_ERR_CUDA;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return CSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_index_scratch) != cudaSuccess || p == nullptr) return CSA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  if (g_scratch_ptr[dev] == nullptr) return CSA_ERR_CUDA;  // first call on this device inside a capture
  *out = g_scratch_ptr[dev];
  return CSA_OK;
}

}  // namespace

extern "C" int csa_index_topk_noalloc(const csa_index_params* p, csa_stream_t stream) {
  int st = check_index(p);
  if (st != CSA_OK) return st;
  if (p->num_queries == 0) return CSA_OK;
  const size_t need = csa_index_topk_workspace_size(p);
  CSA_CHECK(need <= kNoAllocScratchBytes, CSA_ERR_WORKSPACE);
  cudaStream_t s = (cudaStream_t)stream;
  void* ws = nullptr;
  st = scratch_address(s, &ws);
  if (st != CSA_OK) return st;
  // the array keeps the previous call's contents: the status word starts at CSA_OK
  if (cudaMemsetAsync(ws, 0, sizeof(int32_t), s) != cudaSuccess) return CSA_ERR_CUDA;
  st = launch_score(p, ws, s);
  if (st != CSA_OK) return st;
  return launch_select(p, ws, s);
}

extern "C" int csa_index_topk_noalloc_status(int32_t* out, csa_stream_t stream) {
  CSA_CHECK(out != nullptr, CSA_ERR_INVALID_ARG);
  cudaStream_t s = (cudaStream_t)stream;
  // the status word is the first word of the array; the runtime resolves the
  // symbol on the current device
  if (cudaMemcpyFromSymbolAsync(out, g_index_scratch, sizeof(int32_t), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return CSA_ERR_CUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}
