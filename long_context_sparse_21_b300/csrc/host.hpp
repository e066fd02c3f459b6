// Host-side helpers shared by the C-ABI entry points: argument checks that run
// before any launch, and the conversion of csa_store into the device struct.
#pragma once

#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <cmath>

#include "common.cuh"

namespace csa {

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

#define CSA_CHECK(cond, code) \
  do {                        \
    if (!(cond)) return (code); \
  } while (0)

// The CUDA error behind the calling thread's last CSA_ERR_CUDA (the status
// enum only says that one happened).
inline cudaError_t& last_cuda_error() {
  static thread_local cudaError_t e = cudaSuccess;
  return e;
}
inline int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return CSA_OK;
  last_cuda_error() = e;
  return CSA_ERR_CUDA;
}

inline int launch_status() { return cuda_status(cudaGetLastError()); }

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (nullptr when the driver does not provide it).
inline PFN_cuTensorMapEncodeTiled_v12000 tiled_map_encoder() {
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

inline bool is_pool(int f) {
  return f == CSA_FMT_KV_POOL_FP8 || f == CSA_FMT_INDEX_POOL_BF16 || f == CSA_FMT_INDEX_POOL_E2M1;
}

// Validates a store for `batch` sequences that must hold entries [0, need).
inline int check_store(const csa_store& s, int batch, int64_t need) {
  CSA_CHECK(s.base != nullptr, CSA_ERR_INVALID_ARG);
  switch (s.format) {
    case CSA_FMT_DENSE_F32:
    case CSA_FMT_DENSE_BF16:
      CSA_CHECK(aligned(s.base, 16), CSA_ERR_ALIGN);
      CSA_CHECK(s.dim > 0 && s.capacity >= 0, CSA_ERR_SHAPE);
      CSA_CHECK(need <= s.capacity, CSA_ERR_SHAPE);
      return CSA_OK;
    case CSA_FMT_KV_POOL_FP8:
      CSA_CHECK(s.dim == kKvDim, CSA_ERR_UNSUPPORTED);
      break;
    case CSA_FMT_INDEX_POOL_BF16:
    case CSA_FMT_INDEX_POOL_E2M1:
      CSA_CHECK(s.dim == kIdxDim, CSA_ERR_UNSUPPORTED);
      break;
    default:
      return CSA_ERR_INVALID_ARG;
  }
  CSA_CHECK(aligned(s.base, 1024), CSA_ERR_ALIGN);
  CSA_CHECK(s.page_table != nullptr && aligned(s.page_table, 4), CSA_ERR_INVALID_ARG);
  CSA_CHECK(s.page_entries > 0 && s.page_entries % kTile == 0, CSA_ERR_SHAPE);
  CSA_CHECK(s.max_pages > 0 && s.num_pages > 0, CSA_ERR_SHAPE);
  CSA_CHECK(need <= (int64_t)s.max_pages * s.page_entries, CSA_ERR_SHAPE);
  (void)batch;
  return CSA_OK;
}

inline Store to_device(const csa_store& s) {
  Store d;
  d.format = s.format;
  d.dim = s.dim;
  d.base = static_cast<uint8_t*>(s.base);
  d.capacity = s.capacity;
  d.page_entries = s.page_entries;
  d.page_table = s.page_table;
  d.max_pages = s.max_pages;
  d.num_pages = s.num_pages;
  return d;
}

// Launches `kernel` on `s` with cudaLaunchKernelEx: optionally with
// programmatic stream serialization (the kernel may start while the previous
// kernel of the stream finishes; it must call pdl_wait() before reading that
// kernel's results) and a thread-block cluster of (cx, cy, 1) CTAs.
// Every kernel of the library asks for the largest shared-memory carveout, so
// an SM keeps one configuration across the kernels of a step: a kernel whose
// CTAs need a larger carveout than the SM's current one can only start there
// once the SM has drained (a kernel with little shared memory before one with
// much would otherwise delay its CTAs by the whole of the first kernel).  Set
// once per kernel and device.
template <typename K>
inline void prefer_max_shared(K kernel) {
  static std::atomic<uint64_t> done{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return;
  const uint64_t bit = 1ull << dev;
  if (done.load(std::memory_order_relaxed) & bit) return;
  cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  cudaGetLastError();
  done.fetch_or(bit);
}

template <typename... KArgs, typename... Args>
inline int launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                     int cx, int cy, Args... args) {
  prefer_max_shared(kernel);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cx * cy > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cx;
    attr[n].val.clusterDim.y = cy;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
  if (e != cudaSuccess) {
    cudaGetLastError();  // a launch-configuration error is not sticky: clear it
    return cuda_status(e);
  }
  return launch_status();
}

// Rotary frequencies base^(-2i / 64) in double precision.
inline RopeFreq rope_freq(double base) {
  RopeFreq r;
  for (int i = 0; i < kRopePairs; ++i) r.f[i] = base > 0.0 ? std::pow(base, -2.0 * i / kRopeDims) : 0.0;
  return r;
}

// SMs of the current device (queried per call: the library caches nothing).
inline int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}

}  // namespace csa
