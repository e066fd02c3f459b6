// Version and status strings of the C ABI (include/csa.h).
#include "common.cuh"
#include "host.hpp"

extern "C" int csa_abi_version(void) { return CSA_ABI_VERSION; }

extern "C" const char* csa_status_string(int status) {
  switch (status) {
    case CSA_OK: return "ok";
    case CSA_ERR_INVALID_ARG: return "invalid argument";
    case CSA_ERR_SHAPE: return "inconsistent or unsupported sizes";
    case CSA_ERR_ALIGN: return "misaligned pointer";
    case CSA_ERR_UNSUPPORTED: return "unsupported dtype/shape combination";
    case CSA_ERR_WORKSPACE: return "workspace missing or too small";
    case CSA_ERR_CUDA: return "CUDA runtime error";
    case CSA_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

extern "C" const char* csa_last_cuda_error(void) {
  return cudaGetErrorString(csa::last_cuda_error());
}
