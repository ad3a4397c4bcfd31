// fg_gemm_noalloc: the split-K GEMM with its scratch in library-owned device
// memory, for callers that cannot allocate device memory themselves.
//
// Who needs it: a caller whose device memory is fixed once it is running --
// a serving loop that sized every buffer at start-up and must not call
// cudaMalloc later (an allocation can synchronise the device and stall every
// stream), or a plug-in hosted by a framework that owns all device memory and
// hands the plug-in no allocator.  Such a caller can still pass its inputs
// and outputs, but not the fp32 split-K workspace that fg_gemm asks for.
//
// The scratch is one file-scope device array of kScratchBytes; every device
// that loads this library holds it until the process exits.  Host code must
// not use the array's name as an address (on the host it is only a stand-in
// for the symbol), so the first call on each device looks up the device
// address with cudaGetSymbolAddress while that device is current, and later
// calls reuse it.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/fg.h"

namespace fg {
void set_error_message(const char* fmt, ...);
}

namespace {

constexpr unsigned long long kScratchBytes = 8ull << 20;  // 8 MiB

}  // namespace

static __device__ __align__(256) float fg_noalloc_scratch[kScratchBytes / sizeof(float)];

namespace {

// Device address of fg_noalloc_scratch on the current device (set up once per
// device).  Returns nullptr and writes the CUDA error on failure.
void* scratch_address(cudaError_t* err) {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, fg_noalloc_scratch);
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" FG_API fg_status fg_gemm_noalloc(const void* A, const void* a_scales, int64_t M, const fg_bshuf* b,
                                            int mode, int split_k, void* Y, uint32_t flags, void* stream) {
  if (flags & FG_FLAG_DEFER_REDUCE) {
    fg::set_error_message("fg_gemm_noalloc: FG_FLAG_DEFER_REDUCE would leave the partials in the library's "
                          "private scratch; use fg_gemm with a workspace");
    return FG_ERR_INVALID_ARG;
  }
  if (b && b->magic == FG_BSHUF_MAGIC && b->version == FG_BSHUF_VERSION && M > 0) {
    // Only what fg_gemm cannot do without is checked against the scratch:
    // the fp32 partials of a split above the cluster limit, and the A scale
    // image of the large-M MX kernel.  The large-M bf16 / fp8 kernel's
    // stream-K buffer is optional: when it does not fit, fg_gemm runs every
    // tile whole.
    fg_plan plan;
    uint64_t need = 0;
    if (fg_gemm_plan(mode, M, b->N, b->K, split_k, &plan) == FG_OK &&
        fg_gemm_workspace_size(mode, M, b->N, b->K, split_k, &need) == FG_OK) {
      const bool large_mx = plan.path == 1 && mode != FG_BF16 && mode != FG_FP8_TENSOR;
      if (plan.path == 0 && need > kScratchBytes) {
        fg::set_error_message("fg_gemm_noalloc: split_k=%d needs split_k*M*N*4 = %llu bytes of fp32 partials, more "
                              "than the %llu-byte built-in scratch; use a split of at most 8 (no partials in "
                              "memory), a smaller split, or fg_gemm with a caller workspace",
                              plan.split_k, (unsigned long long)need, kScratchBytes);
        return FG_ERR_WORKSPACE;
      }
      if (large_mx && need > kScratchBytes) {
        fg::set_error_message("fg_gemm_noalloc: the large-M MX kernel's A scale image takes %llu bytes for M=%lld, "
                              "more than the %llu-byte built-in scratch; use fg_gemm with a caller workspace",
                              (unsigned long long)need, (long long)M, kScratchBytes);
        return FG_ERR_WORKSPACE;
      }
    }
  }
  cudaError_t e = cudaSuccess;
  void* scratch = scratch_address(&e);
  if (!scratch) {
    fg::set_error_message("fg_gemm_noalloc: scratch address lookup failed: %s", cudaGetErrorString(e));
    return FG_ERR_CUDA;
  }
  // fg_gemm does every other check.  No part of the scratch has to start at
  // zero: each split writes all of its [M][N] partial before the reduce
  // reads it, the A scale image is rewritten whole by every large-M MX call,
  // and a stream-K flag only matches the launch that wrote it.
  return fg_gemm(A, a_scales, M, b, mode, split_k, Y, scratch, kScratchBytes, flags, stream);
}
