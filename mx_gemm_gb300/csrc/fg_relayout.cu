// HBM-bound helper kernels: the one-time weight relayout (and its inverse),
// the scale-factor relayout for MX weights, and the split-K reduce.
//
// The weight relayout is the preshuffle step of the aiter PR "FlyDSL split-K
// preshuffle decode GEMM for small-M shapes (FP8 + MX, gfx950/gfx942)"
// (Copilot file table: the weight/scale preshuffle helpers).  The pages do
// not give a layout; this one makes each 128-row x 128-byte K slab the exact
// shared-memory image of a 128-byte-swizzled K-major tensor-core operand.
//
// The reduce is that PR's second pass ("fp32 split-K reduction kernel
// (downcast once at final store)"): sum the fp32 partials in split order,
// apply the per-tensor scale, round to bf16 once.
#include <cuda_bf16.h>

#include "fg_internal.cuh"
#include "fg_ptx.cuh"

namespace fg {

namespace {

int grid_for(int64_t work, int threads) {
  int64_t blocks = (work + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 16;
  if (blocks > cap) blocks = cap;
  return static_cast<int>(blocks < 1 ? 1 : blocks);
}

// One thread per 16-byte chunk.  Chunk c (0..7) of row r in slab (nb, kb)
// goes to chunk (c ^ (r % 8)) of image row r of slab nb*KB + kb.
__global__ void relayout_b_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t N, int64_t Kb,
                                  int inverse) {
  const int64_t chunks_per_row = Kb >> 4;
  const int64_t KB = Kb >> 7;
  const int64_t total = N * chunks_per_row;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t n = i / chunks_per_row, cc = i - n * chunks_per_row;
    const int64_t kb = cc >> 3, c = cc & 7, nb = n >> 7, r = n & 127;
    const int64_t img = (((nb * KB + kb) << 7) + r) * 8 + (c ^ (r & 7));
    if (!inverse)
      dst[img] = __ldg(src + i);
    else
      dst[i] = __ldg(src + img);
  }
}

// Packed fp4 weights [N][Kb] <-> blocks of 128 rows x 64 bytes: block
// (nb, u) at index nb*(Kb/64) + u, row r of it at byte r*64 (no swizzle).
// One thread per 16-byte chunk.
__global__ void block64_b_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t N, int64_t Kb,
                                 int inverse) {
  const int64_t cpr = Kb / 16;  // chunks per row
  const int64_t total = N * cpr;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t n = i / cpr, cb = i - n * cpr;
    const int64_t img = ((n >> 7) * (Kb / 64) + (cb >> 2)) * 512 + (n & 127) * 4 + (cb & 3);
    if (!inverse)
      dst[img] = __ldg(src + i);
    else
      dst[i] = __ldg(src + img);
  }
}

// MX weight scales [N][K/blk] (E8M0 bytes) <-> atoms of 512 bytes whose byte
// 16*(r%32) + 4*(r/32) + j belongs to row nb*128 + r.  mxfp4 and the 32-K
// modes: for slab u and atom a of the slab, byte j is the scale of the 32-K
// block (u*APS + a)*4 + j.  mxfp8 (one scale per 128-K slab): four slabs to
// an atom, byte j the scale of slab 4g + j (zero past the last slab).
__global__ void relayout_sf_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int64_t N, int64_t K,
                                   int mode, int inverse) {
  if (mode == kMXFP8) {
    const int64_t KB = K / 128, G = (KB + 3) / 4;
    const int64_t total = (N / 128) * G * 512;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
      const int64_t atom = i >> 9;
      const int off = static_cast<int>(i & 511);
      const int r = (off >> 4) + 32 * ((off & 15) >> 2);
      const int64_t nb = atom / G, u = (atom - nb * G) * 4 + (off & 3);
      const int64_t n = nb * 128 + r;
      if (!inverse)
        dst[i] = u < KB ? __ldg(src + n * KB + u) : uint8_t(0);
      else if (u < KB)
        dst[n * KB + u] = __ldg(src + i);
    }
    return;
  }
  const int aps = mode == kMXFP4 ? 2 : 1;
  const int64_t KB = mode == kMXFP4 ? K / 256 : K / 128;  // slabs per row
  const int64_t sf_cols = mode == kMXFP8 ? K / 128 : K / 32;
  const int64_t total = (N / 128) * KB * aps * 512;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t atom = i >> 9;
    const int off = static_cast<int>(i & 511);
    const int r = (off >> 4) + 32 * ((off & 15) >> 2);
    const int j = off & 3;
    const int64_t nb = atom / (KB * aps);
    const int64_t rem = atom - nb * KB * aps;
    const int64_t q32 = rem * 4 + j;  // (u*aps + a)*4 + j
    const int64_t n = nb * 128 + r;
    const int64_t col = mode == kMXFP8 ? (q32 >> 2) : q32;
    if (!inverse) {
      dst[i] = __ldg(src + n * sf_cols + col);
    } else if (mode != kMXFP8 || j == 0) {
      dst[n * sf_cols + col] = __ldg(src + i);
    }
  }
}

// Activation scales of the MX modes, [rows][K/blk] E8M0 bytes, into the same
// 512-byte atoms as the weight image (mxfp8: four slabs to an atom), per
// 128-row tile of A; rows past the end read as 2^0 (their A values are
// zero-filled by the tile loads).
__global__ void relayout_sf_rows_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int64_t rows,
                                        int64_t K, int mode) {
  if (mode == kMXFP8) {
    const int64_t KB = K / 128, G = (KB + 3) / 4;
    const int64_t total = ((rows + 127) / 128) * G * 512;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
      const int64_t atom = i >> 9;
      const int off = static_cast<int>(i & 511);
      const int r = (off >> 4) + 32 * ((off & 15) >> 2);
      const int64_t mb = atom / G, u = (atom - mb * G) * 4 + (off & 3);
      const int64_t m = mb * 128 + r;
      dst[i] = u >= KB ? uint8_t(0) : (m < rows ? __ldg(src + m * KB + u) : uint8_t(127));
    }
    return;
  }
  const int aps = mode == kMXFP4 ? 2 : 1;
  const int64_t KB = mode == kMXFP4 ? K / 256 : K / 128;
  const int64_t sf_cols = mode == kMXFP8 ? K / 128 : K / 32;
  const int64_t total = ((rows + 127) / 128) * KB * aps * 512;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t atom = i >> 9;
    const int off = static_cast<int>(i & 511);
    const int r = (off >> 4) + 32 * ((off & 15) >> 2);
    const int j = off & 3;
    const int64_t mb = atom / (KB * aps);
    const int64_t q32 = (atom - mb * KB * aps) * 4 + j;
    const int64_t m = mb * 128 + r;
    const int64_t col = mode == kMXFP8 ? (q32 >> 2) : q32;
    dst[i] = m < rows ? __ldg(src + m * sf_cols + col) : uint8_t(127);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Y[i] = bf16_rne(scale * sum_s ws[s][i]) over the flattened M*N outputs,
// four consecutive outputs per thread.  All S partial loads of a thread are
// issued before the first add (S is a template constant), so the kernel
// costs one memory round trip instead of S; the adds then run in split
// order.
template <int S>
__global__ void reduce_kernel(const float4* __restrict__ ws, int64_t mn4, const float* __restrict__ a_s,
                              const float* __restrict__ b_s, uint2* __restrict__ y) {
  pdl_wait();  // the partials come from the kernel before this one
  pdl_launch_dependents();
  const float scale = (a_s != nullptr) ? __ldg(a_s) * __ldg(b_s) : 1.0f;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < mn4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float4 v[S];
#pragma unroll
    for (int s = 0; s < S; ++s) v[s] = __ldcs(ws + s * mn4 + i);
    float4 a = v[0];
#pragma unroll
    for (int s = 1; s < S; ++s) {
      a.x += v[s].x; a.y += v[s].y; a.z += v[s].z; a.w += v[s].w;
    }
    uint2 o;
    o.x = pack_bf16x2(a.x * scale, a.y * scale);
    o.y = pack_bf16x2(a.z * scale, a.w * scale);
    y[i] = o;
  }
}

template <int S>
cudaError_t launch_reduce_s(const float* ws, int64_t mn4, const float* a_s, const float* b_s, __nv_bfloat16* y,
                            cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid_for(mn4, 128));
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, reduce_kernel<S>, reinterpret_cast<const float4*>(ws), mn4, a_s, b_s,
                            reinterpret_cast<uint2*>(y));
}

}  // namespace

cudaError_t launch_relayout_b(const uint8_t* src, uint8_t* dst, int64_t N, int64_t Kb, bool inverse,
                              cudaStream_t stream) {
  const int64_t work = N * (Kb / 16);
  if (work == 0) return cudaSuccess;
  relayout_b_kernel<<<grid_for(work, 256), 256, 0, stream>>>(reinterpret_cast<const uint4*>(src),
                                                             reinterpret_cast<uint4*>(dst), N, Kb, inverse ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_block64_b(const uint8_t* src, uint8_t* dst, int64_t N, int64_t Kb, bool inverse,
                             cudaStream_t stream) {
  const int64_t work = N * (Kb / 16);
  if (work == 0) return cudaSuccess;
  block64_b_kernel<<<grid_for(work, 256), 256, 0, stream>>>(reinterpret_cast<const uint4*>(src),
                                                            reinterpret_cast<uint4*>(dst), N, Kb, inverse ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_relayout_sf(int mode, const uint8_t* src, uint8_t* dst, int64_t N, int64_t K, bool inverse,
                               cudaStream_t stream) {
  const int aps = mode == kMXFP4 ? 2 : 1;
  const int64_t KB = mode == kMXFP4 ? K / 256 : K / 128;
  const int64_t work = mode == kMXFP8 ? (N / 128) * ((KB + 3) / 4) * 512 : (N / 128) * KB * aps * 512;
  if (work == 0) return cudaSuccess;
  relayout_sf_kernel<<<grid_for(work, 256), 256, 0, stream>>>(src, dst, N, K, mode, inverse ? 1 : 0);
  return cudaGetLastError();
}

uint64_t sf_rows_image_bytes(int mode, int64_t rows, int64_t K) {
  const int aps = mode == kMXFP4 ? 2 : 1;
  const int64_t KB = mode == kMXFP4 ? K / 256 : K / 128;
  if (mode == kMXFP8) return static_cast<uint64_t>((rows + 127) / 128) * ((KB + 3) / 4) * 512;
  return static_cast<uint64_t>((rows + 127) / 128) * KB * aps * 512;
}

cudaError_t launch_relayout_sf_rows(int mode, const uint8_t* src, uint8_t* dst, int64_t rows, int64_t K,
                                    cudaStream_t stream) {
  const int64_t work = static_cast<int64_t>(sf_rows_image_bytes(mode, rows, K));
  if (work == 0) return cudaSuccess;
  relayout_sf_rows_kernel<<<grid_for(work, 256), 256, 0, stream>>>(src, dst, rows, K, mode);
  return cudaGetLastError();
}

cudaError_t launch_reduce(const float* ws, int split, int64_t M, int64_t N, const float* a_s, const float* b_s,
                          __nv_bfloat16* y, cudaStream_t stream) {
  const int64_t mn4 = M * N / 4;
  if (mn4 == 0) return cudaSuccess;
  switch (split) {
#define FG_RED(S_) \
  case S_: return launch_reduce_s<S_>(ws, mn4, a_s, b_s, y, stream);
    FG_RED(1) FG_RED(2) FG_RED(3) FG_RED(4) FG_RED(5) FG_RED(6) FG_RED(7) FG_RED(8)
    FG_RED(9) FG_RED(10) FG_RED(11) FG_RED(12) FG_RED(13) FG_RED(14) FG_RED(15) FG_RED(16)
#undef FG_RED
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fg
