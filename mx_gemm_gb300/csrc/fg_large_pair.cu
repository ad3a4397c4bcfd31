// Large-M block-scaled (MX) GEMM on CTA pairs: the compute-bound form of the
// aiter PR "FlyDSL split-K preshuffle decode GEMM for small-M shapes (FP8 +
// MX, gfx950/gfx942)" scale modes at M = 4096 (What's included; Notes: MX
// performance left to later work), written for sm_103a's two-SM tensor-core
// operations (tcgen05 .cta_group::2).
//
// What the pair form changes.  A one-CTA 128 x 256 tile brings 48 KiB into
// its SM per 128-byte K slab (16 KiB of A, 32 KiB of weights).  Two CTAs on
// two SMs computing one 256 x 256 tile with pair MMAs each stage only their
// own 128 rows of A and their own 128-row half of the weights (32 KiB per SM
// per slab): the MMA issued by the even CTA reads A from each CTA's shared
// memory and both weight halves, and writes each CTA's 128 accumulator rows
// into its own tensor memory (256 columns, leaving room for the scale-factor
// ring -- the one-CTA 256 x 256 form has no such room).
//
// Measured on GB300 (M = 4096, N = 16384, K = 7168): the MMA pipe alone
// sustains a slab's four pair MMAs (with their scale copies and commit) in
// 512-640 cycles, yet both forms take about 1000-1300 cycles per slab.  A
// time stamp trace puts the gap on the copies (about 2 us from issue to the
// stage being full), and a copy-only probe shows why: an SM streams distinct
// L2 lines into shared memory at about 60 GB/s (about 9 TB/s over the GPU)
// whatever the copy form, and the pair form's 32 KiB per slab at ~50 GB/s
// per SM meets that bound, while the one-CTA form gets more than it out of
// L2 because the SMs that share a weight slab read it at the same time.  So
// the pair form is 2-6 % slower and is selected only on request.
//
// Roles (320 threads per CTA):
//   warp 0    producer, in both CTAs: per slab, tensor copies of the CTA's A
//             tile, its weight slab (the image is already in the MMA's
//             128-byte-swizzled layout), its A scale atoms and the weight
//             scale atoms; every copy counts its bytes on the even CTA's
//             stage barrier, whose producer arms it for both CTAs;
//   warp 1    both CTAs allocate the pair's tensor memory together; in the
//             even CTA lane 0 copies the stage's scale factors into tensor
//             memory (pair tcgen05.cp: each CTA's shared memory into its own
//             tensor memory), issues the four pair MMAs, and commits the
//             stage back to both CTAs' producers;
//   warps 2-9 epilogue, in both CTAs: each warp pulls its lane quarter x 128
//             columns of the CTA's accumulator rows into registers, tells the
//             even CTA the accumulator may be overwritten, then converts to
//             bf16 and stores.
//
// Every wait is bounded.  After an abort the even CTA makes every stage phase
// that either producer started complete (arming phases only the odd CTA
// started, standing in for the bytes of copies the odd CTA never issued)
// before the pair releases its shared and tensor memory.
#include <atomic>
#include <cuda_bf16.h>

#include "fg_internal.cuh"
#include "fg_ptx.cuh"
#include "fg_tiles.cuh"

namespace fg {

namespace {

constexpr int kThreads = 320;
constexpr int kTileM = 256;      // rows of A per pair tile (128 per CTA)
constexpr int kTileN = 256;      // weight rows per pair tile (128 staged by each CTA)
constexpr int kABytes = 128 * 128;
constexpr int kBBytes = 128 * 128;
constexpr int kTmemCols = 512;

// Each CTA stages the scale atoms of both 128-row halves of the weight tile:
// the pair MMA reads all 256 weight rows' scales from each CTA's tensor memory
// (measured: with only its own half's scales in each CTA the results are
// wrong), while A's scales are per CTA (its own 128 rows).
template <int MODE>
struct PairCfg {
  static constexpr int APS = MODE == kMXFP4 ? 2 : 1;  // atoms per 128-row block per slab
  static constexpr int SFA_BYTES = APS * 512;
  static constexpr int SFB_BYTES = 2 * APS * 512;
  static constexpr int SFA_OFF = kABytes + kBBytes;
  static constexpr int SFB_OFF = SFA_OFF + SFA_BYTES;
  static constexpr int STAGE_RAW = SFB_OFF + SFB_BYTES;
  static constexpr int STAGE_BYTES = (STAGE_RAW + 1023) / 1024 * 1024;
  static constexpr int STAGES = 5;  // room beside the ring for the output staging boxes
  static constexpr int OUT_BYTES = 8 * 32 * 64;  // per epilogue warp: a 32-row x 32-column bf16 staging box
  static constexpr int SMEM = STAGES * STAGE_BYTES + OUT_BYTES + 1024;
  // bytes one weight slab counts: the packed fp4 block of fp8 x fp4, else 16 KiB
  static constexpr int B_TX = MODE == kMXFP4FP8A ? 8192 : kBBytes;
  // mxfp8: one atom holds four slabs' scales (copied at the first slab of each
  // group of four, into a ring of four group buffers); the other modes copy
  // every slab's atoms into a per-stage ring
  static constexpr bool GROUP4 = MODE == kMXFP8;
  static constexpr int SF_COLS = APS * 4 + 2 * APS * 4;
  static constexpr int SF_BUFS = GROUP4 ? 4 : STAGES;
  __host__ __device__ static constexpr uint32_t cta_tx(bool sf_here) {
    return static_cast<uint32_t>(kABytes + B_TX + (sf_here ? SFA_BYTES + SFB_BYTES : 0));
  }
  static_assert(SMEM + 1024 <= 232448, "shared memory budget (with the static barriers)");
  static_assert(256 + SF_BUFS * SF_COLS <= kTmemCols, "TMEM budget");
};

// First 512-byte atom of 128-row block r at slab kb in a scale image (the
// image's rows are atoms): GROUP4 images hold one atom per four slabs.
template <typename C>
__device__ __forceinline__ int sf_row(int r, int kb, int KB) {
  const int G = (KB + 3) / 4;
  return C::GROUP4 ? r * G + kb / 4 : (r * KB + kb) * C::APS;
}

// tmap_b: the weight image as 2 KiB rows of 8-byte elements (box: one 16 KiB
// slab, 8 rows), or for fp8 x fp4 the packed fp4 blocks as 4-bit codes (box:
// one block, spread); tmap_asf / tmap_bsf: the A and weight scale images as
// 512-byte atoms (box: the atoms of one 128-row block and slab).
template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    large_mx_pair_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                         const __grid_constant__ CUtensorMap tmap_asf, const __grid_constant__ CUtensorMap tmap_bsf,
                         const __grid_constant__ CUtensorMap tmap_y, const LargeParams p) {
  using C = PairCfg<MODE>;
  extern __shared__ uint8_t dsmem[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[C::STAGES];   // even CTA: both CTAs' copies of a stage landed
  __shared__ __align__(8) uint64_t empty_bar[C::STAGES];  // both: the stage's MMAs are done
  __shared__ __align__(8) uint64_t accf_bar, acce_bar, stall_bar, drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh, issued_sh, consumed_sh, mma_any_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the pair's MMAs
  const int pair = static_cast<int>(blockIdx.x >> 1), npairs = static_cast<int>(gridDim.x >> 1);
  const int tiles = p.tiles_m * p.tiles_n;
  const int KB = p.KB;
  const uint64_t T = p.timeout_ns;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    mbar_init(&accf_bar, 1);
    mbar_init(&acce_bar, 16);  // the eight epilogue warps of each CTA
    mbar_init(&stall_bar, 1);
    mbar_init(&drain_bar, 1);
    abort_sh = 0;
    issued_sh = 0;
    consumed_sh = 0;
    mma_any_sh = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(&tmem_base_sh, kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
    prefetch_tmap(&tmap_asf);
    prefetch_tmap(&tmap_bsf);
  }
  tc_fence_before();
  __syncthreads();
  // both CTAs' barriers exist before either CTA's copies or commits reach them
  cluster_arrive();
  cluster_wait();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int t = pair; ok && t < tiles; t += npairs) {
        const TileCoord tc = tile_coord(t, p.tiles_m, p.tiles_n, p.group_n);
        const int a128 = 2 * tc.m + static_cast<int>(rank);  // this CTA's 128-row block of A
        const int n128 = 2 * tc.n + static_cast<int>(rank);  // its half of the weight tile
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int slot = it % C::STAGES;
          if (!mbar_wait(&empty_bar[slot], ((it / C::STAGES) & 1) ^ 1u, T, p.err, 41)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + slot * C::STAGE_BYTES;
          const bool sf_here = !C::GROUP4 || (kb & 3) == 0;
          const uint32_t fb = mapa_u32(&full_bar[slot], 0);
          if (rank == 0) mbar_arrive_expect_tx(&full_bar[slot], 2 * C::cta_tx(sf_here));
          // rows of A past M, a weight half past N and their scale atoms read
          // as zeros (whole boxes are counted either way)
          tma_load_2d_pair(st, &tmap_a, kb * 128, a128 * 128, fb);
          if (MODE == kMXFP4FP8A)
            tma_load_3d_pair(st + kABytes, &tmap_b, 0, 0, n128 * KB + kb, fb);
          else
            tma_load_2d_pair(st + kABytes, &tmap_b, 0, (n128 * KB + kb) * 8, fb);
          if (sf_here) {
            tma_load_2d_pair(st + C::SFA_OFF, &tmap_asf, 0, sf_row<C>(a128, kb, KB), fb);
            tma_load_2d_pair(st + C::SFB_OFF, &tmap_bsf, 0, sf_row<C>(2 * tc.n, kb, KB), fb);
            tma_load_2d_pair(st + C::SFB_OFF + C::APS * 512, &tmap_bsf, 0, sf_row<C>(2 * tc.n + 1, kb, KB), fb);
          }
        }
      }
      issued_sh = it;
      if (!ok) abort_sh = 1;
    }
  } else if (warp == 1) {
    // -------------------------------------------- MMA issuer (even CTA only)
    if (rank == 0 && lane == 0) {
      bool ok = true;
      if (p.debug_stall) ok = mbar_wait(&stall_bar, 0, T, p.err, 42);
      int it = 0, ti = 0, gc = 0;  // gc: scale groups copied so far (mxfp8)
      for (int t = pair; ok && t < tiles; t += npairs, ++ti) {
        if (!mbar_wait(&acce_bar, (ti & 1) ^ 1u, T, p.err, 43)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < KB; ++kb) {
          const int slot = it % C::STAGES;
          if (!mbar_wait(&full_bar[slot], (it / C::STAGES) & 1, T, p.err, 44)) {
            ok = false;
            break;
          }
          ++it;  // this stage's copies have all landed
          tc_fence_after();
          mma_any_sh = 1;
          uint8_t* st = smem + slot * C::STAGE_BYTES;
          const bool sf_here = !C::GROUP4 || (kb & 3) == 0;
          if (C::GROUP4 && sf_here) ++gc;
          const uint32_t sfa = 256 + (C::GROUP4 ? ((gc - 1) & 3) : slot) * C::SF_COLS;
          const uint32_t sfb = sfa + C::APS * 4;
          if (sf_here) {
#pragma unroll
            for (int g = 0; g < C::APS; ++g) {
              tc_cp_pair_32x128b_warpx4(tmem + sfa + 4 * g, sdesc_plain_rows16(smem_u32(st + C::SFA_OFF + 512 * g)));
              // weight rows 0-127 of the tile at columns +0..3, rows 128-255 at +4..7
              tc_cp_pair_32x128b_warpx4(tmem + sfb + 8 * g, sdesc_plain_rows16(smem_u32(st + C::SFB_OFF + 512 * g)));
              tc_cp_pair_32x128b_warpx4(tmem + sfb + 8 * g + 4,
                                        sdesc_plain_rows16(smem_u32(st + C::SFB_OFF + C::APS * 512 + 512 * g)));
            }
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint64_t adesc = sdesc_sw128(smem_u32(st + j * 32));
            const uint64_t bdesc = sdesc_sw128(smem_u32(st + kABytes + j * 32));
            const uint32_t acc = (kb | j) != 0;
            if (MODE == kMXFP8) {  // byte kb % 4 of the group's atoms
              mma_mxf8f6f4_pair(tmem, adesc, bdesc, idesc_mx(kTileM, kTileN, kF8f6f4E4M3, kb & 3, kb & 3),
                                tmem + sfa, tmem + sfb, acc);
            } else if (MODE == kMXFP8B32) {
              mma_mxf8f6f4_pair(tmem, adesc, bdesc, idesc_mx(kTileM, kTileN, kF8f6f4E4M3, j, j), tmem + sfa,
                                tmem + sfb, acc);
            } else if (MODE == kMXFP4FP8A) {
              mma_mxf8f6f4_pair(tmem, adesc, bdesc, idesc_mx_ab(kTileM, kTileN, kF8f6f4E4M3, kF8f6f4E2M1, j, j),
                                tmem + sfa, tmem + sfb, acc);
            } else {
              const int g = j >> 1, id = 2 * (j & 1);
              mma_mxf4_pair(tmem, adesc, bdesc, idesc_mx(kTileM, kTileN, kMxf4E2M1, id, id), tmem + sfa + 4 * g,
                            tmem + sfb + 8 * g, acc);
            }
          }
          tc_commit_pair_mc(&empty_bar[slot], 3);  // the stage is free again in both CTAs
        }
        if (!ok) break;
        tc_commit_pair_mc(&accf_bar, 3);  // both CTAs' accumulator rows are complete
      }
      consumed_sh = it;
      if (!ok) abort_sh = 1;
      if (mma_any_sh) {
        // every MMA, copy and commit issued has landed before teardown
        tc_commit_pair_mc(&drain_bar, 1);
        mbar_wait(&drain_bar, 0, T, p.err, 45);
      }
    }
  } else {
    // ------------------------------------- epilogue (eight warps, both CTAs)
    // lane quarter warp % 4 (the tensor-memory lanes this warp may read),
    // column half (warp - 2) / 4 of the 256 accumulator columns
    const int qd = warp & 3;
    const int half = (warp - 2) >> 2;
    // this warp's 32-row x 32-column bf16 staging box (64-byte swizzle)
    uint8_t* stg = smem + C::STAGES * C::STAGE_BYTES + (warp - 2) * (32 * 64);
    int ti = 0;
    for (int t = pair; t < tiles; t += npairs, ++ti) {
      const bool w = mbar_wait(&accf_bar, ti & 1, T, p.err, 46);
      if (!__all_sync(0xffffffffu, w)) {
        if (lane == 0) abort_sh = 1;
        break;
      }
      tc_fence_after();
      uint32_t v[128];
      const uint32_t taddr = tmem + half * 128 + (static_cast<uint32_t>(qd * 32) << 16);
      tmem_ld32(taddr + 0, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
      tmem_ld32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
      tmem_ld32(taddr + 64, *reinterpret_cast<uint32_t(*)[32]>(&v[64]));
      tmem_ld32(taddr + 96, *reinterpret_cast<uint32_t(*)[32]>(&v[96]));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(&acce_bar, 0);  // the pair's next tile may overwrite the accumulator
      const TileCoord tc = tile_coord(t, p.tiles_m, p.tiles_n, p.group_n);
      const int row0 = tc.m * kTileM + static_cast<int>(rank) * 128 + qd * 32;
      const int col0 = tc.n * kTileN + half * 128;
      if (col0 < p.N) {
        // bf16 out through the staging box, 32 columns at a time, by tensor
        // store (rows past M are not written)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          if (lane == 0) bulk_wait_group_read0();  // the previous store has read the box
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int q = 4 * r + j;
            uint4 o;
            o.x = pack_bf16x2(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1]));
            o.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3]));
            o.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5]));
            o.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]));
            // 64-byte rows, 16-byte chunk j at j ^ (row / 2 % 4)
            *reinterpret_cast<uint4*>(stg + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) = o;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmap_y, stg, (col0 + 32 * r) * 2, row0);
            bulk_commit_group();
          }
        }
      }
    }
    if (lane == 0) bulk_wait_group0();  // every store has landed
  }

  // ------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  cluster_arrive();  // both CTAs have stopped issuing; their counters are visible across the pair
  cluster_wait();
  if (rank == 0 && threadIdx.x == 0) {
    const int peer_abort = static_cast<int>(ld_cluster_u32(mapa_u32(&abort_sh, 1)));
    if (abort_sh || peer_abort) {
      // Every stage phase either producer started must complete before the
      // pair's shared memory goes away: those copies count on these barriers.
      const int L = issued_sh;
      const int P = static_cast<int>(ld_cluster_u32(mapa_u32(&issued_sh, 1)));
      const int hi = L > P ? L : P;
      for (int it = consumed_sh; it < hi; ++it) {
        const int slot = it % C::STAGES;
        const uint32_t tx = C::cta_tx(!C::GROUP4 || ((it % KB) & 3) == 0);
        if (it >= L)
          mbar_arrive_expect_tx(&full_bar[slot], tx);  // only the odd CTA issued this stage: arm it for its bytes
        else if (it >= P)
          mbar_complete_tx(&full_bar[slot], tx);  // the odd CTA never issued its half of this stage
        mbar_wait(&full_bar[slot], (it / C::STAGES) & 1, T, nullptr, 0);
      }
    }
  }
  __syncthreads();
  cluster_arrive();  // nothing is in flight towards either CTA any more
  cluster_wait();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, kTmemCols);
}

template <int MODE>
cudaError_t launch_pair(const CUtensorMap& tmap_a, const CUtensorMap& tmap_b, const CUtensorMap& tmap_asf,
                        const CUtensorMap& tmap_bsf, const CUtensorMap& tmap_y, const LargeParams& p, int ctas,
                        cudaStream_t stream) {
  using C = PairCfg<MODE>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(&large_mx_pair_kernel<MODE>), C::SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, large_mx_pair_kernel<MODE>, tmap_a, tmap_b, tmap_asf, tmap_bsf, tmap_y, p);
}

}  // namespace

int pair_max_clusters() {
  static std::atomic<int> cached[64];  // per device, computed once (threads may race to the same value)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (const int c = cached[dev].load(std::memory_order_relaxed)) return c;
  using C = PairCfg<kMXFP4>;  // the largest shared-memory footprint of the pair kernels
  if (ensure_smem_attr(reinterpret_cast<const void*>(&large_mx_pair_kernel<kMXFP4>), C::SMEM) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 256);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void*>(&large_mx_pair_kernel<kMXFP4>), &cfg) !=
          cudaSuccess ||
      n <= 0)
    return 0;
  cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

uint32_t pair_sf_box_rows(int mode) { return mode == kMXFP4 ? 2u : 1u; }

cudaError_t launch_large_pair(int mode, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                              const CUtensorMap& tmap_asf, const CUtensorMap& tmap_bsf, const CUtensorMap& tmap_y,
                              const LargeParams& p, int ctas, cudaStream_t stream) {
  switch (mode) {
    case kMXFP8: return launch_pair<kMXFP8>(tmap_a, tmap_b, tmap_asf, tmap_bsf, tmap_y, p, ctas, stream);
    case kMXFP8B32: return launch_pair<kMXFP8B32>(tmap_a, tmap_b, tmap_asf, tmap_bsf, tmap_y, p, ctas, stream);
    case kMXFP4: return launch_pair<kMXFP4>(tmap_a, tmap_b, tmap_asf, tmap_bsf, tmap_y, p, ctas, stream);
    case kMXFP4FP8A: return launch_pair<kMXFP4FP8A>(tmap_a, tmap_b, tmap_asf, tmap_bsf, tmap_y, p, ctas, stream);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace fg
