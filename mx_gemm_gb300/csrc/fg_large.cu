// Large-M preshuffled-weight GEMM for sm_103a: the compute-bound form of the
// FlyDSL PR "Enable the gmem->LDS async copy for f16/bf16 preshuffle GEMM"
// (Performance: bf16 M=54560, N=K=8192) and of the fp8 shape in the FlyDSL PR
// "Migrate kernels to fx.copy / .llvm_ptr" (Validation: M=N=4096, K=8192).
//
// Persistent kernel, one CTA per SM, 128 x 256 output tiles (A rows on the
// MMA M side, two 128-row weight slabs on the N side).  Per 128-byte K slab
// the producer issues one TMA load of the A tile (128 rows x 128 bytes,
// 128-byte swizzle, rows past M read as zero) and one bulk copy per weight
// slab (16 KiB each, already in the swizzled image layout), into a 4-stage
// ring.  The MMA thread issues four tcgen05.mma (128 x 256 x 32 bytes of K)
// per slab into one of two TMEM accumulators (256 fp32 columns each), so the
// four epilogue warps can drain tile t (TMEM -> registers -> scale -> bf16 ->
// global) while tile t+1 accumulates -- the issue-rate lesson of the FlyDSL
// pages (A-fragment reads interleaved with the MMAs, async copies instead of
// register round trips) in tcgen05 form.
//
// Tile order: tiles are walked in groups of `group_n` weight tiles; inside a
// group the weight tile index runs fastest, so the CTAs resident at one time
// share a band of weights (kept in L2) and a few A row blocks.
//
// Stream-K tail (bf16 / fp8, when the caller gives the workspace): when the
// tile count is not a multiple of the CTA count, the last partial wave would
// leave most SMs idle.  Instead each CTA takes its whole tiles for all but
// the last full wave, then an equal contiguous range of the remaining K
// iterations; a tile split between CTAs c and c+1 is finished by c after c+1
// published its fp32 partial (cooperative launch, bounded waits).
#include <cuda_bf16.h>

#include "fg_internal.cuh"
#include "fg_ptx.cuh"
#include "fg_tiles.cuh"

namespace fg {

namespace {

constexpr int kThreads = 192;
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kStages = 4;
constexpr int kABytes = kBM * 128;        // 16 KiB
constexpr int kBBytes = kBN * 128;        // 32 KiB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kSmem = kStages * kStageBytes + 1024;
// the 128 x 256 bf16 / fp8 form: + a 32-row x 32-column bf16 staging box per epilogue warp
constexpr int kSmemOut = kSmem + 4 * 32 * 64;
constexpr int kTmemCols = 512;            // two 256-column accumulators
static_assert(kSmem <= 232448, "shared memory budget");

// One unit of a CTA's work: K iterations [k0, k1) of tile t.
struct Chunk {
  int t, k0, k1;
};

__device__ __forceinline__ int chunk_count(const LargeParams& p, int c, int G, int tiles, int KB) {
  if (p.sk_iters == 0) return c < tiles ? (tiles - c + G - 1) / G : 0;
  const long long s = p.sk_iters * c / G, e = p.sk_iters * (c + 1) / G;
  return p.dp_rounds + (e > s ? static_cast<int>((e - 1) / KB - s / KB + 1) : 0);
}

__device__ __forceinline__ Chunk chunk_at(const LargeParams& p, int c, int G, int KB, int i) {
  Chunk ch;
  if (p.sk_iters == 0 || i < p.dp_rounds) {
    ch.t = c + i * G;
    ch.k0 = 0;
    ch.k1 = KB;
    return ch;
  }
  const long long s = p.sk_iters * c / G, e = p.sk_iters * (c + 1) / G;
  const int j = i - p.dp_rounds;
  const long long tf = s / KB + j;
  ch.t = p.dp_tiles + static_cast<int>(tf);
  ch.k0 = j == 0 ? static_cast<int>(s - tf * KB) : 0;
  ch.k1 = static_cast<int>(e - tf * KB < KB ? e - tf * KB : KB);
  return ch;
}

template <int MODE>
// tmap_y: Y as rows of 2N bytes, boxes of 32 rows x 64 bytes (64-byte
// swizzle): the bf16 tiles leave by tensor store.
__global__ void __launch_bounds__(kThreads, 1)
    large_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_y,
                 const LargeParams p) {
  extern __shared__ uint8_t dsmem[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t accf_bar[2];
  __shared__ __align__(8) uint64_t acce_bar[2];
  __shared__ __align__(8) uint64_t stall_bar, drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh, issued_sh, consumed_sh, mma_any_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles = p.tiles_m * p.tiles_n;
  const int KB = p.KB;
  const uint64_t T = p.timeout_ns;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&accf_bar[i], 1);
      mbar_init(&acce_bar[i], 4);
    }
    mbar_init(&stall_bar, 1);
    mbar_init(&drain_bar, 1);
    abort_sh = 0;
    issued_sh = 0;
    consumed_sh = 0;
    mma_any_sh = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) prefetch_tmap(&tmap_a);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      const int nch = chunk_count(p, blockIdx.x, gridDim.x, tiles, KB);
      for (int ci = 0; ok && ci < nch; ++ci) {
        const Chunk ch = chunk_at(p, blockIdx.x, gridDim.x, KB, ci);
        const TileCoord tc = tile_coord(ch.t, p.tiles_m, p.tiles_n, p.group_n);
        const int nslabs_n = min(2, p.N / 128 - 2 * tc.n);  // weight slabs in this tile (1 or 2)
        for (int kb = ch.k0; kb < ch.k1; ++kb, ++it) {
          const int slot = it % kStages;
          if (!mbar_wait(&empty_bar[slot], ((it / kStages) & 1) ^ 1u, T, p.err, 11)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + slot * kStageBytes;
          mbar_arrive_expect_tx(&full_bar[slot], kABytes + nslabs_n * 16384);
          tma_load_2d(st, &tmap_a, kb * 128, tc.m * kBM, &full_bar[slot]);
          for (int h = 0; h < nslabs_n; ++h)
            bulk_g2s(st + kABytes + h * 16384,
                     p.b_img + (static_cast<size_t>(2 * tc.n + h) * KB + kb) * 16384, 16384, &full_bar[slot]);
        }
      }
      issued_sh = it;
      if (!ok) abort_sh = 1;
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      bool ok = true;
      if (p.debug_stall) ok = mbar_wait(&stall_bar, 0, T, p.err, 12);
      int it = 0, ti = 0;
      const uint32_t idesc = MODE == kBF16 ? idesc_bf16(kBM, kBN) : idesc_e4m3(kBM, kBN);
      const int nch = chunk_count(p, blockIdx.x, gridDim.x, tiles, KB);
      for (; ok && ti < nch; ++ti) {
        const Chunk ch = chunk_at(p, blockIdx.x, gridDim.x, KB, ti);
        const int acc = ti & 1;
        if (!mbar_wait(&acce_bar[acc], ((ti >> 1) & 1) ^ 1u, T, p.err, 13)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + acc * kBN;
        for (int kb = ch.k0; kb < ch.k1; ++kb, ++it) {
          const int slot = it % kStages;
          if (!mbar_wait(&full_bar[slot], (it / kStages) & 1, T, p.err, 14)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_any_sh = 1;
          uint8_t* st = smem + slot * kStageBytes;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint64_t adesc = sdesc_sw128(smem_u32(st + j * 32));
            const uint64_t bdesc = sdesc_sw128(smem_u32(st + kABytes + j * 32));
            const uint32_t accum = (kb > ch.k0 || j > 0) ? 1u : 0u;
            if (MODE == kBF16)
              mma_f16(d, adesc, bdesc, idesc, accum);
            else
              mma_f8f6f4(d, adesc, bdesc, idesc, accum);
          }
          tc_commit(&empty_bar[slot]);
        }
        if (!ok) {
          ++it;
          break;
        }
        tc_commit(&accf_bar[acc]);
      }
      consumed_sh = it;
      if (!ok) abort_sh = 1;
      if (mma_any_sh) {
        tc_commit(&drain_bar);
        mbar_wait(&drain_bar, 0, T, p.err, 15);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int qd = warp & 3;
    float scale = 1.f;
    if (MODE == kTensor) scale = __ldg(static_cast<const float*>(p.a_scales)) * __ldg(p.b_s);
    // this warp's 32-row x 32-column bf16 staging box (64-byte swizzle)
    uint8_t* stg = smem + kStages * kStageBytes + (warp - 2) * (32 * 64);
    const int nch = chunk_count(p, blockIdx.x, gridDim.x, tiles, KB);
    for (int ti = 0; ti < nch; ++ti) {
      const Chunk ch = chunk_at(p, blockIdx.x, gridDim.x, KB, ti);
      const int acc = ti & 1;
      const bool w = mbar_wait(&accf_bar[acc], (ti >> 1) & 1, T, p.err, 16);
      if (!__all_sync(0xffffffffu, w)) {
        if (lane == 0) abort_sh = 1;
        break;
      }
      tc_fence_after();
      const TileCoord tc = tile_coord(ch.t, p.tiles_m, p.tiles_n, p.group_n);
      const int lrow = qd * 32 + lane;
      const int row = tc.m * kBM + lrow;
      const int ncols = min(kBN, p.N - tc.n * kBN);
      const uint32_t taddr = tmem + acc * kBN + (static_cast<uint32_t>(qd * 32) << 16);
      if (ch.k0 > 0) {
        // Stream-K: this CTA holds the last iterations of the tile; publish
        // the raw fp32 partial ([column][row], this warp's 32 rows) for the
        // CTA that finishes the tile.
        float* part = p.sk_part + static_cast<size_t>(blockIdx.x) * kBN * kBM;
        for (int c = 0; c < kBN; c += 32) {
          uint32_t v[32];
          tmem_ld32(taddr + c, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) __stcg(part + (c + i) * kBM + lrow, __uint_as_float(v[i]));
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release_u64(p.sk_flag + blockIdx.x * 4 + qd, p.epoch);
      } else {
        const bool finish = ch.k1 < KB;  // the rest of the tile comes from CTA blockIdx.x + 1
        const float* peer = p.sk_part + static_cast<size_t>(blockIdx.x + 1) * kBN * kBM;
        bool have_peer = true;
        if (finish) {
          bool fw = true;
          if (lane == 0) fw = wait_flag_eq(p.sk_flag + (blockIdx.x + 1) * 4 + qd, p.epoch, T, p.err, 17);
          have_peer = __shfl_sync(0xffffffffu, fw ? 1 : 0, 0) != 0;
          if (have_peer) (void)ld_acquire_u64(p.sk_flag + (blockIdx.x + 1) * 4 + qd);
          else if (lane == 0) abort_sh = 1;
        }
        for (int c = 0; c < ncols; c += 32) {
          uint32_t v[32];
          tmem_ld32(taddr + c, v);
          tmem_wait_ld();
          float f[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(v[i]);
          if (finish && have_peer) {
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] += __ldcg(peer + (c + i) * kBM + lrow);
          }
          if (have_peer) {
            // bf16 out through the staging box by tensor store (rows past M
            // are not written)
            if (lane == 0) bulk_wait_group_read0();  // the previous store has read the box
            __syncwarp();
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 o;
              o.x = pack_bf16x2(f[8 * q + 0] * scale, f[8 * q + 1] * scale);
              o.y = pack_bf16x2(f[8 * q + 2] * scale, f[8 * q + 3] * scale);
              o.z = pack_bf16x2(f[8 * q + 4] * scale, f[8 * q + 5] * scale);
              o.w = pack_bf16x2(f[8 * q + 6] * scale, f[8 * q + 7] * scale);
              // 64-byte rows, 16-byte chunk q at q ^ (row / 2 % 4)
              *reinterpret_cast<uint4*>(stg + lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4)) = o;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmap_y, stg, (tc.n * kBN + c) * 2, tc.m * kBM + qd * 32);
              bulk_commit_group();
            }
          }
        }
        if (finish && have_peer) {
          // consumed: clear the flag, so that a replay of this launch (same
          // epoch, e.g. in a CUDA graph) waits for the partial it writes
          __syncwarp();
          if (lane == 0) p.sk_flag[(blockIdx.x + 1) * 4 + qd] = 0;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce_bar[acc]);
    }
    if (lane == 0) bulk_wait_group0();  // every store has landed
  }

  // ------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (abort_sh && threadIdx.x == 0) {
    for (int it = consumed_sh; it < issued_sh; ++it)
      mbar_wait(&full_bar[it % kStages], (it / kStages) & 1, T, nullptr, 0);
  }
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <int MODE>
cudaError_t launch_mode(const CUtensorMap& tmap_a, const CUtensorMap& tmap_y, const LargeParams& p, int ctas,
                        cudaStream_t stream) {
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(&large_kernel<MODE>), kSmemOut);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemOut;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeCooperative;  // stream-K CTAs wait on one another: all must be resident
  attr.val.cooperative = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = p.sk_iters > 0 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, large_kernel<MODE>, tmap_a, tmap_y, p);
}


// ---------------------------------------------------------- 256 x 256 form
//
// bf16 / fp8 per-tensor with 256 x 256 output tiles: per 128-byte K slab the
// stage holds both 128-row halves of A (two TMA boxes) and both weight slabs,
// and the MMA thread issues the four MMAs of each half against the same
// weight slabs in shared memory.  Per 128 x 256 of output a stage then moves
// 80 KiB through shared memory (TMA writes + MMA operand reads) instead of the
// 96 KiB of the 128 x 256 tile -- the port that bounds the 128 x 256 kernel.
// The two halves' accumulators fill TMEM (2 x 256 columns), so there is no
// second accumulator to overlap the epilogue with: eight epilogue warps pull
// half 0 into registers and release it (the next tile's half-0 MMAs may
// start), store it, then do the same for half 1.
//
// Stream-K tail as in the 128 x 256 form (same chunk walk): a CTA holding a
// tile's last K iterations publishes both halves' fp32 partials, one flag
// per epilogue warp; the CTA holding the tile's first iterations adds them.
constexpr int kWideThreads = 320;
constexpr int kWideBM = 256;
constexpr int kWideStages = 3;
constexpr int kWideABytes = kWideBM * 128;  // 32 KiB
constexpr int kWideStageBytes = kWideABytes + kBBytes;
constexpr int kWideStageOut = 32 * 128;  // per epilogue warp: a 32-row x 64-column bf16 staging box
constexpr int kWideSmem = kWideStages * kWideStageBytes + 8 * kWideStageOut + 1024;
static_assert(kWideSmem <= 232448, "shared memory budget");

// tmap_y: Y as rows of 2N bytes, boxes of 32 rows x 128 bytes (128-byte
// swizzle): the bf16 tiles leave by tensor store.
template <int MODE>
__global__ void __launch_bounds__(kWideThreads, 1)
    large_wide_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_y,
                      const LargeParams p) {
  extern __shared__ uint8_t dsmem[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[kWideStages];
  __shared__ __align__(8) uint64_t empty_bar[kWideStages];
  __shared__ __align__(8) uint64_t acce_bar[2];
  __shared__ __align__(8) uint64_t accf_bar, stall_bar, drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh, issued_sh, consumed_sh, mma_any_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles = p.tiles_m * p.tiles_n;
  const int KB = p.KB;
  const uint64_t T = p.timeout_ns;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kWideStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    mbar_init(&acce_bar[0], 8);
    mbar_init(&acce_bar[1], 8);
    mbar_init(&accf_bar, 1);
    mbar_init(&stall_bar, 1);
    mbar_init(&drain_bar, 1);
    abort_sh = 0;
    issued_sh = 0;
    consumed_sh = 0;
    mma_any_sh = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) prefetch_tmap(&tmap_a);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      const int nch = chunk_count(p, blockIdx.x, gridDim.x, tiles, KB);
      for (int ci = 0; ok && ci < nch; ++ci) {
        const Chunk ch = chunk_at(p, blockIdx.x, gridDim.x, KB, ci);
        const TileCoord tc = tile_coord(ch.t, p.tiles_m, p.tiles_n, p.group_n);
        const int nslabs_n = min(2, p.N / 128 - 2 * tc.n);
        for (int kb = ch.k0; kb < ch.k1; ++kb, ++it) {
          const int slot = it % kWideStages;
          if (!mbar_wait(&empty_bar[slot], ((it / kWideStages) & 1) ^ 1u, T, p.err, 31)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + slot * kWideStageBytes;
          mbar_arrive_expect_tx(&full_bar[slot], kWideABytes + nslabs_n * 16384);
          tma_load_2d(st, &tmap_a, kb * 128, tc.m * kWideBM, &full_bar[slot]);
          tma_load_2d(st + kABytes, &tmap_a, kb * 128, tc.m * kWideBM + kBM, &full_bar[slot]);
          for (int h = 0; h < nslabs_n; ++h)
            bulk_g2s(st + kWideABytes + h * 16384,
                     p.b_img + (static_cast<size_t>(2 * tc.n + h) * KB + kb) * 16384, 16384, &full_bar[slot]);
        }
      }
      issued_sh = it;
      if (!ok) abort_sh = 1;
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      bool ok = true;
      if (p.debug_stall) ok = mbar_wait(&stall_bar, 0, T, p.err, 32);
      int it = 0;
      const uint32_t idesc = MODE == kBF16 ? idesc_bf16(kBM, kBN) : idesc_e4m3(kBM, kBN);
      const int nch = chunk_count(p, blockIdx.x, gridDim.x, tiles, KB);
      for (int ti = 0; ok && ti < nch; ++ti) {
        const Chunk ch = chunk_at(p, blockIdx.x, gridDim.x, KB, ti);
        for (int kb = ch.k0; kb < ch.k1; ++kb, ++it) {
          const int slot = it % kWideStages;
          if (!mbar_wait(&full_bar[slot], (it / kWideStages) & 1, T, p.err, 33)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_any_sh = 1;
          uint8_t* st = smem + slot * kWideStageBytes;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (kb == ch.k0) {
              // half h of the accumulator: drained by the epilogue of the previous chunk
              if (!mbar_wait(&acce_bar[h], (ti & 1) ^ 1u, T, p.err, 34)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            const uint32_t d = tmem + h * kBN;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint64_t adesc = sdesc_sw128(smem_u32(st + h * kABytes + j * 32));
              const uint64_t bdesc = sdesc_sw128(smem_u32(st + kWideABytes + j * 32));
              const uint32_t accum = (kb > ch.k0 || j > 0) ? 1u : 0u;
              if (MODE == kBF16)
                mma_f16(d, adesc, bdesc, idesc, accum);
              else
                mma_f8f6f4(d, adesc, bdesc, idesc, accum);
            }
          }
          if (!ok) {
            ++it;  // this stage's fill was consumed
            break;
          }
          tc_commit(&empty_bar[slot]);
        }
        if (!ok) break;
        tc_commit(&accf_bar);
      }
      consumed_sh = it;
      if (!ok) abort_sh = 1;
      if (mma_any_sh) {
        tc_commit(&drain_bar);
        mbar_wait(&drain_bar, 0, T, p.err, 35);
      }
    }
  } else {
    // -------------------------------------------- epilogue (eight warps)
    // lane quarter warp % 4 (the TMEM lanes this warp may read), column half
    // (warp - 2) / 4 of each accumulator half
    const int qd = warp & 3;
    const int chalf = (warp - 2) >> 2;
    float scale = 1.f;
    if (MODE == kTensor) scale = __ldg(static_cast<const float*>(p.a_scales)) * __ldg(p.b_s);
    const int ew = warp - 2;  // epilogue warp 0..7: its stream-K flag
    uint8_t* stg = smem + kWideStages * kWideStageBytes + ew * kWideStageOut;
    const int nch = chunk_count(p, blockIdx.x, gridDim.x, tiles, KB);
    for (int ti = 0; ti < nch; ++ti) {
      const Chunk ch = chunk_at(p, blockIdx.x, gridDim.x, KB, ti);
      const bool w = mbar_wait(&accf_bar, ti & 1, T, p.err, 36);
      if (!__all_sync(0xffffffffu, w)) {
        if (lane == 0) abort_sh = 1;
        break;
      }
      tc_fence_after();
      const TileCoord tc = tile_coord(ch.t, p.tiles_m, p.tiles_n, p.group_n);
      const int col0 = tc.n * kBN + chalf * 128;
      const int lrow = qd * 32 + lane;
      // stream-K partials: [CTA][half][256 columns][128 rows] fp32
      const bool publish = ch.k0 > 0;   // this CTA holds the tile's last iterations
      const bool finish = !publish && ch.k1 < KB;  // the rest comes from CTA blockIdx.x + 1
      bool have_peer = true;
      if (finish) {
        bool fw = true;
        if (lane == 0) fw = wait_flag_eq(p.sk_flag + (blockIdx.x + 1) * 8 + ew, p.epoch, T, p.err, 37);
        have_peer = __shfl_sync(0xffffffffu, fw ? 1 : 0, 0) != 0;
        if (have_peer) (void)ld_acquire_u64(p.sk_flag + (blockIdx.x + 1) * 8 + ew);
        else if (lane == 0) abort_sh = 1;
      }
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        uint32_t v[128];
        const uint32_t taddr = tmem + h * kBN + chalf * 128 + (static_cast<uint32_t>(qd * 32) << 16);
        tmem_ld32(taddr + 0, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        tmem_ld32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        tmem_ld32(taddr + 64, *reinterpret_cast<uint32_t(*)[32]>(&v[64]));
        tmem_ld32(taddr + 96, *reinterpret_cast<uint32_t(*)[32]>(&v[96]));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acce_bar[h]);  // half h free: the next chunk's MMAs may write it
        const size_t pbase = static_cast<size_t>(h) * kBN * kBM + static_cast<size_t>(chalf) * 128 * kBM + lrow;
        if (publish) {
          float* part = p.sk_part + static_cast<size_t>(blockIdx.x) * 2 * kBN * kBM + pbase;
#pragma unroll
          for (int i = 0; i < 128; ++i) __stcg(part + i * kBM, __uint_as_float(v[i]));
          continue;
        }
        if (finish && have_peer) {
          const float* peer = p.sk_part + static_cast<size_t>(blockIdx.x + 1) * 2 * kBN * kBM + pbase;
#pragma unroll
          for (int i = 0; i < 128; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) + __ldcg(peer + i * kBM));
        }
        if (col0 < p.N && have_peer) {
          // bf16 out through this warp's staging box, 64 columns at a time,
          // by tensor store (rows past M are not written)
          const int row0 = tc.m * kWideBM + h * kBM + qd * 32;
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            if (lane == 0) bulk_wait_group_read0();  // the previous store has read the box
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int q = 8 * r + j;
              uint4 o;
              o.x = pack_bf16x2(__uint_as_float(v[8 * q + 0]) * scale, __uint_as_float(v[8 * q + 1]) * scale);
              o.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]) * scale, __uint_as_float(v[8 * q + 3]) * scale);
              o.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]) * scale, __uint_as_float(v[8 * q + 5]) * scale);
              o.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]) * scale, __uint_as_float(v[8 * q + 7]) * scale);
              *reinterpret_cast<uint4*>(stg + lane * 128 + ((j ^ (lane & 7)) << 4)) = o;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmap_y, stg, (col0 + 64 * r) * 2, row0);
              bulk_commit_group();
            }
          }
        }
      }
      if (publish) {
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release_u64(p.sk_flag + blockIdx.x * 8 + ew, p.epoch);
      } else if (finish && have_peer) {
        // consumed: clear the flag, so that a replay of this launch (same
        // epoch, e.g. in a CUDA graph) waits for the partial it writes
        __syncwarp();
        if (lane == 0) p.sk_flag[(blockIdx.x + 1) * 8 + ew] = 0;
      }
    }
    if (lane == 0) bulk_wait_group0();  // every store has landed
  }

  // ------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (abort_sh && threadIdx.x == 0) {
    for (int it = consumed_sh; it < issued_sh; ++it)
      mbar_wait(&full_bar[it % kWideStages], (it / kWideStages) & 1, T, nullptr, 0);
  }
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <int MODE>
cudaError_t launch_wide(const CUtensorMap& tmap_a, const CUtensorMap& tmap_y, const LargeParams& p, int ctas,
                        cudaStream_t stream) {
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(&large_wide_kernel<MODE>), kWideSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kWideThreads);
  cfg.dynamicSmemBytes = kWideSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeCooperative;  // stream-K CTAs wait on one another: all must be resident
  attr.val.cooperative = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = p.sk_iters > 0 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, large_wide_kernel<MODE>, tmap_a, tmap_y, p);
}


// ------------------------------------------------------------------ MX form
//
// Block-scaled variant (mxfp8: kind::mxf8f6f4, one E8M0 per 32 K of the
// hardware block -- the 128-K mxfp8 scale repeated four times in the atoms;
// mxfp4: kind::mxf4 with two E8M0 per 64-K MMA; fp8 activations against fp4
// weights: kind::mxf8f6f4 with an e4m3 A and an e2m1 B, the weight blocks
// loaded by a tensor copy that spreads every 16 packed codes over a 16-byte
// shared-memory chunk -- the sub-byte operand form this kind reads -- so the
// weight tile has the geometry of an e4m3 tile and HBM moves the packed
// bytes).  Per stage the producer also bulk-copies the scale atoms of the A
// tile (from the per-call A scale image) and of the two weight slabs; the MMA
// thread moves them into a TMEM ring with tcgen05.cp before the stage's MMAs.  TMEM holds one 256-column
// accumulator plus that ring, so the epilogue runs on eight warps that each
// pull their 128 columns into registers and release the accumulator before
// converting and storing -- the next tile's MMAs overlap the stores.
constexpr int kMxThreads = 320;

template <int MODE>
struct MxCfg {
  static constexpr int APS = MODE == kMXFP4 ? 2 : 1;  // atoms per slab (4 K-blocks of 32 each)
  static constexpr int SFA_BYTES = APS * 512;
  static constexpr int SFB_BYTES = 2 * APS * 512;
  static constexpr int STAGE_RAW = kABytes + kBBytes + SFA_BYTES + SFB_BYTES;
  static constexpr int STAGE_BYTES = (STAGE_RAW + 1023) / 1024 * 1024;
  static constexpr int OUT_BYTES = 8 * 32 * 64;  // per epilogue warp: a 32-row x 32-column bf16 staging box
  static constexpr int SMEM = kStages * STAGE_BYTES + OUT_BYTES + 1024;
  static constexpr int SF_COLS = APS * 4 + APS * 8;  // TMEM columns per stage: A (128 rows) + B (256 rows)
  // mxfp8: one atom holds four slabs' scales, so the scales are copied at
  // the first slab of each group of four, into a ring of four group buffers
  // (SF_COLS each) -- rewritten at least four slabs later, after the refill
  // of that slab's stage has waited for the MMAs that read it
  static constexpr bool GROUP4 = MODE == kMXFP8;
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(256 + kStages * SF_COLS <= kTmemCols, "TMEM budget");
};

// tmap_b: fp8 x fp4 only, the weight image as 4-bit codes {128 codes, 128
// rows, N/128 * K/128 blocks}; unused otherwise.
template <int MODE>
__global__ void __launch_bounds__(kMxThreads, 1)
    large_mx_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                    const __grid_constant__ CUtensorMap tmap_y, const LargeParams p) {
  using C = MxCfg<MODE>;
  extern __shared__ uint8_t dsmem[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t accf_bar, acce_bar, stall_bar, drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh, issued_sh, consumed_sh, mma_any_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles = p.tiles_m * p.tiles_n;
  const int KB = p.KB;
  const uint64_t T = p.timeout_ns;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    mbar_init(&accf_bar, 1);
    mbar_init(&acce_bar, 8);
    mbar_init(&stall_bar, 1);
    mbar_init(&drain_bar, 1);
    abort_sh = 0;
    issued_sh = 0;
    consumed_sh = 0;
    mma_any_sh = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmap_a);
    if (MODE == kMXFP4FP8A) prefetch_tmap(&tmap_b);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  // bytes one weight slab counts on the stage barrier: the packed fp4 block
  // (8 KiB, written to 16 KiB of shared memory) or the 16 KiB slab
  constexpr int kBSlabTx = MODE == kMXFP4FP8A ? 8192 : 16384;

  if (warp == 0) {
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
        const TileCoord tc = tile_coord(t, p.tiles_m, p.tiles_n, p.group_n);
        const int nslabs_n = min(2, p.N / 128 - 2 * tc.n);
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int slot = it % kStages;
          if (!mbar_wait(&empty_bar[slot], ((it / kStages) & 1) ^ 1u, T, p.err, 21)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + slot * C::STAGE_BYTES;
          const bool sf_here = !C::GROUP4 || (kb & 3) == 0;  // mxfp8: scales once per four slabs
          const int G = (KB + 3) / 4;
          mbar_arrive_expect_tx(&full_bar[slot], kABytes + nslabs_n * kBSlabTx +
                                                     (sf_here ? C::SFA_BYTES + nslabs_n * C::APS * 512 : 0));
          tma_load_2d(st, &tmap_a, kb * 128, tc.m * kBM, &full_bar[slot]);
          if (sf_here)
            bulk_g2s(st + kABytes + kBBytes,
                     p.a_sf + (C::GROUP4 ? static_cast<size_t>(tc.m) * G + kb / 4 : static_cast<size_t>(tc.m) * KB + kb) *
                                  C::SFA_BYTES,
                     C::SFA_BYTES, &full_bar[slot]);
          for (int h = 0; h < nslabs_n; ++h) {
            const size_t slab = static_cast<size_t>(2 * tc.n + h) * KB + kb;
            if (MODE == kMXFP4FP8A)
              tma_load_3d(st + kABytes + h * 16384, &tmap_b, 0, 0, static_cast<int32_t>(slab), &full_bar[slot]);
            else
              bulk_g2s(st + kABytes + h * 16384, p.b_img + slab * 16384, 16384, &full_bar[slot]);
            if (sf_here) {
              const size_t atom = C::GROUP4 ? static_cast<size_t>(2 * tc.n + h) * G + kb / 4 : slab * C::APS;
              bulk_g2s(st + kABytes + kBBytes + C::SFA_BYTES + h * C::APS * 512, p.b_sf + atom * 512, C::APS * 512,
                       &full_bar[slot]);
            }
          }
        }
      }
      issued_sh = it;
      if (!ok) abort_sh = 1;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      bool ok = true;
      if (p.debug_stall) ok = mbar_wait(&stall_bar, 0, T, p.err, 22);
      int it = 0, ti = 0, gc = 0;  // gc: scale groups copied so far (mxfp8)
      for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x, ++ti) {
        if (!mbar_wait(&acce_bar, (ti & 1) ^ 1u, T, p.err, 23)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int slot = it % kStages;
          if (!mbar_wait(&full_bar[slot], (it / kStages) & 1, T, p.err, 24)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_any_sh = 1;
          uint8_t* st = smem + slot * C::STAGE_BYTES;
          const bool sf_here = !C::GROUP4 || (kb & 3) == 0;
          if (C::GROUP4 && sf_here) ++gc;
          const uint32_t sfa = 256 + (C::GROUP4 ? ((gc - 1) & 3) : slot) * C::SF_COLS;
          const uint32_t sfb = sfa + C::APS * 4;
          uint8_t* sfa_sm = st + kABytes + kBBytes;
          uint8_t* sfb_sm = sfa_sm + C::SFA_BYTES;
          if (sf_here) {
#pragma unroll
            for (int g = 0; g < C::APS; ++g) {
              tc_cp_32x128b_warpx4(tmem + sfa + 4 * g, sdesc_plain_rows16(smem_u32(sfa_sm + 512 * g)));
              tc_cp_32x128b_warpx4(tmem + sfb + 8 * g, sdesc_plain_rows16(smem_u32(sfb_sm + 512 * g)));
              tc_cp_32x128b_warpx4(tmem + sfb + 8 * g + 4,
                                   sdesc_plain_rows16(smem_u32(sfb_sm + C::APS * 512 + 512 * g)));
            }
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint64_t adesc = sdesc_sw128(smem_u32(st + j * 32));
            const uint64_t bdesc = sdesc_sw128(smem_u32(st + kABytes + j * 32));
            if (MODE == kMXFP8) {  // byte kb % 4 of the group's atoms
              mma_mxf8f6f4(tmem, adesc, bdesc, idesc_mx(kBM, kBN, kF8f6f4E4M3, kb & 3, kb & 3), tmem + sfa, tmem + sfb,
                           (kb | j) != 0);
            } else if (MODE == kMXFP8B32) {
              mma_mxf8f6f4(tmem, adesc, bdesc, idesc_mx(kBM, kBN, kF8f6f4E4M3, j, j), tmem + sfa, tmem + sfb,
                           (kb | j) != 0);
            } else if (MODE == kMXFP4FP8A) {
              mma_mxf8f6f4(tmem, adesc, bdesc, idesc_mx_ab(kBM, kBN, kF8f6f4E4M3, kF8f6f4E2M1, j, j), tmem + sfa,
                           tmem + sfb, (kb | j) != 0);
            } else {
              const int g = j >> 1, id = 2 * (j & 1);
              mma_mxf4(tmem, adesc, bdesc, idesc_mx(kBM, kBN, kMxf4E2M1, id, id), tmem + sfa + 4 * g, tmem + sfb + 8 * g,
                       (kb | j) != 0);
            }
          }
          tc_commit(&empty_bar[slot]);
        }
        if (!ok) {
          ++it;
          break;
        }
        tc_commit(&accf_bar);
      }
      consumed_sh = it;
      if (!ok) abort_sh = 1;
      if (mma_any_sh) {
        tc_commit(&drain_bar);
        mbar_wait(&drain_bar, 0, T, p.err, 25);
      }
    }
  } else {
    // eight epilogue warps: lane quarter warp % 4, column half (warp - 2) / 4
    const int qd = warp & 3;
    const int half = (warp - 2) >> 2;
    // this warp's 32-row x 32-column bf16 staging box (64-byte swizzle)
    uint8_t* stg = smem + kStages * C::STAGE_BYTES + (warp - 2) * (32 * 64);
    int ti = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++ti) {
      const bool w = mbar_wait(&accf_bar, ti & 1, T, p.err, 26);
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
      if (lane == 0) mbar_arrive(&acce_bar);  // accumulator free: the next tile may start
      const TileCoord tc = tile_coord(t, p.tiles_m, p.tiles_n, p.group_n);
      const int col0 = tc.n * kBN + half * 128;
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
            tma_store_2d(&tmap_y, stg, (col0 + 32 * r) * 2, tc.m * kBM + qd * 32);
            bulk_commit_group();
          }
        }
      }
    }
    if (lane == 0) bulk_wait_group0();  // every store has landed
  }

  tc_fence_before();
  __syncthreads();
  if (abort_sh && threadIdx.x == 0) {
    for (int it = consumed_sh; it < issued_sh; ++it)
      mbar_wait(&full_bar[it % kStages], (it / kStages) & 1, T, nullptr, 0);
  }
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <int MODE>
cudaError_t launch_mx(const CUtensorMap& tmap_a, const CUtensorMap& tmap_b, const CUtensorMap& tmap_y,
                      const LargeParams& p, int ctas, cudaStream_t stream) {
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(&large_mx_kernel<MODE>), MxCfg<MODE>::SMEM);
  if (e != cudaSuccess) return e;
  large_mx_kernel<MODE><<<ctas, kMxThreads, MxCfg<MODE>::SMEM, stream>>>(tmap_a, tmap_b, tmap_y, p);
  return cudaGetLastError();
}

// ------------------------------------------------------ FP8 blockscale form
//
// FP8 with fp32 scales per (row of A, 128-K block) and per (128 weight rows,
// 128-K block) -- the aiter PR "FlyDSL split-K preshuffle decode GEMM for
// small-M shapes" blockscale mode, at large M.  The scales are fp32, not
// E8M0, so the block-scaled MMA cannot apply them; instead each 128-byte K
// slab (exactly one 128-K scale block) is multiplied into one of two TMEM
// partial buffers (the page's gfx942 software-dequant design: one plain MMA
// pass per scale block), and eight epilogue warps fold every partial into
// fp32 register accumulators as acc += a_s[row][kb] * b_s[nb][kb] * partial,
// storing bf16 at the end of the tile.  Per thread: its TMEM lane (a row of
// A) x 128 of the tile's 256 columns (one 128-row weight block, one b_s).
// The 128 fp32 accumulators per thread need more registers than an even
// split of the file gives, so the first warpgroup (producer, MMA issuer, two
// idle warps) gives registers up to the two epilogue warpgroups:
// 128 x 24 + 256 x 240 = 384 x 168, the launch's total.
constexpr int kBlockThreads = 384;
constexpr int kBlockRegsLow = 24, kBlockRegsHigh = 240;
static_assert(128 * kBlockRegsLow + 256 * kBlockRegsHigh <= kBlockThreads * 168, "register split over the launch");
constexpr int kBlockStageOut = 32 * 128;  // per epilogue warp: 32 rows x 64 bf16 columns
constexpr int kBlockSmem = kStages * kStageBytes + 8 * kBlockStageOut + 1024;
static_assert(kBlockSmem <= 232448, "shared memory per CTA");


__device__ __forceinline__ uint64_t f32x2_splat(float w) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(w));
  return r;
}

// a0 += v0 * w, a1 += v1 * w: two fused multiply-adds, each rounded once
__device__ __forceinline__ void fma_f32x2(float& a0, float& a1, uint32_t v0, uint32_t v1, uint64_t w2) {
  asm("{\n .reg .b64 a, v;\n mov.b64 a, {%0, %1};\n mov.b64 v, {%2, %3};\n"
      " fma.rn.f32x2 a, v, %4, a;\n mov.b64 {%0, %1}, a;\n}"
      : "+f"(a0), "+f"(a1)
      : "r"(v0), "r"(v1), "l"(w2));
}


__global__ void __launch_bounds__(kBlockThreads, 1)
    large_block_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_y,
                       const LargeParams p) {
  extern __shared__ uint8_t dsmem[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t pfull_bar[2], pempty_bar[2];  // the two partial buffers
  __shared__ __align__(8) uint64_t stall_bar, drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh, issued_sh, consumed_sh, mma_any_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles = p.tiles_m * p.tiles_n;
  const int KB = p.KB;
  const uint64_t T = p.timeout_ns;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&pfull_bar[i], 1);
      mbar_init(&pempty_bar[i], 8);  // the eight epilogue warps
    }
    mbar_init(&stall_bar, 1);
    mbar_init(&drain_bar, 1);
    abort_sh = 0;
    issued_sh = 0;
    consumed_sh = 0;
    mma_any_sh = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) prefetch_tmap(&tmap_a);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp < 4) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kBlockRegsLow));
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
        const TileCoord tc = tile_coord(t, p.tiles_m, p.tiles_n, p.group_n);
        const int nslabs_n = min(2, p.N / 128 - 2 * tc.n);
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int slot = it % kStages;
          if (!mbar_wait(&empty_bar[slot], ((it / kStages) & 1) ^ 1u, T, p.err, 51)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + slot * kStageBytes;
          mbar_arrive_expect_tx(&full_bar[slot], kABytes + nslabs_n * 16384);
          tma_load_2d(st, &tmap_a, kb * 128, tc.m * kBM, &full_bar[slot]);
          for (int h = 0; h < nslabs_n; ++h)
            bulk_g2s(st + kABytes + h * 16384, p.b_img + (static_cast<size_t>(2 * tc.n + h) * KB + kb) * 16384,
                     16384, &full_bar[slot]);
        }
      }
      issued_sh = it;
      if (!ok) abort_sh = 1;
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      bool ok = true;
      if (p.debug_stall) ok = mbar_wait(&stall_bar, 0, T, p.err, 52);
      int it = 0;
      const uint32_t idesc = idesc_e4m3(kBM, kBN);
      for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
        for (int kb = 0; kb < KB; ++kb) {
          const int slot = it % kStages;
          const int b = it & 1;  // partial buffer of this slab
          if (!mbar_wait(&full_bar[slot], (it / kStages) & 1, T, p.err, 53) ||
              !mbar_wait(&pempty_bar[b], ((it >> 1) & 1) ^ 1u, T, p.err, 54)) {
            ok = false;
            break;
          }
          ++it;  // this stage's copies have landed
          tc_fence_after();
          mma_any_sh = 1;
          uint8_t* st = smem + slot * kStageBytes;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint64_t adesc = sdesc_sw128(smem_u32(st + j * 32));
            const uint64_t bdesc = sdesc_sw128(smem_u32(st + kABytes + j * 32));
            mma_f8f6f4(tmem + b * kBN, adesc, bdesc, idesc, j > 0 ? 1u : 0u);
          }
          tc_commit(&pfull_bar[b]);      // the slab's partial is ready
          tc_commit(&empty_bar[slot]);   // and its stage may be refilled
        }
      }
      consumed_sh = it;
      if (!ok) abort_sh = 1;
      if (mma_any_sh) {
        tc_commit(&drain_bar);
        mbar_wait(&drain_bar, 0, T, p.err, 55);
      }
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kBlockRegsHigh));
    // ------------------------------------ epilogue (two warpgroups, 8 warps)
    // lane quarter warp % 4 (the TMEM lanes this warp may read), column half
    // (warp - 4) / 4: one 128-row weight block of the 256-column tile
    const int qd = warp & 3;
    const int half = (warp - 4) >> 2;
    const int KS = p.K / 128;
    const float* a_s = static_cast<const float*>(p.a_scales);
    // scales are read four slabs at a time, a group ahead of their use
    const bool vec4 = KS % 4 == 0 && ((reinterpret_cast<uintptr_t>(a_s) | reinterpret_cast<uintptr_t>(p.b_s)) & 15) == 0;
    // this warp's 32-row x 64-column bf16 staging box (128-byte swizzle)
    uint8_t* stg = smem + kStages * kStageBytes + (warp - 4) * kBlockStageOut;
    // scale rows of tile t for this thread (a row past M or a weight block
    // past N reads row / block 0; nothing of it is stored)
    auto scale_rows = [&](int t, const float*& arow, const float*& bcol) {
      const TileCoord tc = tile_coord(t, p.tiles_m, p.tiles_n, p.group_n);
      const int row = tc.m * kBM + qd * 32 + lane;
      const int nb = 2 * tc.n + half;
      arow = a_s + static_cast<size_t>(row < p.M ? row : 0) * KS;
      bcol = p.b_s + static_cast<size_t>(nb < p.N / 128 ? nb : 0) * KS;
    };
    auto load_group = [&](const float* arow, const float* bcol, int kb0, float4& an, float4& bn) {
      if (vec4) {
        an = __ldg(reinterpret_cast<const float4*>(arow + kb0));
        bn = __ldg(reinterpret_cast<const float4*>(bcol + kb0));
      } else {
        an.x = __ldg(arow + kb0);
        bn.x = __ldg(bcol + kb0);
        an.y = kb0 + 1 < KS ? __ldg(arow + kb0 + 1) : 0.f;
        bn.y = kb0 + 1 < KS ? __ldg(bcol + kb0 + 1) : 0.f;
        an.z = kb0 + 2 < KS ? __ldg(arow + kb0 + 2) : 0.f;
        bn.z = kb0 + 2 < KS ? __ldg(bcol + kb0 + 2) : 0.f;
        an.w = kb0 + 3 < KS ? __ldg(arow + kb0 + 3) : 0.f;
        bn.w = kb0 + 3 < KS ? __ldg(bcol + kb0 + 3) : 0.f;
      }
    };
    const float* arow = a_s;
    const float* bcol = p.b_s;
    float4 an = make_float4(0.f, 0.f, 0.f, 0.f), bn = an;
    if (static_cast<int>(blockIdx.x) < tiles) {
      scale_rows(blockIdx.x, arow, bcol);
      load_group(arow, bcol, 0, an, bn);
    }
    int it = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
      const TileCoord tc = tile_coord(t, p.tiles_m, p.tiles_n, p.group_n);
      const bool have_nb = 2 * tc.n + half < p.N / 128;
      const float* ar = arow;
      const float* bc = bcol;
      float acc[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) acc[i] = 0.f;
#pragma unroll 1
      for (int kb0 = 0; ok && kb0 < KB; kb0 += 4) {
        const float wg[4] = {an.x * bn.x, an.y * bn.y, an.z * bn.z, an.w * bn.w};
        // the next group's scales (the next tile's first) load while this group runs
        if (kb0 + 4 < KB) {
          load_group(ar, bc, kb0 + 4, an, bn);
        } else if (t + static_cast<int>(gridDim.x) < tiles) {
          scale_rows(t + gridDim.x, arow, bcol);
          load_group(arow, bcol, 0, an, bn);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (kb0 + j >= KB) break;
          const int b = it & 1;
          const bool ready = mbar_wait(&pfull_bar[b], (it >> 1) & 1, T, p.err, 56);
          if (!__all_sync(0xffffffffu, ready)) {
            ok = false;
            break;
          }
          ++it;
          tc_fence_after();
          const uint32_t taddr = tmem + b * kBN + half * 128 + (static_cast<uint32_t>(qd * 32) << 16);
          const uint64_t w2 = f32x2_splat(wg[j]);
          // eight 16-column loads; each chunk is folded while the next loads
          uint32_t va[16], vb[16];
          tmem_ld16(taddr, va);
          tmem_wait_ld();
#pragma unroll
          for (int c = 1; c < 8; ++c) {
            if (c & 1) {
              tmem_ld16(taddr + 16 * c, vb);
#pragma unroll
              for (int i = 0; i < 16; i += 2)
                fma_f32x2(acc[16 * (c - 1) + i], acc[16 * (c - 1) + i + 1], va[i], va[i + 1], w2);
            } else {
              tmem_ld16(taddr + 16 * c, va);
#pragma unroll
              for (int i = 0; i < 16; i += 2)
                fma_f32x2(acc[16 * (c - 1) + i], acc[16 * (c - 1) + i + 1], vb[i], vb[i + 1], w2);
            }
            tmem_wait_ld();
          }
          // the whole partial is in registers: the buffer may take the slab after next
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&pempty_bar[b]);
#pragma unroll
          for (int i = 0; i < 16; i += 2) fma_f32x2(acc[112 + i], acc[113 + i], vb[i], vb[i + 1], w2);
        }
      }
      if (!ok) break;
      if (have_nb) {
        // bf16 out through the staging box, 64 columns at a time, by tensor
        // store (rows past M are not written)
        const int col0 = tc.n * kBN + half * 128;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          if (lane == 0) bulk_wait_group_read0();  // the previous store has read the box
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            uint4 o;
            o.x = pack_bf16x2(acc[64 * r + 8 * j + 0], acc[64 * r + 8 * j + 1]);
            o.y = pack_bf16x2(acc[64 * r + 8 * j + 2], acc[64 * r + 8 * j + 3]);
            o.z = pack_bf16x2(acc[64 * r + 8 * j + 4], acc[64 * r + 8 * j + 5]);
            o.w = pack_bf16x2(acc[64 * r + 8 * j + 6], acc[64 * r + 8 * j + 7]);
            *reinterpret_cast<uint4*>(stg + lane * 128 + ((j ^ (lane & 7)) << 4)) = o;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmap_y, stg, (col0 + 64 * r) * 2, tc.m * kBM + qd * 32);
            bulk_commit_group();
          }
        }
      }
    }
    if (lane == 0) bulk_wait_group0();  // every store has landed
    if (!ok && lane == 0) abort_sh = 1;
  }

  // ------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (abort_sh && threadIdx.x == 0) {
    for (int it = consumed_sh; it < issued_sh; ++it)
      mbar_wait(&full_bar[it % kStages], (it / kStages) & 1, T, nullptr, 0);
  }
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

cudaError_t launch_block(const CUtensorMap& tmap_a, const CUtensorMap& tmap_y, const LargeParams& p, int ctas,
                         cudaStream_t stream) {
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(&large_block_kernel), kBlockSmem);
  if (e != cudaSuccess) return e;
  large_block_kernel<<<ctas, kBlockThreads, kBlockSmem, stream>>>(tmap_a, tmap_y, p);
  return cudaGetLastError();
}

}  // namespace

uint64_t large_streamk_bytes(int ctas, bool wide) {
  return wide ? static_cast<uint64_t>(ctas) * (2ull * kBN * kBM * 4 + 8 * 8)
              : static_cast<uint64_t>(ctas) * (static_cast<uint64_t>(kBN) * kBM * 4 + 4 * 8);
}

bool large_supported(int mode) { return mode == kBF16 || mode == kTensor || mode == kBlock || is_mx(mode); }

cudaError_t launch_large(int mode, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b, const CUtensorMap& tmap_y,
                         const LargeParams& p, int ctas, cudaStream_t stream) {
  if (p.wide) {
    if (mode == kBF16) return launch_wide<kBF16>(tmap_a, tmap_y, p, ctas, stream);
    if (mode == kTensor) return launch_wide<kTensor>(tmap_a, tmap_y, p, ctas, stream);
    return cudaErrorNotSupported;
  }
  if (mode == kBlock) return launch_block(tmap_a, tmap_y, p, ctas, stream);
  if (mode == kBF16) return launch_mode<kBF16>(tmap_a, tmap_y, p, ctas, stream);
  if (mode == kTensor) return launch_mode<kTensor>(tmap_a, tmap_y, p, ctas, stream);
  if (mode == kMXFP8) return launch_mx<kMXFP8>(tmap_a, tmap_b, tmap_y, p, ctas, stream);
  if (mode == kMXFP8B32) return launch_mx<kMXFP8B32>(tmap_a, tmap_b, tmap_y, p, ctas, stream);
  if (mode == kMXFP4) return launch_mx<kMXFP4>(tmap_a, tmap_b, tmap_y, p, ctas, stream);
  if (mode == kMXFP4FP8A) return launch_mx<kMXFP4FP8A>(tmap_a, tmap_b, tmap_y, p, ctas, stream);
  return cudaErrorNotSupported;
}

}  // namespace fg
