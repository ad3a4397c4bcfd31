// Split-K decode GEMM for small M (aiter PR "FlyDSL split-K preshuffle
// decode GEMM for small-M shapes (FP8 + MX, gfx950/gfx942)", Summary and
// What's included), written for sm_103a tensor cores.
//
// Orientation ("swap AB"): the weight B is the MMA's M operand (128 rows of
// N per CTA), a tile of TOK token rows of A is the MMA's N operand -- 16, or
// 32 when there are more than 16 tokens, so that 17..32 tokens stream the
// weights once -- so one tcgen05.mma is 128 x TOK x (32 bytes of K) and the
// fp32 accumulator lives in TOK TMEM columns.  CTA (nt, s, mt) covers weight
// rows [128 nt, +128), token rows [TOK mt, +TOK) and split s of the K slabs.
//
// Warp roles (192 threads):
//   warp 0    producer: one bulk copy per stage for the contiguous weight
//             slabs of the preshuffled image, one TMA tensor load per slab
//             for the token tile (rows beyond M are zero-filled), and for MX
//             the weight scale atoms (bulk).  fp4 weights against fp8
//             activations come as packed blocks (128 rows x 64 bytes) through
//             a tensor load that spreads every 16 codes over a 16-byte
//             shared-memory chunk (codes in its low 8 bytes), 128-byte
//             swizzled: the sub-byte operand form of the fp8/fp6/fp4 MMA, so
//             the MMA reads fp4 straight from the copy while HBM moves only
//             the packed bytes;
//   warp 1    allocates TMEM; lane 0 issues tcgen05.cp (MX scale factors)
//             and tcgen05.mma, and commits stage releases;
//   warps 2-5 for MX, first build the token scale atoms of each stage from
//             the caller's E8M0 bytes (ahead of the MMA, one arrival per warp
//             on the stage's full barrier); then
//             epilogue: TMEM -> registers -> fp32 partials (split > 1) or
//             scaled bf16 Y (split == 1).  For FP8_BLOCK128 they also run
//             the per-128-K promotion: each K slab (one 128-K scale block)
//             is multiplied into its own TMEM partial, which they read and
//             fold into fp32 registers as acc += a_s[m][kb] * b_s[nb][kb] *
//             partial (the software-dequant path the page describes for
//             gfx942: one plain MMA pass per 128-K scale block).  bf16 uses
//             the same per-slab partials with a weight of 1: the fold is a
//             compensated sum, which keeps the fp32 partials of long K
//             splits within the workspace bound.
//
// Split-K reduction: with split > 1 the S split CTAs of a tile run as one
// thread-block cluster, and CTA r owns rows [ceil(128 r/S), ceil(128 (r+1)/S))
// of the tile.  Each CTA's receive area is the stage buffer its last
// iterations leave idle first; once the MMAs that read that buffer are done,
// the producer thread tells every peer so (one remote mbarrier arrival each).
// When a CTA's fp32 partial [128 rows][TOK tokens] is in registers and all
// peers are ready, its epilogue threads store each row's tokens straight into
// the owner's receive area (st.async, 16 bytes at a time, counted on the
// owner's mbarrier).  The owner then sums its rows over the S slices in split
// order 0..S-1 (the order of the two-pass reduce, so both paths give the same
// bits), applies the per-tensor scale and stores bf16.  A cluster barrier
// split into arrive (after a CTA has received everything) and wait (at exit)
// keeps every CTA alive until all stores into it have landed.  The two-pass
// form (fp32 workspace + reduce kernel) remains for FG_FLAG_DEFER_REDUCE and
// for splits beyond the cluster size limit.
//
// Launch order: every launch allows the next kernel of the stream to start
// early (programmatic dependent launch).  The producer streams its first
// stages of weights -- which no kernel writes -- before waiting for the
// previous kernel; activations, scales and outputs are touched only after.
//
// MX scale factors: the block-scaled MMA reads, for row i of an operand, the
// byte selected by the instruction's scale-factor id in TMEM lane i, column
// (base + i/32).  tcgen05.cp.32x128b.warpx4 copies a 32-row x 16-byte
// shared-memory atom into four TMEM columns of every 32-lane quarter, which
// gives exactly that layout for atoms whose byte 16*(i%32) + 4*(i/32) + j
// holds row i's scale for the j-th 32-K block.  For a 16-token tile the
// MMA reads column 0 at lanes 32q + m (m < 16) of every quarter q -- which
// the warpx4 copy fills from source rows 0-15 -- so token atoms are laid out
// 256 bytes apart and overlap (rows 16-31 of one atom are rows 0-15 of the
// next); a 32-token tile fills whole atoms, 512 bytes apart.  (A copy that
// filled the quarters from different rows gave wrong token scales: quarters
// 1-3 are read too.)
#include <cuda_bf16.h>

#include <cstdio>

#include "fg_internal.cuh"
#include "fg_ptx.cuh"

namespace fg {

namespace {

constexpr int kThreads = 192;
constexpr int kSlabBytes = 16384;   // 128 rows x 128 bytes
// fp4 weight block of one slab: 128 rows x 64 packed bytes.  Its tensor load
// writes kSlabBytes of shared memory and counts these bytes on the barrier.
constexpr int kFp4SlabBytes = 8192;

// TOK: token rows per CTA tile (the MMA's N): 16, or 32 for 17..32 tokens so
// that the weights stream once
template <int MODE, int SPS, int STAGES, int TOK>
struct DCfg {
  static constexpr int APS = MODE == kMXFP4 ? 2 : (is_mx(MODE) ? 1 : 0);
  static constexpr int TOK_BYTES = TOK * 128;  // one slab of the token tile
  // fp8 activations x fp4 weights: packed fp4 blocks through the spreading
  // tensor load (a 16 KiB tile per slab in shared memory, 8 KiB from HBM)
  static constexpr bool FP4W = MODE == kMXFP4FP8A;
  static constexpr int B_BYTES = SPS * kSlabBytes;
  static constexpr int A_BYTES = SPS * TOK_BYTES;
  static constexpr int SFW_BYTES = SPS * APS * 512;
  // token scale atoms: 16 tokens fill rows 0-15 of an atom, so atoms are laid
  // 256 bytes apart and overlap (rows 16-31 of one are rows 0-15 of the next);
  // 32 tokens fill whole 512-byte atoms
  static constexpr int TOK_ATOM_STRIDE = TOK == 16 ? 256 : 512;
  static constexpr int SFT_BYTES = APS ? SPS * APS * TOK_ATOM_STRIDE + (TOK == 16 ? 256 : 0) : 0;
  static constexpr int PREPASS_WARPS = 4;  // warps 2-5: arrivals on an MX stage's full barrier
  static constexpr int STAGE_RAW = B_BYTES + A_BYTES + SFW_BYTES + SFT_BYTES;
  static constexpr int STAGE_BYTES = (STAGE_RAW + 1023) / 1024 * 1024;
  static constexpr int NBUF = 8;  // blockscale TMEM partial buffers
  static constexpr int SF_COLS = SPS * APS * 4;  // TMEM columns per operand per stage
  // bf16 and fp8-blockscale accumulate each K slab in its own TMEM partial
  // and fold the partials in registers (compensated), see the epilogue
  static constexpr bool PROMOTE = MODE == kBlock || MODE == kBF16;
  // PROMOTE modes commit every slab's partial (pfull); when the partial
  // buffers outnumber the slabs the MMA can run ahead of a waiting producer,
  // ((STAGES - 1) * SPS + 1), that commit also tells the producer the stage
  // is free, and the separate release commit (a few hundred cycles of the MMA
  // pipe per stage) is left out
  static constexpr bool PF_RELEASE = PROMOTE && NBUF >= (STAGES - 1) * SPS + 1;
  static constexpr int TMEM_NEED = PROMOTE ? NBUF * TOK : 32 + STAGES * 2 * SF_COLS;
  static constexpr int TMEM_COLS =
      TMEM_NEED <= 32 ? 32 : (TMEM_NEED <= 64 ? 64 : (TMEM_NEED <= 128 ? 128 : (TMEM_NEED <= 256 ? 256 : 512)));
  static constexpr int SMEM = STAGES * STAGE_BYTES + 1024;
  // CTAs per SM the registers must leave room for: FP8 blockscale with 32
  // tokens folds 32-wide register arrays (the sums, their compensation, the
  // slab's partial) and would otherwise take every register, leaving no room
  // beside it for the next launch
  static constexpr int MIN_CTAS = (MODE == kBlock && TOK == 32) ? 2 : 1;
  static_assert(TMEM_NEED <= 512, "TMEM budget");
  static_assert(TOK == 16 || TOK == 32, "token tile");
  static_assert(SPS * APS * TOK <= 128, "one token scale word per pre-pass thread");
  static_assert(SMEM <= 232448, "shared memory budget");
};

// The weight is the MMA's A operand, the tokens its B operand (N = TOK).
template <int TOK>
__device__ __forceinline__ uint32_t mx_idesc(int mode, int sfid) {
  return mode == kMXFP4        ? idesc_mx(128, TOK, kMxf4E2M1, sfid, sfid)
         : mode == kMXFP4FP8A ? idesc_mx_ab(128, TOK, kF8f6f4E2M1, kF8f6f4E4M3, sfid, sfid)
                               : idesc_mx(128, TOK, kF8f6f4E4M3, sfid, sfid);
}

// A row of the accumulator (TOK fp32 columns of this thread's TMEM lane).
template <int TOK>
__device__ __forceinline__ void tmem_ld_tok(uint32_t taddr, uint32_t (&v)[TOK]) {
  if constexpr (TOK == 16)
    tmem_ld16(taddr, v);
  else
    tmem_ld32(taddr, v);
}

// tmap_b: fp8 x fp4 only, the weight image as [blocks][128 rows][128 codes]
// (see the producer); unused otherwise.
template <int MODE, int SPS, int STAGES, int TOK>
__global__ void __launch_bounds__(kThreads, (DCfg<MODE, SPS, STAGES, TOK>::MIN_CTAS))
    decode_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                  const DecodeParams p) {
  using C = DCfg<MODE, SPS, STAGES, TOK>;
  constexpr int kTokRows = TOK;
  constexpr int kTokSlabBytes = C::TOK_BYTES;
  extern __shared__ uint8_t dsmem[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem) + 1023) & ~uintptr_t(1023));

  __shared__ __align__(8) uint64_t full_bar[STAGES];
  __shared__ __align__(8) uint64_t empty_bar[STAGES];
  __shared__ __align__(8) uint64_t pfull_bar[C::NBUF];
  __shared__ __align__(8) uint64_t pempty_bar[C::NBUF];
  __shared__ __align__(8) uint64_t acc_bar, stall_bar, drain_bar;
  __shared__ __align__(8) uint64_t ready_bar, recv_bar;  // fused split-K reduce
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh, issued_sh, consumed_sh, mma_any_sh;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = blockIdx.x, split = blockIdx.y, mt = blockIdx.z;
  const int q = p.KB / p.split, r = p.KB % p.split;
  const int u0 = split * q + min(split, r);
  const int nslab = q + (split < r ? 1 : 0);
  const int niter = (nslab + SPS - 1) / SPS;
  const uint64_t T = p.timeout_ns;
  // Per-slab partial modes: slab i's partial is announced by one commit for
  // its group of 2^pg slabs (the split's last group may be shorter), on
  // barrier (i >> pg) mod (NBUF >> pg); fewer commits keep the MMA pipe busy.
  static_assert(C::NBUF == 8, "partial barrier indexing");
  const int pg = C::PROMOTE ? p.pgroup_log : 0;
  const int pg_nlog = 3 - pg;
  auto pf_bar = [&](int i) { return &pfull_bar[(i >> pg) & ((1 << pg_nlog) - 1)]; };
  auto pf_par = [&](int i) { return static_cast<uint32_t>((i >> (pg + pg_nlog)) & 1); };
  // fused reduce: the stage buffer that holds split s's receive area
  auto recv_slot = [&](int s) {
    const int ns = q + (s < r ? 1 : 0);
    return ((ns + SPS - 1) / SPS) % STAGES;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full_bar[i], C::APS ? 1 + C::PREPASS_WARPS : 1);  // MX: + one arrival per pre-pass warp
      mbar_init(&empty_bar[i], 1);
    }
    for (int i = 0; i < C::NBUF; ++i) {
      mbar_init(&pfull_bar[i], 1);
      mbar_init(&pempty_bar[i], 4);
    }
    mbar_init(&acc_bar, 1);
    mbar_init(&stall_bar, 1);
    mbar_init(&drain_bar, 1);
    mbar_init(&ready_bar, p.split > 1 ? p.split - 1 : 1);
    mbar_init(&recv_bar, 1);
    abort_sh = 0;
    issued_sh = 0;
    consumed_sh = 0;
    mma_any_sh = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmap_a);
    if (C::FP4W) prefetch_tmap(&tmap_b);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // phase 1 of the cluster barrier: waited on before the first access to a
  // peer, it guarantees the peer's mbarriers are initialised
  if (p.fused_reduce) cluster_arrive_relaxed();
  const uint32_t tmem = tmem_base_sh;
  if (threadIdx.x == 0) pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The first min(STAGES, niter) stages get their weight slabs (and weight
    // scale atoms) before the wait for the previous kernel; their token tiles
    // follow right after it.  Later stages load both together.
    const int pre = min(STAGES, niter);
    int it = 0;
    for (; it < niter; ++it) {
      const int slot = it % STAGES;
      const uint32_t ph = (it / STAGES) & 1;
      bool ok = true;
      if (!C::PF_RELEASE) {
        ok = mbar_wait(&empty_bar[slot], ph ^ 1u, T, p.err, 1);
      } else if (it >= STAGES) {
        // the partial of the last slab of stage it - STAGES (slab commits
        // arrive in order, so every earlier MMA of the stage is done too)
        const int s_last = (it - STAGES + 1) * SPS - 1;
        ok = mbar_wait(pf_bar(s_last), pf_par(s_last), T, p.err, 1);
      }
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) abort_sh = 1;
        break;
      }
      const int ub = it * SPS;
      const int nsl = min(SPS, nslab - ub);
      uint8_t* st = smem + slot * C::STAGE_BYTES;
      if (lane == 0) {
        if (C::FP4W) {
          // block (nt, u) of the image is z = nt * KB + u of the tensor map
          mbar_arrive_expect_tx(&full_bar[slot], nsl * (kFp4SlabBytes + kTokSlabBytes + C::APS * 512));
          for (int v = 0; v < nsl; ++v)
            tma_load_3d(st + v * kSlabBytes, &tmap_b, 0, 0, nt * p.KB + u0 + ub + v, &full_bar[slot]);
        } else {
          mbar_arrive_expect_tx(&full_bar[slot], nsl * (kSlabBytes + kTokSlabBytes + C::APS * 512));
          bulk_g2s(st, p.b_img + (static_cast<size_t>(nt) * p.KB + u0 + ub) * kSlabBytes, nsl * kSlabBytes,
                   &full_bar[slot]);
        }
        if (MODE == kMXFP8) {
          // four slabs' scales to an atom: slab u's is byte u%4 of atom u/4
          const int G = (p.KB + 3) / 4;
          for (int v = 0; v < nsl; ++v)
            bulk_g2s(st + C::B_BYTES + C::A_BYTES + v * 512,
                     p.b_sf + (static_cast<size_t>(nt) * G + (u0 + ub + v) / 4) * 512, 512, &full_bar[slot]);
        } else if (C::APS) {
          bulk_g2s(st + C::B_BYTES + C::A_BYTES,
                   p.b_sf + (static_cast<size_t>(nt) * p.KB + u0 + ub) * C::APS * 512, nsl * C::APS * 512,
                   &full_bar[slot]);
        }
        if (it >= pre) {
          for (int v = 0; v < nsl; ++v)
            tma_load_2d(st + C::B_BYTES + v * kTokSlabBytes, &tmap_a, (u0 + ub + v) * 128, mt * kTokRows,
                        &full_bar[slot]);
        }
      }
      if (it + 1 == pre) {
        // Weights of the first stages are on their way.  When the rest of
        // this CTA's K range is short (at most one more window: the latency-
        // bound shapes), its weights and the token tiles go to L2 meanwhile.
        // A prefetch only warms L2, which every writer of the tokens goes
        // through, so it cannot hand out stale data; the copies into shared
        // memory still wait for the previous kernel.
        if (lane == 0 && nslab <= 2 * pre * SPS) {
          const int ub = pre * SPS;
          const int wb = C::FP4W ? kFp4SlabBytes : kSlabBytes;
          if (nslab > ub)
            prefetch_l2(p.b_img + (static_cast<size_t>(nt) * p.KB + u0 + ub) * wb,
                        static_cast<uint32_t>((nslab - ub) * wb));
          for (int u = 0; u < nslab; ++u) prefetch_l2_box(&tmap_a, (u0 + u) * 128, mt * kTokRows);
        }
        // now wait for the previous kernel, then fetch the token tiles of the
        // first stages
        pdl_wait();
        if (lane == 0) {
          for (int jt = 0; jt < pre; ++jt) {
            const int ubj = jt * SPS;
            const int nslj = min(SPS, nslab - ubj);
            uint8_t* stj = smem + (jt % STAGES) * C::STAGE_BYTES;
            for (int v = 0; v < nslj; ++v)
              tma_load_2d(stj + C::B_BYTES + v * kTokSlabBytes, &tmap_a, (u0 + ubj + v) * 128, mt * kTokRows,
                          &full_bar[jt % STAGES]);
          }
        }
      }
    }
    if (it < pre) pdl_wait();  // aborted before the prefetch window closed
    if (lane == 0) issued_sh = it;
    __syncwarp();
    if (p.fused_reduce) {
      cluster_wait();  // phase 1
      if (lane == 0) {
        // The receive area lives in stage buffer niter % STAGES, idle once the
        // MMAs of the last iteration that used it (niter - STAGES) are done.
        // After an abort (it < niter) the signal goes out at once; the peers
        // then run out of time waiting for data that never comes.
        const int itf = niter - STAGES;
        if (itf >= 0 && it == niter) {
          if (C::PF_RELEASE) {
            const int s_last = (itf + 1) * SPS - 1;
            mbar_wait(pf_bar(s_last), pf_par(s_last), T, p.err, 9);
          } else {
            mbar_wait(&empty_bar[niter % STAGES], (itf / STAGES) & 1, T, p.err, 9);
          }
        }
        const int S = p.split;
        const int Mt = min(kTokRows, p.M - mt * kTokRows);
        const int myR = (128 * (split + 1) + S - 1) / S - (128 * split + S - 1) / S;
        mbar_arrive_expect_tx(&recv_bar, static_cast<uint32_t>((S - 1) * myR * ((Mt + 3) / 4) * 16));
        for (int s2 = 0; s2 < S; ++s2)
          if (s2 != split) mbar_arrive_remote(&ready_bar, s2);
      }
      __syncwarp();
      // phase 2; the release keeps it behind the arrivals just sent to the
      // peers, so no peer can leave before they have landed
      cluster_arrive();
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      bool ok = true;
      if (p.debug_stall) ok = mbar_wait(&stall_bar, 0, T, p.err, 2);
      int it = 0, slab_ctr = 0;
      for (; ok && it < niter; ++it) {
        const int slot = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!mbar_wait(&full_bar[slot], ph, T, p.err, 3)) {
          ok = false;
          break;
        }
        tc_fence_after();
        mma_any_sh = 1;
        const int nsl = min(SPS, nslab - it * SPS);
        uint8_t* st = smem + slot * C::STAGE_BYTES;
        const uint32_t sfw_col = 32 + slot * 2 * C::SF_COLS;
        const uint32_t sft_col = sfw_col + C::SF_COLS;
        if (C::APS) {
          for (int t = 0; t < nsl * C::APS; ++t) {
            tc_cp_32x128b_warpx4(tmem + sfw_col + 4 * t, sdesc_plain_rows16(smem_u32(st + C::B_BYTES + C::A_BYTES + 512 * t)));
            tc_cp_32x128b_warpx4(tmem + sft_col + 4 * t,
                                 sdesc_plain_rows16(smem_u32(st + C::B_BYTES + C::A_BYTES + C::SFW_BYTES +
                                                             C::TOK_ATOM_STRIDE * t)));
          }
        }
        for (int v = 0; v < nsl; ++v) {
          uint32_t d = tmem;
          int pb = 0;
          if (C::PROMOTE) {
            pb = slab_ctr % C::NBUF;
            if (!mbar_wait(&pempty_bar[pb], ((slab_ctr / C::NBUF) & 1) ^ 1u, T, p.err, 4)) {
              ok = false;
              break;
            }
            tc_fence_after();
            d = tmem + pb * TOK;
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint64_t adesc = sdesc_sw128(smem_u32(st + v * kSlabBytes + j * 32));
            const uint64_t bdesc = sdesc_sw128(smem_u32(st + C::B_BYTES + v * kTokSlabBytes + j * 32));
            const uint32_t acc = C::PROMOTE ? (j > 0) : ((it | v | j) != 0);
            if (MODE == kBF16) {
              mma_f16(d, adesc, bdesc, idesc_bf16(128, kTokRows), acc);
            } else if (MODE == kTensor || MODE == kBlock) {
              mma_f8f6f4(d, adesc, bdesc, idesc_e4m3(128, kTokRows), acc);
            } else if (MODE == kMXFP8) {
              // the weight's scale is byte (slab % 4) of its atom; the token
              // atoms repeat theirs in all four bytes
              mma_mxf8f6f4(d, adesc, bdesc, idesc_mx(128, kTokRows, 0u, (u0 + it * SPS + v) & 3, j),
                           tmem + sfw_col + 4 * v, tmem + sft_col + 4 * v, acc);
            } else if (MODE == kMXFP8B32 || MODE == kMXFP4FP8A) {
              mma_mxf8f6f4(d, adesc, bdesc, mx_idesc<TOK>(MODE, j), tmem + sfw_col + 4 * v, tmem + sft_col + 4 * v,
                           acc);
            } else {
              const int t = v * 2 + (j >> 1);
              mma_mxf4(d, adesc, bdesc, mx_idesc<TOK>(MODE, 2 * (j & 1)), tmem + sfw_col + 4 * t,
                       tmem + sft_col + 4 * t, acc);
            }
          }
          if (C::PROMOTE) {
            // the last slab of a group (or of the split) announces the group
            if (((slab_ctr + 1) & ((1 << pg) - 1)) == 0 || slab_ctr + 1 == nslab) tc_commit(pf_bar(slab_ctr));
            ++slab_ctr;
          }
        }
        if (!ok) {
          ++it;  // this stage's fill was consumed
          break;
        }
        // Release the stage only if something waits for that: a refill
        // (iteration it + STAGES) or, for the last such stage, the split-K
        // receive area.  A commit stalls the MMA pipe for about as long as
        // five of these MMAs, and the final commit covers the rest.
        if (!C::PF_RELEASE && it + STAGES <= niter) tc_commit(&empty_bar[slot]);
      }
      consumed_sh = it;
      if (ok && !C::PROMOTE) tc_commit(&acc_bar);
      if (!ok) abort_sh = 1;
      // every MMA and every commit this thread issued has landed before the
      // CTA can release TMEM or its barriers
      if (mma_any_sh) {
        tc_commit(&drain_bar);
        mbar_wait(&drain_bar, 0, T, p.err, 7);
      }
    }
    __syncwarp();
    if (p.fused_reduce) {
      cluster_wait();            // phase 1
      cluster_arrive_relaxed();  // phase 2 (this warp stores nothing into peers)
    }
  } else {
    // ------------------------------------------------------------ epilogue
    if (C::APS) {
      // Before the epilogue proper, these four warps build the token scale
      // atoms of every stage (atom t, token row m -> the 4 E8M0 bytes of the
      // atom's four 32-K blocks), running ahead of the MMA by up to STAGES
      // stages so the global-load latency stays hidden.
      const uint8_t* asf = static_cast<const uint8_t*>(p.a_scales);
      const int et = threadIdx.x - 64;  // 0..127
      bool okb = true;
      // One word per (atom t, token row m) of a stage, at most one per thread
      // (SPS * APS * 16 <= 128): the four E8M0 bytes of the atom's 32-K
      // blocks.  The next stage's word is loaded while this stage is
      // processed, so the global-load latency is not paid stage after stage.
      auto tok_sf = [&](int it) -> uint32_t {
        const int nsl = min(SPS, nslab - it * SPS);
        if (et >= nsl * C::APS * kTokRows) return 0u;
        const int t = et / kTokRows, m = et % kTokRows;
        const int row = mt * kTokRows + m;
        if (row >= p.M) return 0x7F7F7F7Fu;  // 2^0 for padded rows (their values are zero)
        const int q32 = ((u0 + it * SPS) * C::APS + t) * 4;  // first 32-K block of the atom
        if (MODE != kMXFP8) {  // one scale per 32-K block
          const uint8_t* src = asf + static_cast<size_t>(row) * (p.K / 32) + q32;
          // K % 128 == 0 keeps the offset a multiple of 4: one word load
          // unless the caller's scale array itself is not 4-byte aligned
          if ((reinterpret_cast<uintptr_t>(asf) & 3u) == 0) return __ldg(reinterpret_cast<const uint32_t*>(src));
          return static_cast<uint32_t>(src[0]) | (static_cast<uint32_t>(src[1]) << 8) |
                 (static_cast<uint32_t>(src[2]) << 16) | (static_cast<uint32_t>(src[3]) << 24);
        }
        return static_cast<uint32_t>(asf[static_cast<size_t>(row) * (p.K / 128) + (q32 >> 2)]) * 0x01010101u;
      };
      pdl_wait();
      uint32_t wv_next = tok_sf(0);
      for (int it = 0; it < niter; ++it) {
        const int slot = it % STAGES;
        const bool w = mbar_wait(&empty_bar[slot], ((it / STAGES) & 1) ^ 1u, T, p.err, 8);
        if (!__all_sync(0xffffffffu, w)) {
          okb = false;
          break;
        }
        const int ub = it * SPS;
        const int nsl = min(SPS, nslab - ub);
        const uint32_t wv = wv_next;
        if (it + 1 < niter) wv_next = tok_sf(it + 1);
        uint8_t* sft = smem + slot * C::STAGE_BYTES + C::B_BYTES + C::A_BYTES + C::SFW_BYTES;
        if (et < nsl * C::APS * kTokRows)
          *reinterpret_cast<uint32_t*>(sft + (et / kTokRows) * C::TOK_ATOM_STRIDE + (et % kTokRows) * 16) = wv;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full_bar[slot]);
      }
      if (!okb && lane == 0) abort_sh = 1;
    }
    pdl_wait();
    // per-tensor output scale, loaded long before it is needed
    const float out_scale = MODE == kTensor ? __ldg(static_cast<const float*>(p.a_scales)) * __ldg(p.b_s) : 1.f;
    const int qd = warp & 3;
    const int nrow = nt * 128 + qd * 32 + lane;
    const uint32_t trow = tmem + (static_cast<uint32_t>(qd * 32) << 16);
    float acc[kTokRows];
#pragma unroll
    for (int m = 0; m < kTokRows; ++m) acc[m] = 0.f;
    bool ok = true;
    if (C::PROMOTE) {
      // Fold per-slab partials with compensated (Kahan) addition:
      //   acc += w * partial,  w = a_s[m][kb] * b_s[nb][kb] (fp8 blockscale) or 1 (bf16).
      // Each partial holds at most 128 K of products, so the fp32 rounding
      // inside the tensor core stays at the scale of one slab, and the sum
      // over slabs loses almost nothing.
      float comp[kTokRows];
#pragma unroll
      for (int m = 0; m < kTokRows; ++m) comp[m] = 0.f;
      const float* a_s = static_cast<const float*>(p.a_scales);
      const int KS = p.K / 128;
      // FP8_BLOCK128 scales of a slab: lane m holds token row m's a_s[row][kb]
      // (one load per lane, shuffled to every lane in the fold) and every lane
      // the weight tile's b_s[nb][kb]; both are loaded one slab ahead.
      const int arow = mt * kTokRows + lane;
      const bool arow_ok = MODE == kBlock && lane < kTokRows && arow < p.M;
      const float* a_srow = arow_ok ? a_s + static_cast<size_t>(arow) * KS + u0 : nullptr;
      const float* b_srow = MODE == kBlock ? p.b_s + static_cast<size_t>(nt) * KS + u0 : nullptr;
      float a_next = 0.f, b_next = 0.f;
      if (MODE == kBlock) {
        a_next = arow_ok ? ld_nc_f32(a_srow) : 0.f;
        b_next = ld_nc_f32(b_srow);
      }
#pragma unroll 1
      for (int i = 0; i < nslab; ++i) {
        const int pb = i % C::NBUF;
        const float a_cur = a_next, bsc = b_next;
        if (MODE == kBlock && i + 1 < nslab) {
          a_next = arow_ok ? ld_nc_f32(a_srow + i + 1) : 0.f;
          b_next = ld_nc_f32(b_srow + i + 1);
        }
        if ((i & ((1 << pg) - 1)) == 0) {  // the first slab of a group waits for the whole group
          const bool w = mbar_wait(pf_bar(i), pf_par(i), T, p.err, 5);
          if (!__all_sync(0xffffffffu, w)) {
            ok = false;
            break;
          }
        }
        tc_fence_after();
        uint32_t v[kTokRows];
        tmem_ld_tok<TOK>(trow + pb * TOK, v);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pempty_bar[pb]);
#pragma unroll
        for (int m = 0; m < kTokRows; ++m) {
          float term = __uint_as_float(v[m]);
          if (MODE == kBlock) term *= __shfl_sync(0xffffffffu, a_cur, m) * bsc;
          const float yk = term - comp[m];
          const float t = acc[m] + yk;
          comp[m] = (t - acc[m]) - yk;
          acc[m] = t;
        }
      }
    } else {
      const bool w = mbar_wait(&acc_bar, 0, T, p.err, 6);
      if (!__all_sync(0xffffffffu, w)) {
        ok = false;
      } else {
        tc_fence_after();
        uint32_t v[kTokRows];
        tmem_ld_tok<TOK>(trow, v);
        tmem_wait_ld();
#pragma unroll
        for (int m = 0; m < kTokRows; ++m) acc[m] = __uint_as_float(v[m]);
      }
    }
    if (!ok && lane == 0) abort_sh = 1;
    if (p.fused_reduce) {
      // Receive area of split s2: fp32 [S][RM][MV][4], slice s, local row j,
      // tokens 4v..4v+3 (tokens >= Mt are the zero rows of the token tile).
      const int S = p.split;
      const int RM = (128 + S - 1) / S;
      const int Mt = min(kTokRows, p.M - mt * kTokRows);
      const int MV = (Mt + 3) / 4;
      const int lr = qd * 32 + lane;
      const int owner = lr * S / 128;
      const int j = lr - (128 * owner + S - 1) / S;
      cluster_wait();  // phase 1
      const bool rd = mbar_wait_cluster<false>(&ready_bar, 0, T, p.err, 10);
      if (ok && rd) {
        float* dst = reinterpret_cast<float*>(smem + recv_slot(owner) * C::STAGE_BYTES) +
                     ((split * RM + j) * MV) * 4;
#pragma unroll
        for (int v = 0; v < kTokRows / 4; ++v) {
          if (v < MV) {
            const float4 val = make_float4(acc[4 * v], acc[4 * v + 1], acc[4 * v + 2], acc[4 * v + 3]);
            if (owner == split)
              *reinterpret_cast<float4*>(dst + 4 * v) = val;
            else
              st_async_f32x4(dst + 4 * v, owner, val, &recv_bar);
          }
        }
      }
      const bool rv = mbar_wait_cluster<true>(&recv_bar, 0, T, p.err, 11);
      cluster_arrive_relaxed();  // phase 2: everything bound for this CTA has landed
      bar_sync_named(1, 128);   // this CTA's own slice, written by all four warps
      if (ok && rd && rv) {
        const int rlo = (128 * split + S - 1) / S;
        const int myR = (128 * (split + 1) + S - 1) / S - rlo;
        const float* rbuf = reinterpret_cast<const float*>(smem + recv_slot(split) * C::STAGE_BYTES);
        const int et = threadIdx.x - 64;
        for (int e = et; e < myR * MV; e += 128) {
          const int jj = e % myR, v = e / myR;
          float4 a = *reinterpret_cast<const float4*>(rbuf + (jj * MV + v) * 4);
          for (int s2 = 1; s2 < S; ++s2) {
            const float4 b = *reinterpret_cast<const float4*>(rbuf + ((s2 * RM + jj) * MV + v) * 4);
            a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
          }
          const float av[4] = {a.x, a.y, a.z, a.w};
          __nv_bfloat16* yc = p.y + static_cast<size_t>(mt * kTokRows + 4 * v) * p.N + nt * 128 + rlo + jj;
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (4 * v + c < Mt) yc[static_cast<size_t>(c) * p.N] = __float2bfloat16_rn(av[c] * out_scale);
        }
      }
    } else if (ok && p.split > 1) {
#pragma unroll
      for (int m = 0; m < kTokRows; ++m) {
        const int row = mt * kTokRows + m;
        if (row < p.M) p.ws[(static_cast<size_t>(split) * p.M + row) * p.N + nrow] = acc[m];
      }
    } else if (ok) {
#pragma unroll
      for (int m = 0; m < kTokRows; ++m) {
        const int row = mt * kTokRows + m;
        if (row < p.M) p.y[static_cast<size_t>(row) * p.N + nrow] = __float2bfloat16_rn(acc[m] * out_scale);
      }
    }
  }

  // ------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (abort_sh) {
    // Let every copy this CTA started land before its shared memory goes
    // away, and every MMA it issued finish before TMEM is released.
    if (threadIdx.x == 0) {
      for (int it = consumed_sh; it < issued_sh; ++it) {
        mbar_wait(&full_bar[it % STAGES], (it / STAGES) & 1, T, nullptr, 0);
      }
    }
  }
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
  if (p.fused_reduce) cluster_wait();  // phase 2: no peer stores into this CTA any more
}

template <int MODE, int SPS, int STAGES, int TOK>
cudaError_t launch_one(const CUtensorMap& tmap_a, const CUtensorMap& tmap_b, const DecodeParams& p, dim3 grid,
                       cudaStream_t stream) {
  using C = DCfg<MODE, SPS, STAGES, TOK>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(&decode_kernel<MODE, SPS, STAGES, TOK>), C::SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  if (pdl_enabled()) {
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (p.fused_reduce) {
    attrs[na].id = cudaLaunchAttributeClusterDimension;
    attrs[na].val.clusterDim.x = 1;
    attrs[na].val.clusterDim.y = static_cast<unsigned>(p.split);
    attrs[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, decode_kernel<MODE, SPS, STAGES, TOK>, tmap_a, tmap_b, p);
}

// Instantiated configurations: (slabs per stage, stages).
#define FG_DECODE_CONFIGS(X, MODE) \
  X(MODE, 1, 4)                    \
  X(MODE, 1, 5)                    \
  X(MODE, 1, 6)                    \
  X(MODE, 1, 8)                    \
  X(MODE, 2, 3)                    \
  X(MODE, 2, 5)                    \
  X(MODE, 4, 2)

}  // namespace

bool decode_config_supported(const DecodeConfig& c) {
  if (c.mode < kBF16 || c.mode > kMXFP4FP8A) return false;
  if (c.tok == 32) return c.sps == 1 && (c.stages == 4 || c.stages == 5 || c.stages == 6 || c.stages == 8);
  if (c.tok != 16) return false;
  return (c.sps == 1 && (c.stages == 4 || c.stages == 5 || c.stages == 6 || c.stages == 8)) ||
         (c.sps == 2 && (c.stages == 3 || c.stages == 5)) || (c.sps == 4 && c.stages == 2);
}

cudaError_t launch_decode(const DecodeConfig& c, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                          const DecodeParams& p, dim3 grid, cudaStream_t stream) {
  // 32-token tiles: the one-slab-per-stage pipelines only
#define FG_TRY(MODE_, SPS_, ST_)                                                   \
  if (c.mode == MODE_ && c.sps == SPS_ && c.stages == ST_) {                       \
    if constexpr (SPS_ == 1) {                                                     \
      if (c.tok == 32) return launch_one<MODE_, SPS_, ST_, 32>(tmap_a, tmap_b, p, grid, stream); \
    }                                                                              \
    if (c.tok != 16) return cudaErrorInvalidValue;                                 \
    return launch_one<MODE_, SPS_, ST_, 16>(tmap_a, tmap_b, p, grid, stream);      \
  }
  FG_DECODE_CONFIGS(FG_TRY, kBF16)
  FG_DECODE_CONFIGS(FG_TRY, kTensor)
  FG_DECODE_CONFIGS(FG_TRY, kBlock)
  FG_DECODE_CONFIGS(FG_TRY, kMXFP8)
  FG_DECODE_CONFIGS(FG_TRY, kMXFP4)
  FG_DECODE_CONFIGS(FG_TRY, kMXFP8B32)
  FG_DECODE_CONFIGS(FG_TRY, kMXFP4FP8A)
#undef FG_TRY
  return cudaErrorInvalidValue;
}

}  // namespace fg
