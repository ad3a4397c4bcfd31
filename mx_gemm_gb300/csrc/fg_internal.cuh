// Internal declarations shared by the library's translation units (host side
// launchers and the parameter blocks the kernels receive).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace fg {

// kMXFP4FP8A: e4m3 activations with 32-K E8M0 scales against packed e2m1
// weights with 32-K E8M0 scales.
enum Mode : int { kBF16 = 0, kTensor = 1, kBlock = 2, kMXFP8 = 3, kMXFP4 = 4, kMXFP8B32 = 5, kMXFP4FP8A = 6 };

constexpr bool is_mx(int mode) { return mode == kMXFP8 || mode == kMXFP4 || mode == kMXFP8B32 || mode == kMXFP4FP8A; }
// MX scale columns per row: one per 128 K (mxfp8) or per 32 K.
inline int64_t mx_sf_cols(int mode, int64_t K) { return mode == kMXFP8 ? K / 128 : K / 32; }

// Bytes per row of A (and of B, except for kMXFP4FP8A's packed fp4 weights).
inline int elem_bits(int mode) { return mode == kBF16 ? 16 : (mode == kMXFP4 ? 4 : 8); }
inline int64_t row_bytes(int mode, int64_t K) { return K * elem_bits(mode) / 8; }
inline int64_t b_row_bytes(int mode, int64_t K) { return mode == kMXFP4FP8A ? K / 2 : row_bytes(mode, K); }
// 512-byte scale-factor atoms per 128-byte K slab of the weight image.
inline int sf_atoms_per_slab(int mode) { return mode == kMXFP4 ? 2 : (is_mx(mode) ? 1 : 0); }

// Parameters of the split-K decode kernel (weights on the MMA M side,
// tokens on the N side, 16 or 32 tokens per CTA tile).
struct DecodeParams {
  const uint8_t* b_img;    // weight image
  const uint8_t* b_sf;     // MX: weight scale image (atoms)
  const float* b_s;        // FP8_TENSOR: scalar; FP8_BLOCK128: [N/128][K/128]
  const void* a_scales;    // FP8_TENSOR: fp32 scalar; BLOCK128: fp32 [M][K/128]; MX: E8M0 [M][K/blk]
  float* ws;               // [split][M][N] fp32 partials (split > 1)
  __nv_bfloat16* y;        // [M][N] (split == 1)
  uint32_t* err;           // device error word
  uint64_t timeout_ns;     // limit of every wait
  int M, N, K;
  int KB;                  // 128-byte slabs per row
  int split;
  int fused_reduce;        // split > 1: the split CTAs of a tile form a cluster and reduce in DSMEM
  int debug_stall;
  int pgroup_log;          // bf16 / FP8_BLOCK128: one partial-ready commit per 2^pgroup_log slabs (0..2)
};

struct DecodeConfig {
  int mode;
  int sps;     // slabs per stage
  int stages;  // pipeline depth
  int tok;     // token rows per CTA tile: 16, or 32 (one-slab-per-stage pipelines only)
};

// Parameters of the large-M kernel (A on the MMA M side, 128 x 256 tiles).
struct LargeParams {
  const uint8_t* b_img;
  const uint8_t* b_sf;     // MX weight scale image
  const uint8_t* a_sf;     // MX activation scale image (atoms per 128-row tile of A)
  const float* b_s;        // FP8_TENSOR scalar
  const void* a_scales;    // FP8_TENSOR scalar / MX E8M0 [M][K/blk]
  __nv_bfloat16* y;
  uint32_t* err;
  uint64_t timeout_ns;
  int M, N, K;
  int KB;
  int tiles_m, tiles_n;
  int debug_stall;
  int wide;                // bf16 / fp8 per-tensor: 256 x 256 tiles (tiles_m counts 256-row blocks)
  int group_n;             // weight tiles per band of the tile walk
  // Stream-K tail (bf16 / fp8 per-tensor; sk_iters == 0: all tiles whole).
  // Each CTA first takes dp_rounds whole tiles (c, c + G, ...), then an equal
  // contiguous range of the remaining K iterations.  A tile split between
  // CTAs c and c+1 is finished by c (which holds its first iterations and
  // reaches them last) after c+1 published its fp32 partial.
  int dp_rounds;
  int dp_tiles;
  long long sk_iters;
  float* sk_part;                  // [G][256 columns][128 rows] fp32 ([G][2 halves][256][128] when wide)
  unsigned long long* sk_flag;     // [G][4 warps] ([G][8 warps] when wide): equals `epoch` once published
  unsigned long long epoch;
};

// Bytes of the optional stream-K workspace of the large-M bf16 / fp8 kernel
// (128 x 256 or, wide, 256 x 256 tiles).
uint64_t large_streamk_bytes(int ctas, bool wide);

bool decode_config_supported(const DecodeConfig& c);
// Kernels are launched with programmatic dependent launch (they may start
// while the previous kernel of the stream finishes; they wait for it before
// touching anything it could write or read).  tmap_b: kMXFP4FP8A's weight
// image as a 3-D map of 4-bit codes {128 codes, 128 rows, N/128 * K/128
// blocks}, loaded one block at a time with each 16 codes spread over 16
// bytes of shared memory (unused by the other modes).
cudaError_t launch_decode(const DecodeConfig& cfg, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                          const DecodeParams& p, dim3 grid, cudaStream_t stream);

bool large_supported(int mode);
// CTA-pair form of the large-M MX kernel (256 x 256 tiles on two SMs):
// clusters of two that fit on the device at once (0 if unknown), the atom
// count of one scale box (the atoms of one 128-row block and slab), and the
// launch.  tmap_b: the weight image as 2 KiB rows of 8-byte elements (box 8
// rows) or, for kMXFP4FP8A, the 3-D map above; tmap_asf / tmap_bsf: the A and
// weight scale images as 512-byte rows (one atom each); tmap_y: Y as rows of
// 2N bytes, boxes of 32 rows x 64 bytes, 64-byte swizzle (tensor stores).
int pair_max_clusters();
uint32_t pair_sf_box_rows(int mode);
cudaError_t launch_large_pair(int mode, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b,
                              const CUtensorMap& tmap_asf, const CUtensorMap& tmap_bsf, const CUtensorMap& tmap_y,
                              const LargeParams& p, int ctas, cudaStream_t stream);
// One-CTA large-M kernels.  tmap_b: the MXFP4_FP8A weight image's map
// (unused otherwise).  tmap_y: the output Y as rows of 2N bytes; all these
// kernels write their bf16 tiles by tensor store -- kBlock and the 256 x 256
// form (p.wide): boxes of 32 rows x 128 bytes, 128-byte swizzle; the MX
// modes and the 128 x 256 bf16 / fp8 form: boxes of 32 rows x 64 bytes,
// 64-byte swizzle.
cudaError_t launch_large(int mode, const CUtensorMap& tmap_a, const CUtensorMap& tmap_b, const CUtensorMap& tmap_y,
                         const LargeParams& p, int ctas, cudaStream_t stream);

cudaError_t launch_relayout_b(const uint8_t* src, uint8_t* dst, int64_t N, int64_t Kb, bool inverse,
                              cudaStream_t stream);
cudaError_t launch_relayout_sf(int mode, const uint8_t* src, uint8_t* dst, int64_t N, int64_t K, bool inverse,
                               cudaStream_t stream);
// kMXFP4FP8A weight image: packed fp4 [N][Kb] <-> 128-row x 64-byte blocks.
cudaError_t launch_block64_b(const uint8_t* src, uint8_t* dst, int64_t N, int64_t Kb, bool inverse,
                             cudaStream_t stream);
uint64_t sf_rows_image_bytes(int mode, int64_t rows, int64_t K);
cudaError_t launch_relayout_sf_rows(int mode, const uint8_t* src, uint8_t* dst, int64_t rows, int64_t K,
                                    cudaStream_t stream);
cudaError_t launch_reduce(const float* ws, int split, int64_t M, int64_t N, const float* a_s, const float* b_s,
                          __nv_bfloat16* y, cudaStream_t stream);

int sm_count();

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per (kernel, device) pair; thread-safe.
cudaError_t ensure_smem_attr(const void* kernel, int bytes);

// Programmatic dependent launch is on unless FG_NO_PDL is set (a sweep hook
// for measuring what the overlap is worth).
bool pdl_enabled();

}  // namespace fg
