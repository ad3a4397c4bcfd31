/*
 * fg.h -- C ABI of the GB300 (sm_103a) preshuffled-weight GEMM library.
 *
 *   Y[M,N] = dequant(A[M,K]) . dequant(B[N,K])^T,  fp32 accumulation, bf16 Y.
 *
 * Sources of the operation (titles of the pages that state the method):
 *  - aiter PR "FlyDSL split-K preshuffle decode GEMM for small-M shapes
 *    (FP8 + MX, gfx950/gfx942)", sections Summary and What's included: the
 *    two-pass split-K GEMM for small M (fp32 partials in a workspace, then a
 *    reduce that downcasts once at the final store), the direct-output
 *    epilogue for split_k = 1, the three scale modes (FP8 per-tensor, FP8
 *    128-block blockscale, MX: mxfp8 with one E8M0 per 128 K, mxfp4 with
 *    one E8M0 per 32 K; the OCP-standard 32-element mxfp8 block is offered
 *    beside the pages' 128-element one), the weight/scale preshuffle helpers and the
 *    shape-keyed dispatch; Copilot review: K must be a multiple of the scale
 *    block, and already-preshuffled weights must not be shuffled again.
 *  - FlyDSL PR "Enable the gmem->LDS async copy for f16/bf16 preshuffle
 *    GEMM", Summary and Performance: the large-M bf16 preshuffle GEMM
 *    (M=54560, N=K=8192), and the early, clear error off the supported arch.
 *  - FlyDSL PR "Migrate kernels to fx.copy / .llvm_ptr; expand
 *    kernel-code-cleanup skill", Validation and the later commit "Reject
 *    tiles whose A tile is only partially loaded": the fp8 large-M shape
 *    (M=N=4096, K=8192) and the rule that a shape the kernel cannot load
 *    whole is refused up front instead of computed wrongly.
 *
 * Conventions for every call:
 *  - Device pointers are caller-owned (allocate them with any allocator).
 *    The library never allocates, frees or synchronises device memory, and
 *    never writes outside the buffers it is given.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Launches are asynchronous; errors found on the host are
 *    returned before anything is launched.  A kernel that gives up on a
 *    bounded wait records FG_ERR_TIMEOUT in a device word that
 *    fg_get_error() returns.
 *  - Only compute capability 10.3 devices are accepted
 *    (FG_ERR_UNSUPPORTED_ARCH otherwise).
 *  - Layouts are row-major.  A: [M][K] bf16 | e4m3 bytes | packed e2m1
 *    ([M][K/2] bytes, low nibble = even k).  B likewise [N][K] (for
 *    MXFP4_FP8A, A is e4m3 [M][K] and B packed e2m1 [N][K/2]).
 *    Y: [M][N] bf16.  Workspace: [split_k][M][N] fp32.
 *  - Shapes: N % 128 == 0; K * element bits / 8 must be a multiple of 128
 *    bytes (K % 64 for bf16, K % 128 for fp8 and MXFP4_FP8A, K % 256 for
 *    mxfp4); the 128-K scale blocks of FP8_BLOCK128 / MXFP8 and the 32-K
 *    blocks of MXFP4 then divide K exactly.  M >= 0 (M == 0 is a no-op).
 */
#ifndef FG_H
#define FG_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FG_API __attribute__((visibility("default")))
#else
#define FG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fg_status {
  FG_OK = 0,
  FG_ERR_INVALID_ARG = 1,      /* null pointer, bad enum, bad flag, bad split_k   */
  FG_ERR_SHAPE = 2,            /* N, K or M violate the shape rules above          */
  FG_ERR_ALIGN = 3,            /* a pointer is not 16-byte aligned (4 for scales)  */
  FG_ERR_LAYOUT = 4,           /* descriptor is not one fg_preshuffle_b made, or   */
                               /* its mode differs from the call's                 */
  FG_ERR_WORKSPACE = 5,        /* workspace missing or too small                   */
  FG_ERR_UNSUPPORTED_ARCH = 6, /* current device is not compute capability 10.3    */
  FG_ERR_CUDA = 7,             /* a CUDA runtime/driver call failed                */
  FG_ERR_TIMEOUT = 8           /* a kernel gave up on a bounded wait               */
} fg_status;

typedef enum fg_mode {
  FG_BF16 = 0,         /* bf16 A and B, no scales                                   */
  FG_FP8_TENSOR = 1,   /* e4m3 A and B; fp32 scalars a_s, b_s                       */
  FG_FP8_BLOCK128 = 2, /* e4m3; a_s fp32 [M][K/128]; b_s fp32 [N/128][K/128]        */
  FG_MXFP8 = 3,        /* e4m3; E8M0 a_sf [M][K/128], b_sf [N][K/128]               */
  FG_MXFP4 = 4,        /* packed e2m1; E8M0 a_sf [M][K/32], b_sf [N][K/32]          */
  FG_MXFP8_B32 = 5,    /* e4m3; E8M0 a_sf [M][K/32], b_sf [N][K/32] (OCP MX block)  */
  FG_MXFP4_FP8A = 6    /* A e4m3, E8M0 a_sf [M][K/32]; B packed e2m1, E8M0 b_sf     */
                       /* [N][K/32] ("MXFP4 fp8-A": fp8 activations, fp4 weights)   */
} fg_mode;

/* fg_gemm flags */
#define FG_FLAG_DEFER_REDUCE 0x1u /* split_k > 1: stop after writing the fp32 partials */
#define FG_FLAG_DEBUG_STALL 0x40000000u /* test hook: the MMA issuer waits on a barrier */
                                        /* nothing arrives at, so every bounded wait    */
                                        /* runs out and the call ends in FG_ERR_TIMEOUT */

#define FG_BSHUF_MAGIC 0x31424746u /* "FGB1" */
#define FG_BSHUF_VERSION 1u

/*
 * Descriptor of a preshuffled weight, filled by fg_preshuffle_b.  It points
 * at caller-owned device buffers and carries a check word over its fields;
 * fg_gemm accepts only descriptors whose check word matches (a raw pointer,
 * a hand-made or edited descriptor, or one of another mode is rejected with
 * FG_ERR_LAYOUT).  Keep the buffers alive while the descriptor is used.
 *
 * Weight image layout: B viewed as N rows of Kb bytes (Kb = 2K bf16, K fp8,
 * K/2 fp4) cut into slabs of 128 rows x 128 bytes, slab (nb, kb) at index
 * nb*(Kb/128)+kb (16 KiB each); in a slab, 16-byte chunk c of row r sits at
 * byte r*128 + ((c ^ (r%8))*16) -- the image a 128-byte-swizzled K-major
 * tensor-core operand has in shared memory, so one pipeline stage of one
 * 128-row tile is one contiguous copy.  MXFP4_FP8A instead keeps the packed
 * fp4 bytes (Kb = K/2) in unswizzled blocks of 128 rows x 64 bytes (128 K),
 * block (nb, kb) at index nb*(K/128)+kb, row r at byte r*64; the image must
 * be 32-byte aligned.  The kernels load one block per tensor copy that puts
 * every 16 codes in the low half of a 16-byte shared-memory chunk (the
 * e2m1 operand form of the fp8/fp6/fp4 block-scaled MMA), so HBM moves
 * only the packed bytes.
 *
 * Scale image (sf): FP8_TENSOR: the fp32 b_s (16 bytes reserved);
 * FP8_BLOCK128: b_s fp32 [N/128][K/128] unchanged; MXFP8_B32 / MXFP4_FP8A
 * (one atom per 128 K) / MXFP4 (two atoms per 256 K): for each 128-row tile
 * and slab, atoms of 512 bytes, atom byte 16*(r%32) + 4*(r/32) + j = the
 * E8M0 of row r for the j-th 32-K block the atom covers; MXFP8 (one scale
 * per 128 K): one atom per four consecutive 128-K slabs of a 128-row tile,
 * byte j of row r = the E8M0 of slab 4g + j (zero past the last slab);
 * BF16: none.
 */
typedef struct fg_bshuf {
  uint32_t magic;
  uint32_t version;
  int32_t mode;
  int32_t tile_rows; /* 128 */
  int64_t N;
  int64_t K;
  void* data;        /* device: weight image, data_bytes long */
  void* sf;          /* device: scale image, sf_bytes long (NULL for BF16) */
  uint64_t data_bytes;
  uint64_t sf_bytes;
  uint64_t check;
} fg_bshuf;

/* Chosen kernel configuration for one GEMM shape (fg_gemm_plan). */
typedef struct fg_plan {
  int32_t path;        /* 0 = split-K decode kernel (weights on the MMA M side), 1 = large-M kernel */
  int32_t split_k;     /* K splits (1 = direct bf16 output, no workspace)                          */
  int32_t tile_m;      /* rows of A per CTA tile                                                   */
  int32_t tile_n;      /* rows of B per CTA tile                                                   */
  int32_t stage_slabs; /* 128-byte K slabs per pipeline stage                                      */
  int32_t stages;      /* pipeline depth                                                           */
  int32_t ctas;        /* CTAs launched by the main kernel                                         */
  int32_t from_table;  /* 1 if an exact dispatch-table row matched, 0 if the heuristic chose       */
  char name[96];       /* kernel/config name: arch, mode, shape identity                          */
} fg_plan;

/* Library version (major*10000 + minor*100 + patch). */
FG_API int fg_version(void);

/* Human-readable name of a status code. */
FG_API const char* fg_status_str(int status);

/* Message with the details of the last error returned on this host thread. */
FG_API const char* fg_last_error_message(void);

/*
 * Sizes of the buffers fg_preshuffle_b writes for a weight of the given mode
 * and shape: the weight image (N*Kb bytes) and the scale image (0 for BF16).
 * Errors: FG_ERR_INVALID_ARG (mode, null outputs), FG_ERR_SHAPE.
 */
FG_API fg_status fg_preshuffle_b_size(int mode, int64_t N, int64_t K, uint64_t* b_bytes, uint64_t* sf_bytes);

/*
 * One-time relayout of the weight B[N][K] (and of its scales) into the
 * images described above; fills *desc_out.  b_scales: FP8_TENSOR: device
 * fp32 scalar; FP8_BLOCK128: device fp32 [N/128][K/128]; MX: device uint8
 * E8M0 [N][K/128] (MXFP8) or [N][K/32] (MXFP4, MXFP8_B32, MXFP4_FP8A); BF16: must be NULL.  B and the images must
 * not overlap.  Errors: INVALID_ARG, SHAPE, ALIGN (16 bytes for B and the
 * images -- 32 for the MXFP4_FP8A weight image --, 4 for fp32 scales),
 * WORKSPACE (an image buffer smaller than
 * fg_preshuffle_b_size says), UNSUPPORTED_ARCH, CUDA.
 */
FG_API fg_status fg_preshuffle_b(int mode, const void* B, const void* b_scales, int64_t N, int64_t K, void* b_image,
                          uint64_t b_image_bytes, void* sf_image, uint64_t sf_image_bytes, fg_bshuf* desc_out,
                          void* stream);

/*
 * Inverse of fg_preshuffle_b: writes B[N][K] (and, if b_scales_out is not
 * NULL, the scales in the caller's layout) back from the images.  Used to
 * check that the relayout is a bijection.  Errors as fg_preshuffle_b, plus
 * FG_ERR_LAYOUT for a bad descriptor.
 */
FG_API fg_status fg_unshuffle_b(const fg_bshuf* desc, void* B_out, void* b_scales_out, void* stream);

/*
 * The configuration fg_gemm would use (split_k = 0 lets the dispatch table
 * choose; a positive split_k is taken as given).  Errors: INVALID_ARG, SHAPE.
 */
FG_API fg_status fg_gemm_plan(int mode, int64_t M, int64_t N, int64_t K, int split_k, fg_plan* out);

/*
 * Workspace bytes a call of fg_gemm without FG_FLAG_DEFER_REDUCE needs for
 * this shape and split: 0 when the split resolves to 1 or to at most 8 (the
 * splits of a tile then reduce inside one thread-block cluster, with no
 * global scratch), split_k*M*N*4 for larger splits, and the A scale image
 * for large-M MX shapes.  For large-M bf16 / fp8 shapes whose tiles leave a
 * partial last wave it is the optional stream-K workspace (fp32 partial
 * tiles of the CTAs that split a tile): with less, those shapes still run,
 * every tile whole.  A call with FG_FLAG_DEFER_REDUCE always needs
 * split_k*M*N*4 bytes.
 */
FG_API fg_status fg_gemm_workspace_size(int mode, int64_t M, int64_t N, int64_t K, int split_k, uint64_t* bytes);

/*
 * Y = dequant(A) . dequant(B)^T for the preshuffled weight `b`.
 *  A        device [M][K] codes (layout per mode, see top).
 *  a_scales FP8_TENSOR: device fp32 scalar; FP8_BLOCK128: fp32 [M][K/128];
 *           MXFP8: uint8 E8M0 [M][K/128]; MXFP4, MXFP8_B32, MXFP4_FP8A:
 *           uint8 E8M0 [M][K/32];
 *           BF16: ignored (pass NULL).
 *  mode     must equal b->mode (FG_ERR_LAYOUT otherwise).
 *  split_k  0 = dispatch chooses; 1..16 = number of K splits.  Split s takes
 *           the contiguous run of 128-byte K slabs [s*q + min(s,r), ...) of
 *           length q + (s < r), q = U/S, r = U%S, U = Kb/128 (for
 *           MXFP4_FP8A, U = K/128: the slabs of the fp8 A).
 *  Y        device bf16 [M][N].
 *  workspace / workspace_bytes: as fg_gemm_workspace_size says; may be
 *           NULL when that is 0.  With FG_FLAG_DEFER_REDUCE (or a split
 *           above 8) it holds fp32 [split_k][M][N], per split the partial
 *           sum: unscaled for FP8_TENSOR (the per-tensor scale is applied
 *           once, in the reduce), fully scaled for the other modes.  Splits
 *           of 2..8 without the flag sum their partials in split order
 *           inside one thread-block cluster, which gives the same bits as
 *           the workspace + fg_gemm_splitk_reduce pair.
 *  flags    FG_FLAG_DEFER_REDUCE: leave the partials in the workspace and do
 *           not write Y (call fg_gemm_splitk_reduce later).
 * Errors: INVALID_ARG, SHAPE, ALIGN, LAYOUT, WORKSPACE, UNSUPPORTED_ARCH, CUDA.
 */
FG_API fg_status fg_gemm(const void* A, const void* a_scales, int64_t M, const fg_bshuf* b, int mode, int split_k,
                  void* Y, void* workspace, uint64_t workspace_bytes, uint32_t flags, void* stream);

/*
 * Second pass of the split-K GEMM:
 *   Y[m][n] = bf16_rne( a_s * b_s * sum_{s=0}^{split_k-1} ws[s][m][n] )
 * summed in split order; a_s and b_s are device fp32 scalars (both NULL
 * means a factor of 1; exactly one NULL is an error).  Errors: INVALID_ARG,
 * SHAPE (N % 8 != 0, split_k outside 1..16), ALIGN, UNSUPPORTED_ARCH, CUDA.
 */
FG_API fg_status fg_gemm_splitk_reduce(const float* ws, int split_k, int64_t M, int64_t N, const float* a_s,
                                const float* b_s, void* Y, void* stream);

/*
 * fg_gemm without a caller workspace (no counterpart in the pages).  For
 * callers that cannot allocate device memory while they run -- a serving
 * loop whose buffers are all sized at start-up (cudaMalloc can synchronise
 * the device and stall every stream), or a plug-in whose host framework owns
 * all device memory and offers no allocator.  Whatever fg_gemm would keep in
 * a caller workspace goes to one 8 MiB array that the library keeps in every
 * device's memory until the process exits; this call allocates nothing.
 * The array holds, depending on the call:
 *  - the fp32 split-K partials of a split above 8 (splits 9..16):
 *    split_k * M * N * 4 bytes, refused with FG_ERR_WORKSPACE (before
 *    anything is launched) when above 8 MiB;
 *  - the A scale image of a large-M MX call (M > 32, MX modes):
 *    M/128 rounded up * K/128 * 512 bytes (twice that for MXFP4; a quarter,
 *    rounded up, for MXFP8), refused with FG_ERR_WORKSPACE when above 8 MiB;
 *  - the optional stream-K partials and flags of a large-M bf16 / fp8 call,
 *    when they fit (about 128 KiB per CTA for 128 x 256 tiles, 256 KiB for
 *    256 x 256 tiles; more than 8 MiB once the grid has more than 63 / 31
 *    CTAs).  When they do not fit the call is not refused: every tile then
 *    runs whole, as fg_gemm does with a smaller workspace.
 * Splits of 2..8 and split 1 need no scratch.
 *  - Arguments as fg_gemm, minus the workspace.  FG_FLAG_DEFER_REDUCE is
 *    refused (FG_ERR_INVALID_ARG): the partials would stay in the private
 *    scratch.
 *  - The first call on a device looks up the scratch's device address (once
 *    per device, with that device current); make that first call before any
 *    stream capture.
 *  - All calls share the one array and it keeps the last call's contents.
 *    Nothing in it has to start at zero (every split writes its whole
 *    partial before the reduce reads it, every large-M MX call rewrites its
 *    whole A scale image, a partial's flag matches only the launch that
 *    wrote it and is cleared once read), but two calls that overlap on the
 *    GPU (e.g. on two streams) race on it: serialise them.
 * Errors: as fg_gemm.
 */
FG_API fg_status fg_gemm_noalloc(const void* A, const void* a_scales, int64_t M, const fg_bshuf* b, int mode,
                                 int split_k, void* Y, uint32_t flags, void* stream);

/*
 * Synchronises the current device and returns (and clears) the error word
 * the library's kernels write when a bounded wait runs out: FG_OK or
 * FG_ERR_TIMEOUT.  A failed synchronisation returns FG_ERR_CUDA.
 */
FG_API fg_status fg_get_error(void);

/*
 * Limit for every wait inside the kernels, in nanoseconds (default 4e9).
 * Values below 1e6 (1 ms) are raised to 1 ms: a wait that gives up must not
 * end while the cluster peers' shared-memory stores it waits for (a few
 * microseconds apart) may still be on their way.
 */
FG_API void fg_set_wait_timeout_ns(uint64_t ns);

/*
 * Test hook: make the architecture check see the given compute capability
 * instead of the device's (major < 0 restores the real one).  Lets host
 * tests reach FG_ERR_UNSUPPORTED_ARCH without a second kind of GPU.
 */
FG_API void fg_debug_override_cc(int major, int minor);

#ifdef __cplusplus
}
#endif

#endif /* FG_H */
