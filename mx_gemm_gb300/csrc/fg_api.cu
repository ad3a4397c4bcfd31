// C ABI of the preshuffled-weight GEMM library: argument and shape checks,
// the weight descriptor, the shape-keyed dispatch table, TMA descriptor
// set-up and kernel launches.  Host code only (plus the device error word).
//
// Checks follow the pages' rules: a clear, early error off the supported
// arch (FlyDSL PR "Enable the gmem->LDS async copy for f16/bf16 preshuffle
// GEMM", review reply on the arch guard), K must be a multiple of the scale
// block (aiter PR "FlyDSL split-K preshuffle decode GEMM for small-M
// shapes", Copilot review), never shuffle already-preshuffled weights (same
// PR, last Copilot review), and refuse a tile shape the kernel cannot load
// whole (FlyDSL PR "Migrate kernels to fx.copy / .llvm_ptr", commit
// "Reject tiles whose A tile is only partially loaded").
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <ctime>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/fg.h"
#include "fg_internal.cuh"

namespace fg {

static __device__ uint32_t g_dev_error;

namespace {

thread_local char g_msg[512] = "";
std::atomic<uint64_t> g_timeout_ns{4000000000ull};
std::atomic<int> g_cc_major_override{-1}, g_cc_minor_override{0};

fg_status fail(fg_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
  return s;
}

fg_status cuda_fail(cudaError_t e, const char* what) {
  return fail(FG_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool mode_ok(int mode) { return mode >= FG_BF16 && mode <= FG_MXFP4_FP8A; }

const char* mode_name(int mode) {
  static const char* names[] = {"bf16", "fp8_tensor", "fp8_block128", "mxfp8", "mxfp4", "mxfp8_b32", "mxfp4_fp8a"};
  return mode_ok(mode) ? names[mode] : "?";
}

// Shape rules shared by every call.
fg_status check_nk(int mode, int64_t N, int64_t K) {
  if (N <= 0 || K <= 0) return fail(FG_ERR_SHAPE, "N=%lld and K=%lld must be positive", (long long)N, (long long)K);
  if (N % 128) return fail(FG_ERR_SHAPE, "N=%lld must be a multiple of 128", (long long)N);
  const int64_t need = mode == FG_BF16 ? 64 : (mode == FG_MXFP4 ? 256 : 128);
  if (K % need)
    return fail(FG_ERR_SHAPE, "K=%lld must be a multiple of %lld for %s (whole 128-byte K slabs%s)", (long long)K,
                (long long)need, mode_name(mode),
                (mode == FG_FP8_BLOCK128 || mode == FG_MXFP8) ? " and whole 128-K scale blocks" : "");
  if (N > (int64_t(1) << 24) || K > (int64_t(1) << 20))
    return fail(FG_ERR_SHAPE, "N=%lld or K=%lld too large", (long long)N, (long long)K);
  return FG_OK;
}

fg_status check_arch() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int major = g_cc_major_override.load(), minor = g_cc_minor_override.load();
  if (major < 0) {
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
  }
  if (major != 10 || minor != 3)
    return fail(FG_ERR_UNSUPPORTED_ARCH, "device compute capability %d.%d; this library runs on 10.3 (sm_103a) only",
                major, minor);
  return FG_OK;
}

// Device address of the error word, per device (looked up once each).
uint32_t* dev_error_ptr() {
  static std::mutex mu;
  static uint32_t* ptrs[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dev_error) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<uint32_t*>(p);
  }
  return ptrs[dev];
}

uint64_t fnv1a(const void* data, size_t n, uint64_t h = 1469598103934665603ull) {
  const uint8_t* b = static_cast<const uint8_t*>(data);
  for (size_t i = 0; i < n; ++i) h = (h ^ b[i]) * 1099511628211ull;
  return h;
}

uint64_t desc_check(const fg_bshuf* d) { return fnv1a(d, offsetof(fg_bshuf, check)) ^ 0x5eedf00dcafe1234ull; }

fg_status check_desc(const fg_bshuf* d) {
  if (!d) return fail(FG_ERR_INVALID_ARG, "null weight descriptor");
  if (d->magic != FG_BSHUF_MAGIC || d->version != FG_BSHUF_VERSION || d->check != desc_check(d))
    return fail(FG_ERR_LAYOUT, "weight descriptor was not produced by fg_preshuffle_b (or was modified)");
  return FG_OK;
}

uint64_t sf_image_bytes(int mode, int64_t N, int64_t K) {
  switch (mode) {
    case FG_FP8_TENSOR: return 16;
    case FG_FP8_BLOCK128: return static_cast<uint64_t>(N / 128) * (K / 128) * 4;
    case FG_MXFP8: return static_cast<uint64_t>(N / 128) * ((K / 128 + 3) / 4) * 512;  // four slabs per atom
    case FG_MXFP8_B32:
    case FG_MXFP4_FP8A: return static_cast<uint64_t>(N / 128) * (K / 128) * 512;
    case FG_MXFP4: return static_cast<uint64_t>(N / 128) * (K / 256) * 2 * 512;
    default: return 0;
  }
}

// Workspace of the large-M MX kernel: A's scale atoms, relaid per call.
uint64_t large_mx_workspace(int mode, int64_t M, int64_t K) { return sf_rows_image_bytes(mode, M, K); }

// ------------------------------------------------------------ dispatch

struct TableRow {
  int mode;
  int64_t m_max;  // rows of A up to which the row applies (bucket upper bound)
  int64_t N, K;
  int split, sps, stages;
};

// Exact-shape rows: the decode shapes of the split-K page (K=7168), each
// the fastest (split, slabs per stage, stages) of a sweep on GB300 over
// splits {1,2,4,8} and every instantiated pipeline (per shape: a CUDA graph
// of back-to-back launches cycling through weight copies larger than twice
// the L2).  Anything else falls through to the heuristic below; an explicit
// split_k other than the row's keeps the heuristic's pipeline.
// Every row keeps a CTA within half of an SM's shared memory, so that while
// one GEMM runs, the CTAs of the next launch (programmatic dependent launch)
// find room beside it and start streaming their weights.  Measured on the fp8
// sweep run as one sequence (M=1/16 x N=2048/16384 in turn): the M=16
// N=16384 shape alone is fastest at split 1 with 2 x 5 stages (185 KB a CTA,
// 19.4 us against 20.1 us at split 2, 2 x 3), but in the sequence that
// footprint shut out the next launch and the step took 51.8 us against 49.6.
// Nor may a row let three CTAs share an SM where its 256 CTAs (N=16384,
// split 2) should spread two to an SM over all of them: FP8_BLOCK128 at
// 1 x 4 stages (74 KB, 96 registers) measured 20.7 / 23.7 us (M=1 / 16)
// against 19.5 / 20.8 at 1 x 5 (90 KB).
const TableRow kTable[] = {
    {FG_FP8_TENSOR, 1, 2048, 7168, 8, 2, 3},     {FG_FP8_TENSOR, 16, 2048, 7168, 8, 2, 3},
    {FG_FP8_TENSOR, 1, 2048, 7168, 4, 2, 5},  // an explicit split of 4 at this shape (timed alone)
    {FG_FP8_TENSOR, 1, 16384, 7168, 2, 2, 3},    {FG_FP8_TENSOR, 16, 16384, 7168, 2, 2, 3},
    {FG_FP8_BLOCK128, 1, 2048, 7168, 8, 1, 4},   {FG_FP8_BLOCK128, 16, 2048, 7168, 8, 1, 4},
    {FG_FP8_BLOCK128, 1, 16384, 7168, 2, 1, 5},  {FG_FP8_BLOCK128, 16, 16384, 7168, 2, 1, 5},
    {FG_MXFP8, 1, 2048, 7168, 8, 1, 5},          {FG_MXFP8, 16, 2048, 7168, 8, 1, 4},
    {FG_MXFP8, 1, 16384, 7168, 2, 1, 4},         {FG_MXFP8, 16, 16384, 7168, 2, 1, 4},
    {FG_MXFP4, 1, 2048, 7168, 8, 1, 4},          {FG_MXFP4, 16, 2048, 7168, 8, 1, 4},
    {FG_MXFP4, 1, 16384, 7168, 2, 1, 4},         {FG_MXFP4, 16, 16384, 7168, 2, 1, 4},
    {FG_MXFP8_B32, 1, 2048, 7168, 8, 1, 5},      {FG_MXFP8_B32, 16, 2048, 7168, 8, 1, 4},
    {FG_MXFP8_B32, 1, 16384, 7168, 2, 1, 4},     {FG_MXFP8_B32, 16, 16384, 7168, 2, 1, 4},
    {FG_BF16, 1, 2048, 7168, 8, 1, 6},           {FG_BF16, 16, 2048, 7168, 8, 1, 6},
    {FG_BF16, 1, 16384, 7168, 2, 2, 3},          {FG_BF16, 16, 16384, 7168, 2, 2, 3},
};

int64_t decode_row_limit() { return 32; }

// Splits up to this many reduce inside one thread-block cluster (portable
// cluster size); larger splits take the two-pass workspace + reduce path.
constexpr int kMaxClusterSplit = 8;

// Output tile height of the large-M kernel: 256 x 256 tiles (both 128-row
// halves of A against the same weight slabs in shared memory) for bf16 and
// fp8 per-tensor once there are enough of them to fill the GPU's CTAs;
// 128 x 256 (with the stream-K tail) otherwise and for MX.
// FG_LARGE_TILE=128|256 overrides the choice for bf16 / fp8 (sweep hook).
int large_tile_m(int mode, int64_t M, int64_t N) {
  if (mode != FG_BF16 && mode != FG_FP8_TENSOR) return 128;
  if (const char* ov = getenv("FG_LARGE_TILE")) {
    if (strcmp(ov, "128") == 0) return 128;
    if (strcmp(ov, "256") == 0) return 256;
  }
  const int64_t wide_tiles = ((M + 255) / 256) * (N / 256 + (N % 256 ? 1 : 0));
  return wide_tiles >= sm_count() ? 256 : 128;
}

// Weight tiles per band of the large-M tile walk (the band stays in L2 while
// the row blocks of A go by): 4 for MX (measured 1-2 % faster than 16 on the
// 8-bit MX modes at 4096 x 16384 x 7168, the same for mxfp4), 16 otherwise
// (bands of 4-16 within 1 % for bf16 / fp8).  FG_LARGE_GROUP_N=<tiles>
// overrides it (sweep hook).
int large_group_n(int mode) {
  if (const char* ov = getenv("FG_LARGE_GROUP_N")) {
    const int g = atoi(ov);
    if (g >= 1 && g <= 4096) return g;
  }
  return is_mx(mode) ? 4 : 16;
}

// bf16 / FP8_BLOCK128 decode: slabs per partial-ready commit, as log2 (each
// slab still has its own TMEM partial; a commit stalls the MMA pipe for about
// as long as five 128 x 16 MMAs).  Any of 1, 2, 4 is valid for every
// instantiated pipeline: a group ends at most three slabs after a stage's
// last slab, inside a stage the producer has already filled.  Pairs when the
// grid is at most one CTA per SM (a latency-bound chain of a few slabs per
// CTA: N = 2048, split 8 measured 2-3 % faster); one slab otherwise, since
// a stage is released only when its group is done, which shortens a
// streaming pipeline (N = 16384: pairs 3 % slower, groups of 4 20 % slower).
// FG_DECODE_PGROUP=1|2|4 overrides it (sweep hook).
int decode_pgroup_log(int64_t ctas) {
  if (const char* ov = getenv("FG_DECODE_PGROUP")) {
    if (strcmp(ov, "1") == 0) return 0;
    if (strcmp(ov, "2") == 0) return 1;
    if (strcmp(ov, "4") == 0) return 2;
  }
  return ctas <= sm_count() ? 1 : 0;
}

// Large-M MX on CTA pairs (256 x 256 tiles, two SMs per tile): built and
// correct, but measured 2-6 % slower than the one-CTA 128 x 256 form at the
// pages' M = 4096 shapes (both are bound by the L2 -> SM stream, see the pair
// kernel's file), so the dispatch keeps the one-CTA form.  FG_LARGE_PAIR=1
// selects the pair form (when the device can hold clusters of two).
bool large_pair(int mode, int64_t /*M*/, int64_t /*N*/) {
  if (!is_mx(mode)) return false;
  const char* ov = getenv("FG_LARGE_PAIR");
  return ov && strcmp(ov, "1") == 0 && pair_max_clusters() > 0;
}

fg_status make_plan(int mode, int64_t M, int64_t N, int64_t K, int split_k, fg_plan* out) {
  memset(out, 0, sizeof *out);
  const int64_t Kb = row_bytes(mode, K);
  const int64_t KB = Kb / 128;
  const int64_t tiles_n = N / 128;
  const int tok = M > 16 ? 32 : 16;
  const int64_t tiles_m = (M + tok - 1) / tok;
  // The large-M kernel has no K split; an explicit split_k > 1 keeps any M on
  // the split-K kernel (which covers M in 16-row tiles).
  const bool large = M > decode_row_limit() && large_supported(mode) && split_k <= 1;
  if (large) {
    out->path = 1;
    out->split_k = 1;
    out->tile_n = 256;
    out->stage_slabs = 1;
    if (large_pair(mode, M, N)) {
      out->tile_m = 256;
      out->stages = 5;
      const int64_t tiles = ((M + 255) / 256) * ((N + 255) / 256);
      const int64_t clusters = pair_max_clusters();
      out->ctas = static_cast<int32_t>(2 * (tiles < clusters ? tiles : clusters));
      snprintf(out->name, sizeof out->name, "fg_large_sm103a_%s_m%lld_n%lld_k%lld_pair256x256", mode_name(mode),
               (long long)M, (long long)N, (long long)K);
      return FG_OK;
    }
    out->tile_m = large_tile_m(mode, M, N);
    out->stages = out->tile_m == 256 ? 3 : 4;
    const int64_t tiles = ((M + out->tile_m - 1) / out->tile_m) * (N / 256 + (N % 256 ? 1 : 0));
    out->ctas = static_cast<int32_t>(tiles < sm_count() ? tiles : sm_count());
    snprintf(out->name, sizeof out->name, "fg_large_sm103a_%s_m%lld_n%lld_k%lld_%dx256", mode_name(mode),
             (long long)M, (long long)N, (long long)K, out->tile_m);
    return FG_OK;
  }
  int split = split_k, sps = 1, stages = 4;
  bool from_table = false;
  // 17..32 tokens (and more, where no large-M form exists) take 32-token
  // tiles: the weights stream once per 32 tokens instead of per 16
  for (const TableRow& r : kTable) {
    if (r.mode == mode && r.N == N && r.K == K && M <= r.m_max && (r.m_max == 1 ? M == 1 : M > 1) &&
        (split == 0 || split == r.split)) {
      split = r.split;
      sps = r.sps;
      stages = r.stages;
      from_table = true;
      break;
    }
  }
  if (split == 0) {
    // Heuristic (measured trend on GB300): the small-footprint pipeline (one
    // slab per stage, four stages, up to three CTAs per SM) with the
    // smallest split in {1,2,4,8} that gives at least 1.5 CTAs per SM,
    // keeping >= 4 slabs per split.
    const int64_t want = (static_cast<int64_t>(sm_count()) * 3) / 2;
    split = 1;
    while (split < 8 && tiles_n * tiles_m * split < want && KB / (split * 2) >= 4) split *= 2;
    // fp8 per-tensor and blockscale CTAs of 1 x 4 stages (74 KB, few
    // registers) fit three to an SM.  Where the grid needs between one and two
    // CTAs per SM and each streams a long K range, that lets CTAs pile up
    // three to an SM while others hold one; 1 x 5 (90 KB) keeps two to an SM.
    // Measured (M = 1 / 16, K = 7168): N = 8192 split 4 11.9 / 12.5 us at 1 x 4
    // against 11.1 / 11.5 at 1 x 5; with more CTAs than two per SM hold
    // (N = 12288, K = 5120: 384 CTAs) or a few slabs per CTA (K = 2048 or
    // 4096) 1 x 4 stays ahead (11.4 against 15.5 us; 4.6 against 5.1).
    const int64_t ctas = tiles_n * tiles_m * split;
    if ((mode == FG_FP8_TENSOR || mode == FG_FP8_BLOCK128) && tok == 16 && ctas > sm_count() &&
        ctas <= 2 * static_cast<int64_t>(sm_count()) && KB / split >= 12)
      stages = 5;
  }
  // Sweep hook: FG_DECODE_CONFIG="<slabs per stage>,<stages>" overrides the
  // pipeline shape of every decode launch (refused when not instantiated).
  if (const char* ov = getenv("FG_DECODE_CONFIG")) {
    int a = 0, b = 0;
    char tail = 0;
    if (sscanf(ov, "%d,%d%c", &a, &b, &tail) != 2 || !decode_config_supported(DecodeConfig{mode, a, b, tok}))
      return fail(FG_ERR_INVALID_ARG, "FG_DECODE_CONFIG=\"%s\" is not an instantiated <slabs>,<stages> pair%s", ov,
                  tok == 32 ? " for 32-token tiles (one slab per stage)" : "");
    sps = a;
    stages = b;
  }
  if (split < 1 || split > 16) return fail(FG_ERR_INVALID_ARG, "split_k=%d outside 1..16", split);
  if (split > KB)
    return fail(FG_ERR_SHAPE, "split_k=%d exceeds the %lld 128-byte K slabs of K=%lld", split, (long long)KB,
                (long long)K);
  out->path = 0;
  out->split_k = split;
  out->tile_m = tok;
  out->tile_n = 128;
  out->stage_slabs = sps;
  out->stages = stages;
  out->ctas = static_cast<int32_t>(tiles_n * tiles_m * split);
  out->from_table = from_table ? 1 : 0;
  snprintf(out->name, sizeof out->name, "fg_decode_sm103a_%s_m%lld_n%lld_k%lld_s%d_%dx%d", mode_name(mode),
           (long long)M, (long long)N, (long long)K, split, sps, stages);
  return FG_OK;
}

// Stream-K tail of the large-M bf16 / fp8 kernel: used when the tile count
// leaves a partial last wave.  Fills the schedule fields of p; returns the
// workspace bytes it needs (0 = every tile is processed whole).
uint64_t large_streamk_plan(int mode, int64_t tiles, int64_t KB, int ctas, LargeParams* p, bool wide) {
  if (p) {
    p->dp_rounds = 0;
    p->dp_tiles = 0;
    p->sk_iters = 0;
  }
  if ((mode != FG_BF16 && mode != FG_FP8_TENSOR) || ctas <= 0 || tiles <= ctas || tiles % ctas == 0) return 0;
  const int64_t full_waves = tiles / ctas;
  // 256 x 256 tiles: measured slower (by ~20 us) when every tile is split,
  // i.e. with fewer than two full waves; there the whole-tile schedule is kept
  if (wide && full_waves < 2) return 0;
  const int64_t dp_rounds = full_waves - 1;
  const int64_t sk_tiles = tiles - dp_rounds * ctas;  // >= ctas: every CTA range spans >= one tile of K
  if (p) {
    p->dp_rounds = static_cast<int>(dp_rounds);
    p->dp_tiles = static_cast<int>(dp_rounds * ctas);
    p->sk_iters = sk_tiles * KB;
  }
  return large_streamk_bytes(ctas, wide);
}

// A 64-bit tag per call: a partial's flag matches only the launch that wrote
// it (workspace contents from earlier calls never do), and the CTA that
// consumes a partial clears its flag, so a replay of a captured launch (which
// reuses its tag) waits for its own partial.
uint64_t next_epoch() {
  static std::atomic<uint64_t> counter{0};
  static const uint64_t salt = (static_cast<uint64_t>(reinterpret_cast<uintptr_t>(&counter)) * 0x9E3779B97F4A7C15ull) ^
                               (static_cast<uint64_t>(time(nullptr)) << 32);
  return salt + 2 * (counter.fetch_add(1) + 1);
}

// ---------------------------------------------------------- TMA set-up

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Byte-typed 2-D map over A ([rows][row_bytes]) with a box of box_rows x 128
// bytes in the 128-byte swizzle; rows past the end read as zero.
fg_status make_tmap(CUtensorMap* map, const void* base, int64_t rows, int64_t rbytes, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return fail(FG_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(rbytes), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(rbytes)};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FG_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return FG_OK;
}

// The bf16 output Y [rows][n] as rows of 2n bytes, boxes of 32 rows x 64
// bytes (32 columns) in the 64-byte swizzle: the store map of the large-M MX
// and 128 x 256 bf16 / fp8 kernels.
fg_status make_tmap_out64(CUtensorMap* map, void* y, int64_t rows, int64_t n) {
  auto fn = encode_fn();
  if (!fn) return fail(FG_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(2 * n), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(2 * n)};
  cuuint32_t box[2] = {64, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, y, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FG_ERR_CUDA, "cuTensorMapEncodeTiled (output) failed (%d)", static_cast<int>(r));
  return FG_OK;
}

// Plain (unswizzled) 2-D map over `rows` rows of `rbytes` bytes (a multiple
// of 8, at most 2048) in 8-byte elements, with a box of box_rows whole rows:
// the weight image as 2 KiB rows (a 16 KiB slab is 8 of them) or a scale
// image as 512-byte atoms.  Long rows keep the number of row requests per
// copy small.  Rows past the end read as zero.
fg_status make_tmap_rows(CUtensorMap* map, const void* base, int64_t rows, uint32_t rbytes, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return fail(FG_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(rbytes / 8), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(rbytes)};
  cuuint32_t box[2] = {rbytes / 8, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_INT64, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FG_ERR_CUDA, "cuTensorMapEncodeTiled (rows) failed (%d)", static_cast<int>(r));
  return FG_OK;
}

// MXFP4_FP8A weight image (blocks of 128 rows x 64 bytes of packed e2m1, see
// fg_preshuffle_b) as a 3-D map of 4-bit codes {128 codes, 128 rows,
// N/128 * K/128 blocks}.  Its box is one block, loaded with every 16 codes
// spread over 16 bytes of shared memory (codes in the low 8 bytes) in the
// 128-byte swizzle: the e2m1 operand form of the mxf8f6f4 MMA.  The copy
// counts the 8192 packed bytes of a block on its barrier.  The image must be
// 32-byte aligned.
fg_status make_tmap_fp4w(CUtensorMap* map, const void* base, int64_t N, int64_t K) {
  auto fn = encode_fn();
  if (!fn) return fail(FG_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[3] = {128, 128, static_cast<cuuint64_t>((N / 128) * (K / 128))};
  cuuint64_t strides[2] = {64, 8192};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(FG_ERR_CUDA, "cuTensorMapEncodeTiled (fp4 weight image) failed (%d)", static_cast<int>(r));
  return FG_OK;
}

}  // namespace

bool pdl_enabled() { return getenv("FG_NO_PDL") == nullptr; }

void set_error_message(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
}

cudaError_t ensure_smem_attr(const void* kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::mutex mu;
  static std::vector<std::pair<const void*, int>> done;  // (kernel, device) pairs already set
  std::lock_guard<std::mutex> lock(mu);
  for (const auto& d : done)
    if (d.first == kernel && d.second == dev) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.emplace_back(kernel, dev);
  return e;
}

int sm_count() {
  static std::atomic<int> count[64];  // per device, looked up once (threads may race to the same value)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int c = count[dev].load(std::memory_order_relaxed);
  if (!c) {
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0) c = 148;
    count[dev].store(c, std::memory_order_relaxed);
  }
  return c;
}

}  // namespace fg

using namespace fg;

extern "C" {

int fg_version(void) { return 100; }

const char* fg_status_str(int s) {
  switch (s) {
    case FG_OK: return "FG_OK";
    case FG_ERR_INVALID_ARG: return "FG_ERR_INVALID_ARG";
    case FG_ERR_SHAPE: return "FG_ERR_SHAPE";
    case FG_ERR_ALIGN: return "FG_ERR_ALIGN";
    case FG_ERR_LAYOUT: return "FG_ERR_LAYOUT";
    case FG_ERR_WORKSPACE: return "FG_ERR_WORKSPACE";
    case FG_ERR_UNSUPPORTED_ARCH: return "FG_ERR_UNSUPPORTED_ARCH";
    case FG_ERR_CUDA: return "FG_ERR_CUDA";
    case FG_ERR_TIMEOUT: return "FG_ERR_TIMEOUT";
    default: return "FG_ERR_UNKNOWN";
  }
}

const char* fg_last_error_message(void) { return g_msg; }

void fg_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns < 1000000 ? 1000000 : ns); }

void fg_debug_override_cc(int major, int minor) {
  g_cc_minor_override.store(minor);
  g_cc_major_override.store(major);
}

fg_status fg_preshuffle_b_size(int mode, int64_t N, int64_t K, uint64_t* b_bytes, uint64_t* sf_bytes) {
  if (!mode_ok(mode)) return fail(FG_ERR_INVALID_ARG, "bad mode %d", mode);
  if (!b_bytes || !sf_bytes) return fail(FG_ERR_INVALID_ARG, "null output pointer");
  fg_status s = check_nk(mode, N, K);
  if (s != FG_OK) return s;
  *b_bytes = static_cast<uint64_t>(N) * b_row_bytes(mode, K);
  *sf_bytes = sf_image_bytes(mode, N, K);
  return FG_OK;
}

fg_status fg_preshuffle_b(int mode, const void* B, const void* b_scales, int64_t N, int64_t K, void* b_image,
                          uint64_t b_image_bytes, void* sf_image, uint64_t sf_image_bytes, fg_bshuf* desc_out,
                          void* stream) {
  uint64_t need_b = 0, need_sf = 0;
  fg_status s = fg_preshuffle_b_size(mode, N, K, &need_b, &need_sf);
  if (s != FG_OK) return s;
  if (!B || !b_image || !desc_out) return fail(FG_ERR_INVALID_ARG, "null B, image or descriptor");
  if (mode == FG_BF16 && b_scales) return fail(FG_ERR_INVALID_ARG, "bf16 weights take no scales");
  if (mode != FG_BF16 && (!b_scales || !sf_image)) return fail(FG_ERR_INVALID_ARG, "%s needs B scales and a scale image", mode_name(mode));
  if (!aligned(B, 16) || !aligned(b_image, 16) || (sf_image && !aligned(sf_image, 16)))
    return fail(FG_ERR_ALIGN, "B and the images must be 16-byte aligned");
  if (mode == FG_MXFP4_FP8A && !aligned(b_image, 32))
    return fail(FG_ERR_ALIGN, "the MXFP4_FP8A weight image must be 32-byte aligned");
  if (b_scales && !aligned(b_scales, is_mx(mode) ? 1 : 4))
    return fail(FG_ERR_ALIGN, "fp32 scales must be 4-byte aligned");
  if (b_image_bytes < need_b || sf_image_bytes < need_sf)
    return fail(FG_ERR_WORKSPACE, "image buffers too small (need %llu and %llu bytes)", (unsigned long long)need_b,
                (unsigned long long)need_sf);
  const uint8_t* b0 = static_cast<const uint8_t*>(B);
  const uint8_t* i0 = static_cast<const uint8_t*>(b_image);
  if (b0 < i0 + need_b && i0 < b0 + need_b) return fail(FG_ERR_INVALID_ARG, "B and its image overlap");
  if ((s = check_arch()) != FG_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = mode == FG_MXFP4_FP8A
                      ? launch_block64_b(b0, static_cast<uint8_t*>(b_image), N, b_row_bytes(mode, K), false, st)
                      : launch_relayout_b(b0, static_cast<uint8_t*>(b_image), N, row_bytes(mode, K), false, st);
  if (e != cudaSuccess) return cuda_fail(e, "weight relayout launch");
  if (mode == FG_FP8_TENSOR || mode == FG_FP8_BLOCK128) {
    e = cudaMemcpyAsync(sf_image, b_scales, mode == FG_FP8_TENSOR ? 4 : need_sf, cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "scale copy");
  } else if (is_mx(mode)) {
    e = launch_relayout_sf(mode, static_cast<const uint8_t*>(b_scales), static_cast<uint8_t*>(sf_image), N, K, false,
                           st);
    if (e != cudaSuccess) return cuda_fail(e, "scale relayout launch");
  }
  fg_bshuf d;
  memset(&d, 0, sizeof d);
  d.magic = FG_BSHUF_MAGIC;
  d.version = FG_BSHUF_VERSION;
  d.mode = mode;
  d.tile_rows = 128;
  d.N = N;
  d.K = K;
  d.data = b_image;
  d.sf = mode == FG_BF16 ? nullptr : sf_image;
  d.data_bytes = need_b;
  d.sf_bytes = need_sf;
  d.check = desc_check(&d);
  *desc_out = d;
  return FG_OK;
}

fg_status fg_unshuffle_b(const fg_bshuf* desc, void* B_out, void* b_scales_out, void* stream) {
  fg_status s = check_desc(desc);
  if (s != FG_OK) return s;
  if (!B_out) return fail(FG_ERR_INVALID_ARG, "null output");
  if (!aligned(B_out, 16)) return fail(FG_ERR_ALIGN, "B_out must be 16-byte aligned");
  if ((s = check_arch()) != FG_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e =
      desc->mode == FG_MXFP4_FP8A
          ? launch_block64_b(static_cast<const uint8_t*>(desc->data), static_cast<uint8_t*>(B_out), desc->N,
                             b_row_bytes(desc->mode, desc->K), true, st)
          : launch_relayout_b(static_cast<const uint8_t*>(desc->data), static_cast<uint8_t*>(B_out), desc->N,
                              row_bytes(desc->mode, desc->K), true, st);
  if (e != cudaSuccess) return cuda_fail(e, "inverse relayout launch");
  if (b_scales_out && desc->sf) {
    if (desc->mode == FG_FP8_TENSOR || desc->mode == FG_FP8_BLOCK128) {
      e = cudaMemcpyAsync(b_scales_out, desc->sf, desc->mode == FG_FP8_TENSOR ? 4 : desc->sf_bytes,
                          cudaMemcpyDeviceToDevice, st);
    } else {
      e = launch_relayout_sf(desc->mode, static_cast<const uint8_t*>(desc->sf), static_cast<uint8_t*>(b_scales_out),
                             desc->N, desc->K, true, st);
    }
    if (e != cudaSuccess) return cuda_fail(e, "inverse scale relayout");
  }
  return FG_OK;
}

fg_status fg_gemm_plan(int mode, int64_t M, int64_t N, int64_t K, int split_k, fg_plan* out) {
  if (!mode_ok(mode)) return fail(FG_ERR_INVALID_ARG, "bad mode %d", mode);
  if (!out) return fail(FG_ERR_INVALID_ARG, "null plan");
  if (M < 0) return fail(FG_ERR_SHAPE, "M=%lld is negative", (long long)M);
  if (split_k < 0 || split_k > 16) return fail(FG_ERR_INVALID_ARG, "split_k=%d outside 0..16", split_k);
  fg_status s = check_nk(mode, N, K);
  if (s != FG_OK) return s;
  return make_plan(mode, M > 0 ? M : 1, N, K, split_k, out);
}

fg_status fg_gemm_workspace_size(int mode, int64_t M, int64_t N, int64_t K, int split_k, uint64_t* bytes) {
  if (!bytes) return fail(FG_ERR_INVALID_ARG, "null output");
  fg_plan plan;
  fg_status s = fg_gemm_plan(mode, M, N, K, split_k, &plan);
  if (s != FG_OK) return s;
  if (M == 0) {
    *bytes = 0;
  } else if (plan.path == 1) {
    const int64_t tiles = ((M + plan.tile_m - 1) / plan.tile_m) * (N / 256 + (N % 256 ? 1 : 0));
    *bytes = is_mx(mode) ? large_mx_workspace(mode, M, K)
                         : large_streamk_plan(mode, tiles, row_bytes(mode, K) / 128, plan.ctas, nullptr,
                                              plan.tile_m == 256);
  }
  else
    *bytes = plan.split_k > kMaxClusterSplit ? static_cast<uint64_t>(plan.split_k) * M * N * 4 : 0;
  return FG_OK;
}

fg_status fg_gemm(const void* A, const void* a_scales, int64_t M, const fg_bshuf* b, int mode, int split_k, void* Y,
                  void* workspace, uint64_t workspace_bytes, uint32_t flags, void* stream) {
  fg_status s = check_desc(b);
  if (s != FG_OK) return s;
  if (!mode_ok(mode)) return fail(FG_ERR_INVALID_ARG, "bad mode %d", mode);
  if (b->mode != mode)
    return fail(FG_ERR_LAYOUT, "weight was preshuffled for %s, call asks for %s", mode_name(b->mode), mode_name(mode));
  if (flags & ~(FG_FLAG_DEFER_REDUCE | FG_FLAG_DEBUG_STALL)) return fail(FG_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
  if (M < 0) return fail(FG_ERR_SHAPE, "M=%lld is negative", (long long)M);
  if (M > (int64_t(1) << 24)) return fail(FG_ERR_SHAPE, "M=%lld too large", (long long)M);
  if (split_k < 0 || split_k > 16) return fail(FG_ERR_INVALID_ARG, "split_k=%d outside 0..16", split_k);
  const int64_t N = b->N, K = b->K;
  if ((s = check_nk(mode, N, K)) != FG_OK) return s;
  if (M == 0) return FG_OK;
  if (!A || !Y) return fail(FG_ERR_INVALID_ARG, "null A or Y");
  if (mode != FG_BF16 && !a_scales) return fail(FG_ERR_INVALID_ARG, "%s needs A scales", mode_name(mode));
  if (!aligned(A, 16) || !aligned(Y, 16)) return fail(FG_ERR_ALIGN, "A and Y must be 16-byte aligned");
  if ((mode == FG_FP8_TENSOR || mode == FG_FP8_BLOCK128) && !aligned(a_scales, 4))
    return fail(FG_ERR_ALIGN, "fp32 A scales must be 4-byte aligned");
  fg_plan plan;
  if ((s = make_plan(mode, M, N, K, split_k, &plan)) != FG_OK) return s;
  const int split = plan.split_k;
  const bool defer = (flags & FG_FLAG_DEFER_REDUCE) != 0;
  const bool mx = is_mx(mode);
  const bool fused = plan.path == 0 && split > 1 && split <= kMaxClusterSplit && !defer;
  if (split > 1 && !fused) {
    const uint64_t need = static_cast<uint64_t>(split) * M * N * 4;
    if (!workspace || workspace_bytes < need)
      return fail(FG_ERR_WORKSPACE, "split_k=%d needs a %llu-byte fp32 workspace", split, (unsigned long long)need);
    if (!aligned(workspace, 16)) return fail(FG_ERR_ALIGN, "workspace must be 16-byte aligned");
  } else if (defer) {
    return fail(FG_ERR_INVALID_ARG, "FG_FLAG_DEFER_REDUCE needs split_k > 1");
  }
  if (plan.path == 1 && mx) {
    // the large-M MX kernel reads A's scales as 512-byte atoms relaid per call
    const uint64_t need = large_mx_workspace(mode, M, K);
    if (!workspace || workspace_bytes < need)
      return fail(FG_ERR_WORKSPACE, "large-M %s needs a %llu-byte workspace for the A scale image", mode_name(mode),
                  (unsigned long long)need);
    if (!aligned(workspace, 16)) return fail(FG_ERR_ALIGN, "workspace must be 16-byte aligned");
  }
  if ((s = check_arch()) != FG_OK) return s;
  uint32_t* err = dev_error_ptr();
  if (!err) return fail(FG_ERR_CUDA, "device error word unavailable");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t rb = row_bytes(mode, K);
  CUtensorMap tmap;
  CUtensorMap tmap_b;
  memset(&tmap_b, 0, sizeof tmap_b);
  if (mode == FG_MXFP4_FP8A && (s = make_tmap_fp4w(&tmap_b, b->data, N, K)) != FG_OK) return s;
  cudaError_t e;
  if (plan.path == 1 && mx && plan.tile_m == 256) {
    // CTA-pair form: every operand arrives by tensor copy (their byte counts
    // complete on the even CTA's barriers)
    if ((s = make_tmap(&tmap, A, M, rb, 128)) != FG_OK) return s;
    const int64_t KBb = row_bytes(mode, K) / 128;
    if (mode != FG_MXFP4_FP8A && (s = make_tmap_rows(&tmap_b, b->data, (N / 128) * KBb * 8, 2048, 8)) != FG_OK)
      return s;
    const uint64_t asf_bytes = large_mx_workspace(mode, M, K);
    CUtensorMap tmap_asf, tmap_bsf;
    const uint32_t box = pair_sf_box_rows(mode);
    if ((s = make_tmap_rows(&tmap_asf, workspace, static_cast<int64_t>(asf_bytes / 512), 512, box)) != FG_OK) return s;
    if ((s = make_tmap_rows(&tmap_bsf, b->sf, static_cast<int64_t>(b->sf_bytes / 512), 512, box)) != FG_OK) return s;
    LargeParams p;
    memset(&p, 0, sizeof p);
    p.b_img = static_cast<const uint8_t*>(b->data);
    p.b_sf = static_cast<const uint8_t*>(b->sf);
    p.a_scales = a_scales;
    p.y = static_cast<__nv_bfloat16*>(Y);
    p.err = err;
    p.timeout_ns = g_timeout_ns.load();
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.KB = static_cast<int>(KBb);
    p.tiles_m = static_cast<int>((M + 255) / 256);
    p.tiles_n = static_cast<int>((N + 255) / 256);
    p.group_n = large_group_n(mode);
    p.debug_stall = (flags & FG_FLAG_DEBUG_STALL) ? 1 : 0;
    e = launch_relayout_sf_rows(mode, static_cast<const uint8_t*>(a_scales), static_cast<uint8_t*>(workspace), M, K,
                                st);
    if (e != cudaSuccess) return cuda_fail(e, "A scale relayout launch");
    p.a_sf = static_cast<const uint8_t*>(workspace);
    CUtensorMap tmap_y;
    if ((s = make_tmap_out64(&tmap_y, Y, M, N)) != FG_OK) return s;
    e = launch_large_pair(mode, tmap, tmap_b, tmap_asf, tmap_bsf, tmap_y, p, plan.ctas, st);
    if (e != cudaSuccess) return cuda_fail(e, "large-M pair kernel launch");
    return FG_OK;
  }
  if (plan.path == 1) {
    if ((s = make_tmap(&tmap, A, M, rb, 128)) != FG_OK) return s;
    // every large-M kernel writes Y by tensor store: boxes of 32 rows x 64
    // bf16 (blockscale, 256 x 256) or 32 rows x 32 (MX and 128 x 256 bf16 /
    // fp8, whose stages leave less room)
    CUtensorMap tmap_y;
    const bool box64 = mode == FG_FP8_BLOCK128 || plan.tile_m == 256;
    if ((s = box64 ? make_tmap(&tmap_y, Y, M, N * 2, 32) : make_tmap_out64(&tmap_y, Y, M, N)) != FG_OK) return s;
    LargeParams p;
    memset(&p, 0, sizeof p);
    p.b_img = static_cast<const uint8_t*>(b->data);
    p.b_sf = static_cast<const uint8_t*>(b->sf);
    p.b_s = static_cast<const float*>(b->sf);
    p.a_scales = a_scales;
    p.y = static_cast<__nv_bfloat16*>(Y);
    p.err = err;
    p.timeout_ns = g_timeout_ns.load();
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.KB = static_cast<int>(rb / 128);
    p.tiles_m = static_cast<int>((M + plan.tile_m - 1) / plan.tile_m);
    p.tiles_n = static_cast<int>(N / 256 + (N % 256 ? 1 : 0));
    p.group_n = large_group_n(mode);
    p.debug_stall = (flags & FG_FLAG_DEBUG_STALL) ? 1 : 0;
    p.wide = plan.tile_m == 256 ? 1 : 0;
    if (!mx) {
      // the stream-K tail is an optimisation: only with a large enough workspace
      const uint64_t need =
          large_streamk_plan(mode, static_cast<int64_t>(p.tiles_m) * p.tiles_n, p.KB, plan.ctas, &p, p.wide != 0);
      if (need && workspace && workspace_bytes >= need && aligned(workspace, 16)) {
        p.sk_part = static_cast<float*>(workspace);
        p.sk_flag = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(workspace) + need -
                                                           static_cast<uint64_t>(plan.ctas) * (p.wide ? 64 : 32));
        p.epoch = next_epoch();
      } else {
        large_streamk_plan(mode, 0, 0, 0, &p, false);  // all tiles whole
      }
    }
    if (mx) {
      e = launch_relayout_sf_rows(mode, static_cast<const uint8_t*>(a_scales), static_cast<uint8_t*>(workspace), M, K,
                                  st);
      if (e != cudaSuccess) return cuda_fail(e, "A scale relayout launch");
      p.a_sf = static_cast<const uint8_t*>(workspace);
    }
    e = launch_large(mode, tmap, tmap_b, tmap_y, p, plan.ctas, st);
    if (e != cudaSuccess) return cuda_fail(e, "large-M kernel launch");
    return FG_OK;
  }
  if ((s = make_tmap(&tmap, A, M, rb, static_cast<uint32_t>(plan.tile_m))) != FG_OK) return s;
  DecodeParams p;
  memset(&p, 0, sizeof p);
  p.b_img = static_cast<const uint8_t*>(b->data);
  p.b_sf = static_cast<const uint8_t*>(b->sf);
  p.b_s = static_cast<const float*>(b->sf);
  p.a_scales = a_scales;
  p.ws = static_cast<float*>(workspace);
  p.y = static_cast<__nv_bfloat16*>(Y);
  p.err = err;
  p.timeout_ns = g_timeout_ns.load();
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.KB = static_cast<int>(rb / 128);
  p.split = split;
  p.fused_reduce = fused ? 1 : 0;
  p.debug_stall = (flags & FG_FLAG_DEBUG_STALL) ? 1 : 0;
  p.pgroup_log = decode_pgroup_log(plan.ctas);
  DecodeConfig cfg{mode, plan.stage_slabs, plan.stages, plan.tile_m};
  if (!decode_config_supported(cfg)) return fail(FG_ERR_INVALID_ARG, "no kernel for config %s", plan.name);
  dim3 grid(static_cast<unsigned>(N / 128), static_cast<unsigned>(split),
            static_cast<unsigned>((M + plan.tile_m - 1) / plan.tile_m));
  if (grid.z > 65535) return fail(FG_ERR_SHAPE, "M=%lld too large for the decode path", (long long)M);
  e = launch_decode(cfg, tmap, tmap_b, p, grid, st);
  if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");
  if (split > 1 && !defer && !fused) {
    const float* as = mode == FG_FP8_TENSOR ? static_cast<const float*>(a_scales) : nullptr;
    const float* bs = mode == FG_FP8_TENSOR ? static_cast<const float*>(b->sf) : nullptr;
    e = launch_reduce(p.ws, split, M, N, as, bs, p.y, st);
    if (e != cudaSuccess) return cuda_fail(e, "split-K reduce launch");
  }
  return FG_OK;
}

fg_status fg_gemm_splitk_reduce(const float* ws, int split_k, int64_t M, int64_t N, const float* a_s,
                                const float* b_s, void* Y, void* stream) {
  if (!ws || !Y) return fail(FG_ERR_INVALID_ARG, "null workspace or Y");
  if ((a_s == nullptr) != (b_s == nullptr)) return fail(FG_ERR_INVALID_ARG, "pass both scales or neither");
  if (split_k < 1 || split_k > 16) return fail(FG_ERR_SHAPE, "split_k=%d outside 1..16", split_k);
  if (M < 0 || N < 0 || N % 8) return fail(FG_ERR_SHAPE, "need M >= 0 and N a multiple of 8");
  if (!aligned(ws, 16) || !aligned(Y, 16)) return fail(FG_ERR_ALIGN, "workspace and Y must be 16-byte aligned");
  if ((a_s && !aligned(a_s, 4)) || (b_s && !aligned(b_s, 4))) return fail(FG_ERR_ALIGN, "scales must be 4-byte aligned");
  if (M == 0) return FG_OK;
  fg_status s = check_arch();
  if (s != FG_OK) return s;
  cudaError_t e = launch_reduce(ws, split_k, M, N, a_s, b_s, static_cast<__nv_bfloat16*>(Y), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "reduce launch");
  return FG_OK;
}

fg_status fg_get_error(void) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  uint32_t* p = dev_error_ptr();
  if (!p) return fail(FG_ERR_CUDA, "device error word unavailable");
  uint32_t v = 0;
  if ((e = cudaMemcpy(&v, p, 4, cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail(e, "error word read");
  const uint32_t zero = 0;
  if ((e = cudaMemcpy(p, &zero, 4, cudaMemcpyHostToDevice)) != cudaSuccess) return cuda_fail(e, "error word reset");
  if (v == 0) return FG_OK;
  fail(static_cast<fg_status>(v & 0xff), "kernel error word 0x%x (wait site %u)", v, v >> 8);
  return static_cast<fg_status>(v & 0xff);
}

}  // extern "C"
