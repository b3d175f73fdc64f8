// api.cu -- the C ABI declared in include/sgemm.h: argument checks, the
// degenerate cases, dispatch by shape / layout / alignment, TMA descriptor
// encoding and the launches.  Everything here is host code except the device
// status word.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <mutex>

#include "dispatch.h"
#include "internal.h"
#include "sgemm.h"

namespace {
// Device status word: a kernel that gives up a bounded wait records
// SGEMM_ERR_DEVICE_TIMEOUT here (one copy per device that loads the library).
__device__ int g_device_status;
sg::DeviceState g_dev[sg::kMaxDevices];
}  // namespace

namespace sg {

std::atomic<uint64_t> g_wait_budget_ns{kDefaultWaitBudgetNs};
thread_local int t_last_launches = 0;

// SGEMM_VERBOSE=1 in the environment: every CUDA-core product prints the plan
// it queued (kernel form, tile, grid, split) to stderr.
bool verbose() {
  static const bool v = [] {
    const char *e = std::getenv("SGEMM_VERBOSE");
    return e && e[0] && !(e[0] == '0' && e[1] == '\0');
  }();
  return v;
}

// Returns the current device's state (initialised once per device) or null.
DeviceState *device_state(sgemm_status_t *why) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    *why = SGEMM_ERR_UNSUPPORTED;
    return nullptr;
  }
  DeviceState &d = g_dev[dev];
  std::call_once(d.once, [&d, dev]() {
    cudaError_t e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess) e = cudaGetSymbolAddress(reinterpret_cast<void **>(&d.status), g_device_status);
    // SGEMM_SCRATCH_LIMIT=<bytes>: the initial scratch limit of every device
    if (const char *env = std::getenv("SGEMM_SCRATCH_LIMIT")) {
      char *end = nullptr;
      const unsigned long long v = std::strtoull(env, &end, 10);
      if (end != env && *end == '\0') d.limit.store(v);
    }
    d.err = e;
    if (e != cudaSuccess) cudaGetLastError();
  });
  if (d.err != cudaSuccess) {
    *why = SGEMM_ERR_UNSUPPORTED;
    return nullptr;
  }
  if (d.cc_major != 10 || d.cc_minor != 3) {
    *why = SGEMM_ERR_UNSUPPORTED;
    return nullptr;
  }
  cudaGetLastError();   // a stale error of someone else's call is not ours
  return &d;
}

const SimtKernelInfo *kernel_info(DeviceState &d, int producer, int ta, int tb, int tile, int csk) {
  const int c = csk ? 1 : 0;
  std::call_once(d.kinfo_once[producer][ta][tb][tile][c], [&]() {
    d.kinfo_err[producer][ta][tb][tile][c] =
        simt_entry(producer, ta, tb, tile, c).info(&d.kinfo[producer][ta][tb][tile][c]);
    if (d.kinfo_err[producer][ta][tb][tile][c] != cudaSuccess) cudaGetLastError();
  });
  if (d.kinfo_err[producer][ta][tb][tile][c] != cudaSuccess) return nullptr;
  return &d.kinfo[producer][ta][tb][tile][c];
}

const TcKernelInfo *tc_kernel_info(DeviceState &d, int ta, int tb) {
  std::call_once(d.tcinfo_once[ta][tb], [&]() {
    d.tcinfo_err[ta][tb] = tc3_entry(ta, tb).info(&d.tcinfo[ta][tb]);
    if (d.tcinfo_err[ta][tb] != cudaSuccess) cudaGetLastError();
  });
  if (d.tcinfo_err[ta][tb] != cudaSuccess) return nullptr;
  return &d.tcinfo[ta][tb];
}

const TcKernelInfo *tc_kernel_info_pair(DeviceState &d, int bn, bool fold_a, bool fold_b) {
  const int i = bn == 256 ? 1 : 0, fa = fold_a ? 1 : 0, fb = fold_b ? 1 : 0;
  std::call_once(d.tcpair_once[i][fa][fb], [&]() {
    d.tcpair_err[i][fa][fb] = tc3_pair_entry(bn, fold_a, fold_b).info(&d.tcpair[i][fa][fb]);
    if (d.tcpair_err[i][fa][fb] != cudaSuccess) cudaGetLastError();
  });
  return d.tcpair_err[i][fa][fb] == cudaSuccess ? &d.tcpair[i][fa][fb] : nullptr;
}

const TcKernelInfo *tc_kernel_info_presplit(DeviceState &d, int bn) {
  if (bn == 256) {
    std::call_once(d.tcpre_wide_once, [&]() {
      d.tcpre_wide_err = tc3_presplit_entry(256).info(&d.tcpre_wide);
      if (d.tcpre_wide_err != cudaSuccess) cudaGetLastError();
    });
    return d.tcpre_wide_err == cudaSuccess ? &d.tcpre_wide : nullptr;
  }
  std::call_once(d.tcpre_once, [&]() {
    d.tcpre_err = tc3_presplit_entry(128).info(&d.tcpre);
    if (d.tcpre_err != cudaSuccess) cudaGetLastError();
  });
  return d.tcpre_err == cudaSuccess ? &d.tcpre : nullptr;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// 2-D FP32 tensor map over a row-major matrix of `rows` x `cols` (row stride
// ld elements), box box_cols x box_rows, zero fill outside.
// The last few 2-D maps encoded on this thread: a map depends only on these
// arguments, so repeated calls on the same buffers skip the driver encode.
struct TmapCacheEntry {
  const float *base = nullptr;
  int64_t rows = 0, cols = 0, ld = 0;
  int box_cols = 0, box_rows = 0;
  bool swizzle128 = false, valid = false;
  CUtensorMap map;
};
constexpr int kTmapCacheSize = 8;
thread_local TmapCacheEntry t_tmap_cache[kTmapCacheSize];
thread_local int t_tmap_next = 0;

bool encode_tmap_uncached(CUtensorMap *m, const float *base, int64_t rows, int64_t cols, int64_t ld,
                          int box_cols, int box_rows, bool swizzle128);

bool encode_tmap(CUtensorMap *m, const float *base, int64_t rows, int64_t cols, int64_t ld,
                 int box_cols, int box_rows, bool swizzle128) {
  for (const TmapCacheEntry &e : t_tmap_cache) {
    if (e.valid && e.base == base && e.rows == rows && e.cols == cols && e.ld == ld &&
        e.box_cols == box_cols && e.box_rows == box_rows && e.swizzle128 == swizzle128) {
      *m = e.map;
      return true;
    }
  }
  if (!encode_tmap_uncached(m, base, rows, cols, ld, box_cols, box_rows, swizzle128)) return false;
  TmapCacheEntry &e = t_tmap_cache[t_tmap_next];
  t_tmap_next = (t_tmap_next + 1) % kTmapCacheSize;
  e.base = base;
  e.rows = rows;
  e.cols = cols;
  e.ld = ld;
  e.box_cols = box_cols;
  e.box_rows = box_rows;
  e.swizzle128 = swizzle128;
  e.map = *m;
  e.valid = true;
  return true;
}

bool encode_tmap_uncached(CUtensorMap *m, const float *base, int64_t rows, int64_t cols, int64_t ld,
                          int box_cols, int box_rows, bool swizzle128) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4u};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D form for a strided batch: dims {cols, rows, batch}, strides {ld, stride}
// elements, box box_cols x box_rows x 1.
bool encode_tmap_batched(CUtensorMap *m, const float *base, int64_t rows, int64_t cols, int64_t ld,
                         int64_t batch, int64_t stride, int box_cols, int box_rows, bool swizzle128) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(batch)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 4u, static_cast<cuuint64_t>(stride) * 4u};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int norm_op(int t) {
  switch (t) {
    case 0: case 'N': case 'n': return 0;
    case 1: case 'T': case 't': return 1;
    default: return -1;
  }
}

// [lo, hi) byte range of a stored rows x cols matrix with leading dim ld, in
// 128-bit arithmetic: rows < 2^31 and ld <= 2^40 make (rows - 1) * ld + cols
// reach 2^71 elements, past int64, and the end may lie past the address space.
using u128 = unsigned __int128;
static void byte_range(const void *p, int64_t rows, int64_t cols, int64_t ld, u128 *lo, u128 *hi) {
  *lo = reinterpret_cast<uintptr_t>(p);
  *hi = *lo + 4 * (static_cast<u128>(rows - 1) * static_cast<u128>(ld) + static_cast<u128>(cols));
}

static bool overlaps(u128 a0, u128 a1, u128 b0, u128 b1) { return a0 < b1 && b0 < a1; }

// Host-side validation shared by sgemm_ex and sgemm_select_algo.
sgemm_status_t validate_shape(const Args &a) {
  if (a.ta < 0 || a.tb < 0) return SGEMM_ERR_INVALID_VALUE;
  if (a.M < 0 || a.N < 0 || a.K < 0) return SGEMM_ERR_INVALID_VALUE;
  if (a.M > kMaxDim || a.N > kMaxDim || a.K > kMaxDim) return SGEMM_ERR_INVALID_VALUE;
  const int64_t a_cols = a.ta ? a.M : a.K, b_cols = a.tb ? a.K : a.N;
  if (a.lda < (a_cols > 1 ? a_cols : 1) || a.lda > kMaxLd) return SGEMM_ERR_INVALID_VALUE;
  if (a.ldb < (b_cols > 1 ? b_cols : 1) || a.ldb > kMaxLd) return SGEMM_ERR_INVALID_VALUE;
  if (a.ldc < (a.N > 1 ? a.N : 1) || a.ldc > kMaxLd) return SGEMM_ERR_INVALID_VALUE;
  return SGEMM_SUCCESS;
}

sgemm_status_t validate(const Args &a, bool c_writable) {
  const sgemm_status_t shape = validate_shape(a);
  if (shape != SGEMM_SUCCESS) return shape;
  const int64_t a_cols = a.ta ? a.M : a.K, b_cols = a.tb ? a.K : a.N;
  if (a.M == 0 || a.N == 0) return SGEMM_SUCCESS;
  if (c_writable && a.C == nullptr) return SGEMM_ERR_INVALID_VALUE;
  const bool need_ab = a.K > 0 && a.alpha != 0.0f;
  if (need_ab && (a.A == nullptr || a.B == nullptr)) return SGEMM_ERR_INVALID_VALUE;
  // A matrix that the call touches must fit in the 64-bit address space; then
  // every element offset the kernels form (row * ld + col) fits in int64.
  const u128 kAddressEnd = static_cast<u128>(1) << 64;
  u128 c0 = 0, c1 = 0, x0, x1;
  if (a.C != nullptr) {
    byte_range(a.C, a.M, a.N, a.ldc, &c0, &c1);
    if (c1 > kAddressEnd) return SGEMM_ERR_INVALID_VALUE;
  }
  if (need_ab) {
    byte_range(a.A, a.ta ? a.K : a.M, a_cols, a.lda, &x0, &x1);
    if (x1 > kAddressEnd) return SGEMM_ERR_INVALID_VALUE;
    if (a.C != nullptr && overlaps(c0, c1, x0, x1)) return SGEMM_ERR_ALIASING;
    byte_range(a.B, a.tb ? a.N : a.K, b_cols, a.ldb, &x0, &x1);
    if (x1 > kAddressEnd) return SGEMM_ERR_INVALID_VALUE;
    if (a.C != nullptr && overlaps(c0, c1, x0, x1)) return SGEMM_ERR_ALIASING;
  }
  return SGEMM_SUCCESS;
}

bool tma_eligible(const Args &a) {
  return (reinterpret_cast<uintptr_t>(a.A) % 16 == 0) && (reinterpret_cast<uintptr_t>(a.B) % 16 == 0) &&
         (a.lda % 4 == 0) && (a.ldb % 4 == 0);
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Tile choice for the CUDA-core kernels (eight math warps, one CTA per SM):
// 128 x 256 with 8 x 16 thread tiles when both operands are m/n-contiguous
// (op = TN), N is wide enough and the TMA producer runs; 128 x 128 otherwise;
// 128 x 64 (two CTAs per SM) when N <= 64 or the product is small.  (Measured on 4096^3: the wide
// tile gives TN 67.7 vs 63.0 TFLOP/s; NN, whose k-contiguous A costs more
// registers in the wide tile, is faster narrow, 59.1 vs 58.4.)  Stream-K
// spreads the k-iterations when the tile count does not fill whole waves.
#ifndef SG_SIMT_WIDE_TILE
#define SG_SIMT_WIDE_TILE 1
#endif
// SG_WIDE_MIN_FILL_PCT: the 128 x 256 tile (and with it the transpose ahead)
// is used once that many percent of the SMs get a whole tile; stream-K spreads
// the rest.  Measured on GB300 (graph-timed): requiring a full wave left
// 2048^3 on 128 x 128 tiles (NN 58.3, NT 54.5, TN 59.3 TFLOP/s); from 75 %
// down to 25 % it runs wide (60.7 / 59.1 / 63.2), 3072^3 and larger
// unchanged, 1536^3 (47 %) slightly faster.
#ifndef SG_WIDE_MIN_FILL_PCT
#define SG_WIDE_MIN_FILL_PCT 40
#endif
// Small products (M * N * K, times the batch count, <= SG_SMALL_TILE_WORK)
// take the 128 x 64 tile (four math warps, two CTAs per SM): twice the
// tiles, so stream-K cuts the k-loop into fewer, longer segments per tile
// and the fixup adds fewer partials.  GB300, NN graph replays: 256^3 12.2 -> 11.0 us, 512^3 20.2 ->
// 17.1 us; from 768^3 on the 128 x 128 tile is as fast or faster.
#ifndef SG_SMALL_TILE_WORK
#define SG_SMALL_TILE_WORK (int64_t(1) << 27)
#endif
int pick_simt_tile(const Args &a, int producer, int sm_count, int64_t batch) {
  if (a.N <= 64) return kTile128x64;
  if (static_cast<double>(a.M) * a.N * a.K * batch <= static_cast<double>(SG_SMALL_TILE_WORK))
    return kTile128x64;
  // the math warps read A m-contiguous when it is stored K x M, or when the
  // TMA producer transposes a k-contiguous A in shared memory
  const bool a_mn_in_smem = a.ta == 1 || (producer == kTma && SG_SIMT_TRANSPOSE_A);
  // the wide tile only once enough SMs get a whole tile: far below that,
  // stream-K would cut its k-loop into short, fixup-heavy segments.  A batch
  // (every product counted) takes it once it fills a whole wave, and only
  // where it pads each product's N no further than the 128-wide tile does
  // (GB300, 128 x 128 -> 128 x 256, TFLOP/s: 96 x 512x512x64 NN 41.1 -> 42.7,
  // TN 41.5 -> 43.0, 8 x 2048^3 NN 61.7 -> 64.5; 12 x 512x512x1024 NN, 96
  // wide tiles, 53.1 -> 51.5, so below a wave it stays narrow).
  const bool fills = batch == 1 ? cdiv(a.M, 128) * cdiv(a.N, 256) * 100 >=
                                      SG_WIDE_MIN_FILL_PCT * sm_count
                                : cdiv(a.M, 128) * cdiv(a.N, 256) * batch >= sm_count;
  const bool pad_ok = batch == 1 || cdiv(a.N, 256) * 2 == cdiv(a.N, 128);
  if (SG_SIMT_WIDE_TILE && producer == kTma && a_mn_in_smem && a.tb == 0 && fills && pad_ok)
    return kTile128x256;
  return kTile128x128;
}

// Tile-rows per raster group of the CUDA-core kernels: consecutive tiles walk
// down a group of this many tile-rows before moving right, so that the tiles
// in flight share op(A) row blocks and op(B) column blocks in L2.
#ifndef SG_SIMT_GROUP_M
#define SG_SIMT_GROUP_M 8
#endif
#ifndef SG_SK_REMAINDER
#define SG_SK_REMAINDER 0
#endif
#ifndef SG_SK_FIXUP_LAUNCH
#define SG_SK_FIXUP_LAUNCH 0
#endif
// Split tiles are finished in-kernel while grid <= SG_SK_INKERNEL_RATIO x
// the number of split tiles (at most about RATIO + 1 segments per tile).
#ifndef SG_SK_INKERNEL_RATIO
#define SG_SK_INKERNEL_RATIO 2
#endif
// SG_EPI_TMA 1: the 128 x 128 TMA kernels write C through a staged tile and
// TMA stores when beta == 0 (0: always from registers).
#ifndef SG_EPI_TMA
#define SG_EPI_TMA 1
#endif
// SG_SK_MIN_GAIN: with at least a wave of tiles, stream-K only where
// balancing the k-tiles over every slot shortens the busiest slot's work by
// this many k-tiles (0: wherever the last wave is partial).  Short k-loops
// gain less than the split segments and the fixup cost (GB300, graph-free
// calls, 0 -> 4: 96 x 512x512x64 NT 36.6 -> 38.9 TFLOP/s, NN 39.1 -> 40.4,
// 512 x 128x128x64 NT 27.6 -> 31.9; single products unchanged).
#ifndef SG_SK_MIN_GAIN
#define SG_SK_MIN_GAIN 4
#endif
SkPlan plan_stream_k(int64_t tiles, int64_t k_tiles, int64_t slots, bool have_ws) {
  SkPlan pl{static_cast<int>(tiles), 0, 0, static_cast<int>(tiles < slots ? tiles : slots)};
  if (!have_ws || k_tiles < 2 * kMinSkSegment) return pl;
  if (tiles >= slots && tiles % slots == 0) return pl;
  if (SG_SK_MIN_GAIN > 0 && tiles >= slots &&
      cdiv(tiles, slots) * k_tiles * slots - tiles * k_tiles < SG_SK_MIN_GAIN * slots)
    return pl;
  // SG_SK_REMAINDER 1: split only the tiles beyond whole waves; 0: the last
  // one to two waves' worth
  const int64_t sk = tiles < slots ? tiles
                     : SG_SK_REMAINDER ? tiles % slots
                     : (tiles >= 2 * slots ? slots + tiles % slots : tiles);
  int64_t grid = slots;
  // fewer CTAs than slots only when every tile is split (whole tiles are
  // spread over the whole grid)
  if (sk == tiles && sk * k_tiles < grid * kMinSkSegment) grid = (sk * k_tiles) / kMinSkSegment;
  // the fixup pass handles at most 126 segments per tile (ranges >= k_tiles/120)
  if (grid > sk * 120) grid = sk * 120;
  if (grid < 2 || sk % grid == 0) return pl;  // whole tiles per CTA: plain waves
  pl.dp_tiles = static_cast<int>(tiles - sk);
  pl.sk_tiles = static_cast<int>(sk);
  pl.sk_iters = sk * k_tiles;
  pl.grid = static_cast<int>(grid);
  return pl;
}

// Cluster split-K (SimtParams::csk): a product whose tiles leave CTA slots
// idle splits each tile's k-tiles over a cluster of S CTAs that add their
// partials through distributed shared memory -- one launch, no workspace,
// no fixup pass.  It pays where each CTA's share is short; with longer
// shares stream-K, which balances the k-tiles over every CTA slot, is the
// faster (GB300, graph replays, us per call, stream-K -> clusters of <= 4:
// 512^3 NN 19.6 -> 13.5, NT 20.8 -> 14.8, 640^3 23.2 -> 22.0, 768^3 29.7 ->
// 24.6; but 8192 x 64 x 4096 89.1 -> 98.4, 2048 x 64 x 2048 26.9 -> 30.8,
// 1000 x 1013 x 997 57.9 -> 63.5, 1024^3 50.4 -> 50.8; clusters of 8 lost to
// clusters of 4: 512^3 16.0 against 13.5).  So S is the larger of 4 and 2
// for which every cluster is resident at once and each CTA gets between
// SG_CSK_MIN_K and SG_CSK_MAX_K k-tiles.  SG_CSK 0 turns it off.
#ifndef SG_CSK
#define SG_CSK 1
#endif
#ifndef SG_CSK_MIN_K
#define SG_CSK_MIN_K 2
#endif
#ifndef SG_CSK_MAX_K
#define SG_CSK_MAX_K 8
#endif
#ifndef SG_CSK_MAX
#define SG_CSK_MAX 4
#endif
// Without a stream-K workspace (scratch limit, a capture before the first
// allocation) the alternative is whole tiles in waves, so cluster split-K is
// then taken whatever the length of the shares (GB300, 1024^3 under a scratch
// limit of 0: 87.0 us per call in whole tiles, 50.8 in clusters of two).
int pick_csk(const SimtKernelInfo &ki, int64_t tiles, int64_t k_tiles, int64_t slots, bool have_ws) {
  if (!SG_CSK || tiles >= slots) return 0;
  for (int i = 2; i >= 0; --i) {
    const int S = 2 << i;
    if (S > SG_CSK_MAX || ki.bm % S != 0) continue;
    if (ki.max_clusters[i] >= tiles && k_tiles >= int64_t(S) * SG_CSK_MIN_K &&
        (!have_ws || k_tiles <= int64_t(S) * SG_CSK_MAX_K))
      return S;
  }
  return 0;
}


bool stream_capturing(cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return cs == cudaStreamCaptureStatusActive;
}

// Id of the capture sequence `s` is recording into, or 0.
unsigned long long capture_id(cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  unsigned long long id = 0;
  if (cudaStreamGetCaptureInfo(s, &cs, &id) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return cs == cudaStreamCaptureStatusActive ? id : 0;
}

cudaError_t order_before_use(BufferOrder &o, cudaStream_t s, bool capturing) {
  if (!o.used) return cudaSuccess;
  if (capturing) {
    // the previous use was captured earlier on this stream into the same
    // graph: the graph orders the two, and a wait node here would only cut
    // the programmatic launch chain
    if (o.last == s && o.capture != 0 && o.capture == capture_id(s)) return cudaSuccess;
    return cudaStreamWaitEvent(s, o.ev, cudaEventWaitExternal);
  }
  if (o.in_graph || o.last != s) return cudaStreamWaitEvent(s, o.ev, 0);
  return cudaSuccess;
}

bool reserve_scratch(DeviceState &d, uint64_t bytes) {
  uint64_t cur = d.held.load();
  do {
    const uint64_t lim = d.limit.load();
    if (cur > lim || bytes > lim - cur) return false;
  } while (!d.held.compare_exchange_weak(cur, cur + bytes));
  return true;
}

void release_scratch(DeviceState &d, uint64_t bytes) { d.held.fetch_sub(bytes); }

cudaError_t order_after_use(BufferOrder &o, cudaStream_t s, bool capturing) {
  const cudaError_t e = capturing ? cudaEventRecordWithFlags(o.ev, s, cudaEventRecordExternal)
                                  : cudaEventRecord(o.ev, s);
  o.used = true;
  o.last = s;
  o.in_graph = o.in_graph || capturing;
  o.capture = capturing ? capture_id(s) : 0;
  return e;
}

}  // namespace sg

namespace {

using namespace sg;

// The device's stream-K workspace (2 partial tiles per CTA slot of the largest
// configuration), allocated on first use; null if that failed, or if it does
// not exist yet and `capturing` (no allocation inside a stream capture).
// Bytes of the stream-K workspace: two 128 x 256 partial tiles per SM (the
// largest need, one CTA per SM), then the arrival counters of the in-kernel
// fixup (zero between launches).
size_t stream_k_workspace_bytes(const DeviceState &d) {
  return static_cast<size_t>(2) * d.sm_count * 128 * 256 * sizeof(float) + kSkCounters * sizeof(int);
}

// Whether a stream-K workspace exists or could be allocated now.
bool stream_k_workspace_possible(DeviceState &d, bool capturing) {
  if (d.ws_failed) return false;
  if (d.ws) return true;
  if (capturing) return false;
  const uint64_t lim = d.limit.load(), held = d.held.load();
  return held <= lim && stream_k_workspace_bytes(d) <= lim - held;
}

float *stream_k_workspace(DeviceState &d, size_t need, bool capturing) {
  if (d.ws_failed) return nullptr;
  if (!d.ws) {
    if (capturing) return nullptr;
    const size_t total = stream_k_workspace_bytes(d), bytes = total - kSkCounters * sizeof(int);
    // over the scratch limit: no workspace (not a failure; the limit may rise)
    if (!reserve_scratch(d, total)) return nullptr;
    if (!d.ws_order.ev && cudaEventCreateWithFlags(&d.ws_order.ev, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      release_scratch(d, total);
      d.ws_failed = true;
      return nullptr;
    }
    if (cudaMalloc(&d.ws, total) != cudaSuccess ||
        cudaMemset(reinterpret_cast<char *>(d.ws) + bytes, 0, kSkCounters * sizeof(int)) != cudaSuccess) {
      cudaGetLastError();
      if (d.ws) cudaFree(d.ws);
      d.ws = nullptr;
      d.ws_failed = true;
      release_scratch(d, total);
      return nullptr;
    }
    d.ws_bytes = bytes;
    d.sk_count = reinterpret_cast<int *>(reinterpret_cast<char *>(d.ws) + bytes);
  }
  return need <= d.ws_bytes ? d.ws : nullptr;
}

// Products of at most 2^26 multiply-adds with K <= 1024 and at most 608
// tiles of 32 x 32 (four per SM of a GB300) run the small-product kernel:
// one launch, no stream-K pass (GB300, CUDA-graph replays: 256^3 12.0 ->
// 5.3 us, 384^3 15.3 -> 8.4 us, 65 x 4097 x 129 20.8 -> 9.7 us,
// 4096 x 128 x 128 16.4 -> 12.8 us).  The persistent kernels are faster from
// 768^3, with K = 4096, and when many tiles have a short K (2048 x 2048 x 32:
// 15.5 against 133 us).
#ifndef SG_SMALL_MAX_WORK
#define SG_SMALL_MAX_WORK (int64_t(1) << 26)
#endif
#ifndef SG_SMALL_MAX_TILES
#define SG_SMALL_MAX_TILES 608
#endif
bool small_wanted(const Args &a) {
  const double work = static_cast<double>(a.M) * static_cast<double>(a.N) * static_cast<double>(a.K);
  return work <= static_cast<double>(SG_SMALL_MAX_WORK) && a.K <= 1024 &&
         cdiv(a.M, 32) * cdiv(a.N, 32) <= SG_SMALL_MAX_TILES;
}

sgemm_algo_t auto_algo(const Args &a) {
  if (small_wanted(a)) return SGEMM_ALGO_SMALL;
  return tma_eligible(a) ? SGEMM_ALGO_SIMT_TMA : SGEMM_ALGO_SIMT_CPASYNC;
}

// A strided batch of products (count 1 for a plain product).
struct Batch {
  int64_t count, sa, sb, sc;
};

// pdl: the product directly follows another kernel of the same call on the
// stream (an operand transpose) and may be scheduled before it ends.
// Launches queued right before the product (the operand copies of
// run_pretransposed): after every wait the product needs, so that the copies
// and the product form one programmatic launch chain.
using PreLaunch = std::function<cudaError_t()>;

// SG_SIMT_PDL 1: every CUDA-core product kernel is launched as a programmatic
// dependent of the stream's previous kernel, whatever that kernel is: its
// set-up (barriers, tensor-map prefetch, register split) overlaps that
// kernel's tail, and it touches memory only after griddepcontrol.wait, which
// returns once the previous grid has completed and its writes are visible.
// 0: only after a kernel of the same call.  GB300, back-to-back calls, 0 ->
// 1: 512^3 NN 14.06 -> 13.64 us and NT 15.32 -> 14.68 us (graph replays),
// strided batches 96 x 512x512x64 NT 38.7 -> 39.5 and NN 42.5 -> 44.0,
// 512 x 128x128x64 NT 31.6 -> 33.5 TFLOP/s; large products unchanged.
#ifndef SG_SIMT_PDL
#define SG_SIMT_PDL 1
#endif

sgemm_status_t run_simt(const Args &a, DeviceState &d, int producer, cudaStream_t stream,
                        const Batch &bt = Batch{1, 0, 0, 0}, bool pdl = false,
                        const PreLaunch *pre = nullptr) {
  const int tile = pick_simt_tile(a, producer, d.sm_count, bt.count);
  const SimtKernelInfo *ki = kernel_info(d, producer, a.ta, a.tb, tile);
  if (!ki || ki->ctas_per_sm < 1) return SGEMM_ERR_LAUNCH;
  pdl = pdl || SG_SIMT_PDL;

  SimtParams p;
  p.A = a.A;
  p.B = a.B;
  p.C = a.C;
  p.lda = a.lda;
  p.ldb = a.ldb;
  p.ldc = a.ldc;
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.alpha = a.alpha;
  p.beta = a.beta;
  p.tiles_m = static_cast<int>(cdiv(a.M, ki->bm));
  p.tiles_n = static_cast<int>(cdiv(a.N, ki->bn));
  p.k_tiles = static_cast<int>(cdiv(a.K, 32));
  const int64_t tiles_per_batch = static_cast<int64_t>(p.tiles_m) * p.tiles_n;
  const int64_t num_tiles = tiles_per_batch * bt.count;
  if (num_tiles > kMaxDim) return SGEMM_ERR_UNSUPPORTED;
  p.num_tiles = static_cast<int>(num_tiles);
  p.tiles_per_batch = static_cast<int>(tiles_per_batch);
  p.strideA = bt.sa;
  p.strideB = bt.sb;
  p.strideC = bt.sc;
  p.a_map3d = producer == kTma && bt.count > 1 && bt.sa != 0;
  p.b_map3d = producer == kTma && bt.count > 1 && bt.sb != 0;
  p.group_m = SG_SIMT_GROUP_M;
  p.c_vec4 = (a.ldc % 4 == 0) && (reinterpret_cast<uintptr_t>(a.C) % 16 == 0) &&
             (bt.count == 1 || bt.sc % 4 == 0);
  p.wait_budget_ns = g_wait_budget_ns.load(std::memory_order_relaxed);
  p.status = d.status;
  p.workspace = nullptr;

  CUtensorMap tmA, tmB;
  std::memset(&tmA, 0, sizeof(tmA));
  std::memset(&tmB, 0, sizeof(tmB));
  if (producer == kTma) {
    // op(A): K-major when stored M x K, MN-major when stored K x M; a strided
    // operand of a batch gets a third (batch) dimension.
    const int64_t ar = a.ta == 0 ? a.M : a.K, ac = a.ta == 0 ? a.K : a.M;
    const int abc = a.ta == 0 ? 32 : ki->bm, abr = a.ta == 0 ? ki->bm : 32;
    const int64_t br = a.tb == 0 ? a.K : a.N, bc = a.tb == 0 ? a.N : a.K;
    const int bbc = a.tb == 0 ? ki->bn : 32, bbr = a.tb == 0 ? 32 : ki->bn;
    const bool okA = p.a_map3d
                         ? encode_tmap_batched(&tmA, a.A, ar, ac, a.lda, bt.count, bt.sa, abc, abr, a.ta == 0)
                         : encode_tmap(&tmA, a.A, ar, ac, a.lda, abc, abr, a.ta == 0);
    const bool okB = p.b_map3d
                         ? encode_tmap_batched(&tmB, a.B, br, bc, a.ldb, bt.count, bt.sb, bbc, bbr, a.tb == 1)
                         : encode_tmap(&tmB, a.B, br, bc, a.ldb, bbc, bbr, a.tb == 1);
    if (!okA || !okB) {
      // a batch layout the tensor-map encoder refuses is still a valid batch:
      // load it with cp.async instead
      if (bt.count > 1) return run_simt(a, d, kCpAsync, stream, bt, pdl, pre);
      return SGEMM_ERR_LAUNCH;
    }
  }

  // C through staged TMA stores (the 128 x 128 TMA kernels, beta == 0, C
  // addressable by a tensor map)
  // A tensor map of C (32-column x 128-row boxes, 128-byte swizzle), when C
  // is TMA-addressable: for the staged stores (beta == 0) or the producer's
  // L2 prefetch of C (beta != 0).
  CUtensorMap tmC;
  std::memset(&tmC, 0, sizeof(tmC));
  p.c_tma = 0;
  p.c_pref = 0;
  int c_map = 0;   // 1: 2-D, 2: 3-D (strided batch)
  if (producer == kTma && reinterpret_cast<uintptr_t>(a.C) % 16 == 0 && a.ldc % 4 == 0 &&
      (SG_EPI_TMA || a.beta != 0.0f)) {
    if (bt.count == 1) {
      if (encode_tmap(&tmC, a.C, a.M, a.N, a.ldc, 32, 128, true)) c_map = 1;
    } else if (bt.sc % 4 == 0 &&
               encode_tmap_batched(&tmC, a.C, a.M, a.N, a.ldc, bt.count, bt.sc, 32, 128, true)) {
      c_map = 2;
    }
  }
  // Staged stores: the 128 x 128 tiles, not the NT kernel that transposes A
  // in shared memory, and N % 4 == 0 -- a TMA store writes whole 16-byte
  // granules at the inner edge of the tensor, so a ragged row end would get
  // up to three floats past N.
  const bool nt_transposing = a.ta == 0 && a.tb == 1 && SG_SIMT_TRANSPOSE_A;
  if (SG_EPI_TMA && c_map && tile == kTile128x128 && !nt_transposing && a.beta == 0.0f && a.N % 4 == 0)
    p.c_tma = c_map;
  if (a.beta != 0.0f) p.c_pref = c_map;

  const int64_t slots = static_cast<int64_t>(d.sm_count) * ki->ctas_per_sm;
  // Under-filled products: cluster split-K (its own instantiation of the
  // kernel, 128 x 128 and 128 x 64 tiles), one launch and no workspace
  const SimtKernelInfo *kc = tile != kTile128x256 && num_tiles < slots
                                 ? kernel_info(d, producer, a.ta, a.tb, tile, 1)
                                 : nullptr;
  const int csk = kc ? pick_csk(*kc, num_tiles, p.k_tiles, static_cast<int64_t>(d.sm_count) * kc->ctas_per_sm,
                               stream_k_workspace_possible(d, stream_capturing(stream)))
                     : 0;
  if (csk > 1) {
    p.csk = csk;
    p.dp_tiles = 0;
    p.sk_iters = 0;
    p.workspace = nullptr;
    p.sk_count = nullptr;
    if (pre && (*pre)() != cudaSuccess) return SGEMM_ERR_LAUNCH;
    if (simt_entry(producer, a.ta, a.tb, tile, 1)
            .launch(p, &tmA, &tmB, &tmC, static_cast<int>(num_tiles * csk), stream, pdl, csk) != cudaSuccess)
      return SGEMM_ERR_LAUNCH;
    t_last_launches = 1;
    if (verbose())
      std::fprintf(stderr, "sgemm: %lldx%lldx%lld %c%c batch %lld: %s %dx%d tiles %lld, cluster split-K S=%d, grid %lld\n",
                   (long long)a.M, (long long)a.N, (long long)a.K, "NT"[a.ta], "NT"[a.tb], (long long)bt.count,
                   producer == kTma ? "tma" : "cp.async", ki->bm, ki->bn, (long long)num_tiles, csk,
                   (long long)(num_tiles * csk));
    return SGEMM_SUCCESS;
  }
  const bool capturing = stream_capturing(stream);
  std::unique_lock<std::mutex> ws_lock(d.ws_mu);
  SkPlan plan = plan_stream_k(num_tiles, p.k_tiles, slots, !d.ws_failed);
  if (plan.sk_tiles > 0) {
    const size_t need = static_cast<size_t>(2) * plan.grid * ki->bm * ki->bn * sizeof(float);
    p.workspace = stream_k_workspace(d, need, capturing);
    if (!p.workspace) plan = plan_stream_k(num_tiles, p.k_tiles, slots, false);
  }
  if (plan.sk_tiles == 0) ws_lock.unlock();
  p.dp_tiles = plan.dp_tiles;
  p.sk_iters = plan.sk_iters;
  // Split tiles of at most about three segments (grid <= 2 * split tiles)
  // are finished inside the TMA kernel that reads A m-contiguous (tiles of
  // eight math warps), by the CTA
  // that arrives last at each; otherwise sk_fixup_kernel does it, which
  // spreads a tile of many segments over many blocks (GB300, per call: 4096^3
  // 2042.5 -> 2034.6 us and 2048^3 TN 268.3 -> 265.3 us in-kernel, but 1536^3
  // NN 125.3 -> 129.3 us and 256^3 11.0 -> 19.5 us).  SG_SK_FIXUP_LAUNCH 1:
  // always the separate pass.
  const bool in_kernel_fixup_kernel =
      producer == kTma && (!(a.ta == 0 && SG_SIMT_TRANSPOSE_A) || SG_SK_INKERNEL_ATRANS) &&
      tile != kTile128x64;
  p.sk_count = (plan.sk_tiles > 0 && !SG_SK_FIXUP_LAUNCH && in_kernel_fixup_kernel &&
                plan.grid <= SG_SK_INKERNEL_RATIO * static_cast<int64_t>(plan.sk_tiles) &&
                plan.sk_tiles <= kSkCounters)
                   ? d.sk_count
                   : nullptr;

  // the previous stream-K call (another stream, or a graph) may still be
  // using the workspace
  if (plan.sk_tiles > 0 && order_before_use(d.ws_order, stream, capturing) != cudaSuccess)
    return SGEMM_ERR_LAUNCH;
  if (pre && (*pre)() != cudaSuccess) return SGEMM_ERR_LAUNCH;
  cudaError_t e =
      simt_entry(producer, a.ta, a.tb, tile).launch(p, &tmA, &tmB, &tmC, plan.grid, stream, pdl, 1);
  if (e != cudaSuccess) return SGEMM_ERR_LAUNCH;
  t_last_launches = 1;
  if (plan.sk_tiles > 0) {
    if (p.sk_count == nullptr) {
      if (launch_sk_fixup(p, ki->bm, ki->bn, plan.grid, plan.sk_tiles, d.sm_count, stream) != cudaSuccess)
        return SGEMM_ERR_LAUNCH;
      t_last_launches = 2;
    }
    if (order_after_use(d.ws_order, stream, capturing) != cudaSuccess) return SGEMM_ERR_LAUNCH;
  }
  if (verbose())
    std::fprintf(stderr, "sgemm: %lldx%lldx%lld %c%c batch %lld: %s %dx%d tiles %lld (%d whole), stream-K tiles %d, grid %d, fixup %s, C %s\n",
                 (long long)a.M, (long long)a.N, (long long)a.K, "NT"[a.ta], "NT"[a.tb], (long long)bt.count,
                 producer == kTma ? "tma" : "cp.async", ki->bm, ki->bn, (long long)num_tiles, plan.dp_tiles,
                 plan.sk_tiles, plan.grid, plan.sk_tiles == 0 ? "none" : p.sk_count ? "in-kernel" : "launch",
                 p.c_tma ? "staged TMA stores" : "from registers");
  return SGEMM_SUCCESS;
}

// Products whose op(A) is k-contiguous (A stored M x K) or whose op(B) is
// k-contiguous (B stored N x K) can instead have that operand transposed once
// into library scratch by the transpose kernel, after which the product runs
// with A m-contiguous and B n-contiguous -- the layout whose tiles need no
// shared-memory rewrite and take the 128 x 256 tile.  The math is the same
// as the in-kernel transpose's (same shared-memory tiles, same k order), so
// the result is bit-identical; the cost is 8 bytes of HBM traffic per
// transposed element, small against 2 * M * N * K FLOP once the other
// dimension is large.  Measured on GB300 at 4096^3 (TFLOP/s, in-kernel ->
// transposed ahead): NN 63.9 -> 66.8, NT 54.0 -> 64.2, TT 58.2 -> 66.9
// (TN 67.6 needs nothing).
#ifndef SG_PRETRANSPOSE
#define SG_PRETRANSPOSE 1
#endif
constexpr int64_t kPretransposeMinOther = 1024;        // the other dimension
constexpr int64_t kPretransposeMinWork = int64_t(1) << 30;   // M * N * K
constexpr size_t kPretransposeMaxBytes = size_t(2) << 30;    // 2 GiB of scratch

// Operands copied into library scratch ahead of the product: transposed
// (a, b), or repacked into 16-byte aligned rows (ra, rb) so that the TMA
// producer can load them.
struct Pretranspose {
  bool a, b;
  bool ra = false, rb = false;
  bool any() const { return a || b || ra || rb; }
};
// Repacking: AUTO runs a product whose A or B is not TMA-eligible (base not
// 16-byte aligned, or a leading dimension not a multiple of 4) on the TMA
// path after copying that operand into aligned scratch, once M * N * K
// reaches this: the cp.async producer moves 4 bytes per instruction and is
// far slower (GB300, NN, TFLOP/s in place -> repacked: 767 x 769 x 771
// 16.2 -> 21.0, 2047 x 2049 x 2051 23.9 -> 50.6; below about 2^27 the extra
// launch costs more than it saves: 383 x 385 x 387 4.5 -> 3.7).
#ifndef SG_REPACK_MIN_WORK
#define SG_REPACK_MIN_WORK (int64_t(1) << 27)
#endif
// The tensor-core product after a transpose is launched the ordinary way:
// as a programmatic dependent it ran slower (4096^3 NN 140.8 vs 167.8
// TFLOP/s on GB300), while the CUDA-core kernel gains a little from it.
#ifndef SG_TC_PDL
#define SG_TC_PDL 0
#endif
// Tile-rows per raster group of the tensor-core kernel (L2 reuse of the
// operand panels that concurrently running tiles share).
#ifndef SG_TC_GROUP_M
#define SG_TC_GROUP_M 8
#endif

sgemm_status_t run_tc3(const Args &a, DeviceState &d, cudaStream_t stream, bool pdl = false);

// tile_n: the N extent of the tiles the transposed product runs with (256
// for the CUDA-core kernel's wide tile, 128 for the tensor-core kernel).
Pretranspose transpose_plan_any(const Args &a, int sm_count, int64_t tile_n) {
  Pretranspose t{false, false};
  if (!SG_PRETRANSPOSE) return t;
  const double work = static_cast<double>(a.M) * static_cast<double>(a.N) * static_cast<double>(a.K);
  // only where the transposed product fills the GPU with 128 x 256 tiles:
  // below that both layouts run 128 x 128 tiles and the extra launch loses
  // (measured at 2048^3 NN: 57.4 in-kernel vs 56.2 TFLOP/s transposed ahead)
  // (GB300, graph replays: transposing ahead into 128 x 128 tiles costs
  // 768^3 NN 28.4 -> 38.2 us, 1024^3 49.2 -> 58.2 us)
  const bool fills =
      cdiv(a.M, 128) * cdiv(a.N, tile_n) * 100 >= (tile_n == 256 ? SG_WIDE_MIN_FILL_PCT : 100) * sm_count;
  if (work < static_cast<double>(kPretransposeMinWork) || !fills) return t;
  t.a = a.ta == 0 && a.N >= kPretransposeMinOther;
  t.b = a.tb == 1 && a.M >= kPretransposeMinOther;
  return t;
}

int64_t round4(int64_t x) { return (x + 3) & ~int64_t(3); }

Pretranspose pretranspose_plan(const Args &a, int sm_count, int64_t tile_n) {
  return tma_eligible(a) ? transpose_plan_any(a, sm_count, tile_n) : Pretranspose{false, false};
}

bool a_tma_ok(const Args &a) { return reinterpret_cast<uintptr_t>(a.A) % 16 == 0 && a.lda % 4 == 0; }
bool b_tma_ok(const Args &a) { return reinterpret_cast<uintptr_t>(a.B) % 16 == 0 && a.ldb % 4 == 0; }

// AUTO on operands that are not TMA-eligible: large enough products copy
// each offending operand into aligned scratch -- transposed where the plan
// transposes it anyway, else repacked as it is (same values, same layout).
bool repack_wanted(const Args &a) {
  const double work = static_cast<double>(a.M) * static_cast<double>(a.N) * static_cast<double>(a.K);
  return !tma_eligible(a) && work >= static_cast<double>(SG_REPACK_MIN_WORK);
}
Pretranspose repack_plan(const Args &a, int sm_count) {
  Pretranspose t = transpose_plan_any(a, sm_count, 256);
  t.ra = !t.a && !a_tma_ok(a);
  t.rb = !t.b && !b_tma_ok(a);
  return t;
}

// Products large enough for the split pass of the tensor-core path: the size
// rule of pretranspose_plan with 128 x 128 tiles, any layout.
bool presplit_size_ok(const Args &a, int sm_count) {
  const double work = static_cast<double>(a.M) * static_cast<double>(a.N) * static_cast<double>(a.K);
  return tma_eligible(a) && work >= static_cast<double>(kPretransposeMinWork) &&
         cdiv(a.M, 128) * cdiv(a.N, 128) >= sm_count;
}

// Scratch of at least `bytes` (grown in 64 MiB steps), or null (also when it
// would have to be allocated or grown inside a stream capture).
float *pretranspose_scratch(DeviceState &d, size_t bytes, bool capturing) {
  if (d.tr_failed || bytes > kPretransposeMaxBytes) return nullptr;
  if (capturing) return bytes <= d.tr_bytes ? d.tr : nullptr;
  if (!d.tr_order.ev && cudaEventCreateWithFlags(&d.tr_order.ev, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    d.tr_failed = true;
    return nullptr;
  }
  if (bytes > d.tr_bytes) {
    const size_t step = size_t(64) << 20;
    size_t want = (bytes + step - 1) / step * step;
    // a captured graph holds the current buffer's address: once one exists
    // the buffer is kept for good and a new one taken (at least twice as
    // large, so that the kept buffers add up to less than the live one)
    const bool keep = d.tr_order.in_graph && d.tr;
    if (keep && want < 2 * d.tr_bytes) want = 2 * d.tr_bytes;
    if (want > kPretransposeMaxBytes) want = bytes;
    // the old buffer is freed (unless kept) once the new one exists: both
    // count against the scratch limit meanwhile; over the limit, try the
    // exact size before giving up
    if (!reserve_scratch(d, want)) {
      want = bytes;
      if (!reserve_scratch(d, want)) return nullptr;   // the product runs in place
    }
    float *fresh = nullptr;
    if (cudaMalloc(&fresh, want) != cudaSuccess) {
      cudaGetLastError();
      release_scratch(d, want);
      return nullptr;   // not fatal: this product runs on its operands in place
    }
    if (keep) {
      d.tr_retired.emplace_back(d.tr, d.tr_bytes);
    } else if (d.tr) {
      // cudaFree waits for work still using the old buffer
      cudaFree(d.tr);
      release_scratch(d, d.tr_bytes);
    }
    d.tr = fresh;
    d.tr_bytes = want;
  }
  return d.tr;
}

// Runs the product with the planned operands transposed into scratch.
// Returns SGEMM_ERR_UNSUPPORTED (and queues nothing) when no scratch can be
// had, so that the caller runs the product as it is.
sgemm_status_t run_pretransposed(const Args &a, DeviceState &d, cudaStream_t s, Pretranspose t,
                                 bool tensor) {
  // stored shapes of A and B, and the leading dimension of each copy
  const int64_t a_rows = a.ta ? a.K : a.M, a_cols = a.ta ? a.M : a.K;
  const int64_t b_rows = a.tb ? a.N : a.K, b_cols = a.tb ? a.K : a.N;
  const int64_t lda2 = t.a ? round4(a.M) : round4(a_cols), ldb2 = t.b ? round4(a.N) : round4(b_cols);
  const size_t a_elems = t.a ? static_cast<size_t>(a.K) * lda2 : t.ra ? static_cast<size_t>(a_rows) * lda2 : 0;
  const size_t b_elems = t.b ? static_cast<size_t>(a.K) * ldb2 : t.rb ? static_cast<size_t>(b_rows) * ldb2 : 0;
  const size_t a_bytes = (a_elems * sizeof(float) + 255) & ~size_t(255);
  const size_t bytes = a_bytes + b_elems * sizeof(float);
  const bool capturing = stream_capturing(s);
  std::lock_guard<std::mutex> lock(d.tr_mu);
  float *scratch = pretranspose_scratch(d, bytes, capturing);
  if (!scratch) return SGEMM_ERR_UNSUPPORTED;
  // a call on another stream (or a graph) may still be reading the scratch
  if (order_before_use(d.tr_order, s, capturing) != cudaSuccess) return SGEMM_ERR_LAUNCH;
  // the product's operands: the copies in scratch
  Args b = a;
  float *b_copy = reinterpret_cast<float *>(reinterpret_cast<char *>(scratch) + a_bytes);
  const bool ra = t.ra && !t.a, rb = t.rb && !t.b;   // kept as they are, moved to aligned rows
  if (t.a || ra) {
    b.A = scratch;
    b.lda = lda2;
    if (t.a) b.ta = 1;
  }
  if (t.b || rb) {
    b.B = b_copy;
    b.ldb = ldb2;
    if (t.b) b.tb = 0;
  }
  const int launches = int(t.a) + int(t.b) + int(ra || rb);
  // the copies, queued by the product's launcher after its own waits
  const PreLaunch copies = [&]() -> cudaError_t {
    if (t.a) {   // A is M x K (lda): A^T is K x M (lda2)
      const cudaError_t e = launch_transpose(a.A, a.lda, scratch, lda2, static_cast<int>(a.M),
                                             static_cast<int>(a.K), d.sm_count, d.status, s);
      if (e != cudaSuccess) return e;
    }
    if (t.b) {   // B is N x K (ldb): B^T is K x N (ldb2)
      const cudaError_t e = launch_transpose(a.B, a.ldb, b_copy, ldb2, static_cast<int>(a.N),
                                             static_cast<int>(a.K), d.sm_count, d.status, s);
      if (e != cudaSuccess) return e;
    }
    if (ra)   // one launch for both
      return launch_repack(a.A, a.lda, static_cast<int>(a_rows), static_cast<int>(a_cols), scratch, lda2,
                           rb ? a.B : nullptr, a.ldb, static_cast<int>(b_rows), static_cast<int>(b_cols),
                           b_copy, ldb2, s);
    if (rb)
      return launch_repack(a.B, a.ldb, static_cast<int>(b_rows), static_cast<int>(b_cols), b_copy, ldb2,
                           nullptr, 0, 0, 0, nullptr, 0, s);
    return cudaSuccess;
  };
  sgemm_status_t st;
  if (tensor) {
    st = copies() == cudaSuccess ? run_tc3(b, d, s, /*pdl=*/SG_TC_PDL != 0) : SGEMM_ERR_LAUNCH;
  } else {
    st = run_simt(b, d, kTma, s, Batch{1, 0, 0, 0}, /*pdl=*/true, &copies);
  }
  if (st != SGEMM_SUCCESS) return st;
  t_last_launches += launches;
  if (order_after_use(d.tr_order, s, capturing) != cudaSuccess) return SGEMM_ERR_LAUNCH;
  return SGEMM_SUCCESS;
}

// 3xTF32 on the tensor cores: 128 x 128 tiles, TMA loads (needs TMA-eligible
// operands), one persistent CTA per SM.
sgemm_status_t run_tc3(const Args &a, DeviceState &d, cudaStream_t stream, bool pdl) {
  const TcKernelInfo *ki = tc_kernel_info(d, a.ta, a.tb);
  if (!ki || ki->ctas_per_sm < 1) return SGEMM_ERR_LAUNCH;
  TcParams p;
  p.C = a.C;
  p.ldc = a.ldc;
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.alpha = a.alpha;
  p.beta = a.beta;
  p.tiles_m = static_cast<int>(cdiv(a.M, ki->bm));
  p.tiles_n = static_cast<int>(cdiv(a.N, ki->bn));
  p.k_tiles = static_cast<int>(cdiv(a.K, 32));
  const int64_t num_tiles = static_cast<int64_t>(p.tiles_m) * p.tiles_n;
  if (num_tiles > kMaxDim) return SGEMM_ERR_UNSUPPORTED;
  p.num_tiles = static_cast<int>(num_tiles);
  p.wide_tiles = p.num_tiles;
  p.group_m = SG_TC_GROUP_M;
  p.c_vec4 = (a.ldc % 4 == 0) && (reinterpret_cast<uintptr_t>(a.C) % 16 == 0);
  p.wait_budget_ns = g_wait_budget_ns.load(std::memory_order_relaxed);
  p.status = d.status;
  CUtensorMap tmA, tmB;
  // k-contiguous operands: one [128 rows][32 k] box with the 128-byte swizzle
  // (read by the MMA directly); m/n-contiguous ones: a dense [32 k][128 mn]
  // box (read by the converters).
  const bool okA = a.ta == 0 ? encode_tmap(&tmA, a.A, a.M, a.K, a.lda, 32, 128, true)
                             : encode_tmap(&tmA, a.A, a.K, a.M, a.lda, 128, 32, false);
  const bool okB = a.tb == 0 ? encode_tmap(&tmB, a.B, a.K, a.N, a.ldb, 128, 32, false)
                             : encode_tmap(&tmB, a.B, a.N, a.K, a.ldb, 32, 128, true);
  if (!okA || !okB) return SGEMM_ERR_LAUNCH;
  const int64_t slots = static_cast<int64_t>(d.sm_count) * ki->ctas_per_sm;
  const int grid = static_cast<int>(num_tiles < slots ? num_tiles : slots);
  if (tc3_entry(a.ta, a.tb).launch(p, &tmA, &tmB, &tmA, &tmB, grid, stream, pdl) != cudaSuccess)
    return SGEMM_ERR_LAUNCH;
  t_last_launches = 1;
  return SGEMM_SUCCESS;
}

// 3xTF32 with the split done ahead: a memory-bound pass writes each operand's
// TF32 small parts K-major into library scratch (and, for an m/n-contiguous
// operand, the operand itself transposed, which serves as its big parts);
// the tensor-core kernel then loads big and small tiles with TMA and converts
// nothing.  Every block of A and B is split once per product instead of once
// per output tile that uses it.  Returns SGEMM_ERR_UNSUPPORTED with nothing
// queued when the scratch or a pass is unavailable.
#ifndef SG_TC_PRESPLIT
#define SG_TC_PRESPLIT 1
#endif
// SG_TC_WIDE  1: the pre-split kernel may run 256-wide tiles (0: never,
//             2: always).
#ifndef SG_TC_WIDE
#define SG_TC_WIDE 1
#endif
// Tile width of the pre-split kernel.  A 128 x 256 tile costs about 1.9
// times a 128 x 128 one on GB300 (8192^3 NN: 14 rounds of wide tiles in
// 4.09 ms against 27 rounds of narrow ones in 4.13 ms, split passes
// included); the wide tile is taken when its rounds of one tile per SM,
// times 1.9, come to fewer than the narrow tile's (2048^3: 1 round against 2;
// not 4096^3: 4 against 7).
int presplit_tile_n(const Args &a, int sm_count) {
  if (SG_TC_WIDE != 1) return SG_TC_WIDE ? 256 : 128;
  const int64_t tm = cdiv(a.M, 128);
  const int64_t narrow = cdiv(tm * cdiv(a.N, 128), sm_count), wide = cdiv(tm * cdiv(a.N, 256), sm_count);
  return 19 * wide < 10 * narrow ? 256 : 128;
}

// SG_TC_PAIR  1: run the pre-split product on CTA pairs (0: never).
#ifndef SG_TC_PAIR
#define SG_TC_PAIR 1
#endif
// SG_TC_FOLD  1: on CTA pairs, compute a k-contiguous operand's small parts
// in the kernel instead of in a split pass; 0 (default): split ahead.  The
// folded form gives the same bits but is slower on GB300 (4096^3 NT: 0.64 ms
// against 0.48 ms for the three launches split ahead): with three 64 KiB
// stages the tensor cores' two stages of lead must cover the copy, the
// conversion, the odd CTA's cluster-scope release and the accumulator
// hand-overs that share the converter warps.
#ifndef SG_TC_FOLD
#define SG_TC_FOLD 0
#endif

// Work plan on CTA pairs.  A 256 x 256 pair tile costs about 1.6 times a
// 256 x 128 one on GB300 (4096^3 NN: 4 rounds of wide tiles in 0.46 ms
// against 7 rounds of narrow ones in 0.50 ms, kernel alone).  Of three plans
// -- all narrow, all wide, or whole rounds of wide tiles with the rest of the
// tiles cut into column halves (so the last, partial round is spread over
// twice the units) -- the one of least cost in rounds is taken.
struct PairPlan {
  int bn;              // tile width of the kernel: 128 or 256
  int64_t wide_tiles;  // units [0, wide_tiles) are whole tiles
  int64_t units;       // whole tiles, then column halves of the rest
};
PairPlan plan_pair(const Args &a, int64_t clusters) {
  const int64_t tm = cdiv(a.M, 256);
  const int64_t narrow = tm * cdiv(a.N, 128), wide = tm * cdiv(a.N, 256);
  const int64_t full = wide / clusters, rest = wide - full * clusters;
  const int64_t cost_narrow = 10 * cdiv(narrow, clusters);
  const int64_t cost_wide = 16 * cdiv(wide, clusters);
  const int64_t cost_mixed = full > 0 && rest > 0 ? 16 * full + 10 * cdiv(2 * rest, clusters)
                                                  : cost_wide;
  if (SG_TC_WIDE == 0 || (SG_TC_WIDE == 1 && cost_narrow < cost_wide && cost_narrow < cost_mixed))
    return PairPlan{128, narrow, narrow};
  if (SG_TC_WIDE == 2 || cost_wide <= cost_mixed) return PairPlan{256, wide, wide};
  return PairPlan{256, full * clusters, full * clusters + 2 * rest};
}

sgemm_status_t run_tc3_presplit(const Args &a, DeviceState &d, cudaStream_t s) {
  const bool tA = a.ta == 1, tB = a.tb == 0;   // operands to transpose to K-major
  // CTA pairs if the device runs them, else one CTA per tile; on pairs a
  // k-contiguous operand's small parts are computed in the kernel (fold)
  PairPlan plan{0, 0, 0};
  const TcKernelInfo *ki = nullptr;
  bool fold_a = false, fold_b = false;
  if (SG_TC_PAIR) {
    fold_a = SG_TC_FOLD && !tA;
    fold_b = SG_TC_FOLD && !tB;
    const TcKernelInfo *k128 = tc_kernel_info_pair(d, 128, fold_a, fold_b),
                       *k256 = tc_kernel_info_pair(d, 256, fold_a, fold_b);
    if (k128 && k256) {
      plan = plan_pair(a, k256->max_ctas / 2);
      ki = plan.bn == 256 ? k256 : k128;
    }
  }
  const bool pair = ki != nullptr;
  if (!pair) {
    fold_a = fold_b = false;
    ki = tc_kernel_info_presplit(d, presplit_tile_n(a, d.sm_count));
  }
  if (!ki || ki->ctas_per_sm < 1) return SGEMM_ERR_UNSUPPORTED;
  const int64_t ldk = a.K;   // K % 4 == 0 on this path
  const size_t mat_a = (static_cast<size_t>(a.M) * ldk * sizeof(float) + 255) & ~size_t(255);
  const size_t mat_b = (static_cast<size_t>(a.N) * ldk * sizeof(float) + 255) & ~size_t(255);
  const size_t bytes_a = fold_a ? 0 : mat_a * (tA ? 2 : 1);
  const size_t bytes_b = fold_b ? 0 : mat_b * (tB ? 2 : 1);
  const bool scratch_used = bytes_a + bytes_b > 0;
  const bool capturing = stream_capturing(s);
  std::lock_guard<std::mutex> lock(d.tr_mu);
  float *scratch = nullptr;
  if (scratch_used) {
    scratch = pretranspose_scratch(d, bytes_a + bytes_b, capturing);
    if (!scratch) return SGEMM_ERR_UNSUPPORTED;
  }
  char *cur = reinterpret_cast<char *>(scratch);
  auto take = [&cur](size_t n) {
    float *q = reinterpret_cast<float *>(cur);
    cur += n;
    return q;
  };
  float *a_small = fold_a ? nullptr : take(mat_a), *a_big = (!fold_a && tA) ? take(mat_a) : nullptr;
  float *b_small = fold_b ? nullptr : take(mat_b), *b_big = (!fold_b && tB) ? take(mat_b) : nullptr;
  if (scratch_used && order_before_use(d.tr_order, s, capturing) != cudaSuccess)
    return SGEMM_ERR_LAUNCH;
  int passes = 0;
  bool done = false;
  // A: stored M x K (k along rows) or K x M
  if (!fold_a) {
    if (launch_tf32_split(a.A, a.lda, tA ? static_cast<int>(a.K) : static_cast<int>(a.M),
                          tA ? static_cast<int>(a.M) : static_cast<int>(a.K), tA, a_big, a_small,
                          ldk, d.sm_count, d.status, s, &done) != cudaSuccess)
      return SGEMM_ERR_LAUNCH;
    if (!done) return SGEMM_ERR_UNSUPPORTED;   // nothing queued yet
    ++passes;
  }
  // B: stored N x K or K x N
  if (!fold_b) {
    if (launch_tf32_split(a.B, a.ldb, tB ? static_cast<int>(a.K) : static_cast<int>(a.N),
                          tB ? static_cast<int>(a.N) : static_cast<int>(a.K), tB, b_big, b_small,
                          ldk, d.sm_count, d.status, s, &done) != cudaSuccess)
      return SGEMM_ERR_LAUNCH;
    // with the A pass queued, failing here is an error
    if (!done) return passes ? SGEMM_ERR_LAUNCH : SGEMM_ERR_UNSUPPORTED;
    ++passes;
  }
  const float *A_big = tA ? a_big : a.A, *B_big = tB ? b_big : a.B;
  const int64_t lda_big = tA ? ldk : a.lda, ldb_big = tB ? ldk : a.ldb;

  TcParams p;
  p.C = a.C;
  p.ldc = a.ldc;
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.alpha = a.alpha;
  p.beta = a.beta;
  p.tiles_m = static_cast<int>(cdiv(a.M, ki->bm));
  p.tiles_n = static_cast<int>(cdiv(a.N, ki->bn));
  p.k_tiles = static_cast<int>(cdiv(a.K, 32));
  const int64_t num_tiles = pair ? plan.units : static_cast<int64_t>(p.tiles_m) * p.tiles_n;
  if (num_tiles > kMaxDim) return SGEMM_ERR_LAUNCH;
  p.num_tiles = static_cast<int>(num_tiles);   // work units
  p.wide_tiles = pair ? static_cast<int>(plan.wide_tiles) : p.num_tiles;
  p.group_m = SG_TC_GROUP_M;
  p.c_vec4 = (a.ldc % 4 == 0) && (reinterpret_cast<uintptr_t>(a.C) % 16 == 0);
  p.wait_budget_ns = g_wait_budget_ns.load(std::memory_order_relaxed);
  p.status = d.status;
  // all K-major [rows][32 k] boxes, 128-byte swizzle: 128 rows, except
  // op(B) on CTA pairs, where each CTA loads half of a tile's n-rows
  const int b_rows = pair ? ki->bn / 2 : 128;
  // a folded operand's small-part map is not read: its big-part map stands in
  CUtensorMap tmA, tmB, tmAs, tmBs;
  if (!encode_tmap(&tmA, A_big, a.M, a.K, lda_big, 32, 128, true) ||
      !encode_tmap(&tmB, B_big, a.N, a.K, ldb_big, 32, b_rows, true))
    return SGEMM_ERR_LAUNCH;
  tmAs = tmA;
  tmBs = tmB;
  if ((!fold_a && !encode_tmap(&tmAs, a_small, a.M, a.K, ldk, 32, 128, true)) ||
      (!fold_b && !encode_tmap(&tmBs, b_small, a.N, a.K, ldk, 32, b_rows, true)))
    return SGEMM_ERR_LAUNCH;
  // persistent grid: one CTA (pair: two) per tile, at most what fits at once
  const int per_tile = pair ? 2 : 1;
  const int64_t slots = pair ? ki->max_ctas : static_cast<int64_t>(d.sm_count) * ki->ctas_per_sm;
  const int64_t want = num_tiles * per_tile;
  const int grid = static_cast<int>(want < slots ? want : slots - slots % per_tile);
  const TcEntry entry =
      pair ? tc3_pair_entry(ki->bn, fold_a, fold_b) : tc3_presplit_entry(ki->bn);
  if (entry.launch(p, &tmA, &tmB, &tmAs, &tmBs, grid, s, false) != cudaSuccess)
    return SGEMM_ERR_LAUNCH;
  t_last_launches = 1 + passes;
  if (scratch_used && order_after_use(d.tr_order, s, capturing) != cudaSuccess)
    return SGEMM_ERR_LAUNCH;
  return SGEMM_SUCCESS;
}

}  // namespace

namespace sg {
SimtEntry simt_entry_kTma_0(int transB, int tile, int csk);
SimtEntry simt_entry_kTma_1(int transB, int tile, int csk);
SimtEntry simt_entry_kCpAsync_0(int transB, int tile, int csk);
SimtEntry simt_entry_kCpAsync_1(int transB, int tile, int csk);

SimtEntry simt_entry(int producer, int transA, int transB, int tile, int csk) {
  if (producer == kTma)
    return transA ? simt_entry_kTma_1(transB, tile, csk) : simt_entry_kTma_0(transB, tile, csk);
  return transA ? simt_entry_kCpAsync_1(transB, tile, csk) : simt_entry_kCpAsync_0(transB, tile, csk);
}
}  // namespace sg

extern "C" {

sgemm_status_t sgemm_ex(int transA, int transB, int64_t M, int64_t N, int64_t K, float alpha,
                        const float *A, int64_t lda, const float *B, int64_t ldb, float beta,
                        float *C, int64_t ldc, void *stream, sgemm_algo_t algo) {
  Args a{norm_op(transA), norm_op(transB), M, N, K, alpha, beta, A, lda, B, ldb, C, ldc};
  if (static_cast<int>(algo) < SGEMM_ALGO_AUTO || static_cast<int>(algo) > SGEMM_ALGO_REG_4X4)
    return SGEMM_ERR_INVALID_VALUE;
  sgemm_status_t st = validate(a, true);
  if (st != SGEMM_SUCCESS) return st;
  t_last_launches = 0;
  if (M == 0 || N == 0) return SGEMM_SUCCESS;

  sgemm_status_t why = SGEMM_SUCCESS;
  DeviceState *d = device_state(&why);
  if (!d) return why;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  if (K == 0 || alpha == 0.0f) {
    if (launch_scale_c(C, ldc, static_cast<int>(M), static_cast<int>(N), beta, s) != cudaSuccess)
      return SGEMM_ERR_LAUNCH;
    t_last_launches = 1;
    return SGEMM_SUCCESS;
  }

  if (algo == SGEMM_ALGO_AUTO && !small_wanted(a) && repack_wanted(a)) {
    const sgemm_status_t st = run_pretransposed(a, *d, s, repack_plan(a, d->sm_count), false);
    if (st != SGEMM_ERR_UNSUPPORTED) return st;
    algo = SGEMM_ALGO_SIMT_CPASYNC;   // no scratch: run in place
  }
  if (algo == SGEMM_ALGO_AUTO) algo = auto_algo(a);
  switch (algo) {
    case SGEMM_ALGO_SIMT_TMA: {
      if (!tma_eligible(a)) return SGEMM_ERR_UNSUPPORTED;
      const Pretranspose t = pretranspose_plan(a, d->sm_count, 256);
      if (t.any()) {
        const sgemm_status_t st = run_pretransposed(a, *d, s, t, false);
        if (st != SGEMM_ERR_UNSUPPORTED) return st;
      }
      return run_simt(a, *d, kTma, s);
    }
    case SGEMM_ALGO_SIMT_CPASYNC:
      return run_simt(a, *d, kCpAsync, s);
    case SGEMM_ALGO_NAIVE:
    case SGEMM_ALGO_SMEM_TILED:
    case SGEMM_ALGO_SMALL:
    case SGEMM_ALGO_REG_2X2:
    case SGEMM_ALGO_REG_4X4: {
      PlainParams p{A, B, C, lda, ldb, ldc, static_cast<int>(M), static_cast<int>(N),
                    static_cast<int>(K), a.ta, a.tb, alpha, beta, d->status};
      cudaError_t e = algo == SGEMM_ALGO_NAIVE       ? launch_naive(p, s)
                      : algo == SGEMM_ALGO_SMEM_TILED ? launch_smem_tiled(p, s)
                      : algo == SGEMM_ALGO_REG_2X2    ? launch_reg_tiled(p, 2, s)
                      : algo == SGEMM_ALGO_REG_4X4    ? launch_reg_tiled(p, 4, s)
                                                      : launch_small(p, s);
      if (e == cudaErrorInvalidValue) return SGEMM_ERR_UNSUPPORTED;
      if (e != cudaSuccess) return SGEMM_ERR_LAUNCH;
      t_last_launches = 1;
      return SGEMM_SUCCESS;
    }
    case SGEMM_ALGO_TC_3XTF32: {
      if (!tma_eligible(a)) return SGEMM_ERR_UNSUPPORTED;
      // the tensor-core kernel is fastest with both operands m/n-contiguous
      // (they pass through its raw ring, which decouples TMA from the MMA
      // stages), so large products transpose k-contiguous operands ahead too
      const Pretranspose t = pretranspose_plan(a, d->sm_count, 128);
      // large products: split ahead (K % 4 == 0 keeps the split pass vectorised)
      if (SG_TC_PRESPLIT && presplit_size_ok(a, d->sm_count) && a.K % 4 == 0) {
        const sgemm_status_t st = run_tc3_presplit(a, *d, s);
        if (st != SGEMM_ERR_UNSUPPORTED) return st;
      }
      if (t.any()) {
        const sgemm_status_t st = run_pretransposed(a, *d, s, t, true);
        if (st != SGEMM_ERR_UNSUPPORTED) return st;
      }
      return run_tc3(a, *d, s);
    }
    default:
      return SGEMM_ERR_UNSUPPORTED;
  }
}

sgemm_status_t sgemm(int transA, int transB, int64_t M, int64_t N, int64_t K, float alpha,
                     const float *A, int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                     int64_t ldc, void *stream) {
  return sgemm_ex(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream,
                  SGEMM_ALGO_AUTO);
}

// SG_BATCH_TRANSPOSE_B 1: a strided batch of k-contiguous op(B) stored as
// dense consecutive N x K blocks is transposed once, as one (batch * N) x K
// matrix, into library scratch: product b's op(B) becomes columns
// [b * N, (b + 1) * N) of the K x (batch * N) copy (ldb = batch * N rounded
// to 4, batch stride N), n-contiguous, so the batch runs the 128 x 256 tile
// that a k-contiguous op(B) cannot use.  Taken only where that tile is the
// one the transposed batch gets and each product has at least
// SG_BATCH_TRANSPOSE_B_MIN_M rows: the copy costs a launch and 8 bytes per
// element of B, the wider tile saves about a tenth of the product (GB300,
// 64 x 1024x1024x64 NT 195.0 -> 174.7 us; 96 x 512x512x64 NT 81.5 -> 82.4,
// so not taken there).  0: never.
#ifndef SG_BATCH_TRANSPOSE_B
#define SG_BATCH_TRANSPOSE_B 1
#endif
#ifndef SG_BATCH_TRANSPOSE_B_MIN_M
#define SG_BATCH_TRANSPOSE_B_MIN_M 1024
#endif

namespace {
sgemm_status_t run_batched_transposed_b(const Args &a, DeviceState &d, cudaStream_t s, int64_t batch,
                                        int64_t strideA, int64_t strideC) {
  const int64_t rows = batch * a.N, ld2 = round4(rows);
  if (!SG_BATCH_TRANSPOSE_B || a.tb != 1 || a.N % 4 != 0 || a.M < SG_BATCH_TRANSPOSE_B_MIN_M ||
      rows > kMaxDim)
    return SGEMM_ERR_UNSUPPORTED;
  Args b = a;
  b.tb = 0;
  b.ldb = ld2;
  if (pick_simt_tile(b, kTma, d.sm_count, batch) != kTile128x256) return SGEMM_ERR_UNSUPPORTED;
  const size_t bytes = static_cast<size_t>(a.K) * ld2 * sizeof(float);
  const bool capturing = stream_capturing(s);
  std::lock_guard<std::mutex> lock(d.tr_mu);
  float *scratch = pretranspose_scratch(d, bytes, capturing);
  if (!scratch) return SGEMM_ERR_UNSUPPORTED;
  // a call on another stream (or a graph) may still be reading the scratch
  if (order_before_use(d.tr_order, s, capturing) != cudaSuccess) return SGEMM_ERR_LAUNCH;
  b.B = scratch;
  const PreLaunch copy = [&]() -> cudaError_t {
    return launch_transpose(a.B, a.ldb, scratch, ld2, static_cast<int>(rows), static_cast<int>(a.K),
                            d.sm_count, d.status, s);
  };
  const sgemm_status_t st =
      run_simt(b, d, kTma, s, Batch{batch, strideA, a.N, strideC}, /*pdl=*/true, &copy);
  if (st != SGEMM_SUCCESS) return st;
  t_last_launches += 1;
  if (order_after_use(d.tr_order, s, capturing) != cudaSuccess) return SGEMM_ERR_LAUNCH;
  return SGEMM_SUCCESS;
}
}  // namespace

sgemm_status_t sgemm_strided_batched(int transA, int transB, int64_t M, int64_t N, int64_t K,
                                     float alpha, const float *A, int64_t lda, int64_t strideA,
                                     const float *B, int64_t ldb, int64_t strideB, float beta,
                                     float *C, int64_t ldc, int64_t strideC, int64_t batch,
                                     void *stream) {
  Args a{norm_op(transA), norm_op(transB), M, N, K, alpha, beta, A, lda, B, ldb, C, ldc};
  if (batch < 0 || batch > kMaxDim || strideA < 0 || strideB < 0 || strideC < 0 ||
      strideA > kMaxLd || strideB > kMaxLd || strideC > kMaxLd)
    return SGEMM_ERR_INVALID_VALUE;
  t_last_launches = 0;
  sgemm_status_t st = batch == 0 ? validate_shape(a) : validate(a, true);
  if (st != SGEMM_SUCCESS || batch == 0 || M == 0 || N == 0) return st;
  const bool need_ab = K > 0 && alpha != 0.0f;
  using u128 = unsigned __int128;
  // elements spanned by one stored operand of rows x cols with leading dimension ld
  auto span = [](int64_t rows, int64_t cols, int64_t ld) -> u128 {
    return static_cast<u128>(rows - 1) * static_cast<u128>(ld) + static_cast<u128>(cols);
  };
  const int64_t ar = a.ta ? K : M, ac = a.ta ? M : K, br = a.tb ? N : K, bc = a.tb ? K : N;
  if (batch > 1) {
    // the C_b must not overlap one another, and the byte range of all C_b must
    // not overlap that of all A_b or all B_b
    if (static_cast<u128>(strideC) < span(M, N, ldc)) return SGEMM_ERR_ALIASING;
    auto range = [&](const void *ptr, u128 one, int64_t stride, u128 *lo, u128 *hi) {
      *lo = reinterpret_cast<uintptr_t>(ptr);
      *hi = *lo + 4 * (one + static_cast<u128>(batch - 1) * static_cast<u128>(stride));
    };
    if (need_ab) {
      u128 c0, c1, x0, x1;
      range(C, span(M, N, ldc), strideC, &c0, &c1);
      range(A, span(ar, ac, lda), strideA, &x0, &x1);
      if (c0 < x1 && x0 < c1) return SGEMM_ERR_ALIASING;
      range(B, span(br, bc, ldb), strideB, &x0, &x1);
      if (c0 < x1 && x0 < c1) return SGEMM_ERR_ALIASING;
    }
  }
  sgemm_status_t why = SGEMM_SUCCESS;
  DeviceState *d = device_state(&why);
  if (!d) return why;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!need_ab) {
    if (launch_scale_c_batched(C, ldc, strideC, static_cast<int>(M), static_cast<int>(N), batch,
                               beta, s) != cudaSuccess)
      return SGEMM_ERR_LAUNCH;
    t_last_launches = 1;
    return SGEMM_SUCCESS;
  }
  // TMA: 16-byte aligned bases, rows and batch strides
  const bool tma = tma_eligible(a) && (batch == 1 || (strideA % 4 == 0 && strideB % 4 == 0));
  // k-contiguous op(B) in dense consecutive blocks: transposed once, ahead
  if (tma && batch > 1 && a.tb == 1 && strideB == N * ldb) {
    const sgemm_status_t tst = run_batched_transposed_b(a, *d, s, batch, strideA, strideC);
    if (tst != SGEMM_ERR_UNSUPPORTED) return tst;
  }
  return run_simt(a, *d, tma ? kTma : kCpAsync, s, Batch{batch, strideA, strideB, strideC});
}

int sgemm_select_algo(int transA, int transB, int64_t M, int64_t N, int64_t K, const float *A,
                      int64_t lda, const float *B, int64_t ldb, float alpha, float beta,
                      const float *C, int64_t ldc) {
  Args a{norm_op(transA), norm_op(transB), M, N, K, alpha, beta, A, lda, B, ldb,
         const_cast<float *>(C), ldc};
  if (validate(a, false) != SGEMM_SUCCESS) return -1;
  if (!small_wanted(a) && repack_wanted(a)) return SGEMM_ALGO_SIMT_TMA;
  return static_cast<int>(auto_algo(a));
}

int sgemm_last_launch_count(void) { return t_last_launches; }

sgemm_status_t sgemm_last_device_status(void *stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return SGEMM_ERR_LAUNCH;
  }
  sgemm_status_t why = SGEMM_SUCCESS;
  DeviceState *d = device_state(&why);
  if (!d) return why;
  int v = 0;
  if (cudaMemcpy(&v, d->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return SGEMM_ERR_LAUNCH;
  }
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(d->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) {
      cudaGetLastError();
      return SGEMM_ERR_LAUNCH;
    }
    // a kernel that gave up a wait may have left arrival counters mid-count
    std::lock_guard<std::mutex> lock(d->ws_mu);
    if (d->sk_count && cudaMemset(d->sk_count, 0, kSkCounters * sizeof(int)) != cudaSuccess) {
      cudaGetLastError();
      return SGEMM_ERR_LAUNCH;
    }
  }
  if (v == 0) return SGEMM_SUCCESS;
  return v == kDevBounds ? SGEMM_ERR_DEVICE_BOUNDS : SGEMM_ERR_DEVICE_TIMEOUT;
}

sgemm_status_t sgemm_set_scratch_limit(uint64_t bytes) {
  sgemm_status_t why = SGEMM_SUCCESS;
  DeviceState *d = device_state(&why);
  if (!d) return why;
  d->limit.store(bytes);
  if (d->held.load() <= bytes) return SGEMM_SUCCESS;
  // Over the new limit: free the buffers no captured graph may still use
  // (cudaFree waits for the device's queued work, which may still read them).
  {
    std::lock_guard<std::mutex> lock(d->ws_mu);
    if (d->ws && !d->ws_order.in_graph) {
      if (cudaFree(d->ws) != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_LAUNCH;
      }
      release_scratch(*d, stream_k_workspace_bytes(*d));
      d->ws = nullptr;
      d->ws_bytes = 0;
      d->sk_count = nullptr;
    }
  }
  std::lock_guard<std::mutex> lock(d->tr_mu);
  if (d->tr && !d->tr_order.in_graph) {
    if (cudaFree(d->tr) != cudaSuccess) {
      cudaGetLastError();
      return SGEMM_ERR_LAUNCH;
    }
    release_scratch(*d, d->tr_bytes);
    d->tr = nullptr;
    d->tr_bytes = 0;
  }
  return SGEMM_SUCCESS;
}

sgemm_status_t sgemm_get_scratch_limit(uint64_t *limit, uint64_t *held) {
  sgemm_status_t why = SGEMM_SUCCESS;
  DeviceState *d = device_state(&why);
  if (!d) return why;
  if (limit) *limit = d->limit.load();
  if (held) *held = d->held.load();
  return SGEMM_SUCCESS;
}

void sgemm_set_wait_budget_ns(uint64_t budget_ns) {
  g_wait_budget_ns.store(budget_ns ? budget_ns : kDefaultWaitBudgetNs, std::memory_order_relaxed);
}

sgemm_status_t sgemm_selftest_wait_timeout(uint64_t budget_ns, void *stream) {
  sgemm_status_t why = SGEMM_SUCCESS;
  DeviceState *d = device_state(&why);
  if (!d) return why;
  if (launch_wait_selftest(budget_ns, d->status, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SGEMM_ERR_LAUNCH;
  return SGEMM_SUCCESS;
}

const char *sgemm_status_string(sgemm_status_t status) {
  switch (status) {
    case SGEMM_SUCCESS: return "success";
    case SGEMM_ERR_INVALID_VALUE: return "invalid value";
    case SGEMM_ERR_ALIASING: return "C overlaps A or B";
    case SGEMM_ERR_UNSUPPORTED: return "unsupported device or arguments";
    case SGEMM_ERR_LAUNCH: return "CUDA launch failure";
    case SGEMM_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait";
    case SGEMM_ERR_SCRATCH_LIMIT: return "needs more scratch than the fixed no-allocation array holds";
    case SGEMM_ERR_DEVICE_BOUNDS: return "a kernel caught an out-of-range index (debug-bounds build)";
    default: return "unknown status";
  }
}

const char *sgemm_algo_name(sgemm_algo_t algo) {
  switch (algo) {
    case SGEMM_ALGO_AUTO: return "auto";
    case SGEMM_ALGO_SIMT_TMA: return "simt_tma";
    case SGEMM_ALGO_SIMT_CPASYNC: return "simt_cpasync";
    case SGEMM_ALGO_TC_3XTF32: return "tc_3xtf32";
    case SGEMM_ALGO_NAIVE: return "naive";
    case SGEMM_ALGO_SMEM_TILED: return "smem_tiled";
    case SGEMM_ALGO_SMALL: return "small";
    case SGEMM_ALGO_REG_2X2: return "reg_2x2";
    case SGEMM_ALGO_REG_4X4: return "reg_4x4";
    default: return "unknown";
  }
}

const char *sgemm_version(void) { return "0.1.0"; }

}  // extern "C"
