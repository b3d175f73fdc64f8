// transpose.cu -- out = in^T for a row-major FP32 matrix, and its C-ABI entry
// point sgemm_transpose().
//
// The workload of "现代 CUDA 工具箱实战：从朴素代码到硬件极限的优化之路" (hankli.space):
// a matrix transpose whose cost is all memory traffic.  The page moves each
// 32 x 32 tile through shared memory (one padding column against bank
// conflicts) so that both the global read and the global write run along
// rows.  Here no shared memory is needed: each thread reads a 4 x 4 block
// with four 16-byte loads (four input rows), swaps it in registers and writes
// four 16-byte stores (four output rows).  The lanes of a warp form 4 rows x 8
// columns of such blocks, so
//   * each load instruction reads 4 input rows x 128 contiguous bytes (whole
//     128-byte lines), and
//   * each store instruction writes 8 output rows x 64 contiguous bytes (whole
//     32-byte sectors; a CTA's 64 x 64 tile completes 256 contiguous bytes of
//     each of its 64 output rows).
// Loads and stores use the streaming cache hint: nothing is read twice.
//
// Edges: a thread whose 4 x 4 block is not entirely inside the matrix, or any
// call whose pointers / leading dimensions are not 16-byte aligned, copies
// element by element with bounds checks (same mapping, scalar accesses).
//
// Roofline: HBM, 2 * rows * cols * 4 bytes per launch.
#include <cstdint>
#include <cstring>
#include <mutex>

#include "dispatch.h"
#include "internal.h"
#include "sgemm.h"

namespace sg {
namespace {

// CTA tile: 64 x 64 input elements; its 8 warps are 4 (down) x 2 (across),
// each warp 16 rows x 32 columns of 4 x 4 thread blocks.
constexpr int kWarps = 8;
constexpr int kTile = 64;
constexpr int kCtasPerSm = 8;                   // 2048 threads per SM
// Tiles are visited in groups of kGroup tile-rows, column by column inside a
// group, so the CTAs in flight cover a compact band: long contiguous runs of
// both the input rows and the output rows (DRAM page locality).
#ifndef SG_TRANSPOSE_GROUP
#define SG_TRANSPOSE_GROUP 16
#endif
constexpr int kGroup = SG_TRANSPOSE_GROUP;
// 1: streaming (evict-first) cache hints on the loads and stores.
#ifndef SG_TRANSPOSE_STREAMING
#define SG_TRANSPOSE_STREAMING 1
#endif

__device__ __forceinline__ float4 load4(const float *p) {
  if (SG_TRANSPOSE_STREAMING) return __ldcs(reinterpret_cast<const float4 *>(p));
  return *reinterpret_cast<const float4 *>(p);
}
__device__ __forceinline__ void store4(float *p, float4 v) {
  if (SG_TRANSPOSE_STREAMING)
    __stcs(reinterpret_cast<float4 *>(p), v);
  else
    *reinterpret_cast<float4 *>(p) = v;
}

struct TransposeParams {
  const float *in;
  float *out;
  int64_t ld_in, ld_out;
  int rows, cols;
  int tiles_r, tiles_c;   // ceil(rows / 64), ceil(cols / 64)
  int64_t num_tiles;
  int vec;                // 16-byte aligned bases and leading dimensions
};

// SG_TRANSPOSE_ILP tiles per loop trip: all their loads are issued before
// any store, so each thread keeps ILP * 64 bytes of reads in flight.
#ifndef SG_TRANSPOSE_ILP
#define SG_TRANSPOSE_ILP 1
#endif
constexpr int kIlp = SG_TRANSPOSE_ILP;

// Origin (r, c) of this thread's 4 x 4 block in tile t, or r = -1 past the end.
__device__ __forceinline__ void block_origin(const TransposeParams &p, int64_t t, int r_in, int c_in,
                                             int &r, int &c) {
  r = -1;
  c = 0;
  if (t >= p.num_tiles) return;
  const int64_t per_group = static_cast<int64_t>(kGroup) * p.tiles_c;
  const int64_t g = t / per_group, i = t - g * per_group;
  const int64_t first = g * kGroup;
  const int64_t rows_here = (p.tiles_r - first < kGroup) ? p.tiles_r - first : kGroup;
  const int64_t tr = first + i % rows_here, tc = i / rows_here;
  r = static_cast<int>(tr * kTile) + r_in;
  c = static_cast<int>(tc * kTile) + c_in;
  if (r >= p.rows || c >= p.cols) r = -1;
}

__device__ __forceinline__ void copy_block_scalar(const TransposeParams &p, int r, int c) {
  const int ra = min(4, p.rows - r), cb = min(4, p.cols - c);
  for (int a = 0; a < ra; ++a)
    for (int b = 0; b < cb; ++b)
      p.out[static_cast<int64_t>(c + b) * p.ld_out + r + a] = p.in[static_cast<int64_t>(r + a) * p.ld_in + c + b];
}

__global__ void __launch_bounds__(kWarps * 32) transpose_kernel(const TransposeParams p) {
  griddep_launch_dependents();   // a product that reads our output may be scheduled
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r_in = (warp >> 1) * 16 + 4 * (lane >> 3);   // thread block origin inside the tile
  const int c_in = (warp & 1) * 32 + 4 * (lane & 7);
  const int64_t step = static_cast<int64_t>(gridDim.x) * kIlp;
  for (int64_t t0 = blockIdx.x; t0 < p.num_tiles; t0 += step) {
    int r[kIlp], c[kIlp];
    bool fast = p.vec != 0;
#pragma unroll
    for (int u = 0; u < kIlp; ++u) {
      block_origin(p, t0 + static_cast<int64_t>(u) * gridDim.x, r_in, c_in, r[u], c[u]);
      fast = fast && r[u] >= 0 && r[u] + 4 <= p.rows && c[u] + 4 <= p.cols;
    }
    if (fast) {
      float4 v[kIlp][4];
#pragma unroll
      for (int u = 0; u < kIlp; ++u)
#pragma unroll
        for (int a = 0; a < 4; ++a) v[u][a] = load4(p.in + static_cast<int64_t>(r[u] + a) * p.ld_in + c[u]);
#pragma unroll
      for (int u = 0; u < kIlp; ++u) {
        float *o = p.out + static_cast<int64_t>(c[u]) * p.ld_out + r[u];
        store4(o, make_float4(v[u][0].x, v[u][1].x, v[u][2].x, v[u][3].x));
        store4(o + p.ld_out, make_float4(v[u][0].y, v[u][1].y, v[u][2].y, v[u][3].y));
        store4(o + 2 * p.ld_out, make_float4(v[u][0].z, v[u][1].z, v[u][2].z, v[u][3].z));
        store4(o + 3 * p.ld_out, make_float4(v[u][0].w, v[u][1].w, v[u][2].w, v[u][3].w));
      }
    } else {
      for (int u = 0; u < kIlp; ++u)
        if (r[u] >= 0) copy_block_scalar(p, r[u], c[u]);
    }
  }
}

// ------------------------------------------------------------ TMA-staged form
// For 16-byte aligned layouts.  A tile is 128 input rows x 32 input columns.
// One producer thread loads it with a TMA box (32 x 128, 128-byte swizzle:
// 16-byte chunk j of row r sits at chunk j ^ (r mod 8)) into a 4-deep ring;
// four consumer warps read it column-wise -- thread t takes row t, one
// 16-byte chunk (4 columns) per LDS.128, conflict-free thanks to the swizzle
// -- and write the 32 x 128 output tile densely (a warp's 32 stores of one
// output row are consecutive words); one consumer thread then stores it with
// a TMA box (128 x 32), which also clips the ragged edges.  Shared memory,
// not registers, holds the bytes in flight: up to 4 input and 2 output tiles
// (96 KiB) per CTA, two CTAs per SM.
constexpr int kTmRows = 128, kTmCols = 32;
constexpr int kTmTileBytes = kTmRows * kTmCols * 4;   // 16 KiB, same for in and out
constexpr int kTmOutStages = 2;
constexpr int kTmConsumers = 128;                     // warps 1..4
constexpr int kTmThreads = 32 + kTmConsumers;
// SPLIT: the split pass of the 3xTF32 product -- besides the transposed
// values (which serve as the TF32 big parts) each output tile gets a twin
// holding the small parts; one input stage fewer keeps two CTAs per SM.
// Input stages of the plain form (16 KiB each): 4 fit two CTAs per SM, 2
// fit three.
#ifndef SG_TRANSPOSE_IN_STAGES
#define SG_TRANSPOSE_IN_STAGES 4
#endif
template <bool SPLIT>
struct TmShape {
  static constexpr int IN_STAGES = SPLIT ? 3 : SG_TRANSPOSE_IN_STAGES;
  static constexpr int OUT_TILES = SPLIT ? 2 : 1;   // per output stage
  static constexpr int SMEM = (IN_STAGES + kTmOutStages * OUT_TILES) * kTmTileBytes + 1024 /*align*/ +
                              64 /*barriers*/;
};
#ifndef SG_TRANSPOSE_TMA_GROUP
#define SG_TRANSPOSE_TMA_GROUP 8
#endif

struct TmaTransposeParams {
  int rows, cols;
  int tiles_r, tiles_c;          // ceil(rows / 128), ceil(cols / 32)
  int64_t num_tiles;
  uint64_t wait_budget_ns;
  int *status;
};

// Input-tile origin (r0, c0) of linear tile t: groups of G 32-column strips,
// walked down the rows inside a group.
__device__ __forceinline__ void tma_tile_origin(const TmaTransposeParams &p, int64_t t, int &r0, int &c0) {
  constexpr int G = SG_TRANSPOSE_TMA_GROUP;
  const int64_t per_group = static_cast<int64_t>(G) * p.tiles_r;
  const int64_t g = t / per_group, i = t - g * per_group;
  const int64_t first = g * G;
  const int64_t cols_here = (p.tiles_c - first < G) ? p.tiles_c - first : G;
  const int64_t tc = first + i % cols_here, tr = i / cols_here;
  r0 = static_cast<int>(tr * kTmRows);
  c0 = static_cast<int>(tc * kTmCols);
}

template <bool SPLIT>
__global__ void __launch_bounds__(kTmThreads) transpose_tma_kernel(const __grid_constant__ CUtensorMap in_map,
                                                                   const __grid_constant__ CUtensorMap out_map,
                                                                   const __grid_constant__ CUtensorMap small_map,
                                                                   const TmaTransposeParams p) {
  constexpr int kTmInStages = TmShape<SPLIT>::IN_STAGES, OUT_TILES = TmShape<SPLIT>::OUT_TILES;
  griddep_launch_dependents();   // a product that reads our output may be scheduled
  extern __shared__ unsigned char smem_raw[];
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;   // 128-byte swizzle wants 1 KiB
  const uint32_t in0 = base, out0 = base + kTmInStages * kTmTileBytes;
  const uint32_t bars = out0 + kTmOutStages * OUT_TILES * kTmTileBytes;
  const uint32_t full0 = bars, empty0 = bars + 8 * kTmInStages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTmInStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kTmConsumers / 32);
    }
    fence_mbar_init();
    tma_prefetch_desc(&in_map);
    tma_prefetch_desc(&out_map);
    if (SPLIT) tma_prefetch_desc(&small_map);
  }
  __syncthreads();

  if (warp == 0) {
    // ---- producer: one thread issues the tile loads
    if (lane != 0) return;
    uint32_t i = 0;
    for (int64_t t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++i) {
      const uint32_t s = i % kTmInStages, round = i / kTmInStages;
      if (round > 0 && !wait_parity_bounded(empty0 + 8 * s, (round - 1) & 1, p.wait_budget_ns, p.status))
        break;   // consumers give up on their own bounded waits
      int r0, c0;
      tma_tile_origin(p, t, r0, c0);
      mbar_arrive_expect_tx(full0 + 8 * s, kTmTileBytes);
      // (a debug-bounds build still issues the load, so that the barrier
      // completes; it records a tile origin outside the matrix)
      SG_CHECK(r0 >= 0 && c0 >= 0 && r0 < p.rows && c0 < p.cols, p.status);
      tma_load_2d(in0 + s * kTmTileBytes, &in_map, full0 + 8 * s, c0, r0);
    }
    // do not let the CTA end with a load of ours still landing: wait (bounded)
    // for the last loads issued in each stage
    for (uint32_t k = (i > kTmInStages ? i - kTmInStages : 0); k < i; ++k)
      wait_parity_bounded(full0 + 8 * (k % kTmInStages), (k / kTmInStages) & 1, p.wait_budget_ns, p.status);
    return;
  }

  // ---- consumers: thread ct owns input row ct of every tile
  const int ct = threadIdx.x - 32;
  uint32_t i = 0;
  for (int64_t t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++i) {
    const uint32_t s = i % kTmInStages, round = i / kTmInStages, o = i % kTmOutStages;
    bool ok = wait_parity_bounded(full0 + 8 * s, round & 1, p.wait_budget_ns, p.status);
    // the output buffer is free once the store issued kTmOutStages tiles ago
    // has read it (only the issuing thread can wait for its bulk groups)
    if (ct == 0) bulk_wait_group_read<kTmOutStages - 1>();
    if (!bar_and(1, kTmConsumers, ok)) break;   // all consumers leave together
    const uint32_t src = in0 + s * kTmTileBytes + ct * 128;
    const uint32_t dst = out0 + o * OUT_TILES * kTmTileBytes + ct * 4;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 v = lds128(src + ((j ^ (ct & 7)) << 4));
      // output row 4j + q, column ct
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(dst + (4 * j + 0) * 512), "f"(v.x) : "memory");
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(dst + (4 * j + 1) * 512), "f"(v.y) : "memory");
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(dst + (4 * j + 2) * 512), "f"(v.z) : "memory");
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(dst + (4 * j + 3) * 512), "f"(v.w) : "memory");
      if (SPLIT) {   // the small parts into the twin tile
        float b0, b1, b2, b3, s0, s1, s2, s3;
        split_pair(v.x, v.y, b0, b1, s0, s1);
        split_pair(v.z, v.w, b2, b3, s2, s3);
        const uint32_t d2 = dst + kTmTileBytes;
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(d2 + (4 * j + 0) * 512), "f"(s0) : "memory");
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(d2 + (4 * j + 1) * 512), "f"(s1) : "memory");
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(d2 + (4 * j + 2) * 512), "f"(s2) : "memory");
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(d2 + (4 * j + 3) * 512), "f"(s3) : "memory");
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
    fence_proxy_async_smem();                     // make the tile visible to the TMA store
    bar_and(1, kTmConsumers, true);
    if (ct == 0) {
      int r0, c0;
      tma_tile_origin(p, t, r0, c0);
      const uint32_t ob = out0 + o * OUT_TILES * kTmTileBytes;
      if (SG_CHECK(r0 >= 0 && c0 >= 0 && r0 < p.rows && c0 < p.cols, p.status)) {
        tma_store_2d(&out_map, ob, r0, c0);   // out: x = input row, y = input col
        if (SPLIT) tma_store_2d(&small_map, ob + kTmTileBytes, r0, c0);
      }
      bulk_commit_group();
    }
  }
  if (ct == 0) bulk_wait_group_all();
}

// Per device and form: dynamic shared memory set once, CTAs per SM.
std::once_flag g_tma_attr_once[2][kMaxDevices];
cudaError_t g_tma_attr_err[2][kMaxDevices];
int g_tma_ctas[2][kMaxDevices];

template <bool SPLIT>
cudaError_t launch_transpose_tma(const float *in, int64_t ld_in, float *out, float *small,
                                 int64_t ld_out, int rows, int cols, int sm_count, int *status,
                                 cudaStream_t s, bool *used) {
  *used = false;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cudaGetLastError();
  std::call_once(g_tma_attr_once[SPLIT][dev], [dev]() {
    cudaError_t &e = g_tma_attr_err[SPLIT][dev];
    e = cudaFuncSetAttribute(transpose_tma_kernel<SPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             TmShape<SPLIT>::SMEM);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&g_tma_ctas[SPLIT][dev], transpose_tma_kernel<SPLIT>,
                                                        kTmThreads, TmShape<SPLIT>::SMEM);
    if (e == cudaSuccess && g_tma_ctas[SPLIT][dev] < 1) e = cudaErrorInvalidConfiguration;
    if (e != cudaSuccess) cudaGetLastError();
  });
  if (g_tma_attr_err[SPLIT][dev] != cudaSuccess) return cudaSuccess;   // not used: caller decides
  CUtensorMap in_map, out_map, small_map;
  std::memset(&small_map, 0, sizeof(small_map));
  if (!encode_tmap(&in_map, in, rows, cols, ld_in, kTmCols, kTmRows, true) ||
      !encode_tmap(&out_map, out, cols, rows, ld_out, kTmRows, kTmCols, false) ||
      (SPLIT && !encode_tmap(&small_map, small, cols, rows, ld_out, kTmRows, kTmCols, false)))
    return cudaSuccess;                                            // likewise
  TmaTransposeParams p;
  p.rows = rows;
  p.cols = cols;
  p.tiles_r = static_cast<int>(cdiv(rows, kTmRows));
  p.tiles_c = static_cast<int>(cdiv(cols, kTmCols));
  p.num_tiles = static_cast<int64_t>(p.tiles_r) * p.tiles_c;
  p.wait_budget_ns = g_wait_budget_ns.load(std::memory_order_relaxed);
  p.status = status;
  const int64_t slots = static_cast<int64_t>(sm_count) * g_tma_ctas[SPLIT][dev];
  const int64_t grid = p.num_tiles < slots ? p.num_tiles : slots;
  transpose_tma_kernel<SPLIT><<<static_cast<unsigned>(grid), kTmThreads, TmShape<SPLIT>::SMEM, s>>>(
      in_map, out_map, small_map, p);
  *used = true;
  return cudaGetLastError();
}

// Small TF32 parts of a k-contiguous operand, elementwise: out[r][c] =
// small(in[r][c]) (16-byte rows on both sides).
__global__ void __launch_bounds__(256) tf32_small_kernel(const float *in, int64_t ld_in, float *out,
                                                         int64_t ld_out, int rows, int cols4) {
  griddep_launch_dependents();
  const int64_t total = static_cast<int64_t>(rows) * cols4;
  for (int64_t e = blockIdx.x * 256ll + threadIdx.x; e < total; e += static_cast<int64_t>(gridDim.x) * 256) {
    const int64_t r = e / cols4, c = 4 * (e - r * cols4);
    const float4 x = __ldcs(reinterpret_cast<const float4 *>(in + r * ld_in + c));
    float4 sm;
    float b0, b1, b2, b3;
    split_pair(x.x, x.y, b0, b1, sm.x, sm.y);
    split_pair(x.z, x.w, b2, b3, sm.z, sm.w);
    *reinterpret_cast<float4 *>(out + r * ld_out + c) = sm;
  }
}

}  // namespace

#ifndef SG_TRANSPOSE_TMA
#define SG_TRANSPOSE_TMA 1
#endif

cudaError_t launch_transpose(const float *in, int64_t ld_in, float *out, int64_t ld_out, int rows,
                             int cols, int sm_count, int *status, cudaStream_t s, bool exact_edges) {
  const bool aligned = (reinterpret_cast<uintptr_t>(in) % 16 == 0) &&
                       (reinterpret_cast<uintptr_t>(out) % 16 == 0) && (ld_in % 4 == 0) &&
                       (ld_out % 4 == 0);
  // A TMA store writes whole 16-byte granules at the inner edge of the
  // tensor: an output row of `rows` floats, rows % 4 != 0, gets up to three
  // floats written past its end (into the row's padding, or past the last
  // row).  Where nothing outside the rows may change, such shapes take the
  // register kernel.
  if (SG_TRANSPOSE_TMA && aligned && (!exact_edges || rows % 4 == 0)) {
    bool used = false;
    const cudaError_t e =
        launch_transpose_tma<false>(in, ld_in, out, nullptr, ld_out, rows, cols, sm_count, status, s, &used);
    if (used || e != cudaSuccess) return e;
  }
  TransposeParams p;
  p.in = in;
  p.out = out;
  p.ld_in = ld_in;
  p.ld_out = ld_out;
  p.rows = rows;
  p.cols = cols;
  p.tiles_r = static_cast<int>(cdiv(rows, kTile));
  p.tiles_c = static_cast<int>(cdiv(cols, kTile));
  p.num_tiles = static_cast<int64_t>(p.tiles_r) * p.tiles_c;
  p.vec = aligned;
  const int64_t slots = static_cast<int64_t>(sm_count) * kCtasPerSm;
  const int64_t grid = p.num_tiles < slots ? p.num_tiles : slots;
  transpose_kernel<<<static_cast<unsigned>(grid), kWarps * 32, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_tf32_split(const float *in, int64_t ld_in, int rows, int cols, bool transpose,
                              float *big, float *small, int64_t ld_out, int sm_count, int *status,
                              cudaStream_t s, bool *done) {
  *done = false;
  if (transpose) {
    bool used = false;
    const cudaError_t e =
        launch_transpose_tma<true>(in, ld_in, big, small, ld_out, rows, cols, sm_count, status, s, &used);
    *done = used && e == cudaSuccess;
    return e;
  }
  const int cols4 = cols / 4;   // cols % 4 == 0 for the tensor-core layouts
  const int64_t total = static_cast<int64_t>(rows) * cols4;
  int64_t grid = (total + 255) / 256;
  if (grid > sm_count * 8ll) grid = sm_count * 8ll;
  tf32_small_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(in, ld_in, small, ld_out, rows, cols4);
  const cudaError_t e = cudaGetLastError();
  *done = e == cudaSuccess;
  return e;
}

}  // namespace sg

using namespace sg;

extern "C" sgemm_status_t sgemm_transpose(int64_t rows, int64_t cols, const float *in,
                                          int64_t ld_in, float *out, int64_t ld_out,
                                          void *stream) {
  if (rows < 0 || cols < 0 || rows > kMaxDim || cols > kMaxDim) return SGEMM_ERR_INVALID_VALUE;
  if (ld_in < (cols > 1 ? cols : 1) || ld_in > kMaxLd) return SGEMM_ERR_INVALID_VALUE;
  if (ld_out < (rows > 1 ? rows : 1) || ld_out > kMaxLd) return SGEMM_ERR_INVALID_VALUE;
  t_last_launches = 0;
  if (rows == 0 || cols == 0) return SGEMM_SUCCESS;
  if (in == nullptr || out == nullptr) return SGEMM_ERR_INVALID_VALUE;
  {
    using u128 = unsigned __int128;
    const u128 i0 = reinterpret_cast<uintptr_t>(in), o0 = reinterpret_cast<uintptr_t>(out);
    const u128 i1 = i0 + 4 * (static_cast<u128>(rows - 1) * static_cast<u128>(ld_in) + cols);
    const u128 o1 = o0 + 4 * (static_cast<u128>(cols - 1) * static_cast<u128>(ld_out) + rows);
    if (i0 < o1 && o0 < i1) return SGEMM_ERR_ALIASING;   // in-place is not supported
  }
  sgemm_status_t why = SGEMM_SUCCESS;
  DeviceState *d = device_state(&why);
  if (!d) return why;

  if (launch_transpose(in, ld_in, out, ld_out, static_cast<int>(rows), static_cast<int>(cols),
                       d->sm_count, d->status, reinterpret_cast<cudaStream_t>(stream),
                       /*exact_edges=*/true) != cudaSuccess)
    return SGEMM_ERR_LAUNCH;
  t_last_launches = 1;
  return SGEMM_SUCCESS;
}
