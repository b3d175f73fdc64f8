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
//     32-byte sectors; the eight warps of a CTA, stacked down the input,
//     complete 512 contiguous bytes of every output row they touch).
// Loads and stores use the streaming cache hint: nothing is read twice.
//
// Edges: a thread whose 4 x 4 block is not entirely inside the matrix, or any
// call whose pointers / leading dimensions are not 16-byte aligned, copies
// element by element with bounds checks (same mapping, scalar accesses).
//
// Roofline: HBM, 2 * rows * cols * 4 bytes per launch.
#include <cstdint>

#include "dispatch.h"
#include "internal.h"
#include "sgemm.h"

namespace sg {
namespace {

constexpr int kWarps = 8;                       // CTA: 8 warps stacked along the rows
constexpr int kCtaRows = kWarps * 16;           // 16 input rows per warp
constexpr int kCtaCols = 32;                    // 8 lanes x 4 columns
constexpr int kCtasPerSm = 8;                   // 2048 threads per SM

struct TransposeParams {
  const float *in;
  float *out;
  int64_t ld_in, ld_out;
  int rows, cols;
  int64_t row_blocks;   // ceil(rows / kCtaRows)
  int64_t num_blocks;   // row_blocks * ceil(cols / kCtaCols)
  int vec;              // 16-byte aligned bases and leading dimensions
};

__global__ void __launch_bounds__(kWarps * 32) transpose_kernel(const TransposeParams p) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int bi = lane >> 3, bj = lane & 7;   // this thread's 4 x 4 block within the warp's 16 x 32
  for (int64_t blk = blockIdx.x; blk < p.num_blocks; blk += gridDim.x) {
    // consecutive CTAs walk down the rows of one 32-column strip, so the
    // output rows of that strip fill contiguously
    const int64_t strip = blk / p.row_blocks, rb = blk - strip * p.row_blocks;
    const int r = static_cast<int>(rb * kCtaRows) + warp * 16 + 4 * bi;
    const int c = static_cast<int>(strip * kCtaCols) + 4 * bj;
    if (r >= p.rows || c >= p.cols) continue;
    if (p.vec && r + 4 <= p.rows && c + 4 <= p.cols) {
      float4 v[4];
#pragma unroll
      for (int a = 0; a < 4; ++a)
        v[a] = __ldcs(reinterpret_cast<const float4 *>(p.in + static_cast<int64_t>(r + a) * p.ld_in + c));
      __stcs(reinterpret_cast<float4 *>(p.out + static_cast<int64_t>(c + 0) * p.ld_out + r),
             make_float4(v[0].x, v[1].x, v[2].x, v[3].x));
      __stcs(reinterpret_cast<float4 *>(p.out + static_cast<int64_t>(c + 1) * p.ld_out + r),
             make_float4(v[0].y, v[1].y, v[2].y, v[3].y));
      __stcs(reinterpret_cast<float4 *>(p.out + static_cast<int64_t>(c + 2) * p.ld_out + r),
             make_float4(v[0].z, v[1].z, v[2].z, v[3].z));
      __stcs(reinterpret_cast<float4 *>(p.out + static_cast<int64_t>(c + 3) * p.ld_out + r),
             make_float4(v[0].w, v[1].w, v[2].w, v[3].w));
    } else {
      const int ra = min(4, p.rows - r), cb = min(4, p.cols - c);
      for (int a = 0; a < ra; ++a)
        for (int b = 0; b < cb; ++b)
          p.out[static_cast<int64_t>(c + b) * p.ld_out + r + a] =
              p.in[static_cast<int64_t>(r + a) * p.ld_in + c + b];
    }
  }
}

}  // namespace
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

  TransposeParams p;
  p.in = in;
  p.out = out;
  p.ld_in = ld_in;
  p.ld_out = ld_out;
  p.rows = static_cast<int>(rows);
  p.cols = static_cast<int>(cols);
  p.row_blocks = cdiv(rows, kCtaRows);
  p.num_blocks = p.row_blocks * cdiv(cols, kCtaCols);
  p.vec = (reinterpret_cast<uintptr_t>(in) % 16 == 0) && (reinterpret_cast<uintptr_t>(out) % 16 == 0) &&
          (ld_in % 4 == 0) && (ld_out % 4 == 0);
  const int64_t slots = static_cast<int64_t>(d->sm_count) * kCtasPerSm;
  const int64_t grid = p.num_blocks < slots ? p.num_blocks : slots;
  transpose_kernel<<<static_cast<unsigned>(grid), kWarps * 32, 0,
                     reinterpret_cast<cudaStream_t>(stream)>>>(p);
  if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
  t_last_launches = 1;
  return SGEMM_SUCCESS;
}
