// repack.cu -- copies of matrices with any alignment into 16-byte aligned
// rows, so that a product on operands the TMA unit cannot address (a leading
// dimension not a multiple of 4 floats, or a base not 16-byte aligned) can
// run on the TMA kernel from library scratch instead of the 4-byte cp.async
// producer.  Values are copied bit for bit.
#include <cstdint>

#include "dispatch.h"
#include "ptx.cuh"

namespace sg {

// Copies of up to two rows x cols matrices of any alignment into 16-byte
// aligned rows (ld_out a multiple of 4), in one launch.  A unit is one float4
// of output; units are numbered row by row, cols4 = ceil(cols / 4) per row.
// Each warp takes 128 consecutive units: its lanes read the 512 source floats
// with consecutive addresses (coalesced whatever the source alignment),
// stage them in shared memory and store float4s.  Row padding gets zeros.
struct RepackJob {
  const float *in;
  int64_t ld_in;
  float *out;
  int64_t ld_out;
  int cols, cols4;
  int64_t units;   // rows * cols4
};
constexpr int kRepackThreads = 256, kRepackUnitsPerWarp = 128;
constexpr int kRepackUnitsPerBlock = kRepackUnitsPerWarp * kRepackThreads / 32;

__global__ void __launch_bounds__(kRepackThreads) repack_kernel(const RepackJob j0, const RepackJob j1,
                                                                int64_t blocks0) {
  griddep_launch_dependents();
  __shared__ __align__(16) float stage[kRepackThreads / 32][4 * kRepackUnitsPerWarp];
  const bool first = blockIdx.x < blocks0;
  const RepackJob &j = first ? j0 : j1;
  const int64_t block = first ? blockIdx.x : blockIdx.x - blocks0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t u0 = block * kRepackUnitsPerBlock + warp * kRepackUnitsPerWarp;
  if (u0 >= j.units) return;
  float *sw = stage[warp];
  // row and column (in units) of the span's first unit; the others follow
  // by a 32-bit division only where the span wraps to a later row
  const int64_t r0 = u0 / j.cols4;
  const int c0 = static_cast<int>(u0 - r0 * j.cols4);
  const auto locate = [&](int w, int64_t &r, int &cu) {
    r = r0;
    cu = c0 + w;
    if (cu >= j.cols4) {
      const int d = cu / j.cols4;
      r += d;
      cu -= d * j.cols4;
    }
  };
  // all loads first (each lane has kLoads in flight), then the stage
  constexpr int kLoads = 4 * kRepackUnitsPerWarp / 32;
  float v[kLoads];
#pragma unroll
  for (int q = 0; q < kLoads; ++q) {
    const int e = q * 32 + lane;            // element of this warp's span
    v[q] = 0.0f;
    if (u0 + (e >> 2) < j.units) {
      int64_t r;
      int cu;
      locate(e >> 2, r, cu);
      const int c = 4 * cu + (e & 3);
      if (c < j.cols) v[q] = __ldcs(j.in + r * j.ld_in + c);
    }
  }
#pragma unroll
  for (int q = 0; q < kLoads; ++q) sw[q * 32 + lane] = v[q];
  __syncwarp();
#pragma unroll
  for (int q = 0; q < kRepackUnitsPerWarp / 32; ++q) {
    const int w = q * 32 + lane;            // unit of this warp's span
    if (u0 + w >= j.units) break;
    int64_t r;
    int cu;
    locate(w, r, cu);
    *reinterpret_cast<float4 *>(j.out + r * j.ld_out + 4 * cu) = *reinterpret_cast<const float4 *>(sw + 4 * w);
  }
}

RepackJob repack_job(const float *in, int64_t ld_in, int rows, int cols, float *out, int64_t ld_out) {
  RepackJob j;
  j.in = in;
  j.ld_in = ld_in;
  j.out = out;
  j.ld_out = ld_out;
  j.cols = cols;
  j.cols4 = (cols + 3) / 4;
  j.units = static_cast<int64_t>(rows) * j.cols4;
  return j;
}

cudaError_t launch_repack(const float *in0, int64_t ld_in0, int rows0, int cols0, float *out0,
                          int64_t ld_out0, const float *in1, int64_t ld_in1, int rows1, int cols1,
                          float *out1, int64_t ld_out1, cudaStream_t s) {
  const RepackJob j0 = repack_job(in0, ld_in0, rows0, cols0, out0, ld_out0);
  const RepackJob j1 = in1 ? repack_job(in1, ld_in1, rows1, cols1, out1, ld_out1)
                           : repack_job(nullptr, 0, 0, 0, nullptr, 4);
  const int64_t b0 = (j0.units + kRepackUnitsPerBlock - 1) / kRepackUnitsPerBlock;
  const int64_t b1 = (j1.units + kRepackUnitsPerBlock - 1) / kRepackUnitsPerBlock;
  if (b0 + b1 == 0) return cudaSuccess;
  if (b0 + b1 > 0x7fffffff) return cudaErrorInvalidValue;
  repack_kernel<<<static_cast<unsigned>(b0 + b1), kRepackThreads, 0, s>>>(j0, j1, b0);
  return cudaGetLastError();
}

}  // namespace sg
