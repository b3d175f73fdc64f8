// sk_fixup.cu -- second pass of a stream-K launch of the CUDA-core kernel.
//
// The k-iterations of the last sk tiles were divided evenly over the G CTAs of
// the main kernel; a tile whose iterations were spread over several CTAs left
// one raw partial sum per CTA segment in the workspace.  Each block takes one
// 1024-element chunk of such a tile (one float4 per thread, so even a handful
// of split tiles spreads over many SMs and no thread waits on a chain of
// loads), adds the partials in increasing k order (so the result is the same
// on every run) and writes C = alpha * sum + beta * C (C not read when
// beta == 0).
#include "internal.h"
#include "ptx.cuh"

namespace sg {

constexpr int kMaxSkSegments = 128;  // the host keeps every tile below this
constexpr int kFixupThreads = 256;
constexpr int kChunk = 4 * kFixupThreads;  // elements per block

__device__ __forceinline__ int64_t sk_start(int64_t g, int64_t S, int64_t G) { return g * S / G; }

// BATCH: partials loaded per round (all in flight at once).  Tiles split
// into many segments (small products) take 8, which costs registers; the
// usual two or three segments per tile take 1 and keep eight blocks per SM.
template <int BATCH>
__global__ void __launch_bounds__(kFixupThreads) sk_fixup_kernel(const SimtParams p, int bm, int bn,
                                                                 int grid_main) {
  const int chunks = bm * bn / kChunk;   // bm * bn is a multiple of 8192
  const int tile = blockIdx.x / chunks, chunk = blockIdx.x - tile * chunks;
  __shared__ int s_slot[kMaxSkSegments];
  __shared__ int s_count;
  if (threadIdx.x == 0) {
    const int64_t KT = p.k_tiles, S = p.sk_iters, G = grid_main;
    const int64_t it0 = static_cast<int64_t>(tile) * KT, it1 = it0 + KT;
    // CTAs whose iteration ranges meet [it0, it1), in increasing k order
    int64_t g = it0 * G / S;
    while (g + 1 < G && sk_start(g + 1, S, G) <= it0) ++g;
    while (g > 0 && sk_start(g, S, G) > it0) --g;
    int n = 0;
    for (; g < G; ++g) {
      const int64_t a = sk_start(g, S, G), b = sk_start(g + 1, S, G);
      if (a >= it1) break;
      if ((a > it0 ? a : it0) >= (b < it1 ? b : it1)) continue;  // empty segment
      if (n < kMaxSkSegments) s_slot[n] = static_cast<int>(2 * g + (a >= it0 ? 0 : 1));
      ++n;
    }
    // one segment: that CTA covered the whole tile and wrote C itself
    s_count = (n <= 1 || n > kMaxSkSegments) ? 0 : n;
  }
  __syncthreads();
  const int n = s_count;
  if (n == 0) return;
  // launched as the main kernel's dependent: its partials and C are complete
  // and visible only after this
  griddep_wait();

  int bi, tm, tn;
  unit_coords(p, p.dp_tiles + tile, bi, tm, tn);
  float *Cb = p.C + static_cast<int64_t>(bi) * p.strideC;
  const int64_t tile_elems = static_cast<int64_t>(bm) * bn;
  const bool read_c = p.beta != 0.0f;
  // 4 consecutive columns per thread (bn is a multiple of 64)
  {
    const int e = chunk * kChunk + 4 * threadIdx.x;
    const int row = tm * bm + e / bn, col = tn * bn + e % bn;
    if (row >= p.M) return;
    if (!SG_CHECK(e + 4 <= tile_elems && tile < p.num_tiles - p.dp_tiles, p.status)) return;
    float4 sum = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    // partials in groups of BATCH loads in flight, added in slot order
    for (int i0 = 0; i0 < n; i0 += BATCH) {
      float4 v[BATCH];
#pragma unroll
      for (int j = 0; j < BATCH; ++j)
        if (i0 + j < n && SG_CHECK(s_slot[i0 + j] >= 0 && s_slot[i0 + j] < 2 * grid_main, p.status))
          v[j] = __ldcg(reinterpret_cast<const float4 *>(p.workspace + s_slot[i0 + j] * tile_elems + e));
        else if (i0 + j < n)
          v[j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
      for (int j = 0; j < BATCH; ++j) {
        if (i0 + j < n) {
          sum.x += v[j].x;
          sum.y += v[j].y;
          sum.z += v[j].z;
          sum.w += v[j].w;
        }
      }
    }
    float *c = Cb + static_cast<int64_t>(row) * p.ldc + col;
    const float s4[4] = {sum.x, sum.y, sum.z, sum.w};
    if (p.c_vec4 && col + 3 < p.N) {
      float4 o;
      if (read_c) {
        const float4 cv = *reinterpret_cast<const float4 *>(c);
        o = make_float4(fmaf(p.alpha, s4[0], p.beta * cv.x), fmaf(p.alpha, s4[1], p.beta * cv.y),
                        fmaf(p.alpha, s4[2], p.beta * cv.z), fmaf(p.alpha, s4[3], p.beta * cv.w));
      } else {
        o = make_float4(p.alpha * s4[0], p.alpha * s4[1], p.alpha * s4[2], p.alpha * s4[3]);
      }
      *reinterpret_cast<float4 *>(c) = o;
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (col + q < p.N) c[q] = read_c ? fmaf(p.alpha, s4[q], p.beta * c[q]) : p.alpha * s4[q];
    }
  }
}

cudaError_t load_sk_fixup() {
  cudaFuncAttributes attr;
  cudaError_t e = cudaFuncGetAttributes(&attr, sk_fixup_kernel<1>);
  return e == cudaSuccess ? cudaFuncGetAttributes(&attr, sk_fixup_kernel<8>) : e;
}

cudaError_t launch_sk_fixup(const SimtParams &p, int bm, int bn, int grid_main, int sk_tiles,
                            int sm_count, cudaStream_t s) {
  const dim3 grid(sk_tiles * (bm * bn / kChunk));
  // 8 loads in flight where tiles have many segments (at most
  // ceil(grid_main / sk_tiles) + 1) and the grid is one wave at the four
  // blocks per SM its registers allow (GB300, graph replays: 256^3 13.2 ->
  // 12.5 us, 768^3 29.8 -> 28.5 us; 1024^3, two waves, 49.2 -> 51.0 us)
  if ((grid_main + sk_tiles - 1) / sk_tiles + 1 >= 4 && grid.x <= 4u * static_cast<unsigned>(sm_count))
    return launch_maybe_pdl(sk_fixup_kernel<8>, grid, dim3(kFixupThreads), 0, s, true, p, bm, bn, grid_main);
  return launch_maybe_pdl(sk_fixup_kernel<1>, grid, dim3(kFixupThreads), 0, s, true, p, bm, bn, grid_main);
}

}  // namespace sg
