// noalloc.cu -- sgemm_noalloc(): the CUDA-core GEMM with its stream-K scratch
// in a fixed __device__ array instead of a cudaMalloc'd workspace, so that a
// call never allocates device memory.
//
// Why: sgemm() gets the scratch for split tiles (the partial sums that
// stream-K scheduling leaves for its fixup pass) from a cudaMalloc made the
// first time a product needs it.  Some callers cannot let a library call do
// that:
//   * applications that hand (nearly) all device memory to their own pool or
//     caching allocator at start-up -- a cudaMalloc behind its back can fail,
//     or shrink what the pool may use;
//   * latency-sensitive loops: cudaMalloc may synchronise the device, stalling
//     work queued on other streams, and it can fail part-way through a run
//     when memory is tight;
//   * services whose device-memory footprint is fixed and checked up front.
// Here the scratch is g_noalloc_scratch, SGEMM_NOALLOC_SCRATCH_BYTES of
// __device__ memory that stays reserved on every GPU where it has been loaded
// until the process exits.
//
// Set-up, once per device, by the first call made with that device current
// (any call whose arguments are valid, an empty one with M = 0 included):
// it looks up the array's device address with cudaGetSymbolAddress (host code
// cannot use the symbol itself: on the host it names a stand-in, not device
// memory) and queries every kernel this entry point launches.  Under CUDA's
// lazy module loading (the default since CUDA 12.2) those lookups are what
// make the runtime load this library's code and reserve the array on that
// device, so the one-time reservation happens there and not at library load.
// Make that first call before handing the remaining device memory to your own
// pool, and before any stream capture begins; every later call allocates
// nothing.
//
// Sharing: every call on a device uses the same array and leaves its contents
// behind.  Nothing in it has to start at zero -- the main kernel writes every
// partial tile that the fixup pass of the same call reads -- but two calls
// whose work overlaps on the GPU (different streams, no ordering between
// them) race on the array and may produce wrong results.  Order such calls
// yourself, or use sgemm().
#include <cstring>
#include <mutex>

#include "dispatch.h"
#include "internal.h"
#include "sgemm.h"

namespace {

using namespace sg;

// Two partial 128 x 128 tiles (64 KiB each) for each of up to 160 CTAs, or two
// 128 x 64 tiles for each of up to 320.
__device__ __align__(256) float g_noalloc_scratch[SGEMM_NOALLOC_SCRATCH_BYTES / sizeof(float)];

struct NoAllocDevice {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  float *scratch = nullptr;
};
NoAllocDevice g_noalloc[kMaxDevices];

// One-time set-up on the current device (see the file comment): the array's
// device address, and every kernel this entry point may launch loaded.
// Returns the address, or null if the set-up failed.
float *noalloc_setup(DeviceState &d) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  NoAllocDevice &n = g_noalloc[dev];
  std::call_once(n.once, [&n, &d]() {
    n.err = cudaGetSymbolAddress(reinterpret_cast<void **>(&n.scratch), g_noalloc_scratch);
    for (int producer = 0; producer < 2 && n.err == cudaSuccess; ++producer)
      for (int ta = 0; ta < 2; ++ta)
        for (int tb = 0; tb < 2; ++tb)
          for (int tile : {kTile128x128, kTile128x64})
            if (n.err == cudaSuccess && !kernel_info(d, producer, ta, tb, tile))
              n.err = cudaErrorInvalidDeviceFunction;
    if (n.err == cudaSuccess) n.err = load_sk_fixup();
    if (n.err == cudaSuccess) n.err = load_scale_c();
    if (n.err != cudaSuccess) {
      cudaGetLastError();
      n.scratch = nullptr;
    }
  });
  return n.scratch;
}

}  // namespace

extern "C" sgemm_status_t sgemm_noalloc(int transA, int transB, int64_t M, int64_t N, int64_t K,
                                        float alpha, const float *A, int64_t lda, const float *B,
                                        int64_t ldb, float beta, float *C, int64_t ldc,
                                        void *stream) {
  Args a{norm_op(transA), norm_op(transB), M, N, K, alpha, beta, A, lda, B, ldb, C, ldc};
  sgemm_status_t st = validate(a, true);
  if (st != SGEMM_SUCCESS) return st;
  t_last_launches = 0;

  // the set-up comes first, so that an empty call (M = 0) can be used to do it
  sgemm_status_t why = SGEMM_SUCCESS;
  DeviceState *d = device_state(&why);
  if (!d) return why;
  float *scratch = noalloc_setup(*d);
  if (!scratch) return SGEMM_ERR_LAUNCH;
  if (M == 0 || N == 0) return SGEMM_SUCCESS;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  if (K == 0 || alpha == 0.0f) {
    if (launch_scale_c(C, ldc, static_cast<int>(M), static_cast<int>(N), beta, s) != cudaSuccess)
      return SGEMM_ERR_LAUNCH;
    t_last_launches = 1;
    return SGEMM_SUCCESS;
  }

  // Same kernels as sgemm()'s CUDA-core path, but only the tiles whose
  // partial sums fit the array at one CTA slot per SM (no 128 x 256 tile).
  const int producer = tma_eligible(a) ? kTma : kCpAsync;
  const int tile = (a.N <= 64) ? kTile128x64 : kTile128x128;
  const SimtKernelInfo *ki = kernel_info(*d, producer, a.ta, a.tb, tile);
  if (!ki || ki->ctas_per_sm < 1) return SGEMM_ERR_LAUNCH;

  SimtParams p;
  p.A = A;
  p.B = B;
  p.C = C;
  p.lda = lda;
  p.ldb = ldb;
  p.ldc = ldc;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.alpha = alpha;
  p.beta = beta;
  p.tiles_m = static_cast<int>(cdiv(M, ki->bm));
  p.tiles_n = static_cast<int>(cdiv(N, ki->bn));
  p.k_tiles = static_cast<int>(cdiv(K, 32));
  const int64_t num_tiles = static_cast<int64_t>(p.tiles_m) * p.tiles_n;
  if (num_tiles > kMaxDim) return SGEMM_ERR_UNSUPPORTED;
  p.num_tiles = static_cast<int>(num_tiles);
  p.tiles_per_batch = p.num_tiles;  // one product
  p.strideA = p.strideB = p.strideC = 0;
  p.a_map3d = p.b_map3d = 0;
  p.group_m = 8;
  p.c_vec4 = (ldc % 4 == 0) && (reinterpret_cast<uintptr_t>(C) % 16 == 0);
  p.wait_budget_ns = g_wait_budget_ns.load(std::memory_order_relaxed);
  p.status = d->status;

  const int64_t slots = static_cast<int64_t>(d->sm_count) * ki->ctas_per_sm;
  SkPlan plan = plan_stream_k(num_tiles, p.k_tiles, slots, true);
  const size_t need =
      plan.sk_tiles > 0 ? static_cast<size_t>(2) * plan.grid * ki->bm * ki->bn * sizeof(float) : 0;
  // split tiles whose partials would not fit the array: whole tiles only
  // (plain waves, no scratch), as sgemm() does without a workspace
  if (need > SGEMM_NOALLOC_SCRATCH_BYTES) plan = plan_stream_k(num_tiles, p.k_tiles, slots, false);
  p.dp_tiles = plan.dp_tiles;
  p.sk_iters = plan.sk_iters;
  p.workspace = plan.sk_tiles > 0 ? scratch : nullptr;

  CUtensorMap tmA, tmB;
  std::memset(&tmA, 0, sizeof(tmA));
  std::memset(&tmB, 0, sizeof(tmB));
  if (producer == kTma) {
    const bool okA = a.ta == 0 ? encode_tmap(&tmA, A, M, K, lda, 32, ki->bm, true)
                               : encode_tmap(&tmA, A, K, M, lda, ki->bm, 32, false);
    const bool okB = a.tb == 0 ? encode_tmap(&tmB, B, K, N, ldb, ki->bn, 32, false)
                               : encode_tmap(&tmB, B, N, K, ldb, 32, ki->bn, true);
    if (!okA || !okB) return SGEMM_ERR_LAUNCH;
  }
  CUtensorMap tmC;   // C written straight from registers (p.c_tma == 0)
  std::memset(&tmC, 0, sizeof(tmC));
  if (simt_entry(producer, a.ta, a.tb, tile).launch(p, &tmA, &tmB, &tmC, plan.grid, s, false, 1) != cudaSuccess)
    return SGEMM_ERR_LAUNCH;
  t_last_launches = 1;
  if (plan.sk_tiles > 0) {
    if (launch_sk_fixup(p, ki->bm, ki->bn, plan.grid, plan.sk_tiles, d->sm_count, s) != cudaSuccess)
      return SGEMM_ERR_LAUNCH;
    t_last_launches = 2;
  }
  return SGEMM_SUCCESS;
}
