// dispatch.h -- host-side helpers of the C ABI shared between its translation
// units: argument checks, per-device state, kernel attributes, TMA descriptor
// encoding and the stream-K planner (defined in api.cu).  Not part of the
// public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>
#include <utility>
#include <vector>

#include "internal.h"
#include "sgemm.h"

namespace sg {

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultWaitBudgetNs = 2000000000ull;  // 2 s
extern std::atomic<uint64_t> g_wait_budget_ns;
extern thread_local int t_last_launches;

// Orders the users of one library-owned device buffer (stream-K workspace,
// transposed-operand scratch) across streams and captured CUDA graphs: every
// use waits for the previous use's event and records its own.  Eager uses on
// the stream that used the buffer last need no wait; uses inside a stream
// capture wait and record through external event nodes, which take effect
// each time the graph is launched (a graph launch records the event like
// cudaEventRecord would); after the first captured use, eager uses always
// wait, since graph launches do not pass through this library.
struct BufferOrder {
  cudaEvent_t ev = nullptr;
  cudaStream_t last = nullptr;
  bool used = false;
  // a use has been captured into a graph at some point: its launches are
  // invisible to the host-side bookkeeping, so every later use waits
  bool in_graph = false;
  // capture sequence of the last use (0: an eager use)
  unsigned long long capture = 0;
};
cudaError_t order_before_use(BufferOrder &o, cudaStream_t s, bool capturing);
cudaError_t order_after_use(BufferOrder &o, cudaStream_t s, bool capturing);
// Copies of one or two (in1 != nullptr) rows x cols matrices into 16-byte
// aligned rows (ld_out % 4 == 0, out 16-byte aligned), zero-padded, in one
// launch (repack.cu).
cudaError_t launch_repack(const float *in0, int64_t ld_in0, int rows0, int cols0, float *out0,
                          int64_t ld_out0, const float *in1, int64_t ld_in1, int rows1, int cols1,
                          float *out1, int64_t ld_out1, cudaStream_t s);
// True while `s` is being captured into a CUDA graph.
bool stream_capturing(cudaStream_t s);

struct DeviceState {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  int sm_count = 0, cc_major = 0, cc_minor = 0;
  int *status = nullptr;
  // Device memory the library may own on this device (sgemm_set_scratch_limit;
  // initial value from the SGEMM_SCRATCH_LIMIT environment variable, else no
  // limit) and what it holds now: the stream-K workspace, the operand scratch
  // and scratch buffers retired under captured graphs.  An allocation first
  // reserves its bytes against the limit (reserve_scratch) and gives them back
  // if cudaMalloc fails.
  std::atomic<uint64_t> limit{UINT64_MAX};
  std::atomic<uint64_t> held{0};
  // Stream-K workspace: allocated on first use, kept until exit.  Calls that
  // use it on different streams or in graphs are ordered by ws_order.
  std::mutex ws_mu;
  float *ws = nullptr;
  size_t ws_bytes = 0;
  int *sk_count = nullptr;   // kSkCounters arrival counters after the partial tiles
  bool ws_failed = false;
  BufferOrder ws_order;
  // Scratch for operands copied ahead of a product (see run_pretransposed):
  // grown on demand up to kPretransposeMaxBytes, kept until exit; calls on
  // different streams or in graphs that use it are ordered by tr_order.  A
  // buffer that a captured graph may hold is never freed: growing past it
  // retires it to tr_retired.
  std::mutex tr_mu;
  float *tr = nullptr;
  size_t tr_bytes = 0;
  std::vector<std::pair<float *, size_t>> tr_retired;
  bool tr_failed = false;
  BufferOrder tr_order;
  // [producer][transA][transB][tile][cluster split-K form]
  std::once_flag kinfo_once[2][2][2][kNumSimtTiles][2];
  cudaError_t kinfo_err[2][2][2][kNumSimtTiles][2] = {};
  SimtKernelInfo kinfo[2][2][2][kNumSimtTiles][2] = {};
  std::once_flag tcinfo_once[2][2];
  cudaError_t tcinfo_err[2][2] = {};
  TcKernelInfo tcinfo[2][2] = {};
  std::once_flag tcpre_once, tcpre_wide_once, tcpair_once[2][2][2];
  cudaError_t tcpre_err = cudaSuccess, tcpre_wide_err = cudaSuccess, tcpair_err[2][2][2] = {};
  // 128 x 128 / 128 x 256 tiles on one CTA, 256 x 128 / 256 x 256 tiles on
  // CTA pairs [wide][fold_a][fold_b]
  TcKernelInfo tcpre = {}, tcpre_wide = {}, tcpair[2][2][2] = {};
};
// Indices are 32-bit inside the kernels; tile origins may run up to one tile
// past the end of a dimension.
constexpr int64_t kMaxDim = 0x7fffffff - 1024;
// stream-K tiles a launch may finish in-kernel (at most two waves' worth of
// tiles are split, far below this)
constexpr int kSkCounters = 4096;
// Leading dimensions and batch strides are bounded by kMaxLd; validate() also
// rejects a matrix whose byte range would end past 2^64 (it cannot exist), so
// every element offset the kernels form stays below 2^62 and fits in int64.
constexpr int64_t kMaxLd = int64_t(1) << 40;

struct Args {
  int ta, tb;
  int64_t M, N, K;
  float alpha, beta;
  const float *A;
  int64_t lda;
  const float *B;
  int64_t ldb;
  float *C;
  int64_t ldc;
};

// Host-side validation shared by the entry points (status codes, no launch).
// Dimension and leading-dimension checks only (no pointers).
sgemm_status_t validate_shape(const Args &a);
sgemm_status_t validate(const Args &a, bool c_writable);
bool tma_eligible(const Args &a);
int64_t cdiv(int64_t a, int64_t b);
int norm_op(int t);

// The current device's state (initialised once per device) or null with the
// reason in *why.  Also clears a pending error left by earlier, unrelated
// runtime calls, so that the launches that follow report only their own.
DeviceState *device_state(sgemm_status_t *why);
const SimtKernelInfo *kernel_info(DeviceState &d, int producer, int ta, int tb, int tile, int csk = 0);
const TcKernelInfo *tc_kernel_info(DeviceState &d, int ta, int tb);
const TcKernelInfo *tc_kernel_info_presplit(DeviceState &d, int bn);
const TcKernelInfo *tc_kernel_info_pair(DeviceState &d, int bn, bool fold_a = false, bool fold_b = false);

// 2-D FP32 tensor map over a row-major rows x cols matrix (row stride ld
// elements), box box_cols x box_rows, zero fill outside; false on failure.
bool encode_tmap(CUtensorMap *m, const float *base, int64_t rows, int64_t cols, int64_t ld,
                 int box_cols, int box_rows, bool swizzle128);

int pick_simt_tile(const Args &a, int producer, int sm_count, int64_t batch = 1);

// Smallest stream-K segment worth a partial tile (k-tiles of 32).
#ifndef SG_MIN_SK_SEGMENT
#define SG_MIN_SK_SEGMENT 1
#endif
constexpr int64_t kMinSkSegment = SG_MIN_SK_SEGMENT;

struct SkPlan {
  int dp_tiles;     // whole tiles, round-robin
  int sk_tiles;     // tiles whose k-iterations are spread over the grid
  int64_t sk_iters;
  int grid;
};

SkPlan plan_stream_k(int64_t tiles, int64_t k_tiles, int64_t slots, bool have_ws);
// CTAs per cluster of cluster split-K for this product (0: not used);
// have_ws: a stream-K workspace is available as the alternative.
int pick_csk(const SimtKernelInfo &ki, int64_t tiles, int64_t k_tiles, int64_t slots, bool have_ws);

// Reserves `bytes` of the device's scratch limit (false, nothing reserved, if
// they do not fit); release_scratch gives bytes back.
bool reserve_scratch(DeviceState &d, uint64_t bytes);
void release_scratch(DeviceState &d, uint64_t bytes);

}  // namespace sg
