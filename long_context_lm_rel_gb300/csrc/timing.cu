// Opt-in device timing of the main attention kernels (rxl_kernel_timing):
// when enabled, the launchers record a CUDA event pair on the launching stream
// around each launch of the forward kernel and of the backward's main kernel;
// reading sums the elapsed times of the recorded pairs. Off by default, and
// then it costs one relaxed atomic load per launch.
#include <atomic>
#include <mutex>

#include "internal.cuh"

namespace rxl {
namespace {

constexpr int kPairs = 1024;  // timed launches kept per kernel between reads

struct Timer {
  std::mutex mu;
  cudaEvent_t start[kPairs], stop[kPairs];
  int created = 0;  // event pairs created so far
  int used = 0;     // pairs recorded since the last read
  int dropped = 0;  // launches not timed because every pair was in use
};

std::atomic<bool> g_enabled{false};
Timer g_timers[kTimedKernels];

}  // namespace

bool timing_enabled() { return g_enabled.load(std::memory_order_relaxed); }

int timing_begin(int kernel, cudaStream_t st) {
  if (!timing_enabled() || kernel < 0 || kernel >= kTimedKernels) return -1;
  // a launch being captured into a graph is not timed (its event records
  // would become graph nodes)
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return -1;
  Timer &t = g_timers[kernel];
  std::lock_guard<std::mutex> lock(t.mu);
  if (t.used == kPairs) {
    ++t.dropped;
    return -1;
  }
  if (t.used == t.created) {
    if (cudaEventCreate(&t.start[t.created]) != cudaSuccess) return -1;
    if (cudaEventCreate(&t.stop[t.created]) != cudaSuccess) {
      cudaEventDestroy(t.start[t.created]);
      return -1;
    }
    ++t.created;
  }
  const int slot = t.used++;
  cudaEventRecord(t.start[slot], st);
  return slot;
}

void timing_end(int kernel, int slot, cudaStream_t st) {
  if (slot < 0) return;
  Timer &t = g_timers[kernel];
  std::lock_guard<std::mutex> lock(t.mu);
  cudaEventRecord(t.stop[slot], st);
}

}  // namespace rxl

extern "C" {

int rxl_kernel_timing(int enable) {
  rxl::g_enabled.store(enable != 0);
  return 0;
}

int rxl_kernel_timing_read(int kernel, double *total_ms, int *launches) {
  if (kernel < 0 || kernel >= rxl::kTimedKernels || !total_ms || !launches) return (int)cudaErrorInvalidValue;
  rxl::Timer &t = rxl::g_timers[kernel];
  std::lock_guard<std::mutex> lock(t.mu);
  double sum = 0.0;
  for (int i = 0; i < t.used; ++i) {
    cudaError_t e = cudaEventSynchronize(t.stop[i]);
    float ms = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, t.start[i], t.stop[i]);
    if (e != cudaSuccess) return (int)e;
    sum += ms;
  }
  *total_ms = sum;
  *launches = t.used;
  t.used = 0;
  t.dropped = 0;
  return 0;
}

}  // extern "C"
