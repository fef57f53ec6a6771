// Launch counter and opt-in per-kernel event timer.  When enabled, every
// kernel the library launches is bracketed by two CUDA events recorded on
// its own stream, so a caller can read each kernel's device time after
// synchronising.  Disabled (the default) it only counts launches.  Not for
// use while a stream is being captured into a CUDA graph.
#include <mutex>
#include <vector>

#include "ktimer.h"

namespace ret {

namespace {
constexpr int kMaxPairs = 16384;
const char *kNames[kKernelCount] = {
    "rotate_scale", "chunk_simt", "parallel_simt", "groupnorm", "recurrent_step",
    "gemm_simt", "chunk_tc", "gemm_tc", "state_pass", "swish_gate",
    "bwd_rows", "bwd_values", "unrotate",
    "layernorm", "residual_add", "gelu", "gemm_skinny", "skinny_reduce",
    "state_combine", "state_simt", "bwd_prep", "bwd_finish", "parallel_tc"};

struct Slot {
  std::vector<cudaEvent_t> start, stop;
  int used = 0;
  long long launches = 0;
};

std::mutex g_mu;
Slot g_slots[kKernelCount];
bool g_enabled = false;
long long g_total_launches = 0;
}  // namespace

int ktimer_begin(int id, cudaStream_t st) {
  std::lock_guard<std::mutex> lk(g_mu);
  ++g_total_launches;
  Slot &s = g_slots[id];
  ++s.launches;
  if (!g_enabled || s.used >= kMaxPairs) return -1;
  if ((int)s.start.size() <= s.used) {
    cudaEvent_t a, b;
    if (cudaEventCreate(&a) != cudaSuccess) return -1;
    if (cudaEventCreate(&b) != cudaSuccess) {
      cudaEventDestroy(a);
      return -1;
    }
    s.start.push_back(a);
    s.stop.push_back(b);
  }
  const int idx = s.used++;
  cudaEventRecord(s.start[idx], st);
  return idx;
}

void ktimer_end(int id, int idx, cudaStream_t st) {
  if (idx < 0) return;
  std::lock_guard<std::mutex> lk(g_mu);
  cudaEventRecord(g_slots[id].stop[idx], st);
}

}  // namespace ret

using namespace ret;

extern "C" {

void retention_kernel_timer_enable(int on) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_enabled = on != 0;
}

void retention_kernel_timer_reset(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (auto &s : g_slots) {
    s.used = 0;
    s.launches = 0;
  }
  g_total_launches = 0;
}

int retention_kernel_count(void) { return kKernelCount; }

const char *retention_kernel_name(int id) {
  return (id >= 0 && id < kKernelCount) ? kNames[id] : nullptr;
}

long long retention_launch_count(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  return g_total_launches;
}

int retention_kernel_timer_read(int id, double *total_ms, long long *launches, int *timed) {
  if (id < 0 || id >= kKernelCount) return (int)RET_EINVAL;
  std::lock_guard<std::mutex> lk(g_mu);
  Slot &s = g_slots[id];
  double tot = 0.0;
  for (int i = 0; i < s.used; ++i) {
    float ms = 0.f;
    cudaError_t e = cudaEventElapsedTime(&ms, s.start[i], s.stop[i]);
    if (e != cudaSuccess) return (int)RET_ECUDA;
    tot += ms;
  }
  if (total_ms) *total_ms = tot;
  if (launches) *launches = s.launches;
  if (timed) *timed = s.used;
  return (int)RET_OK;
}

}  // extern "C"
