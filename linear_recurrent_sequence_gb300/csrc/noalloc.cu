// Chunkwise retention for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a workspace: a plugin hosted by an
// inference runtime that hands it only its input and output tensors, or a
// latency-critical loop where a cudaMalloc (which may synchronise the whole
// device) is not allowed after start-up.  For them this entry point runs
// the ordinary chunkwise forward with its workspace taken from a fixed
// device array that lives in this library (kNoAllocScratchBytes on every
// GPU that loads the library, held until the process exits).  Nothing here
// calls cudaMalloc, cudaFree or any allocating routine.
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)RET_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a stand-in for the
// symbol; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (the first call on a device does this set-up).
cudaError_t scratch_on_current_device(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" ret_status retention_chunkwise_fwd_noalloc(const ret_desc *d, const void *q,
                                                      const void *k, const void *v,
                                                      const float *S_in, const float *z_in,
                                                      float *S_out, float *z_out, void *o,
                                                      ret_stream_t stream) {
  const size_t need = retention_workspace_size(d);
  if (need == 0) return RET_EINVAL;
  if (need > kNoAllocScratchBytes) return RET_EUNSUPPORTED;
  void *ws = nullptr;
  if (scratch_on_current_device(&ws) != cudaSuccess) return RET_ECUDA;
  // The array keeps the previous call's contents; the status word at its
  // start must begin at zero.  Everything else is overwritten by the call.
  if (cudaMemsetAsync(ws, 0, 256, (cudaStream_t)stream) != cudaSuccess) return RET_ECUDA;
  return retention_chunkwise_fwd(d, q, k, v, S_in, z_in, S_out, z_out, o, ws,
                                 kNoAllocScratchBytes, stream);
}
