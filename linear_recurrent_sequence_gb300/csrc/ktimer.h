// Internal interface of the launch counter / kernel timer (ktimer.cu).
#pragma once

#include <cuda_runtime.h>

#include "../../include/retention.h"

namespace ret {

enum KernelId {
  kKRotate = 0,
  kKChunkSimt,
  kKParallelSimt,
  kKGroupNorm,
  kKRecurrent,
  kKGemmSimt,
  kKChunkTc,
  kKGemmTc,
  kKStatePass,
  kKGate,
  kKBwdRows,
  kKBwdValues,
  kKUnrotate,
  kKLayerNorm,
  kKResidual,
  kKGelu,
  kKGemmSkinny,
  kKSkinnyReduce,
  kKStateCombine,
  kKStateSimt,
  kKBwdPrep,
  kKBwdFinish,
  kKParallelTc,
  kKernelCount
};

int ktimer_begin(int id, cudaStream_t st);
void ktimer_end(int id, int idx, cudaStream_t st);

// Runs one launch expression between the timer's two events.
#define RET_TIMED_LAUNCH(id, st, expr)            \
  ([&]() -> cudaError_t {                         \
    const int ti_ = ::ret::ktimer_begin((id), (st)); \
    cudaError_t e_ = (expr);                      \
    ::ret::ktimer_end((id), ti_, (st));           \
    return e_;                                    \
  }())

}  // namespace ret
