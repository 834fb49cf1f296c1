// trace.h — per-phase timing of the library's calls (TPMLP_TRACE=1); see trace.cu.
#pragma once

#include <cuda_runtime.h>

namespace tpmlp {

bool trace_enabled();

// Records a CUDA event on `s` when constructed and another when destroyed,
// and logs the pair under `phase` (a string literal) when tracing is on.
class TraceScope {
 public:
  TraceScope(const char* phase, cudaStream_t s);
  ~TraceScope();
  TraceScope(const TraceScope&) = delete;
  TraceScope& operator=(const TraceScope&) = delete;

 private:
  const char* phase_;
  cudaStream_t stream_;
  cudaEvent_t begin_ = nullptr, end_ = nullptr;
  int device_ = 0;
  bool active_ = false;
};

}  // namespace tpmlp
