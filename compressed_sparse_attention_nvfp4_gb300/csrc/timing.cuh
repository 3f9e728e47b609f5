// Per-kernel device-time accounting: when enabled (csa2_timing_enable), each
// kernel launch of the library is bracketed by two CUDA events recorded on its
// launch stream; csa2_kernel_times() waits for the recorded pairs and sums
// their elapsed times per kernel name.
#pragma once

#include <cuda_runtime.h>

namespace csa2 {

bool timing_on();
void timing_record(const char* name, cudaEvent_t start, cudaEvent_t stop);
bool timing_events(cudaEvent_t* start, cudaEvent_t* stop);

// Brackets the launches made during its lifetime (one kernel) when timing is on.
class KernelTimer {
 public:
  KernelTimer(const char* name, cudaStream_t st) : name_(name), st_(st) {
    if (timing_on() && timing_events(&start_, &stop_)) cudaEventRecord(start_, st_);
  }
  ~KernelTimer() {
    if (start_) {
      cudaEventRecord(stop_, st_);
      timing_record(name_, start_, stop_);
    }
  }
  KernelTimer(const KernelTimer&) = delete;
  KernelTimer& operator=(const KernelTimer&) = delete;

 private:
  const char* name_;
  cudaStream_t st_;
  cudaEvent_t start_ = nullptr, stop_ = nullptr;
};

}  // namespace csa2
