// profile.h -- RAII event bracket around a kernel launch (internal).
#pragma once
#include <cuda_runtime.h>

namespace rnnt {

bool prof_enabled();

// Records a start event on construction and an end event on destruction
// while a profiling session is open; otherwise does nothing.
class ProfScope {
 public:
  ProfScope(const char* name, cudaStream_t s);
  ~ProfScope();
  // number of kernel launches the bracket holds (1 unless set)
  void set_kernels(int n);
  ProfScope(const ProfScope&) = delete;
  ProfScope& operator=(const ProfScope&) = delete;

 private:
  int slot_;
  cudaStream_t s_;
};

}  // namespace rnnt
