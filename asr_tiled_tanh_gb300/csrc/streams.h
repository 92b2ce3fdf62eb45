// streams.h -- side streams for the independent launches of one call (internal).
#pragma once
#include <cuda_runtime.h>

#include <mutex>

namespace rnnt {

constexpr int kMaxSide = 3;

// Launches of one library call that do not depend on one another can run at
// the same time on up to kMaxSide side streams.  The constructor makes each
// side stream wait for everything enqueued on `main` so far; join() (or the
// destructor) makes `main` wait for everything enqueued on the side streams,
// so the call stays ordered on `main` as a whole and works under stream
// capture.  The side streams and events are created once per device, on the
// first fork made with that device current.  One fork is open at a time in
// the process (a lock held from fork to join, so that calls from several
// host threads never interleave their event records); a fork made while
// another is open, or when n is 0 or the streams cannot be created, has
// side() return `main`, and its launches simply run one after another.
class Fork {
 public:
  Fork(cudaStream_t main, int n);
  ~Fork();
  Fork(const Fork&) = delete;
  Fork& operator=(const Fork&) = delete;
  cudaStream_t side(int i) const { return n_ > 0 ? sides_[i % n_] : main_; }
  cudaError_t join();

 private:
  cudaStream_t main_;
  cudaStream_t sides_[kMaxSide] = {};
  cudaEvent_t joins_[kMaxSide] = {};
  int n_ = 0;
  bool joined_ = false;
  std::unique_lock<std::mutex> lock_;
};

}  // namespace rnnt
