// streams.h -- side streams for the independent launches of one call (internal).
#pragma once
#include <cuda_runtime.h>

#include <mutex>

namespace rnnt {

constexpr int kMaxSide = 3;   // side streams of one fork
constexpr int kMaxDepth = 2;  // forks open at once in one thread (nested)

// Launches of one library call that do not depend on one another can run at
// the same time on up to kMaxSide side streams.  The constructor makes each
// side stream wait for everything enqueued on `main` so far; join() (or the
// destructor) makes `main` wait for everything enqueued on the side streams,
// so the call stays ordered on `main` as a whole and works under stream
// capture.  The side streams and events are created once per device, on the
// first fork made with that device current, one set per nesting level: a
// fork opened while another is open in the same thread (its `main` may be a
// side stream of the outer one) uses the next level's streams.  Calls from
// other host threads wait for nothing: while one thread has forks open, a
// fork made in another thread (or past kMaxDepth levels, or when n is 0 or
// the streams cannot be created) has side() return `main`, and its launches
// simply run one after another.
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
  int depth_ = -1;
  bool joined_ = false;
  std::unique_lock<std::recursive_mutex> lock_;
};

}  // namespace rnnt
