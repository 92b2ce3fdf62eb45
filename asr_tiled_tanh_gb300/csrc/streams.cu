// streams.cu -- side streams for the independent launches of one call.
#include "streams.h"

namespace rnnt {
namespace {

constexpr int kMaxDevices = 64;
struct DeviceStreams {
  bool tried = false;
  bool ok = false;
  cudaStream_t side[kMaxSide] = {};
  cudaEvent_t fork = nullptr;
  cudaEvent_t join[kMaxSide] = {};
};
DeviceStreams g_dev[kMaxDevices];
std::mutex g_mu;

// Streams and events of the current device, created on first use (lock held).
DeviceStreams* device_streams() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  DeviceStreams& d = g_dev[dev];
  if (!d.tried) {
    d.tried = true;
    bool ok = cudaEventCreateWithFlags(&d.fork, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; i < kMaxSide && ok; ++i) {
      ok = cudaStreamCreateWithFlags(&d.side[i], cudaStreamNonBlocking) == cudaSuccess &&
           cudaEventCreateWithFlags(&d.join[i], cudaEventDisableTiming) == cudaSuccess;
    }
    d.ok = ok;
  }
  return d.ok ? &d : nullptr;
}

}  // namespace

Fork::Fork(cudaStream_t main, int n) : main_(main), lock_(g_mu, std::try_to_lock) {
  // a fork already open (another thread's, or an enclosing one) means this
  // one runs everything on main
  if (n <= 0 || !lock_.owns_lock()) return;
  if (n > kMaxSide) n = kMaxSide;
  DeviceStreams* d = device_streams();
  if (!d || cudaEventRecord(d->fork, main) != cudaSuccess) return;
  for (int i = 0; i < n; ++i) {
    if (cudaStreamWaitEvent(d->side[i], d->fork, 0) != cudaSuccess) {
      // the streams that already wait are joined back; the rest run on main
      n_ = i;
      for (int k = 0; k < n_; ++k) { sides_[k] = d->side[k]; joins_[k] = d->join[k]; }
      return;
    }
  }
  n_ = n;
  for (int k = 0; k < n_; ++k) { sides_[k] = d->side[k]; joins_[k] = d->join[k]; }
}

cudaError_t Fork::join() {
  if (joined_) return cudaSuccess;
  joined_ = true;
  cudaError_t err = cudaSuccess;
  for (int i = 0; i < n_; ++i) {
    cudaError_t e = cudaEventRecord(joins_[i], sides_[i]);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(main_, joins_[i], 0);
    if (e != cudaSuccess && err == cudaSuccess) err = e;
  }
  return err;
}

Fork::~Fork() { join(); }

}  // namespace rnnt
