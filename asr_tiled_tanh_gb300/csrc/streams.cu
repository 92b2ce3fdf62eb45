// streams.cu -- side streams for the independent launches of one call.
#include "streams.h"

namespace rnnt {
namespace {

constexpr int kMaxDevices = 64;
struct DeviceStreams {
  bool tried = false;
  bool ok = false;
  cudaStream_t side[kMaxDepth][kMaxSide] = {};
  cudaEvent_t fork[kMaxDepth] = {};
  cudaEvent_t join[kMaxDepth][kMaxSide] = {};
};
DeviceStreams g_dev[kMaxDevices];
std::recursive_mutex g_mu;
thread_local int t_depth = 0;  // forks this thread has open

// Streams and events of the current device, created on first use (lock held).
DeviceStreams* device_streams() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  DeviceStreams& d = g_dev[dev];
  if (!d.tried) {
    d.tried = true;
    bool ok = true;
    for (int l = 0; l < kMaxDepth && ok; ++l) {
      ok = cudaEventCreateWithFlags(&d.fork[l], cudaEventDisableTiming) == cudaSuccess;
      for (int i = 0; i < kMaxSide && ok; ++i) {
        ok = cudaStreamCreateWithFlags(&d.side[l][i], cudaStreamNonBlocking) == cudaSuccess &&
             cudaEventCreateWithFlags(&d.join[l][i], cudaEventDisableTiming) == cudaSuccess;
      }
    }
    d.ok = ok;
  }
  return d.ok ? &d : nullptr;
}

}  // namespace

Fork::Fork(cudaStream_t main, int n) : main_(main), lock_(g_mu, std::try_to_lock) {
  // another thread's forks are open: run everything on main
  if (!lock_.owns_lock()) return;
  depth_ = t_depth++;
  if (n <= 0 || depth_ >= kMaxDepth) return;
  if (n > kMaxSide) n = kMaxSide;
  DeviceStreams* d = device_streams();
  if (!d || cudaEventRecord(d->fork[depth_], main) != cudaSuccess) return;
  int ready = 0;
  while (ready < n && cudaStreamWaitEvent(d->side[depth_][ready], d->fork[depth_], 0) ==
                          cudaSuccess)
    ++ready;
  // the streams that wait are joined back; the rest of the work runs on main
  n_ = ready;
  for (int k = 0; k < n_; ++k) {
    sides_[k] = d->side[depth_][k];
    joins_[k] = d->join[depth_][k];
  }
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

Fork::~Fork() {
  join();
  if (depth_ >= 0) --t_depth;
}

}  // namespace rnnt
