// profile.cu -- per-kernel CUDA-event timing sessions (include/rnnt_profile.h).
#include <algorithm>
#include <atomic>
#include <cstring>
#include <vector>

#include "../../include/rnnt_profile.h"
#include "profile.h"

namespace rnnt {
namespace {
struct Session {
  std::atomic<bool> open{false};
  int capacity = 0;
  std::atomic<int> used{0};  // brackets handed out (may pass capacity)
  std::vector<cudaEvent_t> ev;       // 2 per launch
  std::vector<const char*> name;     // per bracket
  std::vector<int> kernels;          // kernel launches inside each bracket
};
Session g_sess;
struct Entry {
  const char* name;
  double ms;
  int launches;
};
std::vector<Entry> g_last;
}  // namespace

bool prof_enabled() { return g_sess.open.load(); }

// Calls from several threads take distinct slots.
ProfScope::ProfScope(const char* name, cudaStream_t s) : slot_(-1), s_(s) {
  if (!g_sess.open.load()) return;
  const int slot = g_sess.used.fetch_add(1);
  if (slot >= g_sess.capacity) return;
  slot_ = slot;
  g_sess.name[slot_] = name;
  g_sess.kernels[slot_] = 1;
  cudaEventRecord(g_sess.ev[2 * slot_], s);
}

void ProfScope::set_kernels(int n) {
  if (slot_ >= 0) g_sess.kernels[slot_] = n;
}

ProfScope::~ProfScope() {
  if (slot_ >= 0) cudaEventRecord(g_sess.ev[2 * slot_ + 1], s_);
}

}  // namespace rnnt

using namespace rnnt;

extern "C" {

rnnt_status rnnt_profile_start(int capacity) {
  if (capacity < 1 || g_sess.open.load()) return RNNT_ERR_INVALID_ARG;
  g_sess.ev.assign(2 * (size_t)capacity, nullptr);
  g_sess.name.assign(capacity, nullptr);
  g_sess.kernels.assign(capacity, 1);
  for (auto& e : g_sess.ev) {
    if (cudaEventCreate(&e) != cudaSuccess) {
      for (auto& f : g_sess.ev)
        if (f) cudaEventDestroy(f);
      g_sess.ev.clear();
      return RNNT_ERR_CUDA;
    }
  }
  g_sess.capacity = capacity;
  g_sess.used.store(0);
  g_sess.open.store(true);
  return RNNT_OK;
}

int rnnt_profile_stop(void) {
  if (!g_sess.open.load()) return -1;
  g_sess.open.store(false);
  g_last.clear();
  int rc = 0;
  const int used = std::min(g_sess.used.load(), g_sess.capacity);
  for (int i = 0; i < used && rc == 0; ++i) {
    float ms = 0.f;
    if (cudaEventSynchronize(g_sess.ev[2 * i + 1]) != cudaSuccess ||
        cudaEventElapsedTime(&ms, g_sess.ev[2 * i], g_sess.ev[2 * i + 1]) != cudaSuccess) {
      rc = -1;
      break;
    }
    bool found = false;
    for (auto& e : g_last) {
      if (std::strcmp(e.name, g_sess.name[i]) == 0) {
        e.ms += ms;
        e.launches += g_sess.kernels[i];
        found = true;
        break;
      }
    }
    if (!found) g_last.push_back(Entry{g_sess.name[i], (double)ms, g_sess.kernels[i]});
  }
  for (auto& e : g_sess.ev) cudaEventDestroy(e);
  g_sess.ev.clear();
  g_sess.name.clear();
  g_sess.kernels.clear();
  if (rc != 0) {
    g_last.clear();
    return -1;
  }
  return (int)g_last.size();
}

rnnt_status rnnt_profile_entry(int i, const char** name, double* total_ms, int* launches) {
  if (i < 0 || i >= (int)g_last.size()) return RNNT_ERR_INVALID_ARG;
  if (name) *name = g_last[i].name;
  if (total_ms) *total_ms = g_last[i].ms;
  if (launches) *launches = g_last[i].launches;
  return RNNT_OK;
}

}  // extern "C"
