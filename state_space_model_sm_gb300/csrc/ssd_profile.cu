// Optional per-kernel timing and launch counting for libssd.
//
// When enabled, every kernel launch is bracketed by two CUDA events recorded
// on the launch stream; ssd_profile_read() waits for them and reports, per
// kernel name, the number of launches and the summed device time.  The launch
// counter runs always (one relaxed atomic increment per launch).
#include <atomic>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "ssd_internal.h"

namespace ssd {
namespace {

struct Pending {
  int slot;
  cudaEvent_t start, stop;
};

struct Slot {
  std::string name;
  double ms = 0.0;
  int64_t launches = 0;
};

std::mutex g_mu;
std::atomic<bool> g_enabled{false};
std::atomic<int64_t> g_launches{0};
std::vector<Slot> g_slots;
std::vector<Pending> g_pending;
std::vector<cudaEvent_t> g_free;

cudaEvent_t take_event() {
  if (!g_free.empty()) {
    cudaEvent_t e = g_free.back();
    g_free.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

int slot_of(const char* name) {
  for (size_t i = 0; i < g_slots.size(); ++i)
    if (g_slots[i].name == name) return (int)i;
  g_slots.push_back(Slot{name});
  return (int)g_slots.size() - 1;
}

}  // namespace

LaunchScope::LaunchScope(const char* name, cudaStream_t s) : name_(name), s_(s) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (!g_enabled.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_mu);
  start_ = take_event();
  if (start_) cudaEventRecord(start_, s_);
}

LaunchScope::~LaunchScope() {
  if (!start_) return;
  std::lock_guard<std::mutex> lk(g_mu);
  cudaEvent_t stop = take_event();
  if (!stop) {
    g_free.push_back(start_);
    return;
  }
  cudaEventRecord(stop, s_);
  g_pending.push_back(Pending{slot_of(name_), start_, stop});
}

}  // namespace ssd

using namespace ssd;

extern "C" {

int ssd_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (auto& p : g_pending) {
    cudaEventSynchronize(p.stop);
    g_free.push_back(p.start);
    g_free.push_back(p.stop);
  }
  g_pending.clear();
  g_slots.clear();
  g_enabled.store(on != 0);
  return SSD_OK;
}

int ssd_profile_read(int max_kernels, char* names, double* ms, int64_t* launches) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (auto& p : g_pending) {
    if (cudaEventSynchronize(p.stop) != cudaSuccess) return -SSD_ERR_CUDA;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, p.start, p.stop) != cudaSuccess) return -SSD_ERR_CUDA;
    g_slots[p.slot].ms += t;
    g_slots[p.slot].launches += 1;
    g_free.push_back(p.start);
    g_free.push_back(p.stop);
  }
  g_pending.clear();
  const int n = (int)g_slots.size() < max_kernels ? (int)g_slots.size() : max_kernels;
  for (int i = 0; i < n; ++i) {
    if (names) {
      std::strncpy(names + (size_t)i * 64, g_slots[i].name.c_str(), 63);
      names[(size_t)i * 64 + 63] = 0;
    }
    if (ms) ms[i] = g_slots[i].ms;
    if (launches) launches[i] = g_slots[i].launches;
  }
  return n;
}

int64_t ssd_launch_count(void) { return g_launches.load(); }

}  // extern "C"
