// Per-kernel device-time accounting (see timing.cuh and csa2_timing_enable).
#include <atomic>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "timing.cuh"

namespace csa2 {
namespace {

struct Pending {
  const char* name;
  cudaEvent_t start, stop;
};

struct Totals {
  int64_t launches = 0;
  double ms = 0.0;
};

std::atomic<bool> g_on{false};
std::mutex g_mu;
std::vector<Pending> g_pending;                  // recorded, not yet read
std::vector<std::pair<cudaEvent_t, cudaEvent_t>> g_free;  // event pairs to reuse
std::map<std::string, Totals> g_totals;          // read so far, by kernel name

// Folds every recorded pair into the totals (waits for each stop event).
bool drain_locked() {
  bool ok = true;
  for (const Pending& p : g_pending) {
    float ms = 0.0f;
    if (cudaEventSynchronize(p.stop) != cudaSuccess || cudaEventElapsedTime(&ms, p.start, p.stop) != cudaSuccess) {
      ok = false;
    } else {
      Totals& t = g_totals[p.name];
      t.launches += 1;
      t.ms += ms;
    }
    g_free.emplace_back(p.start, p.stop);
  }
  g_pending.clear();
  return ok;
}

}  // namespace

bool timing_on() { return g_on.load(std::memory_order_relaxed); }

bool timing_events(cudaEvent_t* start, cudaEvent_t* stop) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_free.empty()) {
    *start = g_free.back().first;
    *stop = g_free.back().second;
    g_free.pop_back();
    return true;
  }
  if (cudaEventCreate(start) != cudaSuccess) return false;
  if (cudaEventCreate(stop) != cudaSuccess) {
    cudaEventDestroy(*start);
    return false;
  }
  return true;
}

void timing_record(const char* name, cudaEvent_t start, cudaEvent_t stop) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_pending.push_back({name, start, stop});
}

}  // namespace csa2

extern "C" csa2_status csa2_timing_enable(int32_t on) {
  using namespace csa2;
  std::lock_guard<std::mutex> lk(g_mu);
  const bool ok = drain_locked();
  g_totals.clear();
  g_on.store(on != 0, std::memory_order_relaxed);
  return ok ? CSA2_OK : CSA2_ERR_CUDA;
}

extern "C" int32_t csa2_kernel_times(csa2_kernel_time* out, int32_t max) {
  using namespace csa2;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!drain_locked()) return -1;
  int32_t n = 0;
  for (const auto& kv : g_totals) {
    if (out && n < max) {
      out[n].name = kv.first.c_str();  // valid until the next csa2_timing_enable
      out[n].launches = kv.second.launches;
      out[n].total_ms = kv.second.ms;
    }
    ++n;
  }
  return n;
}
