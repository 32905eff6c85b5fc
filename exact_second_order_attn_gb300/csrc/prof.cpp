// Per-kernel CUDA-event timing of the library's launches (measurement aid).
#include "prof.h"

#include <cuda_runtime_api.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <map>
#include <mutex>
#include <string>
#include <vector>

namespace fbob {
namespace {

struct Rec {
  const char* name;
  cudaEvent_t e0, e1;
};

std::atomic<int> g_on{0};
std::mutex g_mu;
std::vector<Rec> g_recs;          // launches recorded since the last report
std::vector<cudaEvent_t> g_pool;  // events free for reuse
struct Agg {
  int n = 0;
  double total = 0, mn = 1e300, mx = 0;
};
std::map<std::string, Agg> g_agg;   // per-kernel totals not yet reported
thread_local Rec t_open{nullptr, nullptr, nullptr};

cudaEvent_t get_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

}  // namespace

void prof_begin(cudaStream_t s, const char* kernel) {
  if (!g_on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lock(g_mu);
  t_open.name = kernel;
  t_open.e0 = get_event();
  t_open.e1 = get_event();
  if (t_open.e0) cudaEventRecord(t_open.e0, s);
}

void prof_end(cudaStream_t s) {
  if (!g_on.load(std::memory_order_relaxed) || !t_open.name) return;
  std::lock_guard<std::mutex> lock(g_mu);
  if (t_open.e0 && t_open.e1 && cudaEventRecord(t_open.e1, s) == cudaSuccess) g_recs.push_back(t_open);
  t_open = Rec{nullptr, nullptr, nullptr};
}

}  // namespace fbob

extern "C" {

int fbob_profile_enable(int on) { return fbob::g_on.exchange(on ? 1 : 0); }

// Waits for every launch recorded so far and adds it to the per-kernel totals,
// writes {"kernel": [launches, total_ms, min_ms, max_ms], ...} into buf
// (NUL-terminated) and returns the text's length.  With buf == NULL (or len
// too small for the whole text) only the length is returned and the totals
// are kept; a call that writes the whole text also clears them.
int fbob_profile_report(char* buf, size_t len) {
  using namespace fbob;
  std::lock_guard<std::mutex> lock(g_mu);
  for (const Rec& r : g_recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.e1) == cudaSuccess && cudaEventElapsedTime(&ms, r.e0, r.e1) == cudaSuccess) {
      Agg& a = g_agg[r.name];
      a.n += 1;
      a.total += ms;
      if (ms < a.mn) a.mn = ms;
      if (ms > a.mx) a.mx = ms;
    }
    g_pool.push_back(r.e0);
    g_pool.push_back(r.e1);
  }
  g_recs.clear();
  std::string out = "{";
  char tmp[256];
  bool first = true;
  for (const auto& kv : g_agg) {
    snprintf(tmp, sizeof(tmp), "%s\"%s\": [%d, %.6f, %.6f, %.6f]", first ? "" : ", ", kv.first.c_str(), kv.second.n,
             kv.second.total, kv.second.mn, kv.second.mx);
    out += tmp;
    first = false;
  }
  out += "}";
  if (buf && len > out.size()) {
    memcpy(buf, out.data(), out.size());
    buf[out.size()] = '\0';
    g_agg.clear();
  }
  return (int)out.size();
}

}  // extern "C"
