// Per-kernel CUDA-event timing behind lca_profile_enable / lca_profile_read.
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/lca.h"
#include "profile.h"

namespace lca {

namespace {

const char* kNames[K_COUNT] = {"mask_classify", "mask_scan", "mask_collen", "mask_fill",
                               "mask_lpt", "attn_fwd", "bwd_preprocess", "bwd",
                               "block_scores", "block_topk"};

struct Rec {
  int id, launches;
  cudaEvent_t a, b;
};

std::atomic<bool> g_on{false};
std::mutex g_mu;
std::vector<Rec> g_recs;
std::vector<cudaEvent_t> g_pool;

cudaEvent_t take_event() {
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

bool profiling_on() { return g_on.load(std::memory_order_relaxed); }

long profile_begin(int id, int launches, cudaStream_t st) {
  std::lock_guard<std::mutex> lk(g_mu);
  Rec r{id, launches, take_event(), take_event()};
  if (!r.a || !r.b) return 0;
  cudaEventRecord(r.a, st);
  g_recs.push_back(r);
  return static_cast<long>(g_recs.size());
}

void profile_end(long token, cudaStream_t st) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (token < 1 || token > static_cast<long>(g_recs.size())) return;
  cudaEventRecord(g_recs[token - 1].b, st);
}

}  // namespace lca

extern "C" {

void lca_profile_enable(int on) { lca::g_on.store(on != 0); }

int lca_profile_read(lca_kernel_time* out, int max_entries) {
  using namespace lca;
  std::lock_guard<std::mutex> lk(g_mu);
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  double ms[K_COUNT] = {0};
  int64_t n[K_COUNT] = {0};
  for (const Rec& r : g_recs) {
    float t = 0.f;
    if (cudaEventElapsedTime(&t, r.a, r.b) == cudaSuccess) ms[r.id] += t;
    n[r.id] += r.launches;
    g_pool.push_back(r.a);
    g_pool.push_back(r.b);
  }
  g_recs.clear();
  int k = 0;
  for (int id = 0; id < K_COUNT; ++id) {
    if (n[id] == 0) continue;
    if (out && k < max_entries) {
      std::memset(out[k].name, 0, sizeof(out[k].name));
      std::strncpy(out[k].name, kNames[id], sizeof(out[k].name) - 1);
      out[k].launches = n[id];
      out[k].total_ms = ms[id];
    }
    ++k;
  }
  return k < max_entries ? k : max_entries;
}

}  // extern "C"
