// Optional per-stage device timing (det_stage_timing / det_stage_report).
// While enabled, every stage of det_gemm / det_gemm_partial is bracketed by a
// pair of CUDA events recorded on the call's own stream; the report sums the
// elapsed times per stage once the caller has synchronised.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "det_gemm.h"
#include "det_kernels.h"

namespace det {
namespace {

struct Record {
  int stage;
  cudaEvent_t start, stop;
};

std::atomic<int> g_enabled{0};
std::mutex g_mu;
std::vector<Record> g_records;

const char* const kStageNames[kNumStages] = {"prepass", "residue_planes", "residue_gemm",
                                             "reconstruct", "general_kulisch", "band",
                                             "wide_stats", "wide_planes", "wide_gemm",
                                             "wide_reconstruct"};

}  // namespace

StageScope::StageScope(int stage, cudaStream_t stream) : stage_(stage), stream_(stream) {
  if (!g_enabled.load(std::memory_order_relaxed)) return;
  if (cudaEventCreate(&start_) != cudaSuccess) return;
  if (cudaEventCreate(&stop_) != cudaSuccess) {
    cudaEventDestroy(start_);
    return;
  }
  active_ = cudaEventRecord(start_, stream_) == cudaSuccess;
  if (!active_) {
    cudaEventDestroy(start_);
    cudaEventDestroy(stop_);
  }
}

StageScope::~StageScope() {
  if (!active_) return;
  cudaEventRecord(stop_, stream_);
  std::lock_guard<std::mutex> lock(g_mu);
  g_records.push_back(Record{stage_, start_, stop_});
}

}  // namespace det

extern "C" {

int det_stage_timing(int enable) {
  return det::g_enabled.exchange(enable ? 1 : 0);
}

int det_stage_report(const char** names, double* total_ms, int* counts, int max) {
  std::lock_guard<std::mutex> lock(det::g_mu);
  double tot[det::kNumStages] = {0};
  int cnt[det::kNumStages] = {0};
  for (const det::Record& r : det::g_records) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.stop) == cudaSuccess &&
        cudaEventElapsedTime(&ms, r.start, r.stop) == cudaSuccess) {
      tot[r.stage] += ms;
      cnt[r.stage] += 1;
    }
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  det::g_records.clear();
  int n = 0;
  for (int s = 0; s < det::kNumStages && n < max; ++s) {
    if (cnt[s] == 0) continue;
    if (names) names[n] = det::kStageNames[s];
    if (total_ms) total_ms[n] = tot[s];
    if (counts) counts[n] = cnt[s];
    ++n;
  }
  return n;
}

int det_stage_timeline(const char** names, double* start_ms, double* stop_ms, int max) {
  std::lock_guard<std::mutex> lock(det::g_mu);
  int n = 0;
  const det::Record* first = det::g_records.empty() ? nullptr : &det::g_records.front();
  for (const det::Record& r : det::g_records) {
    float t0 = 0.f, t1 = 0.f;
    if (n < max && cudaEventSynchronize(r.stop) == cudaSuccess &&
        cudaEventElapsedTime(&t0, first->start, r.start) == cudaSuccess &&
        cudaEventElapsedTime(&t1, first->start, r.stop) == cudaSuccess) {
      if (names) names[n] = det::kStageNames[r.stage];
      if (start_ms) start_ms[n] = t0;
      if (stop_ms) stop_ms[n] = t1;
      ++n;
    }
  }
  for (const det::Record& r : det::g_records) {
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  det::g_records.clear();
  return n;
}

}  // extern "C"
