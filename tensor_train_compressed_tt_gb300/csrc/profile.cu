// Measurement hooks: CUDA-event brackets around the library's kernel phases
// and a launch counter.  Host-side state only; not thread-safe by design.
#include <atomic>
#include <vector>

#include "ttc_internal.h"

namespace ttc {
namespace {

struct Interval {
  int phase;
  cudaEvent_t start, stop;
};

bool g_on = false;
std::vector<Interval> g_records;
std::vector<cudaEvent_t> g_pool;
size_t g_pool_used = 0;
int g_open_phase = -1;
cudaEvent_t g_open_start = nullptr;
std::atomic<uint64_t> g_launches{0};

cudaEvent_t take_event() {
  if (g_pool_used == g_pool.size()) {
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    g_pool.push_back(e);
  }
  return g_pool[g_pool_used++];
}

const char* kNames[TT_NUM_PHASES] = {"merge", "forward_tokens", "backward_tokens",
                                     "merge_backward", "elementwise"};

}  // namespace

// Inside a stream capture the record becomes an event-record node of the
// graph (external), so that every replay stamps it; otherwise a plain record.
void record(cudaEvent_t e, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, st, cudaEventRecordExternal);
  else
    cudaEventRecord(e, st);
}

void prof_begin(int phase, cudaStream_t st) {
  if (!g_on) return;
  cudaEvent_t e = take_event();
  if (!e) return;
  record(e, st);
  g_open_phase = phase;
  g_open_start = e;
}

void prof_end(int phase, cudaStream_t st) {
  if (!g_on || g_open_phase != phase || !g_open_start) return;
  cudaEvent_t e = take_event();
  if (!e) return;
  record(e, st);
  g_records.push_back({phase, g_open_start, e});
  g_open_phase = -1;
  g_open_start = nullptr;
}

void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

}  // namespace ttc

using namespace ttc;

extern "C" {

void tt_profile_enable(int on) {
  g_on = on != 0;
  if (g_on) {
    g_records.clear();
    g_pool_used = 0;
    g_open_phase = -1;
    g_open_start = nullptr;
  }
}

tt_status tt_profile_phase(int phase, double* total_ms, int64_t* intervals) {
  if (phase < 0 || phase >= TT_NUM_PHASES || !total_ms || !intervals) return TT_ERR_INVALID_ARG;
  double tot = 0;
  int64_t n = 0;
  for (const Interval& r : g_records) {
    if (r.phase != phase) continue;
    if (cudaEventSynchronize(r.stop) != cudaSuccess) return TT_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess) return TT_ERR_CUDA;
    tot += ms;
    ++n;
  }
  *total_ms = tot;
  *intervals = n;
  return TT_OK;
}

const char* tt_profile_phase_name(int phase) {
  if (phase < 0 || phase >= TT_NUM_PHASES) return "";
  return kNames[phase];
}

uint64_t tt_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
