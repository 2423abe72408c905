// Launch counting and per-kernel CUDA-event tracing.
//
// Every kernel launch in the library goes through trace_begin / trace_end.
// The launch counter is always on.  When tracing is started, each launch is
// bracketed by a pair of CUDA events recorded on the launch stream (also
// inside a stream capture, where the records become graph nodes that fire on
// every replay); dspark_trace_collect() waits for the recorded pairs and adds
// their elapsed times to per-kernel totals.  Events are host-side objects
// created once; no device memory is allocated.
#include <atomic>
#include <mutex>

#include "dspark.h"
#include "common.cuh"

namespace dspark {

namespace {

constexpr int kPairs = 8192;

const char* const kNames[kKindCount] = {
    "markov_bias",       "draft_partial",  "draft_finish", "confidence",  "schedule",
    "verify_rows",    "verify_decide", "final_partial", "final_pick",
    "draft_fused_tc",    "draft_persistent_tc", "final_tc", "wait_check", "rnn_state",
};

std::mutex g_mu;
std::atomic<long long> g_launches{0};
bool g_on = false;
bool g_created = false;
int g_used = 0;
cudaEvent_t g_ev[kPairs][2];
int g_kind[kPairs];
long long g_cnt[kKindCount];
double g_ms[kKindCount];
thread_local int t_cur = -1;

}  // namespace

// Inside a stream capture an event record must be "external" to become a
// graph node that fires on replay (a plain record only adds a dependency).
cudaError_t record(cudaEvent_t ev, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return cudaErrorUnknown;
  if (cs == cudaStreamCaptureStatusActive)
    return cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal);
  return cudaEventRecord(ev, st);
}

void trace_begin(int kind, cudaStream_t st) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  t_cur = -1;
  if (!g_on) return;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_on || g_used >= kPairs) return;
  const int p = g_used++;
  g_kind[p] = kind;
  if (record(g_ev[p][0], st) == cudaSuccess) t_cur = p;
}

void trace_end(int kind, cudaStream_t st) {
  (void)kind;
  if (t_cur < 0) return;
  record(g_ev[t_cur][1], st);
  t_cur = -1;
}

}  // namespace dspark

using namespace dspark;

extern "C" {

long long dspark_launch_count(void) { return g_launches.load(); }

int dspark_trace_start(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_created) {
    for (int p = 0; p < kPairs; ++p)
      for (int i = 0; i < 2; ++i)
        if (cudaEventCreate(&g_ev[p][i]) != cudaSuccess) return DSPARK_ERR_CUDA;
    g_created = true;
  }
  g_used = 0;
  for (int k = 0; k < kKindCount; ++k) {
    g_cnt[k] = 0;
    g_ms[k] = 0.0;
  }
  g_on = true;
  return DSPARK_OK;
}

int dspark_trace_stop(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_on = false;
  return DSPARK_OK;
}

int dspark_trace_collect(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (int p = 0; p < g_used; ++p) {
    if (cudaEventSynchronize(g_ev[p][1]) != cudaSuccess) return -1;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, g_ev[p][0], g_ev[p][1]) != cudaSuccess) return -1;
    g_cnt[g_kind[p]] += 1;
    g_ms[g_kind[p]] += ms;
  }
  return g_used;
}

int dspark_trace_kinds(void) { return kKindCount; }

int dspark_trace_get(int i, const char** name, long long* launches, double* total_ms) {
  if (i < 0 || i >= kKindCount || !name || !launches || !total_ms) return DSPARK_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  *name = kNames[i];
  *launches = g_cnt[i];
  *total_ms = g_ms[i];
  return DSPARK_OK;
}

}  // extern "C"
