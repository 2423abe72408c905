// Prefix scheduler for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or hand the library a workspace: a
// serving engine that replays a fixed, pre-planned memory map (every buffer
// is reserved once at start-up, and an allocation in the decode loop would
// break the plan or the graph capture that replays it), or a plugin running
// inside a host framework that owns the device heap.  For them this file
// provides dspark_schedule_noalloc: the same scheduler kernel as
// dspark_schedule, with its scratch (candidate ranks, the sort's two key
// buffers, a status word) in a file-scope device array instead of a caller
// workspace.
//
// Limits and rules:
// * at most kNoAllocMaxCandidates (= 32768) candidates, R * gamma; larger
//   problems are rejected with DSPARK_ERR_INVALID_ARG;
// * the array (32768 * 20 + 256 bytes, about 640 KiB) lives on every GPU that
//   loads the library, until the process exits;
// * every call shares it: calls that overlap on the GPU (two streams, or two
//   host threads) race on it and must be serialised by the caller;
// * the first call on each device resolves the array's device address with
//   cudaGetSymbolAddress while that device is current; make that first call
//   before any stream capture.
#include <stdio.h>

#include <mutex>

#include "dspark.h"
#include "common.cuh"

namespace dspark {

namespace {

constexpr int kNoAllocMaxCandidates = 32768;
constexpr size_t kRankBytes = (size_t)kNoAllocMaxCandidates * sizeof(int32_t);
constexpr size_t kKeyBytes = (size_t)kNoAllocMaxCandidates * 2 * sizeof(unsigned long long);
constexpr size_t kScratchBytes = 256 + kRankBytes + kKeyBytes;
static_assert(kRankBytes + kKeyBytes == sched_scratch_bytes(kNoAllocMaxCandidates),
              "the scheduler's scratch layout");

// Layout: [0, 4) status word, [256, 256 + kRankBytes) ranks, then the two
// sort-key buffers (8-byte words).
static __device__ __align__(256) unsigned char g_sched_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch array for the current device (resolved once
// per device).  Returns nullptr and sets *err on failure.
void* scratch_for_current_device(cudaError_t* err) {
  int dev = -1;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_sched_scratch);
    if (*err != cudaSuccess) return nullptr;
    g_addr[dev] = p;
  }
  return g_addr[dev];
}

thread_local char g_msg[200] = "";

}  // namespace

}  // namespace dspark

using namespace dspark;

extern "C" {

int dspark_schedule_noalloc(int R, int gamma, const float* a, const float* sps, int n_sps,
                            int early_stop, int max_B, int32_t* ell, int32_t* row_off,
                            int32_t* B_out, double* E_out, uint32_t* dev_status, void* stream) {
  // Same argument rules as dspark_schedule, plus the size limit of the
  // static scratch array; every rejection leaves a reason for
  // dspark_last_error().
  if (R < 1 || gamma < 1 || gamma > kMaxGamma || (long long)R * gamma > kNoAllocMaxCandidates) {
    snprintf(g_msg, sizeof(g_msg),
             "dspark_schedule_noalloc: R*gamma = %lld (R=%d, gamma=%d) must be in [1, %d] "
             "(the size of its static scratch) with 1 <= gamma <= %d",
             (long long)R * gamma, R, gamma, kNoAllocMaxCandidates, kMaxGamma);
    set_error_text(g_msg);
    return DSPARK_ERR_INVALID_ARG;
  }
  if (!a || !sps || !ell || !row_off || !B_out || !E_out) {
    set_error_text("dspark_schedule_noalloc: a, sps, ell, row_off, B_out and E_out must be non-NULL");
    return DSPARK_ERR_INVALID_ARG;
  }
  const int N = R * gamma;
  if (max_B < 0 || (max_B > 0 && max_B < R)) {
    set_error_text("dspark_schedule_noalloc: max_B must be 0 or >= R");
    return DSPARK_ERR_INVALID_ARG;
  }
  const int imax = max_B > 0 ? (max_B - R < N ? max_B - R : N) : N;
  if ((long long)n_sps <= (long long)R + imax) {
    snprintf(g_msg, sizeof(g_msg),
             "dspark_schedule_noalloc: SPS table has %d entries, needs more than R + imax = %d",
             n_sps, R + imax);
    set_error_text(g_msg);
    return DSPARK_ERR_INVALID_ARG;
  }
  cudaError_t e;
  unsigned char* base = static_cast<unsigned char*>(scratch_for_current_device(&e));
  if (base == nullptr) {
    snprintf(g_msg, sizeof(g_msg), "dspark_schedule_noalloc: scratch set-up failed: %s",
             cudaGetErrorString(e));
    set_error_text(g_msg);
    return DSPARK_ERR_CUDA;
  }
  SchedArgs s{};
  s.R = R;
  s.gamma = gamma;
  s.n_sps = n_sps;
  s.early_stop = early_stop;
  s.max_B = max_B;
  s.a = a;
  s.sps = sps;
  s.ell = ell;
  s.row_off = row_off;
  s.B_out = B_out;
  s.E_out = E_out;
  s.status = dev_status ? dev_status : reinterpret_cast<uint32_t*>(base);
  s.imax = imax;
  s.rank = reinterpret_cast<int32_t*>(base + 256);  // fully overwritten by each call
  s.keys = reinterpret_cast<unsigned long long*>(base + 256 + kRankBytes);  // likewise
  e = launch_schedule(s, (cudaStream_t)stream);
  if (e != cudaSuccess) {
    snprintf(g_msg, sizeof(g_msg), "dspark_schedule_noalloc: %s", cudaGetErrorString(e));
    set_error_text(g_msg);
    return DSPARK_ERR_CUDA;
  }
  return DSPARK_OK;
}

}  // extern "C"
