// Per-device launch set-up shared by the kernels' launchers: the SM count,
// the dynamic shared-memory opt-in (a per-device function attribute) and
// occupancy queries.  Everything is keyed by the current device and guarded
// by one mutex, so a process that drives several GPUs, or calls the library
// from several host threads, sets each device up exactly once and never
// launches on a device whose opt-in was made on another.
#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"

namespace dspark {

namespace {

std::mutex g_mu;
std::map<int, int> g_sms;                                        // device -> SMs
std::map<std::pair<int, const void*>, int> g_smem;               // (device, func) -> bytes set
std::map<std::tuple<int, const void*, int, size_t>, int> g_occ;  // -> blocks per SM

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  return dev;
}

}  // namespace

int sm_count() {
  const int dev = current_device();
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_sms.find(dev);
  if (it != g_sms.end()) return it->second;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    return 148;  // not cached: asked again next time
  g_sms[dev] = n;
  return n;
}

cudaError_t ensure_smem_attr(const void* func, int bytes) {
  const int dev = current_device();
  std::lock_guard<std::mutex> lk(g_mu);
  auto key = std::make_pair(dev, func);
  auto it = g_smem.find(key);
  if (it != g_smem.end() && it->second >= bytes) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) g_smem[key] = bytes;
  return e;
}

int blocks_per_sm(const void* func, int threads, size_t dyn_smem) {
  const int dev = current_device();
  std::lock_guard<std::mutex> lk(g_mu);
  auto key = std::make_tuple(dev, func, threads, dyn_smem);
  auto it = g_occ.find(key);
  if (it != g_occ.end()) return it->second;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, func, threads, dyn_smem) != cudaSuccess ||
      n < 1)
    return 0;  // not cached: asked again next time
  g_occ[key] = n;
  return n;
}

}  // namespace dspark
