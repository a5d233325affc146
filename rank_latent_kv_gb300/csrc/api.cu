// Library-wide entry points: error reporting, version, defaults.
#include <cstdio>
#include <map>
#include <mutex>
#include <string>
#include <tuple>

#include "palu_internal.cuh"

namespace palu {

static thread_local std::string g_last_error;

void set_error(const std::string& msg) { g_last_error = msg; }

palu_status fail(palu_status st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

palu_status cuda_check(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return PALU_OK;
  g_last_error = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return PALU_ERR_CUDA;
}

static std::mutex g_mu;

int device_sm_count() {
  static std::map<int, int> cache;
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = cache.find(dev);
  if (it != cache.end()) return it->second;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
  cache[dev] = n;
  return n;
}

palu_status kernel_occupancy(const void* kernel, int threads, int smem, int* per_sm) {
  static std::map<std::tuple<const void*, int, int, int>, int> cache;
  static std::map<std::pair<const void*, int>, int> attr_max;  // dynamic smem limit set per kernel and device
  int dev = 0;
  palu_status st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != PALU_OK) return st;
  const auto key = std::make_tuple(kernel, threads, smem, dev);
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = cache.find(key);
  if (it != cache.end()) {
    *per_sm = it->second;
    return PALU_OK;
  }
  // the limit is a property of the kernel: only ever raise it, never lower it.
  // Beyond 48 KB of static plus dynamic shared memory a block needs it.
  static std::map<std::pair<const void*, int>, int> static_smem;
  auto sit = static_smem.find(std::make_pair(kernel, dev));
  if (sit == static_smem.end()) {
    cudaFuncAttributes fa;
    st = cuda_check(cudaFuncGetAttributes(&fa, kernel), "cudaFuncGetAttributes");
    if (st != PALU_OK) return st;
    sit = static_smem.emplace(std::make_pair(kernel, dev), (int)fa.sharedSizeBytes).first;
  }
  int& cur = attr_max[std::make_pair(kernel, dev)];
  if (smem + sit->second > 48 * 1024 && smem > cur) {
    st = cuda_check(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem),
                    "cudaFuncSetAttribute(max dynamic shared memory)");
    if (st != PALU_OK) return st;
    cur = smem;
  }
  int n = 0;
  st = cuda_check(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem), "occupancy query");
  if (st != PALU_OK) return st;
  n = n > 0 ? n : 1;
  cache[key] = n;
  *per_sm = n;
  return PALU_OK;
}

}  // namespace palu

extern "C" const char* palu_last_error(void) { return palu::g_last_error.c_str(); }

extern "C" const char* palu_version(void) { return "libpalu 0.1.0 (sm_103a)"; }

extern "C" palu_status palu_config_default(palu_config* cfg) {
  if (!cfg) return palu::fail(PALU_ERR_INVALID_ARG, "config is NULL");
  cfg->head_dim = 128;
  cfg->n_head_groups = 4;
  cfg->rank = 0;
  cfg->energy_mode = PALU_ENERGY_SIGMA;
  cfg->energy_threshold = 0.90;
  cfg->hi_fraction = 0.25;
  cfg->hi_bit = 4;
  cfg->lo_bit = 2;
  cfg->group_size = 32;
  cfg->quantize = 1;
  return PALU_OK;
}
