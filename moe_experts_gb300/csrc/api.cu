// Host-side plumbing of the C ABI: status strings, format sizes, the
// per-device attribute cache and the device error word.
#include <atomic>
#include <mutex>

#include "common.cuh"

namespace epq {

// One error word per device (a separate instance lives on every device that
// loads the library).
__device__ unsigned g_device_error[4] = {0, 0, 0, 0};

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceInfo g_info[kMaxDevices];
unsigned *g_err_slot[kMaxDevices] = {};
thread_local int g_last_cuda_error = 0;
}  // namespace

bool current_device(DeviceInfo *out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return false;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo &d = g_info[dev];
  if (d.device != dev) {
    DeviceInfo t;
    t.device = dev;
    if (cudaDeviceGetAttribute(&t.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&t.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&t.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&t.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&t.l2_bytes, cudaDevAttrL2CacheSize, dev) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    d = t;
  }
  *out = d;
  return true;
}

unsigned *device_error_slot() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_slot[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_err_slot[dev] = static_cast<unsigned *>(p);
  }
  return g_err_slot[dev];
}

namespace {
std::atomic<int> g_tile_bytes{32 * 1024};
std::atomic<int> g_ring_bytes{180 * 1024};
std::atomic<int> g_gemv_engine{0};
std::atomic<int> g_early_stages{4};
std::atomic<int> g_tc_split{0};
std::atomic<int> g_attn_chunk{0};
std::atomic<int> g_vn_chunk{0};
std::atomic<int> g_vn_cluster{0};
}  // namespace

int tune_tile_bytes() { return g_tile_bytes.load(std::memory_order_relaxed); }
int tune_ring_bytes() { return g_ring_bytes.load(std::memory_order_relaxed); }
int tune_gemv_engine() { return g_gemv_engine.load(std::memory_order_relaxed); }
int tune_early_stages() { return g_early_stages.load(std::memory_order_relaxed); }
int tune_tc_split() { return g_tc_split.load(std::memory_order_relaxed); }
int tune_attn_chunk() { return g_attn_chunk.load(std::memory_order_relaxed); }
int tune_vn_chunk() { return g_vn_chunk.load(std::memory_order_relaxed); }
int tune_vn_cluster() { return g_vn_cluster.load(std::memory_order_relaxed); }

epq_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return EPQ_ERR_CUDA;
}

}  // namespace epq

extern "C" {

const char *epq_status_string(epq_status s) {
  switch (s) {
    case EPQ_OK: return "ok";
    case EPQ_ERR_ARG: return "invalid argument";
    case EPQ_ERR_FORMAT: return "unknown block format";
    case EPQ_ERR_SHAPE: return "unsupported shape";
    case EPQ_ERR_ALIGN: return "pointer not 16-byte aligned";
    case EPQ_ERR_WORKSPACE: return "workspace missing or too small";
    case EPQ_ERR_CUDA: return "CUDA runtime error";
    case EPQ_ERR_DEVICE: return "no usable sm_103 device";
  }
  return "unknown status";
}

int epq_last_cuda_error(void) { return epq::g_last_cuda_error; }

int epq_set_tuning(int key, int value) {
  switch (key) {
    case EPQ_TUNE_TILE_BYTES:
      if (value < 4096 || value > 131072) return -1;
      return epq::g_tile_bytes.exchange(value);
    case EPQ_TUNE_RING_BYTES:
      if (value < 32768 || value > 200704) return -1;
      return epq::g_ring_bytes.exchange(value);
    case EPQ_TUNE_GEMV_ENGINE:
      if (value < 0 || value > 4) return -1;
      return epq::g_gemv_engine.exchange(value);
    case EPQ_TUNE_EARLY_STAGES:
      if (value < 0 || value > 16) return -1;
      return epq::g_early_stages.exchange(value);
    case EPQ_TUNE_TC_SPLIT:
      if (value != 0 && value != 1 && value != 2 && value != 4 && value != 8 && value != 16) return -1;
      return epq::g_tc_split.exchange(value);
    case EPQ_TUNE_ATTN_CHUNK:
      if (value != 0 && (value < 8 || value > 4096 || value % 8)) return -1;
      return epq::g_attn_chunk.exchange(value);
    case EPQ_TUNE_VN_CHUNK:
      if (value < 0 || value > 64) return -1;
      return epq::g_vn_chunk.exchange(value);
    case EPQ_TUNE_VN_CLUSTER:
      if (value != 0 && value != 1 && value != 2 && value != 4) return -1;
      return epq::g_vn_cluster.exchange(value);
  }
  return -1;
}

int epq_device_error_detail(int *block, int *where, int *thread) {
  unsigned *slot = epq::device_error_slot();
  if (!slot) return -1;
  unsigned v[4] = {0, 0, 0, 0};
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  if (cudaMemcpyFromSymbol(v, epq::g_device_error, sizeof(v)) != cudaSuccess) return -1;
  const unsigned zero[4] = {0, 0, 0, 0};
  if (cudaMemcpyToSymbol(epq::g_device_error, zero, sizeof(zero)) != cudaSuccess) return -1;
  if (block) *block = static_cast<int>(v[1]);
  if (where) *where = static_cast<int>(v[2]);
  if (thread) *thread = static_cast<int>(v[3]);
  return static_cast<int>(v[0]);
}

int epq_device_error(void) { return epq_device_error_detail(nullptr, nullptr, nullptr); }

int64_t epq_block_weights(epq_fmt fmt) {
  switch (fmt) {
    case EPQ_Q8_0:
    case EPQ_Q4_0:
    case EPQ_Q4_1: return 32;
    case EPQ_Q4_K:
    case EPQ_Q2_K:
    case EPQ_Q6_K: return 256;
  }
  return -1;
}

int64_t epq_block_bytes(epq_fmt fmt) {
  switch (fmt) {
    case EPQ_Q8_0: return 34;
    case EPQ_Q4_0: return 18;
    case EPQ_Q4_1: return 20;
    case EPQ_Q4_K: return 144;
    case EPQ_Q2_K: return 84;
    case EPQ_Q6_K: return 210;
  }
  return -1;
}

int64_t epq_row_bytes(epq_fmt fmt, int64_t cols) {
  const int64_t bw = epq_block_weights(fmt);
  if (bw < 0 || cols <= 0 || cols % bw) return -1;
  return cols / bw * epq_block_bytes(fmt);
}

}  // extern "C"
