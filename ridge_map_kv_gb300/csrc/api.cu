// Library-wide entry points (version, status text, device support, wait limit)
// and the host helpers declared in rf_host.h.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdio>
#include <mutex>
#include <string>
#include <vector>

#include "rf_host.h"

namespace rf {

static thread_local std::string t_last_error;
static std::atomic<int64_t> g_timeout_ms{4000};

rf_status fail(rf_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return st;
}

void clear_error() { t_last_error.clear(); }

rf_status cuda_check(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return RF_OK;
  return fail(RF_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

rf_status current_device(int* sm_count) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_check(e, "cudaGetDevice");
  int major = 0;
  e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e != cudaSuccess) return cuda_check(e, "cudaDeviceGetAttribute(major)");
  if (major != 10) return fail(RF_ERR_UNSUPPORTED, "device %d has compute capability %d.x; need 10.x", dev, major);
  e = cudaDeviceGetAttribute(sm_count, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_check(e, "cudaDeviceGetAttribute(SMs)");
  return RF_OK;
}

uint64_t wait_timeout_ns() { return static_cast<uint64_t>(g_timeout_ms.load()) * 1000000ull; }

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

rf_status make_tmap_bf16_2d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer,
                            uint64_t row_stride_elems, uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return fail(RF_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride_elems * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(RF_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d): dims %llu x %llu, stride %llu B", (int)r,
                (unsigned long long)inner, (unsigned long long)outer, (unsigned long long)(row_stride_elems * 2));
  return RF_OK;
}

rf_status make_tmap_bf16_3d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t mid, uint64_t outer,
                            uint64_t mid_stride_elems, uint64_t outer_stride_elems, uint32_t box_inner,
                            uint32_t box_mid) {
  auto fn = encode_fn();
  if (!fn) return fail(RF_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[3] = {inner, mid, outer};
  cuuint64_t strides[2] = {mid_stride_elems * 2, outer_stride_elems * 2};
  cuuint32_t box[3] = {box_inner, box_mid, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(RF_ERR_CUDA, "cuTensorMapEncodeTiled (3-D) failed (%d)", (int)r);
  return RF_OK;
}

rf_status set_smem_attr(const void* kernel, size_t bytes, uint64_t* done_mask) {
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_check(e, "cudaGetDevice");
  std::lock_guard<std::mutex> g(mu);
  const uint64_t bit = uint64_t(1) << (dev & 63);
  if (*done_mask & bit) return RF_OK;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e != cudaSuccess) return cuda_check(e, "cudaFuncSetAttribute(max dynamic smem)");
  *done_mask |= bit;
  return RF_OK;
}

// How many clusters of 2 CTAs of `kernel` (`threads` threads, `smem_bytes` of
// dynamic shared memory) fit on the device at once. A persistent pair grid larger
// than this would run its last pairs after the others finish. Cached per device.
int max_active_pairs(const void* kernel, size_t smem_bytes, int threads, int sms, int* cache) {
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return std::max(sms / 2, 1);
  }
  std::lock_guard<std::mutex> g(mu);
  int& c = cache[dev & 63];
  if (c > 0) return c;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * std::max(sms / 2, 1));
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem_bytes;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = std::max(sms / 2, 1);
  }
  c = std::min(n, std::max(sms / 2, 1));
  return c;
}

// ----------------------------------------------------------------- profiler
struct ProfRecord {
  cudaEvent_t start = nullptr, stop = nullptr;
  int stage = 0;
};
static std::mutex g_prof_mu;
static std::vector<ProfRecord> g_prof;
static int g_prof_used = 0;
static bool g_prof_on = false;

ProfScope::ProfScope(cudaStream_t s, int stage) : stream(s), slot(-1) {
  std::lock_guard<std::mutex> g(g_prof_mu);
  if (!g_prof_on || g_prof_used >= static_cast<int>(g_prof.size())) return;
  slot = g_prof_used++;
  g_prof[slot].stage = stage;
  cudaEventRecord(g_prof[slot].start, stream);
}

ProfScope::~ProfScope() {
  if (slot < 0) return;
  std::lock_guard<std::mutex> g(g_prof_mu);
  if (slot < static_cast<int>(g_prof.size())) cudaEventRecord(g_prof[slot].stop, stream);
}

static void prof_release() {
  for (auto& r : g_prof) {
    if (r.start) cudaEventDestroy(r.start);
    if (r.stop) cudaEventDestroy(r.stop);
  }
  g_prof.clear();
  g_prof_used = 0;
  g_prof_on = false;
}

}  // namespace rf

extern "C" {

rf_status rf_profile_start(int max_records) {
  using namespace rf;
  clear_error();
  if (max_records <= 0) return fail(RF_ERR_INVALID_ARG, "max_records must be > 0");
  std::lock_guard<std::mutex> g(g_prof_mu);
  prof_release();
  g_prof.resize(max_records);
  for (auto& r : g_prof) {
    if (cudaEventCreate(&r.start) != cudaSuccess || cudaEventCreate(&r.stop) != cudaSuccess) {
      prof_release();
      return cuda_check(cudaGetLastError(), "cudaEventCreate");
    }
  }
  g_prof_on = true;
  return RF_OK;
}

int rf_profile_stop(int32_t* stage_ids, float* ms, int capacity) {
  using namespace rf;
  std::lock_guard<std::mutex> g(g_prof_mu);
  int n = 0;
  bool err = false;
  for (int i = 0; i < g_prof_used; ++i) {
    float t = 0.f;
    if (cudaEventSynchronize(g_prof[i].stop) != cudaSuccess ||
        cudaEventElapsedTime(&t, g_prof[i].start, g_prof[i].stop) != cudaSuccess) {
      err = true;
      break;
    }
    if (n < capacity) {
      if (stage_ids) stage_ids[n] = g_prof[i].stage;
      if (ms) ms[n] = t;
      ++n;
    }
  }
  prof_release();
  return err ? -1 : n;
}

const char* rf_stage_name(int s) {
  switch (s) {
    case RF_STAGE_COMPACT: return "compact";
    case RF_STAGE_GATHER: return "gather";
    case RF_STAGE_ROPE_TABLE: return "rope_table";
    case RF_STAGE_MAP_GEMM: return "map_gemm";
    case RF_STAGE_KV_GEMM: return "kv_gemm";
    case RF_STAGE_FOLD: return "fold";
    case RF_STAGE_CALIB_GEMM: return "calib_gemm";
    case RF_STAGE_COLSUM: return "colsum";
    case RF_STAGE_SOLVE: return "solve";
    case RF_STAGE_UNROPE: return "unrope";
    case RF_STAGE_XMODEL_GEMM: return "xmodel_gemm";
    case RF_STAGE_RESCALE: return "value_rescale";
    case RF_STAGE_EXPAND: return "int8_expand";
    case RF_STAGE_QUANTIZE: return "int8_quantize";
    case RF_STAGE_SOLVE_PRODUCT: return "solve_product";
    case RF_STAGE_SOLVE_REFINE: return "solve_refine";
    case RF_STAGE_ROW_RMS: return "row_rms";
    case RF_STAGE_SELECT_GEMM: return "select_gemm";
    case RF_STAGE_SELECT_FACTOR: return "select_factor";
    case RF_STAGE_SELECT_SCORE: return "select_score";
    case RF_STAGE_SELECT_SPLIT: return "select_split";
    default: return "unknown";
  }
}

int rf_version(void) { return 100; }

const char* rf_status_string(int s) {
  switch (s) {
    case RF_OK: return "ok";
    case RF_ERR_INVALID_ARG: return "invalid argument";
    case RF_ERR_SHAPE: return "unsupported shape";
    case RF_ERR_ALIGN: return "misaligned pointer or stride";
    case RF_ERR_CUDA: return "CUDA error";
    case RF_ERR_NOT_SPD: return "matrix not positive definite";
    case RF_ERR_TIMEOUT: return "device wait timed out";
    case RF_ERR_UNSUPPORTED: return "device not supported (need sm_100 family)";
    case RF_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    default: return "unknown status";
  }
}

const char* rf_last_error(void) { return rf::t_last_error.c_str(); }

int rf_device_supported(int device) {
  int major = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return major == 10 ? 1 : 0;
}

void rf_set_wait_timeout_ms(int64_t ms) { rf::g_timeout_ms.store(ms < 1 ? 4000 : ms); }

}  // extern "C"
