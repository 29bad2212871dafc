// rf_fill_kv_static: the RidgeFill fill for callers that cannot allocate device
// memory.
//
// Some callers have no way to obtain scratch memory on the GPU: a plugin inside a
// serving engine that owns every byte of device memory through its own pool and
// does not lend it out, or a latency-critical path where a cudaMalloc would
// synchronise the device and stall other work. For them this entry point runs
// the same fill as rf_fill_kv, but its scratch is a fixed array that lives in
// this file, in the library's device image:
//
//   static __device__ __align__(256) unsigned char g_fill_scratch[RF_STATIC_SCRATCH_BYTES];
//
// Every GPU that loads the library holds this array (64 MiB) until the process
// exits. Host code cannot use the array's name as a device address (on the host
// it is only a stand-in symbol), so the address is looked up once per device with
// cudaGetSymbolAddress, with that device current, and handed to the kernels as
// their workspace.
//
// No allocation: the call makes no cudaMalloc, cudaFree or any other allocating
// call; it only launches kernels on the caller's stream.
//
// Sharing: all calls on a device use the same array, and it keeps whatever the
// last call left in it. The fill writes every scratch value before it reads it in
// the same call, so nothing has to be cleared between calls. Two calls whose work
// overlaps on the GPU (for example on two streams without ordering) race on the
// array and corrupt each other's results; order such calls on one stream.
#include <mutex>

#include "rf_host.h"

namespace rf {

static __device__ __align__(256) unsigned char g_fill_scratch[RF_STATIC_SCRATCH_BYTES];

static std::mutex g_scratch_mu;
static void* g_scratch_ptr[64] = {nullptr};

// Device address of g_fill_scratch on the current device; set up on first use
// per device (this may load the library's device code on that device).
static rf_status static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_check(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(RF_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> g(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_fill_scratch);
    if (e != cudaSuccess) return cuda_check(e, "cudaGetSymbolAddress(static fill scratch)");
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return RF_OK;
}

}  // namespace rf

extern "C" rf_status rf_fill_kv_static(const rf_fill_desc* desc, const rf_bf16* x_S, int64_t ld_x,
                                       const uint8_t* exact_mask, const rf_bf16* A, const float* b,
                                       const rf_bf16* Wkv, rf_bf16* k_cache, rf_bf16* v_cache,
                                       int64_t layer_stride, int64_t row_stride, int32_t* n_fill_out,
                                       int32_t* dev_status, rf_stream_t stream) {
  rf::clear_error();
  const size_t need = rf_fill_workspace_bytes(desc);
  if (need == 0) return rf_fill_kv(desc, x_S, ld_x, exact_mask, A, b, Wkv, k_cache, v_cache, layer_stride,
                                   row_stride, n_fill_out, dev_status, nullptr, 0, stream);
  if (need > RF_STATIC_SCRATCH_BYTES)
    return rf::fail(RF_ERR_WORKSPACE,
                    "rf_fill_kv_static: this fill needs %zu bytes of scratch; the static scratch holds %zu bytes "
                    "(use rf_fill_kv with a workspace for larger fills)",
                    need, static_cast<size_t>(RF_STATIC_SCRATCH_BYTES));
  void* scratch = nullptr;
  rf_status st = rf::static_scratch(&scratch);
  if (st != RF_OK) return st;
  return rf_fill_kv(desc, x_S, ld_x, exact_mask, A, b, Wkv, k_cache, v_cache, layer_stride, row_stride, n_fill_out,
                    dev_status, scratch, RF_STATIC_SCRATCH_BYTES, stream);
}
