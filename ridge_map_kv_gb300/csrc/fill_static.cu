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
// it is only a stand-in symbol), so every call looks the address up with
// cudaGetSymbolAddress in the caller's current context and hands it to the kernels
// as their workspace. Nothing is cached: after a cudaDeviceReset, or in another
// context of the same device, the array can sit at another address, and a cached
// one would send the fill's writes to memory it does not own. The lookup is a host
// call (the first one in a context loads the library's device code there).
//
// No allocation: the call makes no cudaMalloc, cudaFree or any other allocating
// call; it only launches kernels on the caller's stream.
//
// Sharing: all calls on a device use the same array, and it keeps whatever the
// last call left in it. The fill writes every scratch value before it reads it in
// the same call, so nothing has to be cleared between calls. Two calls whose work
// overlaps on the GPU (for example on two streams without ordering) race on the
// array and corrupt each other's results; order such calls on one stream.
#include "rf_host.h"

namespace rf {

static __device__ __align__(256) unsigned char g_fill_scratch[RF_STATIC_SCRATCH_BYTES];

// Device address of g_fill_scratch in the current context, looked up on every call.
static rf_status static_scratch(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_fill_scratch);
  if (e != cudaSuccess) return cuda_check(e, "cudaGetSymbolAddress(static fill scratch)");
  if (reinterpret_cast<uintptr_t>(p) & 255u) return fail(RF_ERR_CUDA, "static fill scratch is not 256-byte aligned");
  *out = p;
  return RF_OK;
}

}  // namespace rf

extern "C" rf_status rf_fill_kv_static(const rf_fill_desc* desc, const rf_bf16* x_S, int64_t ld_x,
                                       const uint8_t* exact_mask, const rf_bf16* A, const float* b,
                                       const rf_bf16* gain, const rf_bf16* Wk, const rf_bf16* Wv, rf_bf16* k_cache,
                                       rf_bf16* v_cache, int64_t layer_stride, int64_t row_stride,
                                       int32_t* n_fill_out, int32_t* dev_status, rf_stream_t stream) {
  rf::clear_error();
  const size_t need = rf_fill_workspace_bytes(desc);
  if (need == 0)
    return rf_fill_kv(desc, x_S, ld_x, exact_mask, A, b, gain, Wk, Wv, k_cache, v_cache, layer_stride, row_stride,
                      n_fill_out, dev_status, nullptr, 0, stream);
  if (need > RF_STATIC_SCRATCH_BYTES)
    return rf::fail(RF_ERR_WORKSPACE,
                    "rf_fill_kv_static: this fill needs %zu bytes of scratch; the static scratch holds %zu bytes "
                    "(use rf_fill_kv with a workspace for larger fills)",
                    need, static_cast<size_t>(RF_STATIC_SCRATCH_BYTES));
  void* scratch = nullptr;
  rf_status st = rf::static_scratch(&scratch);
  if (st != RF_OK) return st;
  return rf_fill_kv(desc, x_S, ld_x, exact_mask, A, b, gain, Wk, Wv, k_cache, v_cache, layer_stride, row_stride,
                    n_fill_out, dev_status, scratch, RF_STATIC_SCRATCH_BYTES, stream);
}
