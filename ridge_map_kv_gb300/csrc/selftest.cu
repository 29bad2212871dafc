// rf_selftest_wait_timeout: exercises the bounded-wait abort path of the GEMM
// core on the GPU. The problem's producer announces its bytes on the `full`
// barrier but issues no copy, so the MMA thread's wait can only run out: the
// kernel must raise its abort flag, drain, free TMEM, write RF_ERR_TIMEOUT to the
// status word and exit, leaving the context usable. No copy or MMA is ever in
// flight, so nothing can land after the CTA has gone. In the dynamic unit order
// the same run also passes a unit through the shared-memory ring and leaves the
// ring's waits to the abort.
#include "rf_host.h"
#include "tc_gemm.cuh"

namespace rf {

template <bool kPair_>
struct NeverReadyProb {
  int32_t* dev_status;
  uint64_t timeout_ns;
  int* sched;  // unit counter (dynamic unit order), or nullptr
  static constexpr bool kAMN = false;
  static constexpr bool kBMN = false;
  static constexpr bool kPair = kPair_;
  static constexpr int kEpiWarps = 4;
  struct EpiState {};
  struct Coords {};
  using Cfg = GemmCfg<kPair_>;
  __device__ void prefetch() const {}
  __device__ int num_units() const { return 1; }
  __device__ int num_subtiles(int) const { return 1; }
  __device__ int num_kb(int, int) const { return 8; }
  __device__ Coords coords(int, int, uint32_t) const { return {}; }
  __device__ void issue_loads(Coords&, int, uint8_t*, uint8_t*, uint32_t) const {}
  __device__ void epilogue(EpiState&, int, int, int, uint32_t, int, int, uint32_t) const {}
  __device__ void epilogue_after(EpiState&, int, int, int, int, int, uint32_t) const {}
};

// The self-test's unit counter (one int; the launch clears it).
static __device__ int g_selftest_sched;

}  // namespace rf

using namespace rf;

extern "C" rf_status rf_selftest_wait_timeout(int mode, int32_t* dev_status, rf_stream_t stream) {
  clear_error();
  if (dev_status == nullptr) return fail(RF_ERR_INVALID_ARG, "dev_status must be non-NULL");
  if (mode < 0 || mode > 3) return fail(RF_ERR_INVALID_ARG, "mode must be 0..3");
  int sms = 0;
  rf_status st = current_device(&sms);
  if (st != RF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* sched = nullptr;
  if (mode & 2) {
    // looked up in the current context on every call (the host-side name is not a device address)
    if ((st = cuda_check(cudaGetSymbolAddress(reinterpret_cast<void**>(&sched), g_selftest_sched),
                         "self-test counter address")) != RF_OK)
      return st;
  }
  if (mode & 1) {
    NeverReadyProb<true> pr{dev_status, wait_timeout_ns(), sched};
    return launch_gemm(pr, 1, sms, s, "self-test launch");
  }
  NeverReadyProb<false> pr{dev_status, wait_timeout_ns(), sched};
  return launch_gemm(pr, 1, sms, s, "self-test launch");
}
