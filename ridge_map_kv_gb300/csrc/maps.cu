// Map storage: the int8 code of the maps (rf_quantize_maps_int8), the int8 -> bf16
// expansion the layer-by-layer fill runs before each layer's map GEMM, and the
// library's copy stream for host-resident maps.
//
// [RF] RidgeFill review, "Ridge map": at 27B the 48 upper-layer maps "in int8
// total 1.2 GiB", and "maps can be kept resident in GPU memory or streamed from
// host memory one layer at a time". The pages give no int8 scheme; the library's
// is symmetric per output row: s[o] = max_i |A[o][i]| / 127 and
// q[o][i] = rint(A[o][i] / s[o]) (ties to even), both in fp32; a zero row has
// s = 0 and q = 0. Since |q| <= 127 is exact in bf16, expanding q to bf16 is a
// pure type change, and the map GEMM applies s[o] to its output column o.
#include <algorithm>
#include <mutex>

#include "rf_host.h"
#include "rf_device.cuh"

namespace rf {

// One CTA per map row: absmax, scale, then the rounded codes.
__global__ void __launch_bounds__(256) k_quantize_rows(const __nv_bfloat16* __restrict__ A, int8_t* __restrict__ q,
                                                       float* __restrict__ s, int d_in) {
  const size_t row = blockIdx.x;
  const __nv_bfloat16* a = A + row * d_in;
  float m = 0.f;
  for (int i = threadIdx.x; i < d_in; i += blockDim.x) m = fmaxf(m, fabsf(__bfloat162float(a[i])));
  __shared__ float red[8];
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    for (int o = 16; o > 0; o >>= 1) t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, o));
    if (threadIdx.x == 0) red[0] = t;
  }
  __syncthreads();
  const float sc = red[0] / 127.0f;
  if (threadIdx.x == 0) s[row] = sc;
  int8_t* qr = q + row * d_in;
  for (int i = threadIdx.x; i < d_in; i += blockDim.x) {
    float v = 0.f;
    if (sc > 0.f) v = fminf(fmaxf(rintf(__bfloat162float(a[i]) / sc), -127.f), 127.f);
    qr[i] = static_cast<int8_t>(v);
  }
}

// bf16(q) for n int8 codes (n % 16 == 0), 16 per thread-step.
__global__ void __launch_bounds__(256) k_expand_int8(const int4* __restrict__ q, uint4* __restrict__ out, size_t n16) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n16;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int4 v = __ldg(q + i);
    const int8_t* b = reinterpret_cast<const int8_t*>(&v);
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] = pack_bf16x2(static_cast<float>(b[2 * j]), static_cast<float>(b[2 * j + 1]));
    out[2 * i] = make_uint4(w[0], w[1], w[2], w[3]);
    out[2 * i + 1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

rf_status expand_int8(const int8_t* q, __nv_bfloat16* out, size_t n, int sms, cudaStream_t s) {
  const size_t n16 = n / 16;
  const unsigned blocks = static_cast<unsigned>(std::min<size_t>((n16 + 255) / 256, static_cast<size_t>(4) * sms));
  ProfScope prof(s, RF_STAGE_EXPAND);
  k_expand_int8<<<blocks, 256, 0, s>>>(reinterpret_cast<const int4*>(q), reinterpret_cast<uint4*>(out), n16);
  return cuda_check(cudaGetLastError(), "int8 expansion launch");
}

// One non-blocking copy stream per device, created on first use and kept for the
// life of the process.
rf_status copy_stream(cudaStream_t* out) {
  static std::mutex mu;
  static cudaStream_t streams[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_check(e, "cudaGetDevice");
  std::lock_guard<std::mutex> g(mu);
  cudaStream_t& st = streams[dev & 63];
  if (st == nullptr) {
    e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
    if (e != cudaSuccess) {
      st = nullptr;
      return cuda_check(e, "cudaStreamCreateWithFlags (copy stream)");
    }
  }
  *out = st;
  return RF_OK;
}

}  // namespace rf

using namespace rf;

extern "C" rf_status rf_quantize_maps_int8(const rf_fill_desc* desc, const rf_bf16* A, int8_t* q, float* s,
                                           rf_stream_t stream) {
  clear_error();
  if (desc == nullptr) return fail(RF_ERR_INVALID_ARG, "desc is NULL");
  const int64_t P = desc->L - desc->S, d = desc->d, d_in = desc->d_in > 0 ? desc->d_in : desc->d;
  if (P < 0 || d <= 0 || d_in <= 0 || d % 256 != 0 || d_in % 256 != 0)
    return fail(RF_ERR_SHAPE, "need 0 <= S <= L and d, d_in multiples of 256");
  if (P == 0) return RF_OK;
  if (!A || !q || !s) return fail(RF_ERR_INVALID_ARG, "A, q and s must be non-NULL");
  if (P * d >= (int64_t(1) << 31)) return fail(RF_ERR_SHAPE, "too many map rows");
  int sms = 0;
  rf_status st = current_device(&sms);
  if (st != RF_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  ProfScope prof(cs, RF_STAGE_QUANTIZE);
  k_quantize_rows<<<static_cast<unsigned>(P * d), 256, 0, cs>>>(reinterpret_cast<const __nv_bfloat16*>(A), q, s,
                                                                static_cast<int>(d_in));
  return cuda_check(cudaGetLastError(), "k_quantize_rows launch");
}
