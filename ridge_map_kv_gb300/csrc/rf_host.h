// Host-side helpers shared by the entry points: error text, argument checks,
// workspace carving, TMA descriptor encoding and device queries.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstddef>
#include <cstdint>

#include "rf.h"

namespace rf {

// Records a thread-local error text and returns `st`.
rf_status fail(rf_status st, const char* fmt, ...);
void clear_error();

// Maps a CUDA error to RF_ERR_CUDA with its text (RF_OK on success).
rf_status cuda_check(cudaError_t e, const char* what);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Current device: SM count and whether it is sm_100-family; RF_ERR_* on failure.
rf_status current_device(int* sm_count);

// Wait limit for bounded device waits, in ns.
uint64_t wait_timeout_ns();

// Builds a 2-D bf16 TMA descriptor with 128-byte swizzle and zero fill out of
// bounds: dims {inner, outer}, row stride in elements, box {box_inner, box_outer}.
rf_status make_tmap_bf16_2d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer,
                            uint64_t row_stride_elems, uint32_t box_inner, uint32_t box_outer);

// 3-D variant: dims {inner, mid, outer}, strides (elements) of mid and outer,
// box {box_inner, box_mid, 1}.
rf_status make_tmap_bf16_3d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t mid, uint64_t outer,
                            uint64_t mid_stride_elems, uint64_t outer_stride_elems, uint32_t box_inner,
                            uint32_t box_mid);

// Bump allocator over the caller workspace (256-byte aligned regions).
struct Carve {
  uint8_t* base;
  size_t off = 0;
  explicit Carve(void* b) : base(static_cast<uint8_t*>(b)) {}
  template <class T>
  T* take(size_t count) {
    off = (off + 255) & ~size_t(255);
    T* p = reinterpret_cast<T*>(base ? base + off : nullptr);
    off += count * sizeof(T);
    return p;
  }
  size_t bytes() const { return (off + 255) & ~size_t(255); }
};

inline int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// Clusters of 2 CTAs of `kernel` that fit on the device at once (cached per device).
int max_active_pairs(const void* kernel, size_t smem_bytes, int threads, int sms, int* cache);

// Sets the dynamic shared-memory limit of a kernel once per process and device.
rf_status set_smem_attr(const void* kernel, size_t bytes, uint64_t* done_mask);

// int8 map codes -> bf16 (exact), n % 16 == 0 (maps.cu).
rf_status expand_int8(const int8_t* q, __nv_bfloat16* out, size_t n, int sms, cudaStream_t s);
// The library's non-blocking copy stream for the current device (maps.cu).
rf_status copy_stream(cudaStream_t* out);

// From raw sums (solve.cu): μ_x = sx/n, μ_y = sy/n (n_y entries), n as double,
// α = λ tr(Gc)/d_in or λ, and H = Gc + αI in fp32 (and fp64 when H64 is set).
rf_status centre_system(const double* G, const double* sx, const double* sy, const int64_t* n, int d_in, long long n_y,
                        double lambda, int alpha_mode, double* mu_x, double* mu_y, double* n_out, double* alpha,
                        double* alpha_out, double* H64, float* H32, int sms, cudaStream_t s);

// For b < batch (solve.cu): W + b*sW (ld ldw) receives L_b^-1 of the SPD n x n block
// A + b*sA = L_b L_bᵀ (ld lda, n % 128 == 0), in fp32 SIMT (recursive halving,
// 128-wide leaves in shared memory). A is used as scratch; W's blocks above the
// diagonal must already be zero. tmp holds batch * stmp floats, stmp >= n * n / 4.
// A non-positive pivot records RF_ERR_NOT_SPD.
rf_status chol_inv_block(float* A, long long lda, long long sA, float* W, long long ldw, long long sW, int n, int batch,
                         float* tmp, long long stmp, int32_t* dev_status, int sms, cudaStream_t s);

// One SPD n x n matrix H (select.cu; n % 128 == 0; H is consumed): Linv = L^-1 of
// H = L Lᵀ and, when Hinv is set, Hinv = H^-1 = Linvᵀ Linv, exactly symmetric. The
// products of widths that are multiples of 512 and Linvᵀ Linv run as fp32-accurate
// split-bf16 tensor-core GEMMs (CTA pairs when `pair`), the rest as fp32 SIMT.
// ctmp holds n*n/4 floats, planes 3*n*n bf16. A non-positive pivot records
// RF_ERR_NOT_SPD.
rf_status spd_inverse(float* H, int n, float* Linv, float* Hinv, float* ctmp, __nv_bfloat16* planes, bool pair,
                      int32_t* dev_status, int sms, cudaStream_t s);

// Brackets one kernel launch with profiling events when rf_profile_start is active.
struct ProfScope {
  cudaStream_t stream;
  int slot;
  ProfScope(cudaStream_t s, int stage);
  ~ProfScope();
};

}  // namespace rf
