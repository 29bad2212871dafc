// Closed-form ridge solve (rf_solve).
//
// [RF] RidgeFill review, "Ridge map": A_l = Y_lᵀX (XᵀX + αI)^-1, b_l = μ_l − A_l μ_S
// on centred data, α = λ·tr(XᵀX)/d_in; the statistics are read only, so a new λ is
// a re-solve. [XM] per-head ridge regression uses the same closed form (α = λ).
//
// From the one-pass sums (G, C, sx, sy, n) in fp64:
//   k_means, k_trace_alpha  μ_x = sx/n, μ_p = sy_p/n, tr(Gc), α
//   k_build_h               H = Gc + αI with Gc = G − n μ_x μ_xᵀ (fp64 and fp32 copies)
//   chol_lower (recursive)  H = L Lᵀ in fp32: a one-CTA kernel factors 128 x 128
//                           diagonal blocks; panels and trailing updates are fp32
//                           GEMMs (k_sgemm) with the inverse of the diagonal block
//   trinv_lower (recursive) L^-1 from one-CTA diagonal inverses and fp32 GEMMs
//   k_sgemm                 H^-1 = L^-ᵀ L^-1, then A_p = Cc_pᵀ H^-1 for every map
//   refinement (optional)   R_p = Cc_pᵀ − A_p H with fp64 products (k_resid64),
//                           A_p += R_p H^-1 (fp32)
//   k_bias                  b_p = μ_p − A_p μ_x (fp64 accumulation)
#include <algorithm>

#include "rf_host.h"
#include "rf_device.cuh"

namespace rf {

constexpr int kSolveBlock = 128;  // diagonal block size of the recursive factorisation

// --------------------------------------------------------------------------
// fp32 GEMM, C[b] = alpha op(A[b]) op(B[b]) + beta C[b]. 128 x 128 x 8 tiles,
// 256 threads, 8 x 8 outputs per thread, double-buffered shared tiles.
// Requires M % 128 == 0, N % 128 == 0, K % 8 == 0, 16-byte aligned rows.
// op(A)[m][k] = TA ? A[k*lda + m] : A[m*lda + k]; op(B)[k][n] = TB ? B[n*ldb + k] : B[k*ldb + n].
// --------------------------------------------------------------------------
template <bool TA, bool TB>
__global__ void __launch_bounds__(256) k_sgemm(int M, int N, int K, float alpha, const float* __restrict__ A,
                                               long long lda, long long sA, const float* __restrict__ B, long long ldb,
                                               long long sB, float beta, float* C, long long ldc, long long sC) {
  __shared__ __align__(16) float As[2][8][128];
  __shared__ __align__(16) float Bs[2][8][128];
  const int tid = threadIdx.x;
  const int bm = blockIdx.y * 128, bn = blockIdx.x * 128;
  A += blockIdx.z * sA;
  B += blockIdx.z * sB;
  C += blockIdx.z * sC;
  const int ty = tid >> 4, tx = tid & 15;

  auto load_a = [&](int k0, float4& r) {
    if (TA) r = *reinterpret_cast<const float4*>(A + static_cast<long long>(k0 + (tid >> 5)) * lda + bm + (tid & 31) * 4);
    else r = *reinterpret_cast<const float4*>(A + static_cast<long long>(bm + (tid >> 1)) * lda + k0 + (tid & 1) * 4);
  };
  auto load_b = [&](int k0, float4& r) {
    if (TB) r = *reinterpret_cast<const float4*>(B + static_cast<long long>(bn + (tid >> 1)) * ldb + k0 + (tid & 1) * 4);
    else r = *reinterpret_cast<const float4*>(B + static_cast<long long>(k0 + (tid >> 5)) * ldb + bn + (tid & 31) * 4);
  };
  auto store_a = [&](int buf, const float4& r) {
    if (TA) {
      *reinterpret_cast<float4*>(&As[buf][tid >> 5][(tid & 31) * 4]) = r;
    } else {
      const int m = tid >> 1, k = (tid & 1) * 4;
      As[buf][k][m] = r.x;
      As[buf][k + 1][m] = r.y;
      As[buf][k + 2][m] = r.z;
      As[buf][k + 3][m] = r.w;
    }
  };
  auto store_b = [&](int buf, const float4& r) {
    if (TB) {
      const int n = tid >> 1, k = (tid & 1) * 4;
      Bs[buf][k][n] = r.x;
      Bs[buf][k + 1][n] = r.y;
      Bs[buf][k + 2][n] = r.z;
      Bs[buf][k + 3][n] = r.w;
    } else {
      *reinterpret_cast<float4*>(&Bs[buf][tid >> 5][(tid & 31) * 4]) = r;
    }
  };

  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  float4 ra, rb;
  load_a(0, ra);
  load_b(0, rb);
  store_a(0, ra);
  store_b(0, rb);
  __syncthreads();
  int buf = 0;
  for (int k0 = 0; k0 < K; k0 += 8) {
    const bool more = k0 + 8 < K;
    if (more) {
      load_a(k0 + 8, ra);
      load_b(k0 + 8, rb);
    }
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][64 + tx * 4]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    if (more) {
      store_a(buf ^ 1, ra);
      store_b(buf ^ 1, rb);
    }
    __syncthreads();
    buf ^= 1;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int m = bm + (i < 4 ? ty * 4 + i : 64 + ty * 4 + i - 4);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float* cp = C + static_cast<long long>(m) * ldc + bn + h * 64 + tx * 4;
      float4 o = make_float4(alpha * acc[i][4 * h], alpha * acc[i][4 * h + 1], alpha * acc[i][4 * h + 2],
                             alpha * acc[i][4 * h + 3]);
      if (beta != 0.f) {
        const float4 c = *reinterpret_cast<const float4*>(cp);
        o.x = fmaf(beta, c.x, o.x);
        o.y = fmaf(beta, c.y, o.y);
        o.z = fmaf(beta, c.z, o.z);
        o.w = fmaf(beta, c.w, o.w);
      }
      *reinterpret_cast<float4*>(cp) = o;
    }
  }
}

// --------------------------------------------------------------------------
// One-CTA kernels on a 128 x 128 (or smaller) diagonal block held in shared memory.
// --------------------------------------------------------------------------
constexpr int kBlkLd = kSolveBlock + 1;
constexpr size_t kBlkSmem = sizeof(float) * kSolveBlock * kBlkLd;

// In-place lower Cholesky of the n x n block at A (n <= 128); zeroes the upper
// triangle. A non-positive pivot records RF_ERR_NOT_SPD and continues with 1.
__global__ void __launch_bounds__(256) k_chol_base(float* A, int n, long long lda, int32_t* dev_status) {
  extern __shared__ float S[];
  for (int e = threadIdx.x; e < n * n; e += blockDim.x) {
    const int i = e / n, j = e % n;
    S[i * kBlkLd + j] = A[i * lda + j];
  }
  __syncthreads();
  for (int j = 0; j < n; ++j) {
    if (threadIdx.x == 0) {
      float d = S[j * kBlkLd + j];
      if (!(d > 0.f)) {
        record_status(dev_status, RF_ERR_NOT_SPD);
        d = 1.f;
      }
      S[j * kBlkLd + j] = sqrtf(d);
    }
    __syncthreads();
    const float inv = 1.f / S[j * kBlkLd + j];
    for (int i = j + 1 + threadIdx.x; i < n; i += blockDim.x) S[i * kBlkLd + j] *= inv;
    __syncthreads();
    const int m = n - j - 1;
    for (int e = threadIdx.x; e < m * m; e += blockDim.x) {
      const int i = j + 1 + e / m, k = j + 1 + e % m;
      if (k <= i) S[i * kBlkLd + k] -= S[i * kBlkLd + j] * S[k * kBlkLd + j];
    }
    __syncthreads();
  }
  for (int e = threadIdx.x; e < n * n; e += blockDim.x) {
    const int i = e / n, j = e % n;
    A[i * lda + j] = j <= i ? S[i * kBlkLd + j] : 0.f;
  }
}

// W = L^-1 for the lower n x n block L (n <= 128), by forward substitution of the
// unit vectors, one column per thread; the upper triangle of W is zeroed.
__global__ void __launch_bounds__(128) k_trinv_base(const float* L, int n, long long ldl, float* W, long long ldw) {
  extern __shared__ float S[];
  for (int e = threadIdx.x; e < n * n; e += blockDim.x) {
    const int i = e / n, j = e % n;
    S[i * kBlkLd + j] = L[i * ldl + j];
  }
  __syncthreads();
  const int j = threadIdx.x;
  if (j < n) {
    float x[kSolveBlock];
#pragma unroll 1
    for (int i = 0; i < n; ++i) {
      if (i < j) {
        x[i] = 0.f;
        continue;
      }
      float s = (i == j) ? 1.f : 0.f;
#pragma unroll 1
      for (int k = j; k < i; ++k) s -= S[i * kBlkLd + k] * x[k];
      x[i] = s / S[i * kBlkLd + i];
    }
#pragma unroll 1
    for (int i = 0; i < n; ++i) W[i * ldw + j] = x[i];
  }
}

// --------------------------------------------------------------------------
// Statistics -> centred system (fp64)
// --------------------------------------------------------------------------
__global__ void k_means(const double* sx, const double* sy, const int64_t* n, int d_in, long long n_y, double* mu_x,
                        double* mu_y, double* n_out) {
  const double nn = static_cast<double>(*n);
  const double inv = nn > 0 ? 1.0 / nn : 0.0;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < d_in + n_y;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    if (i < d_in) mu_x[i] = sx[i] * inv;
    else mu_y[i - d_in] = sy[i - d_in] * inv;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) *n_out = nn;
}

__global__ void __launch_bounds__(1024) k_trace_alpha(const double* G, const double* mu_x, const double* n, int d_in,
                                                      double lam, int mode, double* alpha, double* alpha_out) {
  __shared__ double part[32];
  double s = 0.0;
  for (int i = threadIdx.x; i < d_in; i += blockDim.x)
    s += G[static_cast<size_t>(i) * d_in + i] - (*n) * mu_x[i] * mu_x[i];
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x < 32) {
    s = threadIdx.x < blockDim.x / 32 ? part[threadIdx.x] : 0.0;
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (threadIdx.x == 0) {
      const double a = mode == RF_ALPHA_TRACE ? lam * s / d_in : lam;
      *alpha = a;
      if (alpha_out) *alpha_out = a;
    }
  }
}

// H = (G + Gᵀ)/2 − n μ_x μ_xᵀ + αI, stored in fp64 and fp32.
__global__ void k_build_h(const double* G, const double* mu_x, const double* n, const double* alpha, int d_in,
                          double* H64, float* H32) {
  const long long total = static_cast<long long>(d_in) * d_in;
  for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int i = static_cast<int>(e / d_in), j = static_cast<int>(e % d_in);
    double h = 0.5 * (G[e] + G[static_cast<long long>(j) * d_in + i]) - (*n) * mu_x[i] * mu_x[j];
    if (i == j) h += *alpha;
    H64[e] = h;
    H32[e] = static_cast<float>(h);
  }
}

// Cc32[p][i][o] = C[p][i][o] − n μ_x[i] μ_p[o]
__global__ void k_centre_c(const double* C, const double* mu_x, const double* mu_y, const double* n, int d_in,
                           int d_out, long long total, float* Cc) {
  for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long per = static_cast<long long>(d_in) * d_out;
    const int p = static_cast<int>(e / per);
    const long long r = e - p * per;
    const int i = static_cast<int>(r / d_out), o = static_cast<int>(r % d_out);
    Cc[e] = static_cast<float>(C[e] - (*n) * mu_x[i] * mu_y[static_cast<long long>(p) * d_out + o]);
  }
}

// R_p[o][i] = (C_p[i][o] − n μ_x[i] μ_p[o]) − Σ_j A_p[o][j] H[j][i], fp64 products and
// sums, stored as fp32. 64 x 64 tiles, 256 threads, 4 x 4 outputs per thread.
__global__ void __launch_bounds__(256) k_resid64(int d_out, int d_in, const float* __restrict__ A,
                                                 const double* __restrict__ H, const double* __restrict__ C,
                                                 const double* __restrict__ mu_x, const double* __restrict__ mu_y,
                                                 const double* __restrict__ n, float* __restrict__ R) {
  __shared__ double As[16][65];
  __shared__ double Hs[16][64];
  const int p = blockIdx.z;
  const int o0 = blockIdx.y * 64, i0 = blockIdx.x * 64;
  const float* Ap = A + static_cast<long long>(p) * d_out * d_in;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  double acc[4][4] = {};
  for (int k0 = 0; k0 < d_in; k0 += 16) {
    for (int e = tid; e < 16 * 64; e += 256) {
      const int r = e >> 4, c = e & 15;  // A tile: rows o0+r, cols k0+c
      As[c][r] = static_cast<double>(Ap[static_cast<long long>(o0 + r) * d_in + k0 + c]);
      const int kr = e >> 6, ic = e & 63;  // H tile: rows k0+kr, cols i0+ic
      Hs[kr][ic] = H[static_cast<long long>(k0 + kr) * d_in + i0 + ic];
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      double a[4], h[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        a[q] = As[kk][ty * 4 + q];
        h[q] = Hs[kk][tx * 4 + q];
      }
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[x][y] = fma(a[x], h[y], acc[x][y]);
    }
    __syncthreads();
  }
  const double nn = *n;
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const int o = o0 + ty * 4 + x;
#pragma unroll
    for (int y = 0; y < 4; ++y) {
      const int i = i0 + tx * 4 + y;
      const double cc = C[(static_cast<long long>(p) * d_in + i) * d_out + o] -
                        nn * mu_x[i] * mu_y[static_cast<long long>(p) * d_out + o];
      R[(static_cast<long long>(p) * d_out + o) * d_in + i] = static_cast<float>(cc - acc[x][y]);
    }
  }
}

// b_p[o] = μ_p[o] − Σ_i A_p[o][i] μ_x[i] (fp64), one warp per output; also the
// optional bf16 copy of A.
__global__ void k_bias(const float* A, const double* mu_x, const double* mu_y, long long rows, int d_in, float* b) {
  const long long w = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= rows) return;
  const float* a = A + w * d_in;
  double s = 0.0;
  for (int i = lane; i < d_in; i += 32) s += static_cast<double>(a[i]) * mu_x[i];
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) b[w] = static_cast<float>(mu_y[w] - s);
}

__global__ void k_to_bf16(const float* A, long long total, __nv_bfloat16* out) {
  for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * blockDim.x)
    out[e] = __float2bfloat16_rn(A[e]);
}

// --------------------------------------------------------------------------
// Host-side drivers
// --------------------------------------------------------------------------
struct SolveCtx {
  cudaStream_t s;
  int sms;
  float* tmp;    // d_in^2 scratch for panels
  float* tmp2;   // d_in^2 scratch inside the triangular inverse
  int32_t* dev_status;
};

static rf_status sgemm(SolveCtx& c, bool ta, bool tb, int M, int N, int K, float alpha, const float* A, long long lda,
                       long long sA, const float* B, long long ldb, long long sB, float beta, float* C, long long ldc,
                       long long sC, int batch) {
  dim3 grid(N / 128, M / 128, batch);
  if (!ta && !tb) k_sgemm<false, false><<<grid, 256, 0, c.s>>>(M, N, K, alpha, A, lda, sA, B, ldb, sB, beta, C, ldc, sC);
  else if (ta && !tb) k_sgemm<true, false><<<grid, 256, 0, c.s>>>(M, N, K, alpha, A, lda, sA, B, ldb, sB, beta, C, ldc, sC);
  else if (!ta && tb) k_sgemm<false, true><<<grid, 256, 0, c.s>>>(M, N, K, alpha, A, lda, sA, B, ldb, sB, beta, C, ldc, sC);
  else k_sgemm<true, true><<<grid, 256, 0, c.s>>>(M, N, K, alpha, A, lda, sA, B, ldb, sB, beta, C, ldc, sC);
  return cuda_check(cudaGetLastError(), "k_sgemm launch");
}

static int split_point(int n) { return std::max(kSolveBlock, (n / 2) / kSolveBlock * kSolveBlock); }

// W (n x n, ld ldw) = L^-1 for the lower-triangular L (n x n, ld ldl); n % 128 == 0.
static rf_status trinv_lower(SolveCtx& c, const float* L, int n, long long ldl, float* W, long long ldw) {
  if (n <= kSolveBlock) {
    k_trinv_base<<<1, kSolveBlock, kBlkSmem, c.s>>>(L, n, ldl, W, ldw);
    return cuda_check(cudaGetLastError(), "k_trinv_base launch");
  }
  const int n1 = split_point(n), n2 = n - n1;
  rf_status st;
  if ((st = trinv_lower(c, L, n1, ldl, W, ldw)) != RF_OK) return st;
  if ((st = trinv_lower(c, L + n1 * ldl + n1, n2, ldl, W + n1 * ldw + n1, ldw)) != RF_OK) return st;
  // T = L21 W11 ;  W21 = −W22 T ;  W12 = 0
  if ((st = sgemm(c, false, false, n2, n1, n1, 1.f, L + n1 * ldl, ldl, 0, W, ldw, 0, 0.f, c.tmp2, n1, 0, 1)) != RF_OK)
    return st;
  if ((st = sgemm(c, false, false, n2, n1, n2, -1.f, W + n1 * ldw + n1, ldw, 0, c.tmp2, n1, 0, 0.f, W + n1 * ldw, ldw,
                  0, 1)) != RF_OK)
    return st;
  return cuda_check(cudaMemset2DAsync(W + n1, ldw * sizeof(float), 0, n2 * sizeof(float), n1, c.s), "zero W12");
}

// In-place lower Cholesky of the n x n matrix A (ld lda); n % 128 == 0.
static rf_status chol_lower(SolveCtx& c, float* A, int n, long long lda, float* winv) {
  if (n <= kSolveBlock) {
    k_chol_base<<<1, 256, kBlkSmem, c.s>>>(A, n, lda, c.dev_status);
    return cuda_check(cudaGetLastError(), "k_chol_base launch");
  }
  const int n1 = split_point(n), n2 = n - n1;
  rf_status st;
  if ((st = chol_lower(c, A, n1, lda, winv)) != RF_OK) return st;
  // W11 = L11^-1 ;  L21 = A21 W11ᵀ ;  A22 −= L21 L21ᵀ
  if ((st = trinv_lower(c, A, n1, lda, winv, n1)) != RF_OK) return st;
  if ((st = sgemm(c, false, true, n2, n1, n1, 1.f, A + n1 * lda, lda, 0, winv, n1, 0, 0.f, c.tmp, n1, 0, 1)) != RF_OK)
    return st;
  if ((st = cuda_check(cudaMemcpy2DAsync(A + n1 * lda, lda * sizeof(float), c.tmp, n1 * sizeof(float),
                                         n1 * sizeof(float), n2, cudaMemcpyDeviceToDevice, c.s),
                       "copy L21")) != RF_OK)
    return st;
  if ((st = sgemm(c, false, true, n2, n2, n1, -1.f, A + n1 * lda, lda, 0, A + n1 * lda, lda, 0, 1.f,
                  A + n1 * lda + n1, lda, 0, 1)) != RF_OK)
    return st;
  // zero the upper block so that later full-block products see a triangular L
  if ((st = cuda_check(cudaMemset2DAsync(A + n1, lda * sizeof(float), 0, n2 * sizeof(float), n1, c.s), "zero U12")) != RF_OK)
    return st;
  return chol_lower(c, A + n1 * lda + n1, n2, lda, winv);
}

struct SolveLayout {
  double* mu_x;
  double* mu_y;
  double* alpha;
  double* n;
  double* H64;
  float* L;
  float* Linv;
  float* Hinv;
  float* tmp;
  float* tmp2;
  float* work;  // Cc (first solve) then R (refinement), [P][d_in][d_out] floats
  size_t bytes;
};

static SolveLayout solve_layout(const rf_calib_desc* d, void* ws) {
  const int64_t di = d->d_in, dout = d->d_out, P = d->n_maps;
  Carve c(ws);
  SolveLayout l;
  l.mu_x = c.take<double>(di);
  l.mu_y = c.take<double>(std::max<int64_t>(P * dout, 1));
  l.alpha = c.take<double>(1);
  l.n = c.take<double>(1);
  l.H64 = c.take<double>(di * di);
  l.L = c.take<float>(di * di);
  l.Linv = c.take<float>(di * di);
  l.Hinv = c.take<float>(di * di);
  l.tmp = c.take<float>(di * di);
  l.tmp2 = c.take<float>(di * di);
  l.work = c.take<float>(std::max<int64_t>(P * di * dout, 1));
  l.bytes = c.bytes();
  return l;
}

static rf_status check_solve_desc(const rf_calib_desc* d) {
  if (d == nullptr) return fail(RF_ERR_INVALID_ARG, "desc is NULL");
  if (d->d_in <= 0 || d->d_out <= 0 || d->n_maps <= 0) return fail(RF_ERR_INVALID_ARG, "need d_in, d_out, n_maps > 0");
  if (d->d_in % 256 != 0 || d->d_out % 256 != 0)
    return fail(RF_ERR_SHAPE, "d_in and d_out must be multiples of 256");
  if (d->d_in > 32768 || d->n_maps > 65535) return fail(RF_ERR_SHAPE, "d_in must be <= 32768, n_maps <= 65535");
  return RF_OK;
}

static uint64_t g_chol_attr = 0, g_trinv_attr = 0;

}  // namespace rf

using namespace rf;

extern "C" size_t rf_solve_workspace_bytes(const rf_calib_desc* desc) {
  if (check_solve_desc(desc) != RF_OK) return 0;
  return solve_layout(desc, nullptr).bytes;
}

extern "C" rf_status rf_solve(const rf_calib_desc* desc, const rf_calib_stats* st, double lambda, int alpha_mode,
                              int refine_iters, float* A, float* b, rf_bf16* A_bf16, double* alpha_out,
                              int32_t* dev_status, void* workspace, size_t workspace_bytes, rf_stream_t stream) {
  clear_error();
  rf_status s = check_solve_desc(desc);
  if (s != RF_OK) return s;
  if (alpha_mode != RF_ALPHA_TRACE && alpha_mode != RF_ALPHA_ABSOLUTE)
    return fail(RF_ERR_INVALID_ARG, "alpha_mode must be RF_ALPHA_TRACE or RF_ALPHA_ABSOLUTE");
  if (!(lambda >= 0.0) || refine_iters < 0 || refine_iters > 8)
    return fail(RF_ERR_INVALID_ARG, "need lambda >= 0 and 0 <= refine_iters <= 8");
  if (st == nullptr || !st->G || !st->C || !st->sx || !st->sy || !st->n)
    return fail(RF_ERR_INVALID_ARG, "all statistics pointers must be non-NULL");
  if (!A || !b) return fail(RF_ERR_INVALID_ARG, "A and b must be non-NULL");
  if (!aligned16(A) || !aligned16(b) || (A_bf16 && !aligned16(A_bf16)))
    return fail(RF_ERR_ALIGN, "A, b and A_bf16 must be 16-byte aligned");
  SolveLayout lay = solve_layout(desc, workspace);
  if (workspace == nullptr || workspace_bytes < lay.bytes || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(RF_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned (got %zu)", lay.bytes, workspace_bytes);
  int sms = 0;
  if ((s = current_device(&sms)) != RF_OK) return s;
  if ((s = set_smem_attr(reinterpret_cast<const void*>(&k_chol_base), kBlkSmem, &g_chol_attr)) != RF_OK) return s;
  if ((s = set_smem_attr(reinterpret_cast<const void*>(&k_trinv_base), kBlkSmem, &g_trinv_attr)) != RF_OK) return s;

  const int di = static_cast<int>(desc->d_in), dout = static_cast<int>(desc->d_out), P = static_cast<int>(desc->n_maps);
  SolveCtx c{static_cast<cudaStream_t>(stream), sms, lay.tmp, lay.tmp2, dev_status};
  ProfScope prof(c.s, RF_STAGE_SOLVE);
  const int eb = 8 * sms;
  k_means<<<eb, 256, 0, c.s>>>(st->sx, st->sy, st->n, di, static_cast<long long>(P) * dout, lay.mu_x, lay.mu_y, lay.n);
  k_trace_alpha<<<1, 1024, 0, c.s>>>(st->G, lay.mu_x, lay.n, di, lambda, alpha_mode, lay.alpha, alpha_out);
  k_build_h<<<eb, 256, 0, c.s>>>(st->G, lay.mu_x, lay.n, lay.alpha, di, lay.H64, lay.L);
  const long long ctotal = static_cast<long long>(P) * di * dout;
  k_centre_c<<<eb, 256, 0, c.s>>>(st->C, lay.mu_x, lay.mu_y, lay.n, di, dout, ctotal, lay.work);
  if ((s = cuda_check(cudaGetLastError(), "solve set-up launches")) != RF_OK) return s;

  // H = L Lᵀ ; L^-1 ; H^-1 = L^-ᵀ L^-1
  if ((s = chol_lower(c, lay.L, di, di, lay.Linv)) != RF_OK) return s;
  if ((s = trinv_lower(c, lay.L, di, di, lay.Linv, di)) != RF_OK) return s;
  if ((s = sgemm(c, true, false, di, di, di, 1.f, lay.Linv, di, 0, lay.Linv, di, 0, 0.f, lay.Hinv, di, 0, 1)) != RF_OK)
    return s;
  // A_p = Cc_pᵀ H^-1  (Cc_p stored [d_in][d_out])
  if ((s = sgemm(c, true, false, dout, di, di, 1.f, lay.work, dout, static_cast<long long>(di) * dout, lay.Hinv, di, 0,
                 0.f, A, di, static_cast<long long>(dout) * di, P)) != RF_OK)
    return s;
  for (int it = 0; it < refine_iters; ++it) {
    dim3 g(di / 64, dout / 64, P);
    k_resid64<<<g, 256, 0, c.s>>>(dout, di, A, lay.H64, st->C, lay.mu_x, lay.mu_y, lay.n, lay.work);
    if ((s = cuda_check(cudaGetLastError(), "k_resid64 launch")) != RF_OK) return s;
    if ((s = sgemm(c, false, false, dout, di, di, 1.f, lay.work, di, static_cast<long long>(dout) * di, lay.Hinv, di, 0,
                   1.f, A, di, static_cast<long long>(dout) * di, P)) != RF_OK)
      return s;
  }
  const long long rows = static_cast<long long>(P) * dout;
  k_bias<<<static_cast<unsigned>((rows * 32 + 255) / 256), 256, 0, c.s>>>(A, lay.mu_x, lay.mu_y, rows, di, b);
  if (A_bf16) k_to_bf16<<<eb, 256, 0, c.s>>>(A, rows * di, reinterpret_cast<__nv_bfloat16*>(A_bf16));
  return cuda_check(cudaGetLastError(), "solve tail launches");
}
