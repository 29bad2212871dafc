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
//   k_sgemm                 H^-1 = L^-ᵀ L^-1 (fp32 SIMT)
//   split3 + tc_gemm<Split3Prob>  A_p = Cc_pᵀ H^-1 for every map on the tensor
//                           cores: each fp32 operand is the sum of three bf16
//                           planes (hi + mid + lo, exact to fp32 rounding), and
//                           the six products that matter at fp32 precision
//                           (hi·hi, mid·hi, hi·mid, lo·hi, mid·mid, hi·lo) are
//                           summed over 1024-wide K chunks in TMEM, then in fp32
//                           registers across chunks and terms
//   refinement (optional)   R_p = Cc_pᵀ − A_p H with fp64 products (k_resid64),
//                           A_p += R_p H^-1 (the same split tensor-core product)
//   k_bias                  b_p = μ_p − A_p μ_x (fp64 accumulation)
#include <algorithm>

#include "rf_host.h"
#include "rf_device.cuh"
#include "tc_gemm.cuh"

namespace rf {

constexpr int kSolveBlock = 128;  // diagonal block size of the recursive factorisation

// --------------------------------------------------------------------------
// fp32 GEMM, C[b] = alpha op(A[b]) op(B[b]) + beta C[b]. 128 x 128 x 8 tiles,
// 256 threads, 8 x 8 outputs per thread, double-buffered shared tiles.
// Requires M % 128 == 0, N % 128 == 0, K % 8 == 0, 16-byte aligned rows.
// op(A)[m][k] = TA ? A[k*lda + m] : A[m*lda + k]; op(B)[k][n] = TB ? B[n*ldb + k] : B[k*ldb + n].
// `tri` bits skip work that is known to be zero or unused:
//   kSgemmLowerOut  only the output tiles on or below the diagonal (bn <= bm);
//   kSgemmKFromN    op(B) is zero for k < n: an output column tile at bn sums k >= bn;
//   kSgemmKToN      op(B) is zero for k > n: it sums k < bn + 128;
//   kSgemmKToM      op(A) is zero for k > m: an output row tile at bm sums k < bm + 128.
// --------------------------------------------------------------------------
constexpr int kSgemmLowerOut = 1;
constexpr int kSgemmKFromN = 2;
constexpr int kSgemmKToN = 4;
constexpr int kSgemmKToM = 8;

template <bool TA, bool TB>
__global__ void __launch_bounds__(256) k_sgemm(int M, int N, int K, float alpha, const float* __restrict__ A,
                                               long long lda, long long sA, const float* __restrict__ B, long long ldb,
                                               long long sB, float beta, float* C, long long ldc, long long sC,
                                               int tri) {
  __shared__ __align__(16) float As[2][8][128];
  __shared__ __align__(16) float Bs[2][8][128];
  const int tid = threadIdx.x;
  const int bm = blockIdx.y * 128, bn = blockIdx.x * 128;
  if ((tri & kSgemmLowerOut) && bn > bm) return;
  const int kbeg = (tri & kSgemmKFromN) ? bn : 0;
  int kend = K;
  if (tri & kSgemmKToN) kend = min(kend, bn + 128);
  if (tri & kSgemmKToM) kend = min(kend, bm + 128);
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
  load_a(kbeg, ra);
  load_b(kbeg, rb);
  store_a(0, ra);
  store_b(0, rb);
  __syncthreads();
  int buf = 0;
  for (int k0 = kbeg; k0 < kend; k0 += 8) {
    const bool more = k0 + 8 < kend;
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
// Column by column: the pivot, the column scale, then the trailing update with
// two threads per row (no index divisions; the 129-float row pitch keeps both
// the row and the column accesses free of bank conflicts). CTA b works on the
// block at A + b * stride.
__global__ void __launch_bounds__(256) k_chol_base(float* A, int n, long long lda, long long stride,
                                                   int32_t* dev_status) {
  extern __shared__ float S[];
  A += blockIdx.x * stride;
  for (int i = threadIdx.y; i < n; i += blockDim.y)
    for (int k = threadIdx.x; k < n; k += blockDim.x) S[i * kBlkLd + k] = A[i * lda + k];
  const int tid = threadIdx.y * blockDim.x + threadIdx.x;
  const int nthr = blockDim.x * blockDim.y;
  __syncthreads();
  for (int j = 0; j < n; ++j) {
    if (tid == 0) {
      float d = S[j * kBlkLd + j];
      if (!(d > 0.f)) {
        record_status(dev_status, RF_ERR_NOT_SPD);
        d = 1.f;
      }
      S[j * kBlkLd + j] = sqrtf(d);
    }
    __syncthreads();
    const float inv = 1.f / S[j * kBlkLd + j];
    for (int i = j + 1 + tid; i < n; i += nthr) S[i * kBlkLd + j] *= inv;
    __syncthreads();
    for (int i = j + 1 + (tid >> 1); i < n; i += nthr >> 1) {
      const float lij = S[i * kBlkLd + j];
      for (int k = j + 1 + (tid & 1); k <= i; k += 2) S[i * kBlkLd + k] -= lij * S[k * kBlkLd + j];
    }
    __syncthreads();
  }
  for (int i = threadIdx.y; i < n; i += blockDim.y)
    for (int k = threadIdx.x; k < n; k += blockDim.x) A[i * lda + k] = k <= i ? S[i * kBlkLd + k] : 0.f;
}

// W = L^-1 for the 128 x 128 SPD block A = L Lᵀ, one CTA (8 warps) per matrix b
// (A + b*sA, W + b*sW), in shared memory and blocked by 8 so that a column or row
// block costs a few barriers instead of one per column:
//   factor, per 8-column block k0:  warp 0 factors the 8 x 8 diagonal block
//     (lanes own rows, warp-synchronous); one thread per row below solves its 8
//     panel entries against it; the warps apply the rank-8 update to the trailing
//     lower triangle (warp w takes rows w, w+8, ..., lanes the columns);
//   invert, per 8-row block i0 (rows above already hold W):
//     T = L[i0 block][0:i0] W[0:i0][0:i0]  (all threads), and meanwhile warp 0
//     inverts the diagonal block (lane c forms column c by forward substitution);
//     then W[i0 block][0:i0] = −W_ii T and W_ii replaces L_ii.
// A is only read; W's upper triangle is zero. A non-positive pivot records
// RF_ERR_NOT_SPD and continues with 1.
constexpr int kLeafN = 128;
constexpr int kLeafB = 8;
constexpr size_t kLeafSmem = kBlkSmem + sizeof(float) * (kLeafB * kLeafN + kLeafB * kLeafB);

__global__ void __launch_bounds__(256) k_chol_inv_leaf(const float* __restrict__ A, long long lda, long long sA,
                                                       float* __restrict__ W, long long ldw, long long sW,
                                                       int32_t* dev_status) {
  extern __shared__ float S[];
  float* Tb = S + kLeafN * kBlkLd;  // [8][128]
  float* Wd = Tb + kLeafB * kLeafN;  // [8][8]
  constexpr int n = kLeafN;
  A += blockIdx.x * sA;
  W += blockIdx.x * sW;
  const int lane = threadIdx.x, warp = threadIdx.y, tid = warp * 32 + lane;
  for (int i = warp; i < n; i += 8)
    for (int k = lane; k < n; k += 32) S[i * kBlkLd + k] = A[i * lda + k];
  __syncthreads();
  // ---- factor
  for (int k0 = 0; k0 < n; k0 += kLeafB) {
    if (warp == 0) {
      for (int j = 0; j < kLeafB; ++j) {
        float d = S[(k0 + j) * kBlkLd + k0 + j];
        if (!(d > 0.f)) {
          if (lane == 0) record_status(dev_status, RF_ERR_NOT_SPD);
          d = 1.f;
        }
        d = sqrtf(d);
        __syncwarp();
        if (lane == j) S[(k0 + j) * kBlkLd + k0 + j] = d;
        if (lane > j && lane < kLeafB) S[(k0 + lane) * kBlkLd + k0 + j] /= d;
        __syncwarp();
        if (lane > j && lane < kLeafB) {
          const float lrj = S[(k0 + lane) * kBlkLd + k0 + j];
          for (int c = j + 1; c <= lane; ++c) S[(k0 + lane) * kBlkLd + k0 + c] -= lrj * S[(k0 + c) * kBlkLd + k0 + j];
        }
        __syncwarp();
      }
    }
    __syncthreads();
    // panel: row r solves x L_ddᵀ = S[r][k0..k0+7]
    for (int r = k0 + kLeafB + tid; r < n; r += 256) {
      float x[kLeafB];
#pragma unroll
      for (int j = 0; j < kLeafB; ++j) {
        float v = S[r * kBlkLd + k0 + j];
#pragma unroll
        for (int c = 0; c < j; ++c) v = fmaf(-x[c], S[(k0 + j) * kBlkLd + k0 + c], v);
        x[j] = v / S[(k0 + j) * kBlkLd + k0 + j];
      }
#pragma unroll
      for (int j = 0; j < kLeafB; ++j) S[r * kBlkLd + k0 + j] = x[j];
    }
    __syncthreads();
    // trailing lower triangle, rank 8
    for (int r = k0 + kLeafB + warp; r < n; r += 8) {
      float a[kLeafB];
#pragma unroll
      for (int j = 0; j < kLeafB; ++j) a[j] = S[r * kBlkLd + k0 + j];
      for (int c = k0 + kLeafB + lane; c <= r; c += 32) {
        float v = S[r * kBlkLd + c];
#pragma unroll
        for (int j = 0; j < kLeafB; ++j) v = fmaf(-a[j], S[c * kBlkLd + k0 + j], v);
        S[r * kBlkLd + c] = v;
      }
    }
    __syncthreads();
  }
  // ---- invert in place
  for (int i0 = 0; i0 < n; i0 += kLeafB) {
    for (int e = tid; e < kLeafB * i0; e += 256) {
      const int r = e & (kLeafB - 1), c = e >> 3;
      float s0 = 0.f, s1 = 0.f;
      int k = c;
      for (; k + 1 < i0; k += 2) {
        s0 = fmaf(S[(i0 + r) * kBlkLd + k], S[k * kBlkLd + c], s0);
        s1 = fmaf(S[(i0 + r) * kBlkLd + k + 1], S[(k + 1) * kBlkLd + c], s1);
      }
      if (k < i0) s0 = fmaf(S[(i0 + r) * kBlkLd + k], S[k * kBlkLd + c], s0);
      Tb[r * kLeafN + c] = s0 + s1;
    }
    if (warp == 0 && lane < kLeafB) {
      const int c = lane;
      float col[kLeafB];
#pragma unroll
      for (int r = 0; r < kLeafB; ++r) {
        float v = (r == c) ? 1.f : 0.f;
#pragma unroll
        for (int k = 0; k < r; ++k)
          if (k >= c) v = fmaf(-S[(i0 + r) * kBlkLd + i0 + k], col[k], v);
        col[r] = r >= c ? v / S[(i0 + r) * kBlkLd + i0 + r] : 0.f;
      }
#pragma unroll
      for (int r = 0; r < kLeafB; ++r) Wd[r * kLeafB + c] = col[r];
    }
    __syncthreads();
    for (int e = tid; e < kLeafB * i0; e += 256) {
      const int r = e & (kLeafB - 1), c = e >> 3;
      float v = 0.f;
#pragma unroll
      for (int j = 0; j < kLeafB; ++j)
        if (j <= r) v = fmaf(Wd[r * kLeafB + j], Tb[j * kLeafN + c], v);
      S[(i0 + r) * kBlkLd + c] = -v;
    }
    if (tid < kLeafB * kLeafB) {
      const int r = tid >> 3, c = tid & (kLeafB - 1);
      S[(i0 + r) * kBlkLd + i0 + c] = Wd[r * kLeafB + c];
    }
    __syncthreads();
  }
  for (int i = warp; i < n; i += 8)
    for (int k = lane; k < n; k += 32) W[i * ldw + k] = k <= i ? S[i * kBlkLd + k] : 0.f;
}

// Diagonal blocks of one triangular inverse, inverted by one launch (one CTA each).
constexpr int kMaxLeaves = 256;
struct LeafBlocks {
  int off[kMaxLeaves];
  int size[kMaxLeaves];
};

// W = L^-1 for lower n x n diagonal blocks L (n <= 128), row by row in shared
// memory: W[i][j] = (δ_ij − Σ_{j<=k<i} L[i][k] W[k][j]) / L[i][i], thread j
// computing column j of row i once rows < i are done (four partial sums keep the
// dependent chain short); the upper triangle of W is zero. CTA b inverts the
// block at (off[b], off[b]) of size size[b], in matrix blockIdx.y (L0 + y * sL,
// W0 + y * sW).
__global__ void __launch_bounds__(128) k_trinv_base(const float* L0, long long ldl, long long sL, float* W0,
                                                    long long ldw, long long sW, const __grid_constant__ LeafBlocks lb) {
  const int off = lb.off[blockIdx.x], n = lb.size[blockIdx.x];
  const float* L = L0 + blockIdx.y * sL + static_cast<long long>(off) * ldl + off;
  float* W = W0 + blockIdx.y * sW + static_cast<long long>(off) * ldw + off;
  extern __shared__ float S[];
  float* Wi = S + kSolveBlock * kBlkLd;
  for (int i = 0; i < n; ++i)
    for (int k = threadIdx.x; k < n; k += blockDim.x) S[i * kBlkLd + k] = L[i * ldl + k];
  __syncthreads();
  const int j = threadIdx.x;
  for (int i = 0; i < n; ++i) {
    if (j < n) {
      float s = 0.f;
      if (j <= i) {
        float s0 = (i == j) ? 1.f : 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
        int k = j;
        for (; k + 3 < i; k += 4) {
          s0 = fmaf(-S[i * kBlkLd + k], Wi[k * kBlkLd + j], s0);
          s1 = fmaf(-S[i * kBlkLd + k + 1], Wi[(k + 1) * kBlkLd + j], s1);
          s2 = fmaf(-S[i * kBlkLd + k + 2], Wi[(k + 2) * kBlkLd + j], s2);
          s3 = fmaf(-S[i * kBlkLd + k + 3], Wi[(k + 3) * kBlkLd + j], s3);
        }
        for (; k < i; ++k) s0 = fmaf(-S[i * kBlkLd + k], Wi[k * kBlkLd + j], s0);
        s = ((s0 + s1) + (s2 + s3)) / S[i * kBlkLd + i];
      }
      Wi[i * kBlkLd + j] = s;
    }
    __syncthreads();
  }
  for (int i = 0; i < n; ++i)
    for (int k = threadIdx.x; k < n; k += blockDim.x) W[i * ldw + k] = Wi[i * kBlkLd + k];
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

// H = (G + Gᵀ)/2 − n μ_x μ_xᵀ + αI, stored in fp32 and (when H64 is set) fp64.
// Block (bx, by) writes rows by*32.., columns bx*32.. and reads Gᵀ's matching tile
// through shared memory, so both reads are row-contiguous. 32 x 8 threads.
__global__ void __launch_bounds__(256) k_build_h(const double* __restrict__ G, const double* __restrict__ mu_x,
                                                 const double* __restrict__ n, const double* __restrict__ alpha,
                                                 int d_in, double* __restrict__ H64, float* __restrict__ H32) {
  __shared__ double t[32][33];
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  for (int j = threadIdx.y; j < 32; j += 8)
    t[j][threadIdx.x] = G[static_cast<size_t>(c0 + j) * d_in + r0 + threadIdx.x];  // G[c0 + j][r0 + x]
  __syncthreads();
  const double nn = *n, a = *alpha;
  const int c = c0 + threadIdx.x;
  const double mc = mu_x[c];
  for (int j = threadIdx.y; j < 32; j += 8) {
    const int r = r0 + j;
    const size_t e = static_cast<size_t>(r) * d_in + c;
    double h = 0.5 * (G[e] + t[threadIdx.x][j]) - nn * mu_x[r] * mc;
    if (r == c) h += a;
    if (H64 != nullptr) H64[e] = h;
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
                       long long sC, int batch, int tri = 0) {
  dim3 grid(N / 128, M / 128, batch);
  if (!ta && !tb)
    k_sgemm<false, false><<<grid, 256, 0, c.s>>>(M, N, K, alpha, A, lda, sA, B, ldb, sB, beta, C, ldc, sC, tri);
  else if (ta && !tb)
    k_sgemm<true, false><<<grid, 256, 0, c.s>>>(M, N, K, alpha, A, lda, sA, B, ldb, sB, beta, C, ldc, sC, tri);
  else if (!ta && tb)
    k_sgemm<false, true><<<grid, 256, 0, c.s>>>(M, N, K, alpha, A, lda, sA, B, ldb, sB, beta, C, ldc, sC, tri);
  else
    k_sgemm<true, true><<<grid, 256, 0, c.s>>>(M, N, K, alpha, A, lda, sA, B, ldb, sB, beta, C, ldc, sC, tri);
  return cuda_check(cudaGetLastError(), "k_sgemm launch");
}

// --------------------------------------------------------------------------
// fp32 -> three bf16 planes: x = hi + mid + lo up to the last rounding (x - hi
// and its remainder are exact in fp32). planes[j][p][r][c] for X_p [R][Cn], or
// for X_p's transpose when `tr` (src then holds [P][Cn][R]).
// --------------------------------------------------------------------------
// Row-major copy: 4 consecutive elements per thread-step.
__global__ void __launch_bounds__(256) k_split3(const float* __restrict__ src, __nv_bfloat16* __restrict__ planes,
                                                size_t n4, size_t plane) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(src) + i);
    __nv_bfloat16 h[4], m[4], l[4];
    split3(v.x, h[0], m[0], l[0]);
    split3(v.y, h[1], m[1], l[1]);
    split3(v.z, h[2], m[2], l[2]);
    split3(v.w, h[3], m[3], l[3]);
    *reinterpret_cast<uint2*>(planes + 4 * i) = *reinterpret_cast<const uint2*>(h);
    *reinterpret_cast<uint2*>(planes + plane + 4 * i) = *reinterpret_cast<const uint2*>(m);
    *reinterpret_cast<uint2*>(planes + 2 * plane + 4 * i) = *reinterpret_cast<const uint2*>(l);
  }
}

// Transposed copy through a 32 x 32 shared tile: out rows r < R, columns c < Cn
// of matrix p read src[p][c][r]. Grid (Cn/32, R/32, P), 32 x 8 threads.
__global__ void __launch_bounds__(256) k_split3_t(const float* __restrict__ src, __nv_bfloat16* __restrict__ planes,
                                                  int R, int Cn, size_t plane) {
  __shared__ float t[32][33];
  const int p = blockIdx.z;
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  const float* s = src + static_cast<size_t>(p) * R * Cn;
  for (int j = threadIdx.y; j < 32; j += 8) t[j][threadIdx.x] = s[static_cast<size_t>(c0 + j) * R + r0 + threadIdx.x];
  __syncthreads();
  __nv_bfloat16* out = planes + static_cast<size_t>(p) * R * Cn;
  for (int j = threadIdx.y; j < 32; j += 8) {
    __nv_bfloat16 h, m, l;
    split3(t[threadIdx.x][j], h, m, l);
    const size_t o = static_cast<size_t>(r0 + j) * Cn + c0 + threadIdx.x;
    out[o] = h;
    out[plane + o] = m;
    out[2 * plane + o] = l;
  }
}

// --------------------------------------------------------------------------
// out_p = alpha · A_p B + beta · out_p for p < P on the tensor cores, A_p [M][K]
// and Bᵀ [N][K] given as three bf16 planes each (K-major): planes A [3][P][M][K],
// B [3][N][K]. Unit: (p, M-tile, N-tile), N fastest so an A strip is reused at
// once. Sub-tile sb: product term sb / n_chunks over the K chunk sb % n_chunks.
// Eight epilogue warps keep fp32 running sums of their 128 columns across all
// sub-tiles and write the tile once at the end.
// --------------------------------------------------------------------------
__constant__ int kTermA[6] = {0, 1, 0, 2, 1, 0};  // hi·hi, mid·hi, hi·mid, lo·hi, mid·mid, hi·lo
__constant__ int kTermB[6] = {0, 0, 1, 0, 1, 2};
constexpr int kSplitChunk = 1024;

template <bool kPair_>
struct Split3Prob {
  CUtensorMap tmA;
  CUtensorMap tmB;
  float* out;  // [P][M][N]
  float alpha, beta;
  int P, M, N, K, m_tiles, n_tiles, n_chunks;
  int32_t* dev_status;
  uint64_t timeout_ns;
  static constexpr bool kAMN = false;
  static constexpr bool kBMN = false;
  static constexpr bool kPair = kPair_;
  static constexpr int kEpiWarps = 8;
  static constexpr int kCols = kBN / 2;
  struct EpiState {
    float rs[kCols];
  };
  using Cfg = GemmCfg<kPair_>;

  __device__ void prefetch() const {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  __device__ int num_units() const { return P * m_tiles * n_tiles; }
  __device__ int num_subtiles(int) const { return 6 * n_chunks; }
  __device__ int num_kb(int, int sb) const {
    const int c = sb % n_chunks;
    return (min(kSplitChunk, K - c * kSplitChunk) + kBK - 1) / kBK;
  }
  __device__ void decode(int u, int& p, int& mt, int& nt) const {
    nt = u % n_tiles;
    u /= n_tiles;
    mt = u % m_tiles;
    p = u / m_tiles;
  }
  struct Coords {
    int a_row, b_row, k0;
  };
  __device__ Coords coords(int u, int sb, uint32_t rank) const {
    int p, mt, nt;
    decode(u, p, mt, nt);
    const int t = sb / n_chunks, c = sb - t * n_chunks;
    return {(kTermA[t] * P + p) * M + mt * Cfg::kUnitM + static_cast<int>(rank) * kBM,
            kTermB[t] * N + nt * kBN + static_cast<int>(rank) * Cfg::kBRows, c * kSplitChunk};
  }
  __device__ void issue_loads(Coords& c, int kb, uint8_t* sa, uint8_t* sb, uint32_t bar) const {
    load_operand<kBM, false, kPair>(sa, &tmA, bar, c.k0 + kb * kBK, c.a_row);
    load_operand<Cfg::kBRows, false, kPair>(sb, &tmB, bar, c.k0 + kb * kBK, c.b_row);
  }
  __device__ void epilogue(EpiState& es, int, int sb, int, uint32_t tacc, int, int, uint32_t) const {
#pragma unroll
    for (int ch = 0; ch < kCols / 32; ++ch) {
      uint32_t v[32];
      tmem_ld32(tacc + ch * 32, v);
      tmem_wait_ld32(v);
#pragma unroll
      for (int q = 0; q < 32; ++q) es.rs[ch * 32 + q] = sb == 0 ? u2f(v[q]) : es.rs[ch * 32 + q] + u2f(v[q]);
    }
  }
  __device__ void epilogue_after(EpiState& es, int u, int sb, int nsub, int row, int col0, uint32_t rank) const {
    if (sb != nsub - 1) return;
    int p, mt, nt;
    decode(u, p, mt, nt);
    const size_t m = static_cast<size_t>(mt) * Cfg::kUnitM + rank * kBM + row;
    float4* o = reinterpret_cast<float4*>(out + (static_cast<size_t>(p) * M + m) * N + static_cast<size_t>(nt) * kBN +
                                          col0);
#pragma unroll
    for (int q = 0; q < kCols / 4; ++q) {
      float4 v = make_float4(alpha * es.rs[4 * q], alpha * es.rs[4 * q + 1], alpha * es.rs[4 * q + 2],
                             alpha * es.rs[4 * q + 3]);
      if (beta != 0.f) {
        const float4 c = o[q];
        v.x = fmaf(beta, c.x, v.x);
        v.y = fmaf(beta, c.y, v.y);
        v.z = fmaf(beta, c.z, v.z);
        v.w = fmaf(beta, c.w, v.w);
      }
      o[q] = v;
    }
  }
};

// out_p = alpha A_p B + beta out_p with A_p [M][K] read from `a` ([P][M][K], or
// its transpose [P][K][M] when a_tr) and B [K][N] symmetric (its rows serve as
// Bᵀ), through the split planes in `planes_a` (3·P·M·K) and `planes_b` (3·N·K).
static rf_status split_gemm(SolveCtx& c, const float* a, bool a_tr, const float* Bsym, int P, int M, int N, int K,
                            float alpha, float beta, float* out, __nv_bfloat16* planes_a, __nv_bfloat16* planes_b) {
  rf_status st;
  const size_t pa = static_cast<size_t>(P) * M * K, pb = static_cast<size_t>(N) * K;
  const unsigned eb = static_cast<unsigned>(8 * c.sms);
  if (a_tr) {
    k_split3_t<<<dim3(K / 32, M / 32, P), dim3(32, 8), 0, c.s>>>(a, planes_a, M, K, pa);
  } else {
    k_split3<<<eb, 256, 0, c.s>>>(a, planes_a, pa / 4, pa);
  }
  k_split3<<<eb, 256, 0, c.s>>>(Bsym, planes_b, pb / 4, pb);
  if ((st = cuda_check(cudaGetLastError(), "split launches")) != RF_OK) return st;
  Split3Prob<true> pr;
  if ((st = make_tmap_bf16_2d(&pr.tmA, planes_a, K, 3LL * P * M, K, kBK, kBM)) != RF_OK) return st;
  if ((st = make_tmap_bf16_2d(&pr.tmB, planes_b, K, 3LL * N, K, kBK, GemmCfg<true>::kBRows)) != RF_OK) return st;
  pr.out = out;
  pr.alpha = alpha;
  pr.beta = beta;
  pr.P = P;
  pr.M = M;
  pr.N = N;
  pr.K = K;
  pr.m_tiles = M / GemmCfg<true>::kUnitM;
  pr.n_tiles = N / kBN;
  pr.n_chunks = (K + kSplitChunk - 1) / kSplitChunk;
  pr.dev_status = c.dev_status;
  pr.timeout_ns = wait_timeout_ns();
  return launch_gemm(pr, static_cast<int64_t>(P) * pr.m_tiles * pr.n_tiles, c.sms, c.s, "split GEMM launch");
}

static int split_point(int n) { return std::max(kSolveBlock, (n / 2) / kSolveBlock * kSolveBlock); }

// W (n x n, ld ldw) = L^-1 for the lower-triangular L (n x n, ld ldl); n % 128 == 0.
static void trinv_leaves(int off, int n, LeafBlocks& lb, int& count) {
  if (n <= kSolveBlock) {
    lb.off[count] = off;
    lb.size[count] = n;
    ++count;
    return;
  }
  const int n1 = split_point(n);
  trinv_leaves(off, n1, lb, count);
  trinv_leaves(off + n1, n - n1, lb, count);
}

// Combines the inverted diagonal blocks bottom-up: W21 = −W22 (L21 W11).
static rf_status trinv_combine(SolveCtx& c, const float* L, int n, long long ldl, float* W, long long ldw) {
  if (n <= kSolveBlock) return RF_OK;
  const int n1 = split_point(n), n2 = n - n1;
  rf_status st;
  if ((st = trinv_combine(c, L, n1, ldl, W, ldw)) != RF_OK) return st;
  if ((st = trinv_combine(c, L + n1 * ldl + n1, n2, ldl, W + n1 * ldw + n1, ldw)) != RF_OK) return st;
  // T = L21 W11 ;  W21 = −W22 T ;  W12 = 0
  if ((st = sgemm(c, false, false, n2, n1, n1, 1.f, L + n1 * ldl, ldl, 0, W, ldw, 0, 0.f, c.tmp2, n1, 0, 1)) != RF_OK)
    return st;
  if ((st = sgemm(c, false, false, n2, n1, n2, -1.f, W + n1 * ldw + n1, ldw, 0, c.tmp2, n1, 0, 0.f, W + n1 * ldw, ldw,
                  0, 1)) != RF_OK)
    return st;
  return cuda_check(cudaMemset2DAsync(W + n1, ldw * sizeof(float), 0, n2 * sizeof(float), n1, c.s), "zero W12");
}

// W = L^-1 for the lower n x n L: every diagonal block of the split tree in one
// launch, then the products that join them.
static rf_status trinv_lower(SolveCtx& c, const float* L, int n, long long ldl, float* W, long long ldw) {
  LeafBlocks lb;
  int count = 0;
  trinv_leaves(0, n, lb, count);
  k_trinv_base<<<count, kSolveBlock, 2 * kBlkSmem, c.s>>>(L, ldl, 0, W, ldw, 0, lb);
  rf_status st = cuda_check(cudaGetLastError(), "k_trinv_base launch");
  if (st != RF_OK) return st;
  return trinv_combine(c, L, n, ldl, W, ldw);
}

// In-place lower Cholesky of the n x n matrix A (ld lda); n % 128 == 0.
static rf_status chol_lower(SolveCtx& c, float* A, int n, long long lda, float* winv) {
  if (n <= kSolveBlock) {
    k_chol_base<<<1, dim3(32, 8), kBlkSmem, c.s>>>(A, n, lda, 0, c.dev_status);
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
  __nv_bfloat16* planes_a;  // [3][P][d_out][d_in] bf16 split of Cc_pᵀ or R_p
  __nv_bfloat16* planes_b;  // [3][d_in][d_in] bf16 split of H^-1
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
  l.planes_a = c.take<__nv_bfloat16>(3 * std::max<int64_t>(P * di * dout, 1));
  l.planes_b = c.take<__nv_bfloat16>(3 * di * di);
  l.bytes = c.bytes();
  return l;
}

static rf_status check_solve_desc(const rf_calib_desc* d) {
  if (d == nullptr) return fail(RF_ERR_INVALID_ARG, "desc is NULL");
  if (d->d_in <= 0 || d->d_out <= 0 || d->n_maps <= 0) return fail(RF_ERR_INVALID_ARG, "need d_in, d_out, n_maps > 0");
  if (d->d_in % 256 != 0 || d->d_out % 256 != 0)
    return fail(RF_ERR_SHAPE, "d_in and d_out must be multiples of 256");
  if (d->d_in > 32768 || d->n_maps > 65535) return fail(RF_ERR_SHAPE, "d_in must be <= 32768, n_maps <= 65535");
  // (d_in <= 32768 keeps the triangular inverse's leaf blocks within kMaxLeaves.)
  return RF_OK;
}

static uint64_t g_chol_attr = 0, g_trinv_attr = 0;

static rf_status solve_kernel_attrs() {
  rf_status s = set_smem_attr(reinterpret_cast<const void*>(&k_chol_base), kBlkSmem, &g_chol_attr);
  if (s != RF_OK) return s;
  return set_smem_attr(reinterpret_cast<const void*>(&k_trinv_base), 2 * kBlkSmem, &g_trinv_attr);
}

rf_status centre_system(const double* G, const double* sx, const double* sy, const int64_t* n, int d_in, long long n_y,
                        double lambda, int alpha_mode, double* mu_x, double* mu_y, double* n_out, double* alpha,
                        double* alpha_out, double* H64, float* H32, int sms, cudaStream_t s) {
  const int eb = 8 * sms;
  k_means<<<eb, 256, 0, s>>>(sx, sy, n, d_in, n_y, mu_x, mu_y, n_out);
  k_trace_alpha<<<1, 1024, 0, s>>>(G, mu_x, n_out, d_in, lambda, alpha_mode, alpha, alpha_out);
  k_build_h<<<dim3(d_in / 32, d_in / 32), dim3(32, 8), 0, s>>>(G, mu_x, n_out, alpha, d_in, H64, H32);
  return cuda_check(cudaGetLastError(), "centring launches");
}

static uint64_t g_leaf_attr = 0;

// Batched recursive factorisation: W = L^-1 of every n x n SPD matrix (n % 128 == 0),
// splitting n = n1 + n2 at a multiple of 128 near n/2:
//   W11 = L11^-1                      (recursion on A11)
//   L21 = A21 W11ᵀ                     -> tmp            (W11ᵀ is upper triangular)
//   A22 −= L21 L21ᵀ                    (tiles on and below the diagonal)
//   T = L21 W11                        -> A21's storage  (W11 lower triangular)
//   W22 = L22^-1                       (recursion on A22; it reuses tmp)
//   W21 = −W22 T                       (W22 lower triangular)
// with the 128 x 128 leaves factored and inverted in shared memory by one CTA each.
// Every product is an fp32 SIMT GEMM over the whole batch (k_sgemm, blockIdx.z).
static rf_status chol_inv_rec(SolveCtx& c, float* A, long long lda, long long sA, float* W, long long ldw,
                              long long sW, int n, int batch, float* tmp, long long stmp) {
  rf_status st;
  if (n == kLeafN) {
    k_chol_inv_leaf<<<batch, dim3(32, 8), kLeafSmem, c.s>>>(A, lda, sA, W, ldw, sW, c.dev_status);
    return cuda_check(cudaGetLastError(), "k_chol_inv_leaf launch");
  }
  const int n1 = split_point(n), n2 = n - n1;
  float* A21 = A + static_cast<long long>(n1) * lda;
  float* A22 = A21 + n1;
  float* W21 = W + static_cast<long long>(n1) * ldw;
  float* W22 = W21 + n1;
  if ((st = chol_inv_rec(c, A, lda, sA, W, ldw, sW, n1, batch, tmp, stmp)) != RF_OK) return st;
  if ((st = sgemm(c, false, true, n2, n1, n1, 1.f, A21, lda, sA, W, ldw, sW, 0.f, tmp, n1, stmp, batch,
                  kSgemmKToN)) != RF_OK)
    return st;
  if ((st = sgemm(c, false, true, n2, n2, n1, -1.f, tmp, n1, stmp, tmp, n1, stmp, 1.f, A22, lda, sA, batch,
                  kSgemmLowerOut)) != RF_OK)
    return st;
  if ((st = sgemm(c, false, false, n2, n1, n1, 1.f, tmp, n1, stmp, W, ldw, sW, 0.f, A21, lda, sA, batch,
                  kSgemmKFromN)) != RF_OK)
    return st;
  if ((st = chol_inv_rec(c, A22, lda, sA, W22, ldw, sW, n2, batch, tmp, stmp)) != RF_OK) return st;
  return sgemm(c, false, false, n2, n1, n2, -1.f, W22, ldw, sW, A21, lda, sA, 0.f, W21, ldw, sW, batch, kSgemmKToM);
}

rf_status chol_inv_block(float* A, long long lda, long long sA, float* W, long long ldw, long long sW, int n, int batch,
                         float* tmp, long long stmp, int32_t* dev_status, int sms, cudaStream_t s) {
  rf_status st = set_smem_attr(reinterpret_cast<const void*>(&k_chol_inv_leaf), kLeafSmem, &g_leaf_attr);
  if (st != RF_OK) return st;
  SolveCtx c{s, sms, nullptr, nullptr, dev_status};
  return chol_inv_rec(c, A, lda, sA, W, ldw, sW, n, batch, tmp, stmp);
}

rf_status chol_inv_batched(float* A, long long lda, long long stride, float* Linv, long long ldi, int n, int batch,
                           float* tmp, int32_t* dev_status, int sms, cudaStream_t s) {
  rf_status st = set_smem_attr(reinterpret_cast<const void*>(&k_chol_inv_leaf), kLeafSmem, &g_leaf_attr);
  if (st != RF_OK) return st;
  const long long stride_inv = static_cast<long long>(n) * ldi;
  SolveCtx c{s, sms, nullptr, nullptr, dev_status};
  if ((st = cuda_check(cudaMemsetAsync(Linv, 0, sizeof(float) * stride_inv * batch, s), "zero L^-1")) != RF_OK)
    return st;
  const long long stmp = static_cast<long long>(n) * n / 4;
  return chol_inv_rec(c, A, lda, stride, Linv, ldi, stride_inv, n, batch, tmp, stmp);
}

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
  if ((s = solve_kernel_attrs()) != RF_OK) return s;

  const int di = static_cast<int>(desc->d_in), dout = static_cast<int>(desc->d_out), P = static_cast<int>(desc->n_maps);
  SolveCtx c{static_cast<cudaStream_t>(stream), sms, lay.tmp, lay.tmp2, dev_status};
  const int eb = 8 * sms;
  {
    ProfScope pf(c.s, RF_STAGE_SOLVE);
    k_means<<<eb, 256, 0, c.s>>>(st->sx, st->sy, st->n, di, static_cast<long long>(P) * dout, lay.mu_x, lay.mu_y, lay.n);
    k_trace_alpha<<<1, 1024, 0, c.s>>>(st->G, lay.mu_x, lay.n, di, lambda, alpha_mode, lay.alpha, alpha_out);
    k_build_h<<<dim3(di / 32, di / 32), dim3(32, 8), 0, c.s>>>(st->G, lay.mu_x, lay.n, lay.alpha, di, lay.H64, lay.L);
    const long long ctotal = static_cast<long long>(P) * di * dout;
    k_centre_c<<<eb, 256, 0, c.s>>>(st->C, lay.mu_x, lay.mu_y, lay.n, di, dout, ctotal, lay.work);
    if ((s = cuda_check(cudaGetLastError(), "solve set-up launches")) != RF_OK) return s;

    // H = L Lᵀ ; L^-1 ; H^-1 = L^-ᵀ L^-1
    if ((s = chol_lower(c, lay.L, di, di, lay.Linv)) != RF_OK) return s;
    if ((s = trinv_lower(c, lay.L, di, di, lay.Linv, di)) != RF_OK) return s;
    if ((s = sgemm(c, true, false, di, di, di, 1.f, lay.Linv, di, 0, lay.Linv, di, 0, 0.f, lay.Hinv, di, 0, 1)) != RF_OK)
      return s;
  }
  // A_p = Cc_pᵀ H^-1  (Cc_p stored [d_in][d_out]); H^-1 is symmetric bit for bit
  // (both triangles come from the same products in the same order).
  {
    ProfScope pp(c.s, RF_STAGE_SOLVE_PRODUCT);
    if ((s = split_gemm(c, lay.work, true, lay.Hinv, P, dout, di, di, 1.f, 0.f, A, lay.planes_a, lay.planes_b)) !=
        RF_OK)
      return s;
  }
  for (int it = 0; it < refine_iters; ++it) {
    ProfScope pr(c.s, RF_STAGE_SOLVE_REFINE);
    dim3 g(di / 64, dout / 64, P);
    k_resid64<<<g, 256, 0, c.s>>>(dout, di, A, lay.H64, st->C, lay.mu_x, lay.mu_y, lay.n, lay.work);
    if ((s = cuda_check(cudaGetLastError(), "k_resid64 launch")) != RF_OK) return s;
    if ((s = split_gemm(c, lay.work, false, lay.Hinv, P, dout, di, di, 1.f, 1.f, A, lay.planes_a, lay.planes_b)) !=
        RF_OK)
      return s;
  }
  const long long rows = static_cast<long long>(P) * dout;
  k_bias<<<static_cast<unsigned>((rows * 32 + 255) / 256), 256, 0, c.s>>>(A, lay.mu_x, lay.mu_y, rows, di, b);
  if (A_bf16) k_to_bf16<<<eb, 256, 0, c.s>>>(A, rows * di, reinterpret_cast<__nv_bfloat16*>(A_bf16));
  return cuda_check(cudaGetLastError(), "solve tail launches");
}
