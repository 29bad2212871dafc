// Closed-form ridge solve (rf_solve).
//
// [RF] RidgeFill review, "Ridge map": A_l = Y_lᵀX (XᵀX + αI)^-1, b_l = μ_l − A_l μ_S
// on centred data, α = λ·tr(XᵀX)/d_in; the statistics are read only, so a new λ is
// a re-solve. [XM] per-head ridge regression uses the same closed form (α = λ).
//
// From the one-pass sums (G, C, sx, sy, n) in fp64:
//   k_means, k_trace_alpha  μ_x = sx/n, μ_p = sy_p/n, tr(Gc), α
//   k_build_h               H = Gc + αI with Gc = G − n μ_x μ_xᵀ (fp64 and fp32 copies)
//   spd_inverse (select.cu) H = L Lᵀ, L^-1 by recursive halving (products of widths
//                           that are multiples of 512, from 2,048 up, on the tensor
//                           cores, the narrower ones fp32 SIMT k_sgemm, 128-wide leaves
//                           factored and inverted in shared memory by
//                           k_chol_inv_leaf), then H^-1 = L^-ᵀ L^-1 on the tensor
//                           cores, its upper triangle mirrored
//   split3 + tc_gemm<Split3Prob>  A_p = Cc_pᵀ H^-1 for every map on the tensor
//                           cores: each fp32 operand is the sum of three bf16
//                           planes (hi + mid + lo, exact to fp32 rounding), and
//                           the six products that matter at fp32 precision
//                           (hi·hi, mid·hi, hi·mid, lo·hi, mid·mid, hi·lo) are
//                           summed over 1024-wide K chunks in TMEM, then in fp32
//                           registers across chunks and terms
//   k_centre_split_t        Cc_p = C_p − n μ_x μ_pᵀ, written transposed as the product's
//                           three bf16 planes
//   refinement (optional)   R_p = Cc_pᵀ − A_p H, fp64-accurate on the tensor cores
//                           (k_oz_digits_*: integer digit planes of 8 bits, or 7
//                           above d_in = 21845; OzakiProb: exact int32 sums per
//                           digit weight; k_oz_combine: two exact int64 halves, one
//                           fp64 rounding), then
//                           A_p += R_p H^-1 (the split product)
//   k_bias                  b_p = μ_p − A_p μ_x (compensated fp32 pairs, fp64 across
//                           lanes); k_to_bf16 the optional bf16 copy of A
#include <algorithm>
#include <cstring>

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

// W = L^-1 for the 128 x 128 SPD block A = L Lᵀ, one CTA (8 or 16 warps) per matrix b
// (A + b*sA, W + b*sW), in shared memory and blocked by 8 so that a column or row
// block costs two barriers instead of one per column:
//   factor, per 8-column block k0: one thread per row below the diagonal block
//     solves its 8 panel entries against it (multiplying by the pivots'
//     reciprocals) and also writes them to an aligned copy of the panel; then warp 0
//     applies that panel's rank-8 update to the next diagonal block (two entries a
//     lane) and factors it (every lane the whole block in registers: no shuffles on
//     the chain of pivots), while the other warps update the rows below it, two rows
//     and two columns a step, each element from two 16-byte loads of the panel copy
//     (two float4 arrays, read without bank conflicts);
//   invert, per 8-row block i0 (rows above already hold W):
//     T = L[i0 block][0:i0] W[0:i0][0:i0] with those 8 rows of L staged transposed:
//     a warp takes 32 columns and one of KQ interleaved ranges of k, all its lanes on
//     the same k, so that the staged rows are read by broadcast; meanwhile the last
//     warp inverts the diagonal block (lane c forms column c by forward
//     substitution); then one thread per column adds the KQ partial sums and forms
//     W[i0 block][c] = −W_ii T[:, c], W_ii replaces L_ii, and the next block's rows of
//     L are staged.
// The pivots' reciprocals are rsqrt with one Newton–Raphson step (relative error a
// few units of the last place). A is only read; W's upper triangle is zero. A
// non-positive pivot records RF_ERR_NOT_SPD and continues with 1.
constexpr int kLeafN = 128;
constexpr int kLeafB = 8;
template <int kWarps>
constexpr size_t leaf_smem() {  // S, the panel copy / T's KQ partials, the staged rows, W_ii, 1/L_jj
  return kBlkSmem + sizeof(float) * ((kWarps / 4) * kLeafB * kLeafN + kLeafN * kLeafB + kLeafB * kLeafB + kLeafN);
}
static_assert(kBlkSmem % 16 == 0, "the panel copy must be 16-byte aligned");

template <int kWarps>
__global__ void __launch_bounds__(32 * kWarps) k_chol_inv_leaf(const float* __restrict__ A, long long lda, long long sA,
                                                               float* __restrict__ W, long long ldw, long long sW,
                                                               int32_t* dev_status) {
  constexpr int kThreads = 32 * kWarps;
  constexpr int n = kLeafN, B = kLeafB;
  constexpr int KQ = kWarps / 4;  // ranges of k in T (4 column blocks of 32)
  static_assert(kWarps == 8 || kWarps == 16, "8 or 16 warps");
  extern __shared__ __align__(16) float S[];
  float* P = S + n * kBlkLd;    // the panel's rows as two [n] float4 arrays, entries 0-3 and 4-7
                                // (factor); T's partials [KQ][B][n] (inversion)
  float* Lt = P + KQ * B * n;   // [n][B]: Lt[k][r] = L[i0 + r][k] (inversion)
  float* Wd = Lt + n * B;       // [B][B]: the diagonal block (factor), W_ii (inversion)
  float* Dinv = Wd + B * B;     // [n] 1 / L_jj
  const float4* Plo = reinterpret_cast<const float4*>(P);
  const float4* Phi = Plo + n;
  const float4* Lt4 = reinterpret_cast<const float4*>(Lt);
  A += blockIdx.x * sA;
  W += blockIdx.x * sW;
  const int lane = threadIdx.x, warp = threadIdx.y, tid = warp * 32 + lane;
  {
    // all of a thread's 16-byte loads issued before any is stored (rows of S are 129
    // floats apart, so the stores are scalar); lda % 4 == 0
    constexpr int kLoads = n * n / 4 / kThreads;
    float4 v[kLoads];
#pragma unroll
    for (int q = 0; q < kLoads; ++q) {
      const int e = q * kThreads + tid, i = e / (n / 4), k4 = e % (n / 4);
      v[q] = *reinterpret_cast<const float4*>(A + i * lda + 4 * k4);
    }
#pragma unroll
    for (int q = 0; q < kLoads; ++q) {
      const int e = q * kThreads + tid, i = e / (n / 4), k4 = e % (n / 4);
      float* d = S + i * kBlkLd + 4 * k4;
      d[0] = v[q].x;
      d[1] = v[q].y;
      d[2] = v[q].z;
      d[3] = v[q].w;
    }
  }
  __syncthreads();
  // ---- factor
  // Warp 0 factors the diagonal block at kd. With `update` it first applies the
  // previous panel's rank-8 update to the block (lane: entries (lane/8, lane%8) and
  // (lane/8 + 4, lane%8)), which the other warps skip. Every lane then factors the
  // whole block in registers; lane r < 8 stores row r and 1/L_rr.
  auto factor_diag = [&](int kd, bool update) {
    {
      const int c = lane & 7, r0 = lane >> 3, r1 = r0 + 4;
      float v0 = S[(kd + r0) * kBlkLd + kd + c], v1 = S[(kd + r1) * kBlkLd + kd + c];
      if (update) {
        const float4 q0 = Plo[kd + c], q1 = Phi[kd + c];
        const float4 a0 = Plo[kd + r0], a1 = Phi[kd + r0];
        const float4 b0 = Plo[kd + r1], b1 = Phi[kd + r1];
        v0 -= (a0.x * q0.x + a0.y * q0.y + a0.z * q0.z + a0.w * q0.w) +
              (a1.x * q1.x + a1.y * q1.y + a1.z * q1.z + a1.w * q1.w);
        v1 -= (b0.x * q0.x + b0.y * q0.y + b0.z * q0.z + b0.w * q0.w) +
              (b1.x * q1.x + b1.y * q1.y + b1.z * q1.z + b1.w * q1.w);
      }
      Wd[r0 * B + c] = v0;
      Wd[r1 * B + c] = v1;
    }
    __syncwarp();
    float a[B][B];
#pragma unroll
    for (int r = 0; r < B; ++r)
#pragma unroll
      for (int c = 0; c <= r; ++c) a[r][c] = Wd[r * B + c];
    __syncwarp();  // Wd is rewritten by the next call only after every lane has read it
    float dinv[B];
#pragma unroll
    for (int j = 0; j < B; ++j) {
      float d = a[j][j];
      if (!(d > 0.f)) {
        if (lane == 0) record_status(dev_status, RF_ERR_NOT_SPD);
        d = 1.f;
      }
      float inv = rsqrtf(d);
      inv = inv * fmaf(-0.5f * d * inv, inv, 1.5f);  // one Newton–Raphson step for d^-1/2
      dinv[j] = inv;
      a[j][j] = d * inv;
#pragma unroll
      for (int r = j + 1; r < B; ++r) a[r][j] *= inv;
#pragma unroll
      for (int c = j + 1; c < B; ++c)
#pragma unroll
        for (int r = c; r < B; ++r) a[r][c] = fmaf(-a[r][j], a[c][j], a[r][c]);
    }
#pragma unroll
    for (int r = 0; r < B; ++r)
      if (lane == r) {
#pragma unroll
        for (int c = 0; c <= r; ++c) S[(kd + r) * kBlkLd + kd + c] = a[r][c];
        Dinv[kd + r] = dinv[r];
      }
  };
  if (warp == 0) factor_diag(0, false);
  __syncthreads();
  for (int k0 = 0; k0 < n; k0 += B) {
    // panel: row r solves x L_ddᵀ = S[r][k0..k0+7]; x into S and into the panel copy
    for (int r = k0 + B + tid; r < n; r += kThreads) {
      float x[B];
#pragma unroll
      for (int j = 0; j < B; ++j) {
        float v = S[r * kBlkLd + k0 + j];
#pragma unroll
        for (int c = 0; c < j; ++c) v = fmaf(-x[c], S[(k0 + j) * kBlkLd + k0 + c], v);
        x[j] = v * Dinv[k0 + j];
      }
#pragma unroll
      for (int j = 0; j < B; ++j) S[r * kBlkLd + k0 + j] = x[j];
      float4* pl = reinterpret_cast<float4*>(P);
      pl[r] = make_float4(x[0], x[1], x[2], x[3]);
      pl[n + r] = make_float4(x[4], x[5], x[6], x[7]);
    }
    __syncthreads();
    if (warp == 0) {
      // look-ahead: the next diagonal block, updated and factored while the other
      // warps update the rows below it
      if (k0 + B < n) factor_diag(k0 + B, true);
    } else {
      // trailing lower triangle below the next diagonal block, rank 8: rows ra and
      // rb = ra + (warps − 1) together, columns k0 + 8 .. r, two columns a step
      constexpr int WU = kWarps - 1;
      auto upd = [&](float* dst, const float4& a0, const float4& a1, const float4& q0, const float4& q1) {
        float s0 = a0.x * q0.x, s1 = a0.y * q0.y;
        s0 = fmaf(a0.z, q0.z, s0);
        s1 = fmaf(a0.w, q0.w, s1);
        s0 = fmaf(a1.x, q1.x, s0);
        s1 = fmaf(a1.y, q1.y, s1);
        s0 = fmaf(a1.z, q1.z, s0);
        s1 = fmaf(a1.w, q1.w, s1);
        *dst -= s0 + s1;
      };
      for (int ra = k0 + 2 * B + warp - 1; ra < n; ra += 2 * WU) {
        const int rb = ra + WU;
        const bool hb = rb < n;
        const int rr = hb ? rb : ra;
        const float4 a0 = Plo[ra], a1 = Phi[ra], b0 = Plo[rr], b1 = Phi[rr];
        for (int c = k0 + B + lane; c <= rr; c += 64) {
          const int c2 = c + 32;
          const bool h2 = c2 <= rr;
          const float4 q0 = Plo[c], q1 = Phi[c];
          const float4 u0 = Plo[h2 ? c2 : c], u1 = Phi[h2 ? c2 : c];
          if (c <= ra) upd(&S[ra * kBlkLd + c], a0, a1, q0, q1);
          if (hb) upd(&S[rb * kBlkLd + c], b0, b1, q0, q1);
          if (h2 && c2 <= ra) upd(&S[ra * kBlkLd + c2], a0, a1, u0, u1);
          if (h2 && hb) upd(&S[rb * kBlkLd + c2], b0, b1, u0, u1);
        }
      }
    }
    __syncthreads();
  }
  // ---- invert in place (block 0 stages nothing: T is empty there)
  for (int i0 = 0; i0 < n; i0 += B) {
    {
      // T's partial sums: column c = 32 (warp % 4) + lane, k = kb + q, kb + q + KQ, ...
      const int cb = warp & 3, q = warp >> 2, c = cb * 32 + lane, kb = cb * 32;
      if (kb < i0) {
        float acc[B];
#pragma unroll
        for (int r = 0; r < B; ++r) acc[r] = 0.f;
#pragma unroll 2
        for (int k = kb + q; k < i0; k += KQ) {
          const float w = k >= c ? S[k * kBlkLd + c] : 0.f;  // W[k][c], lower triangle
          const float4 l0 = Lt4[2 * k], l1 = Lt4[2 * k + 1];
          acc[0] = fmaf(l0.x, w, acc[0]);
          acc[1] = fmaf(l0.y, w, acc[1]);
          acc[2] = fmaf(l0.z, w, acc[2]);
          acc[3] = fmaf(l0.w, w, acc[3]);
          acc[4] = fmaf(l1.x, w, acc[4]);
          acc[5] = fmaf(l1.y, w, acc[5]);
          acc[6] = fmaf(l1.z, w, acc[6]);
          acc[7] = fmaf(l1.w, w, acc[7]);
        }
#pragma unroll
        for (int r = 0; r < B; ++r) P[(q * B + r) * n + c] = acc[r];
      }
    }
    if (warp == kWarps - 1 && lane < B) {
      const int c = lane;
      float col[B];
#pragma unroll
      for (int r = 0; r < B; ++r) {
        float v = (r == c) ? 1.f : 0.f;
#pragma unroll
        for (int k = 0; k < r; ++k)
          if (k >= c) v = fmaf(-S[(i0 + r) * kBlkLd + i0 + k], col[k], v);
        col[r] = r >= c ? v * Dinv[i0 + r] : 0.f;
      }
#pragma unroll
      for (int r = 0; r < B; ++r) Wd[r * B + c] = col[r];
    }
    __syncthreads();
    for (int c = tid; c < i0; c += kThreads) {
      float t[B];
#pragma unroll
      for (int j = 0; j < B; ++j) {
        float v = P[j * n + c];
#pragma unroll
        for (int qq = 1; qq < KQ; ++qq) v += P[(qq * B + j) * n + c];
        t[j] = v;
      }
#pragma unroll
      for (int r = 0; r < B; ++r) {
        float v = 0.f;
#pragma unroll
        for (int j = 0; j <= r; ++j) v = fmaf(Wd[r * B + j], t[j], v);
        S[(i0 + r) * kBlkLd + c] = -v;
      }
    }
    if (tid < B * B) {
      const int r = tid >> 3, c = tid & (B - 1);
      S[(i0 + r) * kBlkLd + i0 + c] = Wd[r * B + c];
    }
    // the next block's rows of L, transposed (rows i0 + 8 .. are still L)
    if (i0 + B < n)
      for (int e = tid; e < B * (i0 + B); e += kThreads) {
        const int k = e >> 3, r = e & (B - 1);
        Lt[k * B + r] = S[(i0 + B + r) * kBlkLd + k];
      }
    __syncthreads();
  }
  for (int i = warp; i < n; i += kWarps)
    for (int k = lane; k < n; k += 32) W[i * ldw + k] = k <= i ? S[i * kBlkLd + k] : 0.f;
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

// x rounded to the nearest float, ties to even (IEEE 754), from the double's bits
// with integer operations only (GB300 runs double-to-float conversions on its slow
// fp64 units; this gives the same bits for every double): the sign, the exponent rebased from 1023 to 127, and
// the 53-bit significand cut to 24 bits (or to a subnormal's width) with the
// remainder deciding the rounding; NaN stays NaN, overflow gives infinity.
__device__ __forceinline__ float f64_to_f32_rn(double x) {
  const unsigned long long b = static_cast<unsigned long long>(__double_as_longlong(x));
  const unsigned sign = static_cast<unsigned>(b >> 32) & 0x80000000u;
  const int E = static_cast<int>((b >> 52) & 0x7ff);
  const unsigned long long frac = b & ((1ull << 52) - 1);
  if (E == 0x7ff) return __uint_as_float(sign | 0x7f800000u | (frac != 0 ? 0x400000u : 0u));
  const unsigned long long M = E != 0 ? (frac | (1ull << 52)) : frac;  // x = M 2^(max(E,1) − 1075)
  const int e = (E != 0 ? E : 1) - 1023 + 127;  // the float's biased exponent if normal
  // bits of M dropped: 29 for a normal float, more below (the subnormal step 2^-149)
  const int drop = e >= 1 ? 29 : 29 + (1 - e);
  if (drop > 54) return __uint_as_float(sign);  // below half the smallest subnormal
  const unsigned long long keep = M >> drop, rem = M & ((1ull << drop) - 1), half = 1ull << (drop - 1);
  unsigned long long r = keep + ((rem > half || (rem == half && (keep & 1))) ? 1 : 0);
  // normal: r holds the implicit bit at 2^23 (r may carry to 2^24: the exponent steps
  // up); subnormal: r < 2^23 (or = 2^23: the smallest normal), exponent field 0
  unsigned bits;
  if (e >= 1) {
    int ee = e;
    if (r >> 24) {
      r >>= 1;
      ++ee;
    }
    if (ee >= 255) return __uint_as_float(sign | 0x7f800000u);
    bits = (static_cast<unsigned>(ee) << 23) | (static_cast<unsigned>(r) & 0x7fffffu);
  } else {
    bits = static_cast<unsigned>(r);  // r = 2^23 reads as the smallest normal
  }
  return __uint_as_float(sign | bits);
}

// v / 2 from the double's bits (an exponent decrement, integer operations only) for
// normal v whose half is normal; otherwise one fp64 multiply.
__device__ __forceinline__ double half_of(double v) {
  const long long bits = __double_as_longlong(v);
  const int E = static_cast<int>((bits >> 52) & 0x7ff);
  return (E > 1 && E < 2047) ? __longlong_as_double(bits - (1ll << 52)) : 0.5 * v;
}

// H = (G + Gᵀ)/2 − n μ_x μ_xᵀ + αI, stored in fp32 and (when H64 is set) fp64.
// Block (bx, by) with bx <= by takes the tile pair P = G[rows by*32.., columns
// bx*32..] and Q = G[rows bx*32.., columns by*32..] through shared memory (row-
// contiguous reads) and writes both H tiles, so every element of G is read once
// (the diagonal tiles alone: P = Q); blocks with bx > by return at once. 32 x 8
// threads. Per element one fp64 addition and one fma (GB300's fp64 rate is low):
// the row factors n μ_x[r] are formed once per tile and the halving is an
// exponent shift.
__global__ void __launch_bounds__(256) k_build_h(const double* __restrict__ G, const double* __restrict__ mu_x,
                                                 const double* __restrict__ n, const double* __restrict__ alpha,
                                                 int d_in, double* __restrict__ H64, float* __restrict__ H32) {
  const int bx = blockIdx.x, by = blockIdx.y;
  if (bx > by) return;
  __shared__ double p[32][33];  // p[j][x] = G[r0 + j][c0 + x]
  __shared__ double q[32][33];  // q[j][x] = G[c0 + j][r0 + x]
  __shared__ double ur[32], uc[32], mr[32], mc[32];
  const int c0 = bx * 32, r0 = by * 32;
  const bool diag = bx == by;
  for (int j = threadIdx.y; j < 32; j += 8) {
    p[j][threadIdx.x] = G[static_cast<size_t>(r0 + j) * d_in + c0 + threadIdx.x];
    if (!diag) q[j][threadIdx.x] = G[static_cast<size_t>(c0 + j) * d_in + r0 + threadIdx.x];
  }
  if (threadIdx.y == 0) {
    const double nn = *n, a = mu_x[r0 + threadIdx.x], b = mu_x[c0 + threadIdx.x];
    mr[threadIdx.x] = a;
    mc[threadIdx.x] = b;
    ur[threadIdx.x] = nn * a;
    uc[threadIdx.x] = nn * b;
  }
  __syncthreads();
  const double al = *alpha;
  const double (*qq)[33] = diag ? p : q;
  // H[r0 + j][c0 + x] from G[r0 + j][c0 + x] + G[c0 + x][r0 + j]
  for (int j = threadIdx.y; j < 32; j += 8) {
    const int r = r0 + j, c = c0 + threadIdx.x;
    const size_t e = static_cast<size_t>(r) * d_in + c;
    double h = fma(-ur[j], mc[threadIdx.x], half_of(p[j][threadIdx.x] + qq[threadIdx.x][j]));
    if (r == c) h += al;
    if (H64 != nullptr) H64[e] = h;
    H32[e] = f64_to_f32_rn(h);
  }
  if (diag) return;
  // H[c0 + j][r0 + x] from G[c0 + j][r0 + x] + G[r0 + x][c0 + j]
  for (int j = threadIdx.y; j < 32; j += 8) {
    const int r = c0 + j, c = r0 + threadIdx.x;
    const size_t e = static_cast<size_t>(r) * d_in + c;
    const double h = fma(-uc[j], mr[threadIdx.x], half_of(q[j][threadIdx.x] + p[threadIdx.x][j]));
    if (H64 != nullptr) H64[e] = h;
    H32[e] = f64_to_f32_rn(h);
  }
}

// Cc_p = C_p − n μ_x μ_pᵀ, transposed and split into the product's A operand:
// planes [3][P][d_out][d_in] (K-major), straight from the fp64 sums. One fp64 fma per
// element (GB300's fp64 rate is low): the row factors −n μ_x[i] are formed once per
// tile, and the rounding to fp32 is done in integers (f64_to_f32_rn). A CTA turns a
// tile of 128 i × 32 o through shared memory ([o][i], rows 16-byte aligned): 16 row
// reads of 256 bytes a thread, then 4 consecutive i of 4 rows o per thread, 8 bytes
// a plane per store. Grid (d_in/128, d_out/32, P), 32 x 8 threads; d_in % 128 == 0.
constexpr int kCentreI = 128;
__global__ void __launch_bounds__(256) k_centre_split_t(const double* __restrict__ C, const double* __restrict__ mu_x,
                                                        const double* __restrict__ mu_y, const double* __restrict__ n,
                                                        int d_in, int d_out, __nv_bfloat16* __restrict__ planes,
                                                        size_t plane) {
  __shared__ __align__(16) float t[32][kCentreI + 4];
  __shared__ double a[kCentreI];
  const int p = blockIdx.z, i0 = blockIdx.x * kCentreI, o0 = blockIdx.y * 32;
  const int tx = threadIdx.x, ty = threadIdx.y, tid = ty * 32 + tx;
  if (tid < kCentreI) a[tid] = -(*n) * mu_x[i0 + tid];
  __syncthreads();
  const double* Cp = C + static_cast<size_t>(p) * d_in * d_out;
  const double my = mu_y[static_cast<size_t>(p) * d_out + o0 + tx];
#pragma unroll 4
  for (int j = ty; j < kCentreI; j += 8)  // t[x][j] = Cc[i0 + j][o0 + x]
    t[tx][j] = f64_to_f32_rn(fma(a[j], my, Cp[static_cast<size_t>(i0 + j) * d_out + o0 + tx]));
  __syncthreads();
  __nv_bfloat16* out = planes + static_cast<size_t>(p) * d_out * d_in;
#pragma unroll
  for (int k = 0; k < 4; ++k) {  // elements (o0 + oo, i0 + 4 tx .. + 3)
    const int oo = ty + 8 * k;
    const float4 v = *reinterpret_cast<const float4*>(&t[oo][4 * tx]);
    __nv_bfloat16 h[4], m[4], l[4];
    split3(v.x, h[0], m[0], l[0]);
    split3(v.y, h[1], m[1], l[1]);
    split3(v.z, h[2], m[2], l[2]);
    split3(v.w, h[3], m[3], l[3]);
    const size_t o = static_cast<size_t>(o0 + oo) * d_in + i0 + 4 * tx;
    *reinterpret_cast<uint2*>(out + o) = *reinterpret_cast<const uint2*>(h);
    *reinterpret_cast<uint2*>(out + plane + o) = *reinterpret_cast<const uint2*>(m);
    *reinterpret_cast<uint2*>(out + 2 * plane + o) = *reinterpret_cast<const uint2*>(l);
  }
}

// μ_x as an unevaluated pair of floats, hi + lo (|lo| <= 2^-24 |hi|), for k_bias.
__global__ void k_split_mu(const double* __restrict__ mu_x, int d_in, float2* __restrict__ mu2) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= d_in) return;
  const float hi = static_cast<float>(mu_x[i]);
  mu2[i] = make_float2(hi, static_cast<float>(mu_x[i] - static_cast<double>(hi)));
}

// b_p[o] = μ_p[o] − Σ_i A_p[o][i] μ_x[i], one warp per output. Each lane sums in
// fp32 pairs (hi, lo) with error-free products (fma) and sums (Knuth's two-sum),
// about 2^-44 of Σ|A||μ|; the lanes combine in fp64.
__global__ void k_bias(const float* __restrict__ A, const float2* __restrict__ mu2, const double* __restrict__ mu_y,
                       long long rows, int d_in, float* __restrict__ b) {
  const long long w = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= rows) return;
  const float* a = A + w * d_in;
  float hi = 0.f, lo = 0.f;
  for (int i = lane; i < d_in; i += 32) {
    const float x = a[i];
    const float2 m = mu2[i];
    // (the _rn intrinsics keep the compiler from fusing these into fma's)
    const float p = __fmul_rn(x, m.x);
    const float pe = fmaf(x, m.x, -p) + x * m.y;  // the product's error and the low part
    const float t = __fadd_rn(hi, p);
    const float bb = __fsub_rn(t, hi);
    lo += __fadd_rn(__fsub_rn(hi, __fsub_rn(t, bb)), __fsub_rn(p, bb)) + pe;  // two-sum error of hi + p
    hi = t;
  }
  double s = static_cast<double>(hi) + static_cast<double>(lo);
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) b[w] = static_cast<float>(mu_y[w] - s);
}

// bf16 copy of A, four elements a thread (total % 4 == 0, 16-byte aligned).
// a[i] += b[i], 16 bytes per step.
__global__ void __launch_bounds__(256) k_add_f32(float4* __restrict__ a, const float4* __restrict__ b, long long n4) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    float4 x = a[i];
    const float4 y = b[i];
    x.x += y.x;
    x.y += y.y;
    x.z += y.z;
    x.w += y.w;
    a[i] = x;
  }
}

__global__ void k_to_bf16(const float* __restrict__ A, long long total, __nv_bfloat16* __restrict__ out) {
  for (long long e = 4 * (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x); e < total;
       e += 4 * static_cast<long long>(gridDim.x) * blockDim.x) {
    const float4 v = *reinterpret_cast<const float4*>(A + e);
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 w;
    memcpy(&w.x, &lo, 4);
    memcpy(&w.y, &hi, 4);
    *reinterpret_cast<uint2*>(out + e) = w;
  }
}

// --------------------------------------------------------------------------
// Host-side drivers
// --------------------------------------------------------------------------
struct SolveCtx {
  cudaStream_t s;
  int sms;
  int32_t* dev_status;
};

// The same product on 64 x 64 x 16 tiles (4 x 4 outputs per thread), for products too
// small to fill the GPU with 128 x 128 tiles (the single matrix's narrow levels):
// four times the CTAs, a quarter of the serial work in each. Every output sums k in
// the same ascending order as k_sgemm, so the results are the same bit for bit (the
// `tri` ranges, now in steps of 64, skip only more zero terms). M % 64 == 0,
// N % 64 == 0, K % 16 == 0.
template <bool TA, bool TB>
__global__ void __launch_bounds__(256) k_sgemm64(int M, int N, int K, float alpha, const float* __restrict__ A,
                                                 long long lda, long long sA, const float* __restrict__ B,
                                                 long long ldb, long long sB, float beta, float* C, long long ldc,
                                                 long long sC, int tri) {
  __shared__ __align__(16) float As[2][16][64];
  __shared__ __align__(16) float Bs[2][16][64];
  const int tid = threadIdx.x;
  const int bm = blockIdx.y * 64, bn = blockIdx.x * 64;
  if ((tri & kSgemmLowerOut) && bn > bm) return;
  const int kbeg = (tri & kSgemmKFromN) ? bn : 0;
  int kend = K;
  if (tri & kSgemmKToN) kend = min(kend, bn + 64);
  if (tri & kSgemmKToM) kend = min(kend, bm + 64);
  A += blockIdx.z * sA;
  B += blockIdx.z * sB;
  C += blockIdx.z * sC;
  const int ty = tid >> 4, tx = tid & 15;

  auto load_a = [&](int k0, float4& r) {
    if (TA) r = *reinterpret_cast<const float4*>(A + static_cast<long long>(k0 + (tid >> 4)) * lda + bm + (tid & 15) * 4);
    else r = *reinterpret_cast<const float4*>(A + static_cast<long long>(bm + (tid >> 2)) * lda + k0 + (tid & 3) * 4);
  };
  auto load_b = [&](int k0, float4& r) {
    if (TB) r = *reinterpret_cast<const float4*>(B + static_cast<long long>(bn + (tid >> 2)) * ldb + k0 + (tid & 3) * 4);
    else r = *reinterpret_cast<const float4*>(B + static_cast<long long>(k0 + (tid >> 4)) * ldb + bn + (tid & 15) * 4);
  };
  auto store_a = [&](int buf, const float4& r) {
    if (TA) {
      *reinterpret_cast<float4*>(&As[buf][tid >> 4][(tid & 15) * 4]) = r;
    } else {
      const int m = tid >> 2, k = (tid & 3) * 4;
      As[buf][k][m] = r.x;
      As[buf][k + 1][m] = r.y;
      As[buf][k + 2][m] = r.z;
      As[buf][k + 3][m] = r.w;
    }
  };
  auto store_b = [&](int buf, const float4& r) {
    if (TB) {
      const int n = tid >> 2, k = (tid & 3) * 4;
      Bs[buf][k][n] = r.x;
      Bs[buf][k + 1][n] = r.y;
      Bs[buf][k + 2][n] = r.z;
      Bs[buf][k + 3][n] = r.w;
    } else {
      *reinterpret_cast<float4*>(&Bs[buf][tid >> 4][(tid & 15) * 4]) = r;
    }
  };

  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  if (kbeg < kend) {
    float4 ra, rb;
    load_a(kbeg, ra);
    load_b(kbeg, rb);
    store_a(0, ra);
    store_b(0, rb);
    __syncthreads();
    int buf = 0;
    for (int k0 = kbeg; k0 < kend; k0 += 16) {
      const bool more = k0 + 16 < kend;
      if (more) {
        load_a(k0 + 16, ra);
        load_b(k0 + 16, rb);
      }
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        const float4 a = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
        const float4 b = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
        const float av[4] = {a.x, a.y, a.z, a.w};
        const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
      }
      if (more) {
        store_a(buf ^ 1, ra);
        store_b(buf ^ 1, rb);
      }
      __syncthreads();
      buf ^= 1;
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float* cp = C + static_cast<long long>(bm + ty * 4 + i) * ldc + bn + tx * 4;
    float4 o = make_float4(alpha * acc[i][0], alpha * acc[i][1], alpha * acc[i][2], alpha * acc[i][3]);
    if (beta != 0.f) {
      const float4 cv = *reinterpret_cast<const float4*>(cp);
      o.x = fmaf(beta, cv.x, o.x);
      o.y = fmaf(beta, cv.y, o.y);
      o.z = fmaf(beta, cv.z, o.z);
      o.w = fmaf(beta, cv.w, o.w);
    }
    *reinterpret_cast<float4*>(cp) = o;
  }
}

static rf_status sgemm(SolveCtx& c, bool ta, bool tb, int M, int N, int K, float alpha, const float* A, long long lda,
                       long long sA, const float* B, long long ldb, long long sB, float beta, float* C, long long ldc,
                       long long sC, int batch, int tri = 0) {
  if (static_cast<long long>(N / 128) * (M / 128) * batch < c.sms) {
    // too few 128 x 128 tiles to fill the GPU: 64 x 64 tiles, same sums
    dim3 g64(N / 64, M / 64, batch);
    if (!ta && !tb)
      k_sgemm64<false, false><<<g64, 256, 0, c.s>>>(M, N, K, alpha, A, lda, sA, B, ldb, sB, beta, C, ldc, sC, tri);
    else if (ta && !tb)
      k_sgemm64<true, false><<<g64, 256, 0, c.s>>>(M, N, K, alpha, A, lda, sA, B, ldb, sB, beta, C, ldc, sC, tri);
    else if (!ta && tb)
      k_sgemm64<false, true><<<g64, 256, 0, c.s>>>(M, N, K, alpha, A, lda, sA, B, ldb, sB, beta, C, ldc, sC, tri);
    else
      k_sgemm64<true, true><<<g64, 256, 0, c.s>>>(M, N, K, alpha, A, lda, sA, B, ldb, sB, beta, C, ldc, sC, tri);
    return cuda_check(cudaGetLastError(), "k_sgemm64 launch");
  }
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

// --------------------------------------------------------------------------
// out_p = alpha · A_p B + beta · out_p for p < P on the tensor cores, A_p [M][K]
// and Bᵀ [N][K] given as three bf16 planes each (K-major): planes A [3][P][M][K],
// B [3][N][K]. Unit: (p, M-tile, N-tile), N fastest so an A strip is reused at
// once. Sub-tile sb = 6 c + j: product term 5 - j over the K chunk c; a chunk's terms
// chain into one TMEM accumulation, smallest first and hi·hi last, so the fp32
// accumulator's rounding is that of hi·hi's own sum, and terms beyond the planned
// count have no K-blocks. Eight epilogue warps keep fp32 running sums of their 128
// columns across the chunks and write the tile once at the end.
// --------------------------------------------------------------------------
__constant__ int kTermA[6] = {0, 1, 0, 2, 1, 0};  // hi·hi, mid·hi, hi·mid, lo·hi, mid·mid, hi·lo
__constant__ int kTermB[6] = {0, 0, 1, 0, 1, 2};
constexpr int kSplitChunk = 1024;

template <bool kPair_>
struct Split3Prob {
  CUtensorMap tmA;
  CUtensorMap tmB;
  float* out;  // [P][M][N]
  const int* n_terms;  // device: product terms to sum, the first of the six in order (nullptr: all six)
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
  __device__ bool acc_continues(int, int sb) const { return sb % 6 != 0; }
  __device__ int num_kb(int, int sb) const {
    const int c = sb / 6, t = 5 - (sb - 6 * c);
    if (n_terms != nullptr && t >= *n_terms) return 0;
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
    const int c = sb / 6, t = 5 - (sb - 6 * c);
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
      for (int q = 0; q < 32; ++q) es.rs[ch * 32 + q] = sb < 6 ? u2f(v[q]) : es.rs[ch * 32 + q] + u2f(v[q]);
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
// A_p is fp32 [P][M][K], split here, or null when planes_a already hold its planes.
static rf_status split_gemm(SolveCtx& c, const float* a, const float* Bsym, int P, int M, int N, int K, float alpha,
                            float beta, float* out, __nv_bfloat16* planes_a, __nv_bfloat16* planes_b,
                            const int* n_terms = nullptr) {
  rf_status st;
  const size_t pa = static_cast<size_t>(P) * M * K, pb = static_cast<size_t>(N) * K;
  const unsigned eb = static_cast<unsigned>(8 * c.sms);
  if (a != nullptr) k_split3<<<eb, 256, 0, c.s>>>(a, planes_a, pa / 4, pa);
  k_split3<<<eb, 256, 0, c.s>>>(Bsym, planes_b, pb / 4, pb);
  if ((st = cuda_check(cudaGetLastError(), "split launches")) != RF_OK) return st;
  Split3Prob<true> pr;
  if ((st = make_tmap_bf16_2d(&pr.tmA, planes_a, K, 3LL * P * M, K, kBK, kBM)) != RF_OK) return st;
  if ((st = make_tmap_bf16_2d(&pr.tmB, planes_b, K, 3LL * N, K, kBK, GemmCfg<true>::kBRows)) != RF_OK) return st;
  pr.out = out;
  pr.n_terms = n_terms;
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

// --------------------------------------------------------------------------
// fp64-accurate residual on the tensor cores (Ozaki-scheme splitting: Ozaki,
// Ogita, Oishi and Rump, "Error-free transformations of matrix multiplication by
// using fast routines of matrix multiplication", 2012), for the refinement
//   R_p = Cc_pᵀ − A_p H.
// Each row of A_p (fp32) and each row of H (fp64; H is symmetric, so its rows are
// its columns) is scaled by a power of two σ ≥ 2 × its largest magnitude and cut
// into integer digits of b bits: x/σ = Σ_s d_s 2^(−bs), |d_s| <= 2^(b−1), every digit
// exact in bf16 (b <= 8). A digit product summed over a K chunk of 2^(26−2b) is an
// integer of magnitude at most 2^24, exact in the fp32 accumulator; the epilogue adds
// the chunks and the digit pairs of one weight m = s + t as exact int32 sums J_m
// (|J_m| <= (m−1) 2^(2b−2) d_in) and stores them (one launch per weight). A last pass
// forms T = Σ_m J_m 2^(b(M−m)) from two exact int64 halves joined in fp64 (one
// rounding, 2^-53 of |T|) and R = Cc − σ_o τ_i 2^(−bM) T. b = 8 wherever the int32
// sums cannot overflow (d_in <= 21845), else 7. Of n digits, the pairs with
// s + t <= n + 1 are kept: a residual within about (n+1)/4 · 2^(−bn) of Σ|A||H| in
// the worst case (the dropped pairs of weight n + 2 and both truncations).
// --------------------------------------------------------------------------
constexpr int kOzDigits = 6;  // digits per operand at most (21 pairs, weights 2 .. 7)
constexpr int kOzMaps = 4;    // maps per residual launch (keeps the last wave of units small)

// Digit width for a contraction of length d_in: 8 bits while the largest weight's
// sum, 6 pairs of 2^14 products over d_in, stays below 2^31; else 7.
static int oz_bits(int d_in) {
  return static_cast<long long>(kOzDigits) * (1ll << 14) * d_in < (1ll << 31) ? 8 : 7;
}

// K chunk over which a digit product's sum stays within 2^24: 2^(26 − 2b).
static int oz_chunk(int bits) { return 1 << (26 - 2 * bits); }

// round(x · 2^(62 − e)) for |x| < 2^(e−1), from the bits of x with integer
// operations only: x = ±m·2^(E−1075) with m its 53-bit significand (E its biased
// exponent; a subnormal has no hidden bit and the exponent of E = 1), so the
// result is m shifted by E − 1013 − e, rounded half away from zero when the
// shift drops bits. Exact when no bit is dropped: always, unless x is below
// 2^(e−63), which lies below the digits kept anyway.
__device__ __forceinline__ long long fixed62(double x, int e) {
  const long long b = __double_as_longlong(x);
  const int E = static_cast<int>((b >> 52) & 0x7ff);
  long long m = b & ((1ll << 52) - 1);
  if (E != 0) m |= 1ll << 52;
  const int sh = (E != 0 ? E : 1) - 1013 - e;  // q = m · 2^sh; sh <= 8 since |q| < 2^61
  long long q;
  if (sh >= 0) q = m << sh;
  else if (sh > -63) q = (m + (1ll << (-sh - 1))) >> (-sh);
  else q = 0;
  return b < 0 ? -q : q;
}

// Digits kept this sweep: plan[0] is the largest digit weight n + 1 (k_refine_plan).
__device__ __forceinline__ int oz_planned_digits(const int* plan) { return max(1, min(kOzDigits, *plan - 1)); }

// The first n digits (n from the plan) of each row of an fp64 matrix [rows][cols]:
// digit d of row r at planes[(d * plane_rows + r) * cols ...] in bf16 (plane_rows >=
// rows), and the row scale σ (a power of two, 0 for a zero row). One warp per row.
// The digits come from integer arithmetic on v = x/σ as a 62-bit fixed-point integer
// q = v·2^62 (fixed62; |v| < 1/2, and a double has 53 significant bits): digit s is
// q's bits from 62 − b·s, rounded half up, and taking it out leaves the remainder
// within half a unit of that position, so |d_s| <= 2^(b−1) as in the fp32 split. (In
// fp64 arithmetic the same split took about 1 ms at d = 4,096: GB300's fp64 rate.)
__global__ void __launch_bounds__(256) k_oz_digits_f64(const double* __restrict__ X, int rows, int plane_rows, int cols,
                                                       int bits, const int* __restrict__ plan,
                                                       __nv_bfloat16* __restrict__ planes, double* __restrict__ scale) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= rows) return;
  const int nd = oz_planned_digits(plan);
  const double2* x = reinterpret_cast<const double2*>(X + static_cast<size_t>(warp) * cols);
  // the largest magnitude from the bit patterns (for non-negative doubles the integer
  // order is the numeric one), four columns a lane (cols % 128 == 0)
  long long mb = 0;
  for (int k = lane; k < cols / 4; k += 32) {
    const double2 a = x[2 * k], b = x[2 * k + 1];
    const long long m0 = max(__double_as_longlong(a.x) & 0x7fffffffffffffffll,
                             __double_as_longlong(a.y) & 0x7fffffffffffffffll);
    const long long m1 = max(__double_as_longlong(b.x) & 0x7fffffffffffffffll,
                             __double_as_longlong(b.y) & 0x7fffffffffffffffll);
    mb = max(mb, max(m0, m1));
  }
  for (int o = 16; o > 0; o >>= 1) mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, o));
  const double mx = __longlong_as_double(mb);
  int e = 0;
  if (mx > 0.0) frexp(mx, &e);  // mx = f 2^e, f in [0.5, 1): σ = 2^(e+1) >= 2 mx
  ++e;
  if (lane == 0) scale[warp] = mx > 0.0 ? ldexp(1.0, e) : 0.0;
  const size_t plane = static_cast<size_t>(plane_rows) * cols;
  for (int k = lane; k < cols / 4; k += 32) {
    const double2 a = x[2 * k], b = x[2 * k + 1];
    long long q[4] = {0, 0, 0, 0};
    if (mb > 0) {
      q[0] = fixed62(a.x, e);
      q[1] = fixed62(a.y, e);
      q[2] = fixed62(b.x, e);
      q[3] = fixed62(b.y, e);
    }
#pragma unroll
    for (int d = 0; d < kOzDigits; ++d) {
      if (d >= nd) break;
      const int sh = 62 - bits * (d + 1);
      __nv_bfloat16 r[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const long long v = (q[j] + (1ll << (sh - 1))) >> sh;  // |v| <= 2^(bits-1)
        q[j] -= v * (1ll << sh);                                // |q| <= 2^(sh-1)
        r[j] = __float2bfloat16_rn(static_cast<float>(static_cast<int>(v)));
      }
      uint2 w;
      memcpy(&w, r, sizeof(w));
      *reinterpret_cast<uint2*>(planes + d * plane + static_cast<size_t>(warp) * cols + 4 * k) = w;
    }
  }
}

// The same digits of an fp32 matrix, from fp32 arithmetic: for |v| <= 1/2, v·2^b,
// its nearest integer and their difference are all exact in fp32, so the digits are
// those of the fp64 procedure without using the (slow) fp64 units. Four columns a
// lane; cols % 128 == 0 and X 16-byte aligned.
__global__ void __launch_bounds__(256) k_oz_digits_f32(const float* __restrict__ X, int rows, int plane_rows, int cols,
                                                       int bits, const int* __restrict__ plan,
                                                       __nv_bfloat16* __restrict__ planes, double* __restrict__ scale) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= rows) return;
  const int nd = oz_planned_digits(plan);
  const float radix = static_cast<float>(1 << bits);
  const float4* x = reinterpret_cast<const float4*>(X + static_cast<size_t>(warp) * cols);
  const int c4 = cols / 4;
  float mx = 0.0f;
  for (int k = lane; k < c4; k += 32) {
    const float4 a = x[k];
    mx = fmaxf(mx, fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))));
  }
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  int e = 0;
  if (mx > 0.0f) frexpf(mx, &e);  // σ = 2^(e+1) >= 2 mx
  ++e;
  if (lane == 0) scale[warp] = mx > 0.0f ? ldexp(1.0, e) : 0.0;
  const size_t plane = static_cast<size_t>(plane_rows) * cols;
  for (int k = lane; k < c4; k += 32) {
    const float4 a = x[k];
    float v[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = mx > 0.0f ? ldexpf(v[j], -e) : 0.0f;  // |v| <= 1/2
#pragma unroll
    for (int d = 0; d < kOzDigits; ++d) {
      if (d >= nd) break;
      __nv_bfloat16 r[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float t = v[j] * radix;
        const float q = rintf(t);
        v[j] = t - q;
        r[j] = __float2bfloat16_rn(q);
      }
      uint2 w;
      memcpy(&w, r, sizeof(w));
      *reinterpret_cast<uint2*>(planes + d * plane + static_cast<size_t>(warp) * cols + 4 * k) = w;
    }
  }
}

// Exponent e of a power of two 2^e held as a normal double.
__device__ __forceinline__ int pow2_exponent(double x) {
  return static_cast<int>((static_cast<unsigned long long>(__double_as_longlong(x)) >> 52) & 0x7ff) - 1023;
}

// 2^e as a double, for -1022 <= e <= 1023.
__device__ __forceinline__ double pow2_double(int e) {
  return __longlong_as_double(static_cast<long long>(static_cast<uint64_t>(e + 1023) << 52));
}

// v · 2^e: an exponent shift (integer operations: GB300's fp64 rate is low) for normal
// v and result, else two products that round only if they must (|e| <= 2044).
__device__ __forceinline__ double scale_pow2(double v, int e) {
  const long long b = __double_as_longlong(v);
  const int E = static_cast<int>((b >> 52) & 0x7ff);
  if (E > 0 && E < 2047 && E + e > 0 && E + e < 2047) return __longlong_as_double(b + (static_cast<long long>(e) << 52));
  return v * pow2_double(e / 2) * pow2_double(e - e / 2);
}

// round(x / 2^k), ties away from zero, from the bits of the double with integer
// operations only (GB300's fp64 rate is low); saturates at ±2^62.
__device__ __forceinline__ long long to_grid(double x, int k) {
  const long long b = __double_as_longlong(x);
  const int E = static_cast<int>((b >> 52) & 0x7ff);
  long long m = b & ((1ll << 52) - 1);
  if (E != 0) m |= 1ll << 52;
  const int sh = (E != 0 ? E : 1) - 1075 - k;  // |x| / 2^k = m · 2^sh, m < 2^53
  long long q;
  if (E == 0x7ff || sh > 9) q = 1ll << 62;
  else if (sh >= 0) q = m << sh;
  else if (sh > -63) q = (m + (1ll << (-sh - 1))) >> (-sh);
  else q = 0;
  return b < 0 ? -q : q;
}

// v as fp32 (within about 2 ulp) from two 32-bit conversions of |v|.
__device__ __forceinline__ float ll_to_float(long long v) {
  const unsigned long long a = v < 0 ? 0ull - static_cast<unsigned long long>(v) : static_cast<unsigned long long>(v);
  const float f = fmaf(static_cast<float>(static_cast<unsigned>(a >> 32)), 4294967296.0f,
                       static_cast<float>(static_cast<unsigned>(a & 0xffffffffull)));
  return v < 0 ? -f : f;
}

// R_p[o][i] = Cc_p[i][o] − σ_o τ_i 2^(−bM) T[o][i] for the maps of a group, with
// Cc_p = C_p − n μ_x μ_pᵀ, M = *m_max (the largest digit weight computed, 7 at most)
// and T = Σ_{m <= M} J_m 2^(b(M−m)). The difference is taken exactly in integers on
// T's grid 2^k, k = log2(σ_o τ_i) − bM: Cc rounded to the grid (half a unit of
// 2^(−bM) σ_o τ_i, below the residual's own accuracy) minus T as an int64, then
// rounded to fp32. For an accurate A, |Cc| and |T| stay within d_in 2^(bM−2) units of
// the grid; where that passes 2^61 (8-bit digits at M = 7) the grid is 2^8 coarser
// and T's lowest weights are rounded to it. A zero row of A (σ_o = 0) has T = 0 and
// takes R = Cc directly. Only the centring (one fma per element) uses the fp64 units. C is [i][o] and R [o][i]: a CTA turns a tile of 32 o × 128 i
// through shared memory, each thread then writing 4 consecutive i of 4 rows o (int4
// sums in, float4 out). Grid (d_out/32, d_in/128, maps), 32 x 8 threads; d_in % 128 == 0.
constexpr int kCombI = 128;
__global__ void __launch_bounds__(256) k_oz_combine(const double* __restrict__ C, const double* __restrict__ mu_x,
                                                    const double* __restrict__ mu_y, const double* __restrict__ n,
                                                    const double* __restrict__ sA, const double* __restrict__ sH,
                                                    const int32_t* __restrict__ J, size_t plane, int d_in, int d_out,
                                                    int bits, const int* __restrict__ m_max, float* __restrict__ R32) {
  __shared__ __align__(16) double t[32][kCombI + 2];  // [o][i], rows 16-byte aligned
  __shared__ double u[kCombI];                         // n μ_x over the tile's i
  const int o0 = blockIdx.x * 32, i0 = blockIdx.y * kCombI, p = blockIdx.z;
  const int tx = threadIdx.x, ty = threadIdx.y, tid = ty * 32 + tx;
  const int mm = *m_max, mid = min(mm, 4);
  const int g = (bits == 8 && mm == 7) ? 8 : 0;  // grid coarsening (see above)
  if (tid < kCombI) u[tid] = *n * mu_x[i0 + tid];
  __syncthreads();
  const double* Cp = C + static_cast<size_t>(p) * d_in * d_out;
  const double my = mu_y[static_cast<size_t>(p) * d_out + o0 + tx];
#pragma unroll 4
  for (int r = ty; r < kCombI; r += 8)
    t[tx][r] = fma(-u[r], my, __ldcs(Cp + static_cast<size_t>(i0 + r) * d_out + o0 + tx));
  __syncthreads();
  int eh[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) eh[q] = pow2_exponent(sH[i0 + 4 * tx + q]);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int oo = ty + 8 * j, o = o0 + oo;
    const size_t e = (static_cast<size_t>(p) * d_out + o) * d_in + i0 + 4 * tx;
    // every planned weight's sums loaded before any is used (the weights above the
    // plan read as 0 and are skipped below)
    int4 v[kOzDigits];
#pragma unroll
    for (int w = 0; w < kOzDigits; ++w)
      v[w] = w + 2 <= mm ? __ldcs(reinterpret_cast<const int4*>(J + w * plane + e)) : make_int4(0, 0, 0, 0);
    long long T1[4] = {0, 0, 0, 0}, T2[4] = {0, 0, 0, 0};
#pragma unroll
    for (int w = 0; w < kOzDigits; ++w) {
      const int m = w + 2;
      if (m > mm) break;
      const int x[4] = {v[w].x, v[w].y, v[w].z, v[w].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (m <= mid) T1[q] = T1[q] * (1ll << bits) + x[q];
        else T2[q] = T2[q] * (1ll << bits) + x[q];
      }
    }
    const double sa = sA[static_cast<size_t>(p) * d_out + o];  // 0 for a zero row of A: then T = 0 and R = Cc
    const int ea = pow2_exponent(sa) - bits * mm + g;
    const double2 c01 = *reinterpret_cast<const double2*>(&t[oo][4 * tx]);
    const double2 c23 = *reinterpret_cast<const double2*>(&t[oo][4 * tx + 2]);
    const double cc[4] = {c01.x, c01.y, c23.x, c23.y};
    float r[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int k = ea + eh[q];  // the grid 2^k
      // T on the grid: T1 2^(b(M−mid) − g) + round(T2 / 2^g)
      const long long tg = T1[q] * (1ll << (bits * (mm - mid) - g)) + (g ? (T2[q] + (1ll << (g - 1))) >> g : T2[q]);
      const long long d = static_cast<long long>(static_cast<unsigned long long>(to_grid(cc[q], k)) -
                                                 static_cast<unsigned long long>(tg));
      r[q] = sa != 0.0 ? ldexpf(ll_to_float(d), k) : static_cast<float>(cc[q]);
    }
    __stcs(reinterpret_cast<float4*>(R32 + e), make_float4(r[0], r[1], r[2], r[3]));
  }
}

template <bool kPair_>
struct OzakiProb {
  CUtensorMap tmA;  // digits of the maps' rows: [kOzDigits * maps * d_out][d_in]
  CUtensorMap tmB;  // digits of H rows:        [kOzDigits * d_in][d_in]
  int32_t* J;        // [maps][d_out][d_in] this weight's exact sums J_m
  const int* m_max;  // device: the largest weight the refinement needs (weights above it run no unit)
  int maps, plane_maps, d_out, d_in, m_tiles, n_tiles, n_chunks;  // maps in this launch; maps per digit plane
  int chunk;  // K chunk (oz_chunk): each chunk's sum is exact in the fp32 accumulator
  int m;      // the digit weight s + t of this launch (pairs s = 1 .. m−1)
  int32_t* dev_status;
  uint64_t timeout_ns;
  static constexpr bool kAMN = false;
  static constexpr bool kBMN = false;
  static constexpr bool kPair = kPair_;
  static constexpr int kEpiWarps = 8;
  static constexpr int kCols = kBN / 2;
  struct EpiState {
    int32_t rs[kCols];
  };
  using Cfg = GemmCfg<kPair_>;

  __device__ void prefetch() const {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  __device__ int num_units() const { return m <= *m_max ? maps * m_tiles * n_tiles : 0; }
  __device__ int num_subtiles(int) const { return (m - 1) * n_chunks; }
  __device__ void decode(int u, int& p, int& mt, int& nt) const {
    nt = u % n_tiles;
    u /= n_tiles;
    mt = u % m_tiles;
    p = u / m_tiles;
  }
  __device__ int num_kb(int, int sb) const {
    const int c = sb % n_chunks;
    return (min(chunk, d_in - c * chunk) + kBK - 1) / kBK;
  }
  struct Coords {
    int a_row, b_row, k0;
  };
  __device__ Coords coords(int u, int sb, uint32_t rank) const {
    int p, mt, nt;
    decode(u, p, mt, nt);
    const int s = sb / n_chunks + 1, c = sb % n_chunks;
    const int t = m - s;
    return {((s - 1) * plane_maps + p) * d_out + mt * Cfg::kUnitM + static_cast<int>(rank) * kBM,
            (t - 1) * d_in + nt * kBN + static_cast<int>(rank) * Cfg::kBRows, c * chunk};
  }
  __device__ void issue_loads(Coords& c, int kb, uint8_t* sa, uint8_t* sb, uint32_t bar) const {
    load_operand<kBM, false, kPair>(sa, &tmA, bar, c.k0 + kb * kBK, c.a_row);
    load_operand<Cfg::kBRows, false, kPair>(sb, &tmB, bar, c.k0 + kb * kBK, c.b_row);
  }
  __device__ void epilogue(EpiState& es, int, int sb, int, uint32_t tacc, int, int, uint32_t) const {
    const bool first = sb == 0;
#pragma unroll
    for (int ch = 0; ch < kCols / 32; ++ch) {
      uint32_t v[32];
      tmem_ld32(tacc + ch * 32, v);
      tmem_wait_ld32(v);
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        const int32_t x = __float2int_rn(u2f(v[q]));  // an exact integer
        es.rs[ch * 32 + q] = first ? x : es.rs[ch * 32 + q] + x;
      }
    }
  }
  __device__ void epilogue_after(EpiState& es, int u, int sb, int nsub, int row, int col0, uint32_t rank) const {
    if (sb != nsub - 1) return;  // weight m not complete yet
    int p, mt, nt;
    decode(u, p, mt, nt);
    const size_t o = static_cast<size_t>(p) * d_out + static_cast<size_t>(mt) * Cfg::kUnitM + rank * kBM + row;
    int4* dst = reinterpret_cast<int4*>(J + o * d_in + static_cast<size_t>(nt) * kBN + col0);
#pragma unroll
    for (int q = 0; q < kCols / 4; ++q)
      dst[q] = make_int4(es.rs[4 * q], es.rs[4 * q + 1], es.rs[4 * q + 2], es.rs[4 * q + 3]);
  }
};

// --------------------------------------------------------------------------
// How much refinement arithmetic the conditioning calls for. κ(H) is estimated as
// λmax(H)·λmax(H^-1), each by power iteration (H read as fp32 from its fp64 copy,
// H^-1 in fp32). The Rayleigh quotients approach from below: after k steps from a
// start vector holding a share w of the top eigenvector, the worst spectrum (the
// rest at the ratio ρ where ρ^(2k) (1−w)/w is a few) leaves a quotient of at least
// 0.79 of its eigenvalue for k = 24, d <= 32768 and w 100 times below a random
// vector's 1/d, so twice the product of the two is above κ. A sweep's correction
// R H^-1 moves A by |R||H^-1|, so to bring A to fp32 accuracy (2^-24) the residual
// must be good to about 2^-(25 + log2 κ) of Σ|A||H|, and the correction product's
// own relative error times κ must stay well below 1. With b-bit digits and the pairs
// s + t <= n + 1 kept, n digits give (n+1)/4 · 2^(−bn): for b = 8, 2^-31.7 at n = 4,
// 2^-39.4 at n = 5, 2^-47.2 at n = 6 (all six, the most there are); for b = 7,
// 2^-27.7, 2^-34.4 and 2^-41.2. The first three split terms of the correction give
// about 2^-16, all six about 2^-24.
// --------------------------------------------------------------------------
constexpr int kPowerSteps = 24;
constexpr double kKappaMargin = 2.0;

// log2 of the inverse worst-case residual error with n digits of b bits.
__device__ __forceinline__ double oz_precision_bits(int n, int bits) {
  return static_cast<double>(bits) * n + 2.0 - log2(static_cast<double>(n + 1));
}

// x_m = a fixed ±1/sqrt(d) vector (signs from a multiplicative hash) for m = 0, 1.
__global__ void k_pow_init(float* __restrict__ x, int d) {
  const float v = rsqrtf(static_cast<float>(d));
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < 2 * d; i += gridDim.x * blockDim.x)
    x[i] = ((static_cast<unsigned>(i % d) * 2654435761u) >> 31) ? -v : v;
}

// Hf = H as fp32 (the power iteration's copy; 8 bytes a step read instead of 12).
// n % 2 == 0, both 16-byte aligned.
__global__ void __launch_bounds__(256) k_to_f32(const double2* __restrict__ H, long long n2, float2* __restrict__ Hf) {
  for (long long i = blockIdx.x * 256ll + threadIdx.x; i < n2; i += static_cast<long long>(gridDim.x) * 256) {
    const double2 v = H[i];
    Hf[i] = make_float2(static_cast<float>(v.x), static_cast<float>(v.y));
  }
}

// Sum of squares of x[0 .. d) over the CTA (d % 4 == 0, x 16-byte aligned),
// returned to every thread.
__device__ __forceinline__ double block_sumsq(const float* __restrict__ x, int d, double* red) {
  double s = 0.0;
  const float4* x4 = reinterpret_cast<const float4*>(x);
  for (int i = threadIdx.x; i < d / 4; i += blockDim.x) {
    const float4 v = x4[i];
    s += static_cast<double>(v.x) * v.x + static_cast<double>(v.y) * v.y + static_cast<double>(v.z) * v.z +
         static_cast<double>(v.w) * v.w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if ((threadIdx.x & 31) == 0) red[w] = s;
  __syncthreads();
  double t = 0.0;
  for (int k = 0; k < nw; ++k) t += red[k];
  return t;
}

// One power step on both matrices: y_m = M_m x_m / ‖x_m‖ (M_0 = H in fp32, M_1 = H^-1),
// so the next step's input needs no separate normalisation. A CTA of 8 warps takes
// 16 rows of one matrix (two a warp, summed side by side); x passes through shared
// memory in chunks of 2,048, and ‖x‖ is summed from the chunks on the way. Grid
// (d/16, 2) of 256 threads; d % 256 == 0.
constexpr int kPowRows = 16, kPowChunk = 2048;
__global__ void __launch_bounds__(256) k_pow_step(const float* __restrict__ Hf, const float* __restrict__ Hinv, int d,
                                                  const float* __restrict__ x, float* __restrict__ y) {
  __shared__ __align__(16) float xs[kPowChunk];
  __shared__ double red[8];
  const int m = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = blockIdx.x * kPowRows + 2 * warp;
  const float* xv = x + static_cast<size_t>(m) * d;
  const float* M = (m == 0 ? Hf : Hinv);
  const float4* row0 = reinterpret_cast<const float4*>(M + static_cast<size_t>(r0) * d);
  const float4* row1 = reinterpret_cast<const float4*>(M + static_cast<size_t>(r0 + 1) * d);
  double ss = 0.0;
  float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
  for (int c0 = 0; c0 < d; c0 += kPowChunk) {
    const int len = min(kPowChunk, d - c0);
    __syncthreads();  // the previous chunk is consumed
    for (int i = threadIdx.x; i < len / 4; i += 256) {
      const float4 v = reinterpret_cast<const float4*>(xv + c0)[i];
      reinterpret_cast<float4*>(xs)[i] = v;
      ss += static_cast<double>(v.x) * v.x + static_cast<double>(v.y) * v.y + static_cast<double>(v.z) * v.z +
            static_cast<double>(v.w) * v.w;
    }
    __syncthreads();
    const float4* x4 = reinterpret_cast<const float4*>(xs);
    const int base = c0 / 4;
#pragma unroll 4
    for (int c = lane; c < len / 4; c += 32) {
      const float4 p = row0[base + c], q = row1[base + c], v = x4[c];
      a0 = fmaf(p.x, v.x, fmaf(p.y, v.y, a0));
      a1 = fmaf(p.z, v.z, fmaf(p.w, v.w, a1));
      b0 = fmaf(q.x, v.x, fmaf(q.y, v.y, b0));
      b1 = fmaf(q.z, v.z, fmaf(q.w, v.w, b1));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) red[warp] = ss;
  float s0 = a0 + a1, s1 = b0 + b1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s0 += __shfl_xor_sync(0xffffffffu, s0, o);
    s1 += __shfl_xor_sync(0xffffffffu, s1, o);
  }
  __syncthreads();
  double tot = 0.0;
#pragma unroll
  for (int k = 0; k < 8; ++k) tot += red[k];
  const float inv = static_cast<float>(tot > 0.0 ? rsqrt(tot) : 0.0);
  if (lane == 0) {
    y[static_cast<size_t>(m) * d + r0] = s0 * inv;
    y[static_cast<size_t>(m) * d + r0 + 1] = s1 * inv;
  }
}

// est[m] = the Rayleigh quotient of x_m / ‖x_m‖ with y_m = M_m x_m / ‖x_m‖ (the last
// step's input and output): x_mᵀ y_m / ‖x_m‖. One CTA of 256 threads per matrix.
__global__ void __launch_bounds__(256) k_pow_est(const float* __restrict__ x, const float* __restrict__ y, int d,
                                                 float* __restrict__ est) {
  __shared__ double red[8];
  const int m = blockIdx.x;
  const float* xv = x + static_cast<size_t>(m) * d;
  const float* yv = y + static_cast<size_t>(m) * d;
  const double ss = block_sumsq(xv, d, red);
  __syncthreads();  // red is reused below
  double xy = 0.0;
  for (int i = threadIdx.x; i < d; i += blockDim.x) xy += static_cast<double>(xv[i]) * yv[i];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) xy += __shfl_xor_sync(0xffffffffu, xy, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = xy;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int k = 0; k < 8; ++k) t += red[k];
    est[m] = static_cast<float>(ss > 0.0 ? t * rsqrt(ss) : 0.0);
  }
}

// plan[0] = the largest digit weight the residual keeps (n + 1), plan[1] = the
// correction's split terms (see above). A non-finite estimate keeps everything.
__global__ void k_refine_plan(const float* __restrict__ est, int bits, int* __restrict__ plan) {
  const double prod = static_cast<double>(est[0]) * static_cast<double>(est[1]);
  const double need = 25.0 + log2(fmax(kKappaMargin * prod, 1.0));
  int n = kOzDigits;
  for (int k = 4; k < kOzDigits; ++k)
    if (oz_precision_bits(k, bits) >= need) {
      n = k;
      break;
    }
  plan[0] = n + 1;
  // the correction's band is kept where twelve steps and a margin of 4 put it
  plan[1] = 4.0 * prod <= 1024.0 ? 3 : 6;
}

static int split_point(int n) { return std::max(kSolveBlock, (n / 2) / kSolveBlock * kSolveBlock); }

struct SolveLayout {
  double* mu_x;
  double* mu_y;
  float2* mu2;  // μ_x as float pairs (the bias)
  double* alpha;
  double* n;
  double* H64;
  float* L;
  float* Linv;
  float* Hinv;
  float* tmp;   // [d_in/2][d_in/2] scratch of the factorisation
  float* work;  // R (refinement), [P][d_out][d_in] floats
  __nv_bfloat16* planes_a;  // [3][P][d_out][d_in] bf16 split of Cc_pᵀ or R_p
  __nv_bfloat16* planes_b;  // [3][d_in][d_in] bf16 split of H^-1
  __nv_bfloat16* ozH;       // [kOzDigits][d_in][d_in] digits of H's rows (refinement)
  double* sH;               // [d_in] their scales
  __nv_bfloat16* ozA;       // [kOzDigits][kOzMaps * d_out][d_in] digits of a group of maps' rows
  double* sA;               // [kOzMaps * d_out]
  int32_t* J;               // [kOzDigits][kOzMaps][d_out][d_in] their sums J_m, one plane per weight
  float* pvec;              // [2][2][d_in] power-iteration vectors (x, y; H and H^-1)
  float* est;               // [2] their Rayleigh quotients
  int* plan;                // [2] refinement plan (largest digit weight, correction terms)
  size_t bytes;
};

static SolveLayout solve_layout(const rf_calib_desc* d, void* ws) {
  const int64_t di = d->d_in, dout = d->d_out, P = d->n_maps;
  Carve c(ws);
  SolveLayout l;
  l.mu_x = c.take<double>(di);
  l.mu2 = c.take<float2>(di);
  l.mu_y = c.take<double>(std::max<int64_t>(P * dout, 1));
  l.alpha = c.take<double>(1);
  l.n = c.take<double>(1);
  l.H64 = c.take<double>(di * di);
  l.L = c.take<float>(di * di);
  l.Linv = c.take<float>(di * di);
  l.Hinv = c.take<float>(di * di);
  l.tmp = c.take<float>(di * di / 4);
  l.work = c.take<float>(std::max<int64_t>(P * di * dout, 1));
  l.planes_a = c.take<__nv_bfloat16>(3 * std::max<int64_t>(P * di * dout, 1));
  l.planes_b = c.take<__nv_bfloat16>(3 * di * di);
  l.ozH = c.take<__nv_bfloat16>(kOzDigits * di * di);
  l.sH = c.take<double>(di);
  const int64_t om = std::min<int64_t>(P, kOzMaps);
  l.ozA = c.take<__nv_bfloat16>(kOzDigits * om * dout * di);
  l.sA = c.take<double>(om * dout);
  l.J = c.take<int32_t>(kOzDigits * om * dout * di);
  l.pvec = c.take<float>(4 * di);
  l.est = c.take<float>(2);
  l.plan = c.take<int>(2);
  l.bytes = c.bytes();
  return l;
}

// R_p = Cc_pᵀ − A_p H for every map, fp64-accurate (OzakiProb), into R32 [P][d_out][d_in].
template <bool kPair>
static rf_status oz_residual(SolveCtx& c, const SolveLayout& lay, const double* C, const float* A, int P, int di,
                             int dout, int bits, float* R32) {
  // the weights above lay.plan[0] run no unit and the combine leaves them out
  using Cfg = GemmCfg<kPair>;
  rf_status st;
  const unsigned hb = static_cast<unsigned>((static_cast<long long>(di) * 32 + 255) / 256);
  const int chunk = oz_chunk(bits);
  k_oz_digits_f64<<<hb, 256, 0, c.s>>>(lay.H64, di, di, di, bits, lay.plan, lay.ozH, lay.sH);
  OzakiProb<kPair> pr;
  const int om = std::min(P, kOzMaps);
  if ((st = make_tmap_bf16_2d(&pr.tmA, lay.ozA, di, static_cast<uint64_t>(kOzDigits) * om * dout, di, kBK, kBM)) !=
      RF_OK)
    return st;
  if ((st = make_tmap_bf16_2d(&pr.tmB, lay.ozH, di, static_cast<uint64_t>(kOzDigits) * di, di, kBK, Cfg::kBRows)) !=
      RF_OK)
    return st;
  pr.d_out = dout;
  pr.d_in = di;
  pr.m_tiles = dout / Cfg::kUnitM;
  pr.n_tiles = di / kBN;
  pr.chunk = chunk;
  pr.n_chunks = (di + chunk - 1) / chunk;
  pr.m_max = lay.plan;
  pr.dev_status = c.dev_status;
  pr.timeout_ns = wait_timeout_ns();
  for (int p0 = 0; p0 < P; p0 += om) {
    const int g = std::min(om, P - p0);
    const size_t off = static_cast<size_t>(p0) * dout * di;
    // digits of the group's rows: the planes hold `om` maps per digit; a short last
    // group leaves the rest unused (its units are not launched)
    const unsigned gb = static_cast<unsigned>((static_cast<long long>(g) * dout * 32 + 255) / 256);
    k_oz_digits_f32<<<gb, 256, 0, c.s>>>(A + off, g * dout, om * dout, di, bits, lay.plan, lay.ozA, lay.sA);
    if ((st = cuda_check(cudaGetLastError(), "residual digit launch")) != RF_OK) return st;
    pr.maps = g;
    pr.plane_maps = om;
    // One launch per digit weight m, each storing its own plane of sums, so that the
    // epilogues only write (fire and forget) and never wait on a read.
    const size_t plane = static_cast<size_t>(om) * dout * di;
    for (int m = 2; m <= kOzDigits + 1; ++m) {
      pr.m = m;
      pr.J = lay.J + (m - 2) * plane;
      if ((st = launch_gemm(pr, static_cast<int64_t>(g) * pr.m_tiles * pr.n_tiles, c.sms, c.s,
                            "residual GEMM launch")) != RF_OK)
        return st;
    }
    k_oz_combine<<<dim3(dout / 32, di / kCombI, g), dim3(32, 8), 0, c.s>>>(
        C + off, lay.mu_x, lay.mu_y + static_cast<size_t>(p0) * dout, lay.n, lay.sA, lay.sH, lay.J, plane, di, dout,
        bits, lay.plan, R32 + off);
    if ((st = cuda_check(cudaGetLastError(), "residual combine launch")) != RF_OK) return st;
  }
  return RF_OK;
}

static rf_status check_solve_desc(const rf_calib_desc* d) {
  if (d == nullptr) return fail(RF_ERR_INVALID_ARG, "desc is NULL");
  if (d->d_in <= 0 || d->d_out <= 0 || d->n_maps <= 0) return fail(RF_ERR_INVALID_ARG, "need d_in, d_out, n_maps > 0");
  if (d->d_in % 256 != 0 || d->d_out % 256 != 0)
    return fail(RF_ERR_SHAPE, "d_in and d_out must be multiples of 256");
  if (d->d_in > 32768 || d->n_maps > 65535) return fail(RF_ERR_SHAPE, "d_in must be <= 32768, n_maps <= 65535");
  // (d_in <= 32768 keeps the d_in x d_in work arrays of the workspace within 32 GB.)
  return RF_OK;
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

static uint64_t g_leaf_attr = 0, g_leaf16_attr = 0;

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
    // A few leaves (the solve's single matrix) are a latency chain: 16 warps share
    // each step's work. Many (the selection's batches) keep 8, for occupancy.
    if (batch < c.sms)
      k_chol_inv_leaf<16><<<batch, dim3(32, 16), leaf_smem<16>(), c.s>>>(A, lda, sA, W, ldw, sW, c.dev_status);
    else
      k_chol_inv_leaf<8><<<batch, dim3(32, 8), leaf_smem<8>(), c.s>>>(A, lda, sA, W, ldw, sW, c.dev_status);
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
  rf_status st = set_smem_attr(reinterpret_cast<const void*>(&k_chol_inv_leaf<8>), leaf_smem<8>(), &g_leaf_attr);
  if (st != RF_OK) return st;
  if ((st = set_smem_attr(reinterpret_cast<const void*>(&k_chol_inv_leaf<16>), leaf_smem<16>(), &g_leaf16_attr)) != RF_OK)
    return st;
  SolveCtx c{s, sms, dev_status};
  return chol_inv_rec(c, A, lda, sA, W, ldw, sW, n, batch, tmp, stmp);
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

  const int di = static_cast<int>(desc->d_in), dout = static_cast<int>(desc->d_out), P = static_cast<int>(desc->n_maps);
  SolveCtx c{static_cast<cudaStream_t>(stream), sms, dev_status};
  const int eb = 8 * sms;
  {
    ProfScope pf(c.s, RF_STAGE_SOLVE);
    k_means<<<eb, 256, 0, c.s>>>(st->sx, st->sy, st->n, di, static_cast<long long>(P) * dout, lay.mu_x, lay.mu_y, lay.n);
    k_trace_alpha<<<1, 1024, 0, c.s>>>(st->G, lay.mu_x, lay.n, di, lambda, alpha_mode, lay.alpha, alpha_out);
    k_build_h<<<dim3(di / 32, di / 32), dim3(32, 8), 0, c.s>>>(st->G, lay.mu_x, lay.n, lay.alpha, di, lay.H64, lay.L);
    k_centre_split_t<<<dim3(di / kCentreI, dout / 32, P), dim3(32, 8), 0, c.s>>>(
        st->C, lay.mu_x, lay.mu_y, lay.n, di, dout, lay.planes_a, static_cast<size_t>(P) * dout * di);
    if ((s = cuda_check(cudaGetLastError(), "solve set-up launches")) != RF_OK) return s;
  }
  // H = L Lᵀ ; L^-1 ; H^-1 = L^-ᵀ L^-1  (planes_b is free until the product below)
  if ((s = spd_inverse(lay.L, di, lay.Linv, lay.Hinv, lay.tmp, lay.planes_b, use_pair(desc->flags, true), dev_status,
                       sms, c.s)) != RF_OK)
    return s;
  // A_p = Cc_pᵀ H^-1 (Cc_pᵀ's planes written by k_centre_split_t); H^-1 is exactly
  // symmetric (its lower triangle mirrors the upper), so its rows serve as the B operand.
  {
    ProfScope pp(c.s, RF_STAGE_SOLVE_PRODUCT);
    if ((s = split_gemm(c, nullptr, lay.Hinv, P, dout, di, di, 1.f, 0.f, A, lay.planes_a, lay.planes_b)) !=
        RF_OK)
      return s;
  }
  const int digit_bits = (desc->flags & RF_SOLVE_DIGITS7) ? 7 : oz_bits(di);
  if (refine_iters > 0) {
    // the refinement's precision from the conditioning (see k_refine_plan), once
    ProfScope pr(c.s, RF_STAGE_SOLVE_REFINE);
    // H in fp32 into L's storage (free once H^-1 exists), then the steps, ping-ponging
    // between the two halves of pvec
    const long long n2 = static_cast<long long>(di) * di / 2;
    k_to_f32<<<eb, 256, 0, c.s>>>(reinterpret_cast<const double2*>(lay.H64), n2, reinterpret_cast<float2*>(lay.L));
    k_pow_init<<<(2 * di + 255) / 256, 256, 0, c.s>>>(lay.pvec, di);
    float* xs = lay.pvec;
    float* ys = lay.pvec + 2 * di;
    for (int k = 0; k < kPowerSteps; ++k) {
      k_pow_step<<<dim3(di / kPowRows, 2), 256, 0, c.s>>>(lay.L, lay.Hinv, di, xs, ys);
      if (k + 1 < kPowerSteps) std::swap(xs, ys);
    }
    k_pow_est<<<2, 256, 0, c.s>>>(xs, ys, di, lay.est);
    k_refine_plan<<<1, 1, 0, c.s>>>(lay.est, digit_bits, lay.plan);
    if ((s = cuda_check(cudaGetLastError(), "refinement plan launches")) != RF_OK) return s;
  }
  for (int it = 0; it < refine_iters; ++it) {
    ProfScope pr(c.s, RF_STAGE_SOLVE_REFINE);
    s = use_pair(desc->flags, true) ? oz_residual<true>(c, lay, st->C, A, P, di, dout, digit_bits, lay.work)
                                    : oz_residual<false>(c, lay, st->C, A, P, di, dout, digit_bits, lay.work);
    if (s != RF_OK) return s;
    // ΔA = R H^-1 into the residual's own buffer (split into planes_a first, so free),
    // then A += ΔA in one coalesced pass: an in-epilogue read-modify-write of A (one
    // thread per row) held the accumulators long enough to stall the MMAs.
    if ((s = split_gemm(c, lay.work, lay.Hinv, P, dout, di, di, 1.f, 0.f, lay.work, lay.planes_a, lay.planes_b,
                        lay.plan + 1)) != RF_OK)
      return s;
    const long long n4 = static_cast<long long>(P) * dout * di / 4;
    k_add_f32<<<eb, 256, 0, c.s>>>(reinterpret_cast<float4*>(A), reinterpret_cast<const float4*>(lay.work), n4);
    if ((s = cuda_check(cudaGetLastError(), "correction add launch")) != RF_OK) return s;
  }
  const long long rows = static_cast<long long>(P) * dout;
  k_split_mu<<<(di + 255) / 256, 256, 0, c.s>>>(lay.mu_x, di, lay.mu2);
  k_bias<<<static_cast<unsigned>((rows * 32 + 255) / 256), 256, 0, c.s>>>(A, lay.mu2, lay.mu_y, rows, di, b);
  if (A_bf16) k_to_bf16<<<eb, 256, 0, c.s>>>(A, rows * di, reinterpret_cast<__nv_bfloat16*>(A_bf16));
  return cuda_check(cudaGetLastError(), "solve tail launches");
}
