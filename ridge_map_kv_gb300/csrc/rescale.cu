// Value rescale (rf_value_scale).
//
// [RF] RidgeFill review, "Hybrid layers and two corrections", value rescale: in
// each upper layer the first c tail rows pass through the layer's value
// projection twice, once with the exact input and once with the map's
// prediction; per KV head, the mean over those rows of the ratio of the exact
// value's norm to the predicted value's norm scales the filled values (the
// scale then enters rf_fill_kv through rf_fill_desc.v_scale).
//
// Launch sequence on the caller's stream:
//   1. k_set_count       n_c = c (the map GEMM reads its row count on the device)
//   2. map_gemm         x̂ = x_S[N-T .. N-T+c) · A_pᵀ + b_p for every layer: the
//                        fill's own map GEMM (launched by fill.cu), reading the
//                        tail rows in place
//   3. k_row_sumsq       Σx² of every exact row x_exact[p][t]
//   4. tc_gemm<VNormProb> v = Wv'_p · x for the predicted and the exact rows;
//                        epilogue: r = (Σx²/d + ε)^-1/2, per-head norms r·‖v_h‖
//   5. k_value_scale     scale[p][h] = mean_t ‖v_exact‖ / ‖v_pred‖
#include <algorithm>

#include "fill_gemm.cuh"
#include "rf_host.h"

namespace rf {

__global__ void k_set_count(int32_t* p, int v) { *p = v; }

// Σ x² (fp32; bf16 squares are exact in fp32) of each of `rows` rows of length d.
__global__ void __launch_bounds__(256) k_row_sumsq(const __nv_bfloat16* __restrict__ x, long long ld, int d,
                                                  float* __restrict__ out) {
  const __nv_bfloat16* r = x + static_cast<long long>(blockIdx.x) * ld;
  float s = 0.f;
  for (int i = threadIdx.x * 8; i < d; i += blockDim.x * 8) {
    const uint4 q = *reinterpret_cast<const uint4*>(r + i);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(h[j]);
      s = fmaf(f.x, f.x, fmaf(f.y, f.y, s));
    }
  }
  __shared__ float red[8];
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) t += red[w];
    out[blockIdx.x] = t;
  }
}

// --------------------------------------------------------------------------
// V-norm GEMM: A operand = the predicted rows x̂ [P][Mc][d] (source 0) or the
// exact rows [P][c][ld_e] (source 1), B operand = the gain-folded V projection
// Wv' [P][KV][d]. Unit u: layer p, source, M-tile, N-tile (N fastest, so a row
// strip is reused at once). When KV % 256 == 128 the last N-tile reaches past the
// layer's V rows (into the next layer's, or past the end, where TMA reads zeros);
// its heads h >= H are not written.
// The epilogue writes, for every valid row and each head of the N-tile,
// norms[p][src][t][h] = r · ‖acc_h‖ with r the row's RMS scale.
// --------------------------------------------------------------------------
template <bool kPair_>
struct VNormProb {
  CUtensorMap tmP;
  CUtensorMap tmX;
  CUtensorMap tmB;
  const float* ssp;   // [P][d/256][Mc] predicted rows' Σx̂² partials
  const float* ssx;   // [P][c] exact rows' Σx²
  float* norms;       // [P][2][c][H]
  int c, Mc, d, P, KV, hd, n_ntiles, m_tiles, n_ss;
  float inv_d, eps;
  int32_t* dev_status;
  uint64_t timeout_ns;
  static constexpr bool kAMN = false;
  static constexpr bool kBMN = false;
  static constexpr bool kPair = kPair_;
  static constexpr int kEpiWarps = 4;
  struct EpiState {};
  __device__ void epilogue_after(EpiState&, int, int, int, int, int, uint32_t) const {}
  using Cfg = GemmCfg<kPair_>;

  __device__ void prefetch() const {
    tma_prefetch_desc(&tmP);
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmB);
  }
  __device__ int num_units() const { return P * 2 * m_tiles * n_ntiles; }
  __device__ int num_subtiles(int) const { return 1; }
  __device__ int num_kb(int, int) const { return d / kBK; }
  __device__ void decode(int u, int& p, int& src, int& mt, int& nt) const {
    nt = u % n_ntiles;
    u /= n_ntiles;
    mt = u % m_tiles;
    u /= m_tiles;
    src = u & 1;
    p = u >> 1;
  }
  struct Coords {
    const CUtensorMap* ta;
    int a_row, b_row;
  };
  __device__ Coords coords(int u, int, uint32_t rank) const {
    int p, src, mt, nt;
    decode(u, p, src, mt, nt);
    const int m0 = mt * Cfg::kUnitM + static_cast<int>(rank) * kBM;
    return {src == 0 ? &tmP : &tmX, src == 0 ? p * Mc + m0 : p * c + m0,
            p * KV + nt * kBN + static_cast<int>(rank) * Cfg::kBRows};
  }
  __device__ void issue_loads(Coords& co, int kb, uint8_t* sa, uint8_t* sb, uint32_t bar) const {
    load_operand<kBM, false, kPair>(sa, co.ta, bar, kb * kBK, co.a_row);
    load_operand<Cfg::kBRows, false, kPair>(sb, &tmB, bar, kb * kBK, co.b_row);
  }
  __device__ void epilogue(EpiState&, int u, int, int, uint32_t tacc, int row, int, uint32_t rank) const {
    int p, src, mt, nt;
    decode(u, p, src, mt, nt);
    const int m = mt * Cfg::kUnitM + static_cast<int>(rank) * kBM + row;
    const bool valid = m < c;
    float rs = 0.f;
    if (valid) {
      float s = 0.f;
      if (src == 0) {
        const float* sp = ssp + static_cast<size_t>(p) * n_ss * Mc + m;
        for (int j = 0; j < n_ss; ++j) s += sp[static_cast<size_t>(j) * Mc];
      } else {
        s = ssx[static_cast<size_t>(p) * c + m];
      }
      rs = rsqrtf(fmaf(s, inv_d, eps));
    }
    const int H = KV / hd;
#pragma unroll 1
    for (int hh = 0; hh < kBN / hd; ++hh) {
      float q = 0.f;
#pragma unroll 1
      for (int i0 = 0; i0 < hd; i0 += 32) {
        uint32_t v[32];
        tmem_ld32(tacc + hh * hd + i0, v);
        tmem_wait_ld32(v);
#pragma unroll
        for (int i = 0; i < 32; ++i) q = fmaf(u2f(v[i]), u2f(v[i]), q);
      }
      const int h = (nt * kBN + hh * hd) / hd;  // >= H past the V rows (KV % 256 == 128)
      if (valid && h < H) norms[((static_cast<size_t>(p) * 2 + src) * c + m) * H + h] = rs * sqrtf(q);
    }
  }
};

// scale[p][h] = mean over rows t with a nonzero predicted norm of exact / predicted
// (1 if there is none). One thread per (p, h); fp64 sum.
__global__ void k_value_scale(const float* __restrict__ norms, int P, int c, int H, float* __restrict__ scale) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= P * H) return;
  const int p = i / H, h = i - p * H;
  const float* np_ = norms + static_cast<size_t>(p) * 2 * c * H + h;
  const float* ne = np_ + static_cast<size_t>(c) * H;
  double s = 0.0;
  int k = 0;
  for (int t = 0; t < c; ++t) {
    const float a = np_[static_cast<size_t>(t) * H];
    if (a > 0.f) {
      s += static_cast<double>(ne[static_cast<size_t>(t) * H]) / static_cast<double>(a);
      ++k;
    }
  }
  scale[i] = k > 0 ? static_cast<float>(s / k) : 1.0f;
}

struct RescaleLayout {
  int32_t* n_c;
  __nv_bfloat16* xhat;
  float* ssp;
  float* ssx;
  float* norms;
  __nv_bfloat16* wv;  // gain-folded V projection [P][KV][d] (without RF_WEIGHTS_PREFOLDED)
  size_t bytes;
};

static RescaleLayout rescale_layout(const rf_fill_desc* d, int64_t c, void* ws) {
  const int64_t P = d->L - d->S, Mc = round_up(c, kFillRowAlign), H = d->n_kv_heads;
  Carve cv(ws);
  RescaleLayout l;
  l.n_c = cv.take<int32_t>(1);
  l.xhat = cv.take<__nv_bfloat16>(P * Mc * d->d);
  l.ssp = cv.take<float>(P * (d->d / kBN) * Mc);
  l.ssx = cv.take<float>(P * c);
  l.norms = cv.take<float>(P * 2 * c * H);
  l.wv = (d->flags & RF_WEIGHTS_PREFOLDED) ? nullptr : cv.take<__nv_bfloat16>(P * H * d->head_dim * d->d);
  l.bytes = cv.bytes();
  return l;
}

static rf_status check_rescale(const rf_fill_desc* d, int64_t c) {
  if (d == nullptr) return fail(RF_ERR_INVALID_ARG, "desc is NULL");
  if (d->d <= 0 || d->L <= 0 || d->S < 0 || d->S >= d->L || d->N < 0 || d->T < 0 || d->T > d->N ||
      d->n_kv_heads <= 0 || (d->head_dim != 64 && d->head_dim != 128) || !(d->rms_eps >= 0.0))
    return fail(RF_ERR_INVALID_ARG, "need d > 0, 0 <= S < L, 0 <= T <= N, H > 0, head_dim 64 or 128, rms_eps >= 0");
  if (d->d % kBN != 0) return fail(RF_ERR_SHAPE, "d = %lld must be a multiple of 256", (long long)d->d);
  if (d->d_in < 0 || d->d_in % kBN != 0 || d->d_in > (int64_t(1) << 20))
    return fail(RF_ERR_SHAPE, "d_in = %lld must be 0 (square maps) or a multiple of 256", (long long)d->d_in);
  const int64_t KV = d->n_kv_heads * d->head_dim;
  if (KV % 128 != 0) return fail(RF_ERR_SHAPE, "n_kv_heads * head_dim = %lld must be a multiple of 128", (long long)KV);
  if (c < 1 || c > d->T) return fail(RF_ERR_INVALID_ARG, "need 1 <= c <= T (c = %lld, T = %lld)", (long long)c,
                                     (long long)d->T);
  if (c > (int64_t(1) << 20)) return fail(RF_ERR_SHAPE, "c must be <= 2^20");
  const int64_t P = d->L - d->S;
  if (P * d->d >= (int64_t(1) << 31) || P * 2 * KV >= (int64_t(1) << 31) || P * round_up(c, kFillRowAlign) >= (1 << 30))
    return fail(RF_ERR_SHAPE, "too many rows");
  return RF_OK;
}

template <bool kPair>
static rf_status rescale_gemms(const rf_fill_desc* desc, int64_t c, const RescaleLayout& lay, const rf_bf16* x_tail,
                               int64_t ld_x, const rf_bf16* x_exact, int64_t ld_e, const rf_bf16* A, const float* b,
                               const void* Wv, int32_t* dev_status, int sms, cudaStream_t s) {
  using Cfg = GemmCfg<kPair>;
  rf_status st;
  const int64_t d = desc->d, P = desc->L - desc->S, KV = desc->n_kv_heads * desc->head_dim;
  const int64_t Mc = round_up(c, kFillRowAlign);
  const uint64_t tmo = wait_timeout_ns();
  {
    const int64_t d_in = desc->d_in > 0 ? desc->d_in : d;
    MapGemmArgs ma{x_tail, ld_x, c, lay.n_c, A, b, nullptr, lay.xhat, lay.ssp, d, d_in, P, Mc, dev_status};
    if ((st = map_gemm(kPair, ma, sms, s)) != RF_OK) return st;
  }
  {
    ProfScope prof(s, RF_STAGE_RESCALE);
    k_row_sumsq<<<static_cast<unsigned>(P * c), 256, 0, s>>>(reinterpret_cast<const __nv_bfloat16*>(x_exact), ld_e,
                                                              static_cast<int>(d), lay.ssx);
  }
  if ((st = cuda_check(cudaGetLastError(), "k_row_sumsq launch")) != RF_OK) return st;
  {
    VNormProb<kPair> pr;
    if ((st = make_tmap_bf16_2d(&pr.tmP, lay.xhat, d, P * Mc, d, kBK, kBM)) != RF_OK) return st;
    if ((st = make_tmap_bf16_2d(&pr.tmX, x_exact, d, P * c, ld_e, kBK, kBM)) != RF_OK) return st;
    if ((st = make_tmap_bf16_2d(&pr.tmB, Wv, d, P * KV, d, kBK, Cfg::kBRows)) != RF_OK) return st;
    pr.ssp = lay.ssp;
    pr.ssx = lay.ssx;
    pr.norms = lay.norms;
    pr.c = static_cast<int>(c);
    pr.Mc = static_cast<int>(Mc);
    pr.d = static_cast<int>(d);
    pr.P = static_cast<int>(P);
    pr.KV = static_cast<int>(KV);
    pr.hd = static_cast<int>(desc->head_dim);
    pr.n_ntiles = static_cast<int>((KV + kBN - 1) / kBN);
    pr.m_tiles = static_cast<int>((c + Cfg::kUnitM - 1) / Cfg::kUnitM);
    pr.n_ss = static_cast<int>(d / kBN);
    pr.inv_d = 1.0f / static_cast<float>(d);
    pr.eps = static_cast<float>(desc->rms_eps);
    pr.dev_status = dev_status;
    pr.timeout_ns = tmo;
    ProfScope prof(s, RF_STAGE_RESCALE);
    if ((st = launch_gemm(pr, int64_t(pr.P) * 2 * pr.m_tiles * pr.n_ntiles, sms, s, "value-norm GEMM launch")) != RF_OK)
      return st;
  }
  return RF_OK;
}

}  // namespace rf

using namespace rf;

extern "C" size_t rf_value_scale_workspace_bytes(const rf_fill_desc* desc, int64_t c) {
  if (check_rescale(desc, c) != RF_OK) return 0;
  return rescale_layout(desc, c, nullptr).bytes;
}

extern "C" rf_status rf_value_scale(const rf_fill_desc* desc, int64_t c, const rf_bf16* x_S, int64_t ld_x,
                                    const rf_bf16* x_exact, int64_t ld_e, const rf_bf16* A, const float* b,
                                    const rf_bf16* gain, const rf_bf16* Wv, float* v_scale, int32_t* dev_status,
                                    void* workspace, size_t workspace_bytes, rf_stream_t stream) {
  clear_error();
  rf_status st = check_rescale(desc, c);
  if (st != RF_OK) return st;
  const bool prefolded = (desc->flags & RF_WEIGHTS_PREFOLDED) != 0;
  if (!x_S || !x_exact || !A || !b || !Wv || !v_scale || (!prefolded && !gain))
    return fail(RF_ERR_INVALID_ARG, "x_S, x_exact, A, b, Wv, v_scale (and gain unless RF_WEIGHTS_PREFOLDED) "
                                    "must be non-NULL");
  const int64_t d = desc->d;
  const int64_t d_in = desc->d_in > 0 ? desc->d_in : d;
  if (ld_x < d_in || ld_x % 8 != 0 || ld_e < d || ld_e % 8 != 0)
    return fail(RF_ERR_ALIGN, "ld_x must be >= d_in, ld_e >= d, both multiples of 8");
  const rf_bf16* x_tail = reinterpret_cast<const rf_bf16*>(reinterpret_cast<const __nv_bfloat16*>(x_S) +
                                                           (desc->N - desc->T) * ld_x);
  if (!aligned16(x_tail) || !aligned16(x_exact) || !aligned16(A) || !aligned16(b) || !aligned16(Wv) ||
      (!prefolded && !aligned16(gain)))
    return fail(RF_ERR_ALIGN, "x_S, x_exact, A, b, gain and Wv must be 16-byte aligned");
  RescaleLayout lay = rescale_layout(desc, c, workspace);
  if (workspace == nullptr || workspace_bytes < lay.bytes || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(RF_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned (got %zu)", lay.bytes, workspace_bytes);
  int sms = 0;
  if ((st = current_device(&sms)) != RF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  k_set_count<<<1, 1, 0, s>>>(lay.n_c, static_cast<int>(c));
  if ((st = cuda_check(cudaGetLastError(), "k_set_count launch")) != RF_OK) return st;
  const void* wv = Wv;
  if (!prefolded) {
    if ((st = fold_gain(gain, Wv, lay.wv, desc->L - desc->S, desc->n_kv_heads * desc->head_dim, d, sms, s)) != RF_OK)
      return st;
    wv = lay.wv;
  }
  st = use_pair(desc->flags, true)
           ? rescale_gemms<true>(desc, c, lay, x_tail, ld_x, x_exact, ld_e, A, b, wv, dev_status, sms, s)
           : rescale_gemms<false>(desc, c, lay, x_tail, ld_x, x_exact, ld_e, A, b, wv, dev_status, sms, s);
  if (st != RF_OK) return st;
  const int64_t PH = (desc->L - desc->S) * desc->n_kv_heads;
  {
    ProfScope prof(s, RF_STAGE_RESCALE);
    k_value_scale<<<static_cast<unsigned>((PH + 255) / 256), 256, 0, s>>>(
        lay.norms, static_cast<int>(desc->L - desc->S), static_cast<int>(c), static_cast<int>(desc->n_kv_heads), v_scale);
  }
  return cuda_check(cudaGetLastError(), "k_value_scale launch");
}
