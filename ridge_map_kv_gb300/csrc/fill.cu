// RidgeFill upper-layer KV fill (rf_fill_kv) and its weight preparation
// (rf_fold_kv_weights).
//
// [RF] RidgeFill review, "Two numbers set the skip range" (which rows are filled)
// and "Ridge map: predict the input, and the original projection runs unchanged"
// (x̂_l = A_l x_S + b_l, then the layer's own norm, K/V projections and RoPE).
//
// Launch sequence on the caller's stream (no host synchronisation):
//   1. k_compact       exact-row mask -> ascending fill_idx, n_fill        (1 CTA)
//   2. k_gather_rows   Xf[m] = x_S[fill_idx[m]], zero pad to the M tile     (HBM)
//   3. k_rope_table    cos/sin of (t + pos_offset) * θ^(-2i/hd), fp64 angle (tiny)
//   4. tc_gemm<MapProb> x̂ = Xf · [A_S; …; A_{L-1}]ᵀ + b, all maps in one GEMM;
//                       epilogue: bf16 x̂ and fp32 Σx̂² per (row, layer, N-tile)
//   5. tc_gemm<KVProb>  [k|v] = r · x̂_l · Wkv_lᵀ for every layer in one GEMM;
//                       epilogue: r = rsqrt(Σx̂²/d + ε), RoPE on k, scatter
//                       into cache[l][fill_idx[m]] with 16-byte stores.
#include <algorithm>

#include "rf_host.h"
#include "epilogue.cuh"
#include "tc_gemm.cuh"

namespace rf {

// Filled rows are padded to whole 256-row units (the M of a CTA-pair tile) in
// the gathered operand, the x̂ buffer and the sum-of-squares partials.
constexpr int kFillRowAlign = 256;

// Bytes of gathered rows Xf that one band of the map GEMM keeps in L2.
#ifndef RF_MAP_BAND_BYTES
#define RF_MAP_BAND_BYTES (32ll << 20)
#endif
constexpr long long kMapBandBytes = RF_MAP_BAND_BYTES;

// --------------------------------------------------------------------------
// 1. Row compaction: one CTA, each thread scans a contiguous chunk of the mask.
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) k_compact(const uint8_t* __restrict__ mask, int n_prefix,
                                                  int32_t* __restrict__ fill_idx, int32_t* __restrict__ n_fill,
                                                  int32_t* __restrict__ n_fill_out) {
  __shared__ int warp_sums[32];
  const int tid = threadIdx.x;
  const int nthr = blockDim.x;
  const int per = (n_prefix + nthr - 1) / nthr;
  const int lo = min(tid * per, n_prefix);
  const int hi = min(lo + per, n_prefix);
  int cnt = 0;
  for (int i = lo; i < hi; ++i) cnt += (mask == nullptr || mask[i] == 0) ? 1 : 0;
  const int lane = tid & 31, w = tid >> 5;
  int x = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[w] = x;
  __syncthreads();
  if (w == 0) {
    int s = (lane < nthr / 32) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;
  }
  __syncthreads();
  int pos = x - cnt + (w > 0 ? warp_sums[w - 1] : 0);
  for (int i = lo; i < hi; ++i)
    if (mask == nullptr || mask[i] == 0) fill_idx[pos++] = i;
  if (tid == nthr - 1) {
    *n_fill = pos;
    if (n_fill_out != nullptr) *n_fill_out = pos;
  }
}

// --------------------------------------------------------------------------
// 2. Gather filled rows into a dense, M-tile padded operand (pad rows zeroed).
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(128) k_gather_rows(const uint4* __restrict__ x, long long ld_vec,
                                                     const int32_t* __restrict__ fill_idx,
                                                     const int32_t* __restrict__ n_fill, uint4* __restrict__ xf,
                                                     int row_vecs, int max_rows) {
  const int m = blockIdx.x;
  const int nf = *n_fill;
  const int pad_end = min((nf + kFillRowAlign - 1) / kFillRowAlign * kFillRowAlign, max_rows);
  if (m >= pad_end) return;
  uint4* dst = xf + static_cast<size_t>(m) * row_vecs;
  if (m < nf) {
    const uint4* src = x + static_cast<size_t>(fill_idx[m]) * ld_vec;
    for (int c = threadIdx.x; c < row_vecs; c += blockDim.x) dst[c] = __ldg(src + c);
  } else {
    for (int c = threadIdx.x; c < row_vecs; c += blockDim.x) dst[c] = make_uint4(0, 0, 0, 0);
  }
}

// --------------------------------------------------------------------------
// 3. RoPE table: angle (t + pos_offset) θ^(-2i/hd) in fp64, reduced mod 2π in
//    fp64 (two-constant Cody–Waite), then sincosf on the reduced angle.
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_rope_table(float* __restrict__ cos_t, float* __restrict__ sin_t, int n_rows,
                                                    int half, double theta, long long pos_offset) {
  __shared__ double inv_freq[128];
  for (int i = threadIdx.x; i < half; i += blockDim.x) inv_freq[i] = pow(theta, -2.0 * i / (2.0 * half));
  __syncthreads();
  const double kInv2Pi = 0.15915494309189535;
  const double k2PiHi = 6.283185307179586;
  const double k2PiLo = 2.4492935982947064e-16;
  const long long total = static_cast<long long>(n_rows) * half;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long t = idx / half;
    const int i = static_cast<int>(idx - t * half);
    const double ang = static_cast<double>(t + pos_offset) * inv_freq[i];
    const double k = rint(ang * kInv2Pi);
    double r = fma(-k, k2PiHi, ang);
    r = fma(-k, k2PiLo, r);
    float s, c;
    sincosf(static_cast<float>(r), &s, &c);
    cos_t[idx] = c;
    sin_t[idx] = s;
  }
}

// --------------------------------------------------------------------------
// Gain fold: Wkv[p][j][i] = bf16(W[p][j][i] * g[p][i]); the bf16 x bf16 product
// is exact in fp32, so the only rounding is the final one.
// --------------------------------------------------------------------------
__global__ void k_fold_gain(const uint4* __restrict__ gain, const uint4* __restrict__ Wk,
                            const uint4* __restrict__ Wv, uint4* __restrict__ Wkv, int P, int KV, int d_vec) {
  const long long total = static_cast<long long>(P) * 2 * KV * d_vec;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(idx % d_vec);
    const long long r = idx / d_vec;
    const int j = static_cast<int>(r % (2 * KV));
    const int p = static_cast<int>(r / (2 * KV));
    const uint4 w = j < KV ? __ldg(Wk + (static_cast<long long>(p) * KV + j) * d_vec + c)
                           : __ldg(Wv + (static_cast<long long>(p) * KV + (j - KV)) * d_vec + c);
    const uint4 g = __ldg(gain + static_cast<long long>(p) * d_vec + c);
    const __nv_bfloat162* wh = reinterpret_cast<const __nv_bfloat162*>(&w);
    const __nv_bfloat162* gh = reinterpret_cast<const __nv_bfloat162*>(&g);
    uint4 o;
    uint32_t* ou = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 a = __bfloat1622float2(wh[q]);
      const float2 b = __bfloat1622float2(gh[q]);
      ou[q] = pack_bf16x2(a.x * b.x, a.y * b.y);
    }
    Wkv[idx] = o;
  }
}

// --------------------------------------------------------------------------
// 4. Map GEMM: A operand Xf [M_pad][d], B operand maps [P*d][d] (both K-major).
//    Units run in bands of m_band M-tiles; within a band, N-tiles outer and the
//    band's M-tiles inner. The CTAs in flight share one map tile through L2,
//    and the band's rows of Xf (about kMapBandBytes) stay in L2 for every N-tile
//    of the band; the maps are read once per band. Without bands, the whole Xf
//    is re-read per N-tile and, once it outgrows the share of L2 left beside the
//    streaming maps and outputs, LRU evicts exactly the rows needed next.
// --------------------------------------------------------------------------
template <bool kPair_>
struct MapProb {
  CUtensorMap tmA;
  CUtensorMap tmB;
  const int32_t* n_fill;
  const float* bias;       // [P][d]
  __nv_bfloat16* xhat;     // [P][M_pad][d]
  float* ssp;              // [P][d/256][M_pad]
  int d, P, M_pad, n_ntiles, m_band;
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
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  __device__ int m_tiles() const { return (*n_fill + Cfg::kUnitM - 1) / Cfg::kUnitM; }
  // Unit -> (M-tile, N-tile): band b holds M-tiles [b*m_band, b*m_band + gb),
  // gb = m_band except in the last band.
  __device__ void decode(int u, int mtc, int& mt, int& nt) const {
    const int per_band = m_band * n_ntiles;
    const int b = u / per_band;
    const int r = u - b * per_band;
    const int gb = min(m_band, mtc - b * m_band);
    nt = r / gb;
    mt = b * m_band + (r - nt * gb);
  }
  __device__ int num_units() const { return m_tiles() * n_ntiles; }
  __device__ int num_subtiles(int) const { return 1; }
  __device__ int num_kb(int, int) const { return d / kBK; }
  struct Coords {
    int a_row, b_row;
  };
  __device__ Coords coords(int u, int, uint32_t rank) const {
    int mt, nt;
    decode(u, m_tiles(), mt, nt);
    return {mt * Cfg::kUnitM + static_cast<int>(rank) * kBM, nt * kBN + static_cast<int>(rank) * Cfg::kBRows};
  }
  __device__ void issue_loads(Coords& c, int kb, uint8_t* sa, uint8_t* sb, uint32_t bar) const {
    load_operand<kBM, false, kPair>(sa, &tmA, bar, kb * kBK, c.a_row);
    load_operand<Cfg::kBRows, false, kPair>(sb, &tmB, bar, kb * kBK, c.b_row);
  }
  __device__ void epilogue(EpiState&, int u, int, int, uint32_t tacc, int row, int, uint32_t rank) const {
    const int nf = *n_fill;
    int mt, nt;
    decode(u, (nf + Cfg::kUnitM - 1) / Cfg::kUnitM, mt, nt);
    const int n0 = nt * kBN;
    const int p = n0 / d;
    const int c0 = n0 - p * d;
    const int m = mt * Cfg::kUnitM + static_cast<int>(rank) * kBM + row;
    const bool valid = m < nf;
    const float* bp = bias + static_cast<size_t>(p) * d + c0;
    __nv_bfloat16* dst = xhat + (static_cast<size_t>(p) * M_pad + m) * d + c0;
    float ss = 0.f;
#pragma unroll 1
    for (int ch = 0; ch < kBN / 32; ++ch) {
      uint32_t v[32];
      tmem_ld32(tacc + ch * 32, v);
      tmem_wait_ld32(v);
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        const float4 bb = __ldg(reinterpret_cast<const float4*>(bp + ch * 32 + i));
        const float x0 = u2f(v[i]) + bb.x, x1 = u2f(v[i + 1]) + bb.y;
        const float x2 = u2f(v[i + 2]) + bb.z, x3 = u2f(v[i + 3]) + bb.w;
        ss = fmaf(x0, x0, ss);
        ss = fmaf(x1, x1, ss);
        ss = fmaf(x2, x2, ss);
        ss = fmaf(x3, x3, ss);
        pk[i / 2] = pack_bf16x2(x0, x1);
        pk[i / 2 + 1] = pack_bf16x2(x2, x3);
      }
      if (valid) {
#pragma unroll
        for (int q = 0; q < 4; ++q) st_global_v4(dst + ch * 32 + 8 * q, pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      }
    }
    if (valid) ssp[(static_cast<size_t>(p) * (d / kBN) + c0 / kBN) * M_pad + m] = ss;
  }
};

// --------------------------------------------------------------------------
// 5. K/V GEMM: A operand x̂ [P*M_pad][d], B operand Wkv [P*2KV][d] (K-major).
//    Unit u: layer p, M-tile mt, N-tile nt (N fastest: the A tile is reused by
//    the CTAs in flight, and a layer's 2KV x d weights stay in L2).
// --------------------------------------------------------------------------
template <bool kPair_>
struct KVProb {
  CUtensorMap tmA;
  CUtensorMap tmB;
  const int32_t* n_fill;
  const int32_t* fill_idx;
  const float* ssp;        // [P][d/256][M_pad]
  const float* rope_cos;   // [n_prefix][hd/2]
  const float* rope_sin;
  __nv_bfloat16* kc;
  __nv_bfloat16* vc;
  long long layer_stride, row_stride;
  int d, P, S, M_pad, KV, hd, n_ntiles, n_ss;
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
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  __device__ int m_tiles() const { return (*n_fill + Cfg::kUnitM - 1) / Cfg::kUnitM; }
  __device__ int num_units() const { return P * m_tiles() * n_ntiles; }
  __device__ int num_subtiles(int) const { return 1; }
  __device__ int num_kb(int, int) const { return d / kBK; }
  __device__ void decode(int u, int mtc, int& p, int& mt, int& nt) const {
    const int per_layer = mtc * n_ntiles;
    p = u / per_layer;
    const int r = u - p * per_layer;
    mt = r / n_ntiles;
    nt = r - mt * n_ntiles;
  }
  struct Coords {
    int a_row, b_row;
  };
  __device__ Coords coords(int u, int, uint32_t rank) const {
    int p, mt, nt;
    decode(u, m_tiles(), p, mt, nt);
    return {p * M_pad + mt * Cfg::kUnitM + static_cast<int>(rank) * kBM,
            p * 2 * KV + nt * kBN + static_cast<int>(rank) * Cfg::kBRows};
  }
  __device__ void issue_loads(Coords& c, int kb, uint8_t* sa, uint8_t* sb, uint32_t bar) const {
    load_operand<kBM, false, kPair>(sa, &tmA, bar, kb * kBK, c.a_row);
    load_operand<Cfg::kBRows, false, kPair>(sb, &tmB, bar, kb * kBK, c.b_row);
  }
  __device__ void epilogue(EpiState&, int u, int, int, uint32_t tacc, int row, int, uint32_t rank) const {
    const int nf = *n_fill;
    int p, mt, nt;
    decode(u, (nf + Cfg::kUnitM - 1) / Cfg::kUnitM, p, mt, nt);
    const int m = mt * Cfg::kUnitM + static_cast<int>(rank) * kBM + row;
    const bool valid = m < nf;
    int t = 0;
    float rs = 0.f;
    if (valid) {
      t = fill_idx[m];
      const float* sp = ssp + static_cast<size_t>(p) * n_ss * M_pad + m;
      float s = 0.f;
      for (int j = 0; j < n_ss; ++j) s += sp[static_cast<size_t>(j) * M_pad];
      rs = rsqrtf(fmaf(s, inv_d, eps));
    }
    const size_t row_off = static_cast<size_t>(S + p) * layer_stride + static_cast<size_t>(t) * row_stride;
    const int half = hd >> 1;
    const float* cs = rope_cos + static_cast<size_t>(t) * half;
    const float* sn = rope_sin + static_cast<size_t>(t) * half;
#pragma unroll 1
    for (int hh = 0; hh < kBN / hd; ++hh) {
      const int col0 = nt * kBN + hh * hd;
      const bool is_k = col0 < KV;
      const int h = (is_k ? col0 : col0 - KV) / hd;
      __nv_bfloat16* dst = (is_k ? kc : vc) + row_off + static_cast<size_t>(h) * hd;
      emit_head(tacc + hh * hd, hd, rs, nullptr, is_k, cs, sn, dst, valid);
    }
  }
};

// --------------------------------------------------------------------------
// Host side
// --------------------------------------------------------------------------
struct FillLayout {
  int32_t* fill_idx;
  int32_t* n_fill;
  __nv_bfloat16* xf;
  __nv_bfloat16* xhat;
  float* ssp;
  float* rope_cos;
  float* rope_sin;
  size_t bytes;
};

static rf_status check_fill_desc(const rf_fill_desc* d) {
  if (d == nullptr) return fail(RF_ERR_INVALID_ARG, "desc is NULL");
  if (d->d <= 0 || d->L <= 0 || d->S < 0 || d->S > d->L || d->N < 0 || d->T < 0 || d->T > d->N ||
      d->n_kv_heads <= 0 || d->head_dim <= 0)
    return fail(RF_ERR_INVALID_ARG, "need d > 0, L > 0, 0 <= S <= L, 0 <= T <= N, H > 0, hd > 0");
  if (!(d->rope_theta > 0.0) || !(d->rms_eps >= 0.0)) return fail(RF_ERR_INVALID_ARG, "need rope_theta > 0, rms_eps >= 0");
  if (d->d % kBN != 0) return fail(RF_ERR_SHAPE, "d = %lld must be a multiple of 256", (long long)d->d);
  if (d->head_dim != 64 && d->head_dim != 128) return fail(RF_ERR_SHAPE, "head_dim must be 64 or 128");
  const int64_t KV = d->n_kv_heads * d->head_dim;
  if (KV % 128 != 0) return fail(RF_ERR_SHAPE, "n_kv_heads * head_dim = %lld must be a multiple of 128", (long long)KV);
  if (d->N - d->T > (int64_t(1) << 24)) return fail(RF_ERR_SHAPE, "N - T must be <= 2^24");
  const int64_t P = d->L - d->S;
  if (P * d->d >= (int64_t(1) << 31) || P * 2 * KV >= (int64_t(1) << 31)) return fail(RF_ERR_SHAPE, "too many map rows");
  return RF_OK;
}

static FillLayout fill_layout(const rf_fill_desc* d, void* ws) {
  const int64_t n_prefix = d->N - d->T;
  const int64_t M_pad = round_up(std::max<int64_t>(n_prefix, 1), kFillRowAlign);
  const int64_t P = d->L - d->S;
  Carve c(ws);
  FillLayout l;
  l.fill_idx = c.take<int32_t>(std::max<int64_t>(n_prefix, 1));
  l.n_fill = c.take<int32_t>(1);
  l.xf = c.take<__nv_bfloat16>(M_pad * d->d);
  l.xhat = c.take<__nv_bfloat16>(P * M_pad * d->d);
  l.ssp = c.take<float>(P * (d->d / kBN) * M_pad);
  l.rope_cos = c.take<float>(std::max<int64_t>(n_prefix, 1) * (d->head_dim / 2));
  l.rope_sin = c.take<float>(std::max<int64_t>(n_prefix, 1) * (d->head_dim / 2));
  l.bytes = c.bytes();
  return l;
}

// The two fill GEMMs, on CTA pairs (kPair) or single CTAs.
template <bool kPair>
rf_status fill_gemms(const rf_fill_desc* desc, const FillLayout& lay, const rf_bf16* A, const float* b,
                     const rf_bf16* Wkv, rf_bf16* k_cache, rf_bf16* v_cache, int64_t layer_stride, int64_t row_stride,
                     int32_t* dev_status, int sms, cudaStream_t s) {
  using Cfg = GemmCfg<kPair>;
  rf_status st;
  const int64_t d = desc->d, P = desc->L - desc->S, KV = desc->n_kv_heads * desc->head_dim;
  const int64_t M_pad = round_up(desc->N - desc->T, kFillRowAlign);
  const int64_t m_tiles_max = M_pad / Cfg::kUnitM;
  const uint64_t tmo = wait_timeout_ns();
  {
    MapProb<kPair> pr;
    if ((st = make_tmap_bf16_2d(&pr.tmA, lay.xf, d, M_pad, d, kBK, kBM)) != RF_OK) return st;
    if ((st = make_tmap_bf16_2d(&pr.tmB, A, d, P * d, d, kBK, Cfg::kBRows)) != RF_OK) return st;
    pr.n_fill = lay.n_fill;
    pr.bias = b;
    pr.xhat = lay.xhat;
    pr.ssp = lay.ssp;
    pr.d = static_cast<int>(d);
    pr.P = static_cast<int>(P);
    pr.M_pad = static_cast<int>(M_pad);
    pr.n_ntiles = static_cast<int>(P * d / kBN);
    pr.m_band = static_cast<int>(
        std::max<long long>(1, std::min<long long>(m_tiles_max, kMapBandBytes / (Cfg::kUnitM * d * 2))));
    pr.dev_status = dev_status;
    pr.timeout_ns = tmo;
    ProfScope prof(s, RF_STAGE_MAP_GEMM);
    if ((st = launch_gemm(pr, m_tiles_max * pr.n_ntiles, sms, s, "map GEMM launch")) != RF_OK) return st;
  }
  {
    KVProb<kPair> pr;
    if ((st = make_tmap_bf16_2d(&pr.tmA, lay.xhat, d, P * M_pad, d, kBK, kBM)) != RF_OK) return st;
    if ((st = make_tmap_bf16_2d(&pr.tmB, Wkv, d, P * 2 * KV, d, kBK, Cfg::kBRows)) != RF_OK) return st;
    pr.n_fill = lay.n_fill;
    pr.fill_idx = lay.fill_idx;
    pr.ssp = lay.ssp;
    pr.rope_cos = lay.rope_cos;
    pr.rope_sin = lay.rope_sin;
    pr.kc = reinterpret_cast<__nv_bfloat16*>(k_cache);
    pr.vc = reinterpret_cast<__nv_bfloat16*>(v_cache);
    pr.layer_stride = layer_stride;
    pr.row_stride = row_stride;
    pr.d = static_cast<int>(d);
    pr.P = static_cast<int>(P);
    pr.S = static_cast<int>(desc->S);
    pr.M_pad = static_cast<int>(M_pad);
    pr.KV = static_cast<int>(KV);
    pr.hd = static_cast<int>(desc->head_dim);
    pr.n_ntiles = static_cast<int>(2 * KV / kBN);
    pr.n_ss = static_cast<int>(d / kBN);
    pr.inv_d = 1.0f / static_cast<float>(d);
    pr.eps = static_cast<float>(desc->rms_eps);
    pr.dev_status = dev_status;
    pr.timeout_ns = tmo;
    ProfScope prof(s, RF_STAGE_KV_GEMM);
    if ((st = launch_gemm(pr, P * m_tiles_max * pr.n_ntiles, sms, s, "K/V GEMM launch")) != RF_OK) return st;
  }
  return RF_OK;
}

}  // namespace rf

using namespace rf;

extern "C" size_t rf_fill_workspace_bytes(const rf_fill_desc* desc) {
  if (check_fill_desc(desc) != RF_OK) return 0;
  return fill_layout(desc, nullptr).bytes;
}

extern "C" rf_status rf_fold_kv_weights(const rf_fill_desc* desc, const rf_bf16* gain, const rf_bf16* Wk,
                                        const rf_bf16* Wv, rf_bf16* Wkv, rf_stream_t stream) {
  clear_error();
  rf_status st = check_fill_desc(desc);
  if (st != RF_OK) return st;
  const int64_t P = desc->L - desc->S;
  if (P == 0) return RF_OK;
  if (!gain || !Wk || !Wv || !Wkv) return fail(RF_ERR_INVALID_ARG, "gain, Wk, Wv and Wkv must be non-NULL");
  if (!aligned16(gain) || !aligned16(Wk) || !aligned16(Wv) || !aligned16(Wkv))
    return fail(RF_ERR_ALIGN, "gain, Wk, Wv, Wkv must be 16-byte aligned");
  int sms = 0;
  if ((st = current_device(&sms)) != RF_OK) return st;
  const int KV = static_cast<int>(desc->n_kv_heads * desc->head_dim);
  const int d_vec = static_cast<int>(desc->d / 8);
  const long long total = P * 2LL * KV * d_vec;
  const int blocks = static_cast<int>(std::min<long long>((total + 255) / 256, 8LL * sms));
  ProfScope prof(static_cast<cudaStream_t>(stream), RF_STAGE_FOLD);
  k_fold_gain<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4*>(gain), reinterpret_cast<const uint4*>(Wk), reinterpret_cast<const uint4*>(Wv),
      reinterpret_cast<uint4*>(Wkv), static_cast<int>(P), KV, d_vec);
  return cuda_check(cudaGetLastError(), "k_fold_gain launch");
}

extern "C" rf_status rf_fill_kv(const rf_fill_desc* desc, const rf_bf16* x_S, int64_t ld_x, const uint8_t* exact_mask,
                                const rf_bf16* A, const float* b, const rf_bf16* Wkv, rf_bf16* k_cache,
                                rf_bf16* v_cache, int64_t layer_stride, int64_t row_stride, int32_t* n_fill_out,
                                int32_t* dev_status, void* workspace, size_t workspace_bytes, rf_stream_t stream) {
  clear_error();
  rf_status st = check_fill_desc(desc);
  if (st != RF_OK) return st;
  const int64_t n_prefix = desc->N - desc->T;
  const int64_t P = desc->L - desc->S;
  const int64_t KV = desc->n_kv_heads * desc->head_dim;
  const int64_t d = desc->d;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool any = n_prefix > 0 && P > 0;
  if (n_prefix > 0) {
    if (!x_S && any) return fail(RF_ERR_INVALID_ARG, "x_S is NULL");
  }
  if (any) {
    if (!A || !b || !Wkv || !k_cache || !v_cache) return fail(RF_ERR_INVALID_ARG, "A, b, Wkv, k_cache, v_cache must be non-NULL");
    if (!aligned16(x_S) || !aligned16(A) || !aligned16(b) || !aligned16(Wkv) || !aligned16(k_cache) || !aligned16(v_cache))
      return fail(RF_ERR_ALIGN, "x_S, A, b, Wkv and the caches must be 16-byte aligned");
    if (ld_x < d || ld_x % 8 != 0) return fail(RF_ERR_ALIGN, "ld_x must be >= d and a multiple of 8");
    if (row_stride < KV || row_stride % 8 != 0 || layer_stride < 0 || layer_stride % 8 != 0)
      return fail(RF_ERR_ALIGN, "row_stride must be >= H*hd and a multiple of 8; layer_stride a multiple of 8");
  }
  FillLayout lay = fill_layout(desc, workspace);
  if (n_prefix > 0) {
    if (workspace == nullptr || workspace_bytes < lay.bytes || (reinterpret_cast<uintptr_t>(workspace) & 255u))
      return fail(RF_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned (got %zu)", lay.bytes, workspace_bytes);
  }
  int sms = 0;
  if ((st = current_device(&sms)) != RF_OK) return st;

  if (n_prefix == 0) {
    if (n_fill_out) return cuda_check(cudaMemsetAsync(n_fill_out, 0, sizeof(int32_t), s), "memset n_fill_out");
    return RF_OK;
  }
  {
    ProfScope prof(s, RF_STAGE_COMPACT);
    k_compact<<<1, 1024, 0, s>>>(exact_mask, static_cast<int>(n_prefix), lay.fill_idx, lay.n_fill, n_fill_out);
  }
  if ((st = cuda_check(cudaGetLastError(), "k_compact launch")) != RF_OK) return st;
  if (P == 0) return RF_OK;

  const int64_t M_pad = round_up(n_prefix, kFillRowAlign);
  {
    ProfScope prof(s, RF_STAGE_GATHER);
    k_gather_rows<<<static_cast<unsigned>(M_pad), 128, 0, s>>>(reinterpret_cast<const uint4*>(x_S), ld_x / 8,
                                                              lay.fill_idx, lay.n_fill, reinterpret_cast<uint4*>(lay.xf),
                                                              static_cast<int>(d / 8), static_cast<int>(M_pad));
  }
  const int half = static_cast<int>(desc->head_dim / 2);
  const int rope_blocks = static_cast<int>(std::min<int64_t>((n_prefix * half + 255) / 256, 4LL * sms));
  {
    ProfScope prof(s, RF_STAGE_ROPE_TABLE);
    k_rope_table<<<rope_blocks, 256, 0, s>>>(lay.rope_cos, lay.rope_sin, static_cast<int>(n_prefix), half,
                                             desc->rope_theta, static_cast<long long>(desc->pos_offset));
  }
  if ((st = cuda_check(cudaGetLastError(), "gather / rope launch")) != RF_OK) return st;

  if (use_pair(desc->flags, true))
    return fill_gemms<true>(desc, lay, A, b, Wkv, k_cache, v_cache, layer_stride, row_stride, dev_status, sms, s);
  return fill_gemms<false>(desc, lay, A, b, Wkv, k_cache, v_cache, layer_stride, row_stride, dev_status, sms, s);
}
