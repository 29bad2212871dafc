// RidgeFill upper-layer KV fill (rf_fill_kv) and its weight preparation
// (rf_fold_kv_weights).
//
// [RF] RidgeFill review, "Two numbers set the skip range" (which rows are filled)
// and "Ridge map: predict the input, and the original projection runs unchanged"
// (x̂_l = A_l x_S + b_l, then the layer's own norm, K/V projections and RoPE).
//
// Launch sequence on the caller's stream (no host synchronisation):
//   0. k_fold_gain     (unless RF_WEIGHTS_PREFOLDED) W_k·diag(g), W_v·diag(g)
//                      into the workspace
//   1. k_compact       exact-row mask -> ascending fill_idx, n_fill        (1 CTA)
//   2. k_gather_rows   Xf[m] = x_S[fill_idx[m]], zero pad to the M tile     (HBM)
//   3. tc_gemm<MapProb> x̂ = Xf · [A_S; …; A_{L-1}]ᵀ + b, all maps in one GEMM;
//                       epilogue: bf16 x̂ and fp32 Σx̂² per (row, layer, N-tile)
//   4. k_row_rms       r = rsqrt(Σx̂²/d + ε) per (row, layer) from the partials
//   5. tc_gemm<KVProb>  [k|v] = r · x̂_l · [Wk'_l; Wv'_l]ᵀ for every layer in one GEMM;
//                       epilogue: the row scale r, RoPE on k at position
//                       t + pos_offset (angle reduced in 64-bit fixed point), and
//                       the scatter into cache[l][fill_idx[m]], whole head rows per
//                       warp store through shared-memory staging.
#include <algorithm>

#include "rf_host.h"
#include "fill_gemm.cuh"

namespace rf {

// --------------------------------------------------------------------------
// 1. Row compaction: one CTA walks the mask in tiles of 4 bytes per thread (one
//    coalesced 32-bit load per thread where the mask is 4-byte aligned), scans the
//    per-thread counts across the block and writes the filled rows' indices in
//    ascending order, carrying the running count from tile to tile.
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) k_compact(const uint8_t* __restrict__ mask, int n_prefix,
                                                  int32_t* __restrict__ fill_idx, int32_t* __restrict__ n_fill,
                                                  int32_t* __restrict__ n_fill_out) {
  __shared__ int warp_sums[32];
  const int tid = threadIdx.x;
  const int lane = tid & 31, w = tid >> 5;
  const bool vec = mask != nullptr && (reinterpret_cast<uintptr_t>(mask) & 3u) == 0;
  int carry = 0;
  for (int base = 0; base < n_prefix; base += 4 * 1024) {
    const int i0 = base + 4 * tid;
    unsigned keep = 0;  // bit j: row i0 + j is filled
    if (vec && i0 + 3 < n_prefix) {
      const uint32_t v = *reinterpret_cast<const uint32_t*>(mask + i0);
#pragma unroll
      for (int j = 0; j < 4; ++j) keep |= (((v >> (8 * j)) & 0xffu) == 0u ? 1u : 0u) << j;
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (i0 + j < n_prefix && (mask == nullptr || mask[i0 + j] == 0)) keep |= 1u << j;
    }
    const int cnt = __popc(keep);
    int x = cnt;  // inclusive scan over the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[w] = x;
    __syncthreads();
    if (w == 0) {
      int s = warp_sums[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += y;
      }
      warp_sums[lane] = s;
    }
    __syncthreads();
    int pos = carry + x - cnt + (w > 0 ? warp_sums[w - 1] : 0);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if ((keep >> j) & 1u) fill_idx[pos++] = i0 + j;
    carry += warp_sums[31];
    __syncthreads();  // warp_sums is rewritten by the next tile
  }
  if (tid == 0) {
    *n_fill = carry;
    if (n_fill_out != nullptr) *n_fill_out = carry;
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
// Gain fold: out[p][j][i] = bf16(W[p][j][i] * g[p][i]) for one projection
// [P][rows][d]; the bf16 x bf16 product is exact in fp32, so the only rounding is
// the final one. 16 bytes per step; in place is allowed.
// --------------------------------------------------------------------------
__global__ void k_fold_gain(const uint4* __restrict__ gain, const uint4* W, uint4* out, int P, int rows, int d_vec) {
  const long long total = static_cast<long long>(P) * rows * d_vec;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(idx % d_vec);
    const int p = static_cast<int>(idx / (static_cast<long long>(rows) * d_vec));
    const uint4 w = W[idx];
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
    out[idx] = o;
  }
}

rf_status fold_gain(const void* gain, const void* W, void* out, int64_t P, int64_t rows, int64_t d, int sms,
                    cudaStream_t s) {
  const long long total = P * rows * (d / 8);
  const int blocks = static_cast<int>(std::max<long long>(1, std::min<long long>((total + 255) / 256, 8LL * sms)));
  ProfScope prof(s, RF_STAGE_FOLD);
  k_fold_gain<<<blocks, 256, 0, s>>>(static_cast<const uint4*>(gain), static_cast<const uint4*>(W),
                                     static_cast<uint4*>(out), static_cast<int>(P), static_cast<int>(rows),
                                     static_cast<int>(d / 8));
  return cuda_check(cudaGetLastError(), "k_fold_gain launch");
}

// --------------------------------------------------------------------------
// Host side
// --------------------------------------------------------------------------
struct FillLayout {
  int32_t* fill_idx;
  int32_t* n_fill;
  int* sched;               // unit counter of the GEMM launches (each clears it first)
  __nv_bfloat16* xf;
  __nv_bfloat16* xhat;      // [P][M_pad][d], or one layer in the layered fill
  float* ssp;
  __nv_bfloat16* slot[2];   // layered fill: bf16 map ring (when maps are copied or expanded)
  int8_t* stage[2];         // layered fill: int8 landing slots for host int8 maps
  __nv_bfloat16* wk;        // gain-folded projections [P][KV][d] (without RF_WEIGHTS_PREFOLDED)
  __nv_bfloat16* wv;
  size_t bytes;
};

// The layered fill computes kLayerChunk layers per step (one map GEMM and one K/V
// GEMM over them): one layer per launch leaves the last wave of 76 CTA pairs
// mostly idle (an 8B layer is 704 map and 352 K/V units), four layers per step
// keep that loss to a few percent while x̂ still exists for 4 layers, not P.
constexpr int64_t kLayerChunk = 4;

// Maps the layered fill reads in place (device bf16) need no ring.
static bool maps_staged(const rf_map_source* m) { return !(m->kind == RF_MAPS_BF16 && !m->on_host); }

// Width of x_S rows and of the maps' input (d_in = 0 means square maps).
static int64_t fill_din(const rf_fill_desc* d) { return d->d_in > 0 ? d->d_in : d->d; }

static bool prefolded(const rf_fill_desc* d) { return (d->flags & RF_WEIGHTS_PREFOLDED) != 0; }

static rf_status check_fill_desc(const rf_fill_desc* d) {
  if (d == nullptr) return fail(RF_ERR_INVALID_ARG, "desc is NULL");
  if (d->d <= 0 || d->L <= 0 || d->S < 0 || d->S > d->L || d->N < 0 || d->T < 0 || d->T > d->N ||
      d->n_kv_heads <= 0 || d->head_dim <= 0)
    return fail(RF_ERR_INVALID_ARG, "need d > 0, L > 0, 0 <= S <= L, 0 <= T <= N, H > 0, hd > 0");
  if (!(d->rope_theta > 0.0) || !(d->rms_eps >= 0.0)) return fail(RF_ERR_INVALID_ARG, "need rope_theta > 0, rms_eps >= 0");
  if (d->d % kBN != 0) return fail(RF_ERR_SHAPE, "d = %lld must be a multiple of 256", (long long)d->d);
  if (d->d_in < 0 || fill_din(d) % kBN != 0)
    return fail(RF_ERR_SHAPE, "d_in = %lld must be 0 (square maps) or a multiple of 256", (long long)d->d_in);
  if (fill_din(d) > (int64_t(1) << 20)) return fail(RF_ERR_SHAPE, "d_in must be <= 2^20");
  if (d->head_dim != 64 && d->head_dim != 128) return fail(RF_ERR_SHAPE, "head_dim must be 64 or 128");
  const int64_t KV = d->n_kv_heads * d->head_dim;
  if (KV % 128 != 0) return fail(RF_ERR_SHAPE, "n_kv_heads * head_dim = %lld must be a multiple of 128", (long long)KV);
  if (d->N - d->T > (int64_t(1) << 24)) return fail(RF_ERR_SHAPE, "N - T must be <= 2^24");
  const int64_t P = d->L - d->S;
  if (P * d->d >= (int64_t(1) << 31) || P * 2 * KV >= (int64_t(1) << 31)) return fail(RF_ERR_SHAPE, "too many map rows");
  return RF_OK;
}

// Workspace of the fill (maps == nullptr) or of the layered fill (x̂ for one
// layer at a time, plus the map ring).
static FillLayout fill_layout(const rf_fill_desc* d, void* ws, const rf_map_source* maps = nullptr) {
  const int64_t n_prefix = d->N - d->T;
  const int64_t M_pad = round_up(std::max<int64_t>(n_prefix, 1), kFillRowAlign);
  const int64_t P = d->L - d->S;
  const int64_t xhat_layers = maps != nullptr ? std::min<int64_t>(P, kLayerChunk) : P;
  Carve c(ws);
  FillLayout l{};
  l.fill_idx = c.take<int32_t>(std::max<int64_t>(n_prefix, 1));
  l.n_fill = c.take<int32_t>(1);
  l.sched = c.take<int>(1);
  l.xf = c.take<__nv_bfloat16>(M_pad * fill_din(d));
  l.xhat = c.take<__nv_bfloat16>(xhat_layers * M_pad * d->d);
  l.ssp = c.take<float>(xhat_layers * (d->d / kBN) * M_pad);
  if (!prefolded(d) && P > 0 && n_prefix > 0) {
    const int64_t w = P * d->n_kv_heads * d->head_dim * d->d;
    l.wk = c.take<__nv_bfloat16>(w);
    l.wv = c.take<__nv_bfloat16>(w);
  }
  if (maps != nullptr && maps_staged(maps)) {
    const int64_t n = xhat_layers * d->d * fill_din(d);
    for (int i = 0; i < 2; ++i) l.slot[i] = c.take<__nv_bfloat16>(n);
    if (maps->kind == RF_MAPS_INT8 && maps->on_host)
      for (int i = 0; i < 2; ++i) l.stage[i] = c.take<int8_t>(n);
  }
  l.bytes = c.bytes();
  return l;
}

// The two fill GEMMs, on CTA pairs or single CTAs.
static rf_status fill_gemms(bool pair, const rf_fill_desc* desc, const FillLayout& lay, const rf_bf16* A,
                            const float* b, const void* Wk, const void* Wv, rf_bf16* k_cache, rf_bf16* v_cache,
                            int64_t layer_stride, int64_t row_stride, int32_t* dev_status, int sms, cudaStream_t s) {
  rf_status st;
  const int64_t d = desc->d, P = desc->L - desc->S, KV = desc->n_kv_heads * desc->head_dim;
  const int64_t M_pad = round_up(desc->N - desc->T, kFillRowAlign);
  const int64_t d_in = fill_din(desc);
  MapGemmArgs ma{lay.xf, d_in, M_pad, lay.n_fill, A, b, nullptr, lay.xhat, lay.ssp, d, d_in, P, M_pad, dev_status,
                 lay.sched};
  if ((st = map_gemm(pair, ma, sms, s)) != RF_OK) return st;
  KvGemmArgs ka{lay.xhat, lay.ssp, lay.n_fill, lay.fill_idx, Wk, Wv, k_cache, v_cache,
                desc->v_scale, desc->k_norm_gain, layer_stride, row_stride, d, P, desc->S, M_pad, KV,
                desc->head_dim, desc->rms_eps, desc->rope_theta, desc->pos_offset, dev_status, lay.sched};
  return kv_gemm(pair, ka, sms, s);
}

template <bool kPair>
static rf_status map_gemm_t(const MapGemmArgs& a, int sms, cudaStream_t s) {
  using Cfg = GemmCfg<kPair>;
  rf_status st;
  MapProb<kPair> pr;
  if ((st = make_tmap_bf16_2d(&pr.tmA, a.x_rows, a.d_in, a.n_rows_max, a.ld_x, kBK, kBM)) != RF_OK) return st;
  if ((st = make_tmap_bf16_2d(&pr.tmB, a.A, a.d_in, a.P * a.d, a.d_in, kBK, Cfg::kBRows)) != RF_OK) return st;
  const int64_t m_tiles_max = a.M_pad / Cfg::kUnitM;
  pr.n_fill = a.n_rows;
  pr.bias = a.b;
  pr.col_scale = a.col_scale;
  pr.xhat = a.xhat;
  pr.ssp = a.ssp;
  pr.d = static_cast<int>(a.d);
  pr.k_in = static_cast<int>(a.d_in);
  pr.P = static_cast<int>(a.P);
  pr.M_pad = static_cast<int>(a.M_pad);
  pr.n_ntiles = static_cast<int>(a.P * a.d / kBN);
  pr.m_band = static_cast<int>(
      std::max<long long>(1, std::min<long long>(m_tiles_max, kMapBandBytes / (Cfg::kUnitM * a.d_in * 2))));
  pr.sched = a.sched;
  pr.dev_status = a.dev_status;
  pr.timeout_ns = wait_timeout_ns();
  ProfScope prof(s, RF_STAGE_MAP_GEMM);
  return launch_gemm(pr, m_tiles_max * pr.n_ntiles, sms, s, "map GEMM launch");
}

rf_status map_gemm(bool pair, const MapGemmArgs& a, int sms, cudaStream_t s) {
  return pair ? map_gemm_t<true>(a, sms, s) : map_gemm_t<false>(a, sms, s);
}

// Row RMS scale from the map GEMM's partial sums of squares: for each filled row
// m and layer p, r = (Σ_j ssp[p][j][m] / d + ε)^-1/2, summed in the order j = 0, 1,
// ... and stored in place in slot j = 0 (each thread reads its own row's slots
// before writing), so the K/V epilogue reads one float per row.
__global__ void __launch_bounds__(256) k_row_rms(float* __restrict__ ssp, const int32_t* __restrict__ n_fill, int n_ss,
                                                 int M_pad, float inv_d, float eps) {
  const int m = blockIdx.x * blockDim.x + threadIdx.x;
  if (m >= *n_fill) return;
  float* sp = ssp + static_cast<size_t>(blockIdx.y) * n_ss * M_pad + m;
  float s = 0.f;
  for (int j = 0; j < n_ss; ++j) s += sp[static_cast<size_t>(j) * M_pad];
  sp[0] = rsqrtf(fmaf(s, inv_d, eps));
}

template <bool kPair>
static rf_status kv_gemm_t(const KvGemmArgs& a, int sms, cudaStream_t s) {
  using Cfg = GemmCfg<kPair>;
  rf_status st;
  KVProb<kPair> pr;
  if ((st = make_tmap_bf16_2d(&pr.tmA, a.xhat, a.d, a.P * a.M_pad, a.d, kBK, kBM)) != RF_OK) return st;
  if ((st = make_tmap_bf16_2d(&pr.tmBk, a.Wk, a.d, a.P * a.KV, a.d, kBK, kKvBoxRows)) != RF_OK) return st;
  if ((st = make_tmap_bf16_2d(&pr.tmBv, a.Wv, a.d, a.P * a.KV, a.d, kBK, kKvBoxRows)) != RF_OK) return st;
  pr.n_fill = a.n_fill;
  pr.fill_idx = a.fill_idx;
  pr.ssp = a.ssp;
  pr.pos_offset = a.pos_offset;
  pr.rope = rope_freqs(a.rope_theta, static_cast<int>(a.hd));
  pr.kc = static_cast<__nv_bfloat16*>(a.k_cache);
  pr.vc = static_cast<__nv_bfloat16*>(a.v_cache);
  pr.v_scale = a.v_scale;
  pr.k_gain = static_cast<const __nv_bfloat16*>(a.k_gain);
  pr.layer_stride = a.layer_stride;
  pr.row_stride = a.row_stride;
  pr.d = static_cast<int>(a.d);
  pr.P = static_cast<int>(a.P);
  pr.S = static_cast<int>(a.S);
  pr.M_pad = static_cast<int>(a.M_pad);
  pr.KV = static_cast<int>(a.KV);
  pr.hd = static_cast<int>(a.hd);
  pr.n_ntiles = static_cast<int>(2 * a.KV / kBN);
  pr.n_ss = static_cast<int>(a.d / kBN);
  pr.inv_d = 1.0f / static_cast<float>(a.d);
  pr.eps = static_cast<float>(a.eps);
  pr.sched = a.sched;
  pr.dev_status = a.dev_status;
  pr.timeout_ns = wait_timeout_ns();
  const int64_t m_tiles_max = a.M_pad / Cfg::kUnitM;
  {
    ProfScope prof(s, RF_STAGE_ROW_RMS);
    k_row_rms<<<dim3(static_cast<unsigned>((a.M_pad + 255) / 256), static_cast<unsigned>(a.P)), 256, 0, s>>>(
        a.ssp, a.n_fill, pr.n_ss, pr.M_pad, pr.inv_d, pr.eps);
  }
  if ((st = cuda_check(cudaGetLastError(), "k_row_rms launch")) != RF_OK) return st;
  ProfScope prof(s, RF_STAGE_KV_GEMM);
  return launch_gemm(pr, a.P * m_tiles_max * pr.n_ntiles, sms, s, "K/V GEMM launch");
}

rf_status kv_gemm(bool pair, const KvGemmArgs& a, int sms, cudaStream_t s) {
  return pair ? kv_gemm_t<true>(a, sms, s) : kv_gemm_t<false>(a, sms, s);
}

}  // namespace rf

using namespace rf;

extern "C" size_t rf_fill_workspace_bytes(const rf_fill_desc* desc) {
  if (check_fill_desc(desc) != RF_OK) return 0;
  return fill_layout(desc, nullptr).bytes;
}

extern "C" rf_status rf_fold_kv_weights(const rf_fill_desc* desc, const rf_bf16* gain, const rf_bf16* Wk,
                                        const rf_bf16* Wv, rf_bf16* Wk_folded, rf_bf16* Wv_folded,
                                        rf_stream_t stream) {
  clear_error();
  rf_status st = check_fill_desc(desc);
  if (st != RF_OK) return st;
  const int64_t P = desc->L - desc->S;
  if (P == 0) return RF_OK;
  if (!gain || !Wk || !Wv || !Wk_folded || !Wv_folded)
    return fail(RF_ERR_INVALID_ARG, "gain, Wk, Wv, Wk_folded and Wv_folded must be non-NULL");
  if (!aligned16(gain) || !aligned16(Wk) || !aligned16(Wv) || !aligned16(Wk_folded) || !aligned16(Wv_folded))
    return fail(RF_ERR_ALIGN, "gain, Wk, Wv, Wk_folded and Wv_folded must be 16-byte aligned");
  int sms = 0;
  if ((st = current_device(&sms)) != RF_OK) return st;
  const int64_t KV = desc->n_kv_heads * desc->head_dim;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = fold_gain(gain, Wk, Wk_folded, P, KV, desc->d, sms, s)) != RF_OK) return st;
  return fold_gain(gain, Wv, Wv_folded, P, KV, desc->d, sms, s);
}

// Argument checks shared by rf_fill_kv and rf_fill_kv_layered (the maps are
// checked by the caller).
static rf_status check_fill_args(const rf_fill_desc* desc, const rf_bf16* x_S, int64_t ld_x, const float* b,
                                 const rf_bf16* gain, const rf_bf16* Wk, const rf_bf16* Wv, const rf_bf16* k_cache,
                                 const rf_bf16* v_cache, int64_t layer_stride, int64_t row_stride) {
  const int64_t n_prefix = desc->N - desc->T;
  const int64_t P = desc->L - desc->S;
  const int64_t KV = desc->n_kv_heads * desc->head_dim;
  if (n_prefix > 0 && P > 0) {
    if (!x_S) return fail(RF_ERR_INVALID_ARG, "x_S is NULL");
    if (!b || !Wk || !Wv || !k_cache || !v_cache)
      return fail(RF_ERR_INVALID_ARG, "A, b, Wk, Wv, k_cache, v_cache must be non-NULL");
    if (!prefolded(desc) && !gain)
      return fail(RF_ERR_INVALID_ARG, "gain is NULL (set RF_WEIGHTS_PREFOLDED when Wk and Wv hold the gain)");
    if (!aligned16(x_S) || !aligned16(b) || !aligned16(Wk) || !aligned16(Wv) || !aligned16(k_cache) ||
        !aligned16(v_cache) || (!prefolded(desc) && !aligned16(gain)))
      return fail(RF_ERR_ALIGN, "x_S, A, b, gain, Wk, Wv and the caches must be 16-byte aligned");
    if (ld_x < fill_din(desc) || ld_x % 8 != 0)
      return fail(RF_ERR_ALIGN, "ld_x must be >= d_in (d for square maps) and a multiple of 8");
    if (row_stride < KV || row_stride % 8 != 0 || layer_stride < 0 || layer_stride % 8 != 0)
      return fail(RF_ERR_ALIGN, "row_stride must be >= H*hd and a multiple of 8; layer_stride a multiple of 8");
  }
  return RF_OK;
}

// The projections the K/V GEMM reads: the caller's when prefolded, else the gain
// folded into the workspace now (on stream s, ahead of the GEMMs).
static rf_status kv_weights(const rf_fill_desc* desc, const FillLayout& lay, const rf_bf16* gain, const rf_bf16* Wk,
                            const rf_bf16* Wv, int sms, cudaStream_t s, const void** wk, const void** wv) {
  *wk = Wk;
  *wv = Wv;
  if (prefolded(desc)) return RF_OK;
  const int64_t P = desc->L - desc->S, KV = desc->n_kv_heads * desc->head_dim;
  rf_status st;
  if ((st = fold_gain(gain, Wk, lay.wk, P, KV, desc->d, sms, s)) != RF_OK) return st;
  if ((st = fold_gain(gain, Wv, lay.wv, P, KV, desc->d, sms, s)) != RF_OK) return st;
  *wk = lay.wk;
  *wv = lay.wv;
  return RF_OK;
}

// Row compaction, and when anything is filled the gather, on stream s. *work is
// false when there is nothing left to fill.
static rf_status fill_prologue(const rf_fill_desc* desc, const rf_bf16* x_S, int64_t ld_x, const uint8_t* exact_mask,
                               int32_t* n_fill_out, const FillLayout& lay, int sms, cudaStream_t s, bool* work) {
  *work = false;
  const int64_t n_prefix = desc->N - desc->T;
  const int64_t P = desc->L - desc->S;
  if (n_prefix == 0) {
    if (n_fill_out) return cuda_check(cudaMemsetAsync(n_fill_out, 0, sizeof(int32_t), s), "memset n_fill_out");
    return RF_OK;
  }
  rf_status st;
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
                                                              static_cast<int>(fill_din(desc) / 8),
                                                              static_cast<int>(M_pad));
  }
  if ((st = cuda_check(cudaGetLastError(), "gather launch")) != RF_OK) return st;
  *work = true;
  return RF_OK;
}

extern "C" rf_status rf_fill_kv(const rf_fill_desc* desc, const rf_bf16* x_S, int64_t ld_x, const uint8_t* exact_mask,
                                const rf_bf16* A, const float* b, const rf_bf16* gain, const rf_bf16* Wk,
                                const rf_bf16* Wv, rf_bf16* k_cache, rf_bf16* v_cache, int64_t layer_stride,
                                int64_t row_stride, int32_t* n_fill_out, int32_t* dev_status, void* workspace,
                                size_t workspace_bytes, rf_stream_t stream) {
  clear_error();
  rf_status st = check_fill_desc(desc);
  if (st != RF_OK) return st;
  if ((st = check_fill_args(desc, x_S, ld_x, b, gain, Wk, Wv, k_cache, v_cache, layer_stride, row_stride)) != RF_OK)
    return st;
  const int64_t n_prefix = desc->N - desc->T;
  if (n_prefix > 0 && desc->L > desc->S) {
    if (!A) return fail(RF_ERR_INVALID_ARG, "A, b, Wk, Wv, k_cache, v_cache must be non-NULL");
    if (!aligned16(A)) return fail(RF_ERR_ALIGN, "x_S, A, b, gain, Wk, Wv and the caches must be 16-byte aligned");
  }
  FillLayout lay = fill_layout(desc, workspace);
  if (n_prefix > 0) {
    if (workspace == nullptr || workspace_bytes < lay.bytes || (reinterpret_cast<uintptr_t>(workspace) & 255u))
      return fail(RF_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned (got %zu)", lay.bytes, workspace_bytes);
  }
  int sms = 0;
  if ((st = current_device(&sms)) != RF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bool work = false;
  if ((st = fill_prologue(desc, x_S, ld_x, exact_mask, n_fill_out, lay, sms, s, &work)) != RF_OK || !work) return st;
  const void *wk = nullptr, *wv = nullptr;
  if ((st = kv_weights(desc, lay, gain, Wk, Wv, sms, s, &wk, &wv)) != RF_OK) return st;
  return fill_gemms(use_pair(desc->flags, true), desc, lay, A, b, wk, wv, k_cache, v_cache, layer_stride, row_stride,
                    dev_status, sms, s);
}

// --------------------------------------------------------------------------
// Layer-by-layer fill (rf_fill_kv_layered): one map GEMM and one K/V GEMM per
// step of kLayerChunk layers, x̂ for those layers only. Maps that live on the host
// or in int8 pass through a two-slot bf16 ring: the library's copy stream copies
// (and expands) the next step's layers while the caller's stream computes the
// current ones; events order slot reuse.
// --------------------------------------------------------------------------
struct EventSet {
  cudaEvent_t e[5] = {};
  int n = 0;
  ~EventSet() {
    for (int i = 0; i < n; ++i) cudaEventDestroy(e[i]);
  }
  rf_status create() {
    for (; n < 5; ++n) {
      cudaError_t err = cudaEventCreateWithFlags(&e[n], cudaEventDisableTiming);
      if (err != cudaSuccess) return cuda_check(err, "cudaEventCreateWithFlags");
    }
    return RF_OK;
  }
};

static rf_status check_maps(const rf_map_source* m) {
  if (m == nullptr) return fail(RF_ERR_INVALID_ARG, "maps is NULL");
  if (m->kind != RF_MAPS_BF16 && m->kind != RF_MAPS_INT8)
    return fail(RF_ERR_INVALID_ARG, "maps->kind must be RF_MAPS_BF16 or RF_MAPS_INT8");
  return RF_OK;
}

extern "C" size_t rf_fill_layered_workspace_bytes(const rf_fill_desc* desc, const rf_map_source* maps) {
  if (check_fill_desc(desc) != RF_OK || check_maps(maps) != RF_OK) return 0;
  return fill_layout(desc, nullptr, maps).bytes;
}

extern "C" rf_status rf_fill_kv_layered(const rf_fill_desc* desc, const rf_bf16* x_S, int64_t ld_x,
                                        const uint8_t* exact_mask, const rf_map_source* maps, const float* b,
                                        const rf_bf16* gain, const rf_bf16* Wk, const rf_bf16* Wv, rf_bf16* k_cache,
                                        rf_bf16* v_cache, int64_t layer_stride,
                                        int64_t row_stride, int32_t* n_fill_out, int32_t* dev_status, void* workspace,
                                        size_t workspace_bytes, rf_stream_t stream) {
  clear_error();
  rf_status st = check_fill_desc(desc);
  if (st != RF_OK) return st;
  if ((st = check_maps(maps)) != RF_OK) return st;
  if ((st = check_fill_args(desc, x_S, ld_x, b, gain, Wk, Wv, k_cache, v_cache, layer_stride, row_stride)) != RF_OK)
    return st;
  const int64_t n_prefix = desc->N - desc->T;
  const int64_t P = desc->L - desc->S, d = desc->d, d_in = fill_din(desc), KV = desc->n_kv_heads * desc->head_dim;
  const bool int8 = maps->kind == RF_MAPS_INT8;
  if (n_prefix > 0 && P > 0) {
    if (!maps->A || (int8 && !maps->row_scale))
      return fail(RF_ERR_INVALID_ARG, "maps->A (and maps->row_scale for int8 maps) must be non-NULL");
    if (!aligned16(maps->A) || (int8 && !aligned16(maps->row_scale)))
      return fail(RF_ERR_ALIGN, "maps->A and maps->row_scale must be 16-byte aligned");
  }
  FillLayout lay = fill_layout(desc, workspace, maps);
  if (n_prefix > 0) {
    if (workspace == nullptr || workspace_bytes < lay.bytes || (reinterpret_cast<uintptr_t>(workspace) & 255u))
      return fail(RF_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned (got %zu)", lay.bytes, workspace_bytes);
  }
  int sms = 0;
  if ((st = current_device(&sms)) != RF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool staged = maps_staged(maps) && n_prefix > 0 && P > 0;
  cudaStream_t cs = nullptr;
  EventSet ev;
  cudaEvent_t* ready = ev.e + 1;
  cudaEvent_t* freed = ev.e + 3;
  if (staged) {
    // The ring lives in the caller's workspace: earlier work on `s` may still use
    // it. The event is taken before this call's prologue (which does not touch
    // the ring), so the first copy overlaps the compaction and the gather.
    if ((st = copy_stream(&cs)) != RF_OK || (st = ev.create()) != RF_OK) return st;
    if ((st = cuda_check(cudaEventRecord(ev.e[0], s), "cudaEventRecord")) != RF_OK) return st;
    if ((st = cuda_check(cudaStreamWaitEvent(cs, ev.e[0], 0), "cudaStreamWaitEvent")) != RF_OK) return st;
  }
  bool work = false;
  if ((st = fill_prologue(desc, x_S, ld_x, exact_mask, n_fill_out, lay, sms, s, &work)) != RF_OK || !work) return st;
  const void *wk = nullptr, *wv = nullptr;
  if ((st = kv_weights(desc, lay, gain, Wk, Wv, sms, s, &wk, &wv)) != RF_OK) return st;

  const bool pair = use_pair(desc->flags, true);
  const int64_t M_pad = round_up(n_prefix, kFillRowAlign);
  const size_t map_elems = static_cast<size_t>(d) * static_cast<size_t>(d_in);
  const size_t elem = int8 ? 1 : 2;
  const int64_t H = desc->n_kv_heads;
  // Staged maps start with chunks of 1 and 2 layers, then kLayerChunk: only the
  // first chunk's copy waits in front of the first GEMM, and every later copy
  // fits under the GEMMs of the chunk before it.
  int64_t g = 0;
  for (int64_t c0 = 0, step = 0; c0 < P; c0 += g, ++step) {
    g = std::min<int64_t>(staged && step < 2 ? int64_t(1) << step : kLayerChunk, P - c0);  // layers S+c0 .. +g-1
    const int r = static_cast<int>(step & 1);
    const size_t n = static_cast<size_t>(g) * map_elems;
    const char* src = static_cast<const char*>(maps->A) + static_cast<size_t>(c0) * map_elems * elem;
    const void* Ap = src;
    if (staged) {
      if (step >= 2 && (st = cuda_check(cudaStreamWaitEvent(cs, freed[r], 0), "cudaStreamWaitEvent")) != RF_OK)
        return st;
      if (!int8) {
        st = cuda_check(cudaMemcpyAsync(lay.slot[r], src, n * 2, cudaMemcpyHostToDevice, cs), "map copy");
      } else if (maps->on_host) {
        st = cuda_check(cudaMemcpyAsync(lay.stage[r], src, n, cudaMemcpyHostToDevice, cs), "map copy");
        if (st == RF_OK) st = expand_int8(lay.stage[r], lay.slot[r], n, sms, cs);
      } else {
        st = expand_int8(reinterpret_cast<const int8_t*>(src), lay.slot[r], n, sms, cs);
      }
      if (st != RF_OK) return st;
      if ((st = cuda_check(cudaEventRecord(ready[r], cs), "cudaEventRecord")) != RF_OK) return st;
      if ((st = cuda_check(cudaStreamWaitEvent(s, ready[r], 0), "cudaStreamWaitEvent")) != RF_OK) return st;
      Ap = lay.slot[r];
    }
    MapGemmArgs ma{lay.xf, d_in, M_pad, lay.n_fill, Ap, b + c0 * d, int8 ? maps->row_scale + c0 * d : nullptr,
                   lay.xhat, lay.ssp, d, d_in, g, M_pad, dev_status, lay.sched};
    if ((st = map_gemm(pair, ma, sms, s)) != RF_OK) return st;
    if (staged && (st = cuda_check(cudaEventRecord(freed[r], s), "cudaEventRecord")) != RF_OK) return st;
    KvGemmArgs ka{lay.xhat, lay.ssp, lay.n_fill, lay.fill_idx,
                  static_cast<const __nv_bfloat16*>(wk) + static_cast<size_t>(c0) * KV * d,
                  static_cast<const __nv_bfloat16*>(wv) + static_cast<size_t>(c0) * KV * d, k_cache, v_cache,
                  desc->v_scale ? desc->v_scale + c0 * H : nullptr,
                  desc->k_norm_gain ? reinterpret_cast<const __nv_bfloat16*>(desc->k_norm_gain) + c0 * desc->head_dim
                                    : nullptr,
                  layer_stride, row_stride, d, g, desc->S + c0, M_pad, KV, desc->head_dim, desc->rms_eps,
                  desc->rope_theta, desc->pos_offset, dev_status, lay.sched};
    if ((st = kv_gemm(pair, ka, sms, s)) != RF_OK) return st;
  }
  return RF_OK;
}
