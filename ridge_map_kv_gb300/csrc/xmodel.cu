// Cross-model per-head ridge mapper (rf_xmodel_map) and RoPE on cache rows
// (rf_rope_rows).
//
// [XM] "Cross-Model KV Cache Transfer in LLM Families", content-space mapping:
//   K̂_t = (K_s R_s^-1(t) W_K + b_K) R_t(t); V is mapped without RoPE. The k source
// layers chosen for a target layer are concatenated (all heads), and mapper
// inference is one batched matmul per target layer.
//
// Launch sequence on the caller's stream:
//   0. k_check_layers    the caller's device table of source layers: range check
//                        (an entry outside [0, L_src) sets RF_ERR_INVALID_ARG and
//                        turns the GEMM into a no-op) and a copy into the workspace
//   1. k_rope_rows       un-rope every source layer's keys once into the workspace
//   2. tc_gemm<XMProb>   for every target layer l, M-tile of rows and N-tile of
//                        [K | V] columns: A = the selected source features (the
//                        K-loop walks the k source layers, 64 features per step,
//                        reading the table src[l][j]), B = W_K or W_V of layer l;
//                        epilogue: + b, target RoPE on K, store into the target
//                        caches, whole head rows per warp store through
//                        shared-memory staging.
// RoPE angles are reduced in 64-bit fixed point (RopeFreqs, epilogue.cuh) and
// their sine and cosine taken on the SFU, in both kernels: no tables.
#include <algorithm>
#include <vector>

#include "epilogue.cuh"
#include "rf_host.h"
#include "tc_gemm.cuh"

namespace rf {

// out[row][h][:] = R^{sign}(pos) in[row][h][:], pos = row % rows_per_position + pos_offset,
// with the frequencies `rf` of (θ, hd). Each thread takes 8 rotation pairs (one chunk)
// of one row for every head: the 8 angles are formed once and serve all the row's
// heads, and a step costs two index divisions (8 lanes cover a head's 128-byte half
// row, so a warp's loads stay whole-sector).
__global__ void __launch_bounds__(256) k_rope_rows(const __nv_bfloat16* __restrict__ in, __nv_bfloat16* out,
                                                   long long n_rows, long long ld_in, long long ld_out, int n_heads,
                                                   int hd, long long rows_per_position, long long pos_offset,
                                                   const __grid_constant__ RopeFreqs rf, float sign) {
  const int half = hd >> 1;
  const int chunks = half / 8;
  const long long total = n_rows * chunks;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = idx / chunks;
    const int i0 = static_cast<int>(idx - row * chunks) * 8;
    const long long t = row % rows_per_position;
    float c[8], s[8];
    const unsigned long long pos = static_cast<unsigned long long>(t + pos_offset);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      rope_cs(pos, rf.g[i0 + q], c[q], s[q]);
      s[q] *= sign;
    }
    const __nv_bfloat16* src = in + row * ld_in + i0;
    __nv_bfloat16* dst = out + row * ld_out + i0;
#pragma unroll 4
    for (int h = 0; h < n_heads; ++h) {
      const uint4 a = *reinterpret_cast<const uint4*>(src + static_cast<long long>(h) * hd);
      const uint4 b = *reinterpret_cast<const uint4*>(src + static_cast<long long>(h) * hd + half);
      const __nv_bfloat162* ah = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* bh = reinterpret_cast<const __nv_bfloat162*>(&b);
      uint4 o1, o2;
      uint32_t* u1 = reinterpret_cast<uint32_t*>(&o1);
      uint32_t* u2 = reinterpret_cast<uint32_t*>(&o2);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 x1 = __bfloat1622float2(ah[q]);
        const float2 x2 = __bfloat1622float2(bh[q]);
        u1[q] = pack_bf16x2(x1.x * c[2 * q] - x2.x * s[2 * q], x1.y * c[2 * q + 1] - x2.y * s[2 * q + 1]);
        u2[q] = pack_bf16x2(x2.x * c[2 * q] + x1.x * s[2 * q], x2.y * c[2 * q + 1] + x1.y * s[2 * q + 1]);
      }
      *reinterpret_cast<uint4*>(dst + static_cast<long long>(h) * hd) = o1;
      *reinterpret_cast<uint4*>(dst + static_cast<long long>(h) * hd + half) = o2;
    }
  }
}

// Checks the source-layer table on the device and copies it to the workspace:
// *ok = 1 if every entry lies in [0, L_src), else 0 with RF_ERR_INVALID_ARG in
// *dev_status (out-of-range entries are copied as 0, so nothing downstream ever
// indexes with them). One CTA.
__global__ void __launch_bounds__(256) k_check_layers(const int32_t* __restrict__ in, int n, int L_src,
                                                      int32_t* __restrict__ out, int32_t* __restrict__ ok,
                                                      int32_t* dev_status) {
  int bad = 0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int v = in[i];
    const bool good = v >= 0 && v < L_src;
    out[i] = good ? v : 0;
    bad |= good ? 0 : 1;
  }
  bad = __syncthreads_or(bad);
  if (threadIdx.x == 0) {
    *ok = bad ? 0 : 1;
    if (bad) record_status(dev_status, RF_ERR_INVALID_ARG);
  }
}

template <bool kPair_>
struct XMProb {
  CUtensorMap tmKu;  // un-roped source keys   {KV, L_src*N}, box {64, 128}
  CUtensorMap tmVs;  // source values          {KV, L_src*N}, box {64, 128}
  CUtensorMap tmWk;  // W_K                    {k*KV, L_tgt*KV}, box {64, 256}
  CUtensorMap tmWv;  // W_V
  const int32_t* src;  // [L_tgt][k]
  const int32_t* ok;   // 1 if the table passed k_check_layers; else the GEMM does nothing
  const float* bk;     // [L_tgt][KV]
  const float* bv;
  RopeFreqs rope_t;      // target RoPE frequencies (θ_tgt, hd)
  long long pos_offset;  // position of row 0
  int* sched;            // unit counter (dynamic unit order)
  __nv_bfloat16* k_tgt;  // [L_tgt][N][KV]
  __nv_bfloat16* v_tgt;
  int N, KV, hd, k, L_tgt, m_tiles, n_half;
  int32_t* dev_status;
  uint64_t timeout_ns;
  static constexpr bool kAMN = false;
  static constexpr bool kBMN = false;
  static constexpr bool kPair = kPair_;
  static constexpr int kEpiWarps = 8;  // 128 columns of a tile each (one head at hd = 128)
  static constexpr size_t kEpiSmemBytes = kEpiWarps * kStageBytesPerWarp;  // staging rows of the target stores
  struct EpiState {};
  __device__ void epilogue_after(EpiState&, int, int, int, int, int, uint32_t) const {}
  using Cfg = GemmCfg<kPair_>;

  __device__ void prefetch() const {
    tma_prefetch_desc(&tmKu);
    tma_prefetch_desc(&tmVs);
    tma_prefetch_desc(&tmWk);
    tma_prefetch_desc(&tmWv);
  }
  __device__ int num_units() const { return *ok ? L_tgt * m_tiles * 2 * n_half : 0; }
  __device__ int num_subtiles(int) const { return 1; }
  __device__ int num_kb(int, int) const { return k * KV / kBK; }
  // Unit order: target layer, M-tile, then the 2*n_half N-tiles (K then V), so
  // the CTAs in flight reuse one strip of features and one layer's W from L2.
  __device__ void decode(int u, int& l, int& mt, int& nt) const {
    const int per_layer = m_tiles * 2 * n_half;
    l = u / per_layer;
    const int r = u - l * per_layer;
    mt = r / (2 * n_half);
    nt = r - mt * 2 * n_half;
  }
  // K-blocks run in order 0, 1, ...; the feature column c walks through one
  // source layer's KV columns, then the next source layer (row base a_src). The
  // next layer's index is read from the table one whole layer (KV/64 K-blocks)
  // before it is needed, so the load is never waited on in the copy loop.
  struct Coords {
    const CUtensorMap* ta;
    const CUtensorMap* tb;
    const int32_t* srcs;  // this target layer's k source layers
    int a_row, b_row, a_src, next_src, c, j;
  };
  __device__ Coords coords(int u, int, uint32_t rank) const {
    int l, mt, nt;
    decode(u, l, mt, nt);
    const bool is_k = nt < n_half;
    Coords c;
    c.ta = is_k ? &tmKu : &tmVs;
    c.tb = is_k ? &tmWk : &tmWv;
    c.srcs = src + l * k;
    c.a_row = mt * Cfg::kUnitM + static_cast<int>(rank) * kBM;
    c.b_row = l * KV + (is_k ? nt : nt - n_half) * kBN + static_cast<int>(rank) * Cfg::kBRows;
    c.j = 0;
    c.c = 0;
    c.a_src = __ldg(c.srcs) * N;
    c.next_src = k > 1 ? __ldg(c.srcs + 1) : 0;
    return c;
  }
  __device__ void issue_loads(Coords& c, int kb, uint8_t* sa, uint8_t* sb, uint32_t bar) const {
    if (c.c == KV) {
      c.c = 0;
      ++c.j;
      c.a_src = c.next_src * N;
      c.next_src = c.j + 1 < k ? __ldg(c.srcs + c.j + 1) : 0;
    }
    tma2<kPair>(sa, c.ta, bar, c.c, c.a_src + c.a_row);
    tma2<kPair>(sb, c.tb, bar, kb * kBK, c.b_row);
    c.c += kBK;
  }
  __device__ void epilogue(EpiState&, int u, int, int, uint32_t tacc, int row, int wcol0, uint32_t rank) const {
    int l, mt, nt;
    decode(u, l, mt, nt);
    const bool is_k = nt < n_half;
    const int col0 = (is_k ? nt : nt - n_half) * kBN + wcol0;  // this warp's first column (tacc points at it)
    const int t = mt * Cfg::kUnitM + static_cast<int>(rank) * kBM + row;
    const bool valid = t < N;
    const int tt = valid ? t : 0;
    const unsigned long long pos = static_cast<unsigned long long>(static_cast<long long>(tt) + pos_offset);
    const float* bias = (is_k ? bk : bv) + static_cast<size_t>(l) * KV + col0;
    __nv_bfloat16* dst = (is_k ? k_tgt : v_tgt) + (static_cast<size_t>(l) * N + tt) * KV + col0;
    const uint32_t stage =
        smem_u32(gemm_epi_smem<kPair_>()) + static_cast<uint32_t>(((threadIdx.x >> 5) - 2) * kStageBytesPerWarp);
#pragma unroll 1
    for (int hh = 0; hh < kBN * 4 / kEpiWarps / hd; ++hh)
      emit_head(tacc + hh * hd, hd, 1.0f, bias + hh * hd, nullptr, is_k ? rope_t.g : nullptr, pos,
                valid ? dst + hh * hd : nullptr, stage);
  }
};


struct XLayout {
  __nv_bfloat16* ku;
  int32_t* src;
  int32_t* ok;
  int* sched;  // the mapping GEMM's unit counter
  size_t bytes;
};

static XLayout xmodel_layout(const rf_xmodel_desc* d, void* ws) {
  const int64_t KV = d->n_kv_heads * d->head_dim;
  Carve c(ws);
  XLayout l;
  l.ku = c.take<__nv_bfloat16>(d->L_src * d->N * KV);
  l.src = c.take<int32_t>(d->L_tgt * d->k);
  l.ok = c.take<int32_t>(1);
  l.sched = c.take<int>(1);
  l.bytes = c.bytes();
  return l;
}

static rf_status check_xmodel_desc(const rf_xmodel_desc* d) {
  if (d == nullptr) return fail(RF_ERR_INVALID_ARG, "desc is NULL");
  if (d->L_src <= 0 || d->L_tgt <= 0 || d->k <= 0 || d->n_kv_heads <= 0 || d->head_dim <= 0 || d->N <= 0)
    return fail(RF_ERR_INVALID_ARG, "need L_src, L_tgt, k, H, hd, N > 0");
  if (!(d->theta_src > 0.0) || !(d->theta_tgt > 0.0)) return fail(RF_ERR_INVALID_ARG, "RoPE bases must be > 0");
  if (d->head_dim != 64 && d->head_dim != 128) return fail(RF_ERR_SHAPE, "head_dim must be 64 or 128");
  const int64_t KV = d->n_kv_heads * d->head_dim;
  if (KV % kBN != 0) return fail(RF_ERR_SHAPE, "n_kv_heads * head_dim = %lld must be a multiple of 256", (long long)KV);
  if (d->L_src * d->N >= (int64_t(1) << 31) || d->L_tgt * KV >= (int64_t(1) << 31) || d->k * KV >= (int64_t(1) << 31))
    return fail(RF_ERR_SHAPE, "sizes exceed 2^31 rows or features");
  if (d->N > (int64_t(1) << 30)) return fail(RF_ERR_SHAPE, "N must be <= 2^30");
  return RF_OK;
}

template <bool kPair>
rf_status xmodel_gemm(const rf_xmodel_desc* desc, const XLayout& lay, const rf_bf16* v_src, const rf_bf16* Wk,
                      const float* bk, const rf_bf16* Wv, const float* bv, rf_bf16* k_tgt, rf_bf16* v_tgt,
                      int32_t* dev_status, int sms, cudaStream_t s) {
  using Cfg = GemmCfg<kPair>;
  rf_status st;
  const int64_t KV = desc->n_kv_heads * desc->head_dim, N = desc->N;
  XMProb<kPair> pr;
  const int64_t rows = desc->L_src * N;
  if ((st = make_tmap_bf16_2d(&pr.tmKu, lay.ku, KV, rows, KV, kBK, kBM)) != RF_OK) return st;
  if ((st = make_tmap_bf16_2d(&pr.tmVs, v_src, KV, rows, KV, kBK, kBM)) != RF_OK) return st;
  if ((st = make_tmap_bf16_2d(&pr.tmWk, Wk, desc->k * KV, desc->L_tgt * KV, desc->k * KV, kBK, Cfg::kBRows)) != RF_OK)
    return st;
  if ((st = make_tmap_bf16_2d(&pr.tmWv, Wv, desc->k * KV, desc->L_tgt * KV, desc->k * KV, kBK, Cfg::kBRows)) != RF_OK)
    return st;
  pr.src = lay.src;
  pr.ok = lay.ok;
  pr.bk = bk;
  pr.bv = bv;
  pr.rope_t = rope_freqs(desc->theta_tgt, static_cast<int>(desc->head_dim));
  pr.sched = lay.sched;
  pr.pos_offset = static_cast<long long>(desc->pos_offset);
  pr.k_tgt = reinterpret_cast<__nv_bfloat16*>(k_tgt);
  pr.v_tgt = reinterpret_cast<__nv_bfloat16*>(v_tgt);
  pr.N = static_cast<int>(N);
  pr.KV = static_cast<int>(KV);
  pr.hd = static_cast<int>(desc->head_dim);
  pr.k = static_cast<int>(desc->k);
  pr.L_tgt = static_cast<int>(desc->L_tgt);
  pr.m_tiles = static_cast<int>((N + Cfg::kUnitM - 1) / Cfg::kUnitM);
  pr.n_half = static_cast<int>(KV / kBN);
  pr.dev_status = dev_status;
  pr.timeout_ns = wait_timeout_ns();
  ProfScope prof(s, RF_STAGE_XMODEL_GEMM);
  return launch_gemm(pr, desc->L_tgt * pr.m_tiles * 2 * pr.n_half, sms, s, "cross-model GEMM launch");
}

}  // namespace rf

using namespace rf;

extern "C" size_t rf_xmodel_workspace_bytes(const rf_xmodel_desc* desc) {
  if (check_xmodel_desc(desc) != RF_OK) return 0;
  return xmodel_layout(desc, nullptr).bytes;
}

extern "C" rf_status rf_xmodel_map(const rf_xmodel_desc* desc, const int32_t* src_layers, const rf_bf16* k_src,
                                   const rf_bf16* v_src, const rf_bf16* Wk, const float* bk, const rf_bf16* Wv,
                                   const float* bv, rf_bf16* k_tgt, rf_bf16* v_tgt, int32_t* dev_status,
                                   void* workspace, size_t workspace_bytes, rf_stream_t stream) {
  clear_error();
  rf_status st = check_xmodel_desc(desc);
  if (st != RF_OK) return st;
  if (src_layers == nullptr) return fail(RF_ERR_INVALID_ARG, "src_layers is NULL");
  if (desc->L_tgt * desc->k > (int64_t(1) << 24)) return fail(RF_ERR_SHAPE, "L_tgt * k must be <= 2^24");
  if (!k_src || !v_src || !Wk || !bk || !Wv || !bv || !k_tgt || !v_tgt)
    return fail(RF_ERR_INVALID_ARG, "tensor pointers must be non-NULL");
  if (!aligned16(k_src) || !aligned16(v_src) || !aligned16(Wk) || !aligned16(bk) || !aligned16(Wv) || !aligned16(bv) ||
      !aligned16(k_tgt) || !aligned16(v_tgt))
    return fail(RF_ERR_ALIGN, "tensor pointers must be 16-byte aligned");
  XLayout lay = xmodel_layout(desc, workspace);
  if (workspace == nullptr || workspace_bytes < lay.bytes || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(RF_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned (got %zu)", lay.bytes, workspace_bytes);
  int sms = 0;
  if ((st = current_device(&sms)) != RF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t KV = desc->n_kv_heads * desc->head_dim, N = desc->N;
  const int half = static_cast<int>(desc->head_dim / 2);
  // the caller's device table, checked and copied on the device (no host round trip)
  k_check_layers<<<1, 256, 0, s>>>(src_layers, static_cast<int>(desc->L_tgt * desc->k), static_cast<int>(desc->L_src),
                                   lay.src, lay.ok, dev_status);
  if ((st = cuda_check(cudaGetLastError(), "k_check_layers launch")) != RF_OK) return st;
  {
    ProfScope prof(s, RF_STAGE_UNROPE);
    const long long n_rows = desc->L_src * N;
    const long long total = n_rows * (half / 8);  // one thread a row and chunk of 8 pairs
    const int blocks = static_cast<int>(std::min<long long>((total + 255) / 256, 16LL * sms));
    k_rope_rows<<<blocks, 256, 0, s>>>(reinterpret_cast<const __nv_bfloat16*>(k_src), lay.ku, n_rows, KV, KV,
                                       static_cast<int>(desc->n_kv_heads), static_cast<int>(desc->head_dim), N,
                                       static_cast<long long>(desc->pos_offset),
                                       rope_freqs(desc->theta_src, static_cast<int>(desc->head_dim)), -1.0f);
  }
  if ((st = cuda_check(cudaGetLastError(), "rope launches")) != RF_OK) return st;

  if (use_pair(desc->flags, true))
    return xmodel_gemm<true>(desc, lay, v_src, Wk, bk, Wv, bv, k_tgt, v_tgt, dev_status, sms, s);
  return xmodel_gemm<false>(desc, lay, v_src, Wk, bk, Wv, bv, k_tgt, v_tgt, dev_status, sms, s);
}

extern "C" rf_status rf_rope_rows(const rf_bf16* in, rf_bf16* out, int64_t n_rows, int64_t ld, int64_t n_heads,
                                  int64_t head_dim, double theta, int64_t pos_offset, int inverse,
                                  rf_stream_t stream) {
  clear_error();
  if (n_rows < 0 || n_heads <= 0 || !(theta > 0.0)) return fail(RF_ERR_INVALID_ARG, "need n_rows >= 0, n_heads > 0, theta > 0");
  if (head_dim != 64 && head_dim != 128) return fail(RF_ERR_SHAPE, "head_dim must be 64 or 128");
  if (ld < n_heads * head_dim || ld % 8 != 0) return fail(RF_ERR_ALIGN, "ld must be >= n_heads*head_dim and a multiple of 8");
  if (n_rows == 0) return RF_OK;
  if (!in || !out) return fail(RF_ERR_INVALID_ARG, "in and out must be non-NULL");
  if (!aligned16(in) || !aligned16(out)) return fail(RF_ERR_ALIGN, "in and out must be 16-byte aligned");
  int sms = 0;
  rf_status st = current_device(&sms);
  if (st != RF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long total = n_rows * (head_dim / 16);
  const int blocks = static_cast<int>(std::min<long long>((total + 255) / 256, 16LL * sms));
  ProfScope prof(s, RF_STAGE_UNROPE);
  k_rope_rows<<<blocks, 256, 0, s>>>(reinterpret_cast<const __nv_bfloat16*>(in), reinterpret_cast<__nv_bfloat16*>(out),
                                     n_rows, ld, ld, static_cast<int>(n_heads), static_cast<int>(head_dim), n_rows,
                                     pos_offset, rope_freqs(theta, static_cast<int>(head_dim)), inverse ? -1.0f : 1.0f);
  return cuda_check(cudaGetLastError(), "k_rope_rows launch");
}

namespace rf {

// out[t][j] = in[t][j] for t < n_rows, j < width (width % 8 == 0), 16 bytes per step.
__global__ void __launch_bounds__(256) k_copy_rows(const __nv_bfloat16* __restrict__ in, __nv_bfloat16* __restrict__ out,
                                                   long long n_rows, long long ld_in, long long ld_out, int width) {
  const int per_row = width / 8;
  const long long total = n_rows * per_row;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long t = i / per_row;
    const int c = static_cast<int>(i - t * per_row) * 8;
    *reinterpret_cast<uint4*>(out + t * ld_out + c) = __ldg(reinterpret_cast<const uint4*>(in + t * ld_in + c));
  }
}

}  // namespace rf

extern "C" rf_status rf_concat_layers(const rf_bf16* src, int64_t n_layers, int64_t layer_stride, int64_t n_rows,
                                      int64_t ld_src, int64_t n_heads, int64_t head_dim, double theta,
                                      int64_t pos_offset, rf_bf16* out, int64_t ld_out, rf_stream_t stream) {
  clear_error();
  if (n_layers < 0 || n_rows < 0 || n_heads <= 0 || head_dim <= 0 || !(theta >= 0.0))
    return fail(RF_ERR_INVALID_ARG, "need n_layers, n_rows >= 0, n_heads, head_dim > 0, theta >= 0");
  if (theta > 0.0 && head_dim != 64 && head_dim != 128)
    return fail(RF_ERR_SHAPE, "head_dim must be 64 or 128 when keys are un-roped");
  const int64_t W = n_heads * head_dim;
  if (W % 8 != 0) return fail(RF_ERR_SHAPE, "n_heads * head_dim must be a multiple of 8");
  if (ld_src < W || ld_src % 8 != 0 || ld_out < n_layers * W || ld_out % 8 != 0 || layer_stride % 8 != 0 ||
      (n_layers > 1 && layer_stride < ld_src * n_rows))
    return fail(RF_ERR_ALIGN, "need ld_src >= W, ld_out >= n_layers*W, layer_stride >= ld_src*n_rows, "
                              "all multiples of 8");
  if (n_layers == 0 || n_rows == 0) return RF_OK;
  if (!src || !out) return fail(RF_ERR_INVALID_ARG, "src and out must be non-NULL");
  if (!aligned16(src) || !aligned16(out)) return fail(RF_ERR_ALIGN, "src and out must be 16-byte aligned");
  int sms = 0;
  rf_status st = current_device(&sms);
  if (st != RF_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const __nv_bfloat16* in = reinterpret_cast<const __nv_bfloat16*>(src);
  __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(out);
  ProfScope prof(s, RF_STAGE_UNROPE);
  const RopeFreqs rf = theta > 0.0 ? rope_freqs(theta, static_cast<int>(head_dim)) : RopeFreqs{};
  for (int64_t l = 0; l < n_layers; ++l) {
    const long long total = theta > 0.0 ? n_rows * (head_dim / 16) : n_rows * (W / 8);
    const int blocks = static_cast<int>(std::min<long long>((total + 255) / 256, 16LL * sms));
    if (theta > 0.0) {
      k_rope_rows<<<blocks, 256, 0, s>>>(in + l * layer_stride, o + l * W, n_rows, ld_src, ld_out,
                                         static_cast<int>(n_heads), static_cast<int>(head_dim), n_rows, pos_offset,
                                         rf, -1.0f);
    } else {
      k_copy_rows<<<blocks, 256, 0, s>>>(in + l * layer_stride, o + l * W, n_rows, ld_src, ld_out,
                                         static_cast<int>(W));
    }
  }
  return cuda_check(cudaGetLastError(), "rf_concat_layers launches");
}
