// The two tensor-core GEMM problems of the fill (map GEMM, K/V GEMM), shared by
// rf_fill_kv and the value rescale (rf_value_scale), which runs the same map
// GEMM on the first tail rows.
#pragma once
#include <cuda_bf16.h>

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
  const float* col_scale;  // [P][d] or nullptr: per output column scale (int8 maps' row scales)
  __nv_bfloat16* xhat;     // [P][M_pad][d]
  float* ssp;              // [P][d/256][M_pad]
  int d, k_in, P, M_pad, n_ntiles, m_band;  // d: map output width; k_in: map input width
  int* sched;              // unit counter (dynamic unit order), or nullptr
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
  __device__ int num_kb(int, int) const { return k_in / kBK; }
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
    const float* sp = col_scale != nullptr ? col_scale + static_cast<size_t>(p) * d + c0 : nullptr;
    __nv_bfloat16* dst = xhat + (static_cast<size_t>(p) * M_pad + m) * d + c0;
    // x̂ goes straight from registers, 16 bytes into each lane's own row: turning
    // it through shared memory first (as the cache stores are) measured 1.4 %
    // slower on the 27B-shaped map GEMM, its shared-memory traffic competing with
    // the MMAs' operand reads, and L2 merges the half-written sectors anyway.
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
        const float4 cs = sp != nullptr ? __ldg(reinterpret_cast<const float4*>(sp + ch * 32 + i))
                                        : make_float4(1.f, 1.f, 1.f, 1.f);
        const float x0 = fmaf(u2f(v[i]), cs.x, bb.x), x1 = fmaf(u2f(v[i + 1]), cs.y, bb.y);
        const float x2 = fmaf(u2f(v[i + 2]), cs.z, bb.z), x3 = fmaf(u2f(v[i + 3]), cs.w, bb.w);
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
// 5. K/V GEMM: A operand x̂ [P*M_pad][d]; B operand the folded projections,
//    Wk [P*KV][d] for output columns [0, KV) and Wv [P*KV][d] for [KV, 2KV) of a
//    layer (both K-major, read in boxes of 128 rows; KV % 128 == 0, so a box lies
//    in one of them). Unit u: layer p, M-tile mt, N-tile nt (N fastest: the A
//    tile is reused by the CTAs in flight, and a layer's 2KV x d weights stay in L2).
// --------------------------------------------------------------------------
constexpr int kKvBoxRows = 128;

template <bool kPair_>
struct KVProb {
  CUtensorMap tmA;
  CUtensorMap tmBk;
  CUtensorMap tmBv;
  const int32_t* n_fill;
  const int32_t* fill_idx;
  const float* ssp;        // [P][d/256][M_pad]; slot 0 holds the row scale r after k_row_rms
  __nv_bfloat16* kc;
  __nv_bfloat16* vc;
  const float* v_scale;    // [P][H] or nullptr (value rescale)
  const __nv_bfloat16* k_gain;  // [P][hd] or nullptr (key normalisation)
  long long layer_stride, row_stride;
  long long pos_offset;    // RoPE position of prefix row 0
  RopeFreqs rope;          // the layers' RoPE frequencies (θ, hd)
  int d, P, S, M_pad, KV, hd, n_ntiles, n_ss;
  float inv_d, eps;
  int* sched;              // unit counter (dynamic unit order), or nullptr
  int32_t* dev_status;
  uint64_t timeout_ns;
  static constexpr bool kAMN = false;
  static constexpr bool kBMN = false;
  static constexpr bool kPair = kPair_;
  // Eight epilogue warps, each on 128 columns of a tile (one head at hd = 128):
  // with four, each on 256 columns, the epilogue held the accumulators long enough
  // to show in the GEMM's time.
  static constexpr int kEpiWarps = 8;
  static constexpr size_t kEpiSmemBytes = kEpiWarps * kStageBytesPerWarp;  // staging rows of the cache stores
  struct EpiState {};
  __device__ void epilogue_after(EpiState&, int, int, int, int, int, uint32_t) const {}
  using Cfg = GemmCfg<kPair_>;

  __device__ void prefetch() const {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmBk);
    tma_prefetch_desc(&tmBv);
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
  static constexpr int kBoxes = Cfg::kBRows / kKvBoxRows;  // B boxes per K-block (1 pair, 2 single)
  struct Coords {
    const CUtensorMap* tb[kBoxes];
    int a_row, b_row[kBoxes];
  };
  __device__ Coords coords(int u, int, uint32_t rank) const {
    int p, mt, nt;
    decode(u, m_tiles(), p, mt, nt);
    Coords c;
    c.a_row = p * M_pad + mt * Cfg::kUnitM + static_cast<int>(rank) * kBM;
#pragma unroll
    for (int j = 0; j < kBoxes; ++j) {
      const int col = nt * kBN + static_cast<int>(rank) * Cfg::kBRows + j * kKvBoxRows;  // output column
      const bool v = col >= KV;
      c.tb[j] = v ? &tmBv : &tmBk;
      c.b_row[j] = p * KV + (v ? col - KV : col);
    }
    return c;
  }
  __device__ void issue_loads(Coords& c, int kb, uint8_t* sa, uint8_t* sb, uint32_t bar) const {
    load_operand<kBM, false, kPair>(sa, &tmA, bar, kb * kBK, c.a_row);
#pragma unroll
    for (int j = 0; j < kBoxes; ++j)
      load_operand<kKvBoxRows, false, kPair>(sb + j * (kKvBoxRows * kBK * 2), c.tb[j], bar, kb * kBK, c.b_row[j]);
  }
  __device__ void epilogue(EpiState&, int u, int, int, uint32_t tacc, int row, int wcol0, uint32_t rank) const {
    const int nf = *n_fill;
    int p, mt, nt;
    decode(u, (nf + Cfg::kUnitM - 1) / Cfg::kUnitM, p, mt, nt);
    const int m = mt * Cfg::kUnitM + static_cast<int>(rank) * kBM + row;
    const bool valid = m < nf;
    int t = 0;
    float rs = 0.f;
    if (valid) {
      t = fill_idx[m];
      rs = ssp[static_cast<size_t>(p) * n_ss * M_pad + m];  // the row's RMS scale (k_row_rms)
    }
    const size_t row_off = static_cast<size_t>(S + p) * layer_stride + static_cast<size_t>(t) * row_stride;
    const unsigned long long pos = static_cast<unsigned long long>(static_cast<long long>(t) + pos_offset);
    const uint32_t stage =
        smem_u32(gemm_epi_smem<kPair_>()) + static_cast<uint32_t>(((threadIdx.x >> 5) - 2) * kStageBytesPerWarp);
    // this warp's columns of the tile: wcol0 .. wcol0 + kBN * 4 / kEpiWarps (tacc points at wcol0)
#pragma unroll 1
    for (int hh = 0; hh < kBN * 4 / kEpiWarps / hd; ++hh) {
      const int col0 = nt * kBN + wcol0 + hh * hd;
      const bool is_k = col0 < KV;
      const int h = (is_k ? col0 : col0 - KV) / hd;
      __nv_bfloat16* dst = (is_k ? kc : vc) + row_off + static_cast<size_t>(h) * hd;
      float sc = rs;
      const __nv_bfloat16* g = nullptr;
      if (!is_k && v_scale != nullptr) sc = rs * __ldg(v_scale + p * (KV / hd) + h);
      if (is_k && k_gain != nullptr) {
        // Key normalisation: RMS of the head's rs-scaled values, then its gain (the
        // TMEM loads are warp-collective; the branch is uniform across the warp).
        float q = 0.f;
#pragma unroll 1
        for (int i0 = 0; i0 < hd; i0 += 32) {
          uint32_t v[32];
          tmem_ld32(tacc + hh * hd + i0, v);
          tmem_wait_ld32(v);
#pragma unroll
          for (int i = 0; i < 32; ++i) q = fmaf(u2f(v[i]), u2f(v[i]), q);
        }
        sc = rs * rsqrtf(fmaf(rs * rs, q / static_cast<float>(hd), eps));
        g = k_gain + static_cast<size_t>(p) * hd;
      }
      emit_head(tacc + hh * hd, hd, sc, nullptr, g, is_k ? rope.g : nullptr, pos, valid ? dst : nullptr, stage);
    }
  }
};

// The map GEMM (x̂ = x_rows · A_pᵀ + b_p for all P maps, bf16 x̂ and Σx̂²
// partials), launched from fill.cu only, so that its kernels exist in one
// translation unit (a kernel instantiated in two units would have two device
// copies, and per-kernel launch attributes would be set on only one of them).
//   x_rows      [n_rows_max][ld_x] bf16 rows of width d_in; rows >= *n_rows are not computed
//   n_rows      device int32: rows to compute (<= n_rows_max <= M_pad)
//   A           [P][d][d_in] bf16, b [P][d] fp32
//   col_scale   [P][d] fp32 or nullptr: x̂[o] = col_scale[o] * (A x)[o] + b[o]
//   xhat        [P][M_pad][d] bf16, ssp [P][d/256][M_pad] fp32
struct MapGemmArgs {
  const void* x_rows;
  int64_t ld_x, n_rows_max;
  const int32_t* n_rows;
  const void* A;
  const float* b;
  const float* col_scale;
  __nv_bfloat16* xhat;
  float* ssp;
  int64_t d, d_in, P, M_pad;
  int32_t* dev_status;
  int* sched = nullptr;       // a device int the launch may use for its dynamic unit order
};
rf_status map_gemm(bool pair, const MapGemmArgs& a, int sms, cudaStream_t s);

// The K/V GEMM (norm scale, optional key norm and value scale, RoPE, cache
// scatter), also launched from fill.cu only. Layers S .. S+P-1 of the caches.
struct KvGemmArgs {
  const __nv_bfloat16* xhat;  // [P][M_pad][d]
  float* ssp;                 // [P][d/256][M_pad]; k_row_rms turns slot 0 into the row scale
  const int32_t* n_fill;
  const int32_t* fill_idx;
  const void* Wk;             // [P][KV][d], gain folded
  const void* Wv;             // [P][KV][d], gain folded
  void* k_cache;
  void* v_cache;
  const float* v_scale;       // [P][H] or nullptr
  const void* k_gain;         // [P][hd] bf16 or nullptr
  int64_t layer_stride, row_stride, d, P, S, M_pad, KV, hd;
  double eps;
  double rope_theta;
  int64_t pos_offset;
  int32_t* dev_status;
  int* sched = nullptr;       // a device int the launch may use for its dynamic unit order
};
rf_status kv_gemm(bool pair, const KvGemmArgs& a, int sms, cudaStream_t s);

// Gain fold of one projection, out[p][j][i] = bf16(W[p][j][i] * gain[p][i]) for
// W [P][rows][d] bf16 and gain [P][d] bf16 (in place allowed; d % 8 == 0), on
// stream s. Defined in fill.cu.
rf_status fold_gain(const void* gain, const void* W, void* out, int64_t P, int64_t rows, int64_t d, int sms,
                    cudaStream_t s);

}  // namespace rf
