// Cross-layer source selection (rf_select_sources).
//
// [XM] "소스 층은 몇 개가 필요한가": greedy forward selection adds, one at a time,
// the source layer that raises the head-mean R² most; "층 교차 소스 선택": the
// mapper takes, per target layer, the k source layers with the highest head-mean
// R² of the un-roped keys and of the values, shared by all heads of that layer.
//
// The ridge fit of a target on the features of a layer set S explains
// e_o = c_oᵀ (Gc_SS + αI)^-1 c_o of each output column o. Greedy selection over
// layers is a block Cholesky factorisation of H = Gc + αI whose next pivot block
// is the layer with the best score. With S chosen (m features) and L_S its factor,
// every other layer s carries
//   W_s   = H_{s,S} L_S^-ᵀ              (its would-be row of the factor)
//   Σ_s   = H_ss − W_s W_sᵀ              (its Schur block given S)
//   R_s   = Cc_s − W_s Z_S               (its residual cross terms; Z_S = L_S^-1 Cc_S)
// and adding s explains z_s = L_s^-1 R_s more (Σ_s = L_s L_sᵀ): e(S ∪ s) =
// e(S) + colsum(z_s²). After choosing b, every layer gets one more block column
//   W_s ← [W_s, (H_{s,b} − W_s W_bᵀ) L_b^-ᵀ],   Σ_s −= w wᵀ,   R_s −= w z_b
// (w the new block). Per pass over a group of target layers, for every kind and
// target ("problem" q) at once, a step runs:
//   k_sel_mask_identity      Σ of already-chosen layers := I (never scored)
//   sel_factor               L_s^-1 for every (q, s), from a copy of Σ: recursive
//                            halving, the products of widths >= 512 on the tensor
//                            cores, narrower ones fp32 SIMT, 128-wide leaves in
//                            shared memory
//   SelGemm (sum of squares) z_sᵀ = R_sᵀ L_s^-ᵀ, only colsum(z_s²) is kept
//   k_sel_layer_scores       every (target, kind, layer)'s score and its table entry
//   k_sel_choose             the joint argmax, the choice, e += gain
//   SelGemm                  z_bᵀ;  H[:, b] − W W_bᵀ;  × L_b^-ᵀ;  Σ_s −= w wᵀ;
//                            Rᵀ −= z_bᵀ wᵀ  (the units of chosen layers run nothing)
// Every product is fp32-accurate on the bf16 tensor cores: each fp32 operand is
// split into three bf16 planes (by k_split_rows, or by the epilogue of the product
// that makes it: the new block column and its × L_b^-ᵀ) and the six plane products
// that matter at fp32 precision are summed: per 1024-wide K chunk the six terms run
// as one TMEM accumulation, smallest first, and the chunks add in fp32 registers.
// Operands are K-major rows of the planes; which rows and columns a batch entry
// reads is linear in (term, problem, layer slot, chosen layer), the chosen layer
// read on the device, so no step waits on the host.
#include <algorithm>
#include <cmath>

#include "rf_host.h"
#include "rf_device.cuh"
#include "tc_gemm.cuh"

namespace rf {

constexpr int kSelChunk = 1024;  // K rows summed in TMEM before the fp32 register sum
constexpr int kSelMaxKinds = 2;
enum { kSkipNone = 0, kSkipSlot = 1, kSkipMRows = 2, kSkipNCols = 3 };  // SelGemmProb::skip

// Six plane products: term t multiplies A plane sel_term_a(t) by B plane sel_term_b(t):
// hi·hi, mid·hi, hi·mid, lo·hi, mid·mid, hi·lo. A chunk's accumulation takes them in
// reverse, t = 5 .. 0: the terms of 2^-16 and 2^-8 of the product first, while the
// accumulator is small, then hi·hi, so the fp32 accumulator's rounding is that of
// hi·hi's own sum (one accumulator per term, added in registers, took the MMA
// thread through six epilogue round trips per chunk).
__device__ __forceinline__ int sel_term_a(int t) { return (0x012010 >> (4 * t)) & 3; }
__device__ __forceinline__ int sel_term_b(int t) { return (0x210100 >> (4 * t)) & 3; }

// Row and K coordinates of one operand in the 2-D view [3 * plane_rows][k_extent]
// of its planes.
struct SelOperand {
  long long plane_rows;
  long long q_rows, s_rows, b_rows;  // per problem, per layer slot, per chosen layer
  long long k0, s_k, b_k;            // K offset: fixed, per layer slot, per chosen layer
};

template <bool kPair_>
struct SelGemmProb {
  CUtensorMap tmA;
  CUtensorMap tmB;
  SelOperand a, b;
  const int32_t* chosen;  // [Q] layer chosen this step by problem q, or nullptr
  int Q, nS;              // batch entry p = q * nS + s
  int M, N, K, m_tiles, n_tiles, n_chunks;
  float alpha, beta;
  // store: out[q*o_q + s*o_s + m*ldo + n] = alpha·acc + beta·C, C at
  //        csrc + (q / q_per_kind)*c_kind + bq*c_b + q*c_q + s*c_s + m*ldc + n
  float* out;
  long long o_q, o_s, ldo;
  const float* csrc;
  long long c_kind, c_b, c_q, c_s, ldc;
  int q_per_kind;
  // sum of squares: part[(p*M + m)*2*n_tiles + 2*nt + half] = Σ (alpha·acc)² over 128 columns
  float* part;
  // or the result as three bf16 planes (split3 of alpha·acc + beta·C): element
  // (q, m, n) of plane j at po + j*po_plane + q*po_q + m*po_ld + po_col + n
  __nv_bfloat16* po;
  long long po_plane, po_q, po_ld, po_col;
  // B lower triangular in (row n, column k), an L^-1: tile column nt reads only
  // k < 256 (nt + 1), the rest of its K range being exact zeros
  int b_tri;
  // unit order: M tiles innermost (for N >> M, so that the units sharing one B tile
  // run together), else N tiles innermost
  int m_inner;
  // Units of a layer already chosen for the problem's target (mask[(q % mask_g) *
  // mask_ls + layer] != 0) run nothing: the layer is the batch slot s (kSkipSlot),
  // the M tile's (kSkipMRows, M = D rows of F per layer) or the N tile's (kSkipNCols).
  const uint8_t* mask;
  int skip, mask_g, mask_ls, layer_f;
  int* sched;  // unit counter (dynamic unit order), or nullptr for round-robin dealing
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
  __device__ int num_units() const { return Q * nS * m_tiles * n_tiles; }
  // K extent of unit u and its number of kSelChunk-wide chunks
  __device__ int k_ext(int u) const {
    if (!b_tri) return K;
    const int nt = m_inner ? (u / m_tiles) % n_tiles : u % n_tiles;
    return min(K, kBN * (nt + 1));
  }
  __device__ int chunks(int u) const { return b_tri ? (k_ext(u) + kSelChunk - 1) / kSelChunk : n_chunks; }
  // Sub-tile sb = 6 c + j is term 5 - j of K chunk c; a chunk's six terms chain into
  // one accumulator, smallest first (see sel_term_a), so the epilogue runs once a chunk.
  __device__ int num_subtiles(int u) const { return skipped(u) ? 0 : 6 * chunks(u); }
  __device__ bool acc_continues(int, int sb) const { return sb % 6 != 0; }
  __device__ int num_kb(int u, int sb) const {
    const int c = sb / 6;
    return (min(kSelChunk, k_ext(u) - c * kSelChunk) + kBK - 1) / kBK;
  }
  __device__ bool skipped(int u) const {
    if (skip == kSkipNone) return false;
    int q, s, mt, nt;
    decode(u, q, s, mt, nt);
    const int layer = skip == kSkipSlot ? s : skip == kSkipMRows ? mt * Cfg::kUnitM / layer_f : nt * kBN / layer_f;
    return mask[(q % mask_g) * mask_ls + layer] != 0;
  }
  __device__ void decode(int u, int& q, int& s, int& mt, int& nt) const {
    if (m_inner) {
      mt = u % m_tiles;
      u /= m_tiles;
      nt = u % n_tiles;
      u /= n_tiles;
    } else {
      nt = u % n_tiles;
      u /= n_tiles;
      mt = u % m_tiles;
      u /= m_tiles;
    }
    q = u / nS;
    s = u - q * nS;
  }
  // This thread's row of the β·C term: kCols floats from column n0 = nt·256 + col0.
  __device__ const float* c_row(int u, int row, int col0, uint32_t rank) const {
    int q, s, mt, nt;
    decode(u, q, s, mt, nt);
    const long long m = static_cast<long long>(mt) * Cfg::kUnitM + rank * kBM + row;
    const long long n0 = static_cast<long long>(nt) * kBN + col0;
    const long long bq = chosen != nullptr ? chosen[q] : 0;
    return csrc + (q / q_per_kind) * c_kind + bq * c_b + q * c_q + s * c_s + m * ldc + n0;
  }
  struct Coords {
    int a_row, a_k, b_row, b_k;
  };
  __device__ Coords coords(int u, int sb, uint32_t rank) const {
    int q, s, mt, nt;
    decode(u, q, s, mt, nt);
    const int c = sb / 6, t = 5 - (sb - 6 * c);
    const long long bq = chosen != nullptr ? chosen[q] : 0;
    Coords r;
    r.a_row = static_cast<int>(sel_term_a(t) * a.plane_rows + q * a.q_rows + s * a.s_rows + bq * a.b_rows +
                               static_cast<long long>(mt) * Cfg::kUnitM + rank * kBM);
    r.a_k = static_cast<int>(a.k0 + s * a.s_k + bq * a.b_k + static_cast<long long>(c) * kSelChunk);
    r.b_row = static_cast<int>(sel_term_b(t) * b.plane_rows + q * b.q_rows + s * b.s_rows + bq * b.b_rows +
                               static_cast<long long>(nt) * kBN + rank * Cfg::kBRows);
    r.b_k = static_cast<int>(b.k0 + s * b.s_k + bq * b.b_k + static_cast<long long>(c) * kSelChunk);
    return r;
  }
  __device__ void issue_loads(Coords& c, int kb, uint8_t* sa, uint8_t* sb, uint32_t bar) const {
    load_operand<kBM, false, kPair>(sa, &tmA, bar, c.a_k + kb * kBK, c.a_row);
    load_operand<Cfg::kBRows, false, kPair>(sb, &tmB, bar, c.b_k + kb * kBK, c.b_row);
  }
  __device__ void epilogue(EpiState& es, int, int sb, int, uint32_t tacc, int, int, uint32_t) const {
#pragma unroll
    for (int ch = 0; ch < kCols / 32; ++ch) {
      uint32_t v[32];
      tmem_ld32(tacc + ch * 32, v);
      tmem_wait_ld32(v);
#pragma unroll
      for (int i = 0; i < 32; ++i) es.rs[ch * 32 + i] = sb < 6 ? u2f(v[i]) : es.rs[ch * 32 + i] + u2f(v[i]);
    }
  }
  __device__ void epilogue_after(EpiState& es, int u, int sb, int nsub, int row, int col0, uint32_t rank) const {
    if (sb != nsub - 1) return;
    int q, s, mt, nt;
    decode(u, q, s, mt, nt);
    const long long m = static_cast<long long>(mt) * Cfg::kUnitM + rank * kBM + row;
    const long long n0 = static_cast<long long>(nt) * kBN + col0;
    if (part != nullptr) {
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < kCols; ++i) {
        const float v = alpha * es.rs[i];
        ss = fmaf(v, v, ss);
      }
      const long long p = static_cast<long long>(q) * nS + s;
      part[(p * M + m) * (2 * n_tiles) + 2 * nt + col0 / kCols] = ss;
      return;
    }
    if (po != nullptr) {
      const float4* cp = beta != 0.f ? reinterpret_cast<const float4*>(c_row(u, row, col0, rank)) : nullptr;
      __nv_bfloat16* d = po + q * po_q + m * po_ld + po_col + n0;
#pragma unroll
      for (int i = 0; i < kCols / 8; ++i) {
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = alpha * es.rs[8 * i + e];
        if (cp != nullptr) {
          const float4 c0 = cp[2 * i], c1 = cp[2 * i + 1];
          v[0] = fmaf(beta, c0.x, v[0]);
          v[1] = fmaf(beta, c0.y, v[1]);
          v[2] = fmaf(beta, c0.z, v[2]);
          v[3] = fmaf(beta, c0.w, v[3]);
          v[4] = fmaf(beta, c1.x, v[4]);
          v[5] = fmaf(beta, c1.y, v[5]);
          v[6] = fmaf(beta, c1.z, v[6]);
          v[7] = fmaf(beta, c1.w, v[7]);
        }
        __align__(16) __nv_bfloat16 hi[8], mi[8], lo[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) split3(v[e], hi[e], mi[e], lo[e]);
        *reinterpret_cast<uint4*>(d + 8 * i) = *reinterpret_cast<const uint4*>(hi);
        *reinterpret_cast<uint4*>(d + po_plane + 8 * i) = *reinterpret_cast<const uint4*>(mi);
        *reinterpret_cast<uint4*>(d + 2 * po_plane + 8 * i) = *reinterpret_cast<const uint4*>(lo);
      }
      return;
    }
    float4* o = reinterpret_cast<float4*>(out + q * o_q + s * o_s + m * ldo + n0);
    const float4* cp = beta != 0.f ? reinterpret_cast<const float4*>(c_row(u, row, col0, rank)) : nullptr;
#pragma unroll
    for (int i = 0; i < kCols / 4; ++i) {
      float4 v = make_float4(alpha * es.rs[4 * i], alpha * es.rs[4 * i + 1], alpha * es.rs[4 * i + 2],
                             alpha * es.rs[4 * i + 3]);
      if (cp != nullptr) {
        const float4 c = cp[i];
        v.x = fmaf(beta, c.x, v.x);
        v.y = fmaf(beta, c.y, v.y);
        v.z = fmaf(beta, c.z, v.z);
        v.w = fmaf(beta, c.w, v.w);
      }
      o[i] = v;
    }
  }
};

// One split product of the factorisation on square 256 x 256 tiles, for every matrix s
// of a batch: out_s = alpha · A_s B_sᵀ + beta · C_s with A_s, B_s the h x h blocks of
// planes [3][batch * h][h] (K-major, matrix s at rows s*h ..; with kAMN the planes
// hold A_sᵀ, row k of block s being A_s's column k, read MN-major). The factors' triangles
// are known, so a unit computes only the output tiles that are read later and only
// the K-range where both operands can be nonzero (whole 256-wide tiles of zeros
// skipped, so the sums are those of the full product up to the fp32 chunking):
//   tiles: kTriAll, kTriLower (nt <= mt), kTriUpper (nt >= mt);
//   K:     kKAll, kKUpToN (k < 256 (nt + 1)), kKUpToM (k < 256 (mt + 1)),
//          kKFromM (k >= 256 mt), kKFromN (k >= 256 nt).
enum { kTriAll = 0, kTriLower = 1, kTriUpper = 2 };
enum { kKAll = 0, kKUpToN = 1, kKUpToM = 2, kKFromM = 3, kKFromN = 4 };
// K rows summed in TMEM per chunk. Skipping the zero triangles packs every chunk with
// nonzero terms, and the tensor core's fp32 accumulation truncates with a bias that
// grows with the chunk (1024-row chunks left the unrefined 2,560-wide solve's normal
// equations at 1.1e-5 against 8.1e-6 for the full products); 512 keeps it below.
constexpr int kTriChunk = 512;

// CTA pairs only: their 256 x 256 unit is square (a single CTA's is 128 x 256).
template <bool kAMN_>
struct TriGemmProb {
  CUtensorMap tmA;
  CUtensorMap tmB;
  long long plane_rows;  // batch * h
  int h, T, tiles, tile_mode, k_mode;  // T = h / 256 tiles a side; tiles per matrix
  float alpha, beta;
  float* out;
  long long o_s, ldo;
  const float* csrc;
  long long c_s, ldc;
  int* sched;  // unit counter (dynamic unit order), or nullptr for round-robin dealing
  int32_t* dev_status;
  uint64_t timeout_ns;
  static constexpr bool kAMN = kAMN_;
  static constexpr bool kBMN = false;
  static constexpr bool kPair = true;
  static constexpr int kEpiWarps = 8;
  static constexpr int kCols = kBN / 2;
  struct EpiState {
    float rs[kCols];
  };
  using Cfg = GemmCfg<true>;
  static_assert(Cfg::kUnitM == kBN, "square tiles");

  __device__ void prefetch() const {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  __device__ int num_units() const { return static_cast<int>(plane_rows / h) * tiles; }
  // unit -> (matrix s, tile row mt, tile column nt)
  __device__ void decode(int u, int& s, int& mt, int& nt) const {
    s = u / tiles;
    const int r = u - s * tiles;
    if (tile_mode == kTriAll) {
      mt = r / T;
      nt = r - mt * T;
      return;
    }
    // r-th entry of the lower triangle in row order: row i holds i + 1 entries
    // (T is at most 128, so a walk down the rows is short)
    int i = 0, j = r;
    while (j > i) {
      ++i;
      j -= i;
    }
    mt = tile_mode == kTriLower ? i : j;
    nt = tile_mode == kTriLower ? j : i;
  }
  __device__ void k_range(int mt, int nt, int& lo, int& hi) const {
    lo = 0;
    hi = h;
    switch (k_mode) {
      case kKUpToN: hi = min(h, kBN * (nt + 1)); break;
      case kKUpToM: hi = min(h, kBN * (mt + 1)); break;
      case kKFromM: lo = kBN * mt; break;
      case kKFromN: lo = kBN * nt; break;
      default: break;
    }
  }
  __device__ int n_chunks(int u) const {
    int s, mt, nt, lo, hi;
    decode(u, s, mt, nt);
    k_range(mt, nt, lo, hi);
    return (hi - lo + kTriChunk - 1) / kTriChunk;
  }
  // Sub-tile sb = 6 c + j is term 5 - j of K chunk c, the six chained into one
  // accumulation, smallest first (as in SelGemmProb).
  __device__ int num_subtiles(int u) const { return 6 * n_chunks(u); }
  __device__ bool acc_continues(int, int sb) const { return sb % 6 != 0; }
  __device__ int num_kb(int u, int sb) const {
    int s, mt, nt, lo, hi;
    decode(u, s, mt, nt);
    k_range(mt, nt, lo, hi);
    const int c = sb / 6;
    return (min(kTriChunk, hi - lo - c * kTriChunk) + kBK - 1) / kBK;
  }
  struct Coords {
    int a_row, b_row, k0;
    int a_k0;  // kAMN: A's plane row of K offset k0 (a_row is then A's M offset)
  };
  __device__ Coords coords(int u, int sb, uint32_t rank) const {
    int s, mt, nt, lo, hi;
    decode(u, s, mt, nt);
    k_range(mt, nt, lo, hi);
    const int c = sb / 6, t = 5 - (sb - 6 * c);
    Coords r;
    const int m0 = mt * Cfg::kUnitM + static_cast<int>(rank) * kBM;
    const int a_block = static_cast<int>(sel_term_a(t) * plane_rows + static_cast<long long>(s) * h);
    r.a_row = kAMN ? m0 : a_block + m0;
    r.b_row = static_cast<int>(sel_term_b(t) * plane_rows + static_cast<long long>(s) * h +
                               static_cast<long long>(nt) * kBN + rank * Cfg::kBRows);
    r.k0 = lo + c * kTriChunk;
    if (kAMN) r.a_k0 = a_block + r.k0;
    return r;
  }
  __device__ void issue_loads(Coords& c, int kb, uint8_t* sa, uint8_t* sb, uint32_t bar) const {
    if constexpr (kAMN) load_operand<kBM, true, kPair>(sa, &tmA, bar, c.a_k0 + kb * kBK, c.a_row);
    else load_operand<kBM, false, kPair>(sa, &tmA, bar, c.k0 + kb * kBK, c.a_row);
    load_operand<Cfg::kBRows, false, kPair>(sb, &tmB, bar, c.k0 + kb * kBK, c.b_row);
  }
  __device__ void epilogue(EpiState& es, int, int sb, int, uint32_t tacc, int, int, uint32_t) const {
#pragma unroll
    for (int ch = 0; ch < kCols / 32; ++ch) {
      uint32_t v[32];
      tmem_ld32(tacc + ch * 32, v);
      tmem_wait_ld32(v);
#pragma unroll
      for (int i = 0; i < 32; ++i) es.rs[ch * 32 + i] = sb < 6 ? u2f(v[i]) : es.rs[ch * 32 + i] + u2f(v[i]);
    }
  }
  __device__ void epilogue_after(EpiState& es, int u, int sb, int nsub, int row, int col0, uint32_t rank) const {
    if (sb != nsub - 1) return;
    int s, mt, nt;
    decode(u, s, mt, nt);
    const long long m = static_cast<long long>(mt) * Cfg::kUnitM + rank * kBM + row;
    const long long n0 = static_cast<long long>(nt) * kBN + col0;
    float4* o = reinterpret_cast<float4*>(out + s * o_s + m * ldo + n0);
    const float4* cp = beta != 0.f ? reinterpret_cast<const float4*>(csrc + s * c_s + m * ldc + n0) : nullptr;
#pragma unroll
    for (int i = 0; i < kCols / 4; ++i) {
      float4 v = make_float4(alpha * es.rs[4 * i], alpha * es.rs[4 * i + 1], alpha * es.rs[4 * i + 2],
                             alpha * es.rs[4 * i + 3]);
      if (cp != nullptr) {
        const float4 c = cp[i];
        v.x = fmaf(beta, c.x, v.x);
        v.y = fmaf(beta, c.y, v.y);
        v.z = fmaf(beta, c.z, v.z);
        v.w = fmaf(beta, c.w, v.w);
      }
      o[i] = v;
    }
  }
};

// fp32 rows -> three bf16 planes: dst[j][r][col_off + c] for r < rows, c < cols
// (cols % 4 == 0); plane j at dst + j * plane_stride. With `tri`, the rows are
// stacked cols x cols lower-triangular matrices and row r stops at the end of its
// diagonal 256-column tile, c < 256 (⌊(r mod cols)/256⌋ + 1): the columns beyond are
// zeros that no product reads (SelGemmProb's b_tri).
__global__ void __launch_bounds__(256) k_split_rows(const float* __restrict__ src, long long ld_src,
                                                    __nv_bfloat16* __restrict__ dst, long long ld_dst, long long col_off,
                                                    long long plane_stride, long long rows, int cols, int tri) {
  const int per = cols / 4;
  const long long total = rows * per;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = i / per;
    const int c = static_cast<int>(i - r * per) * 4;
    if (tri && c >= kBN * (static_cast<int>(r % cols) / kBN + 1)) continue;
    const float4 v = __ldg(reinterpret_cast<const float4*>(src + r * ld_src + c));
    __nv_bfloat16 h[4], m[4], l[4];
    split3(v.x, h[0], m[0], l[0]);
    split3(v.y, h[1], m[1], l[1]);
    split3(v.z, h[2], m[2], l[2]);
    split3(v.w, h[3], m[3], l[3]);
    __nv_bfloat16* d = dst + r * ld_dst + col_off + c;
    *reinterpret_cast<uint2*>(d) = *reinterpret_cast<const uint2*>(h);
    *reinterpret_cast<uint2*>(d + plane_stride) = *reinterpret_cast<const uint2*>(m);
    *reinterpret_cast<uint2*>(d + 2 * plane_stride) = *reinterpret_cast<const uint2*>(l);
  }
}

// fp32 blocks -> three bf16 planes, one block per matrix b of a batch: the rows x cols
// block at src + b*s_src (ld ld_src) becomes rows b*rows_out .. of the planes (ld
// ld_dst), transposed when `tr` (rows_out = cols). Grid (cols/32, rows/32, batch),
// 32 x 8 threads; the transposed copy goes through a shared tile.
__global__ void __launch_bounds__(256) k_split_blocks(const float* __restrict__ src, long long ld_src, long long s_src,
                                                      int rows, int cols, __nv_bfloat16* __restrict__ dst,
                                                      long long ld_dst, long long plane_stride, int tr) {
  __shared__ float t[32][33];
  const int b = blockIdx.z;
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  const float* s = src + b * s_src;
  for (int j = threadIdx.y; j < 32; j += 8) t[j][threadIdx.x] = s[static_cast<long long>(r0 + j) * ld_src + c0 + threadIdx.x];
  __syncthreads();
  const long long rows_out = tr ? cols : rows;
  for (int j = threadIdx.y; j < 32; j += 8) {
    // untransposed: out[r0 + j][c0 + x] = t[j][x];  transposed: out[c0 + j][r0 + x] = t[x][j]
    const float v = tr ? t[threadIdx.x][j] : t[j][threadIdx.x];
    const long long orow = b * rows_out + (tr ? c0 + j : r0 + j);
    const long long ocol = tr ? r0 + threadIdx.x : c0 + threadIdx.x;
    __nv_bfloat16 h, m, l;
    split3(v, h, m, l);
    __nv_bfloat16* d = dst + orow * ld_dst + ocol;
    d[0] = h;
    d[plane_stride] = m;
    d[2 * plane_stride] = l;
  }
}

// The untransposed case, 4 elements per thread-step (cols % 4 == 0).
__global__ void __launch_bounds__(256) k_split_blocks_rows(const float* __restrict__ src, long long ld_src,
                                                           long long s_src, int rows, int cols,
                                                           __nv_bfloat16* __restrict__ dst, long long plane_stride,
                                                           int batch) {
  const int per = cols / 4;
  const long long total = static_cast<long long>(batch) * rows * per;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long br = i / per;  // b * rows + r
    const int c = static_cast<int>(i - br * per) * 4;
    const long long b = br / rows, r = br - b * rows;
    const float4 v = __ldg(reinterpret_cast<const float4*>(src + b * s_src + r * ld_src + c));
    __nv_bfloat16 h[4], m[4], l[4];
    split3(v.x, h[0], m[0], l[0]);
    split3(v.y, h[1], m[1], l[1]);
    split3(v.z, h[2], m[2], l[2]);
    split3(v.w, h[3], m[3], l[3]);
    __nv_bfloat16* d = dst + br * cols + c;
    *reinterpret_cast<uint2*>(d) = *reinterpret_cast<const uint2*>(h);
    *reinterpret_cast<uint2*>(d + plane_stride) = *reinterpret_cast<const uint2*>(m);
    *reinterpret_cast<uint2*>(d + 2 * plane_stride) = *reinterpret_cast<const uint2*>(l);
  }
}

// Per-kind inputs of one call.
struct SelKinds {
  const double* C[kSelMaxKinds];    // [n_targets][D][Ft] raw cross sums
  const double* syy[kSelMaxKinds];  // [n_targets][Ft]
  const double* mu_x[kSelMaxKinds];  // [D]   (workspace)
  const double* mu_y[kSelMaxKinds];  // [n_targets][Ft]
  const double* n[kSelMaxKinds];     // rows, as double
};

// Rᵀ of problem q = (kind, target t0 + g): RT[q][o][i] = C[t][i][o] − n μ_x[i] μ_t[o] in
// fp32, through 32 x 32 shared tiles. Grid (D/32, Ft/32, Q), 32 x 8 threads.
__global__ void __launch_bounds__(256) k_sel_init_rt(const __grid_constant__ SelKinds kinds, int t0, int G, int D,
                                                     int Ft, float* __restrict__ RT) {
  __shared__ float tile[32][33];
  const int q = blockIdx.z, kind = q / G, t = t0 + q % G;
  const int i0 = blockIdx.x * 32, o0 = blockIdx.y * 32;
  const double* C = kinds.C[kind] + static_cast<size_t>(t) * D * Ft;
  const double* mx = kinds.mu_x[kind];
  const double* my = kinds.mu_y[kind] + static_cast<size_t>(t) * Ft;
  const double nn = *kinds.n[kind];
  for (int j = threadIdx.y; j < 32; j += 8) {
    const int i = i0 + j, o = o0 + threadIdx.x;
    tile[j][threadIdx.x] = static_cast<float>(C[static_cast<size_t>(i) * Ft + o] - nn * mx[i] * my[o]);
  }
  __syncthreads();
  float* out = RT + static_cast<size_t>(q) * Ft * D;
  for (int j = threadIdx.y; j < 32; j += 8) out[static_cast<size_t>(o0 + j) * D + i0 + threadIdx.x] = tile[threadIdx.x][j];
}

// Σ[q][s] = H_kind[s block][s block] (F x F), and for every q its TSS and e = 0.
__global__ void __launch_bounds__(256) k_sel_init_sigma(const float* __restrict__ H, int G, int Q, int Ls, int F,
                                                        float* __restrict__ Sig) {
  const long long D = static_cast<long long>(Ls) * F;
  const long long per = static_cast<long long>(F) * F / 4;
  const long long total = static_cast<long long>(Q) * Ls * per;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long qs = i / per;
    const long long e = (i - qs * per) * 4;
    const int q = static_cast<int>(qs / Ls), s = static_cast<int>(qs - static_cast<long long>(q) * Ls);
    const long long r = e / F, c = e - r * F;
    const float* src = H + static_cast<long long>(q / G) * D * D + (s * static_cast<long long>(F) + r) * D +
                       s * static_cast<long long>(F) + c;
    *reinterpret_cast<float4*>(Sig + qs * F * F + e) = *reinterpret_cast<const float4*>(src);
  }
}

__global__ void __launch_bounds__(256) k_sel_init_tss(const __grid_constant__ SelKinds kinds, int t0, int G, int Q,
                                                      int Ft, double* __restrict__ tss, double* __restrict__ expl) {
  const long long total = static_cast<long long>(Q) * Ft;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int q = static_cast<int>(i / Ft), o = static_cast<int>(i - static_cast<long long>(q) * Ft);
    const int kind = q / G, t = t0 + q % G;
    const double mu = kinds.mu_y[kind][static_cast<size_t>(t) * Ft + o];
    tss[i] = kinds.syy[kind][static_cast<size_t>(t) * Ft + o] - (*kinds.n[kind]) * mu * mu;
    expl[i] = 0.0;
  }
}

// Σ[q][s] := I for every layer s already chosen for problem q's target. Grid
// (Ls, Q, 16): CTA z writes rows z*F/16 .. of the block, 4 floats per store.
__global__ void __launch_bounds__(256) k_sel_mask_identity(const uint8_t* __restrict__ mask, int G, int Ls, int F,
                                                           float* __restrict__ Sig) {
  const int q = blockIdx.y, s = blockIdx.x;
  if (!mask[(q % G) * Ls + s]) return;
  const int rows = F / 16, r0 = blockIdx.z * rows, per = F / 4;
  float* S = Sig + (static_cast<long long>(q) * Ls + s) * F * F;
  for (int e = threadIdx.x; e < rows * per; e += blockDim.x) {
    const int r = r0 + e / per, c = (e % per) * 4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r >= c && r < c + 4) (&v.x)[r - c] = 1.f;
    *reinterpret_cast<float4*>(S + static_cast<long long>(r) * F + c) = v;
  }
}

// Scores of every (target g, kind, layer s), one CTA each (grid n_kinds·Ls x G),
// a warp per head (heads beyond the warps taken in turn): gain_o = Σ partials of
// colsum(z_s²), score = mean_h (Σ_{o∈h}(e_o + gain_o)) / Σ_{o∈h} TSS_o (0 for a head
// without variance); a layer already chosen scores 0 and NaN in the table. The heads
// add in order, so with at most 8 heads the sums are those of one warp taking
// every head in turn.
__global__ void __launch_bounds__(256) k_sel_layer_scores(const float* __restrict__ part, int n_part, int G,
                                                          int n_kinds, int Ls, int Ft, int hd, int t0, int n_targets,
                                                          int k, int j, const double* __restrict__ tss,
                                                          const double* __restrict__ expl,
                                                          const uint8_t* __restrict__ mask, double* __restrict__ scores,
                                                          float* __restrict__ r2) {
  __shared__ double hs[8];
  const int ks = blockIdx.x, g = blockIdx.y, t = t0 + g;
  const int kind = ks / Ls, s = ks - kind * Ls, q = kind * G + g;
  const int nh = Ft / hd;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t r2i = ((static_cast<size_t>(kind) * n_targets + t) * k + j) * Ls + s;
  if (mask[g * Ls + s]) {
    if (threadIdx.x == 0) {
      scores[(static_cast<size_t>(g) * n_kinds + kind) * Ls + s] = 0.0;
      if (r2 != nullptr) r2[r2i] = nanf("");
    }
    return;
  }
  const float* pp = part + (static_cast<size_t>(q) * Ls + s) * Ft * n_part;
  double acc = 0.0;
  for (int h = warp; h < nh; h += 8) {
    double num = 0.0, den = 0.0;
    for (int o = h * hd + lane; o < (h + 1) * hd; o += 32) {
      double gsum = 0.0;
      for (int i = 0; i < n_part; ++i) gsum += static_cast<double>(pp[static_cast<size_t>(o) * n_part + i]);
      num += expl[static_cast<size_t>(q) * Ft + o] + gsum;
      den += tss[static_cast<size_t>(q) * Ft + o];
    }
    for (int off = 16; off > 0; off >>= 1) {
      num += __shfl_xor_sync(0xffffffffu, num, off);
      den += __shfl_xor_sync(0xffffffffu, den, off);
    }
    acc += den > 0.0 ? num / den : 0.0;
  }
  if (lane == 0) hs[warp] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double score = 0.0;
    for (int w = 0; w < 8 && w < nh; ++w) score += hs[w];
    score /= nh;
    scores[(static_cast<size_t>(g) * n_kinds + kind) * Ls + s] = score;
    if (r2 != nullptr) r2[r2i] = static_cast<float>(score);
  }
}

// One CTA per target g: the first layer not yet chosen with the highest joint
// score (the mean over kinds) is chosen; writes the choice, the mask and e += gain.
__global__ void __launch_bounds__(256) k_sel_choose(const double* __restrict__ scores, const float* __restrict__ part,
                                                    int n_part, int G, int n_kinds, int Ls, int Ft, int t0, int k,
                                                    int j, double* __restrict__ expl, uint8_t* __restrict__ mask,
                                                    int32_t* __restrict__ chosen, int32_t* __restrict__ sel) {
  const int g = blockIdx.x, t = t0 + g;
  const uint8_t* mk = mask + g * Ls;
  __shared__ int best_s;
  if (threadIdx.x == 0) {
    int best = -1;
    double bv = 0.0;
    for (int s = 0; s < Ls; ++s) {
      if (mk[s]) continue;
      double v = 0.0;
      for (int kind = 0; kind < n_kinds; ++kind) v += scores[(static_cast<size_t>(g) * n_kinds + kind) * Ls + s];
      v /= n_kinds;
      if (best < 0 || v > bv) {
        best = s;
        bv = v;
      }
    }
    best_s = best;
    sel[static_cast<size_t>(t) * k + j] = best;
    mask[g * Ls + best] = 1;
    for (int kind = 0; kind < n_kinds; ++kind) chosen[kind * G + g] = best;
  }
  __syncthreads();
  const int b = best_s;
  for (int i = threadIdx.x; i < n_kinds * Ft; i += blockDim.x) {
    const int kind = i / Ft, o = i - kind * Ft;
    const int q = kind * G + g;
    const float* pp = part + ((static_cast<size_t>(q) * Ls + b) * Ft + o) * n_part;
    double gsum = 0.0;
    for (int p = 0; p < n_part; ++p) gsum += static_cast<double>(pp[p]);
    expl[static_cast<size_t>(q) * Ft + o] += gsum;
  }
}

// X[q][i][f] = H_kind[i][b_q F + f]: the first block column of the factor's input.
// Written straight as the three bf16 planes Xp [3][Q*D][F] (plane stride Q*D*F).
__global__ void __launch_bounds__(256) k_sel_copy_hcols(const float* __restrict__ H, const int32_t* __restrict__ chosen,
                                                        int G, int Q, long long D, int F,
                                                        __nv_bfloat16* __restrict__ Xp) {
  const long long per = D * F / 4;
  const long long total = per * Q;
  const long long plane = total * 4;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int q = static_cast<int>(i / per);
    const long long e = (i - q * per) * 4;
    const long long r = e / F, c = e - r * F;
    const float* src = H + static_cast<long long>(q / G) * D * D + r * D + static_cast<long long>(chosen[q]) * F + c;
    const float4 v = *reinterpret_cast<const float4*>(src);
    __align__(8) __nv_bfloat16 h[4], m[4], l[4];
    split3(v.x, h[0], m[0], l[0]);
    split3(v.y, h[1], m[1], l[1]);
    split3(v.z, h[2], m[2], l[2]);
    split3(v.w, h[3], m[3], l[3]);
    __nv_bfloat16* d = Xp + static_cast<long long>(q) * D * F + e;
    *reinterpret_cast<uint2*>(d) = *reinterpret_cast<const uint2*>(h);
    *reinterpret_cast<uint2*>(d + plane) = *reinterpret_cast<const uint2*>(m);
    *reinterpret_cast<uint2*>(d + 2 * plane) = *reinterpret_cast<const uint2*>(l);
  }
}

// --------------------------------------------------------------------------
// Host side
// --------------------------------------------------------------------------
struct SelLayout {
  float* H;         // [n_kinds][D][D]
  double* mu_x;     // [n_kinds][D]
  double* mu_y;     // [n_kinds][n_targets][Ft]
  double* nn;       // [n_kinds]
  double* alpha;    // [n_kinds]
  __nv_bfloat16* Wp;  // [3][Qmax * D][m_max]
  float* Sig;       // [Qmax * Ls][F][F]  Schur blocks, kept across steps
  float* Lf;        // [Qmax * Ls][F][F]  a copy of Σ that the factorisation consumes
  float* Linv;      // [Qmax * Ls][F][F]
  __nv_bfloat16* Lp;  // [3][Qmax * Ls * F][F]
  float* ctmp;      // [Qmax * Ls][F * F / 4]
  __nv_bfloat16* fpa;  // [3][Qmax * Ls * F / 2][F / 2]  planes of the factorisation's products
  __nv_bfloat16* fpb;  // [3][Qmax * Ls * F / 2][F / 2]
  float* RT;        // [Qmax][Ft][D]
  __nv_bfloat16* RTp;  // [3][Qmax * Ft][D]
  float* part;      // [Qmax * Ls][Ft][2 F / 256]
  float* zb;        // [Qmax][Ft][F]
  __nv_bfloat16* zbp;  // [3][Qmax * Ft][F]
  __nv_bfloat16* Xp;  // [3][Qmax * D][F]  the new block column's planes
  double* tss;      // [Qmax][Ft]
  double* expl;     // [Qmax][Ft]
  double* scores;   // [Gmax][n_kinds][Ls] this step's layer scores
  int32_t* chosen;  // [Qmax]
  uint8_t* mask;    // [Gmax][Ls]
  int* sched;       // unit counter of the dynamically ordered products
  size_t bytes;
};

static int sel_group(const rf_select_desc* d) {
  return static_cast<int>(d->group > 0 ? std::min(d->group, d->n_targets) : d->n_targets);
}

static SelLayout sel_layout(const rf_select_desc* d, void* ws) {
  const long long Ls = d->L_src, F = d->F, D = Ls * F, Ft = d->d_out, NK = d->n_kinds;
  const long long Gm = sel_group(d), Q = NK * Gm;
  const long long m_max = (d->k - 1) * F;
  Carve c(ws);
  SelLayout l;
  l.H = c.take<float>(NK * D * D);
  l.mu_x = c.take<double>(NK * D);
  l.mu_y = c.take<double>(NK * d->n_targets * Ft);
  l.nn = c.take<double>(NK);
  l.alpha = c.take<double>(NK);
  l.Wp = c.take<__nv_bfloat16>(std::max<long long>(3 * Q * D * m_max, 1));
  l.Sig = c.take<float>(Q * Ls * F * F);
  l.Lf = c.take<float>(Q * Ls * F * F);
  l.Linv = c.take<float>(Q * Ls * F * F);
  l.Lp = c.take<__nv_bfloat16>(3 * Q * Ls * F * F);
  l.ctmp = c.take<float>(Q * Ls * F * F / 4);
  const long long fp = F % 512 == 0 ? 3 * Q * Ls * F * F / 4 : 1;
  l.fpa = c.take<__nv_bfloat16>(fp);
  l.fpb = c.take<__nv_bfloat16>(fp);
  l.RT = c.take<float>(Q * Ft * D);
  l.RTp = c.take<__nv_bfloat16>(3 * Q * Ft * D);
  l.part = c.take<float>(Q * Ls * Ft * 2 * (F / kBN));
  l.zb = c.take<float>(Q * Ft * F);
  l.zbp = c.take<__nv_bfloat16>(3 * Q * Ft * F);
  l.Xp = c.take<__nv_bfloat16>(3 * Q * D * F);
  l.tss = c.take<double>(Q * Ft);
  l.expl = c.take<double>(Q * Ft);
  l.scores = c.take<double>(Gm * NK * Ls);
  l.chosen = c.take<int32_t>(Q);
  l.mask = c.take<uint8_t>(Gm * Ls);
  l.sched = c.take<int>(1);
  l.bytes = c.bytes();
  return l;
}

static rf_status check_select_desc(const rf_select_desc* d) {
  if (d == nullptr) return fail(RF_ERR_INVALID_ARG, "desc is NULL");
  if (d->L_src <= 0 || d->F <= 0 || d->n_targets <= 0 || d->d_out <= 0 || d->head_dim <= 0 || d->k <= 0 ||
      d->group < 0)
    return fail(RF_ERR_INVALID_ARG, "need L_src, F, n_targets, d_out, head_dim, k > 0 and group >= 0");
  if (d->k > d->L_src) return fail(RF_ERR_INVALID_ARG, "k = %lld exceeds L_src = %lld", (long long)d->k,
                                   (long long)d->L_src);
  if (d->n_kinds != 1 && d->n_kinds != 2) return fail(RF_ERR_INVALID_ARG, "n_kinds must be 1 or 2");
  if (d->F % kBN != 0 || d->d_out % kBN != 0) return fail(RF_ERR_SHAPE, "F and d_out must be multiples of 256");
  if (d->d_out % d->head_dim != 0) return fail(RF_ERR_SHAPE, "d_out must be a multiple of head_dim");
  if (d->L_src * d->F > 65536) return fail(RF_ERR_SHAPE, "L_src * F must be <= 65536");
  if (d->n_targets > 65535) return fail(RF_ERR_SHAPE, "n_targets must be <= 65535");
  return RF_OK;
}

struct SelCtx {
  cudaStream_t s;
  int sms;
  int32_t* dev_status;
  bool pair;
  int factor_stage = RF_STAGE_SELECT_FACTOR;  // profiler stage of the factorisation's launches
  // A device int for the dynamic unit order of the products whose units differ in
  // length (triangle-skipping ones), or nullptr to deal them round-robin: with 76
  // pairs and 4 tile columns, round-robin gives every pair the same column, so the
  // longest column sets the launch's time.
  int* sched = nullptr;
};

static rf_status split_rows(SelCtx& c, const float* src, long long ld_src, __nv_bfloat16* dst, long long ld_dst,
                            long long col_off, long long plane_stride, long long rows, int cols, bool tri = false) {
  const long long total = rows * (cols / 4);
  const unsigned blocks = static_cast<unsigned>(std::min<long long>((total + 255) / 256, 8LL * c.sms));
  ProfScope prof(c.s, RF_STAGE_SELECT_SPLIT);
  k_split_rows<<<blocks, 256, 0, c.s>>>(src, ld_src, dst, ld_dst, col_off, plane_stride, rows, cols, tri ? 1 : 0);
  return cuda_check(cudaGetLastError(), "k_split_rows launch");
}

// One split product: operands are the planes at pa ([3][a_rows][a_kext]) and
// pb ([3][b_rows][b_kext]).
struct SelGemm {
  const __nv_bfloat16* pa;
  long long a_rows, a_kext;
  SelOperand a;
  const __nv_bfloat16* pb;
  long long b_rows, b_kext;
  SelOperand b;
  const int32_t* chosen = nullptr;
  int Q = 1, nS = 1, M = 0, N = 0, K = 0;
  float alpha = 1.f, beta = 0.f;
  float* out = nullptr;
  long long o_q = 0, o_s = 0, ldo = 0;
  const float* csrc = nullptr;
  long long c_kind = 0, c_b = 0, c_q = 0, c_s = 0, ldc = 0;
  int q_per_kind = 1;
  float* part = nullptr;
  __nv_bfloat16* po = nullptr;  // result as bf16 planes instead of `out`
  long long po_plane = 0, po_q = 0, po_ld = 0, po_col = 0;
  bool b_tri = false;  // B is an L^-1 (lower triangular in row, K): skip its zero K range
  bool m_inner = false;  // M tiles innermost in the unit order (N >> M)
  int skip = kSkipNone;  // which layer index marks a unit of an already chosen layer
  const uint8_t* mask = nullptr;
  int mask_g = 1, mask_ls = 1, layer_f = 1;
  int stage = RF_STAGE_SELECT_GEMM;  // profiler stage of the launch
};

template <bool kPair>
static rf_status run_sel_gemm(SelCtx& c, const SelGemm& g) {
  using Cfg = GemmCfg<kPair>;
  SelGemmProb<kPair> pr;
  rf_status st;
  if ((st = make_tmap_bf16_2d(&pr.tmA, g.pa, g.a_kext, 3 * g.a_rows, g.a_kext, kBK, kBM)) != RF_OK) return st;
  if ((st = make_tmap_bf16_2d(&pr.tmB, g.pb, g.b_kext, 3 * g.b_rows, g.b_kext, kBK, Cfg::kBRows)) != RF_OK) return st;
  pr.a = g.a;
  pr.b = g.b;
  pr.a.plane_rows = g.a_rows;
  pr.b.plane_rows = g.b_rows;
  pr.chosen = g.chosen;
  pr.Q = g.Q;
  pr.nS = g.nS;
  pr.M = g.M;
  pr.N = g.N;
  pr.K = g.K;
  pr.m_tiles = g.M / Cfg::kUnitM;
  pr.n_tiles = g.N / kBN;
  pr.n_chunks = (g.K + kSelChunk - 1) / kSelChunk;
  pr.alpha = g.alpha;
  pr.beta = g.beta;
  pr.out = g.out;
  pr.o_q = g.o_q;
  pr.o_s = g.o_s;
  pr.ldo = g.ldo;
  pr.csrc = g.csrc;
  pr.c_kind = g.c_kind;
  pr.c_b = g.c_b;
  pr.c_q = g.c_q;
  pr.c_s = g.c_s;
  pr.ldc = g.ldc;
  pr.q_per_kind = g.q_per_kind;
  pr.part = g.part;
  pr.po = g.po;
  pr.po_plane = g.po_plane;
  pr.po_q = g.po_q;
  pr.po_ld = g.po_ld;
  pr.po_col = g.po_col;
  pr.b_tri = g.b_tri ? 1 : 0;
  pr.m_inner = g.m_inner ? 1 : 0;
  pr.skip = g.mask != nullptr ? g.skip : kSkipNone;
  pr.mask = g.mask;
  pr.mask_g = g.mask_g;
  pr.mask_ls = g.mask_ls;
  pr.layer_f = g.layer_f;
  // Dynamic order wherever units differ in length (triangle skipping) or some run
  // nothing (chosen layers): dealt round-robin, the pairs that skip run ahead of
  // the ones reading the same operand tiles, and those tiles leave L2 between them.
  pr.sched = g.b_tri || g.mask != nullptr ? c.sched : nullptr;
  pr.dev_status = c.dev_status;
  pr.timeout_ns = wait_timeout_ns();
  ProfScope prof(c.s, g.stage);
  return launch_gemm(pr, static_cast<int64_t>(g.Q) * g.nS * pr.m_tiles * pr.n_tiles, c.sms, c.s,
                     "selection GEMM launch");
}

static rf_status sel_gemm(SelCtx& c, const SelGemm& g) {
  return c.pair ? run_sel_gemm<true>(c, g) : run_sel_gemm<false>(c, g);
}

static SelOperand op(long long q_rows, long long s_rows, long long b_rows, long long k0, long long s_k,
                     long long b_k);

// out_s = alpha · A_s B_sᵀ + beta · C_s for the batch's h x h blocks (planes pa, pb:
// [3][batch * h][h]) with the factors' triangles skipped (TriGemmProb); on single
// CTAs, or for h not a multiple of 256, the plain split product over every tile and K.
template <bool kAMN>
static rf_status tri_gemm_t(SelCtx& c, const __nv_bfloat16* pa, const __nv_bfloat16* pb, int batch, int h,
                            int tile_mode, int k_mode, float alpha, float beta, float* out, long long o_s,
                            long long ldo, const float* csrc, long long c_s, long long ldc, int stage) {
  const long long rows = static_cast<long long>(batch) * h;
  if (!c.pair || h % kBN != 0) {
    if (kAMN) return fail(RF_ERR_SHAPE, "MN-major factorisation product needs CTA pairs and h %% 256 == 0");
    SelGemm g{};
    g.pa = pa, g.a_rows = rows, g.a_kext = h, g.a = op(0, h, 0, 0, 0, 0);
    g.pb = pb, g.b_rows = rows, g.b_kext = h, g.b = op(0, h, 0, 0, 0, 0);
    g.nS = batch, g.M = h, g.N = h, g.K = h, g.stage = stage;
    g.alpha = alpha, g.beta = beta;
    g.out = out, g.o_s = o_s, g.ldo = ldo;
    g.csrc = csrc, g.c_s = c_s, g.ldc = ldc;
    return sel_gemm(c, g);
  }
  using Cfg = GemmCfg<true>;
  TriGemmProb<kAMN> pr;
  rf_status st;
  if ((st = make_tmap_bf16_2d(&pr.tmA, pa, h, 3 * rows, h, kAMN ? 64 : kBK, kAMN ? kBK : kBM)) != RF_OK) return st;
  if ((st = make_tmap_bf16_2d(&pr.tmB, pb, h, 3 * rows, h, kBK, Cfg::kBRows)) != RF_OK) return st;
  pr.plane_rows = rows;
  pr.h = h;
  pr.T = h / kBN;
  pr.tiles = tile_mode == kTriAll ? pr.T * pr.T : pr.T * (pr.T + 1) / 2;
  pr.tile_mode = tile_mode;
  pr.k_mode = k_mode;
  pr.alpha = alpha;
  pr.beta = beta;
  pr.out = out;
  pr.o_s = o_s;
  pr.ldo = ldo;
  pr.csrc = csrc;
  pr.c_s = c_s;
  pr.ldc = ldc;
  pr.sched = c.sched;
  pr.dev_status = c.dev_status;
  pr.timeout_ns = wait_timeout_ns();
  ProfScope prof(c.s, stage);
  return launch_gemm(pr, static_cast<int64_t>(batch) * pr.tiles, c.sms, c.s, "factorisation product launch");
}

static rf_status tri_gemm(SelCtx& c, const __nv_bfloat16* pa, const __nv_bfloat16* pb, int batch, int h,
                          int tile_mode, int k_mode, float alpha, float beta, float* out, long long o_s,
                          long long ldo, const float* csrc, long long c_s, long long ldc, int stage) {
  return tri_gemm_t<false>(c, pa, pb, batch, h, tile_mode, k_mode, alpha, beta, out, o_s, ldo, csrc, c_s, ldc, stage);
}

static SelOperand op(long long q_rows, long long s_rows, long long b_rows, long long k0, long long s_k,
                     long long b_k) {
  SelOperand o;
  o.plane_rows = 0;
  o.q_rows = q_rows;
  o.s_rows = s_rows;
  o.b_rows = b_rows;
  o.k0 = k0;
  o.s_k = s_k;
  o.b_k = b_k;
  return o;
}

// Scratch of the factorisation: ctmp [batch][n/2][n/2] fp32, fpa and fpb
// [3][batch * n/2][n/2] bf16 each (only for widths that are multiples of 512).
struct FactorScratch {
  float* ctmp;
  __nv_bfloat16* fpa;
  __nv_bfloat16* fpb;
};

static rf_status split_blocks(SelCtx& c, const float* src, long long ld_src, long long s_src, int rows, int cols,
                              int batch, __nv_bfloat16* dst, bool tr) {
  const long long rows_out = tr ? cols : rows;
  const long long ld_dst = tr ? rows : cols;
  ProfScope prof(c.s, c.factor_stage);
  if (tr) {
    k_split_blocks<<<dim3(cols / 32, rows / 32, batch), dim3(32, 8), 0, c.s>>>(src, ld_src, s_src, rows, cols, dst,
                                                                               ld_dst, rows_out * batch * ld_dst, 1);
  } else {
    const long long total = static_cast<long long>(batch) * rows * (cols / 4);
    const unsigned blocks = static_cast<unsigned>(std::min<long long>((total + 255) / 256, 8LL * c.sms));
    k_split_blocks_rows<<<blocks, 256, 0, c.s>>>(src, ld_src, s_src, rows, cols, dst, rows_out * batch * ld_dst, batch);
  }
  return cuda_check(cudaGetLastError(), "block split launch");
}

// W = L^-1 for a batch of n x n SPD blocks (matrix b at A + b*sA, W + b*sW; A is
// consumed), W zero above the diagonal on entry. Widths that are multiples of 512
// split in halves with the four products on the tensor cores (fp32-accurate split
// bf16): with W11 = L11^-1 from the first half,
//   L21 = A21 W11ᵀ,  A22 −= L21 L21ᵀ,  Tᵀ = W11ᵀ L21ᵀ (into A21's storage),
//   then W22 = L22^-1 from the second half and W21 = −W22 T.
// Other widths run the fp32 SIMT recursion (chol_inv_block).
static rf_status sel_factor(SelCtx& c, const FactorScratch& lay, float* A, long long lda, long long sA, float* W,
                            long long ldw, long long sW, int n, int batch, long long stmp) {
  rf_status st;
  // A single matrix's nodes below 2,048 (products of at most 512³, a few tiles each)
  // run faster as SIMT products (64-tile k_sgemm64) than as ten launches of plane
  // splits and tensor-core GEMMs: the solve's factorisation stage at d = 4,096 and
  // 8,192 took 5.7 and 11.2 ms this way, 5.9 and 11.6 ms with SIMT below 1,024 only,
  // 5.8 and 11.4 ms with SIMT below 4,096.
  if (n % 512 != 0 || (batch == 1 && n < 2048)) {
    ProfScope prof(c.s, c.factor_stage);
    return chol_inv_block(A, lda, sA, W, ldw, sW, n, batch, lay.ctmp, stmp, c.dev_status, c.sms, c.s);
  }
  const int h = n / 2;
  float* A21 = A + static_cast<long long>(h) * lda;
  float* A22 = A21 + h;
  float* W21 = W + static_cast<long long>(h) * ldw;
  float* W22 = W21 + h;
  float* L21 = lay.ctmp;  // [batch][h][h]
  const long long hh = static_cast<long long>(h) * h;
  if ((st = sel_factor(c, lay, A, lda, sA, W, ldw, sW, h, batch, stmp)) != RF_OK) return st;
  const int fs = c.factor_stage;
  // L21 = A21 W11ᵀ (W11 lower triangular: k <= n)
  if ((st = split_blocks(c, A21, lda, sA, h, h, batch, lay.fpa, false)) != RF_OK) return st;
  if ((st = split_blocks(c, W, ldw, sW, h, h, batch, lay.fpb, false)) != RF_OK) return st;
  if ((st = tri_gemm(c, lay.fpa, lay.fpb, batch, h, kTriAll, kKUpToN, 1.f, 0.f, L21, hh, h, nullptr, 0, 0, fs)) !=
      RF_OK)
    return st;
  // A22 −= L21 L21ᵀ (only the tiles on and below the diagonal are read later)
  if ((st = split_blocks(c, L21, h, hh, h, h, batch, lay.fpa, false)) != RF_OK) return st;
  if ((st = tri_gemm(c, lay.fpa, lay.fpa, batch, h, kTriLower, kKAll, -1.f, 1.f, A22, sA, lda, A22, sA, lda, fs)) !=
      RF_OK)
    return st;
  // Tᵀ = W11ᵀ L21ᵀ, kept in A21's storage (W11ᵀ's row m is zero below k = m). On the
  // triangle-skipping kernel W11ᵀ is read MN-major from W11's planes, still in fpb
  // from L21's product; otherwise W11 is split again, transposed.
  if (c.pair && h % kBN == 0) {
    if ((st = tri_gemm_t<true>(c, lay.fpb, lay.fpa, batch, h, kTriAll, kKFromM, 1.f, 0.f, A21, sA, lda, nullptr, 0,
                               0, fs)) != RF_OK)
      return st;
  } else {
    if ((st = split_blocks(c, W, ldw, sW, h, h, batch, lay.fpb, true)) != RF_OK) return st;
    if ((st = tri_gemm(c, lay.fpb, lay.fpa, batch, h, kTriAll, kKFromM, 1.f, 0.f, A21, sA, lda, nullptr, 0, 0, fs)) !=
        RF_OK)
      return st;
  }
  if ((st = sel_factor(c, lay, A22, lda, sA, W22, ldw, sW, h, batch, stmp)) != RF_OK) return st;
  // W21 = −W22 T (W22 lower triangular: k <= m)
  if ((st = split_blocks(c, W22, ldw, sW, h, h, batch, lay.fpa, false)) != RF_OK) return st;
  if ((st = split_blocks(c, A21, lda, sA, h, h, batch, lay.fpb, false)) != RF_OK) return st;
  return tri_gemm(c, lay.fpa, lay.fpb, batch, h, kTriAll, kKUpToM, -1.f, 0.f, W21, sW, ldw, nullptr, 0, 0, fs);
}

// H = L Lᵀ (n x n SPD, n % 128 == 0, consumed): Linv = L^-1 and, when Hinv is set,
// Hinv = Linvᵀ Linv = H^-1 as one split tensor-core product of Linvᵀ with itself,
// its upper triangle then mirrored so that Hinv is exactly symmetric.
__global__ void __launch_bounds__(256) k_mirror_upper_f32(float* __restrict__ M, int n) {
  const int bx = blockIdx.x, by = blockIdx.y;  // block (bx, by) writes rows by*32.., columns bx*32..
  if (bx > by) return;
  __shared__ float t[32][33];
  for (int j = threadIdx.y; j < 32; j += 8) t[j][threadIdx.x] = M[static_cast<size_t>(bx * 32 + j) * n + by * 32 + threadIdx.x];
  __syncthreads();
  for (int j = threadIdx.y; j < 32; j += 8) {
    const int i = by * 32 + j, c = bx * 32 + threadIdx.x;
    if (i > c) M[static_cast<size_t>(i) * n + c] = t[threadIdx.x][j];
  }
}

rf_status spd_inverse(float* H, int n, float* Linv, float* Hinv, float* ctmp, __nv_bfloat16* planes, bool pair,
                      int32_t* dev_status, int sms, cudaStream_t s) {
  SelCtx c{s, sms, dev_status, pair, RF_STAGE_SOLVE};
  rf_status st;
  if ((st = cuda_check(cudaMemsetAsync(Linv, 0, sizeof(float) * n * n, s), "zero L^-1")) != RF_OK) return st;
  const long long q = 3LL * n * n / 4;  // one plane set of the factorisation's products
  if ((st = sel_factor(c, FactorScratch{ctmp, planes, planes + q}, H, n, 0, Linv, n, 0, n, 1,
                       static_cast<long long>(n) * n / 4)) != RF_OK)
    return st;
  if (Hinv == nullptr) return RF_OK;
  if ((st = split_blocks(c, Linv, n, 0, n, n, 1, planes, true)) != RF_OK) return st;
  // the tiles on and above the diagonal, k >= the column tile (L^-1 is lower triangular)
  if ((st = tri_gemm(c, planes, planes, 1, n, kTriUpper, kKFromN, 1.f, 0.f, Hinv, 0, n, nullptr, 0, 0,
                     RF_STAGE_SOLVE)) != RF_OK)
    return st;
  k_mirror_upper_f32<<<dim3(n / 32, n / 32), dim3(32, 8), 0, s>>>(Hinv, n);
  return cuda_check(cudaGetLastError(), "k_mirror_upper_f32 launch");
}

}  // namespace rf

using namespace rf;

extern "C" size_t rf_select_workspace_bytes(const rf_select_desc* desc) {
  if (check_select_desc(desc) != RF_OK) return 0;
  return sel_layout(desc, nullptr).bytes;
}

extern "C" rf_status rf_select_sources(const rf_select_desc* desc, const rf_calib_stats* stats, double lambda,
                                       int alpha_mode, int32_t* src_layers, float* r2, int32_t* dev_status,
                                       void* workspace, size_t workspace_bytes, rf_stream_t stream) {
  clear_error();
  rf_status st = check_select_desc(desc);
  if (st != RF_OK) return st;
  if (alpha_mode != RF_ALPHA_TRACE && alpha_mode != RF_ALPHA_ABSOLUTE)
    return fail(RF_ERR_INVALID_ARG, "alpha_mode must be RF_ALPHA_TRACE or RF_ALPHA_ABSOLUTE");
  if (!(lambda >= 0.0)) return fail(RF_ERR_INVALID_ARG, "need lambda >= 0");
  if (stats == nullptr || src_layers == nullptr) return fail(RF_ERR_INVALID_ARG, "stats and src_layers must be non-NULL");
  for (int kind = 0; kind < desc->n_kinds; ++kind) {
    const rf_calib_stats& k = stats[kind];
    if (!k.G || !k.C || !k.sx || !k.sy || !k.n || !k.syy)
      return fail(RF_ERR_INVALID_ARG, "stats[%d]: G, C, sx, sy, n and syy must be non-NULL", kind);
  }
  SelLayout lay = sel_layout(desc, workspace);
  if (workspace == nullptr || workspace_bytes < lay.bytes || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(RF_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned (got %zu)", lay.bytes, workspace_bytes);
  int sms = 0;
  if ((st = current_device(&sms)) != RF_OK) return st;
  SelCtx c{static_cast<cudaStream_t>(stream), sms, dev_status, use_pair(desc->flags, true)};
  c.sched = lay.sched;

  const int Ls = static_cast<int>(desc->L_src), F = static_cast<int>(desc->F), Ft = static_cast<int>(desc->d_out);
  const int NK = static_cast<int>(desc->n_kinds), T = static_cast<int>(desc->n_targets), K = static_cast<int>(desc->k);
  const int hd = static_cast<int>(desc->head_dim);
  const long long D = static_cast<long long>(Ls) * F;
  const long long m_max = static_cast<long long>(K - 1) * F;
  const int Gm = sel_group(desc);
  const int n_part = 2 * (F / kBN);
  const int eb = 8 * sms;

  SelKinds kinds{};
  {
    ProfScope pf(c.s, RF_STAGE_SELECT_SCORE);
    for (int kind = 0; kind < NK; ++kind) {
      const rf_calib_stats& k = stats[kind];
      if ((st = centre_system(k.G, k.sx, k.sy, k.n, static_cast<int>(D), static_cast<long long>(T) * Ft, lambda,
                              alpha_mode, lay.mu_x + kind * D, lay.mu_y + static_cast<long long>(kind) * T * Ft,
                              lay.nn + kind, lay.alpha + kind, nullptr, nullptr, lay.H + kind * D * D, sms, c.s)) !=
          RF_OK)
        return st;
      kinds.C[kind] = k.C;
      kinds.syy[kind] = k.syy;
      kinds.mu_x[kind] = lay.mu_x + kind * D;
      kinds.mu_y[kind] = lay.mu_y + static_cast<long long>(kind) * T * Ft;
      kinds.n[kind] = lay.nn + kind;
    }
  }
  for (int t0 = 0; t0 < T; t0 += Gm) {
    const int G = std::min(Gm, T - t0), Q = NK * G;
    {
      ProfScope pf(c.s, RF_STAGE_SELECT_SCORE);
      k_sel_init_rt<<<dim3(static_cast<unsigned>(D / 32), static_cast<unsigned>(Ft / 32), Q), dim3(32, 8), 0, c.s>>>(
          kinds, t0, G, static_cast<int>(D), Ft, lay.RT);
      k_sel_init_sigma<<<eb, 256, 0, c.s>>>(lay.H, G, Q, Ls, F, lay.Sig);
      k_sel_init_tss<<<eb, 256, 0, c.s>>>(kinds, t0, G, Q, Ft, lay.tss, lay.expl);
      if ((st = cuda_check(cudaMemsetAsync(lay.mask, 0, static_cast<size_t>(G) * Ls, c.s), "mask reset")) != RF_OK)
        return st;
      if ((st = cuda_check(cudaGetLastError(), "selection set-up launches")) != RF_OK) return st;
    }
    const long long lrows = static_cast<long long>(Q) * Ls * F;  // rows of the L^-1 planes
    const long long rtrows = static_cast<long long>(Q) * Ft;     // rows of the Rᵀ planes
    const long long wrows = static_cast<long long>(Q) * D;       // rows of the W and X planes
    for (int j = 0; j < K; ++j) {
      const long long m = static_cast<long long>(j) * F;
      {
        ProfScope pf(c.s, RF_STAGE_SELECT_FACTOR);
        if (j > 0) k_sel_mask_identity<<<dim3(Ls, Q, 16), 256, 0, c.s>>>(lay.mask, G, Ls, F, lay.Sig);
        if ((st = cuda_check(cudaMemcpyAsync(lay.Lf, lay.Sig, sizeof(float) * Q * Ls * F * F,
                                             cudaMemcpyDeviceToDevice, c.s),
                             "Schur block copy")) != RF_OK)
          return st;
        if ((st = cuda_check(cudaMemsetAsync(lay.Linv, 0, sizeof(float) * Q * Ls * F * F, c.s), "zero L^-1")) != RF_OK)
          return st;
      }
      if ((st = sel_factor(c, FactorScratch{lay.ctmp, lay.fpa, lay.fpb}, lay.Lf, F, static_cast<long long>(F) * F,
                           lay.Linv, F, static_cast<long long>(F) * F, F, Q * Ls, static_cast<long long>(F) * F / 4)) !=
          RF_OK)
        return st;
      // L^-1 up to each row's diagonal tile: the products read no further (b_tri)
      if ((st = split_rows(c, lay.Linv, F, lay.Lp, F, 0, lrows * F, lrows, F, true)) != RF_OK) return st;
      if ((st = split_rows(c, lay.RT, D, lay.RTp, D, 0, rtrows * D, rtrows, static_cast<int>(D))) != RF_OK) return st;
      // colsum(z_s²) for every (q, s): z_sᵀ = R_sᵀ L_s^-ᵀ
      {
        SelGemm g{};
        g.pa = lay.RTp, g.a_rows = rtrows, g.a_kext = D, g.a = op(Ft, 0, 0, 0, F, 0);
        g.pb = lay.Lp, g.b_rows = lrows, g.b_kext = F, g.b = op(static_cast<long long>(Ls) * F, F, 0, 0, 0, 0);
        g.Q = Q, g.nS = Ls, g.M = Ft, g.N = F, g.K = F, g.b_tri = true;
        g.mask = lay.mask, g.mask_g = G, g.mask_ls = Ls, g.layer_f = F, g.skip = kSkipSlot;
        g.part = lay.part;
        if ((st = sel_gemm(c, g)) != RF_OK) return st;
      }
      {
        ProfScope pf(c.s, RF_STAGE_SELECT_SCORE);
        k_sel_layer_scores<<<dim3(static_cast<unsigned>(NK * Ls), static_cast<unsigned>(G)), 256, 0, c.s>>>(
            lay.part, n_part, G, NK, Ls, Ft, hd, t0, T, K, j, lay.tss, lay.expl, lay.mask, lay.scores, r2);
        k_sel_choose<<<G, 256, 0, c.s>>>(lay.scores, lay.part, n_part, G, NK, Ls, Ft, t0, K, j, lay.expl, lay.mask,
                                         lay.chosen, src_layers);
        if ((st = cuda_check(cudaGetLastError(), "score launches")) != RF_OK) return st;
      }
      if (j == K - 1) break;
      // z_bᵀ = R_bᵀ L_b^-ᵀ
      {
        SelGemm g{};
        g.pa = lay.RTp, g.a_rows = rtrows, g.a_kext = D, g.a = op(Ft, 0, 0, 0, 0, F);
        g.pb = lay.Lp, g.b_rows = lrows, g.b_kext = F, g.b = op(static_cast<long long>(Ls) * F, 0, F, 0, 0, 0);
        g.chosen = lay.chosen, g.Q = Q, g.M = Ft, g.N = F, g.K = F, g.b_tri = true;
        g.out = lay.zb, g.o_q = static_cast<long long>(Ft) * F, g.ldo = F;
        if ((st = sel_gemm(c, g)) != RF_OK) return st;
      }
      if ((st = split_rows(c, lay.zb, F, lay.zbp, F, 0, rtrows * F, rtrows, F)) != RF_OK) return st;
      // X = H[:, b] − W W_bᵀ, written as its planes Xp
      if (j == 0) {
        ProfScope pf(c.s, RF_STAGE_SELECT_SCORE);
        k_sel_copy_hcols<<<eb, 256, 0, c.s>>>(lay.H, lay.chosen, G, Q, D, F, lay.Xp);
        if ((st = cuda_check(cudaGetLastError(), "k_sel_copy_hcols launch")) != RF_OK) return st;
      } else {
        SelGemm g{};
        g.pa = lay.Wp, g.a_rows = wrows, g.a_kext = m_max, g.a = op(D, 0, 0, 0, 0, 0);
        g.pb = lay.Wp, g.b_rows = wrows, g.b_kext = m_max, g.b = op(D, 0, F, 0, 0, 0);
        g.chosen = lay.chosen, g.Q = Q, g.M = static_cast<int>(D), g.N = F, g.K = static_cast<int>(m);
        g.mask = lay.mask, g.mask_g = G, g.mask_ls = Ls, g.layer_f = F, g.skip = kSkipMRows;
        g.alpha = -1.f, g.beta = 1.f;
        g.po = lay.Xp, g.po_plane = wrows * F, g.po_q = D * F, g.po_ld = F, g.po_col = 0;
        g.csrc = lay.H, g.c_kind = D * D, g.c_b = F, g.ldc = D, g.q_per_kind = G;
        if ((st = sel_gemm(c, g)) != RF_OK) return st;
      }
      // w = X L_b^-ᵀ  (the new block column of every layer), written into the W planes
      {
        SelGemm g{};
        g.pa = lay.Xp, g.a_rows = wrows, g.a_kext = F, g.a = op(D, 0, 0, 0, 0, 0);
        g.pb = lay.Lp, g.b_rows = lrows, g.b_kext = F, g.b = op(static_cast<long long>(Ls) * F, 0, F, 0, 0, 0);
        g.chosen = lay.chosen, g.Q = Q, g.M = static_cast<int>(D), g.N = F, g.K = F, g.b_tri = true;
        g.mask = lay.mask, g.mask_g = G, g.mask_ls = Ls, g.layer_f = F, g.skip = kSkipMRows;
        g.po = lay.Wp, g.po_plane = wrows * m_max, g.po_q = D * m_max, g.po_ld = m_max, g.po_col = m;
        if ((st = sel_gemm(c, g)) != RF_OK) return st;
      }
      // Σ_s −= w_s w_sᵀ for every (q, s)
      {
        SelGemm g{};
        g.pa = lay.Wp, g.a_rows = wrows, g.a_kext = m_max, g.a = op(D, F, 0, m, 0, 0);
        g.pb = lay.Wp, g.b_rows = wrows, g.b_kext = m_max, g.b = op(D, F, 0, m, 0, 0);
        g.Q = Q, g.nS = Ls, g.M = F, g.N = F, g.K = F;
        g.mask = lay.mask, g.mask_g = G, g.mask_ls = Ls, g.layer_f = F, g.skip = kSkipSlot;
        g.alpha = -1.f, g.beta = 1.f;
        g.out = lay.Sig, g.o_q = static_cast<long long>(Ls) * F * F, g.o_s = static_cast<long long>(F) * F, g.ldo = F;
        g.csrc = lay.Sig, g.c_q = static_cast<long long>(Ls) * F * F, g.c_s = static_cast<long long>(F) * F,
        g.ldc = F;
        if ((st = sel_gemm(c, g)) != RF_OK) return st;
      }
      // Rᵀ −= z_bᵀ wᵀ
      {
        SelGemm g{};
        g.pa = lay.zbp, g.a_rows = rtrows, g.a_kext = F, g.a = op(Ft, 0, 0, 0, 0, 0);
        g.pb = lay.Wp, g.b_rows = wrows, g.b_kext = m_max, g.b = op(D, 0, 0, m, 0, 0);
        g.Q = Q, g.M = Ft, g.N = static_cast<int>(D), g.K = F, g.m_inner = true;
        g.mask = lay.mask, g.mask_g = G, g.mask_ls = Ls, g.layer_f = F, g.skip = kSkipNCols;
        g.alpha = -1.f, g.beta = 1.f;
        g.out = lay.RT, g.o_q = static_cast<long long>(Ft) * D, g.ldo = D;
        g.csrc = lay.RT, g.c_q = static_cast<long long>(Ft) * D, g.ldc = D;
        if ((st = sel_gemm(c, g)) != RF_OK) return st;
      }
    }
  }
  return RF_OK;
}
