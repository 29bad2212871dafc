// Calibration statistics (rf_calib_accumulate).
//
// [RF] RidgeFill review, "Ridge map": calibration only accumulates XᵀX, XᵀY_l and
// the two means in one pass, so a new λ needs only a re-solve. [XM] per-head
// ridge regression: computing XᵀX is the dominant fitting cost.
//
//   tc_gemm<GramProb>  G += XᵀX and C_p += XᵀY_p on the tensor cores. X and Y are
//                      row-major (samples x features), so both operands are
//                      MN-major tiles of the same rows. Each output tile's K-loop
//                      (the rows) is cut into chunks of kCalibChunk rows; a chunk
//                      is summed in fp32 in TMEM, so the tensor cores never sum
//                      more than kCalibChunk rows. Eight epilogue warps add the
//                      chunk blocks into fp32 running sums in registers and flush
//                      them into the fp64 totals every 16 chunks, with fp64
//                      reductions over whole row segments.
//   k_colsum           Σx, Σy_p, optionally Σy_p² (fp32 over 64 rows, fp64 across)
//                      and n += rows.
#include <algorithm>

#include "rf_host.h"
#include "tc_gemm.cuh"

namespace rf {

// Rows summed in fp32 on the tensor cores before the fp64 add. The accumulator's
// additions truncate: measured on a GB300, the relative bias of a Gram diagonal
// grows linearly with the chunk (-1.9e-6 at 1024 rows, -1.0e-5 at 4096, -1.3e-4
// at 32768), so 1024 keeps it 5x under the 1e-5 tolerance.
#ifndef RF_CALIB_CHUNK
#define RF_CALIB_CHUNK 1024
#endif
constexpr int kCalibChunk = RF_CALIB_CHUNK;
static_assert(kCalibChunk % 64 == 0, "calibration chunk must be a multiple of the K block");

template <bool kPair_>
struct GramProb {
  CUtensorMap tmX;  // X  {d_in, n_rows}, box {64, 64}
  CUtensorMap tmY;  // Y  {d_out, n_rows, P}, box {64, 64, 1}
  double* G;        // [d_in][d_in]
  double* C;        // [P][d_in][d_out]
  int d_in, d_out, P, n_rows, n_chunks;
  int g_mt, g_nt, c_nt, g_units;
  int c_group;  // M-tiles per group of the XᵀY units (their X rows stay in L2 together)
  int* sched;   // unit counter (dynamic unit order) when the caller gave a workspace, else nullptr
  int32_t* dev_status;
  uint64_t timeout_ns;
  static constexpr bool kAMN = true;
  static constexpr bool kBMN = true;
  static constexpr bool kPair = kPair_;
  static constexpr int kEpiWarps = 8;
  static constexpr int kCols = kBN / 2;      // columns per epilogue thread
  static constexpr int kFlushChunks = 16;    // row chunks per fp64 flush
  struct EpiState {
    float rs[kCols];
  };
  using Cfg = GemmCfg<kPair_>;

  __device__ void prefetch() const {
    tma_prefetch_desc(&tmX);
    if (P > 0) tma_prefetch_desc(&tmY);
  }
  __device__ int num_units() const { return g_units + P * g_mt * c_nt; }
  __device__ int num_subtiles(int) const { return n_chunks; }
  __device__ int num_kb(int, int sb) const {
    const int rows = min(kCalibChunk, n_rows - sb * kCalibChunk);
    return (rows + kBK - 1) / kBK;
  }
  // Unit order: the Gram tiles, then for every map p its N-tiles with the
  // M-tiles fastest, so the CTAs in flight share one strip of Y_p.
  __device__ void decode(int u, bool& is_g, int& p, int& mt, int& nt) const {
    if (u < g_units) {
      // Gram tiles on or above the diagonal only, column tile nt holding the
      // (nt + 1) * r row tiles that reach it (r = 256 / kUnitM), M fastest:
      // tiles before column nt number r * nt (nt + 1) / 2.
      constexpr int rr = kBN / Cfg::kUnitM;
      is_g = true;
      p = 0;
      int c = static_cast<int>((sqrtf(8.0f * static_cast<float>(u) / rr + 1.0f) - 1.0f) * 0.5f);
      while (rr * (c + 1) * (c + 2) / 2 <= u) ++c;
      while (rr * c * (c + 1) / 2 > u) --c;
      nt = c;
      mt = u - rr * c * (c + 1) / 2;
    } else {
      // XᵀY units in groups of c_group M-tiles: a group's X rows serve every map
      // and N-tile (map, then N-tile, then the group's M-tiles fastest) before the
      // next group starts, so they stay in L2 while the Y strips stream past.
      is_g = false;
      u -= g_units;
      const int full = c_group * c_nt * P;  // units of a whole group
      const int gi = u / full;
      const int m0 = gi * c_group;
      const int gs = min(c_group, g_mt - m0);  // this group's M-tiles
      const int r0 = u - gi * full;
      const int per = gs * c_nt;
      p = r0 / per;
      const int r = r0 - p * per;
      nt = r / gs;
      mt = m0 + (r - nt * gs);
    }
  }
  struct Coords {
    bool is_g;
    int p, m0, n0, row0;
  };
  __device__ Coords coords(int u, int sb, uint32_t rank) const {
    Coords c;
    int mt, nt;
    decode(u, c.is_g, c.p, mt, nt);
    c.m0 = mt * Cfg::kUnitM + static_cast<int>(rank) * kBM;
    c.n0 = nt * kBN + static_cast<int>(rank) * Cfg::kBRows;
    c.row0 = sb * kCalibChunk;
    return c;
  }
  __device__ void issue_loads(Coords& c, int kb, uint8_t* sa, uint8_t* sbuf, uint32_t bar) const {
    const int row = c.row0 + kb * kBK;
    load_operand<kBM, true, kPair>(sa, &tmX, bar, row, c.m0);
    if (c.is_g) {
      load_operand<Cfg::kBRows, true, kPair>(sbuf, &tmX, bar, row, c.n0);
    } else {
#pragma unroll
      for (int j = 0; j < Cfg::kBRows / 64; ++j)
        tma3<kPair>(sbuf + j * (64 * kBK * 2), &tmY, bar, c.n0 + 64 * j, row, c.p);
    }
  }
  // Each thread owns one row and 128 columns of the unit (8 epilogue warps) and
  // adds every row chunk's fp32 block into fp32 running sums in registers; every
  // kFlushChunks chunks, and at the unit's last chunk, it adds them into the fp64
  // sums in memory. The fp32 running sum over at most 16 chunk partials adds a
  // relative error of at most 16 * 2^-24 (about 1e-6) of sqrt(G_ii G_jj), and
  // the read-modify-write traffic on G and C falls 16-fold against a flush per chunk.
  __device__ void epilogue(EpiState& es, int, int sb, int, uint32_t tacc, int, int, uint32_t) const {
    const bool first = (sb % kFlushChunks) == 0;
#pragma unroll
    for (int ch = 0; ch < kCols / 32; ++ch) {
      uint32_t v[32];
      tmem_ld32(tacc + ch * 32, v);
      tmem_wait_ld32(v);
#pragma unroll
      for (int q = 0; q < 32; ++q) es.rs[ch * 32 + q] = first ? u2f(v[q]) : es.rs[ch * 32 + q] + u2f(v[q]);
    }
  }
  // The flush runs after the accumulator is handed back, overlapping the MMAs of
  // the next chunks. Each warp turns its 32 rows x 16 columns around through shared
  // memory, so that its fp64 reductions cover whole 128-byte row segments, and
  // nothing is read back: a read-modify-write of the totals, one thread per row,
  // waited on its loads for longer than the next unit's MMAs (measured: the 27B-
  // shaped Gram GEMM took 29.8 ms that way, 25.3 ms this way). (Static shared
  // memory, on top of the GEMM stages.)
  __device__ void epilogue_after(EpiState& es, int u, int sb, int nsub, int row, int col0, uint32_t rank) const {
    if ((sb % kFlushChunks) != kFlushChunks - 1 && sb != nsub - 1) return;
    __shared__ float turn[kEpiWarps][32][17];
    bool is_g;
    int p, mt, nt;
    decode(u, is_g, p, mt, nt);
    const int lane = row & 31, w = (row >> 5) + 4 * (col0 / kCols);
    const size_t i = static_cast<size_t>(mt) * Cfg::kUnitM + rank * kBM + (row - lane);  // the warp's first row
    const size_t ld = is_g ? d_in : d_out;
    double* o = (is_g ? G + i * d_in : C + (static_cast<size_t>(p) * d_in + i) * d_out) + static_cast<size_t>(nt) * kBN +
                col0;
    const int half = lane >> 4, col = lane & 15;
    o += half * ld + col;  // lanes 0-15 take the even rows, 16-31 the odd ones
    const float* t = &turn[w][half][col];
#pragma unroll
    for (int c = 0; c < kCols; c += 16) {
#pragma unroll
      for (int j = 0; j < 16; ++j) turn[w][lane][j] = es.rs[c + j];
      __syncwarp();
      double* q = o + c;
#pragma unroll 4
      for (int k = 0; k < 16; ++k, q += 2 * ld) atomicAdd(q, static_cast<double>(t[k * 2 * 17]));
      __syncwarp();
    }
  }
};

// G[i][j] = G[j][i] for i > j: the lower triangle from the upper one, through
// 32 x 32 shared tiles (block (bx, by) writes rows by*32.., columns bx*32..).
__global__ void __launch_bounds__(256) k_mirror_lower(double* __restrict__ G, int d) {
  const int bx = blockIdx.x, by = blockIdx.y;
  if (bx > by) return;
  __shared__ double t[32][33];
  for (int j = threadIdx.y; j < 32; j += 8)
    t[j][threadIdx.x] = G[static_cast<size_t>(bx * 32 + j) * d + by * 32 + threadIdx.x];  // upper block (bx, by)
  __syncthreads();
  for (int j = threadIdx.y; j < 32; j += 8) {
    const int i = by * 32 + j, c = bx * 32 + threadIdx.x;
    if (i > c) G[static_cast<size_t>(i) * d + c] = t[threadIdx.x][j];
  }
}

// Column sums of `n_maps` row-major bf16 matrices [n_rows][ld] (map p at
// base + p*map_stride): out[p][c] += Σ_t M_p[t][c], and out_sq[p][c] += Σ_t M_p[t][c]²
// when out_sq is set. Each thread takes 8 adjacent columns (one 16-byte load per
// row) over 512 rows of a block; fp32 over 64 rows (a bf16 square is exact in
// fp32), then fp64, then one fp64 atomic per column and block. n_cols % 8 == 0.
__global__ void __launch_bounds__(256) k_colsum(const __nv_bfloat16* __restrict__ M, long long ld, long long map_stride,
                                                int n_rows, int n_cols, double* __restrict__ out,
                                                double* __restrict__ out_sq, int64_t* __restrict__ n_counter,
                                                long long add_n) {
  const int c = (blockIdx.x * blockDim.x + threadIdx.x) * 8;
  const int r0 = blockIdx.y * 512;
  const int p = blockIdx.z;
  if (n_counter != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0)
    atomicAdd(reinterpret_cast<unsigned long long*>(n_counter), static_cast<unsigned long long>(add_n));
  if (c >= n_cols) return;
  const __nv_bfloat16* col = M + static_cast<long long>(p) * map_stride + c;
  const int r1 = min(r0 + 512, n_rows);
  double acc[8] = {}, acc_sq[8] = {};
  for (int r = r0; r < r1; r += 64) {
    float s[8] = {}, q[8] = {};
    const int re = min(r + 64, r1);
    for (int t = r; t < re; ++t) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(col + static_cast<long long>(t) * ld));
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(h[j]);
        s[2 * j] += f.x;
        s[2 * j + 1] += f.y;
        q[2 * j] = fmaf(f.x, f.x, q[2 * j]);
        q[2 * j + 1] = fmaf(f.y, f.y, q[2 * j + 1]);
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      acc[j] += static_cast<double>(s[j]);
      acc_sq[j] += static_cast<double>(q[j]);
    }
  }
  double* o = out + static_cast<size_t>(p) * n_cols + c;
#pragma unroll
  for (int j = 0; j < 8; ++j) atomicAdd(o + j, acc[j]);
  if (out_sq != nullptr) {
    double* oq = out_sq + static_cast<size_t>(p) * n_cols + c;
#pragma unroll
    for (int j = 0; j < 8; ++j) atomicAdd(oq + j, acc_sq[j]);
  }
}

// Rows per GEMM launch. Every unit of a launch streams all of its rows, and over
// long launches the pairs drift apart, so that rows they share leave L2 between
// readers (the 8,192-feature Gram over 131,072 rows read 58 GB from DRAM for
// 2.4 GB of operands). Launching slab by slab restarts every pair on the same
// rows. The launches run in stream order and a tile is flushed once per launch,
// so every fp64 total receives its additions in a fixed order.
constexpr int64_t kCalibSlabRows = 16 * kCalibChunk;

template <bool kPair>
rf_status calib_gemm(const rf_calib_desc* desc, const rf_bf16* X, int64_t ld_x, const rf_bf16* Y, int64_t ld_y,
                     int64_t y_map_stride, int64_t n_rows, const rf_calib_stats* st, int32_t* dev_status, int* sched,
                     int sms, cudaStream_t cs) {
  using Cfg = GemmCfg<kPair>;
  const int64_t d_in = desc->d_in, d_out = desc->d_out, P = desc->n_maps;
  rf_status s;
  ProfScope prof(cs, RF_STAGE_CALIB_GEMM);
  for (int64_t r0 = 0; r0 < n_rows; r0 += kCalibSlabRows) {
    const int64_t rows = std::min(kCalibSlabRows, n_rows - r0);
    GramProb<kPair> pr;
    const __nv_bfloat16* Xs = reinterpret_cast<const __nv_bfloat16*>(X) + r0 * ld_x;
    if ((s = make_tmap_bf16_2d(&pr.tmX, Xs, d_in, rows, ld_x, 64, kBK)) != RF_OK) return s;
    if (P > 0) {
      const __nv_bfloat16* Ys = reinterpret_cast<const __nv_bfloat16*>(Y) + r0 * ld_y;
      if ((s = make_tmap_bf16_3d(&pr.tmY, Ys, d_out, rows, P, ld_y, P > 1 ? y_map_stride : ld_y * rows, 64, kBK)) !=
          RF_OK)
        return s;
    } else {
      pr.tmY = pr.tmX;
    }
    pr.G = st->G;
    pr.C = st->C;
    pr.d_in = static_cast<int>(d_in);
    pr.d_out = static_cast<int>(P > 0 ? d_out : 0);
    pr.P = static_cast<int>(P);
    pr.n_rows = static_cast<int>(rows);
    pr.n_chunks = static_cast<int>((rows + kCalibChunk - 1) / kCalibChunk);
    pr.g_mt = static_cast<int>(d_in / Cfg::kUnitM);
    pr.g_nt = static_cast<int>(d_in / kBN);
    pr.c_nt = static_cast<int>(P > 0 ? d_out / kBN : 0);
    pr.g_units = (kBN / Cfg::kUnitM) * pr.g_nt * (pr.g_nt + 1) / 2;  // upper-triangle tiles
    // about 48 MB of X rows per group (a third of L2)
    const int64_t panel = static_cast<int64_t>(Cfg::kUnitM) * rows * 2;
    pr.c_group = static_cast<int>(
        std::max<int64_t>(1, std::min<int64_t>(pr.g_mt, (int64_t(48) << 20) / std::max<int64_t>(panel, 1))));
    pr.sched = sched;
    pr.dev_status = dev_status;
    pr.timeout_ns = wait_timeout_ns();
    if ((s = launch_gemm(pr, pr.g_units + P * pr.g_mt * pr.c_nt, sms, cs, "calibration GEMM launch")) != RF_OK)
      return s;
  }
  // The GEMM accumulates G's tiles on and above the diagonal; the lower triangle
  // becomes their mirror (the accumulated upper triangle is the whole sum).
  k_mirror_lower<<<dim3(static_cast<unsigned>(d_in / 32), static_cast<unsigned>(d_in / 32)), dim3(32, 8), 0, cs>>>(
      st->G, static_cast<int>(d_in));
  return cuda_check(cudaGetLastError(), "k_mirror_lower launch");
}

}  // namespace rf

using namespace rf;

static rf_status check_calib_desc(const rf_calib_desc* d) {
  if (d == nullptr) return fail(RF_ERR_INVALID_ARG, "desc is NULL");
  if (d->d_in <= 0 || d->n_maps < 0 || (d->n_maps > 0 && d->d_out <= 0))
    return fail(RF_ERR_INVALID_ARG, "need d_in > 0, n_maps >= 0, d_out > 0");
  if (d->d_in % kBN != 0) return fail(RF_ERR_SHAPE, "d_in = %lld must be a multiple of 256", (long long)d->d_in);
  if (d->n_maps > 0 && d->d_out % kBN != 0)
    return fail(RF_ERR_SHAPE, "d_out = %lld must be a multiple of 256", (long long)d->d_out);
  if (d->n_maps > 65535) return fail(RF_ERR_SHAPE, "n_maps must be <= 65535");
  return RF_OK;
}

// The optional workspace holds the GEMM's unit counter (dynamic unit order).
constexpr size_t kCalibWorkspace = 256;

extern "C" size_t rf_calib_workspace_bytes(const rf_calib_desc* desc, int64_t) {
  if (check_calib_desc(desc) != RF_OK) return 0;
  return kCalibWorkspace;
}

extern "C" rf_status rf_calib_accumulate(const rf_calib_desc* desc, const rf_bf16* X, int64_t ld_x, const rf_bf16* Y,
                                         int64_t ld_y, int64_t y_map_stride, int64_t n_rows,
                                         const rf_calib_stats* st, int32_t* dev_status, void* workspace,
                                         size_t workspace_bytes, rf_stream_t stream) {
  clear_error();
  rf_status s = check_calib_desc(desc);
  if (s != RF_OK) return s;
  if (st == nullptr || !st->G || !st->sx || !st->n || (desc->n_maps > 0 && (!st->C || !st->sy)))
    return fail(RF_ERR_INVALID_ARG, "stats pointers must be non-NULL (C and sy when n_maps > 0)");
  if (n_rows < 0 || n_rows > (int64_t(1) << 30)) return fail(RF_ERR_INVALID_ARG, "n_rows must be in [0, 2^30]");
  if (n_rows == 0) return RF_OK;
  const int64_t d_in = desc->d_in, d_out = desc->d_out, P = desc->n_maps;
  if (!X || (P > 0 && !Y)) return fail(RF_ERR_INVALID_ARG, "X (and Y when n_maps > 0) must be non-NULL");
  if (!aligned16(X) || (P > 0 && !aligned16(Y)) || !aligned16(st->G) || (P > 0 && !aligned16(st->C)))
    return fail(RF_ERR_ALIGN, "X, Y, G and C must be 16-byte aligned");
  if (ld_x < d_in || ld_x % 8 != 0) return fail(RF_ERR_ALIGN, "ld_x must be >= d_in and a multiple of 8");
  if (P > 0 && (ld_y < d_out || ld_y % 8 != 0 || y_map_stride % 8 != 0 || (P > 1 && y_map_stride < ld_y * n_rows)))
    return fail(RF_ERR_ALIGN, "ld_y must be >= d_out and a multiple of 8; y_map_stride a multiple of 8 "
                              "covering n_rows rows");
  if (workspace != nullptr &&
      (workspace_bytes < kCalibWorkspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
    return fail(RF_ERR_WORKSPACE, "workspace, when given, needs %zu bytes, 256-byte aligned (got %zu)",
                kCalibWorkspace, workspace_bytes);
  int* const sched = static_cast<int*>(workspace);
  int sms = 0;
  if ((s = current_device(&sms)) != RF_OK) return s;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);

  {
    ProfScope prof(cs, RF_STAGE_COLSUM);
    dim3 gx(static_cast<unsigned>((d_in + 2047) / 2048), static_cast<unsigned>((n_rows + 511) / 512), 1);
    k_colsum<<<gx, 256, 0, cs>>>(reinterpret_cast<const __nv_bfloat16*>(X), ld_x, 0, static_cast<int>(n_rows),
                                 static_cast<int>(d_in), st->sx, nullptr, st->n, n_rows);
    if (P > 0) {
      dim3 gy(static_cast<unsigned>((d_out + 2047) / 2048), static_cast<unsigned>((n_rows + 511) / 512),
              static_cast<unsigned>(P));
      k_colsum<<<gy, 256, 0, cs>>>(reinterpret_cast<const __nv_bfloat16*>(Y), ld_y, y_map_stride,
                                   static_cast<int>(n_rows), static_cast<int>(d_out), st->sy, st->syy, nullptr, 0);
    }
  }
  if ((s = cuda_check(cudaGetLastError(), "k_colsum launch")) != RF_OK) return s;

  if (use_pair(desc->flags, true))
    return calib_gemm<true>(desc, X, ld_x, Y, ld_y, y_map_stride, n_rows, st, dev_status, sched, sms, cs);
  return calib_gemm<false>(desc, X, ld_x, Y, ld_y, y_map_stride, n_rows, st, dev_status, sched, sms, cs);
}
