// Persistent, warp-specialised tcgen05 GEMM core for sm_103a.
//
//   D[128 x 256] (fp32, TMEM) = Σ_k A[128 x 64] · B[256 x 64]ᵀ   (bf16 operands)
//
// Roles (192 threads, one CTA per SM):
//   warp 0      one thread issues TMA loads into a kStages-deep ring of
//               128-byte-swizzled shared-memory tiles (full/empty mbarriers);
//   warp 1      allocates 512 TMEM columns (two 256-column accumulators) and one
//               thread issues tcgen05.mma (M=128, N=256, K=16) and commits;
//   warps 2..5  the epilogue warpgroup: tcgen05.ld 32 rows each from the finished
//               accumulator while the MMA warp fills the other one.
//
// The problem type `Prob` decides the work: how many work units there are, how
// many independent accumulations ("sub-tiles") a unit holds, the K-blocks of each,
// which TMA boxes to load for a K-block, and what the epilogue does with a
// finished 128 x 256 fp32 tile. Units are dealt round-robin over the CTAs.
//
// Operands may be K-major (rows of K contiguous: box {64, rows}) or MN-major
// (rows of M/N contiguous: 64-wide boxes {64, 64 k-rows}, one per 64 M/N).
// All waits are bounded (see rf_device.cuh); on a timeout every role stops,
// outstanding TMA copies and MMAs are drained, and TMEM is freed.
#pragma once
#include "rf_device.cuh"

namespace rf {

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kStages = 4;
constexpr int kTileABytes = kBM * kBK * 2;
constexpr int kTileBBytes = kBN * kBK * 2;
constexpr int kStageBytes = kTileABytes + kTileBBytes;
constexpr int kTmemCols = 2 * kBN;
constexpr int kGemmThreads = 192;
constexpr int kEpiThreads = 128;

struct GemmShared {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

constexpr size_t kGemmSmemBytes = 1024 + static_cast<size_t>(kStages) * kStageBytes + sizeof(GemmShared);

// Issue the TMA loads of one operand tile.
//   K-major: one box {64 (k), rows}; the shared tile is rows x 128 B.
//   MN-major: rows/64 boxes {64 (m or n), 64 (k)}; chunk j lands at j * 8 KB.
template <int kRows, bool kMN>
__device__ __forceinline__ void load_operand(uint8_t* dst, const CUtensorMap* tm, uint64_t* bar, int k0, int r0) {
  if constexpr (!kMN) {
    tma_load_2d(dst, tm, bar, k0, r0);
  } else {
#pragma unroll
    for (int j = 0; j < kRows / 64; ++j) tma_load_2d(dst + j * (64 * kBK * 2), tm, bar, r0 + 64 * j, k0);
  }
}

// Shared-memory descriptor of the k-th K=16 slice of a stage's operand tile.
template <bool kMN>
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int k) {
  if constexpr (!kMN) {
    return make_sdesc_sw128(base + k * 32, 16, 1024);  // 8-row groups 1 KB apart
  } else {
    return make_sdesc_sw128(base + k * 2048, 64 * kBK * 2, 1024);  // 64-wide chunks 8 KB apart
  }
}

template <class Prob>
__global__ void __launch_bounds__(kGemmThreads, 1) tc_gemm_kernel(const __grid_constant__ Prob prob) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  GemmShared* sh = reinterpret_cast<GemmShared*>(smem + kStages * kStageBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &sh->abort;
  const uint64_t timeout = prob.timeout_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh->full[s], 1);
      mbar_init(&sh->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh->tmem_full[a], 1);
      mbar_init(&sh->tmem_empty[a], kEpiThreads);
    }
    mbar_init(&sh->mma_done, 1);
    sh->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) prob.prefetch();
  if (warp == 1) {
    tmem_alloc(&sh->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sh->tmem_base;
  const int n_units = prob.num_units();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        const int nsub = prob.num_subtiles(u);
        for (int sb = 0; sb < nsub; ++sb) {
          const int nkb = prob.num_kb(u, sb);
          for (int kb = 0; kb < nkb; ++kb) {
            if (!mbar_wait(&sh->empty[stage], phase ^ 1u, abort_flag, timeout)) goto producer_done;
            mbar_arrive_expect_tx(&sh->full[stage], kStageBytes);
            uint8_t* sa = smem + stage * kStageBytes;
            prob.issue_loads(u, sb, kb, sa, sa + kTileABytes, &sh->full[stage]);
            ++issued;
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
    producer_done:
      // Drain: every issued copy must land before the CTA may exit.
      for (long long i = (issued > kStages ? issued - kStages : 0); i < issued; ++i) {
        const int s = static_cast<int>(i % kStages);
        const uint32_t ph = static_cast<uint32_t>((i / kStages) & 1);
        int dummy = 0;
        mbar_wait(&sh->full[s], ph, &dummy, timeout);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // --------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = make_idesc_bf16(kBM, kBN, Prob::kAMN ? 1 : 0, Prob::kBMN ? 1 : 0);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t it = 0;
      for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        const int nsub = prob.num_subtiles(u);
        for (int sb = 0; sb < nsub; ++sb, ++it) {
          const uint32_t acc = it & 1u;
          const uint32_t acc_phase = (it >> 1) & 1u;
          if (!mbar_wait(&sh->tmem_empty[acc], acc_phase ^ 1u, abort_flag, timeout)) goto mma_done;
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * kBN;
          const int nkb = prob.num_kb(u, sb);
          for (int kb = 0; kb < nkb; ++kb) {
            if (!mbar_wait(&sh->full[stage], phase, abort_flag, timeout)) goto mma_done;
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + stage * kStageBytes);
            const uint32_t sbb = sa + kTileABytes;
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              tc_mma_bf16(d_tmem, operand_desc<Prob::kAMN>(sa, k), operand_desc<Prob::kBMN>(sbb, k), idesc,
                          (kb | k) != 0 ? 1u : 0u);
            }
            tc_commit(&sh->empty[stage]);
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          tc_commit(&sh->tmem_full[acc]);
        }
      }
    mma_done:
      // Drain: wait for every MMA this thread issued before TMEM is released.
      tc_commit(&sh->mma_done);
      int dummy = 0;
      mbar_wait(&sh->mma_done, 0, &dummy, timeout);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const int row = quarter * 32 + lane;
    uint32_t it = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      const int nsub = prob.num_subtiles(u);
      for (int sb = 0; sb < nsub; ++sb, ++it) {
        const uint32_t acc = it & 1u;
        const uint32_t acc_phase = (it >> 1) & 1u;
        bool ok = mbar_wait(&sh->tmem_full[acc], acc_phase, abort_flag, timeout);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) goto epi_done;
        tc_fence_after();
        prob.epilogue(u, sb, tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * kBN, row);
        tc_fence_before();
        mbar_arrive(&sh->tmem_empty[acc]);
      }
    }
  epi_done:;
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && sh->abort) record_status(prob.dev_status, RF_ERR_TIMEOUT);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace rf
