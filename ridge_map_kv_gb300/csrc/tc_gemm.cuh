// Persistent, warp-specialised tcgen05 GEMM cores for sm_103a.
//
// Two kernels share one problem interface:
//
//   tc_gemm_kernel       one CTA per unit of 128 x 256 outputs. Per k-block of 64,
//                        the CTA loads A (128 rows) and B (256 rows) and issues
//                        tcgen05.mma M=128 N=256 K=16 (cta_group::1).
//   tc_gemm_pair_kernel  a CTA pair (cluster of 2) per unit of 256 x 256 outputs.
//                        Each CTA loads its 128 rows of A and its 128 rows of B;
//                        one thread of the even CTA issues tcgen05.mma M=256 N=256
//                        (cta_group::2), which reads B from both CTAs. Per CTA this
//                        moves 32 KB per k-block instead of 48 KB for the same
//                        flops, which relieves shared-memory bandwidth.
//
// D (fp32) lives in TMEM: 512 columns = two 256-column accumulators, so the
// epilogue of one unit overlaps the MMAs of the next.
//
// Roles (64 + 32 * Prob::kEpiWarps threads per CTA, one CTA per SM):
//   warp 0      one thread issues TMA loads into the shared-memory stage ring
//               (full/empty mbarriers);
//   warp 1      allocates TMEM; in the single kernel and in the even CTA of a
//               pair, one thread issues the MMAs and commits;
//   warps 2..   epilogue, 4 or 8 warps. A warp may only read the TMEM lanes
//               32*(warp % 4) .. +31, so warp w takes rows 32*(w % 4) + lane;
//               with 8 warps the second four take the upper 128 columns.
//               The epilogue keeps a per-thread `Prob::EpiState` across the
//               sub-tiles of a unit (e.g. register running sums). It reads the
//               accumulator in `epilogue`, hands the accumulator back to the
//               MMA thread, and may then finish in `epilogue_after` (work that
//               needs no TMEM, such as a flush of running sums to memory).
//
// The problem type `Prob` decides the work: how many units there are, how many
// independent accumulations ("sub-tiles") a unit holds, the K-blocks of each,
// which TMA boxes a CTA loads for a K-block, and what the epilogue does with a
// finished 128-row x 256-column fp32 block. A problem may chain sub-tiles into one
// accumulation with `acc_continues(u, sb)`: true when sub-tile sb adds into the
// accumulator of sub-tile sb - 1, so the MMAs run on without an epilogue between
// them and the epilogue sees only the chain's last sub-tile. Sub-tiles of a chain
// may have no K-blocks (the chain's first MMA, wherever it falls, starts the sum),
// but every chain needs at least one. The producer asks the problem once
// per (unit, sub-tile) for its `Coords` (`coords(u, sb)`), and per K-block only
// issues the loads from them (`issue_loads(c, kb, ...)`): one thread issues every
// copy of the CTA, so any per-K-block arithmetic or memory read there would
// throttle the whole pipeline. Operands may be K-major (box {64, rows}) or
// MN-major (boxes {64, 64} per 64 rows of M or N).
//
// Unit order. By default units are dealt round-robin over CTAs (pairs). A problem
// that holds a non-null `int* sched` (a zeroed device int, one per launch; the
// launcher clears it) is scheduled dynamically instead: the leading CTA's producer
// takes each next unit from that counter with an atomic add, one unit ahead, and
// posts it to every role of both CTAs through a ring of kUnitRing slots in shared
// memory (unit_full / unit_empty mbarriers; -1 ends the sequence). Units then run
// in the order they are asked for, so a CTA pair that runs faster takes more
// units rather than drifting away from the pairs that read the same operand tiles
// through L2 (with round-robin dealing, pairs that ran a few units apart over a
// long launch re-read shared tiles from DRAM).
//
// All waits are bounded (rf_device.cuh); on a timeout every role stops,
// outstanding copies and MMAs are drained, and TMEM is freed.
#pragma once
#include <algorithm>
#include <type_traits>

#include "rf_device.cuh"
#include "rf_host.h"

namespace rf {

constexpr int kBM = 128;  // accumulator rows per CTA (TMEM lanes)
constexpr int kBN = 256;  // accumulator columns (N of a unit)
constexpr int kBK = 64;   // K per stage: one 128-byte swizzle row of bf16
constexpr int kTmemCols = 2 * kBN;
template <class Prob>
constexpr int gemm_threads() {
  return 64 + 32 * Prob::kEpiWarps;
}
constexpr int kAtomABytes = kBM * kBK * 2;

// A stage holds kAtoms consecutive K-blocks of 64 ("atoms") of A, then of B;
// each atom has the layout of a single 64-wide tile. The pair kernel takes two
// atoms per stage, which halves the barrier traffic per unit of K for its one
// producer thread and one MMA thread.
template <bool kPair>
struct GemmCfg {
  static constexpr int kBRows = kPair ? 128 : 256;  // B rows this CTA loads per stage
  static constexpr int kUnitM = kPair ? 256 : 128;  // output rows of a unit
  static constexpr int kAtoms = kPair ? 2 : 1;
  static constexpr int kStages = kPair ? 3 : 4;
  static constexpr int kAtomBBytes = kBRows * kBK * 2;
  static constexpr int kTileABytes = kAtoms * kAtomABytes;
  static constexpr int kTileBBytes = kAtoms * kAtomBBytes;
  static constexpr int kStageBytes = kTileABytes + kTileBBytes;
};

constexpr int kUnitRing = 4;  // posted units in flight (dynamic order)

struct GemmShared {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t mma_done;
  uint64_t unit_full[kUnitRing];   // in each CTA: the leader's producer posted the slot
  uint64_t unit_empty[kUnitRing];  // the leader's only: every consumer of both CTAs took it
  int unit_ring[kUnitRing];
  uint32_t tmem_base;
  int abort;
};

// Dynamic unit order (see above): the problem's `sched` counter, or nullptr.
template <class P, class = void>
struct HasSched : std::false_type {};
template <class P>
struct HasSched<P, std::void_t<decltype(std::declval<const P&>().sched)>> : std::true_type {};
// Chained sub-tiles (see above): the problem's `acc_continues`, or none.
template <class P, class = void>
struct HasAccChain : std::false_type {};
template <class P>
struct HasAccChain<P, std::void_t<decltype(std::declval<const P&>().acc_continues(0, 0))>> : std::true_type {};
template <class Prob>
__device__ __forceinline__ bool acc_continues(const Prob& p, int u, int sb) {
  if constexpr (HasAccChain<Prob>::value) return sb > 0 && p.acc_continues(u, sb);
  else return false;
}

template <class Prob>
__host__ __device__ __forceinline__ int* sched_of(const Prob& p) {
  if constexpr (HasSched<Prob>::value) return p.sched;
  else return nullptr;
}

// The leader's producer: posts unit u (or -1) to slot `slot` of the ring of this
// CTA and, for a pair, of the peer, once every consumer took the slot's previous
// unit. False after an abort. The leader's own CTA is reached with CTA-scope
// operations (its MMA thread, on the critical path, then waits at CTA scope); only
// the peer's copy goes through cluster-scope release.
template <bool kPair>
__device__ __forceinline__ bool post_unit(GemmShared* sh, int u, int& slot, uint32_t& phase, volatile int* abort_flag,
                                          uint64_t timeout) {
  if (!mbar_wait<kPair>(&sh->unit_empty[slot], phase ^ 1u, abort_flag, timeout)) return false;
  *reinterpret_cast<volatile int*>(&sh->unit_ring[slot]) = u;
  mbar_arrive(&sh->unit_full[slot]);  // release at CTA scope
  if constexpr (kPair) {
    st_shared_cluster_s32(mapa_shared(smem_u32(&sh->unit_ring[slot]), 1), u);
    mbar_arrive_cluster(mapa_shared(smem_u32(&sh->unit_full[slot]), 1));  // release at cluster scope
  }
  if (++slot == kUnitRing) {
    slot = 0;
    phase ^= 1u;
  }
  return true;
}
// A consumer thread: the next posted unit (-1 at the end), or -2 after an abort.
// `remote` is true in the peer CTA of a pair (its ring is written by the leader
// from the other CTA). The caller then hands the slot back with give_back_unit
// (once per consumer: one thread, or lane 0 of a warp after __syncwarp) and
// advances with next_unit_slot.
__device__ __forceinline__ int take_unit(GemmShared* sh, int slot, uint32_t phase, bool remote,
                                         volatile int* abort_flag, uint64_t timeout) {
  const bool ok = remote ? mbar_wait<true>(&sh->unit_full[slot], phase, abort_flag, timeout)
                         : mbar_wait<false>(&sh->unit_full[slot], phase, abort_flag, timeout);
  if (!ok) return -2;
  return *reinterpret_cast<volatile int*>(&sh->unit_ring[slot]);
}
__device__ __forceinline__ void give_back_unit(GemmShared* sh, int slot, bool remote) {
  if (remote) mbar_arrive_cluster(mapa_shared(smem_u32(&sh->unit_empty[slot]), 0));
  else mbar_arrive(&sh->unit_empty[slot]);
}
__device__ __forceinline__ void next_unit_slot(int& slot, uint32_t& phase) {
  if (++slot == kUnitRing) {
    slot = 0;
    phase ^= 1u;
  }
}
// The leader's producer: the next unit from the counter, or -1 once all are taken.
__device__ __forceinline__ int fetch_unit(int* sched, int n_units) {
  const int u = atomicAdd(sched, 1);
  return u < n_units ? u : -1;
}

// The leader's producer, dynamic order: fetches and posts the first unit before
// its loop, so that every consumer learns each unit one unit ahead. Returns the
// posted unit (-1 when there is none), or -2 after an abort.
template <bool kPair>
__device__ __forceinline__ int leader_start(GemmShared* sh, int* sched, int n_units, int& slot, uint32_t& phase,
                                            volatile int* abort_flag, uint64_t timeout) {
  if (sched == nullptr) return -1;
  const int u = fetch_unit(sched, n_units);
  return post_unit<kPair>(sh, u, slot, phase, abort_flag, timeout) ? u : -2;
}
// The unit after `cur` for the leader's producer, -1 at the end, -2 after an abort.
// Dynamic order: `next` is the unit posted ahead; it is returned, and the one after
// it is fetched and posted now. Static order: cur + stride. Start with
// cur = first − stride.
template <bool kPair>
__device__ __forceinline__ int leader_next(GemmShared* sh, int* sched, int cur, int stride, int n_units, int& next,
                                           int& slot, uint32_t& phase, volatile int* abort_flag, uint64_t timeout) {
  if (sched == nullptr) {
    const int n = cur + stride;
    return n < n_units ? n : -1;
  }
  const int u = next;
  if (u >= 0) {
    next = fetch_unit(sched, n_units);
    if (!post_unit<kPair>(sh, next, slot, phase, abort_flag, timeout)) return -2;
  }
  return u;
}
// The same for a consumer role: one thread, or a whole warp (`warp_role`: every
// lane takes the unit, lane 0 hands the slot back once for the warp). `remote`:
// the consumer is in the peer CTA of a pair.
__device__ __forceinline__ int consumer_next(GemmShared* sh, int* sched, int cur, int stride, int n_units, int& slot,
                                             uint32_t& phase, bool warp_role, bool remote, volatile int* abort_flag,
                                             uint64_t timeout) {
  if (sched == nullptr) {
    const int n = cur + stride;
    return n < n_units ? n : -1;
  }
  const int u = take_unit(sh, slot, phase, remote, abort_flag, timeout);
  if (warp_role) {
    if (!__all_sync(0xffffffffu, u != -2)) return -2;
    __syncwarp();
    if ((threadIdx.x & 31) == 0) give_back_unit(sh, slot, remote);
  } else {
    if (u == -2) return -2;
    give_back_unit(sh, slot, remote);
  }
  next_unit_slot(slot, phase);
  return u;
}

// Shared memory of a CTA: the stage ring, the barriers, then (from a 128-byte
// boundary) `Prob::kEpiSmemBytes` of epilogue scratch when the problem declares it,
// e.g. the staging rows of the cache-writing epilogues.
template <class P, class = void>
struct EpiSmemBytes {
  static constexpr size_t value = 0;
};
template <class P>
struct EpiSmemBytes<P, std::void_t<decltype(P::kEpiSmemBytes)>> {
  static constexpr size_t value = P::kEpiSmemBytes;
};

template <bool kPair>
constexpr size_t gemm_epi_offset() {
  return (static_cast<size_t>(GemmCfg<kPair>::kStages) * GemmCfg<kPair>::kStageBytes + sizeof(GemmShared) + 127) &
         ~size_t(127);
}
template <class Prob>
constexpr size_t gemm_smem_bytes() {
  return 1024 + gemm_epi_offset<Prob::kPair>() + EpiSmemBytes<Prob>::value;
}

template <bool kPair>
__device__ __forceinline__ void tma2(void* dst, const CUtensorMap* tm, uint32_t bar, int32_t x, int32_t y) {
  if constexpr (kPair) tma_load_2d_pair(dst, tm, bar, x, y);
  else tma_load_2d_u32(dst, tm, bar, x, y);
}
template <bool kPair>
__device__ __forceinline__ void tma3(void* dst, const CUtensorMap* tm, uint32_t bar, int32_t x, int32_t y, int32_t z) {
  if constexpr (kPair) tma_load_3d_pair(dst, tm, bar, x, y, z);
  else tma_load_3d_u32(dst, tm, bar, x, y, z);
}

// Loads one operand tile of kRows rows x 64 K.
//   K-major: one box {64 (k), kRows}; the shared tile is kRows x 128 B.
//   MN-major: kRows/64 boxes {64 (m or n), 64 (k)}; chunk j lands at j * 8 KB.
template <int kRows, bool kMN, bool kPair>
__device__ __forceinline__ void load_operand(uint8_t* dst, const CUtensorMap* tm, uint32_t bar, int k0, int r0) {
  if constexpr (!kMN) {
    tma2<kPair>(dst, tm, bar, k0, r0);
  } else {
#pragma unroll
    for (int j = 0; j < kRows / 64; ++j) tma2<kPair>(dst + j * (64 * kBK * 2), tm, bar, r0 + 64 * j, k0);
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

__device__ __forceinline__ uint8_t* gemm_smem_base(uint8_t* raw) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
}

// The epilogue scratch of the running GEMM kernel (see gemm_smem_bytes), for the
// problem's epilogue to call.
template <bool kPair>
__device__ __forceinline__ uint8_t* gemm_epi_smem() {
  extern __shared__ uint8_t smem_raw[];
  return gemm_smem_base(smem_raw) + gemm_epi_offset<kPair>();
}

// --------------------------------------------------------------------------
// Single-CTA kernel
// --------------------------------------------------------------------------
template <class Prob>
__global__ void __launch_bounds__(gemm_threads<Prob>(), 1) tc_gemm_kernel(const __grid_constant__ Prob prob) {
  static_assert(!Prob::kPair, "pair problems run on tc_gemm_pair_kernel");
  using Cfg = GemmCfg<false>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = gemm_smem_base(smem_raw);
  GemmShared* sh = reinterpret_cast<GemmShared*>(smem + Cfg::kStages * Cfg::kStageBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &sh->abort;
  const uint64_t timeout = prob.timeout_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::kStages; ++s) {
      mbar_init(&sh->full[s], 1);
      mbar_init(&sh->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh->tmem_full[a], 1);
      mbar_init(&sh->tmem_empty[a], 32 * Prob::kEpiWarps);
    }
    for (int i = 0; i < kUnitRing; ++i) {
      mbar_init(&sh->unit_full[i], 1);
      mbar_init(&sh->unit_empty[i], 1 + Prob::kEpiWarps);  // the MMA thread and each epilogue warp
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
  int* const sched = sched_of(prob);
  const int first = static_cast<int>(blockIdx.x) - static_cast<int>(gridDim.x), stride = static_cast<int>(gridDim.x);
  int uslot = 0;
  uint32_t uphase = 0;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      int next = leader_start<false>(sh, sched, n_units, uslot, uphase, abort_flag, timeout);
      for (int u = leader_next<false>(sh, sched, first, stride, n_units, next, uslot, uphase, abort_flag, timeout);
           u >= 0; u = leader_next<false>(sh, sched, u, stride, n_units, next, uslot, uphase, abort_flag, timeout)) {
        const int nsub = prob.num_subtiles(u);
        for (int sb = 0; sb < nsub; ++sb) {
          const int nkb = prob.num_kb(u, sb);
          typename Prob::Coords c = prob.coords(u, sb, 0u);
          for (int kb = 0; kb < nkb; ++kb) {
            if (!mbar_wait(&sh->empty[stage], phase ^ 1u, abort_flag, timeout)) goto producer_done;
            mbar_arrive_expect_tx(&sh->full[stage], Cfg::kStageBytes);
            uint8_t* sa = smem + stage * Cfg::kStageBytes;
            prob.issue_loads(c, kb, sa, sa + Cfg::kTileABytes, smem_u32(&sh->full[stage]));
            ++issued;
            if (++stage == Cfg::kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
    producer_done:
      // Drain: every issued copy must land before the CTA may exit.
      for (long long i = (issued > Cfg::kStages ? issued - Cfg::kStages : 0); i < issued; ++i) {
        int dummy = 0;
        mbar_wait(&sh->full[i % Cfg::kStages], static_cast<uint32_t>((i / Cfg::kStages) & 1), &dummy, timeout);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc_bf16(kBM, kBN, Prob::kAMN ? 1 : 0, Prob::kBMN ? 1 : 0);
      // Stage-0 descriptors of the four K=16 slices; stage s adds its byte offset
      // / 16 to the start-address field (shared addresses stay below 256 KB).
      uint64_t adesc[kBK / 16], bdesc[kBK / 16];
#pragma unroll
      for (int k = 0; k < kBK / 16; ++k) {
        adesc[k] = operand_desc<Prob::kAMN>(smem_u32(smem), k);
        bdesc[k] = operand_desc<Prob::kBMN>(smem_u32(smem) + Cfg::kTileABytes, k);
      }
      int stage = 0;
      uint32_t phase = 0;
      uint32_t it = 0;
      bool fresh = true;  // no MMA has written the current accumulation yet
      for (int u = consumer_next(sh, sched, first, stride, n_units, uslot, uphase, false, false, abort_flag, timeout);
           u >= 0;
           u = consumer_next(sh, sched, u, stride, n_units, uslot, uphase, false, false, abort_flag, timeout)) {
        const int nsub = prob.num_subtiles(u);
        for (int sb = 0; sb < nsub; ++sb) {
          const uint32_t acc = it & 1u;
          const bool cont = acc_continues(prob, u, sb);
          if (!cont) {
            if (!mbar_wait(&sh->tmem_empty[acc], ((it >> 1) & 1u) ^ 1u, abort_flag, timeout)) goto mma_done;
            tc_fence_after();
          }
          const uint32_t d_tmem = tmem_base + acc * kBN;
          if (!cont) fresh = true;
          const int nkb = prob.num_kb(u, sb);
          for (int kb = 0; kb < nkb; ++kb) {
            if (!mbar_wait(&sh->full[stage], phase, abort_flag, timeout)) goto mma_done;
            tc_fence_after();
            const uint64_t soff = static_cast<uint64_t>((stage * Cfg::kStageBytes) >> 4);
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              tc_mma_bf16(d_tmem, adesc[k] + soff, bdesc[k] + soff, idesc, fresh ? 0u : 1u);
              fresh = false;
            }
            tc_commit(&sh->empty[stage]);
            if (++stage == Cfg::kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (sb + 1 == nsub || !acc_continues(prob, u, sb + 1)) {
            tc_commit(&sh->tmem_full[acc]);
            ++it;
          }
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
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const int row = quarter * 32 + lane;
    const int col0 = ((warp - 2) >> 2) * (kBN * 4 / Prob::kEpiWarps);
    typename Prob::EpiState es{};
    uint32_t it = 0;
    for (int u = consumer_next(sh, sched, first, stride, n_units, uslot, uphase, true, false, abort_flag, timeout);
         u >= 0; u = consumer_next(sh, sched, u, stride, n_units, uslot, uphase, true, false, abort_flag, timeout)) {
      const int nsub = prob.num_subtiles(u);
      for (int sb = 0; sb < nsub; ++sb) {
        if (sb + 1 < nsub && acc_continues(prob, u, sb + 1)) continue;  // not the end of a chain
        const uint32_t acc = it & 1u;
        bool ok = mbar_wait(&sh->tmem_full[acc], (it >> 1) & 1u, abort_flag, timeout);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) goto epi_done;
        tc_fence_after();
        prob.epilogue(es, u, sb, nsub,
                      tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * kBN + static_cast<uint32_t>(col0),
                      row, col0, 0u);
        tc_fence_before();
        mbar_arrive(&sh->tmem_empty[acc]);
        prob.epilogue_after(es, u, sb, nsub, row, col0, 0u);
        ++it;
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

// --------------------------------------------------------------------------
// CTA-pair kernel (cluster of 2; rank 0 issues the MMAs)
//   full[s]       rank 0's only: its producer expects both CTAs' bytes, and both
//                 CTAs' TMA loads complete on it;
//   empty[s]      in each CTA: the pair commit arrives on both;
//   tmem_full[a]  in each CTA: the pair commit arrives on both;
//   tmem_empty[a] rank 0's only: the 4 epilogue warps of both CTAs arrive.
// full, empty and tmem_full complete through the async proxy (TMA complete_tx,
// tcgen05.commit) and guard async-proxy accesses (MMA reads, TMA writes, TMEM
// loads after a tcgen05 fence), so CTA-scope waits suffice there. tmem_empty
// orders the peer's generic-proxy threads and uses cluster-scope release/acquire;
// it is waited on once per accumulator, not per k-block.
// --------------------------------------------------------------------------
template <class Prob>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(gemm_threads<Prob>(), 1)
    tc_gemm_pair_kernel(const __grid_constant__ Prob prob) {
  static_assert(Prob::kPair, "single-CTA problems run on tc_gemm_kernel");
  using Cfg = GemmCfg<true>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = gemm_smem_base(smem_raw);
  GemmShared* sh = reinterpret_cast<GemmShared*>(smem + Cfg::kStages * Cfg::kStageBytes);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = blockIdx.x >> 1;
  const int n_pairs = gridDim.x >> 1;
  volatile int* abort_flag = &sh->abort;
  const uint64_t timeout = prob.timeout_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::kStages; ++s) {
      mbar_init(&sh->full[s], 1);
      mbar_init(&sh->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh->tmem_full[a], 1);
      mbar_init(&sh->tmem_empty[a], 2 * Prob::kEpiWarps);
    }
    for (int i = 0; i < kUnitRing; ++i) {
      mbar_init(&sh->unit_full[i], 1);
      // rank 0's: its MMA thread, the odd CTA's producer and every epilogue warp of both
      mbar_init(&sh->unit_empty[i], 2 + 2 * Prob::kEpiWarps);
    }
    mbar_init(&sh->mma_done, 1);
    sh->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) prob.prefetch();
  __syncwarp();
  if (warp == 1) {
    tmem_alloc_pair(&sh->tmem_base, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncwarp();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = sh->tmem_base;
  const int n_units = prob.num_units();
  int* const sched = sched_of(prob);
  const int first = pair - n_pairs;
  int uslot = 0;
  uint32_t uphase = 0;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      // rank 0's full barriers, as shared::cluster addresses (8 bytes apart)
      const uint32_t full_leader = mapa_shared(smem_u32(&sh->full[0]), 0);
      // rank 0's producer leads the unit order; rank 1's follows its posts
      int next = rank == 0 ? leader_start<true>(sh, sched, n_units, uslot, uphase, abort_flag, timeout) : -1;
      auto advance = [&](int cur) {
        return rank == 0
                   ? leader_next<true>(sh, sched, cur, n_pairs, n_units, next, uslot, uphase, abort_flag, timeout)
                   : consumer_next(sh, sched, cur, n_pairs, n_units, uslot, uphase, false, true, abort_flag, timeout);
      };
      for (int u = advance(first); u >= 0; u = advance(u)) {
        const int nsub = prob.num_subtiles(u);
        for (int sb = 0; sb < nsub; ++sb) {
          // K-blocks rounded up to whole stages: a missing last atom is read past
          // the operand's end, where TMA fills zeros (only the ragged last row
          // chunk of the calibration sums has an odd count).
          const int nst = (prob.num_kb(u, sb) + Cfg::kAtoms - 1) / Cfg::kAtoms;
          typename Prob::Coords c = prob.coords(u, sb, rank);
          for (int st = 0; st < nst; ++st) {
            if (!mbar_wait(&sh->empty[stage], phase ^ 1u, abort_flag, timeout)) goto producer_done;
            if (rank == 0) mbar_arrive_expect_tx(&sh->full[stage], 2 * Cfg::kStageBytes);
            uint8_t* sa = smem + stage * Cfg::kStageBytes;
#pragma unroll
            for (int a = 0; a < Cfg::kAtoms; ++a)
              prob.issue_loads(c, st * Cfg::kAtoms + a, sa + a * kAtomABytes,
                               sa + Cfg::kTileABytes + a * Cfg::kAtomBBytes, full_leader + stage * 8u);
            ++issued;
            if (++stage == Cfg::kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
    producer_done:
      // Both CTAs' copies complete on rank 0's full barriers: rank 0 drains them
      // before the closing cluster barrier, which neither CTA passes alone.
      if (rank == 0) {
        for (long long i = (issued > Cfg::kStages ? issued - Cfg::kStages : 0); i < issued; ++i) {
          int dummy = 0;
          mbar_wait(&sh->full[i % Cfg::kStages], static_cast<uint32_t>((i / Cfg::kStages) & 1), &dummy, timeout);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = make_idesc_bf16(2 * kBM, kBN, Prob::kAMN ? 1 : 0, Prob::kBMN ? 1 : 0);
      constexpr int kSlices = Cfg::kAtoms * kBK / 16;
      uint64_t adesc[kSlices], bdesc[kSlices];
#pragma unroll
      for (int k = 0; k < kSlices; ++k) {
        const int a = k / (kBK / 16), kk = k % (kBK / 16);
        adesc[k] = operand_desc<Prob::kAMN>(smem_u32(smem) + a * kAtomABytes, kk);
        bdesc[k] = operand_desc<Prob::kBMN>(smem_u32(smem) + Cfg::kTileABytes + a * Cfg::kAtomBBytes, kk);
      }
      int stage = 0;
      uint32_t phase = 0;
      uint32_t it = 0;
      bool fresh = true;  // no MMA has written the current accumulation yet
      for (int u = consumer_next(sh, sched, first, n_pairs, n_units, uslot, uphase, false, false, abort_flag, timeout);
           u >= 0;
           u = consumer_next(sh, sched, u, n_pairs, n_units, uslot, uphase, false, false, abort_flag, timeout)) {
        const int nsub = prob.num_subtiles(u);
        for (int sb = 0; sb < nsub; ++sb) {
          const uint32_t acc = it & 1u;
          const bool cont = acc_continues(prob, u, sb);
          if (!cont) {
            if (!mbar_wait<true>(&sh->tmem_empty[acc], ((it >> 1) & 1u) ^ 1u, abort_flag, timeout)) goto mma_done;
            tc_fence_after();
          }
          const uint32_t d_tmem = tmem_base + acc * kBN;
          if (!cont) fresh = true;
          const int nst = (prob.num_kb(u, sb) + Cfg::kAtoms - 1) / Cfg::kAtoms;
          for (int st = 0; st < nst; ++st) {
            if (!mbar_wait(&sh->full[stage], phase, abort_flag, timeout)) goto mma_done;
            tc_fence_after();
            const uint64_t soff = static_cast<uint64_t>((stage * Cfg::kStageBytes) >> 4);
#pragma unroll
            for (int k = 0; k < kSlices; ++k) {
              tc_mma_bf16_pair(d_tmem, adesc[k] + soff, bdesc[k] + soff, idesc, fresh ? 0u : 1u);
              fresh = false;
            }
            tc_commit_pair_multicast(&sh->empty[stage], 0x3);
            if (++stage == Cfg::kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (sb + 1 == nsub || !acc_continues(prob, u, sb + 1)) {
            tc_commit_pair_multicast(&sh->tmem_full[acc], 0x3);
            ++it;
          }
        }
      }
    mma_done:
      tc_commit_pair(&sh->mma_done);
      int dummy = 0;
      mbar_wait(&sh->mma_done, 0, &dummy, timeout);
    }
    __syncwarp();
  } else {
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int col0 = ((warp - 2) >> 2) * (kBN * 4 / Prob::kEpiWarps);
    typename Prob::EpiState es{};
    uint32_t it = 0;
    for (int u = consumer_next(sh, sched, first, n_pairs, n_units, uslot, uphase, true, rank != 0, abort_flag, timeout);
         u >= 0; u = consumer_next(sh, sched, u, n_pairs, n_units, uslot, uphase, true, rank != 0, abort_flag, timeout)) {
      const int nsub = prob.num_subtiles(u);
      for (int sb = 0; sb < nsub; ++sb) {
        if (sb + 1 < nsub && acc_continues(prob, u, sb + 1)) continue;  // not the end of a chain
        const uint32_t acc = it & 1u;
        bool ok = mbar_wait(&sh->tmem_full[acc], (it >> 1) & 1u, abort_flag, timeout);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) goto epi_done;
        tc_fence_after();
        prob.epilogue(es, u, sb, nsub,
                      tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * kBN + static_cast<uint32_t>(col0),
                      row, col0, rank);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&sh->tmem_empty[acc]), 0));
        prob.epilogue_after(es, u, sb, nsub, row, col0, rank);
        ++it;
      }
    }
  epi_done:;
  }

  tc_fence_before();
  __syncwarp();
  cluster_sync_all();
  if (threadIdx.x == 0 && sh->abort) record_status(prob.dev_status, RF_ERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// Host launcher: persistent grid of min(units, SMs) CTAs, or of min(units,
// co-resident clusters) CTA pairs, with the kernel's dynamic shared memory opted in once per device.
template <class Prob>
rf_status launch_gemm(const Prob& pr, int64_t max_units, int sms, cudaStream_t s, const char* what) {
  static uint64_t attr_mask = 0;
  static int pair_cap[64] = {};
  constexpr bool kPair = Prob::kPair;
  const void* fn;
  if constexpr (kPair) fn = reinterpret_cast<const void*>(&tc_gemm_pair_kernel<Prob>);
  else fn = reinterpret_cast<const void*>(&tc_gemm_kernel<Prob>);
  constexpr size_t smem = gemm_smem_bytes<Prob>();
  static_assert(smem <= 227 * 1024, "shared memory beyond the 227 KB a CTA may hold");
  rf_status st = set_smem_attr(fn, smem, &attr_mask);
  if (st != RF_OK) return st;
  if (max_units <= 0) max_units = 1;
  if (int* sc = sched_of(pr); sc != nullptr) {
    if ((st = cuda_check(cudaMemsetAsync(sc, 0, sizeof(int), s), "unit counter clear")) != RF_OK) return st;
  }
  if constexpr (kPair) {
    const int cap = max_active_pairs(fn, smem, gemm_threads<Prob>(), sms, pair_cap);
    const int pairs = static_cast<int>(std::min<int64_t>(max_units, cap));
    tc_gemm_pair_kernel<Prob><<<2 * pairs, gemm_threads<Prob>(), smem, s>>>(pr);
  } else {
    const int grid = static_cast<int>(std::min<int64_t>(max_units, sms));
    tc_gemm_kernel<Prob><<<grid, gemm_threads<Prob>(), smem, s>>>(pr);
  }
  return cuda_check(cudaGetLastError(), what);
}

// Chooses CTA pairs or single CTAs from RF_FLAG_* bits; with neither bit set,
// the operation's own default `pair_by_default` applies.
inline bool use_pair(uint64_t flags, bool pair_by_default) {
  if (flags & RF_FLAG_SINGLE_CTA) return false;
  if (flags & RF_FLAG_CTA_PAIR) return true;
  return pair_by_default;
}

}  // namespace rf
