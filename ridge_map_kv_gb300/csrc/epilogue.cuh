// Shared epilogue step: one attention head of 32 accumulator rows (one per lane
// of a warp), read from TMEM, optionally scaled and biased, optionally rotated
// (rotate-half RoPE), rounded to bf16, turned through the warp's staging rows in
// shared memory and written to memory whole head rows at a time.
//
// Every tcgen05.ld here is warp-collective, so all lanes call emit_head with the
// same (tcol, hd, rope); only the lane's own position and destination differ
// (nullptr where the lane's row is not written).
//
// Why the turn: a lane owns one row, so storing straight from registers puts 32
// rows into every warp store, 16 bytes each: 32 sectors per request, each half
// written. Each step of 16 rotation pairs (or 32 columns without rotation) instead
// goes to the warp's staging rows, 64 bytes a row, and the warp then stores 8 rows
// per instruction, two whole 32-byte sectors in each: 16 sectors per request, every
// one written whole.
//
// Why the rotation is computed, not looked up: a cos/sin table row per lane puts
// 32 rows into every table load as well, and on the K/V GEMM those loads kept the
// epilogue long enough to delay the next tile's MMAs (the same GEMM without RoPE
// ran 5.7 % faster). The angle is instead reduced exactly in 64-bit fixed point
// and its sine and cosine come from the SFU.
#pragma once
#include <cmath>

#include "rf_device.cuh"

namespace rf {

constexpr int kHeadDimMax = 128;
// Staging rows of one epilogue warp: 32 rows of 64 bytes (one step of a head).
constexpr int kStageBytesPerWarp = 32 * 64;

// Byte offset of 16-byte piece `pc` (0..3) of staged row `r`. The piece index is
// XOR-swizzled by bits 1-2 of the row, so that the eight lanes of a shared-memory
// phase hit distinct banks both when they write one piece of eight rows and when
// they read the four pieces of two rows.
__device__ __forceinline__ uint32_t stage_off(int r, int pc) {
  return static_cast<uint32_t>(r * 64 + ((pc ^ ((r >> 1) & 3)) << 4));
}

// Writes the warp's 32 staged rows: piece pc of row r (staged by lane r) goes to
// lane r's `dst` + c_lo + 8 pc for pc < 2 and + c_hi + 8 (pc − 2) for pc >= 2, or
// nowhere when lane r's `dst` is nullptr. Starts and ends with the warp converged,
// so the staging rows may be rewritten at once.
__device__ __forceinline__ void store_staged_rows(uint32_t stage, int c_lo, int c_hi, __nv_bfloat16* dst) {
  const int lane = threadIdx.x & 31;
  const int pc = lane & 3;
  const int col = pc < 2 ? c_lo + 8 * pc : c_hi + 8 * (pc - 2);
  const unsigned long long mine = reinterpret_cast<unsigned long long>(dst);
  __syncwarp();
#pragma unroll
  for (int r0 = 0; r0 < 32; r0 += 8) {
    const int r = r0 + (lane >> 2);
    const unsigned long long p = __shfl_sync(0xffffffffu, mine, r);
    const uint4 v = ld_shared_v4(stage + stage_off(r, pc));
    if (p != 0ull) st_global_v4(reinterpret_cast<__nv_bfloat16*>(p) + col, v.x, v.y, v.z, v.w);
  }
  __syncwarp();
}

// RoPE frequencies of one (θ, hd) as fixed-point turns per position:
// g[i] = 2^64 · θ^(-2i/hd) / 2π, i < hd/2, computed in double. For an integer
// position q, the angle q·θ^(-2i/hd) reduced mod 2π is q·g[i] mod 2^64 in units of
// 2π/2^64: integer arithmetic that wraps exactly, so the only error is g[i]'s own
// (a few units in the last place of a double) times |q|, under 2e-7 rad for
// |q| < 2^28. Built on the host; 512 bytes, passed by value in kernel parameters.
struct RopeFreqs {
  unsigned long long g[kHeadDimMax / 2];
};

inline RopeFreqs rope_freqs(double theta, int hd) {
  RopeFreqs f{};
  const double inv_two_pi = 0.15915494309189535;  // 1 / 2π
  for (int i = 0; i < hd / 2; ++i)
    f.g[i] = static_cast<unsigned long long>(std::ldexp(std::pow(theta, -2.0 * i / hd) * inv_two_pi, 64));
  return f;
}

// cos and sin of the angle q·g (see RopeFreqs): the top 32 bits of the wrapped
// product, read as a signed fraction of a turn in [-1/2, 1/2), give the reduced
// angle in [-π, π), where the SFU's sine and cosine are accurate to about 2^-21.
__device__ __forceinline__ void rope_cs(unsigned long long q, unsigned long long g, float& c, float& s) {
  const int turns = static_cast<int>(static_cast<unsigned>((q * g) >> 32));
  __sincosf(static_cast<float>(turns) * 1.4629180792671596e-9f, &s, &c);  // 2π / 2^32
}

// acc column c (0 <= c < hd) of this lane's row lives at TMEM column tcol + c.
// out[c] = bf16(f((acc[c] * scale + bias[c]) * gain[c])), with f = RoPE at position
// `pos` (two's complement) with frequencies `rope` when that is not nullptr, else
// the identity. bias and gain may be nullptr. `stage` is the warp's staging rows
// (kStageBytesPerWarp, 16-byte aligned).
__device__ __forceinline__ float gain_at(const __nv_bfloat16* __restrict__ gain, int c) {
  return gain != nullptr ? __bfloat162float(gain[c]) : 1.0f;
}

__device__ __forceinline__ void emit_head(uint32_t tcol, int hd, float scale, const float* __restrict__ bias,
                                          const __nv_bfloat16* __restrict__ gain,
                                          const unsigned long long* __restrict__ rope, unsigned long long pos,
                                          __nv_bfloat16* dst, uint32_t stage) {
  const int half = hd >> 1;
  const int lane = threadIdx.x & 31;
  if (rope != nullptr) {
#pragma unroll 1
    for (int i0 = 0; i0 < half; i0 += 16) {
      uint32_t a[16], b[16];
      tmem_ld16(tcol + i0, a);
      tmem_ld16(tcol + half + i0, b);
      tmem_wait_ld16(a);
      tmem_wait_ld16(b);
      uint32_t o1[8], o2[8];
#pragma unroll
      for (int i = 0; i < 16; i += 4) {
        float cc[4], ssn[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) rope_cs(pos, rope[i0 + i + q], cc[q], ssn[q]);
        float4 b1 = make_float4(0.f, 0.f, 0.f, 0.f), b2 = b1;
        if (bias != nullptr) {
          b1 = __ldg(reinterpret_cast<const float4*>(bias + i0 + i));
          b2 = __ldg(reinterpret_cast<const float4*>(bias + half + i0 + i));
        }
        const float bb1[4] = {b1.x, b1.y, b1.z, b1.w};
        const float bb2[4] = {b2.x, b2.y, b2.z, b2.w};
        float r1[4], r2[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float x1 = fmaf(u2f(a[i + q]), scale, bb1[q]) * gain_at(gain, i0 + i + q);
          const float x2 = fmaf(u2f(b[i + q]), scale, bb2[q]) * gain_at(gain, half + i0 + i + q);
          r1[q] = x1 * cc[q] - x2 * ssn[q];
          r2[q] = x2 * cc[q] + x1 * ssn[q];
        }
        o1[i / 2] = pack_bf16x2(r1[0], r1[1]);
        o1[i / 2 + 1] = pack_bf16x2(r1[2], r1[3]);
        o2[i / 2] = pack_bf16x2(r2[0], r2[1]);
        o2[i / 2 + 1] = pack_bf16x2(r2[2], r2[3]);
      }
      st_shared_v4(stage + stage_off(lane, 0), o1[0], o1[1], o1[2], o1[3]);
      st_shared_v4(stage + stage_off(lane, 1), o1[4], o1[5], o1[6], o1[7]);
      st_shared_v4(stage + stage_off(lane, 2), o2[0], o2[1], o2[2], o2[3]);
      st_shared_v4(stage + stage_off(lane, 3), o2[4], o2[5], o2[6], o2[7]);
      store_staged_rows(stage, i0, half + i0, dst);  // columns i0.., half + i0..
    }
  } else {
#pragma unroll 1
    for (int i0 = 0; i0 < hd; i0 += 32) {
      uint32_t v[32];
      tmem_ld32(tcol + i0, v);
      tmem_wait_ld32(v);
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        float4 bb = make_float4(0.f, 0.f, 0.f, 0.f);
        if (bias != nullptr) bb = __ldg(reinterpret_cast<const float4*>(bias + i0 + i));
        const int c = i0 + i;
        pk[i / 2] = pack_bf16x2(fmaf(u2f(v[i]), scale, bb.x) * gain_at(gain, c),
                                fmaf(u2f(v[i + 1]), scale, bb.y) * gain_at(gain, c + 1));
        pk[i / 2 + 1] = pack_bf16x2(fmaf(u2f(v[i + 2]), scale, bb.z) * gain_at(gain, c + 2),
                                    fmaf(u2f(v[i + 3]), scale, bb.w) * gain_at(gain, c + 3));
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) st_shared_v4(stage + stage_off(lane, q), pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      store_staged_rows(stage, i0, i0 + 16, dst);  // columns i0 .. i0 + 31
    }
  }
}

}  // namespace rf
