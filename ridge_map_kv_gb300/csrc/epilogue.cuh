// Shared epilogue step: one attention head of one accumulator row, read from
// TMEM, optionally scaled and biased, optionally rotated (rotate-half RoPE with
// a cos/sin table row), rounded to bf16 and written with 16-byte stores.
//
// Every tcgen05.ld here is warp-collective, so all lanes call emit_head with the
// same (tcol, hd, rope) and only `valid` differs per lane (it guards the stores).
#pragma once
#include "rf_device.cuh"

namespace rf {

// acc column c (0 <= c < hd) of this thread's row lives at TMEM column tcol + c.
// out[c] = bf16(f((acc[c] * scale + bias[c]) * gain[c])), with f = RoPE at the
// table row (cs, sn) when `rope`, else the identity. bias and gain may be nullptr.
__device__ __forceinline__ float gain_at(const __nv_bfloat16* __restrict__ gain, int c) {
  return gain != nullptr ? __bfloat162float(gain[c]) : 1.0f;
}

__device__ __forceinline__ void emit_head(uint32_t tcol, int hd, float scale, const float* __restrict__ bias,
                                          const __nv_bfloat16* __restrict__ gain, bool rope,
                                          const float* __restrict__ cs, const float* __restrict__ sn,
                                          __nv_bfloat16* dst, bool valid) {
  const int half = hd >> 1;
  if (rope) {
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
        const float4 c4 = *reinterpret_cast<const float4*>(cs + i0 + i);
        const float4 s4 = *reinterpret_cast<const float4*>(sn + i0 + i);
        float4 b1 = make_float4(0.f, 0.f, 0.f, 0.f), b2 = b1;
        if (bias != nullptr) {
          b1 = __ldg(reinterpret_cast<const float4*>(bias + i0 + i));
          b2 = __ldg(reinterpret_cast<const float4*>(bias + half + i0 + i));
        }
        const float cc[4] = {c4.x, c4.y, c4.z, c4.w};
        const float ssn[4] = {s4.x, s4.y, s4.z, s4.w};
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
      if (valid) {
        st_global_v4(dst + i0, o1[0], o1[1], o1[2], o1[3]);
        st_global_v4(dst + i0 + 8, o1[4], o1[5], o1[6], o1[7]);
        st_global_v4(dst + half + i0, o2[0], o2[1], o2[2], o2[3]);
        st_global_v4(dst + half + i0 + 8, o2[4], o2[5], o2[6], o2[7]);
      }
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
      if (valid) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          st_global_v4(dst + i0 + 8 * q, pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      }
    }
  }
}

}  // namespace rf
