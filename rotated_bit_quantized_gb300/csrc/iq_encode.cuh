// Encoding of one K or V row into the packed cache (shared by the append
// kernel and the fused append + attention kernel).
//
// Method source: page "sparkle mlx_streaming/core/cache/quant_kv.py":
// `rotate_last` (x @ M_b, bf16 result), the asymmetric group quantiser of
// `AsymmetricQuantizedKVCache.update_and_fetch` (64-dim groups, scale =
// (max - min) / (2^b - 1) and bias = min stored as bf16, K at 4 bits and V at
// 3 bits) and `_packed_words` (dim * bits / 32 uint32 words per row), with the
// codes packed LSB-first.
#pragma once

#include "iq_common.cuh"

namespace iq {

// The two M_b blocks 2*lane and 2*lane+1 (32 bf16 = 64 bytes) as floats.
__device__ __forceinline__ void load_row_rotation(const uint16_t* rot, int lane, float (&m)[2][4][4]) {
  const uint4* r4 = reinterpret_cast<const uint4*>(rot) + lane * 4;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 v = __ldg(r4 + c);
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      int idx = c * 8 + e * 2;  // bf16 index within the two blocks
      m[idx >> 4][(idx >> 2) & 3][idx & 3] = bf16_to_f32(w[e] & 0xFFFFu);
      m[(idx + 1) >> 4][((idx + 1) >> 2) & 3][(idx + 1) & 3] = bf16_to_f32(w[e] >> 16);
    }
  }
}

// The lane's 8 dims of a bf16 row (raw) rotated by its two M_b blocks and
// rounded to bf16: y[4c+j] = bf16( sum_{i=0..3} x[4c+i] * M_b[c][i][j] ), f32
// sum in order.  A bf16 x bf16 product is exact in f32, so each fused
// multiply-add rounds exactly like the separate product and sum.
__device__ __forceinline__ void rotate_row_bf16(const uint4 raw, const float (&m)[2][4][4], float (&y)[8]) {
  const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
  float x[8];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    x[2 * e] = bf16_to_f32(rw[e] & 0xFFFFu);
    x[2 * e + 1] = bf16_to_f32(rw[e] >> 16);
  }
  float acc[8];
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float a = __fmul_rn(x[4 * c], m[c][0][j]);
#pragma unroll
      for (int k = 1; k < 4; ++k) a = __fmaf_rn(x[4 * c + k], m[c][k][j], a);
      acc[4 * c + j] = a;
    }
#pragma unroll
  for (int e = 0; e < 8; e += 2) {  // round to bf16 in pairs (one conversion per two outputs)
    uint32_t pr;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(pr) : "f"(acc[e + 1]), "f"(acc[e]));
    y[e] = __uint_as_float(pr << 16);
    y[e + 1] = __uint_as_float(pr & 0xFFFF0000u);
  }
}

// Rotate, quantise and pack one K (BITS = 4) or V (BITS = 3) row held by a
// warp: lane l owns dims 8l..8l+7 (rotation blocks 2l, 2l+1); the 64-dim group
// g is lanes 8g..8g+7.
template <int BITS>
__device__ __forceinline__ void encode_row(const uint4 raw, const float (&m)[2][4][4], int lane, long long dst,
                                           uint32_t* codes_out, uint16_t* scales_out, uint16_t* biases_out) {
  constexpr int levels = (1 << BITS) - 1;
  float y[8];
  rotate_row_bf16(raw, m, y);
  float mn = y[0], mx = y[0];
#pragma unroll
  for (int e = 1; e < 8; ++e) {
    mn = fminf(mn, y[e]);
    mx = fmaxf(mx, y[e]);
  }
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  const float scale = __fdiv_rn(__fsub_rn(mx, mn), static_cast<float>(levels));
  const uint32_t s_bits = f32_to_bf16_bits(scale);
  const float s_hat = bf16_to_f32(s_bits);
  // code = clamp(rint(d / s_hat)) with d = y - mn and the IEEE quotient.  The
  // product d * (1/s_hat), both correctly rounded, is within 2^-19 of that
  // quotient for quotients below 16, so it rounds to the same integer unless
  // the quotient lies within 2^-15 of a half-integer.  Rows where some lane
  // meets such a quotient (or a scale outside [2^-100, 2^100], or a NaN)
  // compute the quotients themselves.  s_hat == 0 gives all-zero codes.
  // Rounding to an integer: adding 1.5 * 2^23 leaves rint(q) (half to even) in
  // the low mantissa bits for 0 <= q < 2^22 (q >= 0 here: y >= mn).
  constexpr float kRound = 12582912.0f;
  const float rcp = __frcp_rn(s_hat);
  float tq[8];
  bool slow = !(s_hat >= 0x1p-100f && s_hat <= 0x1p100f);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float qt = __fmul_rn(__fsub_rn(y[e], mn), rcp);
    tq[e] = __fadd_rn(qt, kRound);
    slow |= !(fabsf(__fsub_rn(qt, __fsub_rn(tq[e], kRound))) <= 0.5f - 0x1p-15f);
  }
  if (__any_sync(0xffffffffu, slow)) {
#pragma unroll
    for (int e = 0; e < 8; ++e)
      tq[e] = __fadd_rn(s_hat != 0.0f ? __fdiv_rn(__fsub_rn(y[e], mn), s_hat) : 0.0f, kRound);
  }
  uint32_t code[8];
#pragma unroll
  for (int e = 0; e < 8; ++e)
    code[e] = static_cast<uint32_t>(min(__float_as_int(tq[e]) - __float_as_int(kRound), levels));
  if constexpr (BITS == 4) {
    uint32_t w = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) w |= code[e] << (4 * e);
    codes_out[dst * kKWords + lane] = w;
  } else {
    uint32_t v24 = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) v24 |= code[e] << (3 * e);
    // output word w covers stream bits [32w, 32w+32): lanes a = 32w/24 and a+1
    const int a = lane < kVWords ? (4 * lane) / 3 : 0;
    const int off = lane < kVWords ? 32 * lane - 24 * a : 0;  // 0, 8 or 16
    const uint32_t lo = __shfl_sync(0xffffffffu, v24, a);
    const uint32_t hi = __shfl_sync(0xffffffffu, v24, min(a + 1, 31));
    if (lane < kVWords) codes_out[dst * kVWords + lane] = (lo >> off) | (hi << (24 - off));
  }
  // scales and biases of the 4 groups: lanes 0, 8, 16, 24 hold them
  const uint32_t b_bits = f32_to_bf16_bits(mn);
  uint32_t sg[4], bg[4];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    sg[g] = __shfl_sync(0xffffffffu, s_bits, 8 * g);
    bg[g] = __shfl_sync(0xffffffffu, b_bits, 8 * g);
  }
  if (lane < 2) {
    const uint32_t* v = lane == 0 ? sg : bg;
    uint16_t* base = lane == 0 ? scales_out : biases_out;
    *reinterpret_cast<uint2*>(base + dst * kGroups) = make_uint2(v[0] | (v[1] << 16), v[2] | (v[3] << 16));
  }
}

}  // namespace iq
