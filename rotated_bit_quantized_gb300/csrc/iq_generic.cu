// libiqkv: every cache format the page's cache class can be built with, other
// than the tuned one (4-bit keys, 3-bit values, 64-dim groups): key and value
// widths of 2, 3, 4, 5, 6 or 8 bits and groups of 32, 64 or 128 dims, head_dim
// 256, bf16 scales and biases.
//
// Method source: page "sparkle mlx_streaming/core/cache/quant_kv.py":
// `AsymmetricQuantizedKVCache(k_bits, v_bits, group_size)` with
// `_packed_words` (dim * bits / 32 uint32 words per row, the page's list of
// widths it is right for: 2/3/4/5/6/8), the affine group quantiser (scale =
// (max - min) / (2^b - 1), bias = min, codes LSB-first), `rotate_last`, and
// `asym_quantized_sdpa` (GQA, causal or explicit masks, softmax, P.V, output
// left in rotated space, undone here by M_b^T).
//
// The arithmetic is the tuned path's (same rotation, same quantiser rounding,
// same bf16 output rounding), written for run-time widths: the append encodes
// a row per warp; the attention dequantises each key and value row in float32
// (k = s * c + b with one rounding) and accumulates scores, softmax and P.V in
// float32, split over the keys, then a merge kernel combines the splits.  It
// is a correctness-first path for these formats: the performance work went to
// the tuned format.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>

#include "iq_common.cuh"
#include "iq_encode.cuh"

namespace iq {
namespace gen {

constexpr int kMaxRowTiles = 8;  // query rows per (sequence, kv head): at most 8 tiles of 8
constexpr int kMaxChunks = 512;  // key splits per (sequence, kv head, row tile)
constexpr float kMaskedScore = -1e6f;  // a key a bool mask hides (as the tuned kernels)

bool supported_bits(int b) { return b == 2 || b == 3 || b == 4 || b == 5 || b == 6 || b == 8; }
bool supported_group(int g) { return g == 32 || g == 64 || g == 128; }

// ------------------------------------------------------------------ encode

// Rotate, quantise and pack one row held by a warp with `bits`-bit codes and
// `gs`-dim groups: lane l owns dims 8l..8l+7, group g is lanes
// g*gs/8 .. (g+1)*gs/8 - 1, the lane's 8 codes are stream bits
// [8*bits*l, 8*bits*(l+1)) of the row's 8*bits words.
__device__ void encode_row_any(const uint4 raw, const float (&m)[2][4][4], int lane, long long dst, int bits, int gs,
                               uint32_t* codes_out, uint16_t* scales_out, uint16_t* biases_out) {
  const int levels = (1 << bits) - 1;
  const int words = 8 * bits, span = 8 * bits, ng = kHeadDim / gs;
  float y[8];
  rotate_row_bf16(raw, m, y);
  float mn = y[0], mx = y[0];
#pragma unroll
  for (int e = 1; e < 8; ++e) {
    mn = fminf(mn, y[e]);
    mx = fmaxf(mx, y[e]);
  }
  for (int o = 1; o < gs / 8; o <<= 1) {  // the group's lanes (xor stays inside it)
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  const float scale = __fdiv_rn(__fsub_rn(mx, mn), static_cast<float>(levels));
  const uint32_t s_bits = f32_to_bf16_bits(scale);
  const float s_hat = bf16_to_f32(s_bits);
  // code = clamp(rint(d / s_hat)), d = y - mn, IEEE quotient.  The product
  // d * (1/s_hat) (both correctly rounded) is within 3 * 2^-24 * q of that
  // quotient, below 2^-14 for q < 256, so it rounds the same way unless it lies
  // within 2^-13 of a half-integer; rows where some lane meets one (or a scale
  // outside [2^-100, 2^100], or a NaN) divide.  Adding 1.5 * 2^23 leaves
  // rint(q) (half to even) in the low mantissa bits for 0 <= q < 2^22.
  constexpr float kRound = 12582912.0f;
  const float rcp = __frcp_rn(s_hat);
  float tq[8];
  bool slow = !(s_hat >= 0x1p-100f && s_hat <= 0x1p100f);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float qt = __fmul_rn(__fsub_rn(y[e], mn), rcp);
    tq[e] = __fadd_rn(qt, kRound);
    slow |= !(fabsf(__fsub_rn(qt, __fsub_rn(tq[e], kRound))) <= 0.5f - 0x1p-13f);
  }
  if (__any_sync(0xffffffffu, slow)) {
#pragma unroll
    for (int e = 0; e < 8; ++e)
      tq[e] = __fadd_rn(s_hat != 0.0f ? __fdiv_rn(__fsub_rn(y[e], mn), s_hat) : 0.0f, kRound);
  }
  unsigned long long chunk = 0;  // the lane's 8*bits stream bits
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const unsigned long long c =
        static_cast<unsigned long long>(min(__float_as_int(tq[e]) - __float_as_int(kRound), levels));
    chunk |= c << (bits * e);
  }
  // output word w = stream bits [32w, 32w+32): from lane a = 32w / span at
  // offset 32w - span*a, and from lane a+1 when the word runs past lane a's bits
  const uint32_t clo = static_cast<uint32_t>(chunk), chi = static_cast<uint32_t>(chunk >> 32);
  for (int it = 0; it < (words + 31) / 32; ++it) {
    const int w = lane + 32 * it;
    const int a = min((32 * w) / span, 31), b = min(a + 1, 31);
    const int off = 32 * w - span * a;
    const unsigned long long ca = static_cast<unsigned long long>(__shfl_sync(0xffffffffu, clo, a)) |
                                  static_cast<unsigned long long>(__shfl_sync(0xffffffffu, chi, a)) << 32;
    const unsigned long long cb = static_cast<unsigned long long>(__shfl_sync(0xffffffffu, clo, b)) |
                                  static_cast<unsigned long long>(__shfl_sync(0xffffffffu, chi, b)) << 32;
    if (w < words) {
      unsigned long long v = ca >> off;
      if (off + 32 > span) v |= cb << (span - off);
      codes_out[dst * words + w] = static_cast<uint32_t>(v);
    }
  }
  // scales and biases: group g's values from its first lane
  const uint32_t b_bits = f32_to_bf16_bits(mn);
  const int src = min(lane, ng - 1) * (gs / 8);
  const uint32_t sg = __shfl_sync(0xffffffffu, s_bits, src);
  const uint32_t bg = __shfl_sync(0xffffffffu, b_bits, src);
  if (lane < ng) {
    scales_out[dst * ng + lane] = static_cast<uint16_t>(sg);
    biases_out[dst * ng + lane] = static_cast<uint16_t>(bg);
  }
}

struct AppendArgs {
  const uint16_t* keys;
  const uint16_t* values;
  uint32_t* k_codes;
  uint16_t* k_scales;
  uint16_t* k_biases;
  uint32_t* v_codes;
  uint16_t* v_scales;
  uint16_t* v_biases;
  const uint16_t* rot;
  int heads, n, cap, kbits, vbits, gs;
  int lens[IQ_MAX_BATCH];
};

// One warp per token row (sequence b, kv head h, token i); blockIdx.y = b * heads + h.
__global__ void __launch_bounds__(256) append_any_kernel(const __grid_constant__ AppendArgs p) {
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  float m[2][4][4];
  load_row_rotation(p.rot, lane, m);
  const long long dst0 = static_cast<long long>(bh) * p.cap + p.lens[bh / p.heads];
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < p.n; i += warps) {
    const long long src = (static_cast<long long>(bh) * p.n + i) * kHeadDim + lane * 8;
    const uint4 rk = __ldg(reinterpret_cast<const uint4*>(p.keys + src));
    const uint4 rv = __ldg(reinterpret_cast<const uint4*>(p.values + src));
    encode_row_any(rk, m, lane, dst0 + i, p.kbits, p.gs, p.k_codes, p.k_scales, p.k_biases);
    encode_row_any(rv, m, lane, dst0 + i, p.vbits, p.gs, p.v_codes, p.v_scales, p.v_biases);
  }
}

// ------------------------------------------------------------------ attention

struct AttendArgs {
  const uint32_t* k_codes;
  const uint16_t* k_scales;
  const uint16_t* k_biases;
  const uint32_t* v_codes;
  const uint16_t* v_scales;
  const uint16_t* v_biases;
  const uint16_t* q;
  const uint16_t* rot;
  void* out;
  float* part_o;   // [B*Hkv][rtiles][nch][8][256]
  float* part_ml;  // [B*Hkv][rtiles][nch][8][2]: max and sum (natural-log units)
  unsigned* status;
  const void* mask;  // mask_kind 2: float added; 3: uint8, 0 = masked; [B][nq][mask_stride]
  long long mask_stride;
  int mask_kind, out_f32;
  int kv_heads, rep, nq, cap, kbits, vbits, gs, causal, nch, rows, rtiles;
  float scale;
  int lens[IQ_MAX_BATCH];
};

// The lane's 8 codes of a packed row: stream bits [8*bits*lane, 8*bits*(lane+1)).
__device__ __forceinline__ unsigned long long lane_codes(const uint32_t* row, int bits, int lane) {
  const int words = 8 * bits;
  const int s = 8 * bits * lane, w0 = s >> 5, sh = s & 31;
  const unsigned long long lo = __ldg(row + w0);
  const unsigned long long hi = w0 + 1 < words ? __ldg(row + w0 + 1) : 0ull;
  unsigned long long v = (lo | hi << 32) >> sh;
  if (sh && w0 + 2 < words) v |= static_cast<unsigned long long>(__ldg(row + w0 + 2)) << (64 - sh);
  return v;
}

// Dequantised dims 8*lane .. 8*lane+7 of a row: s * c + b, one rounding each.
__device__ __forceinline__ void dequant_lane(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases,
                                             long long row, int bits, int gs, int lane, float (&x)[8]) {
  const int ng = kHeadDim / gs, g = 8 * lane / gs;
  const unsigned long long v = lane_codes(codes + row * 8 * bits, bits, lane);
  const float s = bf16_to_f32(__ldg(scales + row * ng + g)), b = bf16_to_f32(__ldg(biases + row * ng + g));
  const unsigned long long mask = (1ull << bits) - 1;
#pragma unroll
  for (int e = 0; e < 8; ++e) x[e] = fmaf(s, static_cast<float>((v >> (bits * e)) & mask), b);
}

// grid (nch, B*Hkv, rtiles), 128 threads.  CTA (x, bh, z): the 8 query rows of
// tile z over key split x; its 4 warps take every 4th key, then merge.
__global__ void __launch_bounds__(128) attend_any_kernel(const __grid_constant__ AttendArgs p) {
  __shared__ float s_ml[4][8][2];
  __shared__ float s_o[4][8][kHeadDim];
  const int x = blockIdx.x, bh = blockIdx.y, z = blockIdx.z;
  const int b = bh / p.kv_heads, h = bh % p.kv_heads;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = p.lens[b];
  const int per = (T + p.nch - 1) / p.nch;
  const int c0 = x * per, c1 = min(T, c0 + per);

  float m[2][4][4];
  load_row_rotation(p.rot, lane, m);
  // q'' = bf16(bf16(q @ M_b) * scale) of the tile's rows, the lane's 8 dims
  float qq[8][8];
  int qpos[8], qidx[8];
  bool rv[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int R = 8 * z + r, i = R / p.rep, hr = R % p.rep;
    rv[r] = R < p.rows;
    qidx[r] = min(i, p.nq - 1);
    qpos[r] = p.causal ? T - p.nq + i : T - 1;
    uint4 raw = make_uint4(0, 0, 0, 0);
    if (rv[r]) {
      const long long qrow = (static_cast<long long>(b) * p.kv_heads * p.rep + h * p.rep + hr) * p.nq + i;
      raw = __ldg(reinterpret_cast<const uint4*>(p.q + qrow * kHeadDim + 8 * lane));
    }
    float y[8];
    rotate_row_bf16(raw, m, y);
#pragma unroll
    for (int d = 0; d < 8; ++d) qq[r][d] = round_bf16(__fmul_rn(y[d], p.scale));
  }

  float mrow[8], lrow[8], o[8][8];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    mrow[r] = -__builtin_huge_valf();
    lrow[r] = 0.f;
#pragma unroll
    for (int d = 0; d < 8; ++d) o[r][d] = 0.f;
  }
  const long long rowbase = static_cast<long long>(bh) * p.cap;
  for (int t = c0 + warp; t < c1; t += 4) {
    float k[8], v[8];
    dequant_lane(p.k_codes, p.k_scales, p.k_biases, rowbase + t, p.kbits, p.gs, lane, k);
    dequant_lane(p.v_codes, p.v_scales, p.v_biases, rowbase + t, p.vbits, p.gs, lane, v);
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      float s = 0.f;
#pragma unroll
      for (int d = 0; d < 8; ++d) s = fmaf(qq[r][d], k[d], s);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      if (!rv[r] || t > qpos[r]) continue;  // warp-uniform
      if (p.mask_kind == 2) {
        s += __ldg(static_cast<const float*>(p.mask) + (static_cast<long long>(b) * p.nq + qidx[r]) * p.mask_stride + t);
      } else if (p.mask_kind == 3) {
        if (__ldg(static_cast<const uint8_t*>(p.mask) + (static_cast<long long>(b) * p.nq + qidx[r]) * p.mask_stride +
                  t) == 0)
          s = kMaskedScore;
      }
      const float mn = fmaxf(mrow[r], s);
      const float a = mrow[r] == -__builtin_huge_valf() ? 0.f : expf(mrow[r] - mn);
      const float pr = s == -__builtin_huge_valf() ? 0.f : expf(s - mn);
      lrow[r] = fmaf(lrow[r], a, pr);
#pragma unroll
      for (int d = 0; d < 8; ++d) o[r][d] = fmaf(o[r][d], a, pr * v[d]);
      mrow[r] = mn;
    }
  }
  // merge the 4 warps, store the split's partial
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    if (lane == 0) {
      s_ml[warp][r][0] = mrow[r];
      s_ml[warp][r][1] = lrow[r];
    }
#pragma unroll
    for (int d = 0; d < 8; ++d) s_o[warp][r][8 * lane + d] = o[r][d];
  }
  __syncthreads();
  const long long slot = (static_cast<long long>(bh) * p.rtiles + z) * p.nch + x;
  for (int it = threadIdx.x; it < 8 * kHeadDim; it += blockDim.x) {
    const int r = it / kHeadDim, d = it % kHeadDim;
    float M = s_ml[0][r][0];
    for (int w = 1; w < 4; ++w) M = fmaxf(M, s_ml[w][r][0]);
    float L = 0.f, acc = 0.f;
    if (M != -__builtin_huge_valf())
      for (int w = 0; w < 4; ++w) {
        if (s_ml[w][r][0] == -__builtin_huge_valf()) continue;
        const float wt = expf(s_ml[w][r][0] - M);
        L = fmaf(s_ml[w][r][1], wt, L);
        acc = fmaf(s_o[w][r][d], wt, acc);
      }
    p.part_o[(slot * 8 + r) * kHeadDim + d] = acc;
    if (d == 0) {
      p.part_ml[(slot * 8 + r) * 2] = M;
      p.part_ml[(slot * 8 + r) * 2 + 1] = L;
    }
  }
}

// grid (B*Hkv, rtiles), 256 threads: thread (row r, lane) merges dims
// 8*lane .. 8*lane+7 of row 8*z + r over the splits, normalises, undoes the
// rotation (out[4c+i] = sum_j o[4c+j] * M_b[c][i][j]) and stores.
__global__ void __launch_bounds__(256) merge_any_kernel(const __grid_constant__ AttendArgs p) {
  const int bh = blockIdx.x, z = blockIdx.y;
  const int r = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = 8 * z + r;
  if (R >= p.rows) return;
  const int b = bh / p.kv_heads, h = bh % p.kv_heads, i = R / p.rep, hr = R % p.rep;
  float M = -__builtin_huge_valf(), L = 0.f, acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int x = 0; x < p.nch; ++x) {
    const long long slot = ((static_cast<long long>(bh) * p.rtiles + z) * p.nch + x) * 8 + r;
    const float mx = p.part_ml[slot * 2], lx = p.part_ml[slot * 2 + 1];
    if (mx == -__builtin_huge_valf()) continue;
    const float Mn = fmaxf(M, mx);
    const float a = M == -__builtin_huge_valf() ? 0.f : expf(M - Mn), w = expf(mx - Mn);
    const float4* ox = reinterpret_cast<const float4*>(p.part_o + slot * kHeadDim + 8 * lane);
    const float4 u0 = ox[0], u1 = ox[1];
    const float u[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    L = fmaf(L, a, lx * w);
#pragma unroll
    for (int d = 0; d < 8; ++d) acc[d] = fmaf(acc[d], a, u[d] * w);
    M = Mn;
  }
  if (!(L > 0.f)) atomicOr(p.status, 4u);  // no key of the row has a finite score
  const float inv = 1.f / L;
  float m[2][4][4];
  load_row_rotation(p.rot, lane, m);
  float yv[8];
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int ii = 0; ii < 4; ++ii) {
      float s = 0.f;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) s = fmaf(acc[4 * c + jj] * inv, m[c][ii][jj], s);
      yv[4 * c + ii] = s;
    }
  const long long orow = (static_cast<long long>(b) * p.kv_heads * p.rep + h * p.rep + hr) * p.nq + i;
  if (p.out_f32) {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow * kHeadDim + 8 * lane);
    dst[0] = make_float4(yv[0], yv[1], yv[2], yv[3]);
    dst[1] = make_float4(yv[4], yv[5], yv[6], yv[7]);
  } else {
    uint4 w;
    w.x = f32_to_bf16_bits(yv[0]) | (f32_to_bf16_bits(yv[1]) << 16);
    w.y = f32_to_bf16_bits(yv[2]) | (f32_to_bf16_bits(yv[3]) << 16);
    w.z = f32_to_bf16_bits(yv[4]) | (f32_to_bf16_bits(yv[5]) << 16);
    w.w = f32_to_bf16_bits(yv[6]) | (f32_to_bf16_bits(yv[7]) << 16);
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + orow * kHeadDim + 8 * lane) = w;
  }
}

// Splits per (sequence, kv head, row tile): about four CTAs per SM in all,
// independent of the lengths (so the workspace size is too).
int chunks(int batch, int kv_heads, int rtiles) {
  const long long units = static_cast<long long>(batch) * kv_heads * rtiles;
  const long long want = (4LL * num_sms() + units - 1) / units;
  return static_cast<int>(std::max(1LL, std::min<long long>(want, kMaxChunks)));
}

}  // namespace gen

// ------------------------------------------------------------------ host entry points

bool tuned_format(const iq_cache* c) { return c->group_size == kGroup && c->k_bits == 4 && c->v_bits == 3; }

bool format_supported(int head_dim, int group_size, int k_bits, int v_bits) {
  return head_dim == kHeadDim && gen::supported_group(group_size) && gen::supported_bits(k_bits) &&
         gen::supported_bits(v_bits);
}

int append_any(iq_cache* c, const uint16_t* keys, const uint16_t* values, int n, const uint16_t* rot,
               iq_stream_t stream) {
  gen::AppendArgs p;
  std::memset(&p, 0, sizeof(p));
  p.keys = keys;
  p.values = values;
  p.k_codes = c->k_codes;
  p.k_scales = static_cast<uint16_t*>(c->k_scales);
  p.k_biases = static_cast<uint16_t*>(c->k_biases);
  p.v_codes = c->v_codes;
  p.v_scales = static_cast<uint16_t*>(c->v_scales);
  p.v_biases = static_cast<uint16_t*>(c->v_biases);
  p.rot = rot;
  p.heads = c->kv_heads;
  p.n = n;
  p.cap = c->capacity;
  p.kbits = c->k_bits;
  p.vbits = c->v_bits;
  p.gs = c->group_size;
  for (int b = 0; b < c->batch; ++b) p.lens[b] = c->lens[b];
  const int bh = c->batch * c->kv_heads;
  long long gx = (static_cast<long long>(n) + 7) / 8;
  gx = std::min<long long>(gx, std::max(1LL, static_cast<long long>(num_sms()) * 8 / bh));
  gen::append_any_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(bh)), 256, 0,
                           static_cast<cudaStream_t>(stream)>>>(p);
  IQ_CUDA(cudaGetLastError());
  return IQ_OK;
}

int attend_any_workspace(const iq_cache* c, int q_heads, int n_queries, size_t* bytes) {
  const int rows = q_heads / c->kv_heads * n_queries;
  const int rtiles = (rows + 7) / 8;
  if (rtiles > gen::kMaxRowTiles)
    return fail(IQ_ERR_UNSUPPORTED, "this cache format serves at most 64 query rows per kv head");
  const int nch = gen::chunks(c->batch, c->kv_heads, rtiles);
  const size_t slots = static_cast<size_t>(c->batch) * c->kv_heads * rtiles * nch * 8;
  *bytes = IQ_WORKSPACE_HEAD_BYTES + slots * (kHeadDim + 2) * sizeof(float);
  return IQ_OK;
}

int attend_any(const iq_cache* c, const uint16_t* q, int q_heads, int n_queries, float scale, int causal,
               const uint16_t* rot, void* out, int out_f32, void* workspace, size_t workspace_bytes,
               iq_stream_t stream, int mask_kind, const void* mask, long long mask_stride) {
  size_t need = 0;
  int st = attend_any_workspace(c, q_heads, n_queries, &need);
  if (st != IQ_OK) return st;
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 256)
    return fail(IQ_ERR_WORKSPACE, "workspace missing or not 256-byte aligned");
  if (workspace_bytes < need) return fail(IQ_ERR_WORKSPACE, "workspace smaller than iq_attend_workspace()");
  gen::AttendArgs p;
  std::memset(&p, 0, sizeof(p));
  p.k_codes = c->k_codes;
  p.k_scales = static_cast<const uint16_t*>(c->k_scales);
  p.k_biases = static_cast<const uint16_t*>(c->k_biases);
  p.v_codes = c->v_codes;
  p.v_scales = static_cast<const uint16_t*>(c->v_scales);
  p.v_biases = static_cast<const uint16_t*>(c->v_biases);
  p.q = q;
  p.rot = rot;
  p.out = out;
  p.out_f32 = out_f32 ? 1 : 0;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.status = reinterpret_cast<unsigned*>(ws);
  p.kv_heads = c->kv_heads;
  p.rep = q_heads / c->kv_heads;
  p.nq = n_queries;
  p.rows = p.rep * n_queries;
  p.rtiles = (p.rows + 7) / 8;
  p.nch = gen::chunks(c->batch, c->kv_heads, p.rtiles);
  const size_t slots = static_cast<size_t>(c->batch) * c->kv_heads * p.rtiles * p.nch * 8;
  p.part_o = reinterpret_cast<float*>(ws + IQ_WORKSPACE_HEAD_BYTES);
  p.part_ml = p.part_o + slots * kHeadDim;
  p.cap = c->capacity;
  p.kbits = c->k_bits;
  p.vbits = c->v_bits;
  p.gs = c->group_size;
  p.causal = causal;
  p.scale = scale;
  p.mask_kind = mask_kind;
  p.mask = mask;
  p.mask_stride = mask_stride;
  for (int b = 0; b < c->batch; ++b) p.lens[b] = c->lens[b];
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const unsigned bh = static_cast<unsigned>(c->batch * c->kv_heads);
  gen::attend_any_kernel<<<dim3(static_cast<unsigned>(p.nch), bh, static_cast<unsigned>(p.rtiles)), 128, 0, s>>>(p);
  IQ_CUDA(cudaGetLastError());
  gen::merge_any_kernel<<<dim3(bh, static_cast<unsigned>(p.rtiles)), 256, 0, s>>>(p);
  IQ_CUDA(cudaGetLastError());
  return IQ_OK;
}

}  // namespace iq
