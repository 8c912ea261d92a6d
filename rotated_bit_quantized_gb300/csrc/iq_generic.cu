// libiqkv: every cache format the page's cache class can be built with, other
// than the tuned one (4-bit keys, 3-bit values, 64-dim groups, bfloat16): key
// and value widths of 2, 3, 4, 5, 6 or 8 bits, groups of 32, 64 or 128 dims,
// head_dim 256, and bfloat16 or float32 data (the page's `_init_quant` stores
// scales and biases in the keys' dtype, and `rotate_last` casts M to it).
//
// Method source: page "sparkle mlx_streaming/core/cache/quant_kv.py":
// `AsymmetricQuantizedKVCache(k_bits, v_bits, group_size)` with
// `_packed_words` (dim * bits / 32 uint32 words per row, the page's list of
// widths it is right for: 2/3/4/5/6/8), the affine group quantiser (scale =
// (max - min) / (2^b - 1), bias = min, codes LSB-first), `rotate_last`, and
// `asym_quantized_sdpa` (GQA, causal or explicit masks, softmax, P.V, output
// left in rotated space, undone here by M_b^T).
//
// The bfloat16 arithmetic is the tuned path's (same rotation, same quantiser
// rounding, same bf16 output rounding), written for run-time widths: the
// append encodes a row per warp; the attention dequantises each key and value
// row in float32 (k = s * c + b with one rounding) and accumulates scores,
// softmax and P.V in float32, split over the keys, then a merge kernel
// combines the splits.  float32 data takes the same steps with float32
// rounding in place of bfloat16: the rotation's products and sums are each
// rounded to float32 in block-row order (the f32 M blocks), the scale is kept
// as computed, queries are rotated and scaled in float32, and the scales and
// biases are read as float32.  It is a correctness-first path for these
// formats: the performance work went to the tuned format.
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

// The two f32 M blocks 2*lane and 2*lane+1 (32 floats) as m[c][i][j].
__device__ __forceinline__ void load_row_rotation_f32(const float* rot, int lane, float (&m)[2][4][4]) {
  const float4* r4 = reinterpret_cast<const float4*>(rot) + lane * 8;
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 v = __ldg(r4 + 4 * c + i);
      m[c][i][0] = v.x;
      m[c][i][1] = v.y;
      m[c][i][2] = v.z;
      m[c][i][3] = v.w;
    }
}

// The lane's 8 float32 dims rotated by its two M blocks:
// y[4c+j] = (((x0*M[0][j] + x1*M[1][j]) + x2*M[2][j]) + x3*M[3][j]) with
// x_i = x[4c+i], every product and every sum rounded to float32 (no fused
// multiply-add), i.e. a float32 row-vector times matrix taken in index order.
__device__ __forceinline__ void rotate_row_f32(const float (&x)[8], const float (&m)[2][4][4], float (&y)[8]) {
#pragma unroll
  for (int c = 0; c < 2; ++c)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float a = __fmul_rn(x[4 * c], m[c][0][j]);
#pragma unroll
      for (int i = 1; i < 4; ++i) a = __fadd_rn(a, __fmul_rn(x[4 * c + i], m[c][i][j]));
      y[4 * c + j] = a;
    }
}

// Load the lane's 8 dims of row `row` of a [.., D] array of the data dtype
// and rotate them (rounded to that dtype).
template <bool F32>
__device__ __forceinline__ void load_rotate_row(const void* base, long long row, int lane, const float (&m)[2][4][4],
                                                float (&y)[8]) {
  if constexpr (F32) {
    const float4* p4 = reinterpret_cast<const float4*>(static_cast<const float*>(base) + row * kHeadDim + lane * 8);
    const float4 a = __ldg(p4), b = __ldg(p4 + 1);
    const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    rotate_row_f32(x, m, y);
  } else {
    const uint4 raw =
        __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + row * kHeadDim + lane * 8));
    rotate_row_bf16(raw, m, y);
  }
}

template <bool F32>
__device__ __forceinline__ void load_rotation(const void* rot, int lane, float (&m)[2][4][4]) {
  if constexpr (F32)
    load_row_rotation_f32(static_cast<const float*>(rot), lane, m);
  else
    load_row_rotation(static_cast<const uint16_t*>(rot), lane, m);
}

// Quantise and pack one rotated row held by a warp (y: the lane's 8 dims,
// already rounded to the data dtype) with `bits`-bit codes and `gs`-dim
// groups: lane l owns dims 8l..8l+7, group g is lanes
// g*gs/8 .. (g+1)*gs/8 - 1, the lane's 8 codes are stream bits
// [8*bits*l, 8*bits*(l+1)) of the row's 8*bits words.  The scale is rounded
// to bfloat16 (bfloat16 data) or kept (float32 data) before the codes are
// formed from it; scales and biases are stored in the data dtype.
template <bool F32>
__device__ void encode_row_any(const float (&y)[8], int lane, long long dst, int bits, int gs, uint32_t* codes_out,
                               void* scales_out, void* biases_out) {
  const int levels = (1 << bits) - 1;
  const int words = 8 * bits, span = 8 * bits, ng = kHeadDim / gs;
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
  const uint32_t s_bits = F32 ? __float_as_uint(scale) : f32_to_bf16_bits(scale);
  const float s_hat = F32 ? scale : bf16_to_f32(s_bits);
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
  const uint32_t b_bits = F32 ? __float_as_uint(mn) : f32_to_bf16_bits(mn);
  const int src = min(lane, ng - 1) * (gs / 8);
  const uint32_t sg = __shfl_sync(0xffffffffu, s_bits, src);
  const uint32_t bg = __shfl_sync(0xffffffffu, b_bits, src);
  if (lane < ng) {
    if constexpr (F32) {
      static_cast<uint32_t*>(scales_out)[dst * ng + lane] = sg;
      static_cast<uint32_t*>(biases_out)[dst * ng + lane] = bg;
    } else {
      static_cast<uint16_t*>(scales_out)[dst * ng + lane] = static_cast<uint16_t>(sg);
      static_cast<uint16_t*>(biases_out)[dst * ng + lane] = static_cast<uint16_t>(bg);
    }
  }
}

struct AppendArgs {
  const void* keys;
  const void* values;
  uint32_t* k_codes;
  void* k_scales;
  void* k_biases;
  uint32_t* v_codes;
  void* v_scales;
  void* v_biases;
  const void* rot;
  int heads, n, cap, kbits, vbits, gs;
  int lens[IQ_MAX_BATCH];
};

// One warp per token row (sequence b, kv head h, token i); blockIdx.y = b * heads + h.
template <bool F32>
__global__ void __launch_bounds__(256) append_any_kernel(const __grid_constant__ AppendArgs p) {
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  float m[2][4][4];
  load_rotation<F32>(p.rot, lane, m);
  const long long dst0 = static_cast<long long>(bh) * p.cap + p.lens[bh / p.heads];
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < p.n; i += warps) {
    const long long row = static_cast<long long>(bh) * p.n + i;
    float yk[8], yv[8];
    load_rotate_row<F32>(p.keys, row, lane, m, yk);
    load_rotate_row<F32>(p.values, row, lane, m, yv);
    encode_row_any<F32>(yk, lane, dst0 + i, p.kbits, p.gs, p.k_codes, p.k_scales, p.k_biases);
    encode_row_any<F32>(yv, lane, dst0 + i, p.vbits, p.gs, p.v_codes, p.v_scales, p.v_biases);
  }
}

// ------------------------------------------------------------------ attention

struct AttendArgs {
  const uint32_t* k_codes;
  const void* k_scales;
  const void* k_biases;
  const uint32_t* v_codes;
  const void* v_scales;
  const void* v_biases;
  const void* q;
  const void* rot;
  void* out;
  float* part_o;   // [B*Hkv][rtiles][nch][8][256]
  float* part_ml;  // [B*Hkv][rtiles][nch][8][2]: max (log2 units) and sum
  unsigned* status;
  const void* mask;  // mask_kind 2: float added; 3: uint8, 0 = masked; [B][nq][mask_stride]
  long long mask_stride;
  int mask_kind, out_f32;
  int kv_heads, rep, nq, cap, kbits, vbits, gs, causal, nch, rows, rtiles;
  float scale;
  int lens[IQ_MAX_BATCH];
};

// Where the lane's 8 codes of a row start: stream bit 8*bits*lane = word w0,
// bit sh (constant per lane and width).
struct LaneBits {
  int w0, sh, g;
};
__device__ __forceinline__ LaneBits lane_bits(int bits, int gs, int lane) {
  const int s = 8 * bits * lane;
  return LaneBits{s >> 5, s & 31, 8 * lane / gs};
}

// Dequantised dims 8*lane .. 8*lane+7 of row r of a staged tile, BITS-bit
// codes: s * c + b with one rounding each (c < 2^23 becomes a float exactly by
// the 2^23 magic number).  The lane's window is at most 64 bits, so two words
// hold it.  Scales and biases are bfloat16 or float32 (F32) values.
template <int BITS, bool F32>
__device__ __forceinline__ void dequant_bits(const uint32_t* codes, const uint32_t* scales, const uint32_t* biases,
                                             int r, int ng, LaneBits lb, float (&x)[8]) {
  constexpr int WORDS = 8 * BITS;
  constexpr uint32_t MASK = (1u << BITS) - 1u;
  const uint32_t* row = codes + r * WORDS;
  const uint32_t a = row[lb.w0];
  const uint32_t b = lb.w0 + 1 < WORDS ? row[lb.w0 + 1] : 0u;
  const uint32_t lo = __funnelshift_r(a, b, lb.sh), hi = __funnelshift_r(b, 0u, lb.sh);
  float s, bb;
  if constexpr (F32) {
    s = __uint_as_float(scales[r * ng + lb.g]);
    bb = __uint_as_float(biases[r * ng + lb.g]);
  } else {
    s = bf16_to_f32(reinterpret_cast<const uint16_t*>(scales)[r * ng + lb.g]);
    bb = bf16_to_f32(reinterpret_cast<const uint16_t*>(biases)[r * ng + lb.g]);
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int off = BITS * e;
    uint32_t c;
    if (off + BITS <= 32)
      c = (lo >> off) & MASK;
    else if (off >= 32)
      c = (hi >> (off - 32)) & MASK;
    else
      c = __funnelshift_r(lo, hi, off) & MASK;
    x[e] = fmaf(s, __uint_as_float(0x4B000000u | c) - 8388608.0f, bb);
  }
}

template <bool F32>
__device__ __forceinline__ void dequant_lane(const uint32_t* codes, const uint32_t* scales, const uint32_t* biases,
                                             int r, int bits, int ng, LaneBits lb, float (&x)[8]) {
  switch (bits) {  // uniform over the grid
    case 2: dequant_bits<2, F32>(codes, scales, biases, r, ng, lb, x); break;
    case 3: dequant_bits<3, F32>(codes, scales, biases, r, ng, lb, x); break;
    case 4: dequant_bits<4, F32>(codes, scales, biases, r, ng, lb, x); break;
    case 5: dequant_bits<5, F32>(codes, scales, biases, r, ng, lb, x); break;
    case 6: dequant_bits<6, F32>(codes, scales, biases, r, ng, lb, x); break;
    default: dequant_bits<8, F32>(codes, scales, biases, r, ng, lb, x); break;
  }
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

constexpr int kTileKeys = 32;                                // keys per staged tile
constexpr int kTileCodeBytes = kTileKeys * kHeadDim;         // 32 rows x 256 B (8-bit codes at most)
constexpr int kTileMetaBytes = kTileKeys * (kHeadDim / 32) * 4;  // 32 rows x 8 groups x f32 at most

struct Stage {
  uint32_t kc[kTileCodeBytes / 4];
  uint32_t vc[kTileCodeBytes / 4];
  uint32_t ks[kTileMetaBytes / 4], kb[kTileMetaBytes / 4], vs[kTileMetaBytes / 4], vb[kTileMetaBytes / 4];
};

// grid (nch, B*Hkv, rtiles), 128 threads.  CTA (x, bh, z): the 8 query rows of
// tile z over key split x (a multiple of 32 keys).  The split's keys pass
// through shared memory in 32-key tiles, two in flight (cp.async, 16-byte
// pieces: every row and every tile's scale block starts 16-byte aligned).
// Warp w takes keys 8w .. 8w+7 of each tile, four at a time, for all 8 rows,
// so every key is dequantised once: lane l holds dims 8l .. 8l+7 of the rows'
// queries and of the keys and values; the 32 (key, row) dot products of a
// batch are summed over the lanes by a butterfly that leaves the sum for key
// l/8 and row l%8 in lane l, which applies the masks and the row's lazily
// moving reference max (softmax in log2 units, P <= 2^8); the 32
// probabilities are gathered back for P.V.  At the end the four warps' states
// merge through shared memory into the CTA's partial.  F32: float32 queries,
// rotation, scales and biases.
template <bool F32>
__global__ void __launch_bounds__(128) attend_any_kernel(const __grid_constant__ AttendArgs p) {
  constexpr float LOG2E = 1.4426950408889634f;
  constexpr float NEG = -__builtin_huge_valf();
  constexpr float TAU = 8.0f;  // a row's reference moves only when a score passes it by 2^8
  __shared__ __align__(16) Stage st[2];
  static_assert(sizeof(Stage) * 2 >= 4 * 8 * kHeadDim * 4 + 4 * 8 * 2 * 4 && sizeof(Stage) >= 8 * kHeadDim * 4,
                "the stages hold the query rows and, after the loop, the warps' states");
  const int x = blockIdx.x, bh = blockIdx.y, z = blockIdx.z;
  const int b = bh / p.kv_heads, h = bh % p.kv_heads;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = p.lens[b];
  const int per = ((T + p.nch - 1) / p.nch + kTileKeys - 1) / kTileKeys * kTileKeys;
  const int c0 = x * per;

  // q'' = rnd(rnd(q @ M) * scale) of the tile's 8 rows (warp w rotates rows 2w,
  // 2w+1), rnd rounding to the data dtype (M = M_b for bfloat16 data); every
  // warp then reads the lane's 8 dims of all 8 rows
  float* qsh = reinterpret_cast<float*>(&st[1]);  // [8 rows][256] (st[1] is staged after this)
  {
    float m[2][4][4];
    load_rotation<F32>(p.rot, lane, m);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int R = 8 * z + 2 * warp + j, i = R / p.rep, hr = R % p.rep;
      float y[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (R < p.rows) {
        const long long qrow = (static_cast<long long>(b) * p.kv_heads * p.rep + h * p.rep + hr) * p.nq + i;
        load_rotate_row<F32>(p.q, qrow, lane, m, y);
      }
#pragma unroll
      for (int d = 0; d < 8; ++d)
        qsh[(2 * warp + j) * kHeadDim + 8 * lane + d] =
            F32 ? __fmul_rn(y[d], p.scale) : round_bf16(__fmul_rn(y[d], p.scale));
    }
  }
  __syncthreads();
  float qq[8][8];
#pragma unroll
  for (int r = 0; r < 8; ++r)
#pragma unroll
    for (int d = 0; d < 8; ++d) qq[r][d] = qsh[r * kHeadDim + 8 * lane + d];
  // this lane's row in the softmax phase: row (lane % 8) of the tile
  const int myr = lane & 7;
  int qpos_l, qidx_l;
  {
    const int R = 8 * z + myr, i = R / p.rep;
    qidx_l = min(i, p.nq - 1);
    qpos_l = R < p.rows ? (p.causal ? T - p.nq + i : T - 1) : -1;
  }
  int cmax;  // the last key some row of the tile may see
  {
    const int R = min(8 * z + 7, p.rows - 1), i = R / p.rep;
    cmax = p.causal ? T - p.nq + i : T - 1;
  }
  const int c1 = min(min(T, c0 + per), cmax + 1);  // keys [c0, c1) of the split matter to the tile
  __syncthreads();  // every warp has its query dims before st[1] is staged

  // staging of tile [t, t + 32): codes rows, then the scale and bias blocks
  const int kbytes = kTileKeys * 32 * p.kbits, vbytes = kTileKeys * 32 * p.vbits;
  constexpr int esz = F32 ? 4 : 2;  // bytes per scale or bias
  const int ng = kHeadDim / p.gs, mbytes = kTileKeys * ng * esz;
  const LaneBits klb = lane_bits(p.kbits, p.gs, lane), vlb = lane_bits(p.vbits, p.gs, lane);
  const long long row0 = static_cast<long long>(bh) * p.cap;
  auto stage = [&](int s, int t) {
    const uint8_t* kc = reinterpret_cast<const uint8_t*>(p.k_codes) + (row0 + t) * 32 * p.kbits;
    const uint8_t* vc = reinterpret_cast<const uint8_t*>(p.v_codes) + (row0 + t) * 32 * p.vbits;
    for (int o = threadIdx.x * 16; o < kbytes; o += blockDim.x * 16)
      cp_async16(reinterpret_cast<uint8_t*>(st[s].kc) + o, kc + o);
    for (int o = threadIdx.x * 16; o < vbytes; o += blockDim.x * 16)
      cp_async16(reinterpret_cast<uint8_t*>(st[s].vc) + o, vc + o);
    const long long mo = (row0 + t) * ng * esz;
    for (int o = threadIdx.x * 16; o < 4 * mbytes; o += blockDim.x * 16) {
      const int which = o / mbytes, oo = o % mbytes;
      const void* src = which == 0 ? p.k_scales : which == 1 ? p.k_biases : which == 2 ? p.v_scales : p.v_biases;
      uint32_t* dst = which == 0 ? st[s].ks : which == 1 ? st[s].kb : which == 2 ? st[s].vs : st[s].vb;
      cp_async16(reinterpret_cast<uint8_t*>(dst) + oo, static_cast<const uint8_t*>(src) + mo + oo);
    }
  };

  // softmax state: the lane's row reference and partial row sum; O of all 8
  // rows over the lane's 8 dims
  float mref = NEG, lpart = 0.f, o[8][8];
#pragma unroll
  for (int r = 0; r < 8; ++r)
#pragma unroll
    for (int d = 0; d < 8; ++d) o[r][d] = 0.f;

  const int ntiles = c1 > c0 ? (c1 - c0 + kTileKeys - 1) / kTileKeys : 0;
  if (ntiles > 0) stage(0, c0);
  cp_async_commit();
  for (int it = 0; it < ntiles; ++it) {
    if (it + 1 < ntiles) stage((it + 1) & 1, c0 + (it + 1) * kTileKeys);
    cp_async_commit();
    cp_async_wait_1();  // tile it has landed (the next one may still be in flight)
    __syncthreads();
    const Stage& S = st[it & 1];
    const int tbase = c0 + it * kTileKeys;
    const int nk = min(kTileKeys, c1 - tbase);
#pragma unroll 1
    for (int k0 = 8 * warp; k0 < 8 * warp + 8 && k0 < nk; k0 += 4) {
      // partial dot products of the batch's 4 keys with the 8 rows: value key*8 + row
      float val[32];
      {
        float kx[4][8];
#pragma unroll
        for (int u = 0; u < 4; ++u) dequant_lane<F32>(S.kc, S.ks, S.kb, min(k0 + u, nk - 1), p.kbits, ng, klb, kx[u]);
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            float acc = 0.f;
#pragma unroll
            for (int d = 0; d < 8; ++d) acc = fmaf(qq[r][d], kx[u][d], acc);
            val[8 * u + r] = acc;
          }
      }
      // butterfly reduce-scatter: after step b the lane keeps the half of its
      // values whose index bit (4 - b) equals its lane bit (4 - b); lane l ends
      // with the full sum of value l
#pragma unroll
      for (int lev = 0; lev < 5; ++lev) {
        const int hn = 16 >> lev, msk = 16 >> lev;
        const bool up = (lane & msk) != 0;
#pragma unroll
        for (int i = 0; i < hn; ++i) {
          const float send = up ? val[i] : val[i + hn];
          const float keep = up ? val[i + hn] : val[i];
          val[i] = keep + __shfl_xor_sync(0xffffffffu, send, msk);
        }
      }
      // the lane's (key, row): masks, then the lazily moving row reference
      const int kr = k0 + (lane >> 3), t = tbase + kr;
      float s = val[0] * LOG2E;
      if (kr >= nk || t > qpos_l) s = NEG;
      if (s != NEG && p.mask_kind == 2) {
        s = fmaf(__ldg(static_cast<const float*>(p.mask) + (static_cast<long long>(b) * p.nq + qidx_l) * p.mask_stride + t),
                 LOG2E, s);
      } else if (s != NEG && p.mask_kind == 3) {
        if (__ldg(static_cast<const uint8_t*>(p.mask) + (static_cast<long long>(b) * p.nq + qidx_l) * p.mask_stride + t) ==
            0)
          s = kMaskedScore * LOG2E;
      }
      const bool move = s != NEG && (mref == NEG || s > mref + TAU);
      if (__any_sync(0xffffffffu, move)) {
        float mx = s;  // the row's max over the batch's 4 keys (lanes l, l^8, l^16, l^24)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const bool mv = mx != NEG && (mref == NEG || mx > mref + TAU);
        const float mnew = mv ? (mref == NEG ? mx : fmaxf(mref, mx)) : mref;
        const float al = !mv ? 1.f : mref == NEG ? 0.f : ex2_approx(mref - mnew);
        lpart *= al;
        mref = mnew;
#pragma unroll
        for (int r = 0; r < 8; ++r) {  // every lane's O of row r: the factor of lane r
          const float ar = __shfl_sync(0xffffffffu, al, r);
#pragma unroll
          for (int d = 0; d < 8; ++d) o[r][d] *= ar;
        }
      }
      const float pr = s == NEG ? 0.f : ex2_approx(s - mref);
      lpart += pr;
      // P.V: the values of the 4 keys, each weighted by the row's probability
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float vx[8];
        dequant_lane<F32>(S.vc, S.vs, S.vb, min(k0 + u, nk - 1), p.vbits, ng, vlb, vx);
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const float pw = __shfl_sync(0xffffffffu, pr, 8 * u + r);  // 0 for keys past the tile
#pragma unroll
          for (int d = 0; d < 8; ++d) o[r][d] = fmaf(pw, vx[d], o[r][d]);
        }
      }
    }
    __syncthreads();  // every warp is done with this stage before it is refilled
  }
  // merge the four warps' states through shared memory (the stages are free):
  // per warp and row the reference max and the row sum, then O
  float lrow = lpart;
  lrow += __shfl_xor_sync(0xffffffffu, lrow, 8);
  lrow += __shfl_xor_sync(0xffffffffu, lrow, 16);
  float* wo = reinterpret_cast<float*>(&st[0]);  // [4 warps][8 rows][256]
  float* wml = wo + 4 * 8 * kHeadDim;            // [4 warps][8 rows][2]
  cp_async_wait_1();
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  if (lane < 8) {
    wml[(warp * 8 + lane) * 2] = mref;
    wml[(warp * 8 + lane) * 2 + 1] = lrow;
  }
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    float4* dst = reinterpret_cast<float4*>(wo + (warp * 8 + r) * kHeadDim + 8 * lane);
    dst[0] = make_float4(o[r][0], o[r][1], o[r][2], o[r][3]);
    dst[1] = make_float4(o[r][4], o[r][5], o[r][6], o[r][7]);
  }
  __syncthreads();
  // the split's partial of the tile's rows: thread (row r = warp*2 + j, lane) merges dims 8*lane .. +7
  const long long slot = (static_cast<long long>(bh) * p.rtiles + z) * p.nch + x;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int r = 2 * warp + j;
    float M = NEG;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, wml[(w * 8 + r) * 2]);
    float L = 0.f, acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float mw = wml[(w * 8 + r) * 2];
      if (mw == NEG) continue;
      const float a = ex2_approx(mw - M);
      L = fmaf(wml[(w * 8 + r) * 2 + 1], a, L);
      const float4* src = reinterpret_cast<const float4*>(wo + (w * 8 + r) * kHeadDim + 8 * lane);
      const float4 u0 = src[0], u1 = src[1];
      const float u[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
      for (int d = 0; d < 8; ++d) acc[d] = fmaf(u[d], a, acc[d]);
    }
    const long long rr = slot * 8 + r;
    float4* dst = reinterpret_cast<float4*>(p.part_o + rr * kHeadDim + 8 * lane);
    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    if (lane == 0) {
      p.part_ml[rr * 2] = M;
      p.part_ml[rr * 2 + 1] = L;
    }
  }
}

// grid (B*Hkv, rtiles), 256 threads: thread (row r, lane) merges dims
// 8*lane .. 8*lane+7 of row 8*z + r over the splits, normalises, undoes the
// rotation (out[4c+i] = sum_j o[4c+j] * M[c][i][j], M = M_b for bfloat16
// data) and stores.
template <bool F32>
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
    const float a = M == -__builtin_huge_valf() ? 0.f : ex2_approx(M - Mn), w = ex2_approx(mx - Mn);
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
  load_rotation<F32>(p.rot, lane, m);
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

bool tuned_format(const iq_cache* c) {
  return c->dtype == IQ_DTYPE_BF16 && c->group_size == kGroup && c->k_bits == 4 && c->v_bits == 3;
}

bool format_supported(int head_dim, int group_size, int k_bits, int v_bits) {
  return head_dim == kHeadDim && gen::supported_group(group_size) && gen::supported_bits(k_bits) &&
         gen::supported_bits(v_bits);
}

int append_any(iq_cache* c, const void* keys, const void* values, int n, const void* rot, iq_stream_t stream) {
  gen::AppendArgs p;
  std::memset(&p, 0, sizeof(p));
  p.keys = keys;
  p.values = values;
  p.k_codes = c->k_codes;
  p.k_scales = c->k_scales;
  p.k_biases = c->k_biases;
  p.v_codes = c->v_codes;
  p.v_scales = c->v_scales;
  p.v_biases = c->v_biases;
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
  const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(bh));
  if (c->dtype == IQ_DTYPE_F32)
    gen::append_any_kernel<true><<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(p);
  else
    gen::append_any_kernel<false><<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(p);
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

int attend_any(const iq_cache* c, const void* q, int q_heads, int n_queries, float scale, int causal,
               const void* rot, void* out, int out_f32, void* workspace, size_t workspace_bytes,
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
  p.k_scales = c->k_scales;
  p.k_biases = c->k_biases;
  p.v_codes = c->v_codes;
  p.v_scales = c->v_scales;
  p.v_biases = c->v_biases;
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
  const dim3 grid(static_cast<unsigned>(p.nch), bh, static_cast<unsigned>(p.rtiles));
  const dim3 mgrid(bh, static_cast<unsigned>(p.rtiles));
  if (c->dtype == IQ_DTYPE_F32) {
    gen::attend_any_kernel<true><<<grid, 128, 0, s>>>(p);
    IQ_CUDA(cudaGetLastError());
    gen::merge_any_kernel<true><<<mgrid, 256, 0, s>>>(p);
  } else {
    gen::attend_any_kernel<false><<<grid, 128, 0, s>>>(p);
    IQ_CUDA(cudaGetLastError());
    gen::merge_any_kernel<false><<<mgrid, 256, 0, s>>>(p);
  }
  IQ_CUDA(cudaGetLastError());
  return IQ_OK;
}

}  // namespace iq
