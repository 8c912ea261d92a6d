// libiqkv: rotation build, cache bookkeeping, append (rotate + quantise + pack)
// and row gather.
//
// Method source: page "sparkle mlx_streaming/core/cache/quant_kv.py"
// (`_quat_left`, `_quat_right_conj`, `build_block_so4`, `rotate_last`,
// `_packed_words`, `AsymmetricQuantizedKVCache`), and page
// "sparkle mlx_streaming/mtp/kv_cache.py" (`_snapshot`/`_restore`,
// `tile_caches`, `commit_tree_row`), which the row gather serves.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "iq_common.cuh"
#include "iq_encode.cuh"

namespace iq {

static thread_local std::string g_last_error;

int fail(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}
int cuda_fail(cudaError_t e, const char* what) {
  return fail(IQ_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}
void clear_error() { g_last_error.clear(); }

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

// ------------------------------------------------------------------ rotation

// One thread per 4x4 block.  Normalisation in float32 with explicit IEEE
// operations (sum of squares in index order, correctly rounded sqrt and
// division); block entries L(qL).R(qR) summed in float64 over k = 0..3 in
// order, rounded once to float32; then rounded to bfloat16 for M_b.
struct RotationDraws {
  float v[kHeadDim / 4][2][4];
};

__global__ void rotation_kernel(const __grid_constant__ RotationDraws draws, float* __restrict__ rot,
                                uint16_t* __restrict__ rotb, int nblocks) {
  int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= nblocks) return;
  float q[2][4];
  for (int s = 0; s < 2; ++s) {
    float v[4];
    for (int i = 0; i < 4; ++i) v[i] = draws.v[b][s][i];
    float acc = __fmul_rn(v[0], v[0]);
    for (int i = 1; i < 4; ++i) acc = __fadd_rn(acc, __fmul_rn(v[i], v[i]));
    float nrm = __fsqrt_rn(acc);
    for (int i = 0; i < 4; ++i) q[s][i] = __fdiv_rn(v[i], nrm);
  }
  const double w = q[0][0], x = q[0][1], y = q[0][2], z = q[0][3];
  // left-multiplication matrix of qL (page `_quat_left`)
  const double L[4][4] = {{w, -x, -y, -z}, {x, w, -z, y}, {y, z, w, -x}, {z, -y, x, w}};
  const double rw = q[1][0], rx = q[1][1], ry = q[1][2], rz = q[1][3];
  // page `_quat_right_conj`, entries exactly as printed
  const double R[4][4] = {{rw, rx, ry, rz}, {-rx, rw, rz, -ry}, {-ry, -rz, rw, rx}, {-rz, ry, -rx, rw}};
  for (int i = 0; i < 4; ++i)
    for (int j = 0; j < 4; ++j) {
      double acc = 0.0;
      for (int k = 0; k < 4; ++k) acc = __dadd_rn(acc, __dmul_rn(L[i][k], R[k][j]));
      float f = __double2float_rn(acc);
      rot[b * 16 + i * 4 + j] = f;
      rotb[b * 16 + i * 4 + j] = static_cast<uint16_t>(f32_to_bf16_bits(f));
    }
}

// ------------------------------------------------------------------ append

struct AppendParams {
  const uint16_t* keys;
  const uint16_t* values;
  uint32_t* k_codes;
  uint16_t* k_scales;
  uint16_t* k_biases;
  uint32_t* v_codes;
  uint16_t* v_scales;
  uint16_t* v_biases;
  const uint16_t* rot;
  int batch, heads, n, cap;
  // row r < 2^31 -> (r / n, r % n): r / n = umulhi(r, n_mul) >> n_shift
  uint32_t n_mul;
  int n_shift;
  int lens[IQ_MAX_BATCH];
};

// One warp per token row (sequence b, kv head h, token i): its K and V rows
// are encoded together.  The rows of every (b, h) are laid end to end (the
// input is [B][Hkv][n][256], so flat row r is at r * 256) and a persistent
// grid strides over them (no second wave of blocks for a small append); each
// warp keeps the bf16 K and V of its next IQ_APPEND_DEPTH rows in flight while
// it encodes the current one.  The encoding is bound by instruction issue, so
// occupancy beats depth: one row ahead at three blocks per SM measured best
// (two or four rows ahead at two or one block per SM were slower).
#ifndef IQ_APPEND_MINB
#define IQ_APPEND_MINB 3
#endif
#ifndef IQ_APPEND_DEPTH
#define IQ_APPEND_DEPTH 1
#endif
__global__ void __launch_bounds__(256, IQ_APPEND_MINB) append_kernel(const __grid_constant__ AppendParams p) {
  constexpr int D = IQ_APPEND_DEPTH;
  // Launched as a programmatic dependent of the previous kernel in the
  // stream: wait for it (and its writes) before touching memory.  It never
  // releases its dependents early: an attention launched after it streams
  // cache tiles before its own wait, so it must start after these rows are
  // written.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  // every row index fits in 31 bits (the host refuses caches of 2^31 rows or more)
  const int gwarp = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int nwarps = static_cast<int>((gridDim.x * blockDim.x) >> 5);
  const int total = p.batch * p.heads * p.n;

  float m[2][4][4];
  load_row_rotation(p.rot, lane, m);

  // streamed once: keep the inputs out of L1
  auto load = [&](const uint16_t* base, int r) {
    return __ldcs(reinterpret_cast<const uint4*>(base + static_cast<long long>(r) * kHeadDim + lane * 8));
  };
  uint4 kb[D], vb[D];
#pragma unroll
  for (int d = 0; d < D; ++d) {
    const int r = gwarp + d * nwarps;
    kb[d] = vb[d] = make_uint4(0, 0, 0, 0);
    if (r < total) {
      kb[d] = load(p.keys, r);
      vb[d] = load(p.values, r);
    }
  }
  for (int r0 = gwarp; r0 < total; r0 += D * nwarps) {
#pragma unroll
    for (int d = 0; d < D; ++d) {
      const int r = r0 + d * nwarps;
      if (r >= total) break;
      const uint4 rk = kb[d], rv = vb[d];
      const int nx = r + D * nwarps;
      if (nx < total) {
        kb[d] = load(p.keys, nx);
        vb[d] = load(p.values, nx);
      }
      const uint32_t r32 = static_cast<uint32_t>(r);
      const int bh = static_cast<int>(p.n_mul ? __umulhi(r32, p.n_mul) >> p.n_shift : r32 >> p.n_shift);
      const int i = static_cast<int>(r32 - static_cast<uint32_t>(bh) * static_cast<uint32_t>(p.n));
      const long long dst = static_cast<long long>(bh) * p.cap + p.lens[bh / p.heads] + i;
      encode_row<4>(rk, m, lane, dst, p.k_codes, p.k_scales, p.k_biases);
      encode_row<3>(rv, m, lane, dst, p.v_codes, p.v_scales, p.v_biases);
    }
  }
}

// ------------------------------------------------------------------ gather

struct GatherParams {
  const void* src[6];
  void* dst[6];
  int row_units[6];  // 4-byte units per row of each buffer
  int dst_batch, heads, src_cap, dst_cap;
  int src_of[IQ_MAX_BATCH];
  int len[IQ_MAX_BATCH];
};

// blockIdx.y = dst sequence * heads + head, blockIdx.z = buffer.
__global__ void __launch_bounds__(256) gather_kernel(const __grid_constant__ GatherParams p) {
  const int seq = blockIdx.y / p.heads, h = blockIdx.y % p.heads, buf = blockIdx.z;
  const long long units = static_cast<long long>(p.len[seq]) * p.row_units[buf];
  const uint32_t* s = static_cast<const uint32_t*>(p.src[buf]) +
                      (static_cast<long long>(p.src_of[seq]) * p.heads + h) * p.src_cap * p.row_units[buf];
  uint32_t* d = static_cast<uint32_t*>(p.dst[buf]) +
                (static_cast<long long>(seq) * p.heads + h) * p.dst_cap * p.row_units[buf];
  for (long long u = blockIdx.x * 256LL + threadIdx.x; u < units; u += 256LL * gridDim.x) d[u] = s[u];
}

}  // namespace iq

using namespace iq;

// ------------------------------------------------------------------ C ABI

extern "C" {

const char* iq_status_string(int status) {
  switch (status) {
    case IQ_OK: return "IQ_OK";
    case IQ_ERR_INVALID_ARG: return "IQ_ERR_INVALID_ARG";
    case IQ_ERR_CAPACITY: return "IQ_ERR_CAPACITY";
    case IQ_ERR_WORKSPACE: return "IQ_ERR_WORKSPACE";
    case IQ_ERR_UNSUPPORTED: return "IQ_ERR_UNSUPPORTED";
    case IQ_ERR_CUDA: return "IQ_ERR_CUDA";
    case IQ_ERR_DEVICE: return "IQ_ERR_DEVICE";
    default: return "IQ_ERR_UNKNOWN";
  }
}

const char* iq_last_error(void) { return g_last_error.c_str(); }

int iq_build_rotation(int head_dim, const float* draws_host, float* rot_f32, uint16_t* rot_bf16,
                      iq_stream_t stream) {
  clear_error();
  if (!draws_host || !rot_f32 || !rot_bf16) return fail(IQ_ERR_INVALID_ARG, "null pointer");
  if (head_dim <= 0 || head_dim % 4) return fail(IQ_ERR_INVALID_ARG, "head_dim must be a positive multiple of 4");
  if (head_dim != kHeadDim) return fail(IQ_ERR_UNSUPPORTED, "only head_dim 256 is built");
  const int nb = head_dim / 4;
  // The draws travel as a by-value kernel parameter, so the host buffer may be
  // reused as soon as this call returns.
  RotationDraws d;
  std::memcpy(d.v, draws_host, sizeof(d.v));
  rotation_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(d, rot_f32, rot_bf16, nb);
  IQ_CUDA(cudaGetLastError());
  return IQ_OK;
}

int iq_cache_bytes(int batch, int kv_heads, int head_dim, int group_size, int k_bits, int v_bits,
                   int capacity, int dtype, size_t out_bytes[6]) {
  clear_error();
  if (!out_bytes) return fail(IQ_ERR_INVALID_ARG, "null out_bytes");
  if (batch <= 0 || kv_heads <= 0 || capacity <= 0 || capacity % IQ_STEP)
    return fail(IQ_ERR_INVALID_ARG, "batch, kv_heads > 0 and capacity a positive multiple of 256 required");
  if (dtype != IQ_DTYPE_BF16 && dtype != IQ_DTYPE_F32)
    return fail(IQ_ERR_INVALID_ARG, "dtype must be IQ_DTYPE_BF16 or IQ_DTYPE_F32");
  if (!format_supported(head_dim, group_size, k_bits, v_bits))
    return fail(IQ_ERR_UNSUPPORTED,
                "built formats: head_dim 256, group 32/64/128, k_bits and v_bits 2/3/4/5/6/8");
  if (batch > IQ_MAX_BATCH) return fail(IQ_ERR_UNSUPPORTED, "batch above IQ_MAX_BATCH");
  const size_t rows = static_cast<size_t>(batch) * kv_heads * capacity;
  const size_t ng = head_dim / group_size, esz = dtype == IQ_DTYPE_F32 ? 4 : 2;
  out_bytes[0] = rows * (head_dim * k_bits / 32) * 4;
  out_bytes[1] = out_bytes[2] = rows * ng * esz;
  out_bytes[3] = rows * (head_dim * v_bits / 32) * 4;
  out_bytes[4] = out_bytes[5] = rows * ng * esz;
  return IQ_OK;
}

int iq_cache_check(const iq_cache* c) {
  clear_error();
  if (!c) return fail(IQ_ERR_INVALID_ARG, "null cache");
  size_t bytes[6];
  int st = iq_cache_bytes(c->batch, c->kv_heads, c->head_dim, c->group_size, c->k_bits, c->v_bits,
                          c->capacity, c->dtype, bytes);
  if (st != IQ_OK) return st;
  const void* ptrs[6] = {c->k_codes, c->k_scales, c->k_biases, c->v_codes, c->v_scales, c->v_biases};
  for (int i = 0; i < 6; ++i) {
    if (!ptrs[i]) return fail(IQ_ERR_INVALID_ARG, "null cache buffer");
    if (reinterpret_cast<uintptr_t>(ptrs[i]) % 16) return fail(IQ_ERR_INVALID_ARG, "cache buffer not 16-byte aligned");
  }
  if (!c->lens) return fail(IQ_ERR_INVALID_ARG, "null lens");
  for (int b = 0; b < c->batch; ++b)
    if (c->lens[b] < 0 || c->lens[b] > c->capacity) return fail(IQ_ERR_INVALID_ARG, "lens[b] outside [0, capacity]");
  return IQ_OK;
}

int iq_cache_alloc(iq_cache* c, int batch, int kv_heads, int head_dim, int group_size, int k_bits, int v_bits,
                   int capacity, int dtype, void* const buffers[6], int32_t* lens_host) {
  clear_error();
  if (!c || !buffers || !lens_host) return fail(IQ_ERR_INVALID_ARG, "null cache, buffers or lens");
  iq_cache d;
  d.batch = batch;
  d.kv_heads = kv_heads;
  d.head_dim = head_dim;
  d.group_size = group_size;
  d.k_bits = k_bits;
  d.v_bits = v_bits;
  d.capacity = capacity;
  d.dtype = dtype;
  d.k_codes = static_cast<uint32_t*>(buffers[0]);
  d.k_scales = buffers[1];
  d.k_biases = buffers[2];
  d.v_codes = static_cast<uint32_t*>(buffers[3]);
  d.v_scales = buffers[4];
  d.v_biases = buffers[5];
  d.lens = lens_host;
  if (batch > 0 && batch <= IQ_MAX_BATCH)
    for (int b = 0; b < batch; ++b) lens_host[b] = 0;  // an empty cache (the page's offset 0)
  int st = iq_cache_check(&d);
  if (st != IQ_OK) return st;
  *c = d;
  return IQ_OK;
}

int iq_cache_grow(const iq_cache* src, iq_cache* dst, iq_stream_t stream) {
  clear_error();
  if (!src || !dst) return fail(IQ_ERR_INVALID_ARG, "null cache");
  if (src->batch != dst->batch) return fail(IQ_ERR_INVALID_ARG, "src and dst batch differ");
  if (src->batch <= 0 || src->batch > IQ_MAX_BATCH) return fail(IQ_ERR_INVALID_ARG, "bad batch");
  int32_t ident[IQ_MAX_BATCH];
  for (int b = 0; b < src->batch; ++b) ident[b] = b;
  return iq_cache_gather(src, dst, ident, stream);
}

size_t iq_cache_nbytes(const iq_cache* c) {
  size_t bytes[6];
  if (!c || iq_cache_bytes(c->batch, c->kv_heads, c->head_dim, c->group_size, c->k_bits, c->v_bits,
                           c->capacity, c->dtype, bytes) != IQ_OK)
    return 0;
  size_t t = 0;
  for (int i = 0; i < 6; ++i) t += bytes[i];
  return t;
}

namespace {
// resident 256-thread append blocks per SM (cached per device)
int append_blocks_per_sm() {
  static int cache[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, iq::append_kernel, 256, 0) != cudaSuccess || n <= 0) n = 1;
    cache[dev] = n;
  }
  return cache[dev];
}
}  // namespace

int iq_cache_append(iq_cache* c, const void* keys, const void* values, int n, const void* rot,
                    iq_stream_t stream) {
  int st = iq_cache_check(c);
  if (st != IQ_OK) return st;
  if (n < 0) return fail(IQ_ERR_INVALID_ARG, "negative token count");
  if (n == 0) return IQ_OK;
  if (!keys || !values || !rot) return fail(IQ_ERR_INVALID_ARG, "null keys/values/rotation");
  if (reinterpret_cast<uintptr_t>(keys) % 16 || reinterpret_cast<uintptr_t>(values) % 16 ||
      reinterpret_cast<uintptr_t>(rot) % 16)
    return fail(IQ_ERR_INVALID_ARG, "keys/values/rotation not 16-byte aligned");
  for (int b = 0; b < c->batch; ++b)
    if (static_cast<long long>(c->lens[b]) + n > c->capacity)
      return fail(IQ_ERR_CAPACITY, "append past capacity (grow the cache first)");
  if (static_cast<long long>(c->batch) * c->kv_heads * c->capacity >= (1LL << 31))
    return fail(IQ_ERR_UNSUPPORTED, "cache rows exceed 2^31");
  if (!tuned_format(c)) {
    st = append_any(c, keys, values, n, rot, stream);
    if (st != IQ_OK) return st;
    for (int b = 0; b < c->batch; ++b) c->lens[b] += n;
    return IQ_OK;
  }
  AppendParams p;
  std::memset(&p, 0, sizeof(p));
  p.keys = static_cast<const uint16_t*>(keys);
  p.values = static_cast<const uint16_t*>(values);
  p.k_codes = c->k_codes;
  p.k_scales = static_cast<uint16_t*>(c->k_scales);
  p.k_biases = static_cast<uint16_t*>(c->k_biases);
  p.v_codes = c->v_codes;
  p.v_scales = static_cast<uint16_t*>(c->v_scales);
  p.v_biases = static_cast<uint16_t*>(c->v_biases);
  p.rot = static_cast<const uint16_t*>(rot);
  p.batch = c->batch;
  p.heads = c->kv_heads;
  p.n = n;
  p.cap = c->capacity;
  // division by n for row indices below 2^31: n = 2^s is a shift; otherwise
  // with s = floor(log2 n) and mul = ceil(2^(32+s) / n) < 2^32, umulhi(r, mul)
  // >> s is floor(r / n) exactly (its error is below r / 2^(32+s) < 1 / n)
  {
    int sh = 0;
    while ((2LL << sh) <= n) ++sh;  // floor(log2 n)
    p.n_shift = sh;
    p.n_mul = (n & (n - 1)) == 0 ? 0u
                                 : static_cast<uint32_t>(((static_cast<unsigned long long>(1) << (32 + sh)) + n - 1) /
                                                         static_cast<unsigned long long>(n));
  }
  for (int b = 0; b < c->batch; ++b) p.lens[b] = c->lens[b];
  // a persistent grid: as many 8-warp blocks as fit at once (one row per warp
  // at most), striding over every (sequence, head, token) row
  const long long rows = static_cast<long long>(c->batch) * c->kv_heads * n;
  long long gx = (rows + 7) / 8;
  const long long cap_x = static_cast<long long>(num_sms()) * append_blocks_per_sm();
  if (gx > cap_x) gx = cap_x;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(gx));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  IQ_CUDA(cudaLaunchKernelEx(&cfg, append_kernel, p));
  for (int b = 0; b < c->batch; ++b) c->lens[b] += n;
  return IQ_OK;
}

int iq_cache_trim(iq_cache* c, const int32_t* n_host, int32_t* trimmed_host) {
  clear_error();
  if (!c || !c->lens || !n_host) return fail(IQ_ERR_INVALID_ARG, "null pointer");
  if (c->batch <= 0 || c->batch > IQ_MAX_BATCH) return fail(IQ_ERR_INVALID_ARG, "bad batch");
  for (int b = 0; b < c->batch; ++b)
    if (n_host[b] < 0) return fail(IQ_ERR_INVALID_ARG, "negative trim count");
  for (int b = 0; b < c->batch; ++b) {
    const int32_t t = n_host[b] < c->lens[b] ? n_host[b] : c->lens[b];
    c->lens[b] -= t;
    if (trimmed_host) trimmed_host[b] = t;
  }
  return IQ_OK;
}

int iq_cache_gather(const iq_cache* src, iq_cache* dst, const int32_t* src_of, iq_stream_t stream) {
  int st = iq_cache_check(src);
  if (st != IQ_OK) return st;
  st = iq_cache_check(dst);
  if (st != IQ_OK) return st;
  if (!src_of) return fail(IQ_ERR_INVALID_ARG, "null src_of");
  if (src->kv_heads != dst->kv_heads || src->head_dim != dst->head_dim ||
      src->group_size != dst->group_size || src->k_bits != dst->k_bits || src->v_bits != dst->v_bits ||
      src->dtype != dst->dtype)
    return fail(IQ_ERR_INVALID_ARG, "src and dst shapes or dtypes differ");
  GatherParams p;
  std::memset(&p, 0, sizeof(p));
  int max_len = 0;
  for (int i = 0; i < dst->batch; ++i) {
    if (src_of[i] < 0 || src_of[i] >= src->batch) return fail(IQ_ERR_INVALID_ARG, "src_of index out of range");
    p.src_of[i] = src_of[i];
    p.len[i] = src->lens[src_of[i]];
    if (p.len[i] > dst->capacity) return fail(IQ_ERR_CAPACITY, "dst capacity below a source length");
    if (p.len[i] > max_len) max_len = p.len[i];
  }
  const void* sp[6] = {src->k_codes, src->k_scales, src->k_biases, src->v_codes, src->v_scales, src->v_biases};
  void* dp[6] = {dst->k_codes, dst->k_scales, dst->k_biases, dst->v_codes, dst->v_scales, dst->v_biases};
  // scales (or biases) per row in 4-byte words: two bf16 or one f32 per word
  const int ngw = dst->head_dim / dst->group_size / (dst->dtype == IQ_DTYPE_F32 ? 1 : 2);
  const int units[6] = {dst->head_dim * dst->k_bits / 32, ngw, ngw, dst->head_dim * dst->v_bits / 32, ngw, ngw};
  for (int i = 0; i < 6; ++i) {
    if (sp[i] == dp[i]) return fail(IQ_ERR_INVALID_ARG, "src and dst share a buffer");
    p.src[i] = sp[i];
    p.dst[i] = dp[i];
    p.row_units[i] = units[i];
  }
  p.dst_batch = dst->batch;
  p.heads = dst->kv_heads;
  p.src_cap = src->capacity;
  p.dst_cap = dst->capacity;
  if (max_len > 0) {
    int gx = (max_len * 32 + 255) / 256;
    if (gx > 64) gx = 64;
    dim3 grid(gx, dst->batch * dst->kv_heads, 6);
    gather_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(p);
    IQ_CUDA(cudaGetLastError());
  }
  for (int i = 0; i < dst->batch; ++i) dst->lens[i] = p.len[i];
  return IQ_OK;
}

}  // extern "C"
