// libiqkv: attention of many query rows per kv head (prefill chunks) over the
// packed K4/V3 cache on the 5th-generation tensor cores (tcgen05, accumulators
// in tensor memory).
//
// Method source: page "sparkle mlx_streaming/core/cache/quant_kv.py",
// `asym_quantized_sdpa` (scaled queries, GQA: query head h reads kv head
// h / rep, quantised q.K^T, causal mask at kL - qL + i, softmax, P.V, output in
// rotated value space, undone here by M_b^T) and `rotate_last` (the query
// rotation).  Same arithmetic readings as the split-KV kernels: q'' =
// bf16(bf16(q @ M_b) * scale); keys enter exactly (codes times q'' per 64-dim
// group, then the group's scale and bias in fp32); fp32 softmax; P and the
// dequantised values enter the P.V product as fp16.
//
// One CTA per (sequence, kv head, tile of 128 query rows); its keys stream in
// 64-key tiles.  Warp roles (448 threads):
//  * warps 0-3 and 10-13, two threads per query row (= tensor-memory lane;
//    warp w reaches lanes 32 (w % 4) .. + 31): rotate and store the row's q''
//    (fp16 MMA operand, half of the dims each) and per-group sums; per key tile
//    each reads the four group products S_g of its 32 keys from tensor memory,
//    folds in the key scales and biases and masks; the two agree on the row's
//    reference max (online softmax in log2 units, a lazily moving reference,
//    P <= 2^8) through shared memory, then each writes its half of P (fp16 MMA
//    operand); at the end they add their row sums, normalise, undo the
//    rotation and store half of the output dims each;
//  * warps 4-7: turn each staged tile's 4-bit key codes into bare fp16 fields
//    (a code masked in place is the subnormal c * 2^(L-24), L = 0 or 4: one AND
//    per two codes; the tensor cores take these subnormals exactly, and the
//    query operand is permuted and scaled to match, so every product carries
//    2^-24) and its 3-bit value codes into fp16 values s*c+b, transposed to
//    dims x keys (the P.V MMA operand);
//  * warp 8, one lane: bulk copies of the packed tiles into a two-stage ring;
//  * warp 9, one lane: issues the MMAs: S_g = Q_g . Khat_g^T (M=128 rows,
//    N=64 keys, K=64 dims, one accumulator per group) and O += P . Vhat
//    (M=128, N=256 dims, K=64 keys), each committed to an mbarrier.
// The key operand of tile i+1 is built while the row threads work on tile i
// (it is free once S(i) is done), and S(i+1) is issued as soon as the row
// threads have read S(i), so it runs under their softmax; P.V(i) follows once
// P(i) is written, and the row threads write P(i+1) after P.V(i) is done.  The
// value operand is double-buffered by tile parity: tile i's is built while
// P.V(i-1) runs.
// Fused append (the FUSED instantiation, for iq_cache_append_attend): before
// its pipeline every CTA encodes chunks of the call's new rows (the append's
// row encoder: rotate, group-quantise, pack, store; page "quant_kv.py",
// `update_and_fetch`), taken from a counter in the workspace, and the
// producer streams a sequence's tiles holding new rows only once all of them
// are stored.
// Shared-memory operands use the 128-byte swizzle (K-major, 8-row groups
// 1024 bytes apart).  Tensor memory: S_0..S_3 in columns 0..255, O in
// 256..511.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>

#include "iq_common.cuh"
#include "iq_encode.cuh"

namespace iq {
namespace pre {

constexpr int ROWS = 128;  // query rows per CTA
constexpr int KT = 64;     // keys per tile
constexpr int NSTG = 2;    // staged packed tiles
constexpr float LOG2E = 1.4426950408889634f;
constexpr float NEG = -__builtin_huge_valf();
constexpr float TAU = 8.0f;  // the reference max moves when a score exceeds it by 2^8

// shared memory (from a 1024-byte aligned base)
constexpr int OFF_Q = 0;                       // 4 blocks x [128 rows x 128 B]: q'' fp16
constexpr int OFF_K = OFF_Q + 4 * ROWS * 128;  // 4 blocks x [64 keys x 128 B]: key codes fp16
constexpr int OFF_V = OFF_K + 4 * KT * 128;    // 2 x [256 dims x 128 B]: values fp16, dims x keys (tile parity)
constexpr int OFF_P = OFF_V + 2 * 256 * 128;   // [128 rows x 128 B]: P fp16
constexpr int OFF_STG = OFF_P + ROWS * 128;    // NSTG packed tiles
constexpr int STG_KC = 0, STG_VC = KT * 128, STG_KS = STG_VC + KT * 96, STG_KB = STG_KS + KT * 8,
              STG_VS = STG_KB + KT * 8, STG_VB = STG_VS + KT * 8, STG_BYTES = STG_VB + KT * 8;
constexpr int OFF_SC = OFF_STG + NSTG * STG_BYTES;  // 2 x [64 keys][8] f32: key scales s_0..3, biases b_0..3
constexpr int OFF_XCH = OFF_SC + 2 * KT * 8 * 4;  // row threads' exchange area (1280 floats)
constexpr int XCH_QS = 2 * 2 * ROWS, XCH_L = XCH_QS + 2 * ROWS * 2;
constexpr int OFF_BAR = OFF_XCH + (XCH_L + 2 * ROWS) * 4;
constexpr int SMEM = OFF_BAR + 128 + 1024;  // + alignment slack
static_assert(13 * 8 + 4 <= 128, "the 13 barriers and the tensor-memory slot fit their area");
static_assert(STG_BYTES == 16384 && OFF_STG % 1024 == 0 && OFF_SC % 16 == 0, "layout");
constexpr int THREADS = 448;
constexpr int ENC_CHUNK = 2 * (THREADS / 32);  // new rows per take of the fused append (two per warp)

struct Params {
  const uint32_t* k_codes;
  const uint16_t* k_scales;
  const uint16_t* k_biases;
  const uint32_t* v_codes;
  const uint16_t* v_scales;
  const uint16_t* v_biases;
  const uint16_t* q;
  const uint16_t* rot;
  void* out;
  unsigned* status;
  int out_f32, kv_heads, rep, nq, cap, causal, rtiles;
  float scale;
  int lens[IQ_MAX_BATCH];
};
// The fused launch's parameters: the same fields (same names, so one kernel
// body serves both) plus the fused append's.  The n_new new rows of every
// (sequence, kv head), bf16 [B][Hkv][n_new][256], unrotated, are encoded into
// the cache at rows lens[b] - n_new .. lens[b] - 1 by the grid; flags (zero at
// launch, zero again when the grid ends): [0] chunks taken, [1] CTAs finished,
// then per (sequence, kv head) the count of its new rows stored.  (The field
// order of each struct is the one measured fastest for its kernel.)
struct FusedParams {
  const uint32_t* k_codes;
  const uint16_t* k_scales;
  const uint16_t* k_biases;
  const uint32_t* v_codes;
  const uint16_t* v_scales;
  const uint16_t* v_biases;
  const uint16_t* q;
  const uint16_t* rot;
  void* out;
  unsigned* status;
  const uint16_t* k_new;
  const uint16_t* v_new;
  unsigned* flags;
  int n_new;
  int out_f32, kv_heads, rep, nq, cap, causal, rtiles;
  float scale;
  int lens[IQ_MAX_BATCH];
};

// Bounded wait on an mbarrier phase: gives up after 100 ms (no stage of this
// kernel takes a fraction of that), so a failure ends the kernel quickly with
// a status bit instead of holding the GPU.
__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity) {
  const unsigned long long t0 = now_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity, 2000u)) return true;
    if (now_ns() - t0 > 100000000ull) return false;
  }
}

// Bounded wait for new rows (other CTAs may still be storing them): true once
// their count reaches want, false after 1 s (the encode takes microseconds).
__device__ __forceinline__ bool wait_stored(const unsigned* count, unsigned want) {
  const unsigned long long t0 = now_ns();
  for (;;) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(count) : "memory");
    if (v >= want) return true;
    if (now_ns() - t0 > 1000000000ull) return false;
    __nanosleep(128);
  }
}

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {  // K-major, 128-byte swizzle
  uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1) << 16;                 // leading byte offset (unused with this swizzle)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;         // 8-row groups 1024 B apart
  d |= static_cast<uint64_t>(1) << 46;                 // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                 // 128-byte swizzle
  return d;
}
// f32 accumulate, fp16 A and B, both K-major, N and M
__host__ __device__ constexpr uint32_t idesc(int n, int m) {
  return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}
__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(id), "r"(acc));
}
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void proxy_fence() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}
__device__ __forceinline__ void st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])));
}
__device__ __forceinline__ void ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// byte offset of the 16-byte chunk `c` (0..7) of row `r` inside one 128-byte
// swizzled column block
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// The fused append's encoding, every CTA of the grid taking ENC_CHUNK rows at
// a time (kept out of line: its registers stay out of the pipeline's budget).
__device__ __noinline__ void encode_new_rows(const FusedParams& p, int nbh, uint8_t* smem, int warp, int lane) {
  unsigned* const row_count = p.flags + 2;  // [bh]: new rows stored
  int* slot = reinterpret_cast<int*>(smem + OFF_SC);
  const long long total = static_cast<long long>(nbh) * p.n_new;
  float m[2][4][4];
  load_row_rotation(p.rot, lane, m);
  for (;;) {
    if (threadIdx.x == 0) *slot = static_cast<int>(atomicAdd(p.flags, 1u));
    __syncthreads();
    const long long c0 = static_cast<long long>(*slot) * ENC_CHUNK;
    __syncthreads();  // the slot is read before the next take overwrites it
    if (c0 >= total) break;
    // two rows per warp, both rows' loads issued before either is encoded
    uint4 rk[2], rv[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const long long item = c0 + warp + h * (THREADS / 32);
      if (item < total) {
        const long long src = item * kHeadDim + lane * 8;
        rk[h] = __ldg(reinterpret_cast<const uint4*>(p.k_new + src));
        rv[h] = __ldg(reinterpret_cast<const uint4*>(p.v_new + src));
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const long long item = c0 + warp + h * (THREADS / 32);
      if (item >= total) break;
      const int ebh = static_cast<int>(item / p.n_new), j = static_cast<int>(item % p.n_new);
      const long long dst = static_cast<long long>(ebh) * p.cap + p.lens[ebh / p.kv_heads] - p.n_new + j;
      encode_row<4>(rk[h], m, lane, dst, const_cast<uint32_t*>(p.k_codes), const_cast<uint16_t*>(p.k_scales),
                    const_cast<uint16_t*>(p.k_biases));
      encode_row<3>(rv[h], m, lane, dst, const_cast<uint32_t*>(p.v_codes), const_cast<uint16_t*>(p.v_scales),
                    const_cast<uint16_t*>(p.v_biases));
      asm volatile("fence.proxy.async.global;" ::: "memory");  // the stores before other CTAs' bulk copies
      __syncwarp();
      if (lane == 0) {
        __threadfence();
        atomicAdd(row_count + ebh, 1u);
      }
    }
  }
}

// FUSED: the grid also encodes the call's new rows (the fused append); a
// separate instantiation, so attention-only launches carry none of its code.
template <bool FUSED, typename P>
__global__ void __launch_bounds__(THREADS, 1) prefill_kernel(const __grid_constant__ P p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + OFF_BAR);  // [NSTG]
  uint64_t* empty = full + NSTG;                                  // [NSTG]
  uint64_t* k_ready = empty + NSTG;                               // key operand (and key scales) of tile i written
  // [2]: value operand of tile i written, on v_ready[i & 1] (phase i / 2).  One
  // barrier would not do: the builders may finish V(i+1) while the MMA lane
  // still waits for P(i), and a parity wait cannot tell phase i from phase i+2
  uint64_t* v_ready = k_ready + 1;
  uint64_t* s_ready = v_ready + 2;                                // S_g of tile i in tensor memory
  uint64_t* p_ready = s_ready + 1;                                // P of tile i written (and O rescaled)
  uint64_t* o_ready = p_ready + 1;  // [2]: P.V of tile i done, on o_ready[i & 1] (phase i / 2)
  uint64_t* s_free = o_ready + 2;                                 // S of tile i read (S(i+1) may be issued)
  uint64_t* row_bar = s_free + 1;                                 // barrier of the 8 row warps (bounded)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(row_bar + 1);
  float* sc = reinterpret_cast<float*>(smem + OFF_SC);
  const uint32_t sbase = smem_u32(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // longest first: causal row tiles late in the chunk see the most keys, and
  // CTAs are dispatched in block order
  const int nbh = gridDim.x / p.rtiles;
  const int z = p.rtiles - 1 - static_cast<int>(blockIdx.x) / nbh, bh = static_cast<int>(blockIdx.x) % nbh;
  const int b = bh / p.kv_heads, h = bh % p.kv_heads;
  const int T = p.lens[b];
  const int rows = p.rep * p.nq;
  const int r_last = min(z * ROWS + ROWS - 1, rows - 1);
  const int kmax = p.causal ? T - p.nq + r_last / p.rep + 1 : T;  // keys some row of the tile sees
  const int ntiles = (kmax + KT - 1) / KT;
  const long long row0 = static_cast<long long>(bh) * p.cap;

  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ---- fused append.  The new rows (B x Hkv x n_new of them, in (sequence,
  // kv head, row) order) are encoded in chunks of ENC_CHUNK rows that every CTA
  // takes from one counter (flags[0]) until none is left, a warp per row; each
  // stored row adds one to its (sequence, kv head)'s count (release).  A CTA's
  // producer, at its first tile holding new rows, waits for the count to reach
  // n_new only once every chunk has been taken, so the rows it waits for are
  // owed only by CTAs already encoding (which wait for nothing), never by a CTA
  // that has not started: the grid needs no co-residency.  The last CTA to
  // finish returns the counters to zero (flags[1] counts finished CTAs).
  if constexpr (FUSED) encode_new_rows(p, nbh, smem, warp, lane);
  if (threadIdx.x == 0) {
    for (int s = 0; s < NSTG; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 4);
    }
    mbar_init(k_ready, 4);
    mbar_init(&v_ready[0], 4);
    mbar_init(&v_ready[1], 4);
    mbar_init(s_ready, 1);
    mbar_init(p_ready, 8);
    mbar_init(&o_ready[0], 1);
    mbar_init(&o_ready[1], 1);
    mbar_init(s_free, 8);
    mbar_init(row_bar, 8);
    mbar_fence_init();
  }
  if (warp == 9) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)), "r"(512));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_before();
  __syncthreads();
  tc_after();
  const uint32_t tmem = *tslot;

  if (warp == 8) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int issued = 0;
      int i_new = -1;  // the first tile holding new rows
      if constexpr (FUSED) i_new = (T - p.n_new) / KT;
      for (int i = 0; i < ntiles; ++i, ++issued) {
        const int st = i % NSTG;
        if (i >= NSTG && !wait_phase(&empty[st], static_cast<uint32_t>(i / NSTG - 1) & 1)) {
          atomicOr(p.status, 1u | 0x100u);
          break;
        }
        if constexpr (FUSED) {
          if (i == i_new) {  // the first tile with new rows: wait until all are stored
            if (!wait_stored(p.flags + 2 + bh, static_cast<unsigned>(p.n_new))) {
              atomicOr(p.status, 1u | 0x20000u);
              break;
            }
            asm volatile("fence.proxy.async.global;" ::: "memory");
          }
        }
        uint8_t* g = smem + OFF_STG + st * STG_BYTES;
        const long long r = row0 + static_cast<long long>(i) * KT;
        mbar_arrive_expect_tx(&full[st], STG_BYTES);
        bulk_g2s(g + STG_KC, p.k_codes + r * kKWords, KT * 128, &full[st], pol);
        bulk_g2s(g + STG_VC, p.v_codes + r * kVWords, KT * 96, &full[st], pol);
        bulk_g2s(g + STG_KS, p.k_scales + r * kGroups, KT * 8, &full[st], pol);
        bulk_g2s(g + STG_KB, p.k_biases + r * kGroups, KT * 8, &full[st], pol);
        bulk_g2s(g + STG_VS, p.v_scales + r * kGroups, KT * 8, &full[st], pol);
        bulk_g2s(g + STG_VB, p.v_biases + r * kGroups, KT * 8, &full[st], pol);
      }
      for (int s = 0; s < NSTG && s < issued; ++s) {  // no copy left in flight
        const int last = s + NSTG * ((issued - 1 - s) / NSTG);
        wait_phase(&full[s], static_cast<uint32_t>(last / NSTG) & 1);
      }
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------------- MMA issuer
    // S(i+1) goes in as soon as the row threads have read S(i) (its keys are
    // built while they work on tile i), so it runs under their softmax; P.V(i)
    // follows once P(i) is written
    named_bar(1, 2 * 128 + 32);  // q'' written by the row threads
    if (lane == 0) {
      tc_after();
      auto issue_s = [&](int i) {
        tc_after();
#pragma unroll
        for (int g = 0; g < 4; ++g)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma(tmem + 64 * g, sdesc(sbase + OFF_Q + g * ROWS * 128 + 32 * ks),
                sdesc(sbase + OFF_K + g * KT * 128 + 32 * ks), idesc(KT, ROWS), ks > 0 ? 1u : 0u);
        commit(s_ready);
      };
      int done = 0;
      bool ok = ntiles > 0 && wait_phase(k_ready, 0u);
      if (ntiles > 0 && !ok) atomicOr(p.status, 2u | 0x200u);
      if (ok) issue_s(0);
      for (int i = 0; ok && i < ntiles; ++i) {
        if (i + 1 < ntiles) {
          if (!wait_phase(s_free, static_cast<uint32_t>(i) & 1) ||
              !wait_phase(k_ready, static_cast<uint32_t>(i + 1) & 1)) {
            atomicOr(p.status, 2u | 0x200u);
            break;
          }
          issue_s(i + 1);
        }
        if (!wait_phase(p_ready, static_cast<uint32_t>(i) & 1) ||
            !wait_phase(&v_ready[i & 1], static_cast<uint32_t>(i >> 1) & 1)) {
          atomicOr(p.status, 2u | 0x400u);
          break;
        }
        tc_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma(tmem + 256, sdesc(sbase + OFF_P + 32 * ks), sdesc(sbase + OFF_V + (i & 1) * 32768 + 32 * ks), idesc(256, ROWS),
              (i > 0 || ks > 0) ? 1u : 0u);
        commit(&o_ready[i & 1]);
        done = i + 1;
      }
      if (done > 0) wait_phase(&o_ready[(done - 1) & 1], static_cast<uint32_t>((done - 1) >> 1) & 1);  // nothing left in flight
    }
  } else if (warp >= 4 && warp < 8) {
    // ---------------------------------------------------------------- operand builders
    const int dt = threadIdx.x - 128;  // 0..127
    for (int i = 0; i < ntiles; ++i) {
      const int st = i % NSTG;
      bool ok = wait_phase(&full[st], static_cast<uint32_t>(i / NSTG) & 1);
      if (!ok) atomicOr(p.status, 0x800u);
      if (ok && i > 0) {  // the key operand is free once S(i-1) is done
        ok = wait_phase(s_ready, static_cast<uint32_t>(i - 1) & 1);
        if (!ok) atomicOr(p.status, 0x1000u);
      }
      if (!ok) {
        atomicOr(p.status, 1u);
        break;
      }
      float* sci = sc + (i & 1) * KT * 8;  // read by the row threads of tile i (tile i-2 was done before S(i-1))
      const uint8_t* g = smem + OFF_STG + st * STG_BYTES;
      // key codes -> bare fp16 fields: item (key t, 8-dim chunk c), the chunk is
      // word c of the row (dims 8c+k at bits 4k); a code masked in place is the
      // fp16 subnormal c * 2^(L-24) (L = 0 or 4), so the chunk holds dims
      // (0, 4, 1, 5, 2, 6, 3, 7) with L = (0, 0, 4, 4, 0, 0, 4, 4), and the
      // query operand is laid out and scaled to match (every product carries 2^-24)
      for (int it = dt; it < KT * 32; it += 128) {
        const int t = it >> 5, c = it & 31;
        const uint32_t w = reinterpret_cast<const uint32_t*>(g + STG_KC)[t * 32 + c];
        const uint32_t w8 = w >> 8;
        *reinterpret_cast<uint4*>(smem + OFF_K + (c >> 3) * KT * 128 + swz(t, c & 7)) =
            make_uint4(w & 0x000F000Fu, w & 0x00F000F0u, w8 & 0x000F000Fu, w8 & 0x00F000F0u);
      }
      // the key scales and biases of the tile, for the row threads
      for (int it = dt; it < KT * 4; it += 128) {
        const int t = it >> 2, gi = it & 3;
        sci[t * 8 + gi] = bf16_to_f32(reinterpret_cast<const uint16_t*>(g + STG_KS)[t * 4 + gi]);
        sci[t * 8 + 4 + gi] = bf16_to_f32(reinterpret_cast<const uint16_t*>(g + STG_KB)[t * 4 + gi]);
      }
      proxy_fence();  // generic-proxy stores before the tensor cores read them
      __syncwarp();
      if (lane == 0) mbar_arrive(k_ready);
      // this tile's value buffer was last read by P.V(i-2) (its own completion
      // barrier, so a phase two tiles back is never confused with the latest)
      if (i > 1 && !wait_phase(&o_ready[i & 1], static_cast<uint32_t>((i - 2) >> 1) & 1)) {
        atomicOr(p.status, 1u | 0x1000u);
        break;
      }
      // values -> fp16 s*c+b, transposed: item (8-dim block db, 8-key block tb);
      // lane db of operand warp w takes key blocks (db + w) % 8 and (db + w + 4) % 8,
      // so a warp's lanes read different key rows (192 words apart: the same bank
      // offset, different words) and store into distinct swizzled chunks
      for (int half = 0; half < 2; ++half) {
        const int db = lane, tb = (lane + (warp - 4) + 4 * half) & 7;
        const int gi = db >> 3;  // 64-dim group
        const int w0 = (3 * db) >> 2, sh = (24 * db) & 31;
        float v[8][8];  // [key][dim]
        float vmax = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int t = 8 * tb + k;
          const uint32_t* row = reinterpret_cast<const uint32_t*>(g + STG_VC) + t * 24;
          const uint32_t f = __funnelshift_r(row[w0], row[w0 + 1 < 24 ? w0 + 1 : w0], sh);
          const uint16_t* vs = reinterpret_cast<const uint16_t*>(g + STG_VS) + t * 4;
          const uint16_t* vb = reinterpret_cast<const uint16_t*>(g + STG_VB) + t * 4;
          const float s = bf16_to_f32(vs[gi]), bb = bf16_to_f32(vb[gi]);
          const bool stale = i * KT + t >= T;  // rows past the length may hold anything: P is 0 there, and 0 * NaN is not
          // the group's values lie between b and b + 7 s (codes 0 .. 7)
          if (!stale) vmax = fmaxf(vmax, fmaxf(fabsf(bb), fabsf(fmaf(s, 7.0f, bb))));
#pragma unroll
          for (int e = 0; e < 8; ++e)
            v[k][e] = stale ? 0.f : fmaf(s, __uint_as_float(0x4B000000u | ((f >> (3 * e)) & 7u)) - 8388608.0f, bb);
        }
        // dequantised values enter the P.V product as fp16: a value at or above
        // 2^15 in magnitude (a value group spanning more than about 3e4) is
        // outside what this kernel serves and is reported (status bit 16)
        if (!(vmax < 32768.f)) atomicOr(p.status, 16u);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int d = 8 * db + e;
          *reinterpret_cast<uint4*>(smem + OFF_V + (i & 1) * 32768 + swz(d, tb)) =
              make_uint4(pack_h2(v[0][e], v[1][e]), pack_h2(v[2][e], v[3][e]), pack_h2(v[4][e], v[5][e]),
                         pack_h2(v[6][e], v[7][e]));
        }
      }
      proxy_fence();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&v_ready[i & 1]);
        mbar_arrive(&empty[st]);
      }
    }
  } else {
    // ---------------------------------------------------------------- row threads
    // Two threads per query row (= tensor-memory lane): warps 0-3 take keys
    // 0..31 of every tile and output dims 0..127, warps 10-13 keys 32..63 and
    // dims 128..255 (a warp reaches the lanes 32 * (warp % 4) ..  + 31).  The
    // two threads of a row agree on its reference max each tile through
    // shared memory and a bounded barrier of the 8 row warps.
    const int hf = warp >= 10 ? 1 : 0;
    const int r = 32 * (warp & 3) + lane;  // row in the tile = tensor-memory lane
    const int R = z * ROWS + r;
    const bool live = R < rows;
    const int qi = live ? R / p.rep : 0, hr = live ? R % p.rep : 0;
    const int qpos = live ? (p.causal ? T - p.nq + qi : T - 1) : -1;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    float* xch = reinterpret_cast<float*>(smem + OFF_XCH);  // [2 parities][2 halves][128 rows]
    uint32_t gph = 0;  // completed phases of row_sync
    auto row_sync = [&]() -> bool {  // every row thread's shared-memory writes before the reads after it
      __syncwarp();
      if (lane == 0) mbar_arrive(row_bar);
      const bool ok = __all_sync(0xffffffffu, wait_phase(row_bar, gph & 1));
      ++gph;
      return ok;
    };
    // q'' = bf16(bf16(q @ M_b) * scale), entering the MMA as the fp16 q_s =
    // q'' * 2^-e, and its per-group sums.  The rotation keeps every |q''|
    // below 2.03 * max|q| * |scale| (a row of M_b has an L1 norm of at most
    // 2, plus bf16 rounding), so with max|q| * |scale| in [2^E0, 2^(E0+1))
    // e = E0 - 12 puts |q_s| below 2^15 (fp16) and its largest entry above 2^8.
    // Each thread of the row takes half of its dims (8-dim chunks 16 hf .. 16 hf + 15).
    float qs[4] = {0.f, 0.f, 0.f, 0.f};
    float kmul = LOG2E;  // raw score -> log2 units: log2(e) * 2^e
    bool ok = true;
    {
      const uint16_t* qrow =
          p.q + ((static_cast<long long>(b) * p.kv_heads * p.rep + h * p.rep + hr) * p.nq + qi) * kHeadDim;
      uint32_t amax = 0;  // largest |q| as bf16 bits (monotonic in the magnitude)
      if (live)
        for (int c = 16 * hf; c < 16 * hf + 16; ++c) {
          const uint4 raw = __ldg(reinterpret_cast<const uint4*>(qrow + 8 * c));
          const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) amax = max(amax, max(rw[j] & 0x7FFFu, (rw[j] >> 16) & 0x7FFFu));
        }
      xch[XCH_L + hf * ROWS + r] = __uint_as_float(amax);
      ok = row_sync();
      amax = max(amax, __float_as_uint(xch[XCH_L + (1 - hf) * ROWS + r]));
      const float m = bf16_to_f32(amax) * fabsf(p.scale);
      int e = 0;
      if (m > 0.f) e = min(max(static_cast<int>((__float_as_uint(m) >> 23) & 0xFF) - 127 - 12, -100), 100);
      const float down = __int_as_float((127 - e) << 23);
      // the scores accumulate in units of 2^-24 (key fields), so the multiplier
      // carries 2^24 and the bias sums below 2^-24
      kmul = LOG2E * __int_as_float((127 + e + 24) << 23);
      float qh[2] = {0.f, 0.f};  // sums of this thread's two groups
      for (int c = 16 * hf; c < 16 * hf + 16; ++c) {  // 8-dim chunk c: rotation blocks 2c, 2c+1
        uint4 raw = make_uint4(0, 0, 0, 0);
        if (live) raw = __ldg(reinterpret_cast<const uint4*>(qrow + 8 * c));
        const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
        float yy[8];  // q_s of the chunk's 8 dims
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          float x[4], y[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t w = rw[(4 * blk + e) >> 1];
            x[e] = bf16_to_f32(((4 * blk + e) & 1) ? (w >> 16) : (w & 0xFFFFu));
          }
          const uint16_t* mb = p.rot + (2 * c + blk) * 16;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float a = __fmul_rn(x[0], bf16_to_f32(__ldg(mb + j)));
#pragma unroll
            for (int k = 1; k < 4; ++k) a = __fadd_rn(a, __fmul_rn(x[k], bf16_to_f32(__ldg(mb + 4 * k + j))));
            y[j] = __fmul_rn(round_bf16(__fmul_rn(round_bf16(a), p.scale)), down);  // exact: a power of two
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) yy[4 * blk + j] = y[j];
        }
        // the key chunk's layout: dims (0, 4, 1, 5, 2, 6, 3, 7), the odd pairs
        // scaled by 2^-4 (their key fields sit 4 bits higher)
        const uint32_t h0 = pack_h2(yy[0], yy[4]), h1 = pack_h2(yy[1] * 0.0625f, yy[5] * 0.0625f);
        const uint32_t h2 = pack_h2(yy[2], yy[6]), h3 = pack_h2(yy[3] * 0.0625f, yy[7] * 0.0625f);
        // the sums use the fp16 values the MMA multiplies, in the query's own scale
        const __half2 a0 = *reinterpret_cast<const __half2*>(&h0), a1 = *reinterpret_cast<const __half2*>(&h1);
        const __half2 a2 = *reinterpret_cast<const __half2*>(&h2), a3 = *reinterpret_cast<const __half2*>(&h3);
        qh[(c >> 3) & 1] += __low2float(a0) + __high2float(a0) + 16.0f * (__low2float(a1) + __high2float(a1)) +
                            __low2float(a2) + __high2float(a2) + 16.0f * (__low2float(a3) + __high2float(a3));
        *reinterpret_cast<uint4*>(smem + OFF_Q + (c >> 3) * ROWS * 128 + swz(r, c & 7)) = make_uint4(h0, h1, h2, h3);
      }
      // exchange the group sums: this thread holds groups 2 hf, 2 hf + 1
      xch[XCH_QS + hf * ROWS * 2 + 2 * r] = qh[0];
      xch[XCH_QS + hf * ROWS * 2 + 2 * r + 1] = qh[1];
      ok = row_sync() && ok;
      qs[2 * hf] = qh[0] * 0x1p-24f;
      qs[2 * hf + 1] = qh[1] * 0x1p-24f;
      qs[2 - 2 * hf] = xch[XCH_QS + (1 - hf) * ROWS * 2 + 2 * r] * 0x1p-24f;
      qs[3 - 2 * hf] = xch[XCH_QS + (1 - hf) * ROWS * 2 + 2 * r + 1] * 0x1p-24f;
    }
    proxy_fence();
    named_bar(1, 2 * 128 + 32);  // (arrive side for the MMA warp)

    float mref = NEG, lsum = 0.f;
    for (int i = 0; i < ntiles && ok; ++i) {
      // tensor-memory loads and stores are warp-collective: every decision that
      // guards them is made the same for the whole warp
      if (!__all_sync(0xffffffffu, wait_phase(s_ready, static_cast<uint32_t>(i) & 1))) {
        atomicOr(p.status, 2u | 0x2000u);
        ok = false;
        break;
      }
      tc_after();
      const float* sci = sc + (i & 1) * KT * 8;
      float x[32];  // scores of this thread's 32 keys, log2 units
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c16 = 2 * hf + cc;  // 16-key chunk of the tile
        float s0[16], s1[16], s2[16], s3[16];
        ld16(lane_addr + 0 * 64 + 16 * c16, s0);
        ld16(lane_addr + 1 * 64 + 16 * c16, s1);
        ld16(lane_addr + 2 * 64 + 16 * c16, s2);
        ld16(lane_addr + 3 * 64 + 16 * c16, s3);
        ld_wait();
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int tl = 16 * c16 + k, t = i * KT + tl;
          const float4 ks = *reinterpret_cast<const float4*>(sci + tl * 8);
          const float4 kb = *reinterpret_cast<const float4*>(sci + tl * 8 + 4);
          float sv = ks.x * s0[k];
          sv = fmaf(ks.y, s1[k], sv);
          sv = fmaf(ks.z, s2[k], sv);
          sv = fmaf(ks.w, s3[k], sv);
          sv = fmaf(kb.x, qs[0], sv);
          sv = fmaf(kb.y, qs[1], sv);
          sv = fmaf(kb.z, qs[2], sv);
          sv = fmaf(kb.w, qs[3], sv);
          x[16 * cc + k] = t <= qpos ? sv * kmul : NEG;
        }
      }
      // S(i) is read: S(i+1) may overwrite it
      tc_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);
      float mx = NEG;
#pragma unroll
      for (int k = 0; k < 32; ++k) mx = fmaxf(mx, x[k]);
      xch[(i & 1) * 2 * ROWS + hf * ROWS + r] = mx;
      if (!row_sync()) {
        atomicOr(p.status, 2u | 0x10000u);
        ok = false;
        break;
      }
      mx = fmaxf(mx, xch[(i & 1) * 2 * ROWS + (1 - hf) * ROWS + r]);  // the row's max over the tile
      const bool move = mx != NEG && (mref == NEG || mx > mref + TAU);
      bool o_done = i == 0;  // O(i-1) complete (P and O may be touched)
      if (__any_sync(0xffffffffu, move)) {  // the same for the row's other warp: the rows are the same
        const float mnew = move ? (mref == NEG ? mx : fmaxf(mref, mx)) : mref;
        const float alpha = !move ? 1.f : mref == NEG ? 0.f : ex2_approx(mref - mnew);
        if (i > 0) {  // O holds earlier tiles' sums: rescale this thread's half of its columns
          if (!__all_sync(0xffffffffu, wait_phase(&o_ready[(i - 1) & 1], static_cast<uint32_t>((i - 1) >> 1) & 1))) {
            atomicOr(p.status, 2u | 0x4000u);
            ok = false;
            break;
          }
          o_done = true;
          tc_after();
#pragma unroll 1
          for (int c = 128 * hf; c < 128 * hf + 128; c += 16) {
            float o[16];
            ld16(lane_addr + 256 + c, o);
            ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) o[j] *= alpha;
            st16(lane_addr + 256 + c, o);
          }
          st_wait();
        }
        lsum *= alpha;
        mref = mnew;
      }
      // P = 2^(x - mref) (fp16) into this thread's half of the row, once P.V(i-1) is done with P
#pragma unroll
      for (int k = 0; k < 32; ++k) x[k] = mref == NEG ? 0.f : ex2_approx(x[k] - mref);
      if (!o_done && !__all_sync(0xffffffffu, wait_phase(&o_ready[(i - 1) & 1], static_cast<uint32_t>((i - 1) >> 1) & 1))) {
        atomicOr(p.status, 2u | 0x4000u);
        ok = false;
        break;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t hv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float a = x[8 * c + 2 * j], bq = x[8 * c + 2 * j + 1];
          lsum += a + bq;
          hv[j] = pack_h2(a, bq);
        }
        *reinterpret_cast<uint4*>(smem + OFF_P + swz(r, 4 * hf + c)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
      }
      proxy_fence();
      tc_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_ready);
    }
    // ---- output: O / l (the row's two partial sums), undo the rotation, store this thread's half
    bool fin = ok && ntiles > 0;
    if (fin) {
      xch[XCH_L + hf * ROWS + r] = lsum;
      fin = row_sync();
    }
    if (fin) lsum += xch[XCH_L + (1 - hf) * ROWS + r];
    if (fin && __all_sync(0xffffffffu, wait_phase(&o_ready[(ntiles - 1) & 1], static_cast<uint32_t>((ntiles - 1) >> 1) & 1))) {
      tc_after();
      const float inv = 1.f / lsum;
      if (live && hf == 0 && !(lsum > 0.f)) atomicOr(p.status, 4u);
      const long long orow = (static_cast<long long>(b) * p.kv_heads * p.rep + h * p.rep + hr) * p.nq + qi;
#pragma unroll 1
      for (int c = 128 * hf; c < 128 * hf + 128; c += 16) {
        float o[16];
        ld16(lane_addr + 256 + c, o);
        ld_wait();
        if (!live) continue;
        float y[16];
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
          const uint16_t* mb = p.rot + ((c >> 2) + blk) * 16;
#pragma unroll
          for (int ii = 0; ii < 4; ++ii) {
            float acc = 0.f;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) acc = fmaf(o[4 * blk + jj] * inv, bf16_to_f32(__ldg(mb + 4 * ii + jj)), acc);
            y[4 * blk + ii] = acc;
          }
        }
        if (p.out_f32) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow * kHeadDim + c);
#pragma unroll
          for (int j = 0; j < 4; ++j) dst[j] = make_float4(y[4 * j], y[4 * j + 1], y[4 * j + 2], y[4 * j + 3]);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + orow * kHeadDim + c);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            uint4 w;
            w.x = f32_to_bf16_bits(y[8 * j]) | (f32_to_bf16_bits(y[8 * j + 1]) << 16);
            w.y = f32_to_bf16_bits(y[8 * j + 2]) | (f32_to_bf16_bits(y[8 * j + 3]) << 16);
            w.z = f32_to_bf16_bits(y[8 * j + 4]) | (f32_to_bf16_bits(y[8 * j + 5]) << 16);
            w.w = f32_to_bf16_bits(y[8 * j + 6]) | (f32_to_bf16_bits(y[8 * j + 7]) << 16);
            dst[j] = w;
          }
        }
      }
    } else if (live && hf == 0) {
      atomicOr(p.status, 2u | 0x8000u);
    }
  }
  tc_before();
  __syncthreads();
  if (warp == 9) {
    tc_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
  }
  if constexpr (FUSED) {  // the grid's last CTA (every take and wait is over) zeroes the fused append's counters
    int* last = reinterpret_cast<int*>(smem + OFF_SC);
    if (threadIdx.x == 0) {
      __threadfence();
      *last = atomicAdd(p.flags + 1, 1u) == gridDim.x - 1u;
    }
    __syncthreads();
    if (*last) {
      __threadfence();
      for (int i = threadIdx.x; i < 2 + nbh; i += THREADS) p.flags[i] = 0u;
    }
  }
}

}  // namespace pre

// Rows per kv head from which attention takes the tensor-memory kernel.
#ifndef IQ_PREFILL_MIN_ROWS
#define IQ_PREFILL_MIN_ROWS 128
#endif

bool prefill_shape(const iq_cache* c, int q_heads, int n_queries, int mask_kind) {
  return tuned_format(c) && mask_kind <= 1 && (q_heads / c->kv_heads) * n_queries >= IQ_PREFILL_MIN_ROWS;
}

long long prefill_fuse_flags(const iq_cache* c, int n_new) {
  return n_new > 0 ? 2 + static_cast<long long>(c->batch) * c->kv_heads : 0;
}

int prefill_attend(const iq_cache* c, const uint16_t* q, int q_heads, int n_queries, float scale, int causal,
                   const uint16_t* rot, void* out, int out_f32, unsigned* status, iq_stream_t stream,
                   const uint16_t* k_new, const uint16_t* v_new, int n_new, unsigned* flags) {
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    IQ_CUDA(cudaFuncSetAttribute(pre::prefill_kernel<false, pre::Params>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 pre::SMEM));
    IQ_CUDA(cudaFuncSetAttribute(pre::prefill_kernel<true, pre::FusedParams>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, pre::SMEM));
    attr_set[dev] = true;
  }
  if (n_new > 0 && (!flags || !k_new || !v_new)) return fail(IQ_ERR_INVALID_ARG, "fused prefill append arguments");
  auto fill = [&](auto& p) {
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
    p.status = status;
    p.out_f32 = out_f32 ? 1 : 0;
    p.kv_heads = c->kv_heads;
    p.rep = q_heads / c->kv_heads;
    p.nq = n_queries;
    p.cap = c->capacity;
    p.causal = causal;
    p.rtiles = (p.rep * n_queries + pre::ROWS - 1) / pre::ROWS;
    p.scale = scale;
    for (int b = 0; b < c->batch; ++b) p.lens[b] = c->lens[b];
  };
  const int rtiles = ((q_heads / c->kv_heads) * n_queries + pre::ROWS - 1) / pre::ROWS;
  const long long grid = static_cast<long long>(c->batch) * c->kv_heads * rtiles;
  if (grid > 0x7FFFFFFFLL) return fail(IQ_ERR_UNSUPPORTED, "too many query tiles");
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(pre::THREADS);
  cfg.dynamicSmemBytes = pre::SMEM;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (n_new > 0) {
    // (the fused append's counters share the workspace's unit counters, zero
    // at every call's start; the grid leaves them zero)
    pre::FusedParams f;
    fill(f);
    f.k_new = k_new;
    f.v_new = v_new;
    f.n_new = n_new;
    f.flags = flags;
    IQ_CUDA(cudaLaunchKernelEx(&cfg, pre::prefill_kernel<true, pre::FusedParams>, f));
  } else {
    pre::Params p;
    fill(p);
    IQ_CUDA(cudaLaunchKernelEx(&cfg, pre::prefill_kernel<false, pre::Params>, p));
  }
  return IQ_OK;
}

}  // namespace iq
