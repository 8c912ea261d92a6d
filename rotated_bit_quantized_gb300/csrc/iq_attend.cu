// libiqkv: GQA attention over the packed K4/V3 cache (persistent split-KV
// kernel with the inverse rotation fused in, and the split combine kernel).
//
// Method source: page "sparkle mlx_streaming/core/cache/quant_kv.py",
// `asym_quantized_sdpa` (scale the queries, GQA reshape so query head h reads
// kv head h / rep, quantised q.K^T, causal mask at query position
// kL - qL + i, softmax, P.V over the quantised values) and the module note
// that the output is still in rotated value space, so the caller undoes the
// rotation; `rotate_last` gives the query rotation.
//
// Work decomposition.  A "unit" is (sequence, kv head, tile of 8*NT query
// rows); its keys form a run of TILE-token tiles.  All units' tiles are laid
// end to end and split over a persistent grid (at most one CTA per resident
// slot); the host gives each CTA an explicit tile range, balanced so that a CTA
// crossing unit starts streams fewer tiles.  A CTA whose range holds a whole
// unit finishes it (normalise, inverse rotation, store); a unit shared by
// several CTAs gets an un-normalised partial (O, running max in log2 units,
// running sum) from each, merged afterwards by combine_kernel, a programmatic
// dependent launch.
//
// Inside a CTA:
//  * a producer warp streams the tiles (packed K codes by a 2-D tensor copy with
//    128-byte swizzle; packed V codes and the four scale/bias rows by 1-D bulk
//    copies) into a multi-stage shared-memory ring guarded by mbarriers, running
//    ahead across unit boundaries; its warpgroup hands most of its registers
//    to the consumer warps;
//  * consumer warps run m16n8k16 tensor-core MMAs on codes that enter as bare
//    bit fields: a code masked in place inside a 16-bit half, with every other
//    bit zero, is the fp16 subnormal c * 2^(L - 24) (L its bit position, at
//    most 10 - width), so one AND per register turns packed codes into exact
//    MMA operands and the power of two is undone once per unit.  Scores:
//    S_G = K_codes . q_s per 64-dim group (q_s = q'' times a per-row power of
//    two that keeps it inside fp16), folded with the group scale on CUDA cores,
//    plus the per-token bias sum_G b_G sum(q_G) from one bf16 MMA over the raw
//    bias words; online softmax in fp32 with a lazily moving reference max;
//    O^T += V_codes^T . (P * s_v) with P transposed in registers by movmatrix;
//    the value bias term sum_t p_t b_t on CUDA cores, the codes centred on
//    3.5 by one more MMA over an all-ones operand.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <type_traits>
#include <unordered_map>
#include <vector>

#include "iq_common.cuh"
#include "iq_encode.cuh"

namespace iq {
namespace attn {

// Shared-memory stage of TILE tokens: the four scale/bias rows, packed K
// codes (128-byte swizzled, 1024-byte aligned) and packed V codes, 256 bytes
// per token with no padding.  The value-field window reads at most 4 bytes
// past a stage's V rows, which land in the next stage or in the area that
// follows the ring.
template <int TILE_>
struct Tiling {
  static constexpr int TILE = TILE_;               // tokens per pipeline stage
  static constexpr int SUBS = TILE / 16;           // 16-token sub-tiles per stage
  static constexpr int K_BYTES = TILE * 128;       // TILE rows x 128 B, 128-byte swizzle
  static constexpr int V_BYTES = TILE * 96;        // TILE rows x 96 B
  static constexpr int SB_BYTES = TILE * 8;        // TILE rows x 4 bf16
  static constexpr int OFF_KS = 0;
  static constexpr int OFF_KB = OFF_KS + SB_BYTES;
  static constexpr int OFF_VS = OFF_KB + SB_BYTES;
  static constexpr int OFF_VB = OFF_VS + SB_BYTES;
  static constexpr int OFF_K = OFF_VB + SB_BYTES;
  static constexpr int OFF_V = OFF_K + K_BYTES;
  static constexpr int STAGE = OFF_V + V_BYTES;
  static_assert(OFF_K % 1024 == 0 && STAGE % 1024 == 0, "swizzle atom alignment");
  static constexpr uint32_t STAGE_TX = K_BYTES + V_BYTES + 4 * SB_BYTES;
  static_assert(TILE % 32 == 0 && TILE <= 256 && 256 % TILE == 0, "tile must divide the capacity granule");
};
constexpr int UNIT_CAP = 1024;  // units per launch (their tile prefix travels by value)
constexpr int GRID_CAP = 1024;  // CTAs per launch (their tile ranges travel by value)
constexpr int MIN_TILES_PER_CTA = 8;
// Rows a fused append writes at most (its new rows sit in one decode tile).
constexpr int kFreshRows = 128;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float NEG_INF = -__builtin_huge_valf();
// Score of a key a bool mask hides: far below any real score (|q.k| * scale
// stays well under 1e5), so it weighs exactly 0 next to one; finite and equal
// for every hidden key, so a row whose keys are all hidden averages them
// uniformly, like the page's where(mask, s, finfo.min) softmax; and small
// enough that its log2 and the running max agree to a fraction of a unit.
constexpr float MASKED_SCORE = -1e6f;
#ifndef IQ_QREG
#define IQ_QREG 0  // 1: keep the query fragments in registers (measured slower: register spills)
#endif
// Lazy running max: the reference of a row moves only when a score exceeds it
// by more than 2^tau (log2 units), so p = 2^(s - m) stays below 2^tau.  The
// reference is kept E above the row max, where E (per warp, 0 until a value
// scale of 2^(9 + E) or more shows up) keeps p * s_v below 2^15, inside fp16:
// tau = TAU - E, and raising E shifts the reference (a common factor of P,
// the row sum and the value bias, so the softmax is unchanged).
constexpr int TAU = 6;
constexpr int kScaleExpBase = 127 + 15 - TAU;  // bf16 exponent field of 2^(15 - TAU)
// Queries enter the score MMAs as fp16 q_s = q'' * 2^-e with e chosen per row
// so that max |q_s| lies in [2^14, 2^15); e is clamped to this range (rows
// whose largest entry is below 2^-86 keep the clamp and lose low bits).
constexpr int kQExpMin = -100, kQExpMax = 100;
// Value code k (0..7) of a lane's 24-bit field sits at bit LPOS(k) of its
// 16-bit window (windows start at field bits 0, 8, 16): the MMA sees
// c * 2^(LPOS - 24), undone per output dim at the end of a unit.
__host__ __device__ constexpr int vpos(int k) { return (0x52741630 >> (4 * k)) & 15; }
static_assert(vpos(0) == 0 && vpos(1) == 3 && vpos(2) == 6 && vpos(3) == 1 && vpos(5) == 7 && vpos(7) == 5,
              "3-bit field positions");
// The P.V product multiplies codes c in [0, 7] by w_hat = fp16(p * s_v); its
// rounding error w - w_hat weighs (c - VCENTRE) instead of c: one more MMA
// against an all-ones operand gives sum_t w_hat exactly as the tensor core
// saw it, VCENTRE times that is taken off, and VCENTRE * sum_t p s_v (fp32)
// joins the bias term.
constexpr float VCENTRE = 3.5f;
constexpr uint32_t kOnesF16x2 = 0x3C003C00u;  // fp16 (1, 1)
// Row of the 16-token sub-tile that MMA token slot m (0..7) reads; slot m+8
// reads row mu(m)+8.  Chosen so the swizzled K reads and the 96-byte-pitch V
// reads are free of shared-memory bank conflicts.
constexpr uint32_t MU_PACK = 0x47126530u;  // mu = {0,3,5,6,2,1,7,4}

struct Params {
  const uint32_t* k_codes;
  const uint16_t* k_scales;
  const uint16_t* k_biases;
  const uint32_t* v_codes;
  const uint16_t* v_scales;
  const uint16_t* v_biases;
  const uint16_t* q;
  const uint16_t* rot;
  float* part_o;       // [slots][GT][256]
  float* part_ml;      // [slots][GT][2] (running max in log2 units, running sum)
  unsigned* status;
  // [UNIT_CAP]: partials stored per unit of this launch; the combine takes its
  // unit's expected count off again (also when its wait runs out), so every
  // counter is back at zero once the attention grid has completed.  Two sets
  // in the workspace, used by alternate launches on it (see early).
  unsigned* counters;
  // 1: every CTA releases the dependent launch (this launch's combine) as soon
  // as it starts, so the combine's CTAs sit beside the attention CTAs from the
  // start and the next launch takes each SM this one leaves.  The host sets it
  // only for a grid of one CTA per SM (two attention CTAs never share an SM,
  // so once all of this grid's CTAs have started, every CTA of the launch two
  // before has completed, and with it the combine before that, which used the
  // same counter set) and when it knows the previous launch on the workspace
  // used the other counter set.  0: release after griddepcontrol.wait, in
  // end_unit (the combine then starts after the previous one has completed).
  int early;
  // bounded waits: mbarrier tests per wait, the combine's wait in ns
  unsigned spin_limit;
  unsigned long long combine_wait_ns;
  // partial blocks (kCombineRows rows of one segment) the combine stages in
  // shared memory per round: as many as fit beside the attention CTA
  int combine_blocks;
  // test hook (iq_debug_inject): bit 0 the combine expects one arrival that
  // never comes; bit 1 the consumers wait on a barrier no one arrives at (in
  // place of their first stage), so that wait runs out
  int inject;
  // fused append (n_new > 0): the new rows [lens[b] - n_new, lens[b]) of every
  // (sequence, kv head) are encoded from these bf16 [B][Hkv][n_new][256] rows
  // by the CTA that streams the unit's last tile, which holds them all
  const uint16_t* k_new;
  const uint16_t* v_new;
  int n_new;
  int encode_wait;  // 1: the previous attention on this cache may still read rows the new rows overwrite
  // explicit mask (mask_kind 2: float32 added to the scores; 3: uint8, 0 =
  // masked): [B][nq][mask_stride] over the keys, shared by every head
  int mask_kind;
  const void* mask;
  long long mask_stride;
  void* out;
  int out_f32;
  int batch, kv_heads, rep, nq, cap, nqt, causal;
  int unit_base, num_units, grid;  // this launch covers units [unit_base, unit_base + num_units)
  float scale;
  int lens[IQ_MAX_BATCH];
  int prefix[UNIT_CAP + 1];  // tile prefix over this launch's units
  int cstart[GRID_CAP + 1];  // CTA k streams tiles [cstart[k], cstart[k+1]) (maybe none)
};

__device__ __forceinline__ int tile_limit(const Params& p, int T, int qt, int gt) {
  if (!p.causal) return T;
  const int rmax = min(qt * gt + gt - 1, p.rep * p.nq - 1);
  return T - p.nq + rmax / p.rep + 1;
}

// The CTA that streams tile x: the last k with cstart[k] <= x (never one with
// an empty range).
__device__ __forceinline__ int cta_of(const Params& p, long long x) {
  int lo = 0, hi = p.grid - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.cstart[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// CTAs holding tiles of unit u of this launch: k_first .. k_last (partial
// slots u + k; CTAs in between with empty ranges hold no partial)
__device__ __forceinline__ void seg_range(const Params& p, int u, int& k_first, int& k_last) {
  k_first = cta_of(p, p.prefix[u]);
  k_last = cta_of(p, p.prefix[u + 1] - 1);
}

// The two M_b blocks of output dims 8*l8 .. 8*l8+7 (32 bf16).
__device__ __forceinline__ void load_rot(const Params& p, int l8, uint32_t (&mw)[16]) {
  const uint4* r4 = reinterpret_cast<const uint4*>(p.rot) + l8 * 4;
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    const uint4 v = __ldg(r4 + q4);
    mw[4 * q4] = v.x; mw[4 * q4 + 1] = v.y; mw[4 * q4 + 2] = v.z; mw[4 * q4 + 3] = v.w;
  }
}

// Output of one (row r of unit ub, 8-dim chunk l8): normalise by L, undo the
// rotation (out[4c+i] = sum_j o[4c+j] * M_b[c][i][j]) and store bf16 or fp32.
template <int GT>
__device__ __forceinline__ void store_out(const Params& p, int ub, int r, int l8, const float (&acc)[8], float L,
                                          const uint32_t (&mw)[16]) {
  const int R = (ub % p.nqt) * GT + r, i = R / p.rep, hr = R % p.rep;
  const int bb = ub / (p.kv_heads * p.nqt), hh = (ub / p.nqt) % p.kv_heads;
  if (!(L > 0.f)) atomicOr(p.status, 4u);
  const float inv = __frcp_rn(L);
  float o[8];
#pragma unroll
  for (int d = 0; d < 8; ++d) o[d] = acc[d] * inv;
  float y[8];
#pragma unroll
  for (int cb = 0; cb < 2; ++cb)
#pragma unroll
    for (int ii = 0; ii < 4; ++ii) {
      float sacc = 0.f;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int e = cb * 16 + ii * 4 + jj;
        const float m = bf16_to_f32((e & 1) ? (mw[e >> 1] >> 16) : (mw[e >> 1] & 0xFFFFu));
        sacc = jj == 0 ? o[4 * cb] * m : fmaf(o[4 * cb + jj], m, sacc);
      }
      y[4 * cb + ii] = sacc;
    }
  const int hq = hh * p.rep + hr;
  const long long orow = (static_cast<long long>(bb) * p.kv_heads * p.rep + hq) * p.nq + i;
  if (p.out_f32) {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow * kHeadDim + 8 * l8);
    dst[0] = make_float4(y[0], y[1], y[2], y[3]);
    dst[1] = make_float4(y[4], y[5], y[6], y[7]);
  } else {
    uint4 v;
    v.x = f32_to_bf16_bits(y[0]) | (f32_to_bf16_bits(y[1]) << 16);
    v.y = f32_to_bf16_bits(y[2]) | (f32_to_bf16_bits(y[3]) << 16);
    v.z = f32_to_bf16_bits(y[4]) | (f32_to_bf16_bits(y[5]) << 16);
    v.w = f32_to_bf16_bits(y[6]) | (f32_to_bf16_bits(y[7]) << 16);
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + orow * kHeadDim + 8 * l8) = v;
  }
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* ptr) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
constexpr unsigned long long kCombineWaitNs = 4000000000ull;  // 4 s: far above any attention grid
// The next attention call of this host thread uses these limits and injected
// failures (iq_debug_inject; zero = the defaults, nothing injected), then they reset.
struct DebugInject {
  int flags = 0;
  unsigned spin_limit = 0;
  unsigned long long wait_ns = 0;
};
thread_local DebugInject t_inject;

// Programmatic dependent launch: a grid launched with programmatic stream
// serialization may start once every CTA of its predecessor has executed
// launch_dependents (or exited); griddepcontrol.wait then blocks until the
// predecessor has completed and its writes are visible.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// group G's bf16 from a packed row of 4 bf16 (uint2)
__device__ __forceinline__ float pick_bf16(uint2 v, int G) {
  const uint32_t w = (G & 2) ? v.y : v.x;
  return bf16_to_f32((G & 1) ? (w >> 16) : (w & 0xFFFFu));
}

// Key codes enter the q.K product as bare fields: the code in the low nibble
// of a byte (an even dim) masked in place is the fp16 subnormal c * 2^-24, the
// code in the high nibble (an odd dim) is c * 2^-20.  Every MMA multiplies
// fp16 codes by fp16 queries (exact products, fp32 accumulation); the odd-dim
// query operand is pre-scaled by 2^-4 so all products carry 2^-24.

// The 16 codes of two consecutive words (dims 0..7 in w0, 8..15 in w1) ->
// eight registers; register m holds the dims k_pair(m, 0..1): even m the
// low-nibble codes (even dims), odd m the high-nibble codes (odd dims).  Two
// byte permutes bring the nibbles of bytes 1 and 3 down; every register is
// then one AND.
__host__ __device__ constexpr int k_pair(int m, int h) {
  // {0,4} {1,5} {8,12} {9,13} {2,10} {3,11} {6,14} {7,15}
  return h == 0 ? (m < 4 ? (m & 1) + 8 * (m >> 1) : (m == 4 ? 2 : m == 5 ? 3 : m)) : k_pair(m, 0) + (m < 4 ? 4 : 8);
}
static_assert(k_pair(0, 1) == 4 && k_pair(3, 0) == 9 && k_pair(3, 1) == 13 && k_pair(4, 1) == 10 &&
                  k_pair(6, 0) == 6 && k_pair(7, 1) == 15 && k_pair(2, 0) == 8,
              "register -> dim map");
// Registers of k-step s of a 16-dim chunk: steps 0, 1 are the even-dim MMAs
// over registers (0, 2) and (4, 6), steps 2, 3 the odd-dim MMAs over (1, 3)
// and (5, 7); h = 0 feeds k-slots 2t, 2t+1, h = 1 slots 2t+8, 2t+9.
__host__ __device__ constexpr int kreg(int s, int h) { return s < 2 ? 4 * s + 2 * h : 4 * (s - 2) + 2 * h + 1; }
static_assert(k_pair(kreg(0, 0), 0) % 2 == 0 && k_pair(kreg(1, 1), 1) % 2 == 0 && k_pair(kreg(2, 0), 0) % 2 == 1 &&
                  k_pair(kreg(3, 1), 1) % 2 == 1,
              "steps 0, 1 hold even dims, steps 2, 3 odd dims");
__device__ __forceinline__ void unpack_k16(uint32_t w0, uint32_t w1, uint32_t* r) {
  constexpr uint32_t LO = 0x000F000Fu, HI = 0x00F000F0u;
  const uint32_t x = __byte_perm(w0, w1, 0x0501);  // bytes w0.b1 (nibbles 2, 3), w1.b1
  const uint32_t y = __byte_perm(w0, w1, 0x0703);  // bytes w0.b3 (nibbles 6, 7), w1.b3
  r[0] = w0 & LO;  // (0, 4)
  r[1] = w0 & HI;  // (1, 5)
  r[2] = w1 & LO;  // (8, 12)
  r[3] = w1 & HI;  // (9, 13)
  r[4] = x & LO;   // (2, 10)
  r[5] = x & HI;   // (3, 11)
  r[6] = y & LO;   // (6, 14)
  r[7] = y & HI;   // (7, 15)
}

// fp32 -> fp16 bits, round to nearest even (subnormal results rounded, not flushed)
__device__ __forceinline__ uint32_t f32_to_f16_bits(float x) {
  return static_cast<uint32_t>(__half_as_ushort(__float2half_rn(x)));
}
__device__ __forceinline__ float f16_bits_to_f32(uint32_t h) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

// Two 24-bit fields (8 codes each; token a in fa, token b in fb) -> 8 fp16x2
// pairs (code k of a in the low half, of b in the high half), code k as the
// bare field c * 2^(vpos(k) - 24).
__device__ __forceinline__ void unpack_v3_pair(uint32_t fa, uint32_t fb, uint32_t* h) {
  const uint32_t x0 = __byte_perm(fa, fb, 0x5410);  // bits 0..15 of each
  const uint32_t x1 = __byte_perm(fa, fb, 0x6521);  // bits 8..23
  const uint32_t x2 = __byte_perm(fa, fb, 0x7632);  // bits 16..31
#pragma unroll
  for (int k = 0; k < 8; ++k) h[k] = (k < 3 ? x0 : k < 6 ? x1 : x2) & (0x00070007u << vpos(k));
}
// 2^k as a float (exponent field), |k| <= 126
__device__ __forceinline__ float exp2i(int k) { return __int_as_float((127 + k) << 23); }

// The split combine runs as small CTAs beside the attention CTAs: registers
// are split evenly over the four warp schedulers of an SM, so next to an
// attention CTA (three warps of 160 registers per scheduler) one warp of at
// most 32 registers per scheduler fits.
constexpr int kCombineThreads = 128, kCombineRegs = 32;

template <int NT, int DS, int STREAMS, int NSTAGE, int MINB, int TILE_, int PAIR, int HALVES>
struct Cfg : Tiling<TILE_> {
  using Tiling<TILE_>::STAGE;
  static constexpr int GT = 8 * NT;            // query rows per unit
  static constexpr int GPW = 4 / DS;           // 64-dim groups per consumer warp
  static constexpr int CW = DS * STREAMS;      // consumer warps of a half
  // HALVES independent halves (each its own tile range, ring, producer lane
  // and CW consumer warps, a multiple of 4), then one producer warpgroup whose
  // warp h streams the tiles of half h; registers move from the producer
  // warpgroup to the consumers (setmaxnreg).  Two halves share an SM as two
  // CTAs would, but their consumer warps alternate over the four warp
  // schedulers, so neither half is served first (two CTAs on one SM are not:
  // the scheduler favours the older one, which finishes ~12% earlier).
  static constexpr int THREADS = (HALVES * CW + 4) * 32;
  // registers left free beside each CTA on its SM: one combine CTA fits next
  // to it, so a split merge never needs an SM of its own (see combine_kernel)
  static constexpr int RESERVE_REGS = kCombineThreads * kCombineRegs;

  static constexpr int LAUNCH_REGS = ((65536 / MINB - RESERVE_REGS) / THREADS) / 8 * 8;
  static_assert(MINB > 1 || (THREADS % 128 == 0 && THREADS / 128 * LAUNCH_REGS * 32 + kCombineRegs * 32 <= 16384),
                "a combine warp fits beside the CTA on every warp scheduler");
  static constexpr int PRODUCER_REGS = 24;
  static constexpr int CONSUMER_REGS =
      ((LAUNCH_REGS * THREADS - 128 * PRODUCER_REGS) / (HALVES * CW * 32)) / 8 * 8 > 248
          ? 248
          : ((LAUNCH_REGS * THREADS - 128 * PRODUCER_REGS) / (HALVES * CW * 32)) / 8 * 8;
  static_assert(CW % 4 == 0, "consumer warps form whole warpgroups");
  static_assert(HALVES == 1 || (HALVES == 2 && CW == 4), "two halves of one consumer warpgroup each");
  static_assert(CONSUMER_REGS >= LAUNCH_REGS && PRODUCER_REGS <= LAUNCH_REGS, "register split");
  static_assert(HALVES * CW * 32 * CONSUMER_REGS + 128 * PRODUCER_REGS <= LAUNCH_REGS * THREADS,
                "the split fits the block's launch allocation");
  static constexpr int OBUF_BYTES = GT * 256 * 4;  // the CTA's merged O of a unit
  static constexpr int OFF_OBUF = NSTAGE * STAGE;
  static constexpr int OFF_QSUM = OFF_OBUF + OBUF_BYTES;
  static constexpr int OFF_MBUF = OFF_QSUM + GT * 32;
  static constexpr int OFF_LBUF = OFF_MBUF + STREAMS * GT * 4;
  static constexpr int OFF_XBUF = OFF_LBUF + STREAMS * GT * 4;
  static constexpr int XBUF_BYTES = DS > 1 ? STREAMS * 2 * 2 * DS * NT * 32 * 16 : 0;  // x2 parities x2 sub-tiles
  static constexpr int OFF_QB = OFF_XBUF + XBUF_BYTES;
  static constexpr int QB_BYTES = DS * GPW * 4 * NT * 32 * 8;       // q_s MMA B fragments
  static constexpr int OFF_RMX = OFF_QB + QB_BYTES;                  // per (row, group): max |q''| (bf16 bits)
  static constexpr int OFF_REXP = OFF_RMX + GT * 4 * 4;              // per row: the query exponent e
  // per row of the segment being finished: max and sum over the streams
  static constexpr int OFF_MLR = (OFF_REXP + GT * 4 + 15) / 16 * 16;
  static constexpr int OFF_BAR = (OFF_MLR + GT * 8 + 7) / 8 * 8;
  static constexpr int OFF_FLAG = OFF_BAR + 2 * NSTAGE * 8 + 8;  // + the fused-append barrier
  // explicit-mask rows of a stage (the unit's queries, at most GT, x TILE keys,
  // 4-byte elements at most): the last area, part of the launch only with a mask
  static constexpr int MSK_STAGE = GT * TILE_ * 4;
  static constexpr int OFF_MSK = (OFF_FLAG + 16 + 127) / 128 * 128;
  // without a mask, that area holds instead the first unit segment of a range
  // that has several (its O, per-row max and sum), kept until the range ends
  static constexpr int OFF_DBUF = OFF_MSK;
  static constexpr int OFF_DML = OFF_DBUF + OBUF_BYTES;
  // one half's area, a multiple of the 1024-byte swizzle atom
  static constexpr int HALF_PLAIN = (OFF_DML + GT * 8 + 1023) / 1024 * 1024;
  static constexpr int HALF_MASK = (OFF_MSK + NSTAGE * MSK_STAGE + 1023) / 1024 * 1024;
  static constexpr int SMEM = HALVES * HALF_PLAIN + 1024;  // + alignment slack
  static constexpr int SMEM_MASK = HALVES * HALF_MASK + 1024;
  static_assert(SMEM <= 227 * 1024 && SMEM_MASK <= 227 * 1024, "shared memory per CTA");
  static_assert(OFF_XBUF % 16 == 0 && OFF_OBUF % 16 == 0 && OFF_BAR % 8 == 0, "alignment");
  static_assert(4 % DS == 0, "shape");
  // the masked variant's producer also copies mask rows: it takes 8 registers
  // per consumer thread from the consumers
  static constexpr int CONSUMER_REGS_MASK = CONSUMER_REGS - 8;
  static constexpr int PRODUCER_REGS_MASK =
      (LAUNCH_REGS * THREADS - HALVES * CW * 32 * CONSUMER_REGS_MASK) / 128 / 8 * 8 > 248
          ? 248
          : (LAUNCH_REGS * THREADS - HALVES * CW * 32 * CONSUMER_REGS_MASK) / 128 / 8 * 8;
  static_assert(CONSUMER_REGS_MASK >= LAUNCH_REGS && PRODUCER_REGS_MASK >= PRODUCER_REGS, "masked register split");
  static_assert(HALVES * CW * 32 * CONSUMER_REGS_MASK + 128 * PRODUCER_REGS_MASK <= LAUNCH_REGS * THREADS,
                "the masked split fits the block's launch allocation");
};

template <int NT, int DS, int STREAMS, int NSTAGE, int MINB, int TILE_, int PAIR, int HALVES, bool MASKED>
__global__ void __maxnreg__((Cfg<NT, DS, STREAMS, NSTAGE, MINB, TILE_, PAIR, HALVES>::LAUNCH_REGS))
    attend_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap kmap) {
  using C = Cfg<NT, DS, STREAMS, NSTAGE, MINB, TILE_, PAIR, HALVES>;
  constexpr int TILE = C::TILE, SUBS = C::SUBS, STAGE = C::STAGE;
  constexpr int OFF_K = C::OFF_K, OFF_V = C::OFF_V, OFF_KS = C::OFF_KS, OFF_KB = C::OFF_KB;
  constexpr int OFF_VS = C::OFF_VS, OFF_VB = C::OFF_VB, V_BYTES = C::V_BYTES, SB_BYTES = C::SB_BYTES;
  constexpr uint32_t STAGE_TX = C::STAGE_TX;
  constexpr int GT = C::GT, GPW = C::GPW, CW = C::CW, NCT = CW * 32;
  constexpr int HALF_BYTES = MASKED ? C::HALF_MASK : C::HALF_PLAIN;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base (128-byte swizzle atom), derived by pointer
  // arithmetic on the shared array so loads through it stay shared-memory loads
  uint8_t* const smem0 = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

  // ---- roles: the half a warp serves and its index among the half's consumers
  // (two halves: half ((w >> 2) ^ w) & 1, index (w >> 1) & 3, so each warp
  // scheduler w % 4 holds one consumer warp of each half); producer warpgroup
  // warp HALVES*CW + h streams for half h, its other warps idle
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool consumer = warp < HALVES * CW;
  const int half = consumer ? (HALVES == 2 ? ((warp >> 2) ^ warp) & 1 : 0) : warp - HALVES * CW;
  const int cw = consumer ? (HALVES == 2 ? (warp >> 1) & 3 : warp) : 0;
  uint8_t* const smem = smem0 + (half < HALVES ? half : 0) * HALF_BYTES;
  float* qsum = reinterpret_cast<float*>(smem + C::OFF_QSUM);
  float* mbuf = reinterpret_cast<float*>(smem + C::OFF_MBUF);
  float* lbuf = reinterpret_cast<float*>(smem + C::OFF_LBUF);
  float4* xbuf = reinterpret_cast<float4*>(smem + C::OFF_XBUF);
  float* obuf = reinterpret_cast<float*>(smem + C::OFF_OBUF);
  uint2* qbs = reinterpret_cast<uint2*>(smem + C::OFF_QB);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + NSTAGE;
  uint64_t* encoded = empty + NSTAGE;  // fused append: every consumer warp has stored its new rows
  // named barriers of this half: every consumer warp, and (DS > 1) one per token stream
  const int bar_all = 1 + half * (1 + STREAMS);

  // Launched as a programmatic dependent of the previous kernel in the stream,
  // this grid may start while that kernel (the previous call's combine) and
  // the attention before it still run.  Of the memory it touches, only these
  // may still be written by them: the output, the partials and counters (every
  // write of this grid to them comes after griddepcontrol.wait, in end_unit),
  // and the cache rows of the previous call's fused append, all among the last
  // kFreshRows + n_new rows of a sequence (the producer waits before a tile
  // that reaches them).  The append kernel releases its dependents only when it
  // completes, and the combine writes no cache rows, so every other cache tile,
  // the queries and the rotation can be streamed before the wait.  The fused
  // append's own writes wait too when the host saw a trim since the previous
  // attention on this cache (that attention may still read those rows).
  if (threadIdx.x == 0) {
    for (int h = 0; h < HALVES; ++h) {
      uint64_t* f = reinterpret_cast<uint64_t*>(smem0 + h * HALF_BYTES + C::OFF_BAR);
      for (int s = 0; s < NSTAGE; ++s) {
        mbar_init(&f[s], 1);
        mbar_init(&f[NSTAGE + s], CW);
      }
      mbar_init(&f[2 * NSTAGE], CW);
    }
    mbar_fence_init();
  }
  __syncthreads();
  if (p.early) pdl_launch_dependents();

  // ---- this half's share of the launch's tiles
  const int k_cta = blockIdx.x * HALVES + (half < HALVES ? half : 0);
  const long long g0 = p.cstart[k_cta], g1 = p.cstart[k_cta + 1];
  int u0 = 0;  // unit holding tile g0: last u with prefix[u] <= g0
  {
    int lo = 0, hi = p.num_units - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.prefix[mid] <= g0) lo = mid; else hi = mid - 1;
    }
    u0 = lo;
  }
  int u1 = u0;  // unit holding tile g1 - 1
  while (g1 > p.prefix[u1 + 1]) ++u1;

  // ------------------------------------------------------------ producer
  // One lane streams the CTA's tiles through the ring, refilling a stage as
  // soon as every consumer warp has released it: packed K codes by a 2-D
  // tensor copy (128-byte swizzle), packed V codes and the four scale/bias rows
  // by 1-D bulk copies, all counted on the stage's full barrier; L2
  // evict-first (the cache is read once).
  if (!consumer) {
    setmaxnreg_dec<MASKED ? C::PRODUCER_REGS_MASK : C::PRODUCER_REGS>();
    if (half < HALVES && lane == 0 && g0 < g1) {
      const uint64_t pol = policy_evict_first();
      long long k = 0;
      bool enc_seen = p.n_new == 0;
      bool waited = false;  // griddepcontrol.wait done
      // the range's unit segments, last unit first (the consumers' order)
      int u = u1;
      int gt = max(static_cast<int>(g0), p.prefix[u1]);
      for (;; ++gt, ++k) {
        if (gt >= min(static_cast<int>(g1), p.prefix[u + 1])) {
          if (u == u0) break;
          --u;
          gt = max(static_cast<int>(g0), p.prefix[u]);
        }
        if (!enc_seen && gt == p.prefix[u + 1] - 1) {  // a last tile: its new rows must be stored first
          if (!mbar_wait(encoded, 0, p.spin_limit)) {
            atomicOr(p.status, 1u);
            break;
          }
          enc_seen = true;
        }
        const int ug = p.unit_base + u;
        const int bb = ug / (p.kv_heads * p.nqt), hh = (ug / p.nqt) % p.kv_heads;
        const int st = static_cast<int>(k % NSTAGE);
        if (k >= NSTAGE && !mbar_wait(&empty[st], static_cast<uint32_t>((k / NSTAGE) - 1) & 1, p.spin_limit)) {
          atomicOr(p.status, 1u);
          break;
        }
        uint8_t* sbp = smem + st * STAGE;
        const long long row0 = (static_cast<long long>(bb) * p.kv_heads + hh) * p.cap + (gt - p.prefix[u]) * TILE;
        if (!waited && (gt - p.prefix[u] + 1) * TILE > p.lens[bb] - p.n_new - kFreshRows) {
          pdl_wait();  // the tile may hold rows the previous call's fused append wrote
          waited = true;
        }
        if constexpr (MASKED) {  // the unit's mask rows for this tile's keys (one copy per query)
          const int qt = ug % p.nqt, elem = p.mask_kind == 2 ? 4 : 1;
          const int i_lo = qt * C::GT / p.rep, i_hi = min((qt * C::GT + C::GT - 1) / p.rep, p.nq - 1);
          const uint32_t bytes = TILE * elem;
          mbar_arrive_expect_tx(&full[st], STAGE_TX + (i_hi - i_lo + 1) * bytes);
          for (int i = i_lo; i <= i_hi; ++i)
            bulk_g2s_plain(smem + C::OFF_MSK + st * C::MSK_STAGE + (i - i_lo) * bytes,
                           static_cast<const uint8_t*>(p.mask) +
                               ((static_cast<long long>(bb) * p.nq + i) * p.mask_stride + (gt - p.prefix[u]) * TILE) *
                                   elem,
                           bytes, &full[st]);
        } else {
          mbar_arrive_expect_tx(&full[st], STAGE_TX);
        }
        tensor2d_g2s(sbp + OFF_K, &kmap, 0, static_cast<int>(row0), &full[st], pol);
        bulk_g2s(sbp + OFF_V, p.v_codes + row0 * kVWords, V_BYTES, &full[st], pol);
        bulk_g2s(sbp + OFF_KS, p.k_scales + row0 * kGroups, SB_BYTES, &full[st], pol);
        bulk_g2s(sbp + OFF_KB, p.k_biases + row0 * kGroups, SB_BYTES, &full[st], pol);
        bulk_g2s(sbp + OFF_VS, p.v_scales + row0 * kGroups, SB_BYTES, &full[st], pol);
        bulk_g2s(sbp + OFF_VB, p.v_biases + row0 * kGroups, SB_BYTES, &full[st], pol);
      }
      // never leave with copies in flight: wait for the last tile issued to each stage
      for (long long s = 0; s < NSTAGE && s < k; ++s) {
        const long long last = s + NSTAGE * ((k - 1 - s) / NSTAGE);
        mbar_wait(&full[s], static_cast<uint32_t>(last / NSTAGE) & 1, p.spin_limit);
      }
    }
    return;
  }
  setmaxnreg_inc<MASKED ? C::CONSUMER_REGS_MASK : C::CONSUMER_REGS>();
  if (g0 >= g1) {  // a half without tiles (it still waits, so its exit implies the previous grid's completion)
    pdl_wait();
    return;
  }

  // ------------------------------------------------------------ consumers
  const int stream = cw / DS, dg = cw % DS;
  const int ctid = cw * 32 + lane;  // thread index among the half's consumers
  const int g = lane >> 2, t = lane & 3;
  const int rS0 = (MU_PACK >> (4 * g)) & 15;      // token slot g
  const int rV0 = (MU_PACK >> (8 * t)) & 15;      // slot 2t
  const int rV1 = (MU_PACK >> (8 * t + 4)) & 15;  // slot 2t+1
  const int vword = (3 * g) >> 2, vshift = (24 * g) & 31;
  const uint32_t kswz = ((t & 1) << 3);

  // per-unit state
  int b = 0, kvh = 0, qt = 0, T = 0, limit = 0, qmin = 0;
  int qpos[NT][2];
  int qrow[NT][2];  // query index of rows 2t, 2t+1 of each n-tile (explicit masks)
  int qlo = 0;      // the unit's first query (its mask row is the stage's first)
  // B fragments of the per-token bias product (one bf16 MMA per n-tile):
  // k-slots [b_0..b_3, b_0..b_3, b_0..b_3, 0 x 4] of a key row against
  // [S_hi, S_mid, S_lo, 0], S_G = 2^-24 * sum of q_s over group G for this
  // lane's query row, split into three bf16 parts that add up to it exactly
  uint32_t kbq[NT][2];
  float kmul[NT][2];  // per row: log2(e) * 2^(24 + e), raw score -> log2 units
  float O[GPW][4][NT][4];
  float bacc[GPW][NT][2];
  float wsum[GPW][NT][4];
#if IQ_QREG
  uint2 qreg[GPW][4][NT];  // this warp's q_s MMA B fragments (from shared memory, once per unit)
#endif  // sum of w_hat per (group, query row) (rows g, g+8 alike)
  float msc[NT][2], lrow[NT][2];  // reference max (log2 units), partial row sum
  int xpar = 0;
  int E = 0;  // value-scale shift of the reference (see TAU)
  float* rmx = reinterpret_cast<float*>(smem + C::OFF_RMX);
  int* rexp = reinterpret_cast<int*>(smem + C::OFF_REXP);
  static_assert(NT * 4 <= CW, "one query item (n-tile, group) per consumer warp");

  // ---- start unit u: rotate and scale its queries, load the MMA fragments, reset the state
  auto begin_unit = [&](int u) {
    const int ug = p.unit_base + u;
    b = ug / (p.kv_heads * p.nqt);
    kvh = (ug / p.nqt) % p.kv_heads;
    qt = ug % p.nqt;
    T = p.lens[b];
    limit = tile_limit(p, T, qt, GT);
    // the first key some row of the unit cannot see (no sub-tile at or past it
    // takes the unmasked path); an explicit mask reads every sub-tile
    qmin = MASKED ? -1 : p.causal ? T - p.nq + (qt * GT) / p.rep : T - 1;
    qlo = (qt * GT) / p.rep;
    named_bar(bar_all, NCT);  // every consumer is done with the previous unit's fragments and sums
    // q' = bf16(q @ M_b), q'' = bf16(q' * scale).  Item (n-tile j, group G)
    // goes to one warp; its thread (g, t) rotates row 8j+g, dims 64G+16t ..
    // +15 (rotation blocks 16G+4t .. +3), whose register m holds the dims
    // k_pair(m, 0..1); k-step s uses registers 2s (slots 2t, 2t+1) and 2s+1.
    // Rows r <-> (query R/rep, head R%rep); rows past the queries are zero.
    // Phase 1: q'' and the row's largest magnitude (per group, in shared
    // memory); phase 2: the row exponent e and the fp16 fragments of
    // q_s = q'' * 2^-e ([dim group][k-step][n-tile][lane] in shared memory).
    const int item = cw;
    const bool has_item = item < NT * 4;
    const int j_it = item >> 2, G_it = item & 3;
    uint32_t yb[16];  // q'' (bf16 bits) of the thread's 16 dims
    if (has_item) {
      const int R = qt * GT + 8 * j_it + g, i = R / p.rep, hr = R % p.rep;
      if (i < p.nq) {
        const long long qrow =
            (static_cast<long long>(b) * p.kv_heads * p.rep + kvh * p.rep + hr) * p.nq + i;
        const uint4* qv = reinterpret_cast<const uint4*>(p.q + qrow * kHeadDim + 64 * G_it + 16 * t);
        const uint4* rv = reinterpret_cast<const uint4*>(p.rot + (16 * G_it + 4 * t) * 16);
        uint4 qw4[2], mw4[8];
#pragma unroll
        for (int c = 0; c < 2; ++c) qw4[c] = __ldg(qv + c);
#pragma unroll
        for (int c = 0; c < 8; ++c) mw4[c] = __ldg(rv + c);
        const uint32_t qw[8] = {qw4[0].x, qw4[0].y, qw4[0].z, qw4[0].w, qw4[1].x, qw4[1].y, qw4[1].z, qw4[1].w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {  // rotation block 16G + 4t + c: dims 4c .. 4c+3 of the thread
          const uint32_t mw[8] = {mw4[2 * c].x, mw4[2 * c].y, mw4[2 * c].z, mw4[2 * c].w,
                                  mw4[2 * c + 1].x, mw4[2 * c + 1].y, mw4[2 * c + 1].z, mw4[2 * c + 1].w};
          float x[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t w = qw[(4 * c + e) >> 1];
            x[e] = bf16_to_f32((e & 1) ? (w >> 16) : (w & 0xFFFFu));
          }
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {  // y[jj] = sum_k x[k] * M_b[k][jj], f32 in order k = 0..3
            float acc = 0.f;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const int e = kk * 4 + jj;
              const float mkj = bf16_to_f32((e & 1) ? (mw[e >> 1] >> 16) : (mw[e >> 1] & 0xFFFFu));
              acc = kk == 0 ? __fmul_rn(x[0], mkj) : __fadd_rn(acc, __fmul_rn(x[kk], mkj));
            }
            yb[4 * c + jj] = f32_to_bf16_bits(__fmul_rn(round_bf16(acc), p.scale));
          }
        }
      } else {
#pragma unroll
        for (int d = 0; d < 16; ++d) yb[d] = 0u;
      }
      uint32_t mx = 0;  // largest |q''| as bf16 bits (monotonic in the magnitude)
#pragma unroll
      for (int d = 0; d < 16; ++d) mx = max(mx, yb[d] & 0x7FFFu);
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      if (t == 0) reinterpret_cast<uint32_t*>(rmx)[(8 * j_it + g) * 4 + G_it] = mx;
    }
    named_bar(bar_all, NCT);  // every row's group maxima stored
    if (has_item) {
      const int row = 8 * j_it + g;
      const uint32_t* rm = reinterpret_cast<const uint32_t*>(rmx) + row * 4;
      const uint32_t mx = max(max(rm[0], rm[1]), max(rm[2], rm[3]));
      // e: max |q''| in [2^(e+14), 2^(e+15)); a zero row keeps e = 0
      int e = mx == 0 ? 0 : static_cast<int>(max(mx >> 7, 1u)) - 127 - 14;
      e = min(max(e, kQExpMin), kQExpMax);
      const float down = exp2i(-e), down16 = exp2i(-e - 4);
      uint32_t hb[16];  // the fp16 operand of each dim (odd dims carry an extra 2^-4)
      float qs = 0.f;   // sum of the operand values at one scale (2^-e q'')
#pragma unroll
      for (int d = 0; d < 16; ++d) {
        const float v = bf16_to_f32(yb[d]);
        hb[d] = f32_to_f16_bits(__fmul_rn(v, (d & 1) ? down16 : down));
        qs += (d & 1) ? 16.0f * f16_bits_to_f32(hb[d]) : f16_bits_to_f32(hb[d]);
      }
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        uint32_t h2[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int m = kreg(s, h);
          h2[h] = hb[k_pair(m, 0)] | (hb[k_pair(m, 1)] << 16);
        }
        qbs[((G_it * 4 + s) * NT + j_it) * 32 + lane] = make_uint2(h2[0], h2[1]);
      }
      qs += __shfl_xor_sync(0xffffffffu, qs, 1);
      qs += __shfl_xor_sync(0xffffffffu, qs, 2);
      if (t == 0) {
        qsum[row * 4 + G_it] = qs;
        if (G_it == 0) rexp[row] = e;
      }
    }
    named_bar(bar_all, NCT);  // fragments, sums and exponents visible to every warp
    // this lane's k-slots: 2t, 2t+1 = groups 2(t&1), 2(t&1)+1 of part t>>1
    // (hi for t < 2, mid for t >= 2); slots 2t+8, 2t+9 = the same groups' lo
    // part (t < 2) or nothing; groups another warp of the stream owns
    // contribute there instead
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      uint32_t parts[3] = {0u, 0u, 0u};  // bf16x2 of (group 2(t&1), group 2(t&1)+1) per part
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int G = 2 * (t & 1) + h;
        const bool mine = G >= dg * GPW && G < dg * GPW + GPW;
        float x = mine ? qsum[(8 * j + g) * 4 + G] * 0x1p-24f : 0.0f;
#pragma unroll
        for (int k = 0; k < 3; ++k) {  // x = hi + mid + lo exactly (each a bf16)
          const uint32_t bits = f32_to_bf16_bits(x);
          parts[k] |= bits << (16 * h);
          x -= bf16_to_f32(bits);
        }
      }
      kbq[j][0] = t < 2 ? parts[0] : parts[1];
      kbq[j][1] = t < 2 ? parts[2] : 0u;
    }
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int R = qt * GT + 8 * j + 2 * t + e;
        const int i = min(R / p.rep, p.nq - 1);
        qpos[j][e] = p.causal ? T - p.nq + i : T - 1;
        qrow[j][e] = i;
        kmul[j][e] = LOG2E * exp2i(24 + rexp[8 * j + 2 * t + e]);
      }
#pragma unroll
    for (int gi = 0; gi < GPW; ++gi)
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        bacc[gi][j][0] = bacc[gi][j][1] = 0.f;
        wsum[gi][j][0] = wsum[gi][j][1] = wsum[gi][j][2] = wsum[gi][j][3] = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) O[gi][i][j][0] = O[gi][i][j][1] = O[gi][i][j][2] = O[gi][i][j][3] = 0.f;
      }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      msc[j][0] = msc[j][1] = NEG_INF;
      lrow[j][0] = lrow[j][1] = 0.f;
    }
    E = 0;
#if IQ_QREG
#pragma unroll
    for (int gi = 0; gi < GPW; ++gi)
#pragma unroll
      for (int s = 0; s < 4; ++s)
#pragma unroll
        for (int j = 0; j < NT; ++j) qreg[gi][s][j] = qbs[(((dg * GPW + gi) * 4 + s) * NT + j) * 32 + lane];
#endif
  };

  // ---- N (1 or 2) of this warp's 16-token sub-tiles of one stage, processed
  // together: both score products, one softmax step, both value products (two
  // independent chains per phase, one vote and one query-fragment load per
  // k-step for both).  FULL: every token of the N sub-tiles is inside the
  // unit's range and visible to every row (no masking work at all).
  auto subtiles = [&](auto n_tag, auto full_tag, const int (&subs)[2], const int (&tokbase)[2], uint32_t sb,
                      uint32_t msk) {
    constexpr int N = decltype(n_tag)::value;
    constexpr bool FULL = decltype(full_tag)::value;
    int rr0[N], rr1[N];
    uint2 ksc0[N], ksc1[N];
    float sc[N][NT][4];
    // per-token bias: sum_G b_G S_G, by one bf16 MMA whose A operand is the
    // raw bias words of the two token rows
    const uint32_t bs_off = OFF_KB + (t & 1) * 4;
#pragma unroll
    for (int n = 0; n < N; ++n) {
      rr0[n] = subs[n] * 16 + rS0;
      rr1[n] = rr0[n] + 8;
      ksc0[n] = lds64(sb + OFF_KS + rr0[n] * 8);
      ksc1[n] = lds64(sb + OFF_KS + rr1[n] * 8);
      const uint32_t w0 = lds32(sb + bs_off + rr0[n] * 8), w1 = lds32(sb + bs_off + rr1[n] * 8);
      const uint32_t A[4] = {w0, w1, w0, w1};
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        sc[n][j][0] = sc[n][j][1] = sc[n][j][2] = sc[n][j][3] = 0.f;
        mma_bf16(sc[n][j], A, kbq[j][0], kbq[j][1]);
      }
    }

    // scores: per group, S_G = codes . q_s (fp32), added as s_G * S_G
#pragma unroll
    for (int gi = 0; gi < GPW; ++gi) {
      const int Gr = dg * GPW + gi;
      uint32_t RA[N][8], RB[N][8];
#pragma unroll
      for (int n = 0; n < N; ++n) {
        const uint32_t chunk16 = 2 * Gr + (t >> 1);
        const uint32_t a0 = sb + OFF_K + rr0[n] * 128 + ((chunk16 ^ (rr0[n] & 7)) << 4) + kswz;
        const uint32_t a1 = sb + OFF_K + rr1[n] * 128 + ((chunk16 ^ (rr1[n] & 7)) << 4) + kswz;
        const uint2 w0 = lds64(a0), w1 = lds64(a1);
        unpack_k16(w0.x, w0.y, RA[n]);
        unpack_k16(w1.x, w1.y, RB[n]);
      }
      float acc[N][NT][4];
#pragma unroll
      for (int n = 0; n < N; ++n)
#pragma unroll
        for (int j = 0; j < NT; ++j) acc[n][j][0] = acc[n][j][1] = acc[n][j][2] = acc[n][j][3] = 0.f;
#pragma unroll
      for (int s = 0; s < 4; ++s)
#pragma unroll
        for (int j = 0; j < NT; ++j) {
#if IQ_QREG
          const uint2 bq = qreg[gi][s][j];
#else
          const uint2 bq = qbs[((Gr * 4 + s) * NT + j) * 32 + lane];
#endif
#pragma unroll
          for (int n = 0; n < N; ++n) {
            const uint32_t A[4] = {RA[n][kreg(s, 0)], RB[n][kreg(s, 0)], RA[n][kreg(s, 1)], RB[n][kreg(s, 1)]};
            mma_f16(acc[n][j], A, bq.x, bq.y);
          }
        }
#pragma unroll
      for (int n = 0; n < N; ++n) {
        const float s0 = pick_bf16(ksc0[n], Gr), s1 = pick_bf16(ksc1[n], Gr);
#pragma unroll
        for (int j = 0; j < NT; ++j) {  // this warp's groups, in group order
          float* c = sc[n][j];
          const float* a = acc[n][j];
          c[0] = fmaf(s0, a[0], c[0]); c[1] = fmaf(s0, a[1], c[1]);
          c[2] = fmaf(s1, a[2], c[2]); c[3] = fmaf(s1, a[3], c[3]);
        }
      }
    }
    if constexpr (DS > 1) {  // sum the group partials of the DS warps, in group order
      float4* xb = xbuf + (stream * 2 + xpar) * 2 * DS * NT * 32;
#pragma unroll
      for (int n = 0; n < N; ++n)
#pragma unroll
        for (int j = 0; j < NT; ++j)
          xb[((n * DS + dg) * NT + j) * 32 + lane] = make_float4(sc[n][j][0], sc[n][j][1], sc[n][j][2], sc[n][j][3]);
      named_bar(bar_all + 1 + stream, DS * 32);
#pragma unroll
      for (int n = 0; n < N; ++n)
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          float4 a = xb[(n * DS * NT + j) * 32 + lane];
#pragma unroll
          for (int d = 1; d < DS; ++d) {
            const float4 v = xb[((n * DS + d) * NT + j) * 32 + lane];
            a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
          }
          sc[n][j][0] = a.x; sc[n][j][1] = a.y; sc[n][j][2] = a.z; sc[n][j][3] = a.w;
        }
      xpar ^= 1;
    }

    // value scales and biases of the two token rows (the scale test below
    // reads the scales before the softmax)
    uint2 vsc0[N], vsc1[N], vbi0[N], vbi1[N];
#pragma unroll
    for (int n = 0; n < N; ++n) {
      vsc0[n] = lds64(sb + OFF_VS + rr0[n] * 8);
      vsc1[n] = lds64(sb + OFF_VS + rr1[n] * 8);
      vbi0[n] = lds64(sb + OFF_VB + rr0[n] * 8);
      vbi1[n] = lds64(sb + OFF_VB + rr1[n] * 8);
    }

    // scores in log2 units relative to the row reference: x = y - m, with
    // y = raw * kmul (masked entries -inf, explicit masks applied to y)
    bool valid[N][NT][4];
    float x[N][NT][4];
    float ysv[N][NT][4];  // y itself (used by the masked sub-tiles' slow path)
    bool in_tok[N][2];
#pragma unroll
    for (int n = 0; n < N; ++n) {
      const int tok0 = tokbase[n] + rS0, tok1 = tok0 + 8;
      in_tok[n][0] = FULL || tok0 < limit;
      in_tok[n][1] = FULL || tok1 < limit;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        if constexpr (FULL) {
#pragma unroll
          for (int e = 0; e < 4; ++e) x[n][j][e] = fmaf(sc[n][j][e], kmul[j][e & 1], -msc[j][e & 1]);
        } else {
          valid[n][j][0] = in_tok[n][0] && tok0 <= qpos[j][0];
          valid[n][j][1] = in_tok[n][0] && tok0 <= qpos[j][1];
          valid[n][j][2] = in_tok[n][1] && tok1 <= qpos[j][0];
          valid[n][j][3] = in_tok[n][1] && tok1 <= qpos[j][1];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float y = sc[n][j][e] * kmul[j][e & 1];
            if constexpr (MASKED) {  // explicit mask (staged with the tile): added, or masked
              if (valid[n][j][e]) {
                const int mi = (qrow[j][e & 1] - qlo) * TILE + subs[n] * 16 + rS0 + (e < 2 ? 0 : 8);
                if (p.mask_kind == 2)
                  y = fmaf(__uint_as_float(lds32(msk + mi * 4)), LOG2E, y);
                else if (lds8(msk + mi) == 0)
                  y = MASKED_SCORE * LOG2E;
              }
            }
            y = valid[n][j][e] ? y : NEG_INF;
            ysv[n][j][e] = y;
            x[n][j][e] = y - msc[j][e & 1];
          }
        }
      }
    }
    // lazy max: a row moves its reference only when a score passes it by
    // 2^tau; the value-scale test: a scale at or above 2^(9 + E) raises E
    const float tau = static_cast<float>(TAU - E);
    bool trig = false;
#pragma unroll
    for (int n = 0; n < N; ++n)
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) trig |= !(x[n][j][e] <= tau);
    const uint32_t thr = static_cast<uint32_t>(min(kScaleExpBase + E, 255)) << 7;
    const uint32_t addc = (0x8000u - thr) * 0x10001u;  // bit 15 of a half set iff the half >= thr
    uint32_t over = 0;
#pragma unroll
    for (int n = 0; n < N; ++n) {
      const uint2 a = in_tok[n][0] ? vsc0[n] : make_uint2(0u, 0u);
      const uint2 c = in_tok[n][1] ? vsc1[n] : make_uint2(0u, 0u);
      over |= (a.x + addc) | (a.y + addc) | (c.x + addc) | (c.y + addc);
    }
    const bool strig = (over & 0x80008000u) != 0;
    if (__any_sync(0xffffffffu, trig || strig)) {
      int dE = 0;
      if (__any_sync(0xffffffffu, strig)) {  // largest valid scale (bf16 bits: monotonic) over the warp
        uint32_t hm = 0;
#pragma unroll
        for (int n = 0; n < N; ++n) {
          const uint2 a = in_tok[n][0] ? vsc0[n] : make_uint2(0u, 0u);
          const uint2 c = in_tok[n][1] ? vsc1[n] : make_uint2(0u, 0u);
          const uint32_t w4[4] = {a.x, a.y, c.x, c.y};
#pragma unroll
          for (int q = 0; q < 4; ++q) hm = max(hm, max(w4[q] & 0xFFFFu, w4[q] >> 16));
        }
        hm = __reduce_max_sync(0xffffffffu, hm);
        // smallest E with hm < 2^(9 + E), i.e. (hm >> 7) < kScaleExpBase + E
        const int En = min(max(E, static_cast<int>(hm >> 7) - kScaleExpBase + 1), 255 - kScaleExpBase);
        dE = En - E;
        E = En;
      }
      float alpha[NT][2];
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float mx = NEG_INF;
#pragma unroll
          for (int n = 0; n < N; ++n)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int ee = e + 2 * h;
              const float y = FULL ? sc[n][j][ee] * kmul[j][e] : ysv[n][j][ee];
              mx = fmaxf(mx, y);
            }
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float mold = msc[j][e];
          // the reference sits E above the row max, and a raised E shifts it
          const float mnew = fmaxf(mold + static_cast<float>(dE), mx + static_cast<float>(E));
          alpha[j][e] = mnew == NEG_INF ? 1.f : ex2_approx(mold - mnew);
          msc[j][e] = mnew;
        }
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        lrow[j][0] *= alpha[j][0];
        lrow[j][1] *= alpha[j][1];
#pragma unroll
        for (int gi = 0; gi < GPW; ++gi) {
          bacc[gi][j][0] *= alpha[j][0];
          bacc[gi][j][1] *= alpha[j][1];
          wsum[gi][j][0] *= alpha[j][0];
          wsum[gi][j][2] *= alpha[j][0];
          wsum[gi][j][1] *= alpha[j][1];
          wsum[gi][j][3] *= alpha[j][1];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            O[gi][i][j][0] *= alpha[j][0];
            O[gi][i][j][2] *= alpha[j][0];
            O[gi][i][j][1] *= alpha[j][1];
            O[gi][i][j][3] *= alpha[j][1];
          }
        }
#pragma unroll
        for (int n = 0; n < N; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float m = msc[j][e & 1];
            const float y = FULL ? sc[n][j][e] * kmul[j][e & 1] : ysv[n][j][e];
            x[n][j][e] = y - (m == NEG_INF ? 0.f : m);
          }
      }
    }
    float pr[N][NT][4];
#pragma unroll
    for (int n = 0; n < N; ++n)
#pragma unroll
      for (int j = 0; j < NT; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) pr[n][j][e] = ex2_approx(x[n][j][e]);
        lrow[j][0] += pr[n][j][0] + pr[n][j][2];
        lrow[j][1] += pr[n][j][1] + pr[n][j][3];
      }

    // values: O^T += V_codes^T . (P * s_v) (codes as bare fields); bias term on CUDA cores
    uint32_t vrow[N][4];
#pragma unroll
    for (int n = 0; n < N; ++n) {
      vrow[n][0] = sb + OFF_V + (subs[n] * 16 + rV0) * 96;
      vrow[n][1] = sb + OFF_V + (subs[n] * 16 + rV1) * 96;
      vrow[n][2] = vrow[n][0] + 8 * 96;
      vrow[n][3] = vrow[n][1] + 8 * 96;
    }
#pragma unroll
    for (int gi = 0; gi < GPW; ++gi) {
      const int Gr = dg * GPW + gi;
      const uint32_t wofs = (6 * Gr + vword) * 4;
#pragma unroll
      for (int n = 0; n < N; ++n) {
        const float vs0 = pick_bf16(vsc0[n], Gr), vs1 = pick_bf16(vsc1[n], Gr);
        const float vb0 = fmaf(VCENTRE, vs0, pick_bf16(vbi0[n], Gr));
        const float vb1 = fmaf(VCENTRE, vs1, pick_bf16(vbi1[n], Gr));
        uint32_t bp[NT][2];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const float* p = pr[n][j];
          float q0 = p[0] * vs0, q1 = p[1] * vs0, q2 = p[2] * vs1, q3 = p[3] * vs1;
          if constexpr (FULL) {
            bacc[gi][j][0] = fmaf(p[0], vb0, fmaf(p[2], vb1, bacc[gi][j][0]));
            bacc[gi][j][1] = fmaf(p[1], vb0, fmaf(p[3], vb1, bacc[gi][j][1]));
          } else {  // masked tokens may hold stale (even NaN) scales: select, never multiply
            const bool* v = valid[n][j];
            q0 = v[0] ? q0 : 0.f;
            q1 = v[1] ? q1 : 0.f;
            q2 = v[2] ? q2 : 0.f;
            q3 = v[3] ? q3 : 0.f;
            bacc[gi][j][0] += (v[0] ? p[0] * vb0 : 0.f) + (v[2] ? p[2] * vb1 : 0.f);
            bacc[gi][j][1] += (v[1] ? p[1] * vb0 : 0.f) + (v[3] ? p[3] * vb1 : 0.f);
          }
          bp[j][0] = movmatrix_trans(pack_f16x2(q0, q1));
          bp[j][1] = movmatrix_trans(pack_f16x2(q2, q3));
          const uint32_t ones[4] = {kOnesF16x2, kOnesF16x2, kOnesF16x2, kOnesF16x2};
          mma_f16(wsum[gi][j], ones, bp[j][0], bp[j][1]);
        }
        uint32_t f[4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
          f[r] = __funnelshift_r(lds32(vrow[n][r] + wofs), lds32(vrow[n][r] + wofs + 4), vshift);
        uint32_t h01[8], h23[8];
        unpack_v3_pair(f[0], f[1], h01);
        unpack_v3_pair(f[2], f[3], h23);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t A[4] = {h01[2 * i], h01[2 * i + 1], h23[2 * i], h23[2 * i + 1]};
#pragma unroll
          for (int j = 0; j < NT; ++j) mma_f16(O[gi][i][j], A, bp[j][0], bp[j][1]);
        }
      }
    }
  };

  // ---- publish this range's segment of unit u (O in buf, per-row running max
  // in log2 units and sum in ml): a unit held by this range alone is
  // finalised; otherwise its partial goes to slot u + k_cta and is counted
  // for the combine.  Every write here follows griddepcontrol.wait.
  float2* mlr = reinterpret_cast<float2*>(smem + C::OFF_MLR);
  const float* dbuf = reinterpret_cast<const float*>(smem + C::OFF_DBUF);
  const float2* dml = reinterpret_cast<const float2*>(smem + C::OFF_DML);
  auto publish = [&](int u, const float* buf, const float2* ml) {
    const int ub = p.unit_base + u;
    if (p.prefix[u] >= g0 && p.prefix[u + 1] <= g1) {  // the whole unit is here: finalise
      for (int idx = ctid; idx < GT * 32; idx += NCT) {
        const int r = idx >> 5, l8 = idx & 31;
        if (((ub % p.nqt) * GT + r) / p.rep >= p.nq) continue;
        uint32_t mw[16];
        load_rot(p, l8, mw);
        const float4 o0 = reinterpret_cast<const float4*>(buf + r * kHeadDim + 8 * l8)[0];
        const float4 o1 = reinterpret_cast<const float4*>(buf + r * kHeadDim + 8 * l8)[1];
        const float acc[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
        store_out<GT>(p, ub, r, l8, acc, ml[r].y, mw);
      }
    } else {  // partial for the combine: slot u + k_cta
      const long long slot = static_cast<long long>(u) + k_cta;
      float4* po = reinterpret_cast<float4*>(p.part_o + slot * GT * kHeadDim);
      for (int idx = ctid; idx < GT * kHeadDim / 4; idx += NCT) po[idx] = reinterpret_cast<const float4*>(buf)[idx];
      for (int r = ctid; r < GT; r += NCT) reinterpret_cast<float2*>(p.part_ml)[slot * GT + r] = ml[r];
      named_bar(bar_all, NCT);  // every thread's partial stores precede the arrival
      if (ctid == 0) {
        __threadfence();
        atomicAdd(p.counters + u, 1u);
      }
    }
  };

  // ---- finish this range's segment of unit u: fold the value-bias sums into
  // O, merge the token streams (log-sum-exp) into obuf with each row's max and
  // sum in mlr, then publish it, or (defer: the first of several segments of
  // the range) keep it in shared memory until the range ends, so the range's
  // first griddepcontrol.wait comes at its end.
  auto end_unit = [&](int u, bool defer) {
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float l = lrow[j][e];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        lrow[j][e] = l;
#pragma unroll
        for (int gi = 0; gi < GPW; ++gi) {
          float bs = bacc[gi][j][e];
          bs += __shfl_xor_sync(0xffffffffu, bs, 4);
          bs += __shfl_xor_sync(0xffffffffu, bs, 8);
          bs += __shfl_xor_sync(0xffffffffu, bs, 16);
          bs = fmaf(-VCENTRE, wsum[gi][j][e], bs);
#pragma unroll
          for (int i = 0; i < 4; ++i) {  // undo the field positions of the value codes (exact powers of two)
            O[gi][i][j][e] = fmaf(O[gi][i][j][e], exp2i(24 - vpos(2 * i)), bs);
            O[gi][i][j][e + 2] = fmaf(O[gi][i][j][e + 2], exp2i(24 - vpos(2 * i + 1)), bs);
          }
        }
      }
    // merge the token streams in turn through obuf
    if (dg == 0 && g == 0)
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) mbuf[stream * GT + 8 * j + 2 * t + e] = msc[j][e];
    named_bar(bar_all, NCT);
    float a_row[NT][2];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int row = 8 * j + 2 * t + e;
        float M = mbuf[row];
#pragma unroll
        for (int s = 1; s < STREAMS; ++s) M = fmaxf(M, mbuf[s * GT + row]);
        a_row[j][e] = msc[j][e] == NEG_INF ? 0.f : ex2_approx(msc[j][e] - M);
        if (dg == 0 && g == 0) lbuf[stream * GT + row] = lrow[j][e] * a_row[j][e];
      }
    if (u == u0) {
      // the range's last unit: the ring is idle (every tile consumed), so each
      // stream writes its scaled O to a slot of its own there, in parallel, and
      // every thread then sums the streams of its elements in stream order
      // (the same sums, in the same order, as the turns below)
      static_assert(STREAMS * GT * kHeadDim * 4 <= NSTAGE * STAGE, "the ring holds every stream's O");
      float* slot = reinterpret_cast<float*>(smem) + stream * GT * kHeadDim;
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int row = 8 * j + 2 * t + e;
          const float a = a_row[j][e];
#pragma unroll
          for (int gi = 0; gi < GPW; ++gi) {
            float4* dst = reinterpret_cast<float4*>(slot + row * kHeadDim + 64 * (dg * GPW + gi) + 8 * g);
            dst[0] = make_float4(O[gi][0][j][e] * a, O[gi][0][j][e + 2] * a, O[gi][1][j][e] * a,
                                 O[gi][1][j][e + 2] * a);
            dst[1] = make_float4(O[gi][2][j][e] * a, O[gi][2][j][e + 2] * a, O[gi][3][j][e] * a,
                                 O[gi][3][j][e + 2] * a);
          }
        }
      named_bar(bar_all, NCT);
      const float4* slots = reinterpret_cast<const float4*>(smem);
      for (int idx = ctid; idx < GT * kHeadDim / 4; idx += NCT) {
        float4 acc = slots[idx];
#pragma unroll
        for (int st = 1; st < STREAMS; ++st) {
          const float4 v = slots[st * GT * kHeadDim / 4 + idx];
          acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        reinterpret_cast<float4*>(obuf)[idx] = acc;
      }
      named_bar(bar_all, NCT);
    } else {
#pragma unroll 1
      for (int turn = 0; turn < STREAMS; ++turn) {
        if (stream == turn) {
#pragma unroll
          for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int row = 8 * j + 2 * t + e;
              const float a = a_row[j][e];
#pragma unroll
              for (int gi = 0; gi < GPW; ++gi) {
                const int col = 64 * (dg * GPW + gi) + 8 * g;
                float4 v0 = make_float4(O[gi][0][j][e] * a, O[gi][0][j][e + 2] * a, O[gi][1][j][e] * a,
                                        O[gi][1][j][e + 2] * a);
                float4 v1 = make_float4(O[gi][2][j][e] * a, O[gi][2][j][e + 2] * a, O[gi][3][j][e] * a,
                                        O[gi][3][j][e + 2] * a);
                float4* acc = reinterpret_cast<float4*>(obuf + row * kHeadDim + col);
                if (turn > 0) {
                  const float4 p0 = acc[0], p1 = acc[1];
                  v0.x += p0.x; v0.y += p0.y; v0.z += p0.z; v0.w += p0.w;
                  v1.x += p1.x; v1.y += p1.y; v1.z += p1.z; v1.w += p1.w;
                }
                acc[0] = v0;
                acc[1] = v1;
              }
            }
        }
        named_bar(bar_all, NCT);
      }
    }
    // obuf holds the range's O for the unit; per row M = max and L = sum over the streams
    for (int r = ctid; r < GT; r += NCT) {
      float M = mbuf[r], L = lbuf[r];
#pragma unroll
      for (int s = 1; s < STREAMS; ++s) {
        M = fmaxf(M, mbuf[s * GT + r]);
        L += lbuf[s * GT + r];
      }
      mlr[r] = make_float2(M, L);
    }
    named_bar(bar_all, NCT);
    if constexpr (!MASKED) {
      if (defer) {
        float4* d4 = reinterpret_cast<float4*>(smem + C::OFF_DBUF);
        for (int idx = ctid; idx < GT * kHeadDim / 4; idx += NCT) d4[idx] = reinterpret_cast<const float4*>(obuf)[idx];
        for (int r = ctid; r < GT; r += NCT) reinterpret_cast<float2*>(smem + C::OFF_DML)[r] = mlr[r];
        named_bar(bar_all, NCT);  // obuf and mlr are free again
        return;
      }
    }
    // the previous grids' writes of the output, partials and counters are done
    // (the first wait of the range blocks, later ones return at once); without
    // the early release, the combine may launch now
    pdl_wait();
    pdl_launch_dependents();
    publish(u, obuf, mlr);
  };


  // ------------------------------------------------------------ fused append
  // This CTA holds the last tile of units u0 .. u1 - 1, and of u1 when its
  // range reaches u1's end; it encodes their new rows (a warp per token row,
  // its K and V), makes the stores visible to the tensor copies and tells the
  // producer.  One unit per (sequence, kv head) here (a single query tile).
  if (p.n_new > 0) {
    const int ulast = p.prefix[u1 + 1] <= g1 ? u1 : u1 - 1;
    const int rows = (ulast - u0 + 1) * p.n_new;
    if (rows > 0) {
      if (p.encode_wait) pdl_wait();
      float m[2][4][4];
      load_row_rotation(p.rot, lane, m);
      for (int item = cw; item < rows; item += CW) {
        const int ue = u0 + item / p.n_new, i = item % p.n_new;
        const int ug = p.unit_base + ue;
        const int bb = ug / p.kv_heads, hh = ug % p.kv_heads;
        const long long src = ((static_cast<long long>(bb) * p.kv_heads + hh) * p.n_new + i) * kHeadDim + lane * 8;
        const uint4 rk = __ldg(reinterpret_cast<const uint4*>(p.k_new + src));
        const uint4 rv = __ldg(reinterpret_cast<const uint4*>(p.v_new + src));
        const long long dst = (static_cast<long long>(bb) * p.kv_heads + hh) * p.cap + p.lens[bb] - p.n_new + i;
        encode_row<4>(rk, m, lane, dst, const_cast<uint32_t*>(p.k_codes), const_cast<uint16_t*>(p.k_scales),
                      const_cast<uint16_t*>(p.k_biases));
        encode_row<3>(rv, m, lane, dst, const_cast<uint32_t*>(p.v_codes), const_cast<uint16_t*>(p.v_scales),
                      const_cast<uint16_t*>(p.v_biases));
      }
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");  // generic stores before the async-proxy reads
    __syncwarp();
    if (lane == 0) mbar_arrive(encoded);
  }

  // ------------------------------------------------------------ main loop over this range's tiles
  // One pass per unit segment, last unit first (the producer's order: a unit's
  // last tiles, which may hold the previous call's fused rows, come at the
  // range's end), so the per-unit prologue and epilogue each have a single
  // call site outside the hot per-tile loop.
  long long k = 0;
  bool ok = true;
  int def_u = -1;  // the unit whose segment waits in shared memory for the range's end
  for (int u = u1; u >= u0; --u) {
    const bool defer = !MASKED && u == u1 && u1 > u0;
    begin_unit(u);
    const long long seg_end = p.prefix[u + 1] < g1 ? p.prefix[u + 1] : g1;
    const int tile0 = static_cast<int>(p.prefix[u]);
    for (long long gt = p.prefix[u] > g0 ? p.prefix[u] : g0; gt < seg_end; ++gt, ++k) {
      const int st = static_cast<int>(k % NSTAGE);
      // (test hook: a wait on the fused-append barrier, which no one arrives at
      // in a call without new rows, runs out like a stage that is never filled)
      if (!mbar_wait((p.inject & 2) ? encoded : &full[st], static_cast<uint32_t>(k / NSTAGE) & 1, p.spin_limit)) {
        atomicOr(p.status, 2u);
        ok = false;
        break;
      }
      const uint32_t sb = smem_u32(smem + st * STAGE);
      const uint32_t msk = smem_u32(smem + C::OFF_MSK + st * C::MSK_STAGE);
      const int tile_tok = static_cast<int>(gt - tile0) * TILE;
      // global sub-tile SUBS*k + sub belongs to stream (SUBS*k + sub) % STREAMS;
      // a stream takes its sub-tiles of the stage PAIR at a time
      const int first = static_cast<int>((stream - (SUBS * k) % STREAMS + STREAMS) % STREAMS);
      for (int sub = first; sub < SUBS; sub += PAIR * STREAMS) {
        const int subs[2] = {sub, sub + STREAMS};
        const int tb[2] = {tile_tok + sub * 16, tile_tok + (sub + STREAMS) * 16};
        if (tb[0] >= limit) break;
        if (PAIR == 2 && subs[1] < SUBS && tb[1] < limit) {
          if (tb[1] + 16 <= limit && tb[1] + 15 <= qmin)
            subtiles(std::integral_constant<int, 2>{}, std::true_type{}, subs, tb, sb, msk);
          else
            subtiles(std::integral_constant<int, 2>{}, std::false_type{}, subs, tb, sb, msk);
        } else {
          if (tb[0] + 16 <= limit && tb[0] + 15 <= qmin)
            subtiles(std::integral_constant<int, 1>{}, std::true_type{}, subs, tb, sb, msk);
          else
            subtiles(std::integral_constant<int, 1>{}, std::false_type{}, subs, tb, sb, msk);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    end_unit(u, defer);
    if (defer) def_u = u;
    if (!ok) break;
  }
  if (def_u >= 0) {
    pdl_wait();
    pdl_launch_dependents();
    publish(def_u, dbuf, dml);
  }
}


// ------------------------------------------------------------------ combine
// One small CTA (kCombineThreads threads of at most kCombineRegs registers:
// it fits beside an attention CTA on any SM) per unit of the launch; units
// held by a single range were finalised by it and are skipped.  The unit's
// rows are merged kCombineRows at a time: per pass, one thread bulk-copies
// those rows of up to p.combine_blocks segments' partials (O and the running
// max and sum) into shared memory, so a pass costs one round trip to L2, then
// every thread merges one (row, 8-dim chunk) item over the segments (online
// log-sum-exp) and, after the last segment, normalises, undoes the rotation
// and stores.
constexpr int kCombineRows = kCombineThreads / 32;
constexpr int kCombineBlockBytes = kCombineRows * kHeadDim * 4 + kCombineRows * 8;  // O rows + (max, sum)

template <int GT>
__device__ __forceinline__ void combine_unit(const Params& p, int u) {
  extern __shared__ __align__(128) uint8_t csm[];
  __shared__ int s_ready;
  __shared__ __align__(8) uint64_t cbar;
  int k_first, k_last;
  seg_range(p, u, k_first, k_last);
  if (k_first == k_last) return;  // finished by the CTA that held the whole unit
  const int nseg = k_last - k_first + 1;
  // Wait (bounded, in time) until every CTA holding tiles of the unit has
  // stored its partial, so units are merged while the attention grid still
  // runs; every attention CTA started before this grid was launched.
  // The count is compared signed and taken off with an atomic subtract, on
  // success and on a timeout alike: the arrivals still missing at a timeout
  // land before this grid completes (it completes after the attention grid),
  // so the counter is zero again before any later launch on this counter set
  // stores a partial.
  unsigned expect = 0;
  for (int k = k_first; k <= k_last; ++k) expect += p.cstart[k] < p.cstart[k + 1];
  if (threadIdx.x == 0) {
    const int want = static_cast<int>(expect) + ((p.inject & 1) ? 1 : 0);
    const unsigned long long limit = p.combine_wait_ns ? p.combine_wait_ns : kCombineWaitNs;
    const unsigned long long t0 = global_ns();
    int ready = 0;
    for (;;) {
      if (static_cast<int>(ld_acquire_gpu(p.counters + u)) >= want) { ready = 1; break; }
      if (global_ns() - t0 > limit) break;
      __nanosleep(256);
    }
    s_ready = ready;
    mbar_init(&cbar, 1);
    mbar_fence_init();
    // the partials (stored by other CTAs, acquired above) are read next by bulk copies
    asm volatile("fence.proxy.async.global;" ::: "memory");
  }
  __syncthreads();
  if (!s_ready) {
    if (threadIdx.x == 0) {
      atomicOr(p.status, 8u);
      atomicSub(p.counters + u, expect);
    }
    return;
  }
  const long long slot0 = static_cast<long long>(u) + k_first;
  const int ub = p.unit_base + u;
  const int nb = p.combine_blocks;
  uint32_t phase = 0;
  bool ok = true;
  for (int r0 = 0; r0 < GT && ok; r0 += kCombineRows) {
    const int r = r0 + (threadIdx.x >> 5), l8 = threadIdx.x & 31;
    float M = NEG_INF, L = 0.f;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int q0 = 0; q0 < nseg; q0 += nb) {
      const int qn = min(nb, nseg - q0);
      if (threadIdx.x == 0) {
        uint32_t bytes = 0;
        for (int j = 0; j < qn; ++j) bytes += p.cstart[k_first + q0 + j] < p.cstart[k_first + q0 + j + 1] ? kCombineBlockBytes : 0;
        mbar_arrive_expect_tx(&cbar, bytes);
        for (int j = 0; j < qn; ++j) {
          const int kk = k_first + q0 + j;
          if (p.cstart[kk] >= p.cstart[kk + 1]) continue;  // a range without tiles stored nothing
          const long long sl = slot0 + q0 + j;
          uint8_t* blk = csm + j * kCombineBlockBytes;
          bulk_g2s_plain(blk, p.part_o + (sl * GT + r0) * kHeadDim, kCombineRows * kHeadDim * 4, &cbar);
          bulk_g2s_plain(blk + kCombineRows * kHeadDim * 4, p.part_ml + (sl * GT + r0) * 2, kCombineRows * 8, &cbar);
        }
      }
      if (!__syncthreads_and(mbar_wait(&cbar, phase, p.spin_limit))) {  // one decision for all threads
        if (threadIdx.x == 0) atomicOr(p.status, 8u);
        ok = false;
        break;
      }
      phase ^= 1;
      for (int j = 0; j < qn; ++j) {  // online log-sum-exp over the round's segments
        const int kk = k_first + q0 + j;
        if (p.cstart[kk] >= p.cstart[kk + 1]) continue;
        const uint8_t* blk = csm + j * kCombineBlockBytes;
        const float2 ml = reinterpret_cast<const float2*>(blk + kCombineRows * kHeadDim * 4)[r - r0];
        if (ml.x == NEG_INF) continue;  // a segment with no visible key weighs 0
        const float4 oa = reinterpret_cast<const float4*>(blk)[((r - r0) * kHeadDim + 8 * l8) / 4];
        const float4 ob = reinterpret_cast<const float4*>(blk)[((r - r0) * kHeadDim + 8 * l8) / 4 + 1];
        const float Mn = fmaxf(M, ml.x);
        const float so = M == NEG_INF ? 0.f : ex2_approx(M - Mn), w = ex2_approx(ml.x - Mn);
        const float v[8] = {oa.x, oa.y, oa.z, oa.w, ob.x, ob.y, ob.z, ob.w};
#pragma unroll
        for (int d = 0; d < 8; ++d) acc[d] = fmaf(w, v[d], acc[d] * so);
        L = fmaf(w, ml.y, L * so);
        M = Mn;
      }
      __syncthreads();  // every read of the blocks precedes the next round's copies
    }
    if (ok && r < GT && ((ub % p.nqt) * GT + r) / p.rep < p.nq) {
      uint32_t mw[16];
      load_rot(p, l8, mw);
      store_out<GT>(p, ub, r, l8, acc, L, mw);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) atomicSub(p.counters + u, expect);  // back to zero for a later launch
}


template <int GT>
__global__ void __launch_bounds__(kCombineThreads, 65536 / (kCombineThreads * kCombineRegs))
    combine_kernel(const __grid_constant__ Params p) {
  pdl_launch_dependents();  // the next kernel may launch; it waits for this grid before reading
  const int u = blockIdx.x;
  if (u < p.num_units) combine_unit<GT>(p, u);
  // This grid may run ahead of the attention grid it depends on; it completes
  // only after that grid has completed, so work behind it in the stream (a copy
  // of the output) sees both grids' stores.
  pdl_wait();
}

// ------------------------------------------------------------------ host plan

constexpr int kMaxLaunches = 64;

struct Plan {
  int nt, gt, nqt, tile, launches, grid[kMaxLaunches];
  bool full[kMaxLaunches];  // one CTA on every SM (the early release may be used)
  size_t units, slots, head_bytes, bytes;
};

// workspace: [status word, padded to 256 B][per-unit partial counters: two
// sets of UNIT_CAP x u32][partial O: slots x GT x 256 f32][partial (max, sum):
// slots x GT x 2 f32].  The head (status word and counters) starts zeroed; the status
// word accumulates failure bits until iq_read_status reads it, and the combine
// returns each counter to zero (iq_read_status re-zeroes the whole head after a
// failure).  Partials are written before they are read.
constexpr size_t kStatusBytes = 256;
constexpr size_t kHeadBytes = kStatusBytes + 2 * UNIT_CAP * sizeof(unsigned);  // status word + unit counters
static_assert(kHeadBytes == IQ_WORKSPACE_HEAD_BYTES, "workspace head size in iqkv.h");

template <int NT, int DS, int STREAMS, int NSTAGE, int MINB, int TILE_, int PAIR, int HALVES>
int blocks_per_sm() {
  static int cache[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (cache[dev] == 0) {
    using C = Cfg<NT, DS, STREAMS, NSTAGE, MINB, TILE_, PAIR, HALVES>;
    int n = 0;
    cudaFuncSetAttribute(attend_kernel<NT, DS, STREAMS, NSTAGE, MINB, TILE_, PAIR, HALVES, false>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    cudaFuncSetAttribute(attend_kernel<NT, DS, STREAMS, NSTAGE, MINB, TILE_, PAIR, HALVES, true>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_MASK);
    // CTAs of different kernels share an SM only under one L1 / shared-memory
    // split: the combine asks for the attention kernels' (all shared), so its
    // small CTAs can sit beside theirs
    cudaFuncSetAttribute(attend_kernel<NT, DS, STREAMS, NSTAGE, MINB, TILE_, PAIR, HALVES, false>,
                         cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    cudaFuncSetAttribute(attend_kernel<NT, DS, STREAMS, NSTAGE, MINB, TILE_, PAIR, HALVES, true>,
                         cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    cudaFuncSetAttribute(combine_kernel<C::GT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                         cudaSharedmemCarveoutMaxShared);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attend_kernel<NT, DS, STREAMS, NSTAGE, MINB, TILE_, PAIR, HALVES, false>,
                                                      C::THREADS, C::SMEM) !=
            cudaSuccess ||
        n <= 0)
      n = 1;
    cache[dev] = n;
  }
  return cache[dev];
}

// <query n-tiles, warps per token stream, token streams, ring stages, CTAs per SM, tile tokens>
// Decode (<= 8 query rows per kv head): one warp owns all four groups; four
// token streams per CTA, two CTAs per SM, two 128-token stages (measured best:
// more streams per CTA make the warps wait on one shared ring; 64-token stages
// cost more handshakes per byte; a consumer warp that issues the refills
// itself instead of a producer warp was slower).  Verify / prefill (more
// rows): 16-row query tiles, two warps per token stream (two 64-dim groups
// each, partial scores summed through shared memory), two streams per CTA, two
// CTAs per SM, two 128-token stages (measured best among 8/16/32-row tiles and
// one/two/four warps per stream).
#ifndef IQ_DECODE_STREAMS
#define IQ_DECODE_STREAMS 4
#endif
#ifndef IQ_DECODE_STAGES
#define IQ_DECODE_STAGES 2
#endif
#ifndef IQ_DECODE_TILE
#define IQ_DECODE_TILE 128
#endif
#ifndef IQ_DECODE_MINB
#define IQ_DECODE_MINB 1
#endif
#ifndef IQ_DECODE_HALVES
#define IQ_DECODE_HALVES 2
#endif
#ifndef IQ_DECODE_PAIR
#define IQ_DECODE_PAIR 2
#endif
#ifndef IQ_DECODE_BOUNDARY
#define IQ_DECODE_BOUNDARY 4
#endif
#define IQ_DECODE_CFG \
  1, 1, IQ_DECODE_STREAMS, IQ_DECODE_STAGES, IQ_DECODE_MINB, IQ_DECODE_TILE, IQ_DECODE_PAIR, IQ_DECODE_HALVES
#ifndef IQ_MULTI_NT
#define IQ_MULTI_NT 2
#endif
#ifndef IQ_MULTI_DS
#define IQ_MULTI_DS 2
#endif
#ifndef IQ_MULTI_STREAMS
#define IQ_MULTI_STREAMS 4
#endif
#ifndef IQ_MULTI_STAGES
#define IQ_MULTI_STAGES 4
#endif
#ifndef IQ_MULTI_MINB
#define IQ_MULTI_MINB 1
#endif
#ifndef IQ_MULTI_TILE
#define IQ_MULTI_TILE 128
#endif
#ifndef IQ_MULTI_PAIR
#define IQ_MULTI_PAIR 2
#endif
#ifndef IQ_MULTI_BOUNDARY
#define IQ_MULTI_BOUNDARY 3
#endif
#define IQ_MULTI_CFG \
  IQ_MULTI_NT, IQ_MULTI_DS, IQ_MULTI_STREAMS, IQ_MULTI_STAGES, IQ_MULTI_MINB, IQ_MULTI_TILE, IQ_MULTI_PAIR, 1

// Tiles of every unit, in unit order: unit u = (b, kv head, query tile).
void unit_tiles(const iq_cache* c, int rep, int nq, int causal, int gt, int nqt, int tile, int* tiles) {
  for (int b = 0; b < c->batch; ++b)
    for (int h = 0; h < c->kv_heads; ++h)
      for (int qt = 0; qt < nqt; ++qt) {
        const int T = c->lens[b];
        int limit = T;
        if (causal) limit = T - nq + std::min(qt * gt + gt - 1, rep * nq - 1) / rep + 1;
        tiles[(b * c->kv_heads + h) * nqt + qt] = (limit + tile - 1) / tile;
      }
}

// tiles == nullptr: size an upper bound (every unit as long as the longest sequence)
int make_plan(const iq_cache* c, int q_heads, int nq, int causal, Plan* pl, const int* tiles) {
  const int rep = q_heads / c->kv_heads;
  const int rows = rep * nq;
  pl->nt = rows <= 8 ? 1 : IQ_MULTI_NT;
  pl->gt = 8 * pl->nt;
  pl->nqt = (rows + pl->gt - 1) / pl->gt;
  pl->tile = pl->nt == 1 ? Cfg<IQ_DECODE_CFG>::TILE : Cfg<IQ_MULTI_CFG>::TILE;
  pl->units = static_cast<size_t>(c->batch) * c->kv_heads * pl->nqt;
  pl->launches = static_cast<int>((pl->units + UNIT_CAP - 1) / UNIT_CAP);
  if (pl->launches > kMaxLaunches) return fail(IQ_ERR_UNSUPPORTED, "too many query tiles for one call");
  // virtual CTAs (tile ranges): CTAs per SM x the halves of a CTA
  const int halves = pl->nt == 1 ? IQ_DECODE_HALVES : 1;
  const int bps = pl->nt == 1 ? blocks_per_sm<IQ_DECODE_CFG>() : blocks_per_sm<IQ_MULTI_CFG>();
  const long long slots_hw = static_cast<long long>(num_sms()) * bps * halves;
  int max_tiles = 0;
  for (int b = 0; b < c->batch; ++b) max_tiles = std::max(max_tiles, (static_cast<int>(c->lens[b]) + pl->tile - 1) / pl->tile);
  pl->slots = 0;
  for (int l = 0; l < pl->launches; ++l) {
    const size_t u0 = static_cast<size_t>(l) * UNIT_CAP;
    const size_t nu = std::min(pl->units - u0, static_cast<size_t>(UNIT_CAP));
    long long W = 0;
    if (tiles) {
      for (size_t u = 0; u < nu; ++u) W += tiles[u0 + u];
    } else {
      W = static_cast<long long>(nu) * max_tiles;
    }
    long long G = std::min(std::min(slots_hw, static_cast<long long>(GRID_CAP)),
                           std::max(1LL, W / MIN_TILES_PER_CTA));
    G = std::max<long long>(halves, G / halves * halves);  // whole CTAs
    pl->grid[l] = static_cast<int>(G);
    pl->full[l] = bps == 1 && G == slots_hw;
    pl->slots = std::max(pl->slots, nu + static_cast<size_t>(G));
  }
  if (!tiles)  // independent of the tile counts, so it bounds every later plan
    pl->slots = std::min(pl->units, static_cast<size_t>(UNIT_CAP)) +
                static_cast<size_t>(std::min(slots_hw, static_cast<long long>(GRID_CAP)));
  pl->head_bytes = kHeadBytes;
  pl->bytes = pl->head_bytes + pl->slots * pl->gt * (kHeadDim + 2) * sizeof(float);
  return IQ_OK;
}

// Tile ranges of the G CTAs of a launch.  Starting a unit costs a CTA about
// `boundary` tiles' worth of time (finishing the previous unit's segment and
// rotating the new queries), so the ranges split evenly a virtual line on
// which every unit after the first is preceded by that many virtual tiles: a
// CTA that crosses unit starts streams correspondingly fewer real tiles.
void split_ranges(const int* prefix, int nu, int G, int boundary, int* cstart) {
  const long long W = prefix[nu];
  const long long V = W + static_cast<long long>(boundary) * (nu - 1);
  int u = 0;
  cstart[0] = 0;
  for (int k = 1; k < G; ++k) {
    const long long v = V * k / G;
    // unit u's real tiles sit at virtual [prefix[u] + boundary*u, prefix[u+1] + boundary*u)
    while (u < nu - 1 && v >= prefix[u + 1] + static_cast<long long>(boundary) * u) ++u;
    const long long vs = prefix[u] + static_cast<long long>(boundary) * u;
    cstart[k] = static_cast<int>(v < vs ? prefix[u] : std::min<long long>(v - static_cast<long long>(boundary) * u, prefix[u + 1]));
  }
  cstart[G] = static_cast<int>(W);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

int validate(const iq_cache* c, const void* q, int q_heads, int nq, int causal, const void* rot, const void* out) {
  int st = iq_cache_check(c);
  if (st != IQ_OK) return st;
  if (!q || !rot || !out) return fail(IQ_ERR_INVALID_ARG, "null q/rotation/out");
  if (reinterpret_cast<uintptr_t>(q) % 16 || reinterpret_cast<uintptr_t>(out) % 16 ||
      reinterpret_cast<uintptr_t>(rot) % 16)
    return fail(IQ_ERR_INVALID_ARG, "q/out/rotation not 16-byte aligned");
  if (causal != 0 && causal != 1) return fail(IQ_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (nq < 1) return fail(IQ_ERR_INVALID_ARG, "n_queries must be >= 1");
  if (q_heads < 1 || q_heads % c->kv_heads) return fail(IQ_ERR_INVALID_ARG, "q_heads must be a multiple of kv_heads");
  const int rep = q_heads / c->kv_heads;
  if (rep > 8 || 8 % rep) return fail(IQ_ERR_UNSUPPORTED, "query heads per kv head must divide 8");
  for (int b = 0; b < c->batch; ++b) {
    if (c->lens[b] < 1) return fail(IQ_ERR_INVALID_ARG, "attention over an empty sequence");
    if (causal && c->lens[b] < nq) return fail(IQ_ERR_INVALID_ARG, "causal: lens[b] < n_queries");
  }
  if (static_cast<long long>(c->batch) * c->kv_heads * c->capacity >= (1LL << 31))
    return fail(IQ_ERR_UNSUPPORTED, "cache rows exceed 2^31");
  return IQ_OK;
}

// Partial blocks the combine can stage while its CTA still fits in the shared
// memory an attention CTA of this configuration leaves on an SM (at least one:
// beside the masked verify kernel it then waits for an SM of its own).
template <int NT, int DS, int STREAMS, int NSTAGE, int MINB, int TILE_, int PAIR, int HALVES>
int combine_blocks_for(bool masked) {
  using C = Cfg<NT, DS, STREAMS, NSTAGE, MINB, TILE_, PAIR, HALVES>;
  static int per_sm = -1, reserved = 0;
  if (per_sm < 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess) per_sm = 0;
    if (cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess) reserved = 1024;
  }
  const long long left = static_cast<long long>(per_sm) - (masked ? C::SMEM_MASK : C::SMEM) - 2LL * reserved - 128;
  return static_cast<int>(std::max(1LL, std::min(8LL, left / kCombineBlockBytes)));
}

template <int NT, int DS, int STREAMS, int NSTAGE, int MINB, int TILE_, int PAIR, int HALVES>
int launch_attend(const Params& prm, const CUtensorMap& map, int grid, cudaStream_t s) {
  using C = Cfg<NT, DS, STREAMS, NSTAGE, MINB, TILE_, PAIR, HALVES>;
  blocks_per_sm<NT, DS, STREAMS, NSTAGE, MINB, TILE_, PAIR, HALVES>();  // sets the shared-memory attribute once
  // The warpgroups move registers between them (setmaxnreg); that split adds
  // up to the block's launch allocation only at the register count it was
  // designed for, so any other build of the kernel is refused, never launched.
  const bool masked = prm.mask_kind >= 2;
  static int launch_regs[2] = {-1, -1};
  if (launch_regs[masked] < 0) {
    cudaFuncAttributes fa;
    IQ_CUDA(cudaFuncGetAttributes(&fa, masked ? attend_kernel<NT, DS, STREAMS, NSTAGE, MINB, TILE_, PAIR, HALVES, true>
                                              : attend_kernel<NT, DS, STREAMS, NSTAGE, MINB, TILE_, PAIR, HALVES, false>));
    launch_regs[masked] = fa.numRegs;
  }
  if (launch_regs[masked] != C::LAUNCH_REGS)
    return fail(IQ_ERR_UNSUPPORTED, "attention kernel built with an unexpected register count");
  // Both kernels are programmatic dependents of their predecessor in the
  // stream: their launch overlaps its tail, and each waits for it
  // (griddepcontrol.wait) before reading anything.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid / HALVES));  // `grid` counts tile ranges: HALVES per CTA
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = prm.mask_kind >= 2 ? C::SMEM_MASK : C::SMEM;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (masked)
    IQ_CUDA(cudaLaunchKernelEx(&cfg, attend_kernel<NT, DS, STREAMS, NSTAGE, MINB, TILE_, PAIR, HALVES, true>, prm, map));
  else
    IQ_CUDA(cudaLaunchKernelEx(&cfg, attend_kernel<NT, DS, STREAMS, NSTAGE, MINB, TILE_, PAIR, HALVES, false>, prm, map));
  // the split combine, after the attention grid
  cfg.gridDim = dim3(static_cast<unsigned>(prm.num_units));
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(prm.combine_blocks) * kCombineBlockBytes;
  IQ_CUDA(cudaLaunchKernelEx(&cfg, combine_kernel<C::GT>, prm));
  return IQ_OK;
}

}  // namespace attn
}  // namespace iq

using namespace iq;
using namespace iq::attn;

extern "C" {

int iq_attend_workspace(const iq_cache* c, int q_heads, int n_queries, size_t* bytes) {
  clear_error();
  int st = iq_cache_check(c);
  if (st != IQ_OK) return st;
  if (!bytes) return fail(IQ_ERR_INVALID_ARG, "null bytes");
  if (n_queries < 1 || q_heads < 1 || q_heads % c->kv_heads)
    return fail(IQ_ERR_INVALID_ARG, "bad head or query count");
  if (!tuned_format(c)) return attend_any_workspace(c, q_heads, n_queries, bytes);
  Plan pl;
  st = make_plan(c, q_heads, n_queries, 0, &pl, nullptr);
  if (st != IQ_OK) return st;
  *bytes = pl.bytes;
  return IQ_OK;
}

}  // extern "C"

namespace iq {
namespace attn {

// Rows [0, hi[b]) that the latest attention launched on a cache (keyed by its
// key-code buffer) reads.  An attention grid may still run while the next call's
// grid starts (see attend_kernel); a fused append may write its new rows at
// once only when none of them lies below that mark, i.e. when no trim since the
// latest attention moved the append point back into rows it reads.  No record
// (first call, or the table was reset) counts as a trim.
class ReadMarks {
 public:
  void record(const iq_cache* c) {
    std::lock_guard<std::mutex> lk(mu_);
    if (marks_.size() >= 256) marks_.clear();  // bounded; a lost record only makes an append wait
    auto& v = marks_[c->k_codes];
    v.assign(c->lens, c->lens + c->batch);
  }
  // true when rows [lens[b], ...) of every sequence are at or above the mark
  bool append_clear(const iq_cache* c) {
    std::lock_guard<std::mutex> lk(mu_);
    auto it = marks_.find(c->k_codes);
    if (it == marks_.end() || static_cast<int>(it->second.size()) != c->batch) return false;
    for (int b = 0; b < c->batch; ++b)
      if (c->lens[b] < it->second[b]) return false;
    return true;
  }

 private:
  std::mutex mu_;
  std::unordered_map<const void*, std::vector<int>> marks_;
};
ReadMarks& read_marks() {
  static ReadMarks m;
  return m;
}

// The unit-counter set of the next split-KV launch on a workspace: launches on
// one workspace alternate between the two sets.  next() returns false when the
// previous launch on it is not on record (first use; the table is bounded);
// such a launch releases its combine late, the order that needs no second set.
class CounterSets {
 public:
  bool next(const void* ws, int* set) {
    std::lock_guard<std::mutex> lk(mu_);
    auto it = sets_.find(ws);
    if (it == sets_.end()) {
      if (sets_.size() >= 4096) sets_.clear();
      sets_[ws] = 0;
      *set = 0;
      return false;
    }
    it->second ^= 1;
    *set = it->second;
    return true;
  }

 private:
  std::mutex mu_;
  std::unordered_map<const void*, int> sets_;
};
CounterSets& counter_sets() {
  static CounterSets c;
  return c;
}

// Attention over the cache; with n_new > 0 the last n_new rows of every
// sequence (already counted in c->lens) are first encoded from k_new / v_new
// inside the same kernel (see the fused append in attend_kernel); encode_wait
// makes those writes wait for the previous grids.
int attend_impl(const iq_cache* c, const void* q_in, int q_heads, int n_queries, float scale, int causal,
                const void* rot_in, void* out, int out_f32, void* workspace, size_t workspace_bytes,
                iq_stream_t stream, const void* k_new_in, const void* v_new_in, int n_new, int mask_kind = 0,
                const void* mask = nullptr, long long mask_stride = 0, int encode_wait = 1) {
  int st = validate(c, q_in, q_heads, n_queries, causal, rot_in, out);
  if (st != IQ_OK) return st;
  if (!tuned_format(c)) {
    if (n_new > 0) return fail(IQ_ERR_UNSUPPORTED, "fused append for this cache format");
    return attend_any(c, q_in, q_heads, n_queries, scale, causal, rot_in, out, out_f32, workspace, workspace_bytes,
                      stream, mask_kind, mask, mask_stride);
  }
  // the tuned format holds bfloat16 data
  const uint16_t* q = static_cast<const uint16_t*>(q_in);
  const uint16_t* rot_bf16 = static_cast<const uint16_t*>(rot_in);
  const uint16_t* k_new = static_cast<const uint16_t*>(k_new_in);
  const uint16_t* v_new = static_cast<const uint16_t*>(v_new_in);
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 256)
    return fail(IQ_ERR_WORKSPACE, "workspace missing or not 256-byte aligned");
  Plan bound;  // what iq_attend_workspace promised: an upper bound of this call's needs
  st = make_plan(c, q_heads, n_queries, causal, &bound, nullptr);
  if (st != IQ_OK) return st;
  if (workspace_bytes < bound.bytes) return fail(IQ_ERR_WORKSPACE, "workspace smaller than iq_attend_workspace()");
  if (prefill_shape(c, q_heads, n_queries, mask_kind)) {  // n_new > 0: the caller checked prefill_fusable
    st = prefill_attend(c, q, q_heads, n_queries, scale, causal, rot_bf16, out, out_f32,
                        reinterpret_cast<unsigned*>(workspace), stream, k_new, v_new, n_new,
                        reinterpret_cast<unsigned*>(static_cast<uint8_t*>(workspace) + kStatusBytes));
    if (st == IQ_OK) read_marks().record(c);
    return st;
  }
  static thread_local std::vector<int> tiles;
  tiles.assign(bound.units, 0);
  unit_tiles(c, q_heads / c->kv_heads, n_queries, causal, bound.gt, bound.nqt, bound.tile, tiles.data());
  Plan pl;
  st = make_plan(c, q_heads, n_queries, causal, &pl, tiles.data());
  if (st != IQ_OK) return st;
  auto encode = encode_fn();
  if (!encode) return fail(IQ_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");

  CUtensorMap map;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kKWords),
                              static_cast<cuuint64_t>(c->batch) * c->kv_heads * c->capacity};
  const cuuint64_t strides[1] = {kKWords * 4};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kKWords), static_cast<cuuint32_t>(pl.tile)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult cr = encode(&map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, c->k_codes, dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return fail(IQ_ERR_CUDA, "cuTensorMapEncodeTiled failed for the key codes");

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  unsigned* status = reinterpret_cast<unsigned*>(ws);
  unsigned* counters = reinterpret_cast<unsigned*>(ws + kStatusBytes);
  float* part_o = reinterpret_cast<float*>(ws + bound.head_bytes);
  float* part_ml = part_o + bound.slots * pl.gt * kHeadDim;

  static thread_local Params prm;  // ~5 KB: kept off the stack
  std::memset(&prm, 0, sizeof(prm));
  prm.k_codes = c->k_codes;
  prm.k_scales = static_cast<const uint16_t*>(c->k_scales);
  prm.k_biases = static_cast<const uint16_t*>(c->k_biases);
  prm.v_codes = c->v_codes;
  prm.v_scales = static_cast<const uint16_t*>(c->v_scales);
  prm.v_biases = static_cast<const uint16_t*>(c->v_biases);
  prm.q = q;
  prm.rot = rot_bf16;
  prm.part_o = part_o;
  prm.part_ml = part_ml;
  prm.status = status;
  prm.counters = counters;
  prm.k_new = k_new;
  prm.v_new = v_new;
  prm.n_new = n_new;
  prm.encode_wait = encode_wait ? 1 : 0;
  prm.spin_limit = t_inject.spin_limit ? t_inject.spin_limit : kSpinLimit;
  prm.combine_wait_ns = t_inject.wait_ns;
  prm.inject = t_inject.flags;
  t_inject = DebugInject{};  // one call only
  prm.mask_kind = mask_kind;
  prm.mask = mask;
  prm.mask_stride = mask_stride;
  prm.out = out;
  prm.out_f32 = out_f32 ? 1 : 0;
  prm.batch = c->batch;
  prm.kv_heads = c->kv_heads;
  prm.rep = q_heads / c->kv_heads;
  prm.nq = n_queries;
  prm.cap = c->capacity;
  prm.nqt = pl.nqt;
  prm.causal = causal;
  prm.scale = scale;
  for (int b = 0; b < c->batch; ++b) prm.lens[b] = c->lens[b];
  // launches run in stream order and reuse the partial slots
  for (int l = 0; l < pl.launches; ++l) {
    const int u0 = l * UNIT_CAP;
    const int nu = static_cast<int>(std::min(pl.units - u0, static_cast<size_t>(UNIT_CAP)));
    prm.unit_base = u0;
    prm.num_units = nu;
    prm.grid = pl.grid[l];
    prm.prefix[0] = 0;
    for (int u = 0; u < nu; ++u) prm.prefix[u + 1] = prm.prefix[u] + tiles[u0 + u];
    split_ranges(prm.prefix, nu, prm.grid, pl.nt == 1 ? IQ_DECODE_BOUNDARY : IQ_MULTI_BOUNDARY, prm.cstart);
    int set = 0;
    const bool known = counter_sets().next(workspace, &set);
    prm.counters = counters + static_cast<size_t>(set) * UNIT_CAP;
    prm.early = known && pl.full[l] ? 1 : 0;
    prm.combine_blocks = pl.nt == 1 ? combine_blocks_for<IQ_DECODE_CFG>(mask_kind >= 2)
                                    : combine_blocks_for<IQ_MULTI_CFG>(mask_kind >= 2);
    st = pl.nt == 1 ? launch_attend<IQ_DECODE_CFG>(prm, map, prm.grid, s)
                    : launch_attend<IQ_MULTI_CFG>(prm, map, prm.grid, s);
    if (st != IQ_OK) return st;
  }
  read_marks().record(c);
  return IQ_OK;
}

}  // namespace attn
}  // namespace iq

extern "C" {

int iq_attend(const iq_cache* c, const void* q, int q_heads, int n_queries, float scale, int causal,
              const void* rot, void* out, int out_f32, void* workspace, size_t workspace_bytes,
              iq_stream_t stream) {
  clear_error();
  return attend_impl(c, q, q_heads, n_queries, scale, causal, rot, out, out_f32, workspace, workspace_bytes,
                     stream, nullptr, nullptr, 0);
}

int iq_cache_append_attend(iq_cache* c, const void* keys, const void* values, int n, const void* q,
                           int q_heads, int n_queries, float scale, int causal, const void* rot,
                           void* out, int out_f32, void* workspace, size_t workspace_bytes, iq_stream_t stream) {
  clear_error();
  int st = iq_cache_check(c);
  if (st != IQ_OK) return st;
  if (n < 1) return fail(IQ_ERR_INVALID_ARG, "append_attend needs n >= 1 new tokens");
  if (!keys || !values || !rot) return fail(IQ_ERR_INVALID_ARG, "null keys/values/rotation");
  if (reinterpret_cast<uintptr_t>(keys) % 16 || reinterpret_cast<uintptr_t>(values) % 16)
    return fail(IQ_ERR_INVALID_ARG, "keys/values not 16-byte aligned");
  for (int b = 0; b < c->batch; ++b)
    if (static_cast<long long>(c->lens[b]) + n > c->capacity)
      return fail(IQ_ERR_CAPACITY, "append past capacity (grow the cache first)");
  // One kernel when every (sequence, kv head) is one query tile and the new
  // rows of each sequence sit in one key tile (the split-KV kernel encodes
  // them), or when the call takes the tensor-memory prefill kernel (its CTAs
  // encode the new rows' key tiles, each tile once, before streaming them);
  // otherwise the append, then the attention.
  const int tile = Cfg<IQ_DECODE_CFG>::TILE;
  const bool shape_ok = tuned_format(c) && q_heads >= c->kv_heads && q_heads % c->kv_heads == 0;
  bool fused = shape_ok && static_cast<long long>(q_heads / c->kv_heads) * n_queries <= 8;
  for (int b = 0; b < c->batch && fused; ++b)
    fused = c->lens[b] / tile == (c->lens[b] + n - 1) / tile;
  const long long pflags = shape_ok && prefill_shape(c, q_heads, n_queries, causal ? 1 : 0) ? prefill_fuse_flags(c, n) : 0;
  const bool fused_prefill = pflags > 0 && kStatusBytes + pflags * sizeof(unsigned) <= kHeadBytes;
  if (!fused && !fused_prefill) {
    st = iq_cache_append(c, keys, values, n, rot, stream);
    if (st != IQ_OK) return st;
    return iq_attend(c, q, q_heads, n_queries, scale, causal, rot, out, out_f32, workspace, workspace_bytes,
                     stream);
  }
  static_assert(Cfg<IQ_DECODE_CFG>::TILE <= kFreshRows, "a fused append writes at most kFreshRows rows");
  // (the prefill kernel waits for the previous grids before it stores)
  const int encode_wait = fused_prefill || read_marks().append_clear(c) ? 0 : 1;
  for (int b = 0; b < c->batch; ++b) c->lens[b] += n;
  st = attend_impl(c, q, q_heads, n_queries, scale, causal, rot, out, out_f32, workspace, workspace_bytes,
                   stream, keys, values, n, 0, nullptr, 0, encode_wait);
  if (st != IQ_OK)
    for (int b = 0; b < c->batch; ++b) c->lens[b] -= n;  // nothing was launched
  return st;
}

int iq_attend_mask(const iq_cache* c, const void* q, int q_heads, int n_queries, float scale, int mask_kind,
                   const void* mask, long long mask_stride, const void* rot, void* out, int out_f32,
                   void* workspace, size_t workspace_bytes, iq_stream_t stream) {
  clear_error();
  if (mask_kind == IQ_MASK_NONE || mask_kind == IQ_MASK_CAUSAL)
    return attend_impl(c, q, q_heads, n_queries, scale, mask_kind, rot, out, out_f32, workspace,
                       workspace_bytes, stream, nullptr, nullptr, 0);
  if (mask_kind != IQ_MASK_ADD_F32 && mask_kind != IQ_MASK_BOOL_U8)
    return fail(IQ_ERR_INVALID_ARG, "unknown mask kind");
  int st = iq_cache_check(c);
  if (st != IQ_OK) return st;
  if (!mask) return fail(IQ_ERR_INVALID_ARG, "null mask");
  if (mask_kind == IQ_MASK_ADD_F32 && reinterpret_cast<uintptr_t>(mask) % 4)
    return fail(IQ_ERR_INVALID_ARG, "float mask not 4-byte aligned");
  if (reinterpret_cast<uintptr_t>(mask) % 16 || mask_stride % 128)
    return fail(IQ_ERR_INVALID_ARG, "mask not 16-byte aligned or its row stride not a multiple of 128");
  for (int b = 0; b < c->batch; ++b)
    if (mask_stride < c->lens[b]) return fail(IQ_ERR_INVALID_ARG, "mask row shorter than a sequence");
  return attend_impl(c, q, q_heads, n_queries, scale, 0, rot, out, out_f32, workspace, workspace_bytes,
                     stream, nullptr, nullptr, 0, mask_kind, mask, mask_stride);
}

int iq_debug_inject(int flags, unsigned spin_limit, unsigned long long combine_wait_ns) {
  clear_error();
  if (flags & ~(IQ_INJECT_COMBINE_WAIT | IQ_INJECT_STAGE_NEVER_FILLED))
    return fail(IQ_ERR_INVALID_ARG, "unknown injection flag");
  t_inject.flags = flags;
  t_inject.spin_limit = spin_limit;
  t_inject.wait_ns = combine_wait_ns;
  return IQ_OK;
}

int iq_read_status(void* workspace, iq_stream_t stream, int* device_status) {
  clear_error();
  if (!workspace || !device_status) return fail(IQ_ERR_INVALID_ARG, "null pointer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned v = 0;
  IQ_CUDA(cudaStreamSynchronize(s));
  IQ_CUDA(cudaMemcpy(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost));
  // after a failure the unit counters may be stale too: clear the whole head
  IQ_CUDA(cudaMemset(workspace, 0, v ? kHeadBytes : sizeof(unsigned)));
  *device_status = static_cast<int>(v);
  return v ? fail(IQ_ERR_DEVICE, "a kernel reported a failure (status bits set)") : IQ_OK;
}

}  // extern "C"
