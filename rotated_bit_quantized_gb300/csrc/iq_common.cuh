// Shared device helpers of libiqkv (sm_103a): status plumbing, mbarrier /
// bulk-copy / tensor-copy wrappers, warp-level MMA and bit tricks.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "../../include/iqkv.h"

namespace iq {

// ------------------------------------------------------------------ host side

// Records a one-line message for iq_last_error() and returns `code`.
int fail(int code, const std::string& msg);
int cuda_fail(cudaError_t e, const char* what);
void clear_error();

#define IQ_CUDA(call)                                   \
  do {                                                  \
    cudaError_t e_ = (call);                            \
    if (e_ != cudaSuccess) return iq::cuda_fail(e_, #call); \
  } while (0)

int num_sms();  // multiprocessor count of the current device (cached per device)

// Cache formats (iq_generic.cu): the tuned one (k 4 bits, v 3 bits, 64-dim
// groups, bfloat16) runs the tuned kernels, every other supported one (any
// float32 cache included) the generic path.
bool tuned_format(const iq_cache* c);
bool format_supported(int head_dim, int group_size, int k_bits, int v_bits);
int append_any(iq_cache* c, const void* keys, const void* values, int n, const void* rot, iq_stream_t stream);
int attend_any_workspace(const iq_cache* c, int q_heads, int n_queries, size_t* bytes);
// Prefill shapes (iq_prefill.cu): many query rows per kv head, tuned format,
// no explicit mask: the tensor-memory kernel.
bool prefill_shape(const iq_cache* c, int q_heads, int n_queries, int mask_kind);
int prefill_attend(const iq_cache* c, const uint16_t* q, int q_heads, int n_queries, float scale, int causal,
                   const uint16_t* rot, void* out, int out_f32, unsigned* status, iq_stream_t stream,
                   const uint16_t* k_new = nullptr, const uint16_t* v_new = nullptr, int n_new = 0,
                   unsigned* flags = nullptr);
// Counter words the fused prefill append needs in the workspace's unit-counter
// area (two, plus one per sequence and kv head).
long long prefill_fuse_flags(const iq_cache* c, int n_new);
int attend_any(const iq_cache* c, const void* q, int q_heads, int n_queries, float scale, int causal,
               const void* rot, void* out, int out_f32, void* workspace, size_t workspace_bytes,
               iq_stream_t stream, int mask_kind, const void* mask, long long mask_stride);

// ------------------------------------------------------------------ device side

constexpr int kHeadDim = 256;
constexpr int kGroup = 64;
constexpr int kKWords = 32;   // 256 dims * 4 bits / 32
constexpr int kVWords = 24;   // 256 dims * 3 bits / 32
constexpr int kGroups = 4;    // 256 / 64
constexpr uint32_t kSpinLimit = 1u << 17;  // bounded waits (seconds at most), then report

__device__ __forceinline__ float bf16_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// Round-to-nearest-even float32 -> bfloat16 bits (NaN kept quiet).
__device__ __forceinline__ uint32_t f32_to_bf16_bits(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (u >> 16) | 0x40u;
  return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

__device__ __forceinline__ float round_bf16(float x) { return bf16_to_f32(f32_to_bf16_bits(x)); }

// The same rounding by the conversion instruction (finite inputs; NaN comes
// back as the canonical bf16 NaN).
__device__ __forceinline__ float round_bf16_rn(float x) {
  unsigned short h;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(x));
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// One potentially blocking test of phase `parity`: the hardware suspends the
// warp for up to `suspend_ns` while the phase is incomplete, so waiting warps
// do not spend issue slots polling.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity, uint32_t suspend_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(suspend_ns)
      : "memory");
  return ok != 0;
}
#ifndef IQ_SUSPEND_NS
#define IQ_SUSPEND_NS 20000u
#endif
// Bounded wait: true when the phase completed, false after `limit` tests
// (each of which may suspend the warp for up to IQ_SUSPEND_NS).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit = kSpinLimit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity, IQ_SUSPEND_NS)) return true;
  return false;
}

// ---- bulk copies (global -> shared, completion counted on an mbarrier)
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// the same without a cache-policy hint (data other CTAs may read again)
__device__ __forceinline__ void bulk_g2s_plain(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tensor2d_g2s(void* dst, const void* tmap, int x, int y, uint64_t* bar,
                                             uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---- register reallocation between warpgroups (every warp of a warpgroup
// executes it; the counts are per thread, multiples of 8 in [24, 256])
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ---- named barrier among a subset of warps
__device__ __forceinline__ void named_bar(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---- shared loads (volatile: measured faster than letting the compiler
// reorder them, and it keeps every load after the mbarrier wait)
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds8(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// ---- bit tricks
template <uint32_t LUT>
__device__ __forceinline__ uint32_t lop3(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, %4;" : "=r"(d) : "r"(a), "r"(b), "r"(c), "n"(LUT));
  return d;
}
// (a & b) | c
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  return lop3<0xEA>(a, b, c);
}
__device__ __forceinline__ uint32_t fma_bf16x2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t fma_f16x2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
// Pack two floats to f16x2: `lo` in bits 0..15, `hi` in bits 16..31.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- warp MMA m16n8k16, fp32 accumulate
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7},"
      " {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7},"
      " {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

}  // namespace iq
