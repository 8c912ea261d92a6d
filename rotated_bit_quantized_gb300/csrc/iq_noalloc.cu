// libiqkv: iq_attend_noalloc — attention for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc: a serving process that has already
// handed all of HBM to its own arena (weights + KV pool), a plugin that only
// sees the buffers its host gives it, or a latency-critical decode loop where
// an allocation (which may synchronise the device) is not acceptable.  For
// them this entry point runs the same split-KV attention as iq_attend, with
// its scratch (the split partials and the status word) in a library-owned,
// file-scope device array instead of a caller workspace.
//
// The array is IQ_NOALLOC_SCRATCH_BYTES large and lives for as long as the
// library is loaded on a device.  Its address is looked up once per device,
// on the first call made with that device current.  Every call shares the
// array, so calls that may run at the same time on the GPU (different streams,
// no ordering between them) race on it and must not overlap.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "iq_common.cuh"

namespace iq {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[IQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (set-up on the
// first call per device).  In host code the array's name is only a host-side
// stand-in, so the real address must come from cudaGetSymbolAddress.
int scratch_address(void** out) {
  int dev = -1;
  IQ_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return fail(IQ_ERR_UNSUPPORTED, "device index above 63");
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return IQ_OK;
}

}  // namespace
}  // namespace iq

extern "C" int iq_attend_noalloc(const iq_cache* cache, const void* q, int q_heads, int n_queries,
                                 float scale, int causal, const void* rot, void* out, int out_f32,
                                 iq_stream_t stream) {
  iq::clear_error();
  int st = iq_cache_check(cache);
  if (st != IQ_OK) return st;
  size_t need = 0;
  if (n_queries >= 1 && q_heads >= 1 && q_heads % cache->kv_heads == 0 &&
      iq::prefill_shape(cache, q_heads, n_queries, 0)) {
    need = IQ_WORKSPACE_HEAD_BYTES;  // the prefill kernel uses only the status word of the head
  } else {
    st = iq_attend_workspace(cache, q_heads, n_queries, &need);
    if (st != IQ_OK) return st;
  }
  if (need > IQ_NOALLOC_SCRATCH_BYTES)
    return iq::fail(IQ_ERR_WORKSPACE,
                    "iq_attend_noalloc: this call needs " + std::to_string(need) +
                        " bytes of scratch, above the built-in " +
                        std::to_string(static_cast<size_t>(IQ_NOALLOC_SCRATCH_BYTES)) +
                        "; use iq_attend with a caller workspace");
  void* scratch = nullptr;
  st = iq::scratch_address(&scratch);
  if (st != IQ_OK) return st;
  // The array is zero when the library loads, so its status word starts
  // clear; the split partials are written before they are read, and the unit
  // counters return to zero after every call (also one whose wait ran out).
  return iq_attend(cache, q, q_heads, n_queries, scale, causal, rot, out, out_f32, scratch,
                   IQ_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" int iq_noalloc_read_status(iq_stream_t stream, int* device_status) {
  iq::clear_error();
  if (!device_status) return iq::fail(IQ_ERR_INVALID_ARG, "null device_status");
  void* scratch = nullptr;
  int st = iq::scratch_address(&scratch);
  if (st != IQ_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned v = 0;
  IQ_CUDA(cudaStreamSynchronize(s));
  IQ_CUDA(cudaMemcpy(&v, scratch, sizeof(v), cudaMemcpyDeviceToHost));
  // after a failure, clear the whole head (status word and unit counters)
  if (v) IQ_CUDA(cudaMemset(scratch, 0, IQ_WORKSPACE_HEAD_BYTES));
  *device_status = static_cast<int>(v);
  return v ? iq::fail(IQ_ERR_DEVICE, "a kernel reported a failure (status bits set)") : IQ_OK;
}
