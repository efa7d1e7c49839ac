// ra_noalloc.cu -- a backward entry point for callers that cannot allocate device memory.
//
// Some callers have no way to hand this library a workspace: a plugin inside a host
// runtime that passes it tensors and a stream but exposes no allocator, or a
// latency-critical service that may not call cudaMalloc on its hot path because the call
// can synchronise the whole device and takes unbounded time.  ra_bwd_noalloc serves
// them: it runs the same backward as ra_bwd, but its scratch (error word, fp32 dQ
// accumulator, D and lse*log2(e)) lives in one fixed array of device memory that belongs
// to the library.  The caller still passes every input and output.
#include <cstdio>
#include <mutex>

#include "ra_internal.h"

namespace {

// The scratch array: every GPU that loads the library reserves it until the process
// exits.  64 MiB covers B*L*H up to about 128K rows at head_dim 128.
constexpr size_t kNoAllocScratchBytes = 64ull << 20;
static __device__ __align__(256) unsigned char ra_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

}  // namespace

extern "C" ra_status_t ra_bwd_noalloc(const ra_params_t* p, const void* q, const void* k,
                                      const void* v, const void* out, int out_dtype,
                                      const float* lse, const void* dout, void* dq, void* dk,
                                      void* dv, void* stream) {
  const size_t need = ra_bwd_workspace_bytes(p);
  if (need == 0) {
    // invalid parameters: let the regular entry point produce the precise status/message
    return ra_bwd(p, q, k, v, out, out_dtype, lse, dout, dq, dk, dv, nullptr, 0, stream);
  }
  if (need > kNoAllocScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "ra_bwd_noalloc: this problem needs %zu bytes of scratch; the built-in scratch "
             "holds %zu bytes (use ra_bwd with a caller-provided workspace)",
             need, kNoAllocScratchBytes);
    ra::set_last_error_message(msg);
    return RA_ERR_WORKSPACE;
  }
  // Set-up, once per device, with that device current: the host-side name of the array
  // is not a device address, so look the address up and keep it.
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    ra::set_last_error_message("ra_bwd_noalloc: no usable current CUDA device");
    return RA_ERR_CUDA;
  }
  void* ptr = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
      void* found = nullptr;
      if (cudaGetSymbolAddress(&found, ra_noalloc_scratch) != cudaSuccess || !found) {
        ra::set_last_error_message("ra_bwd_noalloc: cudaGetSymbolAddress of the scratch failed");
        return RA_ERR_CUDA;
      }
      g_scratch_ptr[dev] = found;
    }
    ptr = g_scratch_ptr[dev];
  }
  // The array keeps the previous call's contents.  The error word must start at zero (the
  // kernels stop early when it is set); the dQ accumulator is zeroed by the preprocess.
  if (cudaMemsetAsync(ptr, 0, ra::kWsHeader, reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess) {
    ra::set_last_error_message("ra_bwd_noalloc: clearing the scratch error word failed");
    return RA_ERR_CUDA;
  }
  return ra_bwd(p, q, k, v, out, out_dtype, lse, dout, dq, dk, dv, ptr, kNoAllocScratchBytes,
                stream);
}
