// flce_forward_noalloc: the forward pass for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc or any allocator of their own. Examples
// are a training loop whose framework forbids allocation once its memory plan
// is fixed, a runtime that owns every byte of device memory through a fixed
// arena, and C hosts that only hand over pointers to tensors they already
// have. This
// entry point runs the same kernels as flce_forward. It takes its scratch
// memory (the per-panel partial states, the target logits and the block sums)
// from a fixed array that lives in this library's device image, not from a
// caller-provided workspace.
#include <cuda_runtime.h>
#include <stdio.h>

#include <mutex>

#include "flce.h"
#include "kernels.h"

namespace {

// 48 MiB holds the forward scratch of every workload this library is
// benchmarked on. The largest, N=16384 x V=151936, needs about 39 MB. Every
// GPU that loads the library keeps this array allocated until the process
// exits.
constexpr size_t kNoAllocScratchBytes = size_t(48) << 20;

static __device__ __align__(256) unsigned char g_forward_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[64] = {};

// Device address of g_forward_scratch on the current device. In host code
// the array's name is only a host-side stand-in, so the address has to be
// looked up once per device, with that device current.
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) return FLCE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_forward_scratch);
    if (e != cudaSuccess || p == nullptr) return FLCE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return FLCE_OK;
}

}  // namespace

extern "C" int flce_forward_noalloc(const flce_params* p, const void* hidden, const void* weight,
                                    const void* bias, const int64_t* targets, float* loss,
                                    float* lse, int64_t* num_correct, float* entropy_sum,
                                    flce_stream_t stream) {
  size_t need = 0;
  int rc = flce_workspace_bytes(p, FLCE_PASS_FORWARD, &need);
  if (rc != FLCE_OK) return rc;
  if (need > kNoAllocScratchBytes) {
    char msg[160];
    snprintf(msg, sizeof(msg),
             "flce_forward_noalloc: this size needs %zu bytes of scratch, above the "
             "fixed maximum of %zu",
             need, kNoAllocScratchBytes);
    flce::set_error_detail(msg);
    fprintf(stderr, "%s\n", msg);
    return FLCE_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  if ((rc = scratch_address(&scratch)) != FLCE_OK) return rc;
  // flce_forward zeroes the status word at the start of the scratch before
  // any kernel runs. Every other scratch byte is written before it is read,
  // except after an expired bounded wait: the forward then skips stores, and
  // the merge, seeing the timeout in the status word, writes NaN outputs
  // instead of combining what an earlier call left in the array.
  return flce_forward(p, hidden, weight, bias, targets, loss, lse, num_correct, entropy_sum,
                      scratch, kNoAllocScratchBytes, stream);
}
