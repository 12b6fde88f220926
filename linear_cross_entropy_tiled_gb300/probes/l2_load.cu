// Bytes per SM clock that bulk copies can move from global memory into shared
// memory, with every SM loading at once.
//
// The tensor-core kernels stage each CTA's operands through shared memory: at
// full MMA rate a 256 x 256 pair tile with 64-deep K slices needs 32 KB per
// CTA per 512 SM clocks, 64 bytes per clock per SM, most of it from L2. This
// program measures what the memory system delivers per SM when all SMs
// stream at once, from an L2-resident window and from one much larger than
// L2. One thread per CTA (one CTA per SM) keeps a ring of 16 KB copies in
// flight, each completing on its stage's mbarrier:
//   bulk     cp.async.bulk of 16 KB contiguous bytes;
//   tensor   cp.async.bulk.tensor.2d of a 64 x 128 bf16 box with the 128-byte
//            swizzle, the kernels' own operand load.
// `share` CTAs read the same sequence of chunks at about the same time (the
// kernels' CTA pairs share each operand slab among several pairs); share = 1
// gives every CTA its own data. Every wait is bounded: a stage that does not
// complete within a second sets an error flag, and the program reports it
// instead of a rate.
//
// Output: one JSON object per line.
//   flce_probe_l2_load                                 every configuration once
//   flce_probe_l2_load WINDOW_MB SHARE TENSOR SECONDS  one configuration, repeated
//                                                      for SECONDS (to read power)
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <algorithm>
#include <vector>

namespace {

constexpr int kChunk = 16384;  // bytes per copy
constexpr int kMaxStages = 12;

#define CHECK(x)                                                                       \
  do {                                                                                 \
    cudaError_t e_ = (x);                                                              \
    if (e_ != cudaSuccess) {                                                           \
      fprintf(stderr, "%s:%d %s: %s\n", __FILE__, __LINE__, #x, cudaGetErrorString(e_)); \
      exit(1);                                                                         \
    }                                                                                  \
  } while (0)

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for phase `parity` of the mbarrier at shared address `bar`, at most
// one second. Returns false if it gave up.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = now_ns();
  while (true) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
    if (now_ns() - t0 > 1000000000ull) return false;
  }
}

// CTA c belongs to group g = c / share of `share` CTAs; it copies chunk
// (g + i * groups) mod nchunks of the window, for i in [0, iters), through
// `stages` shared-memory buffers. With a tensor map the chunk is the box at
// rows 128 * chunk of a [rows][64] bf16 view of the window. out[c] = {cycles, ns}.
__global__ void __launch_bounds__(32) bulk_load_kernel(const char* src,
                                                       const __grid_constant__ CUtensorMap tmap,
                                                       bool tensor, long long nchunks,
                                                       long long iters, int stages, int share,
                                                       unsigned long long* out, int* error) {
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ __align__(8) uint64_t bars[kMaxStages];
  if (threadIdx.x != 0) return;
  for (int s = 0; s < stages; ++s)
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&bars[s])) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  const unsigned long long c0 = clock64(), t0 = now_ns();
  const long long groups = (gridDim.x + share - 1) / share;
  long long chunk = (blockIdx.x / share) % nchunks;
  bool ok = true;
  for (long long i = 0; i < iters && ok; ++i) {
    const int s = static_cast<int>(i % stages);
    const uint32_t bar = smem_addr(&bars[s]);
    if (i >= stages) ok = wait_phase(bar, static_cast<uint32_t>(((i / stages) - 1) & 1));
    if (!ok) break;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(kChunk)
                 : "memory");
    if (tensor) {
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
          " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(smem + s * kChunk)),
          "l"(reinterpret_cast<uint64_t>(&tmap)), "r"(0), "r"(static_cast<int>(chunk * 128)),
          "r"(bar)
          : "memory");
    } else {
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
              smem_addr(smem + s * kChunk)),
          "l"(src + chunk * kChunk), "r"(kChunk), "r"(bar)
          : "memory");
    }
    for (chunk += groups; chunk >= nchunks;) chunk -= nchunks;
  }
  // the copies still in flight
  for (long long i = iters > stages ? iters - stages : 0; i < iters && ok; ++i) {
    const int s = static_cast<int>(i % stages);
    ok = wait_phase(smem_addr(&bars[s]), static_cast<uint32_t>((i / stages) & 1));
  }
  if (!ok) atomicOr(error, 1);
  out[2 * blockIdx.x] = clock64() - c0;
  out[2 * blockIdx.x + 1] = now_ns() - t0;
}

}  // namespace

int main(int argc, char** argv) {
  const bool one = argc == 5;
  int dev = 0, sms = 0;
  CHECK(cudaGetDevice(&dev));
  CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const size_t max_window = size_t(2048) << 20;
  char* buf = nullptr;
  CHECK(cudaMalloc(&buf, max_window));
  CHECK(cudaMemset(buf, 1, max_window));
  unsigned long long* rec = nullptr;
  int* err = nullptr;
  CHECK(cudaMalloc(&rec, sizeof(unsigned long long) * 2 * sms));
  CHECK(cudaMalloc(&err, sizeof(int)));
  CHECK(cudaFuncSetAttribute(bulk_load_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kMaxStages * kChunk));
  printf("{\"sms\": %d, \"chunk_bytes\": %d}\n", sms, kChunk);
  // [rows][64] bf16 view of the whole buffer, 64 x 128 boxes, 128-byte swizzle
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    CHECK(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q));
    if (q != cudaDriverEntryPointSuccess || fn == nullptr) {
      fprintf(stderr, "cuTensorMapEncodeTiled not found\n");
      return 1;
    }
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  CUtensorMap tmap;
  {
    const cuuint64_t dims[2] = {64, max_window / 128};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {64, 128};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, buf, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      fprintf(stderr, "cuTensorMapEncodeTiled failed\n");
      return 1;
    }
  }
  std::vector<long long> windows_mb = {64, 2048};
  std::vector<int> tensors = {0, 1}, shares = {1, 4, 16, 152};
  double seconds = 0.0;
  if (one) {
    windows_mb = {atoll(argv[1])};
    shares = {atoi(argv[2])};
    tensors = {atoi(argv[3])};
    seconds = atof(argv[4]);
    if (windows_mb[0] < 1 || (windows_mb[0] << 20) > static_cast<long long>(max_window) ||
        shares[0] < 1) {
      fprintf(stderr, "window must be 1..2048 MB and share >= 1\n");
      return 1;
    }
  }
  for (long long wmb : windows_mb)
  for (int tensor : tensors)
  for (int share : shares) {
    {
      const int stages = 8;
      const long long nchunks = (wmb << 20) / kChunk;
      const long long iters = (48ll << 30) / (static_cast<long long>(sms) * kChunk);
      CHECK(cudaMemset(err, 0, sizeof(int)));
      auto launch = [&] {
        // the full ring's shared memory in every case, so that one CTA runs per SM
        bulk_load_kernel<<<sms, 32, kMaxStages * kChunk>>>(buf, tmap, tensor != 0, nchunks, iters,
                                                           stages, share, rec, err);
      };
      launch();
      CHECK(cudaDeviceSynchronize());
      if (seconds > 0) {   // repeat for the requested time, then time one more run
        cudaEvent_t a, b;
        CHECK(cudaEventCreate(&a));
        CHECK(cudaEventCreate(&b));
        CHECK(cudaEventRecord(a));
        launch();
        CHECK(cudaEventRecord(b));
        CHECK(cudaEventSynchronize(b));
        float one_ms = 1.f;
        CHECK(cudaEventElapsedTime(&one_ms, a, b));
        const int reps = static_cast<int>(seconds * 1e3 / std::max(one_ms, 0.01f));
        for (int r = 0; r < reps; ++r) launch();
        CHECK(cudaDeviceSynchronize());
        CHECK(cudaEventDestroy(a));
        CHECK(cudaEventDestroy(b));
      }
      cudaEvent_t e0, e1;
      CHECK(cudaEventCreate(&e0));
      CHECK(cudaEventCreate(&e1));
      CHECK(cudaEventRecord(e0));
      launch();
      CHECK(cudaEventRecord(e1));
      CHECK(cudaEventSynchronize(e1));
      CHECK(cudaGetLastError());
      float ms = 0.f;
      CHECK(cudaEventElapsedTime(&ms, e0, e1));
      std::vector<unsigned long long> h(2 * sms);
      CHECK(cudaMemcpy(h.data(), rec, h.size() * 8, cudaMemcpyDeviceToHost));
      int herr = 0;
      CHECK(cudaMemcpy(&herr, err, sizeof(int), cudaMemcpyDeviceToHost));
      double cyc = 0, ns = 0;
      for (int i = 0; i < sms; ++i) {
        cyc += static_cast<double>(h[2 * i]);
        ns += static_cast<double>(h[2 * i + 1]);
      }
      const double bytes = static_cast<double>(sms) * iters * kChunk;
      const double mhz = cyc / ns * 1e3;
      const double per_sm_clk = bytes / sms / (cyc / sms);
      printf("{\"probe\": \"%s\", \"window_bytes\": %lld, \"share\": %d, \"stages\": %d, "
             "\"bytes\": %.0f, \"ms\": %.4f, \"gbps\": %.1f, \"sm_mhz\": %.0f, "
             "\"bytes_per_sm_clock\": %.2f, \"status\": \"%s\"}\n",
             tensor ? "tensor_load" : "bulk_load", wmb << 20, share, stages, bytes, ms,
             bytes / (ms * 1e-3) / 1e9, mhz, per_sm_clk, herr ? "a wait expired" : "ok");
      fflush(stdout);
      CHECK(cudaEventDestroy(e0));
      CHECK(cudaEventDestroy(e1));
    }
  }
  CHECK(cudaFree(buf));
  CHECK(cudaFree(rec));
  CHECK(cudaFree(err));
  return 0;
}
