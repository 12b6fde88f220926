// Throughput of fp32 reduce-add into a window of global memory, on this GPU.
//
// A backward that keeps each dlogits tile on chip and feeds both gradient
// contractions from it cannot hold its outputs on chip: a 256-row block of
// grad_hidden or grad_weight is 256 x H fp32, 4 MB at H = 4096. It has to add
// each tile's fp32 contribution into global memory, a reduction that L2
// resolves if the window of live outputs stays resident there. This program
// measures how fast that can go, three ways, for windows from L2-sized to
// far larger than L2:
//   bulk   one thread per CTA issues cp.reduce.async.bulk .add.f32 of a
//          16 KB shared-memory block into the window (the asynchronous bulk
//          reduction a tile flush would use);
//   red_v4 every thread issues red.global.add.v4.f32 (16 bytes) from
//          registers;
//   store  every thread issues plain 16-byte stores, the write bandwidth of
//          the same window for comparison.
// Each reduction run is checked afterwards: every element of the window must
// hold the exact number of 1.0 additions that the schedule sent to it.
//
// Output: one JSON object per line, with bytes moved per run and GB/s.
//   flce_probe_l2_reduce [max_window_mb]
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <algorithm>
#include <vector>

namespace {

constexpr int kThreads = 256;
constexpr int kBlockBytes = 16384;  // bytes per bulk reduction
constexpr int kCtasPerSm = 2;

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

// Block i of CTA c goes to window block (c + i * gridDim.x) mod nblocks.
__global__ void __launch_bounds__(kThreads) bulk_reduce_kernel(float* dst, long long nblocks,
                                                               long long ops_per_cta) {
  extern __shared__ __align__(128) unsigned char smem[];
  float* src = reinterpret_cast<float*>(smem);
  for (int i = threadIdx.x; i < kBlockBytes / 4; i += blockDim.x) src[i] = 1.0f;
  // The bulk copy reads shared memory through the async proxy.
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  if (threadIdx.x != 0) return;
  long long b = blockIdx.x % nblocks;
  for (long long i = 0; i < ops_per_cta; ++i) {
    char* g = reinterpret_cast<char*>(dst) + b * kBlockBytes;
    asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(g),
                 "r"(smem_addr(src)), "r"(kBlockBytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    // at most 8 groups still reading the (unchanging) source block
    asm volatile("cp.async.bulk.wait_group.read 8;" ::: "memory");
    for (b += gridDim.x; b >= nblocks;) b -= nblocks;
  }
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Thread t, iteration i: 16-byte slot (t + i * threads) mod nslots.
__global__ void __launch_bounds__(kThreads) red_v4_kernel(float* dst, long long nslots,
                                                          long long iters) {
  const long long nt = static_cast<long long>(gridDim.x) * blockDim.x;
  long long s = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) % nslots;
  for (long long i = 0; i < iters; ++i) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 4 * s), "f"(1.f),
                 "f"(1.f), "f"(1.f), "f"(1.f)
                 : "memory");
    for (s += nt; s >= nslots;) s -= nslots;
  }
}

__global__ void __launch_bounds__(kThreads) store_v4_kernel(float4* dst, long long nslots,
                                                            long long iters) {
  const long long nt = static_cast<long long>(gridDim.x) * blockDim.x;
  long long s = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) % nslots;
  for (long long i = 0; i < iters; ++i) {
    dst[s] = make_float4(1.f, 1.f, 1.f, 1.f);
    for (s += nt; s >= nslots;) s -= nslots;
  }
}

// Number of additions each 16-byte slot (or bulk block) received: the same
// index formula the kernels use, counted on the host.
std::vector<uint32_t> expected_counts(long long units, long long n_threads, long long iters) {
  std::vector<uint32_t> c(static_cast<size_t>(units), 0);
  const long long total = n_threads * iters;
  const long long full = total / units, rest = total % units;
  for (auto& x : c) x = static_cast<uint32_t>(full);
  // the (t + i * nt) sequence visits consecutive integers 0 .. total-1 mod units
  for (long long k = 0; k < rest; ++k) c[static_cast<size_t>(k)] += 1;
  return c;
}

bool check(const float* dev, long long units, int floats_per_unit, const std::vector<uint32_t>& want) {
  std::vector<float> h(static_cast<size_t>(units) * floats_per_unit);
  CHECK(cudaMemcpy(h.data(), dev, h.size() * sizeof(float), cudaMemcpyDeviceToHost));
  for (long long u = 0; u < units; ++u)
    for (int k = 0; k < floats_per_unit; ++k)
      if (h[static_cast<size_t>(u) * floats_per_unit + k] != static_cast<float>(want[static_cast<size_t>(u)]))
        return false;
  return true;
}

template <class Launch>
float time_ms(Launch launch, int reps) {
  cudaEvent_t e0, e1;
  CHECK(cudaEventCreate(&e0));
  CHECK(cudaEventCreate(&e1));
  std::vector<float> t;
  for (int r = 0; r < reps; ++r) {
    CHECK(cudaEventRecord(e0));
    launch();
    CHECK(cudaEventRecord(e1));
    CHECK(cudaEventSynchronize(e1));
    CHECK(cudaGetLastError());
    float ms = 0.f;
    CHECK(cudaEventElapsedTime(&ms, e0, e1));
    t.push_back(ms);
  }
  std::sort(t.begin(), t.end());
  CHECK(cudaEventDestroy(e0));
  CHECK(cudaEventDestroy(e1));
  return t[t.size() / 2];
}

}  // namespace

int main(int argc, char** argv) {
  const long long max_mb = argc > 1 ? atoll(argv[1]) : 4096;
  int dev = 0, sms = 0;
  CHECK(cudaGetDevice(&dev));
  CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  cudaDeviceProp prop;
  CHECK(cudaGetDeviceProperties(&prop, dev));
  CHECK(cudaFuncSetAttribute(bulk_reduce_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kBlockBytes));
  const int grid = sms * kCtasPerSm;
  float* buf = nullptr;
  CHECK(cudaMalloc(&buf, static_cast<size_t>(max_mb) << 20));
  printf("{\"device\": \"%s\", \"sms\": %d, \"l2_bytes\": %d, \"ctas\": %d, \"threads\": %d}\n",
         prop.name, sms, prop.l2CacheSize, grid, kThreads);

  const long long windows_mb[] = {16, 48, 96, 256, 1024, 4096};
  for (long long wmb : windows_mb) {
    if (wmb > max_mb) continue;
    const long long wbytes = wmb << 20;
    // about 2 x 10^11 bytes per timed run at L2 speeds, fewer beyond L2
    const long long target = wbytes <= (128ll << 20) ? (200ll << 30) : (64ll << 30);

    // bulk: each CTA issues ops_per_cta 16 KB reductions
    {
      const long long nblocks = wbytes / kBlockBytes;
      const long long ops = std::max<long long>(1, target / (static_cast<long long>(grid) * kBlockBytes));
      auto launch = [&] { bulk_reduce_kernel<<<grid, kThreads, kBlockBytes>>>(buf, nblocks, ops); };
      CHECK(cudaMemset(buf, 0, wbytes));
      launch();
      CHECK(cudaDeviceSynchronize());
      const bool ok = check(buf, nblocks, kBlockBytes / 4, expected_counts(nblocks, grid, ops));
      const float ms = time_ms(launch, 5);
      const double bytes = static_cast<double>(grid) * ops * kBlockBytes;
      printf("{\"probe\": \"bulk_reduce_add_f32\", \"window_bytes\": %lld, \"bytes\": %.0f, "
             "\"ms\": %.4f, \"gbps\": %.1f, \"check\": \"%s\"}\n",
             wbytes, bytes, ms, bytes / (ms * 1e-3) / 1e9, ok ? "ok" : "MISMATCH");
      fflush(stdout);
    }
    // red_v4 and store: each thread issues iters 16-byte operations
    {
      const long long nslots = wbytes / 16;
      const long long nthr = static_cast<long long>(grid) * kThreads;
      const long long iters = std::max<long long>(1, target / (nthr * 16));
      auto launch = [&] { red_v4_kernel<<<grid, kThreads>>>(buf, nslots, iters); };
      CHECK(cudaMemset(buf, 0, wbytes));
      launch();
      CHECK(cudaDeviceSynchronize());
      const bool ok = check(buf, nslots, 4, expected_counts(nslots, nthr, iters));
      const float ms = time_ms(launch, 5);
      const double bytes = static_cast<double>(nthr) * iters * 16;
      printf("{\"probe\": \"red_v4_add_f32\", \"window_bytes\": %lld, \"bytes\": %.0f, "
             "\"ms\": %.4f, \"gbps\": %.1f, \"check\": \"%s\"}\n",
             wbytes, bytes, ms, bytes / (ms * 1e-3) / 1e9, ok ? "ok" : "MISMATCH");
      auto launch_st = [&] {
        store_v4_kernel<<<grid, kThreads>>>(reinterpret_cast<float4*>(buf), nslots, iters);
      };
      launch_st();
      const float ms_st = time_ms(launch_st, 5);
      printf("{\"probe\": \"store_v4_f32\", \"window_bytes\": %lld, \"bytes\": %.0f, "
             "\"ms\": %.4f, \"gbps\": %.1f}\n",
             wbytes, bytes, ms_st, bytes / (ms_st * 1e-3) / 1e9);
      fflush(stdout);
    }
  }
  CHECK(cudaFree(buf));
  return 0;
}
