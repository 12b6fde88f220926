// tcgen05 / TMA kernels of the 16-bit path (bf16 or fp16 operands; sm_103a).
//
// Every kernel here is persistent and warp-specialised. CTAs run in pairs
// (clusters of 2) that share one 2-SM MMA (tcgen05.mma.cta_group::2) per
// 256 x 256 tile. Roles in each CTA of a pair:
//   warp 0     one thread issues TMA loads of this CTA's 128 rows of A and
//              its half of B into a 6-stage shared ring. The completion
//              bytes of both CTAs go to the even CTA's "full" barriers;
//   warp 1     in the even CTA, one thread issues the pair's MMAs into
//              double-buffered TMEM accumulators (each CTA holds its 128
//              rows x 256 fp32 columns) and commits to both CTAs' barriers.
//              In both CTAs this warp owns the TMEM allocation;
//   warps 2-5  the epilogue. Each thread owns one accumulator row, which is
//              one TMEM lane, and reads it with tcgen05.ld.
// The kernels differ only in the tile sequence, the operand layouts and the
// epilogue:
//   fwd_tc   logits tile -> bias, scale, softcap -> online max / sum-exp /
//            sum z*exp / argmax per row, plus the target logit
//            (fused-linear-ce README, "Algorithm" and "Metrics for free").
//   ds_tc    recomputed logits tile -> dlogits = (softmax (1 + 2 zeta lse)
//            - onehot) x softcap' x scale x gamma -> bf16 row chunk, plus
//            per-128-row column sums for grad_bias (same README, "Algorithm";
//            the z-loss term is this library's reading of "Chunked Linear
//            Cross-Entropy", "Usage").
//   gemm_tc  plain D = A B with fp32 accumulation. It serves the two
//            gradient contractions grad_hidden = dS W and grad_weight =
//            dS^T h ("Chunked Linear Loss", "Gradient handling"), and the
//            fp32 accumulation of grad_weight across row chunks ("Chunked
//            Linear Loss", "Weight-gradient accumulation dtype").
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "kernels.h"
#include "ptx.cuh"

namespace flce {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kFull = 0xffffffffu;

// --------------------------------------------------------------- smem map
struct TcSmem {
  uint8_t* a;            // kStages x kStageA
  uint8_t* b;            // kStages x kStageB
  float* scratch;        // 8 KB: column sums of the dlogits epilogue
  uint64_t* full;        // kStages: TMA bytes landed
  uint64_t* empty;       // kStages: MMAs done reading the stage
  uint64_t* tfull;       // 2: accumulator complete
  uint64_t* tempty;      // 2: epilogue done reading the accumulator
  uint64_t* mma_done;    // 1: all MMAs complete (teardown)
  uint32_t* tmem_slot;
  int* abort;
  // Unit queue of the dynamic GEMM schedule (see TileQueue): the even CTA's
  // producer publishes each unit to both CTAs of the pair.
  uint64_t* q_full;      // kQueue: the slot holds a unit (in each CTA)
  uint64_t* q_empty;     // kQueue: every consumer has read it (even CTA only)
  int* q_unit;           // kQueue
  int* ep_unit;          // 2: a unit passed from the dlogits kernel's queue reader to its epilogue warps
};

constexpr int kQueue = 4;
// Readers of each queue slot: the MMA thread, the odd CTA's producer, and the
// four epilogue warps of each CTA (the GEMM and the forward), or one epilogue
// warp of each CTA (the dlogits kernel, whose epilogue warps share units
// through shared memory).
constexpr int kQueueReaders = 2 + 2 * 4;
constexpr int kDsQueueReaders = 2 + 2 * 1;

__device__ __forceinline__ TcSmem carve_smem(uint8_t* raw) {
  TcSmem s;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  s.a = base;
  s.b = base + kStages * kStageA;
  s.scratch = reinterpret_cast<float*>(s.b + kStages * kStageB);
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(s.scratch) + 8192);
  s.full = bars;
  s.empty = bars + kStages;
  s.tfull = bars + 2 * kStages;
  s.tempty = s.tfull + 2;
  s.mma_done = s.tempty + 2;
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.mma_done + 1);
  s.abort = reinterpret_cast<int*>(s.tmem_slot + 1);
  s.q_full = s.mma_done + 2;   // after tmem_slot and abort (8 bytes)
  s.q_empty = s.q_full + kQueue;
  s.q_unit = reinterpret_cast<int*>(s.q_empty + kQueue);
  s.ep_unit = s.q_unit + kQueue;
  return s;
}

// Barriers and TMEM of both CTAs of the pair. The cluster barrier at the end
// makes every barrier initialised before any remote arrive or
// remote-signalling TMA can target it.
__device__ __forceinline__ uint32_t tc_setup(const TcSmem& s, int warp, int epi_warps = 4,
                                             int queue_readers = kQueueReaders) {
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.full[i], 1);   // even CTA: its own arrive.expect_tx
      mbar_init(&s.empty[i], 1);  // the MMA commit, multicast to both CTAs
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.tfull[i], 1);   // the MMA commit, multicast to both CTAs
      mbar_init(&s.tempty[i], 2 * epi_warps);  // even CTA: every epilogue warp of both CTAs
    }
    mbar_init(s.mma_done, 1);
    for (int i = 0; i < kQueue; ++i) {
      mbar_init(&s.q_full[i], 1);
      mbar_init(&s.q_empty[i], queue_readers);
    }
    *s.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(s.tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  return *s.tmem_slot;
}

// Start of a CTA's clock record (thread 0 only; see ClockRecord).
struct ClockStart {
  unsigned long long c0 = 0, t0 = 0;
  __device__ __forceinline__ explicit ClockStart(const ClockRecord* rec) {
    if (rec != nullptr && threadIdx.x == 0) {
      c0 = clock64();
      t0 = global_timer_ns();
    }
  }
  __device__ __forceinline__ void finish(ClockRecord* rec) const {
    if (rec != nullptr && threadIdx.x == 0) {
      atomicAdd(&rec->cycles, static_cast<unsigned long long>(clock64()) - c0);
      atomicAdd(&rec->ns, global_timer_ns() - t0);
    }
  }
};

// The even CTA's MMAs read the odd CTA's shared memory and write its TMEM.
// So neither CTA releases TMEM or exits before the whole pair is done.
__device__ __forceinline__ void tc_teardown(uint32_t tmem, int warp) {
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// Bounded wait that ignores the abort flag. It is used only to drain
// operations that are already in flight before the CTA exits.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (global_timer_ns() - t0 > 200000000ull) return;
  }
}

// --------------------------------------------------------- producer / MMA
// ForEachTile(f) calls f(ta, tb) for every tile of this pair, in order.
// KBlocks(ta, tb) is the number of 64-deep K slices of that tile.
// Issue(ta, tb, kb, a_dst, b_dst, mbar) issues this CTA's TMA loads of one
// K slice; `mbar` is the shared::cluster address of the even CTA's barrier.
template <class ForEachTile, class KBlocks, class Issue>
__device__ __forceinline__ void producer_role(const TcSmem& s, const WaitGuard& g,
                                              KBlocks kblocks_of, bool leader,
                                              ForEachTile for_each_tile, Issue issue) {
  int stage = 0;
  uint32_t phase = 0;
  bool dead = false;
  long long issued = 0;
  for_each_tile([&](int ta, int tb) {
    const int kblocks = kblocks_of(ta, tb);
    for (int kb = 0; kb < kblocks && !dead; ++kb) {
      if (!mbar_wait(&s.empty[stage], phase ^ 1u, g)) {
        dead = true;
        break;
      }
      // The even CTA expects the bytes of both CTAs' loads on its barrier.
      if (leader) mbar_arrive_expect_tx(&s.full[stage], 2 * kStageBytes);
      issue(ta, tb, kb, s.a + stage * kStageA, s.b + stage * kStageB,
            mapa_shared(smem_u32(&s.full[stage]), 0));
      ++issued;
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  });
  if (dead && leader) {
    // Let the loads already in flight land before shared memory is released.
    const long long first = issued > kStages ? issued - kStages : 0;
    for (long long i = first; i < issued; ++i)
      drain_wait(&s.full[i % kStages], static_cast<uint32_t>((i / kStages) & 1));
  }
}

// Runs in the even CTA only. Descs(ta, tb, sa, sb, kk, adesc, bdesc, idesc)
// builds the operand and instruction descriptors of the kk-th 16-deep K
// step within a 64-deep stage of tile (ta, tb).
// With `rec` (profiling), the role's cycles and its waits for operands and
// for a free accumulator are added to the launch's clock record.
template <class ForEachTile, class KBlocks, class Descs>
__device__ __forceinline__ void mma_role(const TcSmem& s, const WaitGuard& g, uint32_t tmem,
                                         KBlocks kblocks_of, ForEachTile for_each_tile,
                                         Descs descs, ClockRecord* rec) {
  int stage = 0;
  uint32_t phase = 0;
  int acc = 0;
  uint32_t acc_phase = 0;
  bool dead = false;
  const bool prof = rec != nullptr;
  const unsigned long long t_start = prof ? clock64() : 0;
  unsigned long long w_ops = 0, w_acc = 0;
  for_each_tile([&](int ta, int tb) {
    if (dead) return;
    const int kblocks = kblocks_of(ta, tb);
    const unsigned long long c0 = prof ? clock64() : 0;
    if (!mbar_wait(&s.tempty[acc], acc_phase ^ 1u, g)) {
      dead = true;
      return;
    }
    if (prof) w_acc += clock64() - c0;
    tc_fence_after();
    const uint32_t d = tmem + static_cast<uint32_t>(acc * kBN);
    for (int kb = 0; kb < kblocks; ++kb) {
      const unsigned long long c1 = prof ? clock64() : 0;
      if (!mbar_wait(&s.full[stage], phase, g)) {
        dead = true;
        return;
      }
      if (prof) w_ops += clock64() - c1;
      tc_fence_after();
      const uint32_t sa = smem_u32(s.a + stage * kStageA);
      const uint32_t sb = smem_u32(s.b + stage * kStageB);
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk) {
        uint64_t ad, bd;
        uint32_t idesc;
        descs(ta, tb, sa, sb, kk, ad, bd, idesc);
        umma_f16_pair(d, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
      }
      umma_commit_pair_multicast(&s.empty[stage], 0x3);
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    umma_commit_pair_multicast(&s.tfull[acc], 0x3);
    acc ^= 1;
    if (acc == 0) acc_phase ^= 1u;
  });
  // Every MMA must have finished before TMEM is released.
  umma_commit_pair(s.mma_done);
  drain_wait(s.mma_done, 0);
  if (prof) {
    atomicAdd(&rec->mma_cycles, static_cast<unsigned long long>(clock64()) - t_start);
    atomicAdd(&rec->mma_wait_operands, w_ops);
    atomicAdd(&rec->mma_wait_accumulator, w_acc);
  }
}

// Both operands K-major; the pair computes M = 256, N = 256.
template <typename T>
__device__ __forceinline__ void kmajor_descs(int, int, uint32_t sa, uint32_t sb, int kk,
                                             uint64_t& ad, uint64_t& bd, uint32_t& idesc) {
  ad = smem_desc_sw128(sa + kk * 32, 16, 1024);
  bd = smem_desc_sw128(sb + kk * 32, 16, 1024);
  idesc = idesc_f16kind_f32(kPairM, kBN, false, false, Elem<T>::kBf16);
}

// Operand descriptor of the kk-th 16-deep K step: K-major rows advance 32 B
// within the swizzle row; MN-major tiles advance 16 k-rows (two 1 KB atoms),
// with the two 64-wide MN atoms 8 KB apart.
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, bool mn_major, int kk) {
  return mn_major ? smem_desc_sw128(base + kk * 2048, 8192, 1024)
                  : smem_desc_sw128(base + kk * 32, 16, 1024);
}

// Epilogue: wait until accumulator `acc` is full. The result is warp-uniform,
// so a warp either reads TMEM with every lane or not at all.
__device__ __forceinline__ bool epi_wait_full(const TcSmem& s, int acc, uint32_t acc_phase,
                                              const WaitGuard& g, bool dead) {
  bool ok = !dead && mbar_wait(&s.tfull[acc], acc_phase, g);
  ok = __all_sync(kFull, ok);
  if (ok) tc_fence_after();
  return ok;
}

// Tells the even CTA's MMA thread that this warp is done with accumulator
// `acc`. Both CTAs' epilogue warps arrive on the even CTA's barrier.
__device__ __forceinline__ void epi_release(const TcSmem& s, int acc, int lane) {
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&s.tempty[acc]), 0));
}

// 32 bias values times scale, for columns col0 .. col0+31. Columns at or
// beyond V read as 0.
template <typename T, bool kRagged>
__device__ __forceinline__ void load_bias32(const T* bias, int col0, int V, float scale,
                                            float (&bs)[32]) {
  if (!kRagged) {
    const uint4* p = reinterpret_cast<const uint4*>(bias + col0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 w = __ldg(p + q);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        bs[q * 8 + 2 * h] = Elem<T>::lo(ws[h]) * scale;
        bs[q * 8 + 2 * h + 1] = Elem<T>::hi(ws[h]) * scale;
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      bs[j] = (col0 + j < V) ? Elem<T>::to_float(bias[col0 + j]) * scale : 0.f;
  }
}

// Transformed logit z from the raw accumulator value.
// tanh from the identity tanh(x) = 1 - 2 / (e^(2x) + 1), with e^(2x) taken as
// 2^(2x log2 e) by ex2.approx (relative error about 2^-22) and a fast
// division. The absolute error stays near 1e-7 for every x, far inside the
// 16-bit paths' tolerances. It is a handful of instructions per logit, which
// matters in the softcapped epilogues. e^(2x) overflowing to +inf gives
// exactly 1, and underflowing to 0 gives exactly -1.
__device__ __forceinline__ float tanh_via_exp2(float x) {
  const float e = ex2_approx(x * (2.f * kLog2e));
  return 1.f - __fdividef(2.f, e + 1.f);
}

template <bool kBias, bool kSoftcap>
__device__ __forceinline__ float transform(uint32_t raw, float bs, float scale, float cap,
                                           float inv_cap) {
  float u = kBias ? fmaf(__uint_as_float(raw), scale, bs) : __uint_as_float(raw) * scale;
  if (kSoftcap) u = cap * tanh_via_exp2(u * inv_cap);
  return u;
}

// ======================================================= forward kernel
// Sum of the 32 values of x by a pairwise tree, the first four levels in
// packed pairs of lanes (x is overwritten).
__device__ __forceinline__ float tree_sum32(float (&x)[32]) {
  add_half_pairs<16>(x);
  add_half_pairs<8>(x);
  add_half_pairs<4>(x);
  add_half_pairs<2>(x);
  return x[0] + x[1];
}

// Largest of the 32 values, by a pairwise tree.
__device__ __forceinline__ float tree_max32(const float (&z)[32]) {
  float t[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) t[j] = fmaxf(z[2 * j], z[2 * j + 1]);
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int j = 0; j < w; ++j) t[j] = fmaxf(t[j], t[j + w]);
  return t[0];
}

// x[i] for a runtime i in [0, 32), as a 5-level multiplexer on the bits of
// i. Every array index stays a compile-time constant, so x stays in
// registers.
__device__ __forceinline__ float select32(const float (&x)[32], int i) {
  float t16[16], t8[8], t4[4], t2[2];
#pragma unroll
  for (int j = 0; j < 16; ++j) t16[j] = (i & 16) ? x[j + 16] : x[j];
#pragma unroll
  for (int j = 0; j < 8; ++j) t8[j] = (i & 8) ? t16[j + 8] : t16[j];
#pragma unroll
  for (int j = 0; j < 4; ++j) t4[j] = (i & 4) ? t8[j + 4] : t8[j];
#pragma unroll
  for (int j = 0; j < 2; ++j) t2[j] = (i & 2) ? t4[j + 2] : t4[j];
  return (i & 1) ? t2[1] : t2[0];
}

// The 256 x 256 logit tile's 32 columns col0 .. col0 + 31 of one row, folded
// into the row's online state (fused-linear-ce README, "Algorithm"): the
// transform, the running max m, sum exp(z - m) and, with kMetrics, the first
// index of the max and sum z exp(z - m) ("Metrics for free"). The arithmetic
// that m and ssum see is the same with and without kMetrics, so loss and lse
// are bit-identical either way. The element-wise steps run in packed pairs of
// lanes (f32x2), rounded as the scalar steps are.
template <typename T, bool kRagged, bool kBias, bool kSoftcap, bool kMetrics>
__device__ __forceinline__ void fwd_chunk(const uint32_t (&v)[32], const FwdArgs& a, int col0,
                                          long long tgt, int row, bool row_ok, float& m,
                                          float& ssum, float& tsum, int& amax) {
  float z[32];
  {
    float raw[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) raw[j] = __uint_as_float(v[j]);
    if (kBias) {
      float bs[32];
      load_bias32<T, kRagged>(static_cast<const T*>(a.bias), col0, a.V, a.scale, bs);
      fma_pairs(z, raw, a.scale, bs);       // (a + b) s, as fma(a, s, b s)
    } else {
      mul_pairs(z, raw, a.scale);
    }
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    if (kSoftcap) z[j] = a.softcap * tanh_via_exp2(z[j] * a.inv_softcap);
    if (kRagged && col0 + j >= a.V) z[j] = -INFINITY;
  }
  // The target logit lives in exactly one chunk of the whole vocabulary sweep.
  const long long rel = tgt - col0;
  if (row_ok && rel >= 0 && rel < 32) {
    const float zt = select32(z, static_cast<int>(rel));
    if (store_allowed(&a.zt[row], 4, a.r_zt, a.status)) a.zt[row] = zt;
  }
  const float cmax = tree_max32(z);
  const float mnew = fmaxf(m, cmax);
  if (kMetrics && cmax > m) {
    // strictly larger: an earlier chunk keeps a tie; within the chunk the
    // lowest index that attains the max
    int idx = 31;
#pragma unroll
    for (int j = 30; j >= 0; --j) idx = (z[j] == cmax) ? j : idx;
    amax = col0 + idx;
  }
  const float alpha = ex2_approx((m - mnew) * kLog2e);
  float e[32];
  fma_pairs(e, z, kLog2e, -mnew * kLog2e);
#pragma unroll
  for (int j = 0; j < 32; ++j) e[j] = ex2_approx(e[j]);
  if (kMetrics) {
    float ze[32];
    if (kRagged) {
      float zc[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) zc[j] = (col0 + j >= a.V) ? 0.f : z[j];
      mul_pairs(ze, zc, e);
    } else {
      mul_pairs(ze, z, e);
    }
    tsum = fmaf(tsum, alpha, tree_sum32(ze));
  }
  ssum = fmaf(ssum, alpha, tree_sum32(e));
  m = mnew;
}

// ==================================================== dynamic schedule
// Units handed out by an atomic counter instead of round-robin (the prior
// art's tile semaphore, quack diff, GemmWrapperBase): a pair that finishes
// early takes the next unit. Only the even CTA's producer thread touches the
// counter; it publishes each unit (or -1 when none is left) through a ring of
// kQueue shared-memory slots, written in both CTAs of the pair, and every
// other role of both CTAs reads the units from its own CTA's copy. A slot is
// reused only after all kQueueReaders readers have released it. Every wait
// is bounded (WaitGuard).
struct TileQueue {
  const TcSmem& s;
  const WaitGuard& g;
  uint32_t rank;
  int i = 0;   // units published or read so far

  // Even CTA's producer: the next unit, published to both CTAs; -1 when the
  // units are exhausted; -2 if a wait gave up.
  __device__ __forceinline__ int publish(int* counter, int units) {
    const int slot = i % kQueue;
    const uint32_t ph = static_cast<uint32_t>(i / kQueue) & 1u;
    if (!mbar_wait_cluster(&s.q_empty[slot], ph ^ 1u, g)) return -2;
    int u = atomicAdd(counter, 1);
    if (u >= units) u = -1;
    s.q_unit[slot] = u;
    st_shared_cluster_u32(mapa_shared(smem_u32(&s.q_unit[slot]), 1), static_cast<uint32_t>(u));
    mbar_arrive(&s.q_full[slot]);
    mbar_arrive_cluster(mapa_shared(smem_u32(&s.q_full[slot]), 1));
    ++i;
    return u;
  }

  // Any other role: the next unit from this CTA's slot (-1: none left, -2: a
  // wait gave up). Each reader then calls release() once it has the value;
  // in a warp that reads together, one lane releases after a __syncwarp.
  __device__ __forceinline__ int read() {
    const int slot = i % kQueue;
    const uint32_t ph = static_cast<uint32_t>(i / kQueue) & 1u;
    const bool ok = rank == 0 ? mbar_wait(&s.q_full[slot], ph, g)
                              : mbar_wait_cluster(&s.q_full[slot], ph, g);
    if (!ok) return -2;
    return *reinterpret_cast<volatile int*>(&s.q_unit[slot]);
  }
  __device__ __forceinline__ void release() {
    const int slot = i % kQueue;
    if (rank == 0)
      mbar_arrive(&s.q_empty[slot]);
    else
      mbar_arrive_cluster(mapa_shared(smem_u32(&s.q_empty[slot]), 0));
    ++i;
  }
};

template <typename T, bool kBias, bool kSoftcap, bool kMetrics>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kTcThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w,
                  const FwdArgs a) {
  const ClockStart clock_start(a.clk);
  extern __shared__ uint8_t smem_raw[];
  const TcSmem s = carve_smem(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t tmem = tc_setup(s, warp);
  const uint32_t rank = cluster_ctarank();  // 0: even CTA (issues the MMAs), 1: odd CTA
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const WaitGuard g{a.status, s.abort, a.wait_ns};
  const int kblocks = (a.H + kBK - 1) / kBK;

  // Units (panel, pair block) round-robin, or with a tile counter from the
  // dynamic schedule: the even CTA's producer takes them off the counter and
  // every other role reads them from the queue, in the same order. Taken in
  // order, the units in flight stay a window of consecutive units, so the
  // pairs keep working on the same few W panels however far apart their
  // progress drifts.
  const bool dynamic = a.tile_counter != nullptr;
  auto for_each_unit = [&](auto&& f) {
    if (!dynamic) {
      for (int u = pair; u < a.num_units; u += npairs) f(u);
      return;
    }
    TileQueue q{s, g, rank};
    if (warp == 0 && rank == 0) {
      while (true) {
        const int u = q.publish(a.tile_counter, a.num_units);
        if (u == -1) {
          // the last pair to run out leaves the counters at zero for the next launch
          if (atomicAdd(a.tile_counter + 1, 1) == npairs - 1) {
            a.tile_counter[0] = 0;
            a.tile_counter[1] = 0;
          }
        }
        if (u < 0) return;
        f(u);
      }
    }
    while (true) {   // the odd CTA's producer, or the MMA thread
      const int u = q.read();
      if (u == -2) return;
      q.release();
      if (u < 0) return;
      f(u);
    }
  };
  auto for_each_tile = [&](auto&& f) {
    for_each_unit([&](int u) {
      int panel, nb;
      decode_unit(u, a.n_blocks, a.group_blocks, a.num_panels, panel, nb);
      const int vt0 = panel * a.panel_tiles;
      const int vt1 = min(a.v_tiles, vt0 + a.panel_tiles);
      for (int vt = vt0; vt < vt1; ++vt) f(nb, vt);
    });
  };

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_h);
      tma_prefetch_desc(&tm_w);
      const uint64_t pol_h = l2_policy_evict_last();
      const uint64_t pol_w = l2_policy_evict_normal();
      producer_role(s, g, [&](int, int) { return kblocks; }, rank == 0, for_each_tile,
                    [&](int nb, int vt, int kb, uint8_t* da, uint8_t* db, uint32_t bar) {
                      // Fault injection for the bounded-wait test: the stage is armed
                      // but its loads never come, so the MMA's wait must time out.
                      // (nb, vt) = (0, 0) is the first tile of unit 0.
                      if (kb == a.drop_kb && rank == 0 && nb == 0 && vt == 0) return;
                      tma_load_2d_pair(da, &tm_h, bar, kb * kBK, nb * kPairM + rank * kBM, pol_h);
                      tma_load_2d_pair(db, &tm_w, bar, kb * kBK, vt * kBN + rank * kBNHalf, pol_w);
                    });
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0)
      mma_role(s, g, tmem, [&](int, int) { return kblocks; }, for_each_tile, kmajor_descs<T>,
               a.clk);
  } else {
    const int q = warp & 3;
    const int r = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool dead = false;
    auto unit_epilogue = [&](int u) {
      int panel, nb;
      decode_unit(u, a.n_blocks, a.group_blocks, a.num_panels, panel, nb);
      const int row = nb * kPairM + static_cast<int>(rank) * kBM + r;
      const bool row_ok = row < a.N;
      // shard-local target id; an ignored row gets one that never matches a column
      long long tgt = row_ok ? a.targets[row] : a.ignore_index;
      tgt = (tgt == a.ignore_index) ? -(1ll << 40) : tgt - a.vocab_start;
      float m = -INFINITY, ssum = 0.f, tsum = 0.f;
      int amax = 0;
      const int vt0 = panel * a.panel_tiles;
      const int vt1 = min(a.v_tiles, vt0 + a.panel_tiles);
      for (int vt = vt0; vt < vt1; ++vt) {
        dead = !epi_wait_full(s, acc, acc_phase, g, dead);
        if (!dead) {
          const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) +
                                 static_cast<uint32_t>(acc * kBN);
          const bool ragged = (vt + 1) * kBN > a.V;
#pragma unroll 1
          for (int c = 0; c < kBN / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(tbase + c * 32, v);
            tmem_ld_wait(v);
            const int col0 = vt * kBN + c * 32;
            if (!ragged) {
              fwd_chunk<T, false, kBias, kSoftcap, kMetrics>(v, a, col0, tgt, row, row_ok, m, ssum, tsum,
                                                   amax);
            } else if (col0 < a.V) {
              fwd_chunk<T, true, kBias, kSoftcap, kMetrics>(v, a, col0, tgt, row, row_ok, m, ssum, tsum,
                                                  amax);
            }
          }
          epi_release(s, acc, lane);
        }
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      float4* const dst = a.partials + static_cast<size_t>(panel) * a.N + row;
      if (row_ok && !dead && store_allowed(dst, 16, a.r_partials, a.status))
        *dst = make_float4(m, ssum, tsum, __int_as_float(amax));
    };
    if (!dynamic) {
      for (int u = pair; u < a.num_units; u += npairs) unit_epilogue(u);
    } else {
      TileQueue q{s, g, rank};
      while (true) {
        const int u = q.read();   // the same value in every lane that got one
        if (!__all_sync(kFull, u != -2)) break;
        __syncwarp();
        if (lane == 0) q.release();
        else ++q.i;
        if (u < 0) break;
        unit_epilogue(u);
      }
    }
  }
  tc_teardown(tmem, warp);
  clock_start.finish(a.clk);
}

// ====================================================== dlogits kernel
__device__ __forceinline__ float warp_transpose_sum32(float (&x)[32], int lane) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int k = 0; k < off; ++k) {
      const float send = upper ? x[k] : x[k + off];
      const float keep = upper ? x[k + off] : x[k];
      x[k] = keep + __shfl_xor_sync(kFull, send, off);
    }
  }
  return x[0];  // lane L now holds the sum of column L over the warp's 32 rows
}

template <typename T, bool kRagged, bool kBias, bool kSoftcap>
__device__ __forceinline__ void ds_chunk(const uint32_t (&v)[32], const DsArgs& a, int col0,
                                         float4 cf, bool row_ok, float (&gout)[32]) {
  float bs[32];
  if (kBias) load_bias32<T, kRagged>(static_cast<const T*>(a.bias), col0, a.V, a.scale, bs);
  const int tgt = __float_as_int(cf.w) - a.tgt_base;  // no target (-1) stays negative
  const float nlse = -cf.z * kLog2e;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float z = transform<kBias, kSoftcap>(v[j], kBias ? bs[j] : 0.f, a.scale, a.softcap,
                                               a.inv_softcap);
    const float p = ex2_approx(fmaf(z, kLog2e, nlse));
    float gj = cf.x * p;
    if (col0 + j == tgt) gj -= cf.y;
    if (kSoftcap) {
      const float zc = z * a.inv_softcap;
      gj *= fmaf(-zc, zc, 1.f);
    }
    if (kRagged && col0 + j >= a.V) gj = 0.f;
    gout[j] = row_ok ? gj : 0.f;
  }
}

// 32 values of one row times mul, as 16 words of two neighbouring columns
// in the element type: word i holds columns 2i (low half) and 2i + 1.
template <typename T>
__device__ __forceinline__ void pack32(const float (&g)[32], float mul, uint32_t (&w)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i] = Elem<T>::pack(g[2 * i] * mul, g[2 * i + 1] * mul);
}

// One row's 32 packed columns, row-major, as four 16-byte pieces; a piece is
// written if its first column is below `cols` (the padding up to the next
// multiple of 8 columns receives the packed zeros).
template <typename T>
__device__ __forceinline__ void store_row_packed(const uint32_t (&w)[16], T* dst, int col0,
                                                 int cols, const DevRegion& r, int* status) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    if (col0 + q * 8 < cols && store_allowed(dst + q * 8, 16, r, status))
      *reinterpret_cast<uint4*>(dst + q * 8) =
          make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
}

// Stores a warp's 32 rows x 32 columns, packed by pack32, transposed: row c
// of dst_t holds column c for every row. Lanes 2k and 2k + 1 (rows row_w + 2k
// and row_w + 2k + 1) swap their word of columns (2i, 2i + 1); a byte
// permute then gives the even lane the word of column 2i for both rows and
// the odd lane that of column 2i + 1, so a warp store covers 64 contiguous
// bytes of two dst_t rows. Rows >= rows and columns >= cols are not written
// (a pair whose first row is below `rows` is written whole; ld_t must be
// even). All 32 lanes must call it (it shuffles).
template <typename T>
__device__ __forceinline__ void store_transposed_packed(const uint32_t (&w)[16], T* dst_t,
                                                        long long ld_t, int col0, int row_w,
                                                        int lane, int rows, int cols, bool live,
                                                        const DevRegion& r, int* status) {
  const bool odd = (lane & 1) != 0;
  const int row_pair = row_w + (lane & ~1);  // the first of this lane's two rows
  // even lane: (own low half, partner's low half); odd: (partner's high, own high)
  const uint32_t sel = odd ? 0x3276u : 0x5410u;
  const int c_first = col0 + (odd ? 1 : 0);
  T* const base = dst_t + static_cast<size_t>(c_first) * ld_t + row_pair;
  const size_t step = 2 * static_cast<size_t>(ld_t);
  // warp-uniform: the whole 32 x 32 block is inside
  const bool inside = live && row_w + 32 <= rows && col0 + 32 <= cols;
  const bool row_in = live && row_pair < rows;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t recv = __shfl_xor_sync(kFull, w[i], 1);
    const uint32_t out = __byte_perm(w[i], recv, sel);
    if ((inside || (row_in && c_first + 2 * i < cols)) &&
        store_allowed(base + i * step, 4, r, status))
      *reinterpret_cast<uint32_t*>(base + i * step) = out;
  }
}

// Adds a warp's 32 rows x 32 fp32 columns, transposed, into dst_t (16-bit):
// the layout and bounds of store_transposed_packed, with the lane pairs
// exchanging fp32 values so that each existing value is read, added to in
// fp32 and rounded once. All 32 lanes must call it (it shuffles).
template <typename T>
__device__ __forceinline__ void add_transposed(const float (&d)[32], T* dst_t, long long ld_t,
                                               int col0, int row_w, int lane, int rows, int cols,
                                               bool live, const DevRegion& r, int* status) {
  const bool odd = (lane & 1) != 0;
  const int row_pair = row_w + (lane & ~1);
  const int c_first = col0 + (odd ? 1 : 0);
  T* const base = dst_t + static_cast<size_t>(c_first) * ld_t + row_pair;
  const size_t step = 2 * static_cast<size_t>(ld_t);
  const bool inside = live && row_w + 32 <= rows && col0 + 32 <= cols;
  const bool row_in = live && row_pair < rows;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    // even lane: column 2i of rows (own, partner); odd lane: column 2i + 1 of
    // rows (partner, own)
    const float recv = __shfl_xor_sync(kFull, odd ? d[2 * i] : d[2 * i + 1], 1);
    const float lo = odd ? recv : d[2 * i];
    const float hi = odd ? d[2 * i + 1] : recv;
    T* const p = base + i * step;
    if ((inside || (row_in && c_first + 2 * i < cols)) && store_allowed(p, 4, r, status)) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
      *reinterpret_cast<uint32_t*>(p) = Elem<T>::pack(Elem<T>::lo(w) + lo, Elem<T>::hi(w) + hi);
    }
  }
}

template <typename T, bool kBias, bool kSoftcap>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kDsThreads, 1)
    ds_tc_kernel(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w,
                 const DsArgs a) {
  const ClockStart clock_start(a.clk);
  extern __shared__ uint8_t smem_raw[];
  const TcSmem s = carve_smem(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t tmem = tc_setup(s, warp, 8, kDsQueueReaders);
  const uint32_t rank = cluster_ctarank();  // 0: even CTA (issues the MMAs), 1: odd CTA
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const WaitGuard g{a.status, s.abort};
  const int kblocks = (a.H + kBK - 1) / kBK;

  // Units round-robin, or in order from the dynamic schedule, as in the
  // forward kernel.
  const bool dynamic = a.tile_counter != nullptr;
  auto for_each_unit = [&](auto&& f) {
    if (!dynamic) {
      for (int u = pair; u < a.num_units; u += npairs) f(u);
      return;
    }
    TileQueue q{s, g, rank};
    if (warp == 0 && rank == 0) {
      while (true) {
        const int u = q.publish(a.tile_counter, a.num_units);
        if (u == -1) {
          // the last pair to run out leaves the counters at zero for the next launch
          if (atomicAdd(a.tile_counter + 1, 1) == npairs - 1) {
            a.tile_counter[0] = 0;
            a.tile_counter[1] = 0;
          }
        }
        if (u < 0) return;
        f(u);
      }
    }
    while (true) {   // the odd CTA's producer, or the MMA thread
      const int u = q.read();
      if (u == -2) return;
      q.release();
      if (u < 0) return;
      f(u);
    }
  };
  auto for_each_tile = [&](auto&& f) {
    for_each_unit([&](int u) {
      int panel, nb;
      decode_unit(u, a.n_blocks, a.group_blocks, a.num_panels, panel, nb);
      const int vt0 = panel * a.panel_tiles;
      const int vt1 = min(a.v_tiles, vt0 + a.panel_tiles);
      for (int vt = vt0; vt < vt1; ++vt) f(nb, vt);
    });
  };

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_h);
      tma_prefetch_desc(&tm_w);
      const uint64_t pol_h = l2_policy_evict_last();
      const uint64_t pol_w = l2_policy_evict_normal();
      producer_role(s, g, [&](int, int) { return kblocks; }, rank == 0, for_each_tile,
                    [&](int nb, int vt, int kb, uint8_t* da, uint8_t* db, uint32_t bar) {
                      tma_load_2d_pair(da, &tm_h, bar, kb * kBK,
                                       a.row0 + nb * kPairM + rank * kBM, pol_h);
                      tma_load_2d_pair(db, &tm_w, bar, kb * kBK, vt * kBN + rank * kBNHalf, pol_w);
                    });
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0)
      mma_role(s, g, tmem, [&](int, int) { return kblocks; }, for_each_tile, kmajor_descs<T>,
               a.clk);
  } else {
    // warps 2-5 take columns 0-127 of each tile, warps 6-9 columns 128-255
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = q * 32 + lane;
    const int et = threadIdx.x - 64;  // 0..255
    const float ds_mul = a.ds_scale != nullptr ? *a.ds_scale : 1.f;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool dead = false;
    int tile_par = 0;
    auto unit_epilogue = [&](int u) {
      int panel, nb;
      decode_unit(u, a.n_blocks, a.group_blocks, a.num_panels, panel, nb);
      const int blk_local = nb * 2 + static_cast<int>(rank);  // this CTA's 128-row block
      const int row_local = blk_local * kBM + r;
      const bool row_ok = row_local < a.rows;
      const bool blk_ok = blk_local * kBM < a.rows;
      const float4 cf = row_ok ? a.coef[a.row0 + row_local] : make_float4(0.f, 0.f, 0.f, __int_as_float(-1));
      const int vt0 = panel * a.panel_tiles;
      const int vt1 = min(a.v_tiles, vt0 + a.panel_tiles);
      for (int vt = vt0; vt < vt1; ++vt) {
        float* colsum = s.scratch + tile_par * (4 * kBN);
        dead = !epi_wait_full(s, acc, acc_phase, g, dead);
        const bool ragged = (vt + 1) * kBN > a.V;
#pragma unroll 1
        for (int cc = 0; cc < kBN / 64; ++cc) {
          const int c = half * (kBN / 64) + cc;
          float gv[32];
          const int col0 = vt * kBN + c * 32;
          if (!dead) {
            uint32_t v[32];
            tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) +
                          static_cast<uint32_t>(acc * kBN + c * 32),
                      v);
            tmem_ld_wait(v);
            if (!ragged) {
              ds_chunk<T, false, kBias, kSoftcap>(v, a, col0, cf, row_ok, gv);
            } else if (col0 < a.V) {
              ds_chunk<T, true, kBias, kSoftcap>(v, a, col0, cf, row_ok, gv);
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) gv[j] = 0.f;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) gv[j] = 0.f;
          }
          // dlogits in the input type, packed once for both layouts. fp16
          // stores dlogits times a power of two (ds_mul), which keeps the
          // small probabilities out of the fp16 subnormal range; the GEMMs
          // undo it exactly. bf16 is stored unscaled.
          uint32_t w[16];
          pack32<T>(gv, Elem<T>::kBf16 ? 1.f : ds_mul, w);
          if (!dead && row_ok && col0 < a.V) {
            T* const row = static_cast<T*>(a.ds) + static_cast<size_t>(row_local) * a.V_pad;
            store_row_packed<T>(w, row + col0, col0, a.V, a.r_ds, a.status);
          }
          if (a.ds_t != nullptr)
            store_transposed_packed<T>(w, static_cast<T*>(a.ds_t), a.ld_t, col0, row_local - lane,
                                       lane, a.rows, a.V, !dead, a.r_ds_t, a.status);
          if (a.bias_part != nullptr) {
            const float cs = warp_transpose_sum32(gv, lane);
            colsum[q * kBN + c * 32 + lane] = cs;
          }
        }
        if (!dead) epi_release(s, acc, lane);
        if (a.bias_part != nullptr) {
          // Every epilogue thread reaches this barrier once per tile, also
          // after an abort, so the barrier cannot hang.
          named_barrier(1, 256);
          const int j = et;
          const int col = vt * kBN + j;
          if (col < a.V && blk_ok) {
            const float t = ((colsum[j] + colsum[kBN + j]) + colsum[2 * kBN + j]) +
                            colsum[3 * kBN + j];
            float* const dst = a.bias_part + static_cast<size_t>(a.bias_blk0 + blk_local) * a.bias_ld + col;
            if (store_allowed(dst, 4, a.r_bias, a.status)) *dst = t;
          }
        }
        tile_par ^= 1;
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
    };
    if (!dynamic) {
      for (int u = pair; u < a.num_units; u += npairs) unit_epilogue(u);
    } else {
      // Warp 2 reads the queue for this CTA's eight epilogue warps and passes
      // each unit (or the end: -1, or -2 after a wait gave up) through
      // alternating shared slots, so that all eight stop at the same unit and
      // the per-tile barrier of the bias sums stays balanced. A slot is
      // rewritten two units later, after every warp has passed the barrier
      // that follows its read of the unit in between.
      TileQueue q{s, g, rank};
      for (int it = 0;; ++it) {
        if (warp == 2) {
          int u = q.read();
          u = __all_sync(kFull, u != -2) ? u : -2;
          __syncwarp();
          if (u != -2) {
            if (lane == 0) q.release();
            else ++q.i;
          }
          if (lane == 0) s.ep_unit[it & 1] = u;
        }
        named_barrier(2, 256);
        const int u = *reinterpret_cast<volatile int*>(&s.ep_unit[it & 1]);
        if (u < 0) break;
        unit_epilogue(u);
      }
    }
  }
  tc_teardown(tmem, warp);
  clock_start.finish(a.clk);
}


// ========================================================= plain GEMM
// D = A B with fp32 accumulation; the two gradient contractions. Units
// (split, tile) go round-robin over the pairs: consecutive units are
// neighbouring tiles of the same K range, which share an operand strip in L2.
// Tiles are rastered in groups of `group_m` row tiles, column after column
// within a group (decode_unit), so that with many column tiles the group's
// A strips stay in L2 while each B strip is read once per group.
// The arguments are copied into registers up front; the role loops read no
// kernel parameters.
template <typename T, bool kMse>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kTcThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const __grid_constant__ CUtensorMap tm_a3,
                   const __grid_constant__ CUtensorMap tm_b3, const GemmArgs a) {
  const ClockStart clock_start(a.clk);
  extern __shared__ uint8_t smem_raw[];
  const TcSmem s = carve_smem(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t tmem = tc_setup(s, warp);
  const uint32_t rank = cluster_ctarank();  // 0: even CTA (issues the MMAs), 1: odd CTA
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const WaitGuard g{a.status, s.abort};
  const int M = a.M, N = a.N, n_tiles = a.n_tiles, num_tiles = a.num_tiles;
  const int m_tiles = a.m_tiles, group_m = a.group_m;
  const int k_blocks = a.k_blocks, kb_per_split = a.kb_per_split;
  const int units = num_tiles * a.k_splits;
  const bool a_mn = a.a_mn != 0, b_mn = a.b_mn != 0;
  const int a_atoms = a.a_atoms, b_atoms = a.b_atoms;

  // Every unit of this pair as (row tile << 8 | split, column tile), decoded
  // once per tile: the per-stage work of the single producer thread stays
  // free of divisions. Splits number at most 255 (the host uses at most 2).
  // With a tile counter the units come from the dynamic schedule (TileQueue):
  // the even CTA's producer takes them off the counter and every other role
  // reads them from the queue, in the same order.
  const bool dynamic = a.tile_counter != nullptr;
  auto decode = [&](int u, int& ta, int& nt) {
    const int sp = u / num_tiles;
    int mt;
    decode_unit(u - sp * num_tiles, m_tiles, group_m, n_tiles, nt, mt);
    ta = (mt << 8) | sp;
  };
  auto for_each_tile = [&](auto&& f) {
    int ta, nt;
    if (!dynamic) {
      for (int u = pair; u < units; u += npairs) {
        decode(u, ta, nt);
        f(ta, nt);
      }
      return;
    }
    TileQueue q{s, g, rank};
    if (warp == 0 && rank == 0) {
      while (true) {
        const int u = q.publish(a.tile_counter, units);
        if (u == -1) {
          // the last pair to run out leaves the counters at zero for the next launch
          if (atomicAdd(a.tile_counter + 1, 1) == npairs - 1) {
            a.tile_counter[0] = 0;
            a.tile_counter[1] = 0;
          }
        }
        if (u < 0) return;
        decode(u, ta, nt);
        f(ta, nt);
      }
    }
    while (true) {   // the odd CTA's producer, or the MMA thread
      const int u = q.read();
      if (u == -2) return;
      q.release();
      if (u < 0) return;
      decode(u, ta, nt);
      f(ta, nt);
    }
  };
  auto kblocks_of = [&](int ta, int) {
    const int sp = ta & 255;
    return min(k_blocks, (sp + 1) * kb_per_split) - sp * kb_per_split;
  };

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_a);
      tma_prefetch_desc(&tm_b);
      if (a_atoms > 0) tma_prefetch_desc(&tm_a3);
      if (b_atoms > 0) tma_prefetch_desc(&tm_b3);
      auto policy = [](int k) {
        return k == kL2EvictFirst ? l2_policy_evict_first()
               : k == kL2EvictLast ? l2_policy_evict_last()
                                   : l2_policy_evict_normal();
      };
      const uint64_t pol_a = policy(a.a_l2), pol_b = policy(a.b_l2);
      const int m_off = static_cast<int>(rank) * kBM, n_off = static_cast<int>(rank) * kBNHalf;
      producer_role(s, g, kblocks_of, rank == 0, for_each_tile,
                    [&](int ta, int nt, int kb_rel, uint8_t* da, uint8_t* db, uint32_t bar) {
                      const int sp = ta & 255, mt = ta >> 8;
                      const int m0 = mt * kPairM + m_off, n0 = nt * kBN + n_off;
                      const int k0 = (sp * kb_per_split + kb_rel) * kBK;
                      if (a_mn) {
                        // [K rows][M cols] in memory: the atoms m0/64 and m0/64 + 1 cover
                        // this CTA's 128 rows of M, one 64 x 64 box each
                        const int at = m0 >> 6;
                        if (at + 2 <= a_atoms) {
                          tma_load_3d_pair(da, &tm_a3, bar, 0, k0, at, pol_a);
                        } else {
                          tma_load_2d_pair(da, &tm_a, bar, m0, k0, pol_a);
                          tma_load_2d_pair(da + 8192, &tm_a, bar, m0 + 64, k0, pol_a);
                        }
                      } else {
                        tma_load_2d_pair(da, &tm_a, bar, k0, m0, pol_a);
                      }
                      if (b_mn) {
                        // [K rows][N cols] in memory: two atoms cover this CTA's 128 columns
                        const int at = n0 >> 6;
                        if (at + 2 <= b_atoms) {
                          tma_load_3d_pair(db, &tm_b3, bar, 0, k0, at, pol_b);
                        } else {
                          tma_load_2d_pair(db, &tm_b, bar, n0, k0, pol_b);
                          tma_load_2d_pair(db + 8192, &tm_b, bar, n0 + 64, k0, pol_b);
                        }
                      } else {
                        tma_load_2d_pair(db, &tm_b, bar, k0, n0, pol_b);
                      }
                    });
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      const uint32_t id = idesc_f16kind_f32(kPairM, kBN, a_mn, b_mn, Elem<T>::kBf16);
      mma_role(s, g, tmem, kblocks_of, for_each_tile,
               [&](int, int, uint32_t sa, uint32_t sb, int kk, uint64_t& ad, uint64_t& bd,
                   uint32_t& idesc) {
                 ad = operand_desc(sa, a_mn, kk);
                 bd = operand_desc(sb, b_mn, kk);
                 idesc = id;
               },
               a.clk);
    }
  } else {
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int mode0 = a.k_splits > 1 ? static_cast<int>(kStorePart) : a.mode;
    const bool add_part = mode0 == kAddPart || mode0 == kAddPartToOut;
    const bool add_out = mode0 == kAddOutToOut || mode0 == kAddOutToPart;
    const bool to_part = mode0 == kStorePart || mode0 == kAddPart || mode0 == kAddOutToPart;
    const bool t_only = mode0 == kStoreOutT || mode0 == kAddOutToOutT || mode0 == kAddPartToOutT;
    constexpr bool mse = kMse;  // the kWeightedMse epilogue is its own instantiation
    const float* const tgt = a.target;
    const float* const feat = a.feat_w;
    const long long ld_target = a.ld_target;
    float* const part0 = a.part;
    const long long ld_part = a.ld_part, split_stride = a.split_stride, ld_out = a.ld_out;
    T* const out = static_cast<T*>(a.out);
    const float acc_mul = a.acc_scale != nullptr ? *a.acc_scale : 1.f;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool dead = false;
    auto unit_epilogue = [&](int u) {
      const int sp = u / num_tiles, t = u - sp * num_tiles;
      int mt, nt;
      decode_unit(t, m_tiles, group_m, n_tiles, nt, mt);
      float* const part = part0 + static_cast<size_t>(sp) * split_stride;
      dead = !epi_wait_full(s, acc, acc_phase, g, dead);
      if (!dead) {
        const int m = mt * kPairM + static_cast<int>(rank) * kBM + r;
        const bool row_ok = m < M;
        const float rm = (mse && row_ok) ? a.row_w[m] : 0.f;
        float lsum = 0.f;
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) +
                        static_cast<uint32_t>(acc * kBN + c * 32),
                    v);
          tmem_ld_wait(v);
          const int col0 = nt * kBN + c * 32;
          // The loss epilogue and the transposed store keep every lane of a
          // warp (the transposed store shuffles); a row past M has zero logits
          // and zero weight there.
          if ((mse || t_only) ? col0 >= N : (!row_ok || col0 >= N)) continue;
          float d[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) d[j] = __uint_as_float(v[j]) * acc_mul;
          if (!mse && t_only) {
            if (mode0 == kAddPartToOutT && row_ok) {
              const float4* src =
                  reinterpret_cast<const float4*>(part + static_cast<size_t>(m) * ld_part + col0);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                if (col0 + i * 4 < N) {
                  const float4 p4 = src[i];
                  d[4 * i] += p4.x;
                  d[4 * i + 1] += p4.y;
                  d[4 * i + 2] += p4.z;
                  d[4 * i + 3] += p4.w;
                }
              }
            }
            if (mode0 == kAddOutToOutT) {
              add_transposed<T>(d, static_cast<T*>(a.out_t), a.ld_out_t, col0, m - lane, lane, M, N,
                                true, a.r_out_t, a.status);
            } else {
              uint32_t w[16];
              pack32<T>(d, 1.f, w);
              store_transposed_packed<T>(w, static_cast<T*>(a.out_t), a.ld_out_t, col0, m - lane,
                                         lane, M, N, true, a.r_out_t, a.status);
            }
            continue;
          }
          if (mse) {
            // d holds the logits z of this row's 32 columns; they become
            // 2 r f (z - y), and r f (z - y)^2 goes into the row's loss.
            float y[32], f[32];
            const float* yrow = tgt + static_cast<size_t>(row_ok ? m : 0) * ld_target + col0;
            if (col0 + 32 <= N) {
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float4 y4 = row_ok ? reinterpret_cast<const float4*>(yrow)[i]
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
                const float4 f4 = __ldg(reinterpret_cast<const float4*>(feat + col0) + i);
                y[4 * i] = y4.x; y[4 * i + 1] = y4.y; y[4 * i + 2] = y4.z; y[4 * i + 3] = y4.w;
                f[4 * i] = f4.x; f[4 * i + 1] = f4.y; f[4 * i + 2] = f4.z; f[4 * i + 3] = f4.w;
              }
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const bool in = col0 + j < N;
                y[j] = (in && row_ok) ? yrow[j] : 0.f;
                f[j] = in ? feat[col0 + j] : 0.f;
              }
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float e = d[j] - y[j];
              const float we = rm * f[j] * e;
              lsum = fmaf(we, e, lsum);
              d[j] = 2.f * we;
            }
            uint32_t w[16];
            pack32<T>(d, 1.f, w);
            if (a.out_t != nullptr)
              store_transposed_packed<T>(w, static_cast<T*>(a.out_t), a.ld_out_t, col0, m - lane,
                                         lane, M, N, true, a.r_out_t, a.status);
            if (row_ok)
              store_row_packed<T>(w, out + static_cast<size_t>(m) * ld_out + col0, col0, N, a.r_out,
                                  a.status);
            continue;
          }
          if (add_part) {
            const float4* src =
                reinterpret_cast<const float4*>(part + static_cast<size_t>(m) * ld_part + col0);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              if (col0 + i * 4 < N) {
                const float4 p4 = src[i];
                d[4 * i] += p4.x;
                d[4 * i + 1] += p4.y;
                d[4 * i + 2] += p4.z;
                d[4 * i + 3] += p4.w;
              }
            }
          }
          if (add_out) {
            const uint4* src = reinterpret_cast<const uint4*>(out + static_cast<size_t>(m) * ld_out + col0);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              if (col0 + i * 8 < N) {
                const uint4 w = src[i];
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                  d[8 * i + 2 * h] += Elem<T>::lo(ws[h]);
                  d[8 * i + 2 * h + 1] += Elem<T>::hi(ws[h]);
                }
              }
            }
          }
          if (to_part) {
            float4* dst = reinterpret_cast<float4*>(part + static_cast<size_t>(m) * ld_part + col0);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if (col0 + i * 4 < N)
                if (store_allowed(dst + i, 16, a.r_part, a.status))
                  dst[i] = make_float4(d[4 * i], d[4 * i + 1], d[4 * i + 2], d[4 * i + 3]);
          } else {
            T* dst = out + static_cast<size_t>(m) * ld_out + col0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              if (col0 + i * 8 < N) {
                uint4 w;
                w.x = Elem<T>::pack(d[8 * i + 0], d[8 * i + 1]);
                w.y = Elem<T>::pack(d[8 * i + 2], d[8 * i + 3]);
                w.z = Elem<T>::pack(d[8 * i + 4], d[8 * i + 5]);
                w.w = Elem<T>::pack(d[8 * i + 6], d[8 * i + 7]);
                if (store_allowed(dst + i * 8, 16, a.r_out, a.status))
                  *reinterpret_cast<uint4*>(dst + i * 8) = w;
              }
            }
          }
        }
        if (mse) {
          // the warp's 32 rows summed by a fixed shuffle tree: one partial per
          // (column tile, 32-row group)
          float t = row_ok ? lsum : 0.f;
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1) t += __shfl_xor_sync(kFull, t, o);
          const int m_base = m - lane;
          if (lane == 0 && m_base < M) {
            float* const dst = a.loss_part + static_cast<size_t>(nt) * ((M + 31) / 32) + (m_base >> 5);
            if (store_allowed(dst, 4, a.r_loss, a.status)) *dst = t;
          }
        }
        epi_release(s, acc, lane);
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    };
    if (!dynamic) {
      for (int u = pair; u < units; u += npairs) unit_epilogue(u);
    } else {
      TileQueue q{s, g, rank};
      while (true) {
        const int u = q.read();   // the same value in every lane that got one
        if (!__all_sync(kFull, u != -2)) break;
        __syncwarp();
        if (lane == 0) q.release();
        else ++q.i;
        if (u < 0) break;
        unit_epilogue(u);
      }
    }
  }
  tc_teardown(tmem, warp);
  clock_start.finish(a.clk);
}

template <class K>
cudaError_t set_smem_attr(K kernel) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemBytes);
}

}  // namespace

cudaError_t tc_max_active_pairs(int* pairs) {
  auto k = fwd_tc_kernel<__nv_bfloat16, false, false, false>;
  cudaError_t e = set_smem_attr(k);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kTcThreads, 1, 1);
  cfg.dynamicSmemBytes = kTcSmemBytes;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, k, &cfg);
  if (e != cudaSuccess) return e;
  *pairs = n;
  return cudaSuccess;
}

namespace {
template <typename T, bool kMetrics>
cudaError_t launch_fwd_t(const CUtensorMap& tm_h, const CUtensorMap& tm_w, const FwdArgs& a,
                         bool has_bias, bool softcap, int grid, cudaStream_t st) {
  auto k = has_bias ? (softcap ? fwd_tc_kernel<T, true, true, kMetrics>
                               : fwd_tc_kernel<T, true, false, kMetrics>)
                    : (softcap ? fwd_tc_kernel<T, false, true, kMetrics>
                               : fwd_tc_kernel<T, false, false, kMetrics>);
  cudaError_t e = set_smem_attr(k);
  if (e != cudaSuccess) return e;
  k<<<2 * grid, kTcThreads, kTcSmemBytes, st>>>(tm_h, tm_w, a);
  note_launch();
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_ds_t(const CUtensorMap& tm_h, const CUtensorMap& tm_w, const DsArgs& a,
                        bool has_bias, bool softcap, int grid, cudaStream_t st) {
  auto k = has_bias ? (softcap ? ds_tc_kernel<T, true, true> : ds_tc_kernel<T, true, false>)
                    : (softcap ? ds_tc_kernel<T, false, true> : ds_tc_kernel<T, false, false>);
  cudaError_t e = set_smem_attr(k);
  if (e != cudaSuccess) return e;
  k<<<2 * grid, kDsThreads, kTcSmemBytes, st>>>(tm_h, tm_w, a);
  note_launch();
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_gemm_t(const GemmOperand& op_a, const GemmOperand& op_b, const GemmArgs& a,
                          int grid, cudaStream_t st) {
  auto k = a.mode == kWeightedMse ? gemm_tc_kernel<T, true> : gemm_tc_kernel<T, false>;
  cudaError_t e = set_smem_attr(k);
  if (e != cudaSuccess) return e;
  k<<<2 * grid, kTcThreads, kTcSmemBytes, st>>>(op_a.map, op_b.map, op_a.map3, op_b.map3, a);
  note_launch();
  return cudaGetLastError();
}
}  // namespace

// `grid` counts CTA pairs; the launch has 2 * grid CTAs.
cudaError_t launch_fwd_tc(const CUtensorMap& tm_h, const CUtensorMap& tm_w, const FwdArgs& a,
                          bool f16, bool has_bias, bool softcap, bool metrics, int grid,
                          cudaStream_t st) {
  if (metrics)
    return f16 ? launch_fwd_t<__half, true>(tm_h, tm_w, a, has_bias, softcap, grid, st)
               : launch_fwd_t<__nv_bfloat16, true>(tm_h, tm_w, a, has_bias, softcap, grid, st);
  return f16 ? launch_fwd_t<__half, false>(tm_h, tm_w, a, has_bias, softcap, grid, st)
             : launch_fwd_t<__nv_bfloat16, false>(tm_h, tm_w, a, has_bias, softcap, grid, st);
}

cudaError_t launch_ds_tc(const CUtensorMap& tm_h, const CUtensorMap& tm_w, const DsArgs& a,
                         bool f16, bool has_bias, bool softcap, int grid, cudaStream_t st) {
  return f16 ? launch_ds_t<__half>(tm_h, tm_w, a, has_bias, softcap, grid, st)
             : launch_ds_t<__nv_bfloat16>(tm_h, tm_w, a, has_bias, softcap, grid, st);
}

cudaError_t launch_gemm_tc(const GemmOperand& op_a, const GemmOperand& op_b, const GemmArgs& a,
                           bool f16, int grid, cudaStream_t st) {
  if (a.group_m < 1 || a.m_tiles < 1 || a.n_tiles < 1 || a.k_splits < 1 || a.k_splits > 255 ||
      a.m_tiles > (1 << 22))
    return cudaErrorInvalidValue;
  return f16 ? launch_gemm_t<__half>(op_a, op_b, a, grid, st)
             : launch_gemm_t<__nv_bfloat16>(op_a, op_b, a, grid, st);
}

}  // namespace flce
