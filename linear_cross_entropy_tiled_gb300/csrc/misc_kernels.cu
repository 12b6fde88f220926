// Small kernels shared by both dtypes:
//   merge       per-row merge of the vocabulary-panel partial states into
//               lse, loss_i, entropy_i and correct_i, plus per-block sums;
//   finalize    fixed-order sum of the block sums into the reduced outputs
//               (run by the last merge block to finish, or as its own kernel);
//   row_coef    per-row backward coefficients (gamma with the reduction and
//               the z-loss folded in);
//   bias_reduce fixed-order sum of per-row-block grad_bias partials;
//   split_reduce fixed-order sum of the K-split partials of grad_hidden;
//   shard_state / combine  export of one vocabulary shard's per-row state and
//               the merge of several shards' states (vocabulary-parallel use).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "kernels.h"
#include "ptx.cuh"

namespace flce {
namespace {

// Deterministic block sum: warp shuffles, then warp 0 over the warp sums.
template <typename Tv>
__device__ __forceinline__ Tv block_sum(Tv v, Tv* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  Tv r = 0;
  if (warp == 0) {
    r = (lane < static_cast<int>(blockDim.x >> 5)) ? sh[lane] : Tv(0);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
  }
  __syncthreads();
  return r;  // valid in thread 0
}

// Fixed-order sum of the block sums (each thread a fixed strided subset, then
// a fixed tree) into the reduced outputs. Called by every thread of one block.
__device__ void finalize_block(const FinalizeArgs& a) {
  __shared__ double sh_d[32];
  __shared__ long long sh_i[32];
  double l = 0.0, e = 0.0;
  long long c = 0, v = 0;
  for (int b = threadIdx.x; b < a.nblk; b += blockDim.x) {
    // L2 loads: other blocks of the same launch may have written these
    l += __ldcg(a.blk_loss + b);
    e += __ldcg(a.blk_ent + b);
    c += __ldcg(a.blk_correct + b);
    v += __ldcg(a.blk_valid + b);
  }
  l = block_sum(l, sh_d);
  e = block_sum(e, sh_d);
  c = block_sum(c, sh_i);
  v = block_sum(v, sh_i);
  if (threadIdx.x == 0 && a.status != nullptr && (*a.status & kDevErrTimeout) != 0) {
    if (a.loss != nullptr) *a.loss = NAN;
    if (a.num_correct != nullptr) *a.num_correct = -1;
    if (a.entropy_sum != nullptr) *a.entropy_sum = NAN;
  } else if (threadIdx.x == 0) {
    if (a.loss != nullptr) {
      if (a.reduction == 0) {
        *a.loss = static_cast<float>(l);
      } else {
        *a.loss = v > 0 ? static_cast<float>(l / static_cast<double>(v)) : NAN;
      }
    }
    if (a.num_correct != nullptr) *a.num_correct = c;
    if (a.entropy_sum != nullptr) *a.entropy_sum = static_cast<float>(e);
  }
}

// After a block has stored its block sums: the last block of the grid to get
// here runs finalize_block (threadfence-reduction pattern: each block makes
// its stores visible before it counts itself, and the last one reads the
// others' stores only after it has seen the full count).
__device__ void finalize_if_last(int* done, const FinalizeArgs& fin) {
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(done, 1) == static_cast<int>(gridDim.x) - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  finalize_block(fin);
}

__global__ void __launch_bounds__(256) finalize_kernel(const FinalizeArgs a) { finalize_block(a); }

// Two online-softmax states of one row merged, `left` covering lower columns
// than `right`: the right one takes the argmax only with a strictly larger
// max, so ties keep the lowest column index. An empty right state (max
// -inf: no panel) leaves the left one as it is.
struct SoftmaxState {
  float m, s, t;
  int a;
};

__device__ __forceinline__ void merge_right(SoftmaxState& l, const SoftmaxState& r) {
  if (r.m == -INFINITY) return;
  if (r.m > l.m) {
    const float f = expf(l.m - r.m);
    l.s = fmaf(l.s, f, r.s);
    l.t = fmaf(l.t, f, r.t);
    l.m = r.m;
    l.a = r.a;
  } else {
    const float f = expf(r.m - l.m);
    l.s = fmaf(r.s, f, l.s);
    l.t = fmaf(r.t, f, l.t);
  }
}

// Merge of the online-softmax states of all vocabulary panels of one row
// (fused-linear-ce README, "Algorithm": the flash-attention style
// rescaling). `lanes` threads share a row: each merges a contiguous range of
// panels in panel order, then the lanes combine in a fixed tree, lower panels
// on the left. The order depends on the shape only, not on timing.
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeArgs a) {
  __shared__ double sh_d[32];
  __shared__ long long sh_i[32];
  const int lanes = a.lanes;
  const long long g = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int i = static_cast<int>(g / lanes), lane = static_cast<int>(g % lanes);
  double loss_i = 0.0, ent_i = 0.0;
  long long corr = 0, valid = 0;
  const bool timed_out = (*a.status & kDevErrTimeout) != 0;
  SoftmaxState st{-INFINITY, 0.f, 0.f, 0};
  if (i < a.N && !timed_out) {
    const int p0 = static_cast<int>(static_cast<long long>(lane) * a.num_panels / lanes);
    const int p1 = static_cast<int>(static_cast<long long>(lane + 1) * a.num_panels / lanes);
    for (int p = p0; p < p1; ++p) {
      const float4 q = a.partials[static_cast<size_t>(p) * a.N + i];
      merge_right(st, SoftmaxState{q.x, q.y, q.z, __float_as_int(q.w)});
    }
  }
  for (int o = 1; o < lanes; o <<= 1) {
    SoftmaxState r;
    r.m = __shfl_down_sync(0xffffffffu, st.m, o, lanes);
    r.s = __shfl_down_sync(0xffffffffu, st.s, o, lanes);
    r.t = __shfl_down_sync(0xffffffffu, st.t, o, lanes);
    r.a = __shfl_down_sync(0xffffffffu, st.a, o, lanes);
    if ((lane & (2 * o - 1)) == 0) merge_right(st, r);
  }
  if (i < a.N && lane == 0 && timed_out) {
    // The forward gave up before storing all of its partial states: no
    // output of this call may look like a result.
    a.lse[i] = NAN;
    loss_i = NAN;
    ent_i = NAN;
    if (a.loss_rows != nullptr) a.loss_rows[i] = NAN;
  } else if (i < a.N && lane == 0) {
    const float lse = st.m + logf(st.s);
    a.lse[i] = lse;
    const long long t = a.targets[i];
    float li = 0.f;
    if (t != a.ignore_index) {
      valid = 1;
      if (t < 0 || t >= a.vocab_total) {
        atomicOr(a.status, kDevErrTargetRange);
        li = NAN;
      } else {
        li = lse - a.zt[i] + a.zeta * lse * lse;
        ent_i = static_cast<double>(lse - st.t / st.s);
        corr = (static_cast<long long>(st.a) + a.vocab_start == t) ? 1 : 0;
      }
    }
    loss_i = li;
    if (a.loss_rows != nullptr) a.loss_rows[i] = li;
  }
  const double bl = block_sum(loss_i, sh_d);
  const double be = block_sum(ent_i, sh_d);
  const long long bc = block_sum(corr, sh_i);
  const long long bv = block_sum(valid, sh_i);
  if (threadIdx.x == 0) {
    a.blk_loss[blockIdx.x] = bl;
    a.blk_ent[blockIdx.x] = be;
    a.blk_correct[blockIdx.x] = bc;
    a.blk_valid[blockIdx.x] = bv;
  }
  if (a.done != nullptr) finalize_if_last(a.done, a.fin);
}

// Per-row state of one vocabulary shard: the panels of this call merged in
// panel order (as in merge_kernel), with the argmax made a global id. The
// target logit is kept only if the target lies in this shard.
__global__ void __launch_bounds__(256) shard_state_kernel(const ShardStateArgs a) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= a.N) return;
  if ((*a.status & kDevErrTimeout) != 0) {
    // the forward gave up before storing all of its partial states
    a.out[i] = ShardState{NAN, NAN, NAN, -1, NAN};
    return;
  }
  float M = -INFINITY, S = 0.f, Tt = 0.f;
  int A = 0;
  for (int p = 0; p < a.num_panels; ++p) {
    const float4 st = a.partials[static_cast<size_t>(p) * a.N + i];
    if (st.x > M) {
      const float f = expf(M - st.x);
      S = fmaf(S, f, st.y);
      Tt = fmaf(Tt, f, st.z);
      M = st.x;
      A = __float_as_int(st.w);
    } else {
      const float f = expf(st.x - M);
      S = fmaf(st.y, f, S);
      Tt = fmaf(st.z, f, Tt);
    }
  }
  const long long t = a.targets[i];
  const long long local = t - a.vocab_start;
  const bool owned = t != a.ignore_index && local >= 0 && local < a.V;
  ShardState o;
  o.m = M;
  o.s = S;
  o.t = Tt;
  o.argmax = static_cast<int>(A + a.vocab_start);
  o.zt = owned ? a.zt[i] : 0.f;
  a.out[i] = o;
}

// Merge of the states of R vocabulary shards, in shard order, into lse,
// loss_i, entropy_i and correct_i per row, plus per-block sums, which the
// last block to finish reduces (finalize_block). The shards must be given in
// increasing vocabulary order:
// a later shard takes the argmax only with a strictly larger max, so ties keep
// the lowest global id. The target logit is the sum over shards; only the owning
// shard contributes a nonzero value.
__global__ void __launch_bounds__(kMergeThreads) combine_kernel(const CombineArgs a) {
  __shared__ double sh_d[32];
  __shared__ long long sh_i[32];
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  double loss_i = 0.0, ent_i = 0.0;
  long long corr = 0, valid = 0;
  if (i < a.N) {
    float M = -INFINITY, S = 0.f, Tt = 0.f, zt = 0.f;
    int A = 0;
    for (int r = 0; r < a.R; ++r) {
      const ShardState st = a.states[static_cast<size_t>(r) * a.N + i];
      zt += st.zt;
      if (st.m > M) {
        const float f = expf(M - st.m);
        S = fmaf(S, f, st.s);
        Tt = fmaf(Tt, f, st.t);
        M = st.m;
        A = st.argmax;
      } else {
        const float f = expf(st.m - M);
        S = fmaf(st.s, f, S);
        Tt = fmaf(st.t, f, Tt);
      }
    }
    const float lse = M + logf(S);
    a.lse[i] = lse;
    const long long t = a.targets[i];
    float li = 0.f;
    if (t != a.ignore_index) {
      valid = 1;
      if (t < 0 || t >= a.vocab_total) {
        atomicOr(a.status, kDevErrTargetRange);
        li = NAN;
      } else {
        li = lse - zt + a.zeta * lse * lse;
        ent_i = static_cast<double>(lse - Tt / S);
        corr = (static_cast<long long>(A) == t) ? 1 : 0;
      }
    }
    loss_i = li;
    if (a.loss_rows != nullptr) a.loss_rows[i] = li;
  }
  const double bl = block_sum(loss_i, sh_d);
  const double be = block_sum(ent_i, sh_d);
  const long long bc = block_sum(corr, sh_i);
  const long long bv = block_sum(valid, sh_i);
  if (threadIdx.x == 0) {
    a.blk_loss[blockIdx.x] = bl;
    a.blk_ent[blockIdx.x] = be;
    a.blk_correct[blockIdx.x] = bc;
    a.blk_valid[blockIdx.x] = bv;
  }
  if (a.done != nullptr) finalize_if_last(a.done, a.fin);
}


// One 32 x 32 tile of the transposition, rows [r0, r0 + 32) and columns
// [c0, c0 + 32) of the source, through shared memory (one element per 32-bit
// word, a 33-word row pitch, so that neither the row reads nor the column
// reads conflict); 32 x 8 threads, four rows each.
template <typename R>
__device__ __forceinline__ void transpose_tile(const TransposeArgs& a, uint32_t (&tile)[32][33],
                                               R r0, int c0, int tx, int ty) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const R r = r0 + ty + 8 * i;
    const int c = c0 + tx;
    tile[ty + 8 * i][tx] = (r < a.rows && c < a.cols) ? a.src[r * a.ld_src + c] : 0u;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = c0 + ty + 8 * i;
    const R r = r0 + tx;
    uint16_t* const dst = a.dst + c * a.ld_dst + r;
    if (c < a.cols && r < a.rows && store_allowed(dst, 2, a.r_dst, a.status))
      *dst = static_cast<uint16_t>(tile[tx][ty + 8 * i]);
  }
}

// blockIdx.x is the column tile and blockIdx.y the row tile. gridDim.y is at
// most 65535; past 65535 row tiles (2,097,120 rows) each block steps through
// the row tiles by gridDim.y, so any number of rows fits one launch. The copy
// is latency-bound: 8 blocks per SM (at most 32 registers a thread) keep
// enough loads in flight; with 48 registers and 5 blocks it ran 30 % slower.
__global__ void __launch_bounds__(256, 8) transpose16_kernel(const TransposeArgs a) {
  __shared__ uint32_t tile[32][33];
  const int c0 = blockIdx.x * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  if (gridDim.y * 32ll >= a.rows) {
    transpose_tile<int>(a, tile, static_cast<int>(blockIdx.y) * 32, c0, tx, ty);
    return;
  }
  for (long long r0 = blockIdx.y * 32ll; r0 < a.rows; r0 += gridDim.y * 32ll) {
    transpose_tile<long long>(a, tile, r0, c0, tx, ty);
    __syncthreads();   // the tile is read out before the next one is written
  }
}

// One block, the backward's first kernel. It zeroes the workspace header and
// tile counters, counts the valid rows (needed for the mean), then writes the
// coefficients of every row.
__global__ void __launch_bounds__(1024) row_coef_kernel(const RowCoefArgs a) {
  __shared__ long long sh_i[32];
  __shared__ long long s_valid;
  __shared__ float sh_max[32];
  for (int i = threadIdx.x; i < a.zero_words; i += blockDim.x) a.zero[i] = 0;
  __syncthreads();
  long long v = 0;
  for (int i = threadIdx.x; i < a.N; i += blockDim.x) v += (a.targets[i] != a.ignore_index) ? 1 : 0;
  v = block_sum(v, sh_i);
  if (threadIdx.x == 0) s_valid = v;
  __syncthreads();
  const long long num_valid = s_valid;
  float g_all = 0.f;
  if (a.reduction == 0) g_all = a.grad_loss[0];
  if (a.reduction == 1) g_all = num_valid > 0 ? a.grad_loss[0] / static_cast<float>(num_valid) : 0.f;
  float cmax = 0.f;  // bound on |dlogits|: |g| <= max(|x|, |y|) because 0 <= p <= 1
  for (int i = threadIdx.x; i < a.N; i += blockDim.x) {
    const long long t = a.targets[i];
    const float lse = a.lse[i];
    float4 c = make_float4(0.f, 0.f, lse, __int_as_float(-1));
    if (t != a.ignore_index) {
      if (t < 0 || t >= a.vocab_total) {
        atomicOr(a.status, kDevErrTargetRange);
      } else {
        const float gam = (a.reduction == 2) ? a.grad_loss[i] : g_all;
        const float sg = a.scale * gam;
        c.x = sg * fmaf(2.f * a.zeta, lse, 1.f);
        c.y = sg;
        // the onehot term belongs to the shard that holds the target
        const long long local = t - a.vocab_start;
        if (local >= 0 && local < a.V) c.w = __int_as_float(static_cast<int>(local));
      }
    }
    a.coef[i] = c;
    cmax = fmaxf(cmax, fmaxf(fabsf(c.x), fabsf(c.y)));
  }
  if (a.ds_scale != nullptr) {
    // fp16 dlogits are stored times S = 2^k with max |dlogits| * S <= 2^14:
    // large values stay below the fp16 maximum (65504) and small probabilities
    // stay above its subnormal range. S is a power of two, so scaling and
    // unscaling are exact.
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
    if ((threadIdx.x & 31) == 0) sh_max[threadIdx.x >> 5] = cmax;
    __syncthreads();
    if (threadIdx.x == 0) {
      float m = 0.f;
      for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) m = fmaxf(m, sh_max[w]);
      int k = 0;
      if (m > 0.f && isfinite(m)) {
        int e;
        frexpf(m, &e);          // m = f * 2^e with 0.5 <= f < 1, so m < 2^e
        k = 14 - e;
        k = k > 120 ? 120 : (k < -120 ? -120 : k);
      }
      a.ds_scale[0] = ldexpf(1.f, k);
      a.ds_scale[1] = ldexpf(1.f, -k);
    }
  }
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}
template <> __device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }

template <typename Tout>
__global__ void __launch_bounds__(256) bias_reduce_kernel(const BiasReduceArgs a) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= a.V) return;
  float s = 0.f;
  for (int b = 0; b < a.nblk; ++b) s += a.bias_part[static_cast<size_t>(b) * a.V_pad + j];
  Tout* gb = static_cast<Tout*>(a.grad_bias);
  if (a.accumulate) s += to_f32(gb[j]);
  gb[j] = from_f32<Tout>(s);
}

// Sums the fp32 K-split partials of a GEMM in split order and casts to the
// 16-bit output type. Each thread handles 4 consecutive columns (N is a
// multiple of 8).
template <typename Tout>
__global__ void __launch_bounds__(256) split_reduce_kernel(const SplitReduceArgs a) {
  const long long q = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long per_row = a.N / 4;
  if (q >= static_cast<long long>(a.M) * per_row) return;
  const long long m = q / per_row;
  const long long n = (q - m * per_row) * 4;
  float4 acc = *reinterpret_cast<const float4*>(a.part + m * a.ld_part + n);
  for (int s = 1; s < a.splits; ++s) {
    const float4 p = *reinterpret_cast<const float4*>(a.part + s * a.split_stride + m * a.ld_part + n);
    acc.x += p.x;
    acc.y += p.y;
    acc.z += p.z;
    acc.w += p.w;
  }
  Tout* dst = static_cast<Tout*>(a.out) + m * a.ld_out + n;
  if (a.accumulate) {
    acc.x += to_f32(dst[0]);
    acc.y += to_f32(dst[1]);
    acc.z += to_f32(dst[2]);
    acc.w += to_f32(dst[3]);
  }
  dst[0] = from_f32<Tout>(acc.x);
  dst[1] = from_f32<Tout>(acc.y);
  dst[2] = from_f32<Tout>(acc.z);
  dst[3] = from_f32<Tout>(acc.w);
}

}  // namespace

cudaError_t launch_split_reduce(const SplitReduceArgs& a, cudaStream_t s) {
  const long long n = static_cast<long long>(a.M) * (a.N / 4);
  const unsigned grid = static_cast<unsigned>((n + 255) / 256);
  if (a.f16)
    split_reduce_kernel<__half><<<grid, 256, 0, s>>>(a);
  else
    split_reduce_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(a);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_merge(const MergeArgs& a, int nblk, cudaStream_t s) {
  merge_kernel<<<nblk, kMergeThreads, 0, s>>>(a);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_shard_state(const ShardStateArgs& a, cudaStream_t s) {
  shard_state_kernel<<<(a.N + 255) / 256, 256, 0, s>>>(a);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_combine(const CombineArgs& a, int nblk, cudaStream_t s) {
  combine_kernel<<<nblk, kMergeThreads, 0, s>>>(a);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_finalize(const FinalizeArgs& a, cudaStream_t s) {
  finalize_kernel<<<1, 256, 0, s>>>(a);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_transpose16(const TransposeArgs& a, cudaStream_t s) {
  const int row_tiles = (a.rows + 31) / 32;
  const dim3 grid((a.cols + 31) / 32, row_tiles < 1 ? 1 : (row_tiles < 65535 ? row_tiles : 65535));
  transpose16_kernel<<<grid, 256, 0, s>>>(a);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_row_coef(const RowCoefArgs& a, cudaStream_t s) {
  row_coef_kernel<<<1, 1024, 0, s>>>(a);
  note_launch();
  return cudaGetLastError();
}

// One block: every thread sums a fixed strided subset in fp64, then a fixed
// tree sums the threads. The result does not depend on timing.
__global__ void __launch_bounds__(1024) loss_reduce_kernel(const LossReduceArgs a) {
  __shared__ double sh[32];
  double s = 0.0;
  for (long long i = threadIdx.x; i < a.count; i += blockDim.x) s += a.part[i];
  s = block_sum(s, sh);
  if (threadIdx.x == 0) a.loss[0] = (a.accumulate ? a.loss[0] : 0.0) + s;
}

// 16 bytes per thread and step when both pointers are 16-byte aligned; the
// rest (or everything, if they are not) element by element.
template <typename T>
__global__ void __launch_bounds__(256) scale_kernel(const ScaleArgs a) {
  const float s = *a.scale;
  if (s == 1.f && a.src == a.dst) return;
  constexpr int kPer = 16 / static_cast<int>(sizeof(T));
  const T* src = static_cast<const T*>(a.src);
  T* dst = static_cast<T*>(a.dst);
  const bool vec = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15u) == 0;
  const long long nv = vec ? a.count / kPer : 0;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long t0 = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  for (long long i = t0; i < nv; i += stride) {
    union {
      uint4 v;
      T e[kPer];
    } u;
    u.v = reinterpret_cast<const uint4*>(src)[i];
#pragma unroll
    for (int k = 0; k < kPer; ++k) u.e[k] = from_f32<T>(to_f32(u.e[k]) * s);
    reinterpret_cast<uint4*>(dst)[i] = u.v;
  }
  for (long long i = nv * kPer + t0; i < a.count; i += stride) dst[i] = from_f32<T>(to_f32(src[i]) * s);
}

cudaError_t launch_scale(const ScaleArgs& a, int sms, cudaStream_t s) {
  const long long blocks = (a.count / 4 + 255) / 256;
  const unsigned grid = static_cast<unsigned>(blocks < 1 ? 1 : (blocks < 8ll * sms ? blocks : 8ll * sms));
  if (a.dtype == 1)
    scale_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(a);
  else if (a.dtype == 2)
    scale_kernel<__half><<<grid, 256, 0, s>>>(a);
  else
    scale_kernel<float><<<grid, 256, 0, s>>>(a);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_loss_reduce(const LossReduceArgs& a, cudaStream_t s) {
  loss_reduce_kernel<<<1, 1024, 0, s>>>(a);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_bias_reduce(const BiasReduceArgs& a, int dtype, cudaStream_t s) {
  const int grid = (a.V + 255) / 256;
  if (dtype == 1)
    bias_reduce_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(a);
  else if (dtype == 2)
    bias_reduce_kernel<__half><<<grid, 256, 0, s>>>(a);
  else
    bias_reduce_kernel<float><<<grid, 256, 0, s>>>(a);
  note_launch();
  return cudaGetLastError();
}

}  // namespace flce
