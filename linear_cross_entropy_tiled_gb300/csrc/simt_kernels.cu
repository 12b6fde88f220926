// fp32 kernels. This is the path for fp32 hidden/weight: plain FFMA
// arithmetic, no tensor cores.
//
// The fused-linear-ce README ("Full signature") accepts fp32 inputs. A loss
// accurate to 1e-5 relative needs fp32 products. TF32 tensor cores round the
// operands to 10 mantissa bits, which is not enough. The schedule is the same
// as the bf16 path: vocabulary panels with an online log-sum-exp (forward),
// and a recompute -> dlogits -> two contractions backward. Only the tile
// arithmetic differs. Speed is secondary to the 1e-5 accuracy bar; the work is
// spread over enough blocks for small problems (forward panels of 64 to 256
// columns, vocabulary chunks over all rows in the backward, and a fixed-order
// K split for grad_hidden, whose output is small).
#include <math.h>

#include "kernels.h"
#include "ptx.cuh"

namespace flce {
namespace {

constexpr int T = kSimtTile;   // 64
constexpr int TK = 32;

// Computes the 64 x 64 tile acc[i][j] += sum_k h[r0+4ty+i][k] * w[c0+4tx+j][k].
// Rows >= nrows and columns >= ncols read as 0.
__device__ __forceinline__ void simt_logit_tile(const float* __restrict__ h,
                                                const float* __restrict__ w, int H, int r0,
                                                int nrows, int c0, int ncols, float (&As)[TK][T + 4],
                                                float (&Bs)[TK][T + 4], float (&acc)[4][4]) {
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  // The next K slice is loaded into registers while the current one is
  // multiplied from shared memory, so global latency overlaps the FMAs.
  constexpr int kPer = T * TK / kSimtThreads;   // elements of each operand per thread
  float ra[kPer], rb[kPer];
  auto load = [&](int k0) {
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int e = tid + q * kSimtThreads;
      const int rr = e / TK, k = k0 + e % TK;
      ra[q] = (r0 + rr < nrows && k < H) ? h[static_cast<size_t>(r0 + rr) * H + k] : 0.f;
      rb[q] = (c0 + rr < ncols && k < H) ? w[static_cast<size_t>(c0 + rr) * H + k] : 0.f;
    }
  };
  load(0);
  for (int k0 = 0; k0 < H; k0 += TK) {
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int e = tid + q * kSimtThreads;
      As[e % TK][e / TK] = ra[q];
      Bs[e % TK][e / TK] = rb[q];
    }
    __syncthreads();
    if (k0 + TK < H) load(k0 + TK);
#pragma unroll 8
    for (int kk = 0; kk < TK; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
}

__device__ __forceinline__ float transform_f32(float a, const float* bias, int col, float scale,
                                               float cap, float inv_cap) {
  float u = (bias != nullptr) ? (a + bias[col]) * scale : a * scale;
  if (cap > 0.f) u = cap * tanhf(u * inv_cap);
  return u;
}

// One block per (panel of 64 x panel_tiles columns, block of 64 rows).
__global__ void __launch_bounds__(kSimtThreads)
    fwd_simt_kernel(const float* __restrict__ h, const float* __restrict__ w, const FwdArgs a) {
  __shared__ float As[TK][T + 4];
  __shared__ float Bs[TK][T + 4];
  __shared__ float Z[T][T + 1];
  const int panel = blockIdx.x / a.n_blocks;
  const int rb = blockIdx.x - panel * a.n_blocks;
  const int r0 = rb * T;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const float* bias = static_cast<const float*>(a.bias);
  float m = -INFINITY, ssum = 0.f, tsum = 0.f;
  int amax = 0;
  const int row = r0 + tid;
  long long tgt = (tid < T && row < a.N) ? a.targets[row] : a.ignore_index;
  tgt = (tgt == a.ignore_index) ? -(1ll << 40) : tgt - a.vocab_start;  // shard-local id
  const int c_begin = panel * a.panel_tiles * T;
  const int c_end = min(a.V, c_begin + a.panel_tiles * T);
  for (int c0 = c_begin; c0 < c_end; c0 += T) {
    float acc[4][4];
    simt_logit_tile(h, w, a.H, r0, a.N, c0, a.V, As, Bs, acc);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int col = c0 + tx * 4 + j;
        Z[ty * 4 + i][tx * 4 + j] =
            col < a.V ? transform_f32(acc[i][j], bias, col, a.scale, a.softcap, a.inv_softcap)
                      : -INFINITY;
      }
    __syncthreads();
    if (tid < T && row < a.N) {
      const int nc = min(T, a.V - c0);
      for (int j = 0; j < nc; ++j) {
        const float z = Z[tid][j];
        if (c0 + j == tgt && store_allowed(&a.zt[row], 4, a.r_zt, a.status)) a.zt[row] = z;
        if (z > m) {
          const float f = expf(m - z);
          ssum = ssum * f + 1.f;
          tsum = tsum * f + z;
          m = z;
          amax = c0 + j;
        } else {
          const float e = expf(z - m);
          ssum += e;
          tsum = fmaf(z, e, tsum);
        }
      }
    }
    __syncthreads();
  }
  if (tid < T && row < a.N)
    a.partials[static_cast<size_t>(panel) * a.N + row] =
        make_float4(m, ssum, tsum, __int_as_float(amax));
}

// One block per (64-column tile, 64-row block of the chunk).
__global__ void __launch_bounds__(kSimtThreads)
    ds_simt_kernel(const float* __restrict__ h, const float* __restrict__ w, const DsArgs a) {
  __shared__ float As[TK][T + 4];
  __shared__ float Bs[TK][T + 4];
  __shared__ float G[T][T + 1];
  const int c0 = blockIdx.x * T;
  const int rb = blockIdx.y;
  const int r0 = rb * T;  // local to the chunk
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const float* bias = static_cast<const float*>(a.bias);
  float acc[4][4];
  simt_logit_tile(h + static_cast<size_t>(a.row0) * a.H, w, a.H, r0, a.rows, c0, a.V, As, Bs, acc);
  float* ds = static_cast<float*>(a.ds);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int rl = r0 + ty * 4 + i;
    const bool row_ok = rl < a.rows;
    const float4 cf = row_ok ? a.coef[a.row0 + rl] : make_float4(0.f, 0.f, 0.f, __int_as_float(-1));
    const int tgt = __float_as_int(cf.w) - a.tgt_base;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = c0 + tx * 4 + j;
      float g = 0.f;
      if (row_ok && col < a.V) {
        const float z = transform_f32(acc[i][j], bias, col, a.scale, a.softcap, a.inv_softcap);
        const float p = expf(z - cf.z);
        g = cf.x * p;
        if (col == tgt) g -= cf.y;
        if (a.softcap > 0.f) {
          const float zc = z * a.inv_softcap;
          g *= (1.f - zc * zc);
        }
        float* const dst = ds + static_cast<size_t>(rl) * a.V_pad + col;
        if (store_allowed(dst, 4, a.r_ds, a.status)) *dst = g;
      }
      G[ty * 4 + i][tx * 4 + j] = g;
    }
  }
  if (a.bias_part != nullptr) {
    __syncthreads();
    if (tid < T && c0 + tid < a.V) {
      float sum = 0.f;
      for (int i = 0; i < T; ++i) sum += G[i][tid];
      float* const dst = a.bias_part + static_cast<size_t>(a.bias_blk0 + rb) * a.bias_ld + c0 + tid;
      if (store_allowed(dst, 4, a.r_bias, a.status)) *dst = sum;
    }
  }
}

constexpr int GK = 16;

// Output tile (bx, by) of 64 x 64 and K split bz of one product.
__device__ __forceinline__ void gemm_simt_block(const SimtGemmArgs& a, int bx, int by, int bz) {
  __shared__ float As[GK][T + 4];
  __shared__ float Bs[GK][T + 4];
  const int m0 = by * T, n0 = bx * T;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  // this block's K range: all of K, or split bz of k_splits
  const int kc = a.k_splits > 1 ? (a.K + a.k_splits - 1) / a.k_splits : a.K;
  const int kb = bz * kc;
  const int ke = min(a.K, kb + kc);
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  // Neighbouring threads read neighbouring addresses: along K for an operand
  // whose K stride is 1, else along M (or N). The next K slice is loaded into
  // registers while the current one is multiplied from shared memory.
  const bool a_k_contig = a.sak == 1, b_k_contig = a.sbk == 1 && a.sbn != 1;
  constexpr int kPer = T * GK / kSimtThreads;   // elements of each operand per thread
  float ra[kPer], rb[kPer];
  auto coords = [&](int e, bool k_contig, int& k, int& mn) {
    k = k_contig ? e % GK : e / T;
    mn = k_contig ? e / GK : e % T;
  };
  auto load = [&](int k0) {
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int e = tid + q * kSimtThreads;
      int ka, ma, kbb, nb;
      coords(e, a_k_contig, ka, ma);
      coords(e, b_k_contig, kbb, nb);
      ra[q] = (m0 + ma < a.M && k0 + ka < ke) ? a.A[(m0 + ma) * a.sam + (k0 + ka) * a.sak] : 0.f;
      rb[q] = (n0 + nb < a.N && k0 + kbb < ke) ? a.B[(k0 + kbb) * a.sbk + (n0 + nb) * a.sbn] : 0.f;
    }
  };
  if (kb < ke) load(kb);
  for (int k0 = kb; k0 < ke; k0 += GK) {
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int e = tid + q * kSimtThreads;
      int ka, ma, kbb, nb;
      coords(e, a_k_contig, ka, ma);
      coords(e, b_k_contig, kbb, nb);
      As[ka][ma] = ra[q];
      Bs[kbb][nb] = rb[q];
    }
    __syncthreads();
    if (k0 + GK < ke) load(k0 + GK);
#pragma unroll
    for (int kk = 0; kk < GK; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= a.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= a.N) continue;
      if (bz > 0) {
        float* const dst = a.part + (static_cast<size_t>(bz - 1) * a.M + m) * a.N + n;
        if (store_allowed(dst, 4, a.r_part, a.status)) *dst = acc[i][j];
      } else {
        float* c = a.C + m * a.ldc + n;
        if (store_allowed(c, 4, a.r_c, a.status)) *c = a.accumulate ? *c + acc[i][j] : acc[i][j];
      }
    }
  }
}

__global__ void __launch_bounds__(kSimtThreads) gemm_simt_kernel(const SimtGemmArgs a) {
  gemm_simt_block(a, blockIdx.x, blockIdx.y, blockIdx.z);
}

// Two independent products in one grid: blocks [0, n1) compute the first,
// the rest the second. The two contractions of a backward chunk are each too
// small to fill the GPU alone; together they do.
__global__ void __launch_bounds__(kSimtThreads) gemm_simt2_kernel(const SimtGemmArgs a1,
                                                                  const SimtGemmArgs a2, int n1) {
  const bool first = static_cast<int>(blockIdx.x) < n1;
  const SimtGemmArgs& a = first ? a1 : a2;
  const int i = first ? static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x) - n1;
  const int gx = (a.N + T - 1) / T, gy = (a.M + T - 1) / T;
  gemm_simt_block(a, i % gx, (i / gx) % gy, i / (gx * gy));
}

// Split 0 of a K-split product has already written C (or added to it); this
// adds the other splits' partials part[0 .. k_splits - 2] in split order.
__global__ void __launch_bounds__(256) simt_split_reduce_kernel(const SimtGemmArgs a) {
  const long long total = static_cast<long long>(a.M) * a.N;
  for (long long i = blockIdx.x * 256ll + threadIdx.x; i < total; i += 256ll * gridDim.x) {
    float s = 0.f;
    for (int z = 0; z + 1 < a.k_splits; ++z) s += a.part[z * total + i];
    const int m = static_cast<int>(i / a.N), n = static_cast<int>(i - static_cast<long long>(m) * a.N);
    float* c = a.C + m * a.ldc + n;
    if (store_allowed(c, 4, a.r_c, a.status)) *c += s;
  }
}

}  // namespace

cudaError_t launch_fwd_simt(const float* h, const float* w, const FwdArgs& a, cudaStream_t s) {
  fwd_simt_kernel<<<a.num_units, kSimtThreads, 0, s>>>(h, w, a);
  return cudaGetLastError();
}

cudaError_t launch_ds_simt(const float* h, const float* w, const DsArgs& a, cudaStream_t s) {
  dim3 grid((a.V + T - 1) / T, (a.rows + T - 1) / T);
  ds_simt_kernel<<<grid, kSimtThreads, 0, s>>>(h, w, a);
  return cudaGetLastError();
}

namespace {
int simt_blocks(const SimtGemmArgs& a) {
  return ((a.N + T - 1) / T) * ((a.M + T - 1) / T) * (a.k_splits > 1 ? a.k_splits : 1);
}
cudaError_t split_reduce_after(const SimtGemmArgs& a, cudaStream_t s) {
  if (a.k_splits <= 1) return cudaSuccess;
  const long long total = static_cast<long long>(a.M) * a.N;
  const int blocks = static_cast<int>(min(4096ll, (total + 255) / 256));
  simt_split_reduce_kernel<<<blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_gemm_simt2(const SimtGemmArgs& a1, const SimtGemmArgs& a2, cudaStream_t s) {
  const int n1 = simt_blocks(a1), n2 = simt_blocks(a2);
  gemm_simt2_kernel<<<n1 + n2, kSimtThreads, 0, s>>>(a1, a2, n1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if ((e = split_reduce_after(a1, s)) != cudaSuccess) return e;
  return split_reduce_after(a2, s);
}

cudaError_t launch_gemm_simt(const SimtGemmArgs& a, cudaStream_t s) {
  const int splits = a.k_splits > 1 ? a.k_splits : 1;
  dim3 grid((a.N + T - 1) / T, (a.M + T - 1) / T, splits);
  gemm_simt_kernel<<<grid, kSimtThreads, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || splits == 1) return e;
  const long long total = static_cast<long long>(a.M) * a.N;
  const int blocks = static_cast<int>(min(4096ll, (total + 255) / 256));
  simt_split_reduce_kernel<<<blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace flce
