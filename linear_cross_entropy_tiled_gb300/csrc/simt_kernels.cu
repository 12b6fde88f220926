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
// K split for grad_hidden, whose output is small). Every kernel multiplies
// 64 x 64 tiles with 4 x 8 outputs per thread from operand slices that
// cp.async brings into a shared-memory ring (tile_product); the backward's
// two contractions share one persistent grid.
#include <math.h>

#include "kernels.h"
#include "ptx.cuh"

namespace flce {
namespace {

constexpr int T = kSimtTile;   // 64
constexpr int KS = 16;         // K slice per group and step
constexpr int NS = 3;          // stages of each group's copy ring
constexpr int kPitch = T + 4;  // shared-memory row pitch in floats: rows stay 16-byte aligned

// A 64 x 64 tile is computed by each 128-thread group of a block. Thread
// (ty, tx) = (lt / 8, lt % 8) of a group holds rows 4ty .. 4ty+3 and the
// columns tile_col(tx, 0 .. 7): 4tx .. 4tx+3 and 32+4tx .. 32+4tx+3, in
// increasing order. Per k it reads one 16-byte row piece and two 16-byte
// column pieces from shared memory for 32 FMAs; a warp's reads are 64 and
// 2 x 128 contiguous bytes. The block's groups split the K range, so that
// small grids still keep several warps per SM busy.
__device__ __forceinline__ int tile_col(int tx, int j) { return (j & 4) * 8 + tx * 4 + (j & 3); }

// One operand of a tile product, as seen from its 64 x KS slices: element
// (k, mn) of the tile (k counted from the start of the K range) is
// p[mn * s_mn + k * s_k]; mn_lim of the 64 mn exist.
struct OperandView {
  const float* p;
  long long s_mn, s_k;
  int mn_lim;
  bool k_contig;
};

// A thread's share of one operand slice: kPer = 64 KS / 128 elements, fixed
// coordinates for the whole K loop. K-contiguous operands: a warp reads 8
// consecutive k of 4 rows (four whole 32-byte sectors), and its transposed
// shared-memory stores fall in 32 different banks (the pitch is 4 mod 32);
// element q is (kt, mt + 8q). MN-contiguous operands: a warp reads 32
// consecutive mn of one k; element q is (kt + 2q, mt).
struct SliceStream {
  static constexpr int kPer = T * KS / kSimtThreads;
  static_assert(KS == 16 && kPer == 8, "coordinates below are for 16-deep slices");
  const float* p;     // element 0 at k = 0
  const float* base;  // the operand's first element
  long long dq, dk;   // address step from element q to q + 1, and per unit of k
  int kt, mt;
  unsigned mask;      // bit q: element q lies inside the operand along mn
  bool kc;
  __device__ __forceinline__ void init(const OperandView& v, int lt) {
    const int lane = lt & 31, w = lt >> 5;
    kc = v.k_contig;
    if (kc) {
      kt = (w & 1) * 8 + (lane & 7);
      mt = (w >> 1) * 4 + (lane >> 3);
      dq = 8 * v.s_mn;
    } else {
      kt = lt >> 6;
      mt = lt & 63;
      dq = 2 * v.s_k;
    }
    dk = v.s_k;
    base = v.p;
    p = v.p + mt * v.s_mn + kt * v.s_k;
    mask = 0;
#pragma unroll
    for (int q = 0; q < kPer; ++q)
      if ((kc ? mt + 8 * q : mt) < v.mn_lim) mask |= 1u << q;
  }
  // Starts the copy of element q of the slice starting at k0 into the
  // stage's slice; outside the operand or past ke it is zero-filled (nothing
  // is read: the address given is then the operand's first element).
  __device__ __forceinline__ void copy(float (&sl)[KS][kPitch], int q, int k0, int ke) const {
    const int k = kc ? kt : kt + 2 * q;
    const bool ok = ((mask >> q) & 1u) && k0 + k < ke;
    float* const dst = kc ? &sl[kt][mt + 8 * q] : &sl[kt + 2 * q][mt];
    cp_async4(dst, ok ? p + k0 * dk + q * dq : base, ok);
  }
};

// acc[i][j] += As[k][4ty + i] * Bs[k][tile_col(tx, j)] for one k.
__device__ __forceinline__ void fma_k(const float* as_k, const float* bs_k, int ty, int tx,
                                      float (&acc)[4][8]) {
  const float4 av = *reinterpret_cast<const float4*>(as_k + ty * 4);
  const float4 b0 = *reinterpret_cast<const float4*>(bs_k + tx * 4);
  const float4 b1 = *reinterpret_cast<const float4*>(bs_k + 32 + tx * 4);
  const float a4[4] = {av.x, av.y, av.z, av.w};
  const float b8[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a4[i], b8[j], acc[i][j]);
}

// Each group waits only for its own threads inside the K loop.
__device__ __forceinline__ void group_sync(int g) {
  asm volatile("bar.sync %0, %1;" ::"r"(g + 1), "r"(kSimtThreads) : "memory");
}

// Shared memory of a block (dynamic: it exceeds the 48 KB of static shared
// memory): each group's ring of NS operand slices. After the K loop the same
// bytes carry the groups' sums to group 0.
template <int KG>
struct alignas(16) SimtSmem {
  float a[KG][NS][KS][kPitch];
  float b[KG][NS][KS][kPitch];
};
static_assert(sizeof(SimtSmem<2>) >= sizeof(float) * 32 * kSimtThreads, "room for one group's sums");

// The 64 x 64 tile acc[i][j] = sum over k in [kb, ke) of A(k, 4ty+i) *
// B(k, tile_col(tx, j)), complete in group 0 (the other groups' acc are
// partial). Group g multiplies the slices g, g + KG, ...; group 0 then adds
// the other groups' sums in group order, so the result does not depend on
// timing. A(k, m) and B(k, n) are read through their views, zero outside
// the operand or the range, by cp.async copies NS - 1 slices ahead of the
// multiplication.
template <int KG>
__device__ __forceinline__ void tile_product(const OperandView& va, const OperandView& vb, int kb,
                                             int ke, SimtSmem<KG>& sm, float (&acc)[4][8]) {
  const int g = threadIdx.x / kSimtThreads, lt = threadIdx.x % kSimtThreads;
  const int tx = lt & 7, ty = lt >> 3;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  constexpr int kPer = SliceStream::kPer;
  SliceStream sa, sb;
  sa.init(va, lt);
  sb.init(vb, lt);
  // Slice `step` of this group starts at k_first + step KG KS and goes to
  // stage step % NS. NS - 1 slices are in flight while one is multiplied.
  const int k_first = kb + g * KS;
  const int nsteps = k_first < ke ? (ke - k_first + KG * KS - 1) / (KG * KS) : 0;
  auto issue = [&](int step) {
    const int k0 = k_first + step * KG * KS;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      sa.copy(sm.a[g][step % NS], q, k0, ke);
      sb.copy(sm.b[g][step % NS], q, k0, ke);
    }
  };
#pragma unroll
  for (int st = 0; st < NS - 1; ++st) {
    if (st < nsteps) issue(st);
    cp_async_commit();
  }
  for (int step = 0; step < nsteps; ++step) {
    cp_async_wait<NS - 2>();   // this thread's copies of slice `step` have landed
    group_sync(g);             // everyone's have; the stage of step - 1 is free
    if (step + NS - 1 < nsteps) issue(step + NS - 1);
    cp_async_commit();
    const int stg = step % NS;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) fma_k(sm.a[g][stg][kk], sm.b[g][stg][kk], ty, tx, acc);
  }
  cp_async_wait<0>();
  float* const red = &sm.a[0][0][0][0];
  __syncthreads();
#pragma unroll
  for (int src = 1; src < KG; ++src) {
    if (g == src)
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) red[(i * 8 + j) * kSimtThreads + lt] = acc[i][j];
    __syncthreads();
    if (g == 0)
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] += red[(i * 8 + j) * kSimtThreads + lt];
    __syncthreads();
  }
}

// Operands of a logit tile: rows r0 .. of h [nrows, H] and rows c0 .. of
// w [ncols, H], both contiguous along K = H.
__device__ __forceinline__ void logit_views(const float* h, const float* w, int H, int r0,
                                            int nrows, int c0, int ncols, OperandView& va,
                                            OperandView& vb) {
  va = OperandView{h + static_cast<size_t>(r0) * H, H, 1, nrows - r0, true};
  vb = OperandView{w + static_cast<size_t>(c0) * H, H, 1, ncols - c0, true};
}

__device__ __forceinline__ float transform_f32(float a, const float* bias, int col, float scale,
                                               float cap, float inv_cap) {
  float u = (bias != nullptr) ? (a + bias[col]) * scale : a * scale;
  if (cap > 0.f) u = cap * tanhf(u * inv_cap);
  return u;
}

// Online-softmax state of one row over some columns: max, sum exp(z - max),
// sum z exp(z - max), and the lowest column holding the max. max = -inf: no
// column yet.
struct RowState {
  float m, s, t;
  int a;
};

// Both merges below give ties of the max to the lower column.
// `r` covers columns after those of `l`: it takes the argmax only with a
// strictly larger max (the merge order of successive tiles of a panel).
__device__ __forceinline__ void merge_after(RowState& l, const RowState& r) {
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

// Symmetric merge of two states over interleaved columns (the lanes of a row
// group): both partners compute the same bits, because each sum is one
// addition of two products, and addition commutes.
__device__ __forceinline__ void merge_lanes(RowState& l, const RowState& r) {
  if (r.m == -INFINITY) return;
  if (l.m == -INFINITY) {
    l = r;
    return;
  }
  const float m = fmaxf(l.m, r.m);
  const float fl = expf(l.m - m), fr = expf(r.m - m);
  l.s = l.s * fl + r.s * fr;
  l.t = l.t * fl + r.t * fr;
  l.a = (r.m > l.m || (r.m == l.m && r.a < l.a)) ? r.a : l.a;
  l.m = m;
}

// One block per (panel of 64 x panel_tiles columns, block of 64 rows). After
// each tile, every thread folds its 8 columns of each of its 4 rows into a
// row state, the 8 threads of a row group merge theirs by shuffles, and the
// result is merged after the panel's earlier tiles.
template <int KG>
__global__ void __launch_bounds__(KG * kSimtThreads, 4 / KG)
    fwd_simt_kernel(const float* __restrict__ h, const float* __restrict__ w, const FwdArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SimtSmem<KG>& sm = *reinterpret_cast<SimtSmem<KG>*>(smem_raw);
  const int panel = blockIdx.x / a.n_blocks;
  const int rb = blockIdx.x - panel * a.n_blocks;
  const int r0 = rb * T;
  const int g = threadIdx.x / kSimtThreads, lt = threadIdx.x % kSimtThreads;
  const int tx = lt & 7, ty = lt >> 3;
  const float* bias = static_cast<const float*>(a.bias);
  RowState run[4];
  int tgt[4];   // shard-local column of the row's target; -1 if ignored or in another shard
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    run[i] = RowState{-INFINITY, 0.f, 0.f, 0};
    const int row = r0 + ty * 4 + i;
    const long long t = row < a.N ? a.targets[row] - a.vocab_start : -1;
    tgt[i] = (row < a.N && a.targets[row] != a.ignore_index && t >= 0 && t < a.V)
                 ? static_cast<int>(t) : -1;
  }
  const int c_begin = panel * a.panel_tiles * T;
  const int c_end = min(a.V, c_begin + a.panel_tiles * T);
  for (int c0 = c_begin; c0 < c_end; c0 += T) {
    float acc[4][8];
    OperandView va, vb;
    logit_views(h, w, a.H, r0, a.N, c0, a.V, va, vb);
    tile_product(va, vb, 0, a.H, sm, acc);
    if (g != 0) continue;   // group 0 holds the tile's sums
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = r0 + ty * 4 + i;
      float z[8];
      RowState st{-INFINITY, 0.f, 0.f, 0};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int col = c0 + tile_col(tx, j);
        z[j] = col < a.V ? transform_f32(acc[i][j], bias, col, a.scale, a.softcap, a.inv_softcap)
                         : -INFINITY;
        if (col == tgt[i] && row < a.N && store_allowed(&a.zt[row], 4, a.r_zt, a.status))
          a.zt[row] = z[j];
        if (z[j] > st.m) {   // columns increase with j: ties keep the first
          st.m = z[j];
          st.a = col;
        }
      }
      if (st.m > -INFINITY) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float e = expf(z[j] - st.m);   // 0 for the -inf of columns past V
          st.s += e;
          st.t = z[j] > -INFINITY ? fmaf(z[j], e, st.t) : st.t;
        }
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) {
        RowState r;
        r.m = __shfl_xor_sync(0xffffffffu, st.m, o);
        r.s = __shfl_xor_sync(0xffffffffu, st.s, o);
        r.t = __shfl_xor_sync(0xffffffffu, st.t, o);
        r.a = __shfl_xor_sync(0xffffffffu, st.a, o);
        merge_lanes(st, r);
      }
      merge_after(run[i], st);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = r0 + ty * 4 + i;
    if (g == 0 && tx == 0 && row < a.N)
      a.partials[static_cast<size_t>(panel) * a.N + row] =
          make_float4(run[i].m, run[i].s, run[i].t, __int_as_float(run[i].a));
  }
}

// One block per (64-column tile, 64-row block of the chunk).
template <int KG>
__global__ void __launch_bounds__(KG * kSimtThreads, 4 / KG)
    ds_simt_kernel(const float* __restrict__ h, const float* __restrict__ w, const DsArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SimtSmem<KG>& sm = *reinterpret_cast<SimtSmem<KG>*>(smem_raw);
  // per-column sums for grad_bias: the tile's dlogits, staged in 16-byte pieces
  float (&G)[T][T + 4] = *reinterpret_cast<float (*)[T][T + 4]>(smem_raw + sizeof(SimtSmem<KG>));
  // one 1-D grid over the chunk's tiles, column tiles fastest (a 2-D grid
  // would cap the row tiles at 65535)
  const int ct = (a.V + T - 1) / T;
  const int c0 = static_cast<int>(blockIdx.x % ct) * T;
  const int rb = static_cast<int>(blockIdx.x / ct);
  const int r0 = rb * T;  // local to the chunk
  const int tid = threadIdx.x, g = tid / kSimtThreads, lt = tid % kSimtThreads;
  const int tx = lt & 7, ty = lt >> 3;
  const float* bias = static_cast<const float*>(a.bias);
  float acc[4][8];
  OperandView va, vb;
  logit_views(h + static_cast<size_t>(a.row0) * a.H, w, a.H, r0, a.rows, c0, a.V, va, vb);
  tile_product(va, vb, 0, a.H, sm, acc);
  float* ds = static_cast<float*>(a.ds);
#pragma unroll
  for (int i = 0; i < 4 && g == 0; ++i) {
    const int rl = r0 + ty * 4 + i;
    const bool row_ok = rl < a.rows;
    const float4 cf = row_ok ? a.coef[a.row0 + rl] : make_float4(0.f, 0.f, 0.f, __int_as_float(-1));
    const int tgt = __float_as_int(cf.w) - a.tgt_base;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float g[4];
      const int col0 = c0 + tile_col(tx, 4 * half);
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int col = col0 + jj;
        g[jj] = 0.f;
        if (row_ok && col < a.V) {
          const float z = transform_f32(acc[i][4 * half + jj], bias, col, a.scale, a.softcap,
                                        a.inv_softcap);
          const float p = expf(z - cf.z);
          g[jj] = cf.x * p;
          if (col == tgt) g[jj] -= cf.y;
          if (a.softcap > 0.f) {
            const float zc = z * a.inv_softcap;
            g[jj] *= (1.f - zc * zc);
          }
        }
      }
      if (a.bias_part != nullptr)
        *reinterpret_cast<float4*>(&G[ty * 4 + i][tile_col(tx, 4 * half)]) =
            make_float4(g[0], g[1], g[2], g[3]);
      if (row_ok && col0 < a.V) {
        float* const dst = ds + static_cast<size_t>(rl) * a.V_pad + col0;
        // four neighbouring columns: one 16-byte store when all are in the row
        if (col0 + 3 < a.V && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
          if (store_allowed(dst, 16, a.r_ds, a.status))
            *reinterpret_cast<float4*>(dst) = make_float4(g[0], g[1], g[2], g[3]);
        } else {
          for (int jj = 0; jj < 4 && col0 + jj < a.V; ++jj)
            if (store_allowed(dst + jj, 4, a.r_ds, a.status)) dst[jj] = g[jj];
        }
      }
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

// Output tile (bx, by) of 64 x 64 and K split bz of one product.
template <int KG>
__device__ __forceinline__ void gemm_simt_block(const SimtGemmArgs& a, int bx, int by, int bz) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SimtSmem<KG>& sm = *reinterpret_cast<SimtSmem<KG>*>(smem_raw);
  const int m0 = by * T, n0 = bx * T;
  const int tid = threadIdx.x, g = tid / kSimtThreads, lt = tid % kSimtThreads;
  const int tx = lt & 7, ty = lt >> 3;
  // this block's K range: all of K, or split bz of k_splits
  const int kc = a.k_splits > 1 ? (a.K + a.k_splits - 1) / a.k_splits : a.K;
  const int kb = bz * kc;
  const int ke = min(a.K, kb + kc);
  // Neighbouring threads read neighbouring addresses: along K for an operand
  // whose K stride is 1, else along M (or N).
  float acc[4][8];
  // A(k, m) = A[m * sam + k * sak], B(k, n) = B[k * sbk + n * sbn], from k = kb
  const OperandView va{a.A + m0 * a.sam + static_cast<long long>(kb) * a.sak, a.sam, a.sak, a.M - m0,
                       a.sak == 1};
  const OperandView vb{a.B + n0 * a.sbn + static_cast<long long>(kb) * a.sbk, a.sbn, a.sbk, a.N - n0,
                       a.sbk == 1 && a.sbn != 1};
  tile_product(va, vb, 0, ke - kb, sm, acc);
#pragma unroll
  for (int i = 0; i < 4 && g == 0; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= a.M) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int n = n0 + tile_col(tx, j);
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
  if (a.k_splits <= 1 || a.tile_count == nullptr) return;
  // The last of this tile's splits to finish adds the other splits' partials
  // to C, in split order, so the sum does not depend on which block that is.
  // Each block makes its stores visible before it counts itself; the last
  // one reads the others' stores (from L2) only after it has seen the count.
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    int* const cnt = a.tile_count + by * ((a.N + T - 1) / T) + bx;
    s_last = atomicAdd(cnt, 1) == a.k_splits - 1;
    if (s_last) *cnt = 0;   // every split has counted: zero again for the next product
  }
  __syncthreads();
  if (!s_last || g != 0) return;
  __threadfence();
  // Row by row; within a row, split by split, so that a thread's loads of
  // one split are in flight together. The sum per element is still
  // ((0 + p_1) + p_2) + ... in split order.
  const size_t plane = static_cast<size_t>(a.M) * a.N;
#pragma unroll 1
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= a.M) break;
    float sum[8], cv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int n = n0 + tile_col(tx, j);
      sum[j] = 0.f;
      cv[j] = n < a.N ? __ldcg(a.C + m * a.ldc + n) : 0.f;
    }
    for (int z = 0; z + 1 < a.k_splits; ++z) {
      const float* const pz = a.part + z * plane + size_t(m) * a.N;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int n = n0 + tile_col(tx, j);
        if (n < a.N) sum[j] += __ldcg(pz + n);
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int n = n0 + tile_col(tx, j);
      if (n >= a.N) continue;
      float* c = a.C + m * a.ldc + n;
      if (store_allowed(c, 4, a.r_c, a.status)) *c = cv[j] + sum[j];
    }
  }
}

template <int KG>
__global__ void __launch_bounds__(KG * kSimtThreads, 4 / KG) gemm_simt_kernel(const SimtGemmArgs a) {
  // one 1-D grid: column tiles fastest, then row tiles, then K splits
  const int nx = (a.N + T - 1) / T, ny = (a.M + T - 1) / T;
  const int b = static_cast<int>(blockIdx.x);
  gemm_simt_block<KG>(a, b % nx, (b / nx) % ny, b / (nx * ny));
}

// Two independent products in one grid: units [0, n1) are the first
// product's (tile, split) blocks, the rest the second's; each alone is too
// small to fill the GPU at the sizes this path serves. With sched == nullptr
// block b computes unit b. Otherwise the grid is persistent and takes units
// in order from sched[0] (the host puts the product with the longer K per
// unit first, so the long units start first and the short ones fill in);
// sched[1] counts the blocks that have finished, and the last one zeroes
// both for the next launch. Which block computes a unit does not change its
// result.
template <int KG>
__global__ void __launch_bounds__(KG * kSimtThreads, 4 / KG)
    gemm_simt2_kernel(const SimtGemmArgs a1, const SimtGemmArgs a2, int n1, int n_units,
                      int* sched) {
  __shared__ int s_unit;
  for (int it = 0;; ++it) {
    if (threadIdx.x == 0)
      s_unit = sched != nullptr ? atomicAdd(sched, 1)
                                : (it == 0 ? static_cast<int>(blockIdx.x) : n_units);
    __syncthreads();
    const int u = s_unit;
    __syncthreads();   // every thread has read s_unit before it changes
    if (u >= n_units) break;
    const bool first = u < n1;
    const SimtGemmArgs& a = first ? a1 : a2;
    const int i = first ? u : u - n1;
    const int gx = (a.N + T - 1) / T, gy = (a.M + T - 1) / T;
    gemm_simt_block<KG>(a, i % gx, (i / gx) % gy, i / (gx * gy));
  }
  if (sched != nullptr && threadIdx.x == 0 &&
      atomicAdd(sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
    // every block is past its last fetch
    sched[0] = 0;
    sched[1] = 0;
  }
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

namespace {
template <class K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(bytes));
}

// K groups per block: two (256 threads, two blocks per SM by registers) while
// the grid has at most two blocks per SM, so that few tiles still bring many
// warps; otherwise one (128 threads, four blocks per SM), so that a larger
// grid runs in one wave.
int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 0;
  return sms;
}

int groups_for(long long blocks) { return blocks <= 2ll * sm_count() ? 2 : 1; }

template <int KG>
cudaError_t launch_fwd_kg(const float* h, const float* w, const FwdArgs& a, cudaStream_t s) {
  const size_t bytes = sizeof(SimtSmem<KG>);
  cudaError_t e = set_smem(fwd_simt_kernel<KG>, bytes);
  if (e != cudaSuccess) return e;
  fwd_simt_kernel<KG><<<a.num_units, KG * kSimtThreads, bytes, s>>>(h, w, a);
  note_launch();
  return cudaGetLastError();
}

template <int KG>
cudaError_t launch_ds_kg(const float* h, const float* w, const DsArgs& a, dim3 grid,
                         cudaStream_t s) {
  const size_t bytes = sizeof(SimtSmem<KG>) + sizeof(float) * T * (T + 4);
  cudaError_t e = set_smem(ds_simt_kernel<KG>, bytes);
  if (e != cudaSuccess) return e;
  ds_simt_kernel<KG><<<grid, KG * kSimtThreads, bytes, s>>>(h, w, a);
  note_launch();
  return cudaGetLastError();
}

template <int KG>
cudaError_t launch_gemm2_kg(const SimtGemmArgs& a1, const SimtGemmArgs& a2, int n1, int n2,
                            int grid, int* sched, cudaStream_t s) {
  const size_t bytes = sizeof(SimtSmem<KG>);
  cudaError_t e = set_smem(gemm_simt2_kernel<KG>, bytes);
  if (e != cudaSuccess) return e;
  gemm_simt2_kernel<KG><<<grid, KG * kSimtThreads, bytes, s>>>(a1, a2, n1, n1 + n2, sched);
  note_launch();
  return cudaGetLastError();
}

template <int KG>
cudaError_t launch_gemm_kg(const SimtGemmArgs& a, dim3 grid, cudaStream_t s) {
  const size_t bytes = sizeof(SimtSmem<KG>);
  cudaError_t e = set_smem(gemm_simt_kernel<KG>, bytes);
  if (e != cudaSuccess) return e;
  gemm_simt_kernel<KG><<<grid, KG * kSimtThreads, bytes, s>>>(a);
  note_launch();
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_fwd_simt(const float* h, const float* w, const FwdArgs& a, cudaStream_t s) {
  return groups_for(a.num_units) == 2 ? launch_fwd_kg<2>(h, w, a, s) : launch_fwd_kg<1>(h, w, a, s);
}

cudaError_t launch_ds_simt(const float* h, const float* w, const DsArgs& a, cudaStream_t s) {
  const long long tiles = static_cast<long long>((a.V + T - 1) / T) * ((a.rows + T - 1) / T);
  if (tiles > 0x7fffffffll) return cudaErrorInvalidConfiguration;
  const dim3 grid(static_cast<unsigned>(tiles));
  // at most one tile per SM: four K groups (16 warps) per block
  if (tiles <= sm_count()) return launch_ds_kg<4>(h, w, a, grid, s);
  return groups_for(tiles) == 2 ? launch_ds_kg<2>(h, w, a, grid, s)
                                : launch_ds_kg<1>(h, w, a, grid, s);
}

namespace {
int simt_blocks(const SimtGemmArgs& a) {
  return ((a.N + T - 1) / T) * ((a.M + T - 1) / T) * (a.k_splits > 1 ? a.k_splits : 1);
}
cudaError_t split_reduce_after(const SimtGemmArgs& a, cudaStream_t s) {
  if (a.k_splits <= 1 || a.tile_count != nullptr) return cudaSuccess;
  const long long total = static_cast<long long>(a.M) * a.N;
  const int blocks = static_cast<int>(min(4096ll, (total + 255) / 256));
  simt_split_reduce_kernel<<<blocks, 256, 0, s>>>(a);
  note_launch();
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_gemm_simt2(const SimtGemmArgs& a1, const SimtGemmArgs& a2, int* sched,
                              cudaStream_t s) {
  // K per unit: the longer units go first
  auto unit_k = [](const SimtGemmArgs& a) {
    return a.k_splits > 1 ? (a.K + a.k_splits - 1) / a.k_splits : a.K;
  };
  const bool swap = unit_k(a2) > unit_k(a1);
  const SimtGemmArgs& p1 = swap ? a2 : a1;
  const SimtGemmArgs& p2 = swap ? a1 : a2;
  const int n1 = simt_blocks(p1), n2 = simt_blocks(p2);
  cudaError_t e;
  if (sched != nullptr) {
    // persistent: two 256-thread blocks per SM
    const int cap = 2 * sm_count();
    const int grid = n1 + n2 < cap || cap < 1 ? n1 + n2 : cap;
    e = launch_gemm2_kg<2>(p1, p2, n1, n2, grid, sched, s);
  } else {
    e = groups_for(n1 + n2) == 2 ? launch_gemm2_kg<2>(p1, p2, n1, n2, n1 + n2, nullptr, s)
                                 : launch_gemm2_kg<1>(p1, p2, n1, n2, n1 + n2, nullptr, s);
  }
  if (e != cudaSuccess) return e;
  if ((e = split_reduce_after(a1, s)) != cudaSuccess) return e;
  return split_reduce_after(a2, s);
}

cudaError_t launch_gemm_simt(const SimtGemmArgs& a, cudaStream_t s) {
  const int splits = a.k_splits > 1 ? a.k_splits : 1;
  const long long blocks =
      static_cast<long long>((a.N + T - 1) / T) * ((a.M + T - 1) / T) * splits;
  if (blocks > 0x7fffffffll) return cudaErrorInvalidConfiguration;
  const dim3 grid(static_cast<unsigned>(blocks));
  cudaError_t e = groups_for(blocks) == 2 ? launch_gemm_kg<2>(a, grid, s)
                                          : launch_gemm_kg<1>(a, grid, s);
  if (e != cudaSuccess) return e;
  return split_reduce_after(a, s);
}

}  // namespace flce
