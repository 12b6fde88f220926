// Internal interface between the host runtime (flce.cu) and the kernel
// translation units. It is not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace flce {

// Device status bits written to the workspace status word. The host maps
// them to FLCE_ERR_* codes. kDevErrBounds is set only by builds with
// FLCE_DEBUG (see DevRegion).
enum : int { kDevErrTargetRange = 1, kDevErrTimeout = 2, kDevErrBounds = 4 };

// A buffer a kernel may write: [base, base + bytes). Builds with FLCE_DEBUG
// check every store of the kernels against the region of its buffer; a store
// that would land outside sets kDevErrBounds in the status word and is
// skipped. Other builds ignore the regions.
struct DevRegion {
  const void* base;
  unsigned long long bytes;
};

// ---- tcgen05 tile shape shared by every bf16 kernel -----------------------
// CTAs run in pairs (clusters of 2) with the 2-SM MMA (cta_group::2).
// - A pair computes a 256 x 256 fp32 tile. Each CTA owns 128 rows of it in
//   its own TMEM, double-buffered (2 x 256 of its 512 TMEM columns).
// - Each CTA stages its 128 rows of A and its half (128 rows) of B in 64-deep
//   K slices, one 128-byte swizzle row of bf16, through a 6-stage TMA ring.
constexpr int kBM = 128;                         // rows of the tile per CTA
constexpr int kPairM = 256;                      // rows of the tile per pair
constexpr int kBN = 256;                         // columns of the tile
constexpr int kBNHalf = 128;                     // B rows staged per CTA
constexpr int kBK = 64;
constexpr int kStages = 6;
constexpr int kStageA = kBM * kBK * 2;           // 16 KB
constexpr int kStageB = kBNHalf * kBK * 2;       // 16 KB
constexpr int kStageBytes = kStageA + kStageB;   // 32 KB per CTA
constexpr int kTcThreads = 192;                  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
// The dlogits kernel has two epilogue warps per TMEM lane quarter (warps 2-9),
// each on half of a tile's 256 columns: its epilogue (exp, softcap, two
// stores, bias sums) outlasts the MMAs of a tile when H is small.
constexpr int kDsThreads = 320;
constexpr int kTmemCols = 512;
// dynamic shared memory: 1 KB alignment slack + stages + 8 KB scratch + control block
constexpr int kTcSmemBytes = 1024 + kStages * kStageBytes + 8192 + 1024;

// ---- fp32 SIMT path tile shape -------------------------------------------
constexpr int kSimtTile = 64;        // 64 x 64 logit tiles
constexpr int kSimtPanelCols = 256;  // widest partial-state panel of the fp32 forward (columns)
constexpr int kSimtThreads = 128;
constexpr int kSimtSplitTiles = 256;  // K-split SIMT GEMMs have fewer output tiles than this
constexpr int kSimtSchedWords = 2;    // unit counter and finished-block count of a persistent SIMT grid

// Per (panel, row) partial state of the online log-sum-exp:
// x = running max m, y = sum exp(z - m), z = sum z exp(z - m), w = argmax (int bits).

// The vocabulary sweeps (forward, dlogits) hand out units (panel, pair block)
// in groups of `group_blocks` pair blocks: within a group panel-major, one
// group after the other. A group's rows of h (group_blocks x 256 x H x 2 bytes,
// about 32 MB) stay in L2 while the W panels stream through once per group.
__host__ __device__ inline void decode_unit(int u, int n_blocks, int group_blocks,
                                            int num_panels, int& panel, int& nb) {
  const int per_group = group_blocks * num_panels;
  const int g = u / per_group;
  const int r = u - g * per_group;
  const int rest = n_blocks - g * group_blocks;
  const int gb = rest < group_blocks ? rest : group_blocks;  // the last group may be smaller
  panel = r / gb;
  nb = g * group_blocks + (r - panel * gb);
}

// Clock record of one launch, filled only while profiling is on: the sum over
// the launch's CTAs of SM clock cycles (clock64) and of nanoseconds
// (%globaltimer) from the CTA's start to its end. Their ratio is the launch's
// mean SM clock. The MMA-issuing threads also add the cycles of their role,
// and the cycles they spent waiting for operands (TMA loads) and for a free
// accumulator (the epilogue).
struct ClockRecord {
  unsigned long long cycles, ns;
  unsigned long long mma_cycles, mma_wait_operands, mma_wait_accumulator;
};

struct FwdArgs {
  int N, H, V;
  ClockRecord* clk;            // nullable (profiling)
  int group_blocks;
  long long vocab_start;       // global id of this call's first vocabulary row
  unsigned long long wait_ns;  // limit of every bounded wait (kWaitLimitNs unless testing)
  int drop_kb;                 // fault injection, off (-1) unless testing: the even CTA of the
                               // pair that has unit 0 arms but never issues the loads of this
                               // K slice of that unit's first tile
  int n_blocks, v_tiles, panel_tiles, num_panels, num_units;
  // Dynamic schedule, as GemmArgs::tile_counter: two zeroed ints (left zero)
  // from which the pairs take (panel, pair block) units in order; nullptr:
  // round-robin.
  int* tile_counter;
  float scale, softcap, inv_softcap;
  const void* bias;            // dtype of the pass, or nullptr
  const int64_t* targets;
  long long ignore_index;
  float4* partials;            // [num_panels][N]
  float* zt;                   // [N] transformed target logit
  int* status;
  DevRegion r_partials, r_zt;
};

struct FinalizeArgs {
  int nblk, reduction;
  const int* status;           // kDevErrTimeout set: loss and entropy NaN, num_correct -1
  const double* blk_loss;
  const double* blk_ent;
  const long long* blk_correct;
  const long long* blk_valid;
  float* loss;                 // [1] for sum/mean, nullptr for none
  int64_t* num_correct;        // nullable
  float* entropy_sum;          // nullable
};

// The merge's blocks count themselves on `done` (a zeroed word of the
// workspace header) after storing their block sums; the last one to arrive
// sums all blocks' sums in block order and writes the reduced outputs, as
// finalize_kernel does, so the forward needs no separate finalize launch.
// done == nullptr: the block sums are left for finalize_kernel.

// A forward whose bounded wait expired skipped some partial-state stores, so
// the merge would combine whatever the workspace held before. merge_kernel
// reads the status word first (the stream orders it after the forward) and
// then writes NaN to every lse and loss instead.
struct MergeArgs {
  int N, V, num_panels, reduction;
  int lanes;                   // threads per row (a power of two <= 32); the grid covers N x lanes
  long long vocab_start, vocab_total;   // shard placement; vocab_total = V when not sharded
  long long ignore_index;
  float zeta;
  const float4* partials;
  const float* zt;
  const int64_t* targets;
  float* lse;                  // [N]
  float* loss_rows;            // [N] when reduction == none, else nullptr
  double* blk_loss;            // [gridDim]
  double* blk_ent;
  long long* blk_correct;
  long long* blk_valid;
  int* status;
  int* done;                   // nullable: blocks-done counter, zero at launch
  FinalizeArgs fin;            // the reduced outputs, when done != nullptr
};

// Exported per-row state of one vocabulary shard (20 bytes): running max,
// sum of exp(z - max), sum of z exp(z - max), global argmax, and the target
// logit if this shard holds the target (0 otherwise).
struct ShardState {
  float m, s, t;
  int argmax;
  float zt;
};

struct ShardStateArgs {
  int N, V, num_panels;
  const int* status;           // kDevErrTimeout set: every state is NaN (the partials are incomplete)
  long long vocab_start;
  long long ignore_index;
  const float4* partials;
  const float* zt;
  const int64_t* targets;
  ShardState* out;             // [N]
};

// Merge of R shards' states into the same outputs merge_kernel produces.
struct CombineArgs {
  int N, R, reduction;
  long long vocab_total;
  long long ignore_index;
  float zeta;
  const ShardState* states;    // [R][N]
  const int64_t* targets;
  float* lse;
  float* loss_rows;
  double* blk_loss;
  double* blk_ent;
  long long* blk_correct;
  long long* blk_valid;
  int* status;
  int* done;                   // nullable: as in MergeArgs
  FinalizeArgs fin;
};

// Backward per-row coefficients: x = s*gamma*(1 + 2 zeta lse), y = s*gamma,
// z = lse, w = target (int bits; -1 if ignored or out of the row range).
struct RowCoefArgs {
  int N, V, reduction;
  long long vocab_start, vocab_total;   // shard placement; vocab_total = V when not sharded
  long long ignore_index;
  float scale, zeta;
  const int64_t* targets;
  const float* lse;
  const float* grad_loss;
  float4* coef;
  float* ds_scale;             // nullable: receives {S, 1/S}, S = 2^k with max |dlogits| * S <= 2^14
  int* status;
  // The first words of the workspace (the header with the status word, then
  // the tile counters of the K-split GEMMs), zeroed before anything else: the
  // backward's first kernel does this in place of a memset.
  int* zero;
  int zero_words;
};

struct DsArgs {
  int rows, row0, H, V, V_pad;
  int* tile_counter;           // dynamic schedule as in FwdArgs; nullptr: round-robin
  ClockRecord* clk;            // nullable (profiling)
  int group_blocks;
  int n_blocks, v_tiles, panel_tiles, num_panels, num_units;
  float scale, softcap, inv_softcap;
  const void* bias;
  const float4* coef;          // indexed by global row
  const float* ds_scale;       // fp16: power of two that dlogits is stored times; else nullptr
  void* ds;                    // chunk buffer [rows][V_pad] in the input dtype (f32 for fp32)
  void* ds_t;                  // the same values transposed, [V][ld_t] (16-bit types); or nullptr
  long long ld_t;              // row stride of ds_t, in elements
  float* bias_part;            // [row blocks][bias_ld], offset to this chunk's first column; or nullptr
  int bias_ld;                 // row stride of bias_part
  int bias_blk0;               // first row block of this chunk
  int tgt_base;                // shard-local column of this chunk's first column
  int* status;
  DevRegion r_ds, r_ds_t, r_bias;
};

enum GemmMode : int {
  kStoreOut = 0,      // out  = acc (output dtype)
  kStorePart = 1,     // part = acc (fp32)
  kAddPart = 2,       // part = part + acc
  kAddPartToOut = 3,  // out  = part + acc
  kAddOutToOut = 4,   // out  = out + acc (read-modify-write in the output dtype)
  kAddOutToPart = 5,  // part = out + acc
  // A row- and feature-weighted squared error on the accumulator, whose
  // logits are never stored: out = 2 r_m f_n (acc - y_mn) in the output dtype,
  // and loss_part[n_tile][m / 32] = sum over the tile's columns and the 32
  // rows m / 32 of r_m f_n (acc - y_mn)^2 (fp32). Needs k_splits == 1.
  kWeightedMse = 6,
  // out_t = acc transposed, in the output dtype: out_t[n * ld_out_t + m] for
  // the tile's rows m and columns n. Needs k_splits == 1.
  kStoreOutT = 7,
  // out_t = out_t + acc transposed (read-modify-write in the output dtype,
  // one rounding). Needs k_splits == 1.
  kAddOutToOutT = 8,
  // out_t = (part + acc) transposed: the fp32 partial is in the tile's own
  // layout, part[m * ld_part + n]. Needs k_splits == 1.
  kAddPartToOutT = 9
};

// One plain GEMM D[M,N] = A[M,K] B[K,N] in 256 x 256 pair tiles. With
// k_splits > 1 the K loop of every tile is cut into k_splits contiguous
// ranges. Split s of tile (m, n) writes its fp32 result to
// part + s * split_stride, and split_reduce_kernel later sums the splits in
// order. Units are ordered split-major, so the units that run at the same
// time share their K range.
struct GemmArgs {
  int M, N, K;
  ClockRecord* clk;            // nullable (profiling)
  int m_tiles, n_tiles, k_blocks, num_tiles;
  int k_splits, kb_per_split;
  int group_m;                 // row tiles per raster group (decode_unit; 1: row after row)
  int a_mn, b_mn;              // 1: operand is MN-major in memory
  int a_atoms, b_atoms;        // full 64-column atoms in the operand's 3-D view (0: none)
  int mode;                    // GemmMode (kStorePart when k_splits > 1)
  void* out;
  long long ld_out;
  float* part;
  long long ld_part;
  long long split_stride;      // elements between split partial buffers
  const float* acc_scale;      // nullable: the accumulator is multiplied by *acc_scale first
  int* status;
  // kWeightedMse only
  const float* target;         // y [M][ld_target], fp32
  long long ld_target;         // multiple of 4
  const float* row_w;          // r [M]
  const float* feat_w;         // f [N]
  float* loss_part;            // [n_tiles][ceil(M / 32)]
  void* out_t;                 // nullable: out transposed as well, [N][ld_out_t]
  long long ld_out_t;
  DevRegion r_out, r_part, r_out_t, r_loss;
  // Dynamic schedule: two ints, zero before the launch and left zero after it.
  // [0] hands out units in order, [1] counts the pairs that have finished
  // taking units. nullptr: every pair takes units u = pair, pair + npairs, ...
  int* tile_counter;
  // L2 policy of each operand's loads: kL2Normal, kL2EvictFirst (a stream
  // read once) or kL2EvictLast (an operand every wave of tiles re-reads).
  int a_l2, b_l2;
};

enum L2Policy : int { kL2Normal = 0, kL2EvictFirst = 1, kL2EvictLast = 2 };

// dst[c * ld_dst + r] = src[r * ld_src + c] for a rows x cols matrix of 16-bit
// elements (bf16 or fp16: the bits are moved, not converted).
struct TransposeArgs {
  const uint16_t* src;
  uint16_t* dst;
  int rows, cols;
  long long ld_src, ld_dst;
  int* status;
  DevRegion r_dst;
};

// dst[i] = src[i] * (*scale), i < count, in the element type (dtype 0 fp32,
// 1 bf16, 2 fp16). src == dst is allowed. With *scale == 1 and src == dst
// every thread returns at once.
struct ScaleArgs {
  const void* src;
  void* dst;
  long long count;
  int dtype;
  const float* scale;
};

// loss = (accumulate ? loss : 0) + sum of part[0 .. count), in a fixed order.
struct LossReduceArgs {
  const float* part;
  long long count;
  double* loss;
  int accumulate;
};

// out[m, n] (bf16) = sum over s of part[s][m, n], in split order.
struct SplitReduceArgs {
  int M, N, splits;
  int accumulate;              // 1: out += sum (read-modify-write)
  int f16;                     // output dtype: 1 fp16, 0 bf16
  const float* part;
  long long ld_part, split_stride;
  void* out;
  long long ld_out;
};

struct SimtGemmArgs {
  int M, N, K;
  const float* A;              // A(m,k) = A[m*sam + k*sak]
  long long sam, sak;
  const float* B;              // B(k,n) = B[k*sbk + n*sbn]
  long long sbk, sbn;
  float* C;                    // C[m*ldc + n]
  long long ldc;
  int accumulate;              // 1: C += A B, 0: C = A B
  // k_splits > 1: split 0 of the K range writes C (adds to it when
  // accumulate); split s > 0 stores its fp32 product to part + (s - 1) * M * N
  // ([M][N], row-major). Those are added to C in split order by the last of
  // a tile's splits to finish when tile_count is given (one zeroed counter
  // per 64 x 64 output tile, left zero again), else by a second kernel. For
  // outputs with few 64 x 64 tiles and a long K.
  int k_splits;
  float* part;
  int* tile_count;
  int* status;                 // nullable; receives kDevErrBounds (FLCE_DEBUG builds)
  DevRegion r_c, r_part;
};

struct BiasReduceArgs {
  int V, V_pad, nblk;
  int accumulate;              // 1: grad_bias += sum
  const float* bias_part;      // [nblk][V_pad]
  void* grad_bias;             // dtype of the pass
};

// Counts one kernel launch of this library (flce_launch_count); called after
// every kernel launch statement.
void note_launch();

// tcgen05 / TMA kernels (bf16). `grid` is the number of CTA pairs.
cudaError_t tc_max_active_pairs(int* pairs);
// f16 selects fp16 operands and outputs; otherwise bf16.
// metrics: also keep each row's argmax and sum z exp(z - m) (needed for
// num_correct, entropy_sum and exported shard states); loss and lse are the
// same bits either way.
cudaError_t launch_fwd_tc(const CUtensorMap& tm_h, const CUtensorMap& tm_w, const FwdArgs& a,
                          bool f16, bool has_bias, bool softcap, bool metrics, int grid,
                          cudaStream_t s);
cudaError_t launch_ds_tc(const CUtensorMap& tm_h, const CUtensorMap& tm_w, const DsArgs& a,
                         bool f16, bool has_bias, bool softcap, int grid, cudaStream_t s);
// A GEMM operand in global memory. `map` is its 2-D tensor map: 64 x 128
// boxes (K x rows) when K-major, 64 x 64 boxes (MN x K) when MN-major. An
// MN-major operand [K rows][MN cols] also gets `map3`, a 3-D view of the same
// memory with the 64-column atoms as the outer dimension, so that one TMA load
// brings a CTA's two atoms (128 columns) instead of two loads. In a plain
// GEMM with both operands MN-major (M = 8192, N = 4096, K = 8192, on the
// GB300) the view on B alone took 0.466 ms to 0.399 ms. The view holds only
// the operand's full atoms, so it never reads past the end of a row; a tile
// that reaches past them (GemmArgs a_atoms / b_atoms) loads through `map`.
struct GemmOperand {
  CUtensorMap map;
  CUtensorMap map3;
};

cudaError_t launch_gemm_tc(const GemmOperand& op_a, const GemmOperand& op_b, const GemmArgs& a,
                           bool f16, int grid, cudaStream_t s);

// SIMT kernels (fp32)
cudaError_t launch_fwd_simt(const float* h, const float* w, const FwdArgs& a, cudaStream_t s);
cudaError_t launch_ds_simt(const float* h, const float* w, const DsArgs& a, cudaStream_t s);
cudaError_t launch_gemm_simt(const SimtGemmArgs& a, cudaStream_t s);
// Two independent products in one launch (then each one's split reduction).
// Both products in one grid. sched: nullable, two zeroed ints (left zero)
// that make the grid persistent, taking (tile, split) units longest first.
cudaError_t launch_gemm_simt2(const SimtGemmArgs& a1, const SimtGemmArgs& a2, int* sched,
                              cudaStream_t s);

// dtype-generic small kernels (dtype: 0 = f32, 1 = bf16, 2 = fp16)
cudaError_t launch_merge(const MergeArgs& a, int nblk, cudaStream_t s);
cudaError_t launch_shard_state(const ShardStateArgs& a, cudaStream_t s);
cudaError_t launch_combine(const CombineArgs& a, int nblk, cudaStream_t s);
cudaError_t launch_finalize(const FinalizeArgs& a, cudaStream_t s);
cudaError_t launch_row_coef(const RowCoefArgs& a, cudaStream_t s);
cudaError_t launch_transpose16(const TransposeArgs& a, cudaStream_t s);
cudaError_t launch_bias_reduce(const BiasReduceArgs& a, int dtype, cudaStream_t s);
cudaError_t launch_split_reduce(const SplitReduceArgs& a, cudaStream_t s);
cudaError_t launch_loss_reduce(const LossReduceArgs& a, cudaStream_t s);
cudaError_t launch_scale(const ScaleArgs& a, int sms, cudaStream_t s);

constexpr int kMergeThreads = 256;

// Host side: sets the text flce_last_error_detail returns on this thread.
void set_error_detail(const char* msg);

}  // namespace flce
