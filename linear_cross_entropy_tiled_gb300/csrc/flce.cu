// Host runtime behind the C ABI declared in include/flce.h: argument
// validation, workspace layout, TMA tensor maps, tile-schedule selection and
// the launch sequence of each pass.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <cmath>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "flce.h"
#include "kernels.h"
#include "ptx.cuh"

#ifndef FLCE_NO_NVTX
#include <nvtx3/nvToolsExt.h>
#endif

using namespace flce;

namespace {

// An NVTX range over one entry point, so that profilers (ncu --nvtx, nsys)
// can select a pass by name. Without an attached tool the calls cost a few
// nanoseconds. Builds with FLCE_NO_NVTX leave them out.
struct NvtxRange {
  explicit NvtxRange(const char* name) {
#ifndef FLCE_NO_NVTX
    nvtxRangePushA(name);
#else
    (void)name;
#endif
  }
  ~NvtxRange() {
#ifndef FLCE_NO_NVTX
    nvtxRangePop();
#endif
  }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// ------------------------------------------------------------ device state
struct DeviceInfo {
  bool init = false;
  int sms = 0;
  int pairs = 0;  // co-resident CTA pairs of the tcgen05 kernels
  int major = 0, minor = 0;
};
std::mutex g_mu;
DeviceInfo g_dev[64];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::atomic<uint64_t> g_launches{0};
thread_local char g_detail[256] = "";

// Test hook for the bounded waits (flce_test_fault): the forward launches of
// this host thread starve one pipeline stage and shorten every wait.
thread_local int g_test_drop_kb = -1;
thread_local unsigned long long g_test_wait_ns = 0;

// Builds with FLCE_DEBUG check every kernel store against its buffer (see
// DevRegion). There, each entry point ends by synchronising its stream and
// returns FLCE_ERR_BOUNDS if a store fell outside; other builds return `v`
// at once and stay asynchronous.
int debug_finish(const void* ws, cudaStream_t st, int v) {
#ifdef FLCE_DEBUG
  if (v != FLCE_OK || ws == nullptr) return v;
  int word = 0;
  if (cudaMemcpyAsync(&word, ws, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return FLCE_ERR_CUDA;
  if (word & kDevErrBounds) {
    snprintf(g_detail, sizeof(g_detail), "debug build: a kernel store fell outside its buffer");
    return FLCE_ERR_BOUNDS;
  }
#else
  (void)ws;
  (void)st;
#endif
  return v;
}

int cuda_fail(cudaError_t e, const char* what) {
  snprintf(g_detail, sizeof(g_detail), "%s: %s", what, cudaGetErrorString(e));
  return FLCE_ERR_CUDA;
}

int device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return FLCE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.init) {
    if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
        return cuda_fail(e, "cuTensorMapEncodeTiled entry point");
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    if (d.major == 10 && d.minor == 3) {
      if ((e = tc_max_active_pairs(&d.pairs)) != cudaSuccess || d.pairs <= 0) d.pairs = d.sms / 2;
    }
    d.init = true;
  }
  *out = d;
  if (d.major != 10 || d.minor != 3) {
    snprintf(g_detail, sizeof(g_detail), "device is sm_%d%d; this library is built for sm_103a",
             d.major, d.minor);
    return FLCE_ERR_UNSUPPORTED;
  }
  return FLCE_OK;
}

// -------------------------------------------------------------- profiling
// While profiling is on, each tensor-core launch also sums its CTAs' SM clock
// cycles and nanoseconds into one record of this fixed array (static device
// memory of the library image; nothing is allocated). flce_profiling_read
// turns them into each kernel's mean SM clock.
constexpr int kClockSlots = 4096;
__device__ ClockRecord g_clock_records[kClockSlots];

struct Pending {
  int name;
  cudaEvent_t e0, e1;
  int dev, slot;   // clock record, or slot -1 when none
};
std::mutex g_prof_mu;
bool g_prof = false;
std::vector<std::string> g_names;
std::vector<uint64_t> g_counts;
std::vector<double> g_ms;
std::vector<Pending> g_pending;
std::vector<cudaEvent_t> g_pool;
std::vector<double> g_cycles, g_clock_ns, g_mma_cycles, g_mma_wait_ops, g_mma_wait_acc;
ClockRecord* g_clock_base[64] = {};
int g_clock_next[64] = {};
cudaStream_t g_clock_stream[64] = {};   // stream that zeroed the array for this read epoch
thread_local ClockRecord* g_cur_clk = nullptr;   // record of the launch being issued

// A zeroed clock record on device `dev` for the next launch, or nullptr. The
// first record of a read epoch zeroes the whole array once, on the launching
// stream, so that the timed launches are not interleaved with a memset each;
// a launch on another stream zeroes its own record.
ClockRecord* take_clock_record(int dev, cudaStream_t s, int* slot) {
  *slot = -1;
  if (dev < 0 || dev >= 64 || g_clock_next[dev] >= kClockSlots) return nullptr;
  if (g_clock_base[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_clock_records) != cudaSuccess || p == nullptr) return nullptr;
    g_clock_base[dev] = static_cast<ClockRecord*>(p);
  }
  ClockRecord* r = g_clock_base[dev] + g_clock_next[dev];
  if (g_clock_next[dev] == 0) {
    if (cudaMemsetAsync(g_clock_base[dev], 0, sizeof(ClockRecord) * kClockSlots, s) != cudaSuccess)
      return nullptr;
    g_clock_stream[dev] = s;
  } else if (s != g_clock_stream[dev] &&
             cudaMemsetAsync(r, 0, sizeof(ClockRecord), s) != cudaSuccess) {
    return nullptr;
  }
  *slot = g_clock_next[dev]++;
  return r;
}

cudaEvent_t pool_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

int name_index(const char* n) {
  for (size_t i = 0; i < g_names.size(); ++i)
    if (g_names[i] == n) return static_cast<int>(i);
  g_names.emplace_back(n);
  g_counts.push_back(0);
  g_ms.push_back(0.0);
  g_cycles.push_back(0.0);
  g_clock_ns.push_back(0.0);
  g_mma_cycles.push_back(0.0);
  g_mma_wait_ops.push_back(0.0);
  g_mma_wait_acc.push_back(0.0);
  return static_cast<int>(g_names.size() - 1);
}

template <class F>
int launch(const char* name, cudaStream_t s, F&& f) {
  std::unique_lock<std::mutex> lk(g_prof_mu);
  const bool prof = g_prof;
  Pending p{};
  p.slot = -1;
  g_cur_clk = nullptr;
  if (prof) {
    p.name = name_index(name);
    cudaGetDevice(&p.dev);
    g_cur_clk = take_clock_record(p.dev, s, &p.slot);
    p.e0 = pool_event();
    cudaEventRecord(p.e0, s);
  }
  lk.unlock();
  const cudaError_t e = f();
  g_cur_clk = nullptr;
  if (prof) {
    lk.lock();
    p.e1 = pool_event();
    cudaEventRecord(p.e1, s);
    g_pending.push_back(p);
  }
  if (e != cudaSuccess) return cuda_fail(e, name);
  return FLCE_OK;
}

// ------------------------------------------------------------ validation
int validate(const flce_params* p) {
  if (p == nullptr) return FLCE_ERR_INVALID_ARG;
  const int64_t lim = (int64_t(1) << 30);
  if (p->N < 0 || p->H < 1 || p->V < 1 || p->N > lim || p->H > lim || p->V > lim)
    return FLCE_ERR_INVALID_ARG;
  if (p->dtype != FLCE_F32 && p->dtype != FLCE_BF16 && p->dtype != FLCE_F16)
    return FLCE_ERR_INVALID_ARG;
  if (p->reduction < FLCE_SUM || p->reduction > FLCE_NONE) return FLCE_ERR_INVALID_ARG;
  if (!isfinite(p->logit_scale) || p->logit_scale == 0.f) return FLCE_ERR_INVALID_ARG;
  if (!isfinite(p->softcap)) return FLCE_ERR_INVALID_ARG;
  if (!isfinite(p->z_loss_multiplier) || p->z_loss_multiplier < 0.f) return FLCE_ERR_INVALID_ARG;
  if (p->has_bias != 0 && p->has_bias != 1) return FLCE_ERR_INVALID_ARG;
  if (p->accumulate != 0 && p->accumulate != 1) return FLCE_ERR_INVALID_ARG;
  if (p->grad_weight_accum != FLCE_ACCUM_FP32 && p->grad_weight_accum != FLCE_ACCUM_WEIGHT)
    return FLCE_ERR_INVALID_ARG;
  if (p->vocab_total == 0) {
    if (p->vocab_start != 0) return FLCE_ERR_INVALID_ARG;
  } else if (p->vocab_start < 0 || p->vocab_total > lim || p->vocab_start + p->V > p->vocab_total) {
    return FLCE_ERR_INVALID_ARG;
  }
  if (p->bwd_chunk_axis < FLCE_CHUNK_AXIS_AUTO || p->bwd_chunk_axis > FLCE_CHUNK_AXIS_VOCAB ||
      p->max_chunk < 0)
    return FLCE_ERR_INVALID_ARG;
  if (p->dtype != FLCE_F32 && (p->H % 8) != 0) return FLCE_ERR_ALIGNMENT;
  return FLCE_OK;
}

bool aligned16(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }

// bf16 and fp16 run on the tensor cores; fp32 on the SIMT path.
bool tensor_path(const flce_params* p) { return p->dtype != FLCE_F32; }

// The tensor path moves 16-byte vectors and TMA boxes; the fp32 SIMT path
// reads single elements, so a row chunk of fp32 data may start anywhere on
// a 4-byte boundary.
bool aligned_for(const flce_params* p, const void* q) {
  return tensor_path(p) ? aligned16(q) : (reinterpret_cast<uintptr_t>(q) & 3u) == 0;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ------------------------------------------------------ workspace layouts
constexpr int kMinPanelTiles = 4;
constexpr int kMaxPanelTiles = 32;
constexpr size_t kHeader = 256;   // status word at 0, fp16 dlogits scale {S, 1/S} at 64,
                                  // the GEMMs' tile counters at 128, the merge's
                                  // blocks-done counter at 136
constexpr size_t kScaleOffset = 64;
constexpr size_t kChunkByteCap = size_t(4) << 30;
constexpr int kMaxKSplits = 2;   // K splits of the grad_hidden GEMM (choose_k_splits)

// K splits of a SIMT (fp32) GEMM: enough 64 x 64 output tiles times splits to
// fill the GPU (about 256 blocks), at least 512 of K per split, at most 16,
// and at most K / N + 1, so that the split partials ((s - 1) x M x N; split 0
// writes the output itself) hold no more than the A operand (M x K, the
// dlogits chunk). A function of the shape only, so the workspace query and
// the launch agree.
int simt_k_splits(int64_t M, int64_t N, int64_t K) {
  const int64_t tiles = ((M + 63) / 64) * ((N + 63) / 64);
  int64_t s = (256 + tiles - 1) / tiles;
  if (s > K / 512) s = K / 512;
  if (s > K / N + 1) s = K / N + 1;
  if (s > 16) s = 16;
  return s < 1 ? 1 : static_cast<int>(s);
}

// Bytes of the fp32 K-split partials of a SIMT GEMM (split 0 needs none).
size_t simt_part_bytes(int64_t M, int64_t N, int64_t K) {
  return size_t(simt_k_splits(M, N, K) - 1) * M * N * 4;
}

// 64-column tiles per panel of the fp32 forward: the widest of 4, 2 and 1
// tiles that still gives at least 152 blocks (one per SM of a GB300), so that
// small problems spread over the GPU, while the merge's per-row loop over the
// panels stays short. A function of the shape only.
int simt_panel_tiles(int64_t N, int64_t V) {
  const int64_t n_blocks = ceil_div(N, kSimtTile);
  for (int pt = kSimtPanelCols / kSimtTile; pt > 1; pt /= 2)
    if (n_blocks * ceil_div(V, int64_t(pt) * kSimtTile) >= 152) return pt;
  return 1;
}

struct FwdLayout {
  int num_panels_max;
  int lanes;   // merge threads per row
  int nblk;    // merge blocks
  size_t partials, zt, blk_loss, blk_ent, blk_correct, blk_valid, total;
  size_t partials_bytes, zt_bytes, blk_bytes;   // bytes the kernels may write in each region
};

FwdLayout fwd_layout(const flce_params* p) {
  FwdLayout L{};
  const int64_t N = p->N, V = p->V;
  if (tensor_path(p))
    L.num_panels_max = static_cast<int>(ceil_div(ceil_div(V, kBN), kMinPanelTiles));
  else
    L.num_panels_max = static_cast<int>(ceil_div(V, int64_t(simt_panel_tiles(N, V)) * kSimtTile));
  // about four panels per merge thread, up to a warp per row
  L.lanes = 1;
  while (L.lanes < 32 && L.lanes * 4 < L.num_panels_max) L.lanes *= 2;
  L.nblk = static_cast<int>(ceil_div(N * L.lanes, kMergeThreads));
  L.partials_bytes = size_t(L.num_panels_max) * N * sizeof(float4);
  L.zt_bytes = size_t(N) * 4;
  L.blk_bytes = size_t(L.nblk) * 8;
  size_t o = kHeader;
  L.partials = o;
  o = align_up(o + L.partials_bytes, 256);
  L.zt = o;
  o = align_up(o + L.zt_bytes, 256);
  L.blk_loss = o;
  o = align_up(o + L.blk_bytes, 256);
  L.blk_ent = o;
  o = align_up(o + L.blk_bytes, 256);
  L.blk_correct = o;
  o = align_up(o + L.blk_bytes, 256);
  L.blk_valid = o;
  o = align_up(o + L.blk_bytes, 256);
  L.total = o;
  return L;
}

struct BwdLayout {
  bool vocab;               // chunks are column ranges of the vocabulary (else row ranges)
  int64_t chunk, V_pad;     // rows (or columns) per chunk
  int64_t ds_ld;            // row stride of the dlogits buffer, in elements
  int64_t ds_t_ld;          // row stride of the transposed dlogits buffer (tensor path)
  int64_t ht_ld;            // row stride of the transposed hidden (tensor path)
  int64_t dw_ld;            // row stride of the fp32 grad_weight partial (row chunks)
  bool wt;                  // grad_weight computed transposed, from h^T and the row-major dlogits
  int nchunks, rowblk, n_rowblocks;
  size_t cnt, coef, ds, ds_t, ht, dw, dh_part, bias_part, total;
  // bytes the kernels may write in each region (0: the region is absent)
  size_t cnt_bytes, coef_bytes, ds_bytes, ds_t_bytes, ht_bytes, dw_bytes, dh_bytes, bias_bytes;
};

// The fp32 path's K-split GEMMs count the finished splits of each output tile
// in a region right after the header, followed by the unit counter of the
// persistent contraction grid; the backward's first kernel zeroes all of it.
void place_counters(const flce_params* p, BwdLayout* L, size_t* o) {
  L->cnt = *o;
  L->cnt_bytes = tensor_path(p) ? 0 : size_t(kSimtSplitTiles + kSimtSchedWords) * 4;
  if (L->cnt_bytes) *o = align_up(*o + L->cnt_bytes, 256);
}

// The backward stores dlogits for one chunk at a time and contracts it into
// both gradients. grad_hidden (K = vocabulary) reads the row-major copy
// K-major. The tensor path computes grad_weight transposed, (h^T dS)^T,
// reading that same copy as its MN-major B operand and a transposed copy of h
// as its K-major A, so one dlogits copy suffices. Only row chunks that add
// into existing gradients through the fp32 grad_weight partial keep a second,
// transposed dlogits copy that grad_weight (K = rows) reads K-major, because
// that partial starts from the output in its own [V, H] layout. The copies
// hold about half of the N x V logits, and at most 4 GiB. Whatever crosses
// chunks is summed in an fp32 partial: grad_weight (as [H, V] when computed
// transposed) when the chunks are row ranges, grad_hidden [N, H] when they
// are vocabulary ranges. The tensor path
// chunks the vocabulary whenever N < V, where that partial is the smaller one:
// each chunk's grad_weight rows are then complete after one GEMM over all N
// rows. flce_params.bwd_chunk_axis fixes the axis, so that callers and tests
// can reach both schedules at any size; the result is the same either way.
bool vocab_chunked(const flce_params* p) {
  if (p->N == 0) return false;
  if (p->bwd_chunk_axis == FLCE_CHUNK_AXIS_ROWS) return false;
  if (p->bwd_chunk_axis == FLCE_CHUNK_AXIS_VOCAB) return true;
  return p->N < p->V;
}

BwdLayout bwd_layout(const flce_params* p) {
  BwdLayout L{};
  const int64_t N = p->N, V = p->V, H = p->H;
  const size_t elem = tensor_path(p) ? 2 : 4;
  L.V_pad = (V + 7) / 8 * 8;
  L.vocab = vocab_chunked(p);
  if (L.vocab) {
    // Column chunks of whole tiles (256 columns on the tensor path, 64 on the
    // fp32 path) over all rows, whose dlogits copy holds about N x V bytes:
    // one 16-bit row-major copy of half of the columns (the tensor path:
    // grad_weight is computed transposed, as (h^T dS)^T, from a transposed
    // copy of h), or one fp32 copy of a quarter (the fp32 path).
    // Fewer columns per chunk if N rows of them would pass the 4 GiB cap;
    // then the columns are spread evenly over the chunks.
    // flce_params.max_chunk (rounded down to whole tiles) lowers the cap.
    L.wt = tensor_path(p);
    const int64_t gran = tensor_path(p) ? kBN : kSimtTile;
    int64_t cap = static_cast<int64_t>(kChunkByteCap / (size_t(N) * elem)) / gran * gran;
    if (cap < gran) cap = gran;
    if (p->max_chunk > 0) {
      const int64_t c = p->max_chunk < gran ? gran : p->max_chunk / gran * gran;
      if (c < cap) cap = c;
    }
    int64_t w = ceil_div(ceil_div(V, int64_t(elem)), gran) * gran;
    if (w > cap) w = cap;
    L.nchunks = static_cast<int>(ceil_div(V, w));
    L.chunk = L.nchunks == 1 ? V : ceil_div(ceil_div(V, L.nchunks), gran) * gran;
    L.nchunks = static_cast<int>(ceil_div(V, L.chunk));
    L.ds_ld = (L.chunk + 7) / 8 * 8;
    L.ht_ld = (N + 7) / 8 * 8;
    L.rowblk = tensor_path(p) ? kBM : kSimtTile;
    L.n_rowblocks = static_cast<int>(ceil_div(N, L.rowblk));
    L.coef_bytes = size_t(N) * sizeof(float4);
    L.ds_bytes = size_t(N) * L.ds_ld * elem;
    L.ht_bytes = L.wt ? size_t(H) * L.ht_ld * 2 : 0;
    if (tensor_path(p)) {
      L.dh_bytes = L.nchunks > 1 ? size_t(N) * H * 4 : 0;
    } else {
      // fp32: grad_hidden accumulates in its own fp32 output; only the K-split
      // partials of one chunk's contraction need room
      L.dh_bytes = simt_part_bytes(N, H, L.chunk);
    }
    L.bias_bytes = p->has_bias ? size_t(L.n_rowblocks) * L.V_pad * 4 : 0;
    size_t o = kHeader;
    place_counters(p, &L, &o);
    L.coef = o;
    o = align_up(o + L.coef_bytes, 256);
    L.ds = o;
    o = align_up(o + L.ds_bytes, 1024);
    L.ds_t = o;   // no transposed copy with vocabulary chunks
    L.ht = o;
    if (L.ht_bytes) o = align_up(o + L.ht_bytes, 1024);
    L.dw = o;
    L.dh_part = o;
    if (L.dh_bytes) o = align_up(o + L.dh_bytes, 1024);
    L.bias_part = o;
    if (L.bias_bytes) o = align_up(o + L.bias_bytes, 256);
    L.total = o;
    return L;
  }
  L.ds_ld = L.V_pad;
  // Row chunks whose dlogits copies hold about N x V bytes, half of the
  // logits in bf16: one 16-bit row-major copy of half of the rows (the tensor
  // path, grad_weight computed transposed from a transposed copy of h), two
  // 16-bit copies of a quarter (the tensor path adding into existing
  // gradients through an fp32 grad_weight partial, which starts from the
  // output in grad_weight's own layout), or one fp32 copy of a quarter (the
  // fp32 path). Chunk boundaries fall on 256-row pair blocks (tensor path)
  // or 64-row SIMT tiles.
  L.wt = tensor_path(p) && !(p->grad_weight_accum == FLCE_ACCUM_FP32 && p->accumulate);
  const int copies = tensor_path(p) && !L.wt ? 2 : 1;
  const int64_t gran = tensor_path(p) ? kPairM : kSimtTile;
  {
    const int64_t parts = L.wt ? 2 : 4;
    const int64_t share = ceil_div(ceil_div(N, parts), gran) * gran;
    int64_t cap = static_cast<int64_t>(kChunkByteCap / (size_t(L.V_pad) * elem * copies)) /
                  gran * gran;
    if (cap < gran) cap = gran;
    // flce_params.max_chunk (rounded down to the granule) lowers the cap. The
    // work and the result are the same, in less workspace.
    if (p->max_chunk > 0) {
      const int64_t r = p->max_chunk < gran ? gran : p->max_chunk / gran * gran;
      if (r < cap) cap = r;
    }
    L.chunk = share < cap ? share : cap;
    if (L.chunk > N && N > 0) L.chunk = N;
  }
  L.nchunks = N > 0 ? static_cast<int>(ceil_div(N, L.chunk)) : 0;
  L.rowblk = tensor_path(p) ? kBM : kSimtTile;
  L.n_rowblocks = static_cast<int>(ceil_div(N, L.rowblk));
  L.ds_t_ld = (L.chunk + 7) / 8 * 8;
  L.ht_ld = (N + 7) / 8 * 8;
  // the fp32 grad_weight partial, in the layout the contraction produces:
  // grad_weight^T [H][V_pad] when it is computed transposed, else [V][H]
  L.dw_ld = L.wt ? L.V_pad : H;
  L.coef_bytes = size_t(N) * sizeof(float4);
  L.ds_bytes = size_t(L.chunk) * L.V_pad * elem;
  L.ds_t_bytes = tensor_path(p) && !L.wt ? size_t(V) * L.ds_t_ld * elem : 0;
  L.ht_bytes = L.wt ? size_t(H) * L.ht_ld * 2 : 0;
  L.dw_bytes = (tensor_path(p) && L.nchunks > 1 && p->grad_weight_accum == FLCE_ACCUM_FP32)
                   ? size_t(L.wt ? H : V) * L.dw_ld * 4 : 0;
  if (tensor_path(p)) {
    L.dh_bytes = size_t(kMaxKSplits) * L.chunk * H * 4;
  } else if (N > 0) {
    L.dh_bytes = simt_part_bytes(L.chunk, H, V);   // fp32 grad_hidden split partials
  }
  L.bias_bytes = p->has_bias ? size_t(L.n_rowblocks) * L.V_pad * 4 : 0;
  size_t o = kHeader;
  place_counters(p, &L, &o);
  L.coef = o;
  o = align_up(o + L.coef_bytes, 256);
  L.ds = o;
  o = align_up(o + L.ds_bytes, 1024);
  L.ds_t = o;
  if (L.ds_t_bytes) o = align_up(o + L.ds_t_bytes, 1024);
  L.ht = o;
  if (L.ht_bytes) o = align_up(o + L.ht_bytes, 1024);
  L.dw = o;
  if (L.dw_bytes) o = align_up(o + L.dw_bytes, 1024);
  L.dh_part = o;
  if (L.dh_bytes) o = align_up(o + L.dh_bytes, 1024);
  L.bias_part = o;
  if (L.bias_bytes) o = align_up(o + L.bias_bytes, 256);
  L.total = o;
  return L;
}

// Pair blocks per unit group: about 32 MB of h rows (256 x H x 2 bytes per
// block). Measured at the headline size, a group of 16 blocks (4096 rows x
// 4096) stays in L2. The forward over all 32 blocks (67 MB of h) read 6.1x
// its algorithmic bytes from DRAM.
int group_blocks_for(int n_blocks, int H) {
  const long long per_block = static_cast<long long>(kPairM) * H * 2;
  long long g = (32ll << 20) / per_block;
  if (g < 1) g = 1;
  return static_cast<int>(g < n_blocks ? g : n_blocks);
}

// Vocabulary tiles per panel. Units (panel, pair block) are handed out
// round-robin to `pairs` persistent CTA pairs, in groups of `group` pair
// blocks, panel-major within a group (decode_unit). So at any moment the pairs
// work on the same few panels of the same group: a W panel is read from HBM
// once per group and shared through L2, and the group's rows of h stay
// resident. The criterion is the busiest pair's tile count (the critical
// path). Among panel lengths within 1 % of the best, the shortest wins,
// because it keeps the W working set small next to h.
int choose_panel_tiles(int n_blocks, int group, int v_tiles, int pairs, int* grid_out) {
  long long cost_of[kMaxPanelTiles + 1];
  int grid_of[kMaxPanelTiles + 1];
  long long best_cost = -1;
  for (int pt = kMinPanelTiles; pt <= kMaxPanelTiles; ++pt) {
    const long long P = ceil_div(v_tiles, pt);
    const long long U = P * n_blocks;
    const long long G = U < pairs ? U : pairs;
    const long long last_len = v_tiles - (P - 1) * pt;
    long long cost = 0;
    for (long long c = 0; c < G; ++c) {
      // units of pair c: c, c + G, ...; count those in [lo, hi)
      auto cnt = [&](long long x) { return x > c ? (x - c - 1) / G + 1 : 0; };
      long long t = 0, pos = 0;
      for (long long b0 = 0; b0 < n_blocks; b0 += group) {
        const long long gb = n_blocks - b0 < group ? n_blocks - b0 : group;
        const long long full = gb * (P - 1);  // units of full panels, then gb of the last panel
        t += (cnt(pos + full) - cnt(pos)) * pt + (cnt(pos + full + gb) - cnt(pos + full)) * last_len;
        pos += full + gb;
      }
      if (t > cost) cost = t;
    }
    cost_of[pt] = cost;
    grid_of[pt] = static_cast<int>(G);
    if (best_cost < 0 || cost < best_cost) best_cost = cost;
  }
  int best = kMinPanelTiles;
  for (int pt = kMinPanelTiles; pt <= kMaxPanelTiles; ++pt) {
    if (cost_of[pt] * 100 <= best_cost * 101) {
      best = pt;
      break;
    }
  }
  *grid_out = grid_of[best];
  return best;
}

// Row tiles per raster group of a plain GEMM (decode_unit). When a wave of
// `pairs` tiles spans fewer than all column tiles, row-after-row order reads
// every B strip once per row tile: the projection of a row chunk (K = H,
// thousands of vocabulary columns) streamed all of W once per 256 rows.
// Groups of row tiles whose A strips (256 x K x 2 bytes each) total about
// 32 MB stay in L2 while the columns sweep past, so each B strip is read
// once per group. Otherwise a wave already covers whole rows of tiles, and
// the order stays row after row (a group of 1).
int gemm_group_m(const GemmArgs& ga, int pairs) {
  if (ga.n_tiles <= pairs) return 1;
  const long long strip = static_cast<long long>(kPairM) * ga.kb_per_split * kBK * 2;
  long long g = (32ll << 20) / strip;
  if (g < 1) g = 1;
  return static_cast<int>(g < ga.m_tiles ? g : ga.m_tiles);
}

// The GEMMs take their units from an atomic counter in the workspace header
// (two ints at kTileCounterOffset, zeroed with the header at every entry and
// left zero by each launch), so that a pair that finishes early takes the
// next unit. Builds with FLCE_STATIC_GEMM_SCHEDULE hand the units out
// round-robin instead.
constexpr size_t kTileCounterOffset = 128;

cudaError_t launch_gemm(const GemmOperand& op_a, const GemmOperand& op_b, GemmArgs ga, bool f16,
                        int pairs, cudaStream_t st) {
  ga.group_m = gemm_group_m(ga, pairs);
  ga.clk = g_cur_clk;
#ifndef FLCE_STATIC_GEMM_SCHEDULE
  if (ga.status != nullptr)
    ga.tile_counter = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(ga.status) + kTileCounterOffset);
#endif
  return launch_gemm_tc(op_a, op_b, ga, f16, pairs, st);
}

// K splits of the grad_hidden GEMM. Its long tiles (K = V) number only
// rows/256 x H/256 (256 at the headline size), which is 3.37 waves on 76
// pairs: the last wave runs a third full. Two K halves give 6.74 waves
// (96 % full). The partials cost an extra fp32 write and read of
// rows x H per split.
int choose_k_splits(int tiles, int k_blocks, int pairs) {
  auto eff = [&](int s) {
    const double w = double(tiles) * s / pairs;
    return w / std::ceil(w);
  };
  int best = 1;
  for (int s = 2; s <= kMaxKSplits; ++s)
    if (k_blocks / s >= 128 && eff(s) > eff(best) + 0.04) best = s;
  return best;
}

// ------------------------------------------------------------ tensor maps
int make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
             uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
             CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(m, dt, 2, const_cast<void*>(base),
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_detail, sizeof(g_detail), "cuTensorMapEncodeTiled failed (%d) dims %llu x %llu",
             static_cast<int>(r), static_cast<unsigned long long>(inner),
             static_cast<unsigned long long>(outer));
    return FLCE_ERR_CUDA;
  }
  return FLCE_OK;
}

// A K-major GEMM operand [rows][k]: the 2-D map with 64 x box_rows boxes.
int make_k_operand(GemmOperand* op, const void* base, uint64_t k, uint64_t rows, uint64_t row_bytes,
                   uint32_t box_rows, CUtensorMapDataType dt) {
  const int v = make_map(&op->map, base, k, rows, row_bytes, kBK, box_rows, dt);
  op->map3 = op->map;
  return v;
}

// An MN-major GEMM operand [k rows][mn cols] of 16-bit elements: the 2-D map
// with 64 x 64 boxes and, when it has two or more full 64-column atoms, the
// 3-D view of those atoms. Element (x, y, z) of the view is column 64 z + x of
// row y, so its strides are row_bytes (y) and 128 bytes (z). *atoms is the
// view's atom count, 0 without a view. The MN-major operands are the B sides
// of both gradient GEMMs: W in grad_hidden and h in grad_weight.
int make_mn_operand(GemmOperand* op, int* atoms, const void* base, uint64_t mn, uint64_t k,
                    uint64_t row_bytes, CUtensorMapDataType dt) {
  int v = make_map(&op->map, base, mn, k, row_bytes, 64, 64, dt);
  if (v != FLCE_OK) return v;
  op->map3 = op->map;
  *atoms = 0;
  const uint64_t full = mn / 64;
  if (full < 2) return FLCE_OK;
  const cuuint64_t dims[3] = {64, k, full};
  const cuuint64_t strides[2] = {row_bytes, 128};
  const cuuint32_t box[3] = {64, 64, 2};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(&op->map3, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_detail, sizeof(g_detail), "cuTensorMapEncodeTiled (3-D) failed (%d) atoms %llu x %llu",
             static_cast<int>(r), static_cast<unsigned long long>(full),
             static_cast<unsigned long long>(k));
    return FLCE_ERR_CUDA;
  }
  *atoms = static_cast<int>(full);
  return FLCE_OK;
}

float inv_cap(const flce_params* p) { return p->softcap > 0.f ? 1.f / p->softcap : 0.f; }

CUtensorMapDataType map_type(const flce_params* p) {
  return p->dtype == FLCE_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
}

// Workspace of flce_chunk_grads: the status header, the fp32 grad_weight
// partial that crosses row chunks, and the K-split partials of grad_hidden.
// The two partials exist on the tensor path only; with
// grad_weight_accum = weight the chunks accumulate in grad_weight itself.
struct ChunkLayout {
  bool wt;              // grad_weight computed transposed, (h^T dlogits)^T
  int64_t ht_ld, dw_ld; // row strides of h^T and of the fp32 grad_weight partial
  size_t dw_part, dh_part, ht, total;
  size_t dw_bytes, dh_bytes, ht_bytes;
};

// flce_chunk_grads on the tensor path computes grad_weight transposed, from
// h^T (transposed into the workspace) and the caller's row-major dlogits as
// an MN-major operand, so it needs no transposed dlogits. The fp32 partial
// across the chunks then has grad_weight^T's layout [H][V]. Only adding the
// fp32-accumulated gradient into an existing one keeps the row-major partial
// and reads dlogits transposed. A function of the parameters, so every chunk
// of one loss takes the same path.
bool chunk_grads_transposed(const flce_params* p) {
  return tensor_path(p) && !(p->grad_weight_accum == FLCE_ACCUM_FP32 && p->accumulate);
}

ChunkLayout chunk_layout(const flce_params* p) {
  ChunkLayout L{};
  L.wt = chunk_grads_transposed(p);
  L.dw_ld = L.wt ? (p->V + 7) / 8 * 8 : p->H;
  L.dw_bytes = (tensor_path(p) && p->grad_weight_accum == FLCE_ACCUM_FP32)
                   ? size_t(L.wt ? p->H : p->V) * L.dw_ld * 4 : 0;
  if (tensor_path(p)) {
    L.dh_bytes = size_t(kMaxKSplits) * p->N * p->H * 4;
  } else {
    L.dh_bytes = simt_part_bytes(p->N, p->H, p->V);
  }
  L.ht_ld = (p->N + 7) / 8 * 8;
  L.ht_bytes = L.wt ? size_t(p->H) * L.ht_ld * 2 : 0;
  // grad_hidden's split partials are done with (split-reduced) before h is
  // transposed for grad_weight, so both share one scratch region. It comes
  // last: its size follows the call's N, its start does not, so every chunk
  // of one loss writes inside the regions of the largest chunk.
  size_t o = kHeader;
  L.dw_part = o;
  if (L.dw_bytes) o = align_up(o + L.dw_bytes, 1024);
  L.dh_part = o;
  L.ht = o;
  const size_t scratch = L.dh_bytes > L.ht_bytes ? L.dh_bytes : L.ht_bytes;
  if (scratch) o = align_up(o + scratch, 1024);
  L.total = o;
  return L;
}

size_t mse_loss_part_bytes(const flce_params* p) {
  return size_t(ceil_div(p->V, kBN)) * ceil_div(p->N, 32) * 4;
}

// The regions of one pass's workspace that the kernels may write, in
// address order: everything else in the workspace stays untouched.
struct WsRegion {
  const char* name;
  size_t offset, bytes;
};

std::vector<WsRegion> workspace_regions(const flce_params* p, int pass) {
  std::vector<WsRegion> r;
  r.push_back({"header", 0, kHeader});
  auto add = [&](const char* n, size_t off, size_t bytes) {
    if (bytes > 0) r.push_back({n, off, bytes});
  };
  if (pass == FLCE_PASS_FORWARD) {
    const FwdLayout L = fwd_layout(p);
    add("partial_states", L.partials, L.partials_bytes);
    add("target_logits", L.zt, L.zt_bytes);
    add("block_loss", L.blk_loss, L.blk_bytes);
    add("block_entropy", L.blk_ent, L.blk_bytes);
    add("block_correct", L.blk_correct, L.blk_bytes);
    add("block_valid", L.blk_valid, L.blk_bytes);
  } else if (pass == FLCE_PASS_BACKWARD) {
    const BwdLayout L = bwd_layout(p);
    add("tile_counters", L.cnt, L.cnt_bytes);
    add("row_coefficients", L.coef, L.coef_bytes);
    add("dlogits", L.ds, L.ds_bytes);
    add("dlogits_transposed", L.ds_t, L.ds_t_bytes);
    add("hidden_transposed", L.ht, L.ht_bytes);
    add("grad_weight_fp32", L.dw, L.dw_bytes);
    add("grad_hidden_fp32", L.dh_part, L.dh_bytes);
    add("grad_bias_partials", L.bias_part, L.bias_bytes);
  } else if (pass == FLCE_PASS_CHUNK_GRADS) {
    const ChunkLayout L = chunk_layout(p);
    add("grad_weight_fp32", L.dw_part, L.dw_bytes);
    add("grad_hidden_fp32", L.dh_part, L.dh_bytes);
    add("hidden_transposed", L.ht, L.ht_bytes);
  } else if (pass == FLCE_PASS_CHUNK_MSE) {
    add("loss_partials", kHeader, mse_loss_part_bytes(p));
  }
  return r;
}

}  // namespace

void flce::note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

void flce::set_error_detail(const char* msg) {
  snprintf(g_detail, sizeof(g_detail), "%s", msg);
}

// ===================================================================== ABI
extern "C" {

const char* flce_error_string(int code) {
  switch (code) {
    case FLCE_OK: return "ok";
    case FLCE_ERR_INVALID_ARG: return "invalid argument";
    case FLCE_ERR_UNSUPPORTED: return "unsupported device (needs sm_103 / GB300)";
    case FLCE_ERR_ALIGNMENT: return "misaligned pointer or H not a multiple of 8";
    case FLCE_ERR_WORKSPACE: return "workspace missing or too small";
    case FLCE_ERR_CUDA: return "CUDA runtime error";
    case FLCE_ERR_TARGET_RANGE: return "target outside [0, V) and not ignore_index";
    case FLCE_ERR_TIMEOUT: return "a bounded wait inside a kernel expired";
    case FLCE_ERR_BOUNDS: return "a kernel store fell outside its buffer (debug build)";
    default: return "unknown error code";
  }
}

const char* flce_last_error_detail(void) { return g_detail; }

int flce_workspace_regions(const flce_params* p, int pass, flce_region* out, int max, int* count) {
  const int v = validate(p);
  if (v != FLCE_OK) return v;
  if (pass < FLCE_PASS_FORWARD || pass > FLCE_PASS_CHUNK_MSE || count == nullptr ||
      (max > 0 && out == nullptr))
    return FLCE_ERR_INVALID_ARG;
  const std::vector<WsRegion> r = workspace_regions(p, pass);
  for (int i = 0; i < static_cast<int>(r.size()) && i < max; ++i) {
    memset(&out[i], 0, sizeof(out[i]));
    strncpy(out[i].name, r[i].name, sizeof(out[i].name) - 1);
    out[i].offset = r[i].offset;
    out[i].bytes = r[i].bytes;
  }
  *count = static_cast<int>(r.size());
  return FLCE_OK;
}

int flce_test_fault(int32_t drop_kblock, int32_t wait_ms) {
  if (drop_kblock < -1 || wait_ms < 0) return FLCE_ERR_INVALID_ARG;
  g_test_drop_kb = drop_kblock;
  g_test_wait_ns = static_cast<unsigned long long>(wait_ms) * 1000000ull;
  return FLCE_OK;
}

uint64_t flce_launch_count(void) { return g_launches.load(); }

int flce_workspace_bytes(const flce_params* p, int pass, size_t* bytes) {
  const int v = validate(p);
  if (v != FLCE_OK) return v;
  if (bytes == nullptr) return FLCE_ERR_INVALID_ARG;
  if (pass == FLCE_PASS_FORWARD) {
    *bytes = fwd_layout(p).total;
  } else if (pass == FLCE_PASS_BACKWARD) {
    *bytes = bwd_layout(p).total;
  } else if (pass == FLCE_PASS_CHUNK_LOGITS) {
    *bytes = kHeader;
  } else if (pass == FLCE_PASS_CHUNK_GRADS) {
    *bytes = chunk_layout(p).total;
  } else if (pass == FLCE_PASS_CHUNK_MSE) {
    *bytes = align_up(kHeader + mse_loss_part_bytes(p), 256);
  } else {
    return FLCE_ERR_INVALID_ARG;
  }
  return FLCE_OK;
}

// Checks and set-up shared by the forward entry points. `rows_out` is the
// per-row output that must be non-NULL when N > 0 (lse or the shard states).
static int forward_prologue(const flce_params* p, const void* hidden, const void* weight,
                            const void* bias, const int64_t* targets, const void* rows_out,
                            void* workspace, size_t ws_bytes, FwdLayout* L, DeviceInfo* d) {
  int v = validate(p);
  if (v != FLCE_OK) return v;
  // Row-indexed pointers may be NULL only when there are no rows.
  const bool rows = p->N > 0;
  if (weight == nullptr || (rows && (hidden == nullptr || targets == nullptr || rows_out == nullptr)))
    return FLCE_ERR_INVALID_ARG;
  if ((p->has_bias != 0) != (bias != nullptr)) return FLCE_ERR_INVALID_ARG;
  if (workspace == nullptr) return FLCE_ERR_WORKSPACE;
  if (!aligned16(hidden) || !aligned16(weight) || (bias && !aligned16(bias)) ||
      !aligned16(workspace) || !aligned16(targets))
    return FLCE_ERR_ALIGNMENT;
  *L = fwd_layout(p);
  if (ws_bytes < L->total) return FLCE_ERR_WORKSPACE;
  return FLCE_OK;
}

// The vocabulary sweep: per-panel online states and the target logits.
static int forward_tiles(const flce_params* p, const void* hidden, const void* weight,
                         const void* bias, const int64_t* targets, uint8_t* ws, const FwdLayout& L,
                         const DeviceInfo& d, bool metrics, cudaStream_t st, FwdArgs* out) {
  const int N = static_cast<int>(p->N), H = static_cast<int>(p->H), V = static_cast<int>(p->V);
  FwdArgs fa{};
  fa.N = N;
  fa.H = H;
  fa.V = V;
  fa.vocab_start = p->vocab_start;
  fa.scale = p->logit_scale;
  fa.softcap = p->softcap > 0.f ? p->softcap : 0.f;
  fa.inv_softcap = inv_cap(p);
  fa.bias = bias;
  fa.targets = targets;
  fa.ignore_index = p->ignore_index;
  fa.partials = reinterpret_cast<float4*>(ws + L.partials);
  fa.zt = reinterpret_cast<float*>(ws + L.zt);
  fa.r_partials = DevRegion{ws + L.partials, L.partials_bytes};
  fa.r_zt = DevRegion{ws + L.zt, L.zt_bytes};
  fa.status = reinterpret_cast<int*>(ws);
  // flce_test_fault arms these for the calling thread only; otherwise no
  // stage is starved and every wait has the default limit.
  fa.wait_ns = g_test_wait_ns > 0 ? g_test_wait_ns : kWaitLimitNs;
  fa.drop_kb = g_test_drop_kb;
  // the header's GEMM counters, zeroed at every forward entry (the forward
  // launches no GEMM)
  fa.tile_counter = reinterpret_cast<int*>(ws + kTileCounterOffset);
  int v;
  if (tensor_path(p)) {
    const CUtensorMapDataType dt = map_type(p);
    fa.n_blocks = static_cast<int>(ceil_div(N, kPairM));
    fa.v_tiles = static_cast<int>(ceil_div(V, kBN));
    fa.group_blocks = group_blocks_for(fa.n_blocks, H);
    int grid = 1;
    fa.panel_tiles = choose_panel_tiles(fa.n_blocks, fa.group_blocks, fa.v_tiles, d.pairs, &grid);
    fa.num_panels = static_cast<int>(ceil_div(fa.v_tiles, fa.panel_tiles));
    fa.num_units = fa.num_panels * fa.n_blocks;
    CUtensorMap tm_h, tm_w;
    if ((v = make_map(&tm_h, hidden, H, N, uint64_t(H) * 2, kBK, kBM, dt)) != FLCE_OK) return v;
    if ((v = make_map(&tm_w, weight, H, V, uint64_t(H) * 2, kBK, kBNHalf, dt)) != FLCE_OK) return v;
    const bool f16 = p->dtype == FLCE_F16;
    v = launch("flce_fwd_tc", st, [&] {
      fa.clk = g_cur_clk;
      return launch_fwd_tc(tm_h, tm_w, fa, f16, bias != nullptr, p->softcap > 0.f, metrics, grid,
                           st);
    });
  } else {
    fa.n_blocks = static_cast<int>(ceil_div(N, kSimtTile));
    fa.panel_tiles = simt_panel_tiles(N, V);
    fa.num_panels = static_cast<int>(ceil_div(V, int64_t(fa.panel_tiles) * kSimtTile));
    fa.num_units = fa.num_panels * fa.n_blocks;
    v = launch("flce_fwd_simt", st, [&] {
      return launch_fwd_simt(static_cast<const float*>(hidden), static_cast<const float*>(weight),
                             fa, st);
    });
  }
  *out = fa;
  return v;
}

// The merge's (or combine's) blocks-done counter: a word of the header, which
// every forward entry zeroes before its first kernel.
constexpr size_t kMergeDoneOffset = 136;

static FinalizeArgs finalize_args(const flce_params* p, uint8_t* ws, const FwdLayout& L, int nblk,
                                  float* loss, int64_t* num_correct, float* entropy_sum) {
  FinalizeArgs fz{};
  fz.nblk = nblk;
  fz.status = reinterpret_cast<const int*>(ws);
  fz.reduction = p->reduction;
  fz.blk_loss = reinterpret_cast<const double*>(ws + L.blk_loss);
  fz.blk_ent = reinterpret_cast<const double*>(ws + L.blk_ent);
  fz.blk_correct = reinterpret_cast<const long long*>(ws + L.blk_correct);
  fz.blk_valid = reinterpret_cast<const long long*>(ws + L.blk_valid);
  fz.loss = p->reduction == FLCE_NONE ? nullptr : loss;
  fz.num_correct = num_correct;
  fz.entropy_sum = entropy_sum;
  return fz;
}

// Reduced outputs of a call without rows (the merge, which otherwise writes
// them, does not run).
static int forward_finalize_empty(const flce_params* p, uint8_t* ws, const FwdLayout& L,
                                  float* loss, int64_t* num_correct, float* entropy_sum,
                                  cudaStream_t st) {
  const FinalizeArgs fz = finalize_args(p, ws, L, 0, loss, num_correct, entropy_sum);
  return launch("flce_finalize", st, [&] { return launch_finalize(fz, st); });
}

int flce_forward(const flce_params* p, const void* hidden, const void* weight, const void* bias,
                 const int64_t* targets, float* loss, float* lse, int64_t* num_correct,
                 float* entropy_sum, void* workspace, size_t ws_bytes, flce_stream_t stream) {
  const NvtxRange nvtx_range("flce_forward");
  FwdLayout L;
  DeviceInfo d;
  int v = forward_prologue(p, hidden, weight, bias, targets, lse, workspace, ws_bytes, &L, &d);
  if (v != FLCE_OK) return v;
  if (loss == nullptr && (p->N > 0 || p->reduction != FLCE_NONE)) return FLCE_ERR_INVALID_ARG;
  // The loss needs the whole vocabulary. Shards go through flce_forward_partial
  // and flce_forward_combine.
  if (p->vocab_total != 0 && (p->vocab_total != p->V || p->vocab_start != 0)) {
    snprintf(g_detail, sizeof(g_detail),
             "flce_forward needs the whole vocabulary; use flce_forward_partial + combine");
    return FLCE_ERR_INVALID_ARG;
  }
  if ((v = device_info(&d)) != FLCE_OK) return v;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t e = cudaMemsetAsync(ws, 0, kHeader, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  const int N = static_cast<int>(p->N);
  if (N > 0) {
    FwdArgs fa;
    const bool metrics = num_correct != nullptr || entropy_sum != nullptr;
    if ((v = forward_tiles(p, hidden, weight, bias, targets, ws, L, d, metrics, st, &fa)) != FLCE_OK)
      return v;
    MergeArgs ma{};
    ma.N = N;
    ma.V = static_cast<int>(p->V);
    ma.vocab_start = 0;
    ma.vocab_total = p->V;
    ma.num_panels = fa.num_panels;
    ma.lanes = L.lanes;
    ma.reduction = p->reduction;
    ma.ignore_index = p->ignore_index;
    ma.zeta = p->z_loss_multiplier;
    ma.partials = fa.partials;
    ma.zt = fa.zt;
    ma.targets = targets;
    ma.lse = lse;
    ma.loss_rows = p->reduction == FLCE_NONE ? loss : nullptr;
    ma.blk_loss = reinterpret_cast<double*>(ws + L.blk_loss);
    ma.blk_ent = reinterpret_cast<double*>(ws + L.blk_ent);
    ma.blk_correct = reinterpret_cast<long long*>(ws + L.blk_correct);
    ma.blk_valid = reinterpret_cast<long long*>(ws + L.blk_valid);
    ma.status = reinterpret_cast<int*>(ws);
    ma.done = reinterpret_cast<int*>(ws + kMergeDoneOffset);
    ma.fin = finalize_args(p, ws, L, L.nblk, loss, num_correct, entropy_sum);
    v = launch("flce_merge", st, [&] { return launch_merge(ma, L.nblk, st); });
    return debug_finish(ws, st, v);
  }
  return debug_finish(ws, st, forward_finalize_empty(p, ws, L, loss, num_correct, entropy_sum, st));
}

int flce_forward_partial(const flce_params* p, const void* hidden, const void* weight,
                         const void* bias, const int64_t* targets, flce_row_state* states,
                         void* workspace, size_t ws_bytes, flce_stream_t stream) {
  const NvtxRange nvtx_range("flce_forward_partial");
  static_assert(sizeof(flce_row_state) == sizeof(ShardState), "row state layout");
  FwdLayout L;
  DeviceInfo d;
  int v = forward_prologue(p, hidden, weight, bias, targets, states, workspace, ws_bytes, &L, &d);
  if (v != FLCE_OK) return v;
  if (reinterpret_cast<uintptr_t>(states) & 3u) return FLCE_ERR_ALIGNMENT;
  if ((v = device_info(&d)) != FLCE_OK) return v;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t e = cudaMemsetAsync(ws, 0, kHeader, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  if (p->N == 0) return FLCE_OK;
  FwdArgs fa;
  // the shard states carry the argmax and sum z exp(z - m) for the merge's metrics
  if ((v = forward_tiles(p, hidden, weight, bias, targets, ws, L, d, true, st, &fa)) != FLCE_OK)
    return v;
  ShardStateArgs sa{};
  sa.N = static_cast<int>(p->N);
  sa.V = static_cast<int>(p->V);
  sa.num_panels = fa.num_panels;
  sa.status = reinterpret_cast<const int*>(ws);
  sa.vocab_start = p->vocab_start;
  sa.ignore_index = p->ignore_index;
  sa.partials = fa.partials;
  sa.zt = fa.zt;
  sa.targets = targets;
  sa.out = reinterpret_cast<ShardState*>(states);
  return debug_finish(ws, st,
                      launch("flce_shard_state", st, [&] { return launch_shard_state(sa, st); }));
}

int flce_forward_combine(const flce_params* p, const flce_row_state* states, int32_t num_shards,
                         const int64_t* targets, float* loss, float* lse, int64_t* num_correct,
                         float* entropy_sum, void* workspace, size_t ws_bytes,
                         flce_stream_t stream) {
  const NvtxRange nvtx_range("flce_forward_combine");
  int v = validate(p);
  if (v != FLCE_OK) return v;
  const bool rows = p->N > 0;
  if (num_shards < 1 || (rows && (states == nullptr || targets == nullptr || lse == nullptr)) ||
      (loss == nullptr && (rows || p->reduction != FLCE_NONE)))
    return FLCE_ERR_INVALID_ARG;
  if (workspace == nullptr) return FLCE_ERR_WORKSPACE;
  if (!aligned16(workspace) || !aligned16(targets)) return FLCE_ERR_ALIGNMENT;
  const FwdLayout L = fwd_layout(p);
  if (ws_bytes < L.total) return FLCE_ERR_WORKSPACE;
  DeviceInfo d;
  if ((v = device_info(&d)) != FLCE_OK) return v;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t e = cudaMemsetAsync(ws, 0, kHeader, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  const int N = static_cast<int>(p->N);
  if (N > 0) {
    CombineArgs ca{};
    ca.N = N;
    ca.R = num_shards;
    ca.reduction = p->reduction;
    ca.vocab_total = p->vocab_total ? p->vocab_total : p->V;
    ca.ignore_index = p->ignore_index;
    ca.zeta = p->z_loss_multiplier;
    ca.states = reinterpret_cast<const ShardState*>(states);
    ca.targets = targets;
    ca.lse = lse;
    ca.loss_rows = p->reduction == FLCE_NONE ? loss : nullptr;
    ca.blk_loss = reinterpret_cast<double*>(ws + L.blk_loss);
    ca.blk_ent = reinterpret_cast<double*>(ws + L.blk_ent);
    ca.blk_correct = reinterpret_cast<long long*>(ws + L.blk_correct);
    ca.blk_valid = reinterpret_cast<long long*>(ws + L.blk_valid);
    ca.status = reinterpret_cast<int*>(ws);
    ca.done = reinterpret_cast<int*>(ws + kMergeDoneOffset);
    ca.fin = finalize_args(p, ws, L, L.nblk, loss, num_correct, entropy_sum);
    v = launch("flce_combine", st, [&] { return launch_combine(ca, L.nblk, st); });
    return debug_finish(ws, st, v);
  }
  return debug_finish(ws, st, forward_finalize_empty(p, ws, L, loss, num_correct, entropy_sum, st));
}

int flce_backward(const flce_params* p, const void* hidden, const void* weight, const void* bias,
                  const int64_t* targets, const float* lse, const float* grad_loss,
                  void* grad_hidden, void* grad_weight, void* grad_bias, void* workspace,
                  size_t ws_bytes, flce_stream_t stream) {
  const NvtxRange nvtx_range("flce_backward");
  int v = validate(p);
  if (v != FLCE_OK) return v;
  const bool rows = p->N > 0;
  if (weight == nullptr ||
      (rows && (hidden == nullptr || targets == nullptr || lse == nullptr || grad_loss == nullptr)))
    return FLCE_ERR_INVALID_ARG;
  if ((p->has_bias != 0) != (bias != nullptr)) return FLCE_ERR_INVALID_ARG;
  if (grad_bias != nullptr && !p->has_bias) return FLCE_ERR_INVALID_ARG;
  if (workspace == nullptr) return FLCE_ERR_WORKSPACE;
  if (!aligned16(hidden) || !aligned16(weight) || (bias && !aligned16(bias)) ||
      !aligned16(workspace) || !aligned16(targets) || (grad_hidden && !aligned16(grad_hidden)) ||
      (grad_weight && !aligned16(grad_weight)) || (grad_bias && !aligned16(grad_bias)))
    return FLCE_ERR_ALIGNMENT;
  const BwdLayout L = bwd_layout(p);
  if (ws_bytes < L.total) return FLCE_ERR_WORKSPACE;
  DeviceInfo d;
  if ((v = device_info(&d)) != FLCE_OK) return v;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* status = reinterpret_cast<int*>(ws);
  const int N = static_cast<int>(p->N), H = static_cast<int>(p->H), V = static_cast<int>(p->V);
  const size_t elem = tensor_path(p) ? 2 : 4;
  cudaError_t e = cudaSuccess;
  const bool no_rows = N == 0 || (grad_hidden == nullptr && grad_weight == nullptr && grad_bias == nullptr);
  // Without rows the status word is cleared here; otherwise the row
  // coefficients kernel, which runs first, clears it with the tile counters.
  if (no_rows && (e = cudaMemsetAsync(ws, 0, kHeader, st)) != cudaSuccess)
    return cuda_fail(e, "cudaMemsetAsync");
  if (grad_hidden == nullptr && grad_weight == nullptr && grad_bias == nullptr) return FLCE_OK;
  if (N == 0) {
    if (p->accumulate) return FLCE_OK;  // nothing to add
    if (grad_weight && (e = cudaMemsetAsync(grad_weight, 0, size_t(V) * H * elem, st)) != cudaSuccess)
      return cuda_fail(e, "cudaMemsetAsync");
    if (grad_bias && (e = cudaMemsetAsync(grad_bias, 0, size_t(V) * elem, st)) != cudaSuccess)
      return cuda_fail(e, "cudaMemsetAsync");
    return FLCE_OK;
  }

  float4* coef = reinterpret_cast<float4*>(ws + L.coef);
  RowCoefArgs ra{};
  ra.N = N;
  ra.V = V;
  ra.reduction = p->reduction;
  ra.vocab_start = p->vocab_start;
  ra.vocab_total = p->vocab_total ? p->vocab_total : p->V;
  ra.ignore_index = p->ignore_index;
  ra.scale = p->logit_scale;
  ra.zeta = p->z_loss_multiplier;
  ra.targets = targets;
  ra.lse = lse;
  ra.grad_loss = grad_loss;
  ra.coef = coef;
  float* ds_scale = p->dtype == FLCE_F16 ? reinterpret_cast<float*>(ws + kScaleOffset) : nullptr;
  ra.ds_scale = ds_scale;
  ra.status = status;
  ra.zero = status;
  ra.zero_words = static_cast<int>((L.cnt + L.cnt_bytes) / 4);
  v = launch("flce_row_coef", st, [&] { return launch_row_coef(ra, st); });
  if (v != FLCE_OK) return v;

  float* bias_part = grad_bias ? reinterpret_cast<float*>(ws + L.bias_part) : nullptr;
  DsArgs da{};
  da.H = H;
  da.V = V;
  da.V_pad = static_cast<int>(L.V_pad);
  da.scale = p->logit_scale;
  da.softcap = p->softcap > 0.f ? p->softcap : 0.f;
  da.inv_softcap = inv_cap(p);
  da.bias = bias;
  da.coef = coef;
  da.ds_scale = ds_scale;
  da.ds = ws + L.ds;
  da.bias_part = bias_part;
  da.bias_ld = static_cast<int>(L.V_pad);
  da.tgt_base = 0;
  da.status = status;
  // the header's unit counters, zeroed by the row coefficients kernel and left
  // zero by every launch that takes units from them
  da.tile_counter = tensor_path(p) ? reinterpret_cast<int*>(ws + kTileCounterOffset) : nullptr;
  da.r_ds = DevRegion{ws + L.ds, L.ds_bytes};
  da.r_ds_t = DevRegion{ws + L.ds_t, L.ds_t_bytes};
  da.r_bias = DevRegion{ws + L.bias_part, L.bias_bytes};
  const DevRegion r_gh{grad_hidden, grad_hidden ? size_t(N) * H * elem : 0};
  const DevRegion r_gw{grad_weight, grad_weight ? size_t(V) * H * elem : 0};
  const DevRegion r_dh{ws + L.dh_part, L.dh_bytes};
  const DevRegion r_dw{ws + L.dw, L.dw_bytes};

  if (tensor_path(p)) {
    const CUtensorMapDataType dt = map_type(p);
    const bool f16 = p->dtype == FLCE_F16;
    // fp16 dlogits are stored times S; the contractions multiply by 1/S
    const float* acc_scale = ds_scale != nullptr ? ds_scale + 1 : nullptr;
    CUtensorMap tm_h, tm_w;
    if ((v = make_map(&tm_h, hidden, H, N, uint64_t(H) * 2, kBK, kBM, dt)) != FLCE_OK) return v;
    if ((v = make_map(&tm_w, weight, H, V, uint64_t(H) * 2, kBK, kBNHalf, dt)) != FLCE_OK) return v;
    float* dw_part = reinterpret_cast<float*>(ws + L.dw);
    const int nchunks_rows = L.vocab ? 0 : L.nchunks;
    if (L.wt && grad_weight) {
      // h^T [H][ht_ld], the K-major A operand of the transposed grad_weight
      TransposeArgs ta{};
      ta.src = static_cast<const uint16_t*>(hidden);
      ta.dst = reinterpret_cast<uint16_t*>(ws + L.ht);
      ta.rows = N;
      ta.cols = H;
      ta.ld_src = H;
      ta.ld_dst = L.ht_ld;
      ta.status = status;
      ta.r_dst = DevRegion{ws + L.ht, L.ht_bytes};
      v = launch("flce_transpose_hidden", st, [&] { return launch_transpose16(ta, st); });
      if (v != FLCE_OK) return v;
    }
    for (int c = 0; L.vocab && c < L.nchunks; ++c) {
      // Columns [v0, v0 + vc) of the vocabulary, all N rows.
      const int v0 = static_cast<int>(c * L.chunk);
      const int vc = static_cast<int>(V - v0 < L.chunk ? V - v0 : L.chunk);
      const uint8_t* wc = static_cast<const uint8_t*>(weight) + size_t(v0) * H * 2;
      const uint64_t ds_row_bytes = uint64_t(L.ds_ld) * 2;
      CUtensorMap tm_wc;
      if ((v = make_map(&tm_wc, wc, H, vc, uint64_t(H) * 2, kBK, kBNHalf, dt)) != FLCE_OK) return v;
      da.rows = N;
      da.row0 = 0;
      da.V = vc;
      da.V_pad = static_cast<int>(L.ds_ld);
      da.bias = bias != nullptr ? static_cast<const uint8_t*>(bias) + size_t(v0) * 2 : nullptr;
      da.bias_part = bias_part != nullptr ? bias_part + v0 : nullptr;
      da.bias_blk0 = 0;
      da.tgt_base = v0;
      da.ds_t = nullptr;
      da.n_blocks = static_cast<int>(ceil_div(N, kPairM));
      da.v_tiles = static_cast<int>(ceil_div(vc, kBN));
      da.group_blocks = group_blocks_for(da.n_blocks, H);
      int grid = 1;
      da.panel_tiles = choose_panel_tiles(da.n_blocks, da.group_blocks, da.v_tiles, d.pairs, &grid);
      da.num_panels = static_cast<int>(ceil_div(da.v_tiles, da.panel_tiles));
      da.num_units = da.num_panels * da.n_blocks;
      v = launch("flce_dlogits_tc", st, [&] {
        da.clk = g_cur_clk;
        return launch_ds_tc(tm_h, tm_wc, da, f16, bias != nullptr, p->softcap > 0.f, grid, st);
      });
      if (v != FLCE_OK) return v;
      if (grad_hidden) {
        // grad_hidden[N, H] (+)= dS[N, vc] (K-major) x W[v0:v0+vc, H] (MN-major). The
        // first chunk starts the fp32 partial (from the existing gradient when
        // accumulating), the middle chunks add to it, and the last adds and casts.
        GemmOperand op_a, op_b;
        GemmArgs ga{};
        if ((v = make_k_operand(&op_a, da.ds, vc, N, ds_row_bytes, kBM, dt)) != FLCE_OK) return v;
        if ((v = make_mn_operand(&op_b, &ga.b_atoms, wc, H, vc, uint64_t(H) * 2, dt)) != FLCE_OK)
          return v;
        ga.M = N;
        ga.N = H;
        ga.K = vc;
        ga.m_tiles = static_cast<int>(ceil_div(N, kPairM));
        ga.n_tiles = static_cast<int>(ceil_div(H, kBN));
        ga.k_blocks = static_cast<int>(ceil_div(vc, kBK));
        ga.num_tiles = ga.m_tiles * ga.n_tiles;
        ga.k_splits = 1;
        ga.kb_per_split = ga.k_blocks;
        ga.a_mn = 0;
        ga.b_mn = 1;
        if (L.nchunks == 1)
          ga.mode = p->accumulate ? kAddOutToOut : kStoreOut;
        else if (c == 0)
          ga.mode = p->accumulate ? kAddOutToPart : kStorePart;
        else if (c == L.nchunks - 1)
          ga.mode = kAddPartToOut;
        else
          ga.mode = kAddPart;
        ga.out = grad_hidden;
        ga.ld_out = H;
        ga.part = reinterpret_cast<float*>(ws + L.dh_part);
        ga.ld_part = H;
        ga.acc_scale = acc_scale;
        ga.status = status;
        ga.r_out = r_gh;
        ga.r_part = r_dh;
        const int g2 = ga.num_tiles < d.pairs ? ga.num_tiles : d.pairs;
        v = launch("flce_grad_hidden_tc", st,
                   [&] { return launch_gemm(op_a, op_b, ga, f16, g2, st); });
        if (v != FLCE_OK) return v;
      }
      if (grad_weight) {
        // grad_weight[v0:v0+vc, H] = (h^T[H, N] (K-major, the transposed copy
        // of h) x dS[N, vc] (MN-major through the 3-D view))^T: complete after
        // this one GEMM, whose epilogue stores its tiles transposed straight
        // into the output.
        GemmOperand op_a, op_b;
        GemmArgs ga{};
        if ((v = make_k_operand(&op_a, ws + L.ht, N, H, uint64_t(L.ht_ld) * 2, kBM, dt)) != FLCE_OK)
          return v;
        if ((v = make_mn_operand(&op_b, &ga.b_atoms, da.ds, vc, N, ds_row_bytes, dt)) != FLCE_OK)
          return v;
        ga.M = H;
        ga.N = vc;
        ga.K = N;
        ga.m_tiles = static_cast<int>(ceil_div(H, kPairM));
        ga.n_tiles = static_cast<int>(ceil_div(vc, kBN));
        ga.k_blocks = static_cast<int>(ceil_div(N, kBK));
        ga.num_tiles = ga.m_tiles * ga.n_tiles;
        ga.k_splits = 1;
        ga.kb_per_split = ga.k_blocks;
        ga.a_mn = 0;
        ga.b_mn = 1;
        ga.mode = p->accumulate ? kAddOutToOutT : kStoreOutT;
        ga.out_t = static_cast<uint8_t*>(grad_weight) + size_t(v0) * H * 2;
        ga.ld_out_t = H;
        ga.part = nullptr;
        ga.acc_scale = acc_scale;
        ga.status = status;
        ga.r_out_t = r_gw;
        // h^T (64 MB at H = 4096, N = 8192) is read by every wave of tiles; the
        // dlogits chunk streams through once per group of row tiles
        ga.a_l2 = kL2EvictLast;
        ga.b_l2 = kL2EvictFirst;
        const int g2 = ga.num_tiles < d.pairs ? ga.num_tiles : d.pairs;
        v = launch("flce_grad_weight_tc", st,
                   [&] { return launch_gemm(op_a, op_b, ga, f16, g2, st); });
        if (v != FLCE_OK) return v;
      }
    }
    for (int c = 0; c < nchunks_rows; ++c) {
      const int row0 = static_cast<int>(c * L.chunk);
      const int rows = static_cast<int>(N - row0 < L.chunk ? N - row0 : L.chunk);
      da.rows = rows;
      da.row0 = row0;
      da.n_blocks = static_cast<int>(ceil_div(rows, kPairM));
      da.v_tiles = static_cast<int>(ceil_div(V, kBN));
      da.group_blocks = group_blocks_for(da.n_blocks, H);
      int grid = 1;
      da.panel_tiles = choose_panel_tiles(da.n_blocks, da.group_blocks, da.v_tiles, d.pairs, &grid);
      da.num_panels = static_cast<int>(ceil_div(da.v_tiles, da.panel_tiles));
      da.num_units = da.num_panels * da.n_blocks;
      da.bias_blk0 = row0 / kBM;
      da.ds_t = grad_weight != nullptr && !L.wt ? ws + L.ds_t : nullptr;
      da.ld_t = L.ds_t_ld;
      v = launch("flce_dlogits_tc", st, [&] {
        da.clk = g_cur_clk;
        return launch_ds_tc(tm_h, tm_w, da, f16, bias != nullptr, p->softcap > 0.f, grid, st);
      });
      if (v != FLCE_OK) return v;
      const uint64_t ds_row_bytes = uint64_t(L.V_pad) * 2;
      if (grad_hidden) {
        // grad_hidden[rows, H] = dS[rows, V] (K-major) x W[V, H] (MN-major)
        GemmOperand op_a, op_b;
        GemmArgs ga{};
        if ((v = make_k_operand(&op_a, da.ds, V, rows, ds_row_bytes, kBM, dt)) != FLCE_OK) return v;
        if ((v = make_mn_operand(&op_b, &ga.b_atoms, weight, H, V, uint64_t(H) * 2, dt)) != FLCE_OK)
          return v;
        ga.M = rows;
        ga.N = H;
        ga.K = V;
        ga.m_tiles = static_cast<int>(ceil_div(rows, kPairM));
        ga.n_tiles = static_cast<int>(ceil_div(H, kBN));
        ga.k_blocks = static_cast<int>(ceil_div(V, kBK));
        ga.num_tiles = ga.m_tiles * ga.n_tiles;
        ga.k_splits = choose_k_splits(ga.num_tiles, ga.k_blocks, d.pairs);
        ga.kb_per_split = static_cast<int>(ceil_div(ga.k_blocks, ga.k_splits));
        ga.a_mn = 0;
        ga.b_mn = 1;
        ga.mode = p->accumulate ? kAddOutToOut : kStoreOut;
        ga.out = static_cast<uint8_t*>(grad_hidden) + size_t(row0) * H * 2;
        ga.ld_out = H;
        ga.part = reinterpret_cast<float*>(ws + L.dh_part);
        ga.ld_part = H;
        ga.split_stride = static_cast<long long>(L.chunk) * H;
        ga.acc_scale = acc_scale;
        ga.status = status;
        ga.r_out = r_gh;
        ga.r_part = r_dh;
        const int units = ga.num_tiles * ga.k_splits;
        const int g2 = units < d.pairs ? units : d.pairs;
        v = launch("flce_grad_hidden_tc", st,
                   [&] { return launch_gemm(op_a, op_b, ga, f16, g2, st); });
        if (v != FLCE_OK) return v;
        if (ga.k_splits > 1) {
          SplitReduceArgs ra2{};
          ra2.M = rows;
          ra2.N = H;
          ra2.splits = ga.k_splits;
          ra2.accumulate = p->accumulate;
          ra2.f16 = f16 ? 1 : 0;
          ra2.part = ga.part;
          ra2.ld_part = H;
          ra2.split_stride = ga.split_stride;
          ra2.out = ga.out;
          ra2.ld_out = H;
          v = launch("flce_split_reduce", st, [&] { return launch_split_reduce(ra2, st); });
          if (v != FLCE_OK) return v;
        }
      }
      if (grad_weight && L.wt) {
        // grad_weight[V, H] (+)= (h^T[H, row0:row0+rows] (K-major, columns of
        // the transposed copy of h) x dS[rows, V] (MN-major through the 3-D
        // view))^T. Across row chunks: the fp32 partial grad_weight^T
        // [H][dw_ld] (started by the first chunk, added to by the middle
        // ones, added and stored transposed by the last), or, accumulating in
        // the weight dtype, the output read, added and rewritten transposed.
        GemmOperand op_a, op_b;
        GemmArgs ga{};
        const uint8_t* htc = ws + L.ht + size_t(row0) * 2;
        if ((v = make_k_operand(&op_a, htc, rows, H, uint64_t(L.ht_ld) * 2, kBM, dt)) != FLCE_OK)
          return v;
        if ((v = make_mn_operand(&op_b, &ga.b_atoms, da.ds, V, rows, ds_row_bytes, dt)) != FLCE_OK)
          return v;
        ga.M = H;
        ga.N = V;
        ga.K = rows;
        ga.m_tiles = static_cast<int>(ceil_div(H, kPairM));
        ga.n_tiles = static_cast<int>(ceil_div(V, kBN));
        ga.k_blocks = static_cast<int>(ceil_div(rows, kBK));
        ga.num_tiles = ga.m_tiles * ga.n_tiles;
        ga.k_splits = 1;
        ga.kb_per_split = ga.k_blocks;
        ga.a_mn = 0;
        ga.b_mn = 1;
        if (p->grad_weight_accum == FLCE_ACCUM_WEIGHT || L.nchunks == 1)
          ga.mode = (c > 0 || p->accumulate) ? kAddOutToOutT : kStoreOutT;
        else if (c == 0)
          ga.mode = kStorePart;
        else if (c == L.nchunks - 1)
          ga.mode = kAddPartToOutT;
        else
          ga.mode = kAddPart;
        ga.out_t = grad_weight;
        ga.ld_out_t = H;
        ga.part = dw_part;
        ga.ld_part = L.dw_ld;
        ga.acc_scale = acc_scale;
        ga.status = status;
        ga.r_out_t = r_gw;
        ga.r_part = r_dw;
        // the chunk's columns of h^T stay in L2 while the dlogits columns
        // stream through once
        ga.a_l2 = kL2EvictLast;
        ga.b_l2 = kL2EvictFirst;
        const int g2 = ga.num_tiles < d.pairs ? ga.num_tiles : d.pairs;
        v = launch("flce_grad_weight_tc", st,
                   [&] { return launch_gemm(op_a, op_b, ga, f16, g2, st); });
        if (v != FLCE_OK) return v;
      } else if (grad_weight) {
        // grad_weight[V, H] (+)= dS^T[V, rows] (K-major, the transposed copy)
        // x h[rows, H] (MN-major)
        GemmOperand op_a, op_b;
        GemmArgs ga{};
        if ((v = make_k_operand(&op_a, da.ds_t, rows, V, uint64_t(L.ds_t_ld) * 2, kBM, dt)) != FLCE_OK)
          return v;
        const void* hc = static_cast<const uint8_t*>(hidden) + size_t(row0) * H * 2;
        if ((v = make_mn_operand(&op_b, &ga.b_atoms, hc, H, rows, uint64_t(H) * 2, dt)) != FLCE_OK)
          return v;
        ga.M = V;
        ga.N = H;
        ga.K = rows;
        ga.m_tiles = static_cast<int>(ceil_div(V, kPairM));
        ga.n_tiles = static_cast<int>(ceil_div(H, kBN));
        ga.k_blocks = static_cast<int>(ceil_div(rows, kBK));
        ga.num_tiles = ga.m_tiles * ga.n_tiles;
        ga.k_splits = 1;
        ga.kb_per_split = ga.k_blocks;
        ga.a_mn = 0;
        ga.b_mn = 1;
        // grad_weight across row chunks. fp32: the first chunk starts the fp32
        // partial (from the existing gradient when accumulating), the middle
        // chunks add to it, and the last adds and casts. Weight dtype: every
        // chunk after the first reads, adds and rewrites the output.
        if (p->grad_weight_accum == FLCE_ACCUM_WEIGHT || L.nchunks == 1)
          ga.mode = (c > 0 || p->accumulate) ? kAddOutToOut : kStoreOut;
        else if (c == 0)
          ga.mode = p->accumulate ? kAddOutToPart : kStorePart;
        else if (c == L.nchunks - 1)
          ga.mode = kAddPartToOut;
        else
          ga.mode = kAddPart;
        ga.out = grad_weight;
        ga.ld_out = H;
        ga.part = dw_part;
        ga.ld_part = H;
        ga.acc_scale = acc_scale;
        ga.status = status;
        ga.r_out = r_gw;
        ga.r_part = r_dw;
        const int g2 = ga.num_tiles < d.pairs ? ga.num_tiles : d.pairs;
        v = launch("flce_grad_weight_tc", st,
                   [&] { return launch_gemm(op_a, op_b, ga, f16, g2, st); });
        if (v != FLCE_OK) return v;
      }
    }
  } else if (L.vocab) {
    // fp32, vocabulary chunks (N < V): dlogits for columns [v0, v0 + vc) of
    // all rows, one fp32 copy. Each chunk's grad_weight rows are complete after
    // one contraction over all N rows; grad_hidden accumulates in its own fp32
    // output across the chunks, in chunk order.
    const float* hf = static_cast<const float*>(hidden);
    const float* wf = static_cast<const float*>(weight);
    for (int c = 0; c < L.nchunks; ++c) {
      const int v0 = static_cast<int>(c * L.chunk);
      const int vc = static_cast<int>(V - v0 < L.chunk ? V - v0 : L.chunk);
      da.rows = N;
      da.row0 = 0;
      da.V = vc;
      da.V_pad = static_cast<int>(L.ds_ld);
      da.bias = bias != nullptr ? static_cast<const float*>(bias) + v0 : nullptr;
      da.bias_part = bias_part != nullptr ? bias_part + v0 : nullptr;
      da.bias_blk0 = 0;
      da.tgt_base = v0;
      const float* wc = wf + size_t(v0) * H;
      v = launch("flce_dlogits_simt", st, [&] { return launch_ds_simt(hf, wc, da, st); });
      if (v != FLCE_OK) return v;
      const float* ds = reinterpret_cast<const float*>(da.ds);
      SimtGemmArgs gh_args{}, gw_args{};
      if (grad_hidden) {
        SimtGemmArgs& ga = gh_args;
        ga.M = N;
        ga.N = H;
        ga.K = vc;
        ga.A = ds;
        ga.sam = L.ds_ld;
        ga.sak = 1;
        ga.B = wc;
        ga.sbk = H;
        ga.sbn = 1;
        ga.C = static_cast<float*>(grad_hidden);
        ga.ldc = H;
        ga.accumulate = (c > 0 || p->accumulate) ? 1 : 0;
        ga.k_splits = simt_k_splits(N, H, vc);
        ga.part = reinterpret_cast<float*>(ws + L.dh_part);
        ga.tile_count = reinterpret_cast<int*>(ws + L.cnt);
        ga.status = status;
        ga.r_c = r_gh;
        ga.r_part = r_dh;
      }
      if (grad_weight) {
        SimtGemmArgs& ga = gw_args;
        ga.M = vc;
        ga.N = H;
        ga.K = N;
        ga.A = ds;  // A(m, k) = dlogits[k][m]
        ga.sam = 1;
        ga.sak = L.ds_ld;
        ga.B = hf;
        ga.sbk = H;
        ga.sbn = 1;
        ga.C = static_cast<float*>(grad_weight) + size_t(v0) * H;
        ga.ldc = H;
        ga.accumulate = p->accumulate;
        ga.status = status;
        ga.r_c = r_gw;
      }
      // Both contractions of the chunk in one grid when both are wanted: each
      // alone is too small to fill the GPU at the sizes this path serves.
      if (grad_hidden && grad_weight)
        v = launch("flce_grads_simt", st, [&] {
          return launch_gemm_simt2(gh_args, gw_args,
                                   reinterpret_cast<int*>(ws + L.cnt) + kSimtSplitTiles, st);
        });
      else if (grad_hidden)
        v = launch("flce_grad_hidden_simt", st, [&] { return launch_gemm_simt(gh_args, st); });
      else if (grad_weight)
        v = launch("flce_grad_weight_simt", st, [&] { return launch_gemm_simt(gw_args, st); });
      if (v != FLCE_OK) return v;
    }
  } else {
    const float* hf = static_cast<const float*>(hidden);
    const float* wf = static_cast<const float*>(weight);
    for (int c = 0; c < L.nchunks; ++c) {
      const int row0 = static_cast<int>(c * L.chunk);
      const int rows = static_cast<int>(N - row0 < L.chunk ? N - row0 : L.chunk);
      da.rows = rows;
      da.row0 = row0;
      da.bias_blk0 = row0 / kSimtTile;
      v = launch("flce_dlogits_simt", st, [&] { return launch_ds_simt(hf, wf, da, st); });
      if (v != FLCE_OK) return v;
      const float* ds = reinterpret_cast<const float*>(da.ds);
      if (grad_hidden) {
        SimtGemmArgs ga{};
        ga.M = rows;
        ga.N = H;
        ga.K = V;
        ga.A = ds;
        ga.sam = L.V_pad;
        ga.sak = 1;
        ga.B = wf;
        ga.sbk = H;
        ga.sbn = 1;
        ga.C = static_cast<float*>(grad_hidden) + size_t(row0) * H;
        ga.ldc = H;
        ga.accumulate = p->accumulate;
        // K = V is long and the chunk's output is small: split K, sized for
        // the full chunk so that the workspace holds every chunk's partials
        ga.k_splits = simt_k_splits(L.chunk, H, V);
        ga.part = reinterpret_cast<float*>(ws + L.dh_part);
        ga.tile_count = reinterpret_cast<int*>(ws + L.cnt);
        ga.status = status;
        ga.r_c = r_gh;
        ga.r_part = r_dh;
        v = launch("flce_grad_hidden_simt", st, [&] { return launch_gemm_simt(ga, st); });
        if (v != FLCE_OK) return v;
      }
      if (grad_weight) {
        SimtGemmArgs ga{};
        ga.M = V;
        ga.N = H;
        ga.K = rows;
        ga.A = ds;
        ga.sam = 1;
        ga.sak = L.V_pad;
        ga.B = hf + size_t(row0) * H;
        ga.sbk = H;
        ga.sbn = 1;
        ga.C = static_cast<float*>(grad_weight);
        ga.ldc = H;
        ga.accumulate = (c > 0 || p->accumulate) ? 1 : 0;
        ga.status = status;
        ga.r_c = r_gw;
        v = launch("flce_grad_weight_simt", st, [&] { return launch_gemm_simt(ga, st); });
        if (v != FLCE_OK) return v;
      }
    }
  }
  if (grad_bias) {
    BiasReduceArgs ba{};
    ba.V = V;
    ba.V_pad = static_cast<int>(L.V_pad);
    ba.nblk = L.n_rowblocks;
    ba.bias_part = bias_part;
    ba.grad_bias = grad_bias;
    ba.accumulate = p->accumulate;
    v = launch("flce_bias_reduce", st, [&] { return launch_bias_reduce(ba, p->dtype, st); });
    if (v != FLCE_OK) return v;
  }
  return debug_finish(ws, st, FLCE_OK);
}

// ---------------------------------------------------------------------------
// Generic chunked linear loss: the projection of one row chunk and the
// folding of its dlogits into the gradients ("Chunked Linear Loss").
int flce_chunk_logits(const flce_params* p, const void* hidden, const void* weight, void* logits,
                      int64_t ld_logits, void* workspace, size_t ws_bytes, flce_stream_t stream) {
  const NvtxRange nvtx_range("flce_chunk_logits");
  int v = validate(p);
  if (v != FLCE_OK) return v;
  if (weight == nullptr || (p->N > 0 && (hidden == nullptr || logits == nullptr)))
    return FLCE_ERR_INVALID_ARG;
  if (ld_logits < p->V || ld_logits % 8 != 0) return FLCE_ERR_INVALID_ARG;
  if (workspace == nullptr || ws_bytes < kHeader) return FLCE_ERR_WORKSPACE;
  if (!aligned_for(p, hidden) || !aligned_for(p, weight) || !aligned_for(p, logits) ||
      !aligned16(workspace))
    return FLCE_ERR_ALIGNMENT;
  DeviceInfo d;
  if ((v = device_info(&d)) != FLCE_OK) return v;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t e = cudaMemsetAsync(ws, 0, kHeader, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  if (p->N == 0) return FLCE_OK;
  const int N = static_cast<int>(p->N), H = static_cast<int>(p->H), V = static_cast<int>(p->V);
  if (tensor_path(p)) {
    // logits[N, V] = h[N, H] (K-major) x W[V, H]^T (K-major B)
    const CUtensorMapDataType dt = map_type(p);
    GemmOperand op_a, op_b;
    GemmArgs ga{};
    if ((v = make_k_operand(&op_a, hidden, H, N, uint64_t(H) * 2, kBM, dt)) != FLCE_OK) return v;
    if ((v = make_k_operand(&op_b, weight, H, V, uint64_t(H) * 2, kBNHalf, dt)) != FLCE_OK) return v;
    ga.M = N;
    ga.N = V;
    ga.K = H;
    ga.m_tiles = static_cast<int>(ceil_div(N, kPairM));
    ga.n_tiles = static_cast<int>(ceil_div(V, kBN));
    ga.k_blocks = static_cast<int>(ceil_div(H, kBK));
    ga.num_tiles = ga.m_tiles * ga.n_tiles;
    ga.k_splits = 1;
    ga.kb_per_split = ga.k_blocks;
    ga.a_mn = 0;
    ga.b_mn = 0;
    ga.mode = kStoreOut;
    ga.out = logits;
    ga.ld_out = ld_logits;
    ga.part = nullptr;
    ga.ld_part = 0;
    ga.status = reinterpret_cast<int*>(ws);
    ga.r_out = DevRegion{logits, size_t(N) * ld_logits * 2};
    const bool f16 = p->dtype == FLCE_F16;
    const int g2 = ga.num_tiles < d.pairs ? ga.num_tiles : d.pairs;
    return debug_finish(ws, st, launch("flce_chunk_logits_tc", st, [&] {
                          return launch_gemm(op_a, op_b, ga, f16, g2, st);
                        }));
  }
  SimtGemmArgs ga{};
  ga.M = N;
  ga.N = V;
  ga.K = H;
  ga.A = static_cast<const float*>(hidden);
  ga.sam = H;
  ga.sak = 1;
  ga.B = static_cast<const float*>(weight);  // B(k, n) = W[n][k]
  ga.sbk = 1;
  ga.sbn = H;
  ga.C = static_cast<float*>(logits);
  ga.ldc = ld_logits;
  ga.accumulate = 0;
  ga.status = reinterpret_cast<int*>(ws);
  ga.r_c = DevRegion{logits, size_t(N) * ld_logits * 4};
  return debug_finish(ws, st,
                      launch("flce_chunk_logits_simt", st, [&] { return launch_gemm_simt(ga, st); }));
}

int flce_chunk_weighted_mse(const flce_params* p, const void* hidden, const void* weight,
                            const float* target, int64_t ld_target, const float* row_weight,
                            const float* feature_weight, void* dlogits, int64_t ld_dlogits,
                            void* dlogits_t, int64_t ld_dlogits_t, double* loss,
                            int32_t accumulate_loss, void* workspace, size_t ws_bytes,
                            flce_stream_t stream) {
  const NvtxRange nvtx_range("flce_chunk_weighted_mse");
  int v = validate(p);
  if (v != FLCE_OK) return v;
  if (!tensor_path(p)) return FLCE_ERR_UNSUPPORTED;
  if (p->N < 1 || hidden == nullptr || weight == nullptr || target == nullptr ||
      row_weight == nullptr || feature_weight == nullptr || dlogits == nullptr || loss == nullptr)
    return FLCE_ERR_INVALID_ARG;
  if (accumulate_loss != 0 && accumulate_loss != 1) return FLCE_ERR_INVALID_ARG;
  if (ld_target < p->V || ld_target % 4 != 0 || ld_dlogits < p->V || ld_dlogits % 8 != 0)
    return FLCE_ERR_INVALID_ARG;
  if (dlogits_t != nullptr && (ld_dlogits_t < p->N || ld_dlogits_t % 8 != 0))
    return FLCE_ERR_INVALID_ARG;
  if (dlogits_t != nullptr && !aligned16(dlogits_t)) return FLCE_ERR_ALIGNMENT;
  const int N = static_cast<int>(p->N), H = static_cast<int>(p->H), V = static_cast<int>(p->V);
  const int n_tiles = static_cast<int>(ceil_div(V, kBN));
  const size_t need = align_up(kHeader + mse_loss_part_bytes(p), 256);
  if (workspace == nullptr || ws_bytes < need) return FLCE_ERR_WORKSPACE;
  if (!aligned16(hidden) || !aligned16(weight) || !aligned16(target) ||
      (reinterpret_cast<uintptr_t>(row_weight) & 3u) != 0 || !aligned16(feature_weight) ||
      !aligned16(dlogits) || !aligned16(workspace) || (reinterpret_cast<uintptr_t>(loss) & 7u) != 0)
    return FLCE_ERR_ALIGNMENT;
  DeviceInfo d;
  if ((v = device_info(&d)) != FLCE_OK) return v;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t e = cudaMemsetAsync(ws, 0, kHeader, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  // dlogits[N, V] = 2 r f (h W^T - y): the GEMM of flce_chunk_logits, with the
  // loss applied to the fp32 accumulator in the epilogue.
  const CUtensorMapDataType dt = map_type(p);
  GemmOperand op_a, op_b;
  GemmArgs ga{};
  if ((v = make_k_operand(&op_a, hidden, H, N, uint64_t(H) * 2, kBM, dt)) != FLCE_OK) return v;
  if ((v = make_k_operand(&op_b, weight, H, V, uint64_t(H) * 2, kBNHalf, dt)) != FLCE_OK) return v;
  ga.M = N;
  ga.N = V;
  ga.K = H;
  ga.m_tiles = static_cast<int>(ceil_div(N, kPairM));
  ga.n_tiles = n_tiles;
  ga.k_blocks = static_cast<int>(ceil_div(H, kBK));
  ga.num_tiles = ga.m_tiles * ga.n_tiles;
  ga.k_splits = 1;
  ga.kb_per_split = ga.k_blocks;
  ga.a_mn = 0;
  ga.b_mn = 0;
  ga.mode = kWeightedMse;
  ga.out = dlogits;
  ga.ld_out = ld_dlogits;
  ga.status = reinterpret_cast<int*>(ws);
  ga.target = target;
  ga.ld_target = ld_target;
  ga.row_w = row_weight;
  ga.feat_w = feature_weight;
  ga.loss_part = reinterpret_cast<float*>(ws + kHeader);
  ga.out_t = dlogits_t;
  ga.ld_out_t = ld_dlogits_t;
  ga.r_out = DevRegion{dlogits, size_t(N) * ld_dlogits * 2};
  ga.r_out_t = DevRegion{dlogits_t, dlogits_t ? size_t(V) * ld_dlogits_t * 2 : 0};
  ga.r_loss = DevRegion{ws + kHeader, mse_loss_part_bytes(p)};
  const bool f16 = p->dtype == FLCE_F16;
  const int g2 = ga.num_tiles < d.pairs ? ga.num_tiles : d.pairs;
  v = launch("flce_chunk_mse_tc", st, [&] { return launch_gemm(op_a, op_b, ga, f16, g2, st); });
  if (v != FLCE_OK) return v;
  LossReduceArgs la{};
  la.part = ga.loss_part;
  la.count = static_cast<long long>(n_tiles) * ceil_div(N, 32);
  la.loss = loss;
  la.accumulate = accumulate_loss;
  return debug_finish(ws, st,
                      launch("flce_loss_reduce", st, [&] { return launch_loss_reduce(la, st); }));
}

int flce_chunk_grads(const flce_params* p, const void* hidden, const void* weight,
                     const void* dlogits, int64_t ld_dlogits, const void* dlogits_t,
                     int64_t ld_dlogits_t, int32_t phase, void* grad_hidden, void* grad_weight,
                     void* workspace, size_t ws_bytes, flce_stream_t stream) {
  const NvtxRange nvtx_range("flce_chunk_grads");
  int v = validate(p);
  if (v != FLCE_OK) return v;
  if (p->N < 1 || phase < FLCE_CHUNK_ONLY || phase > FLCE_CHUNK_LAST) return FLCE_ERR_INVALID_ARG;
  if (hidden == nullptr || weight == nullptr || dlogits == nullptr) return FLCE_ERR_INVALID_ARG;
  if (ld_dlogits < p->V || ld_dlogits % 8 != 0) return FLCE_ERR_INVALID_ARG;
  if (dlogits_t != nullptr && (!tensor_path(p) || ld_dlogits_t < p->N || ld_dlogits_t % 8 != 0))
    return FLCE_ERR_INVALID_ARG;
  if (dlogits_t != nullptr && !aligned16(dlogits_t)) return FLCE_ERR_ALIGNMENT;
  const ChunkLayout L = chunk_layout(p);
  if (workspace == nullptr || ws_bytes < L.total) return FLCE_ERR_WORKSPACE;
  if (!aligned_for(p, hidden) || !aligned_for(p, weight) || !aligned_for(p, dlogits) ||
      !aligned16(workspace) || (grad_hidden && !aligned_for(p, grad_hidden)) ||
      (grad_weight && !aligned_for(p, grad_weight)))
    return FLCE_ERR_ALIGNMENT;
  DeviceInfo d;
  if ((v = device_info(&d)) != FLCE_OK) return v;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* status = reinterpret_cast<int*>(ws);
  cudaError_t e = cudaMemsetAsync(ws, 0, kHeader, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  const int N = static_cast<int>(p->N), H = static_cast<int>(p->H), V = static_cast<int>(p->V);
  // grad_weight: the chunk's rows add dlogits^T h. Across chunks the fp32
  // partial is started by the first chunk (from grad_weight when
  // accumulating), added to by the next ones, and added and cast by the last.
  // In the weight dtype every chunk after the first adds into grad_weight.
  const bool later = phase == FLCE_CHUNK_NEXT || phase == FLCE_CHUNK_LAST;
  if (!tensor_path(p)) {
    const float* df = static_cast<const float*>(dlogits);
    if (grad_hidden) {
      SimtGemmArgs ga{};
      ga.M = N;
      ga.N = H;
      ga.K = V;
      ga.A = df;
      ga.sam = ld_dlogits;
      ga.sak = 1;
      ga.B = static_cast<const float*>(weight);
      ga.sbk = H;
      ga.sbn = 1;
      ga.C = static_cast<float*>(grad_hidden);
      ga.ldc = H;
      ga.accumulate = p->accumulate;
      ga.k_splits = simt_k_splits(N, H, V);
      ga.part = reinterpret_cast<float*>(ws + L.dh_part);
      ga.status = status;
      ga.r_c = DevRegion{grad_hidden, size_t(N) * H * 4};
      ga.r_part = DevRegion{ws + L.dh_part, L.dh_bytes};
      v = launch("flce_chunk_grad_hidden_simt", st, [&] { return launch_gemm_simt(ga, st); });
      if (v != FLCE_OK) return v;
    }
    if (grad_weight) {
      SimtGemmArgs ga{};
      ga.M = V;
      ga.N = H;
      ga.K = N;
      ga.A = df;  // A(m, k) = dlogits[k][m]
      ga.sam = 1;
      ga.sak = ld_dlogits;
      ga.B = static_cast<const float*>(hidden);
      ga.sbk = H;
      ga.sbn = 1;
      ga.C = static_cast<float*>(grad_weight);
      ga.ldc = H;
      ga.accumulate = (later || p->accumulate) ? 1 : 0;
      ga.status = status;
      ga.r_c = DevRegion{grad_weight, size_t(V) * H * 4};
      v = launch("flce_chunk_grad_weight_simt", st, [&] { return launch_gemm_simt(ga, st); });
      if (v != FLCE_OK) return v;
    }
    return debug_finish(ws, st, FLCE_OK);
  }
  const CUtensorMapDataType dt = map_type(p);
  const bool f16 = p->dtype == FLCE_F16;
  const uint64_t dl_row_bytes = uint64_t(ld_dlogits) * 2;
  if (grad_hidden) {
    // grad_hidden[N, H] (+)= dlogits[N, V] (K-major) x W[V, H] (MN-major)
    GemmOperand op_a, op_b;
    GemmArgs ga{};
    if ((v = make_k_operand(&op_a, dlogits, V, N, dl_row_bytes, kBM, dt)) != FLCE_OK) return v;
    if ((v = make_mn_operand(&op_b, &ga.b_atoms, weight, H, V, uint64_t(H) * 2, dt)) != FLCE_OK)
      return v;
    ga.M = N;
    ga.N = H;
    ga.K = V;
    ga.m_tiles = static_cast<int>(ceil_div(N, kPairM));
    ga.n_tiles = static_cast<int>(ceil_div(H, kBN));
    ga.k_blocks = static_cast<int>(ceil_div(V, kBK));
    ga.num_tiles = ga.m_tiles * ga.n_tiles;
    ga.k_splits = choose_k_splits(ga.num_tiles, ga.k_blocks, d.pairs);
    ga.kb_per_split = static_cast<int>(ceil_div(ga.k_blocks, ga.k_splits));
    ga.a_mn = 0;
    ga.b_mn = 1;
    ga.mode = p->accumulate ? kAddOutToOut : kStoreOut;
    ga.out = grad_hidden;
    ga.ld_out = H;
    ga.part = reinterpret_cast<float*>(ws + L.dh_part);
    ga.ld_part = H;
    ga.split_stride = static_cast<long long>(N) * H;
    ga.status = status;
    ga.r_out = DevRegion{grad_hidden, size_t(N) * H * 2};
    ga.r_part = DevRegion{ws + L.dh_part, L.dh_bytes};
    const int units = ga.num_tiles * ga.k_splits;
    const int g2 = units < d.pairs ? units : d.pairs;
    v = launch("flce_chunk_grad_hidden_tc", st,
               [&] { return launch_gemm(op_a, op_b, ga, f16, g2, st); });
    if (v != FLCE_OK) return v;
    if (ga.k_splits > 1) {
      SplitReduceArgs ra{};
      ra.M = N;
      ra.N = H;
      ra.splits = ga.k_splits;
      ra.accumulate = p->accumulate;
      ra.f16 = f16 ? 1 : 0;
      ra.part = ga.part;
      ra.ld_part = H;
      ra.split_stride = ga.split_stride;
      ra.out = grad_hidden;
      ra.ld_out = H;
      v = launch("flce_split_reduce", st, [&] { return launch_split_reduce(ra, st); });
      if (v != FLCE_OK) return v;
    }
  }
  if (grad_weight && L.wt) {
    // grad_weight[V, H] (+)= (h^T[H, N] (K-major) x dlogits[N, V] (MN-major
    // through the 3-D view))^T; the epilogue stores (or adds) its tiles
    // transposed. The fp32 partial across chunks is grad_weight^T [H][dw_ld].
    TransposeArgs ta{};
    ta.src = static_cast<const uint16_t*>(hidden);
    ta.dst = reinterpret_cast<uint16_t*>(ws + L.ht);
    ta.rows = N;
    ta.cols = H;
    ta.ld_src = H;
    ta.ld_dst = L.ht_ld;
    ta.status = status;
    ta.r_dst = DevRegion{ws + L.ht, L.ht_bytes};
    v = launch("flce_transpose_hidden", st, [&] { return launch_transpose16(ta, st); });
    if (v != FLCE_OK) return v;
    GemmOperand op_a, op_b;
    GemmArgs ga{};
    if ((v = make_k_operand(&op_a, ws + L.ht, N, H, uint64_t(L.ht_ld) * 2, kBM, dt)) != FLCE_OK)
      return v;
    if ((v = make_mn_operand(&op_b, &ga.b_atoms, dlogits, V, N, dl_row_bytes, dt)) != FLCE_OK)
      return v;
    ga.M = H;
    ga.N = V;
    ga.K = N;
    ga.m_tiles = static_cast<int>(ceil_div(H, kPairM));
    ga.n_tiles = static_cast<int>(ceil_div(V, kBN));
    ga.k_blocks = static_cast<int>(ceil_div(N, kBK));
    ga.num_tiles = ga.m_tiles * ga.n_tiles;
    ga.k_splits = 1;
    ga.kb_per_split = ga.k_blocks;
    ga.a_mn = 0;
    ga.b_mn = 1;
    if (phase == FLCE_CHUNK_ONLY || p->grad_weight_accum == FLCE_ACCUM_WEIGHT)
      ga.mode = (later || p->accumulate) ? kAddOutToOutT : kStoreOutT;
    else if (phase == FLCE_CHUNK_FIRST)
      ga.mode = kStorePart;
    else if (phase == FLCE_CHUNK_NEXT)
      ga.mode = kAddPart;
    else
      ga.mode = kAddPartToOutT;
    ga.out_t = grad_weight;
    ga.ld_out_t = H;
    ga.part = reinterpret_cast<float*>(ws + L.dw_part);
    ga.ld_part = L.dw_ld;
    ga.status = status;
    ga.r_out_t = DevRegion{grad_weight, size_t(V) * H * 2};
    ga.r_part = DevRegion{ws + L.dw_part, L.dw_bytes};
    ga.a_l2 = kL2EvictLast;
    ga.b_l2 = kL2EvictFirst;
    const int g2 = ga.num_tiles < d.pairs ? ga.num_tiles : d.pairs;
    v = launch("flce_chunk_grad_weight_tc", st,
               [&] { return launch_gemm(op_a, op_b, ga, f16, g2, st); });
    if (v != FLCE_OK) return v;
  } else if (grad_weight) {
    // grad_weight[V, H] (+)= dlogits^T[V, N] x h[N, H] (MN-major). dlogits^T is
    // read K-major from the transposed copy when the caller has one, else
    // MN-major from dlogits (about 20 % slower).
    GemmOperand op_a, op_b;
    GemmArgs ga{};
    if (dlogits_t != nullptr) {
      if ((v = make_k_operand(&op_a, dlogits_t, N, V, uint64_t(ld_dlogits_t) * 2, kBM, dt)) !=
          FLCE_OK)
        return v;
    } else {
      if ((v = make_mn_operand(&op_a, &ga.a_atoms, dlogits, V, N, dl_row_bytes, dt)) != FLCE_OK)
        return v;
      ga.a_atoms = 0;  // the A side loads through the 2-D map (the 3-D view does not help it)
    }
    if ((v = make_mn_operand(&op_b, &ga.b_atoms, hidden, H, N, uint64_t(H) * 2, dt)) != FLCE_OK)
      return v;
    ga.M = V;
    ga.N = H;
    ga.K = N;
    ga.m_tiles = static_cast<int>(ceil_div(V, kPairM));
    ga.n_tiles = static_cast<int>(ceil_div(H, kBN));
    ga.k_blocks = static_cast<int>(ceil_div(N, kBK));
    ga.num_tiles = ga.m_tiles * ga.n_tiles;
    ga.k_splits = 1;
    ga.kb_per_split = ga.k_blocks;
    ga.a_mn = dlogits_t != nullptr ? 0 : 1;
    ga.b_mn = 1;
    if (phase == FLCE_CHUNK_ONLY || p->grad_weight_accum == FLCE_ACCUM_WEIGHT)
      ga.mode = (later || p->accumulate) ? kAddOutToOut : kStoreOut;
    else if (phase == FLCE_CHUNK_FIRST)
      ga.mode = p->accumulate ? kAddOutToPart : kStorePart;
    else if (phase == FLCE_CHUNK_NEXT)
      ga.mode = kAddPart;
    else
      ga.mode = kAddPartToOut;
    ga.out = grad_weight;
    ga.ld_out = H;
    ga.part = reinterpret_cast<float*>(ws + L.dw_part);
    ga.ld_part = H;
    ga.status = status;
    ga.r_out = DevRegion{grad_weight, size_t(V) * H * 2};
    ga.r_part = DevRegion{ws + L.dw_part, L.dw_bytes};
    const int g2 = ga.num_tiles < d.pairs ? ga.num_tiles : d.pairs;
    v = launch("flce_chunk_grad_weight_tc", st,
               [&] { return launch_gemm(op_a, op_b, ga, f16, g2, st); });
    if (v != FLCE_OK) return v;
  }
  return debug_finish(ws, st, FLCE_OK);
}

int flce_scale(const void* src, void* dst, int64_t count, int32_t dtype, const float* scale,
               flce_stream_t stream) {
  if (count < 0 || (dtype != FLCE_F32 && dtype != FLCE_BF16 && dtype != FLCE_F16) ||
      scale == nullptr || (count > 0 && (src == nullptr || dst == nullptr)))
    return FLCE_ERR_INVALID_ARG;
  const size_t elem = dtype == FLCE_F32 ? 4 : 2;
  if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) % elem != 0 ||
      (reinterpret_cast<uintptr_t>(scale) & 3u) != 0)
    return FLCE_ERR_ALIGNMENT;
  if (count == 0) return FLCE_OK;
  DeviceInfo d;
  int v = device_info(&d);
  if (v != FLCE_OK) return v;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  ScaleArgs a{src, dst, static_cast<long long>(count), dtype, scale};
  return launch("flce_scale", st, [&] { return launch_scale(a, d.sms, st); });
}

int flce_check_status(const void* workspace, flce_stream_t stream) {
  if (workspace == nullptr) return FLCE_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync");
  if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  if (word & kDevErrBounds) return FLCE_ERR_BOUNDS;
  if (word & kDevErrTimeout) return FLCE_ERR_TIMEOUT;
  if (word & kDevErrTargetRange) return FLCE_ERR_TARGET_RANGE;
  return FLCE_OK;
}

int flce_profiling_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof = on != 0;
  return FLCE_OK;
}

int flce_profiling_read(flce_kernel_time* out, int max, int* count) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  int cur = 0;
  cudaGetDevice(&cur);
  for (const Pending& p : g_pending) {
    cudaError_t e = cudaEventSynchronize(p.e1);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
    float ms = 0.f;
    cudaEventElapsedTime(&ms, p.e0, p.e1);
    g_counts[p.name] += 1;
    g_ms[p.name] += ms;
    if (p.slot >= 0) {
      ClockRecord r{};
      cudaSetDevice(p.dev);
      e = cudaMemcpy(&r, g_clock_base[p.dev] + p.slot, sizeof(r), cudaMemcpyDeviceToHost);
      cudaSetDevice(cur);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy (clock record)");
      g_cycles[p.name] += static_cast<double>(r.cycles);
      g_clock_ns[p.name] += static_cast<double>(r.ns);
      g_mma_cycles[p.name] += static_cast<double>(r.mma_cycles);
      g_mma_wait_ops[p.name] += static_cast<double>(r.mma_wait_operands);
      g_mma_wait_acc[p.name] += static_cast<double>(r.mma_wait_accumulator);
    }
    g_pool.push_back(p.e0);
    g_pool.push_back(p.e1);
  }
  g_pending.clear();
  for (int& n : g_clock_next) n = 0;
  int n = 0;
  for (size_t i = 0; i < g_names.size(); ++i) {
    if (g_counts[i] == 0) continue;
    if (out != nullptr && n < max) {
      memset(&out[n], 0, sizeof(out[n]));
      strncpy(out[n].name, g_names[i].c_str(), sizeof(out[n].name) - 1);
      out[n].launches = g_counts[i];
      out[n].total_ms = g_ms[i];
      out[n].sm_mhz = g_clock_ns[i] > 0 ? g_cycles[i] / g_clock_ns[i] * 1e3 : 0.0;
      out[n].mma_wait_operands = g_mma_cycles[i] > 0 ? g_mma_wait_ops[i] / g_mma_cycles[i] : 0.0;
      out[n].mma_wait_accumulator = g_mma_cycles[i] > 0 ? g_mma_wait_acc[i] / g_mma_cycles[i] : 0.0;
    }
    ++n;
    g_counts[i] = 0;
    g_ms[i] = 0.0;
    g_cycles[i] = 0.0;
    g_clock_ns[i] = 0.0;
    g_mma_cycles[i] = 0.0;
    g_mma_wait_ops[i] = 0.0;
    g_mma_wait_acc[i] = 0.0;
  }
  if (count != nullptr) *count = n;
  return FLCE_OK;
}

}  // extern "C"
