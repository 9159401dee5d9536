// fsops_api.cu -- host side of the C ABI declared in include/fsops.h:
// argument validation, workspace layout, TMA descriptor encoding, launches.
// No function here allocates device memory or synchronises, except
// fsops_set_workspace and fsops_read_kernel_status, which say so.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "../../include/fsops.h"
#include "mx_internal.h"
#include "mx_tiled.h"
#include "mx_attention.h"
#include "mx_slice.h"
#include "mx_small.h"
#include "mx_blockscale.h"

using namespace fsops;

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kCtlRegionBytes = 16384;

struct DeviceInfo {
  bool init = false;
  bool ok = false;
  int sms = 0;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;

struct Workspace {
  void* ptr = nullptr;
  size_t bytes = 0;
};
Workspace g_ws[kMaxDevices];

std::atomic<uint64_t> g_timeout_ns{1000000000ull};
#ifdef FSOPS_TRACE
unsigned long long* g_trace = nullptr;
#endif
std::atomic<uint32_t> g_extra{0};
// Weight tiles (32 KB each) a block keeps in flight by default: 3 x 32 KB per
// SM covers the loaded HBM latency (~1.5 us) at the SM's share of the
// bandwidth; deeper queues only add latency to every other memory round trip
// (against 4: M = 16, H = 2560, I = 9728: 22.0 against 22.4 us; H = 5120,
// I = 17408: 0.2-0.5 us less at M = 1-32, equal at M = 64-128).
constexpr int kDefaultMaxInflight = 3;
// Plan overrides set through fsops_debug_set_knob (-1: the library's own
// choice).  Read with one atomic load per use; nothing is read from the
// process environment on the call path.
std::atomic<int> g_knob[FSOPS_KNOB_COUNT];
struct KnobInit {
  KnobInit() {
    for (auto& k : g_knob) k.store(-1);
  }
} g_knob_init;
int knob(fsops_knob k) { return g_knob[k].load(std::memory_order_relaxed); }
// The knob's value when it is one of the accepted ones, else `dflt`.
int knob_or(fsops_knob k, int dflt, int lo, int hi) {
  const int v = knob(k);
  return (v >= lo && v <= hi) ? v : dflt;
}
// FSOPS_VERBOSE, read once when the library is loaded.
const bool g_verbose = std::getenv("FSOPS_VERBOSE") != nullptr;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

fsops_status current_device(int* dev_out, const DeviceInfo** info) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return FSOPS_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.init) {
    d.init = true;
    int major = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) {
      d.ok = (major == 10);
      d.sms = sms < 256 ? sms : 256;  // one block per SM; the split arithmetic assumes at most 256
    }
    cudaGetLastError();
    if (g_encode == nullptr) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
              cudaSuccess &&
          q == cudaDriverEntryPointSuccess)
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
      cudaGetLastError();
    }
  }
  if (!d.ok || g_encode == nullptr) return FSOPS_ERR_NO_DEVICE;
  *dev_out = dev;
  *info = &d;
  return FSOPS_OK;
}

thread_local int g_last_cuda_error = 0;
// A failed CUDA step: clears the runtime's error state, records the error for
// fsops_last_cuda_error and, with FSOPS_VERBOSE set, reports it.
fsops_status cuda_failed(cudaError_t e, const char* where) {
  cudaGetLastError();
  g_last_cuda_error = static_cast<int>(e);
  if (g_verbose)
    std::fprintf(stderr, "fsops: %s failed: %s (%d)\n", where, cudaGetErrorString(e), static_cast<int>(e));
  return FSOPS_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
int npad_of(int M) { return (M + 15) / 16 * 16; }

// Accumulators are staged through shared memory (and all four epilogue warps
// share the work) when the tokens fit one TMEM lane quarter.
int stage_tmem_for(int npad) { return npad <= 32 ? 1 : 0; }
// Small M: every block quantises the k-chunks of x it needs itself (no
// grid-wide exchange before the first MMA; one warp, two 32-blocks per lane per
// stage).  Larger M: x is quantised once, each block a slice, shared through L2.
int local_xq_for(int npad) {
  if (npad > 16) return 0;
  return knob_or(FSOPS_KNOB_LOCAL_XQ, 1, 0, 2) ? 1 : 0;
}
// Shared memory besides the stage ring (local_xq is only used with x quantised in-kernel).
uint32_t extra_smem(int npad, int local_xq) {
  return (stage_tmem_for(npad) ? stg_bytes_for(npad) : 0u) + (local_xq ? xring_bytes_for(npad) : 0u) +
         kSmemCtlBytes + 1024u;
}
int stages_for(int npad, int local_xq) {
  int s = static_cast<int>((kMaxSmem - extra_smem(npad, local_xq)) / stage_bytes_for(npad));
  if (s > kMaxStages) s = kMaxStages;
  return s;
}
size_t smem_for(int npad, int local_xq) {
  return static_cast<size_t>(stages_for(npad, local_xq)) * stage_bytes_for(npad) + extra_smem(npad, local_xq);
}
// fp32 accumulators of split tiles: [tiles][M][256]
size_t accum_bytes(int M, int tiles) { return round_up(static_cast<size_t>(tiles) * M * kTileRows * 4, 1024); }

// ---------------------------------------------------------------- workspace layouts
struct GemmLayout {
  size_t ctl, xq, xq_sf, part, total;
};
GemmLayout gemm_layout(int M, int N, int K) {
  GemmLayout l;
  l.ctl = 0;
  l.xq = kCtlRegionBytes;
  l.xq_sf = l.xq + round_up(static_cast<size_t>(M) * K, 1024);
  // scale tiles of ceil(M / 128) row tiles; split-K sums only for M <= 128
  l.part = l.xq_sf + round_up(static_cast<size_t>((M + 127) / 128) * (K / 128) * 512, 1024);
  l.total = l.part + (M <= 128 ? accum_bytes(M, (N + kTileRows - 1) / kTileRows) : 0);
  return l;
}
struct MlpLayout {
  size_t ctl, xq, xq_sf, hq, hq_sf, part0, part1, gu, total;
};
MlpLayout mlp_layout(int M, int H, int I) {
  MlpLayout l;
  l.ctl = 0;
  l.xq = kCtlRegionBytes;
  l.xq_sf = l.xq + round_up(static_cast<size_t>(M) * H, 1024);
  const size_t row_tiles = static_cast<size_t>((M + 127) / 128);
  l.hq = l.xq_sf + round_up(row_tiles * (H / 128) * 512, 1024);
  l.hq_sf = l.hq + round_up(static_cast<size_t>(M) * I, 1024);
  l.part0 = l.hq_sf + round_up(row_tiles * (I / 128) * 512, 1024);
  // split-K accumulators for the smallest tiles (128 rows) either phase may
  // use; above 128 rows every block owns whole tiles and there are none
  l.part1 = l.part0 + (M <= 128 ? accum_bytes(M, 2 * I / 128) : 0);
  l.gu = l.part1 + (M <= 128 ? accum_bytes(M, H / 128) : 0);
  l.total = l.gu + round_up(static_cast<size_t>(M) * 2 * I * 4, 1024);
  return l;
}
// control words of the grid-wide kernel: header | x readiness per block |
// h readiness per block | tile counters phase 0 | tile counters phase 1
size_t ctl_words_needed(int T0, int T1) { return kCtlHeaderWords + 2 * kMaxGrid + T0 + T1; }

bool encode_map(CUtensorMap* m, const void* base, int K, int rows, int box_rows) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kTileK), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Scale tiles (512 bytes each, `tiles` of them) as a 2-D tensor of u32 rows of
// 128 elements, read one tile per TMA box.
bool encode_scale_map(CUtensorMap* m, const void* base, int tiles) {
  cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(tiles)};
  cuuint64_t strides[1] = {512};
  cuuint32_t box[2] = {128, 1};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tile heights and split of one fused MLP launch.
struct MlpPlan {
  int TR0, TR1;  // weight rows per tile: gate/up, down (256 or 128)
  int T0, T1;    // tiles per phase
  int whole0;    // 1: one whole gate/up tile per block, no split-K before the SwiGLU
  int pairs0;    // 1: the two blocks of a cluster split a gate/up tile and add through shared memory
};
// 128 or 256 from the knob, else `dflt`.
int tile_rows_knob(fsops_knob k, int dflt) {
  const int v = knob(k);
  return (v == 128 || v == 256) ? v : dflt;
}
MlpPlan plan_mlp(int M, int H, int I, int grid) {
  MlpPlan pl;
  const int npad = npad_of(M);
  const bool staged = stage_tmem_for(npad) != 0;  // M <= 32
  // gate/up: 256-row tiles.  With M > 32 one whole tile per block when they
  // fit the grid (the SwiGLU then needs no split-K reduction); with M <= 32
  // the tiles are split over all blocks, whose staged reduction is cheap and
  // which each quantise only their half of x.  (128-row whole tiles would
  // need no reduction either, but every block would quantise all of x.)
  pl.TR0 = tile_rows_knob(FSOPS_KNOB_TR0, 256);
  pl.T0 = 2 * I / pl.TR0;
  pl.whole0 = (pl.T0 <= grid && !staged) ? 1 : 0;
  if (knob(FSOPS_KNOB_WHOLE_TILES) >= 0) pl.whole0 = (knob(FSOPS_KNOB_WHOLE_TILES) != 0 && pl.T0 <= grid) ? 1 : 0;
  // M <= 32 with between a quarter and a half as many 256-row gate/up tiles
  // as blocks: each tile goes to one 2-block cluster, whose blocks take a K
  // half each and add their sums through distributed shared memory (no L2
  // reduction before the SwiGLU).  The launch falls back to the split over
  // all blocks when the device cannot hold grid / 2 such clusters at once.
  pl.pairs0 = (staged && !pl.whole0 && pl.TR0 == 256 && grid % 2 == 0 && 4 * pl.T0 > grid && 2 * pl.T0 <= grid &&
               knob_or(FSOPS_KNOB_PAIRS, 1, 0, 1))
                  ? 1
                  : 0;
  // down projection: 256-row tiles.  128-row tiles would halve the split-K
  // sums the blocks add up in L2, but need twice the MMAs for the same
  // weights, and an MMA costs its issuing thread the same whatever its N:
  // with the tile-aligned split 256 rows measured faster at every M (M = 128,
  // H = 5120, I = 17408: 62.2 against 66.7 us; H = 4096, I = 12288: 45.2
  // against 45.7)
  pl.TR1 = tile_rows_knob(FSOPS_KNOB_TR1, 256);
  pl.T1 = (H + pl.TR1 - 1) / pl.TR1;
  return pl;
}
// Output C [M, N] of the tiled GEMM: boxes of 32 rows x 64 bytes (32 bf16 or
// 16 fp32 columns), written from shared memory by TMA stores.
bool encode_out_map(CUtensorMap* m, void* c, int M, int N, bool f32) {
  const cuuint64_t es = f32 ? 4 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(N) * es};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(64 / es), 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c, dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}
// bf16 x [M, H] for the local quantisation: box npad rows x 128 elements.
bool encode_x_map(CUtensorMap* m, const void* x, int H, int M, int npad) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(M)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(H) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kTileK), static_cast<cuuint32_t>(npad)};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

void init_common(KernelArgs& a, int M, uint32_t* ctl) {
  std::memset(&a, 0, sizeof(a));
  a.M = M;
  a.npad = npad_of(M);
  a.nstages = stages_for(a.npad, 0);  // set again once local_xq is known
  a.stage_tmem = stage_tmem_for(a.npad);
  const int inflight = knob_or(FSOPS_KNOB_MAX_INFLIGHT, kDefaultMaxInflight, 1, kMaxStages);
  a.max_inflight = inflight < a.nstages ? inflight : a.nstages;
  a.prime_inflight = knob_or(FSOPS_KNOB_PRIME, kPrimeInflight, 1, kMaxStages);
  a.early_w = knob_or(FSOPS_KNOB_EARLY_W, 1, 0, 1);
  a.stage_bytes = stage_bytes_for(a.npad);
  a.timeout_ns = g_timeout_ns.load();
  a.extra_xready = g_extra.load();
  a.ctl = ctl;
#ifdef FSOPS_TRACE
  a.trace = g_trace;
#endif
}

// Whether grid / 2 two-block clusters of the kernel fit the current device at
// this shared-memory size (queried once per device and size).
bool pairs_fit(int grid, size_t smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  static std::mutex mu;
  static std::map<std::tuple<int, int, size_t>, bool> cache;
  std::lock_guard<std::mutex> lk(mu);
  const auto key = std::make_tuple(dev, grid, smem);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  const bool fit = cluster_pairs_fit(grid, smem);
  cache[key] = fit;
  return fit;
}

// grid_fits, queried once per device, grid and shared-memory size.
bool grid_fits_cached(int grid, size_t smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  static std::mutex mu;
  static std::map<std::tuple<int, int, size_t>, bool> cache;
  std::lock_guard<std::mutex> lk(mu);
  const auto key = std::make_tuple(dev, grid, smem);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  const bool fit = grid_fits(grid, smem);
  cache[key] = fit;
  return fit;
}

// Stream-K (an even split of the T x KS units, so a block may hold the end of
// one tile and the start of the next) or the tile-aligned split (each block
// on one tile; with T <= grid and at least one stage per block).  A block
// holding two tiles runs two accumulator rounds, two readiness waits and two
// split-K reductions, and the tiles it holds finish only after both.  The
// aligned split is taken wherever it applies, although its largest share can
// be a few stages above stream-K's: it measured faster at every decode shape
// (H = 4096, I = 12288, M = 64: 43.4 against 46.9 us; H = 5120, I = 17408,
// M = 32: 60.8 against 66.4 us; equal at M = 128).
void choose_split(PhaseArgs& ph, int grid) {
  ph.aligned = 0;
  if (ph.whole_tiles || ph.pairs || ph.T > grid) return;
  if (ph.KS < (grid + ph.T - 1) / ph.T) return;
  ph.aligned = knob(FSOPS_KNOB_ALIGNED) == 0 ? 0 : 1;
}

fsops_status launch(KernelArgs& a, int grid, cudaStream_t stream) {
  if (grid > kMaxGrid) return FSOPS_ERR_UNSUPPORTED_SHAPE;  // one readiness counter per block
  a.nstages = stages_for(a.npad, a.local_xq);
  if (a.max_inflight > a.nstages) a.max_inflight = a.nstages;
  bool pairs = false;
  for (int p = 0; p < a.nphases; ++p) pairs = pairs || a.ph[p].pairs;
  if (pairs && !pairs_fit(grid, smem_for(a.npad, a.local_xq))) {
    for (int p = 0; p < a.nphases; ++p) a.ph[p].pairs = 0;  // split over all blocks instead
    pairs = false;
  }
  a.cluster_pairs = pairs ? 1 : 0;
  for (int p = 0; p < a.nphases; ++p) choose_split(a.ph[p], grid);
  const size_t smem = smem_for(a.npad, a.local_xq);
  // a plain launch with programmatic dependent launch by default (see
  // launch_mx_kernel); cooperative when forced or when the grid might not be
  // resident at once
  const bool coop = knob(FSOPS_KNOB_COOPERATIVE) == 1 || !grid_fits_cached(grid, smem);
  const cudaError_t e = launch_mx_kernel(a, grid, smem, stream, coop);
  return e == cudaSuccess ? FSOPS_OK : cuda_failed(e, "mx_persistent_kernel launch");
}

// Device buffers of one fused MLP launch (workspace or fixed buffer).
struct MlpBuffers {
  uint8_t *ctl, *xq, *xq_sf, *hq, *hq_sf, *part0, *part1;
};
// Fills the two phases of the fused MLP: phase 0 gate/up (W_gateup rows in
// tiles of pl.TR0, SwiGLU epilogue), phase 1 down (W_down in tiles of pl.TR1).
// x_bf16 == nullptr: x is already quantised into b.xq / b.xq_sf (the
// decoder block's RMSNorm launch); residual (bf16 [M, H]) is added to y.
fsops_status fill_mlp_args(KernelArgs& ka, const MlpPlan& pl, const MlpBuffers& b, const void* x_bf16,
                           const uint8_t* w_gateup, const uint8_t* w_down, const fsops_mlp_scales* scales,
                           void* y_bf16, int M, int H, int I, const void* residual = nullptr,
                           const void* gamma = nullptr, float eps = 0.f) {
  init_common(ka, M, reinterpret_cast<uint32_t*>(b.ctl));
  if (ctl_words_needed(pl.T0, pl.T1) * 4 > kCtlRegionBytes) return FSOPS_ERR_UNSUPPORTED_SHAPE;
  ka.xready = ka.ctl + kCtlHeaderWords;
  ka.hflags = ka.xready + kMaxGrid;
  ka.nphases = 2;
  ka.x = static_cast<const uint16_t*>(x_bf16);
  ka.xq_codes = b.xq;
  ka.xq_sf = b.xq_sf;
  ka.H = H;
  ka.hq_codes = b.hq;
  ka.hq_sf = b.hq_sf;
  ka.I = I;
  ka.out = y_bf16;
  ka.out_f32 = 0;
  ka.residual = static_cast<const uint16_t*>(residual);
  PhaseArgs& p0 = ka.ph[0];
  p0.sf_w = scales->gateup;
  p0.sf_act = ka.xq_sf;
  p0.tile_cnt = ka.hflags + kMaxGrid;
  p0.accum = reinterpret_cast<float*>(b.part0);
  p0.KS = H / kTileK;
  p0.T = pl.T0;
  p0.tile_rows = pl.TR0;
  p0.rows = 2 * I;
  p0.whole_tiles = pl.whole0;
  p0.pairs = pl.pairs0;
  ka.gamma = static_cast<const uint16_t*>(gamma);
  ka.eps = eps;
  // y may be x itself: every read of x (the norm's and the quantisation's)
  // comes before its block's gate/up MMAs, and no tile of y is finished before
  // every gate/up tile is (each down-projection tile reads every chunk of h).
  // With RMSNorm every block quantising locally first reads all M rows of x
  // for their norms, all blocks the same rows at once: that pays only for
  // short rows (M = 1, H = 1024: 16.0 against 17.4 us for the block; M = 16,
  // H = 2560: 27.6 against 26.0 with x quantised grid-wide, each block a
  // slice; LOCAL_XQ = 2 forces it)
  const bool norm_local = gamma == nullptr || static_cast<long long>(M) * H <= 16384 ||
                          knob(FSOPS_KNOB_LOCAL_XQ) == 2;
  ka.local_xq = (x_bf16 != nullptr && norm_local) ? local_xq_for(ka.npad) : 0;
  p0.dep = (ka.local_xq || x_bf16 == nullptr) ? kDepNone : kDepXReady;
  if (ka.local_xq && !encode_x_map(&ka.tm_x, x_bf16, H, M, ka.npad)) return FSOPS_ERR_INVALID_ARG;
  p0.epi = kEpiSwiGLU;
  p0.out_ld = I;
  PhaseArgs& p1 = ka.ph[1];
  p1.sf_w = scales->down;
  p1.sf_act = ka.hq_sf;
  p1.tile_cnt = p0.tile_cnt + pl.T0;
  p1.accum = reinterpret_cast<float*>(b.part1);
  p1.KS = I / kTileK;
  p1.T = pl.T1;
  p1.tile_rows = pl.TR1;
  p1.rows = H;
  p1.dep = kDepHFlags;
  p1.epi = kEpiStore;
  p1.out_ld = H;
  if (!encode_map(&ka.tm_w[0], w_gateup, H, 2 * I, pl.TR0) ||
      !encode_map(&ka.tm_act[0], ka.xq_codes, H, M, ka.npad) || !encode_map(&ka.tm_w[1], w_down, I, H, pl.TR1) ||
      !encode_map(&ka.tm_act[1], ka.hq_codes, I, M, ka.npad))
    return FSOPS_ERR_INVALID_ARG;
  return FSOPS_OK;
}

// The cluster-sliced decode kernel (mx_slice.cu) for up to 32 tokens: NP
// 2-block clusters, each owning NC / NP (at most kSliceMaxChunks) 128-feature
// chunks of I; RT = H / 128 row tiles in the down projection.
struct SlicePlan {
  int NC, NP, RT, npad;
};
bool slice_plan(int M, int H, int I, int sms, SlicePlan* sp) {
  if (M < 1 || M > kSliceMaxM || H < 256 || sms < kSliceCluster) return false;
  const int NC = I / 128;
  const int NP = sms / kSliceCluster < NC ? sms / kSliceCluster : NC;
  if ((NC + NP - 1) / NP > kSliceMaxChunks) return false;
  const int RT = H / 128;
  if ((RT + 1) / 2 > 256 || (kCtlHeaderWords + RT) * 4 > static_cast<int>(kCtlRegionBytes)) return false;
  sp->NC = NC;
  sp->NP = NP;
  sp->RT = RT;
  sp->npad = M <= 16 ? 16 : 32;
  return true;
}
// fp32 [M, H] partial sums of the sliced kernel.
size_t slice_accum_bytes(int M, int H) { return round_up(static_cast<size_t>(M) * H * 4, 1024); }
// 128-token chunks per paged-attention block (knob ATTN_CHUNKS, else the
// library's choice).
int attn_chunks_per_block() { return knob_or(FSOPS_KNOB_ATTN_CHUNKS, kAttnChunksPerBlock, 1, 64); }

// Whether the fused MLP call runs the sliced kernel: only when forced
// (FSOPS_KNOB_DECODE_PATH = 1).  The grid-wide kernel measured faster at
// every decode shape, including the small-I one the sliced kernel was built
// for (M = 1, H = 1024, I = 2816: 14.0 against 14.6 us per call; M = 16,
// H = 2560, I = 9728: 23.6 against 33.9 us), where every cluster adds a full
// [M, H] fp32 partial of y into L2 (12.5 MB of L2 reductions at M = 16).
bool use_slice(int M, int H, int I, const DeviceInfo* di, SlicePlan* sp) {
  if (knob(FSOPS_KNOB_DECODE_PATH) != 1) return false;
  return slice_plan(M, H, I, di->sms, sp);
}
// Whether the fused MLP call runs the small-M kernel (mx_small.cu): by
// default wherever it applies (M <= 8, one block per 32 intermediate
// features and per 16 output rows, each block's weights in shared memory),
// or only when FSOPS_KNOB_DECODE_PATH = 2; never with 0 or 1.
bool use_small(int M, int H, int I, const DeviceInfo* di) {
  const int k = knob(FSOPS_KNOB_DECODE_PATH);
  if (k == 0 || k == 1) return false;
  return small_fits(M, H, I, di->sms);
}
// One launch of the small-M kernel on the workspace's control words and h
// buffers.  gamma != null: RMSNorm(x) * gamma is quantised; residual != null
// is added to y before the bf16 rounding.
fsops_status launch_small(const MlpLayout& l, uint8_t* ws, const void* x_bf16, const void* gamma, float eps,
                          const void* residual, const uint8_t* w_gateup, const uint8_t* w_down,
                          const fsops_mlp_scales* scales, void* y_bf16, int M, int H, int I, const DeviceInfo* di,
                          cudaStream_t stream) {
  SmallArgs sa;
  std::memset(&sa, 0, sizeof(sa));
  if (!encode_map(&sa.tm_wgu, w_gateup, H, 2 * I, 32) || !encode_map(&sa.tm_wd, w_down, I, H, 16))
    return FSOPS_ERR_INVALID_ARG;
  sa.sf_gu = scales->gateup;
  sa.sf_d = scales->down;
  sa.x = static_cast<const uint16_t*>(x_bf16);
  sa.gamma = static_cast<const uint16_t*>(gamma);
  sa.eps = eps;
  sa.residual = static_cast<const uint16_t*>(residual);
  sa.y = static_cast<uint16_t*>(y_bf16);
  sa.hq = ws + l.hq;
  sa.hs = ws + l.hq_sf;
  sa.ctl = reinterpret_cast<uint32_t*>(ws + l.ctl);
  sa.M = M;
  sa.H = H;
  sa.I = I;
  sa.U = I / 32;
  sa.T = H / 16;
  sa.split = small_split(H, I, di->sms);
  sa.timeout_ns = g_timeout_ns.load();
  sa.extra_arrivals = g_extra.load();
#ifdef FSOPS_TRACE
  sa.trace = g_trace;
#endif
  const int grid = sa.split ? sa.U + sa.T : (sa.U > sa.T ? sa.U : sa.T);
  const cudaError_t e = launch_small_kernel(sa, grid, stream);
  return e == cudaSuccess ? FSOPS_OK : cuda_failed(e, "mx_small_kernel launch");
}
// One launch of the sliced kernel.  ctl: the control words (status word,
// then RT tile counters), accum: fp32 [M, H], both zero between launches.  gamma != null: x is normalised (RMSNorm with eps) before its
// quantisation; residual != null is added to y before the bf16 rounding.
fsops_status launch_slice(const SlicePlan& sp, uint8_t* ctl, uint8_t* accum, const void* x_bf16, const void* gamma,
                          float eps, const void* residual, const uint8_t* w_gateup, const uint8_t* w_down,
                          const fsops_mlp_scales* scales, void* y_bf16, int M, int H, int I, cudaStream_t stream) {
  SliceArgs sa;
  std::memset(&sa, 0, sizeof(sa));
  if (!encode_map(&sa.tm_wgu, w_gateup, H, 2 * I, 128) || !encode_map(&sa.tm_wd, w_down, I, H, 128) ||
      !encode_x_map(&sa.tm_x, x_bf16, H, M, sp.npad))
    return FSOPS_ERR_INVALID_ARG;
  sa.sf_gu = scales->gateup;
  sa.sf_d = scales->down;
  sa.x = static_cast<const uint16_t*>(x_bf16);
  sa.gamma = static_cast<const uint16_t*>(gamma);
  sa.eps = eps;
  sa.y = static_cast<uint16_t*>(y_bf16);
  sa.residual = static_cast<const uint16_t*>(residual);
  sa.accum = reinterpret_cast<float*>(accum);
  uint32_t* cw = reinterpret_cast<uint32_t*>(ctl);
  sa.status = cw + kCtlStatus;
  sa.tile_cnt = cw + kCtlHeaderWords;
  sa.M = M;
  sa.H = H;
  sa.I = I;
  sa.NC = sp.NC;
  sa.NP = sp.NP;
  sa.KS0 = H / kTileK;
  sa.RT = sp.RT;
  sa.nstages = slice_stages(sp.npad);
  sa.timeout_ns = g_timeout_ns.load();
  sa.extra_arrivals = g_extra.load();
#ifdef FSOPS_TRACE
  sa.trace = g_trace;
#endif
  const cudaError_t e = launch_slice_kernel(sa, sp.npad, stream);
  return e == cudaSuccess ? FSOPS_OK : cuda_failed(e, "mx_slice_kernel launch");
}

// Up to 128 rows: the decode kernel (stream-K split over all SMs); more rows
// (prefill): whole 128 x 256 output tiles per block.
constexpr int kMaxGemmRows = 16384;
bool gemm_shape_ok(int M, int N, int K) {
  return M >= 1 && M <= kMaxGemmRows && N >= 128 && K >= 128 && N % 128 == 0 && K % 128 == 0 && N <= 65536 &&
         K <= 65536;
}

// The operand half of the tiled GEMM's arguments: A codes and scales
// (pre-quantised), B codes and scales, the shape and the status word.
fsops_status fill_tiled(TiledArgs& ta, const uint8_t* codes, const uint8_t* sfa, const uint8_t* b_codes,
                        const uint8_t* b_scales, int M, int N, int K, uint8_t* ctl, const DeviceInfo* di) {
  std::memset(&ta, 0, sizeof(ta));
  // One block per 128 x 256 tile by default.  FSOPS_KNOB_GEMM_FORM = 1 runs
  // 2-block clusters on vertically adjacent row tiles as one 256-row
  // cta_group::2 MMA (N % 256 == 0, two or more row tiles).
  const int MT = (M + 127) / 128;
  ta.form = knob_or(FSOPS_KNOB_GEMM_FORM, kTiledSingle, kTiledSingle, kTiledPairMma);
  if (MT < 2 || di->sms < 2 || N % 256 != 0) ta.form = kTiledSingle;
  if (!encode_map(&ta.tm_a, codes, K, M, 128) ||
      !encode_map(&ta.tm_b, b_codes, K, N, ta.form == kTiledSingle ? 256 : 128))
    return FSOPS_ERR_INVALID_ARG;
  const int KS = K / kTileK;
  if (ta.form == kTiledPairMma &&
      (!encode_scale_map(&ta.tm_sfa, sfa, MT * KS) || !encode_scale_map(&ta.tm_sfb, b_scales, (N / 128) * KS)))
    return FSOPS_ERR_INVALID_ARG;
  ta.sf_a = sfa;
  ta.sf_b = b_scales;
  ta.M = M;
  ta.N = N;
  ta.K = K;
  ta.KS = K / kTileK;
  ta.MT = MT;
  ta.NT = (N + 255) / 256;
  ta.status = reinterpret_cast<uint32_t*>(ctl) + kCtlStatus;
  ta.timeout_ns = g_timeout_ns.load();
  return FSOPS_OK;
}

fsops_status quantize_a(const void* a, int M, int K, uint8_t* xq, uint8_t* xq_sf, cudaStream_t stream) {
  const cudaError_t e = launch_quantize(static_cast<const uint16_t*>(a), M, K, K, xq, xq_sf, 1, stream);
  return e == cudaSuccess ? FSOPS_OK : cuda_failed(e, "quantize_kernel launch");
}

fsops_status run_tiled(const TiledArgs& ta, const DeviceInfo* di, cudaStream_t stream) {
  const cudaError_t e = launch_gemm_tiled(ta, di->sms, stream);
  return e == cudaSuccess ? FSOPS_OK : cuda_failed(e, "mx_gemm_tiled_kernel launch");
}

// M > 128: A quantised by its own launch when it is bf16, then the tiled GEMM.
fsops_status gemm_tiled_impl(const void* a, const uint8_t* a_scales, bool a_bf16, const uint8_t* b_codes,
                             const uint8_t* b_scales, void* c, bool c_f32, int M, int N, int K, uint8_t* ctl,
                             uint8_t* xq, uint8_t* xq_sf, const DeviceInfo* di, cudaStream_t stream) {
  const uint8_t* codes = a_bf16 ? xq : static_cast<const uint8_t*>(a);
  const uint8_t* sfa = a_bf16 ? xq_sf : a_scales;
  TiledArgs ta;
  fsops_status st = fill_tiled(ta, codes, sfa, b_codes, b_scales, M, N, K, ctl, di);
  if (st != FSOPS_OK) return st;
  if (!encode_out_map(&ta.tm_c, c, M, N, c_f32)) return FSOPS_ERR_INVALID_ARG;
  ta.c = c;
  ta.c_f32 = c_f32 ? 1 : 0;
  if (a_bf16 && (st = quantize_a(a, M, K, xq, xq_sf, stream)) != FSOPS_OK) return st;
  return run_tiled(ta, di, stream);
}

// The MLP above 128 token rows, in three launches: x quantised to MXFP8; the
// gate/up GEMM with the SwiGLU epilogue, which writes h requantised to MXFP8;
// the down GEMM on h.
// x_bf16 == nullptr: x is already quantised in the workspace; residual is
// added to y by the down GEMM's epilogue.
fsops_status mlp_tiled_impl(const void* x_bf16, const uint8_t* w_gateup, const uint8_t* w_down,
                            const fsops_mlp_scales* scales, void* y_bf16, int M, int H, int I, uint8_t* ws,
                            const MlpLayout& l, const DeviceInfo* di, cudaStream_t stream,
                            const void* residual = nullptr) {
  TiledArgs gu;
  fsops_status st = fill_tiled(gu, ws + l.xq, ws + l.xq_sf, w_gateup, scales->gateup, M, 2 * I, H, ws + l.ctl, di);
  if (st != FSOPS_OK) return st;
  gu.swiglu = 1;
  gu.h_codes = ws + l.hq;
  gu.h_sf = ws + l.hq_sf;
  TiledArgs dn;
  st = fill_tiled(dn, ws + l.hq, ws + l.hq_sf, w_down, scales->down, M, H, I, ws + l.ctl, di);
  if (st != FSOPS_OK) return st;
  if (!encode_out_map(&dn.tm_c, y_bf16, M, H, false)) return FSOPS_ERR_INVALID_ARG;
  dn.c = y_bf16;
  dn.residual = static_cast<const uint16_t*>(residual);
  if (x_bf16 != nullptr && (st = quantize_a(x_bf16, M, H, ws + l.xq, ws + l.xq_sf, stream)) != FSOPS_OK) return st;
  if ((st = run_tiled(gu, di, stream)) != FSOPS_OK) return st;
  return run_tiled(dn, di, stream);
}

// Plain GEMM (one phase) with the operand pointers already validated.
// `ctl` is the control region, `xq`/`xq_sf` receive the quantised A (bf16 A
// only), `part` holds the split-K partial sums.
fsops_status gemm_impl(const void* a, const uint8_t* a_scales, bool a_bf16, const uint8_t* b_codes,
                       const uint8_t* b_scales, void* c, bool c_f32, int M, int N, int K, uint8_t* ctl,
                       uint8_t* xq, uint8_t* xq_sf, uint8_t* part, const DeviceInfo* di, cudaStream_t stream) {
  if (M > 128) return gemm_tiled_impl(a, a_scales, a_bf16, b_codes, b_scales, c, c_f32, M, N, K, ctl, xq, xq_sf, di, stream);
  const int grid = di->sms;
  KernelArgs ka;
  init_common(ka, M, reinterpret_cast<uint32_t*>(ctl));
  ka.nphases = 1;
  PhaseArgs& p = ka.ph[0];
  p.sf_w = b_scales;
  p.KS = K / kTileK;
  p.T = (N + kTileRows - 1) / kTileRows;
  p.tile_rows = kTileRows;
  p.rows = N;
  p.epi = kEpiStore;
  p.out_ld = N;
  if (kCtlHeaderWords + kMaxGrid + p.T > static_cast<int>(kCtlRegionBytes / 4)) return FSOPS_ERR_UNSUPPORTED_SHAPE;
  ka.xready = ka.ctl + kCtlHeaderWords;
  p.tile_cnt = ka.xready + kMaxGrid;
  p.accum = reinterpret_cast<float*>(part);
  const uint8_t* act_codes;
  if (a_bf16) {
    ka.x = static_cast<const uint16_t*>(a);
    ka.xq_codes = xq;
    ka.xq_sf = xq_sf;
    ka.H = K;
    act_codes = ka.xq_codes;
    p.sf_act = ka.xq_sf;
    ka.local_xq = local_xq_for(ka.npad);
    p.dep = ka.local_xq ? kDepNone : kDepXReady;
    if (ka.local_xq && !encode_x_map(&ka.tm_x, a, K, M, ka.npad)) return FSOPS_ERR_INVALID_ARG;
  } else {
    act_codes = static_cast<const uint8_t*>(a);
    p.sf_act = a_scales;
    p.dep = kDepNone;
  }
  ka.out = c;
  ka.out_f32 = c_f32 ? 1 : 0;
  if (!encode_map(&ka.tm_w[0], b_codes, K, N, kTileRows) || !encode_map(&ka.tm_act[0], act_codes, K, M, ka.npad))
    return FSOPS_ERR_INVALID_ARG;
  return launch(ka, grid, stream);
}

fsops_status check_ws(int dev, size_t need, uint8_t** ws) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_ws[dev].ptr == nullptr || g_ws[dev].bytes < need) return FSOPS_ERR_INVALID_ARG;
  *ws = static_cast<uint8_t*>(g_ws[dev].ptr);
  return FSOPS_OK;
}

fsops_status mlp_validate(const void* x, const uint8_t* wgu, const uint8_t* wd, const fsops_mlp_scales* sc,
                          const void* y, int M, int H, int I) {
  if (x == nullptr || wgu == nullptr || wd == nullptr || sc == nullptr || sc->gateup == nullptr ||
      sc->down == nullptr || y == nullptr)
    return FSOPS_ERR_INVALID_ARG;
  if (M < 1 || M > kMaxGemmRows || H < 128 || I < 128 || H % 128 != 0 || I % 128 != 0 || H > 65536 ||
      I > 65536)
    return FSOPS_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(wgu) || !aligned16(wd) || !aligned16(sc->gateup) || !aligned16(sc->down) ||
      !aligned16(y))
    return FSOPS_ERR_MISALIGNED;
  return FSOPS_OK;
}

}  // namespace

extern "C" {

int fsops_version(void) { return 100; }

int fsops_last_cuda_error(void) { return g_last_cuda_error; }

const char* fsops_status_string(fsops_status s) {
  switch (s) {
    case FSOPS_OK: return "ok";
    case FSOPS_ERR_INVALID_ARG: return "invalid argument";
    case FSOPS_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case FSOPS_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case FSOPS_ERR_CUDA: return "CUDA error";
    case FSOPS_ERR_TIMEOUT: return "kernel wait timed out";
    case FSOPS_ERR_NO_DEVICE: return "no sm_100-class device current";
  }
  return "unknown status";
}

size_t fsops_scale_bytes(int rows, int K, fsops_scale_layout layout) {
  if (rows < 0 || K < 0) return 0;
  if (layout == FSOPS_SCALES_ROWMAJOR) return static_cast<size_t>(rows) * (K / 32);
  if (layout == FSOPS_SCALES_TCGEN05)
    return static_cast<size_t>((rows + 127) / 128) * static_cast<size_t>((K + 127) / 128) * 512;
  return 0;
}

fsops_status fsops_quantize_mxfp8(const void* x_bf16, int rows, int K, int ld, uint8_t* codes, uint8_t* scales,
                                  fsops_scale_layout layout, void* stream) {
  if (layout != FSOPS_SCALES_ROWMAJOR && layout != FSOPS_SCALES_TCGEN05) return FSOPS_ERR_INVALID_ARG;
  if (rows < 0 || K <= 0 || ld < K) return FSOPS_ERR_UNSUPPORTED_SHAPE;
  if (K % (layout == FSOPS_SCALES_TCGEN05 ? 128 : 32) != 0 || ld % 8 != 0) return FSOPS_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<long long>(rows) * ld >= (1LL << 31)) return FSOPS_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0) return FSOPS_OK;
  if (x_bf16 == nullptr || codes == nullptr || scales == nullptr) return FSOPS_ERR_INVALID_ARG;
  if (!aligned16(x_bf16) || !aligned16(codes)) return FSOPS_ERR_MISALIGNED;
  int dev;
  const DeviceInfo* di;
  fsops_status st = current_device(&dev, &di);
  if (st != FSOPS_OK) return st;
  cudaError_t e = launch_quantize(static_cast<const uint16_t*>(x_bf16), rows, K, ld, codes, scales,
                                  layout == FSOPS_SCALES_TCGEN05 ? 1 : 0, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FSOPS_OK : cuda_failed(e, "quantize_kernel launch");
}

fsops_status fsops_quantize_mxfp8_gateup(const void* w_gate_bf16, const void* w_up_bf16, int I, int H, int ld,
                                         uint8_t* codes, uint8_t* scales, void* stream) {
  if (I < 64 || I % 64 != 0 || H < 128 || H % 128 != 0 || ld < H || ld % 8 != 0) return FSOPS_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<long long>(I) * ld >= (1LL << 31) || static_cast<long long>(2 * I) * H >= (1LL << 31))
    return FSOPS_ERR_UNSUPPORTED_SHAPE;
  if (w_gate_bf16 == nullptr || w_up_bf16 == nullptr || codes == nullptr || scales == nullptr)
    return FSOPS_ERR_INVALID_ARG;
  if (!aligned16(w_gate_bf16) || !aligned16(w_up_bf16) || !aligned16(codes)) return FSOPS_ERR_MISALIGNED;
  int dev;
  const DeviceInfo* di;
  fsops_status st = current_device(&dev, &di);
  if (st != FSOPS_OK) return st;
  const cudaError_t e = launch_quantize(static_cast<const uint16_t*>(w_gate_bf16), 2 * I, H, ld, codes, scales, 1,
                                        static_cast<cudaStream_t>(stream), static_cast<const uint16_t*>(w_up_bf16));
  return e == cudaSuccess ? FSOPS_OK : cuda_failed(e, "quantize_kernel launch");
}

size_t fsops_gemm_workspace_bytes(int M, int N, int K) {
  if (!gemm_shape_ok(M, N, K)) return 0;
  int dev;
  const DeviceInfo* di;
  if (current_device(&dev, &di) != FSOPS_OK) return 0;
  return gemm_layout(M, N, K).total;
}

fsops_status fsops_mxfp8_gemm_ex(const void* a, const uint8_t* a_scales, fsops_dtype a_dtype,
                                 const uint8_t* b_codes, const uint8_t* b_scales, void* c, fsops_dtype c_dtype,
                                 int M, int N, int K, void* workspace, size_t ws_bytes, void* stream) {
  if (a == nullptr || b_codes == nullptr || b_scales == nullptr || c == nullptr || workspace == nullptr)
    return FSOPS_ERR_INVALID_ARG;
  if (a_dtype != FSOPS_DTYPE_BF16 && a_dtype != FSOPS_DTYPE_MXFP8) return FSOPS_ERR_INVALID_ARG;
  if (c_dtype != FSOPS_DTYPE_BF16 && c_dtype != FSOPS_DTYPE_F32) return FSOPS_ERR_INVALID_ARG;
  if ((a_dtype == FSOPS_DTYPE_BF16) != (a_scales == nullptr)) return FSOPS_ERR_INVALID_ARG;
  if (!gemm_shape_ok(M, N, K)) return FSOPS_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(a) || !aligned16(b_codes) || !aligned16(b_scales) || !aligned16(c) || !aligned16(workspace) ||
      (a_scales != nullptr && !aligned16(a_scales)))
    return FSOPS_ERR_MISALIGNED;
  int dev;
  const DeviceInfo* di;
  fsops_status st = current_device(&dev, &di);
  if (st != FSOPS_OK) return st;
  const GemmLayout l = gemm_layout(M, N, K);
  if (ws_bytes < l.total) return FSOPS_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  return gemm_impl(a, a_scales, a_dtype == FSOPS_DTYPE_BF16, b_codes, b_scales, c, c_dtype == FSOPS_DTYPE_F32, M,
                   N, K, ws + l.ctl, ws + l.xq, ws + l.xq_sf, ws + l.part, di, static_cast<cudaStream_t>(stream));
}

fsops_status fsops_mxfp8_gemm(const void* a_bf16, const uint8_t* b_codes, const uint8_t* b_scales, void* c_bf16,
                              int M, int N, int K, void* workspace, size_t ws_bytes, void* stream) {
  return fsops_mxfp8_gemm_ex(a_bf16, nullptr, FSOPS_DTYPE_BF16, b_codes, b_scales, c_bf16, FSOPS_DTYPE_BF16, M, N,
                             K, workspace, ws_bytes, stream);
}

fsops_status fsops_swiglu_quantize_mxfp8(const float* gu, int M, int I, uint8_t* h_codes, uint8_t* h_scales,
                                         void* stream) {
  if (gu == nullptr || h_codes == nullptr || h_scales == nullptr) return FSOPS_ERR_INVALID_ARG;
  if (M < 1 || M > kMaxGemmRows || I < 128 || I % 128 != 0 || I > 65536) return FSOPS_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(gu) || !aligned16(h_codes)) return FSOPS_ERR_MISALIGNED;
  int dev;
  const DeviceInfo* di;
  fsops_status st = current_device(&dev, &di);
  if (st != FSOPS_OK) return st;
  cudaError_t e = launch_swiglu_quantize(gu, M, I, h_codes, h_scales, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FSOPS_OK : cuda_failed(e, "swiglu_quantize_kernel launch");
}

size_t fsops_mlp_workspace_bytes(int M, int H, int I) {
  if (M < 1 || M > kMaxGemmRows || H < 128 || I < 128 || H % 128 != 0 || I % 128 != 0 || H > 65536 ||
      I > 65536)
    return 0;
  int dev;
  const DeviceInfo* di;
  if (current_device(&dev, &di) != FSOPS_OK) return 0;
  return mlp_layout(M, H, I).total;
}

fsops_status fsops_set_workspace(void* ws, size_t bytes) {
  int dev;
  const DeviceInfo* di;
  fsops_status st = current_device(&dev, &di);
  if (st != FSOPS_OK) return st;
  if (ws != nullptr && ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)) return FSOPS_ERR_MISALIGNED;
  if (ws != nullptr && bytes < kCtlRegionBytes) return FSOPS_ERR_INVALID_ARG;
  if (ws != nullptr) {
    cudaError_t e = cudaMemset(ws, 0, bytes);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_failed(e, "workspace clear");
  }
  std::lock_guard<std::mutex> lk(g_mu);
  g_ws[dev].ptr = ws;
  g_ws[dev].bytes = ws != nullptr ? bytes : 0;
  return FSOPS_OK;
}

fsops_status fsops_mxfp8_swiglu_mlp(const void* x_bf16, const uint8_t* w_gateup, const uint8_t* w_down,
                                    const fsops_mlp_scales* scales, void* y_bf16, int M, int H, int I,
                                    void* stream) {
  fsops_status st = mlp_validate(x_bf16, w_gateup, w_down, scales, y_bf16, M, H, I);
  if (st != FSOPS_OK) return st;
  int dev;
  const DeviceInfo* di;
  st = current_device(&dev, &di);
  if (st != FSOPS_OK) return st;
  const int grid = di->sms;
  const MlpLayout l = mlp_layout(M, H, I);
  uint8_t* ws;
  st = check_ws(dev, l.total, &ws);
  if (st != FSOPS_OK) return st;
  if (M > 128)
    return mlp_tiled_impl(x_bf16, w_gateup, w_down, scales, y_bf16, M, H, I, ws, l, di,
                          static_cast<cudaStream_t>(stream));
  SlicePlan sp;
  if (use_slice(M, H, I, di, &sp))
    return launch_slice(sp, ws + l.ctl, ws + l.part1, x_bf16, nullptr, 0.f, nullptr, w_gateup, w_down, scales,
                        y_bf16, M, H, I, static_cast<cudaStream_t>(stream));
  if (use_small(M, H, I, di))
    return launch_small(l, ws, x_bf16, nullptr, 0.f, nullptr, w_gateup, w_down, scales, y_bf16, M, H, I, di,
                        static_cast<cudaStream_t>(stream));

  const MlpPlan pl = plan_mlp(M, H, I, grid);
  const MlpBuffers bufs{ws + l.ctl, ws + l.xq, ws + l.xq_sf, ws + l.hq, ws + l.hq_sf, ws + l.part0, ws + l.part1};
  KernelArgs ka;
  st = fill_mlp_args(ka, pl, bufs, x_bf16, w_gateup, w_down, scales, y_bf16, M, H, I);
  if (st != FSOPS_OK) return st;
  return launch(ka, grid, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {
constexpr size_t kAttnStatusBytes = 256;
// Shape check of the paged decode attention; FSOPS_OK when supported.
fsops_status attn_shape(int B, int Hq, int Hkv, int D, int P, int num_pages, int max_pages) {
  if (B < 1 || B > 65535 || Hkv < 1 || Hkv > 65535 || Hq < Hkv || Hq % Hkv != 0 || Hq > 65535)
    return FSOPS_ERR_UNSUPPORTED_SHAPE;
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return FSOPS_ERR_UNSUPPORTED_SHAPE;
  if (D != kAttnHeadDim || (P != 16 && P != 32 && P != 64 && P != 128)) return FSOPS_ERR_UNSUPPORTED_SHAPE;
  if (num_pages < 1 || max_pages < 1 || static_cast<long long>(max_pages) * P > (1LL << 24))
    return FSOPS_ERR_UNSUPPORTED_SHAPE;
  // the cache's token rows are TMA coordinates (int32)
  if (static_cast<long long>(num_pages) * Hkv * P >= (1LL << 31)) return FSOPS_ERR_UNSUPPORTED_SHAPE;
  return FSOPS_OK;
}
}  // namespace

extern "C" {

size_t fsops_paged_attention_workspace_bytes(int B, int Hq, int Hkv, int D, int page_size, int max_pages) {
  if (attn_shape(B, Hq, Hkv, D, page_size, 1, max_pages) != FSOPS_OK) return 0;
  int dev;
  const DeviceInfo* di;
  if (current_device(&dev, &di) != FSOPS_OK) return 0;
  const int ns = attn_splits(B, Hkv, max_pages, page_size, di->sms, attn_chunks_per_block());
  return kAttnStatusBytes + round_up(attn_part_floats(B, Hq, ns) * sizeof(float), 256);
}

fsops_status fsops_mxfp8_paged_decode_attention(const void* q_bf16, const uint8_t* k_codes, const uint8_t* k_scales,
                                                const uint8_t* v_codes, const uint8_t* v_scales, int num_pages,
                                                const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                                                void* out_bf16, int B, int Hq, int Hkv, int D, int page_size,
                                                float sm_scale, void* workspace, size_t ws_bytes, void* stream) {
  fsops_status st = attn_shape(B, Hq, Hkv, D, page_size, num_pages, max_pages);
  if (st != FSOPS_OK) return st;
  if (q_bf16 == nullptr || k_codes == nullptr || k_scales == nullptr || v_codes == nullptr || v_scales == nullptr ||
      block_table == nullptr || seq_lens == nullptr || out_bf16 == nullptr || workspace == nullptr)
    return FSOPS_ERR_INVALID_ARG;
  if (!(sm_scale == sm_scale) || sm_scale > 1e30f || sm_scale < -1e30f) return FSOPS_ERR_INVALID_ARG;
  if (!aligned16(q_bf16) || !aligned16(k_codes) || !aligned16(k_scales) || !aligned16(v_codes) ||
      !aligned16(v_scales) || !aligned16(out_bf16) || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) != 0 || (reinterpret_cast<uintptr_t>(seq_lens) & 3u) != 0)
    return FSOPS_ERR_MISALIGNED;
  int dev;
  const DeviceInfo* di;
  st = current_device(&dev, &di);
  if (st != FSOPS_OK) return st;
  AttnArgs aa;
  std::memset(&aa, 0, sizeof(aa));
  aa.nsplit = attn_splits(B, Hkv, max_pages, page_size, di->sms, attn_chunks_per_block());
  aa.grid = attn_grid(aa.nsplit * B * Hkv, di->sms);
  if (ws_bytes < kAttnStatusBytes + attn_part_floats(B, Hq, aa.nsplit) * sizeof(float)) return FSOPS_ERR_INVALID_ARG;
  aa.q = static_cast<const uint16_t*>(q_bf16);
  const int cache_rows = num_pages * Hkv * page_size;
  if (!encode_map(&aa.tm_k, k_codes, D, cache_rows, page_size) ||
      !encode_map(&aa.tm_v, v_codes, D, cache_rows, page_size))
    return FSOPS_ERR_INVALID_ARG;
  aa.k_scales = k_scales;
  aa.v_scales = v_scales;
  aa.block_table = block_table;
  aa.seq_lens = seq_lens;
  aa.out = static_cast<uint16_t*>(out_bf16);
  aa.status = static_cast<uint32_t*>(workspace);
  aa.work = static_cast<uint32_t*>(workspace) + 1;
  aa.part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kAttnStatusBytes);
  aa.B = B;
  aa.Hq = Hq;
  aa.Hkv = Hkv;
  aa.P = page_size;
  aa.num_pages = num_pages;
  aa.max_pages = max_pages;
  aa.sm_scale = sm_scale;
  aa.timeout_ns = g_timeout_ns.load();
  aa.trace = nullptr;
#ifdef FSOPS_TRACE
  aa.trace = g_trace;
#endif
  const cudaError_t e = launch_paged_decode(aa, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FSOPS_OK : cuda_failed(e, "paged_decode_kernel launch");
}

fsops_status fsops_rmsnorm_quantize_mxfp8(const void* x_bf16, const void* gamma_bf16, float eps, int rows, int K,
                                          int ld, uint8_t* codes, uint8_t* scales, fsops_scale_layout layout,
                                          void* stream) {
  if (layout != FSOPS_SCALES_ROWMAJOR && layout != FSOPS_SCALES_TCGEN05) return FSOPS_ERR_INVALID_ARG;
  if (!(eps >= 0.0f) || eps > 1e30f) return FSOPS_ERR_INVALID_ARG;  // also rejects NaN
  if (rows < 0 || K <= 0 || ld < K) return FSOPS_ERR_UNSUPPORTED_SHAPE;
  if (K % (layout == FSOPS_SCALES_TCGEN05 ? 128 : 32) != 0 || ld % 8 != 0) return FSOPS_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<long long>(rows) * ld >= (1LL << 31)) return FSOPS_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0) return FSOPS_OK;
  if (x_bf16 == nullptr || gamma_bf16 == nullptr || codes == nullptr || scales == nullptr) return FSOPS_ERR_INVALID_ARG;
  if (!aligned16(x_bf16) || !aligned16(gamma_bf16) || !aligned16(codes)) return FSOPS_ERR_MISALIGNED;
  int dev;
  const DeviceInfo* di;
  fsops_status st = current_device(&dev, &di);
  if (st != FSOPS_OK) return st;
  const cudaError_t e = launch_rmsnorm_quantize(
      static_cast<const uint16_t*>(x_bf16), static_cast<const uint16_t*>(gamma_bf16), eps, rows, K, ld, codes, scales,
      layout == FSOPS_SCALES_TCGEN05 ? 1 : 0, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FSOPS_OK : cuda_failed(e, "rmsnorm_quantize_kernel launch");
}

fsops_status fsops_mxfp8_swiglu_mlp_block(const void* x_bf16, const void* gamma_bf16, float eps, int residual,
                                          const uint8_t* w_gateup, const uint8_t* w_down,
                                          const fsops_mlp_scales* scales, void* y_bf16, int M, int H, int I,
                                          void* stream) {
  fsops_status st = mlp_validate(x_bf16, w_gateup, w_down, scales, y_bf16, M, H, I);
  if (st != FSOPS_OK) return st;
  if (gamma_bf16 == nullptr || !(eps >= 0.0f) || eps > 1e30f || (residual != 0 && residual != 1))
    return FSOPS_ERR_INVALID_ARG;
  if (!aligned16(gamma_bf16)) return FSOPS_ERR_MISALIGNED;
  int dev;
  const DeviceInfo* di;
  st = current_device(&dev, &di);
  if (st != FSOPS_OK) return st;
  const MlpLayout l = mlp_layout(M, H, I);
  uint8_t* ws;
  st = check_ws(dev, l.total, &ws);
  if (st != FSOPS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  SlicePlan sp;
  if (M <= 128 && use_slice(M, H, I, di, &sp))  // one launch: the norm runs inside the MLP kernel
    return launch_slice(sp, ws + l.ctl, ws + l.part1, x_bf16, gamma_bf16, eps, residual ? x_bf16 : nullptr,
                        w_gateup, w_down, scales, y_bf16, M, H, I, s);
  if (use_small(M, H, I, di))  // one launch, the norm inside
    return launch_small(l, ws, x_bf16, gamma_bf16, eps, residual ? x_bf16 : nullptr, w_gateup, w_down, scales,
                        y_bf16, M, H, I, di, s);
  const void* res = residual ? x_bf16 : nullptr;
  if (M <= 128) {
    // one launch: the MLP kernel normalises x in its quantisation prologue
    const int grid = di->sms;
    const MlpPlan pl = plan_mlp(M, H, I, grid);
    const MlpBuffers bufs{ws + l.ctl, ws + l.xq, ws + l.xq_sf, ws + l.hq, ws + l.hq_sf, ws + l.part0, ws + l.part1};
    KernelArgs ka;
    st = fill_mlp_args(ka, pl, bufs, x_bf16, w_gateup, w_down, scales, y_bf16, M, H, I, res, gamma_bf16, eps);
    if (st != FSOPS_OK) return st;
    return launch(ka, grid, s);
  }
  // above 128 rows: RMSNorm(x) * gamma quantised into the workspace's x
  // buffers, then the tiled MLP on them, + x
  const cudaError_t e = launch_rmsnorm_quantize(static_cast<const uint16_t*>(x_bf16),
                                                static_cast<const uint16_t*>(gamma_bf16), eps, M, H, H, ws + l.xq,
                                                ws + l.xq_sf, 1, s);
  if (e != cudaSuccess) return cuda_failed(e, "rmsnorm_quantize_kernel launch");
  return mlp_tiled_impl(nullptr, w_gateup, w_down, scales, y_bf16, M, H, I, ws, l, di, s, res);
}

fsops_status fsops_mxfp8_swiglu_mlp_unfused(const void* x_bf16, const uint8_t* w_gateup, const uint8_t* w_down,
                                            const fsops_mlp_scales* scales, void* y_bf16, int M, int H, int I,
                                            void* stream) {
  fsops_status st = mlp_validate(x_bf16, w_gateup, w_down, scales, y_bf16, M, H, I);
  if (st != FSOPS_OK) return st;
  int dev;
  const DeviceInfo* di;
  st = current_device(&dev, &di);
  if (st != FSOPS_OK) return st;
  const MlpLayout l = mlp_layout(M, H, I);
  uint8_t* ws;
  st = check_ws(dev, l.total, &ws);
  if (st != FSOPS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* gu = reinterpret_cast<float*>(ws + l.gu);
  // launch 1: gate/up GEMM, x quantised in-kernel, fp32 [M, 2I] to HBM
  st = gemm_impl(x_bf16, nullptr, true, w_gateup, scales->gateup, gu, true, M, 2 * I, H, ws + l.ctl, ws + l.xq,
                 ws + l.xq_sf, ws + l.part0, di, s);
  if (st != FSOPS_OK) return st;
  // launch 2: SiLU(g) * u, requantised to MXFP8, to HBM
  cudaError_t e = launch_swiglu_quantize(gu, M, I, ws + l.hq, ws + l.hq_sf, s);
  if (e != cudaSuccess) return cuda_failed(e, "swiglu_quantize_kernel launch");
  // launch 3: down GEMM on the requantised intermediate
  return gemm_impl(ws + l.hq, ws + l.hq_sf, false, w_down, scales->down, y_bf16, false, M, H, I, ws + l.ctl,
                   nullptr, nullptr, ws + l.part1, di, s);
}

size_t fsops_blockscale_scale_count(int rows, int K, int block_rows) {
  if (rows < 0 || K <= 0 || K % 128 != 0 || (block_rows != 1 && block_rows != 128)) return 0;
  return static_cast<size_t>((rows + block_rows - 1) / block_rows) * (K / 128);
}

fsops_status fsops_quantize_fp8_blockscale(const void* x_bf16, int rows, int K, int ld, int block_rows, uint8_t* codes,
                                           float* scales, void* stream) {
  if (block_rows != 1 && block_rows != 128) return FSOPS_ERR_INVALID_ARG;
  if (rows < 0 || K <= 0 || K % 128 != 0 || ld < K || ld % 8 != 0) return FSOPS_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<long long>(rows) * ld >= (1LL << 31)) return FSOPS_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0) return FSOPS_OK;
  if (x_bf16 == nullptr || codes == nullptr || scales == nullptr) return FSOPS_ERR_INVALID_ARG;
  if (!aligned16(x_bf16) || !aligned16(codes) || (reinterpret_cast<uintptr_t>(scales) & 3u) != 0)
    return FSOPS_ERR_MISALIGNED;
  int dev;
  const DeviceInfo* di;
  fsops_status st = current_device(&dev, &di);
  if (st != FSOPS_OK) return st;
  const cudaError_t e = launch_bs_quantize(static_cast<const uint16_t*>(x_bf16), rows, K, ld, block_rows, codes, scales,
                                           static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FSOPS_OK : cuda_failed(e, "blockscale quantise launch");
}

size_t fsops_blockscale_gemm_workspace_bytes(int M, int N, int K) {
  if (M < 1 || M > 128 || N < 128 || N % 128 != 0 || K < 128 || K % 128 != 0 || N > 65536 || K > 65536) return 0;
  return kCtlRegionBytes + round_up(static_cast<size_t>(M) * N * 4, 1024);
}

fsops_status fsops_fp8_blockscale_gemm(const uint8_t* a_codes, const float* a_scales, const uint8_t* w_codes,
                                       const float* w_scales, void* c, fsops_dtype c_dtype, int M, int N, int K,
                                       void* workspace, size_t ws_bytes, void* stream) {
  if (a_codes == nullptr || a_scales == nullptr || w_codes == nullptr || w_scales == nullptr || c == nullptr ||
      workspace == nullptr)
    return FSOPS_ERR_INVALID_ARG;
  if (c_dtype != FSOPS_DTYPE_BF16 && c_dtype != FSOPS_DTYPE_F32) return FSOPS_ERR_INVALID_ARG;
  const size_t need = fsops_blockscale_gemm_workspace_bytes(M, N, K);
  if (need == 0) return FSOPS_ERR_UNSUPPORTED_SHAPE;
  if ((N / 128) + kCtlHeaderWords > static_cast<int>(kCtlRegionBytes / 4)) return FSOPS_ERR_UNSUPPORTED_SHAPE;
  if (ws_bytes < need) return FSOPS_ERR_INVALID_ARG;
  if (!aligned16(a_codes) || !aligned16(w_codes) || !aligned16(c) || (reinterpret_cast<uintptr_t>(workspace) & 255u) ||
      (reinterpret_cast<uintptr_t>(a_scales) & 3u) || (reinterpret_cast<uintptr_t>(w_scales) & 3u))
    return FSOPS_ERR_MISALIGNED;
  int dev;
  const DeviceInfo* di;
  fsops_status st = current_device(&dev, &di);
  if (st != FSOPS_OK) return st;
  const int npad = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128;
  BsArgs ba;
  std::memset(&ba, 0, sizeof(ba));
  if (!encode_map(&ba.tm_a, a_codes, K, M, npad) || !encode_map(&ba.tm_w, w_codes, K, N, 128))
    return FSOPS_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  ba.a_scales = a_scales;
  ba.w_scales = w_scales;
  ba.c = c;
  ba.c_f32 = c_dtype == FSOPS_DTYPE_F32 ? 1 : 0;
  ba.accum = reinterpret_cast<float*>(ws + kCtlRegionBytes);
  ba.status = reinterpret_cast<uint32_t*>(ws) + kCtlStatus;
  ba.tile_cnt = reinterpret_cast<uint32_t*>(ws) + kCtlHeaderWords;
  ba.M = M;
  ba.N = N;
  ba.K = K;
  ba.T = N / 128;
  ba.KB = K / 128;
  ba.timeout_ns = g_timeout_ns.load();
  const cudaError_t e = launch_bs_gemm(ba, npad, di->sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FSOPS_OK : cuda_failed(e, "bs_gemm_kernel launch");
}

fsops_status fsops_read_kernel_status(void* workspace, uint32_t* word) {
  if (word == nullptr) return FSOPS_ERR_INVALID_ARG;
  if (workspace == nullptr) {
    int dev;
    const DeviceInfo* di;
    fsops_status st = current_device(&dev, &di);
    if (st != FSOPS_OK) return st;
    std::lock_guard<std::mutex> lk(g_mu);
    workspace = g_ws[dev].ptr;
    if (workspace == nullptr) return FSOPS_ERR_INVALID_ARG;
  }
  uint32_t v = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(workspace, 0, sizeof(v));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_failed(e, "status word read");
  *word = v;
  return FSOPS_OK;
}

fsops_status fsops_set_wait_timeout_ns(uint64_t ns) {
  if (ns == 0) return FSOPS_ERR_INVALID_ARG;
  g_timeout_ns.store(ns);
  return FSOPS_OK;
}

fsops_status fsops_debug_set_extra_arrivals(uint32_t n) {
  g_extra.store(n);
  return FSOPS_OK;
}

fsops_status fsops_debug_set_knob(int k, int value) {
  if (k < 0 || k >= FSOPS_KNOB_COUNT) return FSOPS_ERR_INVALID_ARG;
  g_knob[k].store(value < 0 ? -1 : value);
  return FSOPS_OK;
}

#ifdef FSOPS_TRACE
// Profiling builds only: device buffer of [grid][64] uint64 timeline stamps.
fsops_status fsops_debug_set_trace_buffer(void* buf) {
  g_trace = static_cast<unsigned long long*>(buf);
  return FSOPS_OK;
}
#endif

}  // extern "C"

// ============================================================================
// No-allocation variant of fsops_mxfp8_swiglu_mlp.
//
// Its scratch is a fixed buffer inside the library's device image instead of a
// caller-registered workspace, so neither the caller nor the library ever
// allocates device memory for it.
// ============================================================================
namespace {

// One buffer per device that loads the library, held until the process exits.
constexpr size_t kNoAllocScratchBytes = 8u << 20;  // 8 MiB
__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];
uint8_t* g_noalloc_base[kMaxDevices] = {};
// Per device: the buffer must be cleared before the next call -- before the
// first call, after a call that failed on the host, and after
// fsops_read_noalloc_status found a kernel error (an aborted launch can
// leave split-K sums behind).  A launch that succeeds leaves its counters and
// accumulators zero itself, so calls in between need no clearing.
bool g_noalloc_dirty[kMaxDevices] = {};

// Byte layout inside the fixed buffer: the MLP workspace layout without the
// three-launch path's fp32 [M, 2I] buffer, and without the gate/up split-K
// accumulators when every gate/up tile is done by one block (the kernel never
// touches them then).
struct NoAllocLayout {
  size_t ctl, xq, xq_sf, hq, hq_sf, part0, part1, end;
};
NoAllocLayout noalloc_layout(int M, int H, int I, const MlpPlan& pl) {
  NoAllocLayout l;
  l.ctl = 0;
  l.xq = kCtlRegionBytes;
  l.xq_sf = l.xq + round_up(static_cast<size_t>(M) * H, 1024);
  l.hq = l.xq_sf + round_up(static_cast<size_t>(H / 128) * 512, 1024);
  l.hq_sf = l.hq + round_up(static_cast<size_t>(M) * I, 1024);
  l.part0 = l.hq_sf + round_up(static_cast<size_t>(I / 128) * 512, 1024);
  l.part1 = l.part0 + (pl.whole0 ? 0 : accum_bytes(M, pl.T0));
  l.end = l.part1 + accum_bytes(M, pl.T1);
  return l;
}

// Device address of this device's fixed buffer (looked up on first use: the
// host-side name of a __device__ array is not a device address).
fsops_status noalloc_base(int dev, uint8_t** base) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_noalloc_base[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return cuda_failed(e, "scratch buffer address");
    g_noalloc_base[dev] = static_cast<uint8_t*>(p);
    g_noalloc_dirty[dev] = true;
  }
  *base = g_noalloc_base[dev];
  return FSOPS_OK;
}

}  // namespace

extern "C" {

fsops_status fsops_mxfp8_swiglu_mlp_noalloc(const void* x_bf16, const uint8_t* w_gateup, const uint8_t* w_down,
                                            const fsops_mlp_scales* scales, void* y_bf16, int M, int H, int I,
                                            void* stream) {
  fsops_status st = mlp_validate(x_bf16, w_gateup, w_down, scales, y_bf16, M, H, I);
  if (st != FSOPS_OK) return st;
  int dev;
  const DeviceInfo* di;
  st = current_device(&dev, &di);
  if (st != FSOPS_OK) return st;
  if (M > 128) return FSOPS_ERR_UNSUPPORTED_SHAPE;  // the fixed buffer serves the single-launch path only
  const int grid = di->sms;
  SlicePlan sp;
  const bool sliced = use_slice(M, H, I, di, &sp);
  const MlpPlan pl = plan_mlp(M, H, I, grid);
  if (!sliced && ctl_words_needed(pl.T0, pl.T1) * 4 > kCtlRegionBytes) return FSOPS_ERR_UNSUPPORTED_SHAPE;
  // the sliced kernel needs the control words and its row-tile sums only
  const size_t slice_end = kCtlRegionBytes + (sliced ? slice_accum_bytes(M, H) : 0);
  const NoAllocLayout l = noalloc_layout(M, H, I, pl);
  if ((sliced ? slice_end : l.end) > kNoAllocScratchBytes) return FSOPS_ERR_UNSUPPORTED_SHAPE;  // does not fit

  uint8_t* ws = nullptr;
  if ((st = noalloc_base(dev, &ws)) != FSOPS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bool dirty;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    dirty = g_noalloc_dirty[dev];
  }
  if (dirty) {
    // zero the counters, flags and split-K accumulators the kernel expects at
    // zero (the whole buffer: a different shape may have used other offsets)
    const cudaError_t e = cudaMemsetAsync(ws, 0, kNoAllocScratchBytes, s);
    if (e != cudaSuccess) return cuda_failed(e, "scratch buffer clear");
    std::lock_guard<std::mutex> lk(g_mu);
    g_noalloc_dirty[dev] = false;
  }
  if (sliced) {
    st = launch_slice(sp, ws, ws + kCtlRegionBytes, x_bf16, nullptr, 0.f, nullptr, w_gateup, w_down, scales, y_bf16,
                      M, H, I, s);
  } else {
    const MlpBuffers bufs{ws + l.ctl, ws + l.xq, ws + l.xq_sf, ws + l.hq, ws + l.hq_sf, ws + l.part0, ws + l.part1};
    KernelArgs ka;
    st = fill_mlp_args(ka, pl, bufs, x_bf16, w_gateup, w_down, scales, y_bf16, M, H, I);
    if (st == FSOPS_OK) st = launch(ka, grid, s);
  }
  if (st != FSOPS_OK) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_noalloc_dirty[dev] = true;
  }
  return st;
}

fsops_status fsops_read_noalloc_status(uint32_t* word) {
  if (word == nullptr) return FSOPS_ERR_INVALID_ARG;
  int dev;
  const DeviceInfo* di;
  fsops_status st = current_device(&dev, &di);
  if (st != FSOPS_OK) return st;
  uint8_t* base;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    base = g_noalloc_base[dev];
  }
  if (base == nullptr) return FSOPS_ERR_INVALID_ARG;  // no no-allocation call on this device yet
  st = fsops_read_kernel_status(base, word);
  if (st == FSOPS_OK && *word != 0) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_noalloc_dirty[dev] = true;
  }
  return st;
}

}  // extern "C"
