// mx_internal.h -- structures shared by the host launcher (fsops_api.cu) and
// the kernels (mx_kernels.cu).  Not part of the public ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fsops {

// Control words at the start of every workspace (uint32 indices).
enum CtlWord : int {
  kCtlStatus = 0,   // first error: (status << 24) | (site << 16) | block
  kCtlCleanup = 1,  // taken by the block that clears the control words after a launch gave up
  kCtlExits = 2,    // words 2-3: 64-bit count of blocks that have left, over all launches
  kCtlHeaderWords = 16,
};
// Readiness counters kept per consuming block (at most kMaxGrid blocks): each
// producer adds to the counter of every block that will read what it wrote,
// and each block clears its own counter once it has seen it complete, so a
// launch that succeeds leaves them zero without a grid-wide last step.
constexpr int kMaxGrid = 256;
// Wait sites reported in the status word.
enum WaitSite : uint32_t {
  kSiteEmpty = 1, kSiteFullW = 2, kSiteFullA = 3, kSiteAccEmpty = 4, kSiteAccFull = 5,
  kSiteXReady = 6, kSiteHFlag = 7, kSiteDrain = 8, kSiteTileSum = 9, kSitePeer = 10,
};

enum : int { kDepNone = 0, kDepXReady = 1, kDepHFlags = 2 };
enum : int { kEpiSwiGLU = 0, kEpiStore = 1 };

constexpr int kThreads = 256;       // 8 warps: 0 weight TMA, 1 activation TMA, 2 MMA, 3 idle, 4-7 epilogue
constexpr int kMaxStages = 8;
constexpr int kTileK = 128;         // K elements (bytes) per pipeline stage
constexpr int kTileRows = 256;      // largest weight tile (rows) = N of the tcgen05 instruction; accumulator row stride
constexpr int kMmaM = 128;          // M of the tcgen05 instruction: token rows (padded)
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxSmem = 232448;    // 227 KB opt-in per block

// W_gateup row order: 128-row blocks j = [W_gate rows 64j..64j+63; W_up rows
// 64j..64j+63], so every 128 rows hold gate/up pairs for 64 intermediate
// features and one 512-byte scale tile covers them.  A weight tile of 128
// rows gives 64 features, one of 256 rows 128 (two pair blocks).
constexpr int kPairRows = 64;
// weight loads in flight per block before its activations are available
constexpr int kPrimeInflight = 1;
// split tiles whose finish an epilogue defers to the end of a phase
constexpr int kMaxPend = 4;

// One GEMM phase of the persistent kernel: T tiles of tile_rows (256 or 128)
// weight rows times KS k-stages of 128, split evenly over the grid (stream-K).
struct PhaseArgs {
  const uint8_t* sf_w;    // weight scales (tiled layout)
  const uint8_t* sf_act;  // activation scales (tiled layout, row tile 0)
  uint32_t* tile_cnt;     // [T] arrival counters for split tiles
  float* accum;           // [T][M][256] fp32 sums of split tiles (row-major), zero between launches
  int KS;                 // K / 128
  int T;                  // number of tiles (ceil(rows / tile_rows))
  int tile_rows;          // weight rows per tile = N of the tcgen05 instruction: 256 or 128
  int rows;               // weight rows (a multiple of 128)
  int whole_tiles;        // 1: block t < T does all of tile t (requires T <= grid), no split-K
  int pairs;              // 1: the two blocks of cluster c split tile c in two K halves and add
                          //    their sums through distributed shared memory (M <= 32, T <= grid / 2)
  int aligned;            // 1: tile t goes to blocks [ceil(t G / T), ceil((t+1) G / T)), which split
                          //    its K range evenly (T <= grid, KS >= ceil(G / T)): no block holds
                          //    parts of two tiles
  int dep;                // what the activation loads wait for (kDep*)
  int epi;                // epilogue kind (kEpi*)
  int out_ld;             // row stride (elements) of the plain output
};

struct KernelArgs {
  CUtensorMap tm_w[2];    // weight codes [rows, K] u8, box tile_rows x 128, 128B swizzle
  CUtensorMap tm_act[2];  // activation codes [M, K] u8, box npad x 128, 128B swizzle
  CUtensorMap tm_x;       // bf16 x [M, H], box npad x 128 elements, no swizzle (local_xq only)
  PhaseArgs ph[2];
  int nphases;
  // activation quantisation (x != nullptr)
  const uint16_t* x;      // bf16 [M, H]
  const uint16_t* gamma;  // bf16 [H]: x is RMSNorm(x) * gamma before quantisation (grid-wide path only), or null
  float eps;
  uint8_t* xq_codes;      // [M, H] (grid-wide quantisation only)
  uint8_t* xq_sf;         // tiled, H / 128 tiles
  int H;
  // SwiGLU epilogue output
  uint8_t* hq_codes;      // [M, I]
  uint8_t* hq_sf;         // tiled, I / 128 tiles
  int I;
  // plain epilogue output
  void* out;              // [M, out_ld]
  int out_f32;
  const uint16_t* residual;  // bf16 [M, out_ld] added to a bf16 output before its rounding, or null
  // control
  uint32_t* ctl;          // kCtlHeaderWords words
  uint32_t* xready;       // [grid]: x slices quantised for block b (grid-wide x quantisation)
  uint32_t* hflags;       // [grid]: SwiGLU tiles written that block b's down-projection stages read
  int M;
  int npad;               // M rounded up to 16: activation rows held in shared memory
  int nstages;
  int local_xq;           // 1: phase 0's activation tiles are quantised from x by each block itself (npad <= 32)
  int stage_tmem;         // 1: accumulators are copied to shared memory before the epilogue (M <= 32)
  int cluster_pairs;      // launched as 2-block clusters (a phase uses pairs)
  int max_inflight;       // weight tiles a block may have in flight at once
  int prime_inflight;     // ... before its activations are available (x quantised grid-wide)
  int early_w;            // 1: the weight producer starts before the block's x loads are issued
  uint32_t stage_bytes;
  uint64_t timeout_ns;
  uint32_t extra_xready;  // test hook: extra arrivals to wait for
  unsigned long long* trace;  // [grid][128] %globaltimer stamps, builds with FSOPS_TRACE only
};

// Shared-memory stage layout: X (activations, npad x 128 B), W (weights,
// 256 x 128 B), two weight scale tiles, one activation scale tile.  The MMA
// reads 128 activation rows; rows past npad alias the start of W and only
// produce accumulator lanes that are never read.
__host__ __device__ inline uint32_t stage_off_w(int npad) { return 128u * npad; }
__host__ __device__ inline uint32_t stage_off_sfw(int npad) { return 128u * npad + 32768u; }
__host__ __device__ inline uint32_t stage_off_sfx(int npad) { return 128u * npad + 32768u + 1024u; }
__host__ __device__ inline uint32_t stage_bytes_for(int npad) {
  return (128u * npad + 32768u + 1536u + 1023u) & ~1023u;
}
constexpr uint32_t kSmemCtlBytes = 1024;
// fp32 staging of one accumulator (npad <= 32 tokens x 256 columns, padded rows)
constexpr int kStageLd = 260;
__host__ __device__ inline uint32_t stg_bytes_for(int npad) {
  return (static_cast<uint32_t>(npad) * kStageLd * 4u + 1023u) & ~1023u;
}
// With local_xq: a ring of bf16 x tiles (npad x 128 elements each) that the
// activation producer warp fills by TMA and quantises into the stages.
constexpr int kMaxXSlots = 4;
__host__ __device__ inline uint32_t xring_bytes_for(int npad) { return kMaxXSlots * 256u * npad; }
// Cluster pairs at npad = 16: once the x stages are filled, the x ring's first
// half holds this block's sums of the partner's half of the columns (16 rows
// x 128 fp32) and its second half receives the partner's.
constexpr uint32_t kPairRecvOff = 8192;
// TMEM columns: accumulator [0, 256), then per pipeline stage 12 scale columns
// (activation tile: 4, weight tiles: 8).
constexpr uint32_t kAccCols = 256;
constexpr uint32_t kSfColsPerStage = 12;

// Launch wrappers (mx_kernels.cu).  The persistent kernel's blocks wait on
// one another, so all `grid` of them must be resident at once.  A cooperative
// launch guarantees that; the plain launch (with programmatic stream
// serialization: it may start while the previous kernel on the stream
// finishes) relies on it holding once that kernel has completed -- every
// wait on another block comes after the grid dependency wait -- which
// grid_fits checks against the device's resources.
cudaError_t launch_mx_kernel(const KernelArgs& a, int grid, size_t smem, cudaStream_t stream, bool cooperative);
bool grid_fits(int grid, size_t smem);
// Whether `grid` blocks of the kernel with `smem` bytes of shared memory run
// as grid / 2 co-resident 2-block clusters on the current device.
bool cluster_pairs_fit(int grid, size_t smem);
// up != nullptr: x is W_gate [rows / 2, K], up is W_up [rows / 2, K], and the
// rows are quantised in the paired W_gateup order (blocks of kPairRows).
cudaError_t launch_quantize(const uint16_t* x, int rows, int K, int ld, uint8_t* codes, uint8_t* scales,
                            int tiled, cudaStream_t stream, const uint16_t* up = nullptr);
cudaError_t launch_swiglu_quantize(const float* gu, int M, int I, uint8_t* hc, uint8_t* hs,
                                   cudaStream_t stream);
cudaError_t launch_rmsnorm_quantize(const uint16_t* x, const uint16_t* gamma, float eps, int rows, int K, int ld,
                                    uint8_t* codes, uint8_t* scales, int tiled, cudaStream_t stream);

}  // namespace fsops
