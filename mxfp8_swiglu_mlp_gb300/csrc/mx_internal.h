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
  kCtlXReady = 1,   // number of blocks that finished quantising their slice of x
  kCtlDone = 2,     // number of blocks that finished the launch
  kCtlHeaderWords = 16,
};
// Wait sites reported in the status word.
enum WaitSite : uint32_t {
  kSiteEmpty = 1, kSiteFullW = 2, kSiteFullA = 3, kSiteAccEmpty = 4, kSiteAccFull = 5,
  kSiteXReady = 6, kSiteHFlag = 7, kSiteDrain = 8,
};

enum : int { kDepNone = 0, kDepXReady = 1, kDepHFlags = 2 };
enum : int { kEpiSwiGLU = 0, kEpiStore = 1 };

constexpr int kThreads = 256;       // 8 warps: 0 weight TMA, 1 activation TMA, 2 MMA, 3 idle, 4-7 epilogue
constexpr int kMaxStages = 12;
constexpr int kTileK = 128;         // K elements (bytes) per pipeline stage
constexpr int kTileRows = 128;      // weight rows per tile = M of the tcgen05 instruction
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxSmem = 232448;    // 227 KB opt-in per block

// W_gateup row order: 128-row blocks j = [W_gate rows 64j..64j+63; W_up rows
// 64j..64j+63], so one 128-row tile holds a gate/up pair for 64 intermediate
// features and its scales form one 512-byte scale tile.
constexpr int kPairFeatures = 64;

// One GEMM phase of the persistent kernel: T tiles of 128 weight rows times KS
// k-stages of 128, split evenly over the grid (stream-K).
struct PhaseArgs {
  const uint8_t* sf_w;    // weight scales (tiled layout)
  const uint8_t* sf_act;  // activation scales (tiled layout, row tile 0)
  uint32_t* tile_cnt;     // [T] arrival counters for split tiles
  float* accum;           // [T][M][128] fp32 sums of split tiles, zero between launches
  int KS;                 // K / 128
  int T;                  // number of tiles (rows / 128)
  int dep;                // what the activation loads wait for (kDep*)
  int epi;                // epilogue kind (kEpi*)
  int out_ld;             // row stride (elements) of the plain output
};

struct KernelArgs {
  CUtensorMap tm_w[2];    // weight codes [rows, K] u8, box 128 x 128, 128B swizzle
  CUtensorMap tm_act[2];  // activation codes [M, K] u8, box 128 x npad, 128B swizzle
  PhaseArgs ph[2];
  int nphases;
  // in-kernel activation quantisation (x != nullptr)
  const uint16_t* x;      // bf16 [M, H]
  uint8_t* xq_codes;      // [M, H]
  uint8_t* xq_sf;         // tiled, H / 128 tiles
  int H;
  // SwiGLU epilogue output
  uint8_t* hq_codes;      // [M, I]
  uint8_t* hq_sf;         // tiled, I / 128 tiles
  int I;
  // plain epilogue output
  void* out;              // [M, out_ld]
  int out_f32;
  // control
  uint32_t* ctl;          // kCtlHeaderWords words
  uint32_t* hflags;       // [I / 128]: SwiGLU tiles finished per 128-feature chunk (2 when ready)
  int M;
  int npad;               // M rounded up to 16 (the MMA N)
  int nstages;
  int nacc;               // accumulator buffers in TMEM
  int chains;             // independent accumulators per tile (k-step k adds into chain k % chains)
  int local_xq;           // 1: phase 0's activation tiles are quantised from x by each block itself
  int max_inflight;       // weight tiles a block may have in flight at once
  uint32_t stage_bytes;
  uint64_t timeout_ns;
  uint32_t extra_xready;  // test hook: extra arrivals to wait for
  unsigned long long* trace;  // [grid][64] %globaltimer stamps, builds with FSOPS_TRACE only
};

// Shared-memory stage layout: A (weights, 128 x 128 B), B (activations,
// npad x 128 B), the A scale tile and the B scale tile (512 B each).
__host__ __device__ constexpr uint32_t stage_off_a() { return 0; }
__host__ __device__ constexpr uint32_t stage_off_b() { return 16384; }
__host__ __device__ inline uint32_t stage_off_sfa(int npad) { return 16384u + 128u * npad; }
__host__ __device__ inline uint32_t stage_off_sfb(int npad) { return 16384u + 128u * npad + 512u; }
__host__ __device__ inline uint32_t stage_bytes_for(int npad) {
  return (16384u + 128u * npad + 1024u + 1023u) & ~1023u;
}
constexpr uint32_t kSmemCtlBytes = 1024;
constexpr uint32_t kSmemXchgBytes = 16 * 128 * 4;  // one 16-token chunk of a 128-row tile, fp32
// TMEM columns of one stage's scale tiles (A, then B).
constexpr uint32_t kSfColsPerStage = 8;

// Launch wrappers (mx_kernels.cu).
cudaError_t launch_mx_kernel(const KernelArgs& a, int grid, size_t smem, cudaStream_t stream);
cudaError_t launch_quantize(const uint16_t* x, int rows, int K, int ld, uint8_t* codes, uint8_t* scales,
                            int tiled, cudaStream_t stream);
cudaError_t launch_swiglu_quantize(const float* gu, int M, int I, uint8_t* hc, uint8_t* hs,
                                   cudaStream_t stream);

}  // namespace fsops
