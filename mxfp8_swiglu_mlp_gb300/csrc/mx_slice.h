// mx_slice.h -- arguments, shared-memory layout and launch of the
// cluster-sliced decode MLP kernel (mx_slice.cu).  Not part of the public ABI.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "mx_internal.h"

namespace fsops {

// Blocks per cluster, the most 128-feature chunks one cluster may own, and
// the tokens per launch the sliced kernel serves (the N of its MMAs).
constexpr int kSliceCluster = 2;
constexpr int kSliceMaxChunks = 4;
constexpr int kSliceMaxM = 32;
constexpr int kSliceMaxStages = 12;
// TMEM accumulators (npad columns each) used round robin, so that an
// accumulator is drained while the next one fills.
constexpr int kSliceAccBufs = 4;
// W tile of one pipeline stage: 128 weight rows x 128 K bytes.
constexpr uint32_t kSliceWBytes = 128u * 128u;

struct SliceArgs {
  CUtensorMap tm_wgu;   // W_gateup codes [2I, H] u8, box 128 rows x 128, 128B swizzle
  CUtensorMap tm_wd;    // W_down codes [H, I] u8, box 128 rows x 128, 128B swizzle
  CUtensorMap tm_x;     // bf16 x [M, H], box npad rows x 128 elements, no swizzle
  const uint8_t* sf_gu; // W_gateup scales (tcgen05 tiled layout)
  const uint8_t* sf_d;  // W_down scales (tcgen05 tiled layout)
  const uint16_t* x;    // bf16 x [M, H] (the RMSNorm row pass reads it directly)
  const uint16_t* gamma;  // bf16 [H] RMSNorm gain, or null: x is quantised as it is
  float eps;
  uint16_t* y;          // bf16 [M, H]
  const uint16_t* residual;  // bf16 [M, H] added to y before its rounding, or null
  float* accum;         // [M][H] fp32 partial sums of y, zero between launches
  uint32_t* tile_cnt;   // [RT] arrival counters of the 128-row tiles of y, zero between launches
  uint32_t* status;     // first error: (status << 24) | (site << 16) | block
  int M, H, I;
  int NC;               // I / 128 feature chunks
  int NP;               // clusters; cluster q owns chunks [q NC / NP, (q + 1) NC / NP)
  int KS0;              // H / 128 k-stages of the gate/up projection
  int RT;               // H / 128 row tiles of the down projection
  int nstages;
  uint64_t timeout_ns;
  uint32_t extra_arrivals;  // test hook: arrivals more than any launch makes on h_full
  unsigned long long* trace;  // [grid][64] %globaltimer stamps, builds with FSOPS_TRACE only
};

// Pipeline stage: X tile (npad x 128 B, E4M3) | W tile (128 x 128 B) | W
// scales (512 B) | X scales (512 B) | bf16 x tile (npad x 128 elements, the
// gate/up stages only); a multiple of 1024 bytes for npad in {16, 32}.
__host__ __device__ inline uint32_t slice_stage_bytes(int npad) { return 384u * npad + kSliceWBytes + 1024u; }
__host__ __device__ inline uint32_t slice_off_w(int npad) { return 128u * npad; }
__host__ __device__ inline uint32_t slice_off_sfw(int npad) { return 128u * npad + kSliceWBytes; }
__host__ __device__ inline uint32_t slice_off_sfx(int npad) { return 128u * npad + kSliceWBytes + 512u; }
__host__ __device__ inline uint32_t slice_off_xb(int npad) { return 128u * npad + kSliceWBytes + 1024u; }
// Shared memory, from a 1024-aligned base:
//   htile  [kSliceMaxChunks][npad][128] E4M3 h, 128B-swizzled (the down MMA's B operand)
//   hsf    [kSliceMaxChunks][512] tcgen05 scale tiles of h
//   ring   nstages stages
//   ubuf   fp32 up sums of the block's 64 features, [64][npad + 4]
//   ctl    barriers and flags
__host__ __device__ inline uint32_t slice_off_hsf(int npad) { return kSliceMaxChunks * 128u * npad; }
__host__ __device__ inline uint32_t slice_off_ring(int npad) { return slice_off_hsf(npad) + kSliceMaxChunks * 512u; }
__host__ __device__ inline uint32_t slice_ubuf_ld(int npad) { return static_cast<uint32_t>(npad) + 4u; }
__host__ __device__ inline uint32_t slice_fixed_bytes(int npad) {
  return slice_off_ring(npad) + 64u * slice_ubuf_ld(npad) * 4u + 2048u + 1024u;
}
__host__ __device__ inline int slice_stages(int npad) {
  int s = static_cast<int>((kMaxSmem - slice_fixed_bytes(npad)) / slice_stage_bytes(npad));
  return s > kSliceMaxStages ? kSliceMaxStages : s;
}
__host__ __device__ inline size_t slice_smem(int npad) {
  return static_cast<size_t>(slice_stages(npad)) * slice_stage_bytes(npad) + slice_fixed_bytes(npad);
}

// grid = NP * kSliceCluster blocks in 2-block clusters, launched with
// programmatic stream serialization (the weight stream of a launch may start
// while the previous kernel on the stream finishes).
cudaError_t launch_slice_kernel(const SliceArgs& a, int npad, cudaStream_t stream);

}  // namespace fsops
