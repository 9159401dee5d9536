// mx_small.h -- arguments, shared-memory layout and launch of the fused
// MXFP8 SwiGLU MLP for up to 8 tokens and small hidden sizes (mx_small.cu).
// Not part of the public ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fsops {

// Tokens one launch serves (the N of its MMAs).
constexpr int kSmallMaxM = 8;
// Control words of the workspace the kernel uses besides the status word:
// units of h published in this launch, blocks that have left it (the last
// one sets both back to zero).
constexpr int kCtlSmallPublished = 4;
constexpr int kCtlSmallExits = 5;

struct SmallArgs {
  CUtensorMap tm_wgu;   // W_gateup codes [2I, H] u8, box 32 rows x 128, 128B swizzle
  CUtensorMap tm_wd;    // W_down codes [H, I] u8, box 16 rows x 128, 128B swizzle
  const uint8_t* sf_gu; // W_gateup scales (tcgen05 tiled layout)
  const uint8_t* sf_d;  // W_down scales (tcgen05 tiled layout)
  const uint16_t* x;    // bf16 [M, H]
  const uint16_t* gamma;  // bf16 [H] RMSNorm gain, or null
  float eps;
  const uint16_t* residual;  // bf16 [M, H] added to y before its rounding, or null
  uint16_t* y;          // bf16 [M, H]
  uint8_t* hq;          // [M, I] E4M3 codes of h (row-major)
  uint8_t* hs;          // [M, I / 32] UE8M0 scales of h (row-major)
  uint32_t* ctl;        // the workspace's control words
  int M, H, I;
  int U;                // I / 32 units of h (block u computes features 32u .. 32u + 31)
  int T;                // H / 16 row tiles of y (rows 16t .. 16t + 15)
  int split;            // 1: blocks U .. U + T - 1 compute the tiles (U + T blocks), 0: block t
                        //    computes tile t after its unit (max(U, T) blocks)
  uint64_t timeout_ns;
  uint32_t extra_arrivals;  // test hook: units more than any launch publishes
  unsigned long long* trace;  // [grid][128] %globaltimer stamps, builds with FSOPS_TRACE only
};

// Weight bytes of one block: a unit's 64 W_gateup rows and a tile's 16
// W_down rows, in one region when the roles are split.
__host__ __device__ inline size_t small_weight_bytes(int H, int I, int split) {
  const size_t wa = 64u * static_cast<size_t>(H), wb = 16u * static_cast<size_t>(I);
  return split ? (wa > wb ? wa : wb) : wa + wb;
}
// Dynamic shared memory of one block (from a 1024-byte aligned base).
__host__ __device__ inline size_t small_smem_bytes(int H, int I, int split) {
  return small_weight_bytes(H, I, split)                                  // weights
         + 8u * (H + 32) + 8u * (I + 32)                                 // x and h codes
         + 4u * 8 * (H / 32) + 4u * 8 * (I / 32)                         // x and h scales
         + 64u * (H / 32) + 16u * (I / 32)                               // weight scales
         + 16 + 4u * 16 * 16 * 8 + 4u * 8 * 32                           // reduction (16 warps), h in fp32
         + 1024;                                                         // alignment
}
// Whether the shape runs on this kernel: M <= 8, H and I multiples of 128,
// one block per unit of h and per row tile of y on `sms` SMs, and the
// block's weights in shared memory.
bool small_fits(int M, int H, int I, int sms);
// Whether the roles are split (U + T blocks fit the SMs).
inline int small_split(int H, int I, int sms) { return I / 32 + H / 16 <= sms ? 1 : 0; }
cudaError_t launch_small_kernel(const SmallArgs& a, int grid, cudaStream_t stream);

}  // namespace fsops
