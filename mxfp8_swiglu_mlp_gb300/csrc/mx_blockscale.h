// mx_blockscale.h -- arguments and launches of the FP8 GEMM with 128 x 128
// block scales (mx_blockscale.cu).  Not part of the public ABI.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fsops {

// C[M, N] = A^[M, K] . W^[N, K]^T with E4M3 codes and fp32 scales: one per
// 1 x 128 group of A (row m, K-block kb) and one per 128 x 128 block of W.
struct BsArgs {
  CUtensorMap tm_a;      // A codes [M, K] u8, box npad rows x 128, 128B swizzle (rows past M read as zero)
  CUtensorMap tm_w;      // W codes [N, K] u8, box 128 rows x 128, 128B swizzle
  const float* a_scales; // [M, K / 128]
  const float* w_scales; // [N / 128, K / 128]
  void* c;               // [M, N] bf16 or fp32
  int c_f32;
  float* accum;          // [M, N] fp32 sums of tiles split between blocks, zero between launches
  uint32_t* tile_cnt;    // [N / 128] arrival counters of split tiles, zero between launches
  uint32_t* status;      // first error: (status << 24) | (site << 16) | block
  int M, N, K;
  int T, KB;             // N / 128 row tiles of W, K / 128 blocks of K
  uint64_t timeout_ns;
};

// One launch of the GEMM (npad = M rounded up to 16, 32, 64 or 128 tokens)
// on `sms` SMs at most, with programmatic stream serialization.
cudaError_t launch_bs_gemm(const BsArgs& a, int npad, int sms, cudaStream_t stream);
// E4M3 codes and fp32 scales of bf16 x [rows, K] (row stride ld) in blocks of
// block_rows (1 or 128) x 128.
cudaError_t launch_bs_quantize(const uint16_t* x, int rows, int K, int ld, int block_rows, uint8_t* codes,
                               float* scales, cudaStream_t stream);

}  // namespace fsops
