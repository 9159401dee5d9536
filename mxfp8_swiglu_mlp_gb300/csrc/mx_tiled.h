// mx_tiled.h -- arguments and launch of the whole-tile block-scaled GEMM
// (mx_gemm_tiled.cu), the path for more than 128 token rows.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fsops {

// Block-scaled GEMM for M > 128 (mx_gemm_tiled.cu): whole output tiles per
// block (or block pair), no split-K.  Launch forms:
//   kTiledSingle     one block per 128 x 256 tile;
//   kTiledPairMma    2-block clusters computing one 256 x 256 tile with
//                    cta_group::2 MMAs (N % 256 == 0, at least two row tiles).
enum { kTiledSingle = 0, kTiledPairMma = 1 };
struct TiledArgs {
  CUtensorMap tm_a;       // A codes [M, K] u8, box 128 rows x 128, 128B swizzle
  CUtensorMap tm_b;       // B codes [N, K] u8, box 256 rows x 128 (128 rows in the pair form), 128B swizzle
  CUtensorMap tm_c;       // C [M, N] bf16 (box 32 rows x 32) or fp32 (box 32 rows x 16), no swizzle
  // the scales as 2-D tensors of 512-byte rows (one tcgen05 scale tile each),
  // u32 elements, box 128 x 1: loaded by TMA in the pair-MMA form
  CUtensorMap tm_sfa;     // ceil(M / 128) * KS rows
  CUtensorMap tm_sfb;     // (N / 128) * KS rows
  const uint8_t* sf_a;    // A scales, tiled layout, ceil(M / 128) row tiles
  const uint8_t* sf_b;    // B scales, tiled layout, N / 128 row tiles
  void* c;                // [M, N] bf16 or fp32
  int c_f32;
  int M, N, K, KS;        // KS = K / 128
  int MT, NT;             // ceil(M / 128), ceil(N / 256)
  uint32_t* status;       // first error (status << 24 | site << 16 | block)
  uint64_t timeout_ns;
  int form;               // kTiledSingle or kTiledPairMma
  const uint16_t* residual;  // bf16 [M, N] added to a bf16 C before its rounding, or null
  // SwiGLU epilogue (swiglu = 1): B is W_gateup, whose 128-row blocks hold 64
  // gate rows and then the 64 up rows of the same features, so a 256-column
  // tile covers 128 whole features.  The epilogue writes h = SiLU(g) * u,
  // requantised to MXFP8 along the features, instead of C (tm_c and c unused).
  int swiglu;
  uint8_t* h_codes;       // [M, N / 2] E4M3
  uint8_t* h_sf;          // h scales, tiled layout, ceil(M / 128) row tiles of N / 256 tiles each
};
// Launches at most one block per SM (`sms`).
cudaError_t launch_gemm_tiled(const TiledArgs& a, int sms, cudaStream_t stream);

}  // namespace fsops
