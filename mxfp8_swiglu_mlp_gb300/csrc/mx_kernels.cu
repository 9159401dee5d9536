// mx_kernels.cu -- the sm_103a kernels of the MXFP8 SwiGLU MLP.
//
//   mx_persistent_kernel   one launch per GEMM (M <= 128) or per whole MLP:
//                          cooperative grid of one block per SM; TMA streams
//                          weight tiles, tcgen05 block-scaled MMAs accumulate
//                          in TMEM; per phase either a stream-K split of the
//                          K loop over all blocks (sums added in L2), one
//                          whole tile per block, or 2-block clusters that add
//                          their two K halves through distributed shared memory.
//   quantize_kernel        bf16 -> E4M3 + UE8M0 (row-major or tiled scales).
//   swiglu_quantize_kernel SiLU(g) * u -> E4M3 + UE8M0 (the unfused path).
//
// Quantisation rule (OCP MX, as the Fish Audio post's mxfp8 format uses it,
// p2 "Estrategia de cuantizacion FP8"): for each 32-block, the UE8M0 byte is
// max(biased_exponent(amax) - 8, 0), i.e. e = floor(log2 amax) - 8 clamped at
// -127; elements are v * 2^-e converted to E4M3 with round-to-nearest-even
// and saturation (cvt ... satfinite).  v * 2^-e is exact in fp32 wherever the
// rounding can depend on it, so the codes are bit-exact with an exact
// computation.
#include <cuda_bf16.h>
#include <atomic>
#include <cuda_fp8.h>

#include "mx_internal.h"
#include "mx_device.cuh"
#include "mx_mxfp8.cuh"
#include "sm103.cuh"

namespace fsops {
using namespace dev;

// ======================================================================
// Standalone quantiser: one thread per 32-block.
// With `up` != null the rows come from two matrices in the paired order of
// W_gateup: destination row r of block j = r / 128 is row 64 j + r % 128 of
// `x` (W_gate) for r % 128 < 64, else row 64 j + r % 128 - 64 of `up` (W_up).
// ======================================================================
__global__ void quantize_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ up, int rows,
                                int rows_pad, int K, int ld, uint8_t* __restrict__ codes,
                                uint8_t* __restrict__ scales, int tiled) {
  const int nb = K / 32;
  const long long total = static_cast<long long>(rows_pad) * nb;
  for (long long b = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; b < total;
       b += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(b / nb), kb = static_cast<int>(b % nb);
    uint32_t s = 0;
    if (r < rows) {
      const uint16_t* src = x;
      int sr = r;
      if (up != nullptr) {
        const int j = r >> 7, w = r & 127;
        src = w < kPairRows ? x : up;
        sr = j * kPairRows + (w & (kPairRows - 1));
      }
      s = quantize_block_bf16(src + static_cast<long long>(sr) * ld + kb * 32,
                              codes + static_cast<long long>(r) * K + kb * 32);
    }
    if (tiled) {
      scales[tiled_sf_offset(r, kb, K / 128)] = static_cast<uint8_t>(s);
    } else if (r < rows) {
      scales[static_cast<long long>(r) * nb + kb] = static_cast<uint8_t>(s);
    }
  }
  // weights quantised here may be streamed by the next kernel on the stream
  // before it waits for this one (the decode kernels' programmatic launch):
  // the writes are made visible before the block leaves
  __threadfence();
}

cudaError_t launch_quantize(const uint16_t* x, int rows, int K, int ld, uint8_t* codes, uint8_t* scales,
                            int tiled, cudaStream_t stream, const uint16_t* up) {
  const int rows_pad = tiled ? (rows + 127) / 128 * 128 : rows;
  const long long total = static_cast<long long>(rows_pad) * (K / 32);
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  long long blocks = (total + threads - 1) / threads;
  if (blocks > 65535LL * 16) blocks = 65535LL * 16;
  quantize_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(x, up, rows, rows_pad, K, ld, codes,
                                                                          scales, tiled);
  return cudaGetLastError();
}

// ======================================================================
// RMSNorm + quantisation: one block per row.  The row's mean square is
// reduced in fp32, then each thread quantises whole 32-blocks of
// x * rsqrt(mean(x^2) + eps) * gamma (fp32) with the rule above.  Rows of the
// last 128-row scale tile past `rows` get scale 0 (tiled layout).
// ======================================================================
constexpr int kNormThreads = 128;
__global__ void __launch_bounds__(kNormThreads) rmsnorm_quantize_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ gamma, float eps, int rows, int K, int ld,
    uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, int tiled) {
  const int r = blockIdx.x, nb = K / 32;
  if (r >= rows) {
    for (int kb = threadIdx.x; kb < nb; kb += kNormThreads) scales[tiled_sf_offset(r, kb, K / 128)] = 0;
    return;
  }
  const uint16_t* xr = x + static_cast<long long>(r) * ld;
  float ss = 0.f;
  for (int i = threadIdx.x; i < K / 8; i += kNormThreads) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(xr) + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = bf16_lo(w[j]), hi = bf16_hi(w[j]);
      ss = fmaf(lo, lo, fmaf(hi, hi, ss));
    }
  }
  __shared__ float part[kNormThreads / 32];
  for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < kNormThreads / 32; ++i) tot += part[i];
  const float inv_rms = rsqrtf(tot / static_cast<float>(K) + eps);
  for (int kb = threadIdx.x; kb < nb; kb += kNormThreads) {
    float v[32];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 xv = __ldg(reinterpret_cast<const uint4*>(xr + kb * 32) + q);
      const uint4 gv = __ldg(reinterpret_cast<const uint4*>(gamma + kb * 32) + q);
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[8 * q + 2 * j] = bf16_lo(xw[j]) * inv_rms * bf16_lo(gw[j]);
        v[8 * q + 2 * j + 1] = bf16_hi(xw[j]) * inv_rms * bf16_hi(gw[j]);
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const uint32_t sc = ue8m0_from_amax(amax);
    const float inv = inv_scale_from_ue8m0(sc);
    uint32_t pk[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      pk[i] = e4m3_code(v[4 * i] * inv) | (e4m3_code(v[4 * i + 1] * inv) << 8) |
              (e4m3_code(v[4 * i + 2] * inv) << 16) | (e4m3_code(v[4 * i + 3] * inv) << 24);
    uint4* d = reinterpret_cast<uint4*>(codes + static_cast<long long>(r) * K + kb * 32);
    d[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    d[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
    if (tiled) scales[tiled_sf_offset(r, kb, K / 128)] = static_cast<uint8_t>(sc);
    else scales[static_cast<long long>(r) * nb + kb] = static_cast<uint8_t>(sc);
  }
}

cudaError_t launch_rmsnorm_quantize(const uint16_t* x, const uint16_t* gamma, float eps, int rows, int K, int ld,
                                    uint8_t* codes, uint8_t* scales, int tiled, cudaStream_t stream) {
  const int grid = tiled ? (rows + 127) / 128 * 128 : rows;
  if (grid == 0) return cudaSuccess;
  rmsnorm_quantize_kernel<<<grid, kNormThreads, 0, stream>>>(x, gamma, eps, rows, K, ld, codes, scales, tiled);
  return cudaGetLastError();
}

// ======================================================================
// SwiGLU + requantisation (the middle launch of the unfused path).
// ======================================================================
// SiLU(g) * u = g * sigmoid(g) * u (silu_mul); for g -> -inf the reciprocal
// of inf is 0.
__global__ void swiglu_quantize_kernel(const float* __restrict__ gu, int M, int npad, int I,
                                       uint8_t* __restrict__ hc, uint8_t* __restrict__ hs) {
  const int nb = I / 32;
  const int total = npad * nb;
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < total; b += gridDim.x * blockDim.x) {
    const int m = b / nb, kb = b % nb;
    uint32_t s = 0;
    if (m < M) {
      // gu columns follow the W_gateup row order: 128-column block j holds gate
      // features 64j..64j+63, then up features 64j..64j+63
      const int f0 = kb * 32;
      const float* g = gu + static_cast<long long>(m) * 2 * I + 2 * (f0 / kPairRows) * kPairRows + (f0 % kPairRows);
      const float* u = g + kPairRows;
      float h[32];
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        const float4 gv = __ldg(reinterpret_cast<const float4*>(g + i));
        const float4 uv = __ldg(reinterpret_cast<const float4*>(u + i));
        h[i] = silu_mul(gv.x, uv.x);
        h[i + 1] = silu_mul(gv.y, uv.y);
        h[i + 2] = silu_mul(gv.z, uv.z);
        h[i + 3] = silu_mul(gv.w, uv.w);
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(h[i]));
      s = ue8m0_from_amax(amax);
      const float inv = inv_scale_from_ue8m0(s);
      uint32_t packed[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        packed[i] = e4m3_code(h[4 * i] * inv) | (e4m3_code(h[4 * i + 1] * inv) << 8) |
                    (e4m3_code(h[4 * i + 2] * inv) << 16) | (e4m3_code(h[4 * i + 3] * inv) << 24);
      uint4* d = reinterpret_cast<uint4*>(hc + static_cast<long long>(m) * I + kb * 32);
      d[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
      d[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    }
    hs[tiled_sf_offset(m, kb, I / 128)] = static_cast<uint8_t>(s);
  }
}

cudaError_t launch_swiglu_quantize(const float* gu, int M, int I, uint8_t* hc, uint8_t* hs,
                                   cudaStream_t stream) {
  const int npad = (M + 15) / 16 * 16;
  const int total = npad * (I / 32);
  const int threads = 128;
  const int blocks = (total + threads - 1) / threads;
  swiglu_quantize_kernel<<<blocks, threads, 0, stream>>>(gu, M, npad, I, hc, hs);
  return cudaGetLastError();
}

// ======================================================================
// The persistent block-scaled GEMM / fused MLP kernel.
//
// Orientation: D[token, weight row] = X[token, :] . W[row, :]^T.  The tcgen05
// instruction's A operand is the activation tile (M = 128 token rows, npad of
// them real) and its B operand is a 256-row weight tile (N = 256).  A
// block-scaled MMA of M = 128, K = 32 takes the same time for every N up to
// 256, so this orientation moves 8 KB of weights per instruction; the
// accumulator holds one token per TMEM lane and one weight row per column.
//
// Roles (one block per SM, 8 warps):
//   warp 0 lane 0  weight producer: TMA of 256 x 128 B weight tiles and their
//                  two 512-byte scale tiles into a ring of stages
//   warp 1 lane 0  activation producer: waits until its operand exists (the
//                  grid-wide x quantisation, or the SwiGLU tile of the k-chunk)
//                  and TMA-loads the npad x 128 B activation tile
//   warp 2 lane 0  MMA issuer: tcgen05.cp of the three scale tiles into TMEM,
//                  four kind::mxf8f6f4 block-scaled MMAs (K = 32 each) per stage
//   warps 4-7      quantise x (grid slice, or each stage's tile when M <= 32),
//                  then run the epilogue of every accumulator
// ======================================================================
// Timeline stamps for profiling builds (compiled with -DFSOPS_TRACE).
#ifdef FSOPS_TRACE
#define FSOPS_STAMP(idx)                                                         \
  do {                                                                           \
    if (a.trace != nullptr) a.trace[blockIdx.x * 128 + (idx)] = globaltimer_ns(); \
  } while (0)
#define FSOPS_STAMP_IF(cond, idx) \
  do {                            \
    if (cond) FSOPS_STAMP(idx);   \
  } while (0)
#else
#define FSOPS_STAMP(idx) \
  do {                   \
  } while (0)
#define FSOPS_STAMP_IF(cond, idx) \
  do {                            \
  } while (0)
#endif


__device__ __forceinline__ long long range_begin(long long c, long long U, long long G) { return c * U / G; }
// Stream-K split of U units over G blocks in 32-bit arithmetic (U <= 2^18 and
// G <= 2^8 keep every product below 2^26): block c owns [c U / G, (c+1) U / G).
__device__ __forceinline__ uint32_t split_begin(uint32_t c, uint32_t U, uint32_t G) { return c * U / G; }
// The block whose range holds unit u.
__device__ __forceinline__ uint32_t split_owner(uint32_t u, uint32_t U, uint32_t G) {
  return ((u + 1) * G + U - 1) / U - 1;
}

// Tile-aligned split: the first block of tile t, ceil(t G / T).
__device__ __forceinline__ uint32_t aligned_first(uint32_t t, uint32_t T, uint32_t G) { return (t * G + T - 1) / T; }
// The blocks that add split sums into tile t of phase ph.
__device__ __forceinline__ uint32_t tile_owners(const PhaseArgs& ph, int t, uint32_t G) {
  const uint32_t T = static_cast<uint32_t>(ph.T), KS = static_cast<uint32_t>(ph.KS);
  if (ph.aligned) return aligned_first(t + 1, T, G) - aligned_first(t, T, G);
  const uint32_t U = T * KS;
  const uint32_t cf = split_owner(t * KS, U, G), cl = split_owner(t * KS + KS - 1, U, G);
  // with U >= G every block owns at least one unit; with U < G each owns at most one
  return U >= G ? cl - cf + 1 : KS;
}

// Walks the segments (tile, ks0, ks1) of one phase assigned to this block.
struct SegIter {
  uint32_t u, ue, KS;
  __device__ SegIter(const PhaseArgs& p, uint32_t G) : SegIter(p, G, blockIdx.x) {}
  // the segments of block c
  __device__ SegIter(const PhaseArgs& p, uint32_t G, uint32_t c) {
    KS = static_cast<uint32_t>(p.KS);
    if (p.aligned) {
      // block c works on tile t = floor(c T / G), as its j-th of n blocks
      const uint32_t T = static_cast<uint32_t>(p.T);
      const uint32_t t = c * T / G, f = aligned_first(t, T, G), n = aligned_first(t + 1, T, G) - f;
      const uint32_t j = c - f;
      u = t * KS + j * KS / n;
      ue = t * KS + (j + 1) * KS / n;
    } else if (p.whole_tiles) {
      u = c < static_cast<uint32_t>(p.T) ? c * KS : 0;
      ue = c < static_cast<uint32_t>(p.T) ? u + KS : 0;
    } else if (p.pairs) {
      // block c takes K half (c & 1) of tile c / 2
      const uint32_t tile = c >> 1, hk = KS / 2;
      u = tile < static_cast<uint32_t>(p.T) ? tile * KS + ((c & 1) ? hk : 0) : 0;
      ue = tile < static_cast<uint32_t>(p.T) ? tile * KS + ((c & 1) ? KS : hk) : 0;
    } else {
      const uint32_t U = static_cast<uint32_t>(p.T) * KS;
      u = split_begin(c, U, G);
      ue = split_begin(c + 1, U, G);
    }
  }
  __device__ bool next(int& t, int& ks0, int& ks1) {
    if (u >= ue) return false;
    const uint32_t tt = u / KS;
    t = static_cast<int>(tt);
    ks0 = static_cast<int>(u - tt * KS);
    ks1 = static_cast<int>(min(KS, ks0 + (ue - u)));
    u += ks1 - ks0;
    return true;
  }
};

// The block that holds unit (tile t, k-stage ks) of phase ph.
__device__ __forceinline__ uint32_t unit_owner(const PhaseArgs& ph, uint32_t t, uint32_t ks, uint32_t G) {
  const uint32_t T = static_cast<uint32_t>(ph.T), KS = static_cast<uint32_t>(ph.KS);
  if (ph.whole_tiles) return t;
  if (ph.pairs) return 2 * t + (ks >= KS / 2 ? 1u : 0u);
  if (ph.aligned) {
    const uint32_t f = aligned_first(t, T, G);
    return f + split_owner(ks, KS, aligned_first(t + 1, T, G) - f);
  }
  return split_owner(t * KS + ks, T * KS, G);
}
// Whether block c holds any unit of phase ph.
__device__ __forceinline__ bool has_units(const PhaseArgs& ph, uint32_t c, uint32_t G) {
  const SegIter it(ph, G, c);
  return it.ue > it.u;
}
// SwiGLU tiles of phase 0 per 128-feature chunk of h.
__device__ __forceinline__ uint32_t tiles_per_chunk(const KernelArgs& a) {
  return (a.ph[0].tile_rows == 128 ? 2u : 1u) * (a.ph[0].pairs ? 2u : 1u);
}
// After SwiGLU tile t of phase 0 (h features [t R / 2, (t + 1) R / 2), R its
// rows) is written and ordered by a barrier: epilogue thread et tells the
// blocks whose down-projection stages read its 128-feature chunk.
__device__ __forceinline__ void publish_h(const KernelArgs& a, int t, int et, uint32_t G) {
  const PhaseArgs& p1 = a.ph[1];
  const uint32_t c = static_cast<uint32_t>((t * a.ph[0].tile_rows) >> 8);
  for (int t1 = et; t1 < p1.T; t1 += 128) red_add_release_gpu(a.hflags + unit_owner(p1, t1, c, G), 1u);
}

// ----------------------------------------------------------------------------
// Epilogue pieces.  A tile's result row for token r is 256 fp32 values (128
// when the weight matrix ends half way through the tile).
// ----------------------------------------------------------------------------

// Scale byte of token r for the 32 intermediate features from f0, in the tiled
// scale layout (512-byte tiles of 128 features).
__device__ __forceinline__ uint32_t hq_sf_offset(int r, int f0) {
  return static_cast<uint32_t>((f0 >> 7) * 512 + (r & 31) * 16 + (r >> 5) * 4 + ((f0 >> 5) & 3));
}
// Accumulator column of the gate sums of 32-block b of a gate/up tile; the up
// sums of the same features sit kPairRows columns further.
__device__ __forceinline__ int gate_col(int b) { return ((b >> 1) << 7) + ((b & 1) << 5); }

// SwiGLU + requantisation of the 32 intermediate features f0.. of token r:
// g[i], u[i] are the gate and up sums of those features.
__device__ __forceinline__ void swiglu_block(const KernelArgs& a, int f0, int r, const float* g, const float* u) {
  float h[32];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    h[i] = silu_mul(g[i], u[i]);
    amax = fmaxf(amax, fabsf(h[i]));
  }
  const uint32_t s = ue8m0_from_amax(amax);
  const float inv = inv_scale_from_ue8m0(s);
  uint32_t pk[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    pk[i] = e4m3_code(h[4 * i] * inv) | (e4m3_code(h[4 * i + 1] * inv) << 8) |
            (e4m3_code(h[4 * i + 2] * inv) << 16) | (e4m3_code(h[4 * i + 3] * inv) << 24);
  uint4* dst = reinterpret_cast<uint4*>(a.hq_codes + static_cast<long long>(r) * a.I + f0);
  dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
  a.hq_sf[hq_sf_offset(r, f0)] = static_cast<uint8_t>(s);
}

// Plain output: 8 consecutive columns c..c+7 of token r.
__device__ __forceinline__ void store8(const KernelArgs& a, const PhaseArgs& p, int r, long long col,
                                       const float* v, bool have_res = false, uint4 res = uint4{}) {
  const long long o = static_cast<long long>(r) * p.out_ld + col;
  if (a.residual != nullptr) {  // y = residual + the sums, rounded once (res: the 8 values, if already loaded)
    const uint4 rv = have_res ? res : *reinterpret_cast<const uint4*>(a.residual + o);
    const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
    float s[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      s[2 * i] = v[2 * i] + bf16_lo(rw[i]);
      s[2 * i + 1] = v[2 * i + 1] + bf16_hi(rw[i]);
    }
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(s[2 * i], s[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&b2);
    }
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + o) = make_uint4(w[0], w[1], w[2], w[3]);
    return;
  }
  if (a.out_f32) {
    float4* d = reinterpret_cast<float4*>(static_cast<float*>(a.out) + o);
    d[0] = make_float4(v[0], v[1], v[2], v[3]);
    d[1] = make_float4(v[4], v[5], v[6], v[7]);
  } else {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&b2);
    }
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + o) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Epilogue over a tile staged in shared memory (M <= 32): stg[r * kStageLd + c].
// The code runs once per tile, mostly cold in the instruction cache, so its
// loops are kept rolled and free of divisions.
//   SwiGLU: each 32-block (token r, features 32 b ..) is shared by four
//   adjacent threads, 8 features each; the block's |max| is combined with
//   two shuffles.  Plain: 8 columns per item.
// SwiGLU: 32-blocks [b0, b0 + nb) of the tile, nb = 2 or 4.
__device__ __forceinline__ void finish_staged(const KernelArgs& a, const PhaseArgs& ph, int t, int ncols,
                                              const float* stg, int et, int b0, int nb) {
  if (ph.epi == kEpiSwiGLU) {
    const int lgb = nb == 4 ? 4 : 3;  // log2(tasks per token): nb blocks x 4 parts
    const int tasks = a.M << lgb;
    const int f_tile = t * (ph.tile_rows >> 1);
#pragma unroll 1
    for (int q0 = 0; q0 < tasks; q0 += 128) {
      const int q = q0 + et;
      const int r = q >> lgb, b = b0 + ((q >> 2) & (nb - 1)), part = q & 3;
      const int rr = r < a.M ? r : a.M - 1;
      const float4* gp = reinterpret_cast<const float4*>(stg + rr * kStageLd + gate_col(b) + 8 * part);
      const float4* up = reinterpret_cast<const float4*>(stg + rr * kStageLd + gate_col(b) + kPairRows + 8 * part);
      const float4 g0 = gp[0], g1 = gp[1], u0 = up[0], u1 = up[1];
      float h[8];
      h[0] = silu_mul(g0.x, u0.x); h[1] = silu_mul(g0.y, u0.y); h[2] = silu_mul(g0.z, u0.z); h[3] = silu_mul(g0.w, u0.w);
      h[4] = silu_mul(g1.x, u1.x); h[5] = silu_mul(g1.y, u1.y); h[6] = silu_mul(g1.z, u1.z); h[7] = silu_mul(g1.w, u1.w);
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(h[i]));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      const uint32_t sc = ue8m0_from_amax(amax);
      const float inv = inv_scale_from_ue8m0(sc);
      const uint32_t lo = e4m3x4_code(h[0] * inv, h[1] * inv, h[2] * inv, h[3] * inv);
      const uint32_t hi = e4m3x4_code(h[4] * inv, h[5] * inv, h[6] * inv, h[7] * inv);
      if (r < a.M) {
        const int f0 = f_tile + 32 * b;
        *reinterpret_cast<uint2*>(a.hq_codes + static_cast<long long>(r) * a.I + f0 + 8 * part) = make_uint2(lo, hi);
        if (part == 0) a.hq_sf[hq_sf_offset(r, f0)] = static_cast<uint8_t>(sc);
      }
    }
  } else {
    const int lg = ncols == 256 ? 5 : 4;  // log2(items per row), 8 columns per item
    const int items = a.M << lg;
#pragma unroll 1
    for (int item = et; item < items; item += 128) {
      const int r = item >> lg, c = (item & ((1 << lg) - 1)) * 8;
      store8(a, ph, r, static_cast<long long>(t) * ph.tile_rows + c, stg + r * kStageLd + c);
    }
  }
}

// Local activation tiles (M <= 16): block b of a stage is the 32-element block
// (row b / 4, block b % 4) of a 128-wide k-chunk of x.  Quantise it into the
// stage's activation tile (128-byte swizzled rows, as the TMA would have
// written them) and its scale tile; rows >= M get zeros.
// gam != null: the block is of RMSNorm(x) * gamma (x * rn * gamma, gam the
// block's 32 gains, rn the row's 1 / rms).
__device__ __forceinline__ void store_x_block(const KernelArgs& a, uint8_t* st, int b, const uint4 (&raw)[4],
                                              const uint16_t* gam = nullptr, float rn = 1.0f) {
  const int r = b >> 2, j = b & 3;
  uint32_t s = 0;
  uint4 c0 = make_uint4(0, 0, 0, 0), c1 = c0;
  if (r < a.M) {
    uint32_t pk[8];
    s = gam != nullptr ? quantize_block_pack_norm(raw, gam, rn, pk) : quantize_block_pack(raw, pk);
    c0 = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    c1 = make_uint4(pk[4], pk[5], pk[6], pk[7]);
  }
  uint8_t* row = st + r * 128;
  *reinterpret_cast<uint4*>(row + (((2 * j) ^ (r & 7)) << 4)) = c0;
  *reinterpret_cast<uint4*>(row + (((2 * j + 1) ^ (r & 7)) << 4)) = c1;
  st[stage_off_sfx(a.npad) + (r & 31) * 16 + (r >> 5) * 4 + j] = static_cast<uint8_t>(s);
}

// 16 accumulator columns c0.. of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16f(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  tmem_ld16(taddr, r);
  tmem_ld_wait();
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// Split tile t of a plain-output phase (M > 32): once all `owners` blocks
// have added their sums, this owner writes the token rows [M a / n, M (a+1) / n)
// of the tile (a = its arrival order, n = owners) and clears them in the
// accumulator for the next launch.  pd = (t, arrival, owners, ncols).
__device__ __noinline__ bool finish_slice(const KernelArgs& a, const PhaseArgs& ph, const Ctx& cx, int4 pd, int et,
                                          volatile int* bcast) {
  const int t = pd.x, arrival = pd.y, owners = pd.z, ncols = pd.w;
  if (et == 0) *bcast = wait_counters(cx, ph.tile_cnt + t, 1, static_cast<uint32_t>(owners), kSiteTileSum) ? 1 : 0;
  epi_bar();
  const bool okw = *bcast != 0;
  epi_bar();
  if (!okw) return false;
  // a second count: the owner that brings it to 2 owners clears the counter,
  // after every owner's wait has seen it complete
  uint32_t seen = 0;
  if (et == 0) seen = atom_add_acq_rel_gpu(ph.tile_cnt + t, 1u);
  float* accg = ph.accum + static_cast<long long>(t) * a.M * kTileRows;
  const int r0 = a.M * arrival / owners, r1 = a.M * (arrival + 1) / owners;
  const int lg = ncols == 256 ? 5 : 4;  // log2(8-column items per row)
  const int items = (r1 - r0) << lg;
  // each pass issues its sums' loads (and the residual's) together; each
  // thread clears what it read right after the loads (its stores follow its
  // own loads of the same words), rows [r0, r1) x columns [0, ncols)
#pragma unroll 1
  for (int i0 = 0; i0 < items; i0 += 4 * 128) {
    float4 v[4][2];
    uint4 rv[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = i0 + et + 128 * j;
      if (i < items) {
        const float4* src = reinterpret_cast<const float4*>(accg + (r0 + (i >> lg)) * kTileRows + (i & ((1 << lg) - 1)) * 8);
        v[j][0] = __ldcg(src);
        v[j][1] = __ldcg(src + 1);
        if (a.residual != nullptr)
          rv[j] = __ldcg(reinterpret_cast<const uint4*>(
              a.residual + static_cast<long long>(r0 + (i >> lg)) * ph.out_ld +
              static_cast<long long>(t) * ph.tile_rows + (i & ((1 << lg) - 1)) * 8));
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = i0 + et + 128 * j;
      if (i < items) {
        float4* dst = const_cast<float4*>(reinterpret_cast<const float4*>(accg + (r0 + (i >> lg)) * kTileRows +
                                                                            (i & ((1 << lg) - 1)) * 8));
        __stcg(dst, make_float4(0.f, 0.f, 0.f, 0.f));
        __stcg(dst + 1, make_float4(0.f, 0.f, 0.f, 0.f));
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = i0 + et + 128 * j;
      if (i < items) {
        const float w[8] = {v[j][0].x, v[j][0].y, v[j][0].z, v[j][0].w, v[j][1].x, v[j][1].y, v[j][1].z, v[j][1].w};
        store8(a, ph, r0 + (i >> lg), static_cast<long long>(t) * ph.tile_rows + (i & ((1 << lg) - 1)) * 8, w,
               a.residual != nullptr, rv[j]);
      }
    }
  }
  if (et == 0 && seen + 1 == 2u * static_cast<uint32_t>(owners)) ph.tile_cnt[t] = 0u;
  return true;
}

// STAGED: the instance for M <= 32 (accumulators staged through shared
// memory, local x quantisation possible); the other serves M > 32.  Each
// instance holds only its own epilogue paths, which keeps the run-once
// epilogue code of a call compact for the instruction caches.
template <bool STAGED>
__global__ void __launch_bounds__(kThreads, 1) mx_persistent_kernel(const __grid_constant__ KernelArgs a) {
  const bool local_xq = STAGED && a.local_xq != 0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align(smem_raw, 1024);
  const int S = a.nstages;
  float* stg = reinterpret_cast<float*>(smem + static_cast<size_t>(S) * a.stage_bytes);
  uint8_t* xring = reinterpret_cast<uint8_t*>(stg) + (STAGED ? stg_bytes_for(a.npad) : 0u);
  uint8_t* ctl_smem = xring + (local_xq ? xring_bytes_for(a.npad) : 0u);
  uint64_t* full_w = reinterpret_cast<uint64_t*>(ctl_smem);
  uint64_t* full_a = full_w + kMaxStages;
  uint64_t* empty = full_a + kMaxStages;
  uint64_t* acc_full = empty + kMaxStages;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  uint64_t* x_issued = drain + 1;
  uint64_t* x_full = x_issued + 1;          // [kMaxXSlots] bf16 x tile landed (local_xq)
  uint64_t* peer_ready = x_full + kMaxXSlots;  // the other block of the pair has pushed its sums of this block's half
  uint64_t* peer_free = peer_ready + 1;          // ... may push them (the receiving buffer is free)
  uint64_t* peer_done = peer_free + 1;           // ... has received this block's push
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(peer_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* bcast = reinterpret_cast<volatile int*>(tmem_slot + 2);
  // 0 until this block's activations are available (x quantised grid-wide,
  // or the first SwiGLU tiles published): until then the weight producer
  // keeps only prime_inflight loads in flight, so that the x quantisation's
  // own memory traffic is not queued behind the whole grid's weight stream
  volatile int* flowing = reinterpret_cast<volatile int*>(tmem_slot + 3);
  float* rnorm = reinterpret_cast<float*>(tmem_slot + 4);  // [kMmaM] 1 / rms of the rows this block quantises

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long G = gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_w[s], 1);
      mbar_init(&full_a[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 128);
    mbar_init(drain, 1);
    mbar_init(x_issued, 128);
    for (int i = 0; i < kMaxXSlots; ++i) mbar_init(&x_full[i], 1);
    mbar_init(peer_ready, 1);
    mbar_init(peer_free, 1);
    mbar_init(peer_done, 1);
    *abort_flag = 0;
    *flowing = (a.x != nullptr && !local_xq) ? 0 : 1;
    mbar_fence_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    for (int p = 0; p < a.nphases; ++p) {
      tma_prefetch_desc(&a.tm_w[p]);
      tma_prefetch_desc(&a.tm_act[p]);
    }
    if (local_xq) tma_prefetch_desc(&a.tm_x);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the pair's barriers are initialised before either block arrives remotely
  if (a.cluster_pairs) cluster_sync_all();
  // the next kernel on the stream may be scheduled as this grid's blocks leave
  griddep_launch_dependents();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) FSOPS_STAMP(0);

  Ctx cx;
  cx.abort_flag = abort_flag;
  cx.status = a.ctl + kCtlStatus;
  cx.timeout_ns = a.timeout_ns;

  const int npad = a.npad;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ weight producer
    const uint64_t pol = l2_policy_evict_first();
    uint32_t issued_mask = 0, issued_parity = 0;
    int stage = 0;
    uint32_t round = 0;
    // issuing waits until the load `max_inflight` stages back has landed
    int lag_stage = 0;
    uint32_t lag_round = 0, n_issued = 0, n_landed = 0;
    bool ok = true;
    // let the epilogue warps' loads of x enter the memory system first
    if (a.x != nullptr && !local_xq && !a.early_w) ok = wait_mbar(cx, x_issued, 0, kSiteEmpty);
    for (int p = 0; p < a.nphases && ok; ++p) {
      const PhaseArgs& ph = a.ph[p];
      SegIter it(ph, static_cast<uint32_t>(G));
      int t, ks0, ks1;
      while (ok && it.next(t, ks0, ks1)) {
        // a 256-row tile holds two 128-row scale tiles unless the matrix ends half way
        const bool v1 = ph.tile_rows == 256 && t * 256 + 128 < ph.rows;
        const uint32_t wbytes = static_cast<uint32_t>(ph.tile_rows) * kTileK;
        for (int ks = ks0; ks < ks1; ++ks) {
          if (!wait_mbar(cx, &empty[stage], (round & 1u) ^ 1u, kSiteEmpty)) { ok = false; break; }
          for (;;) {
            const uint32_t cap = *flowing ? static_cast<uint32_t>(a.max_inflight)
                                          : static_cast<uint32_t>(min(a.max_inflight, a.prime_inflight));
            if (n_issued - n_landed < cap) break;
            if (!wait_mbar(cx, &full_w[lag_stage], lag_round & 1u, kSiteFullW)) { ok = false; break; }
            ++n_landed;
            if (++lag_stage == S) { lag_stage = 0; ++lag_round; }
          }
          if (!ok) break;
          FSOPS_STAMP_IF(n_issued < 16, 40 + n_issued);
          ++n_issued;
          uint8_t* st = smem + static_cast<size_t>(stage) * a.stage_bytes;
          mbar_arrive_expect_tx(&full_w[stage], wbytes + (v1 ? 1024u : 512u));
          tma_load_2d(st + stage_off_w(npad), &a.tm_w[p], &full_w[stage], ks * kTileK, t * ph.tile_rows, pol);
          const uint8_t* sfw = ph.sf_w + (static_cast<size_t>(t * (ph.tile_rows >> 7)) * ph.KS + ks) * 512;
          bulk_load(st + stage_off_sfw(npad), sfw, 512, &full_w[stage], pol);
          if (v1) bulk_load(st + stage_off_sfw(npad) + 512, sfw + static_cast<size_t>(ph.KS) * 512, 512, &full_w[stage], pol);
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | ((round & 1u) << stage);
          if (++stage == S) { stage = 0; ++round; }
        }
      }
    }
    if (!ok) *abort_flag = 1;
    for (int s = 0; s < S; ++s)
      if (issued_mask & (1u << s)) drain_mbar(&full_w[s], (issued_parity >> s) & 1u, 200000000ull);
  } else if (warp == 1) {
    // ------------------------------------------------ activation producer
    // x, the quantised activations and the readiness counters may be in use by
    // the previous kernel on the stream until it completes (the launch lets
    // this grid start while it finishes); the weights never are, so the
    // weight producer starts at once.
    griddep_wait();
    if (lane == 0) FSOPS_STAMP(64);
    // Lane 0 issues the TMA loads.  With local_xq phase 0's activation tiles
    // are quantised by the epilogue warps, which fill those stages themselves.
    const uint64_t pol = l2_policy_evict_last();
    uint32_t issued_mask = 0, issued_parity = 0;
    int stage = 0;
    uint32_t round = 0;
    bool ok = true, x_ready = false, h_seen = false;
    for (int p = 0; p < a.nphases && ok; ++p) {
      const PhaseArgs& ph = a.ph[p];
      SegIter it(ph, static_cast<uint32_t>(G));
      int t, ks0, ks1;
      while (ok && it.next(t, ks0, ks1)) {
        if (p == 0 && local_xq) {
          for (int ks = ks0; ks < ks1; ++ks)
            if (++stage == S) { stage = 0; ++round; }
          continue;
        }
        if (lane != 0) {
          for (int ks = ks0; ks < ks1; ++ks)
            if (++stage == S) { stage = 0; ++round; }
          continue;
        }
        for (int ks = ks0; ks < ks1; ++ks) {
          if (!wait_mbar(cx, &empty[stage], (round & 1u) ^ 1u, kSiteEmpty)) { ok = false; break; }
          if (ph.dep == kDepXReady && !x_ready) {
            // every block's slice of x
            if (!wait_counters(cx, a.xready + blockIdx.x, 1, static_cast<uint32_t>(G) + a.extra_xready,
                               kSiteXReady)) {
              ok = false;
              break;
            }
            a.xready[blockIdx.x] = 0u;  // complete: no further adds this launch
            fence_proxy_async_global();
            x_ready = true;
            *flowing = 1;
            FSOPS_STAMP(2);
          } else if (ph.dep == kDepHFlags && !h_seen) {
            // the SwiGLU tiles of every 128-feature chunk of every stage of this phase
            const SegIter all(ph, static_cast<uint32_t>(G));
            const uint32_t want = (all.ue - all.u) * tiles_per_chunk(a) + a.extra_xready;
            if (!wait_counters(cx, a.hflags + blockIdx.x, 1, want, kSiteHFlag)) {
              ok = false;
              break;
            }
            a.hflags[blockIdx.x] = 0u;  // complete: no further adds this launch
            fence_proxy_async_global();
            FSOPS_STAMP(5);
            h_seen = true;
            *flowing = 1;
            FSOPS_STAMP(6);
          }
          uint8_t* st = smem + static_cast<size_t>(stage) * a.stage_bytes;
          mbar_arrive_expect_tx(&full_a[stage], 128u * npad + 512u);
          tma_load_2d(st, &a.tm_act[p], &full_a[stage], ks * kTileK, 0, pol);
          bulk_load(st + stage_off_sfx(npad), ph.sf_act + static_cast<size_t>(ks) * 512, 512, &full_a[stage], pol);
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | ((round & 1u) << stage);
          if (++stage == S) { stage = 0; ++round; }
        }
      }
    }
    if (!ok) *abort_flag = 1;
    if (lane == 0) {
      for (int s = 0; s < S; ++s)
        if (issued_mask & (1u << s)) drain_mbar(&full_a[s], (issued_parity >> s) & 1u, 200000000ull);
    }
  } else if (warp == 2 && lane == 0) {
    // ------------------------------------------------ MMA issuer
    int stage = 0;
    uint32_t round = 0, acc_round = 0, n_mma = 0;
    bool ok = true;
    const uint32_t sf_base = tmem + kAccCols;
    for (int p = 0; p < a.nphases && ok; ++p) {
      const PhaseArgs& ph = a.ph[p];
      SegIter it(ph, static_cast<uint32_t>(G));
      int t, ks0, ks1;
      while (ok && it.next(t, ks0, ks1)) {
        const bool v1 = ph.tile_rows == 256 && t * 256 + 128 < ph.rows;
        const uint32_t idesc0 = idesc_mxf8_e4m3(v1 ? 256u : 128u, 0, 0);
        if (!wait_mbar(cx, acc_empty, (acc_round & 1u) ^ 1u, kSiteAccEmpty)) { ok = false; break; }
        tc_fence_after();
        for (int ks = ks0; ks < ks1; ++ks) {
          if (!wait_mbar(cx, &full_w[stage], round & 1u, kSiteFullW) ||
              !wait_mbar(cx, &full_a[stage], round & 1u, kSiteFullA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          FSOPS_STAMP_IF(n_mma < 24, 16 + n_mma);
          ++n_mma;
          uint8_t* st = smem + static_cast<size_t>(stage) * a.stage_bytes;
          const uint32_t sfc = sf_base + kSfColsPerStage * stage;
          // A scales (tokens): lanes = row % 32, columns sfc + row / 32.
          // B scales (weight rows n): lanes n % 32, columns sfc + 4 + n / 32.
          tc_cp_32x128b_warpx4(sfc, smem_desc(smem_u32(st + stage_off_sfx(npad)), 0, 128, kSwizzleNone));
          tc_cp_32x128b_warpx4(sfc + 4, smem_desc(smem_u32(st + stage_off_sfw(npad)), 0, 128, kSwizzleNone));
          if (v1) tc_cp_32x128b_warpx4(sfc + 8, smem_desc(smem_u32(st + stage_off_sfw(npad) + 512), 0, 128, kSwizzleNone));
          const uint32_t sx = smem_u32(st);
          const uint32_t sw = smem_u32(st + stage_off_w(npad));
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            // scale byte k of each 32-bit TMEM scale word belongs to K-block k of the stage
            const uint32_t idesc = idesc0 | (static_cast<uint32_t>(k) << 4) | (static_cast<uint32_t>(k) << 29);
            tc_mma_mxf8(tmem, smem_desc(sx + 32 * k, 16, 1024, kSwizzle128B),
                        smem_desc(sw + 32 * k, 16, 1024, kSwizzle128B), idesc, sfc, sfc + 4,
                        (ks > ks0 || k > 0) ? 1u : 0u);
          }
          tc_commit(&empty[stage]);
          if (++stage == S) { stage = 0; ++round; }
        }
        if (!ok) break;
        tc_commit(acc_full);
        ++acc_round;
        FSOPS_STAMP(p == 0 ? 7 : 11);
      }
    }
    if (!ok) *abort_flag = 1;
    // wait until every tcgen05 operation issued by this thread has completed
    tc_commit(drain);
    drain_mbar(drain, 0, 200000000ull);
  } else if (warp >= 4) {
    // ------------------------------------------------ epilogue warps
    const int et = threadIdx.x - 128;  // token row of the accumulator (TMEM lane)
    const int ew = et >> 5;
    const uint32_t pair_h = blockIdx.x & 1u, pair_peer = pair_h ^ 1u;  // cluster pairs: rank, partner
    // bulk pair exchange (thread et == 0): this block's x ring armed to
    // receive, the partner's sums received, this block's sums sent
    bool pair_armed = false, pair_received = false, pair_sent = false;
    griddep_wait();  // x, the workspace and y may be in use by the previous kernel until here
    if (et == 0) FSOPS_STAMP(65);
    // (1) grid-wide: quantise this block's slice of x, the 32-blocks [b0, b1)
    // of the row-major [npad, H/32] block grid (rows >= M only get a zero scale)
    if (a.x != nullptr && !local_xq) {
      const int nbk = a.H / 32;
      const long long NB = static_cast<long long>(npad) * nbk;
      const long long b0 = range_begin(blockIdx.x, NB, G), b1 = range_begin(blockIdx.x + 1, NB, G);
      const bool norm = a.gamma != nullptr;
      long long b = b0 + et;
      uint4 raw[4], gv[4];
      bool have = false;
      // the first block's x (and gamma) loads go out before the norms' row
      // loads and the weight stream, so that both round trips overlap
      if (b < b1) {
        const int m = static_cast<int>(b / nbk), kb = static_cast<int>(b % nbk);
        if (m < a.M) {
          const uint4* src = reinterpret_cast<const uint4*>(a.x + static_cast<long long>(m) * a.H + kb * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) raw[i] = __ldcg(src + i);
          if (norm) {
#pragma unroll
            for (int i = 0; i < 4; ++i) gv[i] = __ldg(reinterpret_cast<const uint4*>(a.gamma + kb * 32) + i);
          }
          have = true;
        }
      }
      mbar_arrive(x_issued);
      if (norm && b1 > b0) {
        // RMSNorm: 1 / rms of every row the slice touches, over the whole row
        // (one warp per row in turn)
        const int m0 = static_cast<int>(b0 / nbk), m1 = static_cast<int>((b1 - 1) / nbk);
        for (int m = m0 + ew; m <= m1 && m < a.M; m += 4) {
          const float rn = row_rnorm(a.x + static_cast<long long>(m) * a.H, a.H, a.eps, lane);
          if (lane == 0) rnorm[m] = rn;
        }
        epi_bar();
      }
      for (; b < b1; b += 128) {
        const int m = static_cast<int>(b / nbk), kb = static_cast<int>(b % nbk);
        uint32_t s = 0;
        if (m < a.M) {
          if (!have) {
            const uint4* src = reinterpret_cast<const uint4*>(a.x + static_cast<long long>(m) * a.H + kb * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) raw[i] = __ldcg(src + i);
            if (norm) {
#pragma unroll
              for (int i = 0; i < 4; ++i) gv[i] = __ldg(reinterpret_cast<const uint4*>(a.gamma + kb * 32) + i);
            }
          }
          if (norm) {
            uint32_t pk[8];
            s = quantize_block_pack_norm(raw, gv, rnorm[m], pk);
            uint4* d = reinterpret_cast<uint4*>(a.xq_codes + static_cast<long long>(m) * a.H + kb * 32);
            d[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            d[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          } else {
            s = quantize_block_regs(raw, a.xq_codes + static_cast<long long>(m) * a.H + kb * 32);
          }
        }
        have = false;
        a.xq_sf[(kb >> 2) * 512 + (m & 31) * 16 + (m >> 5) * 4 + (kb & 3)] = static_cast<uint8_t>(s);
      }
      if (et == 0) FSOPS_STAMP(63);
      fence_proxy_async_global();
      epi_bar();
      // to every block whose first phase reads x (each waits for all G
      // slices): one fence orders the whole slice (every epilogue thread's
      // stores, through the barrier) before this thread's relaxed adds
      if (et < static_cast<int>(G)) fence_acq_rel_gpu();
      for (int c = et; c < static_cast<int>(G); c += 128)
        if (has_units(a.ph[0], static_cast<uint32_t>(c), static_cast<uint32_t>(G)))
          red_add_relaxed_gpu(a.xready + c, 1u);
      if (et == 0) FSOPS_STAMP(1);
    }
    // (2) accumulators
    uint32_t acc_round = 0;
    bool ok = true;
    int4 pend[kMaxPend];  // split tiles to finish at the end of the phase: (t, arrival, owners, ncols)
    int npend = 0;
    const uint32_t tlane = tmem + (static_cast<uint32_t>(ew * 32) << 16);
    // With local_xq the epilogue warps fill phase 0's activation stages: two
    // stages at a time, stage c by warp pair c % 2 (warps 4 + 2 (c % 2) and
    // the next; thread pt of the pair quantises 32-element block pt), so a
    // stage reaches the tensor core soon after its x tile lands and the pairs
    // together keep ahead of the MMAs.  The block's phase-0 stages are its
    // consecutive units u0, u0 + 1, ... (stage c: ring position c % S,
    // k-stage (u0 + c) % KS); their bf16 x tiles stream through a four-slot
    // ring (tile c in slot c % 4: the pair's two slots), issued by the pair's
    // first thread two tiles ahead.  Before the accumulator of a segment
    // ending at stage e is awaited, every stage below e + S is filled: those
    // need no MMA of a later segment (whose accumulator is not yet free) to
    // release their ring position, and the next segment's first stages are
    // ready while this one's epilogue runs.
    uint32_t xu0 = 0, xn0 = 0, xks = 1;
    if (local_xq) {
      SegIter it0(a.ph[0], static_cast<uint32_t>(G));
      xu0 = it0.u;
      xn0 = it0.ue - it0.u;
      xks = it0.KS;
    }
    const uint32_t xq = static_cast<uint32_t>(ew >> 1);  // this warp's pair
    const int pt = et & 63;                              // thread of the pair
    uint32_t xc = xq;                                    // next stage of the pair
    uint32_t xi = xq;                                    // next tile the pair issues
    const uint64_t x_pol = l2_policy_evict_last();
    auto issue_x = [&]() {  // the pair's first thread: tile xi into slot xi % 4
      const uint32_t slot = xi & 3u;
      mbar_arrive_expect_tx(&x_full[slot], 256u * npad);
      tma_load_2d(xring + slot * 256 * npad, &a.tm_x, &x_full[slot], static_cast<int>((xu0 + xi) % xks) * kTileK, 0,
                  x_pol);
      xi += 2;
    };
    if (pt == 0)
      while (xi < xn0 && xi < xq + 4) issue_x();
    if (local_xq && a.gamma != nullptr) {
      // RMSNorm: 1 / rms of every row (M <= 16), each over all of H, before
      // any stage is quantised.  Warp ew takes rows ew, ew + 4, ew + 8 and
      // ew + 12 together (the loads of all four in flight); each row's sum
      // runs in the order of row_rnorm, so every path gets the same norms.
      // (five of each row's 16-byte loads in flight per lane: 20 in all)
      float ss[4] = {0.f, 0.f, 0.f, 0.f};
      const int n8 = a.H / 8;
      for (int i0 = lane; i0 < n8; i0 += 5 * 32) {
        uint4 v[5][4];
#pragma unroll
        for (int u = 0; u < 5; ++u)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (ew + 4 * k < a.M && i0 + 32 * u < n8)
              v[u][k] = __ldg(reinterpret_cast<const uint4*>(a.x + static_cast<long long>(ew + 4 * k) * a.H) + i0 + 32 * u);
#pragma unroll
        for (int u = 0; u < 5; ++u)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if (ew + 4 * k >= a.M || i0 + 32 * u >= n8) continue;
            const uint32_t w[4] = {v[u][k].x, v[u][k].y, v[u][k].z, v[u][k].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float lo = bf16_lo(w[q]), hi = bf16_hi(w[q]);
              ss[k] = fmaf(lo, lo, fmaf(hi, hi, ss[k]));
            }
          }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
#pragma unroll
        for (int o = 16; o; o >>= 1) ss[k] += __shfl_xor_sync(0xFFFFFFFFu, ss[k], o);
        if (lane == 0 && ew + 4 * k < a.M) rnorm[ew + 4 * k] = rsqrtf(ss[k] / static_cast<float>(a.H) + a.eps);
      }
      epi_bar();  // every row's norm is in rnorm before any stage is quantised
    }
    auto quantize_upto = [&](uint32_t L) -> bool {
      for (; xc < L; xc += 2) {
        const uint32_t c = xc, slot = c & 3u;
        const int stage = static_cast<int>(c % static_cast<uint32_t>(S));
        const uint32_t round = c / static_cast<uint32_t>(S);
        if (!pair_and(xq, wait_mbar(cx, &x_full[slot], (c >> 2) & 1u, kSiteFullA) &&
                              wait_mbar(cx, &empty[stage], (round & 1u) ^ 1u, kSiteEmpty)))
          return false;
        if (pt == 0) FSOPS_STAMP_IF(c < 6, 66 + c);
        uint8_t* st = smem + static_cast<size_t>(stage) * a.stage_bytes;
        if (pt < 4 * npad) {
          const uint4* src = reinterpret_cast<const uint4*>(xring + slot * 256 * npad + (pt >> 2) * 256 + (pt & 3) * 64);
          uint4 raw[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) raw[k] = src[k];
          if (a.gamma != nullptr) {
            const int ksx = static_cast<int>((xu0 + c) % xks);
            store_x_block(a, st, pt, raw, a.gamma + ksx * kTileK + (pt & 3) * 32,
                          (pt >> 2) < a.M ? rnorm[pt >> 2] : 1.0f);
          } else {
            store_x_block(a, st, pt, raw);
          }
        }
        fence_proxy_async_shared();
        pair_bar(xq);  // the stage is filled and the slot read by both warps
        if (pt == 0) {
          mbar_arrive(&full_a[stage]);
          if (xi < xn0) issue_x();
          FSOPS_STAMP_IF(c < 6, 72 + c);
        }
      }
      return true;
    };
    uint32_t xseg_end = 0;  // phase-0 stages up to the end of the current segment
    for (int p = 0; p < a.nphases && ok; ++p) {
      const PhaseArgs& ph = a.ph[p];
      SegIter it(ph, static_cast<uint32_t>(G));
      int t, ks0, ks1;
      while (ok && it.next(t, ks0, ks1)) {
        if (p == 0 && local_xq) {
          xseg_end += static_cast<uint32_t>(ks1 - ks0);
          if (!epi_and(quantize_upto(min(xn0, xseg_end + static_cast<uint32_t>(S))))) { ok = false; break; }
          if (ph.pairs && et == 0) {
            // every x tile is consumed: the x ring receives the partner's sums
            mbar_arrive_expect_tx(peer_ready, 512u * a.M);
            mbar_arrive_remote(mapa_shared(peer_free, pair_peer));
            pair_armed = true;
          }
        }
        if (!epi_and(wait_mbar(cx, acc_full, acc_round & 1u, kSiteAccFull))) { ok = false; break; }
        ++acc_round;
        tc_fence_after();
        if (et == 0) FSOPS_STAMP(p == 0 ? 3 : 8);
        const bool whole = (ks0 == 0 && ks1 == ph.KS);
        const int ncols = (ph.tile_rows == 256 && t * 256 + 128 < ph.rows) ? 256 : 128;
        float* accg = ph.accum + static_cast<long long>(t) * a.M * kTileRows;  // M * 256 floats
        bool send_ok = true;  // the bulk pair exchange could send (thread et == 0)
        if (STAGED) {
          // M <= 32: warp 4 copies TMEM lanes 0..31 to shared memory (four
          // loads in flight per wait) and the accumulator is released at once;
          // all four warps share the rest.  Split tiles add their rows into a
          // row-major [M][256] accumulator, four columns per reduction.
          // A cluster pair (ph.pairs) splits the tile's K range: each block
          // keeps the sums of its own half of the columns, [128 h, 128 h + 128),
          // and pushes the other half into the partner's stg, at the columns of
          // its own half there (which the partner does not use), then arrives
          // on the partner's peer_ready.
          // With local_xq (M <= 16) the push is one bulk copy instead: warp 4
          // writes the partner's half as contiguous 512-byte rows into the
          // first half of this block's x ring, and one thread copies them into
          // the second half of the partner's (both rings are free once their
          // block's x stages are all filled).
          const bool push_st = ph.pairs && !local_xq, push_bulk = ph.pairs && local_xq;
          if (ew == 0) {
            const uint32_t pstg = push_st ? mapa_shared(stg, pair_peer) : 0u;
#pragma unroll 1
            for (int c0 = 0; c0 < ncols; c0 += 128) {
              // 128 columns per wait (eight loads in flight)
              uint32_t v[8][16];
#pragma unroll
              for (int q = 0; q < 8; ++q) tmem_ld16(tlane + c0 + 16 * q, v[q]);
              tmem_ld_wait();
              if (lane == 0 && p == 0) FSOPS_STAMP_IF(c0 < 256, 83 + (c0 >> 6));
              if (lane < a.M) {
                const bool other = ph.pairs && static_cast<uint32_t>(c0 >> 7) != pair_h;
                if (push_bulk && other) {
                  // row `lane` of 512 bytes, its 16-byte slots XOR-swizzled by
                  // the row (the rows' same slot would share four banks)
                  float4* d = reinterpret_cast<float4*>(xring + lane * 512);
#pragma unroll
                  for (int q = 0; q < 32; ++q)
                    d[q ^ lane] = make_float4(__uint_as_float(v[q >> 2][4 * (q & 3)]), __uint_as_float(v[q >> 2][4 * (q & 3) + 1]),
                                       __uint_as_float(v[q >> 2][4 * (q & 3) + 2]), __uint_as_float(v[q >> 2][4 * (q & 3) + 3]));
                } else if (push_st && other) {
                  const uint32_t dst = pstg + static_cast<uint32_t>(lane * kStageLd + (c0 ^ 128)) * 4u;
#pragma unroll
                  for (int q = 0; q < 32; ++q)
                    st_shared_cluster_v4(dst + 16u * q, make_uint4(v[q >> 2][4 * (q & 3)], v[q >> 2][4 * (q & 3) + 1],
                                                                   v[q >> 2][4 * (q & 3) + 2], v[q >> 2][4 * (q & 3) + 3]));
                } else {
                  float4* d = reinterpret_cast<float4*>(stg + lane * kStageLd + c0);
#pragma unroll
                  for (int q = 0; q < 32; ++q)
                    d[q] = make_float4(__uint_as_float(v[q >> 2][4 * (q & 3)]), __uint_as_float(v[q >> 2][4 * (q & 3) + 1]),
                                       __uint_as_float(v[q >> 2][4 * (q & 3) + 2]), __uint_as_float(v[q >> 2][4 * (q & 3) + 3]));
                }
              }
            }
            if (push_st) {
              fence_acq_rel_cluster();
              __syncwarp();
              if (lane == 0) mbar_arrive_remote(mapa_shared(peer_ready, pair_peer));
            }
            if (push_bulk) fence_proxy_async_shared();  // the copy engine reads those rows
            if (lane == 0 && p == 0) FSOPS_STAMP(87);
          }
          if (et == 32 && p == 0) FSOPS_STAMP(88);
          tc_fence_before();
          epi_bar();
          mbar_arrive(acc_empty);
          if (push_bulk && et == 0) {
            send_ok = wait_mbar_cluster(cx, peer_free, 0, kSitePeer);
            if (send_ok) {
              bulk_copy_to_cluster(mapa_shared(xring + kPairRecvOff, pair_peer), xring, 512u * a.M,
                                   mapa_shared(peer_ready, pair_peer));
              pair_sent = true;
            }
          }
          if (et == 0) FSOPS_STAMP(p == 0 ? 12 : 60);
          if (!whole && !ph.pairs) {
            const int lg = ncols == 256 ? 6 : 5;  // log2(float4 per row)
#pragma unroll 1
            for (int q = et; q < (a.M << lg); q += 128) {
              const int r = q >> lg, c = (q & ((1 << lg) - 1)) * 4;
              const float4 v = *reinterpret_cast<const float4*>(stg + r * kStageLd + c);
              red_add_v4_f32(accg + r * kTileRows + c, v.x, v.y, v.z, v.w);
            }
          }
        } else {
          // M > 32: thread et owns token et (TMEM lane et); split tiles add
          // its 16-column runs into the row-major accumulator, four at a time
          if (whole) {
            if (ph.epi == kEpiSwiGLU) {
#pragma unroll 1
              for (int b = 0; b < (ncols >> 6); ++b) {
                uint32_t gr[2][16], ur[2][16];
                tmem_ld16(tlane + gate_col(b), gr[0]);
                tmem_ld16(tlane + gate_col(b) + 16, gr[1]);
                tmem_ld16(tlane + gate_col(b) + kPairRows, ur[0]);
                tmem_ld16(tlane + gate_col(b) + kPairRows + 16, ur[1]);
                tmem_ld_wait();
                float g[32], u[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                  g[i] = __uint_as_float(gr[i >> 4][i & 15]);
                  u[i] = __uint_as_float(ur[i >> 4][i & 15]);
                }
                if (et < a.M) swiglu_block(a, t * (ph.tile_rows >> 1) + 32 * b, et, g, u);
              }
            } else {
#pragma unroll 1
              for (int c0 = 0; c0 < ncols; c0 += 16) {
                float v[16];
                tmem_ld16f(tlane + c0, v);
                if (et < a.M) {
                  store8(a, ph, et, static_cast<long long>(t) * ph.tile_rows + c0, v);
                  store8(a, ph, et, static_cast<long long>(t) * ph.tile_rows + c0 + 8, v + 8);
                }
              }
            }
          } else {
#pragma unroll 1
            for (int c0 = 0; c0 < ncols; c0 += 16) {
              float v[16];
              tmem_ld16f(tlane + c0, v);
              if (et < a.M) {
                float* dst = accg + et * kTileRows + c0;
#pragma unroll
                for (int q = 0; q < 4; ++q) red_add_v4_f32(dst + 4 * q, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
              }
            }
          }
          tc_fence_before();
          mbar_arrive(acc_empty);
        }
        if (whole) {
          if (STAGED) finish_staged(a, ph, t, ncols, stg, et, 0, ncols >> 6);
          if (et == 0) FSOPS_STAMP_IF(p == 0, 13);
        } else if (ph.pairs) {
          // The two blocks of this cluster hold the two K halves of tile t
          // (M <= 32, staged in shared memory).  Once the partner's sums of
          // this block's half of the columns, [128 h, 128 h + 128) = 32-blocks
          // 2h, 2h+1, have arrived (pushed into this block's stg at the
          // partner's half's columns), they are added and those features
          // finished.  The partner writes nothing here after that arrival.
          const int h = static_cast<int>(pair_h);
          if (!epi_and(send_ok && wait_mbar_cluster(cx, peer_ready, 0, kSitePeer))) { ok = false; break; }
          if (et == 0) FSOPS_STAMP(58);
          // the partner's sums: pushed by stores into this stg at the other
          // half's columns, or copied into the x ring (row r at 512 r bytes,
          // 16-byte slot q of it at q ^ r)
          const float* recv = local_xq ? reinterpret_cast<const float*>(xring + kPairRecvOff) : stg;
          const int rld = local_xq ? 128 : kStageLd;
#pragma unroll 1
          for (int i = et; i < (a.M << 5); i += 128) {
            const int r = i >> 5, c = 128 * h + (i & 31) * 4;
            const float4 pv =
                *reinterpret_cast<const float4*>(recv + r * rld + (local_xq ? ((i ^ r) & 31) * 4 : (c ^ 128)));
            float4* mine = reinterpret_cast<float4*>(stg + r * kStageLd + c);
            const float4 mv = *mine;
            *mine = make_float4(mv.x + pv.x, mv.y + pv.y, mv.z + pv.z, mv.w + pv.w);
          }
          epi_bar();
          if (et == 0) FSOPS_STAMP(59);
          finish_staged(a, ph, t, 256, stg, et, 2 * h, 2);
          if (et == 0) FSOPS_STAMP_IF(p == 0, 13);
          fence_proxy_async_global();
          epi_bar();
          publish_h(a, t, et, static_cast<uint32_t>(G));
          if (et == 0) FSOPS_STAMP(14);
          // the partner's copy into the x ring is consumed (told after the
          // publication, off the path to the down projection)
          if (et == 0 && local_xq) {
            pair_received = true;
            mbar_arrive_remote(mapa_shared(peer_done, pair_peer));
          }
          if (et == 0) FSOPS_STAMP(p == 0 ? 4 : 9);
          continue;
        } else {
          // The K range of tile t is split over several blocks: every block
          // added its sums into the tile's accumulator in L2; the block that
          // arrives last reads the total, finishes the tile and leaves the
          // accumulator zero for the next launch.
          // (whole_tiles phases never get here)
          const uint32_t expected = tile_owners(ph, t, static_cast<uint32_t>(G));
          // the barrier orders every thread's adds before thread 0's acq_rel
          // counter update, which in turn orders the last arriver's reads
          epi_bar();
          if (et == 0) {
            const uint32_t old = atom_add_acq_rel_gpu(ph.tile_cnt + t, 1u);
            *bcast = static_cast<int>(old);
            // the last arrival finishes the tile (except plain output at
            // M > 32, where every owner finishes rows and finish_slice clears
            // the counter): nothing reads the counter again this launch
            if (old + 1 == expected && (STAGED || ph.epi == kEpiSwiGLU)) ph.tile_cnt[t] = 0u;
          }
          epi_bar();
          const uint32_t arrival = static_cast<uint32_t>(*bcast);
          const bool last = arrival + 1 == expected;
          epi_bar();
          if (!STAGED && ph.epi != kEpiSwiGLU) {
            // M > 32, plain output: every owner finishes the token rows its
            // arrival order names, once all owners have added their sums.  The
            // waits come after the block's last segment, so that no owner
            // holds up its later tiles (and their owners) while it waits.
            if (npend == kMaxPend) {
              ok = finish_slice(a, ph, cx, pend[0], et, bcast);
              for (int i = 1; i < npend; ++i) pend[i - 1] = pend[i];
              --npend;
              if (!ok) break;
            }
            pend[npend++] = make_int4(t, static_cast<int>(arrival), static_cast<int>(expected), ncols);
            if (et == 0) FSOPS_STAMP(p == 0 ? 4 : 9);
            continue;
          }
          if (et == 0) FSOPS_STAMP_IF(p == 1, 61);
          if (last) {
            if (STAGED) {
              // a pass's loads are all issued before its first store: one L2
              // round trip per eight float4 per thread (M * ncols / 512 <= 16)
              const int lg = ncols == 256 ? 6 : 5;
              const int n4 = a.M << lg;
              // plain output: each thread writes the four columns of each
              // float4 it read straight from registers (with the residual's
              // loads in the same round trip), eight float4 per pass; SwiGLU
              // goes through stg, whose 32-blocks span several threads' loads.
              // Each thread leaves what it read zero for the next launch at
              // once (the stores follow its own loads of the same words).
              const bool plain = ph.epi != kEpiSwiGLU, res = plain && a.residual != nullptr;
              if (et == 0) FSOPS_STAMP_IF(p == 1, 56);
#pragma unroll 1
              for (int q0 = 0; q0 < n4; q0 += 8 * 128) {
                float4 v[8];
                uint2 rv[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const int q = q0 + et + 128 * j;
                  if (q < n4) {
                    v[j] = __ldcg(reinterpret_cast<const float4*>(accg + (q >> lg) * kTileRows) + (q & ((1 << lg) - 1)));
                    if (res)
                      rv[j] = __ldcg(reinterpret_cast<const uint2*>(
                          a.residual + static_cast<long long>(q >> lg) * ph.out_ld +
                          static_cast<long long>(t) * ph.tile_rows + (q & ((1 << lg) - 1)) * 4));
                  }
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const int q = q0 + et + 128 * j;
                  if (q < n4)
                    __stcg(reinterpret_cast<float4*>(accg + (q >> lg) * kTileRows) + (q & ((1 << lg) - 1)),
                           make_float4(0.f, 0.f, 0.f, 0.f));
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const int q = q0 + et + 128 * j;
                  if (q >= n4) continue;
                  if (!plain) {
                    *reinterpret_cast<float4*>(stg + (q >> lg) * kStageLd + (q & ((1 << lg) - 1)) * 4) = v[j];
                    continue;
                  }
                  const long long o = static_cast<long long>(q >> lg) * ph.out_ld +
                                      static_cast<long long>(t) * ph.tile_rows + (q & ((1 << lg) - 1)) * 4;
                  float4 y = v[j];
                  if (res) {  // y = residual + the sums, rounded once
                    y.x += bf16_lo(rv[j].x);
                    y.y += bf16_hi(rv[j].x);
                    y.z += bf16_lo(rv[j].y);
                    y.w += bf16_hi(rv[j].y);
                  }
                  if (a.out_f32 && !res) {
                    *reinterpret_cast<float4*>(static_cast<float*>(a.out) + o) = y;
                  } else {
                    const __nv_bfloat162 b0 = __floats2bfloat162_rn(y.x, y.y), b1 = __floats2bfloat162_rn(y.z, y.w);
                    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + o) =
                        make_uint2(*reinterpret_cast<const uint32_t*>(&b0), *reinterpret_cast<const uint32_t*>(&b1));
                  }
                }
              }
              if (!plain) {
                epi_bar();
                finish_staged(a, ph, t, ncols, stg, et, 0, ncols >> 6);
              }
              if (et == 0) FSOPS_STAMP_IF(p == 1, 57);
            } else if (ph.epi == kEpiSwiGLU) {
              // token r's sums are row r of the accumulator; 64 loads are in
              // flight before their use.  With M <= 64 two threads share a
              // token (two 32-blocks each).
              const int halves = a.M <= 64 ? 2 : 1;
              const int r = et % a.M, h = et / a.M;
              if (h < halves) {
                const int nbh = (ncols >> 6) / halves;  // 32-blocks per thread
#pragma unroll 1
                for (int b = h * nbh; b < (h + 1) * nbh; ++b) {
                  float g[32], u[32];
                  const float4* gc = reinterpret_cast<const float4*>(accg + r * kTileRows + gate_col(b));
                  const float4* uc = reinterpret_cast<const float4*>(accg + r * kTileRows + gate_col(b) + kPairRows);
#pragma unroll
                  for (int i = 0; i < 8; ++i) {
                    const float4 gv = __ldcg(gc + i), uv = __ldcg(uc + i);
                    g[4 * i] = gv.x; g[4 * i + 1] = gv.y; g[4 * i + 2] = gv.z; g[4 * i + 3] = gv.w;
                    u[4 * i] = uv.x; u[4 * i + 1] = uv.y; u[4 * i + 2] = uv.z; u[4 * i + 3] = uv.w;
                  }
                  swiglu_block(a, t * (ph.tile_rows >> 1) + 32 * b, r, g, u);
                }
              }
            }
            // leave the tile's accumulator (M * 256 floats) zero for the next
            // launch (the staged path zeroed it as it read it)
            if (!STAGED) {
              epi_bar();
              float4* z = reinterpret_cast<float4*>(accg);
              const int n4 = a.M * (kTileRows / 4);
#pragma unroll 1
              for (int i = et; i < n4; i += 128) __stcg(z + i, make_float4(0.f, 0.f, 0.f, 0.f));
            }
            if (et == 0) FSOPS_STAMP_IF(p == 1, 62);
          }
          if (!last) {
            if (et == 0) FSOPS_STAMP(p == 0 ? 4 : 9);
            if (STAGED) epi_bar();  // stg is reused by the next accumulator
            continue;
          }
        }
        if (ph.epi == kEpiSwiGLU) {
          // publish tile t: each writer orders its stores before later TMA
          // reads, the barrier orders all of them before the release-add
          fence_proxy_async_global();
          if (et == 0) FSOPS_STAMP(14);
          epi_bar();
          publish_h(a, t, et, static_cast<uint32_t>(G));
        } else if (STAGED) {
          epi_bar();  // stg is reused by the next accumulator
        }
        if (et == 0) FSOPS_STAMP(p == 0 ? 4 : 9);
      }
      for (int i = 0; i < npend && ok; ++i) ok = finish_slice(a, ph, cx, pend[i], et, bcast);
      npend = 0;
      if (et == 0) FSOPS_STAMP_IF(p == 1, 62);
    }
    if (!ok) *abort_flag = 1;
    // tiles still in flight into the x ring land before the block leaves
    if (pt == 0)
      for (uint32_t c = xc; c < xi; c += 2) drain_mbar(&x_full[c & 3u], (c >> 2) & 1u, 200000000ull);
    // a copy into this block's x ring has landed, and the partner has
    // received this block's copy, before either block leaves (already so
    // unless the launch gave up)
    if (et == 0) {
      if (pair_armed && !pair_received) {
        drain_mbar(peer_ready, 0, 200000000ull);
        mbar_arrive_remote(mapa_shared(peer_done, pair_peer));
      }
      if (pair_sent) drain_mbar(peer_done, 0, 200000000ull);
    }
    if (et == 0) FSOPS_STAMP(79);
  }

  // ------------------------------------------------ teardown
  // After a launch that completes, every control word it used is back at
  // zero already: each readiness counter was cleared by the block it counts
  // for, each split tile's counter by its last arrival.  A block leaves by
  // counting itself out (a release-add, without waiting for it).  A block that
  // gave up waits (bounded) until every block of the launch has counted
  // itself out, and then one such block clears the counters the launch may
  // have left set.
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // neither block of a pair leaves while the other may still touch its shared memory
  if (a.cluster_pairs) {
    __syncwarp();
    cluster_sync_all();
  }
  if (warp == 2) tmem_dealloc(tmem, kTmemCols);
  if (threadIdx.x == 0) {
    unsigned long long* exits = reinterpret_cast<unsigned long long*>(a.ctl + kCtlExits);
    if (!*abort_flag) {
      red_add_release_gpu_u64(exits, 1ull);
    } else {
      // this launch's blocks bring the count from a multiple of G to the next
      const unsigned long long before = atom_add_acq_rel_gpu_u64(exits, 1ull);
      const unsigned long long all = (before / static_cast<unsigned long long>(G) + 1ull) * static_cast<unsigned long long>(G);
      const uint64_t t0 = globaltimer_ns();
      bool gone = false;
      while (!(gone = ld_acquire_gpu_u64(exits) >= all) && globaltimer_ns() - t0 < 200000000ull) __nanosleep(256);
      if (gone && atomicCAS(a.ctl + kCtlCleanup, 0u, 1u) == 0u) {
        for (int p = 0; p < a.nphases; ++p)
          for (int t = 0; t < a.ph[p].T; ++t) a.ph[p].tile_cnt[t] = 0u;
        for (int c = 0; c < static_cast<int>(G); ++c) {
          if (a.xready != nullptr) a.xready[c] = 0u;
          if (a.hflags != nullptr) a.hflags[c] = 0u;
        }
        __threadfence();
        a.ctl[kCtlCleanup] = 0u;
      }
    }
    FSOPS_STAMP(78);
  }
}

namespace {
// Per device: the kernel's dynamic shared-memory limit has been raised.  The
// flags have internal linkage, so every loaded copy of the library sets the
// limit of its own kernel.
constexpr int kMaxAttrDevices = 64;
std::atomic<bool> g_smem_attr_set[kMaxAttrDevices];
}  // namespace

cudaError_t launch_mx_kernel(const KernelArgs& a, int grid, size_t smem, cudaStream_t stream, bool cooperative) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxAttrDevices) return cudaErrorInvalidDevice;
  if (!g_smem_attr_set[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(mx_persistent_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(mx_persistent_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
    if (e != cudaSuccess) return e;
    g_smem_attr_set[dev].store(true, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[3];
  int n = 0;
  if (cooperative) {
    attr[n].id = cudaLaunchAttributeCooperative;
    attr[n++].val.cooperative = 1;
  } else {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n++].val.programmaticStreamSerializationAllowed = 1;
  }
  if (a.cluster_pairs) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 2;
    attr[n].val.clusterDim.y = 1;
    attr[n++].val.clusterDim.z = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return a.stage_tmem ? cudaLaunchKernelEx(&cfg, mx_persistent_kernel<true>, a)
                      : cudaLaunchKernelEx(&cfg, mx_persistent_kernel<false>, a);
}

bool grid_fits(int grid, size_t smem) {
  if (cudaFuncSetAttribute(mx_persistent_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem) !=
      cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  int per_sm = 0, dev = 0, sms = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mx_persistent_kernel<true>, kThreads, smem) != cudaSuccess ||
      cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return per_sm * sms >= grid;
}

bool cluster_pairs_fit(int grid, size_t smem) {
  if (grid % 2 != 0) return false;
  if (cudaFuncSetAttribute(mx_persistent_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem) !=
      cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, mx_persistent_kernel<true>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return 2 * n >= grid;
}

}  // namespace fsops
