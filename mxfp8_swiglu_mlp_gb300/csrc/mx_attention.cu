// mx_attention.cu -- one decode step of attention over a paged MXFP8 KV cache.
//
//   paged_decode_kernel<G>  block (split, kv head, sequence): streams the
//                           split's chunks of 128 tokens (their K and V pages
//                           and scale rows, by bulk copies into a two-stage
//                           shared-memory ring), scores them for the G query
//                           heads that share the KV head (the GQA broadcast:
//                           K and V are read once for the group), keeps an
//                           online softmax and the unnormalised output.
//   attn_combine_kernel     merges the splits of one (sequence, query head)
//                           and writes the bf16 output.
//
// K and V are MXFP8: E4M3 codes with one UE8M0 scale per 32 elements of the
// head dimension (the Fish Audio post's mxfp8 format, p2 "Estrategia de
// cuantizacion FP8", applied to the cache that its MXFP8 FlashAttention
// reads, p2 "Ya esta disponible").  q, the scores and the probabilities stay
// in fp32: scores = sm_scale * q . k, p = softmax over the sequence,
// out = p . v, rounded once to bf16.
//
// Cache layout: page p, KV head h holds P tokens' codes contiguously
// ([num_pages, Hkv, P, D]) and their scales ([num_pages, Hkv, P, D / 32]);
// token t of a sequence is slot t % P of page block_table[t / P].
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "mx_attention.h"
#include "sm103.cuh"

namespace fsops {
using namespace dev;

namespace {

constexpr int kAThreads = 256;  // two threads per token of a chunk
constexpr int kAWarps = kAThreads / 32;
constexpr int kD = kAttnHeadDim;
constexpr int kC = kAttnChunk;
constexpr uint32_t kCodeBytes = kC * kD;      // 16 KB of K (or V) codes per chunk
constexpr uint32_t kScaleBytes = kC * kD / 32;  // 512 B of scales per chunk
constexpr int kQPiece = 20;                     // floats per padded 16-element piece of q

struct __align__(128) AttnStage {
  uint8_t k[kCodeBytes];
  uint8_t v[kCodeBytes];
  uint8_t ks[kScaleBytes];
  uint8_t vs[kScaleBytes];
};
constexpr size_t kAttnSmem = 2 * sizeof(AttnStage) + 128;  // + alignment slack

// Two E4M3 codes (low byte first) as two floats: exact.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two & 0xFFFFu), __NV_E4M3);
  return __half22float2(__half2(h));
}
// 2^(s - 127) for a UE8M0 byte s (s = 0 is the subnormal 2^-127).
__device__ __forceinline__ float ue8m0_value(uint32_t s) {
  return s != 0 ? __uint_as_float(s << 23) : __uint_as_float(0x00400000u);
}
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

__device__ __forceinline__ void attn_error(const AttnArgs& a, uint32_t code, uint32_t site) {
  atomicCAS(a.status, 0u, (code << 24) | ((site & 0xFFu) << 16) | (blockIdx.z & 0xFFFFu));
}

// Timeline stamps for profiling builds (compiled with -DFSOPS_TRACE).
#ifdef FSOPS_TRACE
#define ATTN_STAMP(idx)                                                                                   \
  do {                                                                                                    \
    if (a.trace != nullptr)                                                                               \
      a.trace[((blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x) * 64 + (idx)] = globaltimer_ns(); \
  } while (0)
#else
#define ATTN_STAMP(idx) \
  do {                  \
  } while (0)
#endif

template <int G>
__global__ void __launch_bounds__(kAThreads, 3) paged_decode_kernel(const __grid_constant__ AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  AttnStage* stg = reinterpret_cast<AttnStage*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  // q of the group's heads, each 16-element piece padded to 20 floats: the
  // threads of a quarter warp read eight different pieces at once, and
  // 80-byte strides put them on distinct banks
  __shared__ __align__(16) float qs[G * 8 * kQPiece];
  // probabilities of each warp's 16 tokens of the chunk: [warp][G][16]
  __shared__ __align__(16) float ps[kAWarps * G * 16];
  __shared__ float red_max[kAWarps * G], red_sum[kAWarps * G];
  __shared__ __align__(8) uint64_t bar[2];
  __shared__ int chunk_ok[2];

  const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int len = a.seq_lens[b];
  const bool len_ok = len >= 1 && len <= a.max_pages * a.P;
  if (!len_ok && t == 0 && split == 0 && hk == 0) attn_error(a, 1u, 1u);  // FSOPS_ERR_INVALID_ARG
  const int n = len_ok ? len : 0;
  const int nchunks = (n + kC - 1) / kC;
  // every split the same number of chunks of the longest sequence's
  const int per = (a.max_pages * a.P + kC * a.nsplit - 1) / (kC * a.nsplit);
  const int c0 = min(nchunks, split * per), c1 = min(nchunks, c0 + per);
  const int npages = (n + a.P - 1) / a.P;
  const int pages_per_chunk = kC / a.P;

  for (int i = t; i < G * kD; i += kAThreads)
    qs[(i / 16) * kQPiece + i % 16] = bf16_bits_to_float(a.q[(static_cast<size_t>(b) * a.Hq + hk * G) * kD + i]);
  if (t == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    mbar_fence_init();
    ATTN_STAMP(0);
  }
  __syncthreads();

  // Warp 0: the bulk copies of chunk c into stage s, lane i those of the
  // chunk's page i, all in flight together (pages past the sequence's last
  // one are not loaded; their tokens are masked).  A page id outside
  // [0, num_pages) is reported and its page skipped.
  auto issue = [&](int c, int s) {
    const int p0 = c * pages_per_chunk;
    const int np = min(pages_per_chunk, npages - p0);
    int pid = -1;
    bool mine = lane < np, good = true;
    if (mine) {
      pid = a.block_table[static_cast<size_t>(b) * a.max_pages + p0 + lane];
      good = pid >= 0 && pid < a.num_pages;
    }
    const bool ok = __all_sync(0xFFFFFFFFu, good);
    const uint32_t npg = __popc(__ballot_sync(0xFFFFFFFFu, mine && good));
    if (lane == 0) {
      if (!ok) attn_error(a, 1u, 2u);
      chunk_ok[s] = ok ? 1 : 0;
    }
    fence_proxy_async_shared();  // the stage's earlier generic reads come before the copies' writes
    if (lane == 0) mbar_arrive_expect_tx(&bar[s], npg * 2u * (a.P * kD + a.P * (kD / 32)));
    __syncwarp();
    if (mine && good) {
      const size_t row = (static_cast<size_t>(pid) * a.Hkv + hk) * a.P;  // first token row of the page-head block
      const uint32_t cb = static_cast<uint32_t>(a.P) * kD, sb = static_cast<uint32_t>(a.P) * (kD / 32);
      const uint64_t pol = l2_policy_evict_first();
      bulk_load(stg[s].k + lane * cb, a.k_codes + row * kD, cb, &bar[s], pol);
      bulk_load(stg[s].v + lane * cb, a.v_codes + row * kD, cb, &bar[s], pol);
      bulk_load(stg[s].ks + lane * sb, a.k_scales + row * (kD / 32), sb, &bar[s], pol);
      bulk_load(stg[s].vs + lane * sb, a.v_scales + row * (kD / 32), sb, &bar[s], pol);
    }
  };

  // Warp w owns tokens w, w + 8, ..., w + 120 of every chunk: it scores them
  // (lanes 2k and 2k + 1 token w + 8k, half of the dimensions each), keeps
  // its own online softmax over them, and adds their p . v into its lanes'
  // four output dimensions.  The warps' states are merged once at the end,
  // so a chunk needs no block barrier besides the one on its copies.
  float m_run[G], l_run[G], acc[G][4];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m_run[g] = -INFINITY;
    l_run[g] = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[g][e] = 0.f;
  }
  bool ok = true;
  int issued = c0;   // chunks whose copies were issued
  int stalled = -1;  // the chunk whose copies did not land in time
  if (warp == 0 && c0 < c1) issue(c0, 0);
  issued = c0 < c1 ? c0 + 1 : c0;
  float* pw = ps + warp * G * 16;
  for (int c = c0; c < c1 && ok; ++c) {
    const int s = (c - c0) & 1;
    stalled = c;
    // bounded wait for the chunk's copies
    {
      const uint32_t parity = static_cast<uint32_t>((c - c0) >> 1) & 1u;
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&bar[s], parity)) {
        if (globaltimer_ns() - t0 > a.timeout_ns) {
          if (t == 0) attn_error(a, 5u, 3u);  // FSOPS_ERR_TIMEOUT
          ok = false;
          break;
        }
      }
    }
    // every warp is past the previous chunk: its stage may be refilled
    if (!__syncthreads_and(ok)) break;
    if (warp == 0 && c + 1 < c1) issue(c + 1, s ^ 1);
    issued = c + 1 < c1 ? c + 2 : issued;
    const bool chunk_valid = chunk_ok[s] != 0;
    if (t == 0 && c - c0 < 12) ATTN_STAMP(4 + 4 * (c - c0));

    // ---- scores: lanes 2k and 2k + 1 score token w + 8k of the chunk for
    // the G heads over dimensions [0, 64) and [64, 128), and add their halves
    const int kk = lane >> 1, half = lane & 1;
    const int tt0 = warp + 8 * kk;
    const int tok = c * kC + tt0;
    float sc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) sc[g] = 0.f;
    if (tok < n && chunk_valid) {
      const uint8_t* krow = stg[s].k + tt0 * kD;
      const uint32_t kscales = *reinterpret_cast<const uint32_t*>(stg[s].ks + tt0 * (kD / 32));
#pragma unroll 2
      for (int i = 0; i < 4; ++i) {
        // 16-code piece of this half, rotated per token against bank conflicts
        const int cc = 4 * half + ((i + kk) & 3);
        const uint4 kv = *reinterpret_cast<const uint4*>(krow + 16 * cc);
        const uint32_t w4[4] = {kv.x, kv.y, kv.z, kv.w};
        float kf[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 lo = e4m3x2_to_float2(w4[j]), hi = e4m3x2_to_float2(w4[j] >> 16);
          kf[4 * j] = lo.x;
          kf[4 * j + 1] = lo.y;
          kf[4 * j + 2] = hi.x;
          kf[4 * j + 3] = hi.y;
        }
        const float scale = ue8m0_value((kscales >> (8 * (cc >> 1))) & 0xFFu);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float4* qv = reinterpret_cast<const float4*>(qs + (g * 8 + cc) * kQPiece);
          float dot = 0.f;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float4 q4 = qv[j];
            dot = fmaf(q4.x, kf[4 * j], dot);
            dot = fmaf(q4.y, kf[4 * j + 1], dot);
            dot = fmaf(q4.z, kf[4 * j + 2], dot);
            dot = fmaf(q4.w, kf[4 * j + 3], dot);
          }
          sc[g] = fmaf(scale, dot, sc[g]);
        }
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      sc[g] += __shfl_xor_sync(0xFFFFFFFFu, sc[g], 1);
      sc[g] = (tok < n && chunk_valid) ? sc[g] * a.sm_scale : -INFINITY;
    }
    if (t == 0 && c - c0 < 12) ATTN_STAMP(5 + 4 * (c - c0));

    // ---- the warp's online softmax over its 16 tokens
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float cm = sc[g];
#pragma unroll
      for (int o = 16; o >= 2; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xFFFFFFFFu, cm, o));
      const float mn = fmaxf(m_run[g], cm);
      // no valid token yet (a bad page, or the tokens past the sequence):
      // mn = -inf and nothing is added
      const float p = (sc[g] == -INFINITY || mn == -INFINITY) ? 0.f : expf(sc[g] - mn);
      const float alpha = (m_run[g] == -INFINITY || mn == -INFINITY) ? (mn == -INFINITY ? 1.f : 0.f)
                                                                      : expf(m_run[g] - mn);
      m_run[g] = mn;
      if (half == 0) pw[g * 16 + kk] = p;
      float sum = half == 0 ? p : 0.f;  // each token once
#pragma unroll
      for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
      l_run[g] = l_run[g] * alpha + sum;
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[g][e] *= alpha;
    }
    __syncwarp();  // pw is written before the lanes read it
    if (t == 0 && c - c0 < 12) ATTN_STAMP(6 + 4 * (c - c0));

    // ---- p . v: lane l owns dimensions 4 l .. 4 l + 3 of the warp's tokens
    const int tmax = min(kC, n - c * kC);
    if (chunk_valid) {
#pragma unroll 4
      for (int k = 0; k < 16; ++k) {
        const int tt = warp + 8 * k;
        if (tt >= tmax) break;
        const uint32_t v4 = *reinterpret_cast<const uint32_t*>(stg[s].v + tt * kD + 4 * lane);
        const float vscale = ue8m0_value(stg[s].vs[tt * (kD / 32) + (lane >> 3)]);
        const float2 lo = e4m3x2_to_float2(v4), hi = e4m3x2_to_float2(v4 >> 16);
        const float vf[4] = {lo.x * vscale, lo.y * vscale, hi.x * vscale, hi.y * vscale};
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float p = pw[g * 16 + k];
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[g][e] = fmaf(p, vf[e], acc[g][e]);
        }
      }
    }
    __syncwarp();  // pw is rewritten by the next chunk
    if (t == 0 && c - c0 < 12) ATTN_STAMP(7 + 4 * (c - c0));
    stalled = -1;
  }
  if (stalled >= 0) {
    // gave up: let the copies still in flight land before the ring is reused
    // or the block leaves
    if (t == 0) {
      for (int c = stalled; c < issued; ++c) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&bar[(c - c0) & 1], static_cast<uint32_t>((c - c0) >> 1) & 1u))
          if (globaltimer_ns() - t0 > 200000000ull) break;
      }
    }
  }
  __syncthreads();  // every warp is done with the ring

  if (t == 0) {
    ATTN_STAMP(1);
    if (a.trace != nullptr) a.trace[((blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x) * 64 + 2] = c1 - c0;
  }
  // ---- merge the warps' states: the block's max, sum and unnormalised
  // output per head, one record each
  float* wacc = reinterpret_cast<float*>(stg);  // reuse the ring: [kAWarps][G][D]
#pragma unroll
  for (int g = 0; g < G; ++g) {
#pragma unroll
    for (int e = 0; e < 4; ++e) wacc[(warp * G + g) * kD + 4 * lane + e] = acc[g][e];
    if (lane == 0) {
      red_max[warp * G + g] = m_run[g];
      red_sum[warp * G + g] = l_run[g];
    }
  }
  __syncthreads();
  for (int i = t; i < G * kD; i += kAThreads) {
    const int g = i / kD, d = i % kD;
    float M = red_max[g];
#pragma unroll
    for (int w = 1; w < kAWarps; ++w) M = fmaxf(M, red_max[w * G + g]);
    float o = 0.f, l = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kAWarps; ++w) {
        const float mw = red_max[w * G + g];
        if (mw == -INFINITY) continue;
        const float f = expf(mw - M);
        o = fmaf(f, wacc[(w * G + g) * kD + d], o);
        l = fmaf(f, red_sum[w * G + g], l);
      }
    }
    float* rec = a.part + ((static_cast<size_t>(b) * a.Hq + hk * G + g) * a.nsplit + split) * (2 + kD);
    rec[2 + d] = o;
    if (d == 0) {
      rec[0] = M;
      rec[1] = l;
    }
  }
}

// One block per (query head, sequence), one thread per dimension.
__global__ void __launch_bounds__(kD) attn_combine_kernel(const __grid_constant__ AttnArgs a) {
  const int h = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
  const float* rec = a.part + (static_cast<size_t>(b) * a.Hq + h) * a.nsplit * (2 + kD);
  float M = -INFINITY;
  for (int s = 0; s < a.nsplit; ++s) M = fmaxf(M, rec[s * (2 + kD)]);
  float num = 0.f, den = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < a.nsplit; ++s) {
      const float m = rec[s * (2 + kD)];
      if (m == -INFINITY) continue;
      const float w = expf(m - M);
      num = fmaf(w, rec[s * (2 + kD) + 2 + d], num);
      den = fmaf(w, rec[s * (2 + kD) + 1], den);
    }
  }
  const float o = den > 0.f ? num / den : 0.f;
  const __nv_bfloat16 ob = __float2bfloat16_rn(o);
  a.out[(static_cast<size_t>(b) * a.Hq + h) * kD + d] = *reinterpret_cast<const uint16_t*>(&ob);
}

template <int G>
cudaError_t launch_group(const AttnArgs& a, cudaStream_t stream) {
  static_assert(G <= kAttnMaxGroup, "group");
  cudaError_t e = cudaFuncSetAttribute(paged_decode_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kAttnSmem));
  if (e != cudaSuccess) return e;
  paged_decode_kernel<G><<<dim3(a.nsplit, a.Hkv, a.B), kAThreads, kAttnSmem, stream>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_combine_kernel<<<dim3(a.Hq, a.B), kD, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

int attn_splits(int B, int Hkv, int max_pages, int P, int sms, int chunks_per_block) {
  // Every block takes the same number of chunks (the last of a sequence
  // fewer, and splits past a short sequence's end none), so the blocks are
  // of even size whatever the length mix; with fewer (B, KV head) pairs than
  // about three blocks per SM the chunks are spread thinner.
  const int max_chunks = (max_pages * P + kC - 1) / kC;
  int per = chunks_per_block;
  const int want = (3 * sms + B * Hkv - 1) / (B * Hkv);  // splits for three blocks per SM
  if ((max_chunks + per - 1) / per < want) per = (max_chunks + want - 1) / want;
  if (per < 1) per = 1;
  return (max_chunks + per - 1) / per;
}

cudaError_t launch_paged_decode(const AttnArgs& a, cudaStream_t stream) {
  switch (a.Hq / a.Hkv) {
    case 1: return launch_group<1>(a, stream);
    case 2: return launch_group<2>(a, stream);
    case 4: return launch_group<4>(a, stream);
    case 8: return launch_group<8>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fsops
