// mx_attention.cu -- one decode step of attention over a paged MXFP8 KV cache.
//
//   paged_decode_kernel<G>  block (split, kv head, sequence): a producer warp
//                           streams the split's chunks of 128 tokens (their K
//                           and V pages by TMA with the 128-byte swizzle, their
//                           scale rows by bulk copies) through a three-stage
//                           shared-memory ring; eight consumer warps, 16
//                           tokens each, score them for the G query heads that
//                           share the KV head (the GQA broadcast: K and V are
//                           read once for the group) and add p . v, both
//                           products on the tensor cores, keeping an online
//                           softmax per warp.
//   attn_combine_kernel     merges the splits of one (sequence, query head)
//                           and writes the bf16 output.
//
// K and V are MXFP8: E4M3 codes with one UE8M0 scale per 32 elements of the
// head dimension (the Fish Audio post's mxfp8 format, p2 "Estrategia de
// cuantizacion FP8", applied to the cache that its MXFP8 FlashAttention
// reads, p2 "Ya esta disponible").  q, the scores and the probabilities keep
// fp32 accuracy: scores = sm_scale * q . k, p = softmax over the sequence,
// out = p . v, rounded once to bf16.
//
// How the products stay exact on f16 tensor cores (mma.sync m16n8k16, fp32
// accumulation):
//   * q . k: the E4M3 codes are exact in f16.  Each query head's q is scaled
//     by a power of two that puts its largest element in [2^13, 2^14), which
//     keeps the bf16 values exact in f16.  One 32-element block of the head
//     dimension (two k-steps) is summed per MMA chain and multiplied by its K
//     scale in fp32; the power of two and sm_scale are taken out afterwards.
//   * p . v: V's scales vary along the summed (token) dimension, so they are
//     applied to the codes: a token's block is multiplied by 2^(s - s_max),
//     s_max the largest scale of that block among the 16 tokens of the MMA,
//     exact in f16 while s_max - s <= 14, and 2^(s_max - 127) is applied to
//     the fp32 sums.  The probabilities are split into two f16 terms (the
//     upper 11 significant bits and the rest), 22 bits in all.  A warp whose
//     16 tokens hold a block scale 2^15 or more below s_max (an all-zero
//     block, for one) adds that chunk's p . v with fp32 FMAs instead.
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

constexpr int kCWarps = 8;                        // consumer warps, 16 tokens of a chunk each
constexpr int kAThreads = 32 * (kCWarps + 1);     // + the producer warp
constexpr int kAStages = 3;
constexpr int kD = kAttnHeadDim;
constexpr int kC = kAttnChunk;
constexpr uint32_t kCodeBytes = kC * kD;          // 16 KB of K (or V) codes per chunk
constexpr uint32_t kScaleBytes = kC * kD / 32;    // 512 B of scales per chunk
constexpr int kPwLd = 20;                         // row stride (floats) of a warp's p[head][token]
static_assert(kC == 16 * kCWarps, "a consumer warp owns 16 tokens of a chunk");

struct __align__(1024) AttnStage {
  uint8_t k[kCodeBytes];  // [token][128] swizzled: 16-byte piece j of row r at piece j ^ (r % 8)
  uint8_t v[kCodeBytes];
  uint8_t ks[kScaleBytes];  // [token][4]
  uint8_t vs[kScaleBytes];
};
static_assert(sizeof(AttnStage) % 1024 == 0, "stages stay 1024-byte aligned");
constexpr size_t kAttnSmem = kAStages * sizeof(AttnStage) + 1024;  // + alignment slack

// Byte offset of (row, byte) in a 128-byte-swizzled tile whose base is
// 1024-byte aligned.
__device__ __forceinline__ int swz(int row, int off) {
  return row * 128 + ((((off >> 4) ^ row) & 7) << 4) + (off & 15);
}
// E4M3 codes in bytes 0-1 (or 2-3) of w as f16x2 (exact), the lower byte in
// the lower half.
__device__ __forceinline__ uint32_t e4m3_lo_f16x2(uint32_t w) {
  uint32_t r;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\t}" : "=r"(r) : "r"(w));
  return r;
}
__device__ __forceinline__ uint32_t e4m3_hi_f16x2(uint32_t w) {
  uint32_t r;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, h;\n\t}" : "=r"(r) : "r"(w));
  return r;
}
// Two floats as f16x2 (round to nearest even), `lo` in the lower half.
__device__ __forceinline__ uint32_t f16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// Byte permute; a selector nibble with bit 3 set replicates the sign bit of
// the byte it names.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
// d += A . B on the tensor core: A 16 x 16 f16 (row), B 16 x 8 f16 (col), fp32 d.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Two E4M3 codes (low byte first) as two floats: exact.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two & 0xFFFFu), __NV_E4M3);
  return __half22float2(__half2(h));
}
// 2^(s - 127) for a UE8M0 byte s (s = 0 is the subnormal 2^-127).
__device__ __forceinline__ float ue8m0_value(uint32_t s) {
  return s != 0 ? __uint_as_float(s << 23) : __uint_as_float(0x00400000u);
}
__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }
// p as the f16 pair hi + lo: hi keeps p's upper 11 significant bits (exact in
// f16 for p >= 2^-14), lo the f16 rounding of the rest.
__device__ __forceinline__ void split_f16x2(float2 p, uint32_t& hi, uint32_t& lo) {
  const float hx = __uint_as_float(__float_as_uint(p.x) & 0xFFFFE000u);
  const float hy = __uint_as_float(__float_as_uint(p.y) & 0xFFFFE000u);
  hi = f16x2_rn(hx, hy);
  lo = f16x2_rn(p.x - hx, p.y - hy);
}

__device__ __forceinline__ void attn_error(const AttnArgs& a, uint32_t code, uint32_t site) {
  atomicCAS(a.status, 0u, (code << 24) | ((site & 0xFFu) << 16) | (blockIdx.z & 0xFFFFu));
}
// Wait for the phase of `bar` with the given parity, at most timeout_ns.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > timeout_ns) return false;
  return true;
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
__global__ void __launch_bounds__(kAThreads, 2) paged_decode_kernel(const __grid_constant__ AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  AttnStage* stg = reinterpret_cast<AttnStage*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // each consumer warp's probabilities of its 16 tokens: [warp][head][token]
  __shared__ __align__(16) float pws[kCWarps * 8 * kPwLd];
  __shared__ float red_max[kCWarps * G], red_sum[kCWarps * G];
  __shared__ __align__(8) uint64_t full[kAStages], empty[kAStages];
  __shared__ int chunk_ok[kAStages];
  // q of the group as the B operand of the score MMA, per lane: block bb's
  // two k-steps in qfrag[bb][lane]; sm_scale / 2^e per head
  __shared__ uint4 qfrag[4][32];
  __shared__ float qscale[8];

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

  if (warp == 0) {
    // Lane (g, tq) holds head g's B fragments: k-step j (dimensions of block
    // j / 2) pairs mma column k = 2 tq + {0, 1} with dimension
    // 32 (j / 2) + 8 tq + 4 (j % 2) + {0, 1} and k = 2 tq + 8 + {0, 1} with
    // + {2, 3}, so that a lane's 8-byte K load feeds two k-steps.  Each head
    // is scaled by the power of two 2^e that puts its largest |q| in
    // [2^13, 2^14): exact in f16.
    const int g = lane >> 2, tq = lane & 3;
    float qv[32];
    if (g < G) {
      const uint4* qp = reinterpret_cast<const uint4*>(a.q + (static_cast<size_t>(b) * a.Hq + hk * G + g) * kD);
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        const uint4 w = qp[4 * bb + tq];
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          qv[8 * bb + 2 * j] = bf16_bits_to_float(ws[j] & 0xFFFFu);
          qv[8 * bb + 2 * j + 1] = bf16_bits_to_float(ws[j] >> 16);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) qv[j] = 0.f;
    }
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(qv[j]));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
    int e = 0;
    if (amax > 0.f) e = min(140 - static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu), 126);
    const float up = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
#pragma unroll
    for (int bb = 0; bb < 4; ++bb)
      qfrag[bb][lane] = make_uint4(f16x2_rn(qv[8 * bb] * up, qv[8 * bb + 1] * up),
                                   f16x2_rn(qv[8 * bb + 2] * up, qv[8 * bb + 3] * up),
                                   f16x2_rn(qv[8 * bb + 4] * up, qv[8 * bb + 5] * up),
                                   f16x2_rn(qv[8 * bb + 6] * up, qv[8 * bb + 7] * up));
    if (tq == 0) qscale[g] = ldexpf(a.sm_scale, -e);
  }
  if (t == 0) {
#pragma unroll
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCWarps);
    }
    mbar_fence_init();
    ATTN_STAMP(0);
  }
  __syncthreads();

  const int g = lane >> 2, tq = lane & 3;  // mma fragment row group and column pair
  // consumer state: the p . v sums O^T[d][head] of the warp's tokens (blocks
  // of 32 dimensions bb, two 16-row tiles each: rows g and g + 8 are
  // dimensions 32 bb + 4 g + {0, 1} of tile 0 and + {2, 3} of tile 1; columns
  // heads 2 tq and 2 tq + 1), and the running max and partial sums of the
  // lane's two heads
  float O[4][2][4];
#pragma unroll
  for (int bb = 0; bb < 4; ++bb)
#pragma unroll
    for (int tt = 0; tt < 2; ++tt)
#pragma unroll
      for (int e = 0; e < 4; ++e) O[bb][tt][e] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_part[2] = {0.f, 0.f};

  if (warp == kCWarps) {
    // ---- producer: chunk c into stage (c - c0) % kAStages once every
    // consumer warp has left the chunk that held it; lane i copies the
    // chunk's page i.  Pages past the sequence's last one are not loaded
    // (their tokens are masked); a page id outside [0, num_pages) is reported
    // and the chunk skipped.
    const int npages = (n + a.P - 1) / a.P;
    const int ppc = kC / a.P;
    const uint32_t cb = static_cast<uint32_t>(a.P) * kD, sb = static_cast<uint32_t>(a.P) * (kD / 32);
    const uint64_t pol = l2_policy_evict_first();
    if (lane == 0) {
      tma_prefetch_desc(&a.tm_k);
      tma_prefetch_desc(&a.tm_v);
    }
    int issued = c0;
    for (int c = c0; c < c1; ++c) {
      const int i = c - c0, s = i % kAStages;
      if (i >= kAStages && !wait_phase(&empty[s], static_cast<uint32_t>(i / kAStages - 1) & 1u, a.timeout_ns)) {
        if (lane == 0) attn_error(a, 5u, 4u);  // FSOPS_ERR_TIMEOUT
        break;
      }
      const int p0 = c * ppc;
      const int np = min(ppc, npages - p0);
      int pid = -1;
      const bool mine = lane < np;
      bool good = true;
      if (mine) {
        pid = a.block_table[static_cast<size_t>(b) * a.max_pages + p0 + lane];
        good = pid >= 0 && pid < a.num_pages;
      }
      const bool all_good = __all_sync(0xFFFFFFFFu, good);
      const uint32_t npg = __popc(__ballot_sync(0xFFFFFFFFu, mine && good));
      if (lane == 0) {
        if (!all_good) attn_error(a, 1u, 2u);
        chunk_ok[s] = all_good ? 1 : 0;
      }
      fence_proxy_async_shared();  // the stage's earlier generic reads come before the copies' writes
      if (lane == 0) mbar_arrive_expect_tx(&full[s], npg * 2u * (cb + sb));
      __syncwarp();
      if (mine && good) {
        const int y = (pid * a.Hkv + hk) * a.P;  // first row of the (page, head) block
        tma_load_2d(stg[s].k + lane * cb, &a.tm_k, &full[s], 0, y, pol);
        tma_load_2d(stg[s].v + lane * cb, &a.tm_v, &full[s], 0, y, pol);
        bulk_load(stg[s].ks + lane * sb, a.k_scales + static_cast<size_t>(y) * (kD / 32), sb, &full[s], pol);
        bulk_load(stg[s].vs + lane * sb, a.v_scales + static_cast<size_t>(y) * (kD / 32), sb, &full[s], pol);
      }
      issued = c + 1;
    }
    // the last chunks' copies land before the ring is reused (every earlier
    // chunk of a stage was consumed before the stage was refilled)
    for (int c = max(c0, issued - kAStages); c < issued; ++c)
      wait_phase(&full[(c - c0) % kAStages], static_cast<uint32_t>((c - c0) / kAStages) & 1u, 200000000ull);
  } else {
    // ---- consumer warp: tokens 16 warp .. 16 warp + 15 of every chunk
    const int wrow = 16 * warp;
    float hs[2];  // sm_scale / 2^e of heads 2 tq and 2 tq + 1
    hs[0] = qscale[2 * tq];
    hs[1] = qscale[2 * tq + 1];
    float* pw = pws + warp * 8 * kPwLd;

    for (int c = c0; c < c1; ++c) {
      const int i = c - c0, s = i % kAStages;
      if (!wait_phase(&full[s], static_cast<uint32_t>(i / kAStages) & 1u, a.timeout_ns)) {
        if (lane == 0) attn_error(a, 5u, 3u);  // FSOPS_ERR_TIMEOUT
        break;
      }
      const int tmax = min(kC, n - c * kC);  // valid rows of the chunk
      if (chunk_ok[s] != 0 && wrow < tmax) {
        const uint8_t* kb = stg[s].k;
        const uint8_t* vb = stg[s].v;
        // ---- scores of tokens r0 and r1 (mma rows g, g + 8) for heads 2 tq, 2 tq + 1
        const int r0 = wrow + g, r1 = r0 + 8;
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
        {
          const uint32_t kw0 = *reinterpret_cast<const uint32_t*>(stg[s].ks + 4 * r0);
          const uint32_t kw1 = *reinterpret_cast<const uint32_t*>(stg[s].ks + 4 * r1);
#pragma unroll
          for (int bb = 0; bb < 4; ++bb) {
            const uint2 x0 = *reinterpret_cast<const uint2*>(kb + swz(r0, 32 * bb + 8 * tq));
            const uint2 x1 = *reinterpret_cast<const uint2*>(kb + swz(r1, 32 * bb + 8 * tq));
            const uint4 bq = qfrag[bb][lane];
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            mma_16816(d, e4m3_lo_f16x2(x0.x), e4m3_lo_f16x2(x1.x), e4m3_hi_f16x2(x0.x), e4m3_hi_f16x2(x1.x), bq.x,
                      bq.y);
            mma_16816(d, e4m3_lo_f16x2(x0.y), e4m3_lo_f16x2(x1.y), e4m3_hi_f16x2(x0.y), e4m3_hi_f16x2(x1.y), bq.z,
                      bq.w);
            const float f0 = ue8m0_value((kw0 >> (8 * bb)) & 0xFFu), f1 = ue8m0_value((kw1 >> (8 * bb)) & 0xFFu);
            sc[0] = fmaf(f0, d[0], sc[0]);
            sc[1] = fmaf(f0, d[1], sc[1]);
            sc[2] = fmaf(f1, d[2], sc[2]);
            sc[3] = fmaf(f1, d[3], sc[3]);
          }
        }
        // ---- the warp's online softmax over its 16 tokens, per head
        const bool v0 = r0 < tmax, v1 = r1 < tmax;
        float al[2];
#pragma unroll
        for (int i2 = 0; i2 < 2; ++i2) {
          const int hh = 2 * tq + i2;
          const bool hv = hh < G;
          const float x0 = (v0 && hv) ? sc[i2] * hs[i2] : -INFINITY;
          const float x1 = (v1 && hv) ? sc[2 + i2] * hs[i2] : -INFINITY;
          float cm = fmaxf(x0, x1);
          cm = fmaxf(cm, __shfl_xor_sync(0xFFFFFFFFu, cm, 4));
          cm = fmaxf(cm, __shfl_xor_sync(0xFFFFFFFFu, cm, 8));
          cm = fmaxf(cm, __shfl_xor_sync(0xFFFFFFFFu, cm, 16));
          const float mn = fmaxf(m_run[i2], cm);
          // no valid token yet: mn = -inf and nothing is added
          al[i2] = mn == -INFINITY ? 1.f : expf(m_run[i2] - mn);
          const float p0 = x0 == -INFINITY ? 0.f : expf(x0 - mn);
          const float p1 = x1 == -INFINITY ? 0.f : expf(x1 - mn);
          m_run[i2] = mn;
          l_part[i2] = fmaf(l_part[i2], al[i2], p0 + p1);
          pw[hh * kPwLd + g] = p0;
          pw[hh * kPwLd + g + 8] = p1;
        }
        if (al[0] != 1.f || al[1] != 1.f) {
#pragma unroll
          for (int bb = 0; bb < 4; ++bb)
#pragma unroll
            for (int tt = 0; tt < 2; ++tt) {
              O[bb][tt][0] *= al[0];
              O[bb][tt][1] *= al[1];
              O[bb][tt][2] *= al[0];
              O[bb][tt][3] *= al[1];
            }
        }
        __syncwarp();  // pw is written before the lanes read it

        // ---- p . v: A = V^T (rows: dimensions, k: tokens rv, rv + 1, rv + 8,
        // rv + 9 of the lane), B = p of head g
        const int rv = wrow + 2 * tq;
        const int rvk[4] = {rv, rv + 1, rv + 8, rv + 9};
        uint32_t sw[4], ex[4];
        bool tv[4];
        uint32_t mref = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          tv[k] = rvk[k] < tmax;
          sw[k] = *reinterpret_cast<const uint32_t*>(stg[s].vs + 4 * rvk[k]);
          if (tv[k]) mref = __vmaxu4(mref, sw[k]);
        }
        mref = __vmaxu4(mref, __shfl_xor_sync(0xFFFFFFFFu, mref, 1));
        mref = __vmaxu4(mref, __shfl_xor_sync(0xFFFFFFFFu, mref, 2));
        bool far = false;  // a valid token's block scale 2^15 or more below its group's largest
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          ex[k] = tv[k] ? __vsubus4(0x0F0F0F0Fu, __vsub4(mref, sw[k])) : 0u;  // 15 - (s_max - s), at least 0
          far |= tv[k] && __vcmpeq4(ex[k], 0u) != 0u;
        }
        if (!__any_sync(0xFFFFFFFFu, far)) {
          uint32_t bh0, bh1, bl0, bl1;
          split_f16x2(*reinterpret_cast<const float2*>(pw + g * kPwLd + 2 * tq), bh0, bl0);
          split_f16x2(*reinterpret_cast<const float2*>(pw + g * kPwLd + 2 * tq + 8), bh1, bl1);
          const bool full16 = wrow + 16 <= tmax;
          const uint32_t k01 = (tv[0] ? 0x0000FFFFu : 0u) | (tv[1] ? 0xFFFF0000u : 0u);
          const uint32_t k89 = (tv[2] ? 0x0000FFFFu : 0u) | (tv[3] ? 0xFFFF0000u : 0u);
#pragma unroll
          for (int bb = 0; bb < 4; ++bb) {
            const int off = 32 * bb + 4 * g;
            const uint32_t w0 = *reinterpret_cast<const uint32_t*>(vb + swz(rvk[0], off));
            const uint32_t w1 = *reinterpret_cast<const uint32_t*>(vb + swz(rvk[1], off));
            const uint32_t w8 = *reinterpret_cast<const uint32_t*>(vb + swz(rvk[2], off));
            const uint32_t w9 = *reinterpret_cast<const uint32_t*>(vb + swz(rvk[3], off));
            // f16x2 2^(s - s_max) of the token pairs (rv, rv + 1), (rv + 8, rv + 9)
            const uint32_t sel = static_cast<uint32_t>(bb) | ((8u | bb) << 4) | ((4u + bb) << 8) | ((12u + bb) << 12);
            const uint32_t m01 = prmt(ex[0], ex[1], sel) << 10, m89 = prmt(ex[2], ex[3], sel) << 10;
            // dimension pairs (d, d + 1) and (d + 2, d + 3) of the token pairs
            const uint32_t x01 = prmt(w0, w1, 0x5140u), y01 = prmt(w0, w1, 0x7362u);
            const uint32_t x89 = prmt(w8, w9, 0x5140u), y89 = prmt(w8, w9, 0x7362u);
            uint32_t A0[4] = {hmul2(e4m3_lo_f16x2(x01), m01), hmul2(e4m3_hi_f16x2(x01), m01),
                              hmul2(e4m3_lo_f16x2(x89), m89), hmul2(e4m3_hi_f16x2(x89), m89)};
            uint32_t A1[4] = {hmul2(e4m3_lo_f16x2(y01), m01), hmul2(e4m3_hi_f16x2(y01), m01),
                              hmul2(e4m3_lo_f16x2(y89), m89), hmul2(e4m3_hi_f16x2(y89), m89)};
            if (!full16) {  // tokens past the sequence: their stale codes may not be finite
              A0[0] &= k01;
              A0[1] &= k01;
              A0[2] &= k89;
              A0[3] &= k89;
              A1[0] &= k01;
              A1[1] &= k01;
              A1[2] &= k89;
              A1[3] &= k89;
            }
            float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
            mma_16816(d0, A0[0], A0[1], A0[2], A0[3], bh0, bh1);
            mma_16816(d0, A0[0], A0[1], A0[2], A0[3], bl0, bl1);
            mma_16816(d1, A1[0], A1[1], A1[2], A1[3], bh0, bh1);
            mma_16816(d1, A1[0], A1[1], A1[2], A1[3], bl0, bl1);
            const float rf = ue8m0_value((mref >> (8 * bb)) & 0xFFu);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              O[bb][0][e] = fmaf(rf, d0[e], O[bb][0][e]);
              O[bb][1][e] = fmaf(rf, d1[e], O[bb][1][e]);
            }
          }
        } else {
          // fp32 FMAs: each lane its 16 dimensions x 2 heads over the 16 tokens
#pragma unroll 1
          for (int kk = 0; kk < 16; ++kk) {
            const int r = wrow + kk;
            if (r >= tmax) break;
            const float q0 = pw[(2 * tq) * kPwLd + kk], q1 = pw[(2 * tq + 1) * kPwLd + kk];
            const uint32_t swd = *reinterpret_cast<const uint32_t*>(stg[s].vs + 4 * r);
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) {
              const uint32_t w = *reinterpret_cast<const uint32_t*>(vb + swz(r, 32 * bb + 4 * g));
              const float f = ue8m0_value((swd >> (8 * bb)) & 0xFFu);
              const float2 lo = e4m3x2_to_float2(w), hi = e4m3x2_to_float2(w >> 16);
              const float vv[4] = {lo.x * f, lo.y * f, hi.x * f, hi.y * f};
#pragma unroll
              for (int tt = 0; tt < 2; ++tt) {
                O[bb][tt][0] = fmaf(q0, vv[2 * tt], O[bb][tt][0]);
                O[bb][tt][1] = fmaf(q1, vv[2 * tt], O[bb][tt][1]);
                O[bb][tt][2] = fmaf(q0, vv[2 * tt + 1], O[bb][tt][2]);
                O[bb][tt][3] = fmaf(q1, vv[2 * tt + 1], O[bb][tt][3]);
              }
            }
          }
        }
      }
      __syncwarp();  // the warp is done with the stage (and pw) before it releases it
      if (lane == 0) mbar_arrive(&empty[s]);
    }
#pragma unroll
    for (int i2 = 0; i2 < 2; ++i2) {
      l_part[i2] += __shfl_xor_sync(0xFFFFFFFFu, l_part[i2], 4);
      l_part[i2] += __shfl_xor_sync(0xFFFFFFFFu, l_part[i2], 8);
      l_part[i2] += __shfl_xor_sync(0xFFFFFFFFu, l_part[i2], 16);
    }
  }
  __syncthreads();  // every warp is done with the ring and every copy has landed

  if (t == 0) {
    ATTN_STAMP(1);
    if (a.trace != nullptr) a.trace[((blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x) * 64 + 2] = c1 - c0;
  }
  // ---- merge the warps' states: the block's max, sum and unnormalised
  // output per head, one record each
  float* wacc = reinterpret_cast<float*>(stg);  // reuse the ring: [kCWarps][G][D]
  if (warp < kCWarps) {
#pragma unroll
    for (int i2 = 0; i2 < 2; ++i2) {
      const int hh = 2 * tq + i2;
      if (hh < G) {
#pragma unroll
        for (int bb = 0; bb < 4; ++bb)
          *reinterpret_cast<float4*>(wacc + (warp * G + hh) * kD + 32 * bb + 4 * g) =
              make_float4(O[bb][0][i2], O[bb][0][2 + i2], O[bb][1][i2], O[bb][1][2 + i2]);
        if (g == 0) {
          red_max[warp * G + hh] = m_run[i2];
          red_sum[warp * G + hh] = l_part[i2];
        }
      }
    }
  }
  __syncthreads();
  for (int i = t; i < G * kD; i += kAThreads) {
    const int hh = i / kD, d = i % kD;
    float M = red_max[hh];
#pragma unroll
    for (int w = 1; w < kCWarps; ++w) M = fmaxf(M, red_max[w * G + hh]);
    float o = 0.f, l = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kCWarps; ++w) {
        const float mw = red_max[w * G + hh];
        if (mw == -INFINITY) continue;
        const float f = expf(mw - M);
        o = fmaf(f, wacc[(w * G + hh) * kD + d], o);
        l = fmaf(f, red_sum[w * G + hh], l);
      }
    }
    float* rec = a.part + ((static_cast<size_t>(b) * a.Hq + hk * G + hh) * a.nsplit + split) * (2 + kD);
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
  // about two blocks per SM (the ring's shared memory lets two be resident)
  // the chunks are spread thinner.
  const int max_chunks = (max_pages * P + kC - 1) / kC;
  int per = chunks_per_block;
  const int want = (2 * sms + B * Hkv - 1) / (B * Hkv);
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
