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
//   attn_combine_kernel<G>  merges the splits of one (sequence, KV head)'s
//                           G query heads and writes the bf16 output.
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
constexpr int kAThreads = 32 * (kCWarps + 2);     // + the copy warp and the scale warp
constexpr int kAStages = 3;
constexpr int kD = kAttnHeadDim;
constexpr int kC = kAttnChunk;
constexpr uint32_t kCodeBytes = kC * kD;          // 16 KB of K (or V) codes per chunk
constexpr uint32_t kScaleBytes = kC * kD / 32;    // 512 B of scales per chunk
constexpr int kPwLd = 16;                         // row stride (floats) of a warp's p[head][token]
static_assert(kC == 16 * kCWarps, "a consumer warp owns 16 tokens of a chunk");

struct __align__(1024) AttnStage {
  uint8_t k[kCodeBytes];  // [token][128] swizzled: 16-byte piece j of row r at piece j ^ (r % 8)
  uint8_t v[kCodeBytes];
  uint8_t ks[kScaleBytes];  // [token][4]
  uint8_t vs[kScaleBytes];
};
static_assert(sizeof(AttnStage) % 1024 == 0, "stages stay 1024-byte aligned");
// What the scale warp derives from a chunk's V scales once, for the consumer
// lanes (warp w, column pair tq) that share tokens rv = 16 w + 2 tq +
// {0, 1, 8, 9}: per 32-dimension block bb the f16x2 multipliers 2^(s - s_max)
// of the token pairs (rv, rv + 1) and (rv + 8, rv + 9), s_max the block's
// largest scale among warp w's tokens of the item so far (byte bb of
// smax[w]; it only grows within an item).
struct AttnPrep {
  uint4 vm[kCWarps * 4][2];
  uint32_t smax[kCWarps];
};
constexpr size_t kAttnSmem = kAStages * sizeof(AttnStage) + 1024;  // + alignment slack

// Byte offset of (row, byte) in a 128-byte-swizzled tile whose base is
// 1024-byte aligned.
__device__ __forceinline__ int swz(int row, int off) {
  return row * 128 + ((((off >> 4) ^ row) & 7) << 4) + (off & 15);
}
// Two floats as f16x2 (round to nearest even), `lo` in the lower half.
__device__ __forceinline__ uint32_t f16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// 2^x (the special-function unit's approximation, relative error below
// 2^-22; results below 2^-126 flush to 0)
__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
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
// Two E4M3 codes (low byte first) as two floats: exact.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two & 0xFFFFu), __NV_E4M3);
  return __half22float2(__half2(h));
}
// 2^(s - 127) for a UE8M0 byte s (s = 0 is the subnormal 2^-127).
__device__ __forceinline__ float ue8m0_value(uint32_t s) {
  return s != 0 ? __uint_as_float(s << 23) : __uint_as_float(0x00400000u);
}
// 2^(s - 127) for byte bb of a word of UE8M0 scales, with s = 0 read as 0
// (a block whose scale is 2^-127 holds values below 2^-118)
template <int bb>
__device__ __forceinline__ float ue8m0_byte(uint32_t w) {
  return __uint_as_float((bb < 3 ? (w << (23 - 8 * bb)) : (w >> 1)) & 0x7F800000u);
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

// One work item: chunks [c0, c1) of KV head hk of sequence b (its split
// `split`); n is the sequence's length (0 when it is out of range).
struct AttnItem {
  int b, hk, split, n, c0, c1;
};
// Items are numbered with the KV head fastest, then the sequence, then the
// split, so that the blocks take the full-size splits first.
__device__ __forceinline__ AttnItem attn_item(const AttnArgs& a, int it) {
  AttnItem w;
  w.hk = it % a.Hkv;
  const int r = it / a.Hkv;
  w.b = r % a.B;
  w.split = r / a.B;
  const int len = a.seq_lens[w.b];
  w.n = (len >= 1 && len <= a.max_pages * a.P) ? len : 0;
  // every split the same number of chunks of the longest sequence's
  const int per = (a.max_pages * a.P + kC * a.nsplit - 1) / (kC * a.nsplit);
  const int nchunks = (w.n + kC - 1) / kC;
  w.c0 = min(nchunks, w.split * per);
  w.c1 = min(nchunks, w.c0 + per);
  return w;
}

// What a stage holds, written by the producer: the chunk's item and position.
enum : uint32_t {
  kMetaFirst = 1,  // the item's first chunk
  kMetaLast = 2,   // the item's last chunk
  kMetaOk = 4,     // every page id of the chunk was in range (else the chunk is skipped)
  kMetaFar = 8,    // p . v in fp32 FMAs (a V scale 2^15 or more below its group's largest)
  kMetaEnd = 16,   // no more work: the consumers leave
};
struct ChunkMeta {
  int b, hk, split, n, c;
  uint32_t flags;
  int pid[kC / 16];  // the chunk's page ids (-1: not loaded)
};

// Persistent: each block takes work items from a counter shared by the grid
// (largest first, by the item order) and streams their chunks as one
// sequence through the ring, so the copies of an item's first chunks are in
// flight while the previous item is finished; at an item's end the consumer
// warps merge their states in the stage of its last chunk and write the
// item's record.  The second launch resets the counter.
template <int G>
__global__ void __launch_bounds__(kAThreads, 2) paged_decode_kernel(const __grid_constant__ AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  AttnStage* stg = reinterpret_cast<AttnStage*>(smem_align(smem_raw, 1024));
  // each consumer warp's probabilities of its 16 tokens: [warp][head][token]
  __shared__ __align__(16) float pws[kCWarps * 8 * kPwLd];
  __shared__ float red_max[kCWarps * G], red_sum[kCWarps * G];
  __shared__ __align__(8) uint64_t full[kAStages], posted[kAStages], ready[kAStages], empty[kAStages], qfree[2],
      mrg[2];
  __shared__ AttnPrep prep[kAStages];
  __shared__ ChunkMeta meta[kAStages];
  // q of an item's group as the B operand of the score MMA (two buffers, by
  // item parity), per lane: block bb's two k-steps in qfrag[.][bb][lane];
  // sm_scale log2(e) / 2^e per head (the softmax runs in base 2)
  __shared__ uint4 qfrag[2][4][32];
  __shared__ float qscale[2][8];

  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int items = a.nsplit * a.B * a.Hkv;
  // the combining launch may be scheduled now; it waits for this grid to finish
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (t == 0) {
#pragma unroll
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&posted[s], 32);
      mbar_init(&ready[s], 32);
      mbar_init(&empty[s], kCWarps);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mbar_init(&qfree[i], kCWarps);
      mbar_init(&mrg[i], kCWarps);
    }
    mbar_fence_init();
    ATTN_STAMP(0);
  }
  __syncthreads();

  const int g = lane >> 2, tq = lane & 3;  // mma fragment row group and column pair

  if (warp >= kCWarps) {
    // ---- producers.  The copy warp puts chunk number q of the block's
    // stream into stage q % kAStages as soon as the consumers have left the
    // chunk that held it; lane i copies the chunk's page i.  Pages past a
    // sequence's last one are not loaded (their tokens are masked); a page id
    // outside [0, num_pages) is reported and the chunk skipped.  The scale
    // warp, once a chunk has landed, derives its V-scale multipliers (and an
    // item's q fragments) and marks it ready.
    const int ppc = kC / a.P;
    const uint32_t cb = static_cast<uint32_t>(a.P) * kD;
    const uint64_t pol = l2_policy_evict_first();
    if (lane == 0) {
      tma_prefetch_desc(&a.tm_k);
      tma_prefetch_desc(&a.tm_v);
    }
    // the next non-empty item from the shared counter (false: none left)
    auto grab = [&](AttnItem& w) -> bool {
      int found = 0;
      if (lane == 0) {
        for (;;) {
          const int it = static_cast<int>(atomicAdd(a.work, 1u));
          if (it >= items) break;
          w = attn_item(a, it);
          if (w.n == 0 && w.split == 0 && w.hk == 0) attn_error(a, 1u, 1u);  // a length outside [1, max_pages P]
          if (w.c0 < w.c1) {
            found = 1;
            break;
          }
        }
      }
      found = __shfl_sync(0xFFFFFFFFu, found, 0);
      w.b = __shfl_sync(0xFFFFFFFFu, w.b, 0);
      w.hk = __shfl_sync(0xFFFFFFFFu, w.hk, 0);
      w.split = __shfl_sync(0xFFFFFFFFu, w.split, 0);
      w.n = __shfl_sync(0xFFFFFFFFu, w.n, 0);
      w.c0 = __shfl_sync(0xFFFFFFFFu, w.c0, 0);
      w.c1 = __shfl_sync(0xFFFFFFFFu, w.c1, 0);
      return found != 0;
    };
    // issue cursor: chunk c of item cur (item nxt grabbed one ahead); lane i
    // holds page id pid of the chunk's page i (loaded one issue ahead)
    AttnItem cur{}, nxt{};
    bool have_cur = false, have_nxt = false, nxt_taken = false;
    int c = 0;
    int pid = -1, np = 0;
    auto load_pids = [&]() {
      const int npages = (cur.n + a.P - 1) / a.P;
      np = min(ppc, npages - c * ppc);
      pid = lane < np ? a.block_table[static_cast<size_t>(cur.b) * a.max_pages + c * ppc + lane] : -1;
    };
    bool ended = false;
    auto issue_next = [&](int s) {
      if (!have_cur) {
        if (lane == 0) {
          meta[s].flags = kMetaEnd;
          mbar_arrive(&full[s]);
        }
        __syncwarp();
        mbar_arrive(&posted[s]);
        ended = true;
        return;
      }
      const bool mine = lane < np;
      const bool good = !mine || (pid >= 0 && pid < a.num_pages);
      const bool all_good = __all_sync(0xFFFFFFFFu, good);
      const uint32_t npg = __popc(__ballot_sync(0xFFFFFFFFu, mine && good));
      if (lane == 0) {
        if (!all_good) attn_error(a, 1u, 2u);
        meta[s].b = cur.b;
        meta[s].hk = cur.hk;
        meta[s].split = cur.split;
        meta[s].n = cur.n;
        meta[s].c = c;
        meta[s].flags = (c == cur.c0 ? kMetaFirst : 0u) | (c + 1 == cur.c1 ? kMetaLast : 0u) |
                        (all_good ? kMetaOk : 0u);
      }
      if (lane < kC / 16) meta[s].pid[lane] = (mine && good) ? pid : -1;
      fence_proxy_async_shared();  // the stage's earlier generic reads come before the copies' writes
      if (lane == 0) mbar_arrive_expect_tx(&full[s], npg * 2u * cb);
      __syncwarp();
      if (mine && good) {
        const int y = (pid * a.Hkv + cur.hk) * a.P;  // first row of the (page, head) block
        tma_load_2d(stg[s].k + lane * cb, &a.tm_k, &full[s], 0, y, pol);
        tma_load_2d(stg[s].v + lane * cb, &a.tm_v, &full[s], 0, y, pol);
      }
      mbar_arrive(&posted[s]);  // the chunk's meta is written: its scales may be fetched
      // the next item is taken once its predecessor's first chunk is on its way
      if (!nxt_taken) {
        have_nxt = grab(nxt);
        nxt_taken = true;
      }
      if (++c >= cur.c1) {
        have_cur = have_nxt;
        cur = nxt;
        c = cur.c0;
        nxt_taken = false;
      }
      if (have_cur) load_pids();
    };
    // q of item (b, hk) into buffer qb: lane (g, tq) holds head g's B
    // fragments: k-step j (dimensions of block j / 2) pairs mma column
    // k = 2 tq + {0, 1} with dimension 32 (j / 2) + 8 tq + 4 (j % 2) + {0, 1}
    // and k = 2 tq + 8 + {0, 1} with + {2, 3}, so that a consumer lane's
    // 8-byte K load feeds two k-steps.  Each head is scaled by the power of
    // two 2^e that puts its largest |q| in [2^13, 2^14): exact in f16.
    auto load_q = [&](int b, int hk, int qb) {
      float qv[32];
      if (g < G) {
        const uint4* qp = reinterpret_cast<const uint4*>(a.q + (static_cast<size_t>(b) * a.Hq + hk * G + g) * kD);
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
          const uint4 v = qp[4 * bb + tq];
          const uint32_t vs4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            qv[8 * bb + 2 * j] = bf16_bits_to_float(vs4[j] & 0xFFFFu);
            qv[8 * bb + 2 * j + 1] = bf16_bits_to_float(vs4[j] >> 16);
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
        qfrag[qb][bb][lane] = make_uint4(f16x2_rn(qv[8 * bb] * up, qv[8 * bb + 1] * up),
                                         f16x2_rn(qv[8 * bb + 2] * up, qv[8 * bb + 3] * up),
                                         f16x2_rn(qv[8 * bb + 4] * up, qv[8 * bb + 5] * up),
                                         f16x2_rn(qv[8 * bb + 6] * up, qv[8 * bb + 7] * up));
      if (tq == 0) qscale[qb][g] = ldexpf(a.sm_scale * 1.4426950408889634f, -e);
    };
    // the V-scale multipliers of the chunk in stage s, lane 4 w + tq those of
    // consumer warp w's column pair tq; rref is warp w's running maximum
    uint32_t rref = 0;
    auto prepare = [&](int s) {
      const int pwp = lane >> 2, ptq = lane & 3;
      const int tmax = min(kC, meta[s].n - meta[s].c * kC);
      const int rv = 16 * pwp + 2 * ptq;
      const int rows[4] = {rv, rv + 1, rv + 8, rv + 9};
      uint32_t sw[4], ex[4];
      bool tv[4];
      uint32_t mref = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        tv[k] = rows[k] < tmax;
        sw[k] = *reinterpret_cast<const uint32_t*>(stg[s].vs + 4 * rows[k]);
        if (tv[k]) mref = __vmaxu4(mref, sw[k]);
      }
      mref = __vmaxu4(mref, __shfl_xor_sync(0xFFFFFFFFu, mref, 1));
      mref = __vmaxu4(mref, __shfl_xor_sync(0xFFFFFFFFu, mref, 2));
      if (meta[s].flags & kMetaFirst) rref = 0;
      mref = __vmaxu4(mref, rref);
      rref = mref;
      bool far = false;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        ex[k] = tv[k] ? __vsubus4(0x0F0F0F0Fu, __vsub4(mref, sw[k])) : 0u;  // 15 - (s_max - s), at least 0
        far |= tv[k] && __vcmpeq4(ex[k], 0u) != 0u;
      }
      far = __any_sync(0xFFFFFFFFu, far);
      uint32_t m01[4], m89[4];
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        // bytes (s0, 0, s1, 0) of the pair's exponents, shifted into f16 exponent fields
        const uint32_t sel = 0xC480u + 0x1111u * bb;
        m01[bb] = prmt(ex[0], ex[1], sel) << 10;
        m89[bb] = prmt(ex[2], ex[3], sel) << 10;
      }
      prep[s].vm[lane][0] = make_uint4(m01[0], m01[1], m01[2], m01[3]);
      prep[s].vm[lane][1] = make_uint4(m89[0], m89[1], m89[2], m89[3]);
      if (ptq == 0) prep[s].smax[pwp] = mref;
      // one warp's far chunk sends the whole chunk to the fp32 path
      if (lane == 0 && far) meta[s].flags |= kMetaFar;
    };

    if (warp == kCWarps) {
      // (only this warp takes work from the counter)
      have_cur = grab(cur);
      c = cur.c0;
      if (have_cur) load_pids();
      int issued = 0;
      for (int q = 0; !ended; ++q) {
        const int s = q % kAStages;
        if (q >= kAStages && !wait_phase(&empty[s], static_cast<uint32_t>(q / kAStages - 1) & 1u, a.timeout_ns)) {
          if (lane == 0) attn_error(a, 5u, 4u);  // FSOPS_ERR_TIMEOUT
          break;
        }
        issue_next(s);
        if (lane == 0 && q < 10) ATTN_STAMP(54 + q);
        issued = q + 1;
      }
      // the last chunks' copies land before the block leaves (every earlier
      // chunk of a stage was consumed before the stage was refilled)
      for (int q = max(0, issued - kAStages); q < issued; ++q)
        wait_phase(&full[q % kAStages], static_cast<uint32_t>(q / kAStages) & 1u, 200000000ull);
    } else {
      int kq = 0;  // items begun
      for (int q = 0;; ++q) {
        const int s = q % kAStages;
        const uint32_t par = static_cast<uint32_t>(q / kAStages) & 1u;
        if (!wait_phase(&posted[s], par, a.timeout_ns)) {
          if (lane == 0) attn_error(a, 5u, 3u);  // FSOPS_ERR_TIMEOUT
          break;
        }
        // the chunk's K and V scales (tokens 4 lane .. 4 lane + 3, 16 bytes
        // each), loaded while its codes are on the way
        const uint32_t fl = meta[s].flags;
        uint4 ksv = make_uint4(0u, 0u, 0u, 0u), vsv = ksv;
        if (!(fl & kMetaEnd)) {
          const int tok = 4 * lane;
          const int id = meta[s].pid[tok / a.P];
          if (id >= 0) {
            const size_t row = (static_cast<size_t>(id) * a.Hkv + meta[s].hk) * a.P + tok % a.P;
            ksv = *reinterpret_cast<const uint4*>(a.k_scales + row * (kD / 32));
            vsv = *reinterpret_cast<const uint4*>(a.v_scales + row * (kD / 32));
          }
        }
        if (!wait_phase(&full[s], par, a.timeout_ns)) {
          if (lane == 0) attn_error(a, 5u, 3u);  // FSOPS_ERR_TIMEOUT
          break;
        }
        if (lane == 0 && q < 10) ATTN_STAMP(44 + q);
        if (fl & kMetaEnd) {
          __syncwarp();
          mbar_arrive(&ready[s]);
          break;
        }
        reinterpret_cast<uint4*>(stg[s].ks)[lane] = ksv;
        reinterpret_cast<uint4*>(stg[s].vs)[lane] = vsv;
        __syncwarp();
        if (fl & kMetaFirst) {
          // the buffer's previous item (two back) is done with it
          const int qb = kq & 1;
          if (kq >= 2 && !wait_phase(&qfree[qb], static_cast<uint32_t>((kq >> 1) - 1) & 1u, a.timeout_ns)) {
            if (lane == 0) attn_error(a, 5u, 5u);  // FSOPS_ERR_TIMEOUT
            break;
          }
          load_q(meta[s].b, meta[s].hk, qb);
          ++kq;
        }
        prepare(s);
        __syncwarp();
        mbar_arrive(&ready[s]);
      }
    }
  } else {
    // ---- consumer warp: tokens 16 warp .. 16 warp + 15 of every chunk.
    // Its state: the p . v sums O^T[d][head] of the warp's tokens in eight
    // 16-row tiles T (rows g and g + 8 are dimensions 16 g + 2 T and
    // 16 g + 2 T + 1, so a lane's 16 dimensions lie in one 32-dimension V
    // scale block, g / 2; columns heads 2 tq and 2 tq + 1) in units of
    // 2^(ref_e - 127), ref_e that block's running largest scale among the
    // warp's tokens; and the running max and partial sums of the lane's two
    // heads.
    const int wrow = 16 * warp;
    float* pw = pws + warp * 8 * kPwLd;
    // the lane's swizzled offsets in a stage: K rows wrow + g (+ 8), bytes
    // 32 bb + 8 tq at kofs + ((32 bb) ^ kxor); V rows wrow + 2 tq (+ 1, + 8,
    // + 9), bytes 16 g .. 16 g + 15 at vofs[k & 1] + 1024 (k >> 1)
    const int kofs = (wrow + g) * 128 + 16 * (((tq >> 1) ^ g) & 1) + 8 * (tq & 1), kxor = 32 * (g >> 1);
    const int vofs[2] = {(wrow + 2 * tq) * 128 + ((g ^ (2 * tq)) << 4),
                         (wrow + 2 * tq + 1) * 128 + ((g ^ (2 * tq + 1)) << 4)};
    int kq = 0, qb = 0;
    const int vbb = g >> 1;  // the lane's V scale block
    float O[8][4];
    float m_run[2], l_part[2];
    int ref_e = 0;
    float hs[2] = {0.f, 0.f};  // sm_scale log2(e) / 2^e of heads 2 tq and 2 tq + 1
    for (int seq = 0;; ++seq) {
      const int s = seq % kAStages;
      const uint32_t par = static_cast<uint32_t>(seq / kAStages) & 1u;
      if (t == 0 && seq < 10) ATTN_STAMP(4 + 4 * seq);
      if (!wait_phase(&full[s], par, a.timeout_ns) || !wait_phase(&ready[s], par, a.timeout_ns)) {
        if (lane == 0) attn_error(a, 5u, 3u);  // FSOPS_ERR_TIMEOUT
        break;
      }
      if (t == 0 && seq < 10) ATTN_STAMP(5 + 4 * seq);
      const ChunkMeta m = meta[s];
      if (m.flags & kMetaEnd) break;
      bool released = false;  // the stage was released before the chunk's p . v
      if (m.flags & kMetaFirst) {
#pragma unroll
        for (int tt = 0; tt < 8; ++tt)
#pragma unroll
          for (int e = 0; e < 4; ++e) O[tt][e] = 0.f;
        m_run[0] = m_run[1] = -INFINITY;
        l_part[0] = l_part[1] = 0.f;
        ref_e = 0;  // the item's running scale maximum starts below any chunk's
        qb = kq & 1;
        hs[0] = qscale[qb][2 * tq];
        hs[1] = qscale[qb][2 * tq + 1];
      }
        const int tmax = min(kC, m.n - m.c * kC);  // valid rows of the chunk
        if ((m.flags & kMetaOk) != 0 && wrow < tmax) {
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
              // swz(r0, 32 bb + 8 tq): rows r0 and r0 + 8 share r0 % 8 = g
              const int ko = kofs + ((32 * bb) ^ kxor);
              const uint2 x0 = *reinterpret_cast<const uint2*>(kb + ko);
              const uint2 x1 = *reinterpret_cast<const uint2*>(kb + ko + 1024);
              const uint4 bq = qfrag[qb][bb][lane];
              float d[4] = {0.f, 0.f, 0.f, 0.f};
              mma_16816(d, e4m3_lo_f16x2(x0.x), e4m3_lo_f16x2(x1.x), e4m3_hi_f16x2(x0.x), e4m3_hi_f16x2(x1.x), bq.x,
                        bq.y);
              mma_16816(d, e4m3_lo_f16x2(x0.y), e4m3_lo_f16x2(x1.y), e4m3_hi_f16x2(x0.y), e4m3_hi_f16x2(x1.y), bq.z,
                        bq.w);
              const float f0 = bb == 0   ? ue8m0_byte<0>(kw0)
                             : bb == 1 ? ue8m0_byte<1>(kw0)
                             : bb == 2 ? ue8m0_byte<2>(kw0)
                                       : ue8m0_byte<3>(kw0);
            const float f1 = bb == 0   ? ue8m0_byte<0>(kw1)
                             : bb == 1 ? ue8m0_byte<1>(kw1)
                             : bb == 2 ? ue8m0_byte<2>(kw1)
                                       : ue8m0_byte<3>(kw1);
              sc[0] = fmaf(f0, d[0], sc[0]);
              sc[1] = fmaf(f0, d[1], sc[1]);
              sc[2] = fmaf(f1, d[2], sc[2]);
              sc[3] = fmaf(f1, d[3], sc[3]);
            }
          }
          // ---- the warp's online softmax over its 16 tokens, per head (the
          // running max is only reduced again when some score exceeds it)
          const bool v0 = r0 < tmax, v1 = r1 < tmax;
          float x[2][2];
          bool grow = false;
#pragma unroll
          for (int i2 = 0; i2 < 2; ++i2) {
            const bool hv = 2 * tq + i2 < G;
            x[i2][0] = (v0 && hv) ? sc[i2] * hs[i2] : -INFINITY;
            x[i2][1] = (v1 && hv) ? sc[2 + i2] * hs[i2] : -INFINITY;
            grow |= fmaxf(x[i2][0], x[i2][1]) > m_run[i2];
          }
          float al[2] = {1.f, 1.f};
          if (__any_sync(0xFFFFFFFFu, grow)) {
#pragma unroll
            for (int i2 = 0; i2 < 2; ++i2) {
              float cm = fmaxf(x[i2][0], x[i2][1]);
              cm = fmaxf(cm, __shfl_xor_sync(0xFFFFFFFFu, cm, 4));
              cm = fmaxf(cm, __shfl_xor_sync(0xFFFFFFFFu, cm, 8));
              cm = fmaxf(cm, __shfl_xor_sync(0xFFFFFFFFu, cm, 16));
              const float mn = fmaxf(m_run[i2], cm);
              // no valid token yet: mn = -inf and nothing is added
              al[i2] = mn == -INFINITY ? 1.f : ex2_approx(m_run[i2] - mn);
              m_run[i2] = mn;
            }
            if (al[0] != 1.f || al[1] != 1.f) {
#pragma unroll
              for (int tt = 0; tt < 8; ++tt) {
                O[tt][0] *= al[0];
                O[tt][1] *= al[1];
                O[tt][2] *= al[0];
                O[tt][3] *= al[1];
              }
            }
          }
#pragma unroll
          for (int i2 = 0; i2 < 2; ++i2) {
            const int hh = 2 * tq + i2;
            const float ms = m_run[i2] == -INFINITY ? 0.f : m_run[i2];
            const float p0 = ex2_approx(x[i2][0] - ms), p1 = ex2_approx(x[i2][1] - ms);  // 0 for -inf
            l_part[i2] = fmaf(l_part[i2], al[i2], p0 + p1);
            pw[hh * kPwLd + g] = p0;
            pw[hh * kPwLd + g + 8] = p1;
          }
          __syncwarp();  // pw is written before the lanes read it
          if (t == 0 && seq < 10) ATTN_STAMP(6 + 4 * seq);

          // ---- p . v: A = V^T (rows: dimensions, k: tokens rv, rv + 1, rv + 8,
          // rv + 9 of the lane), B = p of head g; the sums stay in units of
          // 2^(ref_e - 127), ref_e the running largest scale of block vbb
          const int rv = wrow + 2 * tq;
          const int rvk[4] = {rv, rv + 1, rv + 8, rv + 9};
          const AttnPrep& pr = prep[s];
          {
            const int ne = static_cast<int>((pr.smax[warp] >> (8 * vbb)) & 0xFFu);
            if (ne != ref_e) {
              const float f = __uint_as_float(static_cast<uint32_t>(max(127 + ref_e - ne, 0)) << 23);
#pragma unroll
              for (int tt = 0; tt < 8; ++tt)
#pragma unroll
                for (int e = 0; e < 4; ++e) O[tt][e] *= f;
              ref_e = ne;
            }
          }
          uint4 W[4];  // the lane's 16 dimensions of its four tokens
#pragma unroll
          for (int k = 0; k < 4; ++k) W[k] = *reinterpret_cast<const uint4*>(vb + vofs[k & 1] + 1024 * (k >> 1));
          if ((m.flags & kMetaFar) == 0) {
            // f16x2 2^(s - ref) of the token pairs (rv, rv + 1) and (rv + 8, rv + 9)
            const uint32_t m01 = reinterpret_cast<const uint32_t*>(&pr.vm[4 * warp + tq][0])[vbb];
            const uint32_t m89 = reinterpret_cast<const uint32_t*>(&pr.vm[4 * warp + tq][1])[vbb];
            if (!(m.flags & kMetaLast)) {
              // everything the warp reads of the stage is in registers: release it now
              __syncwarp();
              if (t == 0 && seq < 10) ATTN_STAMP(7 + 4 * seq);
              if (lane == 0) mbar_arrive(&empty[s]);
              released = true;
            }
            uint32_t bh0, bh1, bl0, bl1;
            split_f16x2(*reinterpret_cast<const float2*>(pw + g * kPwLd + 2 * tq), bh0, bl0);
            split_f16x2(*reinterpret_cast<const float2*>(pw + g * kPwLd + 2 * tq + 8), bh1, bl1);
            const bool full16 = wrow + 16 <= tmax;
            const uint32_t k01 = (rvk[0] < tmax ? 0x0000FFFFu : 0u) | (rvk[1] < tmax ? 0xFFFF0000u : 0u);
            const uint32_t k89 = (rvk[2] < tmax ? 0x0000FFFFu : 0u) | (rvk[3] < tmax ? 0xFFFF0000u : 0u);
            const uint32_t w0[4] = {W[0].x, W[0].y, W[0].z, W[0].w}, w1[4] = {W[1].x, W[1].y, W[1].z, W[1].w};
            const uint32_t w8[4] = {W[2].x, W[2].y, W[2].z, W[2].w}, w9[4] = {W[3].x, W[3].y, W[3].z, W[3].w};
#pragma unroll
            for (int tt = 0; tt < 8; ++tt) {
              // dimensions 16 g + 2 tt and + 1 of the token pairs
              const uint32_t sel = (tt & 1) ? 0x7362u : 0x5140u;
              const uint32_t x01 = prmt(w0[tt >> 1], w1[tt >> 1], sel), x89 = prmt(w8[tt >> 1], w9[tt >> 1], sel);
              uint32_t A[4] = {hmul2(e4m3_lo_f16x2(x01), m01), hmul2(e4m3_hi_f16x2(x01), m01),
                               hmul2(e4m3_lo_f16x2(x89), m89), hmul2(e4m3_hi_f16x2(x89), m89)};
              if (!full16) {  // tokens past the sequence: their stale codes may not be finite
                A[0] &= k01;
                A[1] &= k01;
                A[2] &= k89;
                A[3] &= k89;
              }
              mma_16816(O[tt], A[0], A[1], A[2], A[3], bh0, bh1);
              mma_16816(O[tt], A[0], A[1], A[2], A[3], bl0, bl1);
            }
          } else {
            // fp32 FMAs: each lane its 16 dimensions x 2 heads over the 16 tokens
#pragma unroll 1
            for (int kk = 0; kk < 16; ++kk) {
              const int r = wrow + kk;
              if (r >= tmax) break;
              const float q0 = pw[(2 * tq) * kPwLd + kk], q1 = pw[(2 * tq + 1) * kPwLd + kk];
              const int se = static_cast<int>(stg[s].vs[4 * r + vbb]);
              const float f = __uint_as_float(static_cast<uint32_t>(max(127 + se - ref_e, 0)) << 23);
              const uint4 vw = *reinterpret_cast<const uint4*>(vb + swz(r, 16 * g));
              const uint32_t vws[4] = {vw.x, vw.y, vw.z, vw.w};
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float2 lo = e4m3x2_to_float2(vws[j]), hi = e4m3x2_to_float2(vws[j] >> 16);
                const float vv[4] = {lo.x * f, lo.y * f, hi.x * f, hi.y * f};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  // dimension 16 g + 4 j + e: tile (4 j + e) / 2, row half e % 2
                  float* o = O[2 * j + (e >> 1)] + 2 * (e & 1);
                  o[0] = fmaf(q0, vv[e], o[0]);
                  o[1] = fmaf(q1, vv[e], o[1]);
                }
              }
            }
          }
        }
      if (!(m.flags & kMetaLast)) {
        if (!released) {
          __syncwarp();  // the warp is done with the stage before it releases it
          if (t == 0 && seq < 10) ATTN_STAMP(7 + 4 * seq);
          if (lane == 0) mbar_arrive(&empty[s]);
        }
        continue;
      }
      // ---- the item's end: merge the warps' states in its last chunk's
      // stage (the item's max, sum and unnormalised output per head, one
      // record each); the stage is released afterwards
      float l_sum[2];
#pragma unroll
      for (int i2 = 0; i2 < 2; ++i2) {
        l_sum[i2] = l_part[i2];
        l_sum[i2] += __shfl_xor_sync(0xFFFFFFFFu, l_sum[i2], 4);
        l_sum[i2] += __shfl_xor_sync(0xFFFFFFFFu, l_sum[i2], 8);
        l_sum[i2] += __shfl_xor_sync(0xFFFFFFFFu, l_sum[i2], 16);
      }
      const uint32_t mpar = static_cast<uint32_t>(kq) & 1u;
      __syncwarp();
      if (lane == 0) mbar_arrive(&mrg[0]);
      if (!wait_phase(&mrg[0], mpar, a.timeout_ns)) {  // every warp is done with the stage
        if (lane == 0) attn_error(a, 5u, 6u);  // FSOPS_ERR_TIMEOUT
        break;
      }
      float* wacc = reinterpret_cast<float*>(&stg[s]);  // [kCWarps][G][D]
      const float unit = ue8m0_value(static_cast<uint32_t>(ref_e));  // the sums' unit 2^(ref_e - 127)
#pragma unroll
      for (int i2 = 0; i2 < 2; ++i2) {
        const int hh = 2 * tq + i2;
        if (hh < G) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<float4*>(wacc + (warp * G + hh) * kD + 16 * g + 4 * j) =
                make_float4(O[2 * j][i2] * unit, O[2 * j][2 + i2] * unit, O[2 * j + 1][i2] * unit,
                            O[2 * j + 1][2 + i2] * unit);
          if (g == 0) {
            red_max[warp * G + hh] = m_run[i2];
            red_sum[warp * G + hh] = l_sum[i2];
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&mrg[1]);
      if (!wait_phase(&mrg[1], mpar, a.timeout_ns)) {
        if (lane == 0) attn_error(a, 5u, 6u);  // FSOPS_ERR_TIMEOUT
        break;
      }
      for (int i = t; i < G * kD; i += 32 * kCWarps) {
        const int hh = i / kD, d = i % kD;
        float M = red_max[hh];
#pragma unroll
        for (int w2 = 1; w2 < kCWarps; ++w2) M = fmaxf(M, red_max[w2 * G + hh]);
        float o = 0.f, l = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w2 = 0; w2 < kCWarps; ++w2) {
            const float mw = red_max[w2 * G + hh];
            if (mw == -INFINITY) continue;
            const float f = exp2f(mw - M);
            o = fmaf(f, wacc[(w2 * G + hh) * kD + d], o);
            l = fmaf(f, red_sum[w2 * G + hh], l);
          }
        }
        float* rec = a.part + ((static_cast<size_t>(m.b) * a.Hq + m.hk * G + hh) * a.nsplit + m.split) * (2 + kD);
        rec[2 + d] = o;
        if (d == 0) {
          rec[0] = M;
          rec[1] = l;
        }
      }
      __syncwarp();  // the warp is done with wacc and with this item's q
      if (lane == 0) {
        mbar_arrive(&empty[s]);
        mbar_arrive(&qfree[qb]);
      }
      ++kq;
    }
    if (t == 0) ATTN_STAMP(1);
  }
}

// One block per (KV head, sequence): thread (g, d) merges dimension d of
// query head hk G + g over the splits that hold chunks of the sequence (only
// those wrote a record).  Launched as the decode launch's programmatic
// dependent: it waits for that grid before reading.
template <int G>
__global__ void __launch_bounds__(G * kD) attn_combine_kernel(const __grid_constant__ AttnArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int hk = blockIdx.x, b = blockIdx.y, h = hk * G + threadIdx.x / kD, d = threadIdx.x % kD;
  const float* rec = a.part + (static_cast<size_t>(b) * a.Hq + h) * a.nsplit * (2 + kD);
  const int len = a.seq_lens[b];
  const int n = (len >= 1 && len <= a.max_pages * a.P) ? len : 0;
  const int per = (a.max_pages * a.P + kC * a.nsplit - 1) / (kC * a.nsplit);
  const int ns = min(a.nsplit, ((n + kC - 1) / kC + per - 1) / per);
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, rec[s * (2 + kD)]);
  float num = 0.f, den = 0.f;
  if (M != -INFINITY) {
#pragma unroll 4
    for (int s = 0; s < ns; ++s) {
      const float m = rec[s * (2 + kD)];
      const float w = m == -INFINITY ? 0.f : exp2f(m - M);
      num = fmaf(w, rec[s * (2 + kD) + 2 + d], num);
      den = fmaf(w, rec[s * (2 + kD) + 1], den);
    }
  }
  // the decode launch has finished: its work counter starts the next call at zero
  if (hk == 0 && b == 0 && threadIdx.x == 0) *a.work = 0u;
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
  paged_decode_kernel<G><<<a.grid, kAThreads, kAttnSmem, stream>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.Hkv, a.B);
  cfg.blockDim = dim3(G * kD);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_combine_kernel<G>, a);
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

int attn_grid(int items, int sms) {
  const int resident = 2 * sms;  // the ring's shared memory lets two blocks share an SM
  return items < resident ? items : resident;
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
