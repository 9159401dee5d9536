// mx_blockscale.cu -- FP8 GEMM with 128 x 128 block scales on tcgen05.
//
// The second scale format the Fish Audio post names beside mxfp8 (X copy,
// "Custom kernels for the shapes TTS actually uses": "bsgemm" FP8 with
// 128 x 128 block scales, for Hopper; p2 "Estrategia de cuantizacion FP8"):
// W [N, K] holds E4M3 codes with one fp32 scale per 128 x 128 block, A [M, K]
// one fp32 scale per 1 x 128 group (a token's K-block), and
//   C[m, n] = sum_kb  sa[m, kb] * sw[n / 128, kb] * sum_{k in kb} a[m, k] w[n, k].
// Each scale is amax / 448 of its block in fp32 (1 for an all-zero block) and
// each code the E4M3 round-to-nearest-even, saturated, of v / scale in fp32.
//
//   bs_quantize_*          bf16 -> codes + fp32 scales (groups of 1 x 128 or
//                          blocks of 128 x 128).
//   bs_gemm_kernel<NPAD>   the GEMM for up to 128 tokens.  The tensor core has
//                          no fp32 block scales, so every 128-deep K-block is
//                          its own MMA: the block-scaled MMA (kind::mxf8f6f4)
//                          with every UE8M0 scale byte 127 (2^0) gives the
//                          plain E4M3 products summed in fp32, and the
//                          epilogue scales that K-block's sums by sa * sw and
//                          adds them up in fp32 registers.  The weight tile
//                          is the A operand (M = 128 rows of W), the tokens
//                          the B operand (N = NPAD), so each epilogue thread
//                          holds one row of W for every token.  The units
//                          (row tile, K-block) are split evenly over the
//                          blocks (stream-K); a row tile shared by two blocks
//                          is added up in an fp32 accumulator in L2 and
//                          written by the block that arrives last.
#include <cuda_bf16.h>

#include <atomic>

#include "mx_blockscale.h"
#include "mx_device.cuh"

namespace fsops {

namespace {

constexpr int kBsAccBufs = 2;
constexpr int kBsMaxStages = 8;
constexpr uint32_t kBsWBytes = 128u * 128u;

template <int NPAD>
struct BsCfg {
  // epilogue warps: two per TMEM lane quarter from 64 tokens on, each with
  // half of the token columns (128 running sums per thread would spill),
  // four at 128 tokens (each unit's TMEM loads then wait once per thread:
  // 63.6 against 66.4 us for the N = 34816, K = 5120 GEMM)
  static constexpr int EW = NPAD >= 128 ? 16 : NPAD >= 64 ? 8 : 4;
  static constexpr int THREADS = 128 + 32 * EW;
  static constexpr int COLS = NPAD / (EW / 4);  // token columns per epilogue thread
  static constexpr uint32_t SB = 128u * NPAD + kBsWBytes;  // stage: A tile (NPAD x 128) | W tile (128 x 128)
  // unit scale tile, control words (512 B) and the token scales of each accumulator, alignment
  static constexpr uint32_t FIXED = 512u + 512u + kBsAccBufs * 512u + 1024u;
  static constexpr int STAGES = (kMaxSmem - FIXED) / SB < kBsMaxStages ? (kMaxSmem - FIXED) / SB : kBsMaxStages;
  static constexpr size_t SMEM = STAGES * SB + FIXED;
  // TMEM: the accumulators, then 8 columns of unit scales
  static constexpr uint32_t COLS_USED = kBsAccBufs * NPAD + 8;
  static constexpr uint32_t TMEM_COLS = COLS_USED <= 64 ? 64 : COLS_USED <= 128 ? 128 : COLS_USED <= 256 ? 256 : 512;
  // the barriers and words below the token scales (which start 512 bytes in)
  static_assert((2 * kBsMaxStages + 3 * kBsAccBufs + 1) * 8 + 16 <= 512, "control words overlap the token scales");
  static_assert(COLS % 4 == 0, "token columns are read four at a time");
};

// fp32 block scale amax / 448 (1 for an all-zero block) and the four codes of
// v0..v3 divided by it, in fp32 with correctly rounded division.
__device__ __forceinline__ float bs_scale(float amax) { return amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f; }
__device__ __forceinline__ uint32_t bs_codes4(float v0, float v1, float v2, float v3, float s) {
  return e4m3x4_code(__fdiv_rn(v0, s), __fdiv_rn(v1, s), __fdiv_rn(v2, s), __fdiv_rn(v3, s));
}

// Groups of 1 x 128: one warp per (row, K-block), four elements per lane.
__global__ void bs_quantize_rows_kernel(const uint16_t* __restrict__ x, int rows, int K, int ld,
                                        uint8_t* __restrict__ codes, float* __restrict__ scales) {
  const int KB = K / 128;
  const long long g = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (g >= static_cast<long long>(rows) * KB) return;  // whole warps leave together
  const int r = static_cast<int>(g / KB), kb = static_cast<int>(g % KB);
  const uint2 raw = __ldg(reinterpret_cast<const uint2*>(x + static_cast<long long>(r) * ld + kb * 128) + lane);
  const float v0 = bf16_lo(raw.x), v1 = bf16_hi(raw.x), v2 = bf16_lo(raw.y), v3 = bf16_hi(raw.y);
  float amax = fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3)));
#pragma unroll
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  const float s = bs_scale(amax);
  reinterpret_cast<uint32_t*>(codes + static_cast<long long>(r) * K + kb * 128)[lane] = bs_codes4(v0, v1, v2, v3, s);
  if (lane == 0) scales[g] = s;
}

// Blocks of 128 x 128: one 256-thread block per (row block, K-block), two
// threads per row (64 elements each); rows past `rows` count as zero.
__global__ void __launch_bounds__(256) bs_quantize_blocks_kernel(const uint16_t* __restrict__ x, int rows, int K,
                                                                 int ld, uint8_t* __restrict__ codes,
                                                                 float* __restrict__ scales) {
  const int KB = K / 128;
  const int rb = blockIdx.x / KB, kb = blockIdx.x % KB;
  const int r = rb * 128 + (threadIdx.x >> 1), c0 = kb * 128 + (threadIdx.x & 1) * 64;
  uint4 raw[8];
  float amax = 0.f;
  if (r < rows) {
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<long long>(r) * ld + c0);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      raw[i] = __ldg(src + i);
      const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
  __shared__ float part[8];
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = amax;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, part[i]);
  const float s = bs_scale(amax);
  if (threadIdx.x == 0) scales[blockIdx.x] = s;
  if (r < rows) {
    uint4* dst = reinterpret_cast<uint4*>(codes + static_cast<long long>(r) * K + c0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t pk[4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint4 v = raw[2 * i + h];
        pk[2 * h] = bs_codes4(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y), s);
        pk[2 * h + 1] = bs_codes4(bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w), s);
      }
      dst[i] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
  }
  // the GEMM launched next may stream these weights before it waits for this
  // kernel (programmatic launch): the writes are visible before the block leaves
  __threadfence();
}

}  // namespace

// Barrier 1 among the EW epilogue warps, and the AND of a wait's outcome over them.
template <int EW>
__device__ __forceinline__ void bs_epi_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * EW) : "memory");
}
template <int EW>
__device__ __forceinline__ bool bs_epi_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"(v ? 1u : 0u), "n"(32 * EW)
      : "memory");
  return r != 0;
}

template <int NPAD>
__global__ void __launch_bounds__(BsCfg<NPAD>::THREADS, 1) bs_gemm_kernel(const __grid_constant__ BsArgs a) {
  using Cfg = BsCfg<NPAD>;
  constexpr int EW = Cfg::EW, COLS = Cfg::COLS;
  constexpr int S = Cfg::STAGES;
  constexpr uint32_t SB = Cfg::SB;
  constexpr int NB = kBsAccBufs;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align(smem_raw, 1024);
  uint8_t* ring = smem;
  uint8_t* unit_sf = smem + static_cast<size_t>(S) * SB;  // 512 bytes of UE8M0 2^0
  uint8_t* ctl = unit_sf + 512;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctl);  // [S] A and W tiles landed
  uint64_t* empty = full + S;                         // [S] the stage's MMAs completed
  uint64_t* acc_full = empty + S;                     // [NB]
  uint64_t* acc_empty = acc_full + NB;                // [NB]
  uint64_t* drain = acc_empty + NB;
  uint64_t* scl_full = drain + 1;                     // [NB] the unit's scales are in sa_s[b]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(scl_full + NB);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* bcast = reinterpret_cast<volatile int*>(tmem_slot + 2);  // [2] last arrivals
  float* sa_s = reinterpret_cast<float*>(ctl + 512);  // [NB][128] the units' token scales x weight scale (16-byte aligned)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t U = static_cast<uint32_t>(a.T) * a.KB, G = gridDim.x;
  const uint32_t u0 = blockIdx.x * U / G, u1 = (blockIdx.x + 1) * U / G;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < NB; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], EW);  // one arrival per epilogue warp
      mbar_init(&scl_full[b], 32);   // every lane of the scale warp
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (threadIdx.x < 128) reinterpret_cast<uint32_t*>(unit_sf)[threadIdx.x] = 0x7F7F7F7Fu;
  fence_proxy_async_shared();  // tcgen05.cp reads the unit scales
  if (warp == 2) {
    tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&a.tm_a);
    tma_prefetch_desc(&a.tm_w);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_launch_dependents();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sf_col = tmem + NB * NPAD;  // unit scales: A at +0, B at +4
  Ctx cx;
  cx.abort_flag = abort_flag;
  cx.status = a.status;
  cx.timeout_ns = a.timeout_ns;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ producer
    griddep_wait();  // A may be the output of the previous kernel (its quantiser)
    const uint64_t pol_w = l2_policy_evict_first(), pol_a = l2_policy_evict_last();
    int stage = 0;
    uint32_t round = 0, issued_mask = 0, issued_parity = 0;
    bool ok = true;
    for (uint32_t u = u0; u < u1; ++u) {
      const int t = static_cast<int>(u / a.KB), kb = static_cast<int>(u % a.KB);
      if (!wait_mbar(cx, &empty[stage], (round & 1u) ^ 1u, kSiteEmpty)) { ok = false; break; }
      uint8_t* st = ring + static_cast<size_t>(stage) * SB;
      mbar_arrive_expect_tx(&full[stage], SB);
      tma_load_2d(st, &a.tm_a, &full[stage], kb * kTileK, 0, pol_a);
      tma_load_2d(st + 128u * NPAD, &a.tm_w, &full[stage], kb * kTileK, t * 128, pol_w);
      issued_mask |= 1u << stage;
      issued_parity = (issued_parity & ~(1u << stage)) | ((round & 1u) << stage);
      if (++stage == S) { stage = 0; ++round; }
    }
    if (!ok) *abort_flag = 1;
    for (int s = 0; s < S; ++s)
      if (issued_mask & (1u << s)) drain_mbar(&full[s], (issued_parity >> s) & 1u, 200000000ull);
  } else if (warp == 2 && lane == 0) {
    // ------------------------------------------------ MMA issuer: one K-block per accumulator
    tc_cp_32x128b_warpx4(sf_col, smem_desc(smem_u32(unit_sf), 0, 128, kSwizzleNone));
    tc_cp_32x128b_warpx4(sf_col + 4, smem_desc(smem_u32(unit_sf), 0, 128, kSwizzleNone));
    const uint32_t idesc0 = idesc_mxf8_e4m3(static_cast<uint32_t>(NPAD), 0, 0);
    int stage = 0;
    uint32_t round = 0, seq = 0;
    bool ok = true;
    for (uint32_t u = u0; u < u1 && ok; ++u, ++seq) {
      const uint32_t b = seq % NB;
      if (!wait_mbar(cx, &acc_empty[b], ((seq / NB) & 1u) ^ 1u, kSiteAccEmpty) ||
          !wait_mbar(cx, &full[stage], round & 1u, kSiteFullW)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint8_t* st = ring + static_cast<size_t>(stage) * SB;
      const uint32_t sa = smem_u32(st), sw = smem_u32(st + 128u * NPAD);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t idesc = idesc0 | (static_cast<uint32_t>(k) << 4) | (static_cast<uint32_t>(k) << 29);
        tc_mma_mxf8(tmem + b * NPAD, smem_desc(sw + 32 * k, 16, 1024, kSwizzle128B),
                    smem_desc(sa + 32 * k, 16, 1024, kSwizzle128B), idesc, sf_col, sf_col + 4, k > 0 ? 1u : 0u);
      }
      tc_commit(&empty[stage]);
      tc_commit(&acc_full[b]);
      if (++stage == S) { stage = 0; ++round; }
    }
    if (!ok) *abort_flag = 1;
    tc_commit(drain);
    drain_mbar(drain, 0, 200000000ull);
  } else if (warp == 1) {
    // ------------------------------------------------ scale warp: each unit's token scales times the
    // weight block's scale into the shared slot of its accumulator (lane l: tokens l, l + 32, ...),
    // loaded one unit ahead, written once the epilogue has released the slot
    griddep_wait();  // the token scales may be the output of the previous kernel
    const int M = a.M, KB = a.KB;
    float sa_next[4] = {0.f, 0.f, 0.f, 0.f}, sw_next = 0.f;
    auto load_scales = [&](uint32_t u) {
      const int t = static_cast<int>(u / KB), kb = static_cast<int>(u % KB);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = lane + 32 * j;
        sa_next[j] = i < NPAD && i < M ? __ldg(a.a_scales + static_cast<size_t>(i) * KB + kb) : 0.f;
      }
      sw_next = __ldg(a.w_scales + static_cast<size_t>(t) * KB + kb);
    };
    bool ok = true;
    uint32_t seq = 0;
    if (u0 < u1) load_scales(u0);
    for (uint32_t u = u0; u < u1; ++u, ++seq) {
      const uint32_t b = seq % NB;
      float sa[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) sa[j] = sa_next[j];
      const float sw = sw_next;
      if (u + 1 < u1) load_scales(u + 1);
      if (!__all_sync(0xFFFFFFFFu, wait_mbar(cx, &acc_empty[b], ((seq / NB) & 1u) ^ 1u, kSiteAccEmpty))) {
        ok = false;
        break;
      }
      float* dst = sa_s + b * 128;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (lane + 32 * j < NPAD) dst[lane + 32 * j] = sw * sa[j];
      mbar_arrive(&scl_full[b]);
    }
    if (!ok) *abort_flag = 1;
  } else if (warp >= 4) {
    // ------------------------------------------------ epilogue: thread et holds row n = et % 128 of
    // the tile for token columns [r0, r0 + COLS)
    const int et = threadIdx.x - 128, q4 = warp & 3, row = et & 127, r0 = (et >> 7) * COLS;
    griddep_wait();  // C, the accumulator and the counters may be in use by the previous kernel
    const int M = a.M, KB = a.KB;
    float run[COLS];
#pragma unroll
    for (int r = 0; r < COLS; ++r) run[r] = 0.f;
    bool ok = true;
    int split_t[2], nsplit = 0;  // tiles this block shares with another (at most its first and last)
    // this block's sums of tile t (row n = 128 t + et), over all of K (whole) or a part of it
    auto flush = [&](int t, bool whole) {
      const size_t n = static_cast<size_t>(t) * 128 + row;
      if (whole) {
#pragma unroll
        for (int i = 0; i < COLS; ++i) {
          const int r = r0 + i;
          if (r < M) {
            if (a.c_f32) static_cast<float*>(a.c)[r * static_cast<size_t>(a.N) + n] = run[i];
            else static_cast<__nv_bfloat16*>(a.c)[r * static_cast<size_t>(a.N) + n] = __float2bfloat16_rn(run[i]);
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < COLS; ++i)
          if (r0 + i < M) red_add_f32(a.accum + (r0 + i) * static_cast<size_t>(a.N) + n, run[i]);
        if (nsplit < 2) split_t[nsplit++] = t;
      }
#pragma unroll
      for (int i = 0; i < COLS; ++i) run[i] = 0.f;
    };
    int cur_t = -1, first_kb = 0, last_kb = 0;
    uint32_t seq = 0;
    // each warp runs on its own: it waits for the unit's accumulator and its
    // scales (the scale warp's), no barrier with the other epilogue warps
    for (uint32_t u = u0; u < u1; ++u, ++seq) {
      const int t = static_cast<int>(u / KB), kb = static_cast<int>(u % KB);
      if (t != cur_t) {
        if (cur_t >= 0) flush(cur_t, first_kb == 0 && last_kb == KB - 1);
        cur_t = t;
        first_kb = kb;
      }
      last_kb = kb;
      const uint32_t b = seq % NB, par = (seq / NB) & 1u;
      if (!__all_sync(0xFFFFFFFFu, wait_mbar(cx, &acc_full[b], par, kSiteAccFull) &&
                                       wait_mbar(cx, &scl_full[b], par, kSiteAccFull))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float* sa_u = sa_s + b * 128;
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q4 * 32) << 16) + b * NPAD + r0;
      // up to 32 columns of loads in flight per wait
      constexpr int kBatch = COLS < 32 ? COLS : 32;
#pragma unroll
      for (int c = 0; c < COLS; c += kBatch) {
        uint32_t v[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch / 16; ++j)
          tmem_ld16(taddr + c + 16 * j, *reinterpret_cast<uint32_t(*)[16]>(&v[16 * j]));
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < kBatch; i += 4) {
          const float4 s4 = *reinterpret_cast<const float4*>(sa_u + r0 + c + i);
          run[c + i] = fmaf(__uint_as_float(v[i]), s4.x, run[c + i]);
          run[c + i + 1] = fmaf(__uint_as_float(v[i + 1]), s4.y, run[c + i + 1]);
          run[c + i + 2] = fmaf(__uint_as_float(v[i + 2]), s4.z, run[c + i + 2]);
          run[c + i + 3] = fmaf(__uint_as_float(v[i + 3]), s4.w, run[c + i + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
    }
    if (!ok) *abort_flag = 1;  // the other warps' waits end at once
    ok = bs_epi_and<EW>(ok);   // every epilogue warp agrees before the tiles' finish
    if (ok && cur_t >= 0) flush(cur_t, first_kb == 0 && last_kb == KB - 1);
    // shared tiles: the block that adds last writes C and leaves the
    // accumulator and the counter zero
    if (ok && nsplit > 0) {
      fence_acq_rel_gpu();  // this thread's adds are performed before any ticket
      bs_epi_bar<EW>();
      if (et < nsplit) {
        const int t = split_t[et];
        const uint32_t ub = static_cast<uint32_t>(t) * KB, ue = ub + KB - 1;
        const uint32_t owners = ((ue + 1) * G + U - 1) / U - ((ub + 1) * G + U - 1) / U + 1;
        bcast[et] = atom_add_acq_rel_gpu(a.tile_cnt + t, 1u) + 1 == owners ? 1 : 0;
      }
      bs_epi_bar<EW>();
      for (int i = 0; i < nsplit; ++i) {
        if (!bcast[i]) continue;
        const int t = split_t[i];
        const size_t n = static_cast<size_t>(t) * 128 + row;
        // every load is issued before the first store: one L2 round trip
#pragma unroll
        for (int j = 0; j < COLS; ++j)
          if (r0 + j < M) run[j] = __ldcg(a.accum + (r0 + j) * static_cast<size_t>(a.N) + n);
#pragma unroll
        for (int j = 0; j < COLS; ++j) {
          if (r0 + j < M) {
            const size_t o = (r0 + j) * static_cast<size_t>(a.N) + n;
            if (a.c_f32) static_cast<float*>(a.c)[o] = run[j];
            else static_cast<__nv_bfloat16*>(a.c)[o] = __float2bfloat16_rn(run[j]);
            __stcg(a.accum + o, 0.f);
          }
        }
        if (et == 0) a.tile_cnt[t] = 0u;
      }
    }
    if (!ok) *abort_flag = 1;
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, Cfg::TMEM_COLS);
}

namespace {
constexpr int kMaxAttrDevices = 64;
std::atomic<bool> g_bs_attr_set[kMaxAttrDevices];

template <int NPAD>
cudaError_t launch_npad(const BsArgs& a, int grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(BsCfg<NPAD>::THREADS);
  cfg.dynamicSmemBytes = BsCfg<NPAD>::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, bs_gemm_kernel<NPAD>, a);
}
template <int NPAD>
cudaError_t set_limit() {
  return cudaFuncSetAttribute(bs_gemm_kernel<NPAD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(BsCfg<NPAD>::SMEM));
}
}  // namespace

cudaError_t launch_bs_gemm(const BsArgs& a, int npad, int sms, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxAttrDevices) return cudaErrorInvalidDevice;
  if (!g_bs_attr_set[dev].load(std::memory_order_acquire)) {
    const cudaError_t es[4] = {set_limit<16>(), set_limit<32>(), set_limit<64>(), set_limit<128>()};
    for (cudaError_t x : es)
      if (x != cudaSuccess) return x;
    g_bs_attr_set[dev].store(true, std::memory_order_release);
  }
  const long long units = static_cast<long long>(a.T) * a.KB;
  const int grid = units < sms ? static_cast<int>(units) : sms;
  switch (npad) {
    case 16: return launch_npad<16>(a, grid, stream);
    case 32: return launch_npad<32>(a, grid, stream);
    case 64: return launch_npad<64>(a, grid, stream);
    case 128: return launch_npad<128>(a, grid, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_bs_quantize(const uint16_t* x, int rows, int K, int ld, int block_rows, uint8_t* codes,
                               float* scales, cudaStream_t stream) {
  const int KB = K / 128;
  if (rows == 0) return cudaSuccess;
  if (block_rows == 1) {
    const long long warps = static_cast<long long>(rows) * KB;
    const long long blocks = (warps * 32 + 255) / 256;
    bs_quantize_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(x, rows, K, ld, codes, scales);
  } else {
    const long long blocks = static_cast<long long>((rows + 127) / 128) * KB;
    bs_quantize_blocks_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(x, rows, K, ld, codes, scales);
  }
  return cudaGetLastError();
}

}  // namespace fsops
