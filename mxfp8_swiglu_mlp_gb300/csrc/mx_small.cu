// mx_small.cu -- the fused MXFP8 SwiGLU MLP for decode batches of up to 8
// tokens at small hidden sizes, in one launch with a single hand-off between
// blocks.
//
// The MLP (X copy of the Fish Audio post, "Custom kernels for the shapes TTS
// actually uses": gate/up projection, SiLU(gate) * up, down projection on
// MXFP8 operands, the intermediate requantised to MXFP8 along I; p2
// "Resultados de benchmark del kernel") is computed as:
//
//   unit u    (block u < I / 32) the gate and up rows of intermediate
//             features 32u .. 32u + 31 over all of K = H: 64 weight rows,
//             so h's 32-element quantisation block along I is the block's
//             own; SiLU(g) * u in fp32, requantised, written to the
//             workspace, and counted;
//   tile t    (block t < H / 16) rows 16t .. 16t + 15 of y over all of I,
//             once every unit is counted: no split-K, no reduction in L2.
//
// At M <= 8 these are matrix-vector products bound by HBM, not dense
// contractions: each block's weights (64 H + 16 I bytes) are put into shared
// memory by TMA before the grid dependency is waited for, and the products
// run as mma.sync m16n8k32 on E4M3 operands (one 32-element scale block per
// instruction, fp32 sums, block scales applied in fp32 afterwards), tokens as
// the N = 8 columns.
//
// Blocks wait on one another (the tiles on the units), so the grid (at most
// one block per SM) must be resident at once; the launch uses programmatic
// stream serialization and every wait is bounded.
#include <cuda_bf16.h>

#include <atomic>

#include "mx_device.cuh"
#include "mx_small.h"

namespace fsops {

namespace {

constexpr int kSmallWarps = 16;
constexpr int kSmallThreads = 32 * kSmallWarps;

// Timeline stamps for profiling builds (compiled with -DFSOPS_TRACE).
#ifdef FSOPS_TRACE
#define SMALL_STAMP(idx)                                                                   \
  do {                                                                                     \
    if (a.trace != nullptr) a.trace[blockIdx.x * 128 + (idx)] = globaltimer_ns();          \
  } while (0)
#else
#define SMALL_STAMP(idx) \
  do {                   \
  } while (0)
#endif

__device__ __forceinline__ void small_error(const SmallArgs& a, uint32_t code, uint32_t site) {
  atomicCAS(a.ctl + kCtlStatus, 0u, (code << 24) | ((site & 0xFFu) << 16) | (blockIdx.x & 0xFFFFu));
}
__device__ __forceinline__ bool small_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > timeout_ns) return false;
  return true;
}
// 2^(s - 127) for a UE8M0 byte s (s = 0 is the subnormal 2^-127).
__device__ __forceinline__ float ue8m0_f32(uint32_t s) {
  return s != 0 ? __uint_as_float(s << 23) : __uint_as_float(0x00400000u);
}
// d = A . B on the tensor core: A 16 x 32 E4M3 (row), B 32 x 8 E4M3 (col),
// fp32 d (the products are exact).
__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Four 8 x 16-byte matrices from shared memory, one row address per lane
// (lanes 8i .. 8i + 7 the rows of matrix i); lane l gets bytes 4 (l % 4) ..
// 4 (l % 4) + 3 of row l / 4 of each.
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& m0, uint32_t& m1, uint32_t& m2, uint32_t& m3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(m0), "=r"(m1), "=r"(m2), "=r"(m3)
               : "r"(addr));
}

// One warp's share of a 16-row weight tile times 8 token columns, over the
// 32-element K blocks j = j0, j0 + dj, ... < j1 (dj a multiple of 4).
//   w, box_bytes, row0  the tile's rows: TMA boxes of 128-byte rows (128-byte
//                       swizzle, box j / 4 at w + (j / 4) box_bytes), the
//                       tile's first row at row0 of its box;
//   ws, wjs, wof        the rows' scale bytes: rows g and g + 8 of block j at
//                       ws + j wjs + 2 g + wof and + 1 (a warp's 16 bytes
//                       contiguous);
//   xc, ld              the tokens' codes, rows of ld bytes, each 32-element
//                       block stored as [tq][half][4 codes]: codes 16 h + 4 tq
//                       .. + 3 at byte 8 tq + 4 h of the block;
//   xsc                 the tokens' scales as floats, [block][8 tokens].
// A block is one E4M3 MMA (m16n8k32, fp32 sums): k index 4 tq + e is code
// 4 tq + e of the block's first 16-code half and 16 + 4 tq + e code 4 tq + e
// of its second, for the weight rows (ldmatrix from the swizzled boxes) and
// the tokens alike.  acc[0..3]: rows g, g, g + 8, g + 8 of the tile x
// tokens 2 tq, 2 tq + 1.
__device__ __forceinline__ void tile_products(float (&acc)[4], const uint8_t* w, uint32_t box_bytes, int row0,
                                              const uint8_t* ws, int wjs, int wof, const uint8_t* xc, int ld,
                                              const float* xsc, int j0, int j1, int dj, int lane) {
  const int g = lane >> 2, tq = lane & 3;
  // dj is a multiple of 4, so every block this warp takes sits at the same
  // place in its 128-byte box: the addresses only step by a constant
  const int lrow = row0 + (lane & 7) + 8 * ((lane >> 3) & 1), lhalf = lane >> 4;
  uint32_t a_addr = smem_u32(w) + lrow * 128 + (((2 * (j0 & 3) + lhalf) ^ (lrow & 7)) << 4) + (j0 >> 2) * box_bytes;
  const uint32_t a_step = (dj >> 2) * box_bytes;
  const uint8_t* bp = xc + g * ld + 32 * j0 + 8 * tq;
  const uint8_t* wp = ws + j0 * wjs + 2 * g + wof;
  const float* xp = xsc + 8 * j0 + 2 * tq;
  // two blocks per step, every load of both issued first
  float acc2[4] = {0.f, 0.f, 0.f, 0.f};
  for (int j = j0; j < j1; j += 2 * dj) {
    const bool two = j + dj < j1;
    uint32_t m[2][4];
    uint2 Bv[2];
    uint32_t wsv[2];
    float2 xv[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int o = (u && two) ? 1 : 0;  // the second load repeats the first past the end
      ldmatrix_x4(a_addr + o * a_step, m[u][0], m[u][1], m[u][2], m[u][3]);
      Bv[u] = *reinterpret_cast<const uint2*>(bp + o * 32 * dj);
      wsv[u] = *reinterpret_cast<const uint16_t*>(wp + o * dj * wjs);
      xv[u] = *reinterpret_cast<const float2*>(xp + o * 8 * dj);
    }
    a_addr += 2 * a_step;
    bp += 64 * dj;
    wp += 2 * dj * wjs;
    xp += 16 * dj;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (u == 1 && !two) break;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      mma_e4m3_16832(d, m[u][0], m[u][1], m[u][2], m[u][3], Bv[u].x, Bv[u].y);
      // 2^(s - 127) of each row's scale byte (s = 0: 2^-127, the subnormal)
      const float w0 = __uint_as_float(max((wsv[u] << 23) & 0x7F800000u, 0x00400000u));
      const float w1 = __uint_as_float(max((wsv[u] << 15) & 0x7F800000u, 0x00400000u));
      float* ac = u ? acc2 : acc;
      ac[0] = fmaf(d[0], w0 * xv[u].x, ac[0]);
      ac[1] = fmaf(d[1], w0 * xv[u].y, ac[1]);
      ac[2] = fmaf(d[2], w1 * xv[u].x, ac[2]);
      ac[3] = fmaf(d[3], w1 * xv[u].y, ac[3]);
    }
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) acc[e] += acc2[e];
}
// Store a 32-code block (packed[i] = codes 4i .. 4i + 3) in the [tq][half]
// order tile_products reads.
__device__ __forceinline__ void store_block_codes(uint8_t* dst, const uint32_t (&packed)[8]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
  d[0] = make_uint4(packed[0], packed[4], packed[1], packed[5]);
  d[1] = make_uint4(packed[2], packed[6], packed[3], packed[7]);
}

template <bool NORM>
__global__ void __launch_bounds__(kSmallThreads, 2) mx_small_kernel(const __grid_constant__ SmallArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_align(smem_raw, 1024);
  __shared__ __align__(8) uint64_t bar_a, bar_b;
  __shared__ int failed;

  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int H = a.H, I = a.I, M = a.M;
  const int KA = H / 128, KB = I / 128;    // 128-byte K boxes
  const int nka = H / 32, nkb = I / 32;    // 32-element K blocks
  // block b: unit b (b < U) and tile b (b < T), or, with split roles, unit b
  // or tile b - U
  const int b = blockIdx.x, tb = a.split ? b - a.U : b;
  const bool do_a = b < a.U, do_b = tb >= 0 && tb < a.T;
  // shared memory (every region 16-byte aligned; the weight boxes 1024)
  uint8_t* wa = sm;                                        // [2][KA][32 rows][128]: gate rows, then up rows
  uint8_t* wb = a.split ? sm : wa + 64 * H;                // [KB][16 rows][128]
  // token codes in rows of H + 32 (I + 32) bytes: 8 tq + 2 tq' mod 32 banks
  // apart for the 16 lanes of a half warp
  uint8_t* xs = sm + small_weight_bytes(H, I, a.split);    // [8][H + 32] x codes ([tq][half] per block)
  uint8_t* hsm = xs + 8 * (H + 32);                        // [8][I + 32] h codes (likewise)
  float* xsc = reinterpret_cast<float*>(hsm + 8 * (I + 32));  // [nka][8 tokens]
  float* hsc = xsc + 8 * nka;                              // [nkb][8 tokens]
  uint8_t* wsa = reinterpret_cast<uint8_t*>(hsc + 8 * nkb);  // [nka][tile rt][g][row half]: 64 nka bytes
  uint8_t* wsb = wsa + 64 * nka;                           // [nkb][g][row half]: 16 nkb bytes
  float* red = reinterpret_cast<float*>(smem_align(wsb + 16 * nkb, 16));
  float* h32 = red + kSmallWarps * 16 * 8;                 // [8 tokens][32 features]

  // unit b's gate rows (32) and up rows (32) in W_gateup's paired order:
  // 128-row blocks of 64 gate rows then the same features' 64 up rows
  const int gate_row = 128 * (b >> 1) + 32 * (b & 1), up_row = gate_row + 64;
  if (t == 0) {
    mbar_init(&bar_a, 1);
    mbar_init(&bar_b, 1);
    mbar_fence_init();
    failed = 0;
    SMALL_STAMP(0);
  }
  __syncthreads();
  // ---- the weights do not depend on earlier work: fetched before the wait
  if (t == 0) {
    const uint64_t pol = l2_policy_evict_first();
    if (do_a) {
      tma_prefetch_desc(&a.tm_wgu);
      mbar_arrive_expect_tx(&bar_a, static_cast<uint32_t>(64 * H));
      for (int kt = 0; kt < KA; ++kt) {
        tma_load_2d(wa + kt * 4096, &a.tm_wgu, &bar_a, 128 * kt, gate_row, pol);
        tma_load_2d(wa + (KA + kt) * 4096, &a.tm_wgu, &bar_a, 128 * kt, up_row, pol);
      }
    }
    if (do_b) {
      tma_prefetch_desc(&a.tm_wd);
      mbar_arrive_expect_tx(&bar_b, static_cast<uint32_t>(16 * I));
      for (int kt = 0; kt < KB; ++kt) tma_load_2d(wb + kt * 2048, &a.tm_wd, &bar_b, 128 * kt, 16 * tb, pol);
    }
  }
  // weight scales, from the tcgen05 tiled layout into the order the
  // products read: block kb, tile rt, lane group g, rows 16 rt + g (+ 8)
  if (do_a)
    for (int i = t; i < 64 * nka; i += kSmallThreads) {
      const int kb = i >> 6, rt = (i >> 4) & 3, g = (i >> 1) & 7, hf = i & 1;
      const int r = 16 * rt + 8 * hf + g;  // unit row: gate 0-31, up 32-63
      wsa[i] = a.sf_gu[tiled_sf_offset(r < 32 ? gate_row + r : up_row + r - 32, kb, KA)];
    }
  if (do_b)
    for (int i = t; i < 16 * nkb; i += kSmallThreads) {
      const int kb = i >> 4, g = (i >> 1) & 7, hf = i & 1;
      wsb[i] = a.sf_d[tiled_sf_offset(16 * tb + 8 * hf + g, kb, KB)];
    }
  griddep_wait();
  griddep_launch_dependents();
  if (t == 0) SMALL_STAMP(1);

  // ---- x (the units only): token m by warp m, one 32-element block per lane
  // at a time.  The tiles never read x, and write y only once every unit has
  // read it, so y may be x's buffer.
  if (do_a && warp < kSmallMaxM) {
    const int m = warp;
    uint8_t* xr = xs + m * (H + 32);
    if (m < M) {
      const uint16_t* src = a.x + static_cast<size_t>(m) * H;
      const float rn = NORM ? row_rnorm(src, H, a.eps, lane) : 1.f;
      for (int kb = lane; kb < nka; kb += 32) {
        uint4 raw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) raw[i] = __ldg(reinterpret_cast<const uint4*>(src + 32 * kb) + i);
        uint32_t packed[8];
        const uint32_t s = NORM ? quantize_block_pack_norm(raw, a.gamma + 32 * kb, rn, packed)
                                : quantize_block_pack(raw, packed);
        store_block_codes(xr + 32 * kb, packed);
        xsc[kb * 8 + m] = ue8m0_f32(s);
      }
    } else {
      for (int i = lane; i < H / 16; i += 32) reinterpret_cast<uint4*>(xr)[i] = make_uint4(0u, 0u, 0u, 0u);
      for (int kb = lane; kb < nka; kb += 32) xsc[kb * 8 + m] = 0.f;
    }
  }
  __syncthreads();

  // ---- unit b: gate and up sums of 32 features, SwiGLU, h requantised
  if (do_a) {
    if (t == 0) SMALL_STAMP(2);
    if (!small_wait(&bar_a, 0, a.timeout_ns)) {
      if (lane == 0) small_error(a, 5u, 20u);  // FSOPS_ERR_TIMEOUT
      failed = 1;
    }
    __syncthreads();
    if (t == 0) SMALL_STAMP(3);
    if (!failed) {
      // warp w: 16-row tile w % 4 (gate rows 0-15, 16-31, up rows 0-15,
      // 16-31) over the K blocks w / 4, w / 4 + 4, ...
      const int rt = warp & 3, kh = warp >> 2;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      if (t == 0) SMALL_STAMP(10);
      tile_products(acc, wa + (rt >> 1) * KA * 4096, 4096, 16 * (rt & 1), wsa, 64, 16 * rt, xs, H + 32, xsc, kh, nka,
                    kSmallWarps / 4, lane);
      if (lane == 0 && warp == 0) SMALL_STAMP(11);
      if (lane == 0 && warp == kSmallWarps - 1) SMALL_STAMP(12);
      const int g = lane >> 2, tq = lane & 3;
      red[(warp * 16 + g) * 8 + 2 * tq] = acc[0];
      red[(warp * 16 + g) * 8 + 2 * tq + 1] = acc[1];
      red[(warp * 16 + g + 8) * 8 + 2 * tq] = acc[2];
      red[(warp * 16 + g + 8) * 8 + 2 * tq + 1] = acc[3];
    }
    __syncthreads();
    if (t == 0) SMALL_STAMP(4);
    if (!failed && t < 256) {
      // feature f = t / 8 of the unit for token m = t % 8: gate in tile
      // f / 16 (warps f / 16 + 4 q), up in tile 2 + f / 16
      const int f = t >> 3, m = t & 7, gt = f >> 4, fr = f & 15;
      float gs = 0.f, us = 0.f;
#pragma unroll
      for (int q = 0; q < kSmallWarps / 4; ++q) {
        gs += red[((4 * q + gt) * 16 + fr) * 8 + m];
        us += red[((4 * q + 2 + gt) * 16 + fr) * 8 + m];
      }
      h32[m * 32 + f] = silu_mul(gs, us);
    }
    __syncthreads();
    if (!failed && warp < M) {
      // token `warp`'s 32 features: one MXFP8 block along I
      const float v = h32[warp * 32 + lane];
      float amax = fabsf(v);
#pragma unroll
      for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
      const uint32_t s = ue8m0_from_amax(amax);
      a.hq[static_cast<size_t>(warp) * I + 32 * b + lane] = static_cast<uint8_t>(e4m3_code(v * inv_scale_from_ue8m0(s)));
      if (lane == 0) a.hs[static_cast<size_t>(warp) * nkb + b] = static_cast<uint8_t>(s);
    }
    __syncthreads();
    // the release (cumulative over the block's writes before the barrier)
    // publishes the unit
    if (t == 0 && !failed) red_add_release_gpu(a.ctl + kCtlSmallPublished, 1u);
    if (t == 0) SMALL_STAMP(5);
  }

  // ---- tile tb: rows 16 tb .. 16 tb + 15 of y over all of I
  if (do_b) {
    // the rows of h past the tokens hold zeros
    for (int i = t; i < (kSmallMaxM - M) * (I / 16); i += kSmallThreads) {
      const int m = M + i / (I / 16), c = i % (I / 16);
      reinterpret_cast<uint4*>(hsm + m * (I + 32))[c] = make_uint4(0u, 0u, 0u, 0u);
    }
    for (int i = t; i < (kSmallMaxM - M) * nkb; i += kSmallThreads) hsc[(i % nkb) * 8 + M + i / nkb] = 0.f;
    if (t == 0) {
      SMALL_STAMP(6);
      if (!small_wait(&bar_b, 0, a.timeout_ns)) {
        small_error(a, 5u, 21u);  // FSOPS_ERR_TIMEOUT
        failed = 1;
      } else {
        // every unit of h written (bounded wait on the counter)
        const uint32_t want = static_cast<uint32_t>(a.U) + a.extra_arrivals;
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire_gpu(a.ctl + kCtlSmallPublished) < want) {
          if (globaltimer_ns() - t0 > a.timeout_ns || *reinterpret_cast<volatile uint32_t*>(a.ctl + kCtlStatus) != 0) {
            small_error(a, 5u, 22u);  // FSOPS_ERR_TIMEOUT
            failed = 1;
            break;
          }
        }
      }
      SMALL_STAMP(7);
    }
    __syncthreads();
    if (!failed) {
      // h codes and scales of the tokens (written by other blocks in this
      // launch: read through L2)
      // (codes and scales in one pass: one round trip; a block's two 16-code
      // halves are read by one thread and stored in the [tq][half] order)
      const int n32 = I / 32, nblocks = M * n32;
      for (int i = t; i < nblocks + M * nkb; i += kSmallThreads) {
        if (i < nblocks) {
          const int m = i / n32, kb = i % n32;
          const uint4* src = reinterpret_cast<const uint4*>(a.hq + static_cast<size_t>(m) * I + 32 * kb);
          const uint4 lo = __ldcg(src), hi = __ldcg(src + 1);
          const uint32_t packed[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
          store_block_codes(hsm + m * (I + 32) + 32 * kb, packed);
        } else {
          const int k = i - nblocks, m = k / nkb, kb = k % nkb;
          hsc[kb * 8 + m] = ue8m0_f32(__ldcg(a.hs + k));
        }
      }
    }
    __syncthreads();
    if (t == 0) SMALL_STAMP(8);
    if (!failed) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      tile_products(acc, wb, 2048, 0, wsb, 16, 0, hsm, I + 32, hsc, warp, nkb, kSmallWarps, lane);
      const int g = lane >> 2, tq = lane & 3;
      red[(warp * 16 + g) * 8 + 2 * tq] = acc[0];
      red[(warp * 16 + g) * 8 + 2 * tq + 1] = acc[1];
      red[(warp * 16 + g + 8) * 8 + 2 * tq] = acc[2];
      red[(warp * 16 + g + 8) * 8 + 2 * tq + 1] = acc[3];
    }
    __syncthreads();
    if (!failed && t < 128) {
      const int r = t >> 3, m = t & 7;
      if (m < M) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kSmallWarps; ++w) v += red[(w * 16 + r) * 8 + m];
        const size_t o = static_cast<size_t>(m) * H + 16 * tb + r;
        if (a.residual != nullptr) v += __uint_as_float(static_cast<uint32_t>(a.residual[o]) << 16);
        const __nv_bfloat16 ob = __float2bfloat16_rn(v);
        a.y[o] = *reinterpret_cast<const uint16_t*>(&ob);
      }
    }
  }

  // ---- the last block to leave sets the launch's counters back to zero
  __syncthreads();
  if (t == 0) {
    SMALL_STAMP(9);
    const uint32_t left = atom_add_acq_rel_gpu(a.ctl + kCtlSmallExits, 1u);
    if (left == gridDim.x - 1) {
      a.ctl[kCtlSmallPublished] = 0u;
      a.ctl[kCtlSmallExits] = 0u;
    }
  }
}

constexpr int kMaxAttrDevices = 16;
std::atomic<size_t> g_small_attr[kMaxAttrDevices];  // largest shared-memory size set so far

}  // namespace

bool small_fits(int M, int H, int I, int sms) {
  if (M < 1 || M > kSmallMaxM || H % 128 != 0 || I % 128 != 0) return false;
  if (I / 32 > sms || H / 16 > sms) return false;
  return small_smem_bytes(H, I, small_split(H, I, sms)) <= 232448;
}

cudaError_t launch_small_kernel(const SmallArgs& a, int grid, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxAttrDevices) return cudaErrorInvalidDevice;
  const size_t smem = small_smem_bytes(a.H, a.I, a.split);
  if (g_small_attr[dev].load(std::memory_order_acquire) < smem) {
    e = cudaFuncSetAttribute(mx_small_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(mx_small_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    g_small_attr[dev].store(smem, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kSmallThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return a.gamma != nullptr ? cudaLaunchKernelEx(&cfg, mx_small_kernel<true>, a)
                            : cudaLaunchKernelEx(&cfg, mx_small_kernel<false>, a);
}

}  // namespace fsops
