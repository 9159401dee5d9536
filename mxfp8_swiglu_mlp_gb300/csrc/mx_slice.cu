// mx_slice.cu -- the single-launch MXFP8 SwiGLU MLP for decode batches of up
// to 32 tokens, sliced over the intermediate features by 2-block clusters.
//
// The MLP (X copy of the Fish Audio post, "Custom kernels for the shapes TTS
// actually uses": gate/up projection, SiLU(gate) * up, down projection, on
// MXFP8 operands; p2 "Resultados de benchmark del kernel": the intermediate
// never makes a bf16 round trip through HBM) is split by intermediate
// feature.  Cluster q owns whole 128-feature chunks of I; in each chunk block
// `rank` owns 64 features:
//
//   gate/up   the block streams the 128 W_gateup rows of its 64 features (64
//             gate rows, then the 64 up rows: W_gateup's paired order) over all
//             of K and accumulates D = W^ . x^T in TMEM with tcgen05
//             kind::mxf8f6f4 block-scaled MMAs: the weight tile is the A
//             operand (M = 128 rows), the tokens the B operand (N = npad);
//   SwiGLU    TMEM lane quarters 0-1 hold the gate sums, 2-3 the up sums of the
//             same features: the up warps hand theirs over through shared
//             memory, the gate warps form h = SiLU(g) * u, requantise it to
//             MXFP8 along I (a 32-block is one warp's 32 lanes) and write the
//             codes and scales into the block's h tile, which is then pushed
//             into the partner's through distributed shared memory;
//   down      with the cluster's h complete (its features only), each block
//             multiplies it by its half of the 128-row tiles of W_down:
//             D = W_down^ . h^T, partial sums of y over the cluster's features;
//   reduce    each lane of the four epilogue warps holds one y feature for
//             every token and adds it into an fp32 [M, H] accumulator in L2
//             (coalesced 32-float rows); the cluster that arrives last at a
//             128-feature tile rounds it to bf16 into y and leaves it zero.
//             The clusters walk their tiles from different starting points,
//             so the finishing spreads over many blocks.
//
// No block waits on a block outside its own cluster, so the grid needs no
// co-residency guarantee (a plain cluster launch, not a cooperative one), and
// the launch uses programmatic stream serialization: the weight stream starts
// while the previous kernel on the stream finishes, and every access to
// memory that earlier work may write (x, the workspace, y) waits for it
// (griddepcontrol.wait).  x is quantised inside each block by the activation
// warp (optionally after RMSNorm, the decoder block's norm: the mean square of
// each row is reduced first).
//
// Roles (one block per SM, 8 warps):
//   warp 0 lane 0  weight producer: TMA of 128 x 128 B weight tiles and their
//                  512-byte scale tiles into a ring of stages (gate/up, then
//                  down; the down tiles do not depend on h, so they stream
//                  while the SwiGLU runs)
//   warp 1 lane 0  x producer: the bf16 x tile of each gate/up stage by TMA,
//                  into the stage (after the previous kernel completed)
//   warp 2 lane 0  MMA issuer
//   warps 4-7      the activation quantisation of the gate/up stages, then
//                  the epilogues: SwiGLU and the push of h, the split-K adds,
//                  the finish
#include <cuda_bf16.h>

#include <atomic>

#include "mx_device.cuh"
#include "mx_slice.h"

namespace fsops {

namespace {

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void st_shared_cluster_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared::cluster.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_shared_cluster() {
  asm volatile("fence.proxy.async.shared::cluster;" ::: "memory");
}

// One 32-element block of bf16 x (row r, k-group j of a 128-wide k-chunk),
// already in registers, quantised into the stage's activation tile (128-byte
// swizzled rows, as TMA would have written them) and its scale tile; rows
// >= M get zeros.
template <int NPAD>
__device__ __forceinline__ void store_x_block(int M, uint8_t* st, int b, const uint4 (&raw)[4], float scale_row,
                                              const uint16_t* gam, bool norm) {
  const int r = b >> 2, j = b & 3;
  uint32_t s = 0;
  uint4 c0 = make_uint4(0, 0, 0, 0), c1 = c0;
  if (r < M) {
    uint32_t pk[8];
    s = norm ? quantize_block_pack_norm(raw, gam, scale_row, pk) : quantize_block_pack(raw, pk);
    c0 = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    c1 = make_uint4(pk[4], pk[5], pk[6], pk[7]);
  }
  uint8_t* row = st + r * 128;
  *reinterpret_cast<uint4*>(row + (((2 * j) ^ (r & 7)) << 4)) = c0;
  *reinterpret_cast<uint4*>(row + (((2 * j + 1) ^ (r & 7)) << 4)) = c1;
  st[slice_off_sfx(NPAD) + (r & 31) * 16 + (r >> 5) * 4 + j] = static_cast<uint8_t>(s);
}

// bf16 pack of 8 fp32 values (plus, if res != null, the bf16 residual first).
__device__ __forceinline__ uint4 pack_bf16x8(const float* v, const uint16_t* res) {
  float s[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) s[i] = v[i];
  if (res != nullptr) {
    const uint4 rv = *reinterpret_cast<const uint4*>(res);
    const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      s[2 * i] += bf16_lo(rw[i]);
      s[2 * i + 1] += bf16_hi(rw[i]);
    }
  }
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 b2 = __floats2bfloat162_rn(s[2 * i], s[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&b2);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace

// Timeline stamps for profiling builds (compiled with -DFSOPS_TRACE).
#ifdef FSOPS_TRACE
#define SLICE_STAMP(idx)                                                         \
  do {                                                                           \
    if (a.trace != nullptr) a.trace[blockIdx.x * 64 + (idx)] = globaltimer_ns(); \
  } while (0)
#else
#define SLICE_STAMP(idx) \
  do {                   \
  } while (0)
#endif

template <int NPAD>
__global__ void __launch_bounds__(kThreads, 1) mx_slice_kernel(const __grid_constant__ SliceArgs a) {
  constexpr int CL = kSliceCluster;
  constexpr int NB = kSliceAccBufs;
  constexpr uint32_t UL = NPAD + 4;       // ubuf row stride (floats)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align(smem_raw, 1024);
  const int S = a.nstages;
  constexpr uint32_t SB = 384u * NPAD + kSliceWBytes + 1024u;  // slice_stage_bytes
  uint8_t* htile = smem;
  uint8_t* hsf = smem + slice_off_hsf(NPAD);
  uint8_t* ring = smem + slice_off_ring(NPAD);
  float* ubuf = reinterpret_cast<float*>(ring + static_cast<size_t>(S) * SB);
  uint8_t* ctl = reinterpret_cast<uint8_t*>(ubuf + 64 * UL);
  uint64_t* full_w = reinterpret_cast<uint64_t*>(ctl);  // [kSliceMaxStages] weight tile landed
  uint64_t* full_a = full_w + kSliceMaxStages;          // [kSliceMaxStages] activation tile quantised
  uint64_t* empty = full_a + kSliceMaxStages;           // [kSliceMaxStages] the stage's MMAs completed
  uint64_t* acc_full = empty + kSliceMaxStages;         // [NB]
  uint64_t* acc_empty = acc_full + NB;                  // [NB]
  uint64_t* drain = acc_empty + NB;
  uint64_t* x_full = drain + 1;                         // [kSliceMaxStages] the stage's bf16 x tile landed
  uint64_t* h_full = x_full + kSliceMaxStages;          // every h chunk of the cluster is here
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(h_full + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* rnorm = reinterpret_cast<float*>(tmem_slot + 2);  // [kSliceMaxM] 1 / rms of each row
  uint8_t* lastflag = reinterpret_cast<uint8_t*>(rnorm + kSliceMaxM);  // [<= 256] this block finishes row tile i

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int q = static_cast<int>(blockIdx.x) / CL;
  const int c0 = q * a.NC / a.NP, c1 = (q + 1) * a.NC / a.NP, nq = c1 - c0;
  // down-projection row tiles of this block: [rt0, rt0 + nrt), walked from a
  // per-cluster offset, so that the clusters reach each tile in different
  // orders and its finish falls to different blocks
  const int rt0 = static_cast<int>(rank) * a.RT / CL, nrt = (static_cast<int>(rank) + 1) * a.RT / CL - rt0;
  const int rot = nrt > 0 ? q % nrt : 0;
  auto rt_of = [&](int i) { return rt0 + (i + rot) % nrt; };
  const int M = a.M;
  const bool norm = a.gamma != nullptr;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_w[s], 1);
      mbar_init(&full_a[s], 4);  // one arrival per epilogue warp (they quantise the tile)
      mbar_init(&empty[s], 1);
      mbar_init(&x_full[s], 1);
    }
    for (int b = 0; b < NB; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);  // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    // one arrival per chunk from each block of the cluster (+ the test hook's)
    mbar_init(h_full, static_cast<uint32_t>(nq * CL) + a.extra_arrivals);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&a.tm_wgu);
    tma_prefetch_desc(&a.tm_wd);
    tma_prefetch_desc(&a.tm_x);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the partner's barriers are initialised before either block arrives remotely
  cluster_sync_all();
  // the next kernel on the stream may be scheduled as this grid's blocks leave
  griddep_launch_dependents();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) SLICE_STAMP(0);
  Ctx cx;
  cx.abort_flag = abort_flag;
  cx.status = a.status;
  cx.timeout_ns = a.timeout_ns;
  // TMEM columns: accumulators [0, NB * NPAD), stage scales from 128 (8 per
  // stage: weight tile, then activation tile), h scales from 224 (4 per chunk)
  const uint32_t sf_base = tmem + 128u, hsf_col = tmem + 224u;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ weight producer
    // Weights are never written by a kernel, so their loads go out before the
    // previous kernel on the stream has finished.
    const uint64_t pol = l2_policy_evict_first();
    uint32_t issued_mask = 0, issued_parity = 0;
    int stage = 0;
    uint32_t round = 0;
    bool ok = true;
    auto load = [&](const CUtensorMap* map, int x, int y, const uint8_t* sf) -> bool {
      if (!wait_mbar(cx, &empty[stage], (round & 1u) ^ 1u, kSiteEmpty)) return false;
      if (round * S + stage < 16) SLICE_STAMP(16 + round * S + stage);
      uint8_t* st = ring + static_cast<size_t>(stage) * SB;
      mbar_arrive_expect_tx(&full_w[stage], kSliceWBytes + 512u);
      tma_load_2d(st + slice_off_w(NPAD), map, &full_w[stage], x, y, pol);
      bulk_load(st + slice_off_sfw(NPAD), sf, 512, &full_w[stage], pol);
      issued_mask |= 1u << stage;
      issued_parity = (issued_parity & ~(1u << stage)) | ((round & 1u) << stage);
      if (++stage == S) { stage = 0; ++round; }
      return true;
    };
    // gate/up: the 128 W_gateup rows of this block's 64 features of every
    // chunk (64 gate rows, then the 64 up rows of the same features), all of K
    for (int j = 0; j < nq && ok; ++j) {
      const int pb = 2 * (c0 + j) + static_cast<int>(rank);  // 128-row block of W_gateup
      for (int ks = 0; ks < a.KS0 && ok; ++ks)
        ok = load(&a.tm_wgu, ks * kTileK, pb * 128, a.sf_gu + (static_cast<size_t>(pb) * a.KS0 + ks) * 512);
    }
    // down: this block's row tiles of W_down, K = the cluster's chunks
    for (int i = 0; i < nrt && ok; ++i) {
      const int rt = rt_of(i);
      for (int j = 0; j < nq && ok; ++j) {
        const int t = c0 + j;
        ok = load(&a.tm_wd, t * kTileK, rt * 128, a.sf_d + (static_cast<size_t>(rt) * a.NC + t) * 512);
      }
    }
    if (!ok) *abort_flag = 1;
    for (int s = 0; s < S; ++s)
      if (issued_mask & (1u << s)) drain_mbar(&full_w[s], (issued_parity >> s) & 1u, 200000000ull);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------ x producer
    // The bf16 x tile of every gate/up stage, into the same stage as its
    // weights (so that it is in flight as far ahead), once the previous
    // kernel on the stream has completed (x may be its output).  The wait
    // holds the whole warp, so this role has a warp of its own.
    griddep_wait();
    const uint64_t pol = l2_policy_evict_last();
    uint32_t issued_mask = 0, issued_parity = 0;
    int stage = 0;
    uint32_t round = 0;
    bool ok = true;
    for (int j = 0; j < nq && ok; ++j) {
      for (int ks = 0; ks < a.KS0; ++ks) {
        if (!wait_mbar(cx, &empty[stage], (round & 1u) ^ 1u, kSiteEmpty)) { ok = false; break; }
        mbar_arrive_expect_tx(&x_full[stage], 256u * NPAD);
        tma_load_2d(ring + static_cast<size_t>(stage) * SB + slice_off_xb(NPAD), &a.tm_x, &x_full[stage], ks * kTileK,
                    0, pol);
        issued_mask |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | ((round & 1u) << stage);
        if (++stage == S) { stage = 0; ++round; }
      }
    }
    if (!ok) *abort_flag = 1;
    for (int s = 0; s < S; ++s)
      if (issued_mask & (1u << s)) drain_mbar(&x_full[s], (issued_parity >> s) & 1u, 200000000ull);
  } else if (warp == 2 && lane == 0) {
    // ------------------------------------------------ MMA issuer
    // D[128 weight rows, NPAD tokens] = W^ . act^T: the weight tile is the A
    // operand (M = 128), the tokens the B operand (N = NPAD).
    int stage = 0;
    uint32_t round = 0, seq = 0;  // seq: accumulators issued so far
    bool ok = true;
    const uint32_t idesc0 = idesc_mxf8_e4m3(static_cast<uint32_t>(NPAD), 0, 0);
    auto acquire_acc = [&]() -> bool {
      const uint32_t b = seq % NB;
      if (!wait_mbar(cx, &acc_empty[b], ((seq / NB) & 1u) ^ 1u, kSiteAccEmpty)) return false;
      tc_fence_after();
      return true;
    };
    auto mma_stage = [&](uint32_t b_act, uint32_t sfb, bool acc_first) {
      uint8_t* st = ring + static_cast<size_t>(stage) * SB;
      const uint32_t sfc = sf_base + 8u * stage;
      tc_cp_32x128b_warpx4(sfc, smem_desc(smem_u32(st + slice_off_sfw(NPAD)), 0, 128, kSwizzleNone));
      const uint32_t sw = smem_u32(st + slice_off_w(NPAD));
      const uint32_t d = tmem + (seq % NB) * NPAD;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t idesc = idesc0 | (static_cast<uint32_t>(k) << 4) | (static_cast<uint32_t>(k) << 29);
        tc_mma_mxf8(d, smem_desc(sw + 32 * k, 16, 1024, kSwizzle128B), smem_desc(b_act + 32 * k, 16, 1024, kSwizzle128B),
                    idesc, sfc, sfb, (!acc_first || k > 0) ? 1u : 0u);
      }
      tc_commit(&empty[stage]);
      if (++stage == S) { stage = 0; ++round; }
    };
    // gate/up chunks
    for (int j = 0; j < nq && ok; ++j) {
      if (!acquire_acc()) { ok = false; break; }
      for (int ks = 0; ks < a.KS0; ++ks) {
        if (!wait_mbar(cx, &full_w[stage], round & 1u, kSiteFullW) ||
            !wait_mbar(cx, &full_a[stage], round & 1u, kSiteFullA)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (j == 0 && ks >= 8 && ks < 16) SLICE_STAMP(40 + ks - 8);
        uint8_t* st = ring + static_cast<size_t>(stage) * SB;
        const uint32_t sfx = sf_base + 8u * stage + 4u;
        tc_cp_32x128b_warpx4(sfx, smem_desc(smem_u32(st + slice_off_sfx(NPAD)), 0, 128, kSwizzleNone));
        mma_stage(smem_u32(st), sfx, ks == 0);
      }
      if (!ok) break;
      tc_commit(&acc_full[seq % NB]);
      ++seq;
      SLICE_STAMP(2);
    }
    // down: the B operand is the cluster's h, complete once both blocks
    // pushed every chunk
    if (ok && nrt > 0) {
      ok = wait_mbar_cluster(cx, h_full, 0, kSiteHFlag);
      SLICE_STAMP(3);
      if (ok) {
        tc_fence_after();
        for (int j = 0; j < nq; ++j)
          tc_cp_32x128b_warpx4(hsf_col + 4 * j, smem_desc(smem_u32(hsf + 512 * j), 0, 128, kSwizzleNone));
      }
    }
    for (int i = 0; i < nrt && ok; ++i) {
      if (!acquire_acc()) { ok = false; break; }
      for (int j = 0; j < nq; ++j) {
        if (!wait_mbar(cx, &full_w[stage], round & 1u, kSiteFullW)) { ok = false; break; }
        tc_fence_after();
        mma_stage(smem_u32(htile + j * NPAD * 128), hsf_col + 4 * j, j == 0);
      }
      if (!ok) break;
      tc_commit(&acc_full[seq % NB]);
      ++seq;
      if (i == 0) SLICE_STAMP(4);
    }
    SLICE_STAMP(5);
    if (!ok) *abort_flag = 1;
    tc_commit(drain);
    drain_mbar(drain, 0, 200000000ull);
  } else if (warp >= 4) {
    // ------------------------------------------------ epilogue warps
    // Warp 4 + q4 reads TMEM lane quarter q4: weight rows 32 q4 .. 32 q4 + 31
    // of the accumulator, every token column.
    const int et = threadIdx.x - 128;
    const int q4 = warp & 3;
    griddep_wait();  // the workspace, y and x may be in use by the previous kernel until here
    bool ok = true;
    if (norm) {
      // RMSNorm: the mean square of each token row over all of H (fp32), one
      // warp per row in turn; the activation warp waits for it
      for (int r = q4; r < M; r += 4) {
        const float rn = row_rnorm(a.x + static_cast<size_t>(r) * a.H, a.H, a.eps, lane);
        if (lane == 0) rnorm[r] = rn;
      }
      epi_bar();  // every row's norm is in rnorm before any quantisation
    }
    uint32_t seq = 0;
    int qstage = 0;
    uint32_t qround = 0;
    // The activation tiles of one chunk's gate/up stages: thread et quantises
    // 32-block et (row et / 4, k-group et % 4) of each stage's bf16 x tile
    // into its 128B-swizzled E4M3 tile and scale tile.
    auto quantize_chunk = [&]() -> bool {
      for (int i = 0; i < a.KS0; ++i) {
        if (!epi_and(wait_mbar(cx, &x_full[qstage], qround & 1u, kSiteFullA))) return false;
        if (et == 0 && i >= 8 && i < 16 && seq == 0) SLICE_STAMP(48 + i - 8);
        uint8_t* st = ring + static_cast<size_t>(qstage) * SB;
        if (et < 4 * NPAD) {
          const int r = et >> 2;
          uint4 raw[4];
          const uint4* src = reinterpret_cast<const uint4*>(st + slice_off_xb(NPAD) + r * 256 + (et & 3) * 64);
#pragma unroll
          for (int k = 0; k < 4; ++k) raw[k] = src[k];
          store_x_block<NPAD>(M, st, et, raw, norm && r < M ? rnorm[r] : 1.0f,
                              norm ? a.gamma + i * kTileK + (et & 3) * 32 : nullptr, norm);
        }
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full_a[qstage]);
        if (et == 0 && i >= 8 && i < 16 && seq == 0) SLICE_STAMP(32 + i - 8);
        if (++qstage == S) { qstage = 0; ++qround; }
      }
      return true;
    };
    // the accumulator of sequence number seq: this warp's 32 rows, NPAD tokens
    auto read_acc = [&](float (&v)[NPAD]) -> bool {
      const uint32_t b = seq % NB;
      if (!epi_and(wait_mbar(cx, &acc_full[b], (seq / NB) & 1u, kSiteAccFull))) return false;
      tc_fence_after();
      uint32_t r[NPAD];
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q4 * 32) << 16) + b * NPAD;
      tmem_ld16(taddr, *reinterpret_cast<uint32_t(*)[16]>(&r[0]));
      if (NPAD == 32) tmem_ld16(taddr + 16, *reinterpret_cast<uint32_t(*)[16]>(&r[16 % NPAD]));
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < NPAD; ++i) v[i] = __uint_as_float(r[i]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
      ++seq;
      return true;
    };
    // -------- gate/up chunks: quantise x, then SwiGLU, requantise, push h to the partner
    for (int j = 0; j < nq && ok; ++j) {
      if (!quantize_chunk()) { ok = false; break; }
      float v[NPAD];
      if (!read_acc(v)) { ok = false; break; }
      if (et == 0 && j == 0) SLICE_STAMP(6);
      uint8_t* hj = htile + j * NPAD * 128;
      uint8_t* sj = hsf + j * 512;
      // rows 64..127 are the up sums: to shared memory, by feature
      if (q4 >= 2) {
        float4* d = reinterpret_cast<float4*>(ubuf + ((q4 - 2) * 32 + lane) * UL);
#pragma unroll
        for (int i = 0; i < NPAD / 4; ++i) d[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      }
      epi_bar();
      if (q4 < 2) {
        // feature f = 32 q4 + lane of the block's 64: gate sums in v, up sums in ubuf
        const int f = 32 * q4 + lane;
        const float4* up = reinterpret_cast<const float4*>(ubuf + f * UL);
        float h[NPAD];
#pragma unroll
        for (int i = 0; i < NPAD / 4; ++i) {
          const float4 u = up[i];
          h[4 * i] = silu_mul(v[4 * i], u.x);
          h[4 * i + 1] = silu_mul(v[4 * i + 1], u.y);
          h[4 * i + 2] = silu_mul(v[4 * i + 2], u.z);
          h[4 * i + 3] = silu_mul(v[4 * i + 3], u.w);
        }
        // per token: the 32-block's amax over the warp's 32 features
        float m[NPAD];
#pragma unroll
        for (int i = 0; i < NPAD; ++i) m[i] = fabsf(h[i]);
#pragma unroll
        for (int o = 16; o; o >>= 1) {
#pragma unroll
          for (int i = 0; i < NPAD; ++i) m[i] = fmaxf(m[i], __shfl_xor_sync(0xFFFFFFFFu, m[i], o));
        }
        // feature fc of the chunk's 128 (16-byte unit fc / 16 of a token row)
        const int fc = 64 * static_cast<int>(rank) + f;
        const int blk = fc >> 5;  // the chunk's 32-block
#pragma unroll
        for (int r = 0; r < NPAD; ++r) {
          const uint32_t sc = ue8m0_from_amax(m[r]);
          if (r < M) {
            hj[r * 128 + ((((fc >> 4) ^ (r & 7))) << 4) + (fc & 15)] =
                static_cast<uint8_t>(e4m3_code(h[r] * inv_scale_from_ue8m0(sc)));
            if (lane == (r & 31)) sj[(r & 31) * 16 + (r >> 5) * 4 + blk] = static_cast<uint8_t>(sc);
          }
        }
      }
      epi_bar();
      // push this block's 64 features of every token row (four 16-byte units
      // per row) and their two scale bytes into the partner's h
      {
        const uint32_t hj_peer = mapa_shared(hj, peer), sj_peer = mapa_shared(sj, peer);
        for (int it = et; it < M * 4; it += 128) {
          const int r = it >> 2, u = 4 * static_cast<int>(rank) + (it & 3);
          const uint32_t off = static_cast<uint32_t>(r * 128 + ((u ^ (r & 7)) << 4));
          const uint4 w = *reinterpret_cast<const uint4*>(hj + off);
          st_shared_cluster_v4(hj_peer + off, w);
        }
        for (int r = et; r < M; r += 128) {
          const uint32_t off = static_cast<uint32_t>((r & 31) * 16 + (r >> 5) * 4 + 2 * static_cast<int>(rank));
          st_shared_cluster_u16(sj_peer + off, *reinterpret_cast<const uint16_t*>(sj + off));
        }
      }
      // the tensor cores of both blocks read what was written here
      fence_proxy_async_shared();
      fence_proxy_async_shared_cluster();
      fence_acq_rel_cluster();
      epi_bar();
      if (et == 0) {
        SLICE_STAMP(9);
        mbar_arrive_remote(mapa_shared(h_full, rank));
        mbar_arrive_remote(mapa_shared(h_full, peer));
      }
    }
    // -------- down row tiles: add this cluster's partial sums of y into L2
    int done_tiles = 0;
    for (int i = 0; i < nrt && ok; ++i) {
      float v[NPAD];
      if (!read_acc(v)) { ok = false; break; }
      if (et == 0 && i == 0) SLICE_STAMP(10);
      const int n = rt_of(i) * 128 + et;  // y feature of this thread's accumulator row
      float* dst = a.accum + n;
#pragma unroll
      for (int r = 0; r < NPAD; ++r)
        if (r < M) red_add_f32(dst + static_cast<size_t>(r) * a.H, v[r]);
      ++done_tiles;
    }
    // -------- tickets: the cluster that adds last to a row tile finishes it
    if (ok && done_tiles > 0) {
      if (et == 0) SLICE_STAMP(11);
      fence_acq_rel_gpu();  // this thread's adds are performed before any ticket
      epi_bar();
      if (et == 0) SLICE_STAMP(12);
      for (int i = et; i < done_tiles; i += 128) {
        const uint32_t old = atom_add_acq_rel_gpu(a.tile_cnt + rt_of(i), 1u);
        lastflag[i] = (old + 1 == static_cast<uint32_t>(a.NP)) ? 1 : 0;
      }
      epi_bar();
      if (et == 0) SLICE_STAMP(13);
      for (int i = 0; i < done_tiles; ++i) {
        if (!lastflag[i]) continue;
        const int rt = rt_of(i);
        // tokens r < M x the tile's 128 features, 8 per item, all loads in flight
        const int items = M * 16;
        float4 v[4][2];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int it = et + 128 * k;
          if (it < items) {
            const float4* src = reinterpret_cast<const float4*>(a.accum + static_cast<size_t>(it >> 4) * a.H + rt * 128 +
                                                                (it & 15) * 8);
            v[k][0] = __ldcg(src);
            v[k][1] = __ldcg(src + 1);
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int it = et + 128 * k;
          if (it < items) {
            const size_t o = static_cast<size_t>(it >> 4) * a.H + rt * 128 + (it & 15) * 8;
            const float w[8] = {v[k][0].x, v[k][0].y, v[k][0].z, v[k][0].w, v[k][1].x, v[k][1].y, v[k][1].z, v[k][1].w};
            *reinterpret_cast<uint4*>(a.y + o) = pack_bf16x8(w, a.residual != nullptr ? a.residual + o : nullptr);
            float4* z = reinterpret_cast<float4*>(a.accum + o);
            __stcg(z, make_float4(0.f, 0.f, 0.f, 0.f));
            __stcg(z + 1, make_float4(0.f, 0.f, 0.f, 0.f));
          }
        }
        if (et == 0) a.tile_cnt[rt] = 0u;
      }
      if (et == 0) SLICE_STAMP(14);
    }
    if (!ok) *abort_flag = 1;
  }

  // ------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // neither block leaves while the partner may still write into its shared
  // memory or arrive on its barriers
  __syncwarp();
  cluster_sync_all();
  if (threadIdx.x == 0) SLICE_STAMP(15);
  if (warp == 2) tmem_dealloc(tmem, 256);
}

namespace {
// Per device: the kernels' dynamic shared-memory limits have been raised.
// Internal linkage, so every loaded copy of the library sets its own.
constexpr int kMaxAttrDevices = 64;
std::atomic<bool> g_slice_attr_set[kMaxAttrDevices];

template <int NPAD>
cudaError_t launch_npad(const SliceArgs& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.NP * kSliceCluster);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = slice_smem(NPAD);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kSliceCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, mx_slice_kernel<NPAD>, a);
}
}  // namespace

cudaError_t launch_slice_kernel(const SliceArgs& a, int npad, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxAttrDevices) return cudaErrorInvalidDevice;
  if (!g_slice_attr_set[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(mx_slice_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(slice_smem(16)));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(mx_slice_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(slice_smem(32)));
    if (e != cudaSuccess) return e;
    g_slice_attr_set[dev].store(true, std::memory_order_release);
  }
  if (npad == 16) return launch_npad<16>(a, stream);
  if (npad == 32) return launch_npad<32>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fsops
