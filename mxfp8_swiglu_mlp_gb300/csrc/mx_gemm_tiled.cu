// mx_gemm_tiled.cu -- block-scaled MXFP8 GEMM for M > 128 (prefill shapes).
//
//   mx_gemm_tiled_kernel   C[M, N] = A^[M, K] * B^[N, K]^T with A and B E4M3
//                          codes plus UE8M0 scales per 32-block along K
//                          (tcgen05 tiled scale layout), fp32 accumulation in
//                          TMEM, bf16 or fp32 output.
//
// One block per SM walks the 128 x 256 output tiles.  In the pair form the
// grid runs as 2-block clusters that compute one 256 x 256 tile with
// cta_group::2 MMAs: each block loads its own A box and one half of the B box,
// and the pair's tensor cores read both halves.
// Warp 0 streams the A (128 x 128 B) and B (256 x 128 B) boxes of each K
// stage and their scale tiles by TMA into a four-stage ring; warp 1 issues
// the block-scaled MMAs (four K = 32 steps per stage) into one TMEM
// accumulator; warps 4-7 drain the finished tile (one output row per thread)
// while the next tile's stages already stream in.  There is no split-K and no
// communication between blocks: every tile has M rows of 128 tokens, so the
// work is plentiful and each block owns whole tiles.  The same block-scaled
// MMA form (kind::mxf8f6f4, scales copied to TMEM with tcgen05.cp) as the
// decode kernel, per the MXFP8 1x32 format of the Fish Audio post (p2
// "Estrategia de cuantizacion FP8").
#include <cuda_bf16.h>

#include <atomic>

#include "mx_internal.h"
#include "mx_mxfp8.cuh"
#include "mx_tiled.h"
#include "sm103.cuh"

namespace fsops {
using namespace dev;

namespace {

constexpr uint32_t kTBytesA = 128u * kTileK;             // 16 KB: A box of 128 rows
constexpr uint32_t kTBytesB = 256u * kTileK;             // 32 KB: B box of 256 rows (zero fill past N)
constexpr uint32_t kTCtlBytes = 1024u;
// 12 warps: 0 TMA, 1 MMA, 4-11 epilogue (two warps per TMEM lane quarter,
// one per half of the tile's columns)
constexpr int kTThreads = 384;
constexpr int kTEpiWarps = 8;
// output staging: per epilogue warp one 2 KB chunk of 32 rows (32 bf16 or 16
// fp32 columns), written to global memory by a TMA store
constexpr uint32_t kTChunkBytes = 2048u;
constexpr uint32_t kTStgBytes = kTEpiWarps * kTChunkBytes;

// Per launch form: blocks per cluster, pipeline stages and the stage layout.
//   single     one block per 128 x 256 tile; stage = A 16 KB | B 32 KB |
//              A scales 512 B | B scales 2 x 512 B.
//   pair MMA   2-block clusters computing one 256 x 256 tile with
//              cta_group::2 MMAs; each block holds its 128 A rows and its
//              128-row half of B (the pair's tensor cores read both halves),
//              so a block takes in 33.5 KB per K step instead of 49.5 KB;
//              stage = A 16 KB | B half 16 KB | A scales 512 B | B scales
//              2 x 512 B (both halves: each block's MMA scales all 256 B rows).
template <int FORM>
struct TForm {
  static constexpr int CL = FORM == kTiledSingle ? 1 : 2;
  static constexpr bool PAIR = FORM == kTiledPairMma;
  static constexpr int kStages = PAIR ? 6 : 4;
  static constexpr uint32_t kOffSfa = PAIR ? kTBytesA + kTBytesB / 2 : kTBytesA + kTBytesB;
  static constexpr uint32_t kOffSfb = kOffSfa + 512u;
  static constexpr uint32_t kStageBytes = PAIR ? 34816u : 51200u;  // 1024-aligned
  static constexpr size_t kSmem = kStages * kStageBytes + kTCtlBytes + kTStgBytes + 1024u;  // + alignment slack
};
static_assert(TForm<kTiledPairMma>::kSmem <= 232448u && TForm<kTiledSingle>::kSmem <= 232448u, "shared memory");
static_assert(TForm<kTiledPairMma>::kOffSfb + 1024u <= TForm<kTiledPairMma>::kStageBytes, "pair stage layout");
static_assert(kAccCols + kSfColsPerStage * 6 <= kTmemCols, "TMEM columns");

// tcgen05 forms of a CTA pair (cta_group::2): issued by one thread of the
// even block; they act on the TMEM (and read the shared memory) of both.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* smem_result, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_result)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar, uint16_t cta_mask) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "h"(cta_mask)
               : "memory");
}
__device__ __forceinline__ void tc_cp_pair_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
// D[256 x N] (+)= A[256 x 32] * B[N x 32]^T: rows 0..127 of A and D in the
// even block, 128..255 in the odd one; B rows 0..N/2-1 in the even block.
__device__ __forceinline__ void tc_mma_mxf8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%5], [%6], p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}
// Work item -> (row group, column tile).  Items are walked in bands of
// kTileBand row groups: within a band the row group changes fastest, so the
// blocks running at one time share each A band and each B tile among a few
// of them instead of all reading one A band (bounded L2 hot spots, both
// operands reused from L2).
#ifndef FSOPS_TILE_BAND
#define FSOPS_TILE_BAND 8
#endif
constexpr int kTileBand = FSOPS_TILE_BAND;
__device__ __forceinline__ void tile_coords(int item, int mrows, int NT, int& mg, int& nt) {
  const int band_items = kTileBand * NT;
  const int band = item / band_items, r = item - band * band_items;
  const int rows = min(kTileBand, mrows - band * kTileBand);  // the last band may be shorter
  mg = band * kTileBand + r % rows;
  nt = r / rows;
}
// 2-D tiled load into this block's shared memory whose completion (bytes) is
// counted on the mbarrier at cluster address `bar` -- this block's or its
// pair partner's (cta_group::2).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}
// Instruction descriptor of kind::mxf8f6f4 with E4M3 A and B, UE8M0 scales,
// both K-major, M = 256 (a pair), N columns.
__host__ __device__ constexpr uint32_t idesc_mxf8_e4m3_m256(uint32_t n) {
  return (((n >> 3) & 0x3Fu) << 17) | (1u << 23) | ((256u >> 7) << 27);
}

struct TWait {
  volatile int* abort;
  uint32_t* status;
  uint64_t timeout_ns;
};

// Bounded mbarrier wait: gives up when the block aborted or the limit passed
// (then records FSOPS_ERR_TIMEOUT with the wait site and the block).
__device__ __forceinline__ bool twait(const TWait& w, uint64_t* bar, uint32_t parity, uint32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t n = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++n & 15u) == 0) {
      if (*w.abort) return false;
      if (globaltimer_ns() - t0 > w.timeout_ns) {
        *w.abort = 1;
        atomicCAS(w.status, 0u, (5u << 24) | ((site & 0xFFu) << 16) | (blockIdx.x & 0xFFFFu));
        return false;
      }
    }
  }
  return true;
}
// The same for a barrier that blocks of the cluster arrive on remotely:
// acquires at cluster scope.
__device__ __forceinline__ bool twait_cluster(const TWait& w, uint64_t* bar, uint32_t parity, uint32_t site) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t n = 0;
  while (!mbar_try_wait_cluster(bar, parity)) {
    if ((++n & 15u) == 0) {
      if (*w.abort) return false;
      if (globaltimer_ns() - t0 > w.timeout_ns) {
        *w.abort = 1;
        atomicCAS(w.status, 0u, (5u << 24) | ((site & 0xFFu) << 16) | (blockIdx.x & 0xFFFFu));
        return false;
      }
    }
  }
  return true;
}
__device__ __forceinline__ void tdrain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > 200000000ull) return;
}

// SwiGLU epilogue of one 128-column chunk of a gate/up tile, for the warp of
// TMEM lane quarter q4 (token rows mt * 128 + 32 q4 + lane).  The chunk's
// columns 0..63 hold the gate sums of features f0 .. f0 + 63 (f0 = 128 nt +
// 64 half), columns 64..127 the up sums of the same features.
// swiglu_load reads the chunk's raw sums into registers, so the accumulator
// can be released before any arithmetic; swiglu_store then forms h = SiLU(g)
// * u and quantises each 32-block with the rule of the standalone quantiser.
// Each thread owns one token row, so a block's amax is its own.
__device__ __forceinline__ void swiglu_load(uint32_t tcol, uint32_t (&g)[4][16], uint32_t (&u)[4][16]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) tmem_ld16(tcol + 16 * j, g[j]);
#pragma unroll
  for (int j = 0; j < 4; ++j) tmem_ld16(tcol + kPairRows + 16 * j, u[j]);
  tmem_ld_wait();
}
// Rows past M write their scales only (their sums are 0: TMA zero-fills A
// past M, so the scale byte is 0).
__device__ __forceinline__ void swiglu_store(const TiledArgs& a, int r, int f0, const uint32_t (&g)[4][16],
                                             const uint32_t (&u)[4][16]) {
  const int I = a.N >> 1;
  uint32_t sbytes = 0;
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    float h[32];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      h[i] = silu_mul(__uint_as_float(g[2 * b + (i >> 4)][i & 15]), __uint_as_float(u[2 * b + (i >> 4)][i & 15]));
      amax = fmaxf(amax, fabsf(h[i]));
    }
    const uint32_t sc = ue8m0_from_amax(amax);
    const float inv = inv_scale_from_ue8m0(sc);
    sbytes |= sc << (8 * b);
    if (r < a.M) {
      uint32_t pk[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        pk[i] = e4m3_code(h[4 * i] * inv) | (e4m3_code(h[4 * i + 1] * inv) << 8) |
                (e4m3_code(h[4 * i + 2] * inv) << 16) | (e4m3_code(h[4 * i + 3] * inv) << 24);
      uint4* d = reinterpret_cast<uint4*>(a.h_codes + static_cast<size_t>(r) * I + f0 + 32 * b);
      d[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      d[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
    }
  }
  // the scales of 32-blocks f0 / 32 and f0 / 32 + 1 sit in adjacent bytes
  *reinterpret_cast<uint16_t*>(a.h_sf + tiled_sf_offset(r, f0 >> 5, I >> 7)) = static_cast<uint16_t>(sbytes);
}
__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo, uint32_t hi) {
  const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
  return *reinterpret_cast<const uint32_t*>(&b2);
}

}  // namespace

template <int FORM, bool SWIGLU>
__global__ void __launch_bounds__(kTThreads, 1) mx_gemm_tiled_kernel(const __grid_constant__ TiledArgs a) {
  using F = TForm<FORM>;
  constexpr int CL = F::CL;
  constexpr bool PAIR = F::PAIR;
  constexpr int NS = F::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align(smem_raw, 1024);
  uint8_t* ctl = smem + NS * F::kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctl);  // this block's stage has landed
  uint64_t* empty = full + NS;                         // the stage's MMAs have completed
  uint64_t* acc_full = empty + NS;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint8_t* ostg = ctl + kTCtlBytes;  // [kTEpiWarps][kTChunkBytes]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // rank in the 2-block cluster (blockIdx.x % 2 for clusters of 2 along x)
  const int rank = CL > 1 ? static_cast<int>(blockIdx.x % CL) : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      // pair MMA: a stage is free once the one pair MMA (committed to both
      // blocks) has consumed it
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    // one arrival per epilogue warp (of both blocks for the pair MMA)
    mbar_init(acc_empty, (PAIR ? 2 : 1) * kTEpiWarps);
    mbar_init(drain, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    if constexpr (PAIR) {  // one warp of each block of the pair allocates, collectively
      tmem_alloc_pair(tmem_slot, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, kTmemCols);
      tmem_relinquish();
    }
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&a.tm_a);
    tma_prefetch_desc(&a.tm_b);
    if (PAIR) {
      tma_prefetch_desc(&a.tm_sfa);
      tma_prefetch_desc(&a.tm_sfb);
    }
    if (!SWIGLU) tma_prefetch_desc(&a.tm_c);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the cluster's barriers are initialised before any block arrives on its
  // partner's
  if (CL > 1) cluster_sync_all();
  const uint32_t tmem = *tmem_slot;
  const TWait w{abort_flag, a.status, a.timeout_ns};
  // work items: CL vertically adjacent tiles (one per block of the cluster)
  const int G = gridDim.x / CL;
  const int first = blockIdx.x / CL;
  const int mrows = (a.MT + CL - 1) / CL;  // row groups of CL tiles
  const int ntiles = mrows * a.NT;
  const uint16_t all_ctas = static_cast<uint16_t>((1u << CL) - 1u);  // the commit arrives in both blocks of a pair

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ TMA producer
    const uint64_t pol_a = l2_policy_evict_last();   // A tiles are re-read by every N tile
    const uint64_t pol_b = l2_policy_evict_last();   // B tiles by every M tile
    int stage = 0;
    uint32_t round = 0, issued_mask = 0, issued_parity = 0;
    bool ok = true;
    for (int tile = first; tile < ntiles && ok; tile += G) {
      int mg, nt;
      tile_coords(tile, mrows, a.NT, mg, nt);
      const int mt = mg * CL + rank;
      const int mt_sf = mt < a.MT ? mt : a.MT - 1;  // a row tile past M: zero codes, any finite scales
      const bool v1 = nt * 256 + 128 < a.N;        // always for the pair MMA (N % 256 == 0)
      for (int ks = 0; ks < a.KS; ++ks) {
        // (the partner's MMA commit arrives here in the cluster forms)
        const bool free_stage = CL > 1 ? twait_cluster(w, &empty[stage], (round & 1u) ^ 1u, kSiteEmpty)
                                       : twait(w, &empty[stage], (round & 1u) ^ 1u, kSiteEmpty);
        if (!free_stage) { ok = false; break; }
        uint8_t* st = smem + static_cast<size_t>(stage) * F::kStageBytes;
        if constexpr (PAIR) {
          // Both blocks' loads complete on the even block's full[stage], which
          // expects the bytes of both; the odd block does not arrive on it.
          const uint32_t full0 = mapa_shared(&full[stage], 0);
          if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2u * (kTBytesA + kTBytesB / 2 + 1536u));
          tma_load_2d_pair(st, &a.tm_a, full0, ks * kTileK, mt * 128, pol_a);
          tma_load_2d_pair(st + kTBytesA, &a.tm_b, full0, ks * kTileK, nt * 256 + rank * 128, pol_b);
          tma_load_2d_pair(st + F::kOffSfa, &a.tm_sfa, full0, 0, mt_sf * a.KS + ks, pol_a);
          tma_load_2d_pair(st + F::kOffSfb, &a.tm_sfb, full0, 0, 2 * nt * a.KS + ks, pol_b);
          tma_load_2d_pair(st + F::kOffSfb + 512, &a.tm_sfb, full0, 0, (2 * nt + 1) * a.KS + ks, pol_b);
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | ((round & 1u) << stage);
          if (++stage == NS) { stage = 0; ++round; }
          continue;
        }
        mbar_arrive_expect_tx(&full[stage], kTBytesA + kTBytesB + 512u + (v1 ? 1024u : 512u));
        tma_load_2d(st, &a.tm_a, &full[stage], ks * kTileK, mt * 128, pol_a);
        tma_load_2d(st + kTBytesA, &a.tm_b, &full[stage], ks * kTileK, nt * 256, pol_b);
        bulk_load(st + F::kOffSfa, a.sf_a + (static_cast<size_t>(mt_sf) * a.KS + ks) * 512, 512, &full[stage],
                  pol_a);
        const uint8_t* sfb = a.sf_b + (static_cast<size_t>(2 * nt) * a.KS + ks) * 512;
        bulk_load(st + F::kOffSfb, sfb, 512, &full[stage], pol_b);
        if (v1) bulk_load(st + F::kOffSfb + 512, sfb + static_cast<size_t>(a.KS) * 512, 512, &full[stage], pol_b);
        issued_mask |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | ((round & 1u) << stage);
        if (++stage == NS) { stage = 0; ++round; }
      }
    }
    if (!ok) *abort_flag = 1;
    // every load this block issued has landed before it leaves (for the pair,
    // the even block's full[] counts both blocks' loads; an odd block that
    // gave up waits out its loads by time instead)
    if (!PAIR || rank == 0) {
      for (int s = 0; s < NS; ++s)
        if (issued_mask & (1u << s)) tdrain(&full[s], (issued_parity >> s) & 1u);
    } else if (!ok) {
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 1000000ull) {
      }
    }
  } else if (warp == 1 && lane == 0 && (!PAIR || rank == 0)) {
    // ------------------------------------------------ MMA issuer (the even block of a pair)
    int stage = 0;
    uint32_t round = 0, acc_round = 0;
    bool ok = true;
    const uint32_t sf_base = tmem + kAccCols;
    for (int tile = first; tile < ntiles && ok; tile += G) {
      int mg, nt;
      tile_coords(tile, mrows, a.NT, mg, nt);
      const bool v1 = nt * 256 + 128 < a.N;
      const uint32_t idesc0 = PAIR ? idesc_mxf8_e4m3_m256(256u) : idesc_mxf8_e4m3(v1 ? 256u : 128u, 0, 0);
      // both blocks' epilogues have read the accumulator (remote arrivals for the pair)
      const bool free_acc = PAIR ? twait_cluster(w, acc_empty, (acc_round & 1u) ^ 1u, kSiteAccEmpty)
                                 : twait(w, acc_empty, (acc_round & 1u) ^ 1u, kSiteAccEmpty);
      if (!free_acc) { ok = false; break; }
      tc_fence_after();
      for (int ks = 0; ks < a.KS; ++ks) {
        // (the pair's odd block's loads complete on this barrier too)
        const bool landed = PAIR ? twait_cluster(w, &full[stage], round & 1u, kSiteFullW)
                                 : twait(w, &full[stage], round & 1u, kSiteFullW);
        if (!landed) { ok = false; break; }
        tc_fence_after();
        uint8_t* st = smem + static_cast<size_t>(stage) * F::kStageBytes;
        const uint32_t sfc = sf_base + kSfColsPerStage * stage;
        const uint64_t d_sfa = smem_desc(smem_u32(st + F::kOffSfa), 0, 128, kSwizzleNone);
        const uint64_t d_sfb0 = smem_desc(smem_u32(st + F::kOffSfb), 0, 128, kSwizzleNone);
        const uint64_t d_sfb1 = smem_desc(smem_u32(st + F::kOffSfb + 512), 0, 128, kSwizzleNone);
        if constexpr (PAIR) {
          tc_cp_pair_32x128b_warpx4(sfc, d_sfa);
          tc_cp_pair_32x128b_warpx4(sfc + 4, d_sfb0);
          tc_cp_pair_32x128b_warpx4(sfc + 8, d_sfb1);
        } else {
          tc_cp_32x128b_warpx4(sfc, d_sfa);
          tc_cp_32x128b_warpx4(sfc + 4, d_sfb0);
          if (v1) tc_cp_32x128b_warpx4(sfc + 8, d_sfb1);
        }
        const uint32_t sa = smem_u32(st), sb = smem_u32(st + kTBytesA);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t idesc = idesc0 | (static_cast<uint32_t>(k) << 4) | (static_cast<uint32_t>(k) << 29);
          const uint64_t da = smem_desc(sa + 32 * k, 16, 1024, kSwizzle128B);
          const uint64_t db = smem_desc(sb + 32 * k, 16, 1024, kSwizzle128B);
          if constexpr (PAIR) tc_mma_mxf8_pair(tmem, da, db, idesc, sfc, sfc + 4, (ks > 0 || k > 0) ? 1u : 0u);
          else tc_mma_mxf8(tmem, da, db, idesc, sfc, sfc + 4, (ks > 0 || k > 0) ? 1u : 0u);
        }
        // the stage is free in this block (and, for the pair MMA, in the partner)
        if constexpr (FORM == kTiledSingle) tc_commit(&empty[stage]);
        else tc_commit_pair(&empty[stage], all_ctas);
        if (++stage == NS) { stage = 0; ++round; }
      }
      if (!ok) break;
      if constexpr (PAIR) tc_commit_pair(acc_full, all_ctas);
      else tc_commit(acc_full);
      ++acc_round;
    }
    if (!ok) *abort_flag = 1;
    if constexpr (PAIR) tc_commit_pair(drain, 1);
    else tc_commit(drain);
    tdrain(drain, 0);
  } else if (warp >= 4) {
    // ------------------------------------------------ epilogue
    // Warp e (4..11) reads TMEM lane quarter e % 4 (rows 32 (e % 4) .. + 31 of
    // the tile) and half (e - 4) / 4 of the columns.  It turns them into 2 KB
    // chunks in shared memory that TMA stores to C; the accumulator is
    // released as soon as every warp has read its part, while the stores drain.
    const int ew = warp - 4, q4 = warp & 3, half = ew >> 2;
    const uint32_t tlane = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    const int cw = a.c_f32 ? 16 : 32;  // columns per chunk
    uint8_t* buf = ostg + ew * kTChunkBytes;
    // the accumulator's readiness counter sits in the even block for the pair MMA
    const uint32_t acc_empty0 = PAIR ? mapa_shared(acc_empty, 0) : 0u;
    // this warp has read its part of the accumulator: one arrival per warp
    auto release_acc = [&]() {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR && rank == 1) mbar_arrive_remote(acc_empty0);
        else mbar_arrive(acc_empty);
      }
    };
    uint32_t acc_round = 0;
    for (int tile = first; tile < ntiles; tile += G) {
      int mg, nt;
      tile_coords(tile, mrows, a.NT, mg, nt);
      const int mt = mg * CL + rank;
      const int ncols = (nt * 256 + 128 < a.N) ? 256 : 128;
      const bool ready = PAIR ? twait_cluster(w, acc_full, acc_round & 1u, kSiteAccFull)
                              : twait(w, acc_full, acc_round & 1u, kSiteAccFull);
      if (!ready) break;
      ++acc_round;
      tc_fence_after();
      if (SWIGLU) {
        const bool has = ncols > half * 128;
        uint32_t g[4][16], u[4][16];
        if (has) swiglu_load(tlane + half * 128, g, u);
        release_acc();
        if (has) swiglu_store(a, mt * 128 + q4 * 32 + lane, nt * 128 + half * 64, g, u);
        continue;
      }
      const int cbeg = half * (ncols >> 1), cend = cbeg + (ncols >> 1);
      if (!a.c_f32) {
        // bf16 C: the warp's columns are read and packed in registers first,
        // so the accumulator is free again before any store work starts
        const int nch = (cend - cbeg) >> 5;  // 32-column chunks: 4, or 2 on a 128-column tile
        uint32_t pk[4][16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (j < nch) {
            uint32_t v[2][16];
            tmem_ld16(tlane + cbeg + 32 * j, v[0]);
            tmem_ld16(tlane + cbeg + 32 * j + 16, v[1]);
            tmem_ld_wait();
            const int r = mt * 128 + q4 * 32 + lane;
            if (a.residual != nullptr && r < a.M) {  // C = residual + the sums, rounded once
              const uint4* rp =
                  reinterpret_cast<const uint4*>(a.residual + static_cast<size_t>(r) * a.N + nt * 256 + cbeg + 32 * j);
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const uint4 rv = rp[q];
                const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const int e = 8 * q + 2 * i;
                  v[e >> 4][e & 15] = __float_as_uint(__uint_as_float(v[e >> 4][e & 15]) + __uint_as_float(rw[i] << 16));
                  v[e >> 4][(e + 1) & 15] =
                      __float_as_uint(__uint_as_float(v[e >> 4][(e + 1) & 15]) + __uint_as_float(rw[i] & 0xFFFF0000u));
                }
              }
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[j][i] = pack_bf16x2(v[i >> 3][(2 * i) & 15], v[i >> 3][(2 * i + 1) & 15]);
          }
        }
        release_acc();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (j < nch) {
            // the store issued from this buffer before has read it
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
            uint4* rowp = reinterpret_cast<uint4*>(buf + lane * 64);  // 32 rows x 64 B
#pragma unroll
            for (int q = 0; q < 4; ++q) rowp[q] = make_uint4(pk[j][4 * q], pk[j][4 * q + 1], pk[j][4 * q + 2], pk[j][4 * q + 3]);
            fence_proxy_async_shared();  // the TMA store reads what the warp wrote
            __syncwarp();
            if (lane == 0 && mt * 128 + q4 * 32 < a.M) {
              tma_store_2d(&a.tm_c, buf, nt * 256 + cbeg + 32 * j, mt * 128 + q4 * 32);
              bulk_commit_group();
            }
          }
        }
        continue;
      }
#pragma unroll 1
      for (int c0 = cbeg; c0 < cend; c0 += cw) {
        uint32_t v[2][16];
        tmem_ld16(tlane + c0, v[0]);
        if (!a.c_f32) tmem_ld16(tlane + c0 + 16, v[1]);
        tmem_ld_wait();
        // the store issued from this buffer before has read it
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
        uint4* rowp = reinterpret_cast<uint4*>(buf + lane * 64);  // 32 rows x 64 B
        if (a.c_f32) {
#pragma unroll
          for (int q = 0; q < 4; ++q) rowp[q] = make_uint4(v[0][4 * q], v[0][4 * q + 1], v[0][4 * q + 2], v[0][4 * q + 3]);
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t pk[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int e = 8 * q + 2 * j;
              const __nv_bfloat162 b2 =
                  __floats2bfloat162_rn(__uint_as_float(v[e >> 4][e & 15]), __uint_as_float(v[(e + 1) >> 4][(e + 1) & 15]));
              pk[j] = *reinterpret_cast<const uint32_t*>(&b2);
            }
            rowp[q] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        }
        fence_proxy_async_shared();  // the TMA store reads what the warp wrote
        __syncwarp();
        if (lane == 0 && mt * 128 + q4 * 32 < a.M) {  // rows past M are clipped; a box wholly past M is not issued
          tma_store_2d(&a.tm_c, buf, nt * 256 + c0, mt * 128 + q4 * 32);
          bulk_commit_group();
        }
      }
      release_acc();
    }
    if (lane == 0) bulk_wait_all();  // every store has landed before the block ends
  }

  // ------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // no block leaves while its partner may still arrive on its barriers
  if (CL > 1) {
    __syncwarp();
    cluster_sync_all();
  }
  if (warp == 1) {
    if constexpr (PAIR) tmem_dealloc_pair(tmem, kTmemCols);
    else tmem_dealloc(tmem, kTmemCols);
  }
}

namespace {
// Per device: the kernel instances' dynamic shared-memory limits have
// been raised.  Internal linkage (not a static inside a template, which the
// toolchain would merge across every loaded copy of the library), so each
// copy sets the limits of its own kernels.
constexpr int kMaxAttrDevices = 64;
std::atomic<bool> g_smem_attr_set[kMaxAttrDevices];

template <int FORM, bool SWIGLU>
cudaError_t set_smem_limit() {
  return cudaFuncSetAttribute(mx_gemm_tiled_kernel<FORM, SWIGLU>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(TForm<FORM>::kSmem));
}
cudaError_t set_smem_limits() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxAttrDevices) return cudaErrorInvalidDevice;
  if (g_smem_attr_set[dev].load(std::memory_order_acquire)) return cudaSuccess;
  const cudaError_t es[4] = {set_smem_limit<kTiledSingle, false>(), set_smem_limit<kTiledSingle, true>(),
                             set_smem_limit<kTiledPairMma, false>(), set_smem_limit<kTiledPairMma, true>()};
  for (cudaError_t x : es)
    if (x != cudaSuccess) return x;
  g_smem_attr_set[dev].store(true, std::memory_order_release);
  return cudaSuccess;
}

template <int FORM, bool SWIGLU>
cudaError_t launch_tiled(const TiledArgs& a, int grid, cudaStream_t stream) {
  constexpr int CL = TForm<FORM>::CL;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTThreads);
  cfg.dynamicSmemBytes = TForm<FORM>::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = CL > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, mx_gemm_tiled_kernel<FORM, SWIGLU>, a);
}
template <bool SWIGLU>
cudaError_t launch_form(const TiledArgs& a, int grid, cudaStream_t stream) {
  if (a.form == kTiledPairMma) return launch_tiled<kTiledPairMma, SWIGLU>(a, grid, stream);
  return launch_tiled<kTiledSingle, SWIGLU>(a, grid, stream);
}
}  // namespace

cudaError_t launch_gemm_tiled(const TiledArgs& a, int sms, cudaStream_t stream) {
  // The host chose the form (and encoded tm_b with 128-row boxes for the
  // pair form).  The pair form takes CL = 2 vertically adjacent row tiles per
  // work item; grid = one block per SM at most.
  if (a.form == kTiledPairMma && (a.N % 256 != 0 || a.MT < 2)) return cudaErrorInvalidValue;
  const int cl = a.form == kTiledSingle ? 1 : 2;
  const int items = ((a.MT + cl - 1) / cl) * a.NT;
  const int grid = (items < sms / cl ? items : sms / cl) * cl;
  const cudaError_t e = set_smem_limits();
  if (e != cudaSuccess) return e;
  return a.swiglu ? launch_form<true>(a, grid, stream) : launch_form<false>(a, grid, stream);
}

}  // namespace fsops
