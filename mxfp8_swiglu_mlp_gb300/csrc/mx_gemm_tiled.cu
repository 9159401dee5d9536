// mx_gemm_tiled.cu -- block-scaled MXFP8 GEMM for M > 128 (prefill shapes).
//
//   mx_gemm_tiled_kernel   C[M, N] = A^[M, K] * B^[N, K]^T with A and B E4M3
//                          codes plus UE8M0 scales per 32-block along K
//                          (tcgen05 tiled scale layout), fp32 accumulation in
//                          TMEM, bf16 or fp32 output.
//
// One block per SM walks the 128 x 256 output tiles.  With CL = 2 the grid
// runs as 2-block clusters that take vertically adjacent tiles (rows 256 p ..
// 256 p + 255, same columns): each block loads its own A box and one half of
// the shared B box, multicast into both blocks, so the pair reads each B
// stage once from L2 (a third less operand traffic per block).
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

constexpr int kTStages = 4;
constexpr uint32_t kTBytesA = 128u * kTileK;             // 16 KB
constexpr uint32_t kTBytesB = 256u * kTileK;             // 32 KB (box of 256 rows, zero fill past N)
constexpr uint32_t kTOffSfa = kTBytesA + kTBytesB;       // 512 B: A scale tile
constexpr uint32_t kTOffSfb = kTOffSfa + 512u;           // 1024 B: B scale tiles (two row halves)
constexpr uint32_t kTStageBytes = 51200u;                // 1024-aligned
constexpr uint32_t kTCtlBytes = 1024u;
// 12 warps: 0 TMA, 1 MMA, 4-11 epilogue (two warps per TMEM lane quarter,
// one per half of the tile's columns)
constexpr int kTThreads = 384;
constexpr int kTEpiWarps = 8;
// output staging: per epilogue warp one 2 KB chunk of 32 rows (32 bf16 or 16
// fp32 columns), written to global memory by a TMA store
constexpr uint32_t kTChunkBytes = 2048u;
constexpr uint32_t kTStgBytes = kTEpiWarps * kTChunkBytes;
constexpr size_t kTSmem = kTStages * kTStageBytes + kTCtlBytes + kTStgBytes + 1024u;  // + alignment slack

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

template <int CL, bool SWIGLU>
__global__ void __launch_bounds__(kTThreads, 1) mx_gemm_tiled_kernel(const __grid_constant__ TiledArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ctl = smem + kTStages * kTStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctl);
  uint64_t* empty = full + kTStages;
  uint64_t* acc_full = empty + kTStages;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint8_t* ostg = ctl + kTCtlBytes;  // [kTEpiWarps][kTChunkBytes]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kTStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], CL);  // a stage is free once every block of the cluster has consumed it
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 32 * kTEpiWarps);
    mbar_init(drain, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&a.tm_a);
    tma_prefetch_desc(&a.tm_b);
    if (!SWIGLU) tma_prefetch_desc(&a.tm_c);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the cluster's barriers are initialised before any multicast reaches them
  if (CL > 1) cluster_sync_all();
  const uint32_t tmem = *tmem_slot;
  const TWait w{abort_flag, a.status, a.timeout_ns};
  // work items: CL vertically adjacent tiles (one per block of the cluster)
  const int rank = CL > 1 ? static_cast<int>(blockIdx.x % CL) : 0;
  const int G = gridDim.x / CL;
  const int first = blockIdx.x / CL;
  const int mrows = (a.MT + CL - 1) / CL;  // row groups of CL tiles
  const int ntiles = mrows * a.NT;
  const uint16_t all_ctas = static_cast<uint16_t>((1u << CL) - 1u);

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ TMA producer
    const uint64_t pol_a = l2_policy_evict_last();   // A tiles are re-read by every N tile
    const uint64_t pol_b = l2_policy_evict_last();   // B tiles by every M tile
    int stage = 0;
    uint32_t round = 0, issued_mask = 0, issued_parity = 0;
    bool ok = true;
    for (int tile = first; tile < ntiles && ok; tile += G) {
      const int mt = (tile / a.NT) * CL + rank, nt = tile % a.NT;
      const int mt_sf = mt < a.MT ? mt : a.MT - 1;  // a row tile past M: zero codes, any finite scales
      const bool v1 = nt * 256 + 128 < a.N;
      for (int ks = 0; ks < a.KS; ++ks) {
        if (!twait(w, &empty[stage], (round & 1u) ^ 1u, kSiteEmpty)) { ok = false; break; }
        uint8_t* st = smem + static_cast<size_t>(stage) * kTStageBytes;
        mbar_arrive_expect_tx(&full[stage], kTBytesA + kTBytesB + 512u + (v1 ? 1024u : 512u));
        tma_load_2d(st, &a.tm_a, &full[stage], ks * kTileK, mt * 128, pol_a);
        if (CL == 1) {
          tma_load_2d(st + kTBytesA, &a.tm_b, &full[stage], ks * kTileK, nt * 256, pol_b);
        } else {
          // this block's 128-row half of B, into the same place in both blocks
          tma_load_2d_multicast(st + kTBytesA + rank * (kTBytesB / 2), &a.tm_b, &full[stage], ks * kTileK,
                                nt * 256 + rank * 128, all_ctas, pol_b);
        }
        bulk_load(st + kTOffSfa, a.sf_a + (static_cast<size_t>(mt_sf) * a.KS + ks) * 512, 512, &full[stage], pol_a);
        const uint8_t* sfb = a.sf_b + (static_cast<size_t>(2 * nt) * a.KS + ks) * 512;
        bulk_load(st + kTOffSfb, sfb, 512, &full[stage], pol_b);
        if (v1) bulk_load(st + kTOffSfb + 512, sfb + static_cast<size_t>(a.KS) * 512, 512, &full[stage], pol_b);
        issued_mask |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | ((round & 1u) << stage);
        if (++stage == kTStages) { stage = 0; ++round; }
      }
    }
    if (!ok) *abort_flag = 1;
    for (int s = 0; s < kTStages; ++s)
      if (issued_mask & (1u << s)) tdrain(&full[s], (issued_parity >> s) & 1u);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------ MMA issuer
    int stage = 0;
    uint32_t round = 0, acc_round = 0;
    bool ok = true;
    const uint32_t sf_base = tmem + kAccCols;
    for (int tile = first; tile < ntiles && ok; tile += G) {
      const int nt = tile % a.NT;
      const bool v1 = nt * 256 + 128 < a.N;
      const uint32_t idesc0 = idesc_mxf8_e4m3(v1 ? 256u : 128u, 0, 0);
      if (!twait(w, acc_empty, (acc_round & 1u) ^ 1u, kSiteAccEmpty)) { ok = false; break; }
      tc_fence_after();
      for (int ks = 0; ks < a.KS; ++ks) {
        if (!twait(w, &full[stage], round & 1u, kSiteFullW)) { ok = false; break; }
        tc_fence_after();
        uint8_t* st = smem + static_cast<size_t>(stage) * kTStageBytes;
        const uint32_t sfc = sf_base + kSfColsPerStage * stage;
        tc_cp_32x128b_warpx4(sfc, smem_desc(smem_u32(st + kTOffSfa), 0, 128, kSwizzleNone));
        tc_cp_32x128b_warpx4(sfc + 4, smem_desc(smem_u32(st + kTOffSfb), 0, 128, kSwizzleNone));
        if (v1) tc_cp_32x128b_warpx4(sfc + 8, smem_desc(smem_u32(st + kTOffSfb + 512), 0, 128, kSwizzleNone));
        const uint32_t sa = smem_u32(st), sb = smem_u32(st + kTBytesA);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t idesc = idesc0 | (static_cast<uint32_t>(k) << 4) | (static_cast<uint32_t>(k) << 29);
          tc_mma_mxf8(tmem, smem_desc(sa + 32 * k, 16, 1024, kSwizzle128B), smem_desc(sb + 32 * k, 16, 1024, kSwizzle128B),
                      idesc, sfc, sfc + 4, (ks > 0 || k > 0) ? 1u : 0u);
        }
        // the stage is free in this block and (for the multicast half) in the partner
        if (CL == 1) tc_commit(&empty[stage]);
        else tc_commit_multicast(&empty[stage], all_ctas);
        if (++stage == kTStages) { stage = 0; ++round; }
      }
      if (!ok) break;
      tc_commit(acc_full);
      ++acc_round;
    }
    if (!ok) *abort_flag = 1;
    tc_commit(drain);
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
    uint32_t acc_round = 0;
    for (int tile = first; tile < ntiles; tile += G) {
      const int mt = (tile / a.NT) * CL + rank, nt = tile % a.NT;
      const int ncols = (nt * 256 + 128 < a.N) ? 256 : 128;
      if (!twait(w, acc_full, acc_round & 1u, kSiteAccFull)) break;
      ++acc_round;
      tc_fence_after();
      if (SWIGLU) {
        const bool has = ncols > half * 128;
        uint32_t g[4][16], u[4][16];
        if (has) swiglu_load(tlane + half * 128, g, u);
        tc_fence_before();
        mbar_arrive(acc_empty);
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
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[j][i] = pack_bf16x2(v[i >> 3][(2 * i) & 15], v[i >> 3][(2 * i + 1) & 15]);
          }
        }
        tc_fence_before();
        mbar_arrive(acc_empty);
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
      tc_fence_before();
      mbar_arrive(acc_empty);
    }
    if (lane == 0) bulk_wait_all();  // every store has landed before the block ends
  }

  // ------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // no block leaves while its partner may still multicast into it or arrive on it
  if (CL > 1) {
    __syncwarp();
    cluster_sync_all();
  }
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

namespace {
// Per device: the four kernel instances' dynamic shared-memory limits have
// been raised.  Internal linkage (not a static inside a template, which the
// toolchain would merge across every loaded copy of the library), so each
// copy sets the limits of its own kernels.
constexpr int kMaxAttrDevices = 64;
std::atomic<bool> g_smem_attr_set[kMaxAttrDevices];

cudaError_t set_smem_limits() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxAttrDevices) return cudaErrorInvalidDevice;
  if (g_smem_attr_set[dev].load(std::memory_order_acquire)) return cudaSuccess;
  const int smem = static_cast<int>(kTSmem);
  e = cudaFuncSetAttribute(mx_gemm_tiled_kernel<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(mx_gemm_tiled_kernel<2, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(mx_gemm_tiled_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(mx_gemm_tiled_kernel<2, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) g_smem_attr_set[dev].store(true, std::memory_order_release);
  return e;
}

template <int CL, bool SWIGLU>
cudaError_t launch_tiled(const TiledArgs& a, int grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTThreads);
  cfg.dynamicSmemBytes = kTSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = CL > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, mx_gemm_tiled_kernel<CL, SWIGLU>, a);
}
}  // namespace

cudaError_t launch_gemm_tiled(const TiledArgs& a, int sms, cudaStream_t stream) {
  // pairs of blocks on vertically adjacent tiles when there are at least two
  // row tiles; grid = one block per SM at most
  const bool pairs = a.cluster_ok != 0;  // the host chose it and encoded tm_b with 128-row boxes
  const int cl = pairs ? 2 : 1;
  const int items = ((a.MT + cl - 1) / cl) * a.NT;
  const int grid = (items < sms / cl ? items : sms / cl) * cl;
  const cudaError_t e = set_smem_limits();
  if (e != cudaSuccess) return e;
  if (a.swiglu) return pairs ? launch_tiled<2, true>(a, grid, stream) : launch_tiled<1, true>(a, grid, stream);
  return pairs ? launch_tiled<2, false>(a, grid, stream) : launch_tiled<1, false>(a, grid, stream);
}

}  // namespace fsops
