// mx_device.cuh -- device helpers shared by the decode kernels
// (mx_kernels.cu, mx_slice.cu): bf16 blocks to MXFP8 codes, and the bounded
// waits that report a timeout through the status word instead of hanging.
#pragma once
#include <cstdint>

#include "mx_internal.h"
#include "mx_mxfp8.cuh"
#include "sm103.cuh"

namespace fsops {
using namespace dev;

// ----------------------------------------------------------------------------
// bf16 blocks to MXFP8 codes (the rule of mx_mxfp8.cuh)
// ----------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Quantise one 32-element bf16 block already in registers (raw = 64 bytes)
// into 32 codes packed four to a word; returns the scale byte.
__device__ __forceinline__ uint32_t quantize_block_pack(const uint4 (&raw)[4], uint32_t (&packed)[8]) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(raw);
  // largest magnitude: the bf16 bit patterns without sign compare as unsigned
  // integers; a tree of per-halfword maxima keeps the dependency chain short
  uint32_t m[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) m[i] = __vmaxu2(w[2 * i] & 0x7FFF7FFFu, w[2 * i + 1] & 0x7FFF7FFFu);
#pragma unroll
  for (int d = 4; d >= 1; d >>= 1)
#pragma unroll
    for (int i = 0; i < d; ++i) m[i] = __vmaxu2(m[i], m[i + d]);
  const uint32_t amax_bits = max(m[0] & 0xFFFFu, m[0] >> 16) << 16;
  const uint32_t s = ue8m0_from_amax(__uint_as_float(amax_bits));
  const float inv = inv_scale_from_ue8m0(s);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    packed[i] = e4m3x4_code(bf16_lo(w[2 * i]) * inv, bf16_hi(w[2 * i]) * inv, bf16_lo(w[2 * i + 1]) * inv,
                            bf16_hi(w[2 * i + 1]) * inv);
  return s;
}
// The same for RMSNorm(x) * gamma: the 32 values x * rn * gamma (fp32, in
// that order; rn = 1 / rms of the block's row, gv the block's 32 gains as
// bf16), quantised with the rule above.  Returns the scale byte.
__device__ __forceinline__ uint32_t quantize_block_pack_norm(const uint4 (&raw)[4], const uint4 (&gv)[4], float rn,
                                                             uint32_t (&packed)[8]) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(raw);
  float v[32];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t gw[4] = {gv[q].x, gv[q].y, gv[q].z, gv[q].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[8 * q + 2 * i] = bf16_lo(w[4 * q + i]) * rn * bf16_lo(gw[i]);
      v[8 * q + 2 * i + 1] = bf16_hi(w[4 * q + i]) * rn * bf16_hi(gw[i]);
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const uint32_t s = ue8m0_from_amax(amax);
  const float inv = inv_scale_from_ue8m0(s);
#pragma unroll
  for (int i = 0; i < 8; ++i) packed[i] = e4m3x4_code(v[4 * i] * inv, v[4 * i + 1] * inv, v[4 * i + 2] * inv, v[4 * i + 3] * inv);
  return s;
}
// The same with the gains read from global memory (16-byte aligned bf16).
__device__ __forceinline__ uint32_t quantize_block_pack_norm(const uint4 (&raw)[4], const uint16_t* gamma, float rn,
                                                             uint32_t (&packed)[8]) {
  uint4 gv[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) gv[q] = __ldg(reinterpret_cast<const uint4*>(gamma) + q);
  return quantize_block_pack_norm(raw, gv, rn, packed);
}
// 1 / sqrt(mean(x^2) + eps) of a bf16 row of K elements, reduced in fp32 by
// the calling warp (every lane gets the result).
__device__ __forceinline__ float row_rnorm(const uint16_t* xr, int K, float eps, int lane) {
  float ss = 0.f;
  for (int i = lane; i < K / 8; i += 32) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(xr) + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float lo = bf16_lo(w[k]), hi = bf16_hi(w[k]);
      ss = fmaf(lo, lo, fmaf(hi, hi, ss));
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
  return rsqrtf(ss / static_cast<float>(K) + eps);
}
// Same, storing the 32 codes at `dst` (16-byte aligned).
__device__ __forceinline__ uint32_t quantize_block_regs(const uint4 (&raw)[4], uint8_t* dst) {
  uint32_t packed[8];
  const uint32_t s = quantize_block_pack(raw, packed);
  uint4* d = reinterpret_cast<uint4*>(dst);
  d[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  d[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
  return s;
}

// Same, loading the block from `src` (16-byte aligned) first.
__device__ __forceinline__ uint32_t quantize_block_bf16(const uint16_t* src, uint8_t* dst) {
  uint4 raw[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) raw[i] = __ldg(reinterpret_cast<const uint4*>(src) + i);
  return quantize_block_regs(raw, dst);
}

// ----------------------------------------------------------------------------
// Bounded waits.  Every wait gives up when the block was told to abort,
// another block reported an error, or the timeout passes; the first error is
// recorded in the status word as (status << 24) | (site << 16) | block.
// ----------------------------------------------------------------------------
struct Ctx {
  volatile int* abort_flag;
  volatile uint32_t* status;
  uint64_t timeout_ns;
};

static __device__ __noinline__ void raise_error(const Ctx& cx, uint32_t code, uint32_t site) {
  *cx.abort_flag = 1;
  const uint32_t word = (code << 24) | ((site & 0xFFu) << 16) | (blockIdx.x & 0xFFFFu);
  atomicCAS(const_cast<uint32_t*>(cx.status), 0u, word);
}

// Bounded wait on an mbarrier phase.  Gives up (returns false) when the block
// was told to abort, another block reported an error, or the timeout passes.
__device__ __forceinline__ bool wait_mbar(const Ctx& cx, uint64_t* bar, uint32_t parity, uint32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t n = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++n & 15u) == 0) {
      if (*cx.abort_flag || *cx.status != 0) { *cx.abort_flag = 1; return false; }
      if (globaltimer_ns() - t0 > cx.timeout_ns) { raise_error(cx, 5u, site); return false; }
    }
  }
  return true;
}
// The same on a barrier a CTA of the cluster arrives on (acquire at cluster scope).
__device__ __forceinline__ bool wait_mbar_cluster(const Ctx& cx, uint64_t* bar, uint32_t parity, uint32_t site) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t n = 0;
  while (!mbar_try_wait_cluster(bar, parity)) {
    if ((++n & 15u) == 0) {
      if (*cx.abort_flag || *cx.status != 0) { *cx.abort_flag = 1; return false; }
      if (globaltimer_ns() - t0 > cx.timeout_ns) { raise_error(cx, 5u, site); return false; }
    }
  }
  return true;
}
// Bounded wait used only while tearing down (no abort check, fixed limit).
__device__ __forceinline__ void drain_mbar(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
  }
}
// Bounded spin until every counter p[0..n) is >= target.  The polls are
// relaxed loads issued together (one round trip per try); an acquire fence
// follows the successful try.
__device__ __forceinline__ bool wait_counters(const Ctx& cx, const uint32_t* p, int n, uint32_t target,
                                              uint32_t site) {
  uint64_t t0 = 0;
  for (;;) {
    bool all = true;
    for (int i = 0; i < n; ++i) all &= (ld_relaxed_gpu(p + i) >= target);
    if (all) break;
    if (t0 == 0) t0 = globaltimer_ns();
    if (*cx.abort_flag || *cx.status != 0) { *cx.abort_flag = 1; return false; }
    if (globaltimer_ns() - t0 > cx.timeout_ns) { raise_error(cx, 5u, site); return false; }
    __nanosleep(20);
  }
  fence_acq_rel_gpu();
  return true;
}

// Programmatic dependent launch: wait until the kernels this grid depends on
// have completed and their memory is visible (holds the whole warp), and let
// the next kernel on the stream be scheduled as this grid's blocks leave.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// The 128 epilogue threads (warps 4-7) of a block.
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// Warp pair q (warps 4 + 2q, 5 + 2q) of the epilogue warps (barriers 2 and 3).
__device__ __forceinline__ void pair_bar(uint32_t q) { asm volatile("bar.sync %0, 64;" ::"r"(2u + q) : "memory"); }
// AND of `v` over warp pair q (a barrier among its 64 threads).
__device__ __forceinline__ bool pair_and(uint32_t q, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %2, 0;\n\t"
      "bar.red.and.pred q, %1, 64, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"(2u + q), "r"(v ? 1u : 0u)
      : "memory");
  return r != 0;
}
// AND of `v` over the 128 epilogue threads (a barrier among them): every
// epilogue thread takes the same branch after a wait, so none of them is left
// alone at a later barrier when another gave up.
__device__ __forceinline__ bool epi_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"(v ? 1u : 0u)
      : "memory");
  return r != 0;
}


}  // namespace fsops
