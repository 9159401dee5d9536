// mx_attention.h -- paged decode attention over an MXFP8 KV cache
// (mx_attention.cu).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fsops {

constexpr int kAttnHeadDim = 128;   // D
constexpr int kAttnChunk = 128;     // tokens per pipeline chunk (16 per consumer warp)
constexpr int kAttnMaxGroup = 8;    // query heads per KV head

struct AttnArgs {
  // K and V codes as 2-D u8 tensors [num_pages * Hkv * P, D]: one box of P
  // rows x D bytes per (page, KV head), 128-byte swizzle
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  const uint16_t* q;          // bf16 [B, Hq, D]
  const uint8_t* k_scales;    // [num_pages, Hkv, P, D / 32] UE8M0
  const uint8_t* v_scales;
  const int32_t* block_table; // [B, max_pages]
  const int32_t* seq_lens;    // [B]
  uint16_t* out;              // bf16 [B, Hq, D]
  float* part;                // [B, Hq, nsplit, 2 + D]: running max (scores in base 2), sum, unnormalised
                              // output; written for the splits that hold chunks of the sequence only
  uint32_t* status;           // first error (status << 24 | site << 16 | sequence)
  uint32_t* work;             // work items handed out so far (zero before a call; the call leaves it zero)
  int B, Hq, Hkv, P, num_pages, max_pages, nsplit;
  int grid;                   // persistent blocks, taking work items (split * B + b) * Hkv + kv head
                              // from the counter `work`
  float sm_scale;
  uint64_t timeout_ns;
  unsigned long long* trace;  // [blocks][64] %globaltimer stamps, builds with FSOPS_TRACE only
};

// Splits of each sequence's chunks (work items of chunks_per_block chunks
// at most) for B sequences, Hkv KV heads and at most max_pages pages of P
// tokens, on `sms` SMs.
int attn_splits(int B, int Hkv, int max_pages, int P, int sms, int chunks_per_block);
constexpr int kAttnChunksPerBlock = 8;
// Partial-result floats of one call.
inline size_t attn_part_floats(int B, int Hq, int nsplit) {
  return static_cast<size_t>(B) * Hq * nsplit * (2 + kAttnHeadDim);
}
// Blocks of the persistent decode kernel for `items` work items on `sms` SMs.
int attn_grid(int items, int sms);
cudaError_t launch_paged_decode(const AttnArgs& a, cudaStream_t stream);

}  // namespace fsops
