// Internal launch interface between the C-ABI layer (gdn_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

struct DecodeParams {
  int num_seqs, total_tokens, hk, hv;
  gdn_dtype dtype;
  int o_fp32;  // o is float32 regardless of dtype
  const void *q, *k, *v;
  const float *g, *beta, *state_in;
  float *state_out;
  const int32_t *cu_seqlens;  // NULL: one token per sequence
  void *o;
};

struct ChunkParams {
  int num_seqs, total_tokens, hk, hv, chunk;
  gdn_dtype dtype;
  int o_fp32;  // o is float32 regardless of dtype
  const void *q, *k, *v;
  const float *g, *beta, *state_in;
  float *state_out;
  const int32_t *cu_seqlens;
  void *o;
  // Workspace of the two-pass bf16 path (see chunk_bf16.cu): one slot per (v-head,
  // block); block c of sequence n uses slot bos_n / C + n + c, which is unique and
  // below nslots = total_tokens / C + num_seqs.  A slot holds, for the C rows of the
  // block (rows past the sequence end are zero), in the shared-memory layout the
  // pass-2 kernel uses:
  //   W  bf16 [C][128] (swizzled)   W = (I+N)^-1 diag(beta e^G) K
  //   Q  bf16 [C][128] (swizzled)   K  bf16 [C][128] (swizzled)
  //   Ah, Al bf16 [C][C] (swizzled) decay-masked causal Q K^T, hi and lo parts
  //   U  fp32 [128][C+4]            U^T, U = (I+N)^-1 diag(beta) V
  //   G  fp32 [C]                   in-block inclusive cumsum of g
  int nslots;
  char *slot_ws;      // Hv * nslots slots of slot_bytes(C) bytes, 128-byte aligned
  int *err;           // device status word: nonzero if a kernel wait timed out
};

// Bytes of one workspace slot for block length C.
__host__ __device__ constexpr size_t slot_head_bytes(int C) {
  return (size_t)3 * 256 * C + (size_t)4 * C * C;
}
__host__ __device__ constexpr size_t slot_u_bytes(int C) { return (size_t)128 * (C + 4) * 4; }
__host__ __device__ constexpr size_t slot_bytes(int C) {
  return (slot_head_bytes(C) + slot_u_bytes(C) + (size_t)4 * C + 127) / 128 * 128;
}

// Workspace bytes of the bf16 chunk path: a 256-byte header (status word) + slots.
size_t chunk_workspace_bytes(int total_tokens, int num_seqs, int hv, int chunk);

cudaError_t launch_decode(const DecodeParams &p, cudaStream_t stream);
cudaError_t launch_chunk_bf16(const ChunkParams &p, cudaStream_t stream);
cudaError_t launch_chunk_fused(const ChunkParams &p, cudaStream_t stream);
cudaError_t launch_chunk_f32(const ChunkParams &p, cudaStream_t stream);

}  // namespace gdn
