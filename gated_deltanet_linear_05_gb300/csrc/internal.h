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
  // workspace regions of the two-pass bf16 path (see chunk_bf16.cu); "hi"/"lo" are the
  // bf16 high part and the bf16 rounding of the remainder of an fp32 value
  void *w_hi, *w_lo;  // bf16 [Hv, T, 128]: W = (I+N)^-1 diag(beta e^G) K, per token row
  float *u_ws;        // fp32 [Hv, T, 128]: U = (I+N)^-1 diag(beta) V
  void *a_hi, *a_lo;  // bf16 [Hv, T, chunk]: row t of the block's decay-masked causal Q K^T
  float *g_ws;        // fp32 [Hv, T]: in-block inclusive cumsum of g
};

constexpr int kWsRegions = 6;
// Workspace layout of the bf16 chunk path (offsets of w_hi, w_lo, u, a_hi, a_lo, g);
// returns total bytes.
size_t chunk_workspace_layout(int total_tokens, int hv, int chunk, size_t offsets[kWsRegions]);

cudaError_t launch_decode(const DecodeParams &p, cudaStream_t stream);
cudaError_t launch_chunk_bf16(const ChunkParams &p, cudaStream_t stream);
cudaError_t launch_chunk_f32(const ChunkParams &p, cudaStream_t stream);

}  // namespace gdn
