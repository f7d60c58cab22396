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
  float *delta;  // per-token deltas [T, Hv, 128] fp32, or NULL
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
  float *delta;  // per-token deltas [T, Hv, 128] fp32, or NULL (single-pass and fp32 kernels)
  // Workspace of the two-pass bf16 path (chunk_bf16.cu): one slot per (v-head, block);
  // block c of sequence n uses slot bos_n / C + n + c, which is unique and below
  // nslots = total_tokens / C + num_seqs.  A slot holds the block's state-free operands,
  // each region one bulk copy for pass 2 (chunk_bf16.cu; rows of W and U past the
  // sequence end are zero, A's are never used).  WN and U are in the fragment order pass
  // 2's chain warps read (each warp's 32 lane runs contiguous):
  //   WN  fp16, C x 128       -W, W = (I+N)^-1 diag(beta e^G) K (rows: tokens)
  //   A   fp16 [C][2C + 16 B] decay-masked causal Q K^T, padded rows (the 16x16 blocks
  //                           above the diagonal are never written nor read)
  //   U   fp16, C x 128       U = (I+N)^-1 diag(beta) V (rows: tokens), per 16-column block
  //   DEC fp32 [3][C]         G (in-block cumsum), e^G, e^(G_C - G)
  int nslots;
  char *slot_ws;      // Hv * nslots slots of slot_bytes(C) bytes, 128-byte aligned
  unsigned int *err;  // the library's device status word (GDN_STATUS_* bits), or NULL
  // Two-pass path only: which passes to run (1: pass 1, 2: pass 2, 3: the sequence
  // split's state chains -- from state_in, and with U = 0 from state_in2 -- on the slots
  // of a pass 1 run with these q, k, v, g, beta; else both passes)
  int passes;
  bool tc_pass2;  // both passes at C = 64: pass 2 on the tensor cores (chunk_tc.cu)
  const float *state_in2;
  float *state_out2;
};

// Padded row bytes of 16-bit tiles staged in shared memory: 128-element rows and
// C-element rows (16 mod 128, so that eight rows read at one column hit eight bank groups).
constexpr int kP128 = 272;
__host__ __device__ constexpr int row_c(int C) { return 2 * C + 16; }
// Slot layout offsets (bytes) for block length C.
__host__ __device__ constexpr size_t slot_a_off(int C) { return (size_t)C * 256; }
__host__ __device__ constexpr size_t slot_u_off(int C) { return slot_a_off(C) + (size_t)C * row_c(C); }
__host__ __device__ constexpr size_t slot_dec_off(int C) { return slot_u_off(C) + (size_t)C * 256; }
__host__ __device__ constexpr size_t slot_bytes(int C) {
  return (slot_dec_off(C) + (size_t)12 * C + 127) / 128 * 128;
}
// Slot layout of the tensor-memory pass 2 (block length 64, chunk_tc.cu): the chain's
// operands in the shared-memory layouts of its MMAs (tc.cuh), copied by one bulk copy:
//   Wt  W^T fp16, MN-major over tokens (wt_off)      Qt  diag(e^G) Q fp16 (t64_off)
//   K   k fp16 (t64_off)                             At  A fp16, zero above the diagonal (at_off)
//   Ut  U^T fp16 [value col][token], 144-byte rows   DEC fp32 [3][64] G, e^G, e^(G_C - G)
constexpr size_t kTsWt = 0, kTsQt = 16384, kTsK = 32768, kTsAt = 49152, kTsUt = 57344,
                 kTsDec = 75776, kTsBytes = 76544;
// Distance between slots: the tensor-memory layout's (tc, C = 64) or slot_bytes(C).
__host__ __device__ constexpr size_t slot_stride(int C, bool tc) {
  return tc && C == 64 ? kTsBytes : slot_bytes(C);
}

// The block's input prologue (block_io.cu): causal conv + SiLU over [q | k | v] raw
// channels, q/k L2 norm, gates.  conv_state_* are [num_seqs][kConvW - 1][C] in dtype.
constexpr int kConvW = 4;
struct PrologueParams {
  int num_seqs, total_tokens, hk, hv;
  gdn_dtype dtype;
  float eps;
  const void *q_raw, *k_raw, *v_raw;
  const float *a, *b, *conv_w, *A_log, *dt_bias;
  const void *conv_state_in;
  void *conv_state_out;
  const int32_t *cu_seqlens;  // NULL: one token per sequence
  void *q, *k, *v;
  float *g, *beta;
  const int32_t *prefix_len;  // conv_state_kernel only: FIFO after the first prefix_len[n]
                              // tokens of sequence n instead of after all of them
};

// State after a prefix of each sequence's block from the captured per-token deltas:
// S_a = e^{G_a} S_in + sum_{t<a} e^{G_a - G_t} k_t delta_t^T (rollback.cu).
struct RollbackParams {
  int num_seqs, total_tokens, hk, hv;
  gdn_dtype dtype;  // of k
  const void *k;
  const float *g, *delta, *state_in;
  const int32_t *prefix_len, *cu_seqlens;
  float *state_out;
};
cudaError_t launch_rollback(const RollbackParams &p, cudaStream_t stream);
cudaError_t launch_conv_state(const PrologueParams &p, cudaStream_t stream);

// Gated RMSNorm of rows of 128: y = o / sqrt(mean o^2 + eps) * w * SiLU(z).
struct NormParams {
  long long rows;
  gdn_dtype dtype;  // of z and y (and of o unless o_fp32)
  int o_fp32;
  float eps;
  const void *o, *z;
  const float *weight;
  void *y;
};

// The block's fused one-token decode step (decode_block.cu): prologue + state step +
// gated RMSNorm; one token per sequence.  Workspace: counters [N Hv + N Hk] (zero between
// calls), each quarter's sum of o^2 [N Hv 4], o [N Hv 128] fp32.
struct DecodeBlockParams {
  int num_seqs, hk, hv;
  gdn_dtype dtype;  // of the raw projections, the conv state, z and y
  float eps_qk, eps_norm;
  const void *q_raw, *k_raw, *v_raw;
  const float *a, *b, *conv_w, *A_log, *dt_bias;
  const void *conv_state_in;
  void *conv_state_out;
  const float *state_in;
  float *state_out;
  const void *z;
  const float *norm_w;
  void *y;
  float *o;  // the layer output before the norm (fp32), or NULL
  unsigned int *ws_cnt;
  float *ws_part, *ws_o;
};
// Workspace bytes of the fused decode step: counters, partial sums, o (each 256-aligned).
inline size_t decode_block_ws_parts(int n, int hk, int hv, size_t *cnt, size_t *part, size_t *o) {
  auto a = [](size_t x) { return (x + 255) / 256 * 256; };
  *cnt = 0;
  *part = a(sizeof(unsigned int) * ((size_t)n * hv + (size_t)n * hk));
  *o = *part + a(sizeof(float) * (size_t)n * hv * 4);
  return *o + a(sizeof(float) * (size_t)n * hv * 128);
}
cudaError_t launch_decode_block(const DecodeBlockParams &p, cudaStream_t stream);

cudaError_t launch_prologue(const PrologueParams &p, cudaStream_t stream);
cudaError_t launch_gated_rmsnorm(const NormParams &p, cudaStream_t stream);

// Sequence-split prefill (split.cu): segment boundaries, identity states, the combine.
struct SplitPlanParams {
  int num_seqs, total_tokens, seg_len, max_segs;
  const int32_t *cu_seqlens;
  int32_t *cu_seg;     // [max_segs + 1] segment boundaries (unused segments empty, at the end)
  int32_t *seg_first;  // [num_seqs + 1] index of each sequence's first segment; [N]: count
};
struct SplitCombineParams {
  int num_seqs, hv;
  const int32_t *seg_first;
  const float *state_in;  // [N, Hv, 128, 128] or NULL (zero)
  const float *map;       // [segments, Hv, 128, 128] M_s (row index: key)
  const float *local;     // [segments, Hv, 128, 128] L_s, the final state from zero
  float *seg_in;          // [segments, Hv, 128, 128] each segment's incoming state
  float *state_out;       // [N, Hv, 128, 128] the sequence's final state
};
cudaError_t launch_split_plan(const SplitPlanParams &p, cudaStream_t stream);
cudaError_t launch_identity(float *state, long long states, cudaStream_t stream);
cudaError_t launch_split_combine(const SplitCombineParams &p, cudaStream_t stream);

// Workspace bytes of the bf16 chunk path: a 256-byte reserved header + slots.
size_t chunk_workspace_bytes(int total_tokens, int num_seqs, int hv, int chunk, bool tc);

cudaError_t launch_decode(const DecodeParams &p, cudaStream_t stream);
cudaError_t launch_chunk_bf16(const ChunkParams &p, cudaStream_t stream);
// Pass 2 of the two-pass path on the tcgen05 tensor cores (chunk_tc.cu): one CTA per
// (sequence, v-head) over slots in the kTs* layout written by pass 1.
cudaError_t launch_tc_chain(const ChunkParams &p, cudaStream_t stream);
cudaError_t launch_chunk_fused(const ChunkParams &p, cudaStream_t stream);
cudaError_t launch_chunk_tc(const ChunkParams &p, cudaStream_t stream);
cudaError_t launch_chunk_f32(const ChunkParams &p, cudaStream_t stream);

}  // namespace gdn
