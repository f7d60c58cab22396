/*
 * libgdn: the gated delta-rule linear-attention layer on NVIDIA GB300 (sm_103a).
 *
 * The layer ("Qwen3.5-9B-npu" model card, section "How it works"): a per-head
 * state S [dk x dv] (S[i][j]: i indexes the key, j the value) evolves per token
 *
 *     S <- S * exp(g_t)
 *     kv = S^T k_t
 *     S <- S + k_t (x) ((v_t - kv) * beta_t)
 *     o_t = S^T q_t            (the output reads the updated state)
 *
 * Three entry points compute it:
 *   gdn_prefill_chunked  prompt blocks in the chunkwise-parallel form of the same
 *                        section (G = cumsum(g), strictly lower N, per-token deltas
 *                        D = (I + N)^-1 diag(beta)(V - diag(exp G) K S0), block
 *                        output O and carried state S_T);
 *   gdn_decode_step      the token-by-token recurrence (the 1-token matrix form of
 *                        that section: o = d q^T S + (q.k) delta, S' = d S + k delta^T);
 *   gdn_verify_block     a prompt-lookup draft check from a state snapshot (section
 *                        "New in v2", prompt lookup decoding: the state is snapshotted
 *                        before the check, so the snapshot must stay untouched).
 * Two more compute the steps of the block right around the layer:
 *   gdn_input_prologue   causal conv + SiLU, q/k L2 norm and the gates, producing the
 *                        layer's q, k, v, g, beta from the block's projections;
 *   gdn_gated_rmsnorm    the gated RMSNorm of the layer output.
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 * Pointers are DEVICE pointers, row-major and contiguous, each 16-byte aligned
 * (cu_seqlens: 4-byte aligned):
 *     q, k          [total_tokens, Hk, dk]   qkv_dtype
 *     v             [total_tokens, Hv, dv]   qkv_dtype
 *     o             [total_tokens, Hv, dv]   qkv_dtype, or float32 when shape->o_fp32
 *     g, beta       [total_tokens, Hv]       float32 (g: log-decay, used as is)
 *     state_in/out  [num_seqs, Hv, dk, dv]   float32
 *     cu_seqlens    [num_seqs + 1]           int32, cu_seqlens[0] = 0, non-decreasing,
 *                                            cu_seqlens[num_seqs] = total_tokens
 * v-head h reads q/k head h / (Hv / Hk) (grouped heads; Hv % Hk == 0).
 * Sequence n owns tokens [cu_seqlens[n], cu_seqlens[n+1]); blocks never cross a
 * sequence boundary and a partly filled block behaves as if padded with g = 0,
 * beta = 0 tokens (the page's token_valid rule), so the state after it is exactly
 * the state after the sequence's last token.  A zero-length sequence copies its
 * initial state to state_out.
 * state_in == NULL means a zero initial state.  The library applies no 1/sqrt(dk)
 * scale and no normalisation to q or k, and computes no gates: g and beta are inputs.
 *
 * Ownership and execution: the caller owns every buffer.  Calls enqueue work on
 * `stream` (a cudaStream_t; NULL = the legacy default stream) and return without
 * synchronising.  The library allocates no memory; scratch memory, where an entry point
 * needs it, is the caller's `workspace` (query its size with gdn_workspace_size).  The
 * only state it keeps is one 32-bit status word per device (gdn_device_status), whose
 * address the first chunked call on a device looks up (make that call before any stream
 * capture).
 *
 * Errors: arguments are validated on the host before anything is launched; a bad
 * argument returns its status and enqueues nothing.  A failed launch returns
 * GDN_ERR_CUDA.  The kernels' waits on shared-memory barriers are bounded: a wait that
 * gives up (a lost signal) ends the kernel normally with unspecified results and sets
 * GDN_STATUS_WAIT_TIMEOUT in the device status word, which gdn_device_status reports.
 * cu_seqlens lives on the device and is not read by the host: a malformed cu_seqlens
 * (decreasing, or past total_tokens) cannot make a kernel read or write outside the
 * buffers sized by `shape` (every range is clamped to [0, total_tokens]), but the results
 * are then unspecified.  Faults raised later on
 * the device surface at the caller's next synchronisation, as usual in CUDA.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1,  /* null pointer, bad count, misaligned pointer   */
  GDN_ERR_UNSUPPORTED = 2,  /* a shape, dtype or block length not built       */
  GDN_ERR_ALIAS = 3,        /* two buffers overlap in a way not allowed       */
  GDN_ERR_WORKSPACE = 4,    /* workspace missing or smaller than required     */
  GDN_ERR_CUDA = 5          /* a CUDA call or launch failed                   */
} gdn_status;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

typedef enum {
  GDN_OP_PREFILL = 0,
  GDN_OP_DECODE = 1,
  GDN_OP_VERIFY = 2,
  GDN_OP_DECODE_BLOCK = 3  /* gdn_decode_block_step */
} gdn_op;

/* Kernel schedule of the bf16 chunked pass (prefill and verify); f32 q/k/v have one.
 *   TWO_PASS     a parallel pass over all blocks of all heads builds the state-free
 *                operands into the workspace, then a second pass walks each head's
 *                blocks in order, spread over 8 CTAs per head.  Suits few heads.
 *   SINGLE_PASS  one CTA per (sequence, v-head) builds the operands and walks the
 *                blocks itself; no workspace.  Suits batches of >= ~1 head per SM.
 *   AUTO         with num_seqs * num_v_heads >= GDN_SINGLE_PASS_MIN_HEADS: TENSOR_MEMORY for
 *                64-token blocks of bf16 q/k/v, else SINGLE_PASS; with fewer pairs TWO_PASS
 *                (a rule of the shape alone, so that gdn_workspace_size does not depend on
 *                the device).
 *   TENSOR_MEMORY one CTA per (sequence, v-head) on the tcgen05 tensor cores: the whole
 *                state in tensor memory, every block's operands read once per head, the
 *                next block's state-free part prepared while the current one runs; no
 *                workspace.  Block length 64 and bf16 q/k/v only (else GDN_ERR_UNSUPPORTED).
 *   RECURRENT    the per-token rule itself, token by token (the token loop of
 *                gdn_decode_step): one CTA per (sequence, v-head, 32 value columns) with
 *                its state slice in registers for the whole sequence and the tokens staged
 *                16 at a time; fp32 arithmetic on CUDA cores (no product is rounded to
 *                16 bits), no workspace, any valid shape->chunk (not used).  The most
 *                accurate schedule and the slowest: the per-token reductions over the keys
 *                cost several times the chunk schedules' tensor-core work from 16 tokens
 *                up.  AUTO never picks it.
 *   TWO_PASS_TENSOR the two-pass schedule with its second pass on the tcgen05 tensor
 *                cores: the first pass writes each block's operands in the layouts of the
 *                tensor-core products (a larger workspace slot), the second runs one CTA
 *                per (sequence, v-head) with the state in tensor memory.  Block length 64
 *                and bf16 q/k/v only (else GDN_ERR_UNSUPPORTED).  AUTO does not pick it.
 * All give results within the same bounds; they are not bit-identical to each other. */
typedef enum {
  GDN_ALGO_AUTO = 0,
  GDN_ALGO_TWO_PASS = 1,
  GDN_ALGO_SINGLE_PASS = 2,
  GDN_ALGO_TENSOR_MEMORY = 3,
  GDN_ALGO_RECURRENT = 4,
  GDN_ALGO_TWO_PASS_TENSOR = 5
} gdn_algo;
#define GDN_SINGLE_PASS_MIN_HEADS 128

typedef struct {
  int32_t num_seqs;      /* N >= 0                                                  */
  int32_t total_tokens;  /* = cu_seqlens[N]; decode without cu_seqlens: = N         */
  int32_t num_k_heads;   /* Hk: heads of q and k                                    */
  int32_t num_v_heads;   /* Hv, a multiple of Hk: heads of v, g, beta, state and o  */
  int32_t dk, dv;        /* head sizes; 128 and 128 are built                       */
  int32_t chunk;         /* block length for prefill / verify: 16, 32 or 64        */
  gdn_dtype qkv_dtype;   /* dtype of q, k, v (and of o unless o_fp32): F32 or BF16  */
  int32_t o_fp32;        /* 0: o has qkv_dtype; 1: o is float32 (the unrounded       */
                         /* fp32 result; the bf16 o of the same call is exactly its  */
                         /* round-to-nearest-even rounding)                          */
  int32_t algo;          /* a gdn_algo; 0 = GDN_ALGO_AUTO                            */
} gdn_shape;

/*
 * Chunkwise-parallel prompt pass ("How it works", chunkwise form).
 * Runs every sequence from state_in (or zero) through its tokens in blocks of
 * shape->chunk, writes o for every token and the final state to state_out.
 * state_out may equal state_in exactly (in-place update); any other overlap is
 * GDN_ERR_ALIAS.  bf16 q/k/v: products on tensor cores with fp32 accumulation, the
 * state kept in fp32.  f32 q/k/v: all arithmetic in fp32 on CUDA cores.
 * workspace: at least gdn_workspace_size(shape, GDN_OP_PREFILL) bytes, 256-byte
 * aligned (may be NULL when that size is 0, as for f32 q/k/v and the bf16 single-pass
 * schedule); its contents on entry do not matter and are unspecified on return.
 */
gdn_status gdn_prefill_chunked(const gdn_shape *shape, const void *q, const void *k,
                               const void *v, const float *g, const float *beta,
                               const float *state_in, float *state_out,
                               const int32_t *cu_seqlens, void *o, void *workspace,
                               size_t workspace_bytes, void *stream);

/*
 * Token-by-token recurrence ("How it works", the per-token rule in its 1-token
 * matrix form), one pass over each head's state per token.
 * cu_seqlens == NULL: one token per sequence (total_tokens must equal num_seqs;
 * token n belongs to sequence n) -- the decode step.  Otherwise each sequence runs
 * through all its tokens in order.
 * state_out may equal state_in exactly (in-place); other overlap is GDN_ERR_ALIAS.
 * shape->chunk is ignored.  Needs no workspace (workspace may be NULL).
 */
gdn_status gdn_decode_step(const gdn_shape *shape, const void *q, const void *k,
                           const void *v, const float *g, const float *beta,
                           const float *state_in, float *state_out,
                           const int32_t *cu_seqlens, void *o, void *workspace,
                           size_t workspace_bytes, void *stream);

/*
 * Draft-verify block ("New in v2", prompt lookup decoding): the chunkwise pass over
 * each sequence's draft tokens, started from the snapshot state_in, which is left
 * unchanged.  state_in must not be NULL and must not overlap state_out
 * (GDN_ERR_ALIAS).  Writes per-token outputs o and the end-of-block state state_out.
 * Draft blocks are normally at most shape->chunk tokens (one block per sequence);
 * longer ones are processed in several blocks, as by gdn_prefill_chunked.
 * workspace: gdn_workspace_size(shape, GDN_OP_VERIFY) bytes, as for prefill.
 */
gdn_status gdn_verify_block(const gdn_shape *shape, const void *q, const void *k,
                            const void *v, const float *g, const float *beta,
                            const float *state_in, float *state_out,
                            const int32_t *cu_seqlens, void *o, void *workspace,
                            size_t workspace_bytes, void *stream);

/*
 * Draft-verify block that also captures each token's delta ("New in v2", prompt lookup
 * decoding; the deltas are the rows D of the chunkwise form in "How it works"):
 *     delta_t = beta_t * (v_t - S'^T k_t),   S' the decayed state before token t's write.
 * Same arguments and results as gdn_verify_block, plus
 *     delta  [total_tokens, Hv, dv] float32, 16-byte aligned (written for every token).
 * With the deltas, gdn_state_rollback gives the state after any accepted prefix of the
 * draft without re-feeding the accepted tokens.  Runs the single-pass schedule (bf16) or
 * the fp32 kernel, or with GDN_ALGO_RECURRENT the token loop; shape->algo must be
 * GDN_ALGO_AUTO, GDN_ALGO_SINGLE_PASS or GDN_ALGO_RECURRENT (else GDN_ERR_UNSUPPORTED).
 * Needs no workspace.
 */
gdn_status gdn_verify_block_capture(const gdn_shape *shape, const void *q, const void *k,
                                    const void *v, const float *g, const float *beta,
                                    const float *state_in, float *state_out,
                                    const int32_t *cu_seqlens, void *o, float *delta,
                                    void *stream);

/*
 * State after the accepted prefix of each sequence's verified block:
 *     S_a = exp(G_a) S_in + sum_{t<a} exp(G_a - G_t) k_t delta_t^T,
 * G_t the inclusive cumsum of g over the sequence's tokens, a = prefix_len[n] clamped to
 * [0, the sequence's length] -- the chunkwise form's end-of-block state ("How it works")
 * cut after a tokens, equal to the per-token rule run over those a tokens.
 *     k          [total_tokens, Hk, dk]   qkv_dtype (the verified block's keys)
 *     g          [total_tokens, Hv]       float32
 *     delta      [total_tokens, Hv, dv]   float32, from gdn_verify_block_capture
 *     state_in   [num_seqs, Hv, dk, dv]   float32, the snapshot the block started from
 *                                         (NULL: zero)
 *     prefix_len [num_seqs]               int32, on the device (accepted tokens)
 *     state_out  [num_seqs, Hv, dk, dv]   float32; may equal state_in exactly (in place),
 *                                         other overlap is GDN_ERR_ALIAS
 *     cu_seqlens [num_seqs + 1]           int32, the verified block's
 * shape->chunk, o_fp32 and algo are ignored.  One launch; reads and writes each state
 * once.
 */
gdn_status gdn_state_rollback(const gdn_shape *shape, const void *k, const float *g,
                              const float *delta, const float *state_in,
                              const int32_t *prefix_len, float *state_out,
                              const int32_t *cu_seqlens, void *stream);

/*
 * Conv FIFO after the accepted prefix of each sequence's draft: conv_state_out[n][j] is
 * the raw input at position a - (W-1) + j of sequence n (a = prefix_len[n], clamped to
 * the sequence's length; positions before the draft come from conv_state_in, the FIFO
 * the draft's prologue started from).  q_raw, k_raw, v_raw are the draft's raw
 * projections as given to gdn_input_prologue; conv states [num_seqs, W-1, C] in
 * qkv_dtype; conv_state_out may equal conv_state_in exactly.  One launch.
 */
gdn_status gdn_conv_state_rollback(const gdn_shape *shape, const void *q_raw, const void *k_raw,
                                   const void *v_raw, const void *conv_state_in,
                                   const int32_t *prefix_len, void *conv_state_out,
                                   const int32_t *cu_seqlens, void *stream);

/*
 * Scratch size built into gdn_prefill_chunked_noalloc (64 MiB).
 */
#define GDN_NOALLOC_SCRATCH_BYTES (64u << 20)

/*
 * The chunked prompt pass for callers that cannot allocate device memory.  The
 * paper has no counterpart to this entry point: it exists for the library's users.
 *
 * Who needs it: code that may not call cudaMalloc (or any allocator) at the point
 * where it runs the layer -- for example a host runtime that hands out only
 * pre-registered buffers, a plug-in inside another framework's memory pool, or a
 * real-time path where an allocation could block or fail.  Such a caller still
 * owns q, k, v, g, beta, the states, cu_seqlens and o, exactly as for
 * gdn_prefill_chunked; only the scratch (the `workspace` there) comes from a fixed
 * array of GDN_NOALLOC_SCRATCH_BYTES compiled into the library.  When the array is
 * reserved on a GPU depends on CUDA's module loading: with lazy loading (the default)
 * when the first call on that GPU looks up its address; with eager loading
 * (CUDA_MODULE_LOADING=EAGER) on every GPU whose context loads the library.  It stays
 * reserved until the process exits.
 *
 * Same arguments and results as gdn_prefill_chunked, without workspace.  The request
 * must fit: gdn_workspace_size(shape, GDN_OP_PREFILL) <= GDN_NOALLOC_SCRATCH_BYTES,
 * else GDN_ERR_WORKSPACE is returned and nothing is launched (f32 q/k/v need no
 * scratch and always fit).  This size check comes after the shape checks but before the
 * pointer checks: a too-large request with bad pointers reports GDN_ERR_WORKSPACE.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  All calls share the one array: two calls whose work
 * overlaps on the GPU (different streams, or different host threads) race on it and
 * give wrong results, so order them.  No part of the array has to start at zero.
 * It allocates nothing itself: no cudaMalloc, cudaFree or allocating library call.
 */
gdn_status gdn_prefill_chunked_noalloc(const gdn_shape *shape, const void *q, const void *k,
                                       const void *v, const float *g, const float *beta,
                                       const float *state_in, float *state_out,
                                       const int32_t *cu_seqlens, void *o, void *stream);

/* Width of the causal convolution built into gdn_input_prologue. */
#define GDN_CONV_WIDTH 4

/*
 * The GDN block's input prologue, the step that produces this layer's q, k, v, g and
 * beta from the block's projections: the short causal-conv FIFO that precedes the
 * recurrent state ("Qwen3.5-4B — Hexagon NPU (QHexRT) — v81" model card, introduction)
 * and the Softplus-built gates ("Qwen3.5-0.8B on Dragon Q6A NPU via QNN EP", main
 * changes).  The pages print no formulas for this step; the ones below (SiLU after the
 * conv, L2-normalised q and k, the gate forms) are the block's standard definitions.
 *
 * Channels: the raw projections, concatenated per token as x = [q_raw | k_raw | v_raw]
 * (C = 2 Hk dk + Hv dv channels, q heads first, then k heads, then v heads).  For each
 * sequence n, token t and channel c, with W = GDN_CONV_WIDTH:
 *     y_t[c] = SiLU( sum_{i<W} conv_w[c][i] * x_{t-(W-1)+i}[c] ),  SiLU(u) = u / (1 + e^-u)
 * where an input before the sequence's first token (bos) is taken from the state FIFO:
 * x_p = conv_state_in[n][p - bos + W - 1][c] (zero when conv_state_in is NULL).  Then
 *     q = y_q / sqrt(sum(y_q^2) + eps), k likewise, per (token, k-head) row of dk;
 *     v = y_v;
 *     g    = -exp(A_log[h]) * log(1 + exp(a[t][h] + dt_bias[h]))    per (token, v-head);
 *     beta = 1 / (1 + exp(-b[t][h])).
 * The outputs are exactly the inputs of gdn_prefill_chunked / gdn_decode_step /
 * gdn_verify_block (q, k, v rounded to qkv_dtype, round-to-nearest-even for bf16).
 * conv_state_out[n][j][c] = x_{eos-(W-1)+j}[c]: the FIFO advanced by the sequence's
 * tokens (for a sequence shorter than W - 1, partly the old FIFO).
 *
 * Arguments (device pointers, row-major, contiguous, 16-byte aligned; shape->chunk,
 * o_fp32 and algo are ignored):
 *     q_raw, k_raw  [total_tokens, Hk, dk]   qkv_dtype
 *     v_raw         [total_tokens, Hv, dv]   qkv_dtype
 *     a, b          [total_tokens, Hv]       float32
 *     conv_w        [C, W]                   float32 (tap W-1 multiplies the current token)
 *     A_log, dt_bias [Hv]                    float32 (4-byte alignment suffices)
 *     conv_state_in, conv_state_out [num_seqs, W - 1, C]  qkv_dtype (oldest input first);
 *                   conv_state_in may be NULL (zeros), conv_state_out may be NULL (not
 *                   written); they may be the same buffer (in-place update), any other
 *                   overlap is GDN_ERR_ALIAS
 *     cu_seqlens    [num_seqs + 1] int32, or NULL: one token per sequence
 *                   (total_tokens == num_seqs), the decode step
 *     eps           >= 0, added to the sum of squares of each q / k row (1e-6 typical)
 *     q, k, v, g, beta  outputs, shaped as the same-named inputs of gdn_prefill_chunked;
 *                   none may overlap an input (q, k, v overlapping q_raw, k_raw, v_raw is
 *                   GDN_ERR_ALIAS; other overlaps give unspecified results).
 * dk = dv = 128 are built.  Errors, streams and ownership as for the other entry points;
 * no workspace.  One launch (two with cu_seqlens and conv_state_out).
 */
gdn_status gdn_input_prologue(const gdn_shape *shape, const void *q_raw, const void *k_raw,
                              const void *v_raw, const float *a, const float *b,
                              const float *conv_w, const float *A_log, const float *dt_bias,
                              const void *conv_state_in, void *conv_state_out,
                              const int32_t *cu_seqlens, float eps, void *q, void *k, void *v,
                              float *g, float *beta, void *stream);

/*
 * The GDN block's whole one-token decode step in one launch: gdn_input_prologue (conv
 * FIFO + SiLU, q/k L2 norm, gates; "Qwen3.5-4B — Hexagon NPU (QHexRT) — v81" model card,
 * introduction; "Qwen3.5-0.8B on Dragon Q6A NPU via QNN EP", main changes), the
 * delta-rule step of gdn_decode_step ("Qwen3.5-9B-npu" model card, "How it works", the
 * 1-token matrix form) and gdn_gated_rmsnorm (the same card: the output feeds only the
 * scale-invariant norm), with q, k, v, g and beta kept on chip.  It computes what those
 * three calls compute (q, k and v rounded to qkv_dtype as the prologue stores them; the
 * norm taken on the fp32 layer output), up to the order of floating-point sums.
 * One token per sequence (total_tokens == num_seqs).
 *     q_raw, k_raw  [N, Hk, dk]   qkv_dtype     v_raw, z  [N, Hv, dv]   qkv_dtype
 *     a, b          [N, Hv]       float32       conv_w    [C, W] float32 (C = 2 Hk dk + Hv dv)
 *     A_log, dt_bias [Hv]         float32       norm_w    [dv]          float32
 *     conv_state_in/out [N, W-1, C] qkv_dtype; in may be NULL (zeros), out may be NULL
 *                   (not written); they may be the same buffer (in place)
 *     state_in/out  [N, Hv, dk, dv] float32; in may be NULL (zero), may equal out
 *     y             [N, Hv, dv]   qkv_dtype: the block's output after the gated norm
 *                   (may be z exactly; other overlap is GDN_ERR_ALIAS)
 *     o             [N, Hv, dv]   float32, the layer output before the norm, or NULL
 *     eps_qk, eps_norm >= 0 (as for gdn_input_prologue and gdn_gated_rmsnorm)
 *     workspace     gdn_workspace_size(shape, GDN_OP_DECODE_BLOCK) bytes, 256-byte aligned
 *                   (else GDN_ERR_WORKSPACE): per-call scratch through which the CTAs of
 *                   a row and of a k-head meet without waiting for one another.  It must
 *                   be zero before the first call that uses it (one cudaMemsetAsync);
 *                   every call leaves it ready for the next.  Calls sharing a workspace
 *                   must not overlap on the GPU.
 * Device pointers: the vectors 16-byte aligned, a, b, A_log, dt_bias 4-byte aligned.
 * dk = dv = 128.  One launch.  Launched, like gdn_decode_step, as a programmatic
 * dependent of the work before it on `stream`.
 */
gdn_status gdn_decode_block_step(const gdn_shape *shape, const void *q_raw, const void *k_raw,
                                 const void *v_raw, const float *a, const float *b,
                                 const float *conv_w, const float *A_log, const float *dt_bias,
                                 const void *conv_state_in, void *conv_state_out, float eps_qk,
                                 const float *state_in, float *state_out, const void *z,
                                 const float *norm_w, float eps_norm, void *y, float *o,
                                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * The GDN block's output epilogue: the gated RMSNorm of each (token, v-head) row of the
 * layer output ("Qwen3.5-4B — Hexagon NPU (QHexRT) — v81" model card, introduction;
 * "Qwen3.5-9B-npu" model card, "How it works": the output feeds only this
 * scale-invariant norm):
 *     y = o / sqrt(mean(o^2) + eps) * weight * SiLU(z),   mean over the dv values of a row,
 * one weight vector [dv] shared by every head, the norm taken in float32.
 *     o       [total_tokens, Hv, dv]  qkv_dtype, or float32 when shape->o_fp32
 *     z       [total_tokens, Hv, dv]  qkv_dtype (the block's gate projection)
 *     weight  [dv]                    float32
 *     y       [total_tokens, Hv, dv]  qkv_dtype; may be o or z exactly (in place, when the
 *                                     dtypes agree), other overlap is GDN_ERR_ALIAS
 * Device pointers, 16-byte aligned.  Only total_tokens, num_v_heads, dv, qkv_dtype and
 * o_fp32 of `shape` are read (num_k_heads must still be valid).  One launch.
 */
gdn_status gdn_gated_rmsnorm(const gdn_shape *shape, const void *o, const void *z,
                             const float *weight, float eps, void *y, void *stream);

/*
 * Sequence-split prompt pass: the results of gdn_prefill_chunked, for batches with few
 * (sequence, head) chains and long sequences.  Per block the chunkwise form ("How it
 * works") maps the state affinely, S -> M S + L with M = e^{G_C} I - (diag(e^{G_C-G}) K)^T W
 * over the keys, so each sequence is cut into segments of segment_len tokens that run as
 * independent sequences of one batch, three times over:
 *   1. from a zero state: each segment's final state L_s;
 *   2. with v = 0 from the identity state: each segment's map M_s (the product of its
 *      blocks' maps);
 *   3. (a combine, in segment order per sequence: S_in(s+1) = M_s S_in(s) + L_s, fp32)
 *   4. from its incoming state S_in(s): the outputs o.
 * state_out receives each sequence's final state from step 3.  Each step runs on the
 * chunked schedules (shape->algo as for gdn_prefill_chunked; GDN_ALGO_RECURRENT is
 * GDN_ERR_UNSUPPORTED), so the work is about three state chains per segment (with one
 * shared pass 1 on the bf16 two-pass schedule), spread over segments x heads chains
 * instead of heads.  Pays off when the plain pass leaves most of
 * the GPU idle (a handful of heads); results within the same bounds as the chunked pass,
 * not bit-identical to it.  Sizing: on the two-pass schedule a (segment, head) chain
 * takes 8 CTAs of one SM each, so P = floor(SM count / (8 * num_v_heads * num_seqs))
 * segments per sequence fill the GPU in one wave: segment_len = ceil(T / P) rounded up
 * to shape->chunk; e.g. one sequence of 65,536 tokens on 2 heads on 152 SMs: P = 9,
 * segments of 7,296 tokens.
 * Arguments as for gdn_prefill_chunked, plus segment_len (> 0, a multiple of
 * shape->chunk); state_out may equal state_in exactly.  workspace: at least
 * gdn_prefill_split_workspace_size(shape, segment_len) bytes, 256-byte aligned; it holds
 * the segment boundaries, three sets of per-segment states, a zero v and scratch outputs.
 * Six launches on the bf16 two-pass schedule (segment plan, identity states, pass 1,
 * the state chains of steps 1 and 2 together, the combine, pass 2), a few more on the
 * other schedules; all on `stream`, no synchronisation.
 */
gdn_status gdn_prefill_split(const gdn_shape *shape, const void *q, const void *k,
                             const void *v, const float *g, const float *beta,
                             const float *state_in, float *state_out,
                             const int32_t *cu_seqlens, void *o, int32_t segment_len,
                             void *workspace, size_t workspace_bytes, void *stream);
/* Workspace bytes of gdn_prefill_split; (size_t)-1 for an invalid shape or segment_len. */
size_t gdn_prefill_split_workspace_size(const gdn_shape *shape, int32_t segment_len);

/* Bits of the device status word. */
#define GDN_STATUS_WAIT_TIMEOUT 1u /* a kernel gave up a bounded wait on a barrier */

/*
 * Reads and clears the library's status word on the current device: the OR of the
 * GDN_STATUS_* bits that its kernels reported since the last read (0: every bounded wait
 * completed).  A GDN_STATUS_WAIT_TIMEOUT means that some call's results are unspecified;
 * the kernel returned normally and the context stays usable.  Synchronizes `stream`
 * before reading (do not call during stream capture).  status: host pointer.
 */
gdn_status gdn_device_status(uint32_t *status, void *stream);

/*
 * Self-test of that path: one kernel waits `polls` times (1 .. 2^22) on a shared-memory
 * barrier that nothing completes, gives up, reports GDN_STATUS_WAIT_TIMEOUT and returns.
 * No copy or tensor-core operation is left in flight.  One launch on `stream`.
 */
gdn_status gdn_selftest_wait_timeout(int32_t polls, void *stream);

/* Workspace bytes `op` (a gdn_op) needs for `shape` (0 when none); (size_t)-1 for an
 * invalid shape or op. */
size_t gdn_workspace_size(const gdn_shape *shape, int op);

/* Static, human-readable name of a status code. */
const char *gdn_status_string(gdn_status status);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
