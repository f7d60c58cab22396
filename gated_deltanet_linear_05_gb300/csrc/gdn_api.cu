// C-ABI entry points of libgdn: host-side validation, workspace layout and launch.
// Declarations and the argument contract: include/gdn.h.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

// The library's device status word: kernels OR GDN_STATUS_* bits into it when a bounded
// wait gives up; gdn_device_status reads and clears it.  In host code the name is only a
// stand-in for the symbol: its device address is looked up per device.
__device__ unsigned int g_status_word;

constexpr int kMaxDevices = 64;
std::mutex g_status_mutex;
unsigned int *g_status_addr[kMaxDevices] = {};

// Device address of the status word on the current device (looked up on first use), or
// NULL if the lookup fails (kernels then report nowhere).
unsigned int *status_word() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_status_mutex);
  if (!g_status_addr[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_status_word) != cudaSuccess) return nullptr;
    g_status_addr[dev] = static_cast<unsigned int *>(ptr);
  }
  return g_status_addr[dev];
}

// One thread waits `polls` times on a shared-memory barrier that nothing completes and
// reports the timeout: the status path without a lost signal anywhere else.  No copy or
// tensor-core operation targets the barrier, so giving up leaves nothing in flight.
__global__ void selftest_wait_kernel(int polls, unsigned int *word) {
  __shared__ __align__(8) uint64_t bar;
  gdn::mbar_init(&bar, 1);
  gdn::mbar_fence_init();
  if (!gdn::mbar_wait_polls(&bar, 0, polls)) gdn::report_status(word, GDN_STATUS_WAIT_TIMEOUT);
}

using gdn::ChunkParams;
using gdn::DecodeParams;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

gdn_status check_shape(const gdn_shape *s, bool needs_chunk) {
  if (!s) return GDN_ERR_INVALID_ARG;
  if (s->num_seqs < 0 || s->total_tokens < 0 || s->num_k_heads <= 0 || s->num_v_heads <= 0)
    return GDN_ERR_INVALID_ARG;
  if (s->num_v_heads % s->num_k_heads != 0) return GDN_ERR_INVALID_ARG;
  if (s->dk != gdn::kD || s->dv != gdn::kD) return GDN_ERR_UNSUPPORTED;
  if (s->qkv_dtype != GDN_F32 && s->qkv_dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
  if (s->o_fp32 != 0 && s->o_fp32 != 1) return GDN_ERR_INVALID_ARG;
  if (s->algo != GDN_ALGO_AUTO && s->algo != GDN_ALGO_TWO_PASS && s->algo != GDN_ALGO_SINGLE_PASS &&
      s->algo != GDN_ALGO_TENSOR_MEMORY && s->algo != GDN_ALGO_RECURRENT &&
      s->algo != GDN_ALGO_TWO_PASS_TENSOR)
    return GDN_ERR_INVALID_ARG;
  if ((s->algo == GDN_ALGO_TENSOR_MEMORY || s->algo == GDN_ALGO_TWO_PASS_TENSOR) && needs_chunk &&
      (s->chunk != 64 || s->qkv_dtype != GDN_BF16))
    return GDN_ERR_UNSUPPORTED;
  if (needs_chunk && s->chunk != 16 && s->chunk != 32 && s->chunk != 64) return GDN_ERR_UNSUPPORTED;
  // grids are sized (sequences x v-heads x 8) in one dimension
  if ((long long)s->num_seqs * s->num_v_heads * 8 > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
  return GDN_OK;
}

// [a, a+n) and [b, b+n) overlap without being identical
bool partial_overlap(const void *a, const void *b, size_t n) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  if (x == y) return false;
  return x < y + n && y < x + n;
}

struct Common {
  const gdn_shape *s;
  const void *q, *k, *v;
  const float *g, *beta, *state_in;
  float *state_out;
  const int32_t *cu_seqlens;
  void *o;
};

gdn_status check_buffers(const Common &c, bool cu_required) {
  const gdn_shape *s = c.s;
  if (s->total_tokens > 0) {
    if (!c.q || !c.k || !c.v || !c.g || !c.beta || !c.o) return GDN_ERR_INVALID_ARG;
    if (!aligned16(c.q) || !aligned16(c.k) || !aligned16(c.v) || !aligned16(c.o) ||
        !aligned16(c.g) || !aligned16(c.beta))
      return GDN_ERR_INVALID_ARG;
  }
  if (s->num_seqs > 0) {
    if (!c.state_out || !aligned16(c.state_out)) return GDN_ERR_INVALID_ARG;
    if (c.state_in && !aligned16(c.state_in)) return GDN_ERR_INVALID_ARG;
    if (cu_required && !c.cu_seqlens) return GDN_ERR_INVALID_ARG;
  }
  if (c.cu_seqlens && (reinterpret_cast<uintptr_t>(c.cu_seqlens) & 3u)) return GDN_ERR_INVALID_ARG;
  return GDN_OK;
}

size_t state_bytes(const gdn_shape *s) {
  return (size_t)s->num_seqs * s->num_v_heads * s->dk * s->dv * sizeof(float);
}

gdn_status cuda_status(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA; }

// bf16 chunked pass: one CTA per (sequence, v-head) without workspace, or two passes
bool single_pass(const gdn_shape *s) {
  if (s->algo == GDN_ALGO_SINGLE_PASS || s->algo == GDN_ALGO_TENSOR_MEMORY) return true;
  if (s->algo == GDN_ALGO_TWO_PASS || s->algo == GDN_ALGO_TWO_PASS_TENSOR) return false;
  return (long long)s->num_seqs * s->num_v_heads >= GDN_SINGLE_PASS_MIN_HEADS;
}

size_t chunked_workspace(const gdn_shape *s) {
  if (s->qkv_dtype == GDN_F32 || s->algo == GDN_ALGO_RECURRENT || single_pass(s)) return 0;
  return gdn::chunk_workspace_bytes(s->total_tokens, s->num_seqs, s->num_v_heads, s->chunk,
                                    s->algo == GDN_ALGO_TWO_PASS_TENSOR);
}

gdn_status run_chunked(const Common &c, void *workspace, size_t workspace_bytes, void *stream,
                       float *delta = nullptr, int passes = 0,
                       const float *state_in2 = nullptr, float *state_out2 = nullptr) {
  const gdn_shape *s = c.s;
  if (s->algo == GDN_ALGO_RECURRENT) {  // the token loop
    DecodeParams d{};
    d.num_seqs = s->num_seqs;
    d.total_tokens = s->total_tokens;
    d.hk = s->num_k_heads;
    d.hv = s->num_v_heads;
    d.dtype = s->qkv_dtype;
    d.o_fp32 = s->o_fp32 != 0;
    d.q = c.q;
    d.k = c.k;
    d.v = c.v;
    d.g = c.g;
    d.beta = c.beta;
    d.state_in = c.state_in;
    d.state_out = c.state_out;
    d.cu_seqlens = c.cu_seqlens;
    d.o = c.o;
    d.delta = delta;
    return cuda_status(gdn::launch_decode(d, static_cast<cudaStream_t>(stream)));
  }
  ChunkParams p{};
  p.err = status_word();
  p.delta = delta;
  p.passes = passes;
  p.tc_pass2 = s->algo == GDN_ALGO_TWO_PASS_TENSOR;
  p.state_in2 = state_in2;
  p.state_out2 = state_out2;
  p.num_seqs = s->num_seqs;
  p.total_tokens = s->total_tokens;
  p.hk = s->num_k_heads;
  p.hv = s->num_v_heads;
  p.chunk = s->chunk;
  p.dtype = s->qkv_dtype;
  p.o_fp32 = s->o_fp32 != 0;
  p.q = c.q;
  p.k = c.k;
  p.v = c.v;
  p.g = c.g;
  p.beta = c.beta;
  p.state_in = c.state_in;
  p.state_out = c.state_out;
  p.cu_seqlens = c.cu_seqlens;
  p.o = c.o;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (s->qkv_dtype == GDN_F32) return cuda_status(gdn::launch_chunk_f32(p, st));
  if (delta) return cuda_status(gdn::launch_chunk_fused(p, st));  // the capturing schedule
  if (single_pass(s)) {
    // many heads, 64-token blocks: the tcgen05 schedule unless the mma.sync one was asked for
    const bool tc = s->algo == GDN_ALGO_TENSOR_MEMORY ||
                    (s->algo == GDN_ALGO_AUTO && s->chunk == 64);
    return cuda_status(tc ? gdn::launch_chunk_tc(p, st) : gdn::launch_chunk_fused(p, st));
  }
  const size_t need = chunked_workspace(s);
  if (need > 0 && (!workspace || workspace_bytes < need ||
                   (reinterpret_cast<uintptr_t>(workspace) & 255u)))
    return GDN_ERR_WORKSPACE;
  char *ws = static_cast<char *>(workspace);
  p.nslots = s->total_tokens / s->chunk + s->num_seqs;
  p.slot_ws = ws + 256;
  return cuda_status(gdn::launch_chunk_bf16(p, st));
}

// Sequence-split prefill: the workspace regions (each 256-byte aligned), in order:
// segment boundaries, first segment of each sequence, a zero v, scratch outputs, the
// identity states (overwritten by the maps M_s), the local states L_s, the segments'
// incoming states, and the inner chunked pass's own workspace.
struct SplitLayout {
  int max_segs;
  size_t cu_seg, seg_first, v_zero, o_scratch, ident, local, seg_in, inner, total;
  gdn_shape inner_shape;
};

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

SplitLayout split_layout(const gdn_shape *s, int seg_len) {
  SplitLayout L{};
  L.max_segs = (s->total_tokens + seg_len - 1) / seg_len + s->num_seqs;
  L.inner_shape = *s;
  L.inner_shape.num_seqs = L.max_segs;
  const size_t es = s->qkv_dtype == GDN_F32 ? 4 : 2;
  const size_t eo = (s->qkv_dtype == GDN_F32 || s->o_fp32) ? 4 : 2;
  const size_t vals = (size_t)s->total_tokens * s->num_v_heads * s->dv;
  const size_t states = (size_t)L.max_segs * s->num_v_heads * s->dk * s->dv * sizeof(float);
  size_t off = 0;
  L.cu_seg = off;    off += align256(sizeof(int32_t) * (L.max_segs + 1));
  L.seg_first = off; off += align256(sizeof(int32_t) * (s->num_seqs + 1));
  L.v_zero = off;    off += align256(vals * es);
  L.o_scratch = off; off += align256(vals * eo);
  L.ident = off;     off += align256(states);
  L.local = off;     off += align256(states);
  L.seg_in = off;    off += align256(states);
  L.inner = off;     off += align256(chunked_workspace(&L.inner_shape));
  L.total = off;
  return L;
}

gdn_status check_split(const gdn_shape *s, int32_t seg_len) {
  gdn_status st = check_shape(s, true);
  if (st != GDN_OK) return st;
  if (seg_len <= 0 || seg_len % s->chunk != 0) return GDN_ERR_INVALID_ARG;
  if (s->algo == GDN_ALGO_RECURRENT) return GDN_ERR_UNSUPPORTED;
  const long long max_segs = ((long long)s->total_tokens + seg_len - 1) / seg_len + s->num_seqs;
  if (max_segs * s->num_v_heads * 8 > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
  if ((long long)s->num_seqs * s->num_v_heads * 32 > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
  return GDN_OK;
}

}  // namespace

extern "C" {

size_t gdn_prefill_split_workspace_size(const gdn_shape *shape, int32_t segment_len) {
  if (check_split(shape, segment_len) != GDN_OK) return (size_t)-1;
  return split_layout(shape, segment_len).total;
}

gdn_status gdn_prefill_split(const gdn_shape *shape, const void *q, const void *k,
                             const void *v, const float *g, const float *beta,
                             const float *state_in, float *state_out,
                             const int32_t *cu_seqlens, void *o, int32_t segment_len,
                             void *workspace, size_t workspace_bytes, void *stream) {
  gdn_status st = check_split(shape, segment_len);
  if (st != GDN_OK) return st;
  Common c{shape, q, k, v, g, beta, state_in, state_out, cu_seqlens, o};
  if ((st = check_buffers(c, true)) != GDN_OK) return st;
  if (state_in && partial_overlap(state_in, state_out, state_bytes(shape))) return GDN_ERR_ALIAS;
  if (shape->num_seqs == 0) return GDN_OK;
  const SplitLayout L = split_layout(shape, segment_len);
  if (!workspace || workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return GDN_ERR_WORKSPACE;
  char *ws = static_cast<char *>(workspace);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  int32_t *cu_seg = reinterpret_cast<int32_t *>(ws + L.cu_seg);
  int32_t *seg_first = reinterpret_cast<int32_t *>(ws + L.seg_first);
  float *ident = reinterpret_cast<float *>(ws + L.ident);
  float *local = reinterpret_cast<float *>(ws + L.local);
  float *seg_in = reinterpret_cast<float *>(ws + L.seg_in);
  void *inner_ws = ws + L.inner;
  const size_t inner_bytes = L.total - L.inner;

  gdn::SplitPlanParams pp{};
  pp.num_seqs = shape->num_seqs;
  pp.total_tokens = shape->total_tokens;
  pp.seg_len = segment_len;
  pp.max_segs = L.max_segs;
  pp.cu_seqlens = cu_seqlens;
  pp.cu_seg = cu_seg;
  pp.seg_first = seg_first;
  if (gdn::launch_split_plan(pp, cs) != cudaSuccess) return GDN_ERR_CUDA;
  if (gdn::launch_identity(ident, (long long)L.max_segs * shape->num_v_heads, cs) != cudaSuccess)
    return GDN_ERR_CUDA;
  // On the bf16 two-pass schedule the three runs share one pass 1 (its slots depend on q,
  // k, v, g, beta only), and runs 1 and 2 are one launch of state chains (U taken as zero
  // for the maps); other schedules run in full, the map run on a zero v.
  const bool shared = shape->qkv_dtype == GDN_BF16 && !single_pass(&L.inner_shape);
  Common a{&L.inner_shape, q, k, v, g, beta, nullptr, local, cu_seg, ws + L.o_scratch};
  Common b{&L.inner_shape, q, k, ws + L.v_zero, g, beta, ident, ident, cu_seg, ws + L.o_scratch};
  Common d{&L.inner_shape, q, k, v, g, beta, seg_in, seg_in, cu_seg, o};
  const int run = shared ? 2 : 0;
  if (shared) {
    if ((st = run_chunked(a, inner_ws, inner_bytes, stream, nullptr, 1)) != GDN_OK) return st;
  } else {
    if (cudaMemsetAsync(ws + L.v_zero, 0, L.o_scratch - L.v_zero, cs) != cudaSuccess)
      return GDN_ERR_CUDA;
  }
  if (shared) {
    // 1 and 2 in one launch of state chains: every segment from a zero state (its local
    // final state L_s) and, with U = 0, from the identity (its map M_s, in place)
    if ((st = run_chunked(a, inner_ws, inner_bytes, stream, nullptr, 3, ident, ident)) != GDN_OK)
      return st;
  } else {
    // 1. every segment from a zero state: its local final state
    if ((st = run_chunked(a, inner_ws, inner_bytes, stream)) != GDN_OK) return st;
    // 2. every segment with v = 0 from the identity: its map M_s (in place over the identity)
    if ((st = run_chunked(b, inner_ws, inner_bytes, stream)) != GDN_OK) return st;
  }
  // 3. the segments' incoming states in order, and each sequence's final state
  gdn::SplitCombineParams cp{};
  cp.num_seqs = shape->num_seqs;
  cp.hv = shape->num_v_heads;
  cp.seg_first = seg_first;
  cp.state_in = state_in;
  cp.map = ident;
  cp.local = local;
  cp.seg_in = seg_in;
  cp.state_out = state_out;
  if (gdn::launch_split_combine(cp, cs) != cudaSuccess) return GDN_ERR_CUDA;
  // 4. every segment from its incoming state: the outputs (its final state, in place, is
  //    not needed again)
  return run_chunked(d, inner_ws, inner_bytes, stream, nullptr, run);
}

}  // extern "C"

extern "C" {

size_t gdn_workspace_size(const gdn_shape *s, int op) {
  if (op != GDN_OP_PREFILL && op != GDN_OP_DECODE && op != GDN_OP_VERIFY && op != GDN_OP_DECODE_BLOCK)
    return (size_t)-1;
  const bool chunked = (op == GDN_OP_PREFILL || op == GDN_OP_VERIFY);
  if (check_shape(s, chunked) != GDN_OK) return (size_t)-1;
  if (op == GDN_OP_DECODE_BLOCK) {
    size_t a, b, c;
    return gdn::decode_block_ws_parts(s->num_seqs, s->num_k_heads, s->num_v_heads, &a, &b, &c);
  }
  return chunked ? chunked_workspace(s) : 0;
}

gdn_status gdn_device_status(uint32_t *status, void *stream) {
  if (!status) return GDN_ERR_INVALID_ARG;
  unsigned int *word = status_word();
  if (!word) return GDN_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GDN_ERR_CUDA;
  unsigned int v = 0, zero = 0;
  if (cudaMemcpy(&v, word, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return GDN_ERR_CUDA;
  if (cudaMemcpy(word, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return GDN_ERR_CUDA;
  *status = v;
  return GDN_OK;
}

gdn_status gdn_selftest_wait_timeout(int32_t polls, void *stream) {
  if (polls < 1 || polls > (1 << 22)) return GDN_ERR_INVALID_ARG;
  unsigned int *word = status_word();
  if (!word) return GDN_ERR_CUDA;
  selftest_wait_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(polls, word);
  return cuda_status(cudaGetLastError());
}

const char *gdn_status_string(gdn_status status) {
  switch (status) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG: null, misaligned or inconsistent argument";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED: shape, dtype or block length not built";
    case GDN_ERR_ALIAS: return "GDN_ERR_ALIAS: two buffers overlap in a way not allowed";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA: a CUDA call or kernel launch failed";
  }
  return "unknown gdn_status";
}

gdn_status gdn_prefill_chunked(const gdn_shape *shape, const void *q, const void *k,
                               const void *v, const float *g, const float *beta,
                               const float *state_in, float *state_out,
                               const int32_t *cu_seqlens, void *o, void *workspace,
                               size_t workspace_bytes, void *stream) {
  gdn_status st = check_shape(shape, true);
  if (st != GDN_OK) return st;
  Common c{shape, q, k, v, g, beta, state_in, state_out, cu_seqlens, o};
  if ((st = check_buffers(c, true)) != GDN_OK) return st;
  if (state_in && partial_overlap(state_in, state_out, state_bytes(shape))) return GDN_ERR_ALIAS;
  if (shape->num_seqs == 0) return GDN_OK;
  return run_chunked(c, workspace, workspace_bytes, stream);
}

gdn_status gdn_verify_block(const gdn_shape *shape, const void *q, const void *k,
                            const void *v, const float *g, const float *beta,
                            const float *state_in, float *state_out,
                            const int32_t *cu_seqlens, void *o, void *workspace,
                            size_t workspace_bytes, void *stream) {
  gdn_status st = check_shape(shape, true);
  if (st != GDN_OK) return st;
  Common c{shape, q, k, v, g, beta, state_in, state_out, cu_seqlens, o};
  if ((st = check_buffers(c, true)) != GDN_OK) return st;
  if (shape->num_seqs == 0) return GDN_OK;
  if (!state_in) return GDN_ERR_INVALID_ARG;
  const size_t n = state_bytes(shape);
  const uintptr_t a = reinterpret_cast<uintptr_t>(state_in), b = reinterpret_cast<uintptr_t>(state_out);
  if (a < b + n && b < a + n) return GDN_ERR_ALIAS;
  return run_chunked(c, workspace, workspace_bytes, stream);
}

gdn_status gdn_decode_step(const gdn_shape *shape, const void *q, const void *k,
                           const void *v, const float *g, const float *beta,
                           const float *state_in, float *state_out,
                           const int32_t *cu_seqlens, void *o, void *workspace,
                           size_t workspace_bytes, void *stream) {
  (void)workspace;
  (void)workspace_bytes;
  gdn_status st = check_shape(shape, false);
  if (st != GDN_OK) return st;
  Common c{shape, q, k, v, g, beta, state_in, state_out, cu_seqlens, o};
  if ((st = check_buffers(c, false)) != GDN_OK) return st;
  if (!cu_seqlens && shape->total_tokens != shape->num_seqs) return GDN_ERR_INVALID_ARG;
  if (state_in && partial_overlap(state_in, state_out, state_bytes(shape))) return GDN_ERR_ALIAS;
  if (shape->num_seqs == 0) return GDN_OK;
  DecodeParams p{};
  p.num_seqs = shape->num_seqs;
  p.total_tokens = shape->total_tokens;
  p.hk = shape->num_k_heads;
  p.hv = shape->num_v_heads;
  p.dtype = shape->qkv_dtype;
  p.o_fp32 = shape->o_fp32 != 0;
  p.q = q;
  p.k = k;
  p.v = v;
  p.g = g;
  p.beta = beta;
  p.state_in = state_in;
  p.state_out = state_out;
  p.cu_seqlens = cu_seqlens;
  p.o = o;
  return cuda_status(gdn::launch_decode(p, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_input_prologue(const gdn_shape *shape, const void *q_raw, const void *k_raw,
                              const void *v_raw, const float *a, const float *b,
                              const float *conv_w, const float *A_log, const float *dt_bias,
                              const void *conv_state_in, void *conv_state_out,
                              const int32_t *cu_seqlens, float eps, void *q, void *k, void *v,
                              float *g, float *beta, void *stream) {
  gdn_status st = check_shape(shape, false);
  if (st != GDN_OK) return st;
  const gdn_shape *s = shape;
  if (!(eps >= 0.f)) return GDN_ERR_INVALID_ARG;  // also rejects NaN
  if (!cu_seqlens && s->total_tokens != s->num_seqs) return GDN_ERR_INVALID_ARG;
  const size_t es = s->qkv_dtype == GDN_BF16 ? 2 : 4;
  const size_t T = (size_t)s->total_tokens;
  const size_t qk_bytes = T * s->num_k_heads * s->dk * es, v_bytes = T * s->num_v_heads * s->dv * es;
  const size_t C = (size_t)(2 * s->num_k_heads * s->dk + s->num_v_heads * s->dv);
  if (T > 0) {
    const void *need[] = {q_raw, k_raw, v_raw, a, b, q, k, v, g, beta};
    for (const void *ptr : need)
      if (!ptr || !aligned16(ptr)) return GDN_ERR_INVALID_ARG;
    if (!conv_w || !aligned16(conv_w) || !A_log || !dt_bias) return GDN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(A_log) & 3u) || (reinterpret_cast<uintptr_t>(dt_bias) & 3u))
      return GDN_ERR_INVALID_ARG;
    // the outputs q, k, v must not overlap the raw inputs (other warps read rows a
    // warp may already have written)
    const void *ins[] = {q_raw, k_raw, v_raw};
    const size_t in_n[] = {qk_bytes, qk_bytes, v_bytes};
    const void *outs[] = {q, k, v};
    const size_t out_n[] = {qk_bytes, qk_bytes, v_bytes};
    for (int i = 0; i < 3; ++i)
      for (int j = 0; j < 3; ++j) {
        const uintptr_t x = reinterpret_cast<uintptr_t>(ins[i]), y = reinterpret_cast<uintptr_t>(outs[j]);
        if (x < y + out_n[j] && y < x + in_n[i]) return GDN_ERR_ALIAS;
      }
  }
  if (s->num_seqs > 0) {
    if (cu_seqlens && (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u)) return GDN_ERR_INVALID_ARG;
    if ((conv_state_in && !aligned16(conv_state_in)) || (conv_state_out && !aligned16(conv_state_out)))
      return GDN_ERR_INVALID_ARG;
    const size_t cs_bytes = (size_t)s->num_seqs * (GDN_CONV_WIDTH - 1) * C * es;
    if (conv_state_in && conv_state_out && partial_overlap(conv_state_in, conv_state_out, cs_bytes))
      return GDN_ERR_ALIAS;
  }
  if (s->num_seqs == 0) return GDN_OK;
  gdn::PrologueParams p{};
  p.num_seqs = s->num_seqs;
  p.total_tokens = s->total_tokens;
  p.hk = s->num_k_heads;
  p.hv = s->num_v_heads;
  p.dtype = s->qkv_dtype;
  p.eps = eps;
  p.q_raw = q_raw;
  p.k_raw = k_raw;
  p.v_raw = v_raw;
  p.a = a;
  p.b = b;
  p.conv_w = conv_w;
  p.A_log = A_log;
  p.dt_bias = dt_bias;
  p.conv_state_in = conv_state_in;
  p.conv_state_out = conv_state_out;
  p.cu_seqlens = cu_seqlens;
  p.q = q;
  p.k = k;
  p.v = v;
  p.g = g;
  p.beta = beta;
  return cuda_status(gdn::launch_prologue(p, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_decode_block_step(const gdn_shape *shape, const void *q_raw, const void *k_raw,
                                 const void *v_raw, const float *a, const float *b,
                                 const float *conv_w, const float *A_log, const float *dt_bias,
                                 const void *conv_state_in, void *conv_state_out, float eps_qk,
                                 const float *state_in, float *state_out, const void *z,
                                 const float *norm_w, float eps_norm, void *y, float *o,
                                 void *workspace, size_t workspace_bytes, void *stream) {
  gdn_status st = check_shape(shape, false);
  if (st != GDN_OK) return st;
  const gdn_shape *s = shape;
  if (s->total_tokens != s->num_seqs) return GDN_ERR_INVALID_ARG;  // one token per sequence
  if (!(eps_qk >= 0.f) || !(eps_norm >= 0.f)) return GDN_ERR_INVALID_ARG;
  if (s->num_seqs == 0) return GDN_OK;
  const void *need16[] = {q_raw, k_raw, v_raw, conv_w, state_out, z, norm_w, y};
  for (const void *ptr : need16)
    if (!ptr || !aligned16(ptr)) return GDN_ERR_INVALID_ARG;
  const void *need4[] = {a, b, A_log, dt_bias};
  for (const void *ptr : need4)
    if (!ptr || (reinterpret_cast<uintptr_t>(ptr) & 3u)) return GDN_ERR_INVALID_ARG;
  if ((state_in && !aligned16(state_in)) || (o && !aligned16(o)) ||
      (conv_state_in && !aligned16(conv_state_in)) || (conv_state_out && !aligned16(conv_state_out)))
    return GDN_ERR_INVALID_ARG;
  if (state_in && partial_overlap(state_in, state_out, state_bytes(s))) return GDN_ERR_ALIAS;
  const size_t es = s->qkv_dtype == GDN_BF16 ? 2 : 4;
  const size_t C = (size_t)(2 * s->num_k_heads + s->num_v_heads) * s->dk;
  if (conv_state_in && conv_state_out &&
      partial_overlap(conv_state_in, conv_state_out, (size_t)s->num_seqs * (GDN_CONV_WIDTH - 1) * C * es))
    return GDN_ERR_ALIAS;
  if (partial_overlap(y, z, (size_t)s->num_seqs * s->num_v_heads * s->dv * es)) return GDN_ERR_ALIAS;
  size_t off_cnt, off_part, off_o;
  const size_t need = gdn::decode_block_ws_parts(s->num_seqs, s->num_k_heads, s->num_v_heads, &off_cnt,
                                                 &off_part, &off_o);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return GDN_ERR_WORKSPACE;
  char *ws = static_cast<char *>(workspace);
  gdn::DecodeBlockParams p{};
  p.ws_cnt = reinterpret_cast<unsigned int *>(ws + off_cnt);
  p.ws_part = reinterpret_cast<float *>(ws + off_part);
  p.ws_o = reinterpret_cast<float *>(ws + off_o);
  p.num_seqs = s->num_seqs;
  p.hk = s->num_k_heads;
  p.hv = s->num_v_heads;
  p.dtype = s->qkv_dtype;
  p.eps_qk = eps_qk;
  p.eps_norm = eps_norm;
  p.q_raw = q_raw;
  p.k_raw = k_raw;
  p.v_raw = v_raw;
  p.a = a;
  p.b = b;
  p.conv_w = conv_w;
  p.A_log = A_log;
  p.dt_bias = dt_bias;
  p.conv_state_in = conv_state_in;
  p.conv_state_out = conv_state_out;
  p.state_in = state_in;
  p.state_out = state_out;
  p.z = z;
  p.norm_w = norm_w;
  p.y = y;
  p.o = o;
  return cuda_status(gdn::launch_decode_block(p, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_gated_rmsnorm(const gdn_shape *shape, const void *o, const void *z,
                             const float *weight, float eps, void *y, void *stream) {
  gdn_status st = check_shape(shape, false);
  if (st != GDN_OK) return st;
  const gdn_shape *s = shape;
  if (!(eps >= 0.f)) return GDN_ERR_INVALID_ARG;
  const long long rows = (long long)s->total_tokens * s->num_v_heads;
  if (rows == 0) return GDN_OK;
  if (!o || !z || !weight || !y || !aligned16(o) || !aligned16(z) || !aligned16(weight) ||
      !aligned16(y))
    return GDN_ERR_INVALID_ARG;
  const size_t es = s->qkv_dtype == GDN_BF16 ? 2 : 4;
  const size_t eo = s->o_fp32 ? 4 : es;
  const size_t ny = (size_t)rows * s->dv * es;
  const size_t no = (size_t)rows * s->dv * eo;
  const uintptr_t yo = reinterpret_cast<uintptr_t>(y), oo = reinterpret_cast<uintptr_t>(o);
  // in place only onto a buffer of the same element size, exactly
  if (yo < oo + no && oo < yo + ny && !(yo == oo && eo == es)) return GDN_ERR_ALIAS;
  if (partial_overlap(y, z, ny)) return GDN_ERR_ALIAS;
  gdn::NormParams p{};
  p.rows = rows;
  p.dtype = s->qkv_dtype;
  p.o_fp32 = s->o_fp32;
  p.eps = eps;
  p.o = o;
  p.z = z;
  p.weight = weight;
  p.y = y;
  return cuda_status(gdn::launch_gated_rmsnorm(p, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_verify_block_capture(const gdn_shape *shape, const void *q, const void *k,
                                    const void *v, const float *g, const float *beta,
                                    const float *state_in, float *state_out,
                                    const int32_t *cu_seqlens, void *o, float *delta,
                                    void *stream) {
  gdn_status st = check_shape(shape, true);
  if (st != GDN_OK) return st;
  if (shape->algo != GDN_ALGO_AUTO && shape->algo != GDN_ALGO_SINGLE_PASS &&
      shape->algo != GDN_ALGO_RECURRENT)
    return GDN_ERR_UNSUPPORTED;
  Common c{shape, q, k, v, g, beta, state_in, state_out, cu_seqlens, o};
  if ((st = check_buffers(c, true)) != GDN_OK) return st;
  if (shape->total_tokens > 0 && (!delta || !aligned16(delta))) return GDN_ERR_INVALID_ARG;
  if (shape->num_seqs == 0) return GDN_OK;
  if (!state_in) return GDN_ERR_INVALID_ARG;
  const size_t n = state_bytes(shape);
  const uintptr_t a = reinterpret_cast<uintptr_t>(state_in), b = reinterpret_cast<uintptr_t>(state_out);
  if (a < b + n && b < a + n) return GDN_ERR_ALIAS;
  return run_chunked(c, nullptr, 0, stream, delta);
}

gdn_status gdn_state_rollback(const gdn_shape *shape, const void *k, const float *g,
                              const float *delta, const float *state_in,
                              const int32_t *prefix_len, float *state_out,
                              const int32_t *cu_seqlens, void *stream) {
  gdn_status st = check_shape(shape, false);
  if (st != GDN_OK) return st;
  const gdn_shape *s = shape;
  if (s->num_seqs == 0) return GDN_OK;
  if (!prefix_len || !cu_seqlens || !state_out || !aligned16(state_out) ||
      (reinterpret_cast<uintptr_t>(prefix_len) & 3u) || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u))
    return GDN_ERR_INVALID_ARG;
  if (state_in && !aligned16(state_in)) return GDN_ERR_INVALID_ARG;
  if (s->total_tokens > 0 && (!k || !g || !delta || !aligned16(k) || !aligned16(g) || !aligned16(delta)))
    return GDN_ERR_INVALID_ARG;
  if (state_in && partial_overlap(state_in, state_out, state_bytes(s))) return GDN_ERR_ALIAS;
  gdn::RollbackParams p{};
  p.num_seqs = s->num_seqs;
  p.total_tokens = s->total_tokens;
  p.hk = s->num_k_heads;
  p.hv = s->num_v_heads;
  p.dtype = s->qkv_dtype;
  p.k = k;
  p.g = g;
  p.delta = delta;
  p.state_in = state_in;
  p.prefix_len = prefix_len;
  p.cu_seqlens = cu_seqlens;
  p.state_out = state_out;
  return cuda_status(gdn::launch_rollback(p, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_conv_state_rollback(const gdn_shape *shape, const void *q_raw, const void *k_raw,
                                   const void *v_raw, const void *conv_state_in,
                                   const int32_t *prefix_len, void *conv_state_out,
                                   const int32_t *cu_seqlens, void *stream) {
  gdn_status st = check_shape(shape, false);
  if (st != GDN_OK) return st;
  const gdn_shape *s = shape;
  if (s->num_seqs == 0) return GDN_OK;
  if (!prefix_len || !cu_seqlens || !conv_state_out || !aligned16(conv_state_out) ||
      (reinterpret_cast<uintptr_t>(prefix_len) & 3u) || (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u))
    return GDN_ERR_INVALID_ARG;
  if (conv_state_in && !aligned16(conv_state_in)) return GDN_ERR_INVALID_ARG;
  if (s->total_tokens > 0 && (!q_raw || !k_raw || !v_raw || !aligned16(q_raw) || !aligned16(k_raw) ||
                              !aligned16(v_raw)))
    return GDN_ERR_INVALID_ARG;
  const size_t es = s->qkv_dtype == GDN_BF16 ? 2 : 4;
  const size_t C = (size_t)(2 * s->num_k_heads * s->dk + s->num_v_heads * s->dv);
  if (conv_state_in &&
      partial_overlap(conv_state_in, conv_state_out, (size_t)s->num_seqs * (GDN_CONV_WIDTH - 1) * C * es))
    return GDN_ERR_ALIAS;
  gdn::PrologueParams p{};
  p.num_seqs = s->num_seqs;
  p.total_tokens = s->total_tokens;
  p.hk = s->num_k_heads;
  p.hv = s->num_v_heads;
  p.dtype = s->qkv_dtype;
  p.q_raw = q_raw;
  p.k_raw = k_raw;
  p.v_raw = v_raw;
  p.conv_state_in = conv_state_in;
  p.conv_state_out = conv_state_out;
  p.cu_seqlens = cu_seqlens;
  p.prefix_len = prefix_len;
  return cuda_status(gdn::launch_conv_state(p, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
