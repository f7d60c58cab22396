// The steps of the GDN block right before and right after the delta-rule layer: the
// block's short causal-conv FIFO before the recurrent state and the gated RMSNorm
// after it ("Qwen3.5-4B — Hexagon NPU (QHexRT) — v81" model card, introduction), gates
// built with Softplus ("Qwen3.5-0.8B on Dragon Q6A NPU via QNN EP", main changes), and
// the layer output feeding only the scale-invariant gated RMSNorm ("Qwen3.5-9B-npu"
// model card, "How it works", fp16 precision of the DeltaNet output).  The pages give
// no formulas for these steps; the kernels compute the formulas stated in gdn.h.  Both
// are streaming, HBM-bound steps: every byte is read once and written once.
//
// Both kernels are persistent and pipelined per warp: a warp walks units of work with a
// stride of the whole grid and keeps the inputs of its next units in flight as cp.async
// copies into its own shared-memory stages (prologue: two stages, norm: three) while it
// computes the current one from shared memory and stores the results from registers,
// so the bytes in flight do not depend on registers.
//
// Input prologue.  The raw channels are x = [q_raw | k_raw | v_raw] (2 Hk + Hv heads of
// 128); a unit is (a run of RUN tokens, one head), staged as the RUN rows plus the three
// rows before them (and, for a v head, the run's gate inputs a and b).  Lane l computes
// channels 4l .. 4l+3 of the head:
//   y_t = SiLU(w0 x_{t-3} + w1 x_{t-2} + w2 x_{t-1} + w3 x_t),
// the inputs before a sequence's first token coming from the conv state FIFO
// [N][3][C] (oldest first).  q and k rows are scaled by 1 / sqrt(sum y^2 + eps) (a
// warp reduction); v rows are stored as they are; the v heads' units also form the
// gates g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b).  When the run and
// the three rows before it lie in one sequence (nearly always), the tokens are
// independent and their row norms share interleaved butterflies; otherwise the tokens
// are walked in order and the window refilled from each new sequence's FIFO.
//
// When every sequence is one token (cu_seqlens NULL, the decode step) a unit is one
// token: its stage holds the token's three FIFO entries and its raw row, and the same
// lane writes the advanced FIFO, so the state may be updated in place.  With
// cu_seqlens a second, small kernel writes the advanced FIFO after the first has
// finished reading (stream order), which again allows in-place use.
#include "common.cuh"
#include "internal.h"

namespace gdn {

namespace {

constexpr int kIoThreads = 256;
constexpr int kIoWarps = kIoThreads / 32;
constexpr int kStages = 3;          // shared-memory stages per warp (norm)
constexpr int kProStages = 2;       // shared-memory stages per warp (prologue)
constexpr int kNormRun = 8;         // rows per unit of the norm
constexpr int kCuSmem = 256;        // cu_seqlens entries kept in shared memory

// Four consecutive elements of a row, as floats.  Global accesses are plain
// (coherent): a conv state may be overwritten in place by the thread that read it.
template <typename T>
struct Vec4;
template <>
struct Vec4<float> {
  using Raw = float4;
  static __device__ __forceinline__ Raw ld(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
  }
  static __device__ __forceinline__ void cvt(const Raw &r, float (&x)[4]) {
    x[0] = r.x; x[1] = r.y; x[2] = r.z; x[3] = r.w;
  }
  static __device__ __forceinline__ void st(float *p, const float (&x)[4]) {
    *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
  }
  static __device__ __forceinline__ Raw zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
};
template <>
struct Vec4<__nv_bfloat16> {
  using Raw = uint2;
  static __device__ __forceinline__ Raw ld(const __nv_bfloat16 *p) {
    return *reinterpret_cast<const uint2 *>(p);
  }
  static __device__ __forceinline__ void cvt(const Raw &r, float (&x)[4]) {
    x[0] = __uint_as_float(r.x << 16);
    x[1] = __uint_as_float(r.x & 0xffff0000u);
    x[2] = __uint_as_float(r.y << 16);
    x[3] = __uint_as_float(r.y & 0xffff0000u);
  }
  static __device__ __forceinline__ void st(__nv_bfloat16 *p, const float (&x)[4]) {
    *reinterpret_cast<uint2 *>(p) = make_uint2(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]));
  }
  static __device__ __forceinline__ Raw zero() { return make_uint2(0u, 0u); }
};

// This lane's four elements of a staged row (shared memory).
template <typename T>
__device__ __forceinline__ void lds4(const char *row, int lane, float (&x)[4]) {
  Vec4<T>::cvt(*reinterpret_cast<const typename Vec4<T>::Raw *>(row + lane * 4 * (int)sizeof(T)), x);
}

// cp.async group wait that is also a compiler barrier for the shared-memory reads after it
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// SiLU with the base-2 exponential and the fast division: the prologue and the norm are
// otherwise issue-bound on the exponential and the IEEE division.  Relative error a few
// 1e-7 for |u| < 20; below u = -87 the result is 0 (true |value| < 1e-35).
__device__ __forceinline__ float silu(float u) { return __fdividef(u, 1.f + decay_exp(-u)); }
// log(1 + e^u) without overflow: max(u, 0) + log1p(e^-|u|)
__device__ __forceinline__ float softplus(float u) { return fmaxf(u, 0.f) + log1pf(expf(-fabsf(u))); }

__device__ __forceinline__ int clampi(int x, int lo, int hi) { return min(max(x, lo), hi); }

// Largest n in [0, N) with cu[n] <= t (the sequence holding token t), cu clamped to [0, T].
__device__ __forceinline__ int seq_of(const int32_t *cu, int N, int T, int t) {
  int lo = 0, hi = N - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (clampi(cu[mid], 0, T) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Tokens per prologue unit: 16 bf16 rows (8 fp32) per unit when sequences are packed,
// one token when every sequence is one token.
template <typename T, bool PER_TOKEN>
struct ProRun {
  static constexpr int kRun = PER_TOKEN ? 1 : (sizeof(T) == 2 ? 16 : 8);
  static constexpr int kRows = kRun + kConvW - 1;
  static constexpr int kRowBytes = kD * (int)sizeof(T);
  static constexpr int kGateOff = kRows * kRowBytes;                  // a[kRun], b[kRun]
  static constexpr int kStage = (kGateOff + 8 * kRun + 15) / 16 * 16;
  static constexpr int kWarpBytes = kProStages * kStage;
};

template <typename T, bool PER_TOKEN>
__global__ void __launch_bounds__(kIoThreads, 2) prologue_kernel(PrologueParams p) {
  using V = Vec4<T>;
  using R = ProRun<T, PER_TOKEN>;
  constexpr int RUN = R::kRun, kH = kConvW - 1, RB = R::kRowBytes;
  constexpr int kChunks = RB / 16;  // 16-byte pieces of a row
  extern __shared__ __align__(16) char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Tt = p.total_tokens, heads_all = 2 * p.hk + p.hv, C = heads_all * kD;

  // cu_seqlens in shared memory when it is short (every unit searches it)
  int32_t *cu_s = reinterpret_cast<int32_t *>(smem);
  const bool cu_in_smem = !PER_TOKEN && p.num_seqs + 1 <= kCuSmem;
  if (cu_in_smem)
    for (int i = threadIdx.x; i <= p.num_seqs; i += kIoThreads) cu_s[i] = p.cu_seqlens[i];
  __syncthreads();
  const int32_t *cu = cu_in_smem ? cu_s : p.cu_seqlens;
  char *wsm = smem + (PER_TOKEN ? 0 : kCuSmem * 4) + warp * R::kWarpBytes;

  const long long units = (long long)((Tt + RUN - 1) / RUN) * heads_all;
  const long long nw = (long long)gridDim.x * kIoWarps;
  const long long gw = (long long)blockIdx.x * kIoWarps + warp;
  const T *cs_in = static_cast<const T *>(p.conv_state_in);
  T *cs_out = static_cast<T *>(p.conv_state_out);

  // rows of head `head` in the raw input and in the output
  auto head_rows = [&](int head, const T *&src, T *&dst, int &nh, int &hidx) {
    if (head < p.hk) {
      src = static_cast<const T *>(p.q_raw); dst = static_cast<T *>(p.q); nh = p.hk; hidx = head;
    } else if (head < 2 * p.hk) {
      src = static_cast<const T *>(p.k_raw); dst = static_cast<T *>(p.k); nh = p.hk;
      hidx = head - p.hk;
    } else {
      src = static_cast<const T *>(p.v_raw); dst = static_cast<T *>(p.v); nh = p.hv;
      hidx = head - 2 * p.hk;
    }
  };

  // Stage of unit u: rows t0 - 3 .. t0 + RUN - 1 of its head (one token per sequence:
  // the token's three FIFO entries, then its row) and, for a v head, the run's a and b.
  // Rows outside [0, T) are zero-filled.
  auto issue = [&](long long u, int stage) {
    if (u < units) {
      const int head = (int)(u % heads_all);
      const int t0 = (int)(u / heads_all) * RUN;
      const T *src;
      T *dst;
      int nh, hidx;
      head_rows(head, src, dst, nh, hidx);
      char *st = wsm + stage * R::kStage;
      for (int i = lane; i < R::kRows * kChunks; i += 32) {
        const int r = i / kChunks, c16 = i - r * kChunks;
        const int pr = t0 - kH + r;
        const char *g = reinterpret_cast<const char *>(src);
        int bytes = 0;
        if (PER_TOKEN && r < kH) {
          if (cs_in) {
            g = reinterpret_cast<const char *>(cs_in + ((size_t)t0 * kH + r) * C + head * kD) + c16 * 16;
            bytes = 16;
          }
        } else if (pr >= 0 && pr < Tt) {
          g = reinterpret_cast<const char *>(src + ((size_t)pr * nh + hidx) * kD) + c16 * 16;
          bytes = 16;
        }
        cp_async16(st + r * RB + c16 * 16, g, bytes);
      }
      if (head >= 2 * p.hk && lane < 2 * RUN) {  // lanes [0, RUN): a, [RUN, 2 RUN): b
        const int t = t0 + lane % RUN;
        const float *ab = lane < RUN ? p.a : p.b;
        const bool ok = t < Tt;
        cp_async4(st + R::kGateOff + lane * 4, ok ? ab + (size_t)t * p.hv + (head - 2 * p.hk) : ab,
                  ok ? 4 : 0);
      }
    }
    cp_async_commit();
  };

  // this lane's conv weights of unit u's head, w[c][i]: tap i of channel 4 lane + c
  auto weights = [&](long long u, float (&w)[4][kConvW]) {
    const int head = (int)(u % heads_all);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float4 wv = __ldg(reinterpret_cast<const float4 *>(p.conv_w) + head * kD + lane * 4 + c);
      w[c][0] = wv.x; w[c][1] = wv.y; w[c][2] = wv.z; w[c][3] = wv.w;
    }
  };

  auto compute = [&](long long u, int stage, const float (&w)[4][kConvW]) {
    const int head = (int)(u % heads_all);
    const int t0 = (int)(u / heads_all) * RUN;
    const T *src;
    T *dst;
    int nh, hidx;
    head_rows(head, src, dst, nh, hidx);
    const bool normed = head < 2 * p.hk;
    const char *st = wsm + stage * R::kStage;
    const int ch = head * kD + lane * 4;  // first channel of this lane
    auto row = [&](int t) { return ((size_t)t * nh + hidx) * kD + lane * 4; };

    auto conv = [&](const float (&x0)[4], const float (&x1)[4], const float (&x2)[4],
                    const float (&x3)[4], float (&y)[4]) {
      float ss = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float acc = w[c][3] * x3[c];
        acc = fmaf(w[c][2], x2[c], acc);
        acc = fmaf(w[c][1], x1[c], acc);
        acc = fmaf(w[c][0], x0[c], acc);
        y[c] = silu(acc);
        ss = fmaf(y[c], y[c], ss);
      }
      return ss;
    };

    if (PER_TOKEN) {  // the window is the token's FIFO; write the advanced FIFO
      float x[4][4], y[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) lds4<T>(st + r * RB, lane, x[r]);
      float ss = conv(x[0], x[1], x[2], x[3], y);
      if (normed) {
        ss = warp_sum(ss);
        const float sc = rsqrtf(ss + p.eps);  // the same rounding on every path
#pragma unroll
        for (int c = 0; c < 4; ++c) y[c] *= sc;
      }
      V::st(dst + row(t0), y);
      if (cs_out) {
        T *s = cs_out + (size_t)t0 * kH * C + ch;
        V::st(s, x[1]);
        V::st(s + C, x[2]);
        V::st(s + 2 * (size_t)C, x[3]);
      }
    } else {
      int n = seq_of(cu, p.num_seqs, Tt, t0);
      int bos = min(clampi(cu[n], 0, Tt), t0);
      int eos = clampi(cu[n + 1], 0, Tt);
      if (bos <= t0 - kH && eos >= min(t0 + RUN, Tt)) {
        // the run and the three rows before it lie inside one sequence: the tokens are
        // independent; groups of 8 share one interleaved butterfly for their row norms
#pragma unroll
        for (int j0 = 0; j0 < RUN; j0 += 8) {
          float xs[8 + kH][4], y[8][4], ss[8];
#pragma unroll
          for (int r = 0; r < 8 + kH; ++r) lds4<T>(st + (j0 + r) * RB, lane, xs[r]);
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) ss[jj] = conv(xs[jj], xs[jj + 1], xs[jj + 2], xs[jj + 3], y[jj]);
          if (normed) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) ss[jj] += __shfl_xor_sync(0xffffffffu, ss[jj], o);
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              const float sc = rsqrtf(ss[jj] + p.eps);
#pragma unroll
              for (int c = 0; c < 4; ++c) y[jj][c] *= sc;
            }
          }
#pragma unroll
          for (int jj = 0; jj < 8; ++jj)
            if (t0 + j0 + jj < Tt) V::st(dst + row(t0 + j0 + jj), y[jj]);
        }
      } else {
        // a sequence starts inside some token's window: walk the tokens in order and
        // refill the window from the FIFO of each sequence that starts here.  Input p_
        // of sequence n_ (first token bos_): a staged row, or FIFO entry p_ - bos_ + 3.
        auto fetch = [&](int p_, int n_, int bos_, float (&x)[4]) {
          if (p_ >= bos_) {
            lds4<T>(st + (p_ - t0 + kH) * RB, lane, x);
          } else if (cs_in) {
            V::cvt(V::ld(cs_in + ((size_t)n_ * kH + (p_ - bos_ + kH)) * C + ch), x);
          } else {
            x[0] = x[1] = x[2] = x[3] = 0.f;
          }
        };
        float win[kH][4];  // x_{t-3}, x_{t-2}, x_{t-1}
#pragma unroll
        for (int i = 0; i < kH; ++i) fetch(t0 - kH + i, n, bos, win[i]);
        for (int j = 0; j < RUN; ++j) {
          const int t = t0 + j;
          if (t >= Tt) break;
          if (j > 0 && t >= eos) {  // first token of a later sequence
            while (n + 1 < p.num_seqs && t >= eos) {
              ++n;
              eos = clampi(cu[n + 1], 0, Tt);
            }
            bos = min(clampi(cu[n], 0, Tt), t);
#pragma unroll
            for (int i = 0; i < kH; ++i) fetch(t - kH + i, n, bos, win[i]);
          }
          float x[4], y[4];
          lds4<T>(st + (j + kH) * RB, lane, x);
          float ss = conv(win[0], win[1], win[2], x, y);
          if (normed) {
            ss = warp_sum(ss);
            const float sc = rsqrtf(ss + p.eps);
#pragma unroll
            for (int c = 0; c < 4; ++c) y[c] *= sc;
          }
          V::st(dst + row(t), y);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            win[0][c] = win[1][c];
            win[1][c] = win[2][c];
            win[2][c] = x[c];
          }
        }
      }
    }

    if (!normed && lane < RUN && t0 + lane < Tt) {  // gates of this v head
      const int h = head - 2 * p.hk;
      const size_t gi = (size_t)(t0 + lane) * p.hv + h;
      const float av = *reinterpret_cast<const float *>(st + R::kGateOff + lane * 4);
      const float bv = *reinterpret_cast<const float *>(st + R::kGateOff + (RUN + lane) * 4);
      const float A = expf(__ldg(p.A_log + h));
      p.g[gi] = -A * softplus(av + __ldg(p.dt_bias + h));
      p.beta[gi] = 1.f / (1.f + expf(-bv));
    }
  };

  // two stages: the next unit's copies fly while the current one is computed
  issue(gw, 0);
  int stage = 0;
  for (long long u = gw; u < units; u += nw) {
    issue(u + nw, stage ^ 1);
    float w[4][kConvW];
    weights(u, w);
    cp_wait<1>();
    __syncwarp();
    compute(u, stage, w);
    __syncwarp();  // every lane is done with this stage before it is refilled
    stage ^= 1;
  }
  cp_wait<0>();
}

// FIFO after the call for packed sequences: entry j of sequence n is the raw input
// eos - 3 + j (a raw row, or the old FIFO's entry when the sequence is shorter than 3);
// with prefix_len, eos is the end of the sequence's first prefix_len[n] tokens.
// One warp per (sequence, head); every lane reads its three entries before writing.
template <typename T>
__global__ void __launch_bounds__(kIoThreads) conv_state_kernel(PrologueParams p) {
  using V = Vec4<T>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int heads = 2 * p.hk + p.hv;
  const long long unit = (long long)blockIdx.x * kIoWarps + warp;
  if (unit >= (long long)p.num_seqs * heads) return;
  const int n = (int)(unit / heads), head = (int)(unit - (long long)n * heads);
  const int C = heads * kD, ch = head * kD + lane * 4;
  const int Tt = p.total_tokens;
  const int bos = clampi(p.cu_seqlens[n], 0, Tt);
  int eos = clampi(p.cu_seqlens[n + 1], bos, Tt);
  if (p.prefix_len) eos = bos + clampi(p.prefix_len[n], 0, eos - bos);  // accepted prefix
  const T *src;
  int hh, hidx;
  if (head < p.hk) {
    src = static_cast<const T *>(p.q_raw); hh = p.hk; hidx = head;
  } else if (head < 2 * p.hk) {
    src = static_cast<const T *>(p.k_raw); hh = p.hk; hidx = head - p.hk;
  } else {
    src = static_cast<const T *>(p.v_raw); hh = p.hv; hidx = head - 2 * p.hk;
  }
  const T *cs_in = static_cast<const T *>(p.conv_state_in);
  typename V::Raw e[kConvW - 1];
#pragma unroll
  for (int j = 0; j < kConvW - 1; ++j) {
    const int q = eos - (kConvW - 1) + j;
    if (q >= bos)
      e[j] = V::ld(src + ((size_t)q * hh + hidx) * kD + lane * 4);
    else if (cs_in)
      e[j] = V::ld(cs_in + ((size_t)n * (kConvW - 1) + (q - bos + kConvW - 1)) * C + ch);
    else
      e[j] = V::zero();
  }
  T *s = static_cast<T *>(p.conv_state_out) + (size_t)n * (kConvW - 1) * C + ch;
#pragma unroll
  for (int j = 0; j < kConvW - 1; ++j)
    *reinterpret_cast<typename V::Raw *>(s + (size_t)j * C) = e[j];
}

// Gated RMSNorm: a unit is kNormRun consecutive rows of 128 (o and z staged as two
// contiguous pieces); lane l holds elements 4l .. 4l+3 of a row.
template <typename T, typename TOI>
__global__ void __launch_bounds__(kIoThreads, 2) gated_rmsnorm_kernel(NormParams p) {
  constexpr int OB = kD * (int)sizeof(TOI), ZB = kD * (int)sizeof(T);
  constexpr int kStage = kNormRun * (OB + ZB);
  extern __shared__ __align__(16) char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  char *wsm = smem + warp * kStages * kStage;
  const long long units = (p.rows + kNormRun - 1) / kNormRun;
  const long long nw = (long long)gridDim.x * kIoWarps;
  const long long gw = (long long)blockIdx.x * kIoWarps + warp;
  const char *o = static_cast<const char *>(p.o);
  const char *z = static_cast<const char *>(p.z);
  T *y = static_cast<T *>(p.y);
  const float4 wv = __ldg(reinterpret_cast<const float4 *>(p.weight) + lane);
  const float w[4] = {wv.x, wv.y, wv.z, wv.w};

  auto issue = [&](long long u, int stage) {
    if (u < units) {
      const long long r0 = u * kNormRun;
      const int nr = (int)min((long long)kNormRun, p.rows - r0);
      char *so = wsm + stage * kStage, *sz = so + kNormRun * OB;
      for (int off = lane * 16; off < nr * OB; off += 512)
        cp_async16(so + off, o + r0 * OB + off, 16);
      for (int off = lane * 16; off < nr * ZB; off += 512)
        cp_async16(sz + off, z + r0 * ZB + off, 16);
    }
    cp_async_commit();
  };

  auto compute = [&](long long u, int stage) {
    const long long r0 = u * kNormRun;
    const char *so = wsm + stage * kStage, *sz = so + kNormRun * OB;
    // the rows' sums of squares, reduced by one interleaved butterfly
    float ss[kNormRun];
#pragma unroll
    for (int j = 0; j < kNormRun; ++j) {
      float x[4];
      lds4<TOI>(so + j * OB, lane, x);
      ss[j] = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) ss[j] = fmaf(x[c], x[c], ss[j]);
    }
#pragma unroll
    for (int o_ = 16; o_ > 0; o_ >>= 1)
#pragma unroll
      for (int j = 0; j < kNormRun; ++j) ss[j] += __shfl_xor_sync(0xffffffffu, ss[j], o_);
#pragma unroll
    for (int j = 0; j < kNormRun; ++j) {
      if (r0 + j >= p.rows) break;
      float x[4], zz[4], out[4];
      lds4<TOI>(so + j * OB, lane, x);
      lds4<T>(sz + j * ZB, lane, zz);
      const float sc = 1.f / sqrtf(ss[j] * (1.f / kD) + p.eps);
#pragma unroll
      for (int c = 0; c < 4; ++c) out[c] = x[c] * sc * w[c] * silu(zz[c]);
      Vec4<T>::st(y + (size_t)(r0 + j) * kD + lane * 4, out);
    }
  };

  issue(gw, 0);
  issue(gw + nw, 1);
  int stage = 0;
  for (long long u = gw; u < units; u += nw) {
    issue(u + 2 * nw, stage == 0 ? 2 : stage - 1);
    cp_wait<kStages - 1>();
    __syncwarp();
    compute(u, stage);
    __syncwarp();
    stage = stage == kStages - 1 ? 0 : stage + 1;
  }
  cp_wait<0>();
}

template <typename K>
cudaError_t launch_persistent(K kernel, size_t smem, long long units, const void *params,
                              cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0, per_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kIoThreads, smem)) !=
      cudaSuccess)
    return e;
  const long long want = (units + kIoWarps - 1) / kIoWarps;
  const long long most = (long long)sms * (per_sm > 0 ? per_sm : 1);
  const unsigned blocks = (unsigned)(want < most ? want : most);
  void *args[] = {const_cast<void *>(params)};
  return cudaLaunchKernel(reinterpret_cast<const void *>(kernel), dim3(blocks), dim3(kIoThreads),
                          args, smem, stream);
}

}  // namespace

cudaError_t launch_prologue(const PrologueParams &p, cudaStream_t stream) {
  if (p.total_tokens == 0 && (p.cu_seqlens == nullptr || p.num_seqs == 0)) return cudaSuccess;
  const int heads = 2 * p.hk + p.hv;
  if (p.total_tokens > 0) {
    cudaError_t e;
    const bool per_token = p.cu_seqlens == nullptr;
#define GDN_PRO(T, PT)                                                                        \
    {                                                                                         \
      using R = ProRun<T, PT>;                                                                \
      const long long units = (long long)((p.total_tokens + R::kRun - 1) / R::kRun) * heads;  \
      const size_t smem = (PT ? 0 : kCuSmem * 4) + (size_t)kIoWarps * R::kWarpBytes;          \
      e = launch_persistent(prologue_kernel<T, PT>, smem, units, &p, stream);                 \
    }
    if (p.dtype == GDN_BF16 && !per_token) GDN_PRO(__nv_bfloat16, false)
    else if (p.dtype == GDN_BF16) GDN_PRO(__nv_bfloat16, true)
    else if (!per_token) GDN_PRO(float, false)
    else GDN_PRO(float, true)
#undef GDN_PRO
    if (e != cudaSuccess) return e;
  }
  if (p.cu_seqlens && p.conv_state_out && p.num_seqs > 0) return launch_conv_state(p, stream);
  return cudaSuccess;
}

cudaError_t launch_conv_state(const PrologueParams &p, cudaStream_t stream) {
  const long long units = (long long)p.num_seqs * (2 * p.hk + p.hv);
  if (units == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((units + kIoWarps - 1) / kIoWarps);
  if (p.dtype == GDN_BF16)
    conv_state_kernel<__nv_bfloat16><<<blocks, kIoThreads, 0, stream>>>(p);
  else
    conv_state_kernel<float><<<blocks, kIoThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_gated_rmsnorm(const NormParams &p, cudaStream_t stream) {
  if (p.rows == 0) return cudaSuccess;
  const long long units = (p.rows + kNormRun - 1) / kNormRun;
  const size_t s16 = (size_t)kIoWarps * kStages * kNormRun * kD * (2 + 2);
  const size_t s32 = (size_t)kIoWarps * kStages * kNormRun * kD * (4 + 2);
  const size_t s3232 = (size_t)kIoWarps * kStages * kNormRun * kD * (4 + 4);
  if (p.dtype == GDN_BF16 && !p.o_fp32)
    return launch_persistent(gated_rmsnorm_kernel<__nv_bfloat16, __nv_bfloat16>, s16, units, &p, stream);
  if (p.dtype == GDN_BF16)
    return launch_persistent(gated_rmsnorm_kernel<__nv_bfloat16, float>, s32, units, &p, stream);
  return launch_persistent(gated_rmsnorm_kernel<float, float>, s3232, units, &p, stream);
}

}  // namespace gdn
