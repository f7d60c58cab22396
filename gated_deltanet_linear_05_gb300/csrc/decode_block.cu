// The GDN block's whole one-token decode step in one launch: the input prologue (short
// causal-conv FIFO + SiLU, q/k L2 norm, gates; "Qwen3.5-4B — Hexagon NPU (QHexRT) — v81"
// model card, introduction, and "Qwen3.5-0.8B on Dragon Q6A NPU via QNN EP", main
// changes), the delta-rule step in its 1-token matrix form ("Qwen3.5-9B-npu" model card,
// "How it works")
//     d = exp(g);  u = S^T k,  w = S^T q;  delta = beta (v - d u)
//     o = d w + (q.k) delta;   S' = d S + k delta^T
// and the gated RMSNorm of o ("Qwen3.5-9B-npu", "How it works": the output feeds only this
// scale-invariant norm).  q, k, v, g and beta never leave the SM.
//
// One CTA of 64 threads owns a quarter of one (sequence, v-head) state, S[:, 32c .. +32],
// laid out as in the one-token decode kernel (rows 0-63 in registers, rows 64-127 staged
// in shared memory by cp.async; 72 registers, 14 CTAs per SM), so a batch of up to
// 2128 / 4 sequence-heads streams its state in one wave.  Each CTA forms the conv + SiLU
// + L2 norm of its token's 128 q and 128 k channels (the k-head's, shared by its v-heads;
// two adjacent channels per thread) and the conv + SiLU of its 32 v channels, rounded to
// the storage dtype as the standalone prologue stores them, so the fused step computes
// what the three separate launches compute.  The CTAs of a row (a v-head's four quarters)
// and of a k-head (its v-heads' quarters) meet through a small workspace, without waiting
// for one another:
//   - each quarter writes its 32 values of o and its sum of o^2, then counts in on the
//     v-head's counter; the last of the four applies the gated norm to the whole row;
//   - each CTA counts in on the k-head's counter after it has read the k-head's q/k FIFO
//     entries; the last one advances them, so the FIFO may be updated in place.
// The last CTA of a counter resets it to zero for the next call.
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace gdn {

namespace {

constexpr int kDBThreads = 64;
constexpr int kDBCols = 32;  // value columns per CTA

// two consecutive elements kept as loaded (one register for bf16): the FIFO entries that
// move one place down are stored back bit for bit
template <typename T>
using RawPair = typename std::conditional<sizeof(T) == 2, __nv_bfloat162, float2>::type;
template <typename T>
__device__ __forceinline__ RawPair<T> ld_raw(const void *p, size_t i) {
  return *reinterpret_cast<const RawPair<T> *>(static_cast<const T *>(p) + i);
}
template <typename T>
__device__ __forceinline__ float raw_lo(RawPair<T> v) {
  if constexpr (sizeof(T) == 2) return __low2float(v); else return v.x;
}
template <typename T>
__device__ __forceinline__ float raw_hi(RawPair<T> v) {
  if constexpr (sizeof(T) == 2) return __high2float(v); else return v.y;
}
template <typename T>
__device__ __forceinline__ void st_raw(T *p, RawPair<T> v) {
  *reinterpret_cast<RawPair<T> *>(p) = v;
}
template <typename T>
__device__ __forceinline__ void st_pair(T *p, const float (&x)[2]) {
  if constexpr (sizeof(T) == 2)
    *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(x[0], x[1]);
  else
    *reinterpret_cast<float2 *>(p) = make_float2(x[0], x[1]);
}
// x rounded to the storage dtype (what a store and a reload give)
template <typename T>
__device__ __forceinline__ float to_storage(float x) {
  T r;
  Elem<T>::store(&r, x);
  return Elem<T>::load(&r);
}
// SiLU and softplus as the standalone prologue and norm compute them
__device__ __forceinline__ float silu_f(float u) { return __fdividef(u, 1.f + decay_exp(-u)); }
__device__ __forceinline__ float softplus_f(float u) { return fmaxf(u, 0.f) + log1pf(expf(-fabsf(u))); }

template <typename T>
__global__ void __launch_bounds__(kDBThreads, 14) decode_block_kernel(DecodeBlockParams p) {
  const int quarter = blockIdx.x & 3;
  const int nh = blockIdx.x >> 2;
  const int n = nh / p.hv;
  const int h = nh - n * p.hv;
  const int ratio = p.hv / p.hk;
  const int kh = h / ratio;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rsub = lane >> 3;  // row within the warp's group of 4
  const int cg = lane & 7;     // column group of 4
  const int col0 = quarter * kDBCols + cg * 4;
  const size_t C = (size_t)(2 * p.hk + p.hv) * kD;  // conv channels [q | k | v]
  const size_t qc0 = (size_t)kh * kD, kc0 = (size_t)(p.hk + kh) * kD;
  const size_t vc0 = (size_t)(2 * p.hk + h) * kD + quarter * kDBCols;

  __shared__ __align__(16) float4 s_S[64][kDBCols / 4];  // rows 64-127 of the slice
  __shared__ float s_q[kD], s_k[kD], s_v[kDBCols];
  __shared__ float s_red[2][2][kDBCols];
  __shared__ float s_ss[2][2];       // [warp][q, k] partial sums of squares
  __shared__ int s_last[2];          // this CTA is the last of its v-head / of its k-head
  __shared__ float s_gate[2];        // d = e^g, beta

  // the previous step (a programmatic primary) has completed and its writes are visible
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

  const size_t sbase = ((size_t)n * p.hv + h) * kD * kD + quarter * kDBCols;
  if (p.state_in) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = tid + kDBThreads * j, r = e >> 3, g4 = e & 7;
      cp_async16(&s_S[r][g4], p.state_in + sbase + (size_t)(64 + r) * kD + 4 * g4, 16);
    }
    cp_async_commit();
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = tid + kDBThreads * j;
      s_S[e >> 3][e & 7] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  float4 S[8];  // rows s * 8 + warp * 4 + rsub, s = 0..7
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int i = s * 8 + warp * 4 + rsub;
    S[s] = p.state_in
               ? *reinterpret_cast<const float4 *>(p.state_in + sbase + (size_t)i * kD + 4 * cg)
               : make_float4(0.f, 0.f, 0.f, 0.f);
  }

  // ---- prologue: conv (tap 3 on the current token) + SiLU of this thread's channels:
  //      the q and k channel pairs 2tid, 2tid + 1 and, for tid < 16, the v channel pair
  //      2tid, 2tid + 1 of this quarter (pairs: one 32-bit load per FIFO entry)
  const size_t fin = (size_t)n * 3 * C;  // this sequence's FIFO, oldest entry first
  auto conv2 = [&](const void *raw, size_t ri, size_t ch, RawPair<T> (&f)[3], RawPair<T> &x,
                   float (&y)[2]) {
    const float4 w0 = *reinterpret_cast<const float4 *>(p.conv_w + 4 * ch);
    const float4 w1 = *reinterpret_cast<const float4 *>(p.conv_w + 4 * ch + 4);
    x = ld_raw<T>(raw, ri);
#pragma unroll
    for (int i = 0; i < 3; ++i)
      f[i] = p.conv_state_in ? ld_raw<T>(p.conv_state_in, fin + i * C + ch) : RawPair<T>{};
    float a0 = w0.w * raw_lo<T>(x), a1 = w1.w * raw_hi<T>(x);
    a0 = fmaf(w0.z, raw_lo<T>(f[2]), a0);
    a1 = fmaf(w1.z, raw_hi<T>(f[2]), a1);
    a0 = fmaf(w0.y, raw_lo<T>(f[1]), a0);
    a1 = fmaf(w1.y, raw_hi<T>(f[1]), a1);
    a0 = fmaf(w0.x, raw_lo<T>(f[0]), a0);
    a1 = fmaf(w1.x, raw_hi<T>(f[0]), a1);
    y[0] = silu_f(a0);
    y[1] = silu_f(a1);
  };
  T *fo = static_cast<T *>(p.conv_state_out) + fin;
  // the FIFO entries of channels ch, ch + 1 move one place down; the token enters last
  auto adv = [&](size_t ch, const RawPair<T> (&f)[3], RawPair<T> x) {
    st_raw<T>(fo + ch, f[1]);
    st_raw<T>(fo + C + ch, f[2]);
    st_raw<T>(fo + 2 * C + ch, x);
  };
  const size_t qri = ((size_t)n * p.hk + kh) * kD + 2 * tid;
  const size_t vri = ((size_t)n * p.hv + h) * kD + quarter * kDBCols + 2 * tid;
  RawPair<T> fq[3], fk[3], xq, xk;  // the k-head's FIFO entries, kept for the update
  float yq[2], yk[2];
  conv2(p.q_raw, qri, qc0 + 2 * tid, fq, xq, yq);
  conv2(p.k_raw, qri, kc0 + 2 * tid, fk, xk, yk);
  float ssq = fmaf(yq[1], yq[1], yq[0] * yq[0]), ssk = fmaf(yk[1], yk[1], yk[0] * yk[0]);
  if (tid < kDBCols / 2) {
    RawPair<T> fv[3], xv;
    float yv[2];
    conv2(p.v_raw, vri, vc0 + 2 * tid, fv, xv, yv);
    s_v[2 * tid] = to_storage<T>(yv[0]);
    s_v[2 * tid + 1] = to_storage<T>(yv[1]);
    if (p.conv_state_out) adv(vc0 + 2 * tid, fv, xv);  // read by this CTA only, just now
  }
  ssq = warp_sum(ssq);
  ssk = warp_sum(ssk);
  if (lane == 0) {
    s_ss[warp][0] = ssq;
    s_ss[warp][1] = ssk;
  }
  // the gated norm's z and weight for this thread's two columns, loaded now (only the row's
  // last quarter uses them, at the very end)
  const RawPair<T> zr = ld_raw<T>(p.z, ((size_t)n * p.hv + h) * kD + 2 * tid);
  const float2 nw = __ldg(reinterpret_cast<const float2 *>(p.norm_w + 2 * tid));
  if (tid == 0) {
    const size_t gi = (size_t)n * p.hv + h;
    const float g = -expf(__ldg(p.A_log + h)) * softplus_f(p.a[gi] + __ldg(p.dt_bias + h));
    s_gate[0] = expf(g);
    s_gate[1] = 1.f / (1.f + expf(-p.b[gi]));
  }
  __syncthreads();
  {
    const float scq = rsqrtf(s_ss[0][0] + s_ss[1][0] + p.eps_qk);
    const float sck = rsqrtf(s_ss[0][1] + s_ss[1][1] + p.eps_qk);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      s_q[2 * tid + e] = to_storage<T>(yq[e] * scq);
      s_k[2 * tid + e] = to_storage<T>(yk[e] * sck);
    }
  }
  if (p.state_in) cp_async_wait<0>();
  __syncthreads();

  // ---- the state step (as the one-token decode kernel)
  const float d = s_gate[0], b = s_gate[1];
  float qk = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) qk += s_q[lane * 4 + e] * s_k[lane * 4 + e];
  qk = warp_sum(qk);
  float u[4] = {0.f, 0.f, 0.f, 0.f}, w[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int s = 0; s < 16; ++s) {
    const int i = s * 8 + warp * 4 + rsub;
    const float4 x = s < 8 ? S[s & 7] : s_S[i - 64][cg];
    const float ki = s_k[i], qi = s_q[i];
    u[0] += x.x * ki; u[1] += x.y * ki; u[2] += x.z * ki; u[3] += x.w * ki;
    w[0] += x.x * qi; w[1] += x.y * qi; w[2] += x.z * qi; w[3] += x.w * qi;
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    u[e] += __shfl_xor_sync(0xffffffffu, u[e], 8);
    u[e] += __shfl_xor_sync(0xffffffffu, u[e], 16);
    w[e] += __shfl_xor_sync(0xffffffffu, w[e], 8);
    w[e] += __shfl_xor_sync(0xffffffffu, w[e], 16);
  }
  if (rsub == 0) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      s_red[0][warp][cg * 4 + e] = u[e];
      s_red[1][warp][cg * 4 + e] = w[e];
    }
  }
  __syncthreads();
  float delta[4], o[4], oss = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int c = cg * 4 + e;
    const float uu = s_red[0][0][c] + s_red[0][1][c];
    const float ww = s_red[1][0][c] + s_red[1][1][c];
    delta[e] = b * (s_v[c] - d * uu);
    o[e] = d * ww + qk * delta[e];
    oss = fmaf(o[e], o[e], oss);
  }
  // ---- this quarter's o and sum of o^2 to the workspace (warp 0, lanes 0-7 hold the 32
  //      columns); then count in
  oss += __shfl_xor_sync(0xffffffffu, oss, 1);
  oss += __shfl_xor_sync(0xffffffffu, oss, 2);
  oss += __shfl_xor_sync(0xffffffffu, oss, 4);
  const size_t rowh = (size_t)n * p.hv + h;
  // ---- S' = d S + k delta^T for this warp's rows, written straight from the update
  auto store_rows = [&]() {
#pragma unroll
    for (int s = 0; s < 16; ++s) {
      const int i = s * 8 + warp * 4 + rsub;
      float4 x = s < 8 ? S[s & 7] : s_S[i - 64][cg];
      const float ki = s_k[i];
      x.x = d * x.x + ki * delta[0];
      x.y = d * x.y + ki * delta[1];
      x.z = d * x.z + ki * delta[2];
      x.w = d * x.w + ki * delta[3];
      *reinterpret_cast<float4 *>(p.state_out + sbase + (size_t)i * kD + 4 * cg) = x;
    }
  };
  if (warp == 1) store_rows();  // warp 1's rows go out while warp 0 counts in
  if (warp == 0) {
    // this quarter's o and sum of o^2 to the workspace (lanes 0-7 hold the 32 columns)
    if (rsub == 0) {
      const float4 ov = make_float4(o[0], o[1], o[2], o[3]);
      *reinterpret_cast<float4 *>(p.ws_o + rowh * kD + col0) = ov;
      if (p.o) *reinterpret_cast<float4 *>(p.o + rowh * kD + col0) = ov;
      if (lane == 0) p.ws_part[rowh * 4 + quarter] = oss;
    }
    // warp 0 wrote o, the sum and the v FIFO entries, and every FIFO read of the CTA was
    // done before the prologue's barrier: after this warp's barrier and one fence (its
    // writes visible on the GPU), count in
    __syncwarp();
    if (lane == 0) {
      __threadfence();
      unsigned int *cv = p.ws_cnt + rowh, *ck = p.ws_cnt + (size_t)p.num_seqs * p.hv + (size_t)n * p.hk + kh;
      const unsigned int gv = atomicAdd(cv, 1u), gk = atomicAdd(ck, 1u);
      s_last[0] = gv == 3u;
      s_last[1] = gk == 4u * (unsigned int)ratio - 1u;
      if (gv == 3u) *cv = 0u;  // every quarter has counted in: ready for the next call
      if (gk == 4u * (unsigned int)ratio - 1u) *ck = 0u;
    }
  }
  __syncthreads();
  // ---- the last CTA of the k-head advances its q/k FIFO entries (every CTA that reads them
  //      has read them before counting in)
  if (s_last[1] && p.conv_state_out) {
    adv(qc0 + 2 * tid, fq, xq);
    adv(kc0 + 2 * tid, fk, xk);
  }
  // ---- the last quarter of the v-head: the gated RMSNorm of the whole row, two values per
  //      thread, stored in the storage dtype
  if (s_last[0]) {
    __threadfence();
    const float tot = __ldcg(p.ws_part + rowh * 4) + __ldcg(p.ws_part + rowh * 4 + 1) +
                      __ldcg(p.ws_part + rowh * 4 + 2) + __ldcg(p.ws_part + rowh * 4 + 3);
    const float sc = 1.f / sqrtf(tot * (1.f / kD) + p.eps_norm);
    const float2 ov = __ldcg(reinterpret_cast<const float2 *>(p.ws_o + rowh * kD + 2 * tid));
    float yy[2];
    yy[0] = ov.x * sc * nw.x * silu_f(raw_lo<T>(zr));
    yy[1] = ov.y * sc * nw.y * silu_f(raw_hi<T>(zr));
    st_pair<T>(static_cast<T *>(p.y) + rowh * kD + 2 * tid, yy);
  }
  if (warp == 0) store_rows();
}

template <typename T>
cudaError_t launch_t(const DecodeBlockParams &p, cudaStream_t stream) {
  const unsigned units = (unsigned)((long long)p.num_seqs * p.hv * 4);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(units);
  cfg.blockDim = dim3(kDBThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_block_kernel<T>, p);
}

}  // namespace

cudaError_t launch_decode_block(const DecodeBlockParams &p, cudaStream_t stream) {
  if ((long long)p.num_seqs * p.hv == 0) return cudaSuccess;
  return p.dtype == GDN_BF16 ? launch_t<__nv_bfloat16>(p, stream) : launch_t<float>(p, stream);
}

}  // namespace gdn
