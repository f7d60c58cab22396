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
// in shared memory by cp.async), so the whole batch's state streams in one wave.  Each
// CTA forms the conv + SiLU + L2 norm of its token's 128 q and 128 k channels (the
// k-head's, shared by its v-heads; two adjacent channels per thread) and the conv + SiLU
// of its 32 v channels, rounded to
// the storage dtype as the standalone prologue stores them, so the fused step computes
// what the three separate launches compute.  The CTAs of one k-head's v-heads (4 per
// v-head) form a thread-block cluster:
//   - the norm's sum of o^2 over the 128 values of a row is the sum of the four quarters'
//     partial sums, exchanged through distributed shared memory;
//   - the cluster barrier that publishes them also orders every CTA's reads of the q/k
//     FIFO entries before their update, so the FIFO may be updated in place.
#include "common.cuh"
#include "internal.h"

namespace gdn {

namespace {

constexpr int kDBThreads = 64;
constexpr int kDBCols = 32;  // value columns per CTA

template <typename T>
__device__ __forceinline__ float ld_elem(const void *p, size_t i) {
  return Elem<T>::load(static_cast<const T *>(p) + i);
}
// two consecutive elements (an even element index: one 32-bit or 64-bit access)
template <typename T>
__device__ __forceinline__ void ld_pair(const void *p, size_t i, float (&x)[2]) {
  if constexpr (sizeof(T) == 2) {
    const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162 *>(static_cast<const T *>(p) + i);
    x[0] = __low2float(v);
    x[1] = __high2float(v);
  } else {
    const float2 v = *reinterpret_cast<const float2 *>(static_cast<const T *>(p) + i);
    x[0] = v.x;
    x[1] = v.y;
  }
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

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
// store a float into the same variable of the shared memory of cluster CTA `rank`
__device__ __forceinline__ void st_cluster(float *local, uint32_t rank, float x) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;\n" ::"r"(remote), "f"(x) : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

template <typename T>
__global__ void __launch_bounds__(kDBThreads, 12) decode_block_kernel(DecodeBlockParams p) {
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
  // the k-head's q/k FIFO entries are advanced by one CTA of the cluster
  const bool qk_writer = (h % ratio) == 0 && quarter == 0;

  __shared__ __align__(16) float4 s_S[64][kDBCols / 4];  // rows 64-127 of the slice
  __shared__ float s_q[kD], s_k[kD], s_v[kDBCols];
  __shared__ float s_red[2][2][kDBCols];
  __shared__ float s_ss[2][2];       // [warp][q, k] partial sums of squares
  __shared__ float s_norm[4];        // each quarter's sum of o^2 (written by the quarters)
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
  auto conv2 = [&](const void *raw, size_t ri, size_t ch, float (&f)[3][2], float (&x)[2],
                   float (&y)[2]) {
    const float4 w0 = *reinterpret_cast<const float4 *>(p.conv_w + 4 * ch);
    const float4 w1 = *reinterpret_cast<const float4 *>(p.conv_w + 4 * ch + 4);
    ld_pair<T>(raw, ri, x);
#pragma unroll
    for (int i = 0; i < 3; ++i) {
      if (p.conv_state_in)
        ld_pair<T>(p.conv_state_in, fin + i * C + ch, f[i]);
      else
        f[i][0] = f[i][1] = 0.f;
    }
    float a0 = w0.w * x[0], a1 = w1.w * x[1];
    a0 = fmaf(w0.z, f[2][0], a0);
    a1 = fmaf(w1.z, f[2][1], a1);
    a0 = fmaf(w0.y, f[1][0], a0);
    a1 = fmaf(w1.y, f[1][1], a1);
    a0 = fmaf(w0.x, f[0][0], a0);
    a1 = fmaf(w1.x, f[0][1], a1);
    y[0] = silu_f(a0);
    y[1] = silu_f(a1);
  };
  const size_t qri = ((size_t)n * p.hk + kh) * kD + 2 * tid;
  const size_t vri = ((size_t)n * p.hv + h) * kD + quarter * kDBCols + 2 * tid;
  float fq[3][2], fk[3][2], xq[2], xk[2], yq[2], yk[2];  // FIFO entries kept for the update
  conv2(p.q_raw, qri, qc0 + 2 * tid, fq, xq, yq);
  conv2(p.k_raw, qri, kc0 + 2 * tid, fk, xk, yk);
  float ssq = fmaf(yq[1], yq[1], yq[0] * yq[0]), ssk = fmaf(yk[1], yk[1], yk[0] * yk[0]);
  float fv[3][2] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}}, xv[2] = {0.f, 0.f};
  if (tid < kDBCols / 2) {
    float yv[2];
    conv2(p.v_raw, vri, vc0 + 2 * tid, fv, xv, yv);
    s_v[2 * tid] = to_storage<T>(yv[0]);
    s_v[2 * tid + 1] = to_storage<T>(yv[1]);
  }
  ssq = warp_sum(ssq);
  ssk = warp_sum(ssk);
  if (lane == 0) {
    s_ss[warp][0] = ssq;
    s_ss[warp][1] = ssk;
  }
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
  // this quarter's sum of o^2 (warp 0, lanes 0-7 hold the 32 columns) to the v-head's
  // four quarters (cluster ranks 4r .. 4r + 3)
  oss += __shfl_xor_sync(0xffffffffu, oss, 1);
  oss += __shfl_xor_sync(0xffffffffu, oss, 2);
  oss += __shfl_xor_sync(0xffffffffu, oss, 4);
  if (warp == 0 && lane < 4) st_cluster(&s_norm[quarter], (cluster_rank() & ~3u) + lane, oss);
  // every CTA of the cluster has read its FIFO entries and published its sum
  cluster_sync_all();

  // ---- gated RMSNorm of the row, stored in the storage dtype
  if (warp == 0 && rsub == 0) {
    const float sc = 1.f / sqrtf((s_norm[0] + s_norm[1] + s_norm[2] + s_norm[3]) * (1.f / kD) + p.eps_norm);
    const size_t row = ((size_t)n * p.hv + h) * kD + col0;
    T *y = static_cast<T *>(p.y);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float zz = ld_elem<T>(p.z, row + e);
      Elem<T>::store(y + row + e, o[e] * sc * __ldg(p.norm_w + col0 + e) * silu_f(zz));
      if (p.o) p.o[row + e] = o[e];
    }
  }
  // ---- the advanced FIFO: the entries shift by one and the current input enters last
  //      (past the barrier, every CTA that reads the k-head's q/k entries has read them)
  if (p.conv_state_out) {
    T *fo = static_cast<T *>(p.conv_state_out) + fin;
    auto adv = [&](size_t ch, const float (&f)[3][2], const float (&x)[2]) {
      st_pair<T>(fo + ch, f[1]);
      st_pair<T>(fo + C + ch, f[2]);
      st_pair<T>(fo + 2 * C + ch, x);
    };
    if (qk_writer) {
      adv(qc0 + 2 * tid, fq, xq);
      adv(kc0 + 2 * tid, fk, xk);
    }
    if (tid < kDBCols / 2) adv(vc0 + 2 * tid, fv, xv);
  }
  // ---- S' = d S + k delta^T, written straight from the update
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
}

template <typename T>
cudaError_t launch_t(const DecodeBlockParams &p, cudaStream_t stream) {
  const unsigned units = (unsigned)((long long)p.num_seqs * p.hv * 4);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(units);
  cfg.blockDim = dim3(kDBThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;  // one k-head's v-heads x 4 quarters
  attr[0].val.clusterDim.x = 4 * (p.hv / p.hk);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, decode_block_kernel<T>, p);
}

}  // namespace

cudaError_t launch_decode_block(const DecodeBlockParams &p, cudaStream_t stream) {
  if ((long long)p.num_seqs * p.hv == 0) return cudaSuccess;
  return p.dtype == GDN_BF16 ? launch_t<__nv_bfloat16>(p, stream) : launch_t<float>(p, stream);
}

}  // namespace gdn
