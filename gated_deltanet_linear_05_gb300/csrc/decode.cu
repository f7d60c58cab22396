// Token-by-token gated delta rule (decode step), "Qwen3.5-9B-npu" model card,
// section "How it works": the 1-token matrix form
//     d = exp(g);  u = S^T k,  w = S^T q  (one pass over S);  delta = beta (v - d u)
//     o = d w + (q.k) delta;   S' = d S + k delta^T
// which equals the four-line per-token rule (decay, read, write, output from the
// updated state).
//
// Token loop (decode_kernel, any number of tokens per sequence): one CTA of 128 threads
// owns a quarter of one head's state, S[0:128, 32c:32c+32] (value columns are
// independent: every reduction runs over the key index only).  Each thread keeps 8 rows
// x 4 columns of S in registers for the whole sequence, so the state is read from HBM
// once and written once, with 128-bit accesses.  The sequence's tokens are staged in
// shared memory 16 at a time by cp.async (the first tile issued together with the state
// loads); per token the column sums k^T S and q^T S are formed in one pass, reduced
// across the 4 rows a warp covers by shuffles and across the 4 warps through shared
// memory, with one barrier per token.  It optionally writes each token's delta (the
// capture of the draft-verify accept step).
#include "common.cuh"
#include "internal.h"

namespace gdn {

namespace {

constexpr int kDecThreads = 128;
constexpr int kDecCols = 32;  // value columns per CTA

constexpr int kDecTile = 16;  // tokens staged per tile

template <typename T, typename TO>
__global__ void __launch_bounds__(kDecThreads, 8) decode_kernel(DecodeParams p) {
  const int quarter = blockIdx.x & 3;
  const int nh = blockIdx.x >> 2;
  const int n = nh / p.hv;
  const int h = nh - n * p.hv;
  const int kh = h / (p.hv / p.hk);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rsub = lane >> 3;  // row within the warp's group of 4
  const int cg = lane & 7;     // column group of 4
  const int col0 = quarter * kDecCols + cg * 4;

  int bos, eos;
  if (p.cu_seqlens) {
    seq_range(p.cu_seqlens, n, p.total_tokens, bos, eos);
  } else {
    bos = n;
    eos = n + 1;
  }

  // a tile of tokens: q, k rows and this CTA's v columns as stored, gates
  __shared__ __align__(16) T s_q[kDecTile][kD], s_k[kDecTile][kD];
  __shared__ __align__(16) T s_v[kDecTile][kDecCols];
  __shared__ float s_g[kDecTile], s_b[kDecTile];
  __shared__ float s_red[2][2][4][kDecCols];  // [token parity][u, w][warp][column]
  const T *q = static_cast<const T *>(p.q);
  const T *k = static_cast<const T *>(p.k);
  const T *v = static_cast<const T *>(p.v);
  TO *o = static_cast<TO *>(p.o);

  // tokens t0 .. t0 + cnt - 1 (cnt >= 1) by cp.async; rows past cnt are zero-filled
  auto load_tile = [&](int t0, int cnt) {
    constexpr int EG = 16 / (int)sizeof(T), KG = kD / EG, VG = kDecCols / EG;
    for (int e = tid; e < kDecTile * KG; e += kDecThreads) {
      const int r = e / KG, gq = e - r * KG;
      const bool ok = r < cnt;
      const size_t tok = (size_t)t0 + (ok ? r : 0);
      cp_async16(&s_q[r][gq * EG], q + (tok * p.hk + kh) * kD + gq * EG, ok ? 16 : 0);
      cp_async16(&s_k[r][gq * EG], k + (tok * p.hk + kh) * kD + gq * EG, ok ? 16 : 0);
    }
    for (int e = tid; e < kDecTile * VG; e += kDecThreads) {
      const int r = e / VG, gq = e - r * VG;
      const bool ok = r < cnt;
      const size_t tok = (size_t)t0 + (ok ? r : 0);
      cp_async16(&s_v[r][gq * EG], v + (tok * p.hv + h) * kD + quarter * kDecCols + gq * EG,
                 ok ? 16 : 0);
    }
    if (tid < kDecTile) {
      const bool ok = tid < cnt;
      const size_t gi = ((size_t)t0 + (ok ? tid : 0)) * p.hv + h;
      cp_async4(&s_g[tid], p.g + gi, ok ? 4 : 0);
      cp_async4(&s_b[tid], p.beta + gi, ok ? 4 : 0);
    }
    cp_async_commit();
  };

  // the first tile's copies and the state's loads go out together
  if (eos > bos) load_tile(bos, min(kDecTile, eos - bos));
  const size_t sbase = ((size_t)n * p.hv + h) * kD * kD;
  float4 S[8];
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int i = s * 16 + warp * 4 + rsub;
    S[s] = p.state_in
               ? *reinterpret_cast<const float4 *>(p.state_in + sbase + (size_t)i * kD + col0)
               : make_float4(0.f, 0.f, 0.f, 0.f);
  }

  int par = 0;
  for (int t0 = bos; t0 < eos; t0 += kDecTile) {
    const int cnt = min(kDecTile, eos - t0);
    cp_async_wait<0>();
    __syncthreads();
    for (int r = 0; r < cnt; ++r, par ^= 1) {
      const size_t t = (size_t)t0 + r;
      // q.k: every warp forms it (4 products per lane, then a butterfly)
      float qk = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        qk += Elem<T>::load(&s_q[r][lane * 4 + e]) * Elem<T>::load(&s_k[r][lane * 4 + e]);
      qk = warp_sum(qk);
      const float d = expf(s_g[r]), b = s_b[r];

      // partial column sums of S^T k and S^T q over this thread's 8 rows
      float u[4] = {0.f, 0.f, 0.f, 0.f}, w[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const int i = s * 16 + warp * 4 + rsub;
        const float ki = Elem<T>::load(&s_k[r][i]), qi = Elem<T>::load(&s_q[r][i]);
        u[0] += S[s].x * ki; u[1] += S[s].y * ki; u[2] += S[s].z * ki; u[3] += S[s].w * ki;
        w[0] += S[s].x * qi; w[1] += S[s].y * qi; w[2] += S[s].z * qi; w[3] += S[s].w * qi;
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
          s_red[par][0][warp][cg * 4 + e] = u[e];
          s_red[par][1][warp][cg * 4 + e] = w[e];
        }
      }
      // one barrier per token: the partial sums alternate between two buffers, and a
      // buffer is rewritten only after every thread has passed the next token's barrier
      __syncthreads();

      float delta[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = cg * 4 + e;
        const float uu = s_red[par][0][0][c] + s_red[par][0][1][c] + s_red[par][0][2][c] +
                         s_red[par][0][3][c];
        const float ww = s_red[par][1][0][c] + s_red[par][1][1][c] + s_red[par][1][2][c] +
                         s_red[par][1][3][c];
        delta[e] = b * (Elem<T>::load(&s_v[r][c]) - d * uu);
        if (warp == 0 && rsub == 0) {
          Elem<TO>::store(o + (t * p.hv + h) * kD + col0 + e, d * ww + qk * delta[e]);
          if (p.delta) p.delta[(t * p.hv + h) * kD + col0 + e] = delta[e];
        }
      }
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const float ki = Elem<T>::load(&s_k[r][s * 16 + warp * 4 + rsub]);
        S[s].x = d * S[s].x + ki * delta[0];
        S[s].y = d * S[s].y + ki * delta[1];
        S[s].z = d * S[s].z + ki * delta[2];
        S[s].w = d * S[s].w + ki * delta[3];
      }
    }
    if (t0 + kDecTile < eos) {
      __syncthreads();  // every thread is done with this tile
      load_tile(t0 + kDecTile, min(kDecTile, eos - t0 - kDecTile));
    }
  }

#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int i = s * 16 + warp * 4 + rsub;
    *reinterpret_cast<float4 *>(p.state_out + sbase + (size_t)i * kD + col0) = S[s];
  }
}

// One token per sequence: the whole batch's state is read in a single wave.  Holding a
// 32-column slice (16 KB) in registers caps residency at 8 slices per SM, so a batch of
// 512 heads (2048 slices) ran in 1.7 waves with a tail.  Here a slice takes 64 threads:
// rows 0-63 of the slice stay in registers (8 float4 per thread) and rows 64-127 are
// staged in 8 KB of shared memory by cp.async, so 14 slices fit on an SM (2128 on 152
// SMs).  Each slice is read once and written once, as in the token loop above.
// Launched as a programmatic dependent: the next step's CTAs are scheduled while this
// one drains and wait (griddepcontrol.wait) before touching memory.
constexpr int kDec1Threads = 64;

template <typename T, typename TO>
__global__ void __launch_bounds__(kDec1Threads, 14) decode1_kernel(DecodeParams p) {
  const int quarter = blockIdx.x & 3;
  const int nh = blockIdx.x >> 2;
  const int n = nh / p.hv;
  const int h = nh - n * p.hv;
  const int kh = h / (p.hv / p.hk);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rsub = lane >> 3;  // row within the warp's group of 4
  const int cg = lane & 7;     // column group of 4
  const int col0 = quarter * kDecCols + cg * 4;

  __shared__ __align__(16) float4 s_S[64][kDecCols / 4];  // rows 64-127 of the slice
  __shared__ float s_q[kD], s_k[kD], s_v[kDecCols];
  __shared__ float s_red[2][2][kDecCols];

  // the previous step (a programmatic primary) has completed and its writes are visible
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

  const size_t sbase = ((size_t)n * p.hv + h) * kD * kD + quarter * kDecCols;
  if (p.state_in) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = tid + kDec1Threads * j, r = e >> 3, g4 = e & 7;
      cp_async16(&s_S[r][g4], p.state_in + sbase + (size_t)(64 + r) * kD + 4 * g4, 16);
    }
    cp_async_commit();
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = tid + kDec1Threads * j;
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
  const T *q = static_cast<const T *>(p.q);
  const T *k = static_cast<const T *>(p.k);
  const T *v = static_cast<const T *>(p.v);
  const size_t t = n;  // token n is sequence n
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    s_q[tid + 64 * e] = Elem<T>::load(q + (t * p.hk + kh) * kD + tid + 64 * e);
    s_k[tid + 64 * e] = Elem<T>::load(k + (t * p.hk + kh) * kD + tid + 64 * e);
  }
  if (tid < kDecCols) s_v[tid] = Elem<T>::load(v + (t * p.hv + h) * kD + quarter * kDecCols + tid);
  const float d = expf(p.g[t * p.hv + h]);
  const float b = p.beta[t * p.hv + h];
  if (p.state_in) cp_async_wait<0>();
  __syncthreads();

  float qk = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) qk += s_q[lane * 4 + e] * s_k[lane * 4 + e];
  qk = warp_sum(qk);

  // partial column sums of S^T k and S^T q over this thread's 16 rows
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

  float delta[4];
  TO *o = static_cast<TO *>(p.o);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int c = cg * 4 + e;
    const float uu = s_red[0][0][c] + s_red[0][1][c];
    const float ww = s_red[1][0][c] + s_red[1][1][c];
    delta[e] = b * (s_v[c] - d * uu);
    if (warp == 0 && rsub == 0)
      Elem<TO>::store(o + (t * p.hv + h) * kD + col0 + e, d * ww + qk * delta[e]);
  }
  // S' = d S + k delta^T, written straight from the update
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

template <typename T, typename TO>
cudaError_t launch_decode1(const DecodeParams &p, unsigned units, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(units);
  cfg.blockDim = dim3(kDec1Threads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode1_kernel<T, TO>, p);
}

}  // namespace

cudaError_t launch_decode(const DecodeParams &p, cudaStream_t stream) {
  const long long units = (long long)p.num_seqs * p.hv * 4;
  if (units == 0) return cudaSuccess;
  if (!p.cu_seqlens && !p.delta) {  // one token per sequence
    if (p.dtype == GDN_BF16 && !p.o_fp32)
      return launch_decode1<__nv_bfloat16, __nv_bfloat16>(p, (unsigned)units, stream);
    if (p.dtype == GDN_BF16) return launch_decode1<__nv_bfloat16, float>(p, (unsigned)units, stream);
    return launch_decode1<float, float>(p, (unsigned)units, stream);
  }
  if (p.dtype == GDN_BF16 && !p.o_fp32)
    decode_kernel<__nv_bfloat16, __nv_bfloat16><<<(unsigned)units, kDecThreads, 0, stream>>>(p);
  else if (p.dtype == GDN_BF16)
    decode_kernel<__nv_bfloat16, float><<<(unsigned)units, kDecThreads, 0, stream>>>(p);
  else
    decode_kernel<float, float><<<(unsigned)units, kDecThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
