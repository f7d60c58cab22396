// Chunkwise-parallel gated delta rule in fp32 on CUDA cores ("Qwen3.5-9B-npu" model
// card, section "How it works", chunkwise form).  Per block of C tokens with in-block
// inclusive cumsum G of g and incoming state S0:
//   N   = diag(beta) [exp(G_t - G_j) k_t.k_j]_{j<t}
//   D   = (I + N)^-1 diag(beta) (V - diag(exp G) K S0)     (forward substitution)
//   O   = diag(exp G) Q S0 + [exp(G_t - G_j) q_t.k_j]_{j<=t} D
//   S_T = exp(G_T) S0 + K^T diag(exp(G_T - G)) D
// Decay factors between two tokens are always formed as the exp of a difference of
// cumsums.  A block that runs past the sequence end is padded with g = 0, beta = 0,
// q = k = v = 0 tokens (the page's token_valid rule), which leave the state unchanged.
//
// This is the fp32 path (every operand and product in fp32): one CTA of 256 threads per
// (sequence, v-head, 32 value columns), the 128 x 32 state block resident in shared
// memory across all blocks of the sequence.
#include "common.cuh"
#include "internal.h"

namespace gdn {

namespace {

constexpr int kF32Threads = 256;
constexpr int kF32Cols = 32;
constexpr int kKP = kD + 1;  // padded row of the K / Q tiles

template <int C>
struct F32Smem {
  float K[C][kKP], Q[C][kKP];
  float V[C][kF32Cols];
  float N[C][C + 1], A[C][C + 1];
  float R[C][kF32Cols];  // R, then D in place
  float S[kD][kF32Cols];
  float G[C], EG[C], B[C], DEC[C];
};

template <int C>
__global__ void __launch_bounds__(kF32Threads) chunk_f32_kernel(ChunkParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  F32Smem<C> &sm = *reinterpret_cast<F32Smem<C> *>(smem_raw);
  constexpr int NB = kD / kF32Cols;
  const int blk = blockIdx.x % NB;
  const int nh = blockIdx.x / NB;
  const int n = nh / p.hv;
  const int h = nh - n * p.hv;
  const int kh = h / (p.hv / p.hk);
  const int tid = threadIdx.x;
  const int c0 = blk * kF32Cols;
  const float *q = static_cast<const float *>(p.q);
  const float *k = static_cast<const float *>(p.k);
  const float *v = static_cast<const float *>(p.v);
  float *o = static_cast<float *>(p.o);

  int bos, eos;
  seq_range(p.cu_seqlens, n, p.total_tokens, bos, eos);
  const size_t sbase = ((size_t)n * p.hv + h) * kD * kD;

  for (int e = tid; e < kD * kF32Cols; e += kF32Threads) {
    const int i = e / kF32Cols, c = e % kF32Cols;
    sm.S[i][c] = p.state_in ? p.state_in[sbase + (size_t)i * kD + c0 + c] : 0.f;
  }

  for (int tok0 = bos; tok0 < eos; tok0 += C) {
    const int L = min(C, eos - tok0);
    __syncthreads();  // previous block fully consumed
    for (int e = tid; e < C * kD; e += kF32Threads) {
      const int t = e / kD, i = e % kD;
      const bool ok = t < L;
      const size_t row = ((size_t)(tok0 + (ok ? t : 0)) * p.hk + kh) * kD + i;
      sm.K[t][i] = ok ? k[row] : 0.f;
      sm.Q[t][i] = ok ? q[row] : 0.f;
    }
    for (int e = tid; e < C * kF32Cols; e += kF32Threads) {
      const int t = e / kF32Cols, c = e % kF32Cols;
      sm.V[t][c] = t < L ? v[((size_t)(tok0 + t) * p.hv + h) * kD + c0 + c] : 0.f;
    }
    if (tid == 0) {
      float acc = 0.f;
      for (int t = 0; t < C; ++t) {
        const bool ok = t < L;
        acc += ok ? p.g[(size_t)(tok0 + t) * p.hv + h] : 0.f;
        sm.G[t] = acc;
        sm.EG[t] = expf(acc);
        sm.B[t] = ok ? p.beta[(size_t)(tok0 + t) * p.hv + h] : 0.f;
      }
      for (int t = 0; t < C; ++t) sm.DEC[t] = expf(sm.G[C - 1] - sm.G[t]);
    }
    __syncthreads();

    // decay-masked Grams: N strictly lower (times beta_t), A lower with the diagonal
    for (int e = tid; e < C * C; e += kF32Threads) {
      const int t = e / C, j = e % C;
      float nn = 0.f, aa = 0.f;
      if (j <= t) {
        float kk = 0.f, qk = 0.f;
#pragma unroll 8
        for (int i = 0; i < kD; ++i) {
          kk += sm.K[t][i] * sm.K[j][i];
          qk += sm.Q[t][i] * sm.K[j][i];
        }
        const float dec = expf(sm.G[t] - sm.G[j]);
        aa = dec * qk;
        if (j < t) nn = sm.B[t] * dec * kk;
      }
      sm.N[t][j] = nn;
      sm.A[t][j] = aa;
    }
    // R = diag(beta) (V - diag(exp G) K S0)
    for (int e = tid; e < C * kF32Cols; e += kF32Threads) {
      const int t = e / kF32Cols, c = e % kF32Cols;
      float ks = 0.f;
#pragma unroll 8
      for (int i = 0; i < kD; ++i) ks += sm.K[t][i] * sm.S[i][c];
      sm.R[t][c] = sm.B[t] * (sm.V[t][c] - sm.EG[t] * ks);
    }
    __syncthreads();

    // D = (I + N)^-1 R by forward substitution; 8 lanes per value column
    {
      const int c = tid >> 3, part = tid & 7;
      for (int t = 1; t < C; ++t) {
        float acc = 0.f;
        for (int j = part; j < t; j += 8) acc += sm.N[t][j] * sm.R[j][c];
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        acc += __shfl_xor_sync(0xffffffffu, acc, 4);
        if (part == 0) sm.R[t][c] -= acc;
        __syncwarp();
      }
    }
    __syncthreads();

    // O = diag(exp G) Q S0 + A D
    for (int e = tid; e < C * kF32Cols; e += kF32Threads) {
      const int t = e / kF32Cols, c = e % kF32Cols;
      if (t >= L) continue;
      float qs = 0.f, ad = 0.f;
#pragma unroll 8
      for (int i = 0; i < kD; ++i) qs += sm.Q[t][i] * sm.S[i][c];
      for (int j = 0; j <= t; ++j) ad += sm.A[t][j] * sm.R[j][c];
      o[((size_t)(tok0 + t) * p.hv + h) * kD + c0 + c] = sm.EG[t] * qs + ad;
      if (p.delta) p.delta[((size_t)(tok0 + t) * p.hv + h) * kD + c0 + c] = sm.R[t][c];
    }
    __syncthreads();

    // S_T = exp(G_T) S0 + K^T diag(exp(G_T - G)) D
    const float egc = sm.EG[C - 1];
    for (int e = tid; e < kD * kF32Cols; e += kF32Threads) {
      const int i = e / kF32Cols, c = e % kF32Cols;
      float acc = 0.f;
      for (int t = 0; t < C; ++t) acc += sm.K[t][i] * sm.DEC[t] * sm.R[t][c];
      sm.S[i][c] = egc * sm.S[i][c] + acc;
    }
  }
  __syncthreads();
  for (int e = tid; e < kD * kF32Cols; e += kF32Threads) {
    const int i = e / kF32Cols, c = e % kF32Cols;
    p.state_out[sbase + (size_t)i * kD + c0 + c] = sm.S[i][c];
  }
}

template <int C>
cudaError_t launch_f32(const ChunkParams &p, cudaStream_t stream) {
  const size_t smem = sizeof(F32Smem<C>);
  cudaError_t err = cudaFuncSetAttribute(chunk_f32_kernel<C>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const long long ctas = (long long)p.num_seqs * p.hv * (kD / kF32Cols);
  chunk_f32_kernel<C><<<(unsigned)ctas, kF32Threads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_f32(const ChunkParams &p, cudaStream_t stream) {
  if ((long long)p.num_seqs * p.hv == 0) return cudaSuccess;
  switch (p.chunk) {
    case 16: return launch_f32<16>(p, stream);
    case 32: return launch_f32<32>(p, stream);
    case 64: return launch_f32<64>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
