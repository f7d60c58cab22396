// State after an accepted prefix of a verified draft block, from the block's per-token
// deltas.  The chunkwise form ("Qwen3.5-9B-npu" model card, section "How it works")
// writes the state after a block of T tokens as
//     S_T = e^{G_T} S_0 + K^T diag(e^{G_T - G}) D,      G the inclusive cumsum of g,
// with D the per-token deltas; no delta depends on a later token, so cutting the sum
// after the first a tokens gives the state after those tokens:
//     S_a = e^{G_a} S_0 + sum_{t<a} e^{G_a - G_t} k_t delta_t^T.
// The prompt-lookup flow of section "New in v2" snapshots the state before checking a
// draft and re-feeds the accepted tokens; with the deltas captured by
// gdn_verify_block_capture, this rank-a update replaces the re-feed.
//
// One CTA of 128 threads per (sequence, v-head, 32 value columns), laid out like the
// decode step: each thread holds 8 rows x 4 columns of S in registers, so the state is
// read once and written once with 128-bit accesses.  Tokens go in tiles of 32: warp 0
// forms the tile's cumsum by a warp scan (the same scan, in the same order, in both
// passes, so G_a - G_{a-1} is exactly 0), the tile's keys and deltas are staged in
// shared memory, and every thread adds the tile's rank-32 update to its entries.
#include "common.cuh"
#include "internal.h"

namespace gdn {

namespace {

constexpr int kRbThreads = 128;
constexpr int kRbCols = 32;  // value columns per CTA
constexpr int kTile = 32;    // tokens per tile

__device__ __forceinline__ int clampi(int x, int lo, int hi) { return min(max(x, lo), hi); }

// Inclusive scan of g over the tile's tokens [t0, t0 + n) of head h, plus `carry`,
// by warp 0; lane l gets G at token t0 + l (tokens past n repeat the last value).
__device__ __forceinline__ float tile_scan(const RollbackParams &p, int h, int t0, int n,
                                           float carry, int lane) {
  float x = lane < n ? p.g[(size_t)(t0 + lane) * p.hv + h] : 0.f;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return carry + x;
}

template <typename T>
__global__ void __launch_bounds__(kRbThreads) rollback_kernel(RollbackParams p) {
  const int quarter = blockIdx.x & 3;
  const int nh = blockIdx.x >> 2;
  const int n = nh / p.hv;
  const int h = nh - n * p.hv;
  const int kh = h / (p.hv / p.hk);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rsub = lane >> 3, cg = lane & 7;
  const int col0 = quarter * kRbCols + cg * 4;

  int bos, eos;
  seq_range(p.cu_seqlens, n, p.total_tokens, bos, eos);
  const int a = clampi(p.prefix_len[n], 0, eos - bos);

  __shared__ float s_k[kTile][kD];
  __shared__ __align__(16) float s_d[kTile][kRbCols];
  __shared__ float s_c[kTile];
  __shared__ float s_ga;

  // pass 1: G_a, the cumsum over the whole prefix
  if (warp == 0) {
    float carry = 0.f;
    for (int t0 = 0; t0 < a; t0 += kTile) {
      const int cnt = min(kTile, a - t0);
      const float G = tile_scan(p, h, bos + t0, cnt, carry, lane);
      carry = __shfl_sync(0xffffffffu, G, cnt - 1);
    }
    if (lane == 0) s_ga = carry;
  }
  __syncthreads();
  const float ga = s_ga;

  const size_t sbase = ((size_t)n * p.hv + h) * kD * kD;
  const float ega = expf(ga);
  float4 S[8];
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int i = s * 16 + warp * 4 + rsub;
    float4 v = p.state_in
                   ? *reinterpret_cast<const float4 *>(p.state_in + sbase + (size_t)i * kD + col0)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    v.x *= ega; v.y *= ega; v.z *= ega; v.w *= ega;
    S[s] = v;
  }

  // pass 2: the rank-a update, a tile of tokens at a time
  const T *k = static_cast<const T *>(p.k);
  float carry = 0.f;
  for (int t0 = 0; t0 < a; t0 += kTile) {
    const int cnt = min(kTile, a - t0);
    if (warp == 0) {
      const float G = tile_scan(p, h, bos + t0, cnt, carry, lane);
      s_c[lane] = lane < cnt ? expf(ga - G) : 0.f;
      carry = __shfl_sync(0xffffffffu, G, cnt - 1);
    }
    for (int e = tid; e < kTile * kD; e += kRbThreads) {
      const int t = e / kD, i = e - t * kD;
      s_k[t][i] = t < cnt ? Elem<T>::load(k + ((size_t)(bos + t0 + t) * p.hk + kh) * kD + i) : 0.f;
    }
    for (int e = tid; e < kTile * kRbCols; e += kRbThreads) {
      const int t = e / kRbCols, j = e - t * kRbCols;
      s_d[t][j] = t < cnt ? p.delta[((size_t)(bos + t0 + t) * p.hv + h) * kD + quarter * kRbCols + j]
                          : 0.f;
    }
    __syncthreads();
    for (int t = 0; t < cnt; ++t) {
      const float c = s_c[t];
      const float4 d = *reinterpret_cast<const float4 *>(&s_d[t][cg * 4]);
      const float dx = c * d.x, dy = c * d.y, dz = c * d.z, dw = c * d.w;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const float ki = s_k[t][s * 16 + warp * 4 + rsub];
        S[s].x = fmaf(ki, dx, S[s].x);
        S[s].y = fmaf(ki, dy, S[s].y);
        S[s].z = fmaf(ki, dz, S[s].z);
        S[s].w = fmaf(ki, dw, S[s].w);
      }
    }
    __syncthreads();  // the tile's shared memory is rewritten by the next one
  }

#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int i = s * 16 + warp * 4 + rsub;
    *reinterpret_cast<float4 *>(p.state_out + sbase + (size_t)i * kD + col0) = S[s];
  }
}

}  // namespace

cudaError_t launch_rollback(const RollbackParams &p, cudaStream_t stream) {
  const long long units = (long long)p.num_seqs * p.hv * 4;
  if (units == 0) return cudaSuccess;
  if (p.dtype == GDN_BF16)
    rollback_kernel<__nv_bfloat16><<<(unsigned)units, kRbThreads, 0, stream>>>(p);
  else
    rollback_kernel<float><<<(unsigned)units, kRbThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
