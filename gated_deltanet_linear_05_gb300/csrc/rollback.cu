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
// read once and written once with 128-bit accesses.  Tokens go in tiles of 32 (a draft
// block is one tile): the tile's keys, deltas and gates are staged in shared memory by
// cp.async, issued together with the state's loads; warp 0 forms the tile's cumsum by a
// warp scan, and every thread adds the tile's rank-32 update to its entries.
#include "common.cuh"
#include "internal.h"

namespace gdn {

namespace {

constexpr int kRbThreads = 128;
constexpr int kRbCols = 32;  // value columns per CTA
constexpr int kTile = 32;    // tokens per tile

__device__ __forceinline__ int clampi(int x, int lo, int hi) { return min(max(x, lo), hi); }

// Inclusive warp scan of the tile's g values (lane l: token l of the tile, 0 past cnt),
// plus `carry`; lane l gets G at token l (lanes past cnt repeat the last value).
__device__ __forceinline__ float warp_scan(float x, float carry, int lane) {
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

  __shared__ __align__(16) T s_k[kTile][kD];           // the tile's key rows, as stored
  __shared__ __align__(16) float s_d[kTile][kRbCols];  // the tile's deltas, this CTA's columns
  __shared__ float s_g[kTile], s_c[kTile];
  __shared__ float s_ga;
  const T *k = static_cast<const T *>(p.k);

  // keys, deltas and gates of tokens bos + t0 .. bos + t0 + cnt - 1, by cp.async
  auto load_tile = [&](int t0, int cnt) {
    constexpr int EG = 16 / (int)sizeof(T), KG = kD / EG;  // 16-byte granules of a key row
    for (int e = tid; e < kTile * KG; e += kRbThreads) {
      const int t = e / KG, gq = e - t * KG;
      const bool ok = t < cnt;
      const size_t tok = (size_t)bos + t0 + (ok ? t : 0);
      cp_async16(&s_k[t][gq * EG], k + (tok * p.hk + kh) * kD + gq * EG, ok ? 16 : 0);
    }
    for (int e = tid; e < kTile * (kRbCols / 4); e += kRbThreads) {
      const int t = e / (kRbCols / 4), gq = e - t * (kRbCols / 4);
      const bool ok = t < cnt;
      const size_t tok = (size_t)bos + t0 + (ok ? t : 0);
      cp_async16(&s_d[t][gq * 4], p.delta + (tok * p.hv + h) * kD + quarter * kRbCols + gq * 4,
                 ok ? 16 : 0);
    }
    if (tid < kTile) {
      const bool ok = tid < cnt;
      cp_async4(&s_g[tid], p.g + ((size_t)bos + t0 + (ok ? tid : 0)) * p.hv + h, ok ? 4 : 0);
    }
    cp_async_commit();
  };

  // the first tile's copies and the state's loads go out together
  if (a > 0) load_tile(0, min(kTile, a));
  const size_t sbase = ((size_t)n * p.hv + h) * kD * kD;
  float4 S[8];
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int i = s * 16 + warp * 4 + rsub;
    S[s] = p.state_in
               ? *reinterpret_cast<const float4 *>(p.state_in + sbase + (size_t)i * kD + col0)
               : make_float4(0.f, 0.f, 0.f, 0.f);
  }

  // G_a, the cumsum over the whole prefix: from the staged first tile when the prefix
  // fits in one tile (a draft block), else scanned tile by tile from global memory; the
  // same scan, in the same order, gives the G_t of pass 2, so G_a - G_{a-1} is exactly 0
  cp_async_wait<0>();
  __syncthreads();
  if (warp == 0) {
    float carry = 0.f;
    if (a <= kTile) {
      const float G = warp_scan(lane < a ? s_g[lane] : 0.f, 0.f, lane);
      if (a > 0) carry = __shfl_sync(0xffffffffu, G, a - 1);
    } else {
      for (int t0 = 0; t0 < a; t0 += kTile) {
        const int cnt = min(kTile, a - t0);
        const float x = lane < cnt ? p.g[((size_t)bos + t0 + lane) * p.hv + h] : 0.f;
        const float G = warp_scan(x, carry, lane);
        carry = __shfl_sync(0xffffffffu, G, cnt - 1);
      }
    }
    if (lane == 0) s_ga = carry;
  }
  __syncthreads();
  const float ga = s_ga;
  const float ega = expf(ga);
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    S[s].x *= ega; S[s].y *= ega; S[s].z *= ega; S[s].w *= ega;
  }

  // pass 2: the rank-a update, a tile of tokens at a time (the first tile already staged)
  float carry = 0.f;
  for (int t0 = 0; t0 < a; t0 += kTile) {
    const int cnt = min(kTile, a - t0);
    if (t0 > 0) {
      __syncthreads();  // the previous tile's shared memory is free
      load_tile(t0, cnt);
      cp_async_wait<0>();
      __syncthreads();
    }
    if (warp == 0) {
      const float G = warp_scan(lane < cnt ? s_g[lane] : 0.f, carry, lane);
      s_c[lane] = lane < cnt ? expf(ga - G) : 0.f;
      carry = __shfl_sync(0xffffffffu, G, cnt - 1);
    }
    __syncthreads();
    for (int t = 0; t < cnt; ++t) {
      const float c = s_c[t];
      const float4 d = *reinterpret_cast<const float4 *>(&s_d[t][cg * 4]);
      const float dx = c * d.x, dy = c * d.y, dz = c * d.z, dw = c * d.w;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const float ki = Elem<T>::load(&s_k[t][s * 16 + warp * 4 + rsub]);
        S[s].x = fmaf(ki, dx, S[s].x);
        S[s].y = fmaf(ki, dy, S[s].y);
        S[s].z = fmaf(ki, dz, S[s].z);
        S[s].w = fmaf(ki, dw, S[s].w);
      }
    }
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
