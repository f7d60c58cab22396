// Chunkwise-parallel gated delta rule, bf16 q/k/v on tensor cores ("Qwen3.5-9B-npu"
// model card, section "How it works", chunkwise form):
//   N   = diag(beta) [exp(G_t - G_j) k_t.k_j]_{j<t}
//   D   = (I + N)^-1 diag(beta) (V - diag(exp G) K S0)
//   O   = diag(exp G) Q S0 + [exp(G_t - G_j) q_t.k_j]_{j<=t} D
//   S_T = exp(G_T) S0 + K^T diag(exp(G_T - G)) D
//
// The state-independent part of D is split off:  with T = (I + N)^-1,
//   D = U - W S0,   U = T diag(beta) V,   W = T diag(beta exp G) K,
// so the work falls in two passes:
//   pass 1 (prep_kernel, every block of every head in parallel): G, the decay-masked
//     Grams, T by exact block doubling in fp32 (16x16 diagonal blocks by forward
//     substitution, then (D + C)^-1 = D^-1 - D^-1 C D^-1 on 16 -> 32 -> 64), and the
//     products W, U on tensor cores.  Writes W, U (fp32), the masked causal A and G
//     (fp32) to the workspace, indexed by token.
//   pass 2 (recur_kernel, one CTA per (sequence, v-head, DVB value columns)): walks the
//     blocks of the sequence in order with the state block S[:, cols] in fp32 registers
//     (read from state_in once, written to state_out once):
//       D^T = U^T - S^T W^T,  O^T = exp(G) (S^T Q^T) + D^T A^T,
//       S^T <- exp(G_T) S^T + (D^T diag(exp(G_T - G))) K
//     all on mma.sync tensor cores with fp32 accumulation.
// Precision: q, k, v are bf16 inputs and enter the products exactly.  Every other MMA
// operand (T, W, A, the state, D) is an fp32 value x carried as two bf16 numbers,
// hi = bf16(x) and lo = bf16(x - hi), and a product x*y is formed as hi*hi + lo*hi +
// hi*lo (or hi*y + lo*y when y is an input), which keeps ~16 significant bits: the
// layer's outputs have heavy tails (max/rms above 10), so single-bf16 intermediates
// would put errors of a few 1e-2 of the rms on the largest entries.
// Decay factors between two tokens are always the exp of a difference of cumsums.  A
// partly filled block is padded with g = 0, beta = 0, zero q/k/v rows (token_valid),
// which leaves the state exactly as after the sequence's last token.
#include "common.cuh"
#include "internal.h"

namespace gdn {

namespace {

constexpr int kRowB = kD * 2;  // bytes in a 128-element bf16 row

__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
  hi = pack_bf16(__bfloat162float(h0), __bfloat162float(h1));
  lo = pack_bf16(x0 - __bfloat162float(h0), x1 - __bfloat162float(h1));
}

// ================================================================== pass 1

template <int C>
struct PrepSmem {
  alignas(128) char K[C * kRowB];
  alignas(128) char V[C * kRowB];
  // Q tile followed by N (fp32); overlaid after the solve by the four bf16 copies of T
  alignas(128) char X[C * kRowB + C * (C + 4) * 4];
  float T[C][C + 4];
  float M[32 * 33];
  float G[C], EG[C], B[C];
};

template <int C>
__global__ void __launch_bounds__(2 * C) prep_kernel(ChunkParams p, int slots) {
  constexpr int NW = C / 16, NT = 32 * NW, MT = C / 16, RB = 2 * C;
  static_assert(8 * C * C <= C * kRowB + C * (C + 4) * 4, "overlay too small");
  extern __shared__ __align__(128) unsigned char smem_raw[];
  PrepSmem<C> &sm = *reinterpret_cast<PrepSmem<C> *>(smem_raw);
  char *sQ = sm.X;
  float(*sN)[C + 4] = reinterpret_cast<float(*)[C + 4]>(sm.X + C * kRowB);
  char *TWH = sm.X, *TWL = sm.X + C * RB, *TUH = sm.X + 2 * C * RB, *TUL = sm.X + 3 * C * RB;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int slot = blockIdx.x % slots;
  const int nh = blockIdx.x / slots;
  const int n = nh / p.hv;
  const int h = nh - n * p.hv;
  const int kh = h / (p.hv / p.hk);
  const size_t T = (size_t)p.total_tokens;
  const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(p.q);
  const __nv_bfloat16 *k = static_cast<const __nv_bfloat16 *>(p.k);
  const __nv_bfloat16 *v = static_cast<const __nv_bfloat16 *>(p.v);
  __nv_bfloat16 *w_hi = static_cast<__nv_bfloat16 *>(p.w_hi);
  __nv_bfloat16 *w_lo = static_cast<__nv_bfloat16 *>(p.w_lo);
  __nv_bfloat16 *a_hi = static_cast<__nv_bfloat16 *>(p.a_hi);
  __nv_bfloat16 *a_lo = static_cast<__nv_bfloat16 *>(p.a_lo);

  int bos, eos;
  seq_range(p.cu_seqlens, n, p.total_tokens, bos, eos);
  const int nchunks = (eos - bos + C - 1) / C;

  for (int c = slot; c < nchunks; c += slots) {
    const int tok0 = bos + c * C;
    const int L = min(C, eos - tok0);
    __syncthreads();  // the previous block is done with shared memory

    for (int e = tid; e < C * 16; e += NT) {
      const int r = e >> 4, gr = e & 15;
      const bool ok = r < L;
      const size_t tok = (size_t)tok0 + (ok ? r : 0);
      const int nb = ok ? 16 : 0;
      cp_async16(sm.K + swz<kRowB>(r, gr * 16), k + (tok * p.hk + kh) * kD + gr * 8, nb);
      cp_async16(sQ + swz<kRowB>(r, gr * 16), q + (tok * p.hk + kh) * kD + gr * 8, nb);
      cp_async16(sm.V + swz<kRowB>(r, gr * 16), v + (tok * p.hv + h) * kD + gr * 8, nb);
    }
    cp_async_commit();

    // in-block inclusive cumsum of g (padding contributes 0), exp(G), beta
    if (warp == 0) {
      constexpr int E = (C + 31) / 32;
      float gv[E], bv[E], run = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int t = lane * E + e;
        const bool ok = t < L;
        gv[e] = ok ? p.g[((size_t)tok0 + t) * p.hv + h] : 0.f;
        bv[e] = ok ? p.beta[((size_t)tok0 + t) * p.hv + h] : 0.f;
        run += gv[e];
        gv[e] = run;
      }
      float incl = run;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      const float excl = incl - run;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int t = lane * E + e;
        if (t < C) {
          sm.G[t] = gv[e] + excl;
          sm.EG[t] = expf(gv[e] + excl);
          sm.B[t] = bv[e];
        }
      }
    }
    for (int e = tid; e < C * (C + 4); e += NT) (&sm.T[0][0])[e] = 0.f;
    cp_async_wait<0>();
    __syncthreads();

    // ---- decay-masked Grams on tensor cores: warp w takes items 2w, 2w+1 of
    //      [KK(0), KK(MT-1), KK(1), ..., QK(0), QK(MT-1), ...] (balanced triangles)
#pragma unroll 1
    for (int it = 0; it < 2; ++it) {
      const int item = warp * 2 + it;
      const int prod = item / MT;  // 0: K K^T, 1: Q K^T
      const int r = item % MT;
      const int mt = (r & 1) ? (MT - 1 - r / 2) : (r / 2);
      const char *Asrc = prod ? sQ : sm.K;
      float acc[C / 8][4];
#pragma unroll
      for (int a = 0; a < C / 8; ++a)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[a][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < kD / 16; ++ks) {
        uint32_t a[4];
        lda_tile<kRowB>(a, Asrc, 16 * mt, 16 * ks, lane);
#pragma unroll
        for (int np = 0; np < C / 16; ++np) {
          if (np <= mt) {
            uint32_t b[4];
            ldb_nk<kRowB>(b, sm.K, 16 * np, 16 * ks, lane);
            mma_bf16(acc[2 * np], a, b[0], b[1]);
            mma_bf16(acc[2 * np + 1], a, b[2], b[3]);
          }
        }
      }
#pragma unroll
      for (int nt = 0; nt < C / 8; ++nt) {
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int t = 16 * mt + gid + 8 * hr;
          const int j = 8 * nt + 2 * tig;
          if (nt <= 2 * mt + 1) {
            const float d0 = expf(sm.G[t] - sm.G[j]), d1 = expf(sm.G[t] - sm.G[j + 1]);
            const float x0 = acc[nt][2 * hr], x1 = acc[nt][2 * hr + 1];
            if (prod == 0) {
              sN[t][j] = (j < t) ? sm.B[t] * d0 * x0 : 0.f;
              sN[t][j + 1] = (j + 1 < t) ? sm.B[t] * d1 * x1 : 0.f;
            } else if (t < L) {
              const float a0 = (j <= t) ? d0 * x0 : 0.f, a1 = (j + 1 <= t) ? d1 * x1 : 0.f;
              uint32_t hi, lo;
              split_bf16(a0, a1, hi, lo);
              const size_t at = ((size_t)h * T + tok0 + t) * C + j;
              *reinterpret_cast<uint32_t *>(a_hi + at) = hi;
              *reinterpret_cast<uint32_t *>(a_lo + at) = lo;
            }
          } else if (prod == 1 && t < L) {
            const size_t at = ((size_t)h * T + tok0 + t) * C + j;
            *reinterpret_cast<uint32_t *>(a_hi + at) = 0u;
            *reinterpret_cast<uint32_t *>(a_lo + at) = 0u;
          }
        }
      }
    }
    __syncthreads();

    // ---- T = (I + N)^-1 by block doubling in fp32.  Level 0: 16x16 diagonal blocks,
    //      one column per thread, forward substitution.
    if (tid < C) {
      const int base = (tid >> 4) * 16, cc = tid & 15;
      float x[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        float val = (r == cc) ? 1.f : 0.f;
        if (r > cc) {
          float acc = 0.f;
#pragma unroll
          for (int m = 0; m < r; ++m)
            if (m >= cc) acc += sN[base + r][base + m] * x[m];
          val = -acc;
        }
        x[r] = val;
        sm.T[base + r][base + cc] = val;
      }
    }
    __syncthreads();
    if (C >= 32) {  // level 1: 16 -> 32, lower-left block = -T_bot N_bl T_top
      for (int e = tid; e < (C / 32) * 256; e += NT) {
        const int pr = e >> 8, r = (e >> 4) & 15, cc = e & 15, top = 32 * pr, bot = top + 16;
        float acc = 0.f;
        for (int m = cc; m < 16; ++m) acc += sN[bot + r][top + m] * sm.T[top + m][top + cc];
        sm.M[pr * 256 + r * 16 + cc] = acc;
      }
      __syncthreads();
      for (int e = tid; e < (C / 32) * 256; e += NT) {
        const int pr = e >> 8, r = (e >> 4) & 15, cc = e & 15, top = 32 * pr, bot = top + 16;
        float acc = 0.f;
        for (int m = 0; m <= r; ++m) acc += sm.T[bot + r][bot + m] * sm.M[pr * 256 + m * 16 + cc];
        sm.T[bot + r][top + cc] = -acc;
      }
      __syncthreads();
    }
    if (C == 64) {  // level 2: 32 -> 64
      for (int e = tid; e < 1024; e += NT) {
        const int r = e >> 5, cc = e & 31;
        float acc = 0.f;
        for (int m = cc; m < 32; ++m) acc += sN[32 + r][m] * sm.T[m][cc];
        sm.M[r * 33 + cc] = acc;
      }
      __syncthreads();
      for (int e = tid; e < 1024; e += NT) {
        const int r = e >> 5, cc = e & 31;
        float acc = 0.f;
        for (int m = 0; m <= r; ++m) acc += sm.T[32 + r][32 + m] * sm.M[m * 33 + cc];
        sm.T[32 + r][cc] = -acc;
      }
      __syncthreads();
    }

    // ---- bf16 operands T diag(beta exp G) and T diag(beta), each as high + low part
    for (int e = tid; e < C * C / 2; e += NT) {
      const int t = e / (C / 2), j = 2 * (e % (C / 2));
      const float x0 = sm.T[t][j], x1 = sm.T[t][j + 1];
      uint32_t hi, lo;
      split_bf16(x0 * sm.B[j] * sm.EG[j], x1 * sm.B[j + 1] * sm.EG[j + 1], hi, lo);
      *reinterpret_cast<uint32_t *>(TWH + swz<RB>(t, 2 * j)) = hi;
      *reinterpret_cast<uint32_t *>(TWL + swz<RB>(t, 2 * j)) = lo;
      split_bf16(x0 * sm.B[j], x1 * sm.B[j + 1], hi, lo);
      *reinterpret_cast<uint32_t *>(TUH + swz<RB>(t, 2 * j)) = hi;
      *reinterpret_cast<uint32_t *>(TUL + swz<RB>(t, 2 * j)) = lo;
    }
    __syncthreads();

    // ---- W = T diag(beta e^G) K, U = T diag(beta) V: 32 n-tiles (16 of W, 16 of U)
    //      spread over the warps in groups of 8; causal: T[t][j] = 0 for j > t.
    constexpr int NTW = 32 / NW;
#pragma unroll 1
    for (int g0 = 0; g0 < NTW; g0 += 8) {
      const int q0 = warp * NTW + g0;
      const bool isU = q0 >= 16;
      const char *Bsrc = isU ? sm.V : sm.K;
      const char *AH = isU ? TUH : TWH;
      const char *AL = isU ? TUL : TWL;
      const int n0 = (q0 & 15) * 8;
#pragma unroll 1
      for (int mt = 0; mt < MT; ++mt) {
        float acc[8][4];
#pragma unroll
        for (int a = 0; a < 8; ++a)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[a][e] = 0.f;
        for (int ks = 0; ks <= mt; ++ks) {
          uint32_t ah[4], al[4];
          lda_tile<RB>(ah, AH, 16 * mt, 16 * ks, lane);
          lda_tile<RB>(al, AL, 16 * mt, 16 * ks, lane);
#pragma unroll
          for (int np = 0; np < 4; ++np) {
            uint32_t b[4];
            ldb_kn<kRowB>(b, Bsrc, 16 * ks, n0 + 16 * np, lane);
            mma_bf16(acc[2 * np], ah, b[0], b[1]);
            mma_bf16(acc[2 * np], al, b[0], b[1]);
            mma_bf16(acc[2 * np + 1], ah, b[2], b[3]);
            mma_bf16(acc[2 * np + 1], al, b[2], b[3]);
          }
        }
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int t = 16 * mt + gid + 8 * hr;
            const int col = n0 + 8 * nt + 2 * tig;
            if (t < L) {
              const size_t row = ((size_t)h * T + tok0 + t) * kD + col;
              if (isU) {
                *reinterpret_cast<float2 *>(p.u_ws + row) =
                    make_float2(acc[nt][2 * hr], acc[nt][2 * hr + 1]);
              } else {
                uint32_t hi, lo;
                split_bf16(acc[nt][2 * hr], acc[nt][2 * hr + 1], hi, lo);
                *reinterpret_cast<uint32_t *>(w_hi + row) = hi;
                *reinterpret_cast<uint32_t *>(w_lo + row) = lo;
              }
            }
          }
        }
      }
    }
    for (int t = tid; t < L; t += NT) p.g_ws[(size_t)h * T + tok0 + t] = sm.G[t];
  }
}

// ================================================================== pass 2

template <int C, int DVB, typename TO>
struct RecSmem {
  struct Stage {
    alignas(128) char Wh[C * kRowB];
    alignas(128) char Wl[C * kRowB];
    alignas(128) char Q[C * kRowB];
    alignas(128) char K[C * kRowB];
    alignas(128) char Ah[C * 2 * C];
    alignas(128) char Al[C * 2 * C];
    alignas(16) float U[C][DVB];
    alignas(16) float G[C];
  } st[2];
  alignas(128) char Sh[DVB * kRowB];   // S^T as bf16 operands (hi, lo), [DVB][128]
  alignas(128) char Sl[DVB * kRowB];
  alignas(128) char Dh[DVB * 2 * C];   // D^T (hi, lo), [DVB][C]
  alignas(128) char Dl[DVB * 2 * C];
  alignas(128) char Th[DVB * 2 * C];   // (diag(exp(G_T - G)) D)^T (hi, lo)
  alignas(128) char Tl[DVB * 2 * C];
  alignas(16) TO O[C][DVB];            // output staging
  alignas(16) float S32[kD][DVB + 4];  // fp32 staging of the state block
};

template <int C, int DVB, typename TO>
__device__ __forceinline__ void load_stage(typename RecSmem<C, DVB, TO>::Stage &st,
                                           const ChunkParams &p, int h, int kh, int blk,
                                           int tok0, int L) {
  constexpr int RB = 2 * C;
  const size_t T = (size_t)p.total_tokens;
  const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(p.q);
  const __nv_bfloat16 *k = static_cast<const __nv_bfloat16 *>(p.k);
  const __nv_bfloat16 *w_hi = static_cast<const __nv_bfloat16 *>(p.w_hi);
  const __nv_bfloat16 *w_lo = static_cast<const __nv_bfloat16 *>(p.w_lo);
  const __nv_bfloat16 *a_hi = static_cast<const __nv_bfloat16 *>(p.a_hi);
  const __nv_bfloat16 *a_lo = static_cast<const __nv_bfloat16 *>(p.a_lo);
  const int tid = threadIdx.x;
  for (int e = tid; e < C * 16; e += 128) {
    const int r = e >> 4, gr = e & 15;
    const bool ok = r < L;
    const size_t tok = (size_t)tok0 + (ok ? r : 0);
    const int nb = ok ? 16 : 0;
    const int so = swz<kRowB>(r, gr * 16);
    const size_t wrow = ((size_t)h * T + tok) * kD + gr * 8;
    cp_async16(st.Wh + so, w_hi + wrow, nb);
    cp_async16(st.Wl + so, w_lo + wrow, nb);
    cp_async16(st.Q + so, q + (tok * p.hk + kh) * kD + gr * 8, nb);
    cp_async16(st.K + so, k + (tok * p.hk + kh) * kD + gr * 8, nb);
  }
  for (int e = tid; e < C * (C / 8); e += 128) {
    const int r = e / (C / 8), gr = e % (C / 8);
    const bool ok = r < L;
    const size_t tok = (size_t)tok0 + (ok ? r : 0);
    const int so = swz<RB>(r, gr * 16);
    const size_t arow = ((size_t)h * T + tok) * C + gr * 8;
    cp_async16(st.Ah + so, a_hi + arow, ok ? 16 : 0);
    cp_async16(st.Al + so, a_lo + arow, ok ? 16 : 0);
  }
  for (int e = tid; e < C * (DVB / 4); e += 128) {
    const int r = e / (DVB / 4), gr = e % (DVB / 4);
    const bool ok = r < L;
    const size_t tok = (size_t)tok0 + (ok ? r : 0);
    cp_async16(&st.U[r][gr * 4], p.u_ws + ((size_t)h * T + tok) * kD + blk * DVB + gr * 4,
               ok ? 16 : 0);
  }
  for (int e = tid; e < C; e += 128) {
    const bool ok = e < L;
    cp_async4(&st.G[e], p.g_ws + (size_t)h * T + tok0 + (ok ? e : 0), ok ? 4 : 0);
  }
}

template <int C, int DVB, typename TO>
__global__ void __launch_bounds__(128) recur_kernel(ChunkParams p) {
  constexpr int NB = kD / DVB, MB = DVB / 16, TT = C / 16, RB = 2 * C;
  using Smem = RecSmem<C, DVB, TO>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int blk = blockIdx.x % NB;
  const int nh = blockIdx.x / NB;
  const int n = nh / p.hv;
  const int h = nh - n * p.hv;
  const int kh = h / (p.hv / p.hk);
  TO *o = static_cast<TO *>(p.o);

  int bos, eos;
  seq_range(p.cu_seqlens, n, p.total_tokens, bos, eos);
  const int nchunks = (eos - bos + C - 1) / C;
  const size_t sbase = ((size_t)n * p.hv + h) * kD * kD + blk * DVB;

  // state block S[:, blk*DVB .. +DVB) -> fp32 staging (coalesced rows of DVB floats)
  for (int e = tid; e < kD * DVB / 4; e += 128) {
    const int i = e / (DVB / 4), c4 = e % (DVB / 4);
    const float4 val =
        p.state_in ? *reinterpret_cast<const float4 *>(p.state_in + sbase + (size_t)i * kD + 4 * c4)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    *reinterpret_cast<float4 *>(&sm.S32[i][4 * c4]) = val;
  }
  for (int s = 0; s < 2; ++s) {
    if (s < nchunks)
      load_stage<C, DVB, TO>(sm.st[s], p, h, kh, blk, bos + s * C, min(C, eos - bos - s * C));
    cp_async_commit();
  }
  __syncthreads();

  // S^T fragments: rows j (value columns), cols i (keys 32*warp ..)
  float Sa[MB][4][4];
#pragma unroll
  for (int m = 0; m < MB; ++m)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        Sa[m][nt][e] = sm.S32[32 * warp + 8 * nt + 2 * tig + (e & 1)][16 * m + gid + 8 * (e >> 1)];

  auto write_state_operand = [&]() {
#pragma unroll
    for (int m = 0; m < MB; ++m)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int j = 16 * m + gid + 8 * hr, i = 32 * warp + 8 * nt + 2 * tig;
          uint32_t hi, lo;
          split_bf16(Sa[m][nt][2 * hr], Sa[m][nt][2 * hr + 1], hi, lo);
          *reinterpret_cast<uint32_t *>(sm.Sh + swz<kRowB>(j, 2 * i)) = hi;
          *reinterpret_cast<uint32_t *>(sm.Sl + swz<kRowB>(j, 2 * i)) = lo;
        }
  };
  write_state_operand();

#pragma unroll 1
  for (int c = 0; c < nchunks; ++c) {
    typename Smem::Stage &st = sm.st[c & 1];
    cp_async_wait<1>();
    __syncthreads();
    const int tok0 = bos + c * C;
    const int L = min(C, eos - tok0);
    const float gC = st.G[L - 1];
    const float egc = expf(gC);

    float Op[MB][2][4];
    if (warp < TT) {
      // P = S^T W^T and R = S^T Q^T for this warp's 16 tokens (main and correction terms)
      float P[MB][2][4], Pc[MB][2][4], R[MB][2][4], Rc[MB][2][4];
#pragma unroll
      for (int m = 0; m < MB; ++m)
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int e = 0; e < 4; ++e) P[m][a][e] = Pc[m][a][e] = R[m][a][e] = Rc[m][a][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < kD / 16; ++ks) {
        uint32_t bwh[4], bwl[4], bq[4];
        ldb_nk<kRowB>(bwh, st.Wh, 16 * warp, 16 * ks, lane);
        ldb_nk<kRowB>(bwl, st.Wl, 16 * warp, 16 * ks, lane);
        ldb_nk<kRowB>(bq, st.Q, 16 * warp, 16 * ks, lane);
#pragma unroll
        for (int m = 0; m < MB; ++m) {
          uint32_t ah[4], al[4];
          lda_tile<kRowB>(ah, sm.Sh, 16 * m, 16 * ks, lane);
          lda_tile<kRowB>(al, sm.Sl, 16 * m, 16 * ks, lane);
#pragma unroll
          for (int a = 0; a < 2; ++a) {
            mma_bf16(P[m][a], ah, bwh[2 * a], bwh[2 * a + 1]);
            mma_bf16(Pc[m][a], al, bwh[2 * a], bwh[2 * a + 1]);
            mma_bf16(Pc[m][a], ah, bwl[2 * a], bwl[2 * a + 1]);
            mma_bf16(R[m][a], ah, bq[2 * a], bq[2 * a + 1]);
            mma_bf16(Rc[m][a], al, bq[2 * a], bq[2 * a + 1]);
          }
        }
      }
      // D = U - W S (transposed), the exp(G)-scaled output part, and D scaled for the carry
#pragma unroll
      for (int m = 0; m < MB; ++m)
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int j = 16 * m + gid + 8 * hr;
            const int t = 16 * warp + 8 * a + 2 * tig;
            const float g0 = (t < L) ? st.G[t] : gC, g1 = (t + 1 < L) ? st.G[t + 1] : gC;
            const float d0 = st.U[t][j] - (P[m][a][2 * hr] + Pc[m][a][2 * hr]);
            const float d1 = st.U[t + 1][j] - (P[m][a][2 * hr + 1] + Pc[m][a][2 * hr + 1]);
            Op[m][a][2 * hr] = expf(g0) * (R[m][a][2 * hr] + Rc[m][a][2 * hr]);
            Op[m][a][2 * hr + 1] = expf(g1) * (R[m][a][2 * hr + 1] + Rc[m][a][2 * hr + 1]);
            const int so = swz<RB>(j, 2 * t);
            uint32_t hi, lo;
            split_bf16(d0, d1, hi, lo);
            *reinterpret_cast<uint32_t *>(sm.Dh + so) = hi;
            *reinterpret_cast<uint32_t *>(sm.Dl + so) = lo;
            split_bf16(d0 * expf(gC - g0), d1 * expf(gC - g1), hi, lo);
            *reinterpret_cast<uint32_t *>(sm.Th + so) = hi;
            *reinterpret_cast<uint32_t *>(sm.Tl + so) = lo;
          }
    }
    __syncthreads();

    if (warp < TT) {
      // O^T += D^T A^T over the causal part of the block
      for (int ks = 0; ks <= warp; ++ks) {
        uint32_t bh[4], bl[4];
        ldb_nk<RB>(bh, st.Ah, 16 * warp, 16 * ks, lane);
        ldb_nk<RB>(bl, st.Al, 16 * warp, 16 * ks, lane);
#pragma unroll
        for (int m = 0; m < MB; ++m) {
          uint32_t ah[4], al[4];
          lda_tile<RB>(ah, sm.Dh, 16 * m, 16 * ks, lane);
          lda_tile<RB>(al, sm.Dl, 16 * m, 16 * ks, lane);
#pragma unroll
          for (int a = 0; a < 2; ++a) {
            mma_bf16(Op[m][a], ah, bh[2 * a], bh[2 * a + 1]);
            mma_bf16(Op[m][a], al, bh[2 * a], bh[2 * a + 1]);
            mma_bf16(Op[m][a], ah, bl[2 * a], bl[2 * a + 1]);
          }
        }
      }
#pragma unroll
      for (int m = 0; m < MB; ++m)
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            Elem<TO>::store(&sm.O[16 * warp + 8 * a + 2 * tig + (e & 1)][16 * m + gid + 8 * (e >> 1)],
                            Op[m][a][e]);
      __syncwarp();
      constexpr int EPG = 16 / sizeof(TO);        // elements per 16-byte granule
      constexpr int GPR = DVB / EPG;              // granules per output row
      for (int e = lane; e < 16 * GPR; e += 32) {
        const int r = e / GPR, gi = e % GPR, t = 16 * warp + r;
        if (t < L)
          *reinterpret_cast<uint4 *>(o + ((size_t)(tok0 + t) * p.hv + h) * kD + blk * DVB + gi * EPG) =
              *reinterpret_cast<const uint4 *>(&sm.O[t][gi * EPG]);
      }
    }

    // S^T <- exp(G_T) S^T + Dt^T K  (this warp's 32 keys)
#pragma unroll
    for (int m = 0; m < MB; ++m)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) Sa[m][nt][e] *= egc;
#pragma unroll
    for (int ks = 0; ks < TT; ++ks) {
      uint32_t ah[MB][4], al[MB][4];
#pragma unroll
      for (int m = 0; m < MB; ++m) {
        lda_tile<RB>(ah[m], sm.Th, 16 * m, 16 * ks, lane);
        lda_tile<RB>(al[m], sm.Tl, 16 * m, 16 * ks, lane);
      }
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        uint32_t b[4];
        ldb_kn<kRowB>(b, st.K, 16 * ks, 32 * warp + 16 * np, lane);
#pragma unroll
        for (int m = 0; m < MB; ++m) {
          mma_bf16(Sa[m][2 * np], ah[m], b[0], b[1]);
          mma_bf16(Sa[m][2 * np], al[m], b[0], b[1]);
          mma_bf16(Sa[m][2 * np + 1], ah[m], b[2], b[3]);
          mma_bf16(Sa[m][2 * np + 1], al[m], b[2], b[3]);
        }
      }
    }
    write_state_operand();
    __syncthreads();
    if (c + 2 < nchunks)
      load_stage<C, DVB, TO>(st, p, h, kh, blk, bos + (c + 2) * C, min(C, eos - bos - (c + 2) * C));
    cp_async_commit();
  }
  cp_async_wait<0>();

  // final state block -> state_out (coalesced through the fp32 staging)
#pragma unroll
  for (int m = 0; m < MB; ++m)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        sm.S32[32 * warp + 8 * nt + 2 * tig + (e & 1)][16 * m + gid + 8 * (e >> 1)] = Sa[m][nt][e];
  __syncthreads();
  for (int e = tid; e < kD * DVB / 4; e += 128) {
    const int i = e / (DVB / 4), c4 = e % (DVB / 4);
    *reinterpret_cast<float4 *>(p.state_out + sbase + (size_t)i * kD + 4 * c4) =
        *reinterpret_cast<const float4 *>(&sm.S32[i][4 * c4]);
  }
}

template <int C, typename TO>
cudaError_t launch_recur(const ChunkParams &p, long long heads, cudaStream_t stream) {
  constexpr int DVB = 16;
  const size_t s2 = sizeof(RecSmem<C, DVB, TO>);
  cudaError_t err = cudaFuncSetAttribute(recur_kernel<C, DVB, TO>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s2);
  if (err != cudaSuccess) return err;
  recur_kernel<C, DVB, TO><<<(unsigned)(heads * (kD / DVB)), 128, s2, stream>>>(p);
  return cudaGetLastError();
}

template <int C>
cudaError_t launch_c(const ChunkParams &p, cudaStream_t stream) {
  int dev = 0, sms = 148;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  const long long heads = (long long)p.num_seqs * p.hv;
  const long long max_chunks = ((long long)p.total_tokens + C - 1) / C;
  long long slots = (4LL * sms + heads - 1) / heads;
  slots = max(1LL, min(slots, max(1LL, max_chunks)));

  if (p.total_tokens > 0) {
    const size_t s1 = sizeof(PrepSmem<C>);
    err = cudaFuncSetAttribute(prep_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1);
    if (err != cudaSuccess) return err;
    prep_kernel<C><<<(unsigned)(heads * slots), 2 * C, s1, stream>>>(p, (int)slots);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  return p.o_fp32 ? launch_recur<C, float>(p, heads, stream)
                  : launch_recur<C, __nv_bfloat16>(p, heads, stream);
}

}  // namespace

size_t chunk_workspace_layout(int total_tokens, int hv, int chunk, size_t off[kWsRegions]) {
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t rows = (size_t)total_tokens * hv;
  off[0] = 0;                                      // W hi  bf16 [Hv, T, 128]
  off[1] = off[0] + up(rows * kD * 2);             // W lo  bf16 [Hv, T, 128]
  off[2] = off[1] + up(rows * kD * 2);             // U     fp32 [Hv, T, 128]
  off[3] = off[2] + up(rows * kD * 4);             // A hi  bf16 [Hv, T, chunk]
  off[4] = off[3] + up(rows * (size_t)chunk * 2);  // A lo  bf16 [Hv, T, chunk]
  off[5] = off[4] + up(rows * (size_t)chunk * 2);  // G     fp32 [Hv, T]
  return off[5] + up(rows * 4);
}

cudaError_t launch_chunk_bf16(const ChunkParams &p, cudaStream_t stream) {
  if ((long long)p.num_seqs * p.hv == 0) return cudaSuccess;
  switch (p.chunk) {
    case 16: return launch_c<16>(p, stream);
    case 32: return launch_c<32>(p, stream);
    case 64: return launch_c<64>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
