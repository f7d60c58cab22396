// Chunkwise-parallel gated delta rule, bf16 q/k/v, two passes ("Qwen3.5-9B-npu" model
// card, section "How it works", chunkwise form):
//   N   = diag(beta) [exp(G_t - G_j) k_t.k_j]_{j<t}
//   D   = (I + N)^-1 diag(beta) (V - diag(exp G) K S0)
//   O   = diag(exp G) Q S0 + [exp(G_t - G_j) q_t.k_j]_{j<=t} D
//   S_T = exp(G_T) S0 + K^T diag(exp(G_T - G)) D
//
// The state-independent part of D is split off:  with T = (I + N)^-1,
//   D = U - W S0,   U = T diag(beta) V,   W = T diag(beta exp G) K,
// so the work falls in two passes:
//   pass 1 (prep_kernel, one CTA per (block, v-head), all in parallel): the block's q, k,
//     v rows by tensor-map TMA, G, the decay-masked Grams, the inverses
//     T_ii = (I + N_ii)^-1 of the 16x16 diagonal blocks of I + N by forward substitution,
//     and W and U by blocked forward substitution over the 16-token blocks,
//     X_i = T_ii (R_i - sum_{j<i} N_ij X_j) -- the same triangular solve as the block
//     inverse of the page, applied to the right-hand sides instead of forming
//     (I + N)^-1.  Each block's -W, A, U and decays go to its own workspace slot, -W and
//     U in the fragment order pass 2 loads.
//   pass 2 (recur_kernel, one CTA per (sequence, v-head, 16 value columns)): walks the
//     blocks of the sequence in order with the state block S[:, cols] in fp32 registers
//     (read from state_in once, written to state_out once): per block
//       D = U - W S,   O = diag(e^G) Q S + A D,
//       S <- e^(G_C) S + K^T (diag(e^(G_C - G)) D)
//     with q and k rows loaded from the inputs by tensor-map TMA.
// Tensor-core products (mma.sync) take fp16 operands with fp32 accumulation (the Grams:
// bf16): bf16 q, k and v enter exactly (converted to fp16), the state, D, T, W and A are
// rounded to fp16 (11 significant bits) for the products only; the state itself, the
// sums and every decay are fp32.  Decay factors between two tokens are always the exp of a difference
// of cumsums.  A partly filled block is padded with g = 0, beta = 0 and zero q/k/v rows
// (token_valid), which leaves the state exactly as after the sequence's last token.
#include <cuda.h>
#include <string.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace gdn {

namespace {

__device__ __forceinline__ size_t slot_index(int bos, int chunk, int n, int c) {
  return (size_t)(bos / chunk + n + c);
}

// A fragment (16 rows x 16 k) as fp16 from two 16x8 accumulator tiles (k = their column
// index), columns scaled by s0, s1 (first tile) and t0, t1 (second tile)
__device__ __forceinline__ void acc_to_f16(const float (&x)[4], const float (&y)[4], float s0,
                                           float s1, float t0, float t1, uint32_t (&a)[4]) {
  a[0] = pack_f16(x[0] * s0, x[1] * s1);
  a[1] = pack_f16(x[2] * s0, x[3] * s1);
  a[2] = pack_f16(y[0] * t0, y[1] * t1);
  a[3] = pack_f16(y[2] * t0, y[3] * t1);
}

// The contraction over the keys in pass 2's D = U - W S takes the keys in a permuted
// order: in every span of 32 keys, lane (gid, tig) supplies the consecutive keys
// span + 8tig .. +7, elements {4e, 4e+1} as the k pair (2tig, 2tig+1) and {4e+2, 4e+3} as
// (2tig+8, 2tig+9) of the span's k-step e.  W and S use the same order, so the product is
// unchanged and each lane reads one contiguous 16-byte run per row.
//
// Fragment order of the slot's -W and U: the chain kernel loads each group of 32 lane
// runs (512 bytes) with one coalesced warp instruction.  Groups, lane = 4 gid + tig:
//   WN (chain warp w < C/16, key span s < 4, row half rh): lane's run = -W row
//      16w + gid + 8rh, keys 32s + 8tig .. +7                                   (16 B)
//   U  (value-column block b < 8, chain warp w < C/16): the words U[16w + gid + 8rh]
//      [16b + 8nt + 2tig, +1] for (nt, rh) = (0,0), (0,1), (1,0), (1,1)       (16 B)
__device__ __forceinline__ int wn_off(int w, int s, int rh, int lane) {
  return (((w * 4 + s) * 2 + rh) * 32 + lane) * 16;
}
template <int C>
__device__ __forceinline__ int u_off(int b, int w, int lane) {
  return ((b * (C / 16) + w) * 32 + lane) * 16;
}
// Element `col` of row r of a 128-element-row tile of 16-bit values held as two halves
// (columns 0-63 | 64-127) of `half` bytes, each with 128-byte rows in the TMA 128-byte
// swizzle (16-byte granule g of row r at g ^ (r & 7)).
__device__ __forceinline__ char *sw_el(char *tile, int half, int r, int col) {
  return tile + (col >> 6) * half + swz<128>(r, 2 * (col & 63));
}
__device__ __forceinline__ const char *sw_el(const char *tile, int half, int r, int col) {
  return tile + (col >> 6) * half + swz<128>(r, 2 * (col & 63));
}
// ================================================================== pass 1

template <int C>
struct PrepSmem {
  // bf16 rows as loaded by TMA (keys 0-63 | 64-127, 128-byte swizzle; rows past the end
  // of the tensor: zero, past the end of the sequence: the next one's, never used)
  char K[2][C * 128];
  char Q[2][C * 128];
  char V[2][C * 128];
  float Nd[C / 16][16][17];       // diagonal 16x16 blocks of N (fp32)
  alignas(16) char N16[C * row_c(C)];     // -N (fp16) [t][j], blocks below the diagonal
  alignas(16) char T16[C / 16][16 * 48];  // fp16 T_ii = (I + N_ii)^-1, rows of 48 B
  float G[C], EG[C], ED[C], B[C];
  float gRaw[C], bRaw[C];
  alignas(8) uint64_t bar_kq, bar_v;  // the q/k tiles, the v tile have landed
};

constexpr int kPrepThreads = 256;

// LAYOUT 0: the slot layout of recur_kernel (slot_*_off); LAYOUT 1 (C = 64): the layout
// of the tensor-memory pass 2 (kTs*), every operand stored straight from registers.
template <int C, int LAYOUT>
__global__ void __launch_bounds__(kPrepThreads, 3)
    prep_kernel(ChunkParams p, int per_head, const __grid_constant__ CUtensorMap kmap,
                const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap vmap) {
  constexpr int NT = kPrepThreads, MT = C / 16, RC = row_c(C), HB = C * 128;
  extern __shared__ unsigned char smem_raw[];
  PrepSmem<C> &sm = *reinterpret_cast<PrepSmem<C> *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int part = blockIdx.x % per_head;
  const int nh = blockIdx.x / per_head;
  const int n = nh / p.hv;
  const int h = nh - n * p.hv;
  const int kh = h / (p.hv / p.hk);

  int bos, eos;
  seq_range(p.cu_seqlens, n, p.total_tokens, bos, eos);
  const int nchunks = (eos - bos + C - 1) / C;
  if (tid == 0) {
    mbar_init(&sm.bar_kq, 1);
    mbar_init(&sm.bar_v, 1);
    mbar_fence_init();
  }
  bool ok = true;

#pragma unroll 1
  for (int c = part, it = 0; c < nchunks; c += per_head, ++it) {
    const int tok0 = bos + c * C;
    const int L = min(C, eos - tok0);
    char *slot = p.slot_ws + ((size_t)h * p.nslots + slot_index(bos, C, n, c)) * slot_stride(C, LAYOUT == 1);
    char *wn_out = slot, *a_out = slot + slot_a_off(C);
    char *u_out = slot + slot_u_off(C);
    float *dec_out = reinterpret_cast<float *>(slot + slot_dec_off(C));
    __syncthreads();  // the previous block is done with shared memory (and the barriers set up)

    // the q, k tiles (the Grams start on them) and the v tile by TMA on two barriers;
    // the gates by 4-byte copies (zero past the sequence end: g = 0, beta = 0 padding)
    if (tid == 0) {
      fence_async_smem();  // the previous block's W and U stores before the tiles' overwrite
      mbar_arrive_expect_tx(&sm.bar_kq, 4 * HB);
      tma_load_3d(sm.K[0], &kmap, 0, kh, tok0, &sm.bar_kq);
      tma_load_3d(sm.K[1], &kmap, 64, kh, tok0, &sm.bar_kq);
      tma_load_3d(sm.Q[0], &qmap, 0, kh, tok0, &sm.bar_kq);
      tma_load_3d(sm.Q[1], &qmap, 64, kh, tok0, &sm.bar_kq);
      mbar_arrive_expect_tx(&sm.bar_v, 2 * HB);
      tma_load_3d(sm.V[0], &vmap, 0, h, tok0, &sm.bar_v);
      tma_load_3d(sm.V[1], &vmap, 64, h, tok0, &sm.bar_v);
    }
    for (int t = tid; t < C; t += NT) {
      const bool in = t < L;
      const size_t gi = ((size_t)tok0 + (in ? t : 0)) * p.hv + h;
      cp_async4(&sm.gRaw[t], p.g + gi, in ? 4 : 0);
      cp_async4(&sm.bRaw[t], p.beta + gi, in ? 4 : 0);
    }
    cp_async_commit();
    cp_async_wait<0>();
    ok = mbar_wait(&sm.bar_kq, it & 1) && ok;
    __syncthreads();

    // in-block inclusive cumsum of g (padding contributes 0), e^G, e^(G_C - G), beta --
    // warp 0, while the Gram products (which do not need the gates) run
    if (warp == 0) {
      constexpr int E = (C + 31) / 32;
      float gv[E], bv[E], run = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int t = lane * E + e;
        gv[e] = t < C ? sm.gRaw[t] : 0.f;
        bv[e] = t < C ? sm.bRaw[t] : 0.f;
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
      const float gC = __shfl_sync(0xffffffffu, incl, 31);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int t = lane * E + e;
        if (t < C) {
          const float G = gv[e] + excl;
          sm.G[t] = G;
          sm.EG[t] = __expf(G);
          sm.ED[t] = __expf(gC - G);
          sm.B[t] = bv[e];
        }
      }
    }

    // ---- raw Grams on tensor cores (bf16 inputs, exact products): warps 0-3 K K^T,
    //      warps 4-7 Q K^T, each a balanced share of the causal 16x16 tiles (mt, np<=mt):
    //      tiles np0 .. np0+n0-1 of row mt0, plus tile (mt1, 0) for one warp at C = 64
    const int prod = warp >> 2, qw = warp & 3;
    int mt0 = 0, np0 = 0, n0 = 0, mt1 = -1;
    if (C == 64) {  // row 3: {0,1}, {2,3}; row 2: {0,1,2}; row 1: {0,1} and row 0: {0}
      mt0 = qw < 2 ? 3 : (qw == 2 ? 2 : 1);
      np0 = qw == 1 ? 2 : 0;
      n0 = qw == 2 ? 3 : 2;
      if (qw == 3) mt1 = 0;
    } else if (C == 32) {  // row 1: {0}, {1}; row 0: {0}
      mt0 = qw < 2 ? 1 : 0;
      np0 = qw == 1 ? 1 : 0;
      n0 = qw < 3 ? 1 : 0;
    } else {
      n0 = qw == 0 ? 1 : 0;
    }
    float ga[6][4];
#pragma unroll
    for (int u = 0; u < 6; ++u)
#pragma unroll
      for (int e = 0; e < 4; ++e) ga[u][e] = 0.f;
    {
      const char *Asrc = prod ? sm.Q[0] : sm.K[0];
#pragma unroll
      for (int ks = 0; ks < kD / 16; ++ks) {
        const int hf = ks >> 2, kk = 16 * (ks & 3);  // key half, key offset in it
        if (n0 > 0) {
          uint32_t a[4];
          lda_tile<128>(a, Asrc + hf * HB, 16 * mt0, kk, lane);
#pragma unroll
          for (int u = 0; u < 3; ++u) {
            if (u < n0) {
              uint32_t b[4];
              ldb_nk<128>(b, sm.K[hf], 16 * (np0 + u), kk, lane);
              mma_bf16(ga[2 * u], a, b[0], b[1]);
              mma_bf16(ga[2 * u + 1], a, b[2], b[3]);
            }
          }
        }
        if (mt1 >= 0) {
          uint32_t a[4], b[4];
          lda_tile<128>(a, Asrc + hf * HB, 16 * mt1, kk, lane);
          ldb_nk<128>(b, sm.K[hf], 0, kk, lane);
          mma_bf16(ga[4], a, b[0], b[1]);
          mma_bf16(ga[5], a, b[2], b[3]);
        }
      }
    }
    __syncthreads();  // gates ready

    // ---- decay masks.  N = beta_t e^(G_t - G_j) k_t.k_j (j < t): fp32 for the diagonal
    //      blocks, -N in fp16 below them.  A = e^(G_t - G_j) q_t.k_j (j <= t): fp16 to the slot.
    {
      // this warp's tiles, their gates and decays read first (registers), then the masked
      // values, then the stores -- so that no gate read waits behind a store
      int tmt[3], tnp[3];
      bool has[3];
#pragma unroll
      for (int u = 0; u < 3; ++u) {
        has[u] = u < n0 || (u == 2 && mt1 >= 0);
        tmt[u] = u < n0 ? mt0 : mt1;
        tnp[u] = u < n0 ? np0 + u : 0;
      }
      float xv[3][2][2][2];  // [tile][half][row half][pair element]
#pragma unroll
      for (int u = 0; u < 3; ++u) {
        if (!has[u]) continue;
        float gt[2], bt[2], gj[2][2];
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          gt[hr] = sm.G[16 * tmt[u] + gid + 8 * hr];
          bt[hr] = sm.B[16 * tmt[u] + gid + 8 * hr];
        }
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          gj[half][0] = sm.G[16 * tnp[u] + 8 * half + 2 * tig];
          gj[half][1] = sm.G[16 * tnp[u] + 8 * half + 2 * tig + 1];
        }
#pragma unroll
        for (int half = 0; half < 2; ++half)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int t = 16 * tmt[u] + gid + 8 * hr, j = 16 * tnp[u] + 8 * half + 2 * tig;
            const float v0 = ga[2 * u + half][2 * hr], v1 = ga[2 * u + half][2 * hr + 1];
            const float d0 = decay_exp(gt[hr] - gj[half][0]), d1 = decay_exp(gt[hr] - gj[half][1]);
            if (prod == 0) {
              xv[u][half][hr][0] = (j < t) ? bt[hr] * d0 * v0 : 0.f;
              xv[u][half][hr][1] = (j + 1 < t) ? bt[hr] * d1 * v1 : 0.f;
            } else {
              xv[u][half][hr][0] = (j <= t) ? d0 * v0 : 0.f;
              xv[u][half][hr][1] = (j + 1 <= t) ? d1 * v1 : 0.f;
            }
          }
      }
#pragma unroll
      for (int u = 0; u < 3; ++u) {
        if (!has[u]) continue;
#pragma unroll
        for (int half = 0; half < 2; ++half)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int t = 16 * tmt[u] + gid + 8 * hr, j = 16 * tnp[u] + 8 * half + 2 * tig;
            const float x0 = xv[u][half][hr][0], x1 = xv[u][half][hr][1];
            if (prod == 0) {
              if (tmt[u] == tnp[u]) {
                sm.Nd[tmt[u]][t - 16 * tmt[u]][j - 16 * tnp[u]] = x0;
                sm.Nd[tmt[u]][t - 16 * tmt[u]][j + 1 - 16 * tnp[u]] = x1;
              } else {
                *reinterpret_cast<uint32_t *>(sm.N16 + t * RC + 2 * j) = pack_f16(-x0, -x1);
              }
            } else if (LAYOUT == 0) {
              *reinterpret_cast<uint32_t *>(a_out + t * RC + 2 * j) = pack_f16(x0, x1);
            } else {
              *reinterpret_cast<uint32_t *>(slot + kTsAt + tc::at_off(t, j)) = pack_f16(x0, x1);
            }
          }
      }
    }
    if (LAYOUT == 1) {
      // the A tile's 16x16 blocks above the diagonal (never computed) are zero: 6 tiles of
      // 16 rows x 8 column pairs
      for (int e = tid; e < 6 * 128; e += NT) {
        const int tile = e >> 7, row = (e >> 3) & 15, pr = e & 7;
        const int mt = tile < 3 ? 0 : (tile < 5 ? 1 : 2);
        const int np = tile < 3 ? 1 + tile : (tile < 5 ? tile - 1 : 3);
        *reinterpret_cast<uint32_t *>(slot + kTsAt + tc::at_off(16 * mt + row, 16 * np + 2 * pr)) = 0u;
      }
    }
    __syncthreads();

    // ---- T_ii = (I + N_ii)^-1 for the 16x16 diagonal blocks in fp32: one column per
    //      thread, forward substitution.  Meanwhile the other threads write the decays
    //      (and for LAYOUT 1 the fp16 operands K and diag(e^G) Q).
    if (tid < C) {
      const int blk = tid >> 4, cc = tid & 15;
      float x[16];
      unit_tril_inverse_col(&sm.Nd[blk][0][0], 17, cc, x);
#pragma unroll
      for (int r = 0; r < 16; ++r)
        *reinterpret_cast<__half *>(sm.T16[blk] + r * 48 + 2 * cc) = __float2half_rn(x[r]);
    } else {
      float *dec = LAYOUT == 0 ? dec_out : reinterpret_cast<float *>(slot + kTsDec);
      for (int t = tid - C; t < C; t += NT - C) {
        dec[t] = sm.G[t];
        dec[C + t] = sm.EG[t];
        dec[2 * C + t] = sm.ED[t];
      }
      if (LAYOUT == 1) {
        // 16 bytes (8 keys of one token) per step, consecutive threads on consecutive
        // tokens: each warp stores 512 contiguous bytes of the core-matrix layout
        for (int e = tid - C; e < 2 * C * 16; e += NT - C) {
          const int which = e >> 10, t = e & (C - 1), gq = (e >> 6) & 15;
          const uint4 raw = *reinterpret_cast<const uint4 *>(sw_el(which ? sm.Q[0] : sm.K[0], HB, t, 8 * gq));
          const float sc = which ? sm.EG[t] : 1.f;
          const uint32_t in4[4] = {raw.x, raw.y, raw.z, raw.w};
          uint32_t out4[4];
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2)
            out4[e2] = pack_f16(__uint_as_float(in4[e2] << 16) * sc, __uint_as_float(in4[e2] & 0xffff0000u) * sc);
          *reinterpret_cast<uint4 *>(slot + (which ? kTsQt : kTsK) + tc::t64_off(t, 8 * gq)) =
              make_uint4(out4[0], out4[1], out4[2], out4[3]);
        }
      }
    }
    ok = mbar_wait(&sm.bar_v, it & 1) && ok;  // v has landed
    __syncthreads();

    // ---- [W U] = (I + N)^-1 [diag(beta e^G) K  diag(beta) V] by blocked forward
    //      substitution over the 16-token blocks, X_i = T_ii (R_i - sum_{j<i} N_ij X_j),
    //      transposed so that each warp solves its own 32 columns without exchange:
    //      X_i^T = (R_i^T - sum_j X_j^T N_ij^T) T_ii^T.  Warps 0-3: W (32 keys each),
    //      warps 4-7: U (32 value columns each).  Each solved tile goes back to token rows
    //      by a transposing stmatrix: -W into the q tile (no longer needed), U in place
    //      over the rows of v it was solved from (only this warp reads those columns).
    {
      const int kind = warp >> 2, c0 = 32 * (warp & 3);
      const char *X = kind ? sm.V[0] : sm.K[0];
      char *xo = kind ? sm.V[0] : sm.Q[0];
      const float sgn = kind ? 1.f : -1.f;
      uint32_t Xf[MT][2][4];  // fp16 A fragments of the solved blocks X_j^T
#pragma unroll
      for (int i = 0; i < MT; ++i) {
        // R_i^T (cols x tokens) straight in the accumulator layout: ldmatrix.trans of the
        // bf16 rows gives lane (gid, tig) the pair (t = 2tig, 2tig + 1; col = gid)
        float acc[2][2][4];
        {
          float sc[2][2];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int t = 16 * i + 8 * nt + 2 * tig + e;
              sc[nt][e] = kind ? sm.B[t] : sm.B[t] * sm.EG[t];
            }
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            uint32_t r4[4];  // (nt 0, cols lo), (nt 0, cols hi), (nt 1, lo), (nt 1, hi)
            ldsm_x4_t(r4, sw_el(X, HB, 16 * i + (lane & 7) + 8 * (lane >> 4), c0 + 16 * mt + 8 * ((lane >> 3) & 1)));
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int hi = 0; hi < 2; ++hi) {
                const uint32_t w = r4[2 * nt + hi];
                acc[mt][nt][2 * hi] = sc[nt][0] * __uint_as_float(w << 16);
                acc[mt][nt][2 * hi + 1] = sc[nt][1] * __uint_as_float(w & 0xffff0000u);
              }
          }
        }
#pragma unroll
        for (int j = 0; j < i; ++j) {
          uint32_t b[4];
          ldb_nk_p<RC>(b, sm.N16, 16 * i, 16 * j, lane);  // B[k=j][n=t] = -N[t][j]
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            mma_f16(acc[mt][0], Xf[j][mt], b[0], b[1]);
            mma_f16(acc[mt][1], Xf[j][mt], b[2], b[3]);
          }
        }
        uint32_t y[2][4], bt[4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
          acc_to_f16(acc[mt][0], acc[mt][1], 1.f, 1.f, 1.f, 1.f, y[mt]);
        ldb_nk_p<48>(bt, sm.T16[i], 0, 0, lane);  // B[k=j'][n=t'] = T_ii[t'][j']
        float out[2][2][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) out[mt][nt][e] = 0.f;
            mma_f16(out[mt][nt], y[mt], bt[2 * nt], bt[2 * nt + 1]);
          }
        if (LAYOUT == 0) __syncwarp();  // every lane's reads of R_i are done before the in-place stores
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          if (LAYOUT == 0) {
            // 8x8 matrices (columns c0 + 16mt + 8hr.., tokens 16i + 8nt..), m = 2nt + hr,
            // stored transposed to rows 16i + 8nt + r, columns c0 + 16mt + 8hr
            const int m = lane >> 3, r = lane & 7;
            stsm_x4_t(sw_el(xo, HB, 16 * i + 8 * (m >> 1) + r, c0 + 16 * mt + 8 * (m & 1)),
                      pack_f16(sgn * out[mt][0][0], sgn * out[mt][0][1]),
                      pack_f16(sgn * out[mt][0][2], sgn * out[mt][0][3]),
                      pack_f16(sgn * out[mt][1][0], sgn * out[mt][1][1]),
                      pack_f16(sgn * out[mt][1][2], sgn * out[mt][1][3]));
          } else {
            // W^T (wt_off) or U^T ([col][token], 144-byte rows) straight to the slot:
            // lane (gid, tig) holds columns c0 + 16mt + gid (+8), tokens 16i + 8nt + 2tig, +1
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int hr = 0; hr < 2; ++hr) {
                const int col = c0 + 16 * mt + gid + 8 * hr, t = 16 * i + 8 * nt + 2 * tig;
                const uint32_t val = pack_f16(out[mt][nt][2 * hr], out[mt][nt][2 * hr + 1]);
                *reinterpret_cast<uint32_t *>(slot + (kind ? kTsUt + col * 144 + 2 * t : kTsWt + tc::wt_off(t, col))) = val;
              }
          }
          if (i + 1 < MT) acc_to_f16(out[mt][0], out[mt][1], 1.f, 1.f, 1.f, 1.f, Xf[i][mt]);
        }
      }
    }
    if (LAYOUT == 1) continue;  // (the next block's first barrier orders the smem reuse)
    __syncthreads();
    // ---- -W and U to the slot in fragment order (16-byte lane runs, coalesced stores)
    for (int e = tid; e < 2 * C * 16; e += NT) {
      const int which = e / (C * 16), f = e % (C * 16), ln = f & 31, g = ln >> 2, tg = ln & 3;
      uint4 x;
      if (!which) {  // WN group (w, s, rh) = (f >> 8, (f >> 6) & 3, (f >> 5) & 1)
        const int w = f >> 8, sp = (f >> 6) & 3, rh = (f >> 5) & 1;
        x = *reinterpret_cast<const uint4 *>(sw_el(sm.Q[0], HB, 16 * w + g + 8 * rh, 32 * sp + 8 * tg));
      } else {       // U group (b, w) = ((f >> 5) / MT, (f >> 5) % MT)
        const int w = (f >> 5) % MT, b = (f >> 5) / MT, r0 = 16 * w + g, c0 = 16 * b + 2 * tg;
        x.x = *reinterpret_cast<const uint32_t *>(sw_el(sm.V[0], HB, r0, c0));          // nt 0, rh 0
        x.y = *reinterpret_cast<const uint32_t *>(sw_el(sm.V[0], HB, r0 + 8, c0));      // nt 0, rh 1
        x.z = *reinterpret_cast<const uint32_t *>(sw_el(sm.V[0], HB, r0, c0 + 8));      // nt 1, rh 0
        x.w = *reinterpret_cast<const uint32_t *>(sw_el(sm.V[0], HB, r0 + 8, c0 + 8));  // nt 1, rh 1
      }
      *reinterpret_cast<uint4 *>((which ? u_out : wn_out) + 16 * f) = x;
    }
  }
  if (!ok) report_status(p.err, GDN_STATUS_WAIT_TIMEOUT);
}

// ================================================================== pass 2
// One CTA per (sequence, v-head, 16 value columns) walks the sequence's blocks in order.
//   producer warp: per block, bulk (TMA) copies of the slot's chain operands, a
//     tensor-map TMA of the block's k rows and, for the outputs, of its q rows and a bulk
//     copy of A, into a 3-stage shared-memory ring signalled on mbarriers.
//   chain warps 0-3: the state block S[:, cols] in fp32 registers for the whole sequence
//     (read from state_in once, written to state_out once), warp w holding keys
//     32w .. 32w+31.  Per block, for tokens 16w .. 16w+15 (w < C/16),
//       D = U - W S          (fragment-ordered -W and U, S from a shared fp16 snapshot),
//     D and D~ = diag(e^(G_C - G)) D go to shared memory (transposed), then each warp
//     updates its keys from the k rows as loaded,
//       S <- e^(G_C) S + K^T D~,
//     and writes its part of the next snapshot.
//   output warps 4-7: for tokens 16ow .. 16ow+15, O = diag(e^G) Q S + A D from the same
//     snapshot and the exchanged D, once D is published (so that their reads overlap the
//     state update, not the D product).
// Hand-offs between chain and output warps are named barriers over kOutBufs snapshot and
// D^T buffers, so that the output warps may trail the chain by up to two blocks (the
// chain overwrites the buffers of block c - 2 once their outputs are done); the ring's
// hand-offs are mbarriers with bounded waits (a wait that gives up reports
// GDN_STATUS_WAIT_TIMEOUT).
constexpr int kDVB = 16;  // value columns per CTA
constexpr int kChainWarps = 4, kOutWarps = 4;
constexpr int kChain = 32 * kChainWarps;
constexpr int kPair = 32 * (kChainWarps + kOutWarps);

// Named barriers of pass 2 (0 is __syncthreads)
constexpr int kOutBufs = 3;    // snapshot and D^T buffers shared with the output warps
constexpr int kBarChain = 1;   // the chain warps among themselves
constexpr int kBarSReady = 2;  // +c mod kOutBufs: snapshot S_c published (chain arrives, output waits)
constexpr int kBarDone = kBarSReady + kOutBufs;  // +c mod kOutBufs: output warps done with block c
constexpr int kBarDReady = kBarDone + kOutBufs;  // +c mod kOutBufs: D_c published (chain arrives)
static_assert(kBarDReady + kOutBufs <= 16, "named barriers 0-15");

// Byte offset of byte b of row r in a shared tile of RB-byte rows whose 16-byte granules
// are permuted per row (granule g stored at g ^ f(r), f(r) = 4 (r & 1) + ((r >> 1) & 3)):
// the fragment loads (eight lanes read four granules of two rows), ldmatrix (eight rows at
// one granule) and the stmatrix stores all touch eight distinct bank groups.
__device__ __forceinline__ int swz_row(int r, int RB, int b) {
  const int f = ((r & 1) << 2) | ((r >> 1) & 3);
  return r * RB + (((b >> 4) ^ f) << 4) + (b & 15);
}

// The chain's operands of one block, as copied from the slot (fragment order).
template <int C>
struct ChainStage {
  alignas(128) char WN[C * 256];        // -W
  alignas(128) char U[(C / 16) * 512];  // U of this CTA's 16 value columns
  alignas(16) float DEC[3 * C];         // G, e^G, e^(G_C - G)
};
// The block's k rows (the state update's operand).
template <int C>
struct alignas(1024) KStage {
  char K[2][C * 128];    // keys 0-63 | 64-127 (bf16, TMA 128-byte swizzle)
};
// The outputs' operands of one block.
template <int C>
struct alignas(1024) OutStage {
  char Q[2][C * 128];    // q rows, keys 0-63 | 64-127 (bf16, TMA 128-byte swizzle)
  alignas(128) char A[C * row_c(C)];
};

template <int C, int MODE>
struct RecSmem {
  static constexpr int NST = MODE == 0 ? 3 : 2;  // ring depth
  ChainStage<C> cs[NST];
  // snapshot and D^T buffers: kOutBufs with output warps (the chain overwrites those of
  // block c + 1 - kOutBufs while the output warps may still be on a later block), else two
  static constexpr int NSB = MODE == 0 ? kOutBufs : 2;
  alignas(128) char Sn[NSB][kDVB * 256];  // S^T (fp16) [16 value cols][128 keys], by c mod NSB
  alignas(128) char Dt[NSB][kDVB * 128];  // D^T (fp16) [16 value cols][C tokens], by c mod NSB
  alignas(128) char Dst[2][kDVB * 128];  // D~^T, D~ = diag(e^(G_C - G)) D (chain only), by parity
  alignas(16) float S32[kD][kDVB + 4];   // fp32 staging of the state block
  alignas(8) uint64_t full[NST], empty[NST];
};
// Shared memory of pass 2: RecSmem, then NST KStages, then (MODE 0) NST OutStages, each
// 1024-byte aligned from a 1024-aligned base.
template <int C, int MODE>
__host__ __device__ constexpr size_t rec_base_bytes() {
  return (sizeof(RecSmem<C, MODE>) + 1023) / 1024 * 1024;
}
template <int C, int MODE>
constexpr size_t rec_smem_bytes() {
  constexpr int NST = RecSmem<C, MODE>::NST;
  return 1024 + rec_base_bytes<C, MODE>() + NST * sizeof(KStage<C>) +
         (MODE == 0 ? NST * sizeof(OutStage<C>) : 0);  // + alignment slack
}

__device__ __forceinline__ void put4(uint32_t (&d)[4], uint4 x) {
  d[0] = x.x;
  d[1] = x.y;
  d[2] = x.z;
  d[3] = x.w;
}
// Chain warp w's snapshot part: S^T rows (value columns) 0-15, keys 32w .. 32w+31, fp16.
__device__ __forceinline__ void write_snapshot(const float (&Sa)[4][4], char *Sn, int w, int lane) {
  const int m = lane >> 3, r = lane & 7;
#pragma unroll
  for (int hf = 0; hf < 2; ++hf)  // matrices m = 2 (nt - 2hf) + rh: rows 8rh.., keys 32w + 8nt..
    stsm_x4(Sn + swz_row(8 * (m & 1) + r, 256, 2 * (32 * w + 8 * (2 * hf + (m >> 1)))),
            pack_f16(Sa[2 * hf][0], Sa[2 * hf][1]), pack_f16(Sa[2 * hf][2], Sa[2 * hf][3]),
            pack_f16(Sa[2 * hf + 1][0], Sa[2 * hf + 1][1]), pack_f16(Sa[2 * hf + 1][2], Sa[2 * hf + 1][3]));
}

// One block of a chain warp: D for its tokens, the exchange, its keys' state update and
// snapshot.  MODE 0: output warps share the snapshots and D through named barriers.
template <int C, int MODE>
__device__ __forceinline__ void chain_block(int c, const ChainStage<C> &st, const KStage<C> &kst,
                                            float (&Sa)[4][4], RecSmem<C, MODE> &sm, int w, int lane,
                                            bool dwork, bool with_u) {
  constexpr int NSB = RecSmem<C, MODE>::NSB;
  const int gid = lane >> 2, tig = lane & 3, par = c & 1, cur = c % NSB, nxt = (c + 1) % NSB;
  if (dwork) {
    // four independent accumulations per n-tile (key spans s), two products deep each
    float d[4][2][4];  // [key span][n-tile: value columns 8nt..][fragment]
#pragma unroll
    for (int g = 0; g < 4; ++g)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) d[g][nt][i] = 0.f;
    const char *Sn = sm.Sn[cur];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      uint32_t b0[4], b1[4], w0[4], w1[4];
      put4(b0, *reinterpret_cast<const uint4 *>(Sn + swz_row(gid, 256, 64 * s + 16 * tig)));
      put4(b1, *reinterpret_cast<const uint4 *>(Sn + swz_row(gid + 8, 256, 64 * s + 16 * tig)));
      put4(w0, *reinterpret_cast<const uint4 *>(st.WN + wn_off(w, s, 0, lane)));
      put4(w1, *reinterpret_cast<const uint4 *>(st.WN + wn_off(w, s, 1, lane)));
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const uint32_t a[4] = {w0[2 * e], w1[2 * e], w0[2 * e + 1], w1[2 * e + 1]};
        mma_f16(d[s][0], a, b0[2 * e], b0[2 * e + 1]);
        mma_f16(d[s][1], a, b1[2 * e], b1[2 * e + 1]);
      }
    }
    uint32_t u[4] = {0u, 0u, 0u, 0u};  // (nt, rh) = (0,0), (0,1), (1,0), (1,1)
    if (with_u) put4(u, *reinterpret_cast<const uint4 *>(st.U + (32 * w + lane) * 16));
    float D[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int rh = 0; rh < 2; ++rh) {
        const float2 uu = f16x2_to_float2(u[2 * nt + rh]);
        D[nt][2 * rh] = uu.x + ((d[0][nt][2 * rh] + d[1][nt][2 * rh]) + (d[2][nt][2 * rh] + d[3][nt][2 * rh]));
        D[nt][2 * rh + 1] = uu.y + ((d[0][nt][2 * rh + 1] + d[1][nt][2 * rh + 1]) +
                                    (d[2][nt][2 * rh + 1] + d[3][nt][2 * rh + 1]));
      }
    // D^T and D~^T: matrices m = 2nt + rh (tokens 16w + 8rh.., columns 8nt..) stored
    // transposed
    const int m = lane >> 3, r = lane & 7;
    const int doff = swz_row(8 * (m >> 1) + r, 128, 32 * w + 16 * (m & 1));
    stsm_x4_t(sm.Dt[cur] + doff, pack_f16(D[0][0], D[0][1]), pack_f16(D[0][2], D[0][3]),
              pack_f16(D[1][0], D[1][1]), pack_f16(D[1][2], D[1][3]));
    const float ed0 = st.DEC[2 * C + 16 * w + gid], ed1 = st.DEC[2 * C + 16 * w + gid + 8];
    stsm_x4_t(sm.Dst[par] + doff, pack_f16(ed0 * D[0][0], ed0 * D[0][1]),
              pack_f16(ed1 * D[0][2], ed1 * D[0][3]), pack_f16(ed0 * D[1][0], ed0 * D[1][1]),
              pack_f16(ed1 * D[1][2], ed1 * D[1][3]));
  }
  bar_sync(kBarChain, kChain);
  if (MODE == 0) bar_arrive(kBarDReady + cur, kPair);

  // S^T <- e^(G_C) S^T + D~^T K over keys 32w .. 32w+31 (the k rows as loaded, bf16 ->
  // fp16 in registers): two accumulations by token step parity, summed with the scaled
  // state at the end
  float X[2][4][4];
#pragma unroll
  for (int s = 0; s < 2; ++s)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) X[s][nt][i] = 0.f;
  const char *Kh = kst.K[w >> 1];  // keys 64 (w >> 1) .. +63
#pragma unroll
  for (int e = 0; e < C / 16; ++e) {
    uint32_t a[4];
    ldsm_x4(a, sm.Dst[par] + swz_row((lane & 7) + ((lane >> 3) & 1) * 8, 128, 2 * (16 * e + (lane >> 4) * 8)));
#pragma unroll
    for (int pr = 0; pr < 2; ++pr) {
      uint32_t b[4];  // n-tiles keys 32w + 16pr .. +7 (b[0], b[1]) and +8 .. +15 (b[2], b[3])
      ldb_kn<128>(b, Kh, 16 * e, 32 * (w & 1) + 16 * pr, lane);
#pragma unroll
      for (int i = 0; i < 4; ++i) b[i] = bf16x2_to_f16x2(b[i]);
      mma_f16(X[e & 1][2 * pr], a, b[0], b[1]);
      mma_f16(X[e & 1][2 * pr + 1], a, b[2], b[3]);
    }
  }
  const float gam = st.DEC[2 * C - 1];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) Sa[nt][i] = fmaf(gam, Sa[nt][i], X[0][nt][i] + X[1][nt][i]);
  // S_{c+1} into the buffer of S_{c+1-NSB} once the output warps are done with that block
  if (MODE == 0 && c + 1 >= NSB) bar_sync(kBarDone + nxt, kPair);
  write_snapshot(Sa, sm.Sn[nxt], w, lane);
  bar_sync(kBarChain, kChain);
  if (MODE == 0) bar_arrive(kBarSReady + nxt, kPair);
}

template <int C, typename TO>
__device__ __forceinline__ void out_block(int c, const ChainStage<C> &cst, const OutStage<C> &ost,
                                          RecSmem<C, 0> &sm, int ow, int lane, TO *o, int tok0,
                                          int L, int hv, int h, int blk) {
  constexpr int RC = row_c(C);
  const int gid = lane >> 2, tig = lane & 3, cur = c % kOutBufs;
  const bool work = 16 * ow < C;
  bar_sync(kBarSReady + cur, kPair);
  // Q S only once D is formed: the chain's D = U - W S reads the same snapshot and the
  // block's operands, and the two would otherwise share shared memory on the chain's
  // critical phase; after it the output warps overlap the state update instead
  bar_sync(kBarDReady + cur, kPair);
  float R[2][4];
  if (work) {
    float r2[2][2][4];  // [k-step parity][n-tile][fragment]
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) r2[e][nt][i] = 0.f;
    const char *Sn = sm.Sn[cur];
#pragma unroll
    for (int ks = 0; ks < kD / 16; ++ks) {
      uint32_t a[4], b[4];
      lda_tile<128>(a, ost.Q[ks >> 2], 16 * ow, 16 * (ks & 3), lane);
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = bf16x2_to_f16x2(a[i]);
      ldsm_x4(b, Sn + swz_row((lane & 7) + (lane >> 4) * 8, 256, 2 * (16 * ks + ((lane >> 3) & 1) * 8)));
      mma_f16(r2[ks & 1][0], a, b[0], b[1]);
      mma_f16(r2[ks & 1][1], a, b[2], b[3]);
    }
    const float e0 = cst.DEC[C + 16 * ow + gid], e1 = cst.DEC[C + 16 * ow + gid + 8];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) R[nt][i] = (r2[0][nt][i] + r2[1][nt][i]) * (i < 2 ? e0 : e1);
  }
  if (work) {
    // O += A D over the causal part (A is zero above the diagonal)
    for (int ks = 0; ks <= ow; ++ks) {
      uint32_t a[4], b[4];
      lda_p<RC>(a, ost.A, 16 * ow, 16 * ks, lane);
      ldsm_x4(b, sm.Dt[cur] + swz_row((lane & 7) + (lane >> 4) * 8, 128, 2 * (16 * ks + ((lane >> 3) & 1) * 8)));
      mma_f16(R[0], a, b[0], b[1]);
      mma_f16(R[1], a, b[2], b[3]);
    }
#pragma unroll
    for (int rh = 0; rh < 2; ++rh) {
      const int t = 16 * ow + gid + 8 * rh;
      if (t < L) {
        TO *dst = o + ((size_t)(tok0 + t) * hv + h) * kD + kDVB * blk + 2 * tig;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          if constexpr (sizeof(TO) == 4) {
            *reinterpret_cast<float2 *>(dst + 8 * nt) = make_float2(R[nt][2 * rh], R[nt][2 * rh + 1]);
          } else {
            *reinterpret_cast<__nv_bfloat162 *>(dst + 8 * nt) =
                __floats2bfloat162_rn(R[nt][2 * rh], R[nt][2 * rh + 1]);
          }
        }
      }
    }
  }
  __syncwarp();
  bar_arrive(kBarDone + cur, kPair);
}

// MODE 0: pass 2 (state chain and outputs): 4 chain + 4 output warps + 1 producer warp.
// MODE 1: the sequence split's state chains: CTAs [0, heads * 8) run from state_in, the
// next heads * 8 from state_in2 with U taken as zero (-> state_out2); 4 chain warps + the
// producer, no outputs.
template <int C, typename TO, int MODE>
__global__ void __launch_bounds__(MODE == 0 ? kPair + 32 : kChain + 32, C == 64 ? 1 : 2)
    recur_kernel(ChunkParams p, const __grid_constant__ CUtensorMap kmap,
                 const __grid_constant__ CUtensorMap qmap) {
  constexpr int NB = kD / kDVB, MT = C / 16, RC = row_c(C);
  constexpr int NT = MODE == 0 ? kPair + 32 : kChain + 32;
  constexpr int NST = RecSmem<C, MODE>::NST, PW = NT / 32 - 1;  // ring depth, producer warp
  constexpr size_t SB = slot_stride(C, false);
  constexpr uint32_t kChainTx = (uint32_t)(C * 256 + MT * 512 + 12 * C + 2 * C * 128);
  constexpr uint32_t kOutTx = (uint32_t)(2 * C * 128 + C * RC);
  extern __shared__ unsigned char smem_raw[];
  unsigned char *base = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  RecSmem<C, MODE> &sm = *reinterpret_cast<RecSmem<C, MODE> *>(base);
  KStage<C> *ks = reinterpret_cast<KStage<C> *>(base + rec_base_bytes<C, MODE>());
  OutStage<C> *os = reinterpret_cast<OutStage<C> *>(ks + NST);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  long long b = blockIdx.x;
  bool maps = false;
  if (MODE == 1) {
    const long long half = (long long)p.num_seqs * p.hv * NB;
    maps = b >= half;
    if (maps) b -= half;
  }
  const int blk = (int)(b % NB);
  const int nh = (int)(b / NB);
  const int n = nh / p.hv;
  const int h = nh - n * p.hv;
  const int kh = h / (p.hv / p.hk);
  const float *s_in = maps ? p.state_in2 : p.state_in;
  float *s_out = maps ? p.state_out2 : p.state_out;

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], MODE == 0 ? 1 + kOutWarps : 1);  // the chain group, each output warp
    }
    mbar_fence_init();
  }
  // Launched as a programmatic dependent of the kernel before it (pass 1): the set-up above
  // overlaps that kernel's tail; nothing in global memory is read before it has completed
  // and its writes are visible.
  asm volatile("griddepcontrol.wait;\n" ::: "memory");

  int bos, eos;
  seq_range(p.cu_seqlens, n, p.total_tokens, bos, eos);
  const int nchunks = (eos - bos + C - 1) / C;
  const size_t sbase = ((size_t)n * p.hv + h) * kD * kD + blk * kDVB;
  const char *slot0 = p.slot_ws + ((size_t)h * p.nslots + slot_index(bos, C, n, 0)) * SB;
  // state block S[:, blk*16 .. +16) -> fp32 staging (coalesced 64-byte rows)
  for (int e = tid; e < kD * kDVB / 4; e += NT) {
    const int i = e / (kDVB / 4), c4 = e % (kDVB / 4);
    const float4 val = s_in ? *reinterpret_cast<const float4 *>(s_in + sbase + (size_t)i * kD + 4 * c4)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
    *reinterpret_cast<float4 *>(&sm.S32[i][4 * c4]) = val;
  }
  __syncthreads();

  if (warp == PW) {
    // ---- producer: each block's operands into the ring
    if (lane == 0) {
      bool ok = true;
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % NST;
        if (c >= NST) ok = mbar_wait(&sm.empty[s], ((c / NST) - 1) & 1) && ok;
        const char *src = slot0 + (size_t)c * SB;
        ChainStage<C> &cs = sm.cs[s];
        mbar_arrive_expect_tx(&sm.full[s], kChainTx + (MODE == 0 ? kOutTx : 0));
        bulk_g2s(cs.WN, src, C * 256, &sm.full[s]);
        bulk_g2s(cs.U, src + slot_u_off(C) + u_off<C>(blk, 0, 0), MT * 512, &sm.full[s]);
        bulk_g2s(cs.DEC, src + slot_dec_off(C), 12 * C, &sm.full[s]);
        tma_load_3d(ks[s].K[0], &kmap, 0, kh, bos + c * C, &sm.full[s]);
        tma_load_3d(ks[s].K[1], &kmap, 64, kh, bos + c * C, &sm.full[s]);
        if (MODE == 0) {
          tma_load_3d(os[s].Q[0], &qmap, 0, kh, bos + c * C, &sm.full[s]);
          tma_load_3d(os[s].Q[1], &qmap, 64, kh, bos + c * C, &sm.full[s]);
          bulk_g2s(os[s].A, src + slot_a_off(C), C * RC, &sm.full[s]);
        }
      }
      // every copy is consumed (full waited on) before the CTA's final barrier
      if (!ok) report_status(p.err, GDN_STATUS_WAIT_TIMEOUT);
    }
  } else if (warp < kChainWarps) {
    const int w = warp;
    const bool dwork = w < MT;
    float Sa[4][4];  // S^T[j][i], j = gid (+8), i = 32w + 8nt + 2tig (+1)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) Sa[nt][e] = sm.S32[32 * w + 8 * nt + 2 * tig + (e & 1)][gid + 8 * (e >> 1)];
    write_snapshot(Sa, sm.Sn[0], w, lane);
    bar_sync(kBarChain, kChain);
    if (MODE == 0) bar_arrive(kBarSReady + 0, kPair);
    bool ok = true;
#pragma unroll 1
    for (int c = 0; c < nchunks; ++c) {
      const int s = c % NST;
      ok = mbar_wait(&sm.full[s], (c / NST) & 1) && ok;
      chain_block<C, MODE>(c, sm.cs[s], ks[s], Sa, sm, w, lane, dwork, !maps);
      if (tid == 0) mbar_arrive(&sm.empty[s]);  // all chain warps are past the barrier
    }
    if (MODE == 0)  // the output warps' last blocks
      for (int c = max(0, nchunks + 1 - kOutBufs); c < nchunks; ++c) bar_sync(kBarDone + c % kOutBufs, kPair);
    if (!ok && lane == 0) report_status(p.err, GDN_STATUS_WAIT_TIMEOUT);
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sm.S32[32 * w + 8 * nt + 2 * tig + (e & 1)][gid + 8 * (e >> 1)] = Sa[nt][e];
  } else if (MODE == 0) {
    const int ow = warp - kChainWarps;
    TO *o = static_cast<TO *>(p.o);
    bool ok = true;
#pragma unroll 1
    for (int c = 0; c < nchunks; ++c) {
      const int s = c % NST;
      ok = mbar_wait(&sm.full[s], (c / NST) & 1) && ok;
      const int tok0 = bos + c * C;
      out_block<C, TO>(c, sm.cs[s], os[s], *reinterpret_cast<RecSmem<C, 0> *>(&sm), ow, lane, o, tok0,
                       min(C, eos - tok0), p.hv, h, blk);
      if (lane == 0) mbar_arrive(&sm.empty[s]);
    }
    bar_sync(kBarSReady + nchunks % kOutBufs, kPair);
    if (!ok && lane == 0) report_status(p.err, GDN_STATUS_WAIT_TIMEOUT);
  }
  __syncthreads();
  for (int e = tid; e < kD * kDVB / 4; e += NT) {
    const int i = e / (kDVB / 4), c4 = e % (kDVB / 4);
    *reinterpret_cast<float4 *>(s_out + sbase + (size_t)i * kD + 4 * c4) =
        *reinterpret_cast<const float4 *>(&sm.S32[i][4 * c4]);
  }
}

// cuTensorMapEncodeTiled from the driver, looked up once (no link against libcuda).
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// Tensor map of a [T, H, 128] bf16 tensor (q, k or v) for boxes of 64 features x 1 head x
// C tokens, 128-byte swizzle (rows past T read as zero).
cudaError_t tile_map(CUtensorMap *map, const void *x, int total_tokens, int heads, int C) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)heads, (cuuint64_t)total_tokens};
  const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)heads * kD * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)C};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(x), dims, strides,
                         box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The q, k, v tile maps of a call (left zero without tokens: no block, no load).
struct TileMaps {
  CUtensorMap q, k, v;
};
template <int C>
cudaError_t make_tile_maps(TileMaps &m, const ChunkParams &p) {
  memset(&m, 0, sizeof(m));
  if (p.total_tokens <= 0) return cudaSuccess;
  cudaError_t err = tile_map(&m.q, p.q, p.total_tokens, p.hk, C);
  if (err == cudaSuccess) err = tile_map(&m.k, p.k, p.total_tokens, p.hk, C);
  if (err == cudaSuccess) err = tile_map(&m.v, p.v, p.total_tokens, p.hv, C);
  return err;
}

template <int C, typename TO, int MODE>
cudaError_t launch_recur(const ChunkParams &p, const TileMaps &m, long long heads, cudaStream_t stream) {
  constexpr size_t smem = rec_smem_bytes<C, MODE>();
  cudaError_t err = cudaFuncSetAttribute(recur_kernel<C, TO, MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const unsigned grid = (unsigned)((MODE == 1 ? 2 : 1) * heads * (kD / kDVB));
  // a programmatic dependent launch: the CTAs may start (and set up their barriers) as
  // the kernel before them drains; the kernel waits for its completion before any read
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(MODE == 0 ? kPair + 32 : kChain + 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, recur_kernel<C, TO, MODE>, p, m.k, m.q);
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
  // pass-1 CTAs per (sequence, head): one per block up to about 8 CTAs per SM in total
  long long per_head = (8LL * sms + heads - 1) / heads;
  per_head = max(1LL, min(per_head, max(1LL, max_chunks)));

  TileMaps maps;
  err = make_tile_maps<C>(maps, p);
  if (err != cudaSuccess) return err;
  // both passes at C = 64 with tc_pass2: pass 2 on the tcgen05 tensor cores (one CTA per
  // chain) over slots in its operand layout; else the mma.sync pass 2 (recur_kernel)
  constexpr int LT = C == 64 ? 1 : 0;
  const bool tc2 = C == 64 && p.passes == 0 && p.tc_pass2;
  if (p.total_tokens > 0 && p.passes != 2 && p.passes != 3) {
    const size_t s1 = 1024 + sizeof(PrepSmem<C>);  // + alignment slack
    const unsigned grid = (unsigned)(heads * per_head);
    if (tc2) {
      err = cudaFuncSetAttribute(prep_kernel<C, LT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1);
      if (err == cudaSuccess)
        prep_kernel<C, LT><<<grid, kPrepThreads, s1, stream>>>(p, (int)per_head, maps.k, maps.q, maps.v);
    } else {
      err = cudaFuncSetAttribute(prep_kernel<C, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1);
      if (err == cudaSuccess)
        prep_kernel<C, 0><<<grid, kPrepThreads, s1, stream>>>(p, (int)per_head, maps.k, maps.q, maps.v);
    }
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  if (tc2) return launch_tc_chain(p, stream);
  if (p.passes == 1) return cudaSuccess;
  if (p.passes == 3) return launch_recur<C, float, 1>(p, maps, heads, stream);
  return p.o_fp32 ? launch_recur<C, float, 0>(p, maps, heads, stream)
                  : launch_recur<C, __nv_bfloat16, 0>(p, maps, heads, stream);
}

}  // namespace

size_t chunk_workspace_bytes(int total_tokens, int num_seqs, int hv, int chunk, bool tc) {
  const size_t slots = (size_t)hv * ((size_t)total_tokens / chunk + num_seqs);
  return 256 + slots * slot_stride(chunk, tc);
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
