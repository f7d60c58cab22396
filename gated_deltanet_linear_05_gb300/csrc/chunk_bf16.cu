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
//   pass 1 (prep_kernel, one CTA per (block, v-head), all in parallel): G, the
//     decay-masked Grams, the inverses T_ii = (I + N_ii)^-1 of the 16x16 diagonal blocks
//     of I + N by forward substitution, and W and U by blocked forward substitution
//     over the 16-token blocks, X_i = T_ii (R_i - sum_{j<i} N_ij X_j) -- the same
//     triangular solve as the block inverse of the page, applied to the right-hand
//     sides instead of forming (I + N)^-1.  Each block's -W, K~^T = (diag(e^(G_C - G)) K)^T,
//     A, U and decays go to its own workspace slot, in the orientation pass 2 loads
//     straight into its tensor-core fragments.
//   pass 2 (chain_kernel, one CTA per (sequence, v-head, 16 value columns)): walks the
//     blocks of the sequence in order with the state block S[:, cols] in fp32 registers
//     (read from state_in once, written to state_out once): D = U - W S and
//     S <- e^(G_C) S + K~^T D per block, exporting each block's S_c and D_c (fp16).
//   pass 3 (out_kernel, one CTA per (v-head, block), all in parallel): the block outputs
//     O = diag(e^G) Q S_c + A D_c.
// Tensor-core products (mma.sync) take fp16 operands with fp32 accumulation: bf16 q, k
// and v enter exactly (converted to fp16), the state, D, T, W, A and K~ are rounded to
// fp16 (11 significant bits) for the products only; the state itself, the sums and every
// decay are fp32.  Decay factors between two tokens are always the exp of a difference
// of cumsums.  A partly filled block is padded with g = 0, beta = 0 and zero q/k/v rows
// (token_valid), which leaves the state exactly as after the sequence's last token.
#include <cuda.h>
#include <string.h>

#include "common.cuh"
#include "internal.h"

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

// Contractions over the keys and over the tokens in pass 2 take the k index in a
// permuted order: in every span of 32 (for C = 16: 16) indices, lane (gid, tig) supplies
// the consecutive indices span + 8tig .. +7 (4tig .. +3), elements {4e, 4e+1} as the k
// pair (2tig, 2tig+1) and {4e+2, 4e+3} as (2tig+8, 2tig+9) of the span's k-step e.  A and
// B of every product use the same order, so the products are unchanged and each lane
// reads one contiguous run per row.
template <int C>
struct TokSpan {
  static constexpr int SPAN = C < 32 ? C : 32;  // tokens per span
  static constexpr int NSP = C / SPAN;          // spans per block
  static constexpr int KW = SPAN / 8;           // 32-bit words per lane and row run
  static constexpr int KS = SPAN / 16;          // k-steps per span
};

// Fragment order of the slot's -W, K~^T and U: the chain kernel loads each group of 32
// lane runs (512 bytes, or 256 for C = 16) with one coalesced warp instruction.  Groups,
// lane = 4 gid + tig:
//   WN (chain warp w < C/16, key span s < 4, row half rh): lane's run = -W row
//      16w + gid + 8rh, keys 32s + 8tig .. +7                                   (16 B)
//   KT (chain warp w < 4, key tile nt < 4, token span s): K~^T row 32w + 8nt + gid, the
//      lane's token run of span s                                              (4 KW B)
//   U  (value-column block b < 8, chain warp w < C/16): the words U[16w + gid + 8rh]
//      [16b + 8nt + 2tig, +1] for (nt, rh) = (0,0), (0,1), (1,0), (1,1)       (16 B)
__device__ __forceinline__ int wn_off(int w, int s, int rh, int lane) {
  return (((w * 4 + s) * 2 + rh) * 32 + lane) * 16;
}
template <int C>
__device__ __forceinline__ int kt_off(int w, int nt, int s, int lane) {
  using TS = TokSpan<C>;
  return (((w * 4 + nt) * TS::NSP + s) * 32 + lane) * (4 * TS::KW);
}
template <int C>
__device__ __forceinline__ int u_off(int b, int w, int lane) {
  return ((b * (C / 16) + w) * 32 + lane) * 16;
}
// ================================================================== pass 1

template <int C>
struct PrepSmem {
  alignas(16) char K[C * kP128];  // bf16 rows as loaded (rows past the end: zero)
  alignas(16) char Q[C * kP128];
  alignas(16) char V[C * kP128];
  float Nd[C / 16][16][17];       // diagonal 16x16 blocks of N (fp32)
  alignas(16) char N16[C * row_c(C)];     // -N (fp16) [t][j], blocks below the diagonal
  alignas(16) char T16[C / 16][16 * 48];  // fp16 T_ii = (I + N_ii)^-1, rows of 48 B
  float G[C], EG[C], ED[C], B[C];
  float gRaw[C], bRaw[C];
};

constexpr int kPrepThreads = 256;

template <int C>
__global__ void __launch_bounds__(kPrepThreads, 3) prep_kernel(ChunkParams p, int per_head) {
  constexpr int NT = kPrepThreads, MT = C / 16, RC = row_c(C);
  extern __shared__ __align__(128) unsigned char smem_raw[];
  PrepSmem<C> &sm = *reinterpret_cast<PrepSmem<C> *>(smem_raw);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int part = blockIdx.x % per_head;
  const int nh = blockIdx.x / per_head;
  const int n = nh / p.hv;
  const int h = nh - n * p.hv;
  const int kh = h / (p.hv / p.hk);
  const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(p.q);
  const __nv_bfloat16 *k = static_cast<const __nv_bfloat16 *>(p.k);
  const __nv_bfloat16 *v = static_cast<const __nv_bfloat16 *>(p.v);

  int bos, eos;
  seq_range(p.cu_seqlens, n, p.total_tokens, bos, eos);
  const int nchunks = (eos - bos + C - 1) / C;

#pragma unroll 1
  for (int c = part; c < nchunks; c += per_head) {
    const int tok0 = bos + c * C;
    const int L = min(C, eos - tok0);
    char *slot = p.slot_ws + ((size_t)h * p.nslots + slot_index(bos, C, n, c)) * slot_bytes(C);
    char *wn_out = slot, *kt_out = slot + slot_kt_off(C), *a_out = slot + slot_a_off(C);
    char *u_out = slot + slot_u_off(C);
    float *dec_out = reinterpret_cast<float *>(slot + slot_dec_off(C));
    __syncthreads();  // the previous block is done with shared memory

    // two copy groups: q, k and the gates (the Grams start on them), then v
    for (int e = tid; e < C * 16; e += NT) {
      const int r = e >> 4, gr = e & 15;
      const bool ok = r < L;
      const size_t tok = (size_t)tok0 + (ok ? r : 0);
      const int nb = ok ? 16 : 0;
      cp_async16(sm.K + r * kP128 + gr * 16, k + (tok * p.hk + kh) * kD + gr * 8, nb);
      cp_async16(sm.Q + r * kP128 + gr * 16, q + (tok * p.hk + kh) * kD + gr * 8, nb);
    }
    for (int t = tid; t < C; t += NT) {
      const bool ok = t < L;
      const size_t gi = ((size_t)tok0 + (ok ? t : 0)) * p.hv + h;
      cp_async4(&sm.gRaw[t], p.g + gi, ok ? 4 : 0);
      cp_async4(&sm.bRaw[t], p.beta + gi, ok ? 4 : 0);
    }
    cp_async_commit();
    for (int e = tid; e < C * 16; e += NT) {
      const int r = e >> 4, gr = e & 15;
      const bool ok = r < L;
      const size_t tok = (size_t)tok0 + (ok ? r : 0);
      cp_async16(sm.V + r * kP128 + gr * 16, v + (tok * p.hv + h) * kD + gr * 8, ok ? 16 : 0);
    }
    cp_async_commit();
    cp_async_wait<1>();
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
      const char *Asrc = prod ? sm.Q : sm.K;
#pragma unroll
      for (int ks = 0; ks < kD / 16; ++ks) {
        if (n0 > 0) {
          uint32_t a[4];
          lda_p<kP128>(a, Asrc, 16 * mt0, 16 * ks, lane);
#pragma unroll
          for (int u = 0; u < 3; ++u) {
            if (u < n0) {
              uint32_t b[4];
              ldb_nk_p<kP128>(b, sm.K, 16 * (np0 + u), 16 * ks, lane);
              mma_bf16(ga[2 * u], a, b[0], b[1]);
              mma_bf16(ga[2 * u + 1], a, b[2], b[3]);
            }
          }
        }
        if (mt1 >= 0) {
          uint32_t a[4], b[4];
          lda_p<kP128>(a, Asrc, 16 * mt1, 16 * ks, lane);
          ldb_nk_p<kP128>(b, sm.K, 0, 16 * ks, lane);
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
            } else {
              *reinterpret_cast<uint32_t *>(a_out + t * RC + 2 * j) = pack_f16(x0, x1);
            }
          }
      }
    }
    // the A tile's upper 16x16 blocks (never computed) are zero: MT (MT - 1) / 2 tiles of
    // 16 rows x 8 column pairs
    for (int e = tid; e < 64 * MT * (MT - 1); e += NT) {
      const int tile = e >> 7, row = (e >> 3) & 15, pr = e & 7;
      int mt = 0, np = 1, cnt = tile;  // tile -> (mt, np > mt), row-major over the upper part
      while (cnt >= MT - 1 - mt) {
        cnt -= MT - 1 - mt;
        ++mt;
      }
      np = mt + 1 + cnt;
      *reinterpret_cast<uint32_t *>(a_out + (16 * mt + row) * RC + 2 * (16 * np + 2 * pr)) = 0u;
    }
    __syncthreads();

    cp_async_wait<0>();  // v has landed (visible to all after the next barrier)
    // ---- T_ii = (I + N_ii)^-1 for the 16x16 diagonal blocks in fp32: one column per
    //      thread, forward substitution.  Meanwhile the other threads write the slot's
    //      K~^T = (diag(e^(G_C - G)) K)^T (fp16, in fragment order) and the decays.
    if (tid < C) {
      const int blk = tid >> 4, cc = tid & 15;
      float x[16];
      unit_tril_inverse_col(&sm.Nd[blk][0][0], 17, cc, x);
#pragma unroll
      for (int r = 0; r < 16; ++r)
        *reinterpret_cast<__half *>(sm.T16[blk] + r * 48 + 2 * cc) = __float2half_rn(x[r]);
    } else {
      const int t2 = tid - C, n2 = NT - C;
      using TS = TokSpan<C>;
      for (int e = t2; e < 4 * 4 * TS::NSP * 32; e += n2) {  // one lane run of K~^T each
        const int lane_ = e & 31, sp = (e >> 5) % TS::NSP, wn = (e >> 5) / TS::NSP;
        const int key = 8 * wn + (lane_ >> 2);  // 32w + 8nt + gid, wn = 4w + nt
        const int t0 = TS::SPAN * sp + (TS::SPAN / 4) * (lane_ & 3);
        // the token pairs are taken in an order rotated by the lane's token group, so that
        // the four groups of a warp read rows in four different bank groups (their runs
        // start 8 rows apart: with 272-byte rows, the same bank group)
        const int rot = (lane_ & 3) & (TS::KW - 1);
        uint32_t w[TS::KW];
#pragma unroll
        for (int u = 0; u < TS::KW; ++u) {
          const int t = t0 + 2 * ((u + rot) & (TS::KW - 1));
          const float k0 = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(sm.K + t * kP128 + 2 * key));
          const float k1 =
              __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(sm.K + (t + 1) * kP128 + 2 * key));
          w[u] = pack_f16(k0 * sm.ED[t], k1 * sm.ED[t + 1]);
        }
        uint32_t wo[TS::KW];  // back in token order: pair j was computed at step (j - rot)
#pragma unroll
        for (int j = 0; j < TS::KW; ++j) {
          uint32_t x = w[0];
#pragma unroll
          for (int u = 1; u < TS::KW; ++u)
            if (((u + rot) & (TS::KW - 1)) == j) x = w[u];
          wo[j] = x;
        }
        char *dst = kt_out + e * (4 * TS::KW);
        if constexpr (TS::KW == 4)
          *reinterpret_cast<uint4 *>(dst) = make_uint4(wo[0], wo[1], wo[2], wo[3]);
        else
          *reinterpret_cast<uint2 *>(dst) = make_uint2(wo[0], wo[1]);
      }
      for (int t = t2; t < C; t += n2) {
        dec_out[t] = sm.G[t];
        dec_out[C + t] = sm.EG[t];
      }
    }
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
      const char *X = kind ? sm.V : sm.K;
      char *xo = kind ? sm.V : sm.Q;
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
            ldsm_x4_t(r4, X + (16 * i + (lane & 7) + 8 * (lane >> 4)) * kP128 +
                              2 * (c0 + 16 * mt + 8 * ((lane >> 3) & 1)));
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
        __syncwarp();  // every lane's reads of R_i are done before the in-place stores
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          // 8x8 matrices (columns c0 + 16mt + 8hr.., tokens 16i + 8nt..), m = 2nt + hr,
          // stored transposed to rows 16i + 8nt + r, columns c0 + 16mt + 8hr
          const int m = lane >> 3, r = lane & 7;
          stsm_x4_t(xo + (16 * i + 8 * (m >> 1) + r) * kP128 + 2 * (c0 + 16 * mt + 8 * (m & 1)),
                    pack_f16(sgn * out[mt][0][0], sgn * out[mt][0][1]),
                    pack_f16(sgn * out[mt][0][2], sgn * out[mt][0][3]),
                    pack_f16(sgn * out[mt][1][0], sgn * out[mt][1][1]),
                    pack_f16(sgn * out[mt][1][2], sgn * out[mt][1][3]));
          if (i + 1 < MT) acc_to_f16(out[mt][0], out[mt][1], 1.f, 1.f, 1.f, 1.f, Xf[i][mt]);
        }
      }
    }
    __syncthreads();
    // ---- -W and U to the slot in fragment order (16-byte lane runs, coalesced stores)
    for (int e = tid; e < 2 * C * 16; e += NT) {
      const int which = e / (C * 16), f = e % (C * 16), ln = f & 31, g = ln >> 2, tg = ln & 3;
      uint4 x;
      if (!which) {  // WN group (w, s, rh) = (f >> 8, (f >> 6) & 3, (f >> 5) & 1)
        const int w = f >> 8, sp = (f >> 6) & 3, rh = (f >> 5) & 1;
        x = *reinterpret_cast<const uint4 *>(sm.Q + (16 * w + g + 8 * rh) * kP128 + 2 * (32 * sp + 8 * tg));
      } else {       // U group (b, w) = ((f >> 5) / MT, (f >> 5) % MT)
        const int w = (f >> 5) % MT, b = (f >> 5) / MT;
        const char *r0 = sm.V + (16 * w + g) * kP128 + 2 * (16 * b + 2 * tg);
        x.x = *reinterpret_cast<const uint32_t *>(r0);                  // nt 0, rh 0
        x.y = *reinterpret_cast<const uint32_t *>(r0 + 8 * kP128);      // nt 0, rh 1
        x.z = *reinterpret_cast<const uint32_t *>(r0 + 16);             // nt 1, rh 0
        x.w = *reinterpret_cast<const uint32_t *>(r0 + 8 * kP128 + 16); // nt 1, rh 1
      }
      *reinterpret_cast<uint4 *>((which ? u_out : wn_out) + 16 * f) = x;
    }
  }
}

// ================================================================== pass 2
// One CTA per (sequence, v-head, 16 value columns) walks the sequence's blocks in order.
//   producer warp: per block, bulk (TMA) copies of the slot's chain operands and, for the
//     outputs, a tensor-map TMA of the block's q rows and a bulk copy of A, into a
//     3-stage shared-memory ring signalled on mbarriers.
//   chain warps 0-3: the state block S[:, cols] in fp32 registers for the whole sequence
//     (read from state_in once, written to state_out once), warp w holding keys
//     32w .. 32w+31.  Per block, for tokens 16w .. 16w+15 (w < C/16),
//       D = U - W S          (fragment-ordered -W and U, S from a shared fp16 snapshot),
//     D goes to shared memory (transposed), then each warp updates its keys,
//       S <- e^(G_C) S + K~^T D,
//     and writes its part of the next snapshot.
//   output warps 4-7: for tokens 16ow .. 16ow+15, O = diag(e^G) Q S + A D from the same
//     snapshot and the exchanged D.
// Hand-offs between chain and output warps are named barriers; the ring's are mbarriers
// with bounded waits (a wait that gives up reports GDN_STATUS_WAIT_TIMEOUT).
constexpr int kDVB = 16;  // value columns per CTA
constexpr int kChainWarps = 4, kOutWarps = 4;
constexpr int kChain = 32 * kChainWarps;
constexpr int kPair = 32 * (kChainWarps + kOutWarps);

// Named barriers of pass 2 (0 is __syncthreads)
constexpr int kBarChain = 1;   // the chain warps among themselves
constexpr int kBarSReady = 2;  // +parity: snapshot S_c published (chain arrives, output waits)
constexpr int kBarDone = 4;    // +parity: output warps done with block c (output arrives, chain waits)
constexpr int kBarDReady = 6;  // +parity: D_c published (chain arrives, output waits)

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
  alignas(128) char KT[C * 256];        // K~^T
  alignas(128) char U[(C / 16) * 512];  // U of this CTA's 16 value columns
  alignas(16) float DEC[2 * C];         // G, e^G
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
  alignas(128) char Sn[2][kDVB * 256];  // S^T (fp16) [16 value cols][128 keys], by parity
  alignas(128) char Dt[2][kDVB * 128];  // D^T (fp16) [16 value cols][C tokens], by parity
  alignas(16) float S32[kD][kDVB + 4];  // fp32 staging of the state block
  alignas(8) uint64_t full[NST], empty[NST];
};
template <int C, int MODE>
constexpr size_t rec_smem_bytes() {
  const size_t base = (sizeof(RecSmem<C, MODE>) + 1023) / 1024 * 1024;
  return 1024 + base + (MODE == 0 ? 3 * sizeof(OutStage<C>) : 0);  // + alignment slack
}

__device__ __forceinline__ void put4(uint32_t (&d)[4], uint4 x) {
  d[0] = x.x;
  d[1] = x.y;
  d[2] = x.z;
  d[3] = x.w;
}
template <int KW>
__device__ __forceinline__ void lds_words(uint32_t (&d)[KW], const char *p) {
  if constexpr (KW == 4) {
    put4(d, *reinterpret_cast<const uint4 *>(p));
  } else {
    const uint2 x = *reinterpret_cast<const uint2 *>(p);
    d[0] = x.x;
    d[1] = x.y;
  }
}
// Lane (gid, tig)'s token run of span `span` in row r of the swizzled D^T tile.
template <int KW>
__device__ __forceinline__ void lds_run(uint32_t (&d)[KW], const char *tile, int r, int span, int tig) {
  lds_words<KW>(d, tile + swz_row(r, 128, 2 * (KW == 4 ? 32 * span + 8 * tig : 16 * span + 4 * tig)));
}

// 3-D tensor-map TMA load (box of the map) into shared memory, completion on `bar`.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3, %4}], [%5];\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
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
__device__ __forceinline__ void chain_block(int c, const ChainStage<C> &st, float (&Sa)[4][4],
                                            RecSmem<C, MODE> &sm, int w, int lane, bool dwork,
                                            bool with_u) {
  using TS = TokSpan<C>;
  const int gid = lane >> 2, tig = lane & 3, par = c & 1;
  if (dwork) {
    // four independent accumulations per n-tile (key spans s), two products deep each
    float d[4][2][4];  // [key span][n-tile: value columns 8nt..][fragment]
#pragma unroll
    for (int g = 0; g < 4; ++g)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) d[g][nt][i] = 0.f;
    const char *Sn = sm.Sn[par];
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
    // D^T: matrices m = 2nt + rh (tokens 16w + 8rh.., columns 8nt..) stored transposed
    const int m = lane >> 3, r = lane & 7;
    stsm_x4_t(sm.Dt[par] + swz_row(8 * (m >> 1) + r, 128, 32 * w + 16 * (m & 1)),
              pack_f16(D[0][0], D[0][1]), pack_f16(D[0][2], D[0][3]), pack_f16(D[1][0], D[1][1]),
              pack_f16(D[1][2], D[1][3]));
  }
  bar_sync(kBarChain, kChain);
  if (MODE == 0) bar_arrive(kBarDReady + par, kPair);

  // S^T <- e^(G_C) S^T + D^T K~ over keys 32w .. 32w+31: one fresh accumulation per
  // token span, summed with the scaled state at the end
  float X[TS::NSP][4][4];
#pragma unroll
  for (int s = 0; s < TS::NSP; ++s)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) X[s][nt][i] = 0.f;
#pragma unroll
  for (int s = 0; s < TS::NSP; ++s) {
    uint32_t a0[TS::KW], a1[TS::KW], kt[4][TS::KW];
    lds_run<TS::KW>(a0, sm.Dt[par], gid, s, tig);
    lds_run<TS::KW>(a1, sm.Dt[par], gid + 8, s, tig);
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) lds_words<TS::KW>(kt[nt], st.KT + kt_off<C>(w, nt, s, lane));
#pragma unroll
    for (int e = 0; e < TS::KS; ++e) {
      const uint32_t a[4] = {a0[2 * e], a1[2 * e], a0[2 * e + 1], a1[2 * e + 1]};
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) mma_f16(X[s][nt], a, kt[nt][2 * e], kt[nt][2 * e + 1]);
    }
  }
  const float gam = st.DEC[2 * C - 1];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float x = X[0][nt][i];
#pragma unroll
      for (int s = 1; s < TS::NSP; ++s) x += X[s][nt][i];
      Sa[nt][i] = fmaf(gam, Sa[nt][i], x);
    }
  // S_{c+1} into the other snapshot buffer once the output warps are done with block c - 1
  if (MODE == 0 && c >= 1) bar_sync(kBarDone + (par ^ 1), kPair);
  write_snapshot(Sa, sm.Sn[par ^ 1], w, lane);
  bar_sync(kBarChain, kChain);
  if (MODE == 0) bar_arrive(kBarSReady + (par ^ 1), kPair);
}

template <int C, typename TO>
__device__ __forceinline__ void out_block(int c, const ChainStage<C> &cst, const OutStage<C> &ost,
                                          RecSmem<C, 0> &sm, int ow, int lane, TO *o, int tok0,
                                          int L, int hv, int h, int blk) {
  constexpr int RC = row_c(C);
  const int gid = lane >> 2, tig = lane & 3, par = c & 1;
  const bool work = 16 * ow < C;
  bar_sync(kBarSReady + par, kPair);
  float R[2][4];
  if (work) {
    float r2[2][2][4];  // [k-step parity][n-tile][fragment]
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) r2[e][nt][i] = 0.f;
    const char *Sn = sm.Sn[par];
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
  bar_sync(kBarDReady + par, kPair);
  if (work) {
    // O += A D over the causal part (A is zero above the diagonal)
    for (int ks = 0; ks <= ow; ++ks) {
      uint32_t a[4], b[4];
      lda_p<RC>(a, ost.A, 16 * ow, 16 * ks, lane);
      ldsm_x4(b, sm.Dt[par] + swz_row((lane & 7) + (lane >> 4) * 8, 128, 2 * (16 * ks + ((lane >> 3) & 1) * 8)));
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
  bar_arrive(kBarDone + par, kPair);
}

// MODE 0: pass 2 (state chain and outputs): 4 chain + 4 output warps + 1 producer warp.
// MODE 1: the sequence split's state chains: CTAs [0, heads * 8) run from state_in, the
// next heads * 8 from state_in2 with U taken as zero (-> state_out2); 4 chain warps + the
// producer, no outputs.
template <int C, typename TO, int MODE>
__global__ void __launch_bounds__(MODE == 0 ? kPair + 32 : kChain + 32, C == 64 ? 1 : 2)
    recur_kernel(ChunkParams p, const __grid_constant__ CUtensorMap qmap) {
  constexpr int NB = kD / kDVB, MT = C / 16, RC = row_c(C);
  constexpr int NT = MODE == 0 ? kPair + 32 : kChain + 32;
  constexpr int NST = RecSmem<C, MODE>::NST, PW = NT / 32 - 1;  // ring depth, producer warp
  constexpr size_t SB = slot_bytes(C);
  constexpr uint32_t kChainTx = (uint32_t)(2 * C * 256 + MT * 512 + 8 * C);
  constexpr uint32_t kOutTx = (uint32_t)(2 * C * 128 + C * RC);
  extern __shared__ unsigned char smem_raw[];
  unsigned char *base = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  RecSmem<C, MODE> &sm = *reinterpret_cast<RecSmem<C, MODE> *>(base);
  OutStage<C> *os = reinterpret_cast<OutStage<C> *>(base + (sizeof(RecSmem<C, MODE>) + 1023) / 1024 * 1024);
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

  int bos, eos;
  seq_range(p.cu_seqlens, n, p.total_tokens, bos, eos);
  const int nchunks = (eos - bos + C - 1) / C;
  const size_t sbase = ((size_t)n * p.hv + h) * kD * kD + blk * kDVB;
  const char *slot0 = p.slot_ws + ((size_t)h * p.nslots + slot_index(bos, C, n, 0)) * SB;

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], MODE == 0 ? 1 + kOutWarps : 1);  // the chain group, each output warp
    }
    mbar_fence_init();
  }
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
        bulk_g2s(cs.KT, src + slot_kt_off(C), C * 256, &sm.full[s]);
        bulk_g2s(cs.U, src + slot_u_off(C) + u_off<C>(blk, 0, 0), MT * 512, &sm.full[s]);
        bulk_g2s(cs.DEC, src + slot_dec_off(C), 8 * C, &sm.full[s]);
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
      chain_block<C, MODE>(c, sm.cs[s], Sa, sm, w, lane, dwork, !maps);
      if (tid == 0) mbar_arrive(&sm.empty[s]);  // all chain warps are past the barrier
    }
    if (MODE == 0 && nchunks >= 1) bar_sync(kBarDone + ((nchunks - 1) & 1), kPair);
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
    bar_sync(kBarSReady + (nchunks & 1), kPair);
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

// Tensor map of q [T, Hk, 128] bf16 for boxes of 64 keys x 1 head x C tokens, 128-byte
// swizzle (rows past T read as zero).
cudaError_t q_tensor_map(CUtensorMap *map, const void *q, int total_tokens, int hk, int C) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)hk, (cuuint64_t)total_tokens};
  const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)hk * kD * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)C};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides,
                         box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int C, typename TO, int MODE>
cudaError_t launch_recur(const ChunkParams &p, long long heads, cudaStream_t stream) {
  constexpr size_t smem = rec_smem_bytes<C, MODE>();
  cudaError_t err = cudaFuncSetAttribute(recur_kernel<C, TO, MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  CUtensorMap qmap;
  memset(&qmap, 0, sizeof(qmap));
  if (MODE == 0 && p.total_tokens > 0) {  // (no block, no q load, without tokens)
    err = q_tensor_map(&qmap, p.q, p.total_tokens, p.hk, C);
    if (err != cudaSuccess) return err;
  }
  const unsigned grid = (unsigned)((MODE == 1 ? 2 : 1) * heads * (kD / kDVB));
  recur_kernel<C, TO, MODE><<<grid, MODE == 0 ? kPair + 32 : kChain + 32, smem, stream>>>(p, qmap);
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
  // pass-1 CTAs per (sequence, head): one per block up to about 8 CTAs per SM in total
  long long per_head = (8LL * sms + heads - 1) / heads;
  per_head = max(1LL, min(per_head, max(1LL, max_chunks)));

  if (p.total_tokens > 0 && p.passes != 2 && p.passes != 3) {
    const size_t s1 = sizeof(PrepSmem<C>);
    err = cudaFuncSetAttribute(prep_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1);
    if (err != cudaSuccess) return err;
    prep_kernel<C><<<(unsigned)(heads * per_head), kPrepThreads, s1, stream>>>(p, (int)per_head);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  if (p.passes == 1) return cudaSuccess;
  if (p.passes == 3) return launch_recur<C, float, 1>(p, heads, stream);
  return p.o_fp32 ? launch_recur<C, float, 0>(p, heads, stream)
                  : launch_recur<C, __nv_bfloat16, 0>(p, heads, stream);
}

}  // namespace

size_t chunk_workspace_bytes(int total_tokens, int num_seqs, int hv, int chunk) {
  const size_t slots = (size_t)hv * ((size_t)total_tokens / chunk + num_seqs);
  return 256 + slots * slot_bytes(chunk);
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
