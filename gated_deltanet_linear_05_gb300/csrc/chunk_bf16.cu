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
//     sides instead of forming (I + N)^-1.  Each block's W^T, fp16 q and k rows, A,
//     decays and U^T go to its own workspace slot in the padded shared-memory layout
//     pass 2 reads.
//   pass 2 (recur_kernel, one CTA per (sequence, v-head, 16 value columns)): walks the
//     blocks of the sequence in order with the state block S[:, cols] in fp32 registers
//     (read from state_in once, written to state_out once).  A producer warp streams
//     each block's slot part into a 2-stage shared-memory ring with two bulk (TMA)
//     copies signalled on mbarriers.  Eight compute warps each own 8 tokens of the
//     block for
//       D^T = U^T - S^T W^T   and   R^T = S^T Q^T   (sharing the S^T fragments),
//     exchange D once through shared memory, then each carries 16 keys of the state,
//       S^T <- exp(G_T) S^T + (D^T diag(exp(G_T - G))) K,
//     and finishes its tokens' outputs O^T = diag(e^G) R^T + D^T A^T.
// Tensor-core products (mma.sync) take fp16 operands with fp32 accumulation: bf16 q, k
// and v enter exactly (converted to fp16), the state, D, T, W and A are rounded to fp16
// (11 significant bits) for the products only; the state itself, the sums and every
// decay are fp32.  Decay factors between two tokens are always the exp of a difference
// of cumsums.  A partly filled block is padded with g = 0, beta = 0 and zero q/k/v rows
// (token_valid), which leaves the state exactly as after the sequence's last token.
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
  if (blockIdx.x == 0 && tid == 0) *p.err = 0;
  // pass 2 may be scheduled now (programmatic dependent launch): its CTAs set up on SMs
  // that pass 1 has left and wait for pass 1's completion before reading any slot
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

  int bos, eos;
  seq_range(p.cu_seqlens, n, p.total_tokens, bos, eos);
  const int nchunks = (eos - bos + C - 1) / C;

#pragma unroll 1
  for (int c = part; c < nchunks; c += per_head) {
    const int tok0 = bos + c * C;
    const int L = min(C, eos - tok0);
    char *slot = p.slot_ws + ((size_t)h * p.nslots + slot_index(bos, C, n, c)) * slot_bytes(C);
    char *w_out = slot, *a_out = slot + slot_a_off(C), *u_out = slot + slot_u_off(C);
    char *q_out = slot + slot_q_off(C), *k_out = slot + slot_k_off(C);
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
    // 16 rows x two 16-byte halves
    for (int e = tid; e < 16 * MT * (MT - 1); e += NT) {
      const int tile = e >> 5, row = (e >> 1) & 15, hh = e & 1;
      int mt = 0, np = 1, cnt = tile;  // tile -> (mt, np > mt), row-major over the upper part
      while (cnt >= MT - 1 - mt) {
        cnt -= MT - 1 - mt;
        ++mt;
      }
      np = mt + 1 + cnt;
      *reinterpret_cast<uint4 *>(a_out + (16 * mt + row) * RC + 2 * (16 * np + 8 * hh)) =
          make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();

    cp_async_wait<0>();  // v has landed (visible to all after the next barrier)
    // ---- T_ii = (I + N_ii)^-1 for the 16x16 diagonal blocks in fp32: one column per
    //      thread, forward substitution.  Meanwhile the other threads ship the fp16 q, k
    //      rows and the decays to the slot.
    if (tid < C) {
      const int blk = tid >> 4, cc = tid & 15;
      float x[16];
      unit_tril_inverse_col(&sm.Nd[blk][0][0], 17, cc, x);
#pragma unroll
      for (int r = 0; r < 16; ++r)
        *reinterpret_cast<__half *>(sm.T16[blk] + r * 48 + 2 * cc) = __float2half_rn(x[r]);
    } else {
      const int t2 = tid - C, n2 = NT - C;
      for (int e = t2; e < 2 * C * 16; e += n2) {  // 16 granules of 8 elements per row
        const int which = e / (C * 16), r = (e >> 4) & (C - 1), gq = e & 15;
        const uint4 x = *reinterpret_cast<const uint4 *>((which ? sm.Q : sm.K) + r * kP128 + 16 * gq);
        *reinterpret_cast<uint4 *>((which ? q_out : k_out) + r * kP128 + 16 * gq) =
            make_uint4(bf16x2_to_f16x2(x.x), bf16x2_to_f16x2(x.y), bf16x2_to_f16x2(x.z),
                       bf16x2_to_f16x2(x.w));
      }
      for (int t = t2; t < C; t += n2) {
        dec_out[t] = sm.G[t];
        dec_out[C + t] = sm.EG[t];
        dec_out[2 * C + t] = sm.ED[t];
      }
    }
    __syncthreads();

    // ---- [W U] = (I + N)^-1 [diag(beta e^G) K  diag(beta) V] by blocked forward
    //      substitution over the 16-token blocks, X_i = T_ii (R_i - sum_{j<i} N_ij X_j),
    //      transposed so that each warp solves its own 32 columns without exchange:
    //      X_i^T = (R_i^T - sum_j X_j^T N_ij^T) T_ii^T.  Warps 0-3: W (32 keys each),
    //      warps 4-7: U (32 value columns each); both stored by column (W^T, U^T).
    {
      const int kind = warp >> 2, c0 = 32 * (warp & 3);
      const char *X = kind ? sm.V : sm.K;
      char *xo = kind ? u_out : w_out;
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
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
              const int col = c0 + 16 * mt + gid + 8 * hr, t = 16 * i + 8 * nt + 2 * tig;
              *reinterpret_cast<uint32_t *>(xo + col * RC + 2 * t) =
                  pack_f16(out[mt][nt][2 * hr], out[mt][nt][2 * hr + 1]);
            }
          if (i + 1 < MT) acc_to_f16(out[mt][0], out[mt][1], 1.f, 1.f, 1.f, 1.f, Xf[i][mt]);
        }
      }
    }
  }
}

// ================================================================== pass 2

constexpr int kChainWarps = 4, kOutWarps = 4;
constexpr int kRecThreads = 32 * (kChainWarps + kOutWarps + 1);  // + 1 producer warp
constexpr int kChain = 32 * kChainWarps;
constexpr int kPair = 32 * (kChainWarps + kOutWarps);
constexpr int kStages = 3;
constexpr int kDVB = 16;  // value columns per CTA

// Named barriers of pass 2 (0 is __syncthreads)
constexpr int kBarChain = 1;   // the chain warps among themselves
constexpr int kBarSReady = 2;  // +parity: snapshot S_c published (chain arrives, output waits)
constexpr int kBarDone = 4;    // +parity: output warps done with block c (output arrives, chain waits)
constexpr int kBarDReady = 6;  // +parity: D_c published (chain arrives, output waits)

template <int C, typename TO>
struct RecSmem {
  static constexpr int RC = row_c(C);
  struct Stage {
    alignas(128) char H[slot_head_bytes(C)];  // W^T | Q | K | A | DEC, as in the slot
    alignas(16) char U[kDVB * RC];            // U^T rows of this CTA's value columns
  } st[kStages];
  alignas(8) uint64_t full[kStages], empty[kStages];
  alignas(16) char Sn[2][kDVB * kP128];  // S_c^T (fp16) [16 value cols][128 keys], by parity
  alignas(16) char Db[2][kDVB * RC];     // D_c^T (fp16) [16 value cols][C tokens], by parity
  alignas(16) char Dd[kDVB * RC];        // (D diag(e^(G_C - G)))^T (fp16)
  alignas(16) TO O[kOutWarps][16][kDVB];
  alignas(16) float S32[kD][kDVB + 4];  // fp32 staging of the state block
};

template <int C, typename TO>
__global__ void __launch_bounds__(kRecThreads) recur_kernel(ChunkParams p) {
  constexpr int NB = kD / kDVB, MT = C / 16, RC = row_c(C);
  constexpr uint32_t kHeadB = (uint32_t)slot_head_bytes(C);
  constexpr uint32_t kUB = (uint32_t)(kDVB * RC);
  constexpr uint32_t kStageTx = kHeadB + kUB;
  using Smem = RecSmem<C, TO>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int blk = blockIdx.x % NB;
  const int nh = blockIdx.x / NB;
  const int n = nh / p.hv;
  const int h = nh - n * p.hv;
  TO *o = static_cast<TO *>(p.o);

  int bos, eos;
  seq_range(p.cu_seqlens, n, p.total_tokens, bos, eos);
  const int nchunks = (eos - bos + C - 1) / C;
  const size_t sbase = ((size_t)n * p.hv + h) * kD * kD + blk * kDVB;
  const char *slot0 = p.slot_ws + ((size_t)h * p.nslots + slot_index(bos, C, n, 0)) * slot_bytes(C);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1 + kOutWarps);  // the chain warps once, each output warp
    }
    mbar_fence_init();
  }
  // state block S[:, blk*16 .. +16) -> fp32 staging (coalesced 64-byte rows)
  for (int e = tid; e < kD * kDVB / 4; e += kRecThreads) {
    const int i = e / (kDVB / 4), c4 = e % (kDVB / 4);
    const float4 val =
        p.state_in ? *reinterpret_cast<const float4 *>(p.state_in + sbase + (size_t)i * kD + 4 * c4)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    *reinterpret_cast<float4 *>(&sm.S32[i][4 * c4]) = val;
  }
  __syncthreads();
  // pass 1 complete and its slot writes visible (returns at once without a pending
  // prerequisite grid)
  asm volatile("griddepcontrol.wait;\n" ::: "memory");

  if (warp == kChainWarps + kOutWarps) {
    // ---- producer: stream each block's slot part into the ring
    if (lane == 0) {
      bool ok = true;
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % kStages;
        if (c >= kStages) ok = mbar_wait(&sm.empty[s], ((c / kStages) - 1) & 1) && ok;
        typename Smem::Stage &st = sm.st[s];
        const char *src = slot0 + (size_t)c * slot_bytes(C);
        mbar_arrive_expect_tx(&sm.full[s], kStageTx);
        bulk_g2s(st.H, src, kHeadB, &sm.full[s]);
        bulk_g2s(st.U, src + slot_u_off(C) + (size_t)blk * kDVB * RC, kUB, &sm.full[s]);
      }
      // the last copies are consumed before the CTA's final barrier
      if (!ok) atomicExch(p.err, 1);
    }
  } else if (warp < kChainWarps) {
    // ---- chain warp w: D for tokens 16w .. 16w+15, the state for keys 32w .. 32w+31
    const int w = warp;
    float Sa[4][4];  // S^T[j][i], j = gid (+8), i = 32w + 8nt + 2tig (+1)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        Sa[nt][e] = sm.S32[32 * w + 8 * nt + 2 * tig + (e & 1)][gid + 8 * (e >> 1)];
    auto write_snapshot = [&](char *Sn) {
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int j = gid + 8 * hr, i = 32 * w + 8 * nt + 2 * tig;
          *reinterpret_cast<uint32_t *>(Sn + j * kP128 + 2 * i) =
              pack_f16(Sa[nt][2 * hr], Sa[nt][2 * hr + 1]);
        }
    };
    write_snapshot(sm.Sn[0]);
    bar_sync(kBarChain, kChain);
    bar_arrive(kBarSReady + 0, kPair);

    bool ok = true;
#pragma unroll 1
    for (int c = 0; c < nchunks; ++c) {
      const int s = c % kStages, par = c & 1;
      typename Smem::Stage &st = sm.st[s];
      const char *Wt = st.H, *Ks = st.H + slot_k_off(C);
      const float *DG = reinterpret_cast<const float *>(st.H + slot_dec_off(C));
      const float *EG = DG + C, *ED = DG + 2 * C;
      ok = mbar_wait(&sm.full[s], (c / kStages) & 1) && ok;

      if (w < MT) {
        // D^T = U^T - S^T W^T for tokens 16w .. 16w+15, keys split in halves
        float D0[2][4], D1[2][4];
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const float2 u = f16x2_to_float2(*reinterpret_cast<const uint32_t *>(
                st.U + (gid + 8 * hr) * RC + 2 * (16 * w + 8 * a + 2 * tig)));
            D0[a][2 * hr] = u.x;
            D0[a][2 * hr + 1] = u.y;
            D1[a][2 * hr] = D1[a][2 * hr + 1] = 0.f;
          }
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
          uint32_t nf[4], bw[4];
          lda_p<kP128>(nf, sm.Sn[par], 0, 16 * ks, lane);
#pragma unroll
          for (int e = 0; e < 4; ++e) nf[e] ^= 0x80008000u;  // -S
          ldb_kn_p<RC>(bw, Wt, 16 * ks, 16 * w, lane);
          if (ks & 1) {
            mma_f16(D1[0], nf, bw[0], bw[1]);
            mma_f16(D1[1], nf, bw[2], bw[3]);
          } else {
            mma_f16(D0[0], nf, bw[0], bw[1]);
            mma_f16(D0[1], nf, bw[2], bw[3]);
          }
        }
        // D (for the outputs) and its carry-scaled copy (for the state), fp16
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int j = gid + 8 * hr, t = 16 * w + 8 * a + 2 * tig;
            const float d0 = D0[a][2 * hr] + D1[a][2 * hr], d1 = D0[a][2 * hr + 1] + D1[a][2 * hr + 1];
            *reinterpret_cast<uint32_t *>(sm.Db[par] + j * RC + 2 * t) = pack_f16(d0, d1);
            *reinterpret_cast<uint32_t *>(sm.Dd + j * RC + 2 * t) = pack_f16(d0 * ED[t], d1 * ED[t + 1]);
          }
      }
      bar_sync(kBarChain, kChain);
      bar_arrive(kBarDReady + par, kPair);

      // S^T <- e^(G_C) S^T + Dd^T K over keys 32w .. 32w+31
      {
        float X[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int e = 0; e < 4; ++e) X[a][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < MT; ++ks) {
          uint32_t df[4];
          lda_p<RC>(df, sm.Dd, 0, 16 * ks, lane);
#pragma unroll
          for (int np = 0; np < 2; ++np) {
            uint32_t b[4];
            ldb_kn_p<kP128>(b, Ks, 16 * ks, 32 * w + 16 * np, lane);
            mma_f16(X[2 * np], df, b[0], b[1]);
            mma_f16(X[2 * np + 1], df, b[2], b[3]);
          }
        }
        const float egc = EG[C - 1];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) Sa[nt][e] = fmaf(egc, Sa[nt][e], X[nt][e]);
      }
      // S_{c+1} into the other snapshot buffer once the output warps are done with block
      // c - 1 (which read it as S_{c-1})
      if (c >= 1) bar_sync(kBarDone + (par ^ 1), kPair);
      write_snapshot(sm.Sn[par ^ 1]);
      bar_sync(kBarChain, kChain);
      if (tid == 0) mbar_arrive(&sm.empty[s]);
      bar_arrive(kBarSReady + (par ^ 1), kPair);
    }
    if (nchunks >= 1) bar_sync(kBarDone + ((nchunks - 1) & 1), kPair);
    if (!ok && lane == 0) atomicExch(p.err, 1);
    // final state block -> fp32 staging
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        sm.S32[32 * w + 8 * nt + 2 * tig + (e & 1)][gid + 8 * (e >> 1)] = Sa[nt][e];
  } else {
    // ---- output warp: O^T = diag(e^G) S^T Q^T + D^T A^T for tokens 16ow .. 16ow+15
    const int ow = warp - kChainWarps;
    bool ok = true;
#pragma unroll 1
    for (int c = 0; c < nchunks; ++c) {
      const int s = c % kStages, par = c & 1;
      typename Smem::Stage &st = sm.st[s];
      const char *Qs = st.H + slot_q_off(C), *A = st.H + slot_a_off(C);
      const float *EG = reinterpret_cast<const float *>(st.H + slot_dec_off(C)) + C;
      const int tok0 = bos + c * C;
      const int L = min(C, eos - tok0);
      ok = mbar_wait(&sm.full[s], (c / kStages) & 1) && ok;
      bar_sync(kBarSReady + par, kPair);
      float R0[2][4], R1[2][4];
      if (ow < MT) {
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int e = 0; e < 4; ++e) R0[a][e] = R1[a][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
          uint32_t sf[4], bq[4];
          lda_p<kP128>(sf, sm.Sn[par], 0, 16 * ks, lane);
          ldb_nk_p<kP128>(bq, Qs, 16 * ow, 16 * ks, lane);
          if (ks & 1) {
            mma_f16(R1[0], sf, bq[0], bq[1]);
            mma_f16(R1[1], sf, bq[2], bq[3]);
          } else {
            mma_f16(R0[0], sf, bq[0], bq[1]);
            mma_f16(R0[1], sf, bq[2], bq[3]);
          }
        }
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            R0[a][e] = (R0[a][e] + R1[a][e]) * EG[16 * ow + 8 * a + 2 * tig + (e & 1)];
      }
      bar_sync(kBarDReady + par, kPair);
      if (ow < MT) {
        // O^T += D^T A^T over the causal part (A is zero above the diagonal)
        for (int ks = 0; ks <= ow; ++ks) {
          uint32_t df[4], ba[4];
          lda_p<RC>(df, sm.Db[par], 0, 16 * ks, lane);
          ldb_nk_p<RC>(ba, A, 16 * ow, 16 * ks, lane);
          mma_f16(R0[0], df, ba[0], ba[1]);
          mma_f16(R0[1], df, ba[2], ba[3]);
        }
        // stage O^T [t][j] and store this warp's rows that lie in the sequence
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            Elem<TO>::store(&sm.O[ow][8 * a + 2 * tig + (e & 1)][gid + 8 * (e >> 1)], R0[a][e]);
        __syncwarp();
        constexpr int EPG = 16 / sizeof(TO);  // elements per 16-byte granule
        constexpr int GPR = kDVB / EPG;       // granules per output row
        for (int e = lane; e < 16 * GPR; e += 32) {
          const int r = e / GPR, gi = e % GPR, t = 16 * ow + r;
          if (t < L)
            *reinterpret_cast<uint4 *>(o + ((size_t)(tok0 + t) * p.hv + h) * kD + blk * kDVB +
                                       gi * EPG) =
                *reinterpret_cast<const uint4 *>(&sm.O[ow][r][gi * EPG]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[s]);
      bar_arrive(kBarDone + par, kPair);
    }
    if (nchunks >= 0) bar_sync(kBarSReady + (nchunks & 1), kPair);
    if (!ok && lane == 0) atomicExch(p.err, 1);
  }
  __syncthreads();
  for (int e = tid; e < kD * kDVB / 4; e += kRecThreads) {
    const int i = e / (kDVB / 4), c4 = e % (kDVB / 4);
    *reinterpret_cast<float4 *>(p.state_out + sbase + (size_t)i * kD + 4 * c4) =
        *reinterpret_cast<const float4 *>(&sm.S32[i][4 * c4]);
  }
}

template <int C, typename TO>
cudaError_t launch_recur(const ChunkParams &p, long long heads, cudaStream_t stream) {
  const size_t s2 = sizeof(RecSmem<C, TO>);
  cudaError_t err = cudaFuncSetAttribute(recur_kernel<C, TO>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s2);
  if (err != cudaSuccess) return err;
  // launched as a programmatic dependent of pass 1, so that its launch and set-up overlap
  // the tail of pass 1
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(heads * (kD / kDVB)));
  cfg.blockDim = dim3(kRecThreads);
  cfg.dynamicSmemBytes = s2;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, recur_kernel<C, TO>, p);
}

// ================================================================== split: state chains
// The sequence split's runs from zero (-> L_s) and from the identity with U = 0 (-> M_s)
// need only pass 2's state chain.  One launch covers both: CTAs [0, heads * 8) walk the
// L chains, the next heads * 8 the M chains (state_in2 / state_out2, U taken as zero).
// A CTA is the 4 chain warps of recur_kernel plus its producer warp, with a 2-stage ring
// of the chain's operands only (W^T, K, the decays and this CTA's U columns: 38 KB per
// block at C = 64) and one snapshot buffer (no output warps read it): ~99 KB of shared
// memory, so two CTAs share an SM and both kinds of chain run in one wave.
constexpr int kChThreads = 32 * (kChainWarps + 1);
constexpr int kChStages = 2;

template <int C>
struct ChainSmem {
  static constexpr int RC = row_c(C);
  struct Stage {
    alignas(128) char W[slot_q_off(C)];  // W^T, as in the slot
    alignas(16) char K[C * kP128];       // the block's k rows (fp16)
    alignas(16) float DEC[3 * C];        // G, e^G, e^(G_C - G)
    alignas(16) char U[kDVB * RC];       // U^T rows of this CTA's value columns
  } st[kChStages];
  alignas(8) uint64_t full[kChStages], empty[kChStages];
  alignas(16) char Sn[kDVB * kP128];  // S_c^T (fp16) [16 value cols][128 keys]
  alignas(16) char Dd[kDVB * RC];     // (D diag(e^(G_C - G)))^T (fp16)
  alignas(16) float S32[kD][kDVB + 4];
};

template <int C>
__global__ void __launch_bounds__(kChThreads) split_chain_kernel(ChunkParams p) {
  constexpr int NB = kD / kDVB, MT = C / 16, RC = row_c(C);
  constexpr uint32_t kWB = (uint32_t)slot_q_off(C), kKB = (uint32_t)(C * kP128);
  constexpr uint32_t kDB = (uint32_t)(12 * C), kUB = (uint32_t)(kDVB * RC);
  using Smem = ChainSmem<C>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const long long half = (long long)p.num_seqs * p.hv * NB;
  const bool maps = (long long)blockIdx.x >= half;
  const long long b = maps ? (long long)blockIdx.x - half : (long long)blockIdx.x;
  const int blk = (int)(b % NB);
  const int nh = (int)(b / NB);
  const int n = nh / p.hv;
  const int h = nh - n * p.hv;
  const float *s_in = maps ? p.state_in2 : p.state_in;
  float *s_out = maps ? p.state_out2 : p.state_out;

  int bos, eos;
  seq_range(p.cu_seqlens, n, p.total_tokens, bos, eos);
  const int nchunks = (eos - bos + C - 1) / C;
  const size_t sbase = ((size_t)n * p.hv + h) * kD * kD + blk * kDVB;
  const char *slot0 = p.slot_ws + ((size_t)h * p.nslots + slot_index(bos, C, n, 0)) * slot_bytes(C);

  if (tid == 0) {
    for (int s = 0; s < kChStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    mbar_fence_init();
  }
  for (int e = tid; e < kD * kDVB / 4; e += kChThreads) {
    const int i = e / (kDVB / 4), c4 = e % (kDVB / 4);
    const float4 val =
        s_in ? *reinterpret_cast<const float4 *>(s_in + sbase + (size_t)i * kD + 4 * c4)
             : make_float4(0.f, 0.f, 0.f, 0.f);
    *reinterpret_cast<float4 *>(&sm.S32[i][4 * c4]) = val;
  }
  __syncthreads();
  asm volatile("griddepcontrol.wait;\n" ::: "memory");  // pass 1's slots are complete

  if (warp == kChainWarps) {
    // ---- producer: the chain's operands of each block into the ring
    if (lane == 0) {
      bool ok = true;
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % kChStages;
        if (c >= kChStages) ok = mbar_wait(&sm.empty[s], ((c / kChStages) - 1) & 1) && ok;
        typename Smem::Stage &st = sm.st[s];
        const char *src = slot0 + (size_t)c * slot_bytes(C);
        mbar_arrive_expect_tx(&sm.full[s], kWB + kKB + kDB + kUB);
        bulk_g2s(st.W, src, kWB, &sm.full[s]);
        bulk_g2s(st.K, src + slot_k_off(C), kKB, &sm.full[s]);
        bulk_g2s(st.DEC, src + slot_dec_off(C), kDB, &sm.full[s]);
        bulk_g2s(st.U, src + slot_u_off(C) + (size_t)blk * kDVB * RC, kUB, &sm.full[s]);
      }
      if (!ok) atomicExch(p.err, 1);
    }
  } else {
    // ---- chain warp w: D for tokens 16w .. 16w+15, the state for keys 32w .. 32w+31
    const int w = warp;
    float Sa[4][4];  // S^T[j][i], j = gid (+8), i = 32w + 8nt + 2tig (+1)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        Sa[nt][e] = sm.S32[32 * w + 8 * nt + 2 * tig + (e & 1)][gid + 8 * (e >> 1)];
    auto write_snapshot = [&]() {
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int j = gid + 8 * hr, i = 32 * w + 8 * nt + 2 * tig;
          *reinterpret_cast<uint32_t *>(sm.Sn + j * kP128 + 2 * i) =
              pack_f16(Sa[nt][2 * hr], Sa[nt][2 * hr + 1]);
        }
    };
    write_snapshot();
    bar_sync(kBarChain, kChain);

    bool ok = true;
#pragma unroll 1
    for (int c = 0; c < nchunks; ++c) {
      const int s = c % kChStages;
      typename Smem::Stage &st = sm.st[s];
      const float *EG = st.DEC + C, *ED = st.DEC + 2 * C;
      ok = mbar_wait(&sm.full[s], (c / kChStages) & 1) && ok;

      if (w < MT) {
        // D^T = U^T - S^T W^T for tokens 16w .. 16w+15 (U = 0 for the map chains)
        float D0[2][4], D1[2][4];
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const float2 u = f16x2_to_float2(*reinterpret_cast<const uint32_t *>(
                st.U + (gid + 8 * hr) * RC + 2 * (16 * w + 8 * a + 2 * tig)));
            D0[a][2 * hr] = maps ? 0.f : u.x;
            D0[a][2 * hr + 1] = maps ? 0.f : u.y;
            D1[a][2 * hr] = D1[a][2 * hr + 1] = 0.f;
          }
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
          uint32_t nf[4], bw[4];
          lda_p<kP128>(nf, sm.Sn, 0, 16 * ks, lane);
#pragma unroll
          for (int e = 0; e < 4; ++e) nf[e] ^= 0x80008000u;  // -S
          ldb_kn_p<RC>(bw, st.W, 16 * ks, 16 * w, lane);
          if (ks & 1) {
            mma_f16(D1[0], nf, bw[0], bw[1]);
            mma_f16(D1[1], nf, bw[2], bw[3]);
          } else {
            mma_f16(D0[0], nf, bw[0], bw[1]);
            mma_f16(D0[1], nf, bw[2], bw[3]);
          }
        }
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int j = gid + 8 * hr, t = 16 * w + 8 * a + 2 * tig;
            const float d0 = D0[a][2 * hr] + D1[a][2 * hr], d1 = D0[a][2 * hr + 1] + D1[a][2 * hr + 1];
            *reinterpret_cast<uint32_t *>(sm.Dd + j * RC + 2 * t) = pack_f16(d0 * ED[t], d1 * ED[t + 1]);
          }
      }
      bar_sync(kBarChain, kChain);  // Dd complete; every warp is done reading the snapshot

      // S^T <- e^(G_C) S^T + Dd^T K over keys 32w .. 32w+31
      {
        float X[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int e = 0; e < 4; ++e) X[a][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < MT; ++ks) {
          uint32_t df[4];
          lda_p<RC>(df, sm.Dd, 0, 16 * ks, lane);
#pragma unroll
          for (int np = 0; np < 2; ++np) {
            uint32_t bk[4];
            ldb_kn_p<kP128>(bk, st.K, 16 * ks, 32 * w + 16 * np, lane);
            mma_f16(X[2 * np], df, bk[0], bk[1]);
            mma_f16(X[2 * np + 1], df, bk[2], bk[3]);
          }
        }
        const float egc = EG[C - 1];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) Sa[nt][e] = fmaf(egc, Sa[nt][e], X[nt][e]);
      }
      write_snapshot();
      bar_sync(kBarChain, kChain);  // the new snapshot is complete; Dd and the stage are free
      if (tid == 0) mbar_arrive(&sm.empty[s]);
    }
    if (!ok && lane == 0) atomicExch(p.err, 1);
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        sm.S32[32 * w + 8 * nt + 2 * tig + (e & 1)][gid + 8 * (e >> 1)] = Sa[nt][e];
  }
  __syncthreads();
  for (int e = tid; e < kD * kDVB / 4; e += kChThreads) {
    const int i = e / (kDVB / 4), c4 = e % (kDVB / 4);
    *reinterpret_cast<float4 *>(s_out + sbase + (size_t)i * kD + 4 * c4) =
        *reinterpret_cast<const float4 *>(&sm.S32[i][4 * c4]);
  }
}

template <int C>
cudaError_t launch_split_chains(const ChunkParams &p, long long heads, cudaStream_t stream) {
  const size_t sz = sizeof(ChainSmem<C>);
  cudaError_t err = cudaFuncSetAttribute(split_chain_kernel<C>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sz);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * heads * (kD / kDVB)));
  cfg.blockDim = dim3(kChThreads);
  cfg.dynamicSmemBytes = sz;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, split_chain_kernel<C>, p);
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
  if (p.passes == 3) return launch_split_chains<C>(p, heads, stream);
  return p.o_fp32 ? launch_recur<C, float>(p, heads, stream)
                  : launch_recur<C, __nv_bfloat16>(p, heads, stream);
}

}  // namespace

size_t chunk_workspace_bytes(int total_tokens, int num_seqs, int hv, int chunk) {
  const size_t slots = (size_t)hv * ((size_t)total_tokens / chunk + num_seqs);
  size_t sb = 0;
  switch (chunk) {
    case 16: sb = slot_bytes(16); break;
    case 32: sb = slot_bytes(32); break;
    default: sb = slot_bytes(64); break;
  }
  return 256 + slots * sb;
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
