// Single-pass chunkwise gated delta rule for batches with many (sequence, head) pairs
// ("Qwen3.5-9B-npu" model card, section "How it works", chunkwise form):
//   N   = diag(beta) [exp(G_t - G_j) k_t.k_j]_{j<t},   T = (I + N)^-1
//   D   = U - W S,  U = T diag(beta) V,  W = T diag(beta exp G) K
//   O   = diag(exp G) Q S + [exp(G_t - G_j) q_t.k_j]_{j<=t} D
//   S_T = exp(G_T) S + K^T diag(exp(G_T - G)) D
//
// One CTA of 8 warps per (sequence, v-head) walks the sequence's blocks in order.  Per
// block, the warps first build the state-independent operands together in shared
// memory (cumsum G, the decay-masked Grams, T by block doubling, W), then each warp
// carries 16 of the 128 value columns through the dependent part on its own: its slice
// of the state, S^T[16 columns][128 keys], stays in mma accumulators for the whole
// sequence and feeds the next products directly as A fragments, so the state never
// goes through shared memory and the warps never exchange data inside the chain:
//   D^T  = V^T T_u^T - S^T W^T        (starts from U^T, subtracts the state part)
//   O^T  = exp(G) S^T Q^T + D^T A^T
//   S^T <- exp(G_T) S^T + (D^T diag(exp(G_T - G))) K
// This needs no workspace.  With one CTA per head it suits batches of at least about
// one CTA per SM; few-head batches use the two-pass path (chunk_bf16.cu), which spreads
// each head over several CTAs.
// Precision as in the two-pass path: the Grams take the bf16 inputs exactly; every
// other product takes fp16 operands (q, k, v converted exactly; T, W, A, D and the
// state rounded to 11 significant bits for the product only) with fp32 accumulation.
#include "common.cuh"
#include "internal.h"

namespace gdn {

namespace {

constexpr int kFThreads = 256;

template <int C, typename TO>
struct FusedSmem {
  static constexpr int RC = row_c(C);
  static constexpr int LD = C + 4;
  static constexpr size_t kNTBytes = (size_t)2 * C * LD * 4;
  static constexpr size_t kOBytes = (size_t)8 * C * 16 * sizeof(TO);
  // q, k, v rows of the current block and of the next one (prefetched); bf16 as loaded,
  // converted in place to fp16 once the Grams are done
  alignas(128) char K[2][C * kP128];
  alignas(16) char Q[2][C * kP128];
  alignas(16) char V[2][C * kP128];
  alignas(16) char W[C * kP128];  // fp16 W [t][key]
  alignas(16) char A[C * RC];     // fp16 causal decay-masked Q K^T [t][j]
  alignas(16) char TW[C * RC];    // fp16 T diag(beta e^G)
  alignas(16) char TU[C * RC];    // fp16 T diag(beta)
  // N and T (fp32 [C][C+4] each) while the operands are built, then the per-warp
  // output staging [8][C][16]
  alignas(16) char NTO[kNTBytes > kOBytes ? kNTBytes : kOBytes];
  float M[32 * 33];
  // 16-token blocks (the draft-verify size): the whole state staged here, so that it moves
  // between global and shared memory in 16-byte pieces along its rows
  alignas(16) float SS[C == 16 ? kD : 1][kD + 4];
  float G[C], EG[C], ED[C], B[C];
  float gRaw[2][C], bRaw[2][C];
};

// A fragment (16 rows x 16 k) as fp16 from two 16x8 accumulator tiles (k = their column
// index), columns scaled by s0, s1 (first tile) and t0, t1 (second tile)
__device__ __forceinline__ void acc_to_f16(const float (&x)[4], const float (&y)[4], float s0,
                                           float s1, float t0, float t1, uint32_t (&a)[4]) {
  a[0] = pack_f16(x[0] * s0, x[1] * s1);
  a[1] = pack_f16(x[2] * s0, x[3] * s1);
  a[2] = pack_f16(y[0] * t0, y[1] * t1);
  a[3] = pack_f16(y[2] * t0, y[3] * t1);
}

// acc (16x8 tile) += A[r0.., k0..k0+16) * B[k0.., n0..n0+8) for fp32 row-major shared
// matrices, as hi*hi + lo*hi + hi*lo of their bf16 splits (block-doubling products).
__device__ __forceinline__ void mma_f32x3f(float (&acc)[4], const float *A, int lda,
                                           const float *B, int ldb, int r0, int k0, int n0,
                                           int lane) {
  const int gid = lane >> 2, tig = lane & 3;
  uint32_t ah[4], al[4], bh0, bl0, bh1, bl1;
  const float *a0 = A + (r0 + gid) * lda + k0 + 2 * tig;
  const float *a1 = a0 + 8 * lda;
  split_bf16(a0[0], a0[1], ah[0], al[0]);
  split_bf16(a1[0], a1[1], ah[1], al[1]);
  split_bf16(a0[8], a0[9], ah[2], al[2]);
  split_bf16(a1[8], a1[9], ah[3], al[3]);
  const float *b0 = B + (k0 + 2 * tig) * ldb + n0 + gid;
  split_bf16(b0[0], b0[ldb], bh0, bl0);
  split_bf16(b0[8 * ldb], b0[9 * ldb], bh1, bl1);
  mma_bf16(acc, ah, bh0, bh1);
  mma_bf16(acc, al, bh0, bh1);
  mma_bf16(acc, ah, bl0, bl1);
}

// C = 16 fits two CTAs per SM (<= 128 registers), so one CTA's state load and store
// overlap another's arithmetic
template <int C, typename TO>
__global__ void __launch_bounds__(kFThreads, C == 16 ? 2 : 1) fused_kernel(ChunkParams p) {
  constexpr int NT = kFThreads, MT = C / 16, RC = row_c(C), LD = C + 4;
  constexpr int NTC = C / 8;  // 8-wide token tiles
  using Smem = FusedSmem<C, TO>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
  float(*Nm)[LD] = reinterpret_cast<float(*)[LD]>(sm.NTO);
  float(*Tm)[LD] = Nm + C;
  TO(*Ost)[C][16] = reinterpret_cast<TO(*)[C][16]>(sm.NTO);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int n = blockIdx.x / p.hv;
  const int h = blockIdx.x - n * p.hv;
  const int kh = h / (p.hv / p.hk);
  const int j0 = 16 * warp;  // this warp's value columns
  const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(p.q);
  const __nv_bfloat16 *k = static_cast<const __nv_bfloat16 *>(p.k);
  const __nv_bfloat16 *v = static_cast<const __nv_bfloat16 *>(p.v);
  TO *o = static_cast<TO *>(p.o);

  int bos, eos;
  seq_range(p.cu_seqlens, n, p.total_tokens, bos, eos);
  const int nchunks = (eos - bos + C - 1) / C;
  const size_t sbase = ((size_t)n * p.hv + h) * kD * kD;

  // q, k, v rows and gates of block cc into buffer buf (rows past the end: zeros)
  auto issue_loads = [&](int cc, int buf) {
    const int t0 = bos + cc * C, Lc = min(C, eos - t0);
    for (int e = tid; e < C * 16; e += NT) {
      const int r = e >> 4, gr = e & 15;
      const bool ok = r < Lc;
      const size_t tok = (size_t)t0 + (ok ? r : 0);
      const int nb = ok ? 16 : 0;
      cp_async16(sm.K[buf] + r * kP128 + gr * 16, k + (tok * p.hk + kh) * kD + gr * 8, nb);
      cp_async16(sm.Q[buf] + r * kP128 + gr * 16, q + (tok * p.hk + kh) * kD + gr * 8, nb);
      cp_async16(sm.V[buf] + r * kP128 + gr * 16, v + (tok * p.hv + h) * kD + gr * 8, nb);
    }
    for (int t = tid; t < C; t += NT) {
      const bool ok = t < Lc;
      const size_t gi = ((size_t)t0 + (ok ? t : 0)) * p.hv + h;
      cp_async4(&sm.gRaw[buf][t], p.g + gi, ok ? 4 : 0);
      cp_async4(&sm.bRaw[buf][t], p.beta + gi, ok ? 4 : 0);
    }
  };
  if (nchunks > 0) issue_loads(0, 0);
  cp_async_commit();  // block 0's q, k, v and gates
  if constexpr (C == 16) {
    // the state in a group of its own: block 0's state-free work (Grams, T, W, U) runs
    // while it lands, and the chain waits for it only before its first product
    if (p.state_in)
      for (int e = tid; e < kD * kD / 4; e += NT) {
        const int r = e >> 5, c4 = e & 31;
        cp_async16(&sm.SS[r][4 * c4], p.state_in + sbase + (size_t)r * kD + 4 * c4, 16);
      }
    cp_async_commit();
  }

  // S^T[j][i] for j = j0 + gid (+8), i = 8nt + 2tig (+1): 16 accumulator tiles
  float S[16][4];
  auto state_from_staging = [&]() {
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = 8 * nt + 2 * tig + (e & 1), j = j0 + gid + 8 * (e >> 1);
        S[nt][e] = p.state_in ? sm.SS[i][j] : 0.f;
      }
  };
  if constexpr (C == 16) {
    if (nchunks == 0) {  // an empty sequence passes its state through
      cp_async_wait<0>();
      __syncthreads();
      state_from_staging();
    }
  } else {
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = 8 * nt + 2 * tig + (e & 1), j = j0 + gid + 8 * (e >> 1);
        S[nt][e] = p.state_in ? p.state_in[sbase + (size_t)i * kD + j] : 0.f;
      }
  }

  // Gram tiles of this warp: warps 0-3 take K K^T, warps 4-7 Q K^T, each a balanced share
  // of the causal 16x16 tiles (mt, np <= mt): np0 .. np0+n0-1 of row mt0, and for one
  // warp at C = 64 also tile (mt1 = 0, 0)
  const int prod = warp >> 2, qw = warp & 3;
  int mt0 = 0, np0 = 0, n0 = 0, mt1 = -1;
  if (C == 64) {  // rows 3: {0,1}, {2,3}; row 2: {0,1,2}; rows 1: {0,1} and 0: {0}
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

#pragma unroll 1
  for (int c = 0; c < nchunks; ++c) {
    const int buf = c & 1;
    const int tok0 = bos + c * C;
    const int L = min(C, eos - tok0);
    __syncthreads();  // the previous block is done with shared memory
    if (c + 1 < nchunks) issue_loads(c + 1, buf ^ 1);
    cp_async_commit();
    // T starts at zero: the doubling products read whole 32x32 blocks of T, whose upper
    // parts are never written
    for (int e = tid; e < C * LD; e += NT) (&Tm[0][0])[e] = 0.f;
    // this block's group has landed (block 0 of 16-token blocks: the state's group,
    // issued after it, may still be in flight)
    if (C == 16 && c == 0)
      cp_async_wait<2>();
    else
      cp_async_wait<1>();
    __syncthreads();
    char *Kb = sm.K[buf], *Qb = sm.Q[buf], *Vb = sm.V[buf];

    // in-block inclusive cumsum of g (padding contributes 0), e^G, e^(G_C - G), beta --
    // warp 0, while the Gram products (which do not need the gates) run
    if (warp == 0) {
      constexpr int E = (C + 31) / 32;
      float gv[E], bv[E], run = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int t = lane * E + e;
        gv[e] = t < C ? sm.gRaw[buf][t] : 0.f;
        bv[e] = t < C ? sm.bRaw[buf][t] : 0.f;
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

    // ---- decay-masked Grams (bf16 inputs, exact products): N (fp32) and the causal A
    float ga[6][4];
#pragma unroll
    for (int u = 0; u < 6; ++u)
#pragma unroll
      for (int e = 0; e < 4; ++e) ga[u][e] = 0.f;
    {
      const char *Asrc = prod ? Qb : Kb;
#pragma unroll
      for (int ks = 0; ks < kD / 16; ++ks) {
        if (n0 > 0) {
          uint32_t a[4];
          lda_p<kP128>(a, Asrc, 16 * mt0, 16 * ks, lane);
#pragma unroll
          for (int u = 0; u < 3; ++u) {
            if (u < n0) {
              uint32_t b[4];
              ldb_nk_p<kP128>(b, Kb, 16 * (np0 + u), 16 * ks, lane);
              mma_bf16(ga[2 * u], a, b[0], b[1]);
              mma_bf16(ga[2 * u + 1], a, b[2], b[3]);
            }
          }
        }
        if (mt1 >= 0) {
          uint32_t a[4], b[4];
          lda_p<kP128>(a, Asrc, 16 * mt1, 16 * ks, lane);
          ldb_nk_p<kP128>(b, Kb, 0, 16 * ks, lane);
          mma_bf16(ga[4], a, b[0], b[1]);
          mma_bf16(ga[5], a, b[2], b[3]);
        }
      }
    }
    __syncthreads();  // G, EG, ED, B written; Grams done with the bf16 tiles
#pragma unroll
    for (int u = 0; u < 3; ++u) {
      int mt, np;
      if (u < n0) {
        mt = mt0;
        np = np0 + u;
      } else if (u == 2 && mt1 >= 0) {
        mt = mt1;
        np = 0;
      } else {
        continue;
      }
#pragma unroll
      for (int half = 0; half < 2; ++half)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int t = 16 * mt + gid + 8 * hr, j = 16 * np + 8 * half + 2 * tig;
          const float gt = sm.G[t];
          const float d0 = decay_exp(gt - sm.G[j]), d1 = decay_exp(gt - sm.G[j + 1]);
          const float v0 = ga[2 * u + half][2 * hr], v1 = ga[2 * u + half][2 * hr + 1];
          if (prod == 0) {
            const float bt = sm.B[t];
            Nm[t][j] = (j < t) ? bt * d0 * v0 : 0.f;
            Nm[t][j + 1] = (j + 1 < t) ? bt * d1 * v1 : 0.f;
          } else {
            *reinterpret_cast<uint32_t *>(sm.A + t * RC + 2 * j) =
                pack_f16((j <= t) ? d0 * v0 : 0.f, (j + 1 <= t) ? d1 * v1 : 0.f);
          }
        }
    }
    // the A tile's upper 16x16 blocks (never computed) are zero
    for (int e = tid; e < C * C / 2; e += NT) {
      const int t = e / (C / 2), j = 2 * (e % (C / 2));
      if ((j >> 4) > (t >> 4)) *reinterpret_cast<uint32_t *>(sm.A + t * RC + 2 * j) = 0u;
    }
    __syncthreads();

    // ---- T = (I + N)^-1 by block doubling: 16x16 diagonal blocks by forward
    // substitution (a thread per column; x[m] = 0 above the column's diagonal), then
    // (D + C)^-1 = D^-1 - D^-1 C D^-1 on 16 -> 32 -> 64 with tensor-core products.
    // Meanwhile the other threads convert the q, k, v tiles to fp16 in place.
    if (tid < C) {
      const int base = (tid >> 4) * 16, cc = tid & 15;
      float x[16];
      unit_tril_inverse_col(&Nm[base][base], LD, cc, x);
#pragma unroll
      for (int r = 0; r < 16; ++r) Tm[base + r][base + cc] = x[r];
    } else {
      const int t2 = tid - C, n2 = NT - C;
      for (int e = t2; e < C * 64; e += n2) {  // 64 packed pairs per 128-element row
        const int r = e >> 6, cp = e & 63;
        uint32_t *pk = reinterpret_cast<uint32_t *>(Kb + r * kP128) + cp;
        uint32_t *pq = reinterpret_cast<uint32_t *>(Qb + r * kP128) + cp;
        uint32_t *pv = reinterpret_cast<uint32_t *>(Vb + r * kP128) + cp;
        *pk = bf16x2_to_f16x2(*pk);
        *pq = bf16x2_to_f16x2(*pq);
        *pv = bf16x2_to_f16x2(*pv);
      }
    }
    __syncthreads();
    if (C >= 32) {
      const int pr = warp >> 1, top = 32 * pr, bot = top + 16, nb = 8 * (warp & 1);
      const bool act = warp < 2 * (C / 32);
      if (act) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        mma_f32x3f(acc, &Nm[bot][top], LD, &Tm[top][top], LD, 0, 0, nb, lane);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          sm.M[pr * 256 + (gid + 8 * (e >> 1)) * 16 + nb + 2 * tig + (e & 1)] = acc[e];
      }
      __syncthreads();
      if (act) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        mma_f32x3f(acc, &Tm[bot][bot], LD, &sm.M[pr * 256], 16, 0, 0, nb, lane);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          Tm[bot + gid + 8 * (e >> 1)][top + nb + 2 * tig + (e & 1)] = -acc[e];
      }
      __syncthreads();
    }
    if (C == 64) {
      const int r0 = 16 * ((warp >> 1) & 1), nb = 16 * (warp & 1);
      const bool act = warp < 4;
      if (act) {
        float acc[2][4] = {};
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int ks = 0; ks < 2; ++ks)
            mma_f32x3f(acc[a], &Nm[32][0], LD, &Tm[0][0], LD, r0, 16 * ks, nb + 8 * a, lane);
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            sm.M[(r0 + gid + 8 * (e >> 1)) * 33 + nb + 8 * a + 2 * tig + (e & 1)] = acc[a][e];
      }
      __syncthreads();
      if (act) {
        float acc[2][4] = {};
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int ks = 0; ks < 2; ++ks)
            mma_f32x3f(acc[a], &Tm[32][32], LD, sm.M, 33, r0, 16 * ks, nb + 8 * a, lane);
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            Tm[32 + r0 + gid + 8 * (e >> 1)][nb + 8 * a + 2 * tig + (e & 1)] = -acc[a][e];
      }
      __syncthreads();
    }

    // ---- fp16 operands T diag(beta exp G) and T diag(beta) (upper part masked)
    for (int e = tid; e < C * C / 2; e += NT) {
      const int t = e / (C / 2), j = 2 * (e % (C / 2));
      const float x0 = (j <= t) ? Tm[t][j] : 0.f, x1 = (j + 1 <= t) ? Tm[t][j + 1] : 0.f;
      *reinterpret_cast<uint32_t *>(sm.TW + t * RC + 2 * j) =
          pack_f16(x0 * sm.B[j] * sm.EG[j], x1 * sm.B[j + 1] * sm.EG[j + 1]);
      *reinterpret_cast<uint32_t *>(sm.TU + t * RC + 2 * j) =
          pack_f16(x0 * sm.B[j], x1 * sm.B[j + 1]);
    }
    __syncthreads();

    // ---- W = T diag(beta e^G) K  [t][i], this warp's 16 key columns
    {
      const int i0 = 16 * warp;
#pragma unroll 1
      for (int mt = 0; mt < MT; ++mt) {
        float acc[2][4] = {};
        for (int ks = 0; ks <= mt; ++ks) {
          uint32_t a[4], b[4];
          lda_p<RC>(a, sm.TW, 16 * mt, 16 * ks, lane);
          ldb_kn_p<kP128>(b, Kb, 16 * ks, i0, lane);
          mma_f16(acc[0], a, b[0], b[1]);
          mma_f16(acc[1], a, b[2], b[3]);
        }
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int t = 16 * mt + gid + 8 * hr, col = i0 + 8 * a + 2 * tig;
            *reinterpret_cast<uint32_t *>(sm.W + t * kP128 + 2 * col) =
                pack_f16(acc[a][2 * hr], acc[a][2 * hr + 1]);
          }
      }
    }
    if (C == 16 && c == 0) cp_async_wait<1>();  // the state has landed as well
    __syncthreads();
    if constexpr (C == 16) {
      if (c == 0) state_from_staging();
    }

    // ================= per-warp state chain for value columns j0 .. j0+15
    // D^T = V^T T_u^T  (U^T), then minus S^T W^T
    float Dc[NTC][4];
#pragma unroll
    for (int a = 0; a < NTC; ++a)
#pragma unroll
      for (int e = 0; e < 4; ++e) Dc[a][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < MT; ++ks) {
      uint32_t a[4];
      lda_t_p<kP128>(a, Vb, j0, 16 * ks, lane);
#pragma unroll
      for (int np = 0; np < MT; ++np) {
        if (np >= ks) {
          uint32_t b[4];
          ldb_nk_p<RC>(b, sm.TU, 16 * np, 16 * ks, lane);
          mma_f16(Dc[2 * np], a, b[0], b[1]);
          mma_f16(Dc[2 * np + 1], a, b[2], b[3]);
        }
      }
    }
    float Rc[NTC][4];
#pragma unroll
    for (int a = 0; a < NTC; ++a)
#pragma unroll
      for (int e = 0; e < 4; ++e) Rc[a][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < kD / 16; ++ks) {
      uint32_t sf[4], nf[4];
      acc_to_f16(S[2 * ks], S[2 * ks + 1], 1.f, 1.f, 1.f, 1.f, sf);
#pragma unroll
      for (int e = 0; e < 4; ++e) nf[e] = sf[e] ^ 0x80008000u;  // -S
#pragma unroll
      for (int np = 0; np < MT; ++np) {
        uint32_t bw[4], bq[4];
        ldb_nk_p<kP128>(bw, sm.W, 16 * np, 16 * ks, lane);
        ldb_nk_p<kP128>(bq, Qb, 16 * np, 16 * ks, lane);
#pragma unroll
        for (int a = 0; a < 2; ++a) {
          mma_f16(Dc[2 * np + a], nf, bw[2 * a], bw[2 * a + 1]);
          mma_f16(Rc[2 * np + a], sf, bq[2 * a], bq[2 * a + 1]);
        }
      }
    }
    if (p.delta) {  // the block's per-token deltas (fp32, before any rounding)
#pragma unroll
      for (int nt = 0; nt < NTC; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int t = 8 * nt + 2 * tig + (e & 1);
          if (t < L)
            p.delta[((size_t)(tok0 + t) * p.hv + h) * kD + j0 + gid + 8 * (e >> 1)] = Dc[nt][e];
        }
    }
    // O^T = exp(G) R^T + D^T A^T over the causal part
#pragma unroll
    for (int nt = 0; nt < NTC; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) Rc[nt][e] *= sm.EG[8 * nt + 2 * tig + (e & 1)];
#pragma unroll
    for (int ks = 0; ks < MT; ++ks) {
      uint32_t df[4];
      acc_to_f16(Dc[2 * ks], Dc[2 * ks + 1], 1.f, 1.f, 1.f, 1.f, df);
#pragma unroll
      for (int np = 0; np < MT; ++np) {
        if (np >= ks) {
          uint32_t b[4];
          ldb_nk_p<RC>(b, sm.A, 16 * np, 16 * ks, lane);
#pragma unroll
          for (int a = 0; a < 2; ++a) mma_f16(Rc[2 * np + a], df, b[2 * a], b[2 * a + 1]);
        }
      }
    }
    // stage O^T [j][t] as rows t and store this warp's 16 columns of the valid rows
#pragma unroll
    for (int nt = 0; nt < NTC; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        Elem<TO>::store(&Ost[warp][8 * nt + 2 * tig + (e & 1)][gid + 8 * (e >> 1)], Rc[nt][e]);
    __syncwarp();
    {
      constexpr int EPG = 16 / sizeof(TO);
      constexpr int GPR = 16 / EPG;
      for (int e = lane; e < C * GPR; e += 32) {
        const int t = e / GPR, gi = e % GPR;
        if (t < L)
          *reinterpret_cast<uint4 *>(o + ((size_t)(tok0 + t) * p.hv + h) * kD + j0 + gi * EPG) =
              *reinterpret_cast<const uint4 *>(&Ost[warp][t][gi * EPG]);
      }
    }
    // S^T <- exp(G_T) S^T + (D^T diag(exp(G_T - G))) K
    const float egc = sm.EG[C - 1];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) S[nt][e] *= egc;
#pragma unroll
    for (int ks = 0; ks < MT; ++ks) {
      const int t0 = 16 * ks + 2 * tig;
      uint32_t tf[4];
      acc_to_f16(Dc[2 * ks], Dc[2 * ks + 1], sm.ED[t0], sm.ED[t0 + 1], sm.ED[t0 + 8],
                 sm.ED[t0 + 9], tf);
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        uint32_t b[4];
        ldb_kn_p<kP128>(b, Kb, 16 * ks, 16 * np, lane);
        mma_f16(S[2 * np], tf, b[0], b[1]);
        mma_f16(S[2 * np + 1], tf, b[2], b[3]);
      }
    }
  }

  if constexpr (C == 16) {  // back through the staging area, 16-byte stores along rows
    __syncthreads();  // (defensive: nothing else uses the staging area after the start)
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = 8 * nt + 2 * tig + (e & 1), j = j0 + gid + 8 * (e >> 1);
        sm.SS[i][j] = S[nt][e];
      }
    __syncthreads();
    for (int e = tid; e < kD * kD / 4; e += NT) {
      const int r = e >> 5, c4 = e & 31;
      *reinterpret_cast<float4 *>(p.state_out + sbase + (size_t)r * kD + 4 * c4) =
          *reinterpret_cast<const float4 *>(&sm.SS[r][4 * c4]);
    }
  } else {
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = 8 * nt + 2 * tig + (e & 1), j = j0 + gid + 8 * (e >> 1);
        p.state_out[sbase + (size_t)i * kD + j] = S[nt][e];
      }
  }
}

template <int C, typename TO>
cudaError_t launch_fused_t(const ChunkParams &p, cudaStream_t stream) {
  const size_t smem = sizeof(FusedSmem<C, TO>);
  cudaError_t err = cudaFuncSetAttribute(fused_kernel<C, TO>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  fused_kernel<C, TO><<<(unsigned)((long long)p.num_seqs * p.hv), kFThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int C>
cudaError_t launch_fused_c(const ChunkParams &p, cudaStream_t stream) {
  return p.o_fp32 ? launch_fused_t<C, float>(p, stream) : launch_fused_t<C, __nv_bfloat16>(p, stream);
}

}  // namespace

cudaError_t launch_chunk_fused(const ChunkParams &p, cudaStream_t stream) {
  if ((long long)p.num_seqs * p.hv == 0) return cudaSuccess;
  switch (p.chunk) {
    case 16: return launch_fused_c<16>(p, stream);
    case 32: return launch_fused_c<32>(p, stream);
    case 64: return launch_fused_c<64>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace gdn
