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
//     products W, U on tensor cores.
//     The doubling levels run on tensor cores with 3-term bf16 splits of the fp32
//     operands.  Each block's results go to its own workspace slot, already in the
//     swizzled shared-memory layout pass 2 uses.
//   pass 2 (recur_kernel, one CTA per (sequence, v-head, 16 value columns)): walks the
//     blocks of the sequence in order with the state block S[:, cols] in fp32 registers
//     (read from state_in once, written to state_out once).  A producer warp streams
//     each block's slot into a 2-stage shared-memory ring with bulk (TMA) copies
//     signalled on mbarriers.  Four "state" warps run the dependent chain
//       P = W S and D = U - P (each for 16 tokens),
//       S <- exp(G_T) S + K^T diag(exp(G_T - G)) D (each for 32 keys),
//     and four "output" warps form O = exp(G) Q S + A D for the same block from a
//     snapshot of S.  All products run on mma.sync tensor cores, fp32 accumulation.
// Precision: q, k, v are bf16 inputs and enter the products exactly.  T, the state, D
// and A are fp32 values carried as two bf16 numbers, hi = bf16(x), lo = bf16(x - hi),
// with products hi*y + lo*y (~16 significant bits); W is rounded to bf16 once.  The
// layer's outputs have heavy tails (max/rms above 10), so single-bf16 copies of those
// operands would put errors of a few 1e-2 of the rms on the largest entries.
// Decay factors between two tokens are always the exp of a difference of cumsums.  A
// partly filled block is padded with g = 0, beta = 0, zero q/k/v rows (token_valid),
// which leaves the state exactly as after the sequence's last token.
#include "common.cuh"
#include "internal.h"

namespace gdn {

namespace {

constexpr int kRowB = kD * 2;  // bytes in a 128-element bf16 row

__device__ __forceinline__ size_t slot_index(int bos, int chunk, int n, int c) {
  return (size_t)(bos / chunk + n + c);
}

// acc (16x8 tile) += A[r0.., k0..k0+16) * B[k0.., n0..n0+8) for fp32 row-major matrices in
// shared memory, as hi*hi + lo*hi + hi*lo of their bf16 splits (~16 significant bits).
__device__ __forceinline__ void mma_f32x3(float (&acc)[4], const float *A, int lda,
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
  float gRaw[C], bRaw[C];
};

constexpr int kPrepThreads = 256;

template <int C>
__global__ void __launch_bounds__(kPrepThreads) prep_kernel(ChunkParams p, int per_head) {
  constexpr int NW = kPrepThreads / 32, NT = kPrepThreads, MT = C / 16, RB = 2 * C, LD = C + 4;
  static_assert(8 * C * C <= C * kRowB + C * (C + 4) * 4, "overlay too small");
  extern __shared__ __align__(128) unsigned char smem_raw[];
  PrepSmem<C> &sm = *reinterpret_cast<PrepSmem<C> *>(smem_raw);
  char *sQ = sm.X;
  float(*sN)[LD] = reinterpret_cast<float(*)[LD]>(sm.X + C * kRowB);
  char *TWH = sm.X, *TWL = sm.X + C * RB, *TUH = sm.X + 2 * C * RB, *TUL = sm.X + 3 * C * RB;

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

  int bos, eos;
  seq_range(p.cu_seqlens, n, p.total_tokens, bos, eos);
  const int nchunks = (eos - bos + C - 1) / C;

  for (int c = part; c < nchunks; c += per_head) {
    const int tok0 = bos + c * C;
    const int L = min(C, eos - tok0);
    char *slot = p.slot_ws + ((size_t)h * p.nslots + slot_index(bos, C, n, c)) * slot_bytes(C);
    char *w_out = slot, *q_out = slot + 256 * C, *k_out = slot + 512 * C;
    char *ah_out = slot + 768 * C, *al_out = slot + 768 * C + 2 * C * C;
    float *u_out = reinterpret_cast<float *>(slot + slot_head_bytes(C));
    float *g_out = reinterpret_cast<float *>(slot + slot_head_bytes(C) + slot_u_bytes(C));
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
    for (int t = tid; t < C; t += NT) {
      const bool ok = t < L;
      const size_t gi = ((size_t)tok0 + (ok ? t : 0)) * p.hv + h;
      cp_async4(&sm.gRaw[t], p.g + gi, ok ? 4 : 0);
      cp_async4(&sm.bRaw[t], p.beta + gi, ok ? 4 : 0);
    }
    cp_async_commit();
    for (int e = tid; e < C * LD; e += NT) (&sm.T[0][0])[e] = 0.f;
    cp_async_wait<0>();
    __syncthreads();

    // in-block inclusive cumsum of g (padding contributes 0), exp(G), beta
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
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int t = lane * E + e;
        if (t < C) {
          sm.G[t] = gv[e] + excl;
          sm.EG[t] = __expf(gv[e] + excl);
          sm.B[t] = bv[e];
          g_out[t] = gv[e] + excl;
        }
      }
    }

    // the block's q and k rows (swizzled, zero past the sequence end) go to the slot as is
    for (int e = tid; e < C * 16; e += NT) {
      reinterpret_cast<uint4 *>(q_out)[e] = reinterpret_cast<const uint4 *>(sQ)[e];
      reinterpret_cast<uint4 *>(k_out)[e] = reinterpret_cast<const uint4 *>(sm.K)[e];
    }
    __syncthreads();  // G, EG, B written by warp 0

    // ---- decay-masked Grams on tensor cores: warp w takes items 2w, 2w+1 of
    //      [KK(0), KK(MT-1), KK(1), ..., QK(0), QK(MT-1), ...] (balanced triangles)
#pragma unroll 1
    for (int item = warp; item < 2 * MT; item += NW) {
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
          float x0 = 0.f, x1 = 0.f;
          if (nt <= 2 * mt + 1) {
            const float d0 = __expf(sm.G[t] - sm.G[j]), d1 = __expf(sm.G[t] - sm.G[j + 1]);
            if (prod == 0) {
              x0 = (j < t) ? sm.B[t] * d0 * acc[nt][2 * hr] : 0.f;
              x1 = (j + 1 < t) ? sm.B[t] * d1 * acc[nt][2 * hr + 1] : 0.f;
            } else {
              x0 = (j <= t) ? d0 * acc[nt][2 * hr] : 0.f;
              x1 = (j + 1 <= t) ? d1 * acc[nt][2 * hr + 1] : 0.f;
            }
          }
          if (prod == 0) {
            if (nt <= 2 * mt + 1) {
              sN[t][j] = x0;
              sN[t][j + 1] = x1;
            }
          } else {
            uint32_t hi, lo;
            split_bf16(x0, x1, hi, lo);
            *reinterpret_cast<uint32_t *>(ah_out + swz<RB>(t, 2 * j)) = hi;
            *reinterpret_cast<uint32_t *>(al_out + swz<RB>(t, 2 * j)) = lo;
          }
        }
      }
    }
    __syncthreads();

    // ---- T = (I + N)^-1 by block doubling.  Level 0: 16x16 diagonal blocks in fp32,
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
    // Level 1 (16 -> 32): lower-left block = -T_bot (N_bl T_top); one 16x8 tile per warp.
    if (C >= 32) {
      const int pr = warp >> 1, top = 32 * pr, bot = top + 16, n0 = 8 * (warp & 1);
      if (warp < 2 * (C / 32)) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        mma_f32x3(acc, &sN[bot][top], LD, &sm.T[top][top], LD, 0, 0, n0, lane);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          sm.M[pr * 256 + (gid + 8 * (e >> 1)) * 16 + n0 + 2 * tig + (e & 1)] = acc[e];
      }
      __syncthreads();
      if (warp < 2 * (C / 32)) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        mma_f32x3(acc, &sm.T[bot][bot], LD, &sm.M[pr * 256], 16, 0, 0, n0, lane);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          sm.T[bot + gid + 8 * (e >> 1)][top + n0 + 2 * tig + (e & 1)] = -acc[e];
      }
      __syncthreads();
    }
    // Level 2 (32 -> 64): lower-left 32x32 block = -T_BB (N_BA T_AA); two tiles per warp.
    if (C == 64) {
      const int r0 = 16 * ((warp >> 1) & 1), nb = 16 * (warp & 1);
      const bool lv2 = warp < 4;
      if (lv2) {
        float acc[2][4] = {};
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int ks = 0; ks < 2; ++ks)
            mma_f32x3(acc[a], &sN[32][0], LD, &sm.T[0][0], LD, r0, 16 * ks, nb + 8 * a, lane);
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            sm.M[(r0 + gid + 8 * (e >> 1)) * 33 + nb + 8 * a + 2 * tig + (e & 1)] = acc[a][e];
      }
      __syncthreads();
      if (lv2) {
        float acc2[2][4] = {};
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int ks = 0; ks < 2; ++ks)
            mma_f32x3(acc2[a], &sm.T[32][32], LD, sm.M, 33, r0, 16 * ks, nb + 8 * a, lane);
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            sm.T[32 + r0 + gid + 8 * (e >> 1)][nb + 8 * a + 2 * tig + (e & 1)] = -acc2[a][e];
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

    // ---- W = T diag(beta e^G) K  [t][i]: this warp's 128/NW key columns, all rows.
    //      Causal: T[t][j] = 0 for j > t.
    {
      constexpr int NTI = 16 / NW;  // 8-wide n-tiles of keys per warp
      const int i0 = warp * (kD / NW);
#pragma unroll 1
      for (int mt = 0; mt < MT; ++mt) {
        float acc[NTI][4];
#pragma unroll
        for (int a = 0; a < NTI; ++a)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[a][e] = 0.f;
        for (int ks = 0; ks <= mt; ++ks) {
          uint32_t ah[4], al[4];
          lda_tile<RB>(ah, TWH, 16 * mt, 16 * ks, lane);
          lda_tile<RB>(al, TWL, 16 * mt, 16 * ks, lane);
#pragma unroll
          for (int np = 0; np < NTI / 2; ++np) {
            uint32_t b[4];
            ldb_kn<kRowB>(b, sm.K, 16 * ks, i0 + 16 * np, lane);
            mma_bf16(acc[2 * np], ah, b[0], b[1]);
            mma_bf16(acc[2 * np], al, b[0], b[1]);
            mma_bf16(acc[2 * np + 1], ah, b[2], b[3]);
            mma_bf16(acc[2 * np + 1], al, b[2], b[3]);
          }
        }
#pragma unroll
        for (int nt = 0; nt < NTI; ++nt)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int t = 16 * mt + gid + 8 * hr, col = i0 + 8 * nt + 2 * tig;
            *reinterpret_cast<uint32_t *>(w_out + swz<kRowB>(t, 2 * col)) =
                pack_bf16(acc[nt][2 * hr], acc[nt][2 * hr + 1]);
          }
      }
    }
    // ---- U^T = V^T (T diag(beta))^T  [j][t]: this warp's 128/NW value rows.
    {
      constexpr int MJ = 8 / NW;  // 16-row m-tiles of value columns per warp
#pragma unroll 1
      for (int mj = 0; mj < MJ; ++mj) {
        const int j0 = warp * (kD / NW) + 16 * mj;
        float acc[C / 8][4];
#pragma unroll
        for (int a = 0; a < C / 8; ++a)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[a][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < MT; ++ks) {
          uint32_t a[4];
          lda_tile_t<kRowB>(a, sm.V, j0, 16 * ks, lane);
#pragma unroll
          for (int np = 0; np < MT; ++np) {
            if (np >= ks) {
              uint32_t bh[4], bl[4];
              ldb_nk<RB>(bh, TUH, 16 * np, 16 * ks, lane);
              ldb_nk<RB>(bl, TUL, 16 * np, 16 * ks, lane);
              mma_bf16(acc[2 * np], a, bh[0], bh[1]);
              mma_bf16(acc[2 * np], a, bl[0], bl[1]);
              mma_bf16(acc[2 * np + 1], a, bh[2], bh[3]);
              mma_bf16(acc[2 * np + 1], a, bl[2], bl[3]);
            }
          }
        }
#pragma unroll
        for (int nt = 0; nt < C / 8; ++nt)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int j = j0 + gid + 8 * hr, t = 8 * nt + 2 * tig;
            *reinterpret_cast<float2 *>(u_out + j * (C + 4) + t) =
                make_float2(acc[nt][2 * hr], acc[nt][2 * hr + 1]);
          }
      }
    }
  }
}

// ================================================================== pass 2

constexpr int kStateWarps = 4, kOutWarps = 4;
constexpr int kRecThreads = 32 * (kStateWarps + kOutWarps + 1);  // + 1 producer warp
constexpr int kConsumers = 32 * (kStateWarps + kOutWarps);
constexpr int kDVB = 16;  // value columns per CTA

template <int C, typename TO>
struct RecSmem {
  struct Stage {  // mirrors a workspace slot: W | Q | K | Ah | Al contiguous, then U, G
    alignas(128) char W[C * kRowB];
    char Q[C * kRowB];
    char K[C * kRowB];
    char Ah[C * 2 * C];
    char Al[C * 2 * C];
    alignas(16) float U[kDVB][C + 4];  // U^T rows of this CTA's value columns
    alignas(16) float G[C];
  } st[2];
  alignas(8) uint64_t full[2], empty[2];
  alignas(128) char Sh[kDVB * kRowB];  // S^T snapshot (hi, lo)
  alignas(128) char Sl[kDVB * kRowB];
  alignas(128) char Dh[kDVB * 2 * C];  // D^T (hi, lo)
  alignas(128) char Dl[kDVB * 2 * C];
  alignas(128) char Th[kDVB * 2 * C];  // (diag(exp(G_T - G)) D)^T (hi, lo)
  alignas(128) char Tl[kDVB * 2 * C];
  alignas(16) TO O[kOutWarps][16][kDVB];
  alignas(16) float S32[kD][kDVB + 4];  // fp32 staging of the state block
};

template <int C, typename TO>
__global__ void __launch_bounds__(kRecThreads) recur_kernel(ChunkParams p) {
  constexpr int NB = kD / kDVB, TT = C / 16, RB = 2 * C;
  constexpr uint32_t kHeadB = (uint32_t)slot_head_bytes(C);
  constexpr uint32_t kUB = (uint32_t)(kDVB * (C + 4) * 4);
  constexpr uint32_t kStageTx = kHeadB + kUB + 4 * C;
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
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
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

  if (warp == kStateWarps + kOutWarps) {
    // ---- producer: stream block slots into the 2-stage ring
    if (lane == 0) {
      bool ok = true;
      for (int c = 0; c < nchunks; ++c) {
        const int s = c & 1;
        if (c >= 2) ok = mbar_wait(&sm.empty[s], ((c - 2) >> 1) & 1) && ok;
        const char *src = slot0 + (size_t)c * slot_bytes(C);
        mbar_arrive_expect_tx(&sm.full[s], kStageTx);
        bulk_g2s(sm.st[s].W, src, kHeadB, &sm.full[s]);
        bulk_g2s(&sm.st[s].U[0][0], src + kHeadB + (size_t)blk * kUB, kUB, &sm.full[s]);
        bulk_g2s(sm.st[s].G, src + kHeadB + slot_u_bytes(C), 4 * C, &sm.full[s]);
      }
      // the last copies are consumed before the CTA's final barrier
      if (!ok) atomicExch(p.err, 1);
    }
  } else if (warp < kStateWarps) {
    // ---- state warps: wq owns tokens 16wq.. (P, D) and keys 32wq.. (state carry)
    const int wq = warp;
    float Sa[4][4];  // S^T[j][i], j = gid (+8), i = 32wq + 8nt + 2tig (+1)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        Sa[nt][e] = sm.S32[32 * wq + 8 * nt + 2 * tig + (e & 1)][gid + 8 * (e >> 1)];
    auto write_snapshot = [&]() {
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int j = gid + 8 * hr, i = 32 * wq + 8 * nt + 2 * tig;
          uint32_t hi, lo;
          split_bf16(Sa[nt][2 * hr], Sa[nt][2 * hr + 1], hi, lo);
          *reinterpret_cast<uint32_t *>(sm.Sh + swz<kRowB>(j, 2 * i)) = hi;
          *reinterpret_cast<uint32_t *>(sm.Sl + swz<kRowB>(j, 2 * i)) = lo;
        }
    };
    write_snapshot();
    bar_sync(2, kConsumers);
    bool ok = true;
#pragma unroll 1
    for (int c = 0; c < nchunks; ++c) {
      const int s = c & 1;
      typename Smem::Stage &st = sm.st[s];
      ok = mbar_wait(&sm.full[s], (c >> 1) & 1) && ok;
      const float gC = st.G[C - 1];
      if (wq < TT) {
        // P^T = S^T W^T for this warp's 16 tokens (k split in halves for shorter chains)
        float Ph[2][2][4], Pl[2][2][4];
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
          for (int a = 0; a < 2; ++a)
#pragma unroll
            for (int e = 0; e < 4; ++e) Ph[x][a][e] = Pl[x][a][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
          uint32_t sh[4], sl[4], bw[4];
          lda_tile<kRowB>(sh, sm.Sh, 0, 16 * ks, lane);
          lda_tile<kRowB>(sl, sm.Sl, 0, 16 * ks, lane);
          ldb_nk<kRowB>(bw, st.W, 16 * wq, 16 * ks, lane);
          const int x = ks & 1;
#pragma unroll
          for (int a = 0; a < 2; ++a) {
            mma_bf16(Ph[x][a], sh, bw[2 * a], bw[2 * a + 1]);
            mma_bf16(Pl[x][a], sl, bw[2 * a], bw[2 * a + 1]);
          }
        }
        // D = U - P, and its carry-scaled copy, as bf16 (hi, lo) for the other warps
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int j = gid + 8 * hr, t = 16 * wq + 8 * a + 2 * tig;
            const float2 u = *reinterpret_cast<const float2 *>(&st.U[j][t]);
            const int e0 = 2 * hr, e1 = 2 * hr + 1;
            const float d0 = u.x - ((Ph[0][a][e0] + Pl[0][a][e0]) + (Ph[1][a][e0] + Pl[1][a][e0]));
            const float d1 = u.y - ((Ph[0][a][e1] + Pl[0][a][e1]) + (Ph[1][a][e1] + Pl[1][a][e1]));
            const int so = swz<RB>(j, 2 * t);
            uint32_t hi, lo;
            split_bf16(d0, d1, hi, lo);
            *reinterpret_cast<uint32_t *>(sm.Dh + so) = hi;
            *reinterpret_cast<uint32_t *>(sm.Dl + so) = lo;
            split_bf16(d0 * __expf(gC - st.G[t]), d1 * __expf(gC - st.G[t + 1]), hi, lo);
            *reinterpret_cast<uint32_t *>(sm.Th + so) = hi;
            *reinterpret_cast<uint32_t *>(sm.Tl + so) = lo;
          }
      }
      bar_sync(1, kConsumers);
      // S^T <- exp(G_T) S^T + Dt^T K over this warp's 32 keys
      float Xh[4][4], Xl[4][4];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int e = 0; e < 4; ++e) Xh[a][e] = Xl[a][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < TT; ++ks) {
        uint32_t th[4], tl[4];
        lda_tile<RB>(th, sm.Th, 0, 16 * ks, lane);
        lda_tile<RB>(tl, sm.Tl, 0, 16 * ks, lane);
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          uint32_t b[4];
          ldb_kn<kRowB>(b, st.K, 16 * ks, 32 * wq + 16 * np, lane);
          mma_bf16(Xh[2 * np], th, b[0], b[1]);
          mma_bf16(Xl[2 * np], tl, b[0], b[1]);
          mma_bf16(Xh[2 * np + 1], th, b[2], b[3]);
          mma_bf16(Xl[2 * np + 1], tl, b[2], b[3]);
        }
      }
      const float egc = __expf(gC);
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) Sa[nt][e] = egc * Sa[nt][e] + (Xh[nt][e] + Xl[nt][e]);
      write_snapshot();
      bar_sync(2, kConsumers);
      if (tid == 0) mbar_arrive(&sm.empty[s]);
    }
    if (!ok && lane == 0) atomicExch(p.err, 1);
    // final state block -> fp32 staging
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        sm.S32[32 * wq + 8 * nt + 2 * tig + (e & 1)][gid + 8 * (e >> 1)] = Sa[nt][e];
  } else {
    // ---- output warps: wq owns tokens 16wq..16wq+15
    const int wq = warp - kStateWarps;
    bar_sync(2, kConsumers);
    bool ok = true;
#pragma unroll 1
    for (int c = 0; c < nchunks; ++c) {
      const int s = c & 1;
      typename Smem::Stage &st = sm.st[s];
      ok = mbar_wait(&sm.full[s], (c >> 1) & 1) && ok;
      const int tok0 = bos + c * C;
      const int L = min(C, eos - tok0);
      float Rh[2][2][4], Rl[2][2][4];  // [k half][n-tile][.]
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int e = 0; e < 4; ++e) Rh[x][a][e] = Rl[x][a][e] = 0.f;
      if (wq < TT) {
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks) {
          uint32_t sh[4], sl[4], bq[4];
          lda_tile<kRowB>(sh, sm.Sh, 0, 16 * ks, lane);
          lda_tile<kRowB>(sl, sm.Sl, 0, 16 * ks, lane);
          ldb_nk<kRowB>(bq, st.Q, 16 * wq, 16 * ks, lane);
          const int x = ks & 1;
#pragma unroll
          for (int a = 0; a < 2; ++a) {
            mma_bf16(Rh[x][a], sh, bq[2 * a], bq[2 * a + 1]);
            mma_bf16(Rl[x][a], sl, bq[2 * a], bq[2 * a + 1]);
          }
        }
      }
      bar_sync(1, kConsumers);
      if (wq < TT) {
        // O^T = exp(G) R^T + D^T A^T over the causal part of the block
        float O1[2][4], O2[2][4], O3[2][4];
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int e = 0; e < 4; ++e) O1[a][e] = O2[a][e] = O3[a][e] = 0.f;
        for (int ks = 0; ks <= wq; ++ks) {
          uint32_t dh[4], dl[4], bh[4], bl[4];
          lda_tile<RB>(dh, sm.Dh, 0, 16 * ks, lane);
          lda_tile<RB>(dl, sm.Dl, 0, 16 * ks, lane);
          ldb_nk<RB>(bh, st.Ah, 16 * wq, 16 * ks, lane);
          ldb_nk<RB>(bl, st.Al, 16 * wq, 16 * ks, lane);
#pragma unroll
          for (int a = 0; a < 2; ++a) {
            mma_bf16(O1[a], dh, bh[2 * a], bh[2 * a + 1]);
            mma_bf16(O2[a], dl, bh[2 * a], bh[2 * a + 1]);
            mma_bf16(O3[a], dh, bl[2 * a], bl[2 * a + 1]);
          }
        }
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int t = 16 * wq + 8 * a + 2 * tig + (e & 1);
            const float r = (Rh[0][a][e] + Rl[0][a][e]) + (Rh[1][a][e] + Rl[1][a][e]);
            Elem<TO>::store(&sm.O[wq][t - 16 * wq][gid + 8 * (e >> 1)],
                            __expf(st.G[t]) * r + (O1[a][e] + O2[a][e] + O3[a][e]));
          }
        __syncwarp();
        constexpr int EPG = 16 / sizeof(TO);  // elements per 16-byte granule
        constexpr int GPR = kDVB / EPG;       // granules per output row
        for (int e = lane; e < 16 * GPR; e += 32) {
          const int r = e / GPR, gi = e % GPR, t = 16 * wq + r;
          if (t < L)
            *reinterpret_cast<uint4 *>(o + ((size_t)(tok0 + t) * p.hv + h) * kD + blk * kDVB +
                                       gi * EPG) =
                *reinterpret_cast<const uint4 *>(&sm.O[wq][r][gi * EPG]);
        }
      }
      bar_sync(2, kConsumers);
    }
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
  recur_kernel<C, TO><<<(unsigned)(heads * (kD / kDVB)), kRecThreads, s2, stream>>>(p);
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
  // prep CTAs per (sequence, head): enough to fill the GPU a few times over
  long long per_head = (4LL * sms + heads - 1) / heads;
  per_head = max(1LL, min(per_head, max(1LL, max_chunks)));

  if (p.total_tokens > 0) {
    const size_t s1 = sizeof(PrepSmem<C>);
    err = cudaFuncSetAttribute(prep_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1);
    if (err != cudaSuccess) return err;
    prep_kernel<C><<<(unsigned)(heads * per_head), kPrepThreads, s1, stream>>>(p, (int)per_head);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  return p.o_fp32 ? launch_recur<C, float>(p, heads, stream)
                  : launch_recur<C, __nv_bfloat16>(p, heads, stream);
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
