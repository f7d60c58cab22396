// Single-pass chunkwise gated delta rule on the tcgen05 tensor cores, 64-token blocks,
// bf16 q/k/v ("Qwen3.5-9B-npu" model card, section "How it works", chunkwise form):
//   N   = diag(beta) [exp(G_t - G_j) k_t.k_j]_{j<t},   A = [exp(G_t - G_j) q_t.k_j]_{j<=t}
//   [W U] = (I + N)^-1 [diag(beta exp G) K  diag(beta) V]
//   D   = U - W S,   O = diag(exp G) Q S + A D,   S_T = exp(G_T) S + K^T diag(exp(G_T - G)) D
//
// One CTA per (sequence, v-head) walks the sequence's blocks in order; the whole 128 x 128
// state stays in tensor memory (fp32) for the sequence, read from state_in once and
// written to state_out once.  With the 128 value columns as the M = 128 rows of every
// state product, each block's operands are read from shared memory once per head:
//   P1: D^T  = -S^T W^T              (A = S^T fp16 in tensor memory, B = W^T in smem)
//   P3: R^T  =  S^T (diag(e^G) Q)^T  (same A)
//   P2: S^T +=  (D diag(e^(G_T - G)))^T K   (S^T pre-scaled by e^(G_T) in tensor memory)
//   P4: O^T  = R^T + D^T A^T
// Warp roles:
//   warps 0-3  ("E", lane = value column): D = U + P1 into fp16 operands in tensor memory;
//              the state epilogue (fp16 copy of S for the next block's P1/P3, then the
//              pre-scaling by the next block's e^(G_T)); the outputs O -> o.
//   warps 4-11 ("P"): the state-free part of the *next* block while the chain runs: q, k,
//              v loads one block ahead (cp.async), the in-block cumsum, the epilogue of
//              the Gram MMA [K; Q] K^T (decay masks -> N and A), the 16x16 diagonal
//              inverses of I + N by forward substitution, and W, U by blocked forward
//              substitution on mma.sync (as in the two-pass path).
//   warp 12 lane 0: issues every tcgen05 MMA and its commits.
// Hand-offs are mbarriers (bounded waits; a wait that gives up reports
// GDN_STATUS_WAIT_TIMEOUT to the device status word: results are then unspecified, the
// kernel still returns).
// Precision: the Gram MMA takes the exact bf16 q, k; every other product takes fp16
// operands (q, k, v exact; S, D, W, A rounded to 11 bits for the product) with fp32
// accumulation, as in the mma.sync paths.
#include <stddef.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace gdn {

namespace {

using tc::at_off;
using tc::t64_off;
using tc::wt_off;

constexpr int kTcC = 64;                 // block length of this kernel
constexpr int kTcThreads = 32 * 13;      // 4 E + 8 P warps + the MMA issuer warp
constexpr int kTcE = 128, kTcP = 256;    // threads of the E and P groups
constexpr int kBarE = 1, kBarP = 2;      // named barriers of the groups
constexpr int kTcLptSeqs = 64;           // longest-first CTA order up to this many sequences

// tensor-memory columns (512 allocated)
constexpr int kTmS = 0;      // S^T fp32 [128 value cols][128 keys]
constexpr int kTmST = 128;   // S^T fp16 pairs (A operand of P1, P3)
constexpr int kTmD = 192;    // P1 accumulator D^T [value col][64 tokens]
constexpr int kTmR = 256;    // P3 + P4 accumulator O^T
constexpr int kTmDT = 320;   // D^T fp16 pairs (A of P4)
constexpr int kTmDD = 352;   // (D diag(e^(G_T - G)))^T fp16 pairs (A of P2)
constexpr int kTmG = 384;    // Gram [K; Q] K^T fp32 [128 rows][64 tokens]

// [K; Q] bf16, 128 rows (tokens of k, then of q) x 128 keys, K-major (no-swizzle
// core-matrix layout, 8 rows x 16 B per core matrix)
__device__ __forceinline__ int kq_off(int r, int key) {
  return (key >> 3) * 2048 + (r >> 3) * 128 + (r & 7) * 16 + (key & 7) * 2;
}

struct TcSmem {
  alignas(1024) char KQ[2][32768];        // [K; Q] bf16 of blocks c (even/odd)
  alignas(128) char Vb[kTcC * kP128];     // v bf16 rows (272-byte rows) of the next block
  alignas(128) char Wt[16384];            // W^T fp16 (wt_off)
  alignas(128) char Qt[2][16384];         // diag(e^G) Q fp16 (t64_off), by block parity
  alignas(128) char K16[2][16384];        // K fp16 (t64_off), by block parity
  alignas(128) char At[2][8192];          // A fp16 (at_off), by block parity
  alignas(16) char Ut[kD * 144];          // U^T fp16 [value col][token], 144-byte rows
  alignas(16) char N16[kTcC * 144];       // -N fp16 [t][j] below the diagonal blocks
  alignas(16) char T16[4][16 * 48];       // T_ii fp16, 48-byte rows
  float Nd[4][16][17];                    // diagonal blocks of N (fp32)
  float dec[2][3][kTcC];                  // G, e^G, e^(G_T - G) by block parity
  float gRaw[2][kTcC], bRaw[2][kTcC];
  float pB[kTcC];                         // beta of the block being prepared
  alignas(8) uint64_t gram_done, gram_free, prep_done, dec_ready[2];
  alignas(8) uint64_t p1_done, p2_done, p4_done, d_ready, s_ready, r_free, p4_buf[2];
  alignas(8) uint64_t kq_full[2], v_full;  // cp.async completions (one arrive per E thread)
  uint32_t tmem;
};

// A fragment (16 rows x 16 k) as fp16 from two 16x8 mma.sync accumulator tiles
__device__ __forceinline__ void acc_to_f16x(const float (&x)[4], const float (&y)[4], uint32_t (&a)[4]) {
  a[0] = pack_f16(x[0], x[1]);
  a[1] = pack_f16(x[2], x[3]);
  a[2] = pack_f16(y[0], y[1]);
  a[3] = pack_f16(y[2], y[3]);
}

template <typename TO>
__global__ void __launch_bounds__(kTcThreads, 1) tc_kernel(ChunkParams p) {
  constexpr int C = kTcC;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  TcSmem &sm = *reinterpret_cast<TcSmem *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Longest sequences first: with more (sequence, head) chains than SMs, CTAs start in
  // index order as SMs free up, so the long chains should not be the last to start.
  // CTA b takes head b % Hv of the (b / Hv)-th longest sequence (ties by index), for up
  // to kTcLptSeqs sequences; beyond that, in sequence order.
  const int rank = blockIdx.x / p.hv;
  const int h = blockIdx.x - rank * p.hv;
  int n = rank;
  if (p.num_seqs <= kTcLptSeqs) {
    __shared__ int s_pick;
    if (tid < p.num_seqs) {
      int bi, ei;
      seq_range(p.cu_seqlens, tid, p.total_tokens, bi, ei);
      int r = 0;
      for (int m = 0; m < p.num_seqs; ++m) {
        int bm, em;
        seq_range(p.cu_seqlens, m, p.total_tokens, bm, em);
        r += (em - bm > ei - bi) || (em - bm == ei - bi && m < tid);
      }
      if (r == rank) s_pick = tid;
    }
    __syncthreads();
    n = s_pick;
  }
  const int kh = h / (p.hv / p.hk);
  const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(p.q);
  const __nv_bfloat16 *k = static_cast<const __nv_bfloat16 *>(p.k);
  const __nv_bfloat16 *v = static_cast<const __nv_bfloat16 *>(p.v);
  TO *o = static_cast<TO *>(p.o);

  int bos, eos;
  seq_range(p.cu_seqlens, n, p.total_tokens, bos, eos);
  const int nchunks = (eos - bos + C - 1) / C;
  const size_t sbase = ((size_t)n * p.hv + h) * kD * kD;

  if (nchunks == 0) {  // empty sequence: the state passes through
    for (int e = tid; e < kD * kD; e += kTcThreads)
      p.state_out[sbase + e] = p.state_in ? p.state_in[sbase + e] : 0.f;
    return;
  }

  if (warp == 0) tc::alloc<512>(&sm.tmem);
  if (tid == 32) {
    mbar_init(&sm.gram_done, 1);
    mbar_init(&sm.gram_free, 1);
    mbar_init(&sm.prep_done, 1);
    mbar_init(&sm.dec_ready[0], 1);
    mbar_init(&sm.dec_ready[1], 1);
    mbar_init(&sm.p1_done, 1);
    mbar_init(&sm.p2_done, 1);
    mbar_init(&sm.p4_done, 1);
    mbar_init(&sm.d_ready, 1);
    mbar_init(&sm.s_ready, 1);
    mbar_init(&sm.r_free, 1);
    mbar_init(&sm.p4_buf[0], 1);
    mbar_init(&sm.p4_buf[1], 1);
    mbar_init(&sm.kq_full[0], kTcE);
    mbar_init(&sm.kq_full[1], kTcE);
    mbar_init(&sm.v_full, kTcE);
    mbar_fence_init();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = sm.tmem;
  bool ok = true;
  // Loads of q, k, v and the gates are issued by the E threads with cp.async; each E thread
  // then arrives (as its copies complete) on kq_full[buffer] or v_full.
  // (rows past the end of the sequence are zero-filled)
  // q, k and the gates of block cc into buffer cc & 1
  auto load_kq = [&](int cc) {
    const int b = cc & 1, t0 = bos + cc * C, Lc = min(C, eos - t0);
    for (int e = tid; e < 2 * C * 16; e += kTcE) {
      const int r = e & (2 * C - 1), gq = e >> 7, t = r & (C - 1);
      const bool in = t < Lc;
      const size_t tok = (size_t)t0 + (in ? t : 0);
      const __nv_bfloat16 *src = (r < C ? k : q) + (tok * p.hk + kh) * kD + gq * 8;
      cp_async16(sm.KQ[b] + kq_off(r, gq * 8), src, in ? 16 : 0);
    }
    for (int t = tid; t < C; t += kTcE) {
      const bool in = t < Lc;
      const size_t gi = ((size_t)t0 + (in ? t : 0)) * p.hv + h;
      cp_async4(&sm.gRaw[b][t], p.g + gi, in ? 4 : 0);
      cp_async4(&sm.bRaw[b][t], p.beta + gi, in ? 4 : 0);
    }
  };
  auto load_v = [&](int cc) {  // v rows of block cc (single buffer)
    const int t0 = bos + cc * C, Lc = min(C, eos - t0);
    for (int e = tid; e < C * 16; e += kTcE) {
      const int r = e >> 4, gq = e & 15;
      const bool in = r < Lc;
      const size_t tok = (size_t)t0 + (in ? r : 0);
      cp_async16(sm.Vb + r * kP128 + gq * 16, v + (tok * p.hv + h) * kD + gq * 8, in ? 16 : 0);
    }
  };

  if (warp >= 4 && warp < 12) {
    // ======================= P group: the state-free part of each block
    const int pt = tid - kTcE, pw = warp - 4;
    const int gid = lane >> 2, tig = lane & 3;
#pragma unroll 1
    for (int c = 0; c < nchunks; ++c) {
      const int b = c & 1;
      if (ok) ok = mbar_wait_sleep(&sm.kq_full[b], (c >> 1) & 1);  // q, k, gates of block c
      tc::fence_proxy_async();
      bar_sync(kBarP, kTcP);

      // in-block inclusive cumsum of g (padding contributes 0), e^G, e^(G_T - G), beta
      if (pw == 0) {
        float gv[2], bv[2], run = 0.f;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          gv[e] = sm.gRaw[b][2 * lane + e];
          bv[e] = sm.bRaw[b][2 * lane + e];
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
        for (int e = 0; e < 2; ++e) {
          const int t = 2 * lane + e;
          const float G = gv[e] + excl;
          sm.dec[b][0][t] = G;
          sm.dec[b][1][t] = __expf(G);
          sm.dec[b][2][t] = __expf(gC - G);
          sm.pB[t] = bv[e];
        }
      }
      bar_sync(kBarP, kTcP);
      if (pt == 0) mbar_arrive(&sm.dec_ready[b]);
      const float *G = sm.dec[b][0], *EG = sm.dec[b][1];

      // the Gram MMA of this block is done; the chain of block c - 2 no longer reads the
      // operand buffers of this parity
      if (ok) ok = mbar_wait_sleep(&sm.gram_done, c & 1);
      if (c >= 2 && ok) ok = mbar_wait_sleep(&sm.p4_buf[b], ((c - 2) >> 1) & 1);
      tc::fence_after();

      // ---- Gram epilogue: rows 0-63 K K^T -> N, rows 64-127 Q K^T -> A; warp quarter
      //      warp & 3 owns TMEM lanes (rows) 32 (warp & 3) .., column half pw >> 2
      {
        const int hf = pw >> 2, r = 32 * (warp & 3) + lane;
        uint32_t acc[32];
        tc::ld32(tc::lane_addr(tmem, warp, kTmG + 32 * hf), acc);
        // G_j of this column half into registers first (broadcast reads), so that the
        // arithmetic below is not ordered behind the shared-memory stores
        float gj[32];
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 g4 = reinterpret_cast<const float4 *>(G + 32 * hf)[j4];
          gj[4 * j4] = g4.x;
          gj[4 * j4 + 1] = g4.y;
          gj[4 * j4 + 2] = g4.z;
          gj[4 * j4 + 3] = g4.w;
        }
        const int t = r & (C - 1);
        const float Gt = G[t];
        tc::wait_ld();
        if (r < C) {
          // K K^T row t -> N = beta_t e^(G_t - G_j) k_t.k_j (j < t)
          const float bt = sm.pB[t];
          if (32 * hf < 32 * (warp & 3) + 32) {  // else every j of this half is above every t
            float x[32];
#pragma unroll
            for (int jj = 0; jj < 32; ++jj)
              x[jj] = (32 * hf + jj < t) ? bt * decay_exp(Gt - gj[jj]) * __uint_as_float(acc[jj]) : 0.f;
            // -N in fp16 everywhere (only the blocks below the diagonal are read), fp32 N on
            // the diagonal blocks
#pragma unroll
            for (int jj = 0; jj < 32; jj += 2)
              *reinterpret_cast<uint32_t *>(sm.N16 + t * 144 + 2 * (32 * hf + jj)) = pack_f16(-x[jj], -x[jj + 1]);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj)
              if (((32 * hf + jj) >> 4) == (t >> 4)) sm.Nd[t >> 4][t & 15][jj & 15] = x[jj];
          }
        } else {
          // Q K^T row t -> A = e^(G_t - G_j) q_t.k_j (j <= t), zero above the diagonal
#pragma unroll
          for (int j8 = 0; j8 < 32; j8 += 8) {
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int jj = j8 + 2 * e, j = 32 * hf + jj;
              const float a0 = (j <= t) ? decay_exp(Gt - gj[jj]) * __uint_as_float(acc[jj]) : 0.f;
              const float a1 = (j + 1 <= t) ? decay_exp(Gt - gj[jj + 1]) * __uint_as_float(acc[jj + 1]) : 0.f;
              w4[e] = pack_f16(a0, a1);
            }
            *reinterpret_cast<uint4 *>(sm.At[b] + at_off(t, 32 * hf + j8)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        }
      }
      tc::fence_before();
      bar_sync(kBarP, kTcP);
      if (pt == 0) mbar_arrive(&sm.gram_free);  // the Gram accumulator may be reused

      if (pt < C) {
        // ---- T_ii = (I + N_ii)^-1 for the four 16x16 diagonal blocks, one column per thread
        const int blk = pt >> 4, cc = pt & 15;
        float x[16];
        unit_tril_inverse_col(&sm.Nd[blk][0][0], 17, cc, x);
#pragma unroll
        for (int r = 0; r < 16; ++r)
          *reinterpret_cast<__half *>(sm.T16[blk] + r * 48 + 2 * cc) = __float2half_rn(x[r]);
      } else {
        // ---- meanwhile: fp16 operands K and diag(e^G) Q from the bf16 tile (lanes along
        //      rows, so the 16-byte accesses of a warp are contiguous)
        for (int e = pt - C; e < 2 * C * 16; e += kTcP - C) {
          const int which = e >> 10, t = e & (C - 1), gq = (e >> 6) & 15;
          const uint4 raw = *reinterpret_cast<const uint4 *>(sm.KQ[b] + kq_off(which * C + t, gq * 8));
          const float sc = which ? EG[t] : 1.f;
          const uint32_t in4[4] = {raw.x, raw.y, raw.z, raw.w};
          uint32_t out4[4];
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2)
            out4[e2] = pack_f16(__uint_as_float(in4[e2] << 16) * sc, __uint_as_float(in4[e2] & 0xffff0000u) * sc);
          *reinterpret_cast<uint4 *>((which ? sm.Qt[b] : sm.K16[b]) + t64_off(t, gq * 8)) =
              make_uint4(out4[0], out4[1], out4[2], out4[3]);
        }
        tc::fence_proxy_async();
      }
      if (ok) ok = mbar_wait_sleep(&sm.v_full, c & 1);  // v of block c
      bar_sync(kBarP, kTcP);
      // W^T and U^T are single buffers: the previous block's P1 and D epilogue are done
      if (c >= 1) {
        if (ok) ok = mbar_wait_sleep(&sm.p1_done, (c - 1) & 1);
        if (ok) ok = mbar_wait_sleep(&sm.d_ready, (c - 1) & 1);
      }

      // ---- [W U] = (I + N)^-1 [diag(beta e^G) K  diag(beta) V] by blocked forward
      //      substitution X_i^T = (R_i^T - sum_{j<i} X_j^T N_ij^T) T_ii^T; warps pw 0-3:
      //      W (32 keys each, into W^T), pw 4-7: U (32 value columns each, into U^T)
      {
        const int kind = pw >> 2, c0 = 32 * (pw & 3);
        uint32_t Xf[4][2][4];  // fp16 A fragments of the solved blocks X_j^T
#pragma unroll
        for (int i = 0; i < 4; ++i) {
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
                sc[nt][e] = kind ? sm.pB[t] : sm.pB[t] * EG[t];
              }
            const int tr = 16 * i + (lane & 7) + 8 * (lane >> 4);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
              const int cr = c0 + 16 * mt + 8 * ((lane >> 3) & 1);
              uint32_t r4[4];  // (nt 0, cols lo), (nt 0, cols hi), (nt 1, lo), (nt 1, hi)
              ldsm_x4_t(r4, kind ? sm.Vb + tr * kP128 + 2 * cr : sm.KQ[b] + kq_off(tr, cr));
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
            uint32_t bb[4];
            ldb_nk_p<144>(bb, sm.N16, 16 * i, 16 * j, lane);  // B[k=j][n=t] = -N[t][j]
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
              mma_f16(acc[mt][0], Xf[j][mt], bb[0], bb[1]);
              mma_f16(acc[mt][1], Xf[j][mt], bb[2], bb[3]);
            }
          }
          uint32_t y[2][4], bt[4];
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) acc_to_f16x(acc[mt][0], acc[mt][1], y[mt]);
          ldb_nk_p<48>(bt, sm.T16[i], 0, 0, lane);  // B[k=j'][n=t'] = T_ii[t'][j']
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            float out[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
              for (int e = 0; e < 4; ++e) out[nt][e] = 0.f;
              mma_f16(out[nt], y[mt], bt[2 * nt], bt[2 * nt + 1]);
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int hr = 0; hr < 2; ++hr) {
                const int col = c0 + 16 * mt + gid + 8 * hr, t = 16 * i + 8 * nt + 2 * tig;
                const uint32_t val = pack_f16(out[nt][2 * hr], out[nt][2 * hr + 1]);
                if (kind)
                  *reinterpret_cast<uint32_t *>(sm.Ut + col * 144 + 2 * t) = val;
                else
                  *reinterpret_cast<uint32_t *>(sm.Wt + wt_off(t, col)) = val;
              }
            if (i + 1 < 4) acc_to_f16x(out[0], out[1], Xf[i][mt]);
          }
        }
      }
      tc::fence_proxy_async();
      bar_sync(kBarP, kTcP);
      if (pt == 0) mbar_arrive(&sm.prep_done);
    }
  } else if (warp < 4) {
    // ======================= E group: thread j owns value column j (TMEM lane j)
    const int j = tid;
    auto wait = [&](uint64_t *bar, uint32_t par) { if (ok) ok = mbar_wait_sleep(bar, par); };
    auto cp_arrive = [&](uint64_t *bar) {
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(smem_u32(bar)) : "memory");
    };
    load_kq(0);
    cp_arrive(&sm.kq_full[0]);
    load_v(0);
    cp_arrive(&sm.v_full);
    if (nchunks > 1) load_kq(1);
    cp_arrive(&sm.kq_full[1]);
    // initial state: S^T row j = S[:, j]; fp16 copy for P1/P3, fp32 scaled by e^(G_T) of
    // block 0 (P2 accumulates on top of it)
    wait(&sm.dec_ready[0], 0);
    {
      const float eg = sm.dec[0][1][C - 1];
#pragma unroll 1
      for (int s4 = 0; s4 < 4; ++s4) {
        float x[32];
        uint32_t r32[32], h16[16];
#pragma unroll
        for (int i = 0; i < 32; ++i)
          x[i] = p.state_in ? p.state_in[sbase + (size_t)(32 * s4 + i) * kD + j] : 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) h16[i] = pack_f16(x[2 * i], x[2 * i + 1]);
#pragma unroll
        for (int i = 0; i < 32; ++i) r32[i] = __float_as_uint(x[i] * eg);
        tc::st16(tc::lane_addr(tmem, warp, kTmST + 16 * s4), h16);
        tc::st32(tc::lane_addr(tmem, warp, kTmS + 32 * s4), r32);
      }
      tc::wait_st();
    }
    tc::fence_before();
    bar_sync(kBarE, kTcE);
    if (tid == 0) mbar_arrive(&sm.s_ready);

#pragma unroll 1
    for (int c = 0; c < nchunks; ++c) {
      const int b = c & 1, tok0 = bos + c * C, L = min(C, eos - tok0);
      // ---- D = U + (-S W): fp16 D^T and (D diag(e^(G_T - G)))^T into tensor memory
      wait(&sm.p1_done, c & 1);
      wait(&sm.prep_done, c & 1);  // U^T and the decays of this block are written
      tc::fence_after();
      {
        const float *ED = sm.dec[b][2];
        const uint4 *urow = reinterpret_cast<const uint4 *>(sm.Ut + j * 144);
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {  // tokens 32 hh .. 32 hh + 31
          uint32_t a[32], dt[16], dd[16];
          tc::ld32(tc::lane_addr(tmem, warp, kTmD + 32 * hh), a);
          tc::wait_ld();
#pragma unroll
          for (int g8 = 0; g8 < 4; ++g8) {
            const uint4 u4 = urow[4 * hh + g8];
            const uint32_t uw[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int tl = 8 * g8 + 2 * e, t = 32 * hh + tl;
              const float2 u = f16x2_to_float2(uw[e]);
              const float d0 = u.x + __uint_as_float(a[tl]), d1 = u.y + __uint_as_float(a[tl + 1]);
              dt[tl >> 1] = pack_f16(d0, d1);
              dd[tl >> 1] = pack_f16(d0 * ED[t], d1 * ED[t + 1]);
            }
          }
          tc::st16(tc::lane_addr(tmem, warp, kTmDT + 16 * hh), dt);
          tc::st16(tc::lane_addr(tmem, warp, kTmDD + 16 * hh), dd);
        }
        tc::wait_st();
      }
      tc::fence_before();
      bar_sync(kBarE, kTcE);
      if (tid == 0) mbar_arrive(&sm.d_ready);
      // block c's inputs are consumed (prep of block c is done): v of block c + 1, then
      // q, k, gates of block c + 2 into the freed buffers
      if (c + 1 < nchunks) {
        load_v(c + 1);
        cp_arrive(&sm.v_full);
      }
      if (c + 2 < nchunks) {
        load_kq(c + 2);
        cp_arrive(&sm.kq_full[b]);
      }

      // ---- state: S after P2 -> fp16 copy for the next block, then pre-scaled by the
      //      next block's e^(G_T); after the last block, S goes to state_out
      wait(&sm.p2_done, c & 1);
      tc::fence_after();
      const bool last = c + 1 == nchunks;
      float egn = 1.f;
      if (!last) {
        wait(&sm.dec_ready[(c + 1) & 1], ((c + 1) >> 1) & 1);
        egn = sm.dec[(c + 1) & 1][1][C - 1];
      }
#pragma unroll 1
      for (int s4 = 0; s4 < 4; ++s4) {
        uint32_t r32[32];
        tc::ld32(tc::lane_addr(tmem, warp, kTmS + 32 * s4), r32);
        tc::wait_ld();
        if (last) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            p.state_out[sbase + (size_t)(32 * s4 + i) * kD + j] = __uint_as_float(r32[i]);
        } else {
          uint32_t h16[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            h16[i] = pack_f16(__uint_as_float(r32[2 * i]), __uint_as_float(r32[2 * i + 1]));
#pragma unroll
          for (int i = 0; i < 32; ++i) r32[i] = __float_as_uint(__uint_as_float(r32[i]) * egn);
          tc::st16(tc::lane_addr(tmem, warp, kTmST + 16 * s4), h16);
          tc::st32(tc::lane_addr(tmem, warp, kTmS + 32 * s4), r32);
        }
      }
      if (!last) {
        tc::wait_st();
        tc::fence_before();
        bar_sync(kBarE, kTcE);
        if (tid == 0) mbar_arrive(&sm.s_ready);
      }

      // ---- outputs O^T row j -> o[t][h][j] for the block's valid tokens
      wait(&sm.p4_done, c & 1);
      tc::fence_after();
      {
        uint32_t r0[32], r1[32];
        tc::ld32(tc::lane_addr(tmem, warp, kTmR), r0);
        tc::ld32(tc::lane_addr(tmem, warp, kTmR + 32), r1);
        tc::wait_ld();
        TO *orow = o + ((size_t)tok0 * p.hv + h) * kD + j;
        const size_t tstride = (size_t)p.hv * kD;
#pragma unroll
        for (int t = 0; t < C; ++t)
          if (t < L) Elem<TO>::store(orow + t * tstride, __uint_as_float(t < 32 ? r0[t & 31] : r1[t & 31]));
      }
      tc::fence_before();
      bar_sync(kBarE, kTcE);
      if (tid == 0) mbar_arrive(&sm.r_free);
    }
    cp_async_wait<0>();
  } else if (warp == 12 && lane == 0) {
    // ======================= MMA issuer
    auto wait = [&](uint64_t *bar, uint32_t par) { if (ok) ok = mbar_wait_sleep(bar, par); };
    constexpr uint32_t idG = tc::idesc(128, 64, 1, 0, 0);   // [K; Q] K^T, bf16
    constexpr uint32_t idP1 = tc::idesc(128, 64, 0, 1, 1);  // -S^T W^T, W^T MN-major
    constexpr uint32_t idP3 = tc::idesc(128, 64, 0, 0, 0);  // S^T (diag(e^G) Q)^T
    constexpr uint32_t idP2 = tc::idesc(128, 128, 0, 0, 1); // Dd^T K, K MN-major over keys
    constexpr uint32_t idP4 = tc::idesc(128, 64, 0, 0, 0);  // D^T A^T
    const uint32_t sWt = smem_u32(sm.Wt);
    auto gram = [&](int cc) {
      const uint32_t base = smem_u32(sm.KQ[cc & 1]);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {  // 16 keys per step: two core matrices along K
        const uint64_t d = tc::sdesc(base + kk * 4096, 2048, 128);
        tc::mma_ss(tmem + kTmG, d, d, idG, kk > 0);
      }
      tc::commit(&sm.gram_done);
    };
    // The Gram MMA of a block needs only its q and k tiles and a free Gram accumulator,
    // so it is issued as soon as both hold: one block ahead of the chain, while the prep
    // warps are still busy with the current block.
    wait(&sm.kq_full[0], 0);
    tc::fence_proxy_async();  // the cp.async writes, as seen by the tensor cores
    tc::fence_after();
    gram(0);
#pragma unroll 1
    for (int c = 0; c < nchunks; ++c) {
      const uint32_t sQt = smem_u32(sm.Qt[c & 1]), sK = smem_u32(sm.K16[c & 1]);
      const uint32_t sAt = smem_u32(sm.At[c & 1]);
      if (c + 1 < nchunks) {
        wait(&sm.kq_full[(c + 1) & 1], ((c + 1) >> 1) & 1);
        wait(&sm.gram_free, c & 1);
        tc::fence_proxy_async();
        tc::fence_after();
        gram(c + 1);
      }
      wait(&sm.prep_done, c & 1);
      wait(&sm.s_ready, c & 1);
      tc::fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        tc::mma_ts(tmem + kTmD, tmem + kTmST + 8 * kk, tc::sdesc(sWt + kk * 2048, 1024, 128), idP1, kk > 0);
      tc::commit(&sm.p1_done);
      if (c >= 1) wait(&sm.r_free, (c - 1) & 1);
      tc::fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        tc::mma_ts(tmem + kTmR, tmem + kTmST + 8 * kk, tc::sdesc(sQt + kk * 2048, 1024, 128), idP3, kk > 0);
      wait(&sm.d_ready, c & 1);
      tc::fence_after();
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)  // 16 tokens per step
        tc::mma_ts(tmem + kTmS, tmem + kTmDD + 8 * kk, tc::sdesc(sK + kk * 256, 128, 1024), idP2, 1);
      tc::commit(&sm.p2_done);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        tc::mma_ts(tmem + kTmR, tmem + kTmDT + 8 * kk, tc::sdesc(sAt + kk * 2048, 1024, 128), idP4, 1);
      tc::commit(&sm.p4_done);
      tc::commit(&sm.p4_buf[c & 1]);
    }
  }

  if (!ok) report_status(p.err, GDN_STATUS_WAIT_TIMEOUT);
  tc::fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after();
    tc::dealloc<512>(tmem);
  }
}

// ============================================================ the chain over pass-1 slots
// tc_chain_kernel: pass 2 of the two-pass path.  The state-free operands of every block
// come from its workspace slot (written by pass 1 in the kTs* layout), so the CTA runs
// only the state chain and the outputs, with the products of tc_kernel:
//   P1: D^T  = -S^T W^T,  P3: R^T = S^T (diag(e^G) Q)^T,  P2: S^T += Dd^T K,  P4: O^T = R^T + D^T A^T
// Warp roles:
//   warps 0-3 (E, thread j = value column j = TMEM lane j): D = U + P1 into the fp16
//     operands of P2 and P4; the state epilogue after P2: first the fp16 copy of S (the
//     A operand of the next block's P1 and P3), then S pre-scaled by the next block's
//     e^(G_C) (P2 accumulates on top of it).  Only these two steps sit on the chain.
//   warps 4-7 (O, same lanes): the block's outputs O^T after P4 -> o.
//   warp 8 lane 0: the producer, each block's slot into a ring stage with one bulk copy.
//   warp 9 lane 0: issues every MMA and its commits.
constexpr int kChNst = 2;                // ring depth
constexpr int kChThreads = 32 * 10;
constexpr int kBarO = 3;                 // named barrier of the O group

struct alignas(128) ChainSlot {          // one block's operands, as in the slot (kTs*)
  char Wt[16384], Qt[16384], K16[16384], At[8192], Ut[kD * 144];
  float dec[3][kTcC];                    // G, e^G, e^(G_C - G)
};
static_assert(sizeof(ChainSlot) == kTsBytes && offsetof(ChainSlot, Qt) == kTsQt &&
                  offsetof(ChainSlot, K16) == kTsK && offsetof(ChainSlot, At) == kTsAt &&
                  offsetof(ChainSlot, Ut) == kTsUt && offsetof(ChainSlot, dec) == kTsDec,
              "slot layout");
struct ChainSmem {
  ChainSlot st[kChNst];
  alignas(8) uint64_t full[kChNst], empty[kChNst];
  alignas(8) uint64_t p1_done, p2_done, p4_done, d_ready, s_ready, r_free;
  uint32_t tmem;
};

template <typename TO>
__global__ void __launch_bounds__(kChThreads, 1) tc_chain_kernel(ChunkParams p) {
  constexpr int C = kTcC;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  ChainSmem &sm = *reinterpret_cast<ChainSmem *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = blockIdx.x / p.hv, h = blockIdx.x - n * p.hv;
  int bos, eos;
  seq_range(p.cu_seqlens, n, p.total_tokens, bos, eos);
  const int nchunks = (eos - bos + C - 1) / C;
  const size_t sbase = ((size_t)n * p.hv + h) * kD * kD;
  const char *slot0 = p.slot_ws + ((size_t)h * p.nslots + (size_t)(bos / C + n)) * kTsBytes;

  if (nchunks == 0) {  // empty sequence: the state passes through
    for (int e = tid; e < kD * kD; e += kChThreads)
      p.state_out[sbase + e] = p.state_in ? p.state_in[sbase + e] : 0.f;
    return;
  }
  if (warp == 0) tc::alloc<512>(&sm.tmem);
  if (tid == 32) {
    for (int s = 0; s < kChNst; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 2);  // the last MMA reading the stage, the E group
    }
    mbar_init(&sm.p1_done, 1);
    mbar_init(&sm.p2_done, 1);
    mbar_init(&sm.p4_done, 1);
    mbar_init(&sm.d_ready, 1);
    mbar_init(&sm.s_ready, 1);
    mbar_init(&sm.r_free, 1);
    mbar_fence_init();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = sm.tmem;
  bool ok = true;
  auto wait = [&](uint64_t *bar, uint32_t par) { if (ok) ok = mbar_wait(bar, par); };

  if (warp == 8) {
    // ======================= producer: block c's slot into stage c % kChNst
    if (lane == 0) {
#pragma unroll 1
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % kChNst;
        if (c >= kChNst) wait(&sm.empty[s], ((c / kChNst) - 1) & 1);
        mbar_arrive_expect_tx(&sm.full[s], (uint32_t)kTsBytes);
        bulk_g2s(&sm.st[s], slot0 + (size_t)c * kTsBytes, (uint32_t)kTsBytes, &sm.full[s]);
      }
    }
  } else if (warp < 4) {
    // ======================= E group: thread j owns value column j (TMEM lane j)
    const int j = tid;
    // initial state: S^T row j = S[:, j]; fp16 copy for P1/P3, fp32 scaled by e^(G_C) of
    // block 0 (P2 accumulates on top of it)
    wait(&sm.full[0], 0);
    {
      const float eg = sm.st[0].dec[1][C - 1];
#pragma unroll 1
      for (int s4 = 0; s4 < 4; ++s4) {
        float x[32];
        uint32_t r32[32], h16[16];
#pragma unroll
        for (int i = 0; i < 32; ++i)
          x[i] = p.state_in ? p.state_in[sbase + (size_t)(32 * s4 + i) * kD + j] : 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) h16[i] = pack_f16(x[2 * i], x[2 * i + 1]);
#pragma unroll
        for (int i = 0; i < 32; ++i) r32[i] = __float_as_uint(x[i] * eg);
        tc::st16(tc::lane_addr(tmem, warp, kTmST + 16 * s4), h16);
        tc::st32(tc::lane_addr(tmem, warp, kTmS + 32 * s4), r32);
      }
      tc::wait_st();
    }
    tc::fence_before();
    bar_sync(kBarE, kTcE);
    if (tid == 0) mbar_arrive(&sm.s_ready);

#pragma unroll 1
    for (int c = 0; c < nchunks; ++c) {
      const int s = c % kChNst;
      const ChainSlot &st = sm.st[s];
      // ---- D = U + (-S W): fp16 D^T and (D diag(e^(G_C - G)))^T into tensor memory
      wait(&sm.full[s], (c / kChNst) & 1);
      wait(&sm.p1_done, c & 1);
      tc::fence_after();
      {
        const float *ED = st.dec[2];
        const uint4 *urow = reinterpret_cast<const uint4 *>(st.Ut + j * 144);
        uint32_t a[64];
        tc::ld32(tc::lane_addr(tmem, warp, kTmD), *reinterpret_cast<uint32_t(*)[32]>(a));
        tc::ld32(tc::lane_addr(tmem, warp, kTmD + 32), *reinterpret_cast<uint32_t(*)[32]>(a + 32));
        tc::wait_ld();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {  // tokens 32 hh .. 32 hh + 31
          uint32_t dt[16], dd[16];
#pragma unroll
          for (int g8 = 0; g8 < 4; ++g8) {
            const uint4 u4 = urow[4 * hh + g8];
            const uint32_t uw[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int tl = 8 * g8 + 2 * e, t = 32 * hh + tl;
              const float2 u = f16x2_to_float2(uw[e]);
              const float d0 = u.x + __uint_as_float(a[t]), d1 = u.y + __uint_as_float(a[t + 1]);
              dt[tl >> 1] = pack_f16(d0, d1);
              dd[tl >> 1] = pack_f16(d0 * ED[t], d1 * ED[t + 1]);
            }
          }
          tc::st16(tc::lane_addr(tmem, warp, kTmDT + 16 * hh), dt);
          tc::st16(tc::lane_addr(tmem, warp, kTmDD + 16 * hh), dd);
        }
        tc::wait_st();
      }
      tc::fence_before();
      bar_sync(kBarE, kTcE);
      if (tid == 0) {
        mbar_arrive(&sm.d_ready);
        if (c + kChNst < nchunks) mbar_arrive(&sm.empty[s]);  // U^T and the decays of stage s are read
      }

      // ---- state: S after P2 -> fp16 copy for the next block (released first), then
      //      pre-scaled by the next block's e^(G_C); after the last block, S -> state_out
      wait(&sm.p2_done, c & 1);
      tc::fence_after();
      if (c + 1 == nchunks) {
#pragma unroll 1
        for (int s4 = 0; s4 < 4; ++s4) {
          uint32_t r32[32];
          tc::ld32(tc::lane_addr(tmem, warp, kTmS + 32 * s4), r32);
          tc::wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) p.state_out[sbase + (size_t)(32 * s4 + i) * kD + j] = __uint_as_float(r32[i]);
        }
      } else {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {  // keys 64 hf .. 64 hf + 63
          uint32_t r[64], h16[32];
          tc::ld32(tc::lane_addr(tmem, warp, kTmS + 64 * hf), *reinterpret_cast<uint32_t(*)[32]>(r));
          tc::ld32(tc::lane_addr(tmem, warp, kTmS + 64 * hf + 32), *reinterpret_cast<uint32_t(*)[32]>(r + 32));
          tc::wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) h16[i] = pack_f16(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
          tc::st32(tc::lane_addr(tmem, warp, kTmST + 32 * hf), h16);
        }
        tc::wait_st();
        tc::fence_before();
        bar_sync(kBarE, kTcE);
        if (tid == 0) mbar_arrive(&sm.s_ready);  // P1 and P3 of block c + 1 may start
        const int s1 = (c + 1) % kChNst;
        wait(&sm.full[s1], ((c + 1) / kChNst) & 1);
        const float egn = sm.st[s1].dec[1][C - 1];
#pragma unroll 1
        for (int s4 = 0; s4 < 4; ++s4) {
          uint32_t r32[32];
          tc::ld32(tc::lane_addr(tmem, warp, kTmS + 32 * s4), r32);
          tc::wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) r32[i] = __float_as_uint(__uint_as_float(r32[i]) * egn);
          tc::st32(tc::lane_addr(tmem, warp, kTmS + 32 * s4), r32);
        }
        tc::wait_st();  // (ordered before P2 of block c + 1 by the d_ready hand-off)
      }
    }
  } else if (warp < 8) {
    // ======================= O group: the block's outputs, O^T row j -> o[t][h][j]
    const int j = tid - 128;
    TO *o = static_cast<TO *>(p.o);
#pragma unroll 1
    for (int c = 0; c < nchunks; ++c) {
      const int tok0 = bos + c * C, L = min(C, eos - tok0);
      wait(&sm.p4_done, c & 1);
      tc::fence_after();
      uint32_t r0[32], r1[32];
      tc::ld32(tc::lane_addr(tmem, warp, kTmR), r0);
      tc::ld32(tc::lane_addr(tmem, warp, kTmR + 32), r1);
      tc::wait_ld();
      tc::fence_before();
      bar_sync(kBarO, kTcE);
      if (j == 0) mbar_arrive(&sm.r_free);  // the accumulator is read: P3 of block c + 1 may start
      TO *dst = o + ((size_t)tok0 * p.hv + h) * kD + j;
      const size_t tstride = (size_t)p.hv * kD;
#pragma unroll
      for (int t = 0; t < C; ++t) {
        if (t < L) Elem<TO>::store(dst, __uint_as_float(t < 32 ? r0[t & 31] : r1[t & 31]));
        dst += tstride;
      }
    }
  } else if (warp == 9 && lane == 0) {
    // ======================= MMA issuer
    constexpr uint32_t idP1 = tc::idesc(128, 64, 0, 1, 1);  // -S^T W^T, W^T MN-major
    constexpr uint32_t idP3 = tc::idesc(128, 64, 0, 0, 0);  // S^T (diag(e^G) Q)^T
    constexpr uint32_t idP2 = tc::idesc(128, 128, 0, 0, 1); // Dd^T K, K MN-major over keys
    constexpr uint32_t idP4 = tc::idesc(128, 64, 0, 0, 0);  // D^T A^T
#pragma unroll 1
    for (int c = 0; c < nchunks; ++c) {
      const int s = c % kChNst;
      const uint32_t sWt = smem_u32(sm.st[s].Wt), sQt = smem_u32(sm.st[s].Qt);
      const uint32_t sK = smem_u32(sm.st[s].K16), sAt = smem_u32(sm.st[s].At);
      wait(&sm.full[s], (c / kChNst) & 1);
      wait(&sm.s_ready, c & 1);
      tc::fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        tc::mma_ts(tmem + kTmD, tmem + kTmST + 8 * kk, tc::sdesc(sWt + kk * 2048, 1024, 128), idP1, kk > 0);
      tc::commit(&sm.p1_done);
      if (c >= 1) wait(&sm.r_free, (c - 1) & 1);
      tc::fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        tc::mma_ts(tmem + kTmR, tmem + kTmST + 8 * kk, tc::sdesc(sQt + kk * 2048, 1024, 128), idP3, kk > 0);
      wait(&sm.d_ready, c & 1);
      tc::fence_after();
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)  // 16 tokens per step
        tc::mma_ts(tmem + kTmS, tmem + kTmDD + 8 * kk, tc::sdesc(sK + kk * 256, 128, 1024), idP2, 1);
      tc::commit(&sm.p2_done);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        tc::mma_ts(tmem + kTmR, tmem + kTmDT + 8 * kk, tc::sdesc(sAt + kk * 2048, 1024, 128), idP4, 1);
      tc::commit(&sm.p4_done);
      // every MMA reading stage s is done (only where the producer refills it: no arrive
      // may land after the CTA has finished)
      if (c + kChNst < nchunks) tc::commit(&sm.empty[s]);
    }
  }

  if (!ok) report_status(p.err, GDN_STATUS_WAIT_TIMEOUT);
  tc::fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after();
    tc::dealloc<512>(tmem);
  }
}

template <typename TO>
cudaError_t launch_tc_chain_t(const ChunkParams &p, cudaStream_t stream) {
  const size_t smem = sizeof(ChainSmem);
  cudaError_t err =
      cudaFuncSetAttribute(tc_chain_kernel<TO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  tc_chain_kernel<TO><<<(unsigned)((long long)p.num_seqs * p.hv), kChThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <typename TO>
cudaError_t launch_tc_t(const ChunkParams &p, cudaStream_t stream) {
  const size_t smem = sizeof(TcSmem);
  cudaError_t err =
      cudaFuncSetAttribute(tc_kernel<TO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  tc_kernel<TO><<<(unsigned)((long long)p.num_seqs * p.hv), kTcThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_chain(const ChunkParams &p, cudaStream_t stream) {
  if ((long long)p.num_seqs * p.hv == 0) return cudaSuccess;
  return p.o_fp32 ? launch_tc_chain_t<float>(p, stream) : launch_tc_chain_t<__nv_bfloat16>(p, stream);
}

cudaError_t launch_chunk_tc(const ChunkParams &p, cudaStream_t stream) {
  if ((long long)p.num_seqs * p.hv == 0) return cudaSuccess;
  if (p.chunk != kTcC) return cudaErrorInvalidValue;
  return p.o_fp32 ? launch_tc_t<float>(p, stream) : launch_tc_t<__nv_bfloat16>(p, stream);
}

}  // namespace gdn
