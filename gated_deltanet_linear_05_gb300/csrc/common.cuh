// Device helpers shared by the libgdn kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

constexpr int kD = 128;  // dk = dv = 128, the head size built

// ------------------------------------------------------------------ dtype traits

template <typename T>
struct Elem;
template <>
struct Elem<float> {
  static __device__ __forceinline__ float load(const float *p) { return *p; }
  static __device__ __forceinline__ void store(float *p, float x) { *p = x; }
};
template <>
struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float load(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
  }
  static __device__ __forceinline__ void store(__nv_bfloat16 *p, float x) {
    *p = __float2bfloat16_rn(x);
  }
};

// ------------------------------------------------------------------ sequences

// Token range [bos, eos) of sequence n, clamped to [0, total] so that a malformed
// cu_seqlens can never move an access outside the buffers.
__device__ __forceinline__ void seq_range(const int32_t *cu, int n, int total, int &bos,
                                          int &eos) {
  int a = cu[n], b = cu[n + 1];
  a = min(max(a, 0), total);
  b = min(max(b, a), total);
  bos = a;
  eos = b;
}

// ------------------------------------------------------------------ cp.async

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global->shared copy; src_bytes == 0 fills the destination with zeros.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem)),
               "l"(gmem), "r"(src_bytes));
}
// 4-byte global->shared copy; src_bytes == 0 writes a zero.
__device__ __forceinline__ void cp_async4(void *smem, const void *gmem, int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(smem_u32(smem)),
               "l"(gmem), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// ------------------------------------------------------------------ mbarrier / bulk copy

__device__ __forceinline__ void mbar_init(uint64_t *bar, int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
// Wait for the phase with the given parity to complete.  Bounded: gives up after about
// 2^22 polls (far beyond any legitimate wait) and returns false, so that a lost
// signal ends in wrong results and an error flag instead of a hung GPU.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  uint32_t done = 0;
  for (int it = 0; it < (1 << 22) && !done; ++it) {
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
  }
  return done != 0;
}
// mbar_wait with a caller-given number of polls.
__device__ __forceinline__ bool mbar_wait_polls(uint64_t *bar, uint32_t parity, int polls) {
  uint32_t done = 0;
  for (int it = 0; it < polls && !done; ++it) {
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
  }
  return done != 0;
}
// Set status bits in the library's device status word (see gdn_device_status).
__device__ __forceinline__ void report_status(unsigned int *word, unsigned int bits) {
  if (word) atomicOr(word, bits);
}
// Like mbar_wait, but each try suspends the thread until the phase completes or about
// 50 us pass, so that waiting warps do not take issue slots from working ones.  Gives up
// after 2^15 tries (over a second) and returns false.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t *bar, uint32_t parity) {
  uint32_t done = 0;
  for (int it = 0; it < (1 << 15) && !done; ++it) {
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity), "r"(50000u)
        : "memory");
  }
  return done != 0;
}
// Orders this thread's (and, after a barrier, the CTA's) generic-proxy accesses to shared
// memory before later async-proxy ones (a bulk or tensor copy into the same bytes).
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
// 3-D tensor-map (TMA) load of the map's box at coordinates (x, y, z) into shared memory
// (1024-byte aligned for a 128-byte swizzle), completion counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_3d(void *dst, const void *map, int x, int y, int z,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3, %4}], [%5];\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}
// Bulk (TMA) copy global -> shared of `bytes` (multiple of 16, both ends 16-byte
// aligned); completion is counted in bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ------------------------------------------------------------------ tensor cores
// mma.sync m16n8k16, bf16 inputs, fp32 accumulate.  Fragment ownership (lane l,
// gid = l >> 2, tig = l & 3):
//   A 16x16 (row-major): a0:(gid, 2tig..+1) a1:(gid+8, 2tig..) a2:(gid, 2tig+8..) a3:(gid+8, 2tig+8..)
//   B 16x8  (k x n):     b0:(k=2tig..+1, n=gid) b1:(k=2tig+8..+9, n=gid)
//   C 16x8:              c0,c1:(gid, 2tig..+1) c2,c3:(gid+8, 2tig..+1)

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *smem) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(smem)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void *smem) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(smem)));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// Swizzled tile of bf16 rows: row r holds ROWB bytes (a multiple of 16) split in
// 16-byte granules.  Granule g of row r is stored at granule g ^ ((r / RPL) & MASK),
// RPL = rows per 128-byte line, so that an ldmatrix read of eight consecutive rows at
// one column touches eight different 16-byte bank groups.
template <int ROWB>
__device__ __forceinline__ int swz(int r, int byte_col) {
  constexpr int GP = ROWB / 16;
  constexpr int RPL = ROWB >= 128 ? 1 : 128 / ROWB;
  constexpr int MASK = (GP >= 8 ? 8 : GP) - 1;
  const int g = byte_col >> 4;
  return r * ROWB + (((g ^ ((r / RPL) & MASK)) << 4) | (byte_col & 15));
}

// A-operand (16x16 at rows r0.., bf16 cols c0..) from a swizzled row-major tile.
template <int ROWB>
__device__ __forceinline__ void lda_tile(uint32_t (&a)[4], const char *base, int r0, int c0,
                                         int lane) {
  const int r = r0 + (lane & 7) + ((lane >> 3) & 1) * 8;
  const int c = c0 + (lane >> 4) * 8;
  ldsm_x4(a, base + swz<ROWB>(r, c * 2));
}
// A-operand (16x16: rows m0.., k cols k0..) from a swizzled tile stored [k][m].
template <int ROWB>
__device__ __forceinline__ void lda_tile_t(uint32_t (&a)[4], const char *base, int m0, int k0,
                                           int lane) {
  const int r = k0 + (lane & 7) + (lane >> 4) * 8;
  const int c = m0 + ((lane >> 3) & 1) * 8;
  ldsm_x4_t(a, base + swz<ROWB>(r, c * 2));
}
// Two B-operands (n-tiles n0 and n0+8, k 16 wide at k0) from a tile stored [n][k].
// b[0], b[1]: n-tile n0 (k lo, k hi); b[2], b[3]: n-tile n0 + 8.
template <int ROWB>
__device__ __forceinline__ void ldb_nk(uint32_t (&b)[4], const char *base, int n0, int k0,
                                       int lane) {
  const int r = n0 + (lane & 7) + (lane >> 4) * 8;
  const int c = k0 + ((lane >> 3) & 1) * 8;
  ldsm_x4(b, base + swz<ROWB>(r, c * 2));
}
// Two B-operands (n-tiles n0 and n0+8, k 16 wide at k0) from a tile stored [k][n].
template <int ROWB>
__device__ __forceinline__ void ldb_kn(uint32_t (&b)[4], const char *base, int k0, int n0,
                                       int lane) {
  const int r = k0 + (lane & 7) + ((lane >> 3) & 1) * 8;
  const int c = n0 + (lane >> 4) * 8;
  ldsm_x4_t(b, base + swz<ROWB>(r, c * 2));
}

// x0, x1 -> bf16 pair hi = bf16(x), lo = bf16(x - hi): together ~16 significant bits.
__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  const __nv_bfloat16 h0 = __float2bfloat16_rn(x0), h1 = __float2bfloat16_rn(x1);
  hi = pack_bf16(__bfloat162float(h0), __bfloat162float(h1));
  lo = pack_bf16(x0 - __bfloat162float(h0), x1 - __bfloat162float(h1));
}

// ------------------------------------------------------------------ fp16 operands
// mma.sync m16n8k16 with fp16 inputs and fp32 accumulation (same fragment ownership as
// mma_bf16).  fp16 keeps 11 significant bits against bf16's 8.
__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// (lo, hi) -> packed fp16 pair, round to nearest even
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// packed bf16 pair -> packed fp16 pair (exact for |x| >= 2^-14 and below 65504; tiny
// values round to the fp16 subnormal grid, an absolute change below 2^-25)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t x) {
  return pack_f16(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
}

__device__ __forceinline__ float2 f16x2_to_float2(uint32_t x) {
  __half2 h = *reinterpret_cast<__half2 *>(&x);
  return __half22float2(h);
}

// Padded row-major 16-bit tiles: row r starts at r * STRIDE bytes, STRIDE = 16 mod 128
// (272 for 128-element rows, 2C + 16 for C-element rows), so the eight 16-byte rows
// of an ldmatrix read fall on eight different bank groups.
template <int STRIDE>
__device__ __forceinline__ const char *pad_at(const char *base, int r, int col) {
  return base + r * STRIDE + col * 2;
}
// A-operand 16x16 (rows m0.., k cols k0..) from a tile stored [m][k]
template <int STRIDE>
__device__ __forceinline__ void lda_p(uint32_t (&a)[4], const char *base, int m0, int k0,
                                      int lane) {
  ldsm_x4(a, pad_at<STRIDE>(base, m0 + (lane & 7) + ((lane >> 3) & 1) * 8, k0 + (lane >> 4) * 8));
}
// A-operand 16x16 (rows m0.., k cols k0..) from a tile stored [k][m]
template <int STRIDE>
__device__ __forceinline__ void lda_t_p(uint32_t (&a)[4], const char *base, int m0, int k0,
                                        int lane) {
  ldsm_x4_t(a, pad_at<STRIDE>(base, k0 + (lane & 7) + (lane >> 4) * 8, m0 + ((lane >> 3) & 1) * 8));
}
// Two B-operands (n-tiles n0, n0+8; k 16 wide at k0) from a tile stored [n][k]:
// b[0], b[1] for n-tile n0, b[2], b[3] for n-tile n0 + 8
template <int STRIDE>
__device__ __forceinline__ void ldb_nk_p(uint32_t (&b)[4], const char *base, int n0, int k0,
                                         int lane) {
  ldsm_x4(b, pad_at<STRIDE>(base, n0 + (lane & 7) + (lane >> 4) * 8, k0 + ((lane >> 3) & 1) * 8));
}
// Two B-operands (n-tiles n0, n0+8; k 16 wide at k0) from a tile stored [k][n]
template <int STRIDE>
__device__ __forceinline__ void ldb_kn_p(uint32_t (&b)[4], const char *base, int k0, int n0,
                                         int lane) {
  ldsm_x4_t(b, pad_at<STRIDE>(base, k0 + (lane & 7) + ((lane >> 3) & 1) * 8, n0 + (lane >> 4) * 8));
}

// One B-operand (n-tile n0, k 16 wide at k0) from a tile stored [n][k]: b[0] k lo, b[1] k hi
template <int STRIDE>
__device__ __forceinline__ void ldb1_nk_p(uint32_t (&b)[2], const char *base, int n0, int k0,
                                          int lane) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n"
               : "=r"(b[0]), "=r"(b[1])
               : "r"(smem_u32(pad_at<STRIDE>(base, n0 + (lane & 7), k0 + ((lane >> 3) & 1) * 8))));
}
// One B-operand (n-tile n0, k 16 wide at k0) from a tile stored [k][n]
template <int STRIDE>
__device__ __forceinline__ void ldb1_kn_p(uint32_t (&b)[2], const char *base, int k0, int n0,
                                          int lane) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];\n"
               : "=r"(b[0]), "=r"(b[1])
               : "r"(smem_u32(pad_at<STRIDE>(base, k0 + (lane & 7) + ((lane >> 3) & 1) * 8, n0))));
}

// Four 8x8 16-bit matrices from the mma fragment layout (lane (gid, tig) holds row gid,
// columns 2tig, 2tig + 1 of matrix i in r_i) to shared memory; lane l gives the address
// of row l % 8 of matrix l / 8.  The .trans form stores each matrix transposed.
__device__ __forceinline__ void stsm_x4(void *smem, uint32_t r0, uint32_t r1, uint32_t r2,
                                        uint32_t r3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};\n" ::"r"(
                   smem_u32(smem)),
               "r"(r0), "r"(r1), "r"(r2), "r"(r3)
               : "memory");
}
__device__ __forceinline__ void stsm_x4_t(void *smem, uint32_t r0, uint32_t r1, uint32_t r2,
                                          uint32_t r3) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1,%2,%3,%4};\n" ::"r"(
                   smem_u32(smem)),
               "r"(r0), "r"(r1), "r"(r2), "r"(r3)
               : "memory");
}

// Named barrier over `count` threads (a multiple of 32); id 0 is __syncthreads.
__device__ __forceinline__ void bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(count) : "memory");
}
// Arrive on named barrier `id` without waiting (producer side of a bar.sync by others).
__device__ __forceinline__ void bar_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;\n" ::"r"(id), "r"(count) : "memory");
}

// e^d by the change-of-base identity e^d = 2^(d log2 e) on the hardware base-2
// exponential (PTX ex2.approx.ftz): relative error a few 1e-7 plus |d| 6e-8, results
// below 2^-126 flushed to zero.  Used for the in-block decays and the SiLU gate, where
// it replaced a measurably slower exponential.
__device__ __forceinline__ float decay_exp(float d) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(r) : "f"(d * 1.4426950408889634f));
  return r;
}

// Column cc of (I + N)^-1 for a strictly lower triangular 16 x 16 block N (N(r, m) at
// N0[r * stride + m]): x[r] = 0 above the diagonal, 1 on it and
// -sum_{cc <= m < r} N(r, m) x[m] below, by column-oriented forward substitution: each
// x[m] is pushed into every later row's sum as soon as it is known, so the dependent
// chain is one fused multiply-add per row.
__device__ __forceinline__ void unit_tril_inverse_col(const float *N0, int stride, int cc,
                                                      float (&x)[16]) {
  float acc[16];
#pragma unroll
  for (int r = 0; r < 16; ++r) acc[r] = 0.f;
#pragma unroll
  for (int m = 0; m < 16; ++m) {
    const float xm = (m < cc) ? 0.f : (m == cc ? 1.f : -acc[m]);
    x[m] = xm;
#pragma unroll
    for (int r = m + 1; r < 16; ++r) acc[r] = fmaf(N0[r * stride + m], xm, acc[r]);
  }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

}  // namespace gdn
