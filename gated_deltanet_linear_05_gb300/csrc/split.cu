// Sequence-split prefill: the helper kernels.  Per block the chunkwise form ("Qwen3.5-9B-npu"
// model card, section "How it works") is an affine map of the state,
//     S_{c+1} = M_c S_c + B_c,   M_c = e^{G_C} I - K~^T W,   B_c = K~^T U,
// (K~ = diag(e^{G_C - G}) K), so a segment of blocks maps its incoming state S through
// M_s S + L_s, with M_s the product of its blocks' M_c and L_s its final state from a
// zero start.  A long sequence is cut into segments; the host side (gdn_api.cu) runs
//   1. every segment from a zero state                        -> L_s
//   2. every segment with v = 0 from the identity state       -> M_s (B_c = 0 when V = 0)
//   3. the combine below, in segment order per sequence: S_in(s+1) = M_s S_in(s) + L_s
//   4. every segment from its S_in(s)                         -> o and the final states
// with passes 1, 2 and 4 on the ordinary chunked schedules, every segment an independent
// sequence of their batch.
#include "common.cuh"
#include "internal.h"

namespace gdn {

namespace {

// Segment boundaries: sequence n (tokens [bos, eos)) becomes ceil((eos - bos) / seg)
// segments of seg tokens (the last one shorter); seg_first[n] is the index of its first
// segment, seg_first[N] the number used; unused entries up to max_segs are empty
// segments at the end of the token range.  One CTA: thread 0 scans the sequences, then
// every thread fills boundaries.
__global__ void __launch_bounds__(256) split_plan_kernel(SplitPlanParams p) {
  __shared__ int s_used;
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int n = 0; n < p.num_seqs; ++n) {
      int bos, eos;
      seq_range(p.cu_seqlens, n, p.total_tokens, bos, eos);
      p.seg_first[n] = acc;
      acc += (eos - bos + p.seg_len - 1) / p.seg_len;
    }
    p.seg_first[p.num_seqs] = acc;
    s_used = acc;
  }
  __syncthreads();
  const int used = s_used;
  for (int n = threadIdx.x; n < p.num_seqs; n += blockDim.x) {
    int bos, eos;
    seq_range(p.cu_seqlens, n, p.total_tokens, bos, eos);
    const int first = p.seg_first[n], cnt = p.seg_first[n + 1] - first;
    for (int j = 0; j < cnt; ++j) p.cu_seg[first + j] = bos + j * p.seg_len;
  }
  for (int i = used + threadIdx.x; i <= p.max_segs; i += blockDim.x) p.cu_seg[i] = p.total_tokens;
}

// state[i][h] = I for every segment i < max_segs and head h (float4 stores)
__global__ void identity_kernel(float *state, long long count4) {
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < count4;
       e += (long long)gridDim.x * blockDim.x) {
    const long long flat = 4 * e;
    const int ij = (int)(flat % (kD * kD)), i = ij / kD, j0 = ij % kD;
    float4 x;
    x.x = (i == j0) ? 1.f : 0.f;
    x.y = (i == j0 + 1) ? 1.f : 0.f;
    x.z = (i == j0 + 2) ? 1.f : 0.f;
    x.w = (i == j0 + 3) ? 1.f : 0.f;
    reinterpret_cast<float4 *>(state)[e] = x;
  }
}

constexpr int kCmbCols = 4;     // value columns per combine CTA
constexpr int kMPitch = kD + 4;  // padded row of a staged map: row r's float4 k lands in
                                 // bank group (r + k) mod 8, no conflict across 8 lanes

struct CombineSmem {
  alignas(16) float M[2][kD][kMPitch];  // M_i and M_{i+1} (cp.async double buffer)
  alignas(16) float4 S[kD];             // row k: S[k][c0 .. c0 + 3]
};

// One CTA of 128 threads per (sequence, v-head, 4 value columns): walks the sequence's
// segments in order with S[:, cols] in shared memory; segment i's incoming state is
// written to seg_in[i], then S <- M_i S + L_i, thread r forming row r in fp32 on CUDA
// cores (two partial sums over the keys).  M_{i+1} is staged into shared memory by
// cp.async while step i computes.  The final S is the sequence's state_out.
__global__ void __launch_bounds__(kD) split_combine_kernel(SplitCombineParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  CombineSmem &sm = *reinterpret_cast<CombineSmem *>(smem_raw);
  const int blk = blockIdx.x % (kD / kCmbCols);
  const int nh = blockIdx.x / (kD / kCmbCols);
  const int n = nh / p.hv, h = nh - n * p.hv;
  const int r = threadIdx.x, c0 = blk * kCmbCols;
  const size_t sb = ((size_t)n * p.hv + h) * kD * kD;
  const int first = p.seg_first[n], last = p.seg_first[n + 1];
  auto stage = [&](int i, int buf) {  // M_i into buffer buf, 16-byte pieces along rows
    const float *src = p.map + ((size_t)i * p.hv + h) * kD * kD;
    for (int e = r; e < kD * kD / 4; e += kD) {
      const int row = e >> 5, q4 = e & 31;
      cp_async16(&sm.M[buf][row][4 * q4], src + (size_t)row * kD + 4 * q4, 16);
    }
    cp_async_commit();
  };
  if (first < last) stage(first, 0);
  sm.S[r] = p.state_in ? *reinterpret_cast<const float4 *>(p.state_in + sb + (size_t)r * kD + c0)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i = first; i < last; ++i) {
    const int buf = (i - first) & 1;
    if (i + 1 < last) {
      stage(i + 1, buf ^ 1);  // the other buffer's last reader passed the previous barrier
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();  // M_i landed for every thread; S is current
    const size_t ib = ((size_t)i * p.hv + h) * kD * kD + (size_t)r * kD;
    *reinterpret_cast<float4 *>(p.seg_in + ib + c0) = sm.S[r];
    // L_i's row is added last, so that its load overlaps the products
    const float4 l = *reinterpret_cast<const float4 *>(p.local + ib + c0);
    float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
    const float4 *Mr = reinterpret_cast<const float4 *>(&sm.M[buf][r][0]);
#pragma unroll 8
    for (int k4 = 0; k4 < kD / 4; ++k4) {
      const float4 m = Mr[k4];
      const float4 s0 = sm.S[4 * k4], s1 = sm.S[4 * k4 + 1], s2 = sm.S[4 * k4 + 2],
                   s3 = sm.S[4 * k4 + 3];
      a0.x = fmaf(m.x, s0.x, a0.x); a0.y = fmaf(m.x, s0.y, a0.y);
      a0.z = fmaf(m.x, s0.z, a0.z); a0.w = fmaf(m.x, s0.w, a0.w);
      a1.x = fmaf(m.y, s1.x, a1.x); a1.y = fmaf(m.y, s1.y, a1.y);
      a1.z = fmaf(m.y, s1.z, a1.z); a1.w = fmaf(m.y, s1.w, a1.w);
      a0.x = fmaf(m.z, s2.x, a0.x); a0.y = fmaf(m.z, s2.y, a0.y);
      a0.z = fmaf(m.z, s2.z, a0.z); a0.w = fmaf(m.z, s2.w, a0.w);
      a1.x = fmaf(m.w, s3.x, a1.x); a1.y = fmaf(m.w, s3.y, a1.y);
      a1.z = fmaf(m.w, s3.z, a1.z); a1.w = fmaf(m.w, s3.w, a1.w);
    }
    __syncthreads();  // every row of the old S (and of M_i) has been read
    sm.S[r] = make_float4(a0.x + a1.x + l.x, a0.y + a1.y + l.y, a0.z + a1.z + l.z,
                          a0.w + a1.w + l.w);
  }
  __syncthreads();
  *reinterpret_cast<float4 *>(p.state_out + sb + (size_t)r * kD + c0) = sm.S[r];
}

}  // namespace

cudaError_t launch_split_plan(const SplitPlanParams &p, cudaStream_t stream) {
  split_plan_kernel<<<1, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_identity(float *state, long long states, cudaStream_t stream) {
  const long long count4 = states * (kD * kD / 4);
  if (count4 == 0) return cudaSuccess;
  const long long want = (count4 + 255) / 256;
  identity_kernel<<<(unsigned)(want < 4096 ? want : 4096), 256, 0, stream>>>(state, count4);
  return cudaGetLastError();
}

cudaError_t launch_split_combine(const SplitCombineParams &p, cudaStream_t stream) {
  const long long units = (long long)p.num_seqs * p.hv * (kD / kCmbCols);
  if (units == 0) return cudaSuccess;
  const size_t smem = sizeof(CombineSmem);
  cudaError_t err = cudaFuncSetAttribute(split_combine_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  split_combine_kernel<<<(unsigned)units, kD, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
