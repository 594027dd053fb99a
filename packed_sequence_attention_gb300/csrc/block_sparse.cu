// Sol-Attn block selection (Sol-H3, arXiv 2609.35110, section 3.4
// "Per-step dynamic sparsity" and "Safety rails and the exact prefix KV
// sink"): 128-row block means of Q and K, block-level scores, and per query
// block the list of KV blocks whose score exceeds mu + tau * sigma, with the
// prefix query blocks dense and the prefix KV blocks always kept.
//
// Readings where the page leaves the method open: the block-level score is
// scale * <mean query of the block, mean key of the block>; sigma is the
// population standard deviation over all KV blocks; "exceed" is strict;
// a block holding any prefix row is a prefix block.  Arithmetic is fp32 in
// a fixed order, so the selection is deterministic run to run.
#include <atomic>
#include <cmath>

#include "h3_internal.h"

namespace h3 {
namespace {

constexpr int kBlk = 128;

__device__ __forceinline__ uint4 ld_stream16(const uint4* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void add8(float* acc, const uint4 v) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] += __uint_as_float(u[i] << 16);
    acc[2 * i + 1] += __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

// grid (n_heads, n_blocks, n_tensors), 128 threads: 16 chunks of 8 channels
// x 8 row slices.  Consecutive CTAs take consecutive heads of the same
// block, so the CTAs running together read whole rows between them.  A
// thread sums rows slice, slice + 8, ... of its chunk in that order, then
// the 8 slices are added in order: a fixed summation order, so the means
// are deterministic.  A full block issues all 16 of a thread's loads before
// the first add.
__global__ void __launch_bounds__(128) block_means_kernel(MeansJob job, int64_t n_rows, int H) {
  __shared__ float red[8][kHeadDim];
  const int h = blockIdx.x, b = blockIdx.y;
  const bool second = blockIdx.z != 0;
  const __nv_bfloat16* x = second ? job.x[1] : job.x[0];
  const int64_t stride = second ? job.stride[1] : job.stride[0];
  float* out = second ? job.out[1] : job.out[0];
  const int chunk = threadIdx.x & 15, slice = threadIdx.x >> 4;
  const int64_t r0 = static_cast<int64_t>(b) * kBlk;
  const int rows = static_cast<int>(n_rows - r0 < kBlk ? n_rows - r0 : kBlk);
  const uint4* src = reinterpret_cast<const uint4*>(x + (r0 + slice) * stride + h * kHeadDim) + chunk;
  const int64_t step = stride;  // 8 rows apart, in 16-byte units: 8 * stride * 2 B / 16 B
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (rows == kBlk) {
    uint4 v[kBlk / 8];
#pragma unroll
    for (int i = 0; i < kBlk / 8; ++i) v[i] = ld_stream16(src + i * step);
#pragma unroll
    for (int i = 0; i < kBlk / 8; ++i) add8(acc, v[i]);
  } else {
    for (int r = slice, i = 0; r < rows; r += 8, ++i) add8(acc, ld_stream16(src + i * step));
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) red[slice][chunk * 8 + i] = acc[i];
  __syncthreads();
  const int c = threadIdx.x;
  float sum = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) sum += red[k][c];
  out[(static_cast<int64_t>(b) * H + h) * kHeadDim + c] = sum / static_cast<float>(rows);
}

constexpr int kSelThreads = 256;
constexpr int kSelQB = kSelThreads / 32;  // query blocks per CTA: one warp each

// grid (ceil(nqb / kSelQB), n_heads): the scores of kSelQB query blocks
// against every KV block (each key mean is read once per CTA and dotted with
// all kSelQB query means), then per query block -- one warp each -- the mean
// and population std of its scores and the ordered list of kept blocks.
// Dynamic shared memory: kSelQB x nkb scores.
__global__ void __launch_bounds__(kSelThreads) block_select_kernel(
    const float* __restrict__ qm, const float* __restrict__ km, int nqb, int nkb, int H,
    float scale, float tau, int n_prefix, float* __restrict__ scores_out,
    int32_t* __restrict__ lists, int32_t* __restrict__ counts) {
  extern __shared__ float sc[];  // [kSelQB][nkb]
  __shared__ float4 qv[kSelQB][kHeadDim / 4];
  const int a0 = blockIdx.x * kSelQB, h = blockIdx.y, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < kSelQB * kHeadDim / 4; i += kSelThreads) {
    const int qb = i / (kHeadDim / 4), c4 = i % (kHeadDim / 4);
    qv[qb][c4] = a0 + qb < nqb
                     ? __ldg(reinterpret_cast<const float4*>(qm + (static_cast<int64_t>(a0 + qb) * H + h) * kHeadDim) + c4)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  __syncthreads();
  for (int b = tid; b < nkb; b += kSelThreads) {
    const float4* kr = reinterpret_cast<const float4*>(km + (static_cast<int64_t>(b) * H + h) * kHeadDim);
    float s[kSelQB];
#pragma unroll
    for (int qb = 0; qb < kSelQB; ++qb) s[qb] = 0.f;
#pragma unroll 4
    for (int c4 = 0; c4 < kHeadDim / 4; ++c4) {
      const float4 kv = __ldg(kr + c4);
#pragma unroll
      for (int qb = 0; qb < kSelQB; ++qb) {  // channel order fixed: the sum is deterministic
        const float4 q = qv[qb][c4];
        s[qb] = fmaf(q.x, kv.x, s[qb]);
        s[qb] = fmaf(q.y, kv.y, s[qb]);
        s[qb] = fmaf(q.z, kv.z, s[qb]);
        s[qb] = fmaf(q.w, kv.w, s[qb]);
      }
    }
#pragma unroll
    for (int qb = 0; qb < kSelQB; ++qb) sc[qb * nkb + b] = s[qb] * scale;
  }
  __syncthreads();
  const int a = a0 + warp;
  if (a >= nqb) return;
  const float* row = sc + warp * nkb;
  // mean, then the population variance about it (two passes, fixed order)
  float part = 0.f;
  for (int b = lane; b < nkb; b += 32) part += row[b];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  const float mu = part / static_cast<float>(nkb);
  part = 0.f;
  for (int b = lane; b < nkb; b += 32) part += (row[b] - mu) * (row[b] - mu);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  const float thr = mu + tau * sqrtf(part / static_cast<float>(nkb));
  // ordered compaction of the kept blocks
  int32_t* list = lists + (static_cast<int64_t>(h) * nqb + a) * nkb;
  int base = 0;
  for (int b0 = 0; b0 < nkb; b0 += 32) {
    const int b = b0 + lane;
    const bool keep = b < nkb && (a < n_prefix || b < n_prefix || row[b] > thr);
    const unsigned m = __ballot_sync(0xffffffffu, keep);
    if (keep) list[base + __popc(m & ((1u << lane) - 1u))] = b;
    base += __popc(m);
  }
  if (lane == 0) counts[static_cast<int64_t>(h) * nqb + a] = base;
  if (scores_out != nullptr)
    for (int b = lane; b < nkb; b += 32)
      scores_out[(static_cast<int64_t>(h) * nqb + a) * nkb + b] = row[b];
}

}  // namespace

cudaError_t launch_block_means(const MeansJob& job, int n_tensors, int64_t n_rows, int H,
                               cudaStream_t stream) {
  const int nb = static_cast<int>((n_rows + kBlk - 1) / kBlk);
  block_means_kernel<<<dim3(H, nb, n_tensors), 128, 0, stream>>>(job, n_rows, H);
  return cudaGetLastError();
}

cudaError_t launch_block_select(const float* qm, const float* km, int nqb, int nkb, int H,
                                float scale, float tau, int n_prefix, float* scores,
                                int32_t* lists, int32_t* counts, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(kSelQB) * nkb * sizeof(float);  // <= 64 KB
  static std::atomic<int> attr_set[64];  // opt-in above 48 KB, once per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (attr_set[dev].load() == 0) {
    e = cudaFuncSetAttribute(block_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSelQB * kMaxSparseBlocks * sizeof(float)));
    if (e != cudaSuccess) return e;
    attr_set[dev].store(1);
  }
  block_select_kernel<<<dim3((nqb + kSelQB - 1) / kSelQB, H), kSelThreads, smem, stream>>>(
      qm, km, nqb, nkb, H, scale, tau, n_prefix, scores, lists, counts);
  return cudaGetLastError();
}

}  // namespace h3
