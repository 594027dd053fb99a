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
#include <cmath>

#include "h3_internal.h"

namespace h3 {
namespace {

constexpr int kBlk = 128;

// grid (n_blocks, n_heads), 128 threads: 16 chunks of 8 channels x 8 row slices.
__global__ void __launch_bounds__(128) block_means_kernel(const __nv_bfloat16* __restrict__ x,
                                                          int64_t stride, int64_t n_rows, int H,
                                                          float* __restrict__ out) {
  __shared__ float red[8][kHeadDim];
  const int b = blockIdx.x, h = blockIdx.y;
  const int chunk = threadIdx.x & 15, slice = threadIdx.x >> 4;
  const int64_t r0 = static_cast<int64_t>(b) * kBlk;
  const int rows = static_cast<int>(n_rows - r0 < kBlk ? n_rows - r0 : kBlk);
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int r = slice; r < rows; r += 8) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + (r0 + r) * stride + h * kHeadDim) + chunk);
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] += __uint_as_float(u[i] << 16);
      acc[2 * i + 1] += __uint_as_float(u[i] & 0xFFFF0000u);
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) red[slice][chunk * 8 + i] = acc[i];
  __syncthreads();
  const int c = threadIdx.x;
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) s += red[k][c];
  out[(static_cast<int64_t>(b) * H + h) * kHeadDim + c] = s / static_cast<float>(rows);
}

constexpr int kSelThreads = 256;

// grid (n_q_blocks, n_heads): scores of one query block against every KV
// block, their mean and population std, and the ordered list of kept blocks.
__global__ void __launch_bounds__(kSelThreads) block_select_kernel(
    const float* __restrict__ qm, const float* __restrict__ km, int nqb, int nkb, int H,
    float scale, float tau, int n_prefix, float* __restrict__ scores_out,
    int32_t* __restrict__ lists, int32_t* __restrict__ counts) {
  __shared__ float qv[kHeadDim];
  __shared__ float sc[kMaxSparseBlocks];
  __shared__ float red[kSelThreads / 32];
  __shared__ int warp_base[kSelThreads / 32 + 1];
  const int a = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  if (tid < kHeadDim) qv[tid] = qm[(static_cast<int64_t>(a) * H + h) * kHeadDim + tid];
  __syncthreads();
  for (int b = tid; b < nkb; b += kSelThreads) {
    const float4* kr = reinterpret_cast<const float4*>(km + (static_cast<int64_t>(b) * H + h) * kHeadDim);
    float s = 0.f;
#pragma unroll 8
    for (int c4 = 0; c4 < kHeadDim / 4; ++c4) {
      const float4 kv = __ldg(kr + c4);
      s = fmaf(qv[4 * c4], kv.x, s);
      s = fmaf(qv[4 * c4 + 1], kv.y, s);
      s = fmaf(qv[4 * c4 + 2], kv.z, s);
      s = fmaf(qv[4 * c4 + 3], kv.w, s);
    }
    sc[b] = s * scale;
  }
  __syncthreads();
  // mean, then the population variance about it (two passes, fixed order)
  auto block_sum = [&](float v) -> float {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.f;
    for (int w = 0; w < kSelThreads / 32; ++w) t += red[w];
    __syncthreads();
    return t;
  };
  float part = 0.f;
  for (int b = tid; b < nkb; b += kSelThreads) part += sc[b];
  const float mu = block_sum(part) / static_cast<float>(nkb);
  part = 0.f;
  for (int b = tid; b < nkb; b += kSelThreads) part += (sc[b] - mu) * (sc[b] - mu);
  const float sd = sqrtf(block_sum(part) / static_cast<float>(nkb));
  const float thr = mu + tau * sd;
  // ordered compaction of the kept blocks
  int32_t* list = lists + (static_cast<int64_t>(h) * nqb + a) * nkb;
  int base = 0;
  for (int b0 = 0; b0 < nkb; b0 += kSelThreads) {
    const int b = b0 + tid;
    const bool keep = b < nkb && (a < n_prefix || b < n_prefix || sc[b] > thr);
    const unsigned m = __ballot_sync(0xffffffffu, keep);
    if (lane == 0) warp_base[warp + 1] = __popc(m);
    __syncthreads();
    if (tid == 0) {
      warp_base[0] = 0;
      for (int w = 1; w <= kSelThreads / 32; ++w) warp_base[w] += warp_base[w - 1];
    }
    __syncthreads();
    if (keep) list[base + warp_base[warp] + __popc(m & ((1u << lane) - 1u))] = b;
    base += warp_base[kSelThreads / 32];
    __syncthreads();
  }
  if (tid == 0) counts[static_cast<int64_t>(h) * nqb + a] = base;
  if (scores_out != nullptr)
    for (int b = tid; b < nkb; b += kSelThreads)
      scores_out[(static_cast<int64_t>(h) * nqb + a) * nkb + b] = sc[b];
}

}  // namespace

cudaError_t launch_block_means(const __nv_bfloat16* x, int64_t stride, int64_t n_rows, int H,
                               float* out, cudaStream_t stream) {
  const int nb = static_cast<int>((n_rows + kBlk - 1) / kBlk);
  block_means_kernel<<<dim3(nb, H), 128, 0, stream>>>(x, stride, n_rows, H, out);
  return cudaGetLastError();
}

cudaError_t launch_block_select(const float* qm, const float* km, int nqb, int nkb, int H,
                                float scale, float tau, int n_prefix, float* scores,
                                int32_t* lists, int32_t* counts, cudaStream_t stream) {
  block_select_kernel<<<dim3(nqb, H), kSelThreads, 0, stream>>>(qm, km, nqb, nkb, H, scale, tau,
                                                               n_prefix, scores, lists, counts);
  return cudaGetLastError();
}

}  // namespace h3
