// Fused Q/K RMSNorm + axial 3-D RoPE, in place, one pass over HBM.
//
// "QK normalization with partial RoPE" is operator group 2 of Sol-H3
// (arXiv 2609.35110), section 3.5 "Kernel Fusion"; the vLLM-Omni blog
// ("MiniMax H3 on vLLM-Omni"), section 3.2, fuses the same Q/K RMSNorm and
// RoPE.  The point of the fusion is to read each wide activation once and
// write it once.
//
// Work split: one warp per row r, covering both tensors and every head.
// Lane l owns channel chunks [8s, 8s+8) and [64+8s, 64+8s+8) with s = l % 8,
// and head-units u = l/8, l/8 + 4, ... of the 2*H units (q heads, then k
// heads) of the row.  Each warp-wide 16-byte load therefore covers four
// whole 128-byte segments, the 8 lanes of a head reduce the sum of squares
// with three xor-shuffles, and the 8 (cos, sin) pairs a lane needs are
// computed once per row and reused across all 2*H units.  Loads are issued
// for kBatch units before any arithmetic so that each lane keeps
// kBatch * 32 bytes in flight.
#include "h3_internal.h"

namespace h3 {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kBatch = 7;  // units per lane in flight (7 * 32 B)

struct NormRopeParams {
  __nv_bfloat16* x[2];
  int64_t stride[2];
  const __nv_bfloat16* w[2];
  const int32_t* pos;
  int64_t n_rows;
  int n_heads;
  float eps;
  float inv_freq[64];  // per channel pair p = (2p, 2p+1): theta^(-2j/d) of its section
  int32_t axis[64];    // 0 = t, 1 = h, 2 = w, -1 = not rotated
};

__device__ __forceinline__ void unpack8(const uint4 v, float* f) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(u[i] << 16);
    f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // round to nearest even
  return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    qk_norm_rope_kernel(const __grid_constant__ NormRopeParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  if (row >= p.n_rows) return;
  const int sub = lane & 7;
  const int grp = lane >> 3;

  // Rotation of this lane's 8 channel pairs for this row.
  const int32_t* pr = p.pos + row * 3;
  const float pos3[3] = {static_cast<float>(__ldg(pr)), static_cast<float>(__ldg(pr + 1)),
                         static_cast<float>(__ldg(pr + 2))};
  float cs[8], sn[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int pair = (i < 4) ? 4 * sub + i : 32 + 4 * sub + (i - 4);
    const int ax = p.axis[pair];
    if (ax < 0) {
      cs[i] = 1.0f;
      sn[i] = 0.0f;
    } else {
      sincosf(pos3[ax] * p.inv_freq[pair], &sn[i], &cs[i]);
    }
  }

  const int n_units = 2 * p.n_heads;
  for (int base = 0; base < n_units; base += 4 * kBatch) {
    uint4 xa[kBatch], xb[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int u = base + 4 * b + grp;
      if (u < n_units) {
        const int t = u >= p.n_heads;
        const int h = u - t * p.n_heads;
        const uint4* src =
            reinterpret_cast<const uint4*>(p.x[t] + row * p.stride[t] + h * kHeadDim);
        xa[b] = __ldcs(src + sub);
        xb[b] = __ldcs(src + 8 + sub);
      } else {
        xa[b] = make_uint4(0, 0, 0, 0);
        xb[b] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int u = base + 4 * b + grp;
      float x[16];
      unpack8(xa[b], x);
      unpack8(xb[b], x + 8);
      float ss0 = 0.f, ss1 = 0.f;
#pragma unroll
      for (int c = 0; c < 16; c += 2) {
        ss0 = fmaf(x[c], x[c], ss0);
        ss1 = fmaf(x[c + 1], x[c + 1], ss1);
      }
      float ss = ss0 + ss1;
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      ss += __shfl_xor_sync(0xffffffffu, ss, 2);
      ss += __shfl_xor_sync(0xffffffffu, ss, 4);
      if (u >= n_units) continue;  // uniform across the 8 lanes of a unit
      const float r = rsqrtf(ss * (1.0f / kHeadDim) + p.eps);
      const int t = u >= p.n_heads;
      const int h = u - t * p.n_heads;
      const uint4* wsrc = reinterpret_cast<const uint4*>(p.w[t] + h * kHeadDim);
      float w[16];
      unpack8(__ldg(wsrc + sub), w);
      unpack8(__ldg(wsrc + 8 + sub), w + 8);
      uint32_t o[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float y0 = x[2 * i] * r * w[2 * i];
        const float y1 = x[2 * i + 1] * r * w[2 * i + 1];
        const float z0 = y0 * cs[i] - y1 * sn[i];
        const float z1 = y0 * sn[i] + y1 * cs[i];
        o[i] = pack2(z0, z1);
      }
      uint4* dst = reinterpret_cast<uint4*>(p.x[t] + row * p.stride[t] + h * kHeadDim);
      __stcs(dst + sub, make_uint4(o[0], o[1], o[2], o[3]));
      __stcs(dst + 8 + sub, make_uint4(o[4], o[5], o[6], o[7]));
    }
  }
}

}  // namespace

cudaError_t launch_qk_norm_rope(const NormRopeArgs& a, cudaStream_t stream) {
  NormRopeParams p{};
  p.x[0] = a.q;
  p.x[1] = a.k;
  p.stride[0] = a.q_stride;
  p.stride[1] = a.k_stride;
  p.w[0] = a.wq;
  p.w[1] = a.wk;
  p.pos = a.pos;
  p.n_rows = a.n_rows;
  p.n_heads = a.n_heads;
  p.eps = a.eps;
  // Per-pair section and inverse frequency, in double, rounded once.
  const int edges[3] = {a.rot[0], a.rot[0] + a.rot[1], a.rot[0] + a.rot[1] + a.rot[2]};
  for (int pair = 0; pair < 64; ++pair) {
    const int c = 2 * pair;
    int ax = -1, off = 0;
    for (int s = 0; s < 3; ++s) {
      if (c < edges[s]) {
        ax = s;
        break;
      }
      off = edges[s];
    }
    p.axis[pair] = ax;
    if (ax >= 0) {
      const double d = static_cast<double>(a.rot[ax]);
      const double j = static_cast<double>((c - off) / 2);
      p.inv_freq[pair] = static_cast<float>(std::pow(static_cast<double>(a.theta), -2.0 * j / d));
    } else {
      p.inv_freq[pair] = 0.0f;
    }
  }
  const int64_t blocks = (a.n_rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
  qk_norm_rope_kernel<<<static_cast<unsigned>(blocks), kWarpsPerBlock * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace h3
