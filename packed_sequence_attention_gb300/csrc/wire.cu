// Wire formats at the attention boundary (Sol-H3, arXiv 2609.35110, section
// 3.2 "Optimized attention collectives" and "Quantized communication").
//
// * Packed QKV, destination-major: Q, K and V are read through their own row
//   strides and written in one pass into [n_dest][rows][H/n_dest] records of
//   q, k, v back to back -- bf16 (768 B, a pure permutation) or block-INT8
//   (400 B: 3 x 128 int8 values, 12 group-32 UE5M3 scale codes, 4 zero bytes).
// * Attention output records [rows][H_local]: bf16 (256 B), block-INT8
//   (144 B: 128 values, 4 scale codes, 12 zero bytes) or raw FP8 E4M3
//   (128 B, round-to-nearest-even saturated at +-448); the inverse head merge
//   turns [n_src][rows][H/n_src] records back into [rows][H][128].
//
// UE5M3 (the page names it without spelling it out): unsigned, 5 exponent
// bits with bias 15, 3 mantissa bits, every code finite and positive:
// value(c) = 2^((c >> 3) - 15) * (1 + (c & 7) / 8).  A group of 32 values
// takes the smallest code with 127 * value >= max|x| -- a comparison that is
// exact in fp32 -- and stores rint(x / value) as int8.
//
// One warp handles one (token, head) record; lane l owns channels 4l..4l+3
// of each tensor, so the 8 lanes of a 32-channel group reduce its max with
// three xor-shuffles.
#include <cuda_fp16.h>

#include <atomic>

#include "h3_internal.h"
#include "ptx.cuh"

namespace h3 {
namespace {

constexpr int kWarps = 8;
using ptx::ffma2;
using ptx::fadd2;
using ptx::fmax3;

// value(c) = 2^((c >> 3) - 15) * (1 + (c & 7) / 8), built as fp32 bits
// (biased exponent (c >> 3) + 112, top 3 mantissa bits c & 7): exact.
__device__ __forceinline__ float ue5m3_value(int c) {
  return __uint_as_float((static_cast<uint32_t>((c >> 3) + 112) << 23) |
                         (static_cast<uint32_t>(c & 7) << 20));
}

// Smallest code c with 127 * value(c) >= amax.  The code just above
// fl(amax / 127) is at most one step from the answer (code values are 1/16
// apart relatively, the two roundings 2^-23), so one exact compare settles
// it (127 * value has at most 11 significant bits).
__device__ __forceinline__ int ue5m3_code(float amax) {
  const uint32_t b = __float_as_uint(amax * (1.0f / 127.0f));
  int c = (static_cast<int>(b >> 23) - 112) * 8 + static_cast<int>((b >> 20) & 7u) +
          ((b & 0xFFFFFu) != 0u ? 1 : 0);
  c = min(max(c, 0), 255);
  if (c > 0 && 127.0f * ue5m3_value(c - 1) >= amax) --c;
  else if (c < 255 && 127.0f * ue5m3_value(c) < amax) ++c;
  return c;
}

__device__ __forceinline__ void unpack4(uint2 u, float* f) {
  f[0] = __uint_as_float(u.x << 16);
  f[1] = __uint_as_float(u.x & 0xFFFF0000u);
  f[2] = __uint_as_float(u.y << 16);
  f[3] = __uint_as_float(u.y & 0xFFFF0000u);
}

__device__ __forceinline__ uint2 pack4_bf16(const float* f) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(f[0], f[1]);
  const __nv_bfloat162 b = __floats2bfloat162_rn(f[2], f[3]);
  return make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
}

__device__ __forceinline__ uint2 ld8(const void* p) {
  return __ldg(reinterpret_cast<const uint2*>(p));
}

// rint(x / s), ties to even, for 4 values with |x| <= 127 s, without a
// division and on the FMA pipe only (paired fp32 operations): the 4 int8
// results in two's complement, one byte each.  Adding M = 1.5 * 2^23
// rounds to an integer (ties to even).
// With r = 1/s correctly rounded, q' = rint(x * r) is within one of the
// answer and the remainder x - q' s is exact in fp32 (24 bits span it).
// t = q' + (x - q' s) * r is then within 2^-25 of x / s: an exact tie
// k + 1/2 comes out as exactly k + 1/2 (the error is below half an ulp),
// and any other quotient stays more than 2^-6 / 30 away from a half-integer
// (x has 8 significant bits, s = m 2^b with m in 8..15), so rounding t
// gives rint(x / s) in every case.  The low byte of t + M is the result.
__device__ __forceinline__ uint32_t quant4(const float* x, float s, float r) {
  constexpr float kMagic = 12582912.0f;
  float q[4], e[4], t[4];
#pragma unroll
  for (int i = 0; i < 4; i += 2) {
    ffma2(q[i], q[i + 1], x[i], x[i + 1], r, r, kMagic, kMagic);
    fadd2(q[i], q[i + 1], q[i], q[i + 1], -kMagic, -kMagic);      // q' = rint(x r)
    ffma2(e[i], e[i + 1], q[i], q[i + 1], -s, -s, x[i], x[i + 1]);  // x - q' s, exact
    ffma2(t[i], t[i + 1], e[i], e[i + 1], r, r, q[i], q[i + 1]);   // q' + (x - q' s) r
    fadd2(t[i], t[i + 1], t[i], t[i + 1], kMagic, kMagic);
  }
  return __byte_perm(__byte_perm(__float_as_uint(t[0]), __float_as_uint(t[1]), 0x0040),
                     __byte_perm(__float_as_uint(t[2]), __float_as_uint(t[3]), 0x0040), 0x5410);
}

// max |x| over a 32-channel group (its 8 lanes hold 4 values each).
__device__ __forceinline__ float group_amax(const float* f) {
  float a = fmaxf(fmax3(fabsf(f[0]), fabsf(f[1]), fabsf(f[2])), fabsf(f[3]));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
  return fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
}

// Scale codes of N <= 8 items (tensors or records) at once: lane j of each
// 8-lane group computes the code of item j of that group, then every lane
// fetches s and 1/s of its group for all items.  Returns this lane's code
// (item lane & 7, meaningful when that is < N); *sat tells the whole warp
// whether some group's max lies past 127 s (possible with the largest code
// only), in which case values must be clamped to +-127 s first.
template <int N>
__device__ __forceinline__ int group_scales(const float (&amax)[N], float (&s)[N], float (&r)[N],
                                            bool* sat) {
  const int lane = threadIdx.x & 31, j = lane & 7;
  float a = amax[0];
#pragma unroll
  for (int i = 1; i < N; ++i) a = j == i ? amax[i] : a;
  const int c = ue5m3_code(a);
  const float sc = ue5m3_value(c), rc = __frcp_rn(sc);
  *sat = __any_sync(0xffffffffu, j < N && a > 127.0f * sc);
#pragma unroll
  for (int i = 0; i < N; ++i) {
    s[i] = __shfl_sync(0xffffffffu, sc, (lane & 24) | i);
    r[i] = __shfl_sync(0xffffffffu, rc, (lane & 24) | i);
  }
  return c;
}

__device__ __forceinline__ void clamp4(float* f, float s) {
  const float lim = 127.0f * s;
#pragma unroll
  for (int i = 0; i < 4; ++i) f[i] = fminf(fmaxf(f[i], -lim), lim);
}

__device__ __forceinline__ uint2 dequant4(uint32_t bytes, int code) {
  const float s = ue5m3_value(code);
  float f[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) f[i] = static_cast<float>(static_cast<int8_t>(bytes >> (8 * i))) * s;
  return pack4_bf16(f);
}

__device__ __forceinline__ uint32_t fp8x4(const float* f) {
  uint16_t lo, hi;
  // cvt.rn.satfinite.e4m3x2.f32 d, a, b: a -> upper byte, b -> lower byte
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(f[1]), "f"(f[0]));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(f[3]), "f"(f[2]));
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

__device__ __forceinline__ uint2 fp8x4_to_bf16(uint32_t w) {
  uint32_t h01, h23;  // e4m3x2 -> f16x2 is exact; f16 -> fp32 -> bf16 is exact too
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h01) : "h"(static_cast<uint16_t>(w & 0xFFFF)));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h23) : "h"(static_cast<uint16_t>(w >> 16)));
  const __half2 a = *reinterpret_cast<const __half2*>(&h01);
  const __half2 b = *reinterpret_cast<const __half2*>(&h23);
  const float f[4] = {__low2float(a), __high2float(a), __low2float(b), __high2float(b)};
  return pack4_bf16(f);
}

// Every kernel below: warp w of block b takes the kU consecutive units
// (row, head) starting at (b * kWarps + w) * kU and issues all their loads
// before it computes, so a lane has kU loads in flight; lane l owns
// channels 4l..4l+3 of a head.
template <int kU>
struct Units {
  int64_t r[kU];
  int h[kU];
  bool ok[kU];
  // total < 2^31 (checked on the host), so 32-bit arithmetic suffices.
  __device__ __forceinline__ Units(int64_t total, int H)
      : Units(total, H, blockIdx.x * kWarps + (threadIdx.x >> 5)) {}
  // The kU units of pass p: p * kU, p * kU + 1, ...
  __device__ __forceinline__ Units(int64_t total, int H, uint32_t pass) {
    const uint32_t u0 = pass * kU;
    int64_t row = u0 / static_cast<uint32_t>(H);
    int head = static_cast<int>(u0 - static_cast<uint32_t>(row) * static_cast<uint32_t>(H));
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      r[u] = row;
      h[u] = head;
      ok[u] = static_cast<int64_t>(u0) + u < total;
      if (++head == H) {
        head = 0;
        ++row;
      }
    }
  }
};

__global__ void __launch_bounds__(kWarps * 32) pack_qkv_bf16_kernel(
    const __nv_bfloat16* __restrict__ q, int64_t qs, const __nv_bfloat16* __restrict__ k, int64_t ks,
    const __nv_bfloat16* __restrict__ v, int64_t vs, int64_t n_rows, int H, int n_dest,
    uint8_t* __restrict__ wire) {
  constexpr int kU = 2;
  const int lane = threadIdx.x & 31;
  const Units<kU> un(n_rows * H, H);
  const int hl = H / n_dest;
  uint2 in[kU][3] = {};
#pragma unroll
  for (int u = 0; u < kU; ++u) {
    if (un.ok[u]) {
      const int64_t c = un.h[u] * kHeadDim + lane * 4;
      in[u][0] = ld8(q + un.r[u] * qs + c);
      in[u][1] = ld8(k + un.r[u] * ks + c);
      in[u][2] = ld8(v + un.r[u] * vs + c);
    }
  }
#pragma unroll
  for (int u = 0; u < kU; ++u) {
    if (!un.ok[u]) break;
    const int d = un.h[u] / hl, hloc = un.h[u] - d * hl;
    uint8_t* dst = wire + ((static_cast<int64_t>(d) * n_rows + un.r[u]) * hl + hloc) * 768;
#pragma unroll
    for (int t = 0; t < 3; ++t) *reinterpret_cast<uint2*>(dst + t * 256 + lane * 8) = in[u][t];
  }
}

// Block-INT8 QKV records.  Quantising costs more issue slots than the bytes
// take to move, so the layout is chosen to share work: a half-warp handles
// one (token, head) unit, lane l owning channels 8 (l & 15) .. + 7 of each of
// q, k and v (16-byte loads), so the 4 lanes of a 32-channel group reduce its
// max with two xor-shuffles and lane j < 3 of the group derives the scale
// code of tensor j once for the whole group.  The kernel is persistent and
// software-pipelined: a warp loads its next pair of units before it
// quantises the current one, and steps its unit indices without divisions.
constexpr int kInt8Warps = 8;

// 8 values of one tensor -> 8 int8 (two words), scale s, reciprocal r.
__device__ __forceinline__ uint2 quant8(const float* x, float s, float r) {
  return make_uint2(quant4(x, s, r), quant4(x + 4, s, r));
}

__device__ __forceinline__ void unpack8(const uint4 u, float* f) {
  unpack4(make_uint2(u.x, u.y), f);
  unpack4(make_uint2(u.z, u.w), f + 4);
}

__global__ void __launch_bounds__(kInt8Warps * 32, 4) pack_qkv_int8_kernel(
    const __nv_bfloat16* __restrict__ q, int64_t qs, const __nv_bfloat16* __restrict__ k, int64_t ks,
    const __nv_bfloat16* __restrict__ v, int64_t vs, int64_t n_rows, int H, int n_dest,
    uint8_t* __restrict__ wire) {
  constexpr int kRec = 400;
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4, l16 = lane & 15;
  const int j = lane & 3;               // lane within its 32-channel group
  const int grp = l16 >> 2;             // the group (0..3) of this lane's channels
  const int hl = H / n_dest;
  const uint32_t total = static_cast<uint32_t>(n_rows * H);  // < 2^31, checked on the host
  // 8 / (8 + m), correctly rounded, for m = lane & 7: 1 / value(c) is this
  // times 2^(15 - (c >> 3)), with m = c & 7 (exact scaling by a power of 2).
  const float recip_tbl = __fdiv_rn(8.0f, static_cast<float>(8 + (lane & 7)));
  // This lane's unit of pass p is u = (p * 2) + half = row H + d hl + hloc.
  // The next pass is `stride` passes on: u grows by adv = stride * 2 = drow H
  // + dd hl + dh, so (row, d, hloc) advance by constants with carries.
  const uint32_t stride = gridDim.x * kInt8Warps;
  const uint32_t adv = stride * 2;
  const uint32_t drow = adv / static_cast<uint32_t>(H);
  const uint32_t rem = adv - drow * static_cast<uint32_t>(H);
  const int dd = static_cast<int>(rem) / hl, dh = static_cast<int>(rem) - dd * hl;
  uint32_t u = (blockIdx.x * kInt8Warps + (threadIdx.x >> 5)) * 2 + half;
  int64_t row = u / static_cast<uint32_t>(H);
  int d, hloc;
  {
    const int head = static_cast<int>(u - static_cast<uint32_t>(row) * static_cast<uint32_t>(H));
    d = head / hl;
    hloc = head - d * hl;
  }
  const int c8 = l16 * 8;
  auto load = [&](uint32_t uu, int64_t r, int dx, int hx, uint4 (&in)[3]) {
    if (uu < total) {
      const int64_t c = static_cast<int64_t>(dx * hl + hx) * kHeadDim + c8;
      in[0] = __ldg(reinterpret_cast<const uint4*>(q + r * qs + c));
      in[1] = __ldg(reinterpret_cast<const uint4*>(k + r * ks + c));
      in[2] = __ldg(reinterpret_cast<const uint4*>(v + r * vs + c));
    } else {
      in[0] = in[1] = in[2] = make_uint4(0u, 0u, 0u, 0u);
    }
  };
  uint4 in[3];
  load(u, row, d, hloc, in);
  // Whole warps leave together: the pass loop runs while either half has a unit.
  while (__any_sync(0xffffffffu, u < total)) {
    const uint32_t nu = u + adv;
    int64_t nrow = row + drow;
    int nd = d + dd, nh = hloc + dh;
    if (nh >= hl) {
      nh -= hl;
      ++nd;
    }
    if (nd >= n_dest) {
      nd -= n_dest;
      ++nrow;
    }
    uint4 nin[3];
    load(nu, nrow, nd, nh, nin);
    // this lane's 8 values of each tensor and the group maxima
    float f[3][8], amax[3];
#pragma unroll
    for (int t = 0; t < 3; ++t) {
      unpack8(in[t], f[t]);
      float a = fmax3(fabsf(f[t][0]), fabsf(f[t][1]), fabsf(f[t][2]));
      a = fmax3(a, fabsf(f[t][3]), fabsf(f[t][4]));
      a = fmax3(a, fabsf(f[t][5]), fabsf(f[t][6]));
      a = fmaxf(a, fabsf(f[t][7]));
      a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
      amax[t] = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    }
    // lane j < 3 of each group: the code of tensor j; then s and 1/s of all
    // three tensors for every lane of the group
    const float a = j == 0 ? amax[0] : (j == 1 ? amax[1] : amax[2]);
    const int code = ue5m3_code(a);
    const float sc = ue5m3_value(code);
    const float rc = __uint_as_float(
        __float_as_uint(__shfl_sync(0xffffffffu, recip_tbl, code & 7)) +
        (static_cast<uint32_t>(15 - (code >> 3)) << 23));
    const bool sat = __any_sync(0xffffffffu, j < 3 && a > 127.0f * sc);
    float s[3], r[3];
#pragma unroll
    for (int t = 0; t < 3; ++t) {
      s[t] = __shfl_sync(0xffffffffu, sc, (lane & ~3) | t);
      r[t] = __shfl_sync(0xffffffffu, rc, (lane & ~3) | t);
    }
    if (sat) {
#pragma unroll
      for (int t = 0; t < 3; ++t) {
        clamp4(f[t], s[t]);
        clamp4(f[t] + 4, s[t]);
      }
    }
    if (u < total) {
      uint8_t* dst = wire + ((static_cast<int64_t>(d) * n_rows + row) * hl + hloc) * kRec;
#pragma unroll
      for (int t = 0; t < 3; ++t)
        *reinterpret_cast<uint2*>(dst + t * 128 + c8) = quant8(f[t], s[t], r[t]);
      // codes: tensor j, group grp at byte 384 + 4 j + grp; lane 15 of the
      // half clears the 4 pad bytes
      if (j < 3) dst[384 + 4 * j + grp] = static_cast<uint8_t>(code);
      if (l16 == 15) *reinterpret_cast<uint32_t*>(dst + 396) = 0u;
    }
    u = nu;
    row = nrow;
    d = nd;
    hloc = nh;
#pragma unroll
    for (int t = 0; t < 3; ++t) in[t] = nin[t];
  }
}

// BF16 QKV unpack.  Records of one part are [rows][hl], so unit u is record u.
__global__ void __launch_bounds__(kWarps * 32) unpack_qkv_bf16_kernel(
    const uint8_t* __restrict__ wire, int64_t n_rows, int hl, __nv_bfloat16* __restrict__ q,
    int64_t qs, __nv_bfloat16* __restrict__ k, int64_t ks, __nv_bfloat16* __restrict__ v,
    int64_t vs) {
  constexpr int kU = 2;
  const int lane = threadIdx.x & 31;
  const Units<kU> un(n_rows * hl, hl);
  uint2 in[kU][3];
#pragma unroll
  for (int u = 0; u < kU; ++u) {
    if (un.ok[u]) {
      const uint8_t* src = wire + (un.r[u] * hl + un.h[u]) * 768;
#pragma unroll
      for (int t = 0; t < 3; ++t) in[u][t] = ld8(src + t * 256 + lane * 8);
    }
  }
#pragma unroll
  for (int u = 0; u < kU; ++u) {
    if (!un.ok[u]) break;
    const int64_t c = un.h[u] * kHeadDim + lane * 4;
    __nv_bfloat16* dst[3] = {q + un.r[u] * qs + c, k + un.r[u] * ks + c, v + un.r[u] * vs + c};
#pragma unroll
    for (int t = 0; t < 3; ++t) *reinterpret_cast<uint2*>(dst[t]) = in[u][t];
  }
}

// Block-INT8 QKV unpack.  A quarter-warp decodes one tensor row (the 128
// values of q, k or v of one record) per pass; lane s of the quarter owns
// channels 8s .. 8s+7 and 64+8s .. 64+8s+7, so that each of its two 16-byte
// stores covers, across the quarter, 128 contiguous bytes (whole sectors),
// and each of its two 8-byte loads 64 contiguous bytes; one 4-byte load
// brings the tensor's four scale codes.  Tensor rows are numbered
// f = 3 * record + tensor, and the grid's warp count is a multiple of 3, so a
// quarter-warp that advances by 4 * warps keeps its tensor and moves its
// (row, head) by constants with a carry, without dividing.  The next pass's
// bytes are loaded before the current ones are decoded.
constexpr int kUnpackWarps = 8;

__global__ void __launch_bounds__(kUnpackWarps * 32) unpack_qkv_int8_kernel(
    const uint8_t* __restrict__ wire, uint32_t n_rec, uint32_t hl, __nv_bfloat16* __restrict__ q,
    int64_t qs, __nv_bfloat16* __restrict__ k, int64_t ks, __nv_bfloat16* __restrict__ v,
    int64_t vs) {
  const int lane = threadIdx.x & 31;
  const int sub = lane & 7;
  const uint32_t f0 = (blockIdx.x * kUnpackWarps + (threadIdx.x >> 5)) * 4 + (lane >> 3);
  const int t = static_cast<int>(f0 % 3);
  const uint32_t du = gridDim.x * kUnpackWarps / 3 * 4;  // records per pass
  const uint32_t du_row = du / hl, du_head = du - du_row * hl;
  uint32_t u = f0 / 3;
  uint32_t row = u / hl, head = u - row * hl;
  __nv_bfloat16* const base = t == 0 ? q : (t == 1 ? k : v);
  const int64_t stride = t == 0 ? qs : (t == 1 ? ks : vs);
  const uint32_t off = t * 128 + sub * 8;  // value bytes of channels 8s.. (and 64 + 8s.. at +64)
  const int g0 = sub >> 2;                 // 32-channel groups of the two chunks: g0 and g0 + 2
  uint2 b0 = make_uint2(0u, 0u), b1 = b0;
  uint32_t codes = 0u;
  if (u < n_rec) {
    const uint8_t* rec = wire + static_cast<size_t>(u) * 400;
    b0 = __ldg(reinterpret_cast<const uint2*>(rec + off));
    b1 = __ldg(reinterpret_cast<const uint2*>(rec + off + 64));
    codes = __ldg(reinterpret_cast<const uint32_t*>(rec + 384 + t * 4));
  }
  while (u < n_rec) {
    const uint32_t un = u + du;  // < 2^32: both terms are below 2^31
    uint2 n0 = b0, n1 = b1;
    uint32_t nc = codes;
    if (un < n_rec) {
      const uint8_t* rec = wire + static_cast<size_t>(un) * 400;
      n0 = __ldg(reinterpret_cast<const uint2*>(rec + off));
      n1 = __ldg(reinterpret_cast<const uint2*>(rec + off + 64));
      nc = __ldg(reinterpret_cast<const uint32_t*>(rec + 384 + t * 4));
    }
    const int c0 = static_cast<int>((codes >> (8 * g0)) & 0xFFu);
    const int c1 = static_cast<int>((codes >> (8 * (g0 + 2))) & 0xFFu);
    const uint2 o0 = dequant4(b0.x, c0), o1 = dequant4(b0.y, c0);
    const uint2 o2 = dequant4(b1.x, c1), o3 = dequant4(b1.y, c1);
    __nv_bfloat16* dst = base + static_cast<int64_t>(row) * stride + head * kHeadDim + sub * 8;
    *reinterpret_cast<uint4*>(dst) = make_uint4(o0.x, o0.y, o1.x, o1.y);
    *reinterpret_cast<uint4*>(dst + 64) = make_uint4(o2.x, o2.y, o3.x, o3.y);
    u = un;
    b0 = n0;
    b1 = n1;
    codes = nc;
    head += du_head;
    row += du_row;
    if (head >= hl) {
      head -= hl;
      ++row;
    }
  }
}

template <int kFmt>
__global__ void __launch_bounds__(kWarps * 32) pack_out_kernel(
    const __nv_bfloat16* __restrict__ out, int64_t os, int64_t n_rows, int hl,
    uint8_t* __restrict__ wire) {
  constexpr int kU = 4;
  constexpr int kRec = kFmt == H3_WIRE_BF16 ? 256 : (kFmt == H3_WIRE_INT8 ? 144 : 128);
  const int lane = threadIdx.x & 31;
  const Units<kU> un(n_rows * hl, hl);
  uint2 in[kU] = {};
#pragma unroll
  for (int u = 0; u < kU; ++u)
    if (un.ok[u]) in[u] = ld8(out + un.r[u] * os + un.h[u] * kHeadDim + lane * 4);
  uint8_t* dst[kU];
#pragma unroll
  for (int u = 0; u < kU; ++u) dst[u] = wire + (un.r[u] * hl + un.h[u]) * kRec;
  if constexpr (kFmt == H3_WIRE_INT8) {
    float f[kU][4], amax[kU], s[kU], rs[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      unpack4(in[u], f[u]);
      amax[u] = group_amax(f[u]);
    }
    bool sat;
    const int code = group_scales<kU>(amax, s, rs, &sat);
    if (sat) {
#pragma unroll
      for (int u = 0; u < kU; ++u) clamp4(f[u], s[u]);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (un.ok[u]) *reinterpret_cast<uint32_t*>(dst[u] + lane * 4) = quant4(f[u], s[u], rs[u]);
    // lane (g, j) holds the code of record j, group g; lane u < kU clears
    // the pad bytes of record u
    const int j = lane & 7, g = lane >> 3;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (!un.ok[u]) break;
      if (j == u) dst[u][128 + g] = static_cast<uint8_t>(code);
      if (lane == u) {
        *reinterpret_cast<uint32_t*>(dst[u] + 132) = 0u;
        *reinterpret_cast<uint2*>(dst[u] + 136) = make_uint2(0u, 0u);
      }
    }
  } else {
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (!un.ok[u]) break;
      if (kFmt == H3_WIRE_BF16) {
        *reinterpret_cast<uint2*>(dst[u] + lane * 8) = in[u];
      } else {
        float f[4];
        unpack4(in[u], f);
        *reinterpret_cast<uint32_t*>(dst[u] + lane * 4) = fp8x4(f);
      }
    }
  }
}

template <int kFmt>
__global__ void __launch_bounds__(kWarps * 32) merge_heads_kernel(
    const uint8_t* __restrict__ wire, int64_t n_rows, int H, int n_src,
    __nv_bfloat16* __restrict__ out, int64_t os) {
  constexpr int kU = 4;
  constexpr int kRec = kFmt == H3_WIRE_BF16 ? 256 : (kFmt == H3_WIRE_INT8 ? 144 : 128);
  const int lane = threadIdx.x & 31;
  const Units<kU> un(n_rows * H, H);
  const int hl = H / n_src;
  uint2 in[kU];
  int codes[kU];
#pragma unroll
  for (int u = 0; u < kU; ++u) {
    if (un.ok[u]) {
      const int sidx = un.h[u] / hl, hloc = un.h[u] - sidx * hl;
      const uint8_t* src = wire + ((static_cast<int64_t>(sidx) * n_rows + un.r[u]) * hl + hloc) * kRec;
      if (kFmt == H3_WIRE_BF16) {
        in[u] = ld8(src + lane * 8);
      } else {
        in[u].x = __ldg(reinterpret_cast<const uint32_t*>(src + lane * 4));
        if (kFmt == H3_WIRE_INT8) codes[u] = src[128 + (lane >> 3)];
      }
    }
  }
#pragma unroll
  for (int u = 0; u < kU; ++u) {
    if (!un.ok[u]) break;
    uint2 o;
    if (kFmt == H3_WIRE_BF16) o = in[u];
    else if (kFmt == H3_WIRE_INT8) o = dequant4(in[u].x, codes[u]);
    else o = fp8x4_to_bf16(in[u].x);
    *reinterpret_cast<uint2*>(out + un.r[u] * os + un.h[u] * kHeadDim + lane * 4) = o;
  }
}

// Blocks for `units` (row, head) units at kU units per warp.
unsigned blocks_for(int64_t units, int ku) {
  return static_cast<unsigned>((units + kWarps * ku - 1) / (kWarps * ku));
}

}  // namespace

cudaError_t launch_pack_qkv(const WireQkvArgs& a, cudaStream_t s) {
  if (a.format == H3_WIRE_BF16) {
    pack_qkv_bf16_kernel<<<blocks_for(a.n_rows * a.n_heads, 2), kWarps * 32, 0, s>>>(
        a.q, a.qs, a.k, a.ks, a.v, a.vs, a.n_rows, a.n_heads, a.n_parts, a.wire);
    return cudaGetLastError();
  }
  // persistent: as many blocks as fit at once, or fewer for a small input
  // resident blocks of the whole device, looked up once per device (racing
  // threads store the same value)
  static std::atomic<int64_t> full_cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int64_t full = full_cache[dev].load();
  if (full == 0) {
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, pack_qkv_int8_kernel,
                                                      kInt8Warps * 32, 0);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    full = static_cast<int64_t>(sms) * (per_sm < 1 ? 1 : per_sm);
    full_cache[dev].store(full);
  }
  const int64_t units = a.n_rows * a.n_heads;
  const int64_t need = (units + kInt8Warps * 2 - 1) / (kInt8Warps * 2);
  const unsigned g = static_cast<unsigned>(need < full ? need : full);
  pack_qkv_int8_kernel<<<g, kInt8Warps * 32, 0, s>>>(a.q, a.qs, a.k, a.ks, a.v, a.vs, a.n_rows,
                                                     a.n_heads, a.n_parts, a.wire);
  return cudaGetLastError();
}

cudaError_t launch_unpack_qkv(const WireQkvArgs& a, cudaStream_t s) {
  if (a.format == H3_WIRE_BF16) {
    const unsigned g = blocks_for(a.n_rows * a.n_heads, 2);
    unpack_qkv_bf16_kernel<<<g, kWarps * 32, 0, s>>>(a.wire, a.n_rows, a.n_heads, a.qm, a.qs,
                                                     a.km, a.ks, a.vm, a.vs);
    return cudaGetLastError();
  }
  // Block-INT8: persistent, as many blocks as fit at once (or fewer for a
  // small input), rounded to a multiple of 3 blocks (see the kernel).
  static std::atomic<int64_t> full_cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int64_t full = full_cache[dev].load();
  if (full == 0) {
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, unpack_qkv_int8_kernel,
                                                      kUnpackWarps * 32, 0);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    full = static_cast<int64_t>(sms) * (per_sm < 1 ? 1 : per_sm) / 3 * 3;
    if (full < 3) full = 3;
    full_cache[dev].store(full);
  }
  const int64_t rows_of_tensors = 3 * a.n_rows * a.n_heads;      // q, k and v of every record
  int64_t need = (rows_of_tensors + kUnpackWarps * 4 - 1) / (kUnpackWarps * 4);
  need = (need + 2) / 3 * 3;
  const unsigned g = static_cast<unsigned>(need < full ? need : full);
  unpack_qkv_int8_kernel<<<g, kUnpackWarps * 32, 0, s>>>(
      a.wire, static_cast<uint32_t>(a.n_rows * a.n_heads), static_cast<uint32_t>(a.n_heads), a.qm,
      a.qs, a.km, a.ks, a.vm, a.vs);
  return cudaGetLastError();
}

cudaError_t launch_pack_out(const WireOutArgs& a, cudaStream_t s) {
  const unsigned g = blocks_for(a.n_rows * a.n_heads, 4);
  switch (a.format) {
    case H3_WIRE_BF16:
      pack_out_kernel<H3_WIRE_BF16><<<g, kWarps * 32, 0, s>>>(a.out, a.os, a.n_rows, a.n_heads, a.wire);
      break;
    case H3_WIRE_INT8:
      pack_out_kernel<H3_WIRE_INT8><<<g, kWarps * 32, 0, s>>>(a.out, a.os, a.n_rows, a.n_heads, a.wire);
      break;
    default:
      pack_out_kernel<H3_WIRE_FP8><<<g, kWarps * 32, 0, s>>>(a.out, a.os, a.n_rows, a.n_heads, a.wire);
  }
  return cudaGetLastError();
}

cudaError_t launch_merge_heads(const WireOutArgs& a, cudaStream_t s) {
  const unsigned g = blocks_for(a.n_rows * a.n_heads, 4);
  switch (a.format) {
    case H3_WIRE_BF16:
      merge_heads_kernel<H3_WIRE_BF16><<<g, kWarps * 32, 0, s>>>(a.wire, a.n_rows, a.n_heads,
                                                                 a.n_parts, a.outm, a.os);
      break;
    case H3_WIRE_INT8:
      merge_heads_kernel<H3_WIRE_INT8><<<g, kWarps * 32, 0, s>>>(a.wire, a.n_rows, a.n_heads,
                                                                 a.n_parts, a.outm, a.os);
      break;
    default:
      merge_heads_kernel<H3_WIRE_FP8><<<g, kWarps * 32, 0, s>>>(a.wire, a.n_rows, a.n_heads,
                                                                a.n_parts, a.outm, a.os);
  }
  return cudaGetLastError();
}

}  // namespace h3
