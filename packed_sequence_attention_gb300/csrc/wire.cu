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

#include "h3_internal.h"

namespace h3 {
namespace {

constexpr int kWarps = 8;

// value(c) = 2^((c >> 3) - 15) * (1 + (c & 7) / 8), built as fp32 bits
// (biased exponent (c >> 3) + 112, top 3 mantissa bits c & 7): exact.
__device__ __forceinline__ float ue5m3_value(int c) {
  return __uint_as_float((static_cast<uint32_t>((c >> 3) + 112) << 23) |
                         (static_cast<uint32_t>(c & 7) << 20));
}

// Smallest code c with 127 * value(c) >= amax.  A first guess from the
// exponent and leading mantissa bits of amax / 127 is corrected with the
// exact comparison (127 * value has at most 11 significant bits).
__device__ __forceinline__ int ue5m3_code(float amax) {
  if (!(amax > 127.0f * ue5m3_value(0))) return 0;
  const uint32_t b = __float_as_uint(amax * (1.0f / 127.0f));
  int e = static_cast<int>(b >> 23) - 112;
  int c = e * 8 + static_cast<int>((b >> 20) & 7u) + 1;  // round the mantissa up
  c = c < 0 ? 0 : (c > 255 ? 255 : c);
  while (c > 0 && 127.0f * ue5m3_value(c - 1) >= amax) --c;
  while (c < 255 && 127.0f * ue5m3_value(c) < amax) ++c;
  return c;
}

__device__ __forceinline__ void load4(const __nv_bfloat16* p, float* f) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
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

// Quantise this lane's 4 values of a 32-channel group: returns the 4 int8
// bytes; *code receives the group's scale code (same in all 8 lanes).
__device__ __forceinline__ uint32_t quant4(const float* f, int* code) {
  float a = fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3])));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
  const int c = ue5m3_code(a);
  *code = c;
  const float s = ue5m3_value(c);
  uint32_t out = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int q = __float2int_rn(__fdiv_rn(f[i], s));
    q = q > 127 ? 127 : (q < -127 ? -127 : q);
    out |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * i);
  }
  return out;
}

__device__ __forceinline__ void dequant4(uint32_t bytes, int code, float* f) {
  const float s = ue5m3_value(code);
#pragma unroll
  for (int i = 0; i < 4; ++i) f[i] = static_cast<float>(static_cast<int8_t>(bytes >> (8 * i))) * s;
}

// Gather the group codes of one tensor (lanes 0, 8, 16, 24 hold groups 0-3)
// into one little-endian word.
__device__ __forceinline__ uint32_t gather_codes(int code) {
  uint32_t w = 0;
#pragma unroll
  for (int g = 0; g < 4; ++g) w |= static_cast<uint32_t>(__shfl_sync(0xffffffffu, code, 8 * g)) << (8 * g);
  return w;
}

template <int kFmt>
__global__ void __launch_bounds__(kWarps * 32) pack_qkv_kernel(
    const __nv_bfloat16* __restrict__ q, int64_t qs, const __nv_bfloat16* __restrict__ k, int64_t ks,
    const __nv_bfloat16* __restrict__ v, int64_t vs, int64_t n_rows, int H, int n_dest,
    uint8_t* __restrict__ wire) {
  const int lane = threadIdx.x & 31;
  const int64_t unit = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (unit >= n_rows * H) return;
  const int64_t r = unit / H;
  const int h = static_cast<int>(unit - r * H);
  const int hl = H / n_dest, d = h / hl, hloc = h - d * hl;
  const int64_t rec = (static_cast<int64_t>(d) * n_rows + r) * hl + hloc;
  const __nv_bfloat16* src[3] = {q + r * qs, k + r * ks, v + r * vs};
  if (kFmt == H3_WIRE_BF16) {
    uint8_t* dst = wire + rec * 768;
#pragma unroll
    for (int t = 0; t < 3; ++t)
      *reinterpret_cast<uint2*>(dst + t * 256 + lane * 8) =
          *reinterpret_cast<const uint2*>(src[t] + h * kHeadDim + lane * 4);
  } else {
    uint8_t* dst = wire + rec * 400;
    uint32_t codes[3];
#pragma unroll
    for (int t = 0; t < 3; ++t) {
      float f[4];
      load4(src[t] + h * kHeadDim + lane * 4, f);
      int code;
      *reinterpret_cast<uint32_t*>(dst + t * 128 + lane * 4) = quant4(f, &code);
      codes[t] = gather_codes(code);
    }
    if (lane == 0) *reinterpret_cast<uint4*>(dst + 384) = make_uint4(codes[0], codes[1], codes[2], 0u);
  }
}

template <int kFmt>
__global__ void __launch_bounds__(kWarps * 32) unpack_qkv_kernel(
    const uint8_t* __restrict__ wire, int64_t n_rows, int hl, __nv_bfloat16* __restrict__ q,
    int64_t qs, __nv_bfloat16* __restrict__ k, int64_t ks, __nv_bfloat16* __restrict__ v,
    int64_t vs) {
  const int lane = threadIdx.x & 31;
  const int64_t unit = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (unit >= n_rows * hl) return;
  const int64_t r = unit / hl;
  const int h = static_cast<int>(unit - r * hl);
  __nv_bfloat16* dst[3] = {q + r * qs, k + r * ks, v + r * vs};
  if (kFmt == H3_WIRE_BF16) {
    const uint8_t* src = wire + unit * 768;
#pragma unroll
    for (int t = 0; t < 3; ++t)
      *reinterpret_cast<uint2*>(dst[t] + h * kHeadDim + lane * 4) =
          *reinterpret_cast<const uint2*>(src + t * 256 + lane * 8);
  } else {
    const uint8_t* src = wire + unit * 400;
    const uint4 cw = *reinterpret_cast<const uint4*>(src + 384);
    const uint32_t cws[3] = {cw.x, cw.y, cw.z};
#pragma unroll
    for (int t = 0; t < 3; ++t) {
      float f[4];
      dequant4(*reinterpret_cast<const uint32_t*>(src + t * 128 + lane * 4),
               (cws[t] >> (8 * (lane >> 3))) & 0xFF, f);
      *reinterpret_cast<uint2*>(dst[t] + h * kHeadDim + lane * 4) = pack4_bf16(f);
    }
  }
}

template <int kFmt>
__global__ void __launch_bounds__(kWarps * 32) pack_out_kernel(
    const __nv_bfloat16* __restrict__ out, int64_t os, int64_t n_rows, int hl,
    uint8_t* __restrict__ wire) {
  const int lane = threadIdx.x & 31;
  const int64_t unit = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (unit >= n_rows * hl) return;
  const int64_t r = unit / hl;
  const int h = static_cast<int>(unit - r * hl);
  const __nv_bfloat16* src = out + r * os + h * kHeadDim + lane * 4;
  if (kFmt == H3_WIRE_BF16) {
    *reinterpret_cast<uint2*>(wire + unit * 256 + lane * 8) = *reinterpret_cast<const uint2*>(src);
  } else if (kFmt == H3_WIRE_INT8) {
    float f[4];
    load4(src, f);
    int code;
    uint8_t* dst = wire + unit * 144;
    *reinterpret_cast<uint32_t*>(dst + lane * 4) = quant4(f, &code);
    const uint32_t c = gather_codes(code);
    if (lane == 0) *reinterpret_cast<uint4*>(dst + 128) = make_uint4(c, 0u, 0u, 0u);
  } else {
    float f[4];
    load4(src, f);
    uint16_t lo, hi;
    // cvt.rn.satfinite.e4m3x2.f32 d, a, b: a -> upper byte, b -> lower byte
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(f[1]), "f"(f[0]));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(f[3]), "f"(f[2]));
    *reinterpret_cast<uint32_t*>(wire + unit * 128 + lane * 4) =
        static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
}

template <int kFmt>
__global__ void __launch_bounds__(kWarps * 32) merge_heads_kernel(
    const uint8_t* __restrict__ wire, int64_t n_rows, int H, int n_src,
    __nv_bfloat16* __restrict__ out, int64_t os) {
  const int lane = threadIdx.x & 31;
  const int64_t unit = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (unit >= n_rows * H) return;
  const int64_t r = unit / H;
  const int h = static_cast<int>(unit - r * H);
  const int hl = H / n_src, sidx = h / hl, hloc = h - sidx * hl;
  const int64_t rec = (static_cast<int64_t>(sidx) * n_rows + r) * hl + hloc;
  __nv_bfloat16* dst = out + r * os + h * kHeadDim + lane * 4;
  if (kFmt == H3_WIRE_BF16) {
    *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(wire + rec * 256 + lane * 8);
  } else if (kFmt == H3_WIRE_INT8) {
    const uint8_t* src = wire + rec * 144;
    float f[4];
    dequant4(*reinterpret_cast<const uint32_t*>(src + lane * 4),
             src[128 + (lane >> 3)], f);
    *reinterpret_cast<uint2*>(dst) = pack4_bf16(f);
  } else {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(wire + rec * 128 + lane * 4);
    uint32_t h01, h23;  // e4m3x2 -> f16x2 is exact; f16 -> fp32 -> bf16 is exact too
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h01) : "h"(static_cast<uint16_t>(w & 0xFFFF)));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h23) : "h"(static_cast<uint16_t>(w >> 16)));
    const __half2 a = *reinterpret_cast<const __half2*>(&h01);
    const __half2 b = *reinterpret_cast<const __half2*>(&h23);
    float f[4] = {__low2float(a), __high2float(a), __low2float(b), __high2float(b)};
    *reinterpret_cast<uint2*>(dst) = pack4_bf16(f);
  }
}

unsigned blocks_for(int64_t units) { return static_cast<unsigned>((units + kWarps - 1) / kWarps); }

}  // namespace

cudaError_t launch_pack_qkv(const WireQkvArgs& a, cudaStream_t s) {
  const unsigned g = blocks_for(a.n_rows * a.n_heads);
  if (a.format == H3_WIRE_BF16)
    pack_qkv_kernel<H3_WIRE_BF16><<<g, kWarps * 32, 0, s>>>(a.q, a.qs, a.k, a.ks, a.v, a.vs,
                                                            a.n_rows, a.n_heads, a.n_parts, a.wire);
  else
    pack_qkv_kernel<H3_WIRE_INT8><<<g, kWarps * 32, 0, s>>>(a.q, a.qs, a.k, a.ks, a.v, a.vs,
                                                            a.n_rows, a.n_heads, a.n_parts, a.wire);
  return cudaGetLastError();
}

cudaError_t launch_unpack_qkv(const WireQkvArgs& a, cudaStream_t s) {
  const unsigned g = blocks_for(a.n_rows * a.n_heads);
  if (a.format == H3_WIRE_BF16)
    unpack_qkv_kernel<H3_WIRE_BF16><<<g, kWarps * 32, 0, s>>>(a.wire, a.n_rows, a.n_heads, a.qm,
                                                              a.qs, a.km, a.ks, a.vm, a.vs);
  else
    unpack_qkv_kernel<H3_WIRE_INT8><<<g, kWarps * 32, 0, s>>>(a.wire, a.n_rows, a.n_heads, a.qm,
                                                              a.qs, a.km, a.ks, a.vm, a.vs);
  return cudaGetLastError();
}

cudaError_t launch_pack_out(const WireOutArgs& a, cudaStream_t s) {
  const unsigned g = blocks_for(a.n_rows * a.n_heads);
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
  const unsigned g = blocks_for(a.n_rows * a.n_heads);
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
