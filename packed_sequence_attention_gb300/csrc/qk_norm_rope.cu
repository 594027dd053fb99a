// Fused Q/K RMSNorm + axial 3-D RoPE, in place, one pass over HBM.
//
// "QK normalization with partial RoPE" is operator group 2 of Sol-H3
// (arXiv 2609.35110), section 3.5 "Kernel Fusion"; the vLLM-Omni blog
// ("MiniMax H3 on vLLM-Omni"), section 3.2, fuses the same Q/K RMSNorm and
// RoPE.  The point of the fusion is to read each wide activation once and
// write it once, so the kernel is built around keeping HBM busy:
//
// * Persistent CTAs walk items g = blockIdx.x + i * gridDim.x: items
//   0 .. n-1 are the n valid rows of Q, items n .. 2n-1 those of K, each
//   n_heads * 256 contiguous bytes.  All CTAs thus stream through Q, then
//   through K, one address window at a time (interleaving Q and K rows put
//   two windows in flight and was ~1 % slower).  Valid rows are numbered across the packed sequences of the
//   launch (the valid rows of each, in order), so several sequences share one
//   persistent grid and pay one tail.  The streaming warp holds the sequence
//   table (at most 16 entries) in its lanes' registers, maps each item's valid
//   row to its buffer row with a ballot and two shuffles, and hands that row
//   to the compute warps in the item's stage.  (Reading the table from the
//   kernel parameters with a run-time index on every item cost 4 % on the
//   58,758-row workload.)
// * Warp roles.  One streaming warp copies items into a 3-stage shared-memory
//   ring with 1-D bulk async copies (cp.async.bulk, completion on a "full"
//   mbarrier) and fills each stage's (cos, sin) table for the item's
//   position; four compute warps consume the stages and give each one back
//   through an "empty" mbarrier.  No block-wide barrier is left in the loop,
//   so a compute warp never waits for a slower one.  On the 58,758-row
//   workload this runs at 401 us against 412 us for the same arithmetic with
//   all threads computing and a block barrier per item; 2 or 4 stages, or
//   7 CTAs per SM, were no faster.
// * Per item, the streaming warp computes the (cos, sin) of the 64 channel
//   pairs once (two pairs per lane, positions fetched one item ahead); every
//   head of the item reuses them.
// * A head-vector (128 channels) is handled by 8 lanes, each owning channel
//   chunks [8s, 8s+8) and [64+8s, 64+8s+8); the sum of squares is reduced with
//   three xor-shuffles; results are rounded once to bf16 (RNE) and stored
//   straight to global memory with 16-byte streaming stores.
// * The squares and the products x * w are taken straight from the bf16x2
//   words with the mixed-precision fma (bf16 x bf16 + f32), so neither the
//   input nor the weight is unpacked; each output is ((x * w) * r) rotated,
//   r = 1 / rms.  Behind the attention, on a power-capped SM clock, this took
//   the 58,758-row launch from 427-430 us to 408-412 us.
// * Every mbarrier wait is bounded; a wait that gives up sets a bit in the
//   device status word and the role stops (the streaming warp first lets its
//   copies in flight land).
#include <cmath>
#include <mutex>

#include "h3_internal.h"
#include "ptx.cuh"

namespace h3 {
namespace {

using namespace ptx;

constexpr int kComputeWarps = 4;
constexpr int kThreads = 32 * (kComputeWarps + 1);
constexpr int kMaxStages = 4;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr size_t kMaxSmemPerBlock = 227 * 1024;  // opt-in dynamic shared memory per CTA

struct NormRopeParams {
  __nv_bfloat16* x[2];
  int64_t stride[2];
  const __nv_bfloat16* d[2];  // LoRA branch outputs (delta) of Q and K, or null
  int64_t dstride[2];
  const __nv_bfloat16* w[2];
  const int32_t* pos;
  uint32_t* status;
  int64_t n_rows;  // valid rows over all segments
  int n_heads;
  int n_stages;
  float eps;
  int n_seg;
  int32_t seg_cum[kPrologueMaxSegments + 1];  // valid rows before segment b; [n_seg] = n_rows
  int64_t seg_row0[kPrologueMaxSegments];     // buffer row of segment b's first valid row
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

// d = lo(a) * lo(b) + c and d = hi(a) * hi(b) + c for bf16x2 words a, b: the
// mixed-precision fma (bf16 multiplicands, f32 addend and result, one
// rounding; PTX ISA 8.6, sm_100 and later).  The input is used as it sits in
// shared memory, with no unpacking to f32 first; the product of two bf16
// values is exact in f32, so with c = -0 the result is that exact product.
__device__ __forceinline__ float fma_lo(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{ .reg .b16 al, ah, bl, bh;\n mov.b32 {al, ah}, %1;\n mov.b32 {bl, bh}, %2;\n"
      " fma.rn.f32.bf16 %0, al, bl, %3; }" : "=f"(d) : "r"(a), "r"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fma_hi(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{ .reg .b16 al, ah, bl, bh;\n mov.b32 {al, ah}, %1;\n mov.b32 {bl, bh}, %2;\n"
      " fma.rn.f32.bf16 %0, ah, bh, %3; }" : "=f"(d) : "r"(a), "r"(b), "f"(c));
  return d;
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// (cos, sin) table layout: a compute lane with chunk index sub reads its 8
// pairs as four 16-byte reads k = 0..3 at [k][sub], so the 8 lanes of a
// quarter-warp read 128 contiguous bytes (no bank conflict).  Pair p sits in
// read k = (p >> 5) * 2 + ((p & 3) >> 1) of lane sub = (p & 31) >> 2, entry p & 1.
__device__ __forceinline__ int tab_slot(int p) {
  return (((p >> 5) * 2 + ((p & 3) >> 1)) * 16) + ((p & 31) >> 2) * 2 + (p & 1);
}

// kLora: the item is base + delta; the sum is rounded to bf16 first, as the
// separate branches would store it (Sol-H3 section 3.5, precision-preserving
// LoRA fusion), then normalised and rotated.
//
// Warp roles: warps 0..3 compute, warp 4 streams.  The streaming warp waits
// until every compute warp has released a stage, copies the next row into
// it and fills the stage's (cos, sin) table; compute warps never wait for
// one another.
template <bool kLora>
__global__ void __launch_bounds__(kThreads) qk_norm_rope_kernel(const __grid_constant__ NormRopeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int H = p.n_heads;
  const uint32_t row_bytes = static_cast<uint32_t>(H) * kHeadDim * 2;
  const uint32_t stage_bytes = (kLora ? 2 : 1) * row_bytes;  // one tensor row (+ its delta row)
  const int NST = p.n_stages;
  const uint32_t sbase = smem_u32(smem);
  float2* tab = reinterpret_cast<float2*>(smem + NST * stage_bytes);  // [NST][64] (cos, sin)
  const uint32_t full_bar = sbase + NST * stage_bytes + NST * 64 * 8;  // mbarriers [NST]
  const uint32_t empty_bar = full_bar + 8 * kMaxStages;                // mbarriers [NST]
  // Buffer row of the item in each stage, written by the streaming warp
  // before it arrives on the stage's full barrier.
  int64_t* stage_row = reinterpret_cast<int64_t*>(smem + NST * stage_bytes + NST * 64 * 8 +
                                                  16 * kMaxStages);

  const int64_t first = blockIdx.x;
  const int64_t step = gridDim.x;
  const int64_t n_items = 2 * p.n_rows;  // item g: Q row g, or K row g - n_rows
  const int64_t n_mine = first < n_items ? (n_items - 1 - first) / step + 1 : 0;

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(full_bar + 8 * s, 1 + 32);            // the copy's arrive + one per table lane
      mbar_init(empty_bar + 8 * s, kComputeWarps);  // one per compute warp
    }
    fence_mbar_init();
  }
  __syncthreads();

  // Bounded wait; false = gave up.
  auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
      if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    return true;
  };

  if (warp == kComputeWarps) {
    // ------------------------------------------------------------ streaming
    const int ax0 = p.axis[lane], ax1 = p.axis[lane + 32];
    const float f0 = p.inv_freq[lane], f1 = p.inv_freq[lane + 32];
    // The segment table in registers: lane b < n_seg holds segment b's
    // cumulative valid count and first buffer row.  The segment of valid row
    // r is the last one whose count is <= r (empty segments share their
    // count with the next one, which comes later): one ballot, two shuffles.
    const int32_t cum_l = lane < p.n_seg ? p.seg_cum[lane] : INT32_MAX;
    const int64_t row0_l = lane < p.n_seg ? p.seg_row0[lane] : 0;
    auto row_of = [&](int64_t i) -> int64_t {
      const int64_t g = first + i * step;
      const int64_t r = g >= p.n_rows ? g - p.n_rows : g;  // valid row of the item
      const int b = __popc(__ballot_sync(0xffffffffu, cum_l <= r)) - 1;
      return __shfl_sync(0xffffffffu, row0_l, b) + (r - __shfl_sync(0xffffffffu, cum_l, b));
    };
    auto pos_at = [&](int64_t row, int ax) -> int32_t {
      return ax < 0 ? 0 : __ldg(p.pos + row * 3 + ax);
    };
    // Buffer row of the next item and its positions, fetched one item ahead.
    int64_t row_next = n_mine > 0 ? row_of(0) : 0;
    int32_t pn0 = n_mine > 0 ? pos_at(row_next, ax0) : 0;
    int32_t pn1 = n_mine > 0 ? pos_at(row_next, ax1) : 0;
    int64_t i = 0;
    bool ok = true;
    for (; i < n_mine; ++i) {
      const int s = static_cast<int>(i % NST);
      if (i >= NST) {
        const uint32_t par = static_cast<uint32_t>((i / NST - 1) & 1);
        bool w = true;
        if (lane == 0) w = wait(empty_bar + 8 * s, par);
        if (!__shfl_sync(0xffffffffu, w ? 1 : 0, 0)) {
          ok = false;
          break;
        }
      }
      const uint32_t bar = full_bar + 8 * s;
      const int64_t row = row_next;
      if (lane == 0) {
        stage_row[s] = row;
        const int tt = (first + i * step) >= p.n_rows ? 1 : 0;
        mbar_arrive_expect_tx(bar, stage_bytes);
        bulk_load(sbase + s * stage_bytes, p.x[tt] + row * p.stride[tt], row_bytes, bar);
        if (kLora)
          bulk_load(sbase + s * stage_bytes + row_bytes, p.d[tt] + row * p.dstride[tt], row_bytes, bar);
      }
      const int32_t q0 = pn0, q1 = pn1;
      if (i + 1 < n_mine) {  // next row's positions, in flight meanwhile
        row_next = row_of(i + 1);
        pn0 = pos_at(row_next, ax0);
        pn1 = pos_at(row_next, ax1);
      }
      float c0 = 1.0f, s0 = 0.0f, c1 = 1.0f, s1 = 0.0f;
      if (ax0 >= 0) sincosf(static_cast<float>(q0) * f0, &s0, &c0);
      if (ax1 >= 0) sincosf(static_cast<float>(q1) * f1, &s1, &c1);
      tab[s * 64 + tab_slot(lane)] = make_float2(c0, s0);
      tab[s * 64 + tab_slot(lane + 32)] = make_float2(c1, s1);
      mbar_arrive(bar);
    }
    if (lane == 0) {
      if (!ok) atomicOr(p.status, H3_STATUS_TIMEOUT_PROLOGUE);
      // Let every copy this CTA started land before it exits (bounded): the
      // last NST issued rows.
      for (int64_t j = (i > NST ? i - NST : 0); j < i; ++j)
        wait(full_bar + 8 * (j % NST), static_cast<uint32_t>((j / NST) & 1));
    }
    return;
  }

  // -------------------------------------------------------------- compute
  const int sub = lane & 7;                 // channel chunk of this lane
  const int slot = warp * 4 + (lane >> 3);  // which head-unit of a pass
  constexpr int kSlots = kComputeWarps * 4;
  const int n_units = H;
  for (int64_t i = 0; i < n_mine; ++i) {
    const int s = static_cast<int>(i % NST);
    const uint32_t parity = static_cast<uint32_t>((i / NST) & 1);
    const int tsel = (first + i * step) >= p.n_rows ? 1 : 0;
    // Wait for this row's bytes and table (bounded; uniform across the warp).
    bool ok = mbar_try_wait(full_bar + 8 * s, parity);
    if (!__all_sync(0xffffffffu, ok)) {
      ok = wait(full_bar + 8 * s, parity);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) atomicOr(p.status, H3_STATUS_TIMEOUT_PROLOGUE);
        return;
      }
    }
    const int64_t row = stage_row[s];
    float cs[8], sn[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float2 v = tab[s * 64 + (j >> 1) * 16 + sub * 2 + (j & 1)];
      cs[j] = v.x;
      sn[j] = v.y;
    }
    const uint32_t stage = sbase + s * stage_bytes;
    // The slots of the last, partial pass (n_heads % 16 of them) move to
    // other warps from one item to the next, so that every warp does the
    // same work on average: a stage is released only when its slowest warp
    // is done.
    const int rslot = (slot + 4 * static_cast<int>(i & 3)) & (kSlots - 1);
    for (int u0 = 0; u0 < n_units; u0 += kSlots) {
      const int u = u0 + rslot;
      const bool live = u < n_units;
      const int t = tsel;
      const int h = live ? u : 0;
      const uint32_t src = stage + h * (kHeadDim * 2) + sub * 16;
      const uint4* wsrc = reinterpret_cast<const uint4*>(p.w[t] + h * kHeadDim);
      const uint4 wa = __ldg(wsrc + sub), wb = __ldg(wsrc + 8 + sub);
      uint32_t xw[8];
      if (live) {
        const uint4 a = lds128(src), b = lds128(src + 128);
        xw[0] = a.x; xw[1] = a.y; xw[2] = a.z; xw[3] = a.w;
        xw[4] = b.x; xw[5] = b.y; xw[6] = b.z; xw[7] = b.w;
        if (kLora) {
          float x[16], dx[16];
          unpack8(a, x);
          unpack8(b, x + 8);
          unpack8(lds128(src + row_bytes), dx);
          unpack8(lds128(src + row_bytes + 128), dx + 8);
#pragma unroll
          for (int c = 0; c < 16; c += 2)  // base + delta, rounded to bf16 (RNE)
            xw[c / 2] = pack_bf16x2(x[c] + dx[c], x[c + 1] + dx[c + 1]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) xw[j] = 0u;
      }
      float ss0 = 0.f, ss1 = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        ss0 = fma_lo(xw[j], xw[j], ss0);
        ss1 = fma_hi(xw[j], xw[j], ss1);
      }
      float ss = ss0 + ss1;
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      ss += __shfl_xor_sync(0xffffffffu, ss, 2);
      ss += __shfl_xor_sync(0xffffffffu, ss, 4);
      if (!live) continue;  // uniform across the 8 lanes of a unit
      const float r = rsqrtf(ss * (1.0f / kHeadDim) + p.eps);
      const uint32_t ww[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
      uint32_t o[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float y0 = fma_lo(xw[j], ww[j], -0.0f) * r;
        const float y1 = fma_hi(xw[j], ww[j], -0.0f) * r;
        o[j] = pack_bf16x2(y0 * cs[j] - y1 * sn[j], y0 * sn[j] + y1 * cs[j]);
      }
      uint4* dst = reinterpret_cast<uint4*>(p.x[t] + row * p.stride[t] + h * kHeadDim);
      __stcs(dst + sub, make_uint4(o[0], o[1], o[2], o[3]));
      __stcs(dst + 8 + sub, make_uint4(o[4], o[5], o[6], o[7]));
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_bar + 8 * s);  // this warp is done with stage s
  }
}

}  // namespace

int prologue_max_heads(bool lora) {
  // At least two stages of one tensor row (256 B per head; twice that with
  // the LoRA delta row) plus two cos/sin tables and the barriers must fit in
  // 227 KB of shared memory: 452 heads (225 with LoRA); keep 448 (220).
  return lora ? 220 : 448;
}

cudaError_t launch_qk_norm_rope(const NormRopeArgs& a, cudaStream_t stream) {
  if (a.n_seg < 1 || a.n_seg > kPrologueMaxSegments) return cudaErrorInvalidValue;
  NormRopeParams p{};
  p.x[0] = a.q;
  p.x[1] = a.k;
  p.stride[0] = a.q_stride;
  p.stride[1] = a.k_stride;
  p.w[0] = a.wq;
  p.w[1] = a.wk;
  p.pos = a.pos;
  p.n_heads = a.n_heads;
  p.eps = a.eps;
  p.status = status_word_device_ptr();
  if (p.status == nullptr) return cudaErrorInvalidSymbol;
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
  // Ring depth: three stages where they fit in shared memory, else two
  // (very wide rows).
  const bool lora = a.dq != nullptr;
  p.d[0] = a.dq;
  p.d[1] = a.dk;
  p.dstride[0] = a.dq_stride;
  p.dstride[1] = a.dk_stride;
  const size_t stage_bytes = (lora ? 2ull : 1ull) * a.n_heads * kHeadDim * 2;
  auto smem_for = [&](int nst) { return nst * (stage_bytes + 64 * 8) + 3 * kMaxStages * 8; };
  const int nst = smem_for(3) <= kMaxSmemPerBlock ? 3 : 2;
  p.n_stages = nst;
  const size_t smem = smem_for(nst);
  auto kernel = lora ? qk_norm_rope_kernel<true> : qk_norm_rope_kernel<false>;
  // The attribute only ever grows, so a launch never runs under a smaller
  // limit that another thread set after it checked.
  static std::mutex attr_mu;
  static size_t attr_smem[2][64];  // guarded by attr_mu
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(attr_mu);
    if (attr_smem[lora][dev] < smem) {
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      attr_smem[lora][dev] = smem;
    }
  }
  int per_sm = 0, sms = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  // Valid rows are numbered across the segments; segments with no row are
  // stepped over by the kernel.  The caller has checked that the total fits
  // in int32 and that n_seg <= kPrologueMaxSegments.
  int64_t total = 0;
  for (int b = 0; b < a.n_seg; ++b) {
    p.seg_cum[b] = static_cast<int32_t>(total);
    p.seg_row0[b] = a.seg_row0[b];
    total += a.seg_rows[b];
  }
  p.seg_cum[a.n_seg] = static_cast<int32_t>(total);
  p.n_seg = a.n_seg;
  p.n_rows = total;
  if (total == 0) return cudaSuccess;
  int64_t grid = static_cast<int64_t>(sms) * per_sm;
  if (grid > 2 * total) grid = 2 * total;
  kernel<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace h3
