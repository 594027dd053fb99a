// Packed-sequence attention, sm_103a: TMA + tcgen05/TMEM flash attention.
//
// Computes out = softmax(Q K^T * scale) V per segment (a packed sequence
// with a valid length, vLLM-Omni blog "MiniMax H3 on vLLM-Omni" section 3.1,
// or a query group over its own KV range, SolarWM-H3 Realtime blog stage 2)
// and per head, exactly, with the online-softmax recurrence of the
// FlashAttention line of work: running row max m, running sum l, and a
// rescale of the partial output whenever m moves.
//
// One CTA = one (segment, head, pair of 128-row query tiles).  Roles:
//   warps 0-3  softmax for query tile 0 (thread i owns row i = TMEM lane i)
//   warps 4-7  softmax for query tile 1
//   warp  8    TMA producer: Q tiles once, then K/V tiles into a 2-stage ring
//   warp  9    TMEM owner and single-thread tcgen05.mma issuer
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512);
// P_t (bf16 pairs) overwrites the first 64 columns of S_t and feeds the
// P.V product straight from TMEM.  Per KV tile j the issuer runs, in order,
//   PV0(j)  QK0(j+1)  PV1(j)  QK1(j+1)
// so that the softmax of one tile overlaps the MMAs of the other.  All
// tcgen05.mma ops of the CTA execute in issue order, and a commit tracks
// every earlier op of the issuing thread: S_t(j+1) complete therefore also
// means PV_t(j) complete, which is what lets softmax rescale O_t in place.
//
// Masking: per-segment tensor maps have the segment's VALID row count as
// their outer extent, so TMA zero-fills rows past it and never reads
// padded rows (which may hold NaN/Inf); score columns past the valid
// length are set to -inf with a select; query tiles wholly past it are
// never scheduled.  Output rows past the valid length are written as 0.
//
// Every wait is bounded (wall-clock limit from %globaltimer).  A wait that
// gives up sets a bit in the device status word and an abort epoch; the
// CTA then drains its own in-flight copies and MMAs, frees TMEM and exits,
// and other CTAs of the same launch stop at their next wait.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <vector>

#include "h3_internal.h"
#include "ptx.cuh"

namespace h3 {

__device__ uint32_t g_status;       // OR of H3_STATUS_* bits
__device__ uint32_t g_abort_epoch;  // epoch of the last launch that gave up

namespace {

using namespace ptx;

constexpr int kBM = 128;  // query rows per tile (MMA M)
constexpr int kBN = 128;  // key rows per tile (MMA N of Q.K^T, K of P.V)
constexpr int kNS = 2;    // K/V ring stages
constexpr int kThreads = 320;
constexpr uint32_t kTileBytes = kBM * kHeadDim * 2;  // 32 KB
constexpr uint32_t kHalfBytes = kTileBytes / 2;      // 64 channels x 128 rows
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + 2 * kTileBytes;
constexpr uint32_t kOffV = kOffK + kNS * kTileBytes;
constexpr uint32_t kOffBar = kOffV + kNS * kTileBytes;
enum {
  BAR_Q = 0,
  // K and V rings have their own barriers: a K stage is released as soon as
  // the last Q.K^T reading it completes, an iteration before its V stage.
  BAR_KFULL = 1,
  BAR_VFULL = BAR_KFULL + kNS,
  BAR_KEMPTY = BAR_VFULL + kNS,
  BAR_VEMPTY = BAR_KEMPTY + kNS,
  BAR_SFULL = BAR_VEMPTY + kNS,
  BAR_PFULL = BAR_SFULL + 2,
  BAR_OFINAL = BAR_PFULL + 2,
  BAR_DRAIN = BAR_OFINAL + 2,
  NUM_BARS = BAR_DRAIN + 1
};
constexpr uint32_t kOffTmemSlot = kOffBar + NUM_BARS * 8;
constexpr uint32_t kOffAbort = kOffTmemSlot + 4;
constexpr uint32_t kOffQIssued = kOffAbort + 4;  // 1 once the Q copy is in flight
// Block-sparse mode only: int [4] = union length, steps both tiles keep,
// alternating pairs, the tile of the remaining steps; then the lists.
constexpr uint32_t kOffList = kOffQIssued + 12;
constexpr uint32_t kListWords = kMaxSparseBlocks / 32;
constexpr uint32_t kOffListBits = kOffList + 16;                   // [2][kListWords] u32
constexpr uint32_t kOffListTiles = kOffListBits + 2 * kListWords * 4;  // [kMaxSparseBlocks] u16
constexpr uint32_t kOffListSel = kOffListTiles + kMaxSparseBlocks * 2;  // [kMaxSparseBlocks] u8
constexpr uint32_t kSmemUsed = kOffList;
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;  // slack for 1024-byte alignment
constexpr uint32_t kSmemBytesSparse = kOffListSel + kMaxSparseBlocks + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 256;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale only if max grows by > 2^8
constexpr uint64_t kWaitLimitNs = 2000000000ull;

constexpr uint32_t kIdescQK = idesc_bf16_f32(kBM, kBN, false, false);      // K-major Q, K
constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, kHeadDim, false, true);  // V is MN-major

struct Seg {
  int32_t q_row0;   // first row of the segment in q / out
  int32_t nq;       // valid query rows (> 0)
  int32_t nkv;      // key rows of the first KV view (k / v)
  int32_t nkv2;     // key rows of the second KV view (k_cache / v_cache), may be 0
  int32_t n_pairs;  // ceil(nq / 256)
  int32_t cta0;     // first CTA of the segment
};

struct __align__(128) AttnParams {
  CUtensorMap tm_q[H3_MAX_SEGMENTS];
  CUtensorMap tm_k[H3_MAX_SEGMENTS];   // first KV view
  CUtensorMap tm_v[H3_MAX_SEGMENTS];
  CUtensorMap tm_k2[H3_MAX_SEGMENTS];  // second KV view (cached keys), if any
  CUtensorMap tm_v2[H3_MAX_SEGMENTS];
  Seg seg[H3_MAX_SEGMENTS];  // schedule order (longest KV first)
  int32_t zero_row0[H3_MAX_SEGMENTS];
  int32_t zero_rows[H3_MAX_SEGMENTS];
  __nv_bfloat16* out;
  int64_t out_stride;
  int64_t zero_chunks;  // 16-byte chunks to clear: sum(zero_rows) * n_heads * 16
  int32_t n_seg, n_zero, n_heads, n_compute_ctas;
  float scale_log2;
  uint32_t epoch;
  int32_t fault;  // test hook: 1 = the producer never loads K/V tile 1
  // block-sparse mode: per (head, query block) ordered lists of kept KV blocks
  const int32_t* sp_lists;   // [H, nqb, nkb]
  const int32_t* sp_counts;  // [H, nqb]
  int32_t sp_nqb, sp_nkb;
  int32_t sp_tail;           // valid rows of the last KV block
  int32_t sp_heavy;          // leading query-tile pairs of every head scheduled first
};

struct WaitCtx {
  volatile uint32_t* abort_smem;
  uint32_t epoch;
};

__device__ __noinline__ void give_up(const WaitCtx& w, uint32_t bit) {
  *w.abort_smem = 1u;
  atomicOr(&g_status, bit);
  atomicExch(&g_abort_epoch, w.epoch);
}

__device__ __forceinline__ bool should_stop(const WaitCtx& w) {
  if (*w.abort_smem != 0u) return true;
  if (*reinterpret_cast<volatile uint32_t*>(&g_abort_epoch) == w.epoch) {
    atomicOr(&g_status, H3_STATUS_ABORTED);
    return true;
  }
  return false;
}

// Single-thread bounded wait.  False = gave up (or another role did).  Kept
// inline: as a call, the register saves and reloads around it cost the
// issuing thread more than the spin itself.
__device__ __forceinline__ bool wait1(uint32_t bar, uint32_t parity, const WaitCtx& w, uint32_t bit) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0u) {
      if (should_stop(w)) {
        *w.abort_smem = 1u;
        return false;
      }
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        give_up(w, bit);
        return false;
      }
    }
  }
}

// Two bounded waits whose first try_waits are issued back to back: two
// barriers that have already completed cost one round trip, not two.
__device__ __forceinline__ bool wait2(uint32_t bar_a, uint32_t par_a, uint32_t bar_b, uint32_t par_b,
                                      const WaitCtx& w, uint32_t bit) {
  const bool a = mbar_try_wait(bar_a, par_a);
  const bool b = mbar_try_wait(bar_b, par_b);
  if (a && b) return true;
  if (!a && !wait1(bar_a, par_a, w, bit)) return false;
  return b || wait1(bar_b, par_b, w, bit);
}

// Bounded wait that only ends on completion or time (no early stop): used to
// drain operations already in flight before the CTA exits.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

// Warp-wide bounded wait; the decision is uniform across the warp.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, const WaitCtx& w, uint32_t bit) {
  const int lane = threadIdx.x & 31;
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    const bool ok = mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, ok)) return true;
    if ((it & 63u) == 63u) {
      int stop = 0;
      if (lane == 0) {
        if (t0 == 0) t0 = globaltimer_ns();
        if (should_stop(w)) {
          stop = 1;
        } else if (globaltimer_ns() - t0 > kWaitLimitNs) {
          give_up(w, bit);
          stop = 1;
        }
      }
      if (__shfl_sync(0xffffffffu, stop, 0)) {
        *w.abort_smem = 1u;
        return false;
      }
    }
  }
}

__device__ __forceinline__ void zero_fill(const AttnParams& p) {
  const int64_t n = p.zero_chunks;
  const int64_t per_row = static_cast<int64_t>(p.n_heads) * 16;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * 256;
  for (int64_t c = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x; c < n; c += stride) {
    int64_t rem = c;
    int r = 0;
    while (r + 1 < p.n_zero && rem >= static_cast<int64_t>(p.zero_rows[r]) * per_row) {
      rem -= static_cast<int64_t>(p.zero_rows[r]) * per_row;
      ++r;
    }
    const int64_t row = p.zero_row0[r] + rem / per_row;
    const int64_t col = (rem % per_row) * 8;  // element offset within the row's H*128
    *reinterpret_cast<uint4*>(p.out + row * p.out_stride + col) = make_uint4(0, 0, 0, 0);
  }
}

// kSparse: Sol-Attn block-sparse mode -- one packed sequence, each query
// tile attends to the KV tiles its block list keeps.  A CTA walks the union
// of its two tiles' lists (both-kept blocks, then the tiles' own blocks
// alternating, then the longer list's rest); a tile takes part only in the
// steps its list keeps.
template <bool kSparse>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (p.zero_chunks > 0 && threadIdx.x < 256) zero_fill(p);
  if (static_cast<int>(blockIdx.x) >= p.n_compute_ctas) return;

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * static_cast<uint32_t>(i); };
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gbase + kOffAbort);
  const WaitCtx wctx{abort_flag, p.epoch};

  // ---- work item
  int si = 0;
  while (si + 1 < p.n_seg && static_cast<int>(blockIdx.x) >= p.seg[si + 1].cta0) ++si;
  const Seg sg = p.seg[si];
  const int local = static_cast<int>(blockIdx.x) - sg.cta0;
  int head, pair;
  if (kSparse && local < p.sp_heavy * p.n_heads) {
    // Block-sparse: the tiles of the dense prefix queries (every KV block
    // kept) are several times longer than the rest; they go first, head by
    // head, so that none of them starts in the last waves.
    head = local / p.sp_heavy;
    pair = local - head * p.sp_heavy;
  } else {
    const int heavy = kSparse ? p.sp_heavy : 0;
    const int rest = sg.n_pairs - heavy;
    const int l2 = local - heavy * p.n_heads;
    head = l2 / rest;
    pair = heavy + (l2 - head * rest);
  }
  const int qrow0 = pair * (2 * kBM);  // segment-relative
  const int n_tiles = (qrow0 + kBM < sg.nq) ? 2 : 1;
  // KV tiles: those of the first view, then those of the second; the online
  // softmax does not depend on the order in which keys are visited.
  const int n_kv1 = (sg.nkv + kBN - 1) / kBN;
  int n_kv = n_kv1 + (sg.nkv2 + kBN - 1) / kBN;
  const uint16_t* list_tiles = reinterpret_cast<const uint16_t*>(gbase + kOffListTiles);
  const uint8_t* list_sel = gbase + kOffListSel;
  // Set-up by the producer's lane: barriers, then the Q tiles' load, so that
  // Q lands while the other warps zero padded rows, build the block lists
  // and allocate TMEM.  Nothing else touches a barrier before the block-wide
  // barrier below.
  volatile uint32_t* q_issued = reinterpret_cast<volatile uint32_t*>(gbase + kOffQIssued);
  if (warp == 8 && lane == 0) {
    *q_issued = 0u;
    mbar_init(bar(BAR_Q), 1);
    for (int s = 0; s < kNS; ++s) {
      mbar_init(bar(BAR_KFULL + s), 1);
      mbar_init(bar(BAR_VFULL + s), 1);
      mbar_init(bar(BAR_KEMPTY + s), 1);
      mbar_init(bar(BAR_VEMPTY + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(BAR_SFULL + t), 1);
      mbar_init(bar(BAR_PFULL + t), 4);  // one arrive per softmax warp
      mbar_init(bar(BAR_OFINAL + t), 1);
    }
    mbar_init(bar(BAR_DRAIN), 1);
    fence_mbar_init();
    *abort_flag =
        (*reinterpret_cast<volatile uint32_t*>(&g_abort_epoch) == p.epoch) ? 1u : 0u;
    if (*abort_flag == 0u) {
      const CUtensorMap* tq = &p.tm_q[si];
      prefetch_tmap(tq);
      mbar_arrive_expect_tx(bar(BAR_Q), n_tiles * kTileBytes);
      for (int t = 0; t < n_tiles; ++t)
        for (int h = 0; h < 2; ++h)
          tma_load_3d(sbase + kOffQ + t * kTileBytes + h * kHalfBytes, tq, bar(BAR_Q), h * 64,
                      head, qrow0 + t * kBM);
      *q_issued = 1u;
    }
  }
  if (kSparse) {
    // Ordered union of the two query tiles' kept KV blocks (warp 2).
    if (warp == 2) {
      uint32_t* bits = reinterpret_cast<uint32_t*>(gbase + kOffListBits);
      uint16_t* tiles = reinterpret_cast<uint16_t*>(gbase + kOffListTiles);
      uint8_t* sel = gbase + kOffListSel;
      const int nwords = (p.sp_nkb + 31) / 32;
      for (int w = lane; w < 2 * static_cast<int>(kListWords); w += 32) bits[w] = 0u;
      __syncwarp();
      // Both tiles' counts, then their entries in batches of 8 per lane and
      // tile, every load of a batch in flight before the first is used: a
      // handful of global round trips before the first K/V copy can start,
      // instead of one per 32 entries.
      const int64_t row0 = static_cast<int64_t>(head) * p.sp_nqb + qrow0 / kBM;
      const int32_t* lst0 = p.sp_lists + row0 * p.sp_nkb;
      const int32_t* lst1 = lst0 + p.sp_nkb;
      // The first batch is read before the counts are known (every row holds
      // n_kv_blocks entries), so that it shares their round trip.
      int f0[8], f1[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = u * 32 + lane;
        f0[u] = i < p.sp_nkb ? __ldg(lst0 + i) : -1;
        f1[u] = (n_tiles == 2 && i < p.sp_nkb) ? __ldg(lst1 + i) : -1;
      }
      const int c0 = __ldg(p.sp_counts + row0);
      const int c1 = n_tiles == 2 ? __ldg(p.sp_counts + row0 + 1) : 0;
      const int cnt0 = c0 < 0 ? 0 : (c0 > p.sp_nkb ? p.sp_nkb : c0);  // lists are not trusted
      const int cnt1 = c1 < 0 ? 0 : (c1 > p.sp_nkb ? p.sp_nkb : c1);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = u * 32 + lane;
        if (i < cnt0 && f0[u] >= 0 && f0[u] < p.sp_nkb)
          atomicOr(&bits[f0[u] >> 5], 1u << (f0[u] & 31));
        if (i < cnt1 && f1[u] >= 0 && f1[u] < p.sp_nkb)
          atomicOr(&bits[kListWords + (f1[u] >> 5)], 1u << (f1[u] & 31));
      }
      const int cmax = cnt0 > cnt1 ? cnt0 : cnt1;
      for (int base = 8 * 32; base < cmax; base += 8 * 32) {
        int e0[8], e1[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int i = base + u * 32 + lane;
          e0[u] = i < cnt0 ? __ldg(lst0 + i) : -1;
          e1[u] = i < cnt1 ? __ldg(lst1 + i) : -1;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (e0[u] >= 0 && e0[u] < p.sp_nkb) atomicOr(&bits[e0[u] >> 5], 1u << (e0[u] & 31));
          if (e1[u] >= 0 && e1[u] < p.sp_nkb)
            atomicOr(&bits[kListWords + (e1[u] >> 5)], 1u << (e1[u] & 31));
        }
      }
      __syncwarp();
      // Step order: blocks both tiles keep (B), then the two tiles' own
      // blocks alternating (E0, E1, E0, ...), then the rest of the longer
      // one.  The online softmax does not depend on the order of the keys;
      // this one gives the issuer work from both tiles at every step while
      // both have any, so the tiles' Q.K^T -> softmax -> P.V chains overlap.
      int nb = 0, n0 = 0, n1 = 0;
      for (int w = lane; w < nwords; w += 32) {
        const uint32_t b0 = bits[w], b1 = bits[kListWords + w];
        nb += __popc(b0 & b1);
        n0 += __popc(b0 & ~b1);
        n1 += __popc(b1 & ~b0);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        nb += __shfl_xor_sync(0xffffffffu, nb, o);
        n0 += __shfl_xor_sync(0xffffffffu, n0, o);
        n1 += __shfl_xor_sync(0xffffffffu, n1, o);
      }
      const int m = n0 < n1 ? n0 : n1;
      int rb = 0, r0 = 0, r1 = 0;  // ranks before this group of 32 words
      for (int w0 = 0; w0 < nwords; w0 += 32) {
        const int w = w0 + lane;
        const uint32_t b0 = w < nwords ? bits[w] : 0u;
        const uint32_t b1 = w < nwords ? bits[kListWords + w] : 0u;
        const int cb = __popc(b0 & b1), c0 = __popc(b0 & ~b1), c1 = __popc(b1 & ~b0);
        int ib = cb, i0 = c0, i1 = c1;  // inclusive scans over the lanes
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int yb = __shfl_up_sync(0xffffffffu, ib, o);
          const int y0 = __shfl_up_sync(0xffffffffu, i0, o);
          const int y1 = __shfl_up_sync(0xffffffffu, i1, o);
          if (lane >= o) {
            ib += yb;
            i0 += y0;
            i1 += y1;
          }
        }
        int kb = rb + ib - cb, k0 = r0 + i0 - c0, k1 = r1 + i1 - c1;
        uint32_t u = b0 | b1;
        while (u) {
          const int bit = __ffs(u) - 1;
          u &= u - 1;
          const uint32_t sl = ((b0 >> bit) & 1u) | (((b1 >> bit) & 1u) << 1);
          int pos;
          if (sl == 3u) {
            pos = kb++;
          } else if (sl == 1u) {
            pos = nb + (k0 < m ? 2 * k0 : m + k0);
            ++k0;
          } else {
            pos = nb + (k1 < m ? 2 * k1 + 1 : m + k1);
            ++k1;
          }
          tiles[pos] = static_cast<uint16_t>(w * 32 + bit);
          sel[pos] = static_cast<uint8_t>(sl);
        }
        rb += __shfl_sync(0xffffffffu, ib, 31);
        r0 += __shfl_sync(0xffffffffu, i0, 31);
        r1 += __shfl_sync(0xffffffffu, i1, 31);
      }
      if (lane == 0) {
        volatile int* hdr = reinterpret_cast<volatile int*>(gbase + kOffList);
        hdr[0] = nb + n0 + n1;
        hdr[1] = nb;
        hdr[2] = m;
        hdr[3] = n0 >= n1 ? 0 : 1;  // the tile of the steps after the alternation
      }
    }
  }

  // ---- set-up: TMEM (warp 9)
  if (warp == 9) {
    tmem_alloc(sbase + kOffTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + kOffTmemSlot);
  if (kSparse) n_kv = *reinterpret_cast<volatile int*>(gbase + kOffList);
  // No KV tile at all (block-sparse mode with two empty lists): rows are 0.
  const bool no_keys = n_kv == 0;

  if (warp == 8) {
    // ================================================= TMA producer
    if (lane == 0 && *abort_flag == 0u && !no_keys) {
      const CUtensorMap* tk1 = &p.tm_k[si];
      const CUtensorMap* tv1 = &p.tm_v[si];
      const CUtensorMap* tk2 = &p.tm_k2[si];
      const CUtensorMap* tv2 = &p.tm_v2[si];
      prefetch_tmap(tk1);
      prefetch_tmap(tv1);
      if (sg.nkv2 > 0) {
        prefetch_tmap(tk2);
        prefetch_tmap(tv2);
      }
      int armed_k[kNS], armed_v[kNS];
      for (int s = 0; s < kNS; ++s) armed_k[s] = armed_v[s] = -1;
      auto row_of = [&](int j, bool& first) -> int {
        first = kSparse || j < n_kv1;
        return (kSparse ? static_cast<int>(list_tiles[j]) : (first ? j : j - n_kv1)) * kBN;
      };
      // K(j) / V(j) into stage j % kNS once the tile that used it last is released.
      auto load_k = [&](int j) -> bool {
        const int s = j % kNS, use = j / kNS;
        if (j >= kNS && !wait1(bar(BAR_KEMPTY + s), (use - 1) & 1, wctx, H3_STATUS_TIMEOUT_LOAD))
          return false;
        if (p.fault == 1 && j == 1) return true;  // test hook: leave this stage empty
        bool first;
        const int row = row_of(j, first);
        mbar_arrive_expect_tx(bar(BAR_KFULL + s), kTileBytes);
        for (int h = 0; h < 2; ++h)
          tma_load_3d(sbase + kOffK + s * kTileBytes + h * kHalfBytes, first ? tk1 : tk2,
                      bar(BAR_KFULL + s), h * 64, head, row);
        armed_k[s] = use;
        return true;
      };
      auto load_v = [&](int j) -> bool {
        const int s = j % kNS, use = j / kNS;
        if (j >= kNS && !wait1(bar(BAR_VEMPTY + s), (use - 1) & 1, wctx, H3_STATUS_TIMEOUT_LOAD))
          return false;
        if (p.fault == 1 && j == 1) return true;
        bool first;
        const int row = row_of(j, first);
        mbar_arrive_expect_tx(bar(BAR_VFULL + s), kTileBytes);
        for (int h = 0; h < 2; ++h)
          tma_load_3d(sbase + kOffV + s * kTileBytes + h * kHalfBytes, first ? tv1 : tv2,
                      bar(BAR_VFULL + s), h * 64, head, row);
        armed_v[s] = use;
        return true;
      };
      bool ok = true;
      if (kSparse) {
        // K runs one tile ahead of V.  A single-tile step reads V(j) and
        // K(j + 2), and lasts half as long as a two-tile one: queued behind
        // V(j + 1) the next K landed after the step that needs it had begun
        // (98 % of single-tile steps in a clock64 trace; 1,683 -> 1,559
        // cycles per step with K ahead).
        ok = load_k(0);
        for (int j = 0; j < n_kv && ok; ++j) {
          if (j + 1 < n_kv) ok = load_k(j + 1);
          if (ok) ok = load_v(j);
        }
      } else {
        // Dense: K(j) and V(j) in turn.  V(j) is needed at the start of step
        // j and its stage is released half a step before K's, so it must
        // not wait behind K(j + 1) (1.7 % slower that way).
        for (int j = 0; j < n_kv && ok; ++j) {
          const int s = j % kNS, use = j / kNS;
          if (j >= kNS) ok = wait1(bar(BAR_KEMPTY + s), (use - 1) & 1, wctx, H3_STATUS_TIMEOUT_LOAD);
          if (!ok) break;
          if (p.fault == 1 && j == 1) continue;  // test hook: leave this stage empty
          const bool first = j < n_kv1;
          const CUtensorMap* tk = first ? tk1 : tk2;
          const CUtensorMap* tv = first ? tv1 : tv2;
          const int row = (first ? j : j - n_kv1) * kBN;
          mbar_arrive_expect_tx(bar(BAR_KFULL + s), kTileBytes);
          for (int h = 0; h < 2; ++h)
            tma_load_3d(sbase + kOffK + s * kTileBytes + h * kHalfBytes, tk, bar(BAR_KFULL + s),
                        h * 64, head, row);
          armed_k[s] = use;
          if (j >= kNS) ok = wait1(bar(BAR_VEMPTY + s), (use - 1) & 1, wctx, H3_STATUS_TIMEOUT_LOAD);
          if (!ok) break;
          mbar_arrive_expect_tx(bar(BAR_VFULL + s), kTileBytes);
          for (int h = 0; h < 2; ++h)
            tma_load_3d(sbase + kOffV + s * kTileBytes + h * kHalfBytes, tv, bar(BAR_VFULL + s),
                        h * 64, head, row);
          armed_v[s] = use;
        }
      }
      if (*abort_flag != 0u) {
        // Let every copy this CTA started land before the CTA exits.
        drain_wait(bar(BAR_Q), 0);
        for (int s = 0; s < kNS; ++s) {
          if (armed_k[s] >= 0) drain_wait(bar(BAR_KFULL + s), armed_k[s] & 1);
          if (armed_v[s] >= 0) drain_wait(bar(BAR_VFULL + s), armed_v[s] & 1);
        }
      }
    } else if (lane == 0 && *q_issued != 0u) {
      drain_wait(bar(BAR_Q), 0);  // no K/V to load: let the Q copy land before the CTA exits
    }
    __syncwarp();  // lanes 1-31 wait here for lane 0
  } else if (warp == 9) {
    // ================================================= MMA issuer
    if (lane == 0 && *abort_flag == 0u && !no_keys) {
      // Descriptors are built once; a K step only moves the start address,
      // which is the low field of the descriptor (addresses stay < 256 KB).
      const uint64_t dq0 = sdesc_sw128(sbase + kOffQ, 16, 1024);
      const uint64_t dk0 = sdesc_sw128(sbase + kOffK, 16, 1024);
      const uint64_t dv0 = sdesc_sw128(sbase + kOffV, kHalfBytes, 1024);
      auto qk = [&](int t, int s) {
        const uint64_t qa = dq0 + ((t * kTileBytes) >> 4);
        const uint64_t kb = dk0 + ((s * kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kHeadDim / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
          mma_ss(tmem + kColS + t * 128, qa + off, kb + off, kIdescQK, kk > 0 ? 1u : 0u);
        }
      };
      auto pv = [&](int t, int s, bool acc) {
        const uint64_t vb = dv0 + ((s * kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          mma_ts(tmem + kColO + t * 128, tmem + kColS + t * 128 + kk * 8, vb + ((kk * 2048) >> 4),
                 kIdescPV, (acc || kk > 0) ? 1u : 0u);
        }
      };
      bool ok = wait1(bar(BAR_Q), 0, wctx, H3_STATUS_TIMEOUT_MMA) &&
                wait1(bar(BAR_KFULL), 0, wctx, H3_STATUS_TIMEOUT_MMA);
      // Straight-line pieces for two query tiles.  The issuing thread pays
      // tens of cycles for every branch or dependent scalar op between MMAs
      // while the MMA queue holds only a few, so a two-tile step carries no
      // branch but its waits.
      const uint64_t qa0 = dq0, qa1 = dq0 + (kTileBytes >> 4);
      const uint64_t kb0 = dk0, kb1 = dk0 + (kTileBytes >> 4);
      const uint64_t vb0 = dv0, vb1 = dv0 + (kTileBytes >> 4);
      const uint32_t dS0 = tmem + kColS, dS1 = tmem + kColS + 128;
      const uint32_t dO0 = tmem + kColO, dO1 = tmem + kColO + 128;
      auto qk_ = [&](uint32_t dS, uint64_t qa, uint64_t kb) {
#pragma unroll
        for (int kk = 0; kk < kHeadDim / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
          mma_ss(dS, qa + off, kb + off, kIdescQK, kk > 0 ? 1u : 0u);
        }
      };
      auto pv_ = [&](uint32_t dO, uint32_t dS, uint64_t vb, uint32_t acc) {
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ts(dO, dS + kk * 8, vb + ((kk * 2048) >> 4), kIdescPV, acc | (kk > 0 ? 1u : 0u));
      };
      // One step in which both tiles read V(j) and K(j + 1): P_0.V, Q_0.K^T,
      // P_1.V, release V(j), Q_1.K^T, release K(j + 1).  pp0/pp1: the tiles'
      // P phases; acc0/acc1: whether their O already holds a partial sum.
      auto step2 = [&](int j, uint32_t pp0, uint32_t pp1, uint32_t acc0, uint32_t acc1) -> bool {
        const uint32_t s = static_cast<uint32_t>(j) & 1u;
        const uint64_t vbc = s ? vb1 : vb0, kbn = s ? kb0 : kb1;  // V of this stage, K of the next
        // The step's P and V try_waits and a test of K go out back to back;
        // K, needed only after the first P.V, is waited for there if it had
        // not landed.
        const uint32_t kbar = bar(BAR_KFULL + (s ^ 1u)), kpar = (static_cast<uint32_t>(j + 1) >> 1) & 1u;
        const bool p_ok = mbar_try_wait(bar(BAR_PFULL), pp0);
        const bool v_ok = mbar_try_wait(bar(BAR_VFULL + s), (static_cast<uint32_t>(j) >> 1) & 1u);
        const bool k_ok = mbar_test_wait(kbar, kpar);  // a probe: K must not hold up P.V
        bool r = p_ok || wait1(bar(BAR_PFULL), pp0, wctx, H3_STATUS_TIMEOUT_MMA);
        r = r && (v_ok || wait1(bar(BAR_VFULL + s), (static_cast<uint32_t>(j) >> 1) & 1u, wctx,
                                H3_STATUS_TIMEOUT_MMA));
        tc_fence_after();
        pv_(dO0, dS0, vbc, acc0);
        if (!k_ok) {
          r = r && wait1(kbar, kpar, wctx, H3_STATUS_TIMEOUT_MMA);
          tc_fence_after();
        }
        qk_(dS0, qa0, kbn);
        mma_commit(bar(BAR_SFULL));
        r &= wait1(bar(BAR_PFULL + 1), pp1, wctx, H3_STATUS_TIMEOUT_MMA);
        tc_fence_after();
        pv_(dO1, dS1, vbc, acc1);
        mma_commit(bar(BAR_VEMPTY + s));
        qk_(dS1, qa1, kbn);
        mma_commit(bar(BAR_SFULL + 1));
        mma_commit(bar(BAR_KEMPTY + (s ^ 1u)));
        return r;
      };
      if constexpr (!kSparse) {
       if (n_tiles == 2) {
        // The last step (no next Q.K^T) is peeled off.
        if (ok) {
          tc_fence_after();
          qk_(dS0, qa0, kb0);
          mma_commit(bar(BAR_SFULL));
          qk_(dS1, qa1, kb0);
          mma_commit(bar(BAR_SFULL + 1));
          mma_commit(bar(BAR_KEMPTY));
        }
        int j = 0;
        for (; j + 1 < n_kv && ok; ++j) {
          const uint32_t par = static_cast<uint32_t>(j) & 1u;
          ok = step2(j, par, par, j > 0 ? 1u : 0u, j > 0 ? 1u : 0u);
        }
        if (ok) {  // last step
          const uint32_t s = static_cast<uint32_t>(j) & 1u;
          const uint64_t vbc = s ? vb1 : vb0;
          const uint32_t acc = j > 0 ? 1u : 0u;
          ok = wait2(bar(BAR_PFULL), s, bar(BAR_VFULL + s), (static_cast<uint32_t>(j) >> 1) & 1u,
                     wctx, H3_STATUS_TIMEOUT_MMA);
          tc_fence_after();
          pv_(dO0, dS0, vbc, acc);
          mma_commit(bar(BAR_OFINAL));
          ok &= wait1(bar(BAR_PFULL + 1), s, wctx, H3_STATUS_TIMEOUT_MMA);
          tc_fence_after();
          pv_(dO1, dS1, vbc, acc);
          mma_commit(bar(BAR_OFINAL + 1));
        }
       } else {
        if (ok) {
          tc_fence_after();
          for (int t = 0; t < n_tiles; ++t) {
            qk(t, 0);
            mma_commit(bar(BAR_SFULL + t));
          }
          mma_commit(bar(BAR_KEMPTY));
        }
        // One flat loop over (KV step j, query tile t) groups: wait for
        // P_t(j) (and V(j) for the first tile), P_t(j).V(j), then (K(j + 1)
        // landed) Q_t.K(j + 1)^T; the last tile releases the V and K stages.
        const int n_groups = n_kv * n_tiles;
        for (int g = 0; g < n_groups && ok; ++g) {
          const int j = n_tiles == 2 ? (g >> 1) : g;
          const int t = g - j * n_tiles;
          const int s = j % kNS, s2 = (j + 1) % kNS, use2 = (j + 1) / kNS;
          ok = wait1(bar(BAR_PFULL + t), j & 1, wctx, H3_STATUS_TIMEOUT_MMA);
          if (ok && t == 0) ok = wait1(bar(BAR_VFULL + s), (j / kNS) & 1, wctx, H3_STATUS_TIMEOUT_MMA);
          if (!ok) break;
          tc_fence_after();
          pv(t, s, j > 0);
          if (t == n_tiles - 1) mma_commit(bar(BAR_VEMPTY + s));
          if (j + 1 < n_kv) {
            if (t == 0) {
              ok = wait1(bar(BAR_KFULL + s2), use2 & 1, wctx, H3_STATUS_TIMEOUT_MMA);
              if (!ok) break;
              tc_fence_after();
            }
            qk(t, s2);
            mma_commit(bar(BAR_SFULL + t));
            if (t == n_tiles - 1) mma_commit(bar(BAR_KEMPTY + s2));
          } else {
            mma_commit(bar(BAR_OFINAL + t));
          }
        }
       }
      } else {
        // Block-sparse.  The list builder orders the union of the two tiles'
        // kept KV blocks in three phases: nb steps both tiles keep, then 2m
        // steps alternating tile 0, tile 1 (tile 0 first), then the steps
        // left to one tile (rt).  Each tile's next step is therefore known
        // without a search, and every phase runs straight-line steps: the
        // issuing thread pays tens of cycles for each branch or dependent
        // scalar op between MMAs, while the MMA queue holds only a few.
        // Every Q.K^T of step j is issued before step j, so K(j + 2) can
        // always land; a K stage is released after its last Q.K^T, a V stage
        // after its last P.V.  S/P barrier phases count each tile's steps.
        const volatile int* hdr = reinterpret_cast<const volatile int*>(gbase + kOffList);
        const int nb = hdr[1], m = hdr[2], rt = hdr[3];
        const int na_end = nb + 2 * m;  // first step of the last phase
        int kept0 = 0, kept1 = 0;
        // tile t's first step after the two-tile phase (n_kv: none)
        auto first_after_b = [&](int t) -> int {
          if (m > 0) return nb + t;
          return (na_end < n_kv && rt == t) ? na_end : n_kv;
        };
        // Q_t.K(n)^T, t the last reader of K(n)
        auto qk_last = [&](int t, int n) -> bool {
          const uint32_t sn = static_cast<uint32_t>(n) & 1u;
          if (!wait1(bar(BAR_KFULL + sn), (static_cast<uint32_t>(n) >> 1) & 1u, wctx,
                     H3_STATUS_TIMEOUT_MMA))
            return false;
          tc_fence_after();
          qk_(t ? dS1 : dS0, t ? qa1 : qa0, sn ? kb1 : kb0);
          mma_commit(bar(BAR_SFULL + t));
          mma_commit(bar(BAR_KEMPTY + sn));
          return true;
        };
        // P_t.V(j) then Q_t.K(n)^T (n < n_kv), t the last reader of V(j) and
        // of K(n); the P and V try_waits and a test of K go out back to back.
        auto step1 = [&](int t, int j, int kept, int n) -> bool {
          const uint32_t s = static_cast<uint32_t>(j) & 1u, sn = static_cast<uint32_t>(n) & 1u;
          const uint32_t pbar = bar(BAR_PFULL + t), ppar = static_cast<uint32_t>(kept) & 1u;
          const uint32_t vbar = bar(BAR_VFULL + s), vpar = (static_cast<uint32_t>(j) >> 1) & 1u;
          const uint32_t kbar = bar(BAR_KFULL + sn), kpar = (static_cast<uint32_t>(n) >> 1) & 1u;
          const bool p_ok = mbar_try_wait(pbar, ppar);
          const bool v_ok = mbar_try_wait(vbar, vpar);
          const bool k_ok = n >= n_kv || mbar_test_wait(kbar, kpar);  // a probe: K must not hold up P.V
          bool r = p_ok || wait1(pbar, ppar, wctx, H3_STATUS_TIMEOUT_MMA);
          r = r && (v_ok || wait1(vbar, vpar, wctx, H3_STATUS_TIMEOUT_MMA));
          if (!r) return false;
          tc_fence_after();
          pv_(t ? dO1 : dO0, t ? dS1 : dS0, s ? vb1 : vb0, kept > 0 ? 1u : 0u);
          mma_commit(bar(BAR_VEMPTY + s));
          if (n >= n_kv) return true;
          if (!k_ok) {
            if (!wait1(kbar, kpar, wctx, H3_STATUS_TIMEOUT_MMA)) return false;
            tc_fence_after();
          }
          qk_(t ? dS1 : dS0, t ? qa1 : qa0, sn ? kb1 : kb0);
          mma_commit(bar(BAR_SFULL + t));
          mma_commit(bar(BAR_KEMPTY + sn));
          return true;
        };
        if (ok) {
          if (nb > 0) {
            tc_fence_after();
            qk_(dS0, qa0, kb0);
            mma_commit(bar(BAR_SFULL));
            qk_(dS1, qa1, kb0);
            mma_commit(bar(BAR_SFULL + 1));
            mma_commit(bar(BAR_KEMPTY));
          } else {
            const int f0 = first_after_b(0), f1 = first_after_b(1);
            if (f0 < n_kv) ok = qk_last(0, f0);
            if (ok && f1 < n_kv) ok = qk_last(1, f1);
          }
        }
        // Two-tile phase: the dense kernel's step, then the last step hands
        // each tile over to its first step after the phase.
        int j = 0;
        for (; j + 1 < nb && ok; ++j) {
          ok = step2(j, static_cast<uint32_t>(kept0) & 1u, static_cast<uint32_t>(kept1) & 1u,
                     kept0 > 0 ? 1u : 0u, kept1 > 0 ? 1u : 0u);
          ++kept0;
          ++kept1;
        }
        if (ok && nb > 0) {
          const uint32_t s = static_cast<uint32_t>(j) & 1u;
          ok = wait2(bar(BAR_PFULL), static_cast<uint32_t>(kept0) & 1u, bar(BAR_VFULL + s),
                     (static_cast<uint32_t>(j) >> 1) & 1u, wctx, H3_STATUS_TIMEOUT_MMA);
          tc_fence_after();
          pv_(dO0, dS0, s ? vb1 : vb0, kept0 > 0 ? 1u : 0u);
          ++kept0;
          const int f0 = first_after_b(0), f1 = first_after_b(1);
          if (ok && f0 < n_kv) ok = qk_last(0, f0);
          ok &= wait1(bar(BAR_PFULL + 1), static_cast<uint32_t>(kept1) & 1u, wctx,
                      H3_STATUS_TIMEOUT_MMA);
          tc_fence_after();
          pv_(dO1, dS1, s ? vb1 : vb0, kept1 > 0 ? 1u : 0u);
          mma_commit(bar(BAR_VEMPTY + s));
          ++kept1;
          if (ok && f1 < n_kv) ok = qk_last(1, f1);
          ++j;
        }
        // Alternating phase: step j belongs to tile (j - nb) & 1, whose next
        // step is j + 2, or the first step of the last phase.  Pairs of
        // steps (tile 0 at j, tile 1 at j + 1) whose next steps stay in the
        // phase run as straight-line code in which every barrier and
        // descriptor is fixed (j advances by 2, so the ring stages do not
        // change).  Each step also probes, without waiting, the P and V
        // barriers of the step after it before its commits, so that the next
        // step skips their round trip when they have completed.
        if (ok && j + 3 < na_end) {
          const uint32_t sa = static_cast<uint32_t>(j) & 1u, sb = sa ^ 1u;
          const uint32_t pbar0 = bar(BAR_PFULL), pbar1 = bar(BAR_PFULL + 1);
          const uint32_t vfa = bar(BAR_VFULL + sa), vfb = bar(BAR_VFULL + sb);
          const uint32_t kfa = bar(BAR_KFULL + sa), kfb = bar(BAR_KFULL + sb);
          const uint32_t vea = bar(BAR_VEMPTY + sa), veb = bar(BAR_VEMPTY + sb);
          const uint32_t kea = bar(BAR_KEMPTY + sa), keb = bar(BAR_KEMPTY + sb);
          const uint32_t sf0 = bar(BAR_SFULL), sf1 = bar(BAR_SFULL + 1);
          const uint64_t vda = sa ? vb1 : vb0, vdb = sa ? vb0 : vb1;
          const uint64_t kda = sa ? kb1 : kb0, kdb = sa ? kb0 : kb1;
          bool p_known = false, v_known = false;  // probed complete by the previous step
          for (; j + 3 < na_end && ok; j += 2) {
            const uint32_t hj = static_cast<uint32_t>(j) >> 1;
            // tile 0: P0 . V(j), then Q0 . K(j + 2)^T
            {
              const uint32_t pp = static_cast<uint32_t>(kept0) & 1u, vp = hj & 1u;
              const uint32_t kp = (hj + 1u) & 1u;
              const bool p_ok = p_known || mbar_try_wait(pbar0, pp);
              const bool v_ok = v_known || mbar_try_wait(vfa, vp);
              const bool k_ok = mbar_test_wait(kfa, kp);
              bool r = p_ok || wait1(pbar0, pp, wctx, H3_STATUS_TIMEOUT_MMA);
              r = r && (v_ok || wait1(vfa, vp, wctx, H3_STATUS_TIMEOUT_MMA));
              if (!r) { ok = false; break; }
              tc_fence_after();
              pv_(dO0, dS0, vda, kept0 > 0 ? 1u : 0u);
              mma_commit(vea);
              if (!k_ok) {
                if (!wait1(kfa, kp, wctx, H3_STATUS_TIMEOUT_MMA)) { ok = false; break; }
                tc_fence_after();
              }
              qk_(dS0, qa0, kda);
              p_known = mbar_test_wait(pbar1, static_cast<uint32_t>(kept1) & 1u);
              v_known = mbar_test_wait(vfb, (static_cast<uint32_t>(j + 1) >> 1) & 1u);
              mma_commit(sf0);
              mma_commit(kea);
              ++kept0;
            }
            // tile 1: P1 . V(j + 1), then Q1 . K(j + 3)^T
            {
              const uint32_t pp = static_cast<uint32_t>(kept1) & 1u;
              const uint32_t vp = (static_cast<uint32_t>(j + 1) >> 1) & 1u;
              const uint32_t kp = (static_cast<uint32_t>(j + 3) >> 1) & 1u;
              const bool p_ok = p_known || mbar_try_wait(pbar1, pp);
              const bool v_ok = v_known || mbar_try_wait(vfb, vp);
              const bool k_ok = mbar_test_wait(kfb, kp);
              bool r = p_ok || wait1(pbar1, pp, wctx, H3_STATUS_TIMEOUT_MMA);
              r = r && (v_ok || wait1(vfb, vp, wctx, H3_STATUS_TIMEOUT_MMA));
              if (!r) { ok = false; break; }
              tc_fence_after();
              pv_(dO1, dS1, vdb, kept1 > 0 ? 1u : 0u);
              mma_commit(veb);
              if (!k_ok) {
                if (!wait1(kfb, kp, wctx, H3_STATUS_TIMEOUT_MMA)) { ok = false; break; }
                tc_fence_after();
              }
              qk_(dS1, qa1, kdb);
              p_known = mbar_test_wait(pbar0, static_cast<uint32_t>(kept0) & 1u);
              v_known = mbar_test_wait(vfa, ((hj + 1u) & 1u));
              mma_commit(sf1);
              mma_commit(keb);
              ++kept1;
            }
          }
        }
        // The phase's last pair hands each tile over to its next step.
        for (; j < na_end && ok; j += 2) {
          const int n0 = j + 2 < na_end ? j + 2 : ((rt == 0 && na_end < n_kv) ? na_end : n_kv);
          ok = step1(0, j, kept0, n0);
          ++kept0;
          if (!ok) break;
          const int n1 = j + 3 < na_end ? j + 3 : ((rt == 1 && na_end < n_kv) ? na_end : n_kv);
          ok = step1(1, j + 1, kept1, n1);
          ++kept1;
        }
        // The other tile has no step left: its output can be written while
        // tile rt runs the last phase.
        const int other_kept = rt ? kept0 : kept1;
        if (ok && other_kept > 0) mma_commit(bar(BAR_OFINAL + (1 - rt)));
        // Last phase: one tile, step after step.
        for (; j < n_kv && ok; ++j) {
          ok = step1(rt, j, rt ? kept1 : kept0, j + 1);
          if (rt) ++kept1; else ++kept0;
        }
        if (ok && (rt ? kept1 : kept0) > 0) mma_commit(bar(BAR_OFINAL + rt));
      }
      // Every MMA issued above completes before TMEM is released.
      mma_commit(bar(BAR_DRAIN));
      drain_wait(bar(BAR_DRAIN), 0);
    }
    __syncwarp();
  } else {
    // ================================================= softmax (warps 0-7)
    const int t = warp >> 2;
    if (t < n_tiles && *abort_flag == 0u && no_keys) {
      // Block-sparse mode with nothing kept: the tile's valid rows are 0.
      const int row = qrow0 + t * kBM + (warp & 3) * 32 + lane;
      if (row < sg.nq) {
        uint4* dst = reinterpret_cast<uint4*>(
            p.out + static_cast<int64_t>(sg.q_row0 + row) * p.out_stride + head * kHeadDim);
        for (int v4 = 0; v4 < 16; ++v4) dst[v4] = make_uint4(0, 0, 0, 0);
      }
    } else if (t < n_tiles && *abort_flag == 0u) {
      const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
      const uint32_t tS = tmem + lane_base + kColS + t * 128;
      const uint32_t tO = tmem + lane_base + kColO + t * 128;
      const float c = p.scale_log2;
      // valid columns of the last tile of each view (128 when it is full)
      const int tail1 = sg.nkv - (n_kv1 - 1) * kBN;
      const int tail2 = sg.nkv2 - (n_kv - n_kv1 - 1) * kBN;
      float m_used = -INFINITY;
      float l = 0.0f;
      bool ok = true;
      int kept = 0;  // KV steps this tile has processed (= j in dense mode)
      for (int j = 0; j < n_kv; ++j) {
        // Block-sparse: steps this tile's list does not keep have no S / P.
        if (kSparse && !((list_sel[j] >> t) & 1u)) continue;
        ok = wait_warp(bar(BAR_SFULL + t), kept & 1, wctx, H3_STATUS_TIMEOUT_SOFTMAX);
        if (!ok) break;
        tc_fence_after();
        float s[4][32];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld32(tS + q * 32, s[q]);
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_wait_ld(s[q]);
        const int kv_tail = kSparse ? (list_tiles[j] == p.sp_nkb - 1 ? p.sp_tail : kBN)
                                    : (j == n_kv1 - 1) ? tail1 : (j == n_kv - 1) ? tail2 : kBN;
        if (kv_tail < kBN) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int i = 0; i < 32; ++i) s[q][i] = (q * 32 + i < kv_tail) ? s[q][i] : -INFINITY;
        }
        // Row max: 8 independent chains of three-input max.
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = fmax3(s[0][i], s[0][i + 8], s[0][i + 16]);
#pragma unroll
        for (int i = 24; i < 32; ++i) mx[i & 7] = fmaxf(mx[i & 7], s[0][i]);
#pragma unroll
        for (int q = 1; q < 4; ++q)
#pragma unroll
          for (int i = 0; i < 16; ++i) mx[i & 7] = fmax3(mx[i & 7], s[q][i], s[q][i + 16]);
        const float m_tile =
            fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) * c;
        // Lazy rescaling: the running max only moves when the tile max
        // exceeds it by more than 2^8, so p <= 256 and O / l stay exact.
        const bool need = m_tile > m_used + kRescaleThreshold;
        const float alpha = need ? ex2(m_used - m_tile) : 1.0f;  // 0 on the first tile
        l *= alpha;
        if (need) m_used = m_tile;
        // p = 2^(s*c - m) for pairs: packed FMA, two ex2, packed running sums.
        float ls[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) ls[i] = 0.0f;
        const float neg_m = -m_used;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float a0, a1;
            ffma2(a0, a1, s[q][2 * i], s[q][2 * i + 1], c, c, neg_m, neg_m);
            const float p0 = ex2(a0);
            const float p1 = ex2(a1);
            fadd2(ls[2 * (i & 3)], ls[2 * (i & 3) + 1], ls[2 * (i & 3)], ls[2 * (i & 3) + 1], p0, p1);
            pk[i] = pack_bf16x2(p0, p1);
          }
          tmem_st16(tS + q * 16, pk);  // P columns 16q..16q+15 = scores 32q..32q+31
        }
        fadd2(ls[0], ls[1], ls[0], ls[1], ls[2], ls[3]);
        fadd2(ls[4], ls[5], ls[4], ls[5], ls[6], ls[7]);
        fadd2(ls[0], ls[1], ls[0], ls[1], ls[4], ls[5]);
        l += ls[0] + ls[1];
        if (kept > 0 && __any_sync(0xffffffffu, need)) {
          // O_t holds PV(0..j-1), complete because S_t(j) is (in-order MMAs).
          const float f = alpha;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float o[32];
            tmem_ld32(tO + q * 32, o);
            tmem_wait_ld(o);
#pragma unroll
            for (int i = 0; i < 32; i += 2) fmul2(o[i], o[i + 1], o[i], o[i + 1], f, f);
            tmem_st32(tO + q * 32, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_PFULL + t));
        ++kept;
      }
      // A tile whose list keeps nothing has no O (TMEM never written): its
      // valid rows are 0.
      if (ok && kept == 0) {
        const int row = qrow0 + t * kBM + (warp & 3) * 32 + lane;
        if (row < sg.nq) {
          uint4* dst = reinterpret_cast<uint4*>(
              p.out + static_cast<int64_t>(sg.q_row0 + row) * p.out_stride + head * kHeadDim);
          for (int v4 = 0; v4 < 16; ++v4) dst[v4] = make_uint4(0, 0, 0, 0);
        }
        ok = false;
      }
      if (ok) ok = wait_warp(bar(BAR_OFINAL + t), 0, wctx, H3_STATUS_TIMEOUT_SOFTMAX);
      if (ok) {
        tc_fence_after();
        const float inv_l = l > 0.0f ? 1.0f / l : 0.0f;  // l == 0: no kept key
        const int row = qrow0 + t * kBM + (warp & 3) * 32 + lane;  // segment-relative
        const bool valid_row = row < sg.nq;
        uint4* dst = reinterpret_cast<uint4*>(
            p.out + static_cast<int64_t>(sg.q_row0 + row) * p.out_stride + head * kHeadDim);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float o[32];
          tmem_ld32(tO + q * 32, o);
          tmem_wait_ld(o);
          uint32_t u[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            fmul2(o[2 * i], o[2 * i + 1], o[2 * i], o[2 * i + 1], inv_l, inv_l);
            u[i] = pack_bf16x2(o[2 * i], o[2 * i + 1]);
          }
          if (valid_row) {
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
              dst[q * 4 + v4] = make_uint4(u[4 * v4], u[4 * v4 + 1], u[4 * v4 + 2], u[4 * v4 + 3]);
          }
        }
      }
    }
  }

  // ---- teardown: all TMEM reads and MMAs are complete here
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encoder(std::string& err) {
  static std::atomic<EncodeTiledFn> fn{nullptr};
  if (EncodeTiledFn f = fn.load()) return f;
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q{};
  cudaError_t e =
      cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || ptr == nullptr) {
    err = std::string("cuTensorMapEncodeTiled unavailable: ") + cudaGetErrorString(e);
    return nullptr;
  }
  const EncodeTiledFn f = reinterpret_cast<EncodeTiledFn>(ptr);
  fn.store(f);  // threads racing here store the same entry point
  return f;
}

// [rows, n_heads, 128] bf16 starting at `base`, boxes of 64 channels x 1 head x 128 rows.
bool encode_rows(EncodeTiledFn enc, CUtensorMap* m, const void* base, int64_t row_stride,
                 int n_heads, int rows, std::string& err) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(n_heads),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim) * 2,
                                 static_cast<cuuint64_t>(row_stride) * 2};
  const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(kBN)};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    err = "cuTensorMapEncodeTiled failed with CUresult " + std::to_string(static_cast<int>(r));
    return false;
  }
  return true;
}

std::atomic<uint32_t> g_epoch_counter{0};
std::atomic<int> g_fault_next{0};

}  // namespace

namespace {

struct Item {
  int q0, nq;  // query rows
  int kv0, nkv;  // first KV view: rows of k / v
  int c0, nc;    // second KV view: rows of k_cache / v_cache
};

struct Buffers {
  const __nv_bfloat16 *q, *k, *v, *kc, *vc;
  __nv_bfloat16* out;
  int64_t q_stride, k_stride, v_stride, kc_stride, vc_stride, out_stride;
};

// Work items (at most H3_MAX_SEGMENTS, nq > 0, nkv + nc > 0) and output
// row ranges to zero -> tensor maps, schedule, one launch.
struct SparseLists {
  const int32_t* lists;
  const int32_t* counts;
  int nqb, nkb, tail;
  int heavy_pairs;  // leading query-tile pairs scheduled first
};

int launch_items(const Buffers& b, std::vector<Item>& items,
                 const std::vector<std::pair<int, int>>& zero, int n_heads, float scale,
                 cudaStream_t stream, std::string& err, const SparseLists* sparse = nullptr) {
  EncodeTiledFn enc = get_encoder(err);
  if (!enc) return H3_ERR_DEVICE;
  thread_local AttnParams P;  // ~11 KB of kernel parameters, rebuilt on every call
  std::memset(&P, 0, sizeof(P));
  P.n_zero = 0;
  P.zero_chunks = 0;
  for (const auto& z : zero) {
    if (z.second <= 0) continue;
    P.zero_row0[P.n_zero] = z.first;
    P.zero_rows[P.n_zero] = z.second;
    P.zero_chunks += static_cast<int64_t>(z.second) * n_heads * 16;
    ++P.n_zero;
  }
  // Longest KV extent first, so that long work items start in the first wave.
  std::stable_sort(items.begin(), items.end(), [](const Item& x, const Item& y) {
    return x.nkv + x.nc > y.nkv + y.nc;
  });
  int64_t ctas = 0;
  for (size_t i = 0; i < items.size(); ++i) {
    const Item& it = items[i];
    Seg& s = P.seg[i];
    s.q_row0 = it.q0;
    s.nq = it.nq;
    // A view with no rows is moved second, so that tile 0 always exists.
    const bool swap = it.nkv == 0;
    const int kv0 = swap ? it.c0 : it.kv0, nkv = swap ? it.nc : it.nkv;
    const __nv_bfloat16* k1 = swap ? b.kc : b.k;
    const __nv_bfloat16* v1 = swap ? b.vc : b.v;
    const int64_t ks1 = swap ? b.kc_stride : b.k_stride, vs1 = swap ? b.vc_stride : b.v_stride;
    s.nkv = nkv;
    s.nkv2 = swap ? 0 : it.nc;
    s.n_pairs = (it.nq + 2 * kBM - 1) / (2 * kBM);
    s.cta0 = static_cast<int32_t>(ctas);
    ctas += static_cast<int64_t>(s.n_pairs) * n_heads;
    if (!encode_rows(enc, &P.tm_q[i], b.q + static_cast<int64_t>(it.q0) * b.q_stride, b.q_stride,
                     n_heads, it.nq, err) ||
        !encode_rows(enc, &P.tm_k[i], k1 + static_cast<int64_t>(kv0) * ks1, ks1, n_heads, nkv,
                     err) ||
        !encode_rows(enc, &P.tm_v[i], v1 + static_cast<int64_t>(kv0) * vs1, vs1, n_heads, nkv,
                     err))
      return H3_ERR_DEVICE;
    if (s.nkv2 > 0 &&
        (!encode_rows(enc, &P.tm_k2[i], b.kc + static_cast<int64_t>(it.c0) * b.kc_stride,
                      b.kc_stride, n_heads, it.nc, err) ||
         !encode_rows(enc, &P.tm_v2[i], b.vc + static_cast<int64_t>(it.c0) * b.vc_stride,
                      b.vc_stride, n_heads, it.nc, err)))
      return H3_ERR_DEVICE;
  }
  if (ctas > 0x7fffffff) {
    err = "too many work items for one launch";
    return H3_ERR_SHAPE;
  }
  P.n_seg = static_cast<int32_t>(items.size());
  P.n_heads = n_heads;
  P.n_compute_ctas = static_cast<int32_t>(ctas);
  P.out = b.out;
  P.out_stride = b.out_stride;
  P.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  P.epoch = g_epoch_counter.fetch_add(1) + 1;
  P.fault = g_fault_next.exchange(0);
  if (sparse != nullptr) {
    P.sp_lists = sparse->lists;
    P.sp_counts = sparse->counts;
    P.sp_nqb = sparse->nqb;
    P.sp_nkb = sparse->nkb;
    P.sp_tail = sparse->tail;
    P.sp_heavy = sparse->heavy_pairs;
  }
  int64_t grid = ctas;
  if (grid == 0) {
    if (P.zero_chunks == 0) return H3_OK;  // nothing to do
    grid = std::min<int64_t>((P.zero_chunks + 255) / 256, 1024);
  }

  const bool sp = sparse != nullptr;
  auto kernel = sp ? attn_fwd_kernel<true> : attn_fwd_kernel<false>;
  const uint32_t smem = sp ? kSmemBytesSparse : kSmemBytes;
  static std::atomic<int> attr_done[2][64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && attr_done[sp][dev].load() == 0) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) {
      err = std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e);
      return H3_ERR_DEVICE;
    }
    attr_done[sp][dev].store(1);
  }
  kernel<<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(P);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    err = std::string("attention launch: ") + cudaGetErrorString(e);
    return H3_ERR_LAUNCH;
  }
  return H3_OK;
}

}  // namespace

int launch_attention(const AttnArgs& a, cudaStream_t stream, std::string& err) {
  std::vector<Item> items;
  std::vector<std::pair<int, int>> zero;
  for (int b = 0; b < a.n_seq; ++b) {
    const int q0 = a.cu_q[b], q_ext = a.cu_q[b + 1] - a.cu_q[b];
    const int kv0 = a.cu_kv[b], kv_ext = a.cu_kv[b + 1] - a.cu_kv[b];
    int nq = a.valid ? a.valid[b] : q_ext;
    const int nkv = a.valid ? a.valid[b] : kv_ext;
    if (nkv == 0) nq = 0;  // no key: every query row of the segment is 0
    if (nq > 0) items.push_back({q0, nq, kv0, nkv, 0, 0});
    if (q_ext > nq) zero.push_back({q0 + nq, q_ext - nq});
  }
  const Buffers bufs{a.q, a.k, a.v, nullptr, nullptr, a.out,
                     a.q_stride, a.k_stride, a.v_stride, 0, 0, a.out_stride};
  return launch_items(bufs, items, zero, a.n_heads, a.scale, stream, err);
}

int launch_attention_groups(const AttnGroupArgs& a, cudaStream_t stream, std::string& err) {
  std::vector<Item> items;
  std::vector<std::pair<int, int>> zero;
  for (int g = 0; g < a.n_groups; ++g) {
    const h3_attn_group& G = a.groups[g];
    if (G.q_len == 0) continue;
    if (G.kv_len + G.cache_len == 0)
      zero.push_back({G.q_start, G.q_len});
    else
      items.push_back({G.q_start, G.q_len, G.kv_start, G.kv_len, G.cache_start, G.cache_len});
  }
  const Buffers bufs{a.q, a.k, a.v, a.kc, a.vc, a.out,
                     a.q_stride, a.k_stride, a.v_stride, a.kc_stride, a.vc_stride, a.out_stride};
  return launch_items(bufs, items, zero, a.n_heads, a.scale, stream, err);
}

int launch_sparse_attention(const SparseAttnArgs& a, cudaStream_t stream, std::string& err) {
  std::vector<Item> items;
  std::vector<std::pair<int, int>> zero;
  items.push_back({0, static_cast<int>(a.n_rows), 0, static_cast<int>(a.n_rows), 0, 0});
  const Buffers bufs{a.q, a.k, a.v, nullptr, nullptr, a.out,
                     a.q_stride, a.k_stride, a.v_stride, 0, 0, a.out_stride};
  const int nb = static_cast<int>((a.n_rows + kBN - 1) / kBN);
  const int n_pairs = (nb + 1) / 2;
  const int heavy = std::min((a.n_prefix_blocks + 1) / 2, n_pairs);
  const SparseLists sl{a.lists, a.counts, nb, nb, static_cast<int>(a.n_rows - (nb - 1) * kBN),
                       heavy};
  return launch_items(bufs, items, zero, a.n_heads, a.scale, stream, err, &sl);
}

// Device address of the status word on the current device (looked up once
// per device, with that device current), for kernels in other files.
uint32_t* status_word_device_ptr() {
  static std::atomic<uint32_t*> ptrs[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (uint32_t* q = ptrs[dev].load()) return q;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
  ptrs[dev].store(static_cast<uint32_t*>(p));  // racing threads store the same address
  return static_cast<uint32_t*>(p);
}

cudaError_t read_and_clear_status(uint32_t* out) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(out, g_status, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  const uint32_t zero = 0;
  return cudaMemcpyToSymbol(g_status, &zero, sizeof(uint32_t));
}

// Test hook (not in the public header): the next h3_attention launch on any
// thread runs with the given fault; 1 = the producer never loads K/V tile 1,
// so the MMA issuer's bounded wait runs out.
void set_fault_next(int f) { g_fault_next.store(f); }

}  // namespace h3
