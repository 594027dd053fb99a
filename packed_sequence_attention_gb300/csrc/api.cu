// C-ABI front end of libh3kern: argument checks on the host, device checks,
// then one launch per call.  See include/h3kern.h for the contract.
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <initializer_list>
#include <string>

#include "h3_internal.h"
#include "h3kern_debug.h"

namespace h3 {
void set_fault_next(int f);
}

namespace {

thread_local std::string t_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return code;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Current device must be compute capability 10.3 (the kernels are built for
// sm_103a only).  The answer is cached per device.
int check_device() {
  static std::atomic<int> cache[64];  // 0 unknown, 1 sm_103, 2 other
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(H3_ERR_DEVICE, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev >= 0 && dev < 64) {
    const int c = cache[dev].load();
    if (c == 1) return H3_OK;
    if (c == 2) return fail(H3_ERR_ARCH, "device %d is not sm_103", dev);
  }
  int major = 0, minor = 0;
  e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e != cudaSuccess)
    return fail(H3_ERR_DEVICE, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
  const bool ok = (major == 10 && minor == 3);
  if (dev >= 0 && dev < 64) cache[dev].store(ok ? 1 : 2);
  if (!ok) return fail(H3_ERR_ARCH, "device %d is sm_%d%d, the kernels need sm_103", dev, major, minor);
  return H3_OK;
}

// Every pointer a kernel dereferences (or encodes into a tensor map) must be
// memory of the current device, or managed memory: a host buffer or another
// GPU's memory would otherwise reach the kernel as a bad address.  NULL
// entries (optional outputs) are skipped.  Call after check_device().
struct DevPtr {
  const void* p;
  const char* name;
};

int check_device_memory(std::initializer_list<DevPtr> ptrs) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(H3_ERR_DEVICE, "cudaGetDevice: %s", cudaGetErrorString(e));
  for (const DevPtr& d : ptrs) {
    if (d.p == nullptr) continue;
    cudaPointerAttributes attr{};
    e = cudaPointerGetAttributes(&attr, d.p);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();  // a failed query leaves no sticky error
      return fail(H3_ERR_ARG, "%s: cannot query the pointer (%s)", d.name, cudaGetErrorString(e));
    }
    if (attr.type == cudaMemoryTypeManaged) continue;
    if (attr.type != cudaMemoryTypeDevice)
      return fail(H3_ERR_ARG, "%s is host memory; it must be memory of the current device %d",
                  d.name, dev);
    if (attr.device != dev)
      return fail(H3_ERR_ARG, "%s is memory of device %d, but the current device is %d", d.name,
                  attr.device, dev);
  }
  return H3_OK;
}

}  // namespace

extern "C" {

int h3_version(void) { return 1 * 10000 + 0 * 100 + 0; }

const char* h3_last_error(void) { return t_last_error.c_str(); }

}  // extern "C"

namespace {

// Shared checks and launch of the plain, packed-sequence and LoRA-fused
// prologue.  The rows are n_seg segments [seg_row0[b], seg_row0[b] + seg_rows[b])
// of the buffers (already checked: non-negative, in order, not overlapping).
int norm_rope_entry(void* q, int64_t q_row_stride, void* k, int64_t k_row_stride,
                    const void* dq, int64_t dq_row_stride, const void* dk, int64_t dk_row_stride,
                    bool lora, const void* wq, const void* wk, const int32_t* pos_thw,
                    const int64_t* seg_row0, const int64_t* seg_rows, int n_seg, int n_heads,
                    int head_dim, int rot_t, int rot_h, int rot_w, float theta, float eps,
                    h3_stream_t stream) {
  int64_t n_rows = 0;
  for (int b = 0; b < n_seg; ++b) n_rows += seg_rows[b];
  if (n_heads < 1) return fail(H3_ERR_ARG, "n_heads must be >= 1 (got %d)", n_heads);
  if (head_dim != h3::kHeadDim) return fail(H3_ERR_SHAPE, "head_dim must be 128 (got %d)", head_dim);
  if (n_heads > h3::prologue_max_heads(lora))
    return fail(H3_ERR_SHAPE, "n_heads must be <= %d for this prologue (got %d)",
                h3::prologue_max_heads(lora), n_heads);
  if (rot_t < 0 || rot_h < 0 || rot_w < 0 || (rot_t | rot_h | rot_w) & 1)
    return fail(H3_ERR_SHAPE, "rotary sections must be even and >= 0 (got %d/%d/%d)", rot_t, rot_h,
                rot_w);
  if (rot_t + rot_h + rot_w > head_dim)
    return fail(H3_ERR_SHAPE, "rotary sections sum to %d > head_dim %d", rot_t + rot_h + rot_w,
                head_dim);
  if (!std::isfinite(theta) || !(theta > 0.0f))
    return fail(H3_ERR_ARG, "theta must be finite and > 0");
  if (!std::isfinite(eps) || eps < 0.0f) return fail(H3_ERR_ARG, "eps must be finite and >= 0");
  const int64_t width = static_cast<int64_t>(n_heads) * h3::kHeadDim;
  if (q_row_stride < width || k_row_stride < width)
    return fail(H3_ERR_SHAPE, "row strides (%lld, %lld) must be >= n_heads*128 = %lld",
                (long long)q_row_stride, (long long)k_row_stride, (long long)width);
  if (lora && (dq_row_stride < width || dk_row_stride < width))
    return fail(H3_ERR_SHAPE, "delta row strides (%lld, %lld) must be >= n_heads*128 = %lld",
                (long long)dq_row_stride, (long long)dk_row_stride, (long long)width);
  if (n_rows == 0) return H3_OK;
  if (!q || !k || !wq || !wk || !pos_thw || (lora && (!dq || !dk)))
    return fail(H3_ERR_ARG, "null pointer argument");
  if (q == k) return fail(H3_ERR_ARG, "q and k must be distinct buffers");
  if (!aligned16(q) || !aligned16(k) || !aligned16(wq) || !aligned16(wk) ||
      (lora && (!aligned16(dq) || !aligned16(dk))))
    return fail(H3_ERR_ALIGN, "tensor and weight pointers must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(pos_thw) & 3u) != 0)
    return fail(H3_ERR_ALIGN, "pos_thw must be 4-byte aligned");
  if ((q_row_stride * 2) % 16 != 0 || (k_row_stride * 2) % 16 != 0 ||
      (lora && ((dq_row_stride * 2) % 16 != 0 || (dk_row_stride * 2) % 16 != 0)))
    return fail(H3_ERR_ALIGN, "row strides must be multiples of 8 elements (16 bytes)");
  if (n_rows > (int64_t(1) << 30))
    return fail(H3_ERR_SHAPE, "%lld rows are too many for one launch (at most 2^30)",
                (long long)n_rows);
  int st = check_device();
  if (st != H3_OK) return st;
  st = check_device_memory({{q, "q"}, {k, "k"}, {wq, "wq"}, {wk, "wk"}, {pos_thw, "pos_thw"},
                            {lora ? dq : nullptr, "q_delta"}, {lora ? dk : nullptr, "k_delta"}});
  if (st != H3_OK) return st;
  h3::NormRopeArgs a{};
  a.q = static_cast<__nv_bfloat16*>(q);
  a.k = static_cast<__nv_bfloat16*>(k);
  a.q_stride = q_row_stride;
  a.k_stride = k_row_stride;
  a.wq = static_cast<const __nv_bfloat16*>(wq);
  a.wk = static_cast<const __nv_bfloat16*>(wk);
  a.pos = pos_thw;
  a.seg_row0 = seg_row0;
  a.seg_rows = seg_rows;
  a.n_seg = n_seg;
  a.n_heads = n_heads;
  a.rot[0] = rot_t;
  a.rot[1] = rot_h;
  a.rot[2] = rot_w;
  a.theta = theta;
  a.eps = eps;
  if (lora) {
    a.dq = static_cast<const __nv_bfloat16*>(dq);
    a.dk = static_cast<const __nv_bfloat16*>(dk);
    a.dq_stride = dq_row_stride;
    a.dk_stride = dk_row_stride;
  }
  cudaError_t e = h3::launch_qk_norm_rope(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(H3_ERR_LAUNCH, "qk_norm_rope launch: %s", cudaGetErrorString(e));
  return H3_OK;
}

}  // namespace

extern "C" {

int h3_qk_norm_rope(void* q, int64_t q_row_stride, void* k, int64_t k_row_stride, const void* wq,
                    const void* wk, const int32_t* pos_thw, int64_t n_rows, int n_heads,
                    int head_dim, int rot_t, int rot_h, int rot_w, float theta, float eps,
                    h3_stream_t stream) {
  if (n_rows < 0) return fail(H3_ERR_ARG, "n_rows must be >= 0 (got %lld)", (long long)n_rows);
  const int64_t row0 = 0;
  return norm_rope_entry(q, q_row_stride, k, k_row_stride, nullptr, 0, nullptr, 0, false, wq, wk,
                         pos_thw, &row0, &n_rows, 1, n_heads, head_dim, rot_t, rot_h, rot_w,
                         theta, eps, stream);
}

int h3_qk_norm_rope_varlen(void* q, int64_t q_row_stride, void* k, int64_t k_row_stride,
                           const void* wq, const void* wk, const int32_t* pos_thw,
                           const int32_t* cu_seqlens, const int32_t* valid_len, int n_seq,
                           int n_heads, int head_dim, int rot_t, int rot_h, int rot_w,
                           float theta, float eps, h3_stream_t stream) {
  if (n_seq < 1 || n_seq > H3_MAX_SEGMENTS)
    return fail(H3_ERR_ARG, "n_seq must be in [1, %d] (got %d)", H3_MAX_SEGMENTS, n_seq);
  if (!cu_seqlens) return fail(H3_ERR_ARG, "null cu_seqlens");
  if (cu_seqlens[0] != 0) return fail(H3_ERR_ARG, "cu_seqlens must start at 0");
  int64_t row0[H3_MAX_SEGMENTS], rows[H3_MAX_SEGMENTS];
  for (int b = 0; b < n_seq; ++b) {
    if (cu_seqlens[b + 1] < cu_seqlens[b])
      return fail(H3_ERR_ARG, "cu_seqlens must be non-decreasing (segment %d)", b);
    const int32_t len = cu_seqlens[b + 1] - cu_seqlens[b];
    if (valid_len && (valid_len[b] < 0 || valid_len[b] > len))
      return fail(H3_ERR_ARG, "valid_len[%d] = %d outside [0, %d]", b, valid_len[b], len);
    row0[b] = cu_seqlens[b];
    rows[b] = valid_len ? valid_len[b] : len;
  }
  return norm_rope_entry(q, q_row_stride, k, k_row_stride, nullptr, 0, nullptr, 0, false, wq, wk,
                         pos_thw, row0, rows, n_seq, n_heads, head_dim, rot_t, rot_h, rot_w,
                         theta, eps, stream);
}

int h3_qk_norm_rope_lora(void* q, int64_t q_row_stride, const void* q_delta,
                         int64_t q_delta_row_stride, void* k, int64_t k_row_stride,
                         const void* k_delta, int64_t k_delta_row_stride, const void* wq,
                         const void* wk, const int32_t* pos_thw, int64_t n_rows, int n_heads,
                         int head_dim, int rot_t, int rot_h, int rot_w, float theta, float eps,
                         h3_stream_t stream) {
  if (n_rows < 0) return fail(H3_ERR_ARG, "n_rows must be >= 0 (got %lld)", (long long)n_rows);
  const int64_t row0 = 0;
  return norm_rope_entry(q, q_row_stride, k, k_row_stride, q_delta, q_delta_row_stride, k_delta,
                         k_delta_row_stride, true, wq, wk, pos_thw, &row0, &n_rows, 1, n_heads,
                         head_dim, rot_t, rot_h, rot_w, theta, eps, stream);
}

int h3_attention(const void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride,
                 const void* v, int64_t v_row_stride, void* out, int64_t out_row_stride,
                 const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                 const int32_t* valid_len, int n_seq, int n_heads, int head_dim, float scale,
                 h3_stream_t stream) {
  if (n_seq < 1 || n_seq > H3_MAX_SEGMENTS)
    return fail(H3_ERR_ARG, "n_seq must be in [1, %d] (got %d)", H3_MAX_SEGMENTS, n_seq);
  if (n_heads < 1) return fail(H3_ERR_ARG, "n_heads must be >= 1 (got %d)", n_heads);
  if (head_dim != h3::kHeadDim) return fail(H3_ERR_SHAPE, "head_dim must be 128 (got %d)", head_dim);
  if (!std::isfinite(scale) || !(scale > 0.0f)) return fail(H3_ERR_ARG, "scale must be finite and > 0");
  if (!cu_seqlens_q || !cu_seqlens_kv) return fail(H3_ERR_ARG, "null cu_seqlens");
  if (cu_seqlens_q[0] != 0 || cu_seqlens_kv[0] != 0)
    return fail(H3_ERR_ARG, "cu_seqlens must start at 0");
  for (int b = 0; b < n_seq; ++b) {
    if (cu_seqlens_q[b + 1] < cu_seqlens_q[b] || cu_seqlens_kv[b + 1] < cu_seqlens_kv[b])
      return fail(H3_ERR_ARG, "cu_seqlens must be non-decreasing (segment %d)", b);
    if (valid_len) {
      const int32_t lim = std::min(cu_seqlens_q[b + 1] - cu_seqlens_q[b],
                                   cu_seqlens_kv[b + 1] - cu_seqlens_kv[b]);
      if (valid_len[b] < 0 || valid_len[b] > lim)
        return fail(H3_ERR_ARG, "valid_len[%d] = %d outside [0, %d]", b, valid_len[b], lim);
    }
  }
  const int64_t width = static_cast<int64_t>(n_heads) * h3::kHeadDim;
  if (q_row_stride < width || k_row_stride < width || v_row_stride < width ||
      out_row_stride < width)
    return fail(H3_ERR_SHAPE, "row strides must be >= n_heads*128 = %lld", (long long)width);
  if (!q || !k || !v || !out) return fail(H3_ERR_ARG, "null tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(H3_ERR_ALIGN, "q, k, v, out must be 16-byte aligned");
  if ((q_row_stride * 2) % 16 || (k_row_stride * 2) % 16 || (v_row_stride * 2) % 16 ||
      (out_row_stride * 2) % 16)
    return fail(H3_ERR_ALIGN, "row strides must be multiples of 8 elements (16 bytes)");
  if (q_row_stride * 2 >= (int64_t(1) << 40) || k_row_stride * 2 >= (int64_t(1) << 40) ||
      v_row_stride * 2 >= (int64_t(1) << 40))
    return fail(H3_ERR_SHAPE, "row stride too large for a tensor map");
  int st = check_device();
  if (st != H3_OK) return st;
  st = check_device_memory({{q, "q"}, {k, "k"}, {v, "v"}, {out, "out"}});
  if (st != H3_OK) return st;
  h3::AttnArgs a{};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.q_stride = q_row_stride;
  a.k_stride = k_row_stride;
  a.v_stride = v_row_stride;
  a.out_stride = out_row_stride;
  a.cu_q = cu_seqlens_q;
  a.cu_kv = cu_seqlens_kv;
  a.valid = valid_len;
  a.n_seq = n_seq;
  a.n_heads = n_heads;
  a.scale = scale;
  std::string err;
  st = h3::launch_attention(a, reinterpret_cast<cudaStream_t>(stream), err);
  if (st != H3_OK) return fail(st, "%s", err.c_str());
  return H3_OK;
}

int h3_attention_groups(const void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride,
                        const void* v, int64_t v_row_stride, const void* k_cache,
                        int64_t k_cache_row_stride, const void* v_cache,
                        int64_t v_cache_row_stride, void* out, int64_t out_row_stride,
                        const h3_attn_group* groups, int n_groups, int n_heads, int head_dim,
                        float scale, h3_stream_t stream) {
  if (n_groups < 1 || n_groups > H3_MAX_SEGMENTS)
    return fail(H3_ERR_ARG, "n_groups must be in [1, %d] (got %d)", H3_MAX_SEGMENTS, n_groups);
  if (!groups) return fail(H3_ERR_ARG, "null groups");
  if (n_heads < 1) return fail(H3_ERR_ARG, "n_heads must be >= 1 (got %d)", n_heads);
  if (head_dim != h3::kHeadDim) return fail(H3_ERR_SHAPE, "head_dim must be 128 (got %d)", head_dim);
  if (!std::isfinite(scale) || !(scale > 0.0f)) return fail(H3_ERR_ARG, "scale must be finite and > 0");
  bool uses_cache = false;
  for (int g = 0; g < n_groups; ++g) {
    const h3_attn_group& G = groups[g];
    const int64_t f[6] = {G.q_start, G.q_len, G.kv_start, G.kv_len, G.cache_start, G.cache_len};
    for (int i = 0; i < 6; ++i)
      if (f[i] < 0) return fail(H3_ERR_ARG, "group %d has a negative field", g);
    if (f[0] + f[1] > INT32_MAX || f[2] + f[3] > INT32_MAX || f[4] + f[5] > INT32_MAX)
      return fail(H3_ERR_ARG, "group %d addresses rows past 2^31", g);
    uses_cache = uses_cache || G.cache_len > 0;
    for (int o = 0; o < g; ++o) {  // query ranges must not overlap (racing writes)
      const h3_attn_group& P = groups[o];
      if (G.q_len > 0 && P.q_len > 0 && G.q_start < P.q_start + P.q_len &&
          P.q_start < G.q_start + G.q_len)
        return fail(H3_ERR_ARG, "query ranges of groups %d and %d overlap", o, g);
    }
  }
  const int64_t width = static_cast<int64_t>(n_heads) * h3::kHeadDim;
  if (q_row_stride < width || k_row_stride < width || v_row_stride < width ||
      out_row_stride < width || (uses_cache && (k_cache_row_stride < width ||
                                                v_cache_row_stride < width)))
    return fail(H3_ERR_SHAPE, "row strides must be >= n_heads*128 = %lld", (long long)width);
  if (!q || !k || !v || !out || (uses_cache && (!k_cache || !v_cache)))
    return fail(H3_ERR_ARG, "null tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      (uses_cache && (!aligned16(k_cache) || !aligned16(v_cache))))
    return fail(H3_ERR_ALIGN, "tensor pointers must be 16-byte aligned");
  if ((q_row_stride * 2) % 16 || (k_row_stride * 2) % 16 || (v_row_stride * 2) % 16 ||
      (out_row_stride * 2) % 16 ||
      (uses_cache && ((k_cache_row_stride * 2) % 16 || (v_cache_row_stride * 2) % 16)))
    return fail(H3_ERR_ALIGN, "row strides must be multiples of 8 elements (16 bytes)");
  const int64_t lim = int64_t(1) << 40;
  if (q_row_stride * 2 >= lim || k_row_stride * 2 >= lim || v_row_stride * 2 >= lim ||
      k_cache_row_stride * 2 >= lim || v_cache_row_stride * 2 >= lim)
    return fail(H3_ERR_SHAPE, "row stride too large for a tensor map");
  int st = check_device();
  if (st != H3_OK) return st;
  st = check_device_memory({{q, "q"}, {k, "k"}, {v, "v"}, {out, "out"},
                            {uses_cache ? k_cache : nullptr, "k_cache"},
                            {uses_cache ? v_cache : nullptr, "v_cache"}});
  if (st != H3_OK) return st;
  h3::AttnGroupArgs a{};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.kc = static_cast<const __nv_bfloat16*>(k_cache);
  a.vc = static_cast<const __nv_bfloat16*>(v_cache);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.q_stride = q_row_stride;
  a.k_stride = k_row_stride;
  a.v_stride = v_row_stride;
  a.kc_stride = k_cache_row_stride;
  a.vc_stride = v_cache_row_stride;
  a.out_stride = out_row_stride;
  a.groups = groups;
  a.n_groups = n_groups;
  a.n_heads = n_heads;
  a.scale = scale;
  std::string err;
  st = h3::launch_attention_groups(a, reinterpret_cast<cudaStream_t>(stream), err);
  if (st != H3_OK) return fail(st, "%s", err.c_str());
  return H3_OK;
}

}  // extern "C"

namespace {

// Shared checks of one tensor of a block-means call.
int means_tensor(const void* x, int64_t row_stride, const float* means, int n_heads,
                 const char* name) {
  if (row_stride < static_cast<int64_t>(n_heads) * h3::kHeadDim)
    return fail(H3_ERR_SHAPE, "%s row stride must be >= n_heads*128", name);
  if (!x || !means) return fail(H3_ERR_ARG, "null pointer argument (%s)", name);
  if (!aligned16(x) || (row_stride * 2) % 16)
    return fail(H3_ERR_ALIGN, "%s and its row stride must be 16-byte aligned", name);
  if ((reinterpret_cast<uintptr_t>(means) & 3u) != 0)
    return fail(H3_ERR_ALIGN, "the means of %s must be 4-byte aligned", name);
  return H3_OK;
}

int block_means_entry(const void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride,
                      int64_t n_rows, int n_heads, int head_dim, float* q_means, float* k_means,
                      int n_tensors, h3_stream_t stream) {
  if (n_rows < 1 || n_rows > int64_t(h3::kMaxSparseBlocks) * 128)
    return fail(H3_ERR_ARG, "n_rows must be in [1, %d] (got %lld)", h3::kMaxSparseBlocks * 128,
                (long long)n_rows);
  if (n_heads < 1 || n_heads > 65535) return fail(H3_ERR_ARG, "n_heads out of range (%d)", n_heads);
  if (head_dim != h3::kHeadDim) return fail(H3_ERR_SHAPE, "head_dim must be 128 (got %d)", head_dim);
  int st = means_tensor(q, q_row_stride, q_means, n_heads, n_tensors == 2 ? "q" : "x");
  if (st == H3_OK && n_tensors == 2) st = means_tensor(k, k_row_stride, k_means, n_heads, "k");
  if (st != H3_OK) return st;
  if (n_tensors == 2 && q_means == k_means)
    return fail(H3_ERR_ARG, "q_means and k_means must be distinct buffers");
  if ((st = check_device())) return st;
  if ((st = check_device_memory({{q, "q"}, {q_means, "q_means"},
                                 {n_tensors == 2 ? k : nullptr, "k"},
                                 {n_tensors == 2 ? k_means : nullptr, "k_means"}})))
    return st;
  h3::MeansJob job{};
  job.x[0] = static_cast<const __nv_bfloat16*>(q);
  job.stride[0] = q_row_stride;
  job.out[0] = q_means;
  job.x[1] = static_cast<const __nv_bfloat16*>(k);
  job.stride[1] = k_row_stride;
  job.out[1] = k_means;
  cudaError_t e = h3::launch_block_means(job, n_tensors, n_rows, n_heads,
                                         reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(H3_ERR_LAUNCH, "block means launch: %s", cudaGetErrorString(e));
  return H3_OK;
}

}  // namespace

extern "C" {

int h3_block_means(const void* x, int64_t row_stride, int64_t n_rows, int n_heads, int head_dim,
                   float* means, h3_stream_t stream) {
  return block_means_entry(x, row_stride, nullptr, 0, n_rows, n_heads, head_dim, means, nullptr,
                           1, stream);
}

int h3_block_means_qk(const void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride,
                      int64_t n_rows, int n_heads, int head_dim, float* q_means, float* k_means,
                      h3_stream_t stream) {
  return block_means_entry(q, q_row_stride, k, k_row_stride, n_rows, n_heads, head_dim, q_means,
                           k_means, 2, stream);
}

int h3_block_select(const float* q_means, const float* k_means, int n_q_blocks, int n_kv_blocks,
                    int n_heads, float scale, float tau, int n_prefix_blocks, float* scores,
                    int32_t* lists, int32_t* counts, h3_stream_t stream) {
  if (n_q_blocks < 1 || n_q_blocks > 65535 || n_kv_blocks < 1 || n_kv_blocks > h3::kMaxSparseBlocks)
    return fail(H3_ERR_ARG, "block counts out of range (%d, %d; at most 65535 and %d)", n_q_blocks,
                n_kv_blocks, h3::kMaxSparseBlocks);
  if (n_heads < 1 || n_heads > 65535) return fail(H3_ERR_ARG, "n_heads out of range (%d)", n_heads);
  if (!std::isfinite(scale) || !std::isfinite(tau)) return fail(H3_ERR_ARG, "scale and tau must be finite");
  if (n_prefix_blocks < 0 || n_prefix_blocks > n_kv_blocks)
    return fail(H3_ERR_ARG, "n_prefix_blocks must be in [0, %d]", n_kv_blocks);
  if (!q_means || !k_means || !lists || !counts) return fail(H3_ERR_ARG, "null pointer argument");
  if (!aligned16(q_means) || !aligned16(k_means))
    return fail(H3_ERR_ALIGN, "means must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(lists) & 3u) || (reinterpret_cast<uintptr_t>(counts) & 3u) ||
      (scores && (reinterpret_cast<uintptr_t>(scores) & 3u)))
    return fail(H3_ERR_ALIGN, "lists, counts and scores must be 4-byte aligned");
  int st = check_device();
  if (st != H3_OK) return st;
  st = check_device_memory({{q_means, "q_means"}, {k_means, "k_means"}, {scores, "scores"},
                            {lists, "lists"}, {counts, "counts"}});
  if (st != H3_OK) return st;
  cudaError_t e = h3::launch_block_select(q_means, k_means, n_q_blocks, n_kv_blocks, n_heads, scale,
                                          tau, n_prefix_blocks, scores, lists, counts,
                                          reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(H3_ERR_LAUNCH, "block select launch: %s", cudaGetErrorString(e));
  return H3_OK;
}

int h3_sparse_attention(const void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride,
                        const void* v, int64_t v_row_stride, void* out, int64_t out_row_stride,
                        int64_t n_rows, int n_heads, int head_dim, const int32_t* lists,
                        const int32_t* counts, int n_prefix_blocks, float scale,
                        h3_stream_t stream) {
  if (n_rows < 1 || n_rows > int64_t(h3::kMaxSparseBlocks) * 128)
    return fail(H3_ERR_ARG, "n_rows must be in [1, %d] (got %lld)", h3::kMaxSparseBlocks * 128,
                (long long)n_rows);
  if (n_heads < 1) return fail(H3_ERR_ARG, "n_heads must be >= 1 (got %d)", n_heads);
  if (head_dim != h3::kHeadDim) return fail(H3_ERR_SHAPE, "head_dim must be 128 (got %d)", head_dim);
  if (!std::isfinite(scale) || !(scale > 0.0f)) return fail(H3_ERR_ARG, "scale must be finite and > 0");
  const int64_t n_b = (n_rows + 127) / 128;
  if (n_prefix_blocks < 0 || n_prefix_blocks > n_b)
    return fail(H3_ERR_ARG, "n_prefix_blocks must be in [0, %lld] (got %d)", (long long)n_b,
                n_prefix_blocks);
  const int64_t width = static_cast<int64_t>(n_heads) * h3::kHeadDim;
  if (q_row_stride < width || k_row_stride < width || v_row_stride < width || out_row_stride < width)
    return fail(H3_ERR_SHAPE, "row strides must be >= n_heads*128 = %lld", (long long)width);
  if (!q || !k || !v || !out || !lists || !counts) return fail(H3_ERR_ARG, "null pointer argument");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return fail(H3_ERR_ALIGN, "q, k, v, out must be 16-byte aligned");
  if ((q_row_stride * 2) % 16 || (k_row_stride * 2) % 16 || (v_row_stride * 2) % 16 ||
      (out_row_stride * 2) % 16)
    return fail(H3_ERR_ALIGN, "row strides must be multiples of 8 elements (16 bytes)");
  if ((reinterpret_cast<uintptr_t>(lists) & 3u) || (reinterpret_cast<uintptr_t>(counts) & 3u))
    return fail(H3_ERR_ALIGN, "lists and counts must be 4-byte aligned");
  int st = check_device();
  if (st != H3_OK) return st;
  st = check_device_memory({{q, "q"}, {k, "k"}, {v, "v"}, {out, "out"}, {lists, "lists"},
                            {counts, "counts"}});
  if (st != H3_OK) return st;
  h3::SparseAttnArgs a{};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.q_stride = q_row_stride;
  a.k_stride = k_row_stride;
  a.v_stride = v_row_stride;
  a.out_stride = out_row_stride;
  a.n_rows = n_rows;
  a.n_heads = n_heads;
  a.lists = lists;
  a.counts = counts;
  a.scale = scale;
  a.n_prefix_blocks = n_prefix_blocks;
  std::string err;
  st = h3::launch_sparse_attention(a, reinterpret_cast<cudaStream_t>(stream), err);
  if (st != H3_OK) return fail(st, "%s", err.c_str());
  return H3_OK;
}

int h3_wire_record_bytes(int what, int format) {
  if (what == 0) return format == H3_WIRE_BF16 ? 768 : format == H3_WIRE_INT8 ? 400 : -1;
  if (what == 1)
    return format == H3_WIRE_BF16 ? 256 : format == H3_WIRE_INT8 ? 144 : format == H3_WIRE_FP8 ? 128 : -1;
  return -1;
}

}  // extern "C"

namespace {

int wire_rows_heads(int64_t n_rows, int n_heads, int parts) {
  if (n_rows < 0 || n_rows > (int64_t(1) << 40)) return fail(H3_ERR_ARG, "n_rows out of range");
  if (n_heads < 1 || n_heads > 4096) return fail(H3_ERR_ARG, "n_heads out of range (%d)", n_heads);
  if (parts < 1 || n_heads % parts != 0)
    return fail(H3_ERR_ARG, "the part count (%d) must divide n_heads (%d)", parts, n_heads);
  if (n_rows * n_heads >= (int64_t(1) << 31))
    return fail(H3_ERR_ARG, "n_rows * n_heads must be < 2^31");
  return H3_OK;
}

int bf16_tensor(const void* p, int64_t stride, int64_t width, const char* name) {
  if (!p) return fail(H3_ERR_ARG, "%s is NULL", name);
  if (stride < width) return fail(H3_ERR_SHAPE, "%s row stride must be >= %lld", name, (long long)width);
  if ((reinterpret_cast<uintptr_t>(p) & 7u) || (stride * 2) % 8)
    return fail(H3_ERR_ALIGN, "%s and its row stride must be 8-byte aligned", name);
  return H3_OK;
}

}  // namespace

extern "C" {

int h3_pack_qkv(const void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride,
                const void* v, int64_t v_row_stride, int64_t n_rows, int n_heads, int n_dest,
                int format, void* wire, h3_stream_t stream) {
  int st = wire_rows_heads(n_rows, n_heads, n_dest);
  if (st != H3_OK) return st;
  if (format != H3_WIRE_BF16 && format != H3_WIRE_INT8)
    return fail(H3_ERR_ARG, "QKV wire format must be BF16 or INT8 (got %d)", format);
  const int64_t w = static_cast<int64_t>(n_heads) * h3::kHeadDim;
  if ((st = bf16_tensor(q, q_row_stride, w, "q")) || (st = bf16_tensor(k, k_row_stride, w, "k")) ||
      (st = bf16_tensor(v, v_row_stride, w, "v")))
    return st;
  if (format == H3_WIRE_INT8 &&
      (!aligned16(q) || !aligned16(k) || !aligned16(v) || (q_row_stride * 2) % 16 ||
       (k_row_stride * 2) % 16 || (v_row_stride * 2) % 16))
    return fail(H3_ERR_ALIGN, "INT8 packing reads 16-byte vectors: q, k, v and their row "
                              "strides must be 16-byte aligned");
  if (!wire) return fail(H3_ERR_ARG, "wire is NULL");
  if (!aligned16(wire)) return fail(H3_ERR_ALIGN, "wire must be 16-byte aligned");
  if (n_rows == 0) return H3_OK;
  if ((st = check_device())) return st;
  if ((st = check_device_memory({{q, "q"}, {k, "k"}, {v, "v"}, {wire, "wire"}}))) return st;
  h3::WireQkvArgs a{};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.qs = q_row_stride;
  a.ks = k_row_stride;
  a.vs = v_row_stride;
  a.n_rows = n_rows;
  a.n_heads = n_heads;
  a.n_parts = n_dest;
  a.format = format;
  a.wire = static_cast<uint8_t*>(wire);
  cudaError_t e = h3::launch_pack_qkv(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(H3_ERR_LAUNCH, "pack_qkv launch: %s", cudaGetErrorString(e));
  return H3_OK;
}

int h3_unpack_qkv(const void* wire, int64_t n_rows, int n_heads_local, int format, void* q,
                  int64_t q_row_stride, void* k, int64_t k_row_stride, void* v,
                  int64_t v_row_stride, h3_stream_t stream) {
  int st = wire_rows_heads(n_rows, n_heads_local, 1);
  if (st != H3_OK) return st;
  if (format != H3_WIRE_BF16 && format != H3_WIRE_INT8)
    return fail(H3_ERR_ARG, "QKV wire format must be BF16 or INT8 (got %d)", format);
  const int64_t w = static_cast<int64_t>(n_heads_local) * h3::kHeadDim;
  if ((st = bf16_tensor(q, q_row_stride, w, "q")) || (st = bf16_tensor(k, k_row_stride, w, "k")) ||
      (st = bf16_tensor(v, v_row_stride, w, "v")))
    return st;
  if (format == H3_WIRE_INT8 &&
      (!aligned16(q) || !aligned16(k) || !aligned16(v) || (q_row_stride * 2) % 16 ||
       (k_row_stride * 2) % 16 || (v_row_stride * 2) % 16))
    return fail(H3_ERR_ALIGN, "INT8 unpacking writes 16-byte vectors: q, k, v and their row "
                              "strides must be 16-byte aligned");
  if (!wire) return fail(H3_ERR_ARG, "wire is NULL");
  if (!aligned16(wire)) return fail(H3_ERR_ALIGN, "wire must be 16-byte aligned");
  if (n_rows == 0) return H3_OK;
  if ((st = check_device())) return st;
  if ((st = check_device_memory({{wire, "wire"}, {q, "q"}, {k, "k"}, {v, "v"}}))) return st;
  h3::WireQkvArgs a{};
  a.qm = static_cast<__nv_bfloat16*>(q);
  a.km = static_cast<__nv_bfloat16*>(k);
  a.vm = static_cast<__nv_bfloat16*>(v);
  a.qs = q_row_stride;
  a.ks = k_row_stride;
  a.vs = v_row_stride;
  a.n_rows = n_rows;
  a.n_heads = n_heads_local;
  a.n_parts = 1;
  a.format = format;
  a.wire = const_cast<uint8_t*>(static_cast<const uint8_t*>(wire));
  cudaError_t e = h3::launch_unpack_qkv(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(H3_ERR_LAUNCH, "unpack_qkv launch: %s", cudaGetErrorString(e));
  return H3_OK;
}

int h3_pack_out(const void* out, int64_t out_row_stride, int64_t n_rows, int n_heads_local,
                int format, void* wire, h3_stream_t stream) {
  int st = wire_rows_heads(n_rows, n_heads_local, 1);
  if (st != H3_OK) return st;
  if (format != H3_WIRE_BF16 && format != H3_WIRE_INT8 && format != H3_WIRE_FP8)
    return fail(H3_ERR_ARG, "unknown output wire format %d", format);
  if ((st = bf16_tensor(out, out_row_stride, static_cast<int64_t>(n_heads_local) * h3::kHeadDim, "out")))
    return st;
  if (!wire) return fail(H3_ERR_ARG, "wire is NULL");
  if (!aligned16(wire)) return fail(H3_ERR_ALIGN, "wire must be 16-byte aligned");
  if (n_rows == 0) return H3_OK;
  if ((st = check_device())) return st;
  if ((st = check_device_memory({{out, "out"}, {wire, "wire"}}))) return st;
  h3::WireOutArgs a{};
  a.out = static_cast<const __nv_bfloat16*>(out);
  a.os = out_row_stride;
  a.n_rows = n_rows;
  a.n_heads = n_heads_local;
  a.n_parts = 1;
  a.format = format;
  a.wire = static_cast<uint8_t*>(wire);
  cudaError_t e = h3::launch_pack_out(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(H3_ERR_LAUNCH, "pack_out launch: %s", cudaGetErrorString(e));
  return H3_OK;
}

int h3_merge_heads(const void* wire, int64_t n_rows, int n_heads, int n_src, int format, void* out,
                   int64_t out_row_stride, h3_stream_t stream) {
  int st = wire_rows_heads(n_rows, n_heads, n_src);
  if (st != H3_OK) return st;
  if (format != H3_WIRE_BF16 && format != H3_WIRE_INT8 && format != H3_WIRE_FP8)
    return fail(H3_ERR_ARG, "unknown output wire format %d", format);
  if ((st = bf16_tensor(out, out_row_stride, static_cast<int64_t>(n_heads) * h3::kHeadDim, "out")))
    return st;
  if (!wire) return fail(H3_ERR_ARG, "wire is NULL");
  if (!aligned16(wire)) return fail(H3_ERR_ALIGN, "wire must be 16-byte aligned");
  if (n_rows == 0) return H3_OK;
  if ((st = check_device())) return st;
  if ((st = check_device_memory({{wire, "wire"}, {out, "out"}}))) return st;
  h3::WireOutArgs a{};
  a.outm = static_cast<__nv_bfloat16*>(out);
  a.os = out_row_stride;
  a.n_rows = n_rows;
  a.n_heads = n_heads;
  a.n_parts = n_src;
  a.format = format;
  a.wire = const_cast<uint8_t*>(static_cast<const uint8_t*>(wire));
  cudaError_t e = h3::launch_merge_heads(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(H3_ERR_LAUNCH, "merge_heads launch: %s", cudaGetErrorString(e));
  return H3_OK;
}

int h3_copy_2d(void* dst, int64_t dst_pitch, const void* src, int64_t src_pitch,
               int64_t width_bytes, int64_t height, h3_stream_t stream) {
  if (height < 0 || width_bytes < 0) return fail(H3_ERR_ARG, "negative copy extent");
  if (height == 0 || width_bytes == 0) return H3_OK;
  if (!dst || !src) return fail(H3_ERR_ARG, "dst and src must not be NULL");
  if (dst_pitch < width_bytes || src_pitch < width_bytes)
    return fail(H3_ERR_SHAPE, "pitches (%lld, %lld) must be >= the width (%lld)",
                (long long)dst_pitch, (long long)src_pitch, (long long)width_bytes);
  const cudaError_t e =
      cudaMemcpy2DAsync(dst, static_cast<size_t>(dst_pitch), src, static_cast<size_t>(src_pitch),
                        static_cast<size_t>(width_bytes), static_cast<size_t>(height),
                        cudaMemcpyDefault, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(H3_ERR_LAUNCH, "2-D copy: %s", cudaGetErrorString(e));
  return H3_OK;
}

int h3_status_word(uint32_t* out) {
  if (!out) return fail(H3_ERR_ARG, "out must not be NULL");
  cudaError_t e = h3::read_and_clear_status(out);
  if (e != cudaSuccess) return fail(H3_ERR_DEVICE, "status read: %s", cudaGetErrorString(e));
  if (*out != 0u)
    return fail(H3_ERR_TIMEOUT, "a bounded device wait gave up (status bits 0x%x)", *out);
  return H3_OK;
}

int h3_debug_fault_next_attention(int fault) {
  if (fault < 0 || fault > 1) return fail(H3_ERR_ARG, "unknown fault %d", fault);
  h3::set_fault_next(fault);
  return H3_OK;
}

}  // extern "C"
