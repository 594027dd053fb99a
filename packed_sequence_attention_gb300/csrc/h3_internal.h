// Internal interface between the C-ABI front end (api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "h3kern.h"

namespace h3 {

constexpr int kHeadDim = 128;
// Block-sparse mode: blocks (and attention tiles) of 128 rows; at most
// kMaxSparseBlocks blocks per sequence (262,144 rows).
constexpr int kMaxSparseBlocks = 2048;

// ---------------------------------------------------------------- prologue
// Packed sequences one prologue launch covers at most.
constexpr int kPrologueMaxSegments = H3_MAX_SEGMENTS;

struct NormRopeArgs {
  __nv_bfloat16* q;
  __nv_bfloat16* k;
  int64_t q_stride, k_stride;  // elements
  const __nv_bfloat16* wq;
  const __nv_bfloat16* wk;
  const int32_t* pos;          // indexed by buffer row
  // The rows to process: segment b is buffer rows [seg_row0[b], seg_row0[b] + seg_rows[b]).
  const int64_t* seg_row0;     // host [n_seg]
  const int64_t* seg_rows;     // host [n_seg]
  int n_seg;
  int n_heads;
  int rot[3];
  float theta, eps;
  const __nv_bfloat16* dq = nullptr;  // LoRA deltas (both null: plain prologue)
  const __nv_bfloat16* dk = nullptr;
  int64_t dq_stride = 0, dk_stride = 0;
};
// Validated arguments -> one launch on `stream`.
cudaError_t launch_qk_norm_rope(const NormRopeArgs& a, cudaStream_t stream);
// Largest n_heads the prologue's shared-memory ring holds.
int prologue_max_heads(bool lora);
// Device address of the status word on the current device (nullptr on error).
uint32_t* status_word_device_ptr();

// --------------------------------------------------------------- attention
struct AttnArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  __nv_bfloat16* out;
  int64_t q_stride, k_stride, v_stride, out_stride;  // elements
  const int32_t* cu_q;   // host [n_seq + 1]
  const int32_t* cu_kv;  // host [n_seq + 1]
  const int32_t* valid;  // host [n_seq] or nullptr
  int n_seq, n_heads;
  float scale;
};
// Validated arguments -> tensor maps, schedule, one launch.  Returns an
// H3_* status and fills `err` on failure.
int launch_attention(const AttnArgs& a, cudaStream_t stream, std::string& err);

struct AttnGroupArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const __nv_bfloat16* kc;  // cached K/V (may be null when no group uses them)
  const __nv_bfloat16* vc;
  __nv_bfloat16* out;
  int64_t q_stride, k_stride, v_stride, kc_stride, vc_stride, out_stride;  // elements
  const h3_attn_group* groups;  // host [n_groups]
  int n_groups, n_heads;
  float scale;
};
int launch_attention_groups(const AttnGroupArgs& a, cudaStream_t stream, std::string& err);

// ------------------------------------------------------------ block sparse
// Block means of one or two tensors (x[0] -> out[0], x[1] -> out[1]) in one launch.
struct MeansJob {
  const __nv_bfloat16* x[2];
  int64_t stride[2];  // elements
  float* out[2];
};
cudaError_t launch_block_means(const MeansJob& job, int n_tensors, int64_t n_rows, int H,
                               cudaStream_t stream);
cudaError_t launch_block_select(const float* qm, const float* km, int nqb, int nkb, int H,
                                float scale, float tau, int n_prefix, float* scores,
                                int32_t* lists, int32_t* counts, cudaStream_t stream);
struct SparseAttnArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  __nv_bfloat16* out;
  int64_t q_stride, k_stride, v_stride, out_stride;
  int64_t n_rows;
  int n_heads;
  const int32_t* lists;   // device [H, nb, nb]
  const int32_t* counts;  // device [H, nb]
  float scale;
  int n_prefix_blocks;    // scheduling hint: dense prefix query blocks
};
int launch_sparse_attention(const SparseAttnArgs& a, cudaStream_t stream, std::string& err);

// ------------------------------------------------------------ wire formats
struct WireQkvArgs {
  const __nv_bfloat16 *q, *k, *v;  // pack: sources
  __nv_bfloat16 *qm, *km, *vm;     // unpack: destinations
  int64_t qs, ks, vs;              // row strides (elements)
  int64_t n_rows;
  int n_heads;   // pack: all heads; unpack: heads in the records
  int n_parts;   // pack: destinations
  int format;
  uint8_t* wire;
};
struct WireOutArgs {
  const __nv_bfloat16* out;  // pack: source [rows][n_heads][128]
  __nv_bfloat16* outm;       // merge: destination [rows][n_heads][128]
  int64_t os;
  int64_t n_rows;
  int n_heads;  // pack: heads in the records; merge: all heads
  int n_parts;  // merge: sources
  int format;
  uint8_t* wire;
};
cudaError_t launch_pack_qkv(const WireQkvArgs& a, cudaStream_t s);
cudaError_t launch_unpack_qkv(const WireQkvArgs& a, cudaStream_t s);
cudaError_t launch_pack_out(const WireOutArgs& a, cudaStream_t s);
cudaError_t launch_merge_heads(const WireOutArgs& a, cudaStream_t s);

// Device status word: read (after a device synchronise) and clear.
cudaError_t read_and_clear_status(uint32_t* out);

}  // namespace h3
