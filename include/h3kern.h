/*
 * h3kern -- packed-sequence attention and its fused Q/K RMSNorm + axial RoPE
 * prologue for one DiT block of the MiniMax-H3 joint audio/video model,
 * hand-written for sm_103a (GB300).
 *
 * C ABI: plain pointers and sizes.  Every call is asynchronous on the
 * caller's CUDA stream, allocates no device memory and holds no reference
 * to the caller's buffers after it returns.  The caller owns all device
 * buffers and the stream.
 *
 * Tensor layout ("flat (total, heads, head_dim)", Sol-H3 arXiv 2609.35110,
 * section 3.2 "Optimized attention collectives"): a tensor is
 * [rows, n_heads, 128] bf16 with the 128 channels of a head contiguous,
 * heads 128 elements apart, and rows `row_stride` ELEMENTS apart
 * (row_stride >= n_heads * 128), so that views into a packed
 * [rows, 3, n_heads, 128] QKV buffer can be passed without a copy.
 *
 * Errors: arguments are checked on the host before any launch; a failed
 * check returns a negative status and launches nothing.  Besides the checks
 * each call lists, every pointer a kernel reads or writes is queried with
 * cudaPointerGetAttributes and must be memory of the current device (or
 * managed memory): host memory, pinned or not, and another GPU's memory are
 * rejected with H3_ERR_ARG.  The library never aborts or exits.  The message
 * of the last nonzero status of the calling thread is available from
 * h3_last_error().
 */
#ifndef H3KERN_H
#define H3KERN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* h3_stream_t; /* a cudaStream_t; NULL = legacy default stream */

enum {
  H3_OK = 0,
  H3_ERR_ARG = -1,     /* null or non-device pointer, bad count, non-finite scalar,
                          bad cu_seqlens */
  H3_ERR_ALIGN = -2,   /* base pointer or row stride not 16-byte aligned */
  H3_ERR_SHAPE = -3,   /* head_dim != 128, row stride too small, bad rotary split */
  H3_ERR_ARCH = -4,    /* current device is not compute capability 10.3 (sm_103) */
  H3_ERR_LAUNCH = -5,  /* the kernel launch itself failed */
  H3_ERR_TIMEOUT = -6, /* a bounded device-side wait gave up (see h3_status_word) */
  H3_ERR_DEVICE = -7   /* CUDA runtime / driver error outside a launch */
};

/* Most segments (packed sequences or query groups) one h3_attention call takes. */
#define H3_MAX_SEGMENTS 16

/* Bits of the device status word (h3_status_word). */
#define H3_STATUS_TIMEOUT_LOAD 0x1u   /* producer gave up waiting for a free K/V stage */
#define H3_STATUS_TIMEOUT_MMA 0x2u    /* MMA issuer gave up waiting for data or P */
#define H3_STATUS_TIMEOUT_SOFTMAX 0x4u/* softmax warps gave up waiting for S or O */
#define H3_STATUS_ABORTED 0x8u        /* a CTA stopped early because another gave up */
#define H3_STATUS_TIMEOUT_PROLOGUE 0x10u /* the Q/K prologue gave up waiting for a row */

/*
 * h3_qk_norm_rope -- fused Q/K RMSNorm + axial 3-D RoPE, in place, one pass.
 *
 * Follows "QK normalization with partial RoPE" (Sol-H3, section 3.5 "Kernel
 * Fusion", operator group 2) and the fused Q/K RMSNorm + RoPE of the vLLM-Omni
 * blog (section 3.2).  For every row r < n_rows and head h, with x the 128
 * channels of q[r, h] (and likewise k[r, h] with wk):
 *
 *   y_c  = x_c / sqrt(mean_c(x_c^2) + eps) * w[h, c]            (fp32)
 *   the channels are split into sections t = [0, rot_t),
 *   h = [rot_t, rot_t + rot_h), w = [rot_t + rot_h, rot_t + rot_h + rot_w);
 *   pair j of a section of width d is channels (off + 2j, off + 2j + 1),
 *   turned by phi = pos_thw[r, a] * theta^(-2j/d):
 *   (y0, y1) -> (y0 cos phi - y1 sin phi, y0 sin phi + y1 cos phi);
 *   channels past rot_t + rot_h + rot_w are only normalised;
 *   the result is rounded once to bf16 (round-to-nearest-even) and stored
 *   over x.
 *
 * q, k        device bf16 [n_rows, n_heads, 128], row strides in elements;
 *             modified in place; q and k must not overlap.
 * wq, wk      device bf16 [n_heads, 128], per-head norm weights.
 * pos_thw     device int32 [n_rows, 3]: (t, h, w) position of each row.
 * n_rows      rows to process (0 = nothing to do); typically the valid rows.
 * head_dim    must be 128.
 * n_heads     1 .. 448 (two staged rows must fit in shared memory).
 * rot_t/h/w   even, >= 0, rot_t + rot_h + rot_w <= 128 (the configs use 32/48/48).
 * theta       RoPE base (> 0, finite); eps >= 0, finite.
 * Alignment:  q, k, wq, wk 16-byte aligned; row strides * 2 bytes a multiple of 16;
 *             pos_thw 4-byte aligned.
 * Returns H3_OK or a negative status.
 */
int h3_qk_norm_rope(void* q, int64_t q_row_stride, void* k, int64_t k_row_stride,
                    const void* wq, const void* wk, const int32_t* pos_thw,
                    int64_t n_rows, int n_heads, int head_dim,
                    int rot_t, int rot_h, int rot_w, float theta, float eps,
                    h3_stream_t stream);

/*
 * h3_qk_norm_rope_varlen -- the same prologue over the valid rows of several
 * packed sequences, in one launch.
 *
 * The vLLM-Omni blog (section 3.1) denoises text, audio and video tokens as
 * one packed sequence whose valid rows are followed by padding up to an
 * aligned length.  Several such sequences may sit back to back in one buffer,
 * in the layout h3_attention takes: sequence b is buffer rows
 * [cu_seqlens[b], cu_seqlens[b + 1]), of which the first valid_len[b] are
 * valid, and the prologue applies to those.  Each of those rows is processed
 * exactly as by h3_qk_norm_rope (bitwise the same result); other rows are not
 * read or written.  One persistent launch covers all sequences, so they pay
 * one launch tail instead of one per sequence.
 *
 * q, k        device bf16 [cu_seqlens[n_seq], n_heads, 128], row strides in elements.
 * pos_thw     device int32 [cu_seqlens[n_seq], 3], indexed by buffer row.
 * cu_seqlens  HOST int32 [n_seq + 1], cu_seqlens[0] == 0, non-decreasing.
 * valid_len   HOST int32 [n_seq], 0 <= valid_len[b] <= cu_seqlens[b + 1] - cu_seqlens[b];
 *             NULL = every row of every sequence is valid.
 * n_seq       1 .. H3_MAX_SEGMENTS; the valid rows sum to at most 2^30.
 * All other arguments, alignment rules and errors as h3_qk_norm_rope.  The
 * host arrays are read before the call returns.
 */
int h3_qk_norm_rope_varlen(void* q, int64_t q_row_stride, void* k, int64_t k_row_stride,
                           const void* wq, const void* wk, const int32_t* pos_thw,
                           const int32_t* cu_seqlens, const int32_t* valid_len, int n_seq,
                           int n_heads, int head_dim, int rot_t, int rot_h, int rot_w,
                           float theta, float eps, h3_stream_t stream);

/*
 * h3_qk_norm_rope_lora -- the same fused prologue as a LoRA consumer.
 *
 * Follows "Precision-preserving LoRA fusion" (Sol-H3, section 3.5): the base
 * projection and the LoRA branch output stay separate tensors, and the
 * consumer rounds base + delta to bf16 (fp32 sum, round-to-nearest-even)
 * before the QK normalisation and RoPE, exactly where separate branches
 * would have stored the sum.  The result is therefore bit-identical to
 * adding the branches into a bf16 tensor first and then calling
 * h3_qk_norm_rope, without the wide sum's HBM write and re-read.
 *
 * q, k        device bf16 [n_rows, n_heads, 128]: the base branch on input,
 *             the normalised + rotated result on output (in place).
 * q_delta, k_delta
 *             device bf16 [n_rows, n_heads, 128] LoRA branch outputs, read only;
 *             their row strides are in elements.
 * n_heads     1 .. 220 (two staged rows of base + delta must fit in shared memory).
 * All other arguments, alignment rules and errors as h3_qk_norm_rope; the
 * delta pointers and strides follow the same 16-byte rules.
 */
int h3_qk_norm_rope_lora(void* q, int64_t q_row_stride, const void* q_delta,
                         int64_t q_delta_row_stride, void* k, int64_t k_row_stride,
                         const void* k_delta, int64_t k_delta_row_stride, const void* wq,
                         const void* wk, const int32_t* pos_thw, int64_t n_rows, int n_heads,
                         int head_dim, int rot_t, int rot_h, int rot_w, float theta, float eps,
                         h3_stream_t stream);

/*
 * h3_attention -- non-causal softmax(Q K^T * scale) V over packed sequences
 * or grouped query ranges, in one launch.
 *
 * Follows the packed joint sequence with a valid length (vLLM-Omni blog,
 * section 3.1: the attention backend receives the valid sequence length and
 * the structural suffix padding costs nothing) and the grouped condition /
 * audio / video query ranges over different KV extents of a contiguous
 * history cache (SolarWM-H3 Realtime blog, stages 2 and 3).
 *
 * Segment b (0 <= b < n_seq) owns query rows [cu_seqlens_q[b], cu_seqlens_q[b+1])
 * of q and out, and key/value rows [cu_seqlens_kv[b], cu_seqlens_kv[b+1]) of
 * k and v.  If valid_len is non-NULL only the first valid_len[b] rows of both
 * ranges are valid (self-attention over one padded buffer); otherwise every
 * row of both ranges is.  For each valid query row i and head h:
 *   out[i, h] = sum_j softmax_j(scale * <q[i, h], k[j, h]>) v[j, h]
 * over the segment's valid key rows j.  Output rows past the valid length,
 * and all rows of a segment with no valid key, are written as 0.  Padded
 * input rows are never read, so they may hold anything (NaN, Inf).
 *
 * q, out      device bf16 [cu_seqlens_q[n_seq], n_heads, 128]
 * k, v        device bf16 [cu_seqlens_kv[n_seq], n_heads, 128]
 * cu_seqlens_q, cu_seqlens_kv
 *             HOST int32 [n_seq + 1], start at 0, non-decreasing.
 * valid_len   HOST int32 [n_seq] or NULL; 0 <= valid_len[b] <= both extents.
 * n_seq       1 .. H3_MAX_SEGMENTS.
 * scale       > 0 and finite (1/sqrt(128) for the DiT block).
 * Alignment:  all four base pointers 16-byte aligned; row strides * 2 a
 *             multiple of 16.  out must not overlap q, k or v.
 * The host arrays are read during the call only, so the call can be
 * captured in a CUDA graph.
 * Returns H3_OK or a negative status.
 */
int h3_attention(const void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride,
                 const void* v, int64_t v_row_stride, void* out, int64_t out_row_stride,
                 const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                 const int32_t* valid_len, int n_seq, int n_heads, int head_dim,
                 float scale, h3_stream_t stream);

/*
 * h3_attention_groups -- query groups over KV views, including a cached KV
 * range, in one launch.
 *
 * Follows the reference KV caching of Sol-H3 (section 5, Fig. 4): after the
 * first denoising step the reference query rows are skipped and the text /
 * generation queries attend to the cached reference K/V together with the
 * current tokens' K/V; and the history K/V reuse of the SolarWM-H3 Realtime
 * blog (stage 3), where query groups read a pre-concatenated history.
 *
 * Group g: query rows [q_start, q_start + q_len) of q and out attend to the
 * union of k / v rows [kv_start, kv_start + kv_len) and k_cache / v_cache
 * rows [cache_start, cache_start + cache_len):
 *   out[i, h] = sum_j softmax_j(scale * <q[i, h], key_j[h]>) value_j[h]
 * KV views may overlap between groups; query ranges must not.  Output rows
 * that belong to no group (for instance skipped reference queries) are not
 * written; a group whose two views are both empty writes zeros.
 *
 * q, out          device bf16 [rows, n_heads, 128]
 * k, v            device bf16, rows as addressed by kv_start/kv_len
 * k_cache, v_cache device bf16, rows as addressed by cache_start/cache_len;
 *                 may be NULL when every cache_len is 0
 * groups          HOST array of n_groups entries, 1 <= n_groups <= H3_MAX_SEGMENTS;
 *                 all fields >= 0, start + len < 2^31.
 * The caller guarantees that every addressed row exists.  Alignment, scale
 * and error rules as h3_attention.
 */
typedef struct {
  int32_t q_start, q_len;
  int32_t kv_start, kv_len;
  int32_t cache_start, cache_len;
} h3_attn_group;

int h3_attention_groups(const void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride,
                        const void* v, int64_t v_row_stride, const void* k_cache,
                        int64_t k_cache_row_stride, const void* v_cache,
                        int64_t v_cache_row_stride, void* out, int64_t out_row_stride,
                        const h3_attn_group* groups, int n_groups, int n_heads, int head_dim,
                        float scale, h3_stream_t stream);

/*
 * Sol-Attn block-sparse attention (Sol-H3, section 3.4 "Per-step dynamic
 * sparsity" and "Safety rails and the exact prefix KV sink"), in three
 * stages over one packed sequence of n_rows rows, blocks of 128 rows
 * (n_b = ceil(n_rows / 128) <= 2048, the last block may be partial):
 *
 *   h3_block_means    q_means, k_means = per-block mean rows of Q and K;
 *   h3_block_select   per head and query block a, score(a, b) =
 *                     scale * <q_means[a], k_means[b]>; KV block b is kept when
 *                     score > mean_b(score) + tau * std_b(score) (population
 *                     std), or b < n_prefix_blocks (prefix sink), or
 *                     a < n_prefix_blocks (prefix queries are dense);
 *   h3_sparse_attention  exact softmax attention of each query row over the
 *                     keys of the blocks its query block keeps.
 *
 * The pages leave "block-level score" undefined; the block-mean dot product
 * above is the reading taken.  A block holding any prefix row counts as a
 * prefix block (n_prefix_blocks = ceil(prefix rows / 128)).
 */

/* x: device bf16 [n_rows, n_heads, 128] (row stride in elements, 16-byte
 * aligned); means: device fp32 [n_b, n_heads, 128], 4-byte aligned.  Each
 * mean is an fp32 sum in a fixed order divided by the block's row count
 * (deterministic run to run). */
int h3_block_means(const void* x, int64_t row_stride, int64_t n_rows, int n_heads, int head_dim,
                   float* means, h3_stream_t stream);

/* The block means of Q and of K in one launch: q -> q_means, k -> k_means,
 * each as h3_block_means (same results bit for bit); the two means buffers
 * must be distinct. */
int h3_block_means_qk(const void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride,
                      int64_t n_rows, int n_heads, int head_dim, float* q_means, float* k_means,
                      h3_stream_t stream);

/* q_means [n_q_blocks, n_heads, 128], k_means [n_kv_blocks, n_heads, 128]
 * (device fp32, 16-byte aligned; n_kv_blocks <= 2048).  Outputs (device,
 * 4-byte aligned): lists int32 [n_heads, n_q_blocks, n_kv_blocks], row (h, a)
 * holding the kept KV blocks in ascending order in its first counts[h, a]
 * entries; counts int32 [n_heads, n_q_blocks]; scores fp32 [n_heads,
 * n_q_blocks, n_kv_blocks] or NULL.  Arithmetic is fp32 in a fixed order
 * (the selection is deterministic). */
int h3_block_select(const float* q_means, const float* k_means, int n_q_blocks, int n_kv_blocks,
                    int n_heads, float scale, float tau, int n_prefix_blocks, float* scores,
                    int32_t* lists, int32_t* counts, h3_stream_t stream);

/* q, k, v, out: device bf16 [>= n_rows, n_heads, 128] as in h3_attention;
 * lists / counts as h3_block_select writes them for this sequence
 * (n_q_blocks = n_kv_blocks = n_b).  Rows of a query block that keeps no
 * block are written as 0; rows >= n_rows are not written.  List entries
 * outside [0, n_b) are ignored.
 * n_prefix_blocks (0 .. n_b) is a scheduling hint, the value given to
 * h3_block_select: the prefix query blocks keep every KV block, so their
 * tiles take several times longer than the others and are scheduled first.
 * It never changes the output (0 = no hint). */
int h3_sparse_attention(const void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride,
                        const void* v, int64_t v_row_stride, void* out, int64_t out_row_stride,
                        int64_t n_rows, int n_heads, int head_dim, const int32_t* lists,
                        const int32_t* counts, int n_prefix_blocks, float scale,
                        h3_stream_t stream);

/*
 * Wire formats at the attention boundary (Sol-H3, section 3.2 "Optimized
 * attention collectives" and "Quantized communication").  On one GPU there
 * is no exchange; these calls produce and consume the exchange buffers a
 * sequence-parallel (Ulysses) all-to-all would move.
 *
 *   QKV records, one per (token, head):   H3_WIRE_BF16  768 B  q|k|v bf16
 *                                          H3_WIRE_INT8  400 B  q|k|v int8 (384 B),
 *                                                        12 scale codes, 4 zero bytes
 *   output records, one per (token, head): H3_WIRE_BF16  256 B  bf16
 *                                          H3_WIRE_INT8  144 B  128 int8, 4 codes, 12 zeros
 *                                          H3_WIRE_FP8   128 B  E4M3, RNE, saturated +-448
 * Scale codes are UE5M3 (read as: 5 exponent bits, bias 15, 3 mantissa bits,
 * every code finite and positive, value = 2^(e-15) * (1 + m/8)), one per 32
 * channels; a group takes the smallest code with 127 * value >= max|x| and
 * stores rint(x / value).  INT8 and FP8 are approximate; BF16 records are a
 * pure permutation (bit-exact).  Wire buffers are device memory, 16-byte
 * aligned; sizes per record from h3_wire_record_bytes.  Tensors are bf16
 * device memory with 8-byte aligned bases and row strides; n_rows >= 0 and
 * n_rows * n_heads < 2^31 (more records than device memory holds), else
 * H3_ERR_ARG; n_rows == 0 launches nothing.
 * Values are expected finite (a NaN does not raise the group's scale).
 */
enum { H3_WIRE_BF16 = 0, H3_WIRE_INT8 = 1, H3_WIRE_FP8 = 2 };

/* Bytes of one record: what = 0 for QKV, 1 for the attention output; -1
 * for a combination that does not exist (FP8 QKV). */
int h3_wire_record_bytes(int what, int format);

/* q, k, v [n_rows, n_heads, 128] (own row strides) -> wire
 * [n_dest][n_rows][n_heads / n_dest] QKV records, destination d holding heads
 * d * n_heads / n_dest ...; n_dest divides n_heads.  Format BF16 or INT8;
 * INT8 needs q, k, v and their row strides 16-byte aligned (H3_ERR_ALIGN
 * otherwise). */
int h3_pack_qkv(const void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride,
                const void* v, int64_t v_row_stride, int64_t n_rows, int n_heads, int n_dest,
                int format, void* wire, h3_stream_t stream);

/* wire [n_rows][n_heads_local] QKV records -> q, k, v [n_rows, n_heads_local, 128]
 * (INT8 values decoded and rounded to bf16).  INT8 needs q, k, v and their
 * row strides 16-byte aligned (H3_ERR_ALIGN otherwise). */
int h3_unpack_qkv(const void* wire, int64_t n_rows, int n_heads_local, int format, void* q,
                  int64_t q_row_stride, void* k, int64_t k_row_stride, void* v,
                  int64_t v_row_stride, h3_stream_t stream);

/* out [n_rows, n_heads_local, 128] -> wire [n_rows][n_heads_local] output records. */
int h3_pack_out(const void* out, int64_t out_row_stride, int64_t n_rows, int n_heads_local,
                int format, void* wire, h3_stream_t stream);

/* Inverse head merge: wire [n_src][n_rows][n_heads / n_src] output records
 * -> out [n_rows, n_heads, 128]; n_src divides n_heads. */
int h3_merge_heads(const void* wire, int64_t n_rows, int n_heads, int n_src, int format, void* out,
                   int64_t out_row_stride, h3_stream_t stream);

/*
 * Strided transfer helper (not a step of the method): copies `height` rows
 * of `width_bytes` bytes from src (row pitch src_pitch bytes) to dst (row
 * pitch dst_pitch bytes), asynchronously on `stream`, in whichever direction
 * the two addresses imply (host <-> device or device <-> device).  Used to
 * move a group of heads of a [rows, heads, 128] tensor between pinned host
 * memory and the device while other heads are being computed.  Host memory
 * must be pinned for the copy to be asynchronous.  Returns H3_ERR_ARG for a
 * NULL pointer or a negative extent, H3_ERR_SHAPE for a pitch below the
 * width, H3_ERR_LAUNCH when the runtime rejects the copy; an empty copy
 * returns H3_OK without touching either pointer.
 */
int h3_copy_2d(void* dst, int64_t dst_pitch, const void* src, int64_t src_pitch,
               int64_t width_bytes, int64_t height, h3_stream_t stream);

/* Message for the last nonzero status returned to the calling thread
 * ("" if none).  The pointer stays valid until the thread's next call. */
const char* h3_last_error(void);

/*
 * Synchronise the current device, copy the device status word (an OR of
 * H3_STATUS_* bits set by kernels whose bounded waits gave up) to *out and
 * clear it.  Returns H3_OK when no bit was set, H3_ERR_TIMEOUT when some
 * were (the output of those launches is undefined), H3_ERR_ARG for a NULL
 * out, or H3_ERR_DEVICE.
 */
int h3_status_word(uint32_t* out);

/* Library version, major * 10000 + minor * 100 + patch. */
int h3_version(void);

#ifdef __cplusplus
}
#endif

#endif /* H3KERN_H */
