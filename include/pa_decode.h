/*
 * pa_decode.h -- C ABI of the GB300 (sm_103a) paged-attention decode library
 * (libpa_decode.so).
 *
 * What the library computes.  For every sequence s, query position i < qlen and
 * query head h (KV head hkv = h / G, G = num_q_heads / num_kv_heads):
 *
 *     out[s,i,h,:] = sum_{t < L_s} softmax_t(x_t) * v_t,
 *     x_t = softmax_scale * q_scale * <q[s,i,h,:], k_t>,
 *
 * where token t of sequence s lives in page block_tables[s, t / page_size], slot
 * t mod page_size, and L_s = context_lens[s].  By default queries are not causally
 * masked (every query position sees all L_s tokens); `causal` and `sliding_window` in
 * pa_decode_args restrict what each query position sees.  References: "[FlyDSL] pa_decode:
 * zero V rows past the context before PV" (Root cause, Fix) and "[FlyDSL]
 * pa_decode: MXFP4 K/V in the shared PA tile kernel" (Summary, Self-Review).
 *
 * The work is cut into 256-token tiles (ceil(L_s / 256) per sequence); a plan
 * groups consecutive tiles of one (sequence, KV head) into tasks, one task per
 * partition of the context.  Tasks write partial (max, sum, output) triples
 * that pa_decode_reduce merges; a sequence with a single partition is written
 * directly.  Rows at or past L_s -- padded block-table columns pointing at any
 * block and the unwritten tail of the last page -- never reach the output,
 * whatever bytes they hold (NaN, Inf, e8m0 255): on the boundary tile their
 * scores are replaced by -inf and their V values and per-token scales by 0.
 *
 * Conventions
 *   - Every pointer in pa_decode_args is a DEVICE pointer; the caller owns all
 *     memory, including the workspace.  The library allocates nothing.
 *   - Calls never synchronise with the host and are stream-ordered on the given
 *     stream (a cudaStream_t passed as void*; NULL is the legacy default
 *     stream).  Arguments are validated on the host before any launch; a
 *     refused call launches nothing and returns a negative pa_status.
 *   - Strides are in ELEMENTS for query/output/block tables and in BYTES for the
 *     caches and scale caches.  The head_dim axis of query and output is
 *     contiguous; one token row of a cache is contiguous (row_bytes below).
 *
 * Storage formats (kv_dtype, kv_scale):
 *   PA_KV_BF16     + PA_SCALE_NONE        key/value bf16 [NB, Hkv, S, D]
 *   PA_KV_FP8_E4M3 + PA_SCALE_PER_TENSOR  key/value OCP e4m3 bytes [NB, Hkv, S, D];
 *                                         key_scale/value_scale fp32 [1]
 *   PA_KV_FP8_E4M3 + PA_SCALE_PER_TOKEN   as above; key_scale/value_scale fp32
 *                                         [NB, Hkv, S] (one per token and KV head)
 *   PA_KV_MXFP4    + PA_SCALE_E8M0_32     key/value uint8 [NB, Hkv, S, D/2], two e2m1
 *                                         per byte (element 2j in the low nibble);
 *                                         key_scale/value_scale uint8 e8m0
 *                                         [NB, Hkv, S, D/32], 2^(b-127) per 32 values
 *   ("[FlyDSL] pa_decode: MXFP4 K/V ...", Summary: the MXFP4 page layout.)
 *   row_bytes = 2D (bf16), D (e4m3), D/2 (MXFP4).  q_dtype PA_Q_BF16 reads a bf16
 *   query exactly; PA_Q_FP8_E4M3 reads e4m3 bytes multiplied by q_scale (fp32 [1], or
 *   [B, qlen, Hq] when q_scale_per_row != 0); PA_Q_BF16_TO_E4M3 (MXFP4 KV only) reads a
 *   bf16 query and quantises each head row in the kernel as the MXFP4 page does
 *   ("[FlyDSL] pa_decode: MXFP4 K/V ...", Summary): s = amax / 448 and y = q / s in fp32
 *   (round to nearest), y rounded to the nearest e4m3 (ties to even, saturating at
 *   448), used as e4m3(y) * s; q_scale is not read.
 *
 * Supported shapes (others return PA_ERR_UNSUPPORTED): head_dim 64, 128 or 256
 * (MXFP4: 128); page_size 16, 32, 64, 128 or 256; G * qlen <= 64 (MXFP4: <= 16,
 * qlen 1); kv_stride_token == row_bytes; 16-byte aligned cache, scale and
 * stride values.  fp8 per-tensor caches may store V transposed (`trans_v`).
 */
#ifndef PA_DECODE_H_
#define PA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t pa_status;
#define PA_OK 0
#define PA_ERR_INVALID_ARG (-1)   /* malformed argument: null pointer, bad shape */
#define PA_ERR_UNSUPPORTED (-2)   /* well-formed, but not a combination the library serves */
#define PA_ERR_WORKSPACE (-3)     /* workspace missing, too small or misaligned */
#define PA_ERR_CUDA (-4)          /* a CUDA runtime call or launch failed */

#define PA_KV_BF16 0
#define PA_KV_FP8_E4M3 1
#define PA_KV_MXFP4 2

#define PA_SCALE_NONE 0
#define PA_SCALE_PER_TENSOR 1
#define PA_SCALE_PER_TOKEN 2
#define PA_SCALE_E8M0_32 3

#define PA_Q_BF16 0
#define PA_Q_FP8_E4M3 1
#define PA_Q_BF16_TO_E4M3 2

/* Device status word (first int32 of the workspace), read with pa_decode_read_status. */
#define PA_DEVICE_OK 0
#define PA_DEVICE_WAIT_TIMEOUT 1     /* a pipeline wait gave up; the output is not valid */
#define PA_DEVICE_CONTEXT_CLAMPED 2  /* a context length exceeded the block table width */

typedef struct pa_decode_args {
  /* shapes */
  int32_t batch;              /* B >= 0 sequences */
  int32_t qlen;               /* query tokens per sequence, >= 1 */
  int32_t num_q_heads;        /* Hq, a multiple of num_kv_heads */
  int32_t num_kv_heads;       /* Hkv >= 1 */
  int32_t head_dim;           /* D */
  int32_t page_size;          /* S, tokens per cache block */
  int32_t num_blocks;         /* NB, blocks in each cache */
  int32_t max_blocks_per_seq; /* block-table width W; context lengths are clamped to W*S */
  /* formats */
  int32_t kv_dtype;           /* PA_KV_* */
  int32_t kv_scale;           /* PA_SCALE_* */
  int32_t q_dtype;            /* PA_Q_* */
  int32_t q_scale_per_row;    /* e4m3 query: 0 = q_scale[1], 1 = q_scale[B*qlen*Hq] */
  float softmax_scale;        /* <= 0 selects 1/sqrt(head_dim) */
  /* work split */
  int32_t max_partitions;     /* >= 1 caps partitions per (sequence, KV head) (at most 128);
                                 1 = direct output, no reduce; <= 0 picks 128 */
  int32_t task_budget;        /* work chunks = tile-kernel CTAs; <= 0 picks the SM count */
  int32_t merge_in_decode;    /* 1: pa_decode merges the partitions of split units itself
                                 (the last task of a unit to finish does it) and
                                 pa_decode_reduce launches nothing; 0: pa_decode_reduce merges */
  /* tensors (device pointers) */
  const void* query;          /* [B*qlen, Hq, D] bf16 or e4m3 */
  int64_t q_stride_token;     /* elements between consecutive (s, i) rows */
  int64_t q_stride_head;      /* elements between consecutive heads */
  const float* q_scale;       /* e4m3 query only, else may be NULL */
  const void* key_cache;
  const void* value_cache;
  int64_t kv_stride_block;    /* bytes between blocks (both caches) */
  int64_t kv_stride_head;     /* bytes between KV heads within a block */
  int64_t kv_stride_token;    /* bytes between token rows; must equal row_bytes */
  const void* key_scale;      /* see the format table; NULL for PA_SCALE_NONE */
  const void* value_scale;
  int64_t scale_stride_block; /* per-token / e8m0 scale caches: bytes between blocks */
  int64_t scale_stride_head;  /* bytes between KV heads; the token axis is dense */
  const int32_t* block_tables;/* [B, W] */
  int64_t bt_stride;          /* elements between block-table rows (>= W) */
  const int32_t* context_lens;/* [B] */
  void* out;                  /* [B*qlen, Hq, D] bf16 */
  int64_t out_stride_token;
  int64_t out_stride_head;
  /* 0 or 1.  With 1 and qlen > 1 the context is taken to end with the qlen query tokens:
   * query position i sees tokens t < context_len - qlen + 1 + i only (a position that
   * sees none gets a zero row).  The first page notes such a causal option, added by a
   * later change next to the masking flag.  bf16 and fp8 caches; MXFP4 takes qlen 1. */
  int32_t causal;
  /* Sliding window W >= 0 (0: none).  With W > 0, query position i, whose own place in the
   * context is p = context_len - qlen + i, sees only the tokens t > p - W: the W tokens
   * ending at itself (cut further by `causal` when that is set).  The first page lists
   * sliding-window plans among the variants its probe covers and defines them no further;
   * this is the plain reading.  Tokens before every position's window have no effect,
   * whatever their bytes: pages holding none of a window's tokens are not loaded, and
   * their block-table entries are never used as addresses.  Every format; the tcgen05
   * kernel does not take a window (the tile kernel runs).  Negative: PA_ERR_INVALID_ARG. */
  int32_t sliding_window;
  /* 0 or 1.  With 1 the value cache stores each page head-dim major: value_cache is
   * [NB, Hkv, D, S] e4m3 bytes, the S tokens of one head dim contiguous, with the key
   * cache's block and head strides (the key cache keeps [NB, Hkv, S, D]).  The first page's
   * probe runs fp8 per-tensor caches in a trans_v layout as well as with plain V, and does
   * not define that layout; this is the plain transposed reading.  fp8 with a per-tensor scale only
   * (PA_ERR_UNSUPPORTED otherwise); the tcgen05 kernel does not take it. */
  int32_t trans_v;
  /* Attention sinks: fp32 [Hq], one logit per query head in the units of the
   * softmax-scaled scores, or NULL.  Every row of query head h then takes one more softmax
   * term with a zero value: out = sum_t e^(x_t - M) v_t / (sum_t e^(x_t - M) + e^(s_h - M)),
   * M = max(max_t x_t, s_h); a row that sees no token stays zero.  The pages list sinks
   * beside sliding window among what the MXFP4 path refuses, without defining them; this
   * is the plain reading.  Every format; the tcgen05 kernel does not take them. */
  const float* sinks;
  /* Which decode kernel serves the call (PA_KERNEL_*): the library's choice (0), the
   * mma.sync tile kernel, or the tcgen05 kernel where it covers the shape (head_dim 128, at
   * most 32 query rows, pages of 8 tokens or more, separate reduce, no causal mask, window,
   * sinks, transposed V or in-kernel query quantisation; other shapes run the tile kernel).
   * Every choice computes the same function within the stated tolerances.  Other values:
   * PA_ERR_INVALID_ARG. */
  int32_t kernel;
} pa_decode_args;

#define PA_KERNEL_DEFAULT 0
#define PA_KERNEL_MMA 1
#define PA_KERNEL_TCGEN05 2

/* ABI version of this header; a mismatched library refuses nothing but reports it here.
 * Version 6 appended `kernel`; earlier fields keep their offsets. */
#define PA_DECODE_ABI_VERSION 6
int32_t pa_decode_abi_version(void);

/* Bytes of workspace the three calls need for these shapes (plan, partition scratch,
 * status word).  0 when the arguments are refused. Pure host arithmetic. */
size_t pa_decode_workspace_size(const pa_decode_args* args);

/* Host-side validation only (what every call checks before launching). */
pa_status pa_decode_validate(const pa_decode_args* args);

/* Builds the tile/partition work list on the device from context_lens: ceil(L/256)
 * tiles per (sequence, KV head) unit; the units are laid end to end, each as a gap of
 * two tiles (a task's fixed cost) followed by its tiles, and the line is cut into
 * task_budget chunks of equal length (one per tile-kernel CTA), longer when needed so
 * that no unit touches more than max_partitions chunks.  A unit crossing chunk
 * boundaries becomes one partition per chunk it touches; with max_partitions 1 each
 * unit is one task, run by the chunk it starts in.  The plan also keeps every unit whole
 * (as with max_partitions 1) when no unit is longer than a chunk plus its gap and, so laid
 * out, no chunk carries more than two gaps beyond its length (checked for batches of up
 * to 1024 sequences): splits there would add tasks, partials and reduce work without
 * evening out the chunks.  Clears the device status word.  One
 * launch, 1 CTA.  ("[FlyDSL] pa_decode: MXFP4 K/V ...", commit messages: planned tasks,
 * direct output with one partition, tasks from a CU budget.)
 * All launches of this library use programmatic dependent launch: a kernel may begin
 * before the previous kernel in the stream has finished when that kernel allows it (this
 * library's kernels do; others do only if they execute griddepcontrol.launch_dependents).
 * Each kernel waits for its predecessor before touching the workspace or the output, but
 * the plan reads context_lens before that wait: a kernel that writes context_lens and
 * allows early launch must do so before it allows it. */
pa_status pa_decode_plan(const pa_decode_args* args, void* workspace, size_t workspace_bytes,
                         void* stream);

/* Runs the tile kernel over the planned tasks, task_budget CTAs, each on its chunk:
 * block-table page gather (TMA), QK, online softmax, boundary-tile masking, PV.  Units
 * with one partition get their output rows written here (context 0 gives zeros);
 * others get partials in the workspace.  ("[FlyDSL] pa_decode: zero V rows past the context before PV", Fix.) */
pa_status pa_decode(const pa_decode_args* args, void* workspace, size_t workspace_bytes,
                    void* stream);

/* Merges the partials of every unit with two or more partitions, in a fixed
 * partition order: M = max_p m_p, w_p = l_p 2^(m_p - M), out = sum w_p o_p / sum w_p.
 * A no-op launch-free return when max_partitions is 1 or merge_in_decode is set (the
 * same merge, in the same order, then runs at the end of pa_decode).  ("[FlyDSL] pa_decode: MXFP4
 * K/V ...", Self-Review: the partition reducer.) */
pa_status pa_decode_reduce(const pa_decode_args* args, void* workspace,
                           size_t workspace_bytes, void* stream);

/* plan + decode + reduce in one call, on one stream.  With max_partitions == 1 each
 * (sequence, KV head) unit is a single task, the decode stores its bf16 rows itself and
 * the reduce has nothing to do; this is how the pages' plan-free mode is served here
 * ("[FlyDSL] pa_decode: MXFP4 K/V ...", Summary).
 * Small problems run as one launch instead, with no plan and no reduce kernel: when every
 * (sequence, KV head) unit fits the CTA budget and a unit's tiles (bounded by
 * max_blocks_per_seq * page_size, or by the sliding window) leave at most 3 per CTA, each
 * unit gets a thread-block cluster of up to 8 CTAs (at most max_partitions), each CTA an
 * equal run of the unit's tiles, and after a cluster barrier the cluster's CTAs merge the
 * partials in partition order with the reduce's formula, each CTA a share of the rows.  That launch leaves the workspace without a
 * plan (no chunk holds a task): a pa_decode or pa_decode_reduce on it needs a new
 * pa_decode_plan first.  The tcgen05 tile kernel (kernel = PA_KERNEL_TCGEN05) always takes
 * the planned path. */
pa_status pa_decode_run(const pa_decode_args* args, void* workspace, size_t workspace_bytes,
                        void* stream);

/* Fixed size of the library-owned workspace used by pa_decode_run_static. */
#define PA_DECODE_STATIC_WORKSPACE_BYTES ((size_t)16 << 20)

/* No counterpart in the source pages.  The same plan + decode + reduce as pa_decode_run,
 * for callers that cannot call cudaMalloc (code running inside another runtime's memory
 * budget, or latency-critical loops where an allocation may synchronise the device): the
 * workspace is a fixed PA_DECODE_STATIC_WORKSPACE_BYTES array in device memory that the
 * library defines, so this call allocates nothing; the caller still passes the inputs and
 * the output in args.  Returns PA_ERR_WORKSPACE when the problem needs more workspace than
 * that maximum (pa_decode_workspace_size tells how much it needs).  Every GPU that loads the
 * library holds the array until the process exits.  The first call on a device looks up the
 * array's device address with that device current; make that first call before any stream
 * capture.  All calls on a device share the array and it keeps the previous call's contents:
 * calls that overlap on the GPU race on it. */
pa_status pa_decode_run_static(const pa_decode_args* args, void* stream);

/* Enqueues a copy of the device status word (PA_DEVICE_*) into *host_status; the caller
 * synchronises the stream before reading it. host_status should be pinned memory. */
pa_status pa_decode_read_status(const void* workspace, int32_t* host_status, void* stream);

/* No counterpart in the source pages.  The device status word of the last
 * pa_decode_run_static call on the current device (the word lives in the library-owned
 * array, whose address callers never see): enqueues its copy into *host_status on
 * `stream`, which must belong to the current device (PA_ERR_INVALID_ARG otherwise); the
 * caller synchronises the stream before reading it.  Allocates nothing. */
pa_status pa_decode_read_status_static(int32_t* host_status, void* stream);

/* Static description of a status code. */
const char* pa_status_string(pa_status status);

#ifdef __cplusplus
}
#endif

#endif /* PA_DECODE_H_ */
