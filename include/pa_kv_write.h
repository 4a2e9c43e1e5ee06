/*
 * pa_kv_write.h -- C ABI of the MXFP4 KV-cache write in libpa_decode.so (sm_103a).
 *
 * Writes new key / value rows into the paged MXFP4 caches that pa_decode reads.  The
 * pages say the MXFP4 pages come from a KV write kernel ("[FlyDSL] pa_decode: MXFP4
 * K/V in the shared PA tile kernel", Dependencies) and fix the format (Summary: uint8
 * data [pages, kv_heads, 128, 64], two e2m1 per byte with element 2j in the low nibble;
 * uint8 e8m0 scales [pages, kv_heads, 128, 4], one per 32 values along head_dim); the
 * conversion into it is the OCP MX one.  For every token t with slot_mapping[t] >= 0
 * and KV head h, each block of 32 values x of key[t, h, :] (and of value[t, h, :]):
 *
 *     X      = 2^E,  E = floor(log2 max|x|) - 2, clamped to [-126, 127]
 *     scale  = E + 127                      (an all-zero block: 127, i.e. X = 1)
 *     code_i = the e2m1 value nearest to x_i / X, ties to the code with an even
 *              mantissa bit, saturating at +-6 (the hardware cvt.rn.satfinite)
 *
 * A block holding a NaN or an infinity gets scale 255 (NaN) and zero codes.  Scale
 * bytes are otherwise in 1..254, the range the decode takes as defined.
 *
 * Layout and ownership: all pointers are DEVICE pointers owned by the caller.
 *   key, value      bf16 [T, Hkv, D]; strides in elements; head_dim contiguous, 16-byte
 *                   aligned rows
 *   slot_mapping    int64 [T]: the cache slot block * page_size + offset of token t;
 *                   a negative slot skips the token; slots at or past
 *                   num_blocks * page_size are skipped too (nothing is written)
 *   key_cache,      uint8 [NB, Hkv, S, D/2] with the strides below (bytes; token rows
 *   value_cache     dense, D/2 bytes)
 *   key_scale,      uint8 [NB, Hkv, S, D/32] (bytes; token rows dense, D/32 bytes)
 *   value_scale
 * head_dim 64, 128 or 256; page_size 16, 32, 64, 128 or 256 (the decode's); fewer than
 * 2^29 (token, KV head) pairs per call.  Stream-ordered on `stream` (a cudaStream_t as void*), no
 * host synchronisation, no allocation; arguments are checked on the host before the
 * launch, and a refused call launches nothing (PA_ERR_INVALID_ARG for missing pointers,
 * negative sizes or strides that overlap rows; PA_ERR_UNSUPPORTED for other head_dims
 * or unaligned rows; PA_ERR_CUDA if the launch fails).
 */
#ifndef PA_KV_WRITE_H
#define PA_KV_WRITE_H

#include <stdint.h>

#include "pa_decode.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int32_t num_tokens, num_kv_heads, head_dim, page_size, num_blocks;
  const void* key;            /* bf16 [T, Hkv, D] */
  const void* value;          /* bf16 [T, Hkv, D] */
  int64_t src_stride_token;   /* elements between tokens (key and value) */
  int64_t src_stride_head;    /* elements between KV heads */
  const int64_t* slot_mapping;/* [T] */
  void* key_cache;            /* uint8 [NB, Hkv, S, D/2] */
  void* value_cache;
  int64_t cache_stride_block; /* bytes between blocks (both data caches) */
  int64_t cache_stride_head;  /* bytes between KV heads within a block */
  void* key_scale;            /* uint8 [NB, Hkv, S, D/32] */
  void* value_scale;
  int64_t scale_stride_block; /* bytes between blocks (both scale caches) */
  int64_t scale_stride_head;  /* bytes between KV heads within a block */
} pa_mxfp4_write_args;

pa_status pa_mxfp4_kv_write(const pa_mxfp4_write_args* args, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_KV_WRITE_H */
