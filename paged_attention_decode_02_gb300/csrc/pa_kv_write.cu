// pa_kv_write.cu -- the MXFP4 KV-cache write: bf16 key / value rows into the paged e2m1 +
// e8m0 caches the decode reads ("[FlyDSL] pa_decode: MXFP4 K/V in the shared PA tile
// kernel", Dependencies: the pages come from a KV write kernel; Summary: the page layout).
// The conversion is the OCP MX one; include/pa_kv_write.h states it in full.
//
// One lane per 32-value block: a (token, KV head, K or V) row takes D/32 lanes, a warp
// 1024/D rows per pass, and each lane loads its 64 bytes for two passes before converting
// any.  The block's largest magnitude is an integer maximum over the bf16 bit patterns (no
// shuffles), and each lane writes its 16 bytes of codes with one store and its scale byte
// next to its neighbours'.  HBM-bound: 2D bytes read and D/2 + D/32 written per row.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pa_kv_write.h"

namespace pa {
namespace {

struct WriteParams {
  int T, Hkv, page_shift, NB;  // page_size = 1 << page_shift
  const __nv_bfloat16* key;
  const __nv_bfloat16* value;
  int64_t st, sh;  // source strides (elements)
  const int64_t* slots;
  uint8_t* kc;
  uint8_t* vc;
  int64_t csb, csh;  // data cache strides (bytes)
  uint8_t* ks;
  uint8_t* vs;
  int64_t ssb, ssh;  // scale cache strides (bytes)
};

// e8m0 byte of a finite block whose largest magnitude is amax, and 2^-E:
// E = floor(log2 amax) - 2 clamped to [-126, 127] (read from the exponent field; a
// subnormal amax lies below the clamp, and a finite bf16 amax puts E at most at 125, so
// 2^-E stays a normal fp32); an all-zero block takes byte 127 (X = 1).
__device__ __forceinline__ uint32_t block_scale(float amax, float* inv) {
  if (amax == 0.f) {
    *inv = 1.f;
    return 127u;
  }
  int E = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127 - 2;
  E = E < -126 ? -126 : (E > 125 ? 125 : E);  // bf16 input: floor(log2 amax) <= 127
  *inv = __uint_as_float((uint32_t)(127 - E) << 23);
  return (uint32_t)(E + 127);
}

// Two values to one byte of e2m1 codes (lo in the low nibble), nearest with ties to even,
// saturating at +-6: the hardware conversion.
__device__ __forceinline__ uint32_t e2m1_pair(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

constexpr int kPasses = 2;  // row passes per warp, the loads of all issued first

template <int D>
__global__ void __launch_bounds__(256) mxfp4_write_kernel(const WriteParams p) {
  constexpr int LPR = D / 32;    // lanes per row: one 32-value block each
  constexpr int RPP = 32 / LPR;  // rows per warp and pass
  const int lane = threadIdx.x & 31;
  const int b = lane % LPR;      // this lane's block in its row
  const int rows = p.T * p.Hkv * 2;  // < 2^30 (checked on the host)
  const int warp = blockIdx.x * 8 + (threadIdx.x >> 5);
  // rows (t, h, K|V) in order; this lane's row in each pass, its 32 bf16 values loaded
  // (64 contiguous bytes) for every pass before any is converted
  uint4 raw[kPasses][4];
  int tk[kPasses], hd[kPasses], rw[kPasses];
#pragma unroll
  for (int ps = 0; ps < kPasses; ++ps) {
    const int row = (warp * kPasses + ps) * RPP + lane / LPR;
    rw[ps] = row;
    const int th = row >> 1;
    tk[ps] = th / p.Hkv;
    hd[ps] = th - tk[ps] * p.Hkv;
    if (row < rows) {
      const uint4* src = reinterpret_cast<const uint4*>(((row & 1) ? p.value : p.key) +
                                                       tk[ps] * p.st + hd[ps] * p.sh + 32 * b);
#pragma unroll
      for (int i = 0; i < 4; ++i) raw[ps][i] = src[i];
    }
  }
#pragma unroll
  for (int ps = 0; ps < kPasses; ++ps) {
    const int row = rw[ps];
    if (row >= rows) continue;
    const long long slot = p.slots[tk[ps]];
    if (slot < 0 || slot >= ((long long)p.NB << p.page_shift)) continue;  // skipped token
    const long long blk = slot >> p.page_shift;
    const int off = (int)(slot & ((1 << p.page_shift) - 1));
    const uint32_t w[16] = {raw[ps][0].x, raw[ps][0].y, raw[ps][0].z, raw[ps][0].w,
                            raw[ps][1].x, raw[ps][1].y, raw[ps][1].z, raw[ps][1].w,
                            raw[ps][2].x, raw[ps][2].y, raw[ps][2].z, raw[ps][2].w,
                            raw[ps][3].x, raw[ps][3].y, raw[ps][3].z, raw[ps][3].w};
    // the block's largest magnitude: bf16 magnitudes order like their bit patterns, and an
    // exponent field of all ones (infinity, NaN) orders above every finite value
    uint32_t m2 = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) m2 = __vmaxu2(m2, w[i] & 0x7FFF7FFFu);
    const uint32_t mb = max(m2 & 0xFFFFu, m2 >> 16);
    const bool bad = mb >= 0x7F80u;
    float inv = 0.f;
    const uint32_t sb = bad ? 255u : block_scale(__uint_as_float(mb << 16), &inv);
    uint32_t code[4] = {0u, 0u, 0u, 0u};  // 32 e2m1 codes, value 2i in the low nibble of byte i
    if (!bad) {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        code[i >> 2] |= e2m1_pair(__uint_as_float(w[i] << 16) * inv,
                                  __uint_as_float(w[i] & 0xFFFF0000u) * inv) << (8 * (i & 3));
    }
    uint8_t* dst = ((row & 1) ? p.vc : p.kc) + blk * p.csb + hd[ps] * p.csh +
                   (long long)off * (D / 2) + 16 * b;
    *reinterpret_cast<uint4*>(dst) = make_uint4(code[0], code[1], code[2], code[3]);
    ((row & 1) ? p.vs : p.ks)[blk * p.ssb + hd[ps] * p.ssh + (long long)off * (D / 32) + b] =
        (uint8_t)sb;
  }
}

bool aligned16(const void* q) { return ((uintptr_t)q & 15) == 0; }

}  // namespace
}  // namespace pa

extern "C" pa_status pa_mxfp4_kv_write(const pa_mxfp4_write_args* a, void* stream) {
  if (!a) return PA_ERR_INVALID_ARG;
  const int D = a->head_dim;
  if (a->num_tokens < 0 || a->num_kv_heads < 1 || a->page_size < 1 || a->num_blocks < 1 || D < 1)
    return PA_ERR_INVALID_ARG;
  if (D != 64 && D != 128 && D != 256) return PA_ERR_UNSUPPORTED;
  switch (a->page_size) {  // the decode's page sizes
    case 16: case 32: case 64: case 128: case 256: break;
    default: return PA_ERR_UNSUPPORTED;
  }
  // rows (and the rounded-up grid's row indices) stay well inside int32
  if ((int64_t)a->num_tokens * a->num_kv_heads >= ((int64_t)1 << 29)) return PA_ERR_UNSUPPORTED;
  if (a->num_tokens == 0) return PA_OK;
  if (!a->key || !a->value || !a->slot_mapping || !a->key_cache || !a->value_cache ||
      !a->key_scale || !a->value_scale)
    return PA_ERR_INVALID_ARG;
  if (a->src_stride_head < D || a->src_stride_token < a->src_stride_head * a->num_kv_heads)
    return PA_ERR_INVALID_ARG;
  if (a->cache_stride_head < (int64_t)a->page_size * (D / 2) ||
      a->cache_stride_block < a->cache_stride_head * a->num_kv_heads ||
      a->scale_stride_head < (int64_t)a->page_size * (D / 32) ||
      a->scale_stride_block < a->scale_stride_head * a->num_kv_heads)
    return PA_ERR_INVALID_ARG;
  // vector loads of whole lane chunks; stores of the lanes' bytes on their natural alignment
  if (!pa::aligned16(a->key) || !pa::aligned16(a->value) || (a->src_stride_head * 2) % 16 ||
      (a->src_stride_token * 2) % 16 || !pa::aligned16(a->key_cache) ||
      !pa::aligned16(a->value_cache) || a->cache_stride_head % 16 || a->cache_stride_block % 16)
    return PA_ERR_UNSUPPORTED;
  pa::WriteParams p;
  p.T = a->num_tokens;
  p.Hkv = a->num_kv_heads;
  p.page_shift = __builtin_ctz((unsigned)a->page_size);
  p.NB = a->num_blocks;
  p.key = static_cast<const __nv_bfloat16*>(a->key);
  p.value = static_cast<const __nv_bfloat16*>(a->value);
  p.st = a->src_stride_token;
  p.sh = a->src_stride_head;
  p.slots = a->slot_mapping;
  p.kc = static_cast<uint8_t*>(a->key_cache);
  p.vc = static_cast<uint8_t*>(a->value_cache);
  p.csb = a->cache_stride_block;
  p.csh = a->cache_stride_head;
  p.ks = static_cast<uint8_t*>(a->key_scale);
  p.vs = static_cast<uint8_t*>(a->value_scale);
  p.ssb = a->scale_stride_block;
  p.ssh = a->scale_stride_head;
  const long long rows = (long long)p.T * p.Hkv * 2;
  const long long per_block = 8LL * pa::kPasses * (32 / (D / 32));  // 8 warps
  const long long blocks = (rows + per_block - 1) / per_block;
  if (blocks > 0x7FFFFFFFll) return PA_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (D == 64)
    pa::mxfp4_write_kernel<64><<<(unsigned)blocks, 256, 0, s>>>(p);
  else if (D == 128)
    pa::mxfp4_write_kernel<128><<<(unsigned)blocks, 256, 0, s>>>(p);
  else
    pa::mxfp4_write_kernel<256><<<(unsigned)blocks, 256, 0, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
