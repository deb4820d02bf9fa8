// stv_device.cuh -- device-side building blocks shared by the kernels:
// page addressing, the 3-bit block decode, status reporting.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "stv_internal.h"

namespace stv {

__device__ __forceinline__ void report(int32_t* status, int bit) {
  if (status) atomicOr(status, bit);
}

// Base of KV head h's block in the page holding token `tok` of sequence s,
// or nullptr (and STV_DEV_BAD_PAGE) when the table or the pool is exceeded.
__device__ __forceinline__ const uint8_t* head_block(const SeqDesc& sd, const uint8_t* pool, int64_t page_bytes,
                                                     int32_t pool_pages, int64_t tok, int h, int32_t* status) {
  int64_t lp = tok >> 8;
  if (tok < 0 || lp >= sd.n_pages) {
    report(status, STV_DEV_BAD_PAGE);
    return nullptr;
  }
  int32_t page = __ldg(sd.page_table + lp);
  if (page < 0 || page >= pool_pages) {
    report(status, STV_DEV_BAD_PAGE);
    return nullptr;
  }
  return pool + (int64_t)page * page_bytes + (int64_t)h * kHeadBytes;
}

// Bit b of code i of a 32-code block: word and bit index (the layout stated
// in include/stv.h).
__device__ __forceinline__ void bit_place(int i, int b, int& word, int& bit) {
  if (i < 30) {
    int m = i >> 1;
    word = m / 5;
    bit = ((i & 1) ? 16 : 0) + 3 * (m % 5) + b;
  } else {
    word = b;
    bit = (i == 30) ? 15 : 31;
  }
}

__device__ __forceinline__ int block_code(uint32_t w0, uint32_t w1, uint32_t w2, int i) {
  int c = 0;
#pragma unroll
  for (int b = 0; b < 3; ++b) {
    int wd, bt;
    bit_place(i, b, wd, bt);
    uint32_t w = wd == 0 ? w0 : (wd == 1 ? w1 : w2);
    c |= ((w >> bt) & 1u) << b;
  }
  return c;
}

// Decode one 32-code block into 16 fp16 pairs (codes 2m, 2m+1) of
// scale * (code - 4).  Each code is dropped into the mantissa of an fp16
// constant (1024, 128 or 16, chosen so that the field's lowest bit weighs 1)
// with a single AND/OR, which yields base + code exactly; subtracting
// base + 4 is exact; the product with the scale is one fp16 rounding.
// `scale` holds the two scales of the pair (equal for a K block, the two
// tokens' scales for a V block).
__device__ __forceinline__ __half2 u32_as_h2(uint32_t x) {
  __half2 h;
  *reinterpret_cast<uint32_t*>(&h) = x;
  return h;
}

template <typename ScaleFn>
__device__ __forceinline__ void decode_block_h2(uint32_t w0, uint32_t w1, uint32_t w2, ScaleFn scale,
                                                __half2 (&out)[16]) {
  const __half2 b1024 = u32_as_h2(0x64046404u);  // 1028
  const __half2 b128 = u32_as_h2(0x58205820u);   // 132
  const __half2 b16 = u32_as_h2(0x4D004D00u);    // 20
  const uint32_t w[3] = {w0, w1, w2};
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    uint32_t x = w[j];
    uint32_t xs = x >> 9;
    out[5 * j + 0] = __hmul2(__hsub2(u32_as_h2((x & 0x00070007u) | 0x64006400u), b1024), scale(5 * j + 0));
    out[5 * j + 1] = __hmul2(__hsub2(u32_as_h2((x & 0x00380038u) | 0x58005800u), b128), scale(5 * j + 1));
    out[5 * j + 2] = __hmul2(__hsub2(u32_as_h2((x & 0x01C001C0u) | 0x4C004C00u), b16), scale(5 * j + 2));
    out[5 * j + 3] = __hmul2(__hsub2(u32_as_h2((xs & 0x00070007u) | 0x64006400u), b1024), scale(5 * j + 3));
    out[5 * j + 4] = __hmul2(__hsub2(u32_as_h2((xs & 0x00380038u) | 0x58005800u), b128), scale(5 * j + 4));
  }
  uint32_t x15 = ((w0 >> 15) & 0x00010001u) | ((w1 >> 14) & 0x00020002u) | ((w2 >> 13) & 0x00040004u) | 0x64006400u;
  out[15] = __hmul2(__hsub2(u32_as_h2(x15), b1024), scale(15));
}

// Same decode without the scale: fp16 pairs of (code - 4), exact.
__device__ __forceinline__ void decode_block_raw(uint32_t w0, uint32_t w1, uint32_t w2, __half2 (&out)[16]) {
  const __half2 one = u32_as_h2(0x3C003C00u);
  decode_block_h2(w0, w1, w2, [&](int) { return one; }, out);
}

}  // namespace stv
