// stv_device.cuh -- device-side building blocks shared by the kernels:
// page addressing, the 3-bit block decode, status reporting.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "stv_internal.h"

namespace stv {

// Programmatic dependent launch: the round's kernels are launched with
// programmatic stream serialization (launch_pdl), so a kernel's CTAs may be
// scheduled while the previous kernel in the stream is still finishing.
// grid_dep_wait() returns once that kernel has completed and its writes are
// visible (at once when there is none); every kernel calls it before its
// first global-memory access.  grid_dep_launch() lets the next kernel's CTAs
// be scheduled; they wait in their own grid_dep_wait().
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void report(int32_t* status, int bit) {
  if (status) atomicOr(status, bit);
}

// Base of KV head h's block in the page holding token `tok` of sequence s,
// or nullptr (and STV_DEV_BAD_PAGE) when the table or the pool is exceeded.
__device__ __forceinline__ const uint8_t* head_block(const SeqDesc& sd, const uint8_t* pool, int64_t page_bytes,
                                                     int32_t pool_pages, int64_t tok, int h, int32_t* status,
                                                     int head_bytes = kHeadBytes) {
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
  return pool + (int64_t)page * page_bytes + (int64_t)h * head_bytes;
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

// ---------------------------------------------------------------------------
// a1, the per-row quantizer and packer (kv_append_pack; also run inside the
// verify kernel for the round's tree rows).

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// rne(x / s) for s > 0, exactly, without a division (both quantizers of
// include/stv.h; |x / s| <= 11 for them).  q = x * (1/s) from the
// approximate reciprocal is within far less than 1/2 of x / s, so c = rint(q)
// is rne(x / s) or next to it, and only when x / s lies near a half-integer.
// The residual d = x - c s is exact: either c = 0 (d = x) or |x| >= s/2, and
// then x and c s (fp16 values times integers of at most 4 bits) are a few
// binades apart, so d needs at most about 16 significant bits.  d against
// +-s/2 (exact) settles the rounding, ties to the even integer.  s is an fp16
// value, so a normal fp32 value, and the reciprocal's flush-to-zero mode
// never applies.
__device__ __forceinline__ int rne_quotient(float x, float s) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
  int c = __float2int_rn(x * r);
  const float d = fmaf(-(float)c, s, x), hs = 0.5f * s;
  const bool odd = (c & 1) != 0;
  if (d > hs || (d == hs && odd)) c += 1;        // closer to c + 1, or a tie with odd c
  else if (d < -hs || (d == -hs && odd)) c -= 1;  // closer to c - 1, or a tie with odd c
  return c;
}

// 3-bit code of x for scale s: clamp(rne(x / s) + 4, 0, 7); 4 when s == 0.
__device__ __forceinline__ int quant_code(float x, float s) {
  if (s == 0.f) return 4;
  return min(max(rne_quotient(x, s) + 4, 0), 7);
}

// int4 code u = c + 8 of x for scale s: c = clamp(rne(x / s), -8, 7); 8 when
// s == 0 (the int4 per-token-head cache of include/stv.h).
__device__ __forceinline__ int quant_code_i4(float x, float s) {
  if (s == 0.f) return 8;
  return min(max(rne_quotient(x, s), -8), 7) + 8;
}

// Bit position of element e (0..7) of an int4 word: 4 * (e / 2), plus 16
// for odd e, so that one AND/OR per pair makes an fp16 pair (below).
__device__ __forceinline__ int i4_pos(int e) { return ((e & 1) ? 16 : 0) + 4 * (e >> 1); }

// Bit position of token t (0..15) in a 2-bit V word of the K 4 / V 2-bit
// cache: 2 * (t / 2), plus 16 for odd t, so that one AND/OR per pair makes
// an fp16 pair (decode_v2_block_h2).
__device__ __forceinline__ int v2_pos(int t) { return ((t & 1) ? 16 : 0) + 2 * (t >> 1); }

// Decode one channel's 2-bit V codes for 32 tokens (two words; pairs (2m,
// 2m+1) in order) into 16 fp16 pairs scale * (u - 2).  The pair at bits
// 2k, 16 + 2k (k = 0..3 of each byte-pair) drops into the mantissas of 1024,
// 256, 64 or 16 (lowest field bit weighing 1) with one AND/OR, giving
// base + u exactly; subtracting base + 2 is exact; the product with the
// scale pair is one fp16 rounding.
template <typename ScaleFn>
__device__ __forceinline__ void decode_v2_block_h2(uint32_t w0, uint32_t w1, ScaleFn scale, __half2 (&out)[16]) {
  const __half2 b1026 = u32_as_h2(0x64026402u);  // 1026
  const __half2 b258 = u32_as_h2(0x5C085C08u);   // 258
  const __half2 b66 = u32_as_h2(0x54205420u);    // 66
  const __half2 b18 = u32_as_h2(0x4C804C80u);    // 18
  const uint32_t w[2] = {w0, w1};
#pragma unroll
  for (int j = 0; j < 2; ++j) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const uint32_t x = half ? (w[j] >> 8) : w[j];
      const int m = 8 * j + 4 * half;
      out[m + 0] = __hmul2(__hsub2(u32_as_h2((x & 0x00030003u) | 0x64006400u), b1026), scale(m + 0));
      out[m + 1] = __hmul2(__hsub2(u32_as_h2((x & 0x000C000Cu) | 0x5C005C00u), b258), scale(m + 1));
      out[m + 2] = __hmul2(__hsub2(u32_as_h2((x & 0x00300030u) | 0x54005400u), b66), scale(m + 2));
      out[m + 3] = __hmul2(__hsub2(u32_as_h2((x & 0x00C000C0u) | 0x4C004C00u), b18), scale(m + 3));
    }
  }
}

// Decode four int4 words (32 elements, pairs (2m, 2m+1) in order) into 16
// fp16 pairs of the signed codes c = u - 8.  Elements 0/1 of a word drop into
// the mantissas of 1024 (lowest bit weighs 1) and elements 2/3 into those of
// 64 (bits 4..7 weigh 1) with one AND/OR each, giving base + u exactly; the
// upper byte's elements 4..7 do the same after one shift.  Subtracting
// base + 8 is exact, so every code comes out exact.
__device__ __forceinline__ void decode_i4_codes_h2(const uint32_t (&w)[4], __half2 (&out)[16]) {
  const __half2 b1032 = u32_as_h2(0x64086408u);  // 1032
  const __half2 b72 = u32_as_h2(0x54805480u);    // 72
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t x = w[j], xs = x >> 8;
    out[4 * j + 0] = __hsub2(u32_as_h2((x & 0x000F000Fu) | 0x64006400u), b1032);
    out[4 * j + 1] = __hsub2(u32_as_h2((x & 0x00F000F0u) | 0x54005400u), b72);
    out[4 * j + 2] = __hsub2(u32_as_h2((xs & 0x000F000Fu) | 0x64006400u), b1032);
    out[4 * j + 3] = __hsub2(u32_as_h2((xs & 0x00F000F0u) | 0x54005400u), b72);
  }
}

// The same, times a scale per pair: scale * c with one fp16 rounding.
template <typename ScaleFn>
__device__ __forceinline__ void decode_i4_block_h2(const uint32_t (&w)[4], ScaleFn scale, __half2 (&out)[16]) {
  decode_i4_codes_h2(w, out);
#pragma unroll
  for (int m = 0; m < 16; ++m) out[m] = __hmul2(out[m], scale(m));
}

// One channel of one (row, KV head): called by 256 threads, thread c =
// channel, warp = one 32-channel group (all 32 lanes take part).  K: the
// group maximum is a warp reduction, the block's three words are three
// warp-wide OR reductions, written by lane 0 with the group's scale.  V: the
// group's scale is written by lane 0 and this channel's code is returned; V
// codes are channel-major (a block holds one channel's codes for 32 tokens),
// so the caller places the code's three bits.
__device__ __forceinline__ int append_row_k_vscale(float xk, float xv, uint8_t* hb, int slot, int c) {
  const int g = c >> 5, lane = c & 31;
  {
    __half sh = __float2half_rn(warp_max(fabsf(xk)) * 0.25f);
    int code = quant_code(xk, __half2float(sh));
    uint32_t m0 = 0u, m1 = 0u, m2 = 0u;  // this lane's bits of the block's three words
#pragma unroll
    for (int b = 0; b < 3; ++b) {
      int wd, bt;
      bit_place(lane, b, wd, bt);
      const uint32_t bit = ((code >> b) & 1) ? 1u << bt : 0u;
      m0 |= wd == 0 ? bit : 0u;
      m1 |= wd == 1 ? bit : 0u;
      m2 |= wd == 2 ? bit : 0u;
    }
    uint32_t w0 = __reduce_or_sync(0xffffffffu, m0);
    uint32_t w1 = __reduce_or_sync(0xffffffffu, m1);
    uint32_t w2 = __reduce_or_sync(0xffffffffu, m2);
    if (lane == 0) {
      uint32_t* wp = reinterpret_cast<uint32_t*>(hb + kOffKCodes + slot * 96 + g * 12);
      wp[0] = w0;
      wp[1] = w1;
      wp[2] = w2;
      *reinterpret_cast<__half*>(hb + kOffKScales + slot * 16 + g * 2) = sh;
    }
  }
  __half sh = __float2half_rn(warp_max(fabsf(xv)) * 0.25f);
  const int tile = slot / kTileTok, within = slot % kTileTok;
  if (lane == 0)
    *reinterpret_cast<__half*>(hb + kOffVScales + tile * kVTileScaleBytes + g * (kTileTok * 2) + within * 2) = sh;
  return quant_code(xv, __half2float(sh));
}

// Address of the three V words (one 32-token block of channel c) holding
// slot's code, and the code's index in that block.
__device__ __forceinline__ uint32_t* v_block_words(uint8_t* hb, int slot, int c, int* index) {
  const int tile = slot / kTileTok, within = slot % kTileTok;
  *index = within % 32;
  return reinterpret_cast<uint32_t*>(hb + kOffVCodes + tile * kVTileCodeBytes + c * 24 + (within / 32) * 12);
}

// Replaces code `index` of a 32-code block held in three words.
__device__ __forceinline__ void set_block_code(uint32_t& w0, uint32_t& w1, uint32_t& w2, int index, int code) {
#pragma unroll
  for (int b = 0; b < 3; ++b) {
    int wd, bt;
    bit_place(index, b, wd, bt);
    const uint32_t m = 1u << bt, v = ((code >> b) & 1) ? m : 0u;
    w0 = wd == 0 ? ((w0 & ~m) | v) : w0;
    w1 = wd == 1 ? ((w1 & ~m) | v) : w1;
    w2 = wd == 2 ? ((w2 & ~m) | v) : w2;
  }
}

// a1 for one channel of one row, V bits by atomics: rows packed by other
// threads or CTAs at the same time may share the V block (disjoint bits).
__device__ __forceinline__ void append_row_channel(float xk, float xv, uint8_t* hb, int slot, int c) {
  const int code = append_row_k_vscale(xk, xv, hb, slot, c);
  int i;
  uint32_t* wp = v_block_words(hb, slot, c, &i);
#pragma unroll
  for (int b = 0; b < 3; ++b) {
    int wd, bt;
    bit_place(i, b, wd, bt);
    if ((code >> b) & 1)
      atomicOr(wp + wd, 1u << bt);
    else
      atomicAnd(wp + wd, ~(1u << bt));
  }
}

}  // namespace stv
