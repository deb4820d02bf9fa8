// combine.cuh -- a5, the merge of the split-KV partials of one (sequence,
// KV head, row, 64-channel quarter), shared by split_combine_kernel (its own
// launch) and the verify kernel that merges its own splits (one launch per
// layer).  Both run this code, so their outputs are equal bit for bit.
//
// Sources: Reddit posts (u/iamMess), second post (split-KV verify
// attention: per-split partial outputs, then a merge).
//
// One warp; lane = 2 channels.  Split kb + j's (m, l) sits in lane j of chunk
// kb / 32.  The (m, l) of every split and the partial O of the first kDepth
// splits are loaded together, one memory round trip for up to kDepth splits
// (with kDepth = 64, later chunks of 32 take one more each); then M = max m,
// the weights 2^(m - M), and the sums in split order, so the result depends
// neither on timing nor on kDepth.  kDepth <= 32 requires splits <= kDepth.
// kCg: the loads bypass L1 (partials written by other CTAs of the same
// launch).
#pragma once
#include "stv_device.cuh"

namespace stv {

__device__ __forceinline__ float warp_max_xor(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

template <bool kCg>
__device__ __forceinline__ float2 ld_f2(const float* a) {
  if constexpr (kCg) return __ldcg(reinterpret_cast<const float2*>(a));
  else return *reinterpret_cast<const float2*>(a);
}

// acc += the chunk's N partials weighted by w (lane j's weight is split j's)
template <int N>
__device__ __forceinline__ void combine_chunk(const float2 (&o)[N], float w, float& acc0, float& acc1) {
#pragma unroll
  for (int j = 0; j < N; ++j) {
    const float wk = __shfl_sync(0xffffffffu, w, j);
    // a split with weight 0 (no visible key for this row) adds nothing
    acc0 = wk != 0.f ? fmaf(wk, o[j].x, acc0) : acc0;
    acc1 = wk != 0.f ? fmaf(wk, o[j].y, acc1) : acc1;
  }
}

// Row r of (sequence s, KV head h), channels [64 quarter, 64 quarter + 64):
// O = sum_k 2^(m_k - M) O_k / sum_k 2^(m_k - M) l_k over the head's splits k,
// written as fp16 to o [n_seqs][T][hq][256].  o_part [units][R][256] and
// ml [units][R][2] are indexed by work unit.
template <int kDepth, bool kCg>
__device__ __forceinline__ void combine_row_quarter(const SeqDesc& sd, int s, int h, int r, int quarter, int R, int T,
                                                    int hq, int G, const float* o_part, const float* ml_,
                                                    __half* o) {
  static_assert(kDepth == 16 || kDepth == 32 || kDepth == 64, "depth");
  const int lane = threadIdx.x & 31;
  const int u0 = sd.unit_base + h * sd.splits, splits = sd.splits;
  const int64_t split_stride = (int64_t)R * kHeadDim;
  const float* src = o_part + (int64_t)u0 * split_stride + (int64_t)r * kHeadDim + quarter * 64 + lane * 2;
  // (m, l) of every split, 32 per register: at most kMaxChunks * 32 splits
  constexpr int kMaxChunks = kDepth == 64 ? kMaxSplitsPerHead / 32 : 1;
  float2 mlv[kMaxChunks];
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    const int k = c * 32 + lane;
    mlv[c] = k < splits ? ld_f2<kCg>(ml_ + ((int64_t)(u0 + k) * R + r) * 2) : make_float2(-INFINITY, 0.f);
  }
  // the first kDepth partials, in flight with the (m, l) loads
  constexpr int kA = kDepth < 32 ? kDepth : 32;
  float2 oa[kA], ob[kDepth == 64 ? 32 : 1];
#pragma unroll
  for (int j = 0; j < kA; ++j) oa[j] = j < splits ? ld_f2<kCg>(src + j * split_stride) : make_float2(0.f, 0.f);
  if constexpr (kDepth == 64) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      ob[j] = 32 + j < splits ? ld_f2<kCg>(src + (32 + j) * split_stride) : make_float2(0.f, 0.f);
  }
  float M = -INFINITY;
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) M = fmaxf(M, mlv[c].x);
  M = warp_max_xor(M);
  float L = 0.f, acc0 = 0.f, acc1 = 0.f;
  auto weight = [&](const float2 v) {
    const float w = v.x == -INFINITY ? 0.f : exp2f(v.x - M);
    L += w * v.y;
    return w;
  };
  combine_chunk(oa, weight(mlv[0]), acc0, acc1);
  if constexpr (kDepth == 64) {
    if (splits > 32) combine_chunk(ob, weight(mlv[1]), acc0, acc1);
    // chunks 2 and later (more than 64 splits: contexts past about 500K keys)
#pragma unroll 1
    for (int c = 2; c < kMaxChunks && c * 32 < splits; ++c) {
      float w = 0.f;
#pragma unroll
      for (int i = 2; i < kMaxChunks; ++i)
        if (i == c) w = weight(mlv[i]);
      const int n = min(32, splits - c * 32);
      const float* sp = src + (int64_t)(c * 32) * split_stride;
#pragma unroll
      for (int j = 0; j < 32; ++j) oa[j] = j < n ? ld_f2<kCg>(sp + j * split_stride) : make_float2(0.f, 0.f);
      combine_chunk(oa, w, acc0, acc1);
    }
  }
#pragma unroll
  for (int o2 = 16; o2; o2 >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o2);
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const int node = r / G, qh = h * G + r % G;
  *reinterpret_cast<__half2*>(o + (((int64_t)s * T + node) * hq + qh) * kHeadDim + quarter * 64 + lane * 2) =
      __floats2half2_rn(acc0 * inv, acc1 * inv);
}

// The same merge in about 60 registers, for callers whose register budget is
// tight: a first pass takes M from the splits' m (one load per 32 splits a
// lane, all in flight), a second walks the splits in chunks of 16, loading
// each 32 splits' (m, l) again with their first 16 partials.  Same values,
// same weights, same order of sums as combine_row_quarter: the same result
// bit for bit.
template <bool kCg>
__device__ __forceinline__ void combine_row_quarter_lean(const SeqDesc& sd, int s, int h, int r, int quarter, int R,
                                                         int T, int hq, int G, const float* o_part,
                                                         const float* ml_, __half* o) {
  const int lane = threadIdx.x & 31;
  const int u0 = sd.unit_base + h * sd.splits, splits = sd.splits;
  const int64_t split_stride = (int64_t)R * kHeadDim;
  const float* src = o_part + (int64_t)u0 * split_stride + (int64_t)r * kHeadDim + quarter * 64 + lane * 2;
  const float* mlr = ml_ + ((int64_t)u0 * R + r) * 2;  // split k's (m, l) at mlr + k * 2R
  constexpr int kMaxChunks = kMaxSplitsPerHead / 32;
  float M = -INFINITY;
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    const int k = c * 32 + lane;
    if (k < splits) M = fmaxf(M, ld_f2<kCg>(mlr + (int64_t)k * 2 * R).x);
  }
  M = warp_max_xor(M);
  float L = 0.f, acc0 = 0.f, acc1 = 0.f;
#pragma unroll 1
  for (int c = 0; c * 32 < splits; ++c) {
    const int k = c * 32 + lane;
    const float2 v = k < splits ? ld_f2<kCg>(mlr + (int64_t)k * 2 * R) : make_float2(-INFINITY, 0.f);
#pragma unroll 1
    for (int hf = 0; hf < 2 && c * 32 + hf * 16 < splits; ++hf) {
      const int k0 = c * 32 + hf * 16;
      float2 oa[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        oa[j] = k0 + j < splits ? ld_f2<kCg>(src + (int64_t)(k0 + j) * split_stride) : make_float2(0.f, 0.f);
      const float w = v.x == -INFINITY ? 0.f : exp2f(v.x - M);  // split c * 32 + lane's weight
      if (hf == 0) L += w * v.y;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float wk = __shfl_sync(0xffffffffu, w, hf * 16 + j);
        acc0 = wk != 0.f ? fmaf(wk, oa[j].x, acc0) : acc0;
        acc1 = wk != 0.f ? fmaf(wk, oa[j].y, acc1) : acc1;
      }
    }
  }
#pragma unroll
  for (int o2 = 16; o2; o2 >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o2);
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const int node = r / G, qh = h * G + r % G;
  *reinterpret_cast<__half2*>(o + (((int64_t)s * T + node) * hq + qh) * kHeadDim + quarter * 64 + lane * 2) =
      __floats2half2_rn(acc0 * inv, acc1 * inv);
}

}  // namespace stv
