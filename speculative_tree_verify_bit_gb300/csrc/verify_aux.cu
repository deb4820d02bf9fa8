// verify_aux.cu -- the kernels around the tensor-core verify kernel: the int8
// Q quantizer (a3), split_combine (a5) and the prefill chain parents.
//
// Sources: "elpis" README, "Why fast" (8-row token tree verified in one pass;
// decode verify with 3-bit K codes as exact int8 against int8 Q); Reddit
// posts (u/iamMess), second post (split-KV verify attention).
#include "stv_device.cuh"

namespace stv {

__device__ __forceinline__ float wmax(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
// a3: per (node, Q head) row, m = max|q|, qi = rne(127 q / m), sQ = m / 127.
// 127 q is exact in fp32 and the quotient of two fp16-derived values never
// rounds onto a half-integer, so this matches the exact definition.
__device__ __forceinline__ void quantize_q_row_warp(const __half* __restrict__ q, int8_t* qi, float* sq) {
  const int lane = threadIdx.x & 31;
  uint4 raw = *reinterpret_cast<const uint4*>(q + lane * 8);
  const __half* hv = reinterpret_cast<const __half*>(&raw);
  float x[8], m = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    x[e] = __half2float(hv[e]);
    m = fmaxf(m, fabsf(x[e]));
  }
  m = wmax(m);
  uint32_t packed[2] = {0u, 0u};
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    int v = (m == 0.f) ? 0 : (int)rintf(__fdiv_rn(127.f * x[e], m));
    packed[e >> 2] |= ((uint32_t)(v & 0xff)) << (8 * (e & 3));
  }
  *reinterpret_cast<uint2*>(qi + lane * 8) = make_uint2(packed[0], packed[1]);
  if (lane == 0) *sq = (m == 0.f) ? 0.f : __fdiv_rn(m, 127.f);
}

__global__ void __launch_bounds__(256) quantize_q_kernel(const __half* __restrict__ q, int n_rows,
                                                         int8_t* __restrict__ qi, float* __restrict__ sq) {
  grid_dep_wait();
  grid_dep_launch();
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= n_rows) return;
  quantize_q_row_warp(q + (int64_t)row * kHeadDim, qi + (int64_t)row * kHeadDim, sq + row);
}

cudaError_t launch_quantize_q(const __half* q, int n_rows, int8_t* qi, float* sq, cudaStream_t s) {
  return launch_pdl(quantize_q_kernel, (n_rows + 7) / 8, 256, 0, s, q, n_rows, qi, sq);
}

// ---------------------------------------------------------------------------
// a5: split_combine.  One warp per (sequence, KV head, row, 64-channel
// quarter); lane = 2 channels.  Split kb + j's (m, l) sits in lane j of
// chunk kb / 32.  The (m, l) of every split and the partial O of the first
// kDepth splits are loaded together, one memory round trip for up to kDepth
// splits (with kDepth = 64, later chunks of 32 take one more each); then
// M = max m, the weights 2^(m - M), and the sums in split order, so the
// result does not depend on timing, nor on kDepth.  kDepth is the smallest
// of 16, 32, 64 that covers the launch's largest split count: the partials
// in flight take 2 kDepth registers a lane, and a batch of short sequences
// (many rows, few splits each) runs more warps per SM with fewer.

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

template <int kDepth>
__global__ void __launch_bounds__(256) split_combine_kernel(const __grid_constant__ CombineParams p) {
  static_assert(kDepth == 16 || kDepth == 32 || kDepth == 64, "depth");
  grid_dep_wait();
  grid_dep_launch();
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int quarter = gw & 3, row_id = gw >> 2;
  int s = 0, base = 0;
  while (s < p.n_seqs && row_id >= base + p.hkv * p.R) {
    base += p.hkv * p.R;
    ++s;
  }
  if (s >= p.n_seqs) return;
  const int h = (row_id - base) / p.R, r = (row_id - base) % p.R;
  const SeqDesc& sd = p.seq[s];
  const int u0 = sd.unit_base + h * sd.splits, splits = sd.splits;
  const float2* ml = reinterpret_cast<const float2*>(p.ml);
  const int64_t split_stride = (int64_t)p.R * kHeadDim;
  const float* src = p.o_part + (int64_t)u0 * split_stride + (int64_t)r * kHeadDim + quarter * 64 + lane * 2;
  // (m, l) of every split, 32 per register: at most kMaxChunks * 32 splits
  // (kDepth <= 32: the launch has at most kDepth splits per head)
  constexpr int kMaxChunks = kDepth == 64 ? kMaxSplitsPerHead / 32 : 1;
  float2 mlv[kMaxChunks];
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) {
    const int k = c * 32 + lane;
    mlv[c] = k < splits ? ml[(int64_t)(u0 + k) * p.R + r] : make_float2(-INFINITY, 0.f);
  }
  // the first kDepth partials, in flight with the (m, l) loads
  constexpr int kA = kDepth < 32 ? kDepth : 32;
  float2 oa[kA], ob[kDepth == 64 ? 32 : 1];
#pragma unroll
  for (int j = 0; j < kA; ++j)
    oa[j] = j < splits ? *reinterpret_cast<const float2*>(src + j * split_stride) : make_float2(0.f, 0.f);
  if constexpr (kDepth == 64) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      ob[j] = 32 + j < splits ? *reinterpret_cast<const float2*>(src + (32 + j) * split_stride) : make_float2(0.f, 0.f);
  }
  float M = -INFINITY;
#pragma unroll
  for (int c = 0; c < kMaxChunks; ++c) M = fmaxf(M, mlv[c].x);
  M = wmax(M);
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
      for (int j = 0; j < 32; ++j)
        oa[j] = j < n ? *reinterpret_cast<const float2*>(sp + j * split_stride) : make_float2(0.f, 0.f);
      combine_chunk(oa, w, acc0, acc1);
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const int node = r / p.G, qh = h * p.G + r % p.G;
  *reinterpret_cast<__half2*>(p.o + (((int64_t)s * p.T + node) * p.hq + qh) * kHeadDim + quarter * 64 + lane * 2) =
      __floats2half2_rn(acc0 * inv, acc1 * inv);
}

cudaError_t launch_split_combine(const CombineParams& p, cudaStream_t s) {
  const int warps = p.n_seqs * p.hkv * p.R * 4;  // four channel quarters per row
  int max_splits = 0;
  for (int i = 0; i < p.n_seqs; ++i) max_splits = max(max_splits, p.seq[i].splits);
  const int blocks = (warps + 7) / 8;
  if (max_splits <= 16) return launch_pdl(split_combine_kernel<16>, blocks, 256, 0, s, p);
  if (max_splits <= 32) return launch_pdl(split_combine_kernel<32>, blocks, 256, 0, s, p);
  return launch_pdl(split_combine_kernel<64>, blocks, 256, 0, s, p);
}

// ---------------------------------------------------------------------------
// Prefill (next row f2): chain trees, parent[c][i] = i - 1 for chunks of t
// prompt tokens, whose ancestor-or-self masks are the causal mask.

__global__ void __launch_bounds__(256) chain_parents_t_kernel(int32_t* parent, int chunks, int t) {
  grid_dep_wait();
  grid_dep_launch();
  const int i = blockIdx.x * 256 + threadIdx.x;
  if (i < chunks * t) parent[i] = (i % t) - 1;
}

cudaError_t launch_chain_parents(int32_t* parent, int chunks, int t, cudaStream_t s) {
  const int n = chunks * t;
  return launch_pdl(chain_parents_t_kernel, (n + 255) / 256, 256, 0, s, parent, chunks, t);
}

}  // namespace stv
