// verify_aux.cu -- the kernels around the tensor-core verify kernel: the int8
// Q quantizer (a3), split_combine (a5) and the prefill chain parents.
//
// Sources: "elpis" README, "Why fast" (8-row token tree verified in one pass;
// decode verify with 3-bit K codes as exact int8 against int8 Q); Reddit
// posts (u/iamMess), second post (split-KV verify attention).
#include "combine.cuh"
#include "stv_device.cuh"

namespace stv {

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
  m = warp_max_xor(m);
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
// quarter), the merge of combine.cuh.  kDepth is the smallest of 16, 32, 64
// that covers the launch's largest split count: the partials in flight take
// 2 kDepth registers a lane, and a batch of short sequences (many rows, few
// splits each) runs more warps per SM with fewer.

template <int kDepth>
__global__ void __launch_bounds__(256) split_combine_kernel(const __grid_constant__ CombineParams p) {
  grid_dep_wait();
  grid_dep_launch();
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int quarter = gw & 3, row_id = gw >> 2;
  int s = 0, base = 0;
  while (s < p.n_seqs && row_id >= base + p.hkv * p.R) {
    base += p.hkv * p.R;
    ++s;
  }
  if (s >= p.n_seqs) return;
  const int h = (row_id - base) / p.R, r = (row_id - base) % p.R;
  combine_row_quarter<kDepth, false>(p.seq[s], s, h, r, quarter, p.R, p.T, p.hq, p.G, p.o_part, p.ml, p.o);
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
