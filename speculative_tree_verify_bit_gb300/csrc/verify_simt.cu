// verify_simt.cu -- a2..a5 on CUDA cores: the int8 Q quantizer, a
// straightforward split-KV tree-masked attention kernel, split_combine and the
// int8-dots inspection kernel.
//
// Sources: "elpis" README, "Why fast" (8-row token tree verified in one pass;
// decode verify with 3-bit K codes as exact int8 against int8 Q); Reddit
// posts (u/iamMess), second post (split-KV verify attention).
//
// verify_simt_kernel: one CTA per work unit (sequence, KV head, split), 256
// threads.  Warp w owns rows w, w+8, ... of the T*G rows that share the KV
// head; lane = key within a 32-key sub-tile, so each row's softmax max and
// sum are warp reductions.  K is dequantized to fp16 (exact path) or to the
// exact integers code-4 (int8 path, per-group integer dots, exact in fp32),
// V to fp16; P is rounded to fp16; all sums are fp32.
#include "stv_device.cuh"

namespace stv {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float wmax(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float wsum(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
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
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= n_rows) return;
  quantize_q_row_warp(q + (int64_t)row * kHeadDim, qi + (int64_t)row * kHeadDim, sq + row);
}

cudaError_t launch_quantize_q(const __half* q, int n_rows, int8_t* qi, float* sq, cudaStream_t s) {
  quantize_q_kernel<<<(n_rows + 7) / 8, 256, 0, s>>>(q, n_rows, qi, sq);
  return cudaGetLastError();
}

// Work unit -> (sequence, KV head, split).
__device__ __forceinline__ void locate_unit(const SeqDesc* seq, int n_seqs, int u, int& s, int& h, int& split) {
  s = 0;
  while (s + 1 < n_seqs && u >= seq[s + 1].unit_base) ++s;
  const int local = u - seq[s].unit_base;
  h = local / seq[s].splits;
  split = local % seq[s].splits;
}

// a2: ancestor-or-self bit masks of a tree.  An invalid parent ends the walk
// (and is reported); the walk is bounded by T steps.
__device__ __forceinline__ uint32_t ancestor_mask(const int32_t* parent, int T, int i, int32_t* status) {
  uint32_t m = 1u << i;
  int n = i;
  for (int st = 0; st < T && n > 0; ++st) {
    int pa = __ldg(parent + n);
    if (pa < 0 || pa >= n) {
      report(status, STV_DEV_BAD_TREE);
      break;
    }
    m |= 1u << pa;
    n = pa;
  }
  if (i == 0 && __ldg(parent) != -1) report(status, STV_DEV_BAD_TREE);
  return m;
}

constexpr int kSub = 32;       // keys per sub-tile
constexpr int kKStride = 260;  // floats per K row in shared memory (16-byte rows, no bank conflicts)

template <int RPW>
__global__ void __launch_bounds__(256, 1) verify_simt_kernel(const __grid_constant__ VerifyParams p) {
  extern __shared__ __align__(16) float smem[];
  float* q_s = smem;                         // [8*RPW][256]
  float* k_s = q_s + 8 * RPW * kHeadDim;     // [32][260]
  float* v_s = k_s + kSub * kKStride;        // [32][256]
  float* p_s = v_s + kSub * kHeadDim;        // [8*RPW][32]
  float* sk_s = p_s + 8 * RPW * kSub;        // [32][8]
  __shared__ uint32_t anc_s[kMaxT];
  __shared__ float sq_s[8 * RPW];

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  int s, h, split;
  locate_unit(p.seq, p.n_seqs, blockIdx.x, s, h, split);
  const SeqDesc sd = p.seq[s];
  const int T = p.T, G = p.G, R = p.R;
  const int n_keys = sd.ctx + T;
  const int tok0 = split * p.tiles_per_split * kTileTok;
  const int tok1 = min(n_keys, tok0 + p.tiles_per_split * kTileTok);
  const bool int8 = p.path == STV_PATH_INT8;

  if (tid < T) anc_s[tid] = ancestor_mask(p.parent + (int64_t)s * T, T, tid, split == 0 && h == 0 ? p.status : nullptr);
  for (int idx = tid; idx < 8 * RPW * kHeadDim; idx += 256) {
    const int r = idx / kHeadDim, c = idx % kHeadDim;
    float val = 0.f;
    if (r < R) {
      const int64_t qrow = ((int64_t)s * T + r / G) * p.hq + h * G + r % G;
      val = int8 ? (float)p.qi[qrow * kHeadDim + c] : __half2float(p.q[qrow * kHeadDim + c]);
      if (c == 0) sq_s[r] = int8 ? p.sq[qrow] : 1.f;
    }
    q_s[idx] = val;
  }

  float o[RPW][8], m_r[RPW], l_r[RPW];
#pragma unroll
  for (int k = 0; k < RPW; ++k) {
    m_r[k] = -INFINITY;
    l_r[k] = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) o[k][e] = 0.f;
  }
  __syncthreads();

  for (int t0 = tok0; t0 < tok1; t0 += kSub) {
    // ---- K sub-tile: thread = (key, group) ----
    {
      const int j = tid >> 3, g = tid & 7, tok = t0 + j;
      const uint8_t* hb = tok < tok1 ? head_block(sd, p.pool, p.page_bytes, p.pool_pages, tok, h, p.status) : nullptr;
      float* dst = k_s + j * kKStride + g * kGroup;
      if (hb) {
        const int slot = tok & (kPageTok - 1);
        const uint32_t* wp = reinterpret_cast<const uint32_t*>(hb + kOffKCodes + slot * 96 + g * 12);
        const __half sh = *reinterpret_cast<const __half*>(hb + kOffKScales + slot * 16 + g * 2);
        __half2 out[16];
        if (int8) {
          decode_block_raw(wp[0], wp[1], wp[2], out);
          sk_s[j * 8 + g] = __half2float(sh);
        } else {
          const __half2 s2 = __halves2half2(sh, sh);
          decode_block_h2(wp[0], wp[1], wp[2], [&](int) { return s2; }, out);
        }
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          float2 f = __half22float2(out[m]);
          dst[2 * m] = f.x;
          dst[2 * m + 1] = f.y;
        }
      } else {
#pragma unroll
        for (int e = 0; e < kGroup; ++e) dst[e] = 0.f;
        if (int8) sk_s[j * 8 + g] = 0.f;
      }
    }
    // ---- V sub-tile: thread = channel; the 32 keys are one channel block ----
    {
      const int c = tid;
      const uint8_t* hb = head_block(sd, p.pool, p.page_bytes, p.pool_pages, t0, h, p.status);
      if (hb) {
        const int slot = t0 & (kPageTok - 1), tile = slot / kTileTok, within = slot % kTileTok;
        const uint32_t* wp =
            reinterpret_cast<const uint32_t*>(hb + kOffVCodes + tile * kVTileCodeBytes + c * 24 + (within / 32) * 12);
        const __half2* sp = reinterpret_cast<const __half2*>(hb + kOffVScales + tile * kVTileScaleBytes +
                                                             (c / kGroup) * (kTileTok * 2) + within * 2);
        __half2 out[16];
        decode_block_h2(wp[0], wp[1], wp[2], [&](int m) { return sp[m]; }, out);
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          float2 f = __half22float2(out[m]);
          v_s[(2 * m) * kHeadDim + c] = (t0 + 2 * m < tok1) ? f.x : 0.f;
          v_s[(2 * m + 1) * kHeadDim + c] = (t0 + 2 * m + 1 < tok1) ? f.y : 0.f;
        }
      } else {
        for (int j = 0; j < kSub; ++j) v_s[j * kHeadDim + c] = 0.f;
      }
    }
    __syncthreads();

    // ---- scores: lane = key, warp rows w + 8k ----
    const int tok = t0 + lane;
    float sc[RPW];
#pragma unroll
    for (int k = 0; k < RPW; ++k) sc[k] = 0.f;
    if (!int8) {
      for (int c4 = 0; c4 < kHeadDim / 4; ++c4) {
        const float4 kv = *reinterpret_cast<const float4*>(k_s + lane * kKStride + 4 * c4);
#pragma unroll
        for (int k = 0; k < RPW; ++k) {
          const float4 qv = *reinterpret_cast<const float4*>(q_s + (w + 8 * k) * kHeadDim + 4 * c4);
          sc[k] += qv.x * kv.x + qv.y * kv.y + qv.z * kv.z + qv.w * kv.w;
        }
      }
    } else {
      for (int g = 0; g < kGroups; ++g) {
        float acc[RPW];
#pragma unroll
        for (int k = 0; k < RPW; ++k) acc[k] = 0.f;
        for (int c4 = g * 8; c4 < g * 8 + 8; ++c4) {
          const float4 kv = *reinterpret_cast<const float4*>(k_s + lane * kKStride + 4 * c4);
#pragma unroll
          for (int k = 0; k < RPW; ++k) {
            const float4 qv = *reinterpret_cast<const float4*>(q_s + (w + 8 * k) * kHeadDim + 4 * c4);
            acc[k] += qv.x * kv.x + qv.y * kv.y + qv.z * kv.z + qv.w * kv.w;  // exact integers
          }
        }
        const float skg = sk_s[lane * 8 + g];
#pragma unroll
        for (int k = 0; k < RPW; ++k) sc[k] += skg * acc[k];
      }
    }
#pragma unroll
    for (int k = 0; k < RPW; ++k) {
      const int r = w + 8 * k;
      const int node = r < R ? r / G : 0;
      bool vis = tok < tok1 && r < R;
      if (vis && tok >= sd.ctx) vis = (anc_s[node] >> (tok - sd.ctx)) & 1u;
      const float s2 = vis ? sc[k] * sq_s[r < R ? r : 0] * (kLog2e / 16.f) : -INFINITY;
      const float m_new = fmaxf(m_r[k], wmax(s2));
      float pk = 0.f, corr = 1.f;
      if (m_new != -INFINITY) {
        corr = exp2f(m_r[k] - m_new);
        pk = exp2f(s2 - m_new);
      }
      l_r[k] = l_r[k] * corr + wsum(pk);
      m_r[k] = m_new;
      p_s[r * kSub + lane] = __half2float(__float2half_rn(pk));
#pragma unroll
      for (int e = 0; e < 8; ++e) o[k][e] *= corr;
    }
    __syncwarp();
    // ---- P . V ----
    for (int j = 0; j < kSub; ++j) {
      float vv[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) vv[e] = v_s[j * kHeadDim + lane + 32 * e];
#pragma unroll
      for (int k = 0; k < RPW; ++k) {
        const float pv = p_s[(w + 8 * k) * kSub + j];
#pragma unroll
        for (int e = 0; e < 8; ++e) o[k][e] += pv * vv[e];
      }
    }
    __syncthreads();
  }

  const int u = blockIdx.x;
#pragma unroll
  for (int k = 0; k < RPW; ++k) {
    const int r = w + 8 * k;
    if (r >= R) continue;
    float* dst = p.o_part + ((int64_t)u * R + r) * kHeadDim;
#pragma unroll
    for (int e = 0; e < 8; ++e) dst[lane + 32 * e] = o[k][e];
    if (lane == 0) {
      p.ml[((int64_t)u * R + r) * 2] = m_r[k];
      p.ml[((int64_t)u * R + r) * 2 + 1] = l_r[k];
    }
  }
}

template <int RPW>
static cudaError_t launch_simt(const VerifyParams& p, cudaStream_t s) {
  const size_t smem = sizeof(float) * (8 * RPW * kHeadDim + kSub * kKStride + kSub * kHeadDim + 8 * RPW * kSub + kSub * 8);
  cudaError_t e = cudaFuncSetAttribute(verify_simt_kernel<RPW>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  verify_simt_kernel<RPW><<<p.n_units, 256, smem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_verify(const VerifyParams& p, cudaStream_t s) {
  if (p.R <= 48) return launch_simt<6>(p, s);
  if (p.R <= 96) return launch_simt<12>(p, s);
  return launch_simt<16>(p, s);
}

// ---------------------------------------------------------------------------
// a5: split_combine.  One warp per (sequence, KV head, row); lane = 8 channels.

__global__ void __launch_bounds__(256) split_combine_kernel(const __grid_constant__ CombineParams p) {
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  int s = 0, base = 0;
  while (s < p.n_seqs && gw >= base + p.hkv * p.R) {
    base += p.hkv * p.R;
    ++s;
  }
  if (s >= p.n_seqs) return;
  const int h = (gw - base) / p.R, r = (gw - base) % p.R;
  const SeqDesc& sd = p.seq[s];
  const int u0 = sd.unit_base + h * sd.splits;
  float M = -INFINITY;
  for (int k = 0; k < sd.splits; ++k) M = fmaxf(M, p.ml[((int64_t)(u0 + k) * p.R + r) * 2]);
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, L = 0.f;
  for (int k = 0; k < sd.splits; ++k) {
    const int64_t at = (int64_t)(u0 + k) * p.R + r;
    const float mk = p.ml[at * 2];
    if (mk == -INFINITY) continue;
    const float wk = exp2f(mk - M);
    L += wk * p.ml[at * 2 + 1];
    const float4* src = reinterpret_cast<const float4*>(p.o_part + at * kHeadDim + lane * 8);
    const float4 a = src[0], b = src[1];
    acc[0] += wk * a.x; acc[1] += wk * a.y; acc[2] += wk * a.z; acc[3] += wk * a.w;
    acc[4] += wk * b.x; acc[5] += wk * b.y; acc[6] += wk * b.z; acc[7] += wk * b.w;
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  __align__(16) __half outv[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) outv[e] = __float2half_rn(acc[e] * inv);
  const int node = r / p.G, qh = h * p.G + r % p.G;
  *reinterpret_cast<uint4*>(p.o + (((int64_t)s * p.T + node) * p.hq + qh) * kHeadDim + lane * 8) =
      *reinterpret_cast<const uint4*>(outv);
}

cudaError_t launch_split_combine(const CombineParams& p, cudaStream_t s) {
  int rows = 0;
  for (int i = 0; i < p.n_seqs; ++i) rows += p.hkv * p.R;
  split_combine_kernel<<<(rows + 7) / 8, 256, 0, s>>>(p);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Inspection: exact int8 per-group dots of one Q row against a key range.

__global__ void __launch_bounds__(256) int8_dots_kernel(const __grid_constant__ VerifyParams p, int s,
                                                        const __half* __restrict__ q_row, int q_head, int tok_begin,
                                                        int tok_end, int32_t* __restrict__ dots) {
  __shared__ __align__(16) int8_t qi[kHeadDim];
  __shared__ float sq;
  if (threadIdx.x < 32) quantize_q_row_warp(q_row, qi, &sq);
  __syncthreads();
  const int h = q_head / p.G;
  const int n = tok_end - tok_begin;
  for (int idx = blockIdx.x * 256 + threadIdx.x; idx < n * kGroups; idx += gridDim.x * 256) {
    const int j = idx / kGroups, g = idx % kGroups, tok = tok_begin + j;
    const uint8_t* hb = head_block(p.seq[s], p.pool, p.page_bytes, p.pool_pages, tok, h, p.status);
    int acc = 0;
    if (hb) {
      const int slot = tok & (kPageTok - 1);
      const uint32_t* wp = reinterpret_cast<const uint32_t*>(hb + kOffKCodes + slot * 96 + g * 12);
      __half2 out[16];
      decode_block_raw(wp[0], wp[1], wp[2], out);
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        float2 f = __half22float2(out[m]);
        acc += (int)qi[g * kGroup + 2 * m] * (int)f.x + (int)qi[g * kGroup + 2 * m + 1] * (int)f.y;
      }
    }
    dots[idx] = acc;
  }
}

cudaError_t launch_int8_dots(const VerifyParams& p, int seq, const __half* q_row, int q_head, int tok_begin,
                             int tok_end, int32_t* dots, cudaStream_t s) {
  const int n = (tok_end - tok_begin) * kGroups;
  if (n <= 0) return cudaSuccess;
  int blocks = (n + 255) / 256;
  if (blocks > 1024) blocks = 1024;
  int8_dots_kernel<<<blocks, 256, 0, s>>>(p, seq, q_row, q_head, tok_begin, tok_end, dots);
  return cudaGetLastError();
}

}  // namespace stv
