// kv_pack.cu -- a1 kv_append_pack and a7 kv_commit.
//
// kv_append_pack quantizes fp16 K/V rows into the paged 3-bit cache ("elpis"
// README, header table: 3-bit KV cache, 12 KiB per token over 16 layers).
// One CTA per (row, KV head); thread = channel, warp = one 32-channel group
// (append_row_channel in stv_device.cuh, shared with the verify kernel, which
// packs the round's tree rows itself in stv_append_verify_attn).
//
// kv_commit moves the accepted rows to ctx .. ctx + n_commit - 1 ("elpis"
// README, "Why fast": commit the longest matching path + 1).  One CTA per
// (sequence, layer, KV head) reads every source row into shared memory before
// writing any destination, because a destination slot can be the source slot
// of a later row.  A sequence whose path or pages are bad is left untouched
// in every layer (and its ctx_dev entry too): each CTA validates all of it
// before writing anything.
#include "stv_device.cuh"

namespace stv {

__global__ void __launch_bounds__(256) kv_append_kernel(const __grid_constant__ AppendParams p) {
  grid_dep_wait();
  grid_dep_launch();
  const int row = blockIdx.x / p.hkv, h = blockIdx.x % p.hkv;
  const int c = threadIdx.x;
  // The row's values first: they depend on nothing else, so their memory
  // round trip overlaps the row's sequence/position and page-table reads.
  const int64_t src = ((int64_t)row * p.hkv + h) * kHeadDim + c;
  const float xk = __half2float(p.k[src]), xv = __half2float(p.v[src]);
  const int s = __ldg(p.row_seq + row), pos = __ldg(p.row_pos + row);
  if (s < 0 || s >= p.n_seqs || pos < 0) {
    if (c == 0) report(p.status, STV_DEV_BAD_ROW);
    return;
  }
  uint8_t* hb = const_cast<uint8_t*>(
      head_block(p.seq[s], p.pool, p.page_bytes, p.pool_pages, pos, h, c == 0 ? p.status : nullptr));
  if (!hb) return;
  const int slot = pos & (kPageTok - 1);
  append_row_channel(xk, xv, hb, slot, c);
}

// The int4 per-token-head cache (include/stv.h, group 256): one CTA per
// (row, KV head), thread = channel.  The scale is fp16(max|x| / 7) over the
// whole row: an IEEE single division whose result is never within rounding
// of an fp16 midpoint (m / 7 with m an fp16 value is at least 1/7 of a
// half-ulp away from one), so rounding it to fp16 equals rounding m / 7
// directly.  K: a word holds 8 channels, OR-reduced over 8 lanes; V: a word
// holds one channel's codes for 8 tokens, read-modify-written with atomics
// (rows appended in the same launch may share it; their nibbles differ).
__global__ void __launch_bounds__(256) kv_append_i4_kernel(const __grid_constant__ AppendParams p) {
  grid_dep_wait();
  grid_dep_launch();
  const int row = blockIdx.x / p.hkv, h = blockIdx.x % p.hkv;
  const int c = threadIdx.x, lane = c & 31, warp = c >> 5;
  __shared__ float red[2][kHeadDim / 32];
  // the row's values first (see kv_append_kernel)
  const int64_t src = ((int64_t)row * p.hkv + h) * kHeadDim + c;
  const float xk = __half2float(p.k[src]), xv = __half2float(p.v[src]);
  const int s = __ldg(p.row_seq + row), pos = __ldg(p.row_pos + row);
  if (s < 0 || s >= p.n_seqs || pos < 0) {
    if (c == 0) report(p.status, STV_DEV_BAD_ROW);
    return;
  }
  uint8_t* hb = const_cast<uint8_t*>(head_block(p.seq[s], p.pool, p.page_bytes, p.pool_pages, pos, h,
                                                c == 0 ? p.status : nullptr, kI4HeadBytes));
  if (!hb) return;
  const int slot = pos & (kPageTok - 1);
  const float mk = warp_max(fabsf(xk)), mv = warp_max(fabsf(xv));
  if (lane == 0) {
    red[0][warp] = mk;
    red[1][warp] = mv;
  }
  __syncthreads();
  float m0 = 0.f, m1 = 0.f;
#pragma unroll
  for (int w = 0; w < kHeadDim / 32; ++w) {
    m0 = fmaxf(m0, red[0][w]);
    m1 = fmaxf(m1, red[1][w]);
  }
  const __half sk = __float2half_rn(__fdiv_rn(m0, 7.f)), sv = __float2half_rn(__fdiv_rn(m1, 7.f));
  // K: channel c is element c % 8 of word c / 8
  uint32_t kw = (uint32_t)quant_code_i4(xk, __half2float(sk)) << i4_pos(c & 7);
  kw |= __shfl_xor_sync(0xffffffffu, kw, 1);
  kw |= __shfl_xor_sync(0xffffffffu, kw, 2);
  kw |= __shfl_xor_sync(0xffffffffu, kw, 4);
  if ((c & 7) == 0) *reinterpret_cast<uint32_t*>(hb + kI4OffKCodes + slot * 128 + (c >> 3) * 4) = kw;
  // V: token `slot` is element slot % 8 of channel c's word for its 8 tokens
  const int tile = slot / kTileTok, within = slot % kTileTok;
  uint32_t* wp = reinterpret_cast<uint32_t*>(hb + kI4OffVCodes + tile * kI4VTileCodeBytes + c * 32 + (within / 8) * 4);
  const int sh = i4_pos(within & 7);
  atomicAnd(wp, ~(15u << sh));
  atomicOr(wp, (uint32_t)quant_code_i4(xv, __half2float(sv)) << sh);
  if (c == 0) {
    *reinterpret_cast<__half*>(hb + kI4OffKScales + slot * 2) = sk;
    *reinterpret_cast<__half*>(hb + kI4OffVScales + slot * 2) = sv;
  }
}

// The K 4 / V 2-bit cache (include/stv.h, STV_KV_K4V2): one CTA per (row, KV
// head), thread = channel, warp = 32-channel group.  The 3-bit quantizer at
// 4 bits (K: s = fp16(max / 8), codes -8..7) and 2 bits (V: s = fp16(max /
// 2), codes -2..1); max / 8 and max / 2 are exact in fp32, so rounding them
// to fp16 is fp16(max / h).  The division-free exact rounding of
// rne_quotient gives the codes.  K: a word holds 8 channels, OR-reduced over
// 8 lanes.  V: a word holds one channel's codes for 16 tokens; rows appended
// in the same launch may share it (their bits differ), so it is updated
// with atomics.
__global__ void __launch_bounds__(256) kv_append_k4v2_kernel(const __grid_constant__ AppendParams p) {
  grid_dep_wait();
  grid_dep_launch();
  const int row = blockIdx.x / p.hkv, h = blockIdx.x % p.hkv;
  const int c = threadIdx.x, lane = c & 31, g = c >> 5;
  // the row's values first (see kv_append_kernel)
  const int64_t src = ((int64_t)row * p.hkv + h) * kHeadDim + c;
  const float xk = __half2float(p.k[src]), xv = __half2float(p.v[src]);
  const int s = __ldg(p.row_seq + row), pos = __ldg(p.row_pos + row);
  if (s < 0 || s >= p.n_seqs || pos < 0) {
    if (c == 0) report(p.status, STV_DEV_BAD_ROW);
    return;
  }
  uint8_t* hb = const_cast<uint8_t*>(
      head_block(p.seq[s], p.pool, p.page_bytes, p.pool_pages, pos, h, c == 0 ? p.status : nullptr, kKv2HeadBytes));
  if (!hb) return;
  const int slot = pos & (kPageTok - 1);
  // K, 4 bits
  const __half sk = __float2half_rn(warp_max(fabsf(xk)) * 0.125f);
  const float skf = __half2float(sk);
  const int uk = (skf == 0.f ? 0 : min(max(rne_quotient(xk, skf), -8), 7)) + 8;
  uint32_t kw = (uint32_t)uk << i4_pos(lane & 7);
  kw |= __shfl_xor_sync(0xffffffffu, kw, 1);
  kw |= __shfl_xor_sync(0xffffffffu, kw, 2);
  kw |= __shfl_xor_sync(0xffffffffu, kw, 4);
  if ((lane & 7) == 0)
    *reinterpret_cast<uint32_t*>(hb + kKv2OffKCodes + slot * 128 + g * 16 + (lane >> 3) * 4) = kw;
  if (lane == 0) *reinterpret_cast<__half*>(hb + kKv2OffKScales + slot * 16 + g * 2) = sk;
  // V, 2 bits
  const __half sv = __float2half_rn(warp_max(fabsf(xv)) * 0.5f);
  const float svf = __half2float(sv);
  const uint32_t uv = (uint32_t)((svf == 0.f ? 0 : min(max(rne_quotient(xv, svf), -2), 1)) + 2);
  const int tile = slot / kTileTok, within = slot % kTileTok;
  if (lane == 0)
    *reinterpret_cast<__half*>(hb + kKv2OffVScales + tile * kKv2VTileScaleBytes + g * (kTileTok * 2) + within * 2) = sv;
  uint32_t* wp = reinterpret_cast<uint32_t*>(hb + kKv2OffVCodes + tile * kKv2VTileCodeBytes + c * 16 + (within / 16) * 4);
  const int sh = v2_pos(within & 15);
  atomicAnd(wp, ~(3u << sh));
  atomicOr(wp, uv << sh);
}

cudaError_t launch_kv_append(const AppendParams& p, cudaStream_t s) {
  if (p.n_rows == 0) return cudaSuccess;
  const int blocks = p.n_rows * p.hkv;
  if (p.fmt == kFmtInt4) return launch_pdl(kv_append_i4_kernel, blocks, 256, 0, s, p);
  if (p.fmt == kFmtK4V2) return launch_pdl(kv_append_k4v2_kernel, blocks, 256, 0, s, p);
  return launch_pdl(kv_append_kernel, blocks, 256, 0, s, p);
}

// ---------------------------------------------------------------------------

// Whether every page a sequence's commit touches (sources ctx + path[i] and
// destinations ctx + i, i < n) is in its table and inside every layer's pool
// (min_pool: the smallest pool).  Every CTA of the sequence (one per layer
// and KV head) checks the same entries against the same bound, so they all
// take the same decision: the commit is all or nothing.
__device__ __forceinline__ bool commit_pages_ok(const SeqDesc& sd, const int* path_s, int n, int32_t min_pool) {
  for (int i = 0; i < n; ++i) {
    const int64_t pos[2] = {(int64_t)sd.ctx + path_s[i], (int64_t)sd.ctx + i};
    for (int k = 0; k < 2; ++k) {
      const int64_t lp = pos[k] >> 8;
      if (lp >= sd.n_pages) return false;
      const int32_t page = __ldg(sd.page_table + lp);
      if (page < 0 || page >= min_pool) return false;
    }
  }
  return true;
}

__global__ void __launch_bounds__(256) kv_commit_kernel(const __grid_constant__ CommitParams p) {
  grid_dep_wait();
  grid_dep_launch();
  int b = blockIdx.x;
  const int h = b % p.hkv;
  b /= p.hkv;
  const int layer = b % p.n_layers;
  const int s = b / p.n_layers;
  const int tid = threadIdx.x;
  const bool leader = (layer == 0 && h == 0 && tid == 0);

  __shared__ int path_s[kMaxT];
  __shared__ int n_s, ok_s;
  __shared__ __align__(16) uint8_t krow[kMaxT][112];  // 96 B codes + 16 B scales
  __shared__ __align__(4) __half vscale[kMaxT][kGroups];
  __shared__ uint8_t vcode[kMaxT][kHeadDim];

  if (tid == 0) {
    int n = __ldg(p.n_commit + s);
    int ok = (n >= 1 && n <= p.T);
    int prev = -1;
    for (int i = 0; ok && i < n; ++i) {
      int x = __ldg(p.path + (int64_t)s * p.T + i);
      path_s[i] = x;
      if ((i == 0 && x != 0) || x <= prev || x >= p.T) ok = 0;
      prev = x;
    }
    n_s = n;
    ok_s = ok ? (commit_pages_ok(p.seq[s], path_s, n, p.min_pool_pages) ? 1 : 2) : 0;
  }
  __syncthreads();
  if (ok_s != 1) {
    if (leader) report(p.status, ok_s == 0 ? STV_DEV_BAD_COMMIT : STV_DEV_BAD_PAGE);
    return;
  }
  const int n = n_s;
  const SeqDesc& sd = p.seq[s];
  const uint8_t* pool = p.pools[layer];
  const int32_t pool_pages = p.pool_pages[layer];

  // Read every source row.
  for (int i = 0; i < n; ++i) {
    const int64_t src = (int64_t)sd.ctx + path_s[i];
    const uint8_t* hb = head_block(sd, pool, p.page_bytes, pool_pages, src, h, nullptr);  // validated above
    const int slot = (int)(src & (kPageTok - 1));
    if (tid < 6)
      reinterpret_cast<uint4*>(krow[i])[tid] = reinterpret_cast<const uint4*>(hb + kOffKCodes + slot * 96)[tid];
    else if (tid == 6)
      reinterpret_cast<uint4*>(krow[i])[6] = *reinterpret_cast<const uint4*>(hb + kOffKScales + slot * 16);
    else if (tid >= 8 && tid < 16) {
      const int g = tid - 8, tile = slot / kTileTok, within = slot % kTileTok;
      vscale[i][g] =
          *reinterpret_cast<const __half*>(hb + kOffVScales + tile * kVTileScaleBytes + g * (kTileTok * 2) + within * 2);
    }
    {
      const int tile = slot / kTileTok, within = slot % kTileTok;
      const uint32_t* wp =
          reinterpret_cast<const uint32_t*>(hb + kOffVCodes + tile * kVTileCodeBytes + tid * 24 + (within / 32) * 12);
      vcode[i][tid] = (uint8_t)block_code(wp[0], wp[1], wp[2], within % 32);
    }
  }
  __syncthreads();

  // Write every destination row.
  for (int i = 0; i < n; ++i) {
    const int64_t dst = (int64_t)sd.ctx + i;
    uint8_t* hb = const_cast<uint8_t*>(head_block(sd, pool, p.page_bytes, pool_pages, dst, h, nullptr));
    if (!hb) continue;
    const int slot = (int)(dst & (kPageTok - 1));
    const int tile = slot / kTileTok, within = slot % kTileTok;
    if (tid < 6)
      reinterpret_cast<uint4*>(hb + kOffKCodes + slot * 96)[tid] = reinterpret_cast<const uint4*>(krow[i])[tid];
    else if (tid == 6)
      *reinterpret_cast<uint4*>(hb + kOffKScales + slot * 16) = reinterpret_cast<const uint4*>(krow[i])[6];
    else if (tid >= 8 && tid < 16) {
      const int g = tid - 8;
      *reinterpret_cast<__half*>(hb + kOffVScales + tile * kVTileScaleBytes + g * (kTileTok * 2) + within * 2) =
          vscale[i][g];
    }
    // Channel `tid` owns its V words in this head: plain read-modify-write.
    uint32_t* wp = reinterpret_cast<uint32_t*>(hb + kOffVCodes + tile * kVTileCodeBytes + tid * 24 + (within / 32) * 12);
    const int code = vcode[i][tid], pos = within % 32;
#pragma unroll
    for (int bb = 0; bb < 3; ++bb) {
      int wd, bt;
      bit_place(pos, bb, wd, bt);
      wp[wd] = (wp[wd] & ~(1u << bt)) | ((uint32_t)((code >> bb) & 1) << bt);
    }
  }
  if (leader && p.ctx_dev) p.ctx_dev[s] += n;
}

// kv_commit for the int4 per-token-head cache: the same protocol as above
// (validate the path, read every source row, then write), moving each row's
// K codes and both scales whole and its V code channel by channel.
__global__ void __launch_bounds__(256) kv_commit_i4_kernel(const __grid_constant__ CommitParams p) {
  grid_dep_wait();
  grid_dep_launch();
  int b = blockIdx.x;
  const int h = b % p.hkv;
  b /= p.hkv;
  const int layer = b % p.n_layers;
  const int s = b / p.n_layers;
  const int tid = threadIdx.x;
  const bool leader = (layer == 0 && h == 0 && tid == 0);

  __shared__ int path_s[kMaxT];
  __shared__ int n_s, ok_s;
  __shared__ __align__(16) uint8_t krow[kMaxT][128];  // K codes
  __shared__ __align__(4) __half scl[kMaxT][2];       // K and V scales
  __shared__ uint8_t vcode[kMaxT][kHeadDim];

  if (tid == 0) {
    int n = __ldg(p.n_commit + s);
    int ok = (n >= 1 && n <= p.T);
    int prev = -1;
    for (int i = 0; ok && i < n; ++i) {
      int x = __ldg(p.path + (int64_t)s * p.T + i);
      path_s[i] = x;
      if ((i == 0 && x != 0) || x <= prev || x >= p.T) ok = 0;
      prev = x;
    }
    n_s = n;
    ok_s = ok ? (commit_pages_ok(p.seq[s], path_s, n, p.min_pool_pages) ? 1 : 2) : 0;
  }
  __syncthreads();
  if (ok_s != 1) {
    if (leader) report(p.status, ok_s == 0 ? STV_DEV_BAD_COMMIT : STV_DEV_BAD_PAGE);
    return;
  }
  const int n = n_s;
  const SeqDesc& sd = p.seq[s];
  const uint8_t* pool = p.pools[layer];
  const int32_t pool_pages = p.pool_pages[layer];

  for (int i = 0; i < n; ++i) {
    const int64_t src = (int64_t)sd.ctx + path_s[i];
    const uint8_t* hb = head_block(sd, pool, p.page_bytes, pool_pages, src, h, nullptr, kI4HeadBytes);  // validated
    const int slot = (int)(src & (kPageTok - 1)), tile = slot / kTileTok, within = slot % kTileTok;
    if (tid < 8)
      reinterpret_cast<uint4*>(krow[i])[tid] = reinterpret_cast<const uint4*>(hb + kI4OffKCodes + slot * 128)[tid];
    else if (tid == 8)
      scl[i][0] = *reinterpret_cast<const __half*>(hb + kI4OffKScales + slot * 2);
    else if (tid == 9)
      scl[i][1] = *reinterpret_cast<const __half*>(hb + kI4OffVScales + slot * 2);
    const uint32_t w =
        *reinterpret_cast<const uint32_t*>(hb + kI4OffVCodes + tile * kI4VTileCodeBytes + tid * 32 + (within / 8) * 4);
    vcode[i][tid] = (uint8_t)((w >> i4_pos(within & 7)) & 15u);
  }
  __syncthreads();

  for (int i = 0; i < n; ++i) {
    const int64_t dst = (int64_t)sd.ctx + i;
    uint8_t* hb = const_cast<uint8_t*>(head_block(sd, pool, p.page_bytes, pool_pages, dst, h, nullptr, kI4HeadBytes));
    if (!hb) continue;
    const int slot = (int)(dst & (kPageTok - 1)), tile = slot / kTileTok, within = slot % kTileTok;
    if (tid < 8)
      reinterpret_cast<uint4*>(hb + kI4OffKCodes + slot * 128)[tid] = reinterpret_cast<const uint4*>(krow[i])[tid];
    else if (tid == 8)
      *reinterpret_cast<__half*>(hb + kI4OffKScales + slot * 2) = scl[i][0];
    else if (tid == 9)
      *reinterpret_cast<__half*>(hb + kI4OffVScales + slot * 2) = scl[i][1];
    // Channel `tid` owns its V words in this head: plain read-modify-write.
    uint32_t* wp = reinterpret_cast<uint32_t*>(hb + kI4OffVCodes + tile * kI4VTileCodeBytes + tid * 32 + (within / 8) * 4);
    const int sh = i4_pos(within & 7);
    *wp = (*wp & ~(15u << sh)) | ((uint32_t)vcode[i][tid] << sh);
  }
  if (leader && p.ctx_dev) p.ctx_dev[s] += n;
}

// kv_commit for the K 4 / V 2-bit cache: the same protocol (validate the
// path and every page, read every source row, then write), moving each row's
// K codes and both scale rows whole and its V code channel by channel.
__global__ void __launch_bounds__(256) kv_commit_k4v2_kernel(const __grid_constant__ CommitParams p) {
  grid_dep_wait();
  grid_dep_launch();
  int b = blockIdx.x;
  const int h = b % p.hkv;
  b /= p.hkv;
  const int layer = b % p.n_layers;
  const int s = b / p.n_layers;
  const int tid = threadIdx.x;
  const bool leader = (layer == 0 && h == 0 && tid == 0);

  __shared__ int path_s[kMaxT];
  __shared__ int n_s, ok_s;
  __shared__ __align__(16) uint8_t krow[kMaxT][144];  // 128 B codes + 16 B scales
  __shared__ __align__(4) __half vscale[kMaxT][kGroups];
  __shared__ uint8_t vcode[kMaxT][kHeadDim];

  if (tid == 0) {
    int n = __ldg(p.n_commit + s);
    int ok = (n >= 1 && n <= p.T);
    int prev = -1;
    for (int i = 0; ok && i < n; ++i) {
      int x = __ldg(p.path + (int64_t)s * p.T + i);
      path_s[i] = x;
      if ((i == 0 && x != 0) || x <= prev || x >= p.T) ok = 0;
      prev = x;
    }
    n_s = n;
    ok_s = ok ? (commit_pages_ok(p.seq[s], path_s, n, p.min_pool_pages) ? 1 : 2) : 0;
  }
  __syncthreads();
  if (ok_s != 1) {
    if (leader) report(p.status, ok_s == 0 ? STV_DEV_BAD_COMMIT : STV_DEV_BAD_PAGE);
    return;
  }
  const int n = n_s;
  const SeqDesc& sd = p.seq[s];
  const uint8_t* pool = p.pools[layer];
  const int32_t pool_pages = p.pool_pages[layer];

  for (int i = 0; i < n; ++i) {
    const int64_t src = (int64_t)sd.ctx + path_s[i];
    const uint8_t* hb = head_block(sd, pool, p.page_bytes, pool_pages, src, h, nullptr, kKv2HeadBytes);  // validated
    const int slot = (int)(src & (kPageTok - 1)), tile = slot / kTileTok, within = slot % kTileTok;
    if (tid < 8)
      reinterpret_cast<uint4*>(krow[i])[tid] = reinterpret_cast<const uint4*>(hb + kKv2OffKCodes + slot * 128)[tid];
    else if (tid == 8)
      reinterpret_cast<uint4*>(krow[i])[8] = *reinterpret_cast<const uint4*>(hb + kKv2OffKScales + slot * 16);
    else if (tid >= 16 && tid < 24) {
      const int g = tid - 16;
      vscale[i][g] = *reinterpret_cast<const __half*>(hb + kKv2OffVScales + tile * kKv2VTileScaleBytes +
                                                      g * (kTileTok * 2) + within * 2);
    }
    const uint32_t w =
        *reinterpret_cast<const uint32_t*>(hb + kKv2OffVCodes + tile * kKv2VTileCodeBytes + tid * 16 + (within / 16) * 4);
    vcode[i][tid] = (uint8_t)((w >> v2_pos(within & 15)) & 3u);
  }
  __syncthreads();

  for (int i = 0; i < n; ++i) {
    const int64_t dst = (int64_t)sd.ctx + i;
    uint8_t* hb = const_cast<uint8_t*>(head_block(sd, pool, p.page_bytes, pool_pages, dst, h, nullptr, kKv2HeadBytes));
    const int slot = (int)(dst & (kPageTok - 1)), tile = slot / kTileTok, within = slot % kTileTok;
    if (tid < 8)
      reinterpret_cast<uint4*>(hb + kKv2OffKCodes + slot * 128)[tid] = reinterpret_cast<const uint4*>(krow[i])[tid];
    else if (tid == 8)
      *reinterpret_cast<uint4*>(hb + kKv2OffKScales + slot * 16) = reinterpret_cast<const uint4*>(krow[i])[8];
    else if (tid >= 16 && tid < 24) {
      const int g = tid - 16;
      *reinterpret_cast<__half*>(hb + kKv2OffVScales + tile * kKv2VTileScaleBytes + g * (kTileTok * 2) + within * 2) =
          vscale[i][g];
    }
    // Channel `tid` owns its V words in this head: plain read-modify-write.
    uint32_t* wp = reinterpret_cast<uint32_t*>(hb + kKv2OffVCodes + tile * kKv2VTileCodeBytes + tid * 16 + (within / 16) * 4);
    const int sh = v2_pos(within & 15);
    *wp = (*wp & ~(3u << sh)) | ((uint32_t)vcode[i][tid] << sh);
  }
  if (leader && p.ctx_dev) p.ctx_dev[s] += n;
}

cudaError_t launch_kv_commit(const CommitParams& p, cudaStream_t s) {
  const int blocks = p.n_seqs * p.n_layers * p.hkv;
  if (p.fmt == kFmtInt4) return launch_pdl(kv_commit_i4_kernel, blocks, 256, 0, s, p);
  if (p.fmt == kFmtK4V2) return launch_pdl(kv_commit_k4v2_kernel, blocks, 256, 0, s, p);
  return launch_pdl(kv_commit_kernel, blocks, 256, 0, s, p);
}

}  // namespace stv
