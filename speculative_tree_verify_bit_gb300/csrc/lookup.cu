// lookup.cu -- lookup drafting (next row f4): propose the tokens that
// followed the most recent earlier occurrence of the history's last
// max_len .. min_len tokens.
//
// Sources: Reddit posts (u/iamMess), "Now added" list, lookup-augmented
// drafting (draft tokens copied from earlier in the same request, where its
// trailing six to twelve tokens last appeared); syv-ai README (mirror),
// SPEC=dflash2 section (verify slots past the drafter's come from the
// request's own context).
//
// One pass over the history.  A candidate is the END position e of an
// earlier occurrence (e <= n - 2); its backward match length is
// m(e) = the number of tokens h[e], h[e-1], ... equal to h[n-1], h[n-2], ...,
// capped at max_len.  The answer is the candidate with the largest
// min(m, max_len) >= min_len and, among those, the largest e: one maximum
// over the 64-bit keys (m << 32) | e.  Each CTA stages a chunk of the history
// (plus max_len - 1 tokens to its left) in shared memory with coalesced
// loads, reduces its chunk, and folds the result into the sequence's key
// with a 64-bit atomicMax.  The last CTA of a sequence to finish (a done
// counter; no CTA ever waits for another) writes the proposal and sets the
// sequence's key and counter back to zero, so the workspace, zero before the
// first call, is zero before every call (no clearing launch).  It reads
// 4 bytes of history per token; at one request's history (a megabyte at 262K
// tokens) the call is bound by launch and load latency rather than bandwidth.
#include <stdint.h>
#include <string.h>

#include "stv.h"

namespace stv {
namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 2048;  // candidate end positions per CTA
constexpr int kMaxLen = 32;
constexpr int kMaxK = 64;

struct LookupParams {
  const int32_t* tok[STV_MAX_SEQS];
  int64_t n[STV_MAX_SEQS];
  int cta_base[STV_MAX_SEQS + 1];  // first CTA of each sequence; [n_seqs] = grid size
  int n_seqs, min_len, max_len, k;
  int32_t* n_prop;
  int32_t* prop;
  int32_t* match_len;
  int64_t* match_pos;
  unsigned long long* key;  // per sequence, zero at launch, left zero
  unsigned int* done;       // per sequence, zero at launch, left zero
};

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const unsigned long long y = __shfl_xor_sync(0xffffffffu, x, o);
    x = y > x ? y : x;
  }
  return x;
}

__global__ void __launch_bounds__(kThreads) lookup_kernel(const __grid_constant__ LookupParams p) {
  __shared__ int32_t win[kChunk + kMaxLen];
  __shared__ int32_t suf[kMaxLen];  // suf[i] = h[n - 1 - i]
  __shared__ unsigned long long red[kThreads / 32];
  __shared__ unsigned long long final_key;
  __shared__ int is_last;
  const int tid = threadIdx.x;
  int s = 0;
  while (s + 1 < p.n_seqs && (int)blockIdx.x >= p.cta_base[s + 1]) ++s;
  const int chunk = blockIdx.x - p.cta_base[s];
  const int n_chunks = p.cta_base[s + 1] - p.cta_base[s];
  const int32_t* h = p.tok[s];
  const int64_t n = p.n[s];
  const int max_len = p.max_len;

  // candidates e in [e0, e1), e <= n - 2; the window holds h[w0 .. e1 - 1]
  const int64_t e0 = (int64_t)chunk * kChunk;
  const int64_t e1 = e0 + kChunk < n - 1 ? e0 + kChunk : n - 1;
  const int64_t w0 = e0 - (max_len - 1);
  if (tid < max_len) suf[tid] = n - 1 - tid >= 0 ? h[n - 1 - tid] : 0;
  for (int64_t j = tid; j < e1 - w0; j += kThreads) {
    const int64_t pos = w0 + j;
    win[j] = pos >= 0 ? h[pos] : 0;  // positions left of 0 are never compared
  }
  __syncthreads();

  unsigned long long best = 0;
  const int32_t last = suf[0];
  for (int64_t e = e0 + tid; e < e1; e += kThreads) {
    if (win[e - w0] != last) continue;
    int m = 1;
    while (m < max_len && m <= e && win[e - m - w0] == suf[m]) ++m;
    if (m >= p.min_len) {
      const unsigned long long key = ((unsigned long long)m << 32) | (unsigned long long)e;
      best = key > best ? key : best;
    }
  }
  best = warp_max_u64(best);
  if ((tid & 31) == 0) red[tid >> 5] = best;
  __syncthreads();
  if (tid == 0) {
    unsigned long long b = 0;
    for (int w = 0; w < kThreads / 32; ++w) b = red[w] > b ? red[w] : b;
    if (b) atomicMax(p.key + s, b);
    __threadfence();  // the key is visible before this CTA counts itself done
    is_last = atomicAdd(p.done + s, 1u) == (unsigned)(n_chunks - 1);
  }
  __syncthreads();
  if (!is_last) return;

  // ---- last CTA of sequence s: write the proposal ----
  // One thread reads the final key (every other CTA of this sequence has
  // folded in its key and counted itself) and sets the key and the counter
  // back to zero for the next call; the CTA reads the key from shared memory.
  if (tid == 0) {
    __threadfence();
    final_key = atomicAdd(p.key + s, 0ull);
    p.key[s] = 0ull;
    p.done[s] = 0u;
  }
  __syncthreads();
  const unsigned long long key = final_key;
  const int L = (int)(key >> 32);
  const int64_t e = (int64_t)(key & 0xffffffffull);
  const int64_t avail = L ? n - 1 - e : 0;
  const int cnt = (int)(avail < p.k ? avail : p.k);
  for (int j = tid; j < p.k; j += kThreads) p.prop[(int64_t)s * p.k + j] = j < cnt ? h[e + 1 + j] : 0;
  if (tid == 0) {
    p.n_prop[s] = cnt;
    p.match_len[s] = L;
    p.match_pos[s] = L ? e - L + 1 : -1;
  }
}

}  // namespace
}  // namespace stv

extern "C" int stv_lookup_workspace_bytes(int n_seqs, size_t* bytes) {
  if (!bytes || n_seqs < 1 || n_seqs > STV_MAX_SEQS) return STV_ERR_INVALID_ARG;
  *bytes = (size_t)n_seqs * (sizeof(unsigned long long) + sizeof(unsigned int));
  return STV_OK;
}

extern "C" int stv_lookup_draft(const stv_history* hist, int n_seqs, int min_len, int max_len, int k, int32_t* n_prop,
                                int32_t* prop, int32_t* match_len, int64_t* match_pos, void* workspace,
                                size_t ws_bytes, stv_stream_t stream) {
  using namespace stv;
  size_t need = 0;
  if (stv_lookup_workspace_bytes(n_seqs, &need) != STV_OK || !hist) return STV_ERR_INVALID_ARG;
  if (min_len < 1 || max_len < min_len || max_len > kMaxLen || k < 0 || k > kMaxK) return STV_ERR_INVALID_ARG;
  if (!n_prop || !match_len || !match_pos || (k > 0 && !prop) || !workspace) return STV_ERR_INVALID_ARG;
  if (ws_bytes < need) return STV_ERR_WORKSPACE_TOO_SMALL;
  LookupParams p;
  memset(&p, 0, sizeof(p));
  int ctas = 0;
  for (int s = 0; s < n_seqs; ++s) {
    if (hist[s].n < 0 || hist[s].n > ((int64_t)1 << 31) || (hist[s].n > 0 && !hist[s].tokens))
      return STV_ERR_INVALID_ARG;
    p.tok[s] = hist[s].tokens;
    p.n[s] = hist[s].n;
    p.cta_base[s] = ctas;
    const int64_t cand = hist[s].n > 1 ? hist[s].n - 1 : 0;  // candidate ends 0 .. n-2
    ctas += cand > 0 ? (int)((cand + kChunk - 1) / kChunk) : 1;
  }
  p.cta_base[n_seqs] = ctas;
  p.n_seqs = n_seqs;
  p.min_len = min_len;
  p.max_len = max_len;
  p.k = k;
  p.n_prop = n_prop;
  p.prop = prop;
  p.match_len = match_len;
  p.match_pos = match_pos;
  p.key = static_cast<unsigned long long*>(workspace);
  p.done = reinterpret_cast<unsigned int*>(static_cast<unsigned long long*>(workspace) + n_seqs);
  cudaStream_t st = (cudaStream_t)stream;
  lookup_kernel<<<ctas, kThreads, 0, st>>>(p);
  return cudaGetLastError() == cudaSuccess ? STV_OK : STV_ERR_CUDA;
}
