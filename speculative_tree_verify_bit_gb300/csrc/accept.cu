// accept.cu -- a6 tree_accept: exact greedy acceptance of a token tree
// ("elpis" README, "Why fast": commit the longest matching path + 1;
// "elpis-lossless" README, "How": 7 nodes ranked best first; "Lossless":
// token ids compared exactly, nothing sampled or thresholded).
//
// One warp per sequence, lane i = node i (T <= 32).  The match of every edge
// and each node's depth propagate down the tree by warp shuffles; the longest
// fully matching root path is a warp max; ties are broken toward the
// lexicographically smallest node-index sequence by narrowing the candidates
// one depth at a time with warp min reductions.  Every shuffle is executed by
// all 32 lanes, so nothing diverges around a collective.
#include "stv_device.cuh"

namespace stv {

__global__ void __launch_bounds__(32) tree_accept_kernel(const int32_t* __restrict__ parent,
                                                         const int32_t* __restrict__ draft,
                                                         const int32_t* __restrict__ argmax, int T,
                                                         int32_t* __restrict__ n_commit, int32_t* __restrict__ path,
                                                         int32_t* __restrict__ out_ids, int32_t* status) {
  grid_dep_wait();
  grid_dep_launch();
  const unsigned full = 0xffffffffu;
  const int s = blockIdx.x, i = threadIdx.x;
  const bool act = i < T;
  const int64_t at = (int64_t)s * T + i;
  const int par = act ? __ldg(parent + at) : -1;
  const int dr = act ? __ldg(draft + at) : 0;
  const int am = act ? __ldg(argmax + at) : 0;

  const bool bad = act && (i == 0 ? par != -1 : (par < 0 || par >= i));
  if (__any_sync(full, bad)) {
    if (act) {
      path[at] = -1;
      out_ids[at] = -1;
    }
    if (i == 0) {
      n_commit[s] = 0;
      report(status, STV_DEV_BAD_TREE);
    }
    return;
  }
  const int pl = par < 0 ? 0 : par;  // lane holding the parent
  // Every lane executes the shuffle (no short-circuit around a collective).
  const int parent_am = __shfl_sync(full, am, pl);
  const bool match = (i == 0) || (act && dr == parent_am);

  // ok: every edge root -> i matches; depth: edges from the root.
  int ok = (i == 0) ? 1 : 0, depth = 0;
  for (int it = 0; it < T; ++it) {
    int okp = __shfl_sync(full, ok, pl);
    int dp = __shfl_sync(full, depth, pl);
    if (act && i > 0) {
      ok = match && okp;
      depth = dp + 1;
    }
  }
  const int maxd = __reduce_max_sync(full, (act && ok) ? depth : -1);
  bool cand = act && ok && depth == maxd;

  // Narrow the candidates to the lexicographically smallest root path.
  for (int L = 1; L <= maxd; ++L) {
    int a = i;
    for (int st = 0; st < T; ++st) {
      int pa = __shfl_sync(full, par, a & 31);
      if (st < depth - L) a = pa;
    }
    unsigned key = cand ? (unsigned)a : 0xffffffffu;
    unsigned mn = __reduce_min_sync(full, key);
    cand = cand && (unsigned)a == mn;
  }
  const int best = (int)__reduce_min_sync(full, cand ? (unsigned)i : 0xffffffffu);

  // Lane d <= maxd: the path node at depth d.
  int a = best;
  for (int st = 0; st < T; ++st) {
    int pa = __shfl_sync(full, par, a & 31);
    if (st < maxd - i) a = pa;
  }
  const int next = __shfl_sync(full, a, (i + 1) & 31);          // path node at depth i + 1
  const int next_draft = __shfl_sync(full, dr, next & 31);      // its draft id
  const int best_am = __shfl_sync(full, am, best & 31);         // bonus token
  if (act) {
    if (i <= maxd) {
      path[at] = a;
      out_ids[at] = (i < maxd) ? next_draft : best_am;
    } else {
      path[at] = -1;
      out_ids[at] = -1;
    }
  }
  if (i == 0) n_commit[s] = maxd + 1;
}

cudaError_t launch_tree_accept(const int32_t* parent, const int32_t* draft, const int32_t* argmax, int T, int n_seqs,
                               int32_t* n_commit, int32_t* path, int32_t* out_ids, int32_t* status, cudaStream_t s) {
  return launch_pdl(tree_accept_kernel, n_seqs, 32, 0, s, parent, draft, argmax, T, n_commit, path, out_ids, status);
}

}  // namespace stv
