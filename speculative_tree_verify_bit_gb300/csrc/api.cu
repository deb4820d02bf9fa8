// api.cu -- the extern "C" entry points of include/stv.h: host-side
// validation, the split plan, workspace carve-up and kernel launches.  No
// entry point allocates, frees or synchronises.
#include <string.h>

#include <algorithm>

#include "stv_internal.h"

namespace stv {

static int check_shape(const stv_shape* sh, int t_nodes, ShapeInfo* out) {
  if (!sh) return STV_ERR_INVALID_ARG;
  if (sh->head_dim != kHeadDim || sh->page_tokens != kPageTok) return STV_ERR_SHAPE_UNSUPPORTED;
  if (sh->group != kGroup && sh->group != kGroupI4) return STV_ERR_SHAPE_UNSUPPORTED;
  if (sh->kv_format != STV_KV_BY_GROUP && !(sh->kv_format == STV_KV_K4V2 && sh->group == kGroup))
    return STV_ERR_SHAPE_UNSUPPORTED;
  if (sh->hkv < 1 || sh->hq < sh->hkv || sh->hq % sh->hkv != 0) return STV_ERR_SHAPE_UNSUPPORTED;
  const int G = sh->hq / sh->hkv;
  if (t_nodes >= 0) {
    if (t_nodes < 1 || t_nodes > kMaxT) return STV_ERR_SHAPE_UNSUPPORTED;
    if (t_nodes * G > kMaxRows) return STV_ERR_SHAPE_UNSUPPORTED;
  }
  if (out) {
    out->hq = sh->hq;
    out->hkv = sh->hkv;
    out->G = G;
    out->T = t_nodes;
    out->R = t_nodes * G;
    out->fmt = sh->kv_format == STV_KV_K4V2 ? kFmtK4V2 : (sh->group == kGroupI4 ? kFmtInt4 : kFmtBit3);
  }
  return STV_OK;
}

static int check_layer(const stv_layer_cache* l, const ShapeInfo& sh) {
  if (!l || !l->pool || l->n_pages < 1) return STV_ERR_INVALID_ARG;
  if (l->page_bytes != (int64_t)sh.hkv * (sh.fmt == kFmtInt4 ? kI4HeadBytes : kHeadBytes)) return STV_ERR_SHAPE_UNSUPPORTED;
  return STV_OK;
}

// need_keys < 0: only the table pointer is checked (append: positions are on
// the device); otherwise ctx + need_keys must fit in the sequence's pages.
static int check_seqs(const stv_seq* seqs, int n_seqs, int need_keys) {
  if (!seqs || n_seqs < 1 || n_seqs > STV_MAX_SEQS) return STV_ERR_INVALID_ARG;
  for (int s = 0; s < n_seqs; ++s) {
    if (!seqs[s].page_table || seqs[s].n_pages < 0 || seqs[s].ctx < 0) return STV_ERR_INVALID_ARG;
    if (need_keys >= 0 && (int64_t)seqs[s].ctx + need_keys > (int64_t)seqs[s].n_pages * kPageTok)
      return STV_ERR_INVALID_ARG;
  }
  return STV_OK;
}

static int device_sm_count(int* n) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return STV_ERR_CUDA;
  if (cudaDeviceGetAttribute(n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return STV_ERR_CUDA;
  return STV_OK;
}

// The persistent verify kernel's deal for split k: units longest first (the
// full units of k tiles in unit order, then each sequence's last, shorter
// units, longest first), CTA b taking the b-th, then the (2n - 1 - b)-th,
// ... (snake order over n = min(SMs, units) CTAs).  Returns the makespan in
// tiles, each unit costing its tiles plus kUnitCostTiles (its epilogue and
// the next unit's Q load, about three tiles' time), or -1 past
// kMaxPersistUnits units; fills `order` (unit numbers, sequence-major, then
// KV head, then split) when given.
constexpr int kUnitCostTiles = 3;
static int64_t balanced_deal(const int64_t* tiles, int n_seqs, int hkv, int64_t k, int sm, int16_t* order) {
  int sp[STV_MAX_SEQS], rem[STV_MAX_SEQS], by_rem[STV_MAX_SEQS], base[STV_MAX_SEQS];
  int n = 0;
  for (int s = 0; s < n_seqs; ++s) {
    sp[s] = (int)((tiles[s] + k - 1) / k);
    rem[s] = (int)(tiles[s] - (int64_t)(sp[s] - 1) * k);
    base[s] = n;
    n += hkv * sp[s];
    by_rem[s] = s;
  }
  if (n > kMaxPersistUnits) return -1;
  // sequences by their last unit's length, longest first (ties: lower index)
  for (int i = 1; i < n_seqs; ++i)
    for (int j = i; j > 0 && rem[by_rem[j]] > rem[by_rem[j - 1]]; --j) std::swap(by_rem[j], by_rem[j - 1]);
  const int ctas = std::min(sm, n);
  int64_t load[kMaxPersistUnits];
  for (int b = 0; b < ctas; ++b) load[b] = 0;
  int w = 0;
  auto deal = [&](int unit, int len) {
    const int kk = w / ctas, b = w % ctas;
    load[(kk & 1) ? ctas - 1 - b : b] += len + kUnitCostTiles;
    if (order) order[w] = (int16_t)unit;
    ++w;
  };
  for (int s = 0; s < n_seqs; ++s)  // full units (a last unit of k tiles is one too)
    for (int h = 0; h < hkv; ++h)
      for (int j = 0; j < sp[s]; ++j)
        if (j + 1 < sp[s] || rem[s] == k) deal(base[s] + h * sp[s] + j, (int)k);
  for (int i = 0; i < n_seqs; ++i) {
    const int s = by_rem[i];
    if (rem[s] == k) continue;
    for (int h = 0; h < hkv; ++h) deal(base[s] + h * sp[s] + sp[s] - 1, rem[s]);
  }
  int64_t most = 0;
  for (int b = 0; b < ctas; ++b) most = std::max(most, load[b]);
  return most;
}

// The last balanced plan this thread made, and what it was made for (a
// verify round's calls -- workspace size, verify, merge, for every layer --
// ask for the same plan).
struct PlanMemo {
  bool valid = false;
  int hkv, T, R, fmt, sm, n_seqs;
  int32_t ctx[STV_MAX_SEQS];
  Plan plan;
};

int make_plan(const ShapeInfo& sh, const stv_seq* seqs, int n_seqs, int sm_count, Plan* plan, bool balance) {
  balance = balance && n_seqs > 1 && sh.fmt == kFmtBit3;
  static thread_local PlanMemo memo;
  if (balance && memo.valid && memo.hkv == sh.hkv && memo.T == sh.T && memo.R == sh.R && memo.fmt == sh.fmt &&
      memo.sm == sm_count && memo.n_seqs == n_seqs) {
    bool same = true;
    for (int s = 0; s < n_seqs && same; ++s) same = memo.ctx[s] == seqs[s].ctx;
    if (same) {
      *plan = memo.plan;
      return STV_OK;
    }
  }
  int64_t tiles[STV_MAX_SEQS], total = 0;
  for (int s = 0; s < n_seqs; ++s) {
    tiles[s] = ((int64_t)seqs[s].ctx + sh.T + kTileTok - 1) / kTileTok;
    total += tiles[s] * sh.hkv;
  }
  const int64_t target = sm_count > 0 ? sm_count : 1;
  int64_t k = (total + target - 1) / target;
  if (k < 1) k = 1;
  int64_t k_min = 1;  // at most kMaxSplitsPerHead splits per (sequence, KV head)
  for (int s = 0; s < n_seqs; ++s)
    k_min = std::max<int64_t>(k_min, (tiles[s] + kMaxSplitsPerHead - 1) / kMaxSplitsPerHead);
  k = std::max(k, k_min);
  for (;;) {
    int64_t units = 0;
    for (int s = 0; s < n_seqs; ++s) units += sh.hkv * ((tiles[s] + k - 1) / k);
    if (units <= target || units <= (int64_t)n_seqs * sh.hkv) break;
    ++k;
  }
  // One unit per SM, as above, leaves a batch of unequal sequences waiting
  // for its longest units (each sequence's split count rounds up).  For
  // several sequences on the 3-bit cache, the persistent kernel may take
  // more units than SMs: choose the split whose deal finishes first (ties to
  // the larger split), within kMaxPersistUnits units and 24 MiB of partials.
  plan->persist_ctas = 0;
  if (balance) {
    int64_t best = balanced_deal(tiles, n_seqs, sh.hkv, k, (int)target, nullptr), best_k = k;
    if (best >= 0) {
      for (int64_t kc = k - 1; kc >= std::max(k_min, k / 4); --kc) {
        int64_t units = 0;
        for (int s = 0; s < n_seqs; ++s) units += sh.hkv * ((tiles[s] + kc - 1) / kc);
        if (units > kMaxPersistUnits || units * sh.R * kHeadDim * (int64_t)sizeof(float) > ((int64_t)24 << 20)) break;
        const int64_t cost = balanced_deal(tiles, n_seqs, sh.hkv, kc, (int)target, nullptr);
        if (cost >= 0 && cost < best) {
          best = cost;
          best_k = kc;
        }
      }
      k = best_k;
      balanced_deal(tiles, n_seqs, sh.hkv, k, (int)target, plan->order);
    }
  }
  plan->tiles_per_split = (int)k;
  int base = 0;
  for (int s = 0; s < n_seqs; ++s) {
    plan->splits[s] = (int)((tiles[s] + k - 1) / k);
    plan->unit_base[s] = base;
    base += sh.hkv * plan->splits[s];
  }
  plan->unit_base[n_seqs] = base;
  plan->n_units = base;
  if (balance && base <= kMaxPersistUnits) plan->persist_ctas = (int)std::min<int64_t>(target, base);
  if (balance) {
    memo.valid = true;
    memo.hkv = sh.hkv;
    memo.T = sh.T;
    memo.R = sh.R;
    memo.fmt = sh.fmt;
    memo.sm = sm_count;
    memo.n_seqs = n_seqs;
    for (int s = 0; s < n_seqs; ++s) memo.ctx[s] = seqs[s].ctx;
    memo.plan = *plan;
  }
  return STV_OK;
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

WsLayout ws_layout(const ShapeInfo& sh, int n_seqs, const Plan& plan) {
  WsLayout w;
  const size_t q_rows = (size_t)n_seqs * sh.T * sh.hq;
  size_t at = 0;
  // stv_append_verify_combine's arrival counters: first, at a size fixed by
  // the shape alone, so that calls with other plans on the same workspace
  // never write over them
  w.off_cnt = at;
  at = align256(at + (size_t)(2 + STV_MAX_SEQS * sh.hkv) * sizeof(uint32_t));
  w.off_qi = at;
  at = align256(at + q_rows * kHeadDim);
  w.off_sq = at;
  at = align256(at + q_rows * sizeof(float));
  w.off_opart = at;
  at = align256(at + (size_t)plan.n_units * sh.R * kHeadDim * sizeof(float));
  w.off_ml = at;
  at = align256(at + (size_t)plan.n_units * sh.R * 2 * sizeof(float));
  w.total = at;
  return w;
}

static void fill_seq_descs(SeqDesc* out, const stv_seq* seqs, int n_seqs, const Plan* plan) {
  for (int s = 0; s < n_seqs; ++s) {
    out[s].page_table = seqs[s].page_table;
    out[s].n_pages = seqs[s].n_pages;
    out[s].ctx = seqs[s].ctx;
    out[s].splits = plan ? plan->splits[s] : 0;
    out[s].unit_base = plan ? plan->unit_base[s] : 0;
  }
}

static int to_status(cudaError_t e) { return e == cudaSuccess ? STV_OK : STV_ERR_CUDA; }

}  // namespace stv

using namespace stv;

// Prefill launch planning (used by stv_prefill_* below).
namespace {

constexpr size_t kParentsBytes = ((size_t)STV_MAX_SEQS * kMaxT * sizeof(int32_t) + 255) / 256 * 256;

int prefill_chunk_tokens(const stv_shape* sh) {
  const int g = sh->hq / sh->hkv;
  const int c = 128 / g;
  return c < kMaxT ? c : kMaxT;
}

// The launches of a prefill: for each, the first prompt token, the chunk
// size and the number of chunks.  Full chunks go STV_MAX_SEQS at a time; a
// last partial chunk gets a launch of its own.
struct PrefillLaunch {
  int start, t, count;
};

template <typename F>
int for_each_prefill_launch(int n_tokens, int c, F&& f) {
  int start = 0;
  while (start < n_tokens) {
    const int full = (n_tokens - start) / c;
    PrefillLaunch pl;
    pl.start = start;
    if (full > 0) {
      pl.t = c;
      pl.count = full < STV_MAX_SEQS ? full : STV_MAX_SEQS;
    } else {
      pl.t = n_tokens - start;
      pl.count = 1;
    }
    if (int rc = f(pl)) return rc;
    start += pl.t * pl.count;
  }
  return STV_OK;
}

void prefill_seqs(const stv_seq* seq, const PrefillLaunch& pl, stv_seq* out) {
  for (int i = 0; i < pl.count; ++i) {
    out[i] = *seq;
    out[i].ctx = seq->ctx + pl.start + i * pl.t;
  }
}

}  // namespace

extern "C" {

const char* stv_status_string(int status) {
  switch (status) {
    case STV_OK: return "STV_OK";
    case STV_ERR_INVALID_ARG: return "STV_ERR_INVALID_ARG";
    case STV_ERR_SHAPE_UNSUPPORTED: return "STV_ERR_SHAPE_UNSUPPORTED";
    case STV_ERR_WORKSPACE_TOO_SMALL: return "STV_ERR_WORKSPACE_TOO_SMALL";
    case STV_ERR_CUDA: return "STV_ERR_CUDA";
    case STV_ERR_UNIMPLEMENTED: return "STV_ERR_UNIMPLEMENTED";
    default: return "STV_ERR_UNKNOWN";
  }
}

int stv_version(void) { return 2; }

int stv_page_bytes(const stv_shape* shape, int64_t* bytes) {
  int rc = check_shape(shape, -1, nullptr);
  if (rc) return rc;
  if (!bytes) return STV_ERR_INVALID_ARG;
  *bytes = (int64_t)shape->hkv * (shape->group == kGroupI4 ? kI4HeadBytes : kHeadBytes);
  return STV_OK;
}

int stv_kv_append_pack(const stv_shape* shape, const stv_layer_cache* layer, const stv_seq* seqs, int n_seqs,
                       const void* k, const void* v, const int32_t* row_seq, const int32_t* row_pos, int n_rows,
                       int32_t* dev_status, stv_stream_t stream) {
  ShapeInfo sh;
  int rc = check_shape(shape, -1, &sh);
  if (rc) return rc;
  if ((rc = check_layer(layer, sh)) || (rc = check_seqs(seqs, n_seqs, -1))) return rc;
  if (n_rows < 0 || (n_rows > 0 && (!k || !v || !row_seq || !row_pos))) return STV_ERR_INVALID_ARG;
  if (n_rows == 0) return STV_OK;
  AppendParams p;
  memset(&p, 0, sizeof(p));
  fill_seq_descs(p.seq, seqs, n_seqs, nullptr);
  p.n_seqs = n_seqs;
  p.hkv = sh.hkv;
  p.pool = layer->pool;
  p.page_bytes = layer->page_bytes;
  p.pool_pages = layer->n_pages;
  p.k = static_cast<const __half*>(k);
  p.v = static_cast<const __half*>(v);
  p.row_seq = row_seq;
  p.row_pos = row_pos;
  p.n_rows = n_rows;
  p.fmt = sh.fmt;
  p.status = dev_status;
  return to_status(launch_kv_append(p, (cudaStream_t)stream));
}

static int workspace_bytes(const stv_shape* shape, const stv_seq* seqs, int n_seqs, int t_nodes, int sm_count,
                           size_t* bytes, bool balance) {
  ShapeInfo sh;
  int rc = check_shape(shape, t_nodes, &sh);
  if (rc) return rc;
  if ((rc = check_seqs(seqs, n_seqs, t_nodes))) return rc;
  if (!bytes || sm_count < 0) return STV_ERR_INVALID_ARG;
  if (sm_count == 0 && (rc = device_sm_count(&sm_count))) return rc;
  Plan plan;
  if ((rc = make_plan(sh, seqs, n_seqs, sm_count, &plan, balance))) return rc;
  *bytes = ws_layout(sh, n_seqs, plan).total;
  return STV_OK;
}

int stv_verify_workspace_bytes(const stv_shape* shape, const stv_seq* seqs, int n_seqs, int t_nodes, int sm_count,
                               size_t* bytes) {
  return workspace_bytes(shape, seqs, n_seqs, t_nodes, sm_count, bytes, true);
}

// stv_verify_attn, and stv_append_verify_attn when k_tree / v_tree are given.
// balance: the split plan the public calls share (stv_verify_workspace_bytes,
// stv_split_combine); the library's own launch sequences (chunked prefill)
// use the one-unit-per-SM plan, and so does the one-launch layer, whose
// units wait for one another.
static int verify_common(const stv_shape* shape, const stv_layer_cache* layer, const stv_seq* seqs, int n_seqs,
                         const void* k_tree, const void* v_tree, const void* q, const int32_t* parent, int t_nodes,
                         int path, void* workspace, size_t ws_bytes, int32_t* dev_status, stv_stream_t stream,
                         int32_t* dots = nullptr, int withhold_copies = 0, void* o_fused = nullptr,
                         bool balance = true) {
  ShapeInfo sh;
  int rc = check_shape(shape, t_nodes, &sh);
  if (rc) return rc;
  if ((rc = check_layer(layer, sh)) || (rc = check_seqs(seqs, n_seqs, t_nodes))) return rc;
  if (!q || !parent || !workspace || (path != STV_PATH_EXACT && path != STV_PATH_INT8)) return STV_ERR_INVALID_ARG;
  if (k_tree && sh.fmt != kFmtBit3) return STV_ERR_UNIMPLEMENTED;  // the fused append packs the 3-bit cache only
  if (path == STV_PATH_INT8 && sh.fmt == kFmtK4V2) return STV_ERR_UNIMPLEMENTED;  // exact path only on this cache
  if (o_fused && (path != STV_PATH_EXACT || sh.fmt != kFmtBit3)) return STV_ERR_UNIMPLEMENTED;
  int sm = 0;
  if ((rc = device_sm_count(&sm))) return rc;
  Plan plan;
  if ((rc = make_plan(sh, seqs, n_seqs, sm, &plan, balance && !o_fused))) return rc;
  // the fused launch's units wait for one another: all of them resident at once
  if (o_fused && plan.n_units > sm) return STV_ERR_SHAPE_UNSUPPORTED;
  const WsLayout wl = ws_layout(sh, n_seqs, plan);
  if (ws_bytes < wl.total) return STV_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  VerifyParams p;
  memset(&p, 0, sizeof(p));
  fill_seq_descs(p.seq, seqs, n_seqs, &plan);
  p.n_seqs = n_seqs;
  p.T = sh.T;
  p.hq = sh.hq;
  p.hkv = sh.hkv;
  p.G = sh.G;
  p.R = sh.R;
  p.tiles_per_split = plan.tiles_per_split;
  p.n_units = plan.n_units;
  p.path = path;
  p.pool = layer->pool;
  p.page_bytes = layer->page_bytes;
  p.pool_pages = layer->n_pages;
  p.q = static_cast<const __half*>(q);
  p.parent = parent;
  p.qi = reinterpret_cast<const int8_t*>(ws + wl.off_qi);
  p.sq = reinterpret_cast<const float*>(ws + wl.off_sq);
  p.o_part = reinterpret_cast<float*>(ws + wl.off_opart);
  p.ml = reinterpret_cast<float*>(ws + wl.off_ml);
  p.k_tree = static_cast<const __half*>(k_tree);
  p.v_tree = static_cast<const __half*>(v_tree);
  p.fmt = sh.fmt;
  p.dots = dots;
  p.test_withhold_copies = withhold_copies;
  p.status = dev_status;
  // the persistent kernel runs the exact path on the 3-bit cache (no fused
  // append, no inspection, no failure-path test)
  if (plan.persist_ctas > 0 && path == STV_PATH_EXACT && sh.fmt == kFmtBit3 && !k_tree && !dots && !withhold_copies) {
    p.persist_ctas = plan.persist_ctas;
    memcpy(p.order, plan.order, sizeof(int16_t) * plan.n_units);
  }
  // The fused append's packing warp (tree rows packed by all units, the
  // tile's copy waiting on a device counter) needs every unit resident at
  // once: the exact path on the 3-bit cache with one unit per SM; otherwise
  // (the int8 path, a balanced plan) the units holding tree rows pack them.
  const bool pack_warp = k_tree && !o_fused && path == STV_PATH_EXACT && sh.fmt == kFmtBit3 &&
                         plan.persist_ctas == 0 && plan.n_units <= sm && !withhold_copies;
  if (o_fused || pack_warp) {
    p.o_out = static_cast<__half*>(o_fused);
    p.pack_warp = pack_warp ? 1 : 0;
    p.cnt = reinterpret_cast<uint32_t*>(ws + wl.off_cnt);
    p.n_pairs = n_seqs * sh.T * sh.hkv;
    p.packed_target = std::min(p.n_units, p.n_pairs);  // one packing warp per unit that has a pair
  }
  cudaStream_t s = (cudaStream_t)stream;
  if (path == STV_PATH_INT8) {
    cudaError_t e = launch_quantize_q(p.q, n_seqs * sh.T * sh.hq, reinterpret_cast<int8_t*>(ws + wl.off_qi),
                                      reinterpret_cast<float*>(ws + wl.off_sq), s);
    if (e != cudaSuccess) return STV_ERR_CUDA;
  }
  return to_status(launch_verify(p, s));
}

int stv_verify_attn(const stv_shape* shape, const stv_layer_cache* layer, const stv_seq* seqs, int n_seqs,
                    const void* q, const int32_t* parent, int t_nodes, int path, void* workspace, size_t ws_bytes,
                    int32_t* dev_status, stv_stream_t stream) {
  return verify_common(shape, layer, seqs, n_seqs, nullptr, nullptr, q, parent, t_nodes, path, workspace, ws_bytes,
                       dev_status, stream);
}

int stv_append_verify_attn(const stv_shape* shape, const stv_layer_cache* layer, const stv_seq* seqs, int n_seqs,
                           const void* k_tree, const void* v_tree, const void* q, const int32_t* parent, int t_nodes,
                           int path, void* workspace, size_t ws_bytes, int32_t* dev_status, stv_stream_t stream) {
  if (!k_tree || !v_tree) return STV_ERR_INVALID_ARG;
  return verify_common(shape, layer, seqs, n_seqs, k_tree, v_tree, q, parent, t_nodes, path, workspace, ws_bytes,
                       dev_status, stream);
}

int stv_append_verify_combine(const stv_shape* shape, const stv_layer_cache* layer, const stv_seq* seqs, int n_seqs,
                              const void* k_tree, const void* v_tree, const void* q, const int32_t* parent,
                              int t_nodes, int path, void* workspace, size_t ws_bytes, void* o, int32_t* dev_status,
                              stv_stream_t stream) {
  if (!k_tree || !v_tree || !o) return STV_ERR_INVALID_ARG;
  return verify_common(shape, layer, seqs, n_seqs, k_tree, v_tree, q, parent, t_nodes, path, workspace, ws_bytes,
                       dev_status, stream, nullptr, 0, o);
}

int stv_verify_attn_timeout_test(const stv_shape* shape, const stv_layer_cache* layer, const stv_seq* seqs,
                                 int n_seqs, const void* q, const int32_t* parent, int t_nodes, int path,
                                 void* workspace, size_t ws_bytes, int32_t* dev_status, stv_stream_t stream) {
  return verify_common(shape, layer, seqs, n_seqs, nullptr, nullptr, q, parent, t_nodes, path, workspace, ws_bytes,
                       dev_status, stream, nullptr, 1);
}

static int combine_common(const stv_shape* shape, const stv_seq* seqs, int n_seqs, int t_nodes, const void* workspace,
                          size_t ws_bytes, void* o, stv_stream_t stream, bool balance) {
  ShapeInfo sh;
  int rc = check_shape(shape, t_nodes, &sh);
  if (rc) return rc;
  if ((rc = check_seqs(seqs, n_seqs, t_nodes))) return rc;
  if (!workspace || !o) return STV_ERR_INVALID_ARG;
  int sm = 0;
  if ((rc = device_sm_count(&sm))) return rc;
  Plan plan;
  if ((rc = make_plan(sh, seqs, n_seqs, sm, &plan, balance))) return rc;
  const WsLayout wl = ws_layout(sh, n_seqs, plan);
  if (ws_bytes < wl.total) return STV_ERR_WORKSPACE_TOO_SMALL;
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  CombineParams p;
  memset(&p, 0, sizeof(p));
  fill_seq_descs(p.seq, seqs, n_seqs, &plan);
  p.n_seqs = n_seqs;
  p.T = sh.T;
  p.hq = sh.hq;
  p.hkv = sh.hkv;
  p.G = sh.G;
  p.R = sh.R;
  p.o_part = reinterpret_cast<const float*>(ws + wl.off_opart);
  p.ml = reinterpret_cast<const float*>(ws + wl.off_ml);
  p.o = static_cast<__half*>(o);
  return to_status(launch_split_combine(p, (cudaStream_t)stream));
}

int stv_split_combine(const stv_shape* shape, const stv_seq* seqs, int n_seqs, int t_nodes, const void* workspace,
                      size_t ws_bytes, void* o, stv_stream_t stream) {
  return combine_common(shape, seqs, n_seqs, t_nodes, workspace, ws_bytes, o, stream, true);
}

// ---------------------------------------------------------------------------
// Prefill (next row f2): chunks of C prompt tokens as chain trees, up to
// STV_MAX_SEQS chunks per verify launch, then the split merge.


int stv_prefill_workspace_bytes(const stv_shape* shape, const stv_seq* seq, int n_tokens, size_t* bytes) {
  if (!shape || !seq || !bytes || n_tokens < 1) return STV_ERR_INVALID_ARG;
  ShapeInfo sh;
  int rc = check_shape(shape, 1, &sh);
  if (rc) return rc;
  const int c = prefill_chunk_tokens(shape);
  size_t most = 0;
  rc = for_each_prefill_launch(n_tokens, c, [&](const PrefillLaunch& pl) -> int {
    stv_seq seqs[STV_MAX_SEQS];
    prefill_seqs(seq, pl, seqs);
    size_t b = 0;  // the chunk launches use the one-unit-per-SM plan
    if (int r = workspace_bytes(shape, seqs, pl.count, pl.t, 0, &b, false)) return r;
    most = b > most ? b : most;
    return (int)STV_OK;
  });
  if (rc) return rc;
  *bytes = kParentsBytes + most;
  return STV_OK;
}

static int prefill_common(const stv_shape* shape, const stv_layer_cache* layer, const stv_seq* seq, const void* q,
                          int n_tokens, int path, void* workspace, size_t ws_bytes, void* o, int32_t* dev_status,
                          stv_stream_t stream, bool withhold_copies) {
  size_t need = 0;
  int rc = stv_prefill_workspace_bytes(shape, seq, n_tokens, &need);
  if (rc) return rc;
  if (!layer || !q || !o || !workspace) return STV_ERR_INVALID_ARG;
  if (ws_bytes < need) return STV_ERR_WORKSPACE_TOO_SMALL;
  const int c = prefill_chunk_tokens(shape);
  ShapeInfo sh;
  if ((rc = check_shape(shape, -1, &sh))) return rc;
  if (path == STV_PATH_EXACT && sh.fmt == kFmtBit3) {
    // one persistent launch over (chunk, KV head) units; no workspace used
    if ((rc = check_layer(layer, sh))) return rc;
    if ((rc = check_seqs(seq, 1, n_tokens))) return rc;
    PrefillParams pp;
    memset(&pp, 0, sizeof(pp));
    pp.page_table = seq->page_table;
    pp.n_pages = seq->n_pages;
    pp.ctx0 = seq->ctx;
    pp.n_tokens = n_tokens;
    pp.chunk = c;
    pp.n_chunks = (n_tokens + c - 1) / c;
    pp.n_units = pp.n_chunks * sh.hkv;
    pp.hq = sh.hq;
    pp.hkv = sh.hkv;
    pp.G = sh.G;
    pp.pool = layer->pool;
    pp.page_bytes = layer->page_bytes;
    pp.pool_pages = layer->n_pages;
    pp.q = static_cast<const __half*>(q);
    pp.o = static_cast<__half*>(o);
    pp.status = dev_status;
    int sms = 0;
    if ((rc = device_sm_count(&sms))) return rc;
    return to_status(launch_prefill(pp, std::min(pp.n_units, sms), (cudaStream_t)stream, withhold_copies));
  }
  if (withhold_copies) return STV_ERR_UNIMPLEMENTED;  // the failure-path test runs the persistent kernel only
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* parents = reinterpret_cast<int32_t*>(ws);
  // chain parents for STV_MAX_SEQS chunks of c tokens; a last partial chunk
  // of t < c tokens uses the first t entries, which are its chain too
  if (cudaError_t e = launch_chain_parents(parents, STV_MAX_SEQS, c, (cudaStream_t)stream)) {
    (void)e;
    return STV_ERR_CUDA;
  }
  const size_t row = (size_t)shape->hq * kHeadDim;  // halves per token
  return for_each_prefill_launch(n_tokens, c, [&](const PrefillLaunch& pl) -> int {
    stv_seq seqs[STV_MAX_SEQS];
    prefill_seqs(seq, pl, seqs);
    const __half* qs = static_cast<const __half*>(q) + (size_t)pl.start * row;
    __half* os = static_cast<__half*>(o) + (size_t)pl.start * row;
    if (int r = verify_common(shape, layer, seqs, pl.count, nullptr, nullptr, qs, parents, pl.t, path,
                              ws + kParentsBytes, ws_bytes - kParentsBytes, dev_status, stream, nullptr, 0, nullptr,
                              false))
      return r;
    return combine_common(shape, seqs, pl.count, pl.t, ws + kParentsBytes, ws_bytes - kParentsBytes, os, stream,
                          false);
  });
}

int stv_prefill_attn(const stv_shape* shape, const stv_layer_cache* layer, const stv_seq* seq, const void* q,
                     int n_tokens, int path, void* workspace, size_t ws_bytes, void* o, int32_t* dev_status,
                     stv_stream_t stream) {
  return prefill_common(shape, layer, seq, q, n_tokens, path, workspace, ws_bytes, o, dev_status, stream, false);
}

int stv_prefill_attn_timeout_test(const stv_shape* shape, const stv_layer_cache* layer, const stv_seq* seq,
                                  const void* q, int n_tokens, int path, void* workspace, size_t ws_bytes, void* o,
                                  int32_t* dev_status, stv_stream_t stream) {
  return prefill_common(shape, layer, seq, q, n_tokens, path, workspace, ws_bytes, o, dev_status, stream, true);
}

int stv_tree_accept(const int32_t* parent, const int32_t* draft_ids, const int32_t* target_argmax, int t_nodes,
                    int n_seqs, int32_t* n_commit, int32_t* path, int32_t* out_ids, int32_t* dev_status,
                    stv_stream_t stream) {
  if (!parent || !draft_ids || !target_argmax || !n_commit || !path || !out_ids) return STV_ERR_INVALID_ARG;
  if (n_seqs < 1) return STV_ERR_INVALID_ARG;
  if (t_nodes < 1 || t_nodes > kMaxT) return STV_ERR_SHAPE_UNSUPPORTED;
  return to_status(launch_tree_accept(parent, draft_ids, target_argmax, t_nodes, n_seqs, n_commit, path, out_ids,
                                      dev_status, (cudaStream_t)stream));
}

int stv_kv_commit(const stv_shape* shape, const stv_layer_cache* layers, int n_layers, const stv_seq* seqs,
                  int n_seqs, int t_nodes, const int32_t* n_commit, const int32_t* path, int32_t* ctx_dev,
                  int32_t* dev_status, stv_stream_t stream) {
  ShapeInfo sh;
  int rc = check_shape(shape, t_nodes, &sh);
  if (rc) return rc;
  if (!layers || n_layers < 1 || n_layers > kMaxLayers || !n_commit || !path) return STV_ERR_INVALID_ARG;
  if ((rc = check_seqs(seqs, n_seqs, t_nodes))) return rc;
  CommitParams p;
  memset(&p, 0, sizeof(p));
  p.min_pool_pages = layers[0].n_pages;
  for (int l = 0; l < n_layers; ++l) {
    if ((rc = check_layer(&layers[l], sh))) return rc;
    p.pools[l] = layers[l].pool;
    p.pool_pages[l] = layers[l].n_pages;
    p.min_pool_pages = std::min(p.min_pool_pages, layers[l].n_pages);
  }
  fill_seq_descs(p.seq, seqs, n_seqs, nullptr);
  p.n_seqs = n_seqs;
  p.n_layers = n_layers;
  p.hkv = sh.hkv;
  p.T = sh.T;
  p.page_bytes = layers[0].page_bytes;
  p.n_commit = n_commit;
  p.path = path;
  p.ctx_dev = ctx_dev;
  p.fmt = sh.fmt;
  p.status = dev_status;
  return to_status(launch_kv_commit(p, (cudaStream_t)stream));
}

int stv_int8_qk_dots(const stv_shape* shape, const stv_layer_cache* layer, const stv_seq* seq, const void* q,
                     const int32_t* parent, int t_nodes, void* workspace, size_t ws_bytes, int32_t* dots,
                     int32_t* dev_status, stv_stream_t stream) {
  ShapeInfo sh;
  int rc = check_shape(shape, t_nodes, &sh);
  if (rc) return rc;
  if (sh.fmt != kFmtBit3) return STV_ERR_UNIMPLEMENTED;  // the per-group dots belong to the 3-bit cache
  if (!dots) return STV_ERR_INVALID_ARG;
  return verify_common(shape, layer, seq, 1, nullptr, nullptr, q, parent, t_nodes, STV_PATH_INT8, workspace, ws_bytes,
                       dev_status, stream, dots);
}

}  // extern "C"
