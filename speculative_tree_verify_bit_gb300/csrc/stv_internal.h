// stv_internal.h -- shared definitions of the CUDA library (host and device):
// cache layout constants, the split plan, kernel parameter blocks and the
// launchers that api.cu calls.  Not part of the public ABI (include/stv.h).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "stv.h"

namespace stv {

constexpr int kHeadDim = 256;
constexpr int kGroup = 32;
constexpr int kGroups = kHeadDim / kGroup;  // 8
constexpr int kPageTok = 256;
constexpr int kTileTok = 64;                 // V-code tiles and verify tiles
constexpr int kMaxRows = 128;                // T * G per KV head
constexpr int kMaxT = 32;
constexpr int kMaxSplitsPerHead = 256;  // split_combine keeps one (m, l) per split in 8 registers x 32 lanes
// A balanced plan (several sequences, 3-bit cache) may hold up to this many
// work units; the persistent verify kernel takes them in the order
// VerifyParams::order gives.
constexpr int kMaxPersistUnits = 640;

// Byte offsets inside one KV head's block of a page (see include/stv.h).
constexpr int kOffKCodes = 0;
constexpr int kOffKScales = kPageTok * kGroups * 12;            // 24576
constexpr int kOffVCodes = kOffKScales + kPageTok * kGroups * 2;  // 28672
constexpr int kOffVScales = kOffVCodes + kPageTok * kGroups * 12;  // 53248
constexpr int kHeadBytes = kOffVScales + kPageTok * kGroups * 2;   // 57344
constexpr int kVTileCodeBytes = kHeadDim * 24;                     // 6144: one 64-token tile
constexpr int kVTileScaleBytes = kGroups * kTileTok * 2;           // 1024
constexpr int kKTileCodeBytes = kTileTok * 96;                     // 6144
constexpr int kKTileScaleBytes = kTileTok * 16;                    // 1024
static_assert(kHeadBytes == STV_HEAD_BLOCK_BYTES, "layout");

// The int4 per-token-head format (group 256; see include/stv.h).
constexpr int kGroupI4 = 256;
constexpr int kI4OffKCodes = 0;
constexpr int kI4OffKScales = kPageTok * 128;                 // 32768
constexpr int kI4OffVCodes = kI4OffKScales + kPageTok * 2;    // 33280
constexpr int kI4OffVScales = kI4OffVCodes + kPageTok * 128;  // 66048
constexpr int kI4HeadBytes = kI4OffVScales + kPageTok * 2;    // 66560
constexpr int kI4KTileCodeBytes = kTileTok * 128;             // 8192: one 64-token tile
constexpr int kI4KTileScaleBytes = kTileTok * 2;              // 128
constexpr int kI4VTileCodeBytes = kHeadDim * 32;              // 8192
constexpr int kI4VTileScaleBytes = kTileTok * 2;              // 128
static_assert(kI4HeadBytes == STV_HEAD_BLOCK_BYTES_INT4, "layout");

// The K 4 / V 2-bit format (group 32; see include/stv.h).
constexpr int kKv2OffKCodes = 0;
constexpr int kKv2OffKScales = kPageTok * kGroups * 16;                 // 32768
constexpr int kKv2OffVCodes = kKv2OffKScales + kPageTok * kGroups * 2;  // 36864
constexpr int kKv2OffVScales = kKv2OffVCodes + kPageTok * kHeadDim / 4;  // 53248
constexpr int kKv2HeadBytes = kKv2OffVScales + kPageTok * kGroups * 2;  // 57344
constexpr int kKv2KTileCodeBytes = kTileTok * 128;                      // 8192: one 64-token tile
constexpr int kKv2KTileScaleBytes = kTileTok * 16;                      // 1024
constexpr int kKv2VTileCodeBytes = kHeadDim * 16;                       // 4096
constexpr int kKv2VTileScaleBytes = kGroups * kTileTok * 2;             // 1024
static_assert(kKv2HeadBytes == STV_HEAD_BLOCK_BYTES, "layout");
static_assert(kKv2OffVScales == kOffVScales, "V scales sit where the 3-bit cache's do");

struct SeqDesc {
  const int32_t* page_table;
  int32_t n_pages;
  int32_t ctx;
  int32_t splits;     // splits per KV head for this sequence
  int32_t unit_base;  // first work unit of this sequence
};

// Split plan: every (sequence, KV head) range [0, ctx + T) is cut into pieces
// of `tiles_per_split` 64-token tiles; each piece is one work unit (one CTA),
// numbered sequence-major, then KV head, then split.
struct Plan {
  int n_units;
  int tiles_per_split;
  int splits[STV_MAX_SEQS];
  int unit_base[STV_MAX_SEQS + 1];
  // Balanced plan (make_plan with balance, several sequences, 3-bit cache):
  // the persistent verify kernel's CTAs (0 otherwise) and the units, longest
  // first.
  int persist_ctas;
  int16_t order[kMaxPersistUnits];
};

// Workspace carve-up (byte offsets, each 256-aligned).
struct WsLayout {
  size_t off_qi, off_sq, off_opart, off_ml, off_cnt, total;
};

// Cache formats (include/stv.h): the pages' 3-bit cache, the int4
// per-token-head cache, the K 4 / V 2-bit cache.
enum { kFmtBit3 = 0, kFmtInt4 = 1, kFmtK4V2 = 2 };

struct ShapeInfo {
  int hq, hkv, G, T, R;  // R = T * G rows per KV head
  int fmt;               // kFmtBit3, kFmtInt4 or kFmtK4V2
};

// Parameters of one verify launch (passed by value; < 4 KB).
struct VerifyParams {
  SeqDesc seq[STV_MAX_SEQS];
  int n_seqs;
  int T, hq, hkv, G, R;
  int tiles_per_split;
  int n_units;
  int path;
  const uint8_t* pool;
  int64_t page_bytes;
  int32_t pool_pages;
  const __half* q;        // [n_seqs][T][hq][256]
  const int32_t* parent;  // [n_seqs][T]
  const int8_t* qi;       // [n_seqs][T][hq][256] (int8 path)
  const float* sq;        // [n_seqs][T][hq]
  float* o_part;          // [n_units][R][256]
  float* ml;              // [n_units][R][2] (m in log2 units, l)
  // Tree rows to pack into the cache before they are read (fused append), or
  // null when they are already there: fp16 [n_seqs][T][hkv][256], row i of
  // sequence s goes to position ctx_s + i.
  const __half* k_tree;
  const __half* v_tree;
  int fmt;  // cache format
  // Inspection (int8 path, one sequence): when set, the verify kernel also
  // writes its own per-group integer dots, int32 [hkv][R][ctx + T][8].
  int32_t* dots;
  // Failure-path test (stv_verify_attn_timeout_test): the producer issues no
  // copy, every wait on one runs out and the kernel reports STV_DEV_TIMEOUT.
  int test_withhold_copies;
  int32_t* status;
  // One launch per layer (stv_append_verify_combine), or null: the round's
  // tree rows (k_tree, v_tree) are packed by every work unit, (row, KV head)
  // pair q = (s * T + i) * hkv + h by unit q mod n_units, and the units then
  // merge the splits into o_out, the items dealt over the whole launch.
  // cnt (workspace, zero between launches): [0] packing warps done, [1] units
  // done, [2 + s * hkv + h] units of (s, h) whose partials are written.
  __half* o_out;
  uint32_t* cnt;
  int n_pairs;
  int packed_target;  // packing warps that arrive: min(n_units, n_pairs)
  // The fused append by the packing warp without the merge (o_out null):
  // stv_append_verify_attn when the plan keeps one unit per SM.
  int pack_warp;
  // Balanced plan: the exact path on the 3-bit cache runs the persistent
  // kernel (prefill_tc.cu, verify mode) on persist_ctas CTAs, which take the
  // units order[0], order[1], ... (longest first) in snake order; 0 = one
  // CTA per unit.
  int persist_ctas;
  int16_t order[kMaxPersistUnits];
};

// Parameters of one prefill launch (prefill_tc.cu, exact path, 3-bit cache):
// the prompt of one sequence, cut into chunks of `chunk` tokens; a unit is
// (chunk, KV head), numbered longest first.
struct PrefillParams {
  const int32_t* page_table;  // the sequence's pages
  int32_t n_pages;
  int32_t ctx0;      // cached tokens before the prompt
  int n_tokens;      // prompt tokens, already in the cache at ctx0 ..
  int chunk, n_chunks, n_units;
  int hq, hkv, G;
  const uint8_t* pool;
  int64_t page_bytes;
  int32_t pool_pages;
  const __half* q;   // [n_tokens][hq][256]
  __half* o;         // [n_tokens][hq][256]
  int32_t* status;
};

struct CombineParams {
  SeqDesc seq[STV_MAX_SEQS];
  int n_seqs;
  int T, hq, hkv, G, R;
  const float* o_part;
  const float* ml;
  __half* o;
};

struct AppendParams {
  SeqDesc seq[STV_MAX_SEQS];
  int n_seqs;
  int hkv;
  uint8_t* pool;
  int64_t page_bytes;
  int32_t pool_pages;
  const __half* k;
  const __half* v;
  const int32_t* row_seq;
  const int32_t* row_pos;
  int n_rows;
  int fmt;  // cache format
  int32_t* status;
};

constexpr int kMaxLayers = 128;
struct CommitParams {
  SeqDesc seq[STV_MAX_SEQS];
  uint8_t* pools[kMaxLayers];
  int n_seqs, n_layers, hkv, T;
  int64_t page_bytes;
  int32_t pool_pages[kMaxLayers];
  int32_t min_pool_pages;  // the smallest of pool_pages
  const int32_t* n_commit;
  const int32_t* path;
  int32_t* ctx_dev;
  int fmt;  // cache format
  int32_t* status;
};

// Launch with programmatic stream serialization (see grid_dep_wait in
// stv_device.cuh): the kernel's CTAs may start while the previous kernel in
// the stream finishes; every kernel of this library waits for it before its
// first global-memory access.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), int grid, int block, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  if (e != cudaSuccess) (void)cudaGetLastError();
  return e;
}

// The same launch, cooperative as well: every CTA of the grid is resident at
// once, so CTAs of the launch may wait (bounded) for one another.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_coop(void (*kernel)(KArgs...), int grid, int block, size_t smem, cudaStream_t s,
                            Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  if (e != cudaSuccess) (void)cudaGetLastError();
  return e;
}

// ---- host helpers (api.cu) ----
int make_plan(const ShapeInfo& sh, const stv_seq* seqs, int n_seqs, int sm_count, Plan* plan, bool balance);
WsLayout ws_layout(const ShapeInfo& sh, int n_seqs, const Plan& plan);

// ---- launchers (return cudaError_t of the launch) ----
cudaError_t launch_kv_append(const AppendParams& p, cudaStream_t s);
cudaError_t launch_chain_parents(int32_t* parent, int chunks, int t, cudaStream_t s);
cudaError_t launch_kv_commit(const CommitParams& p, cudaStream_t s);
cudaError_t launch_quantize_q(const __half* q, int n_rows, int8_t* qi, float* sq, cudaStream_t s);
cudaError_t launch_verify(const VerifyParams& p, cudaStream_t s);     // exact path; int4 cache (verify_tc.cu)
cudaError_t launch_verify_i8(const VerifyParams& p, cudaStream_t s);  // int8 path, 3-bit cache (verify_i8.cu)
cudaError_t launch_split_combine(const CombineParams& p, cudaStream_t s);
// prefill_tc.cu; withhold_copies: failure-path test (every wait runs out)
cudaError_t launch_prefill(const PrefillParams& p, int grid, cudaStream_t s, bool withhold_copies = false);
cudaError_t launch_verify_persistent(const VerifyParams& p, cudaStream_t s);  // prefill_tc.cu, verify mode
cudaError_t launch_tree_accept(const int32_t* parent, const int32_t* draft, const int32_t* argmax, int T, int n_seqs,
                               int32_t* n_commit, int32_t* path, int32_t* out_ids, int32_t* status, cudaStream_t s);

}  // namespace stv
