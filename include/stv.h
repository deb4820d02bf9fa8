/*
 * stv.h -- C ABI of the GB300 (sm_103a) tree-verify library: one speculative
 * decoding verify round over a paged 3-bit KV cache.
 *
 * What the round computes (page titles and sections it follows):
 *  - "elpis" README, header table: the target keeps a 3-bit KV cache
 *    (12 KiB per token over 16 attention layers) with a 262,144-token native
 *    context.  -> stv_kv_append_pack
 *  - "elpis" README, "Why fast" table: a draft proposes 7 tokens arranged as
 *    an 8-row token tree; the target verifies all rows in one pass (decode
 *    verify with the 3-bit K codes used as exact int8 values against int8 Q);
 *    the engine commits the longest matching path + 1.
 *    -> stv_verify_attn (STV_PATH_EXACT / STV_PATH_INT8), stv_tree_accept,
 *       stv_kv_commit
 *  - Reddit posts (u/iamMess), second post: the verify step needs split-KV
 *    attention because a few query rows alone cannot fill the GPU.
 *    -> stv_verify_attn writes per-split partials, stv_split_combine merges them
 *  - "elpis" README, "Why fast": host check after launch (tree verify pipe).
 *    -> nothing here synchronises; acceptance and commit stay on the device.
 *  - syv-ai README (mirror), split-KV scratch buffer section: the verify
 *    workspace must be sized and owned by someone.
 *    -> stv_verify_workspace_bytes; the caller owns the workspace.
 *
 * Conventions (every entry point):
 *  - extern "C"; returns STV_OK (0) or a negative STV_ERR_* status.  Host
 *    arguments are validated before anything is enqueued; on a negative
 *    status nothing was enqueued.
 *  - Pointers documented "device" are caller-owned device memory; the library
 *    never allocates, frees or synchronises, and keeps no pointer after the
 *    call returns.  All work is enqueued on `stream` (NULL = legacy default
 *    stream); asynchronous CUDA faults surface at the caller's next sync.
 *  - Kernels are launched with programmatic stream serialization: a launch's
 *    blocks may be scheduled, and do their set-up, while the previous kernel
 *    in the stream is still running, but every kernel waits for that kernel
 *    to complete (and its writes to be visible) before its first read or
 *    write of global memory.  Stream order is kept for any predecessor, the
 *    library's own or not.
 *  - Data that lives on the device (page tables, row positions, parent
 *    arrays, commit counts) cannot be checked on the host.  Kernels check it
 *    as they read it, never touch memory outside the described buffers, and
 *    OR an STV_DEV_* bit into *dev_status (device int32, may be NULL).
 *  - Supported shape: head_dim 256, group 32, page_tokens 256, hq = G * hkv
 *    with T * G <= 128 query rows per KV head, 1 <= T <= 32 tree nodes,
 *    1 <= n_seqs <= STV_MAX_SEQS.
 *
 * Paged cache layout (one pool per layer; page_bytes = hkv * 57,344 for the
 * supported shape).  Inside a page, KV head h owns the block at h * 57,344:
 *    [0, 24576)      K codes   [256 tokens][8 groups][3 x uint32]
 *    [24576, 28672)  K scales  [256 tokens][8 groups] fp16
 *    [28672, 53248)  V codes   [4 tiles of 64 tokens][256 channels][2 blocks][3 x uint32]
 *    [53248, 57344)  V scales  [4 tiles][8 groups][64 tokens] fp16
 * Quantizer, per (token, KV head, group of 32 channels), for K and V alike:
 * s = fp16(max|x| / 4); code c = clamp(rne(x / s) + 4, 0, 7) (round half to
 * even; all codes 4 when s == 0); decoded value s * (c - 4).  A block of 32
 * codes (32 channels of one token for K, 32 tokens of one channel for V) is
 * three little-endian uint32 W0..W2: for j in 0..2, k in 0..4, m = 5j + k,
 * code 2m sits in bits 3k..3k+2 of Wj and code 2m+1 in bits 16+3k..16+3k+2
 * of Wj; bit b of code 30 is bit 15 of Wb, bit b of code 31 is bit 31 of Wb.
 */
#ifndef STV_H_
#define STV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* stv_stream_t;

#define STV_MAX_SEQS 64
#define STV_HEAD_DIM 256
#define STV_GROUP 32
#define STV_PAGE_TOKENS 256
#define STV_HEAD_BLOCK_BYTES 57344
#define STV_GROUP_INT4 256            /* group of the int4 per-token-head cache */
#define STV_HEAD_BLOCK_BYTES_INT4 66560

enum stv_status {
  STV_OK = 0,
  STV_ERR_INVALID_ARG = -1,         /* null pointer, negative count, bad enum */
  STV_ERR_SHAPE_UNSUPPORTED = -2,   /* shape outside the supported set */
  STV_ERR_WORKSPACE_TOO_SMALL = -3, /* ws_bytes below stv_verify_workspace_bytes */
  STV_ERR_CUDA = -4,                /* a CUDA runtime call or launch failed */
  STV_ERR_UNIMPLEMENTED = -5,
};

/* Bits OR-ed into *dev_status by kernels that find bad device-side data. */
enum stv_dev_status {
  STV_DEV_BAD_PAGE = 1,   /* page-table entry outside the pool, or position past the table */
  STV_DEV_BAD_TREE = 2,   /* parent[0] != -1 or parent[i] outside [0, i) */
  STV_DEV_BAD_ROW = 4,    /* row_seq outside [0, n_seqs) or row_pos negative */
  STV_DEV_BAD_COMMIT = 8, /* n_commit outside [1, T] or path not a root path */
  STV_DEV_TIMEOUT = 16,   /* a bounded wait inside a kernel gave up; outputs are invalid */
};

enum stv_path { STV_PATH_EXACT = 0, STV_PATH_INT8 = 1 };

/* Cache formats (stv_shape.kv_format). */
enum stv_kv_format {
  STV_KV_BY_GROUP = 0, /* by stv_shape.group: 32 the 3-bit cache, 256 the int4 per-token-head cache */
  STV_KV_K4V2 = 2,     /* the KVarN-style cache: K 4 bits, V 2 bits, group 32 (see the notes below) */
};

typedef struct {
  int32_t hq;          /* query heads (24 for the pages' model) */
  int32_t hkv;         /* KV heads (4) */
  int32_t head_dim;    /* must be 256 */
  int32_t group;       /* cache format, by its quantization group:
                        *   32  (STV_GROUP): 3-bit codes, one fp16 scale per
                        *       32 channels -- the pages' cache;
                        *   256 (STV_GROUP_INT4): int4 codes, one fp16 scale
                        *       per token and KV head (next row f3; see the
                        *       int4 notes below) */
  int32_t page_tokens; /* must be 256 */
  int32_t kv_format;   /* STV_KV_BY_GROUP, or STV_KV_K4V2 with group 32 */
} stv_shape;

typedef struct {
  uint8_t* pool;      /* device: n_pages * page_bytes bytes */
  int64_t page_bytes; /* must equal hkv * STV_HEAD_BLOCK_BYTES (group 32, both
                       * formats) or hkv * STV_HEAD_BLOCK_BYTES_INT4 (group 256) */
  int32_t n_pages;
} stv_layer_cache;

typedef struct {
  const int32_t* page_table; /* device: n_pages entries, each in [0, pool n_pages) */
  int32_t n_pages;           /* logical pages of this sequence */
  int32_t ctx;               /* cached tokens before this round's tree rows */
} stv_seq;

/* Name of a status code (static string). */
const char* stv_status_string(int status);

/* Library ABI version (monotonic). */
int stv_version(void);

/* Bytes of one page for `shape` (hkv * 57,344; hkv * 66,560 for group 256).
 *
 * The int4 per-token-head cache (group 256; syv-ai README (mirror), int4 KV
 * section: the stock int4_per_token_head cache; the pages give no formula).
 * Reading: per (token, KV head) s = fp16(max|x| / 7), c = clamp(rne(x / s),
 * -8, 7) (all 0 when s == 0), stored as u = c + 8; decoded value s * c.
 * Per KV head (66,560 bytes): K codes [256 tok][32 words] at 0, K scales
 * [256] fp16 at 32,768, V codes [4 tiles of 64 tok][256 ch][8 words] at
 * 33,280 (a word holds one channel's codes for 8 tokens), V scales [256]
 * fp16 at 66,048.  In a word of 8 elements e0..e7, element e sits at bit
 * 4 * (e / 2), plus 16 when e is odd.  stv_kv_append_pack, stv_verify_attn,
 * stv_split_combine, stv_verify_attn_no_alloc, stv_prefill_attn and
 * stv_kv_commit accept it; stv_append_verify_attn and stv_int8_qk_dots return
 * STV_ERR_UNIMPLEMENTED for it. */
/* The KVarN-style 4/2-bit cache (STV_KV_K4V2, group 32; Reddit posts
 * (u/iamMess), "Now added" list: KVarN 4/2-bit KV cache; syv-ai README
 * (mirror), DFlash2 at 240k: CTX=huge; the pages give no formula).  Reading:
 * the 3-bit cache's quantizer at other widths, per (token, KV head, group of
 * 32 channels): at b bits, h = 2^(b-1), s = fp16(max|x| / h),
 * c = clamp(rne(x / s), -h, h - 1), stored as u = c + h; decoded s * c.  K at
 * 4 bits, V at 2 bits.  Per KV head (57,344 bytes, as the 3-bit cache):
 *    [0, 32768)      K codes  [256 tokens][8 groups][4 x uint32]; a word holds
 *                    8 channels, element e at bit 4 * (e / 2) + 16 * (e % 2)
 *    [32768, 36864)  K scales [256 tokens][8 groups] fp16
 *    [36864, 53248)  V codes  [4 tiles of 64 tokens][256 channels][4 x uint32];
 *                    a word holds one channel's codes for 16 tokens, token
 *                    t at bit 2 * (t / 2) + 16 * (t % 2)
 *    [53248, 57344)  V scales [4 tiles][8 groups][64 tokens] fp16
 * stv_kv_append_pack, stv_verify_attn (exact path), stv_split_combine,
 * stv_verify_attn_no_alloc, stv_prefill_attn (exact path) and stv_kv_commit
 * accept it; the int8 path, stv_append_verify_attn and stv_int8_qk_dots
 * return STV_ERR_UNIMPLEMENTED for it. */
int stv_page_bytes(const stv_shape* shape, int64_t* bytes);

/*
 * a1 -- quantize fp16 K/V rows into the paged 3-bit cache ("elpis" README,
 * header table: 3-bit KV cache).
 *  k, v:      device fp16 [n_rows][hkv][256].
 *  row_seq:   device int32 [n_rows], sequence of each row.
 *  row_pos:   device int32 [n_rows], token position of each row in its
 *             sequence; page row_pos / 256 of that sequence's table, slot
 *             row_pos % 256.  Two rows may not share a (sequence, position).
 * A verify round appends its T tree rows at ctx .. ctx + T - 1.
 */
int stv_kv_append_pack(const stv_shape* shape, const stv_layer_cache* layer, const stv_seq* seqs, int n_seqs,
                       const void* k, const void* v, const int32_t* row_seq, const int32_t* row_pos, int n_rows,
                       int32_t* dev_status, stv_stream_t stream);

/*
 * Workspace for stv_verify_attn / stv_split_combine: per-split partial
 * outputs (fp32), their row maxima and sums, the int8 Q rows and scales.
 * sm_count: SMs the split plan targets; 0 = the current device's count
 * (stv_verify_attn and stv_split_combine always plan for the current device).
 * The plan cuts each (sequence, KV head) key range into splits of equal
 * whole 64-key tiles, never more than 256 splits for one (sequence, KV
 * head): as many work units as SMs at most; or, for several sequences on the
 * 3-bit cache, the split whose work units, dealt longest first to the SMs by
 * the persistent verify kernel, finish first (up to 640 units, 24 MiB of
 * partials), so that a batch of unequal sequences keeps every SM busy.
 */
int stv_verify_workspace_bytes(const stv_shape* shape, const stv_seq* seqs, int n_seqs, int t_nodes, int sm_count,
                               size_t* bytes);

/*
 * a2..a4 -- tree-masked split-KV GQA attention of the round's T nodes over
 * every cached token ("elpis" README, "Why fast": 8-row token tree, decode
 * verify; Reddit posts, second post: split-KV verify attention).
 *  q:       device fp16 [n_seqs][T][hq][256] (node-major, then Q head).
 *  parent:  device int32 [n_seqs][T], parent[0] = -1, parent[i] in [0, i).
 *  path:    STV_PATH_EXACT: Q fp16 times K dequantized to fp16, fp32 sums;
 *           STV_PATH_INT8: Q quantized per row to int8 (qi = rne(127 q /
 *           max|q|)) times the 3-bit K codes, scaled per group.
 * Key j < ctx is visible to every node; key ctx + k is visible to node i iff
 * k is i or an ancestor of i.  Scores are q . k / 16; softmax in fp32; P is
 * rounded to fp16 and P . V accumulates in fp32.  On the int4 cache (group
 * 256) a key's one scale covers the whole head, so Q is multiplied by the
 * key's exact codes and the score by the key's scale in fp32 (both paths);
 * V is dequantized to fp16 as on the 3-bit cache.  Writes partials into the
 * workspace; stv_split_combine produces the output.  The round's tree rows
 * must already be in the cache (stv_kv_append_pack).
 */
int stv_verify_attn(const stv_shape* shape, const stv_layer_cache* layer, const stv_seq* seqs, int n_seqs,
                    const void* q, const int32_t* parent, int t_nodes, int path, void* workspace, size_t ws_bytes,
                    int32_t* dev_status, stv_stream_t stream);

/*
 * a1 + a2..a4 in one launch (the round's append fused into verify): packs the
 * round's T tree rows into the cache exactly as stv_kv_append_pack would (row
 * i of sequence s at position ctx_s + i, every KV head, K and V), then runs
 * stv_verify_attn over the cache that now holds them.  The work unit whose
 * key range holds a tree row packs it, before its bulk copies read that tile,
 * so the rows never need a launch of their own ("elpis" README, "Why fast":
 * tree verify pipe, host check after launch; syv-ai README (mirror), CUDA
 * graph notes: an uncaptured verify step is launch-bound).
 *  k_tree, v_tree: device fp16 [n_seqs][T][hkv][256], caller-owned, read only.
 *  All other arguments, the workspace and the results as in stv_verify_attn;
 *  the cache bytes written equal those of stv_kv_append_pack on the same rows.
 *  Exact path, one work unit per SM (one sequence): the rows are packed by an
 *  extra warp of every unit, the pairs (row, KV head) dealt round-robin, and
 *  a unit copies a tile holding tree keys once every pair is packed (a
 *  cooperative launch; the workspace's arrival counters, as for
 *  stv_append_verify_combine, must be zero before the first call and every
 *  completed call leaves them zero).  Otherwise (the int8 path, several
 *  sequences) the unit whose key range holds a tree row packs it.
 *  STV_ERR_INVALID_ARG when k_tree or v_tree is null; a page-table entry
 *  outside the pool sets STV_DEV_BAD_PAGE and that row is not written.
 */
int stv_append_verify_attn(const stv_shape* shape, const stv_layer_cache* layer, const stv_seq* seqs, int n_seqs,
                           const void* k_tree, const void* v_tree, const void* q, const int32_t* parent, int t_nodes,
                           int path, void* workspace, size_t ws_bytes, int32_t* dev_status, stv_stream_t stream);

/*
 * a1 + a2..a4 + a5 in one launch: one layer of a verify round.  Packs the
 * round's tree rows into the cache as stv_kv_append_pack would (row i of
 * sequence s at position ctx_s + i), runs stv_verify_attn over the cache that
 * now holds them, and merges the splits into o as stv_split_combine would
 * ("elpis" README, "Why fast": tree verify pipe; Reddit posts (u/iamMess),
 * second post: split-KV verify then merge; syv-ai README (mirror), CUDA graph
 * notes: an uncaptured verify step is launch-bound).  The tree rows are
 * packed by all work units together, (row, KV head) pairs dealt round-robin;
 * a unit copies a tile holding tree keys once every pair is packed, and the
 * units of each (sequence, KV head) merge their own partials once all of
 * them have written theirs.  The units wait for one another (bounded), so
 * the launch is cooperative: every unit resident at once.
 *  k_tree, v_tree: device fp16 [n_seqs][T][hkv][256], read only.
 *  q, parent, t_nodes: as stv_verify_attn; path: STV_PATH_EXACT only.
 *  o: device fp16 [n_seqs][T][hq][256], the merged attention output.
 *  workspace: as stv_verify_attn (the same size).  Its first
 *   (2 + STV_MAX_SEQS * hkv) * 4 bytes, rounded up to 256, hold arrival
 *   counters that must be zero before the first call on a workspace
 *   (allocate it zero-filled).  Every call that completes leaves them zero,
 *   and no other call writes them, whatever its plan; after STV_DEV_TIMEOUT
 *   the caller zeroes them again.
 * Cache bytes and o equal those of stv_kv_append_pack + stv_verify_attn +
 * stv_split_combine on the same inputs, bit for bit.  On GB300 the three
 * separate launches (in a CUDA graph) are faster: the packing warp's code
 * slows the verify kernel's tile loop, and the merge's waits and dependent
 * loads cost more than the merge launch they replace.
 *  STV_ERR_INVALID_ARG when k_tree, v_tree or o is null;
 *  STV_ERR_UNIMPLEMENTED for the int8 path and for the int4 and 4/2-bit caches;
 *  STV_ERR_SHAPE_UNSUPPORTED when the split plan has more work units than the
 *  device has SMs (more than sm_count / hkv sequences).
 */
int stv_append_verify_combine(const stv_shape* shape, const stv_layer_cache* layer, const stv_seq* seqs, int n_seqs,
                              const void* k_tree, const void* v_tree, const void* q, const int32_t* parent,
                              int t_nodes, int path, void* workspace, size_t ws_bytes, void* o, int32_t* dev_status,
                              stv_stream_t stream);

/*
 * Failure-path test of stv_verify_attn (the pages have no counterpart: it
 * exists to test this library's failure detection without a GPU fault).
 * Same arguments and checks as stv_verify_attn, but the kernel's producer
 * issues none of its copies, so the waits on them never complete: every
 * wait gives up after its bound (about 1.3 s), the kernel stops every role,
 * waits for anything it issued, frees its tensor memory, ORs
 * STV_DEV_TIMEOUT into *dev_status and returns.  The workspace's partials
 * are then invalid; the CUDA context stays usable.
 */
int stv_verify_attn_timeout_test(const stv_shape* shape, const stv_layer_cache* layer, const stv_seq* seqs,
                                 int n_seqs, const void* q, const int32_t* parent, int t_nodes, int path,
                                 void* workspace, size_t ws_bytes, int32_t* dev_status, stv_stream_t stream);

/*
 * a5 -- merge the split partials of the last stv_verify_attn on this
 * workspace: per row M = max_s m_s, O = sum_s 2^(m_s - M) O_s / sum_s
 * 2^(m_s - M) l_s, splits taken in a fixed order (deterministic).
 *  o: device fp16 [n_seqs][T][hq][256].
 */
int stv_split_combine(const stv_shape* shape, const stv_seq* seqs, int n_seqs, int t_nodes, const void* workspace,
                      size_t ws_bytes, void* o, stv_stream_t stream);

/*
 * a6 -- exact greedy tree acceptance ("elpis" README, "Why fast": commit the
 * longest matching path + 1; "elpis-lossless" README, "Lossless": token ids
 * compared exactly).  Edge p -> c matches iff draft_ids[c] ==
 * target_argmax[p].  Longest root path of matching edges; among equally
 * long ones the lexicographically smallest node-index sequence.
 *  parent, draft_ids, target_argmax: device int32 [n_seqs][T].
 *  n_commit: device int32 [n_seqs] = accepted depth + 1 (0 for a bad tree).
 *  path:     device int32 [n_seqs][T], first n_commit entries: node indices
 *            from the root (path[0] = 0); the rest are set to -1.
 *  out_ids:  device int32 [n_seqs][T], first n_commit entries: the accepted
 *            drafts, then the bonus token target_argmax[last node]; rest -1.
 */
int stv_tree_accept(const int32_t* parent, const int32_t* draft_ids, const int32_t* target_argmax, int t_nodes,
                    int n_seqs, int32_t* n_commit, int32_t* path, int32_t* out_ids, int32_t* dev_status,
                    stv_stream_t stream);

/*
 * a7 -- compact the accepted rows: for every layer, KV head and i <
 * n_commit[s], the packed row at slot ctx + path[i] moves to slot ctx + i
 * (all sources are read before any destination is written), then
 * ctx_dev[s] += n_commit[s].  A sequence is committed in every layer or in
 * none: one whose n_commit is outside [1, T] or whose path is not a root
 * path is left untouched (STV_DEV_BAD_COMMIT), and so is one whose source or
 * destination positions are past its page table or map to a page outside
 * any layer's pool (STV_DEV_BAD_PAGE); ctx_dev[s] then stays as it was.
 *  layers:   host array of n_layers caches (device pools).
 *  n_commit, path: device, as written by stv_tree_accept.
 *  ctx_dev:  device int32 [n_seqs] (may be NULL).
 * Uses seqs[s].ctx (host) as the round's context length.
 */
int stv_kv_commit(const stv_shape* shape, const stv_layer_cache* layers, int n_layers, const stv_seq* seqs,
                  int n_seqs, int t_nodes, const int32_t* n_commit, const int32_t* path, int32_t* ctx_dev,
                  int32_t* dev_status, stv_stream_t stream);

/*
 * Inspection of the int8 path ("elpis" README, "Why fast": 3-bit K codes as
 * exact int8): stv_verify_attn with STV_PATH_INT8 on one sequence that also
 * writes out the per-group integer dots the verify kernel itself forms on
 * the tensor cores, I_g = sum_{c in g} qi_c * (code_c - 4), for every key of
 * [0, ctx + T) and every query row (whatever the tree mask says).
 *  q, parent, t_nodes, workspace: as in stv_verify_attn (n_seqs = 1); the
 *            workspace receives the same partials as stv_verify_attn.
 *  dots:     device int32 [hkv][T * G][ctx + T][8]; row r of KV head h is
 *            node r / G, Q head h * G + r % G (G = hq / hkv).
 * STV_ERR_UNIMPLEMENTED on the int4 cache (group 256), whose int8 path has
 * one group per key.
 */
int stv_int8_qk_dots(const stv_shape* shape, const stv_layer_cache* layer, const stv_seq* seq, const void* q,
                     const int32_t* parent, int t_nodes, void* workspace, size_t ws_bytes, int32_t* dots,
                     int32_t* dev_status, stv_stream_t stream);

/*
 * Verify attention and split merge in one call, without a caller workspace
 * (no counterpart on the pages: it exists for callers of this library that
 * cannot allocate device memory -- e.g. a serving engine whose allocator
 * already owns nearly all device memory, where an extra cudaMalloc during a
 * decode step can fail, or a plain C host without a device allocator).
 * Same arguments, checks and results as stv_verify_attn followed by
 * stv_split_combine, with o as in stv_split_combine.  The scratch is a
 * fixed 32 MiB array inside the library: it calls no cudaMalloc, cudaFree
 * or allocating routine, and every GPU that loads the library keeps those
 * 32 MiB until the process exits.  A round whose workspace
 * (stv_verify_workspace_bytes) exceeds 32 MiB returns
 * STV_ERR_WORKSPACE_TOO_SMALL and enqueues nothing.  All calls share the
 * array: calls that overlap on the GPU (other streams or host threads) race
 * and must be serialised by the caller.  The first call on each device looks
 * the array's device address up (a CUDA runtime query, once per device) and
 * should come before any stream capture.
 */
int stv_verify_attn_no_alloc(const stv_shape* shape, const stv_layer_cache* layer, const stv_seq* seqs, int n_seqs,
                             const void* q, const int32_t* parent, int t_nodes, int path, void* o,
                             int32_t* dev_status, stv_stream_t stream);

/*
 * Prefill attention over the 3-bit cache (next row f2): every token of a
 * prompt attends causally to the cache and to the prompt tokens before it.
 * "elpis" README, "Why fast" (prefill int8 Q.K^T, 3021c; prefill K/V
 * double-buffered ring, 3022: the next tile loads while the current one is
 * computed).  A chunk of C consecutive prompt tokens is a chain tree
 * (parent[i] = i - 1), whose ancestor-or-self mask is the causal mask,
 * appended after the tokens before it; C = min(32, floor(128 / (hq / hkv)))
 * rows per chunk fill the 128-row tile.  Exact path on the 3-bit cache: one
 * persistent launch, one CTA per SM walking (chunk, KV head) units longest
 * first, each over the chunk's whole key range, writing O / l directly (the
 * workspace is not used).  int8 path and the other cache formats: up to 64
 * chunks per verify launch, then the split merge.
 *  seq:      ctx = tokens cached before the prompt; the prompt's own K/V
 *            rows must already be in the cache at ctx .. ctx + n_tokens - 1
 *            (stv_kv_append_pack), so attention reads them in 3-bit, like
 *            every cached token.
 *  q:        device fp16 [n_tokens][hq][256].   o: device fp16 [n_tokens][hq][256].
 *  path:     STV_PATH_EXACT or STV_PATH_INT8, as in stv_verify_attn.
 *  workspace: device, at least stv_prefill_workspace_bytes(...) bytes.
 * Errors as in stv_verify_attn; n_tokens < 1 is STV_ERR_INVALID_ARG.
 */
int stv_prefill_workspace_bytes(const stv_shape* shape, const stv_seq* seq, int n_tokens, size_t* bytes);
int stv_prefill_attn(const stv_shape* shape, const stv_layer_cache* layer, const stv_seq* seq, const void* q,
                     int n_tokens, int path, void* workspace, size_t ws_bytes, void* o, int32_t* dev_status,
                     stv_stream_t stream);

/*
 * Failure-path test of stv_prefill_attn's persistent kernel (exact path, the
 * 3-bit cache; the pages have no counterpart: it exists to test this
 * library's failure detection without a GPU fault).  Same arguments and
 * checks as stv_prefill_attn; the kernel's producer issues none of its
 * copies, so every wait on them gives up after its bound (about 1.3 s), the
 * kernel stops every role, waits for anything it issued, frees its tensor
 * memory, ORs STV_DEV_TIMEOUT into *dev_status and returns.  `o` is then
 * invalid; the CUDA context stays usable.  STV_ERR_UNIMPLEMENTED for the
 * int8 path and the other cache formats.
 */
int stv_prefill_attn_timeout_test(const stv_shape* shape, const stv_layer_cache* layer, const stv_seq* seq,
                                  const void* q, int n_tokens, int path, void* workspace, size_t ws_bytes, void* o,
                                  int32_t* dev_status, stv_stream_t stream);

/*
 * Lookup drafting (next row f4).  Reddit posts (u/iamMess), "Now added" list,
 * lookup-augmented drafting (draft tokens copied from earlier in the same
 * request: find where its trailing tokens, between six and twelve of them,
 * last appeared before, and take what came next); syv-ai README (mirror),
 * SPEC=dflash2 section (verify slots past the drafter's come from the
 * request's own context).
 *
 * For each sequence with history h[0 .. n-1]: lengths L = max_len down to
 * min_len are tried; for the first L whose suffix h[n-L .. n-1] occurs at an
 * earlier start p < n - L (the occurrence may overlap the suffix), the
 * latest such p is taken and up to k tokens h[p+L ..] are proposed, never
 * past h[n-1].  With no occurrence nothing is proposed.
 *  hist:      host array of n_seqs descriptors; each tokens pointer is device
 *             int32 [n] owned by the caller (read only); n may be 0.
 *  min_len, max_len: 1 <= min_len <= max_len <= 32.   k: 0 <= k <= 64.
 *  n_prop:    device int32 [n_seqs]: tokens proposed (0..k).
 *  prop:      device int32 [n_seqs][k]: the proposal, zero beyond n_prop.
 *  match_len: device int32 [n_seqs]: L, or 0 when nothing matched.
 *  match_pos: device int64 [n_seqs]: p, or -1 when nothing matched.
 *  workspace: device, at least stv_lookup_workspace_bytes(n_seqs) bytes,
 *             caller-owned, ZERO before the first call (e.g. allocated
 *             zeroed); every call leaves the bytes it used zero again, so
 *             the same workspace serves any later call without clearing.
 * Returns STV_ERR_INVALID_ARG for lengths, k or n_seqs out of range, null
 * pointers or a workspace too small (STV_ERR_WORKSPACE_TOO_SMALL).  The
 * result is unique, so it does not depend on timing.
 */
typedef struct {
  const int32_t* tokens;
  int64_t n;
} stv_history;

int stv_lookup_workspace_bytes(int n_seqs, size_t* bytes);
int stv_lookup_draft(const stv_history* hist, int n_seqs, int min_len, int max_len, int k, int32_t* n_prop,
                     int32_t* prop, int32_t* match_len, int64_t* match_pos, void* workspace, size_t ws_bytes,
                     stv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* STV_H_ */
