// verify_tc.cu -- a2..a4 on the 5th-generation tensor cores (tcgen05, TMEM,
// bulk async copies): split-KV, tree-masked GQA verify attention over the
// paged 3-bit cache.
//
// Sources: "elpis" README, "Why fast" (8-row token tree verified in one pass;
// decode verify with the 3-bit K codes as exact int8 against int8 Q; prefill
// K/V double-buffered ring: the next tile loads while the current one is
// computed); Reddit posts (u/iamMess), second post (split-KV verify kernel).
// The pages' kernels target the RTX 3090 (mma.sync, IMMA); this one is laid
// out for sm_103a.
//
// One CTA per work unit (sequence, KV head, range of 64-key tiles), one CTA
// per SM, 14 warps:
//   warp 0      producer: one bulk copy per array per tile (K codes, K scales,
//               V codes, V scales: 14,336 B) into a 4-stage shared ring.
//   warp 1      TMEM owner and MMA issuer (the warp runs the loop, one
//               elected lane issues).
//   warps 2-5   softmax: thread = query row = TMEM lane (128 rows, the
//               T*G rows sharing the KV head, zero-padded).
//   warps 6-13  unpack: 3-bit codes -> fp16 operands in shared memory.
//   warp 14     (the kFused instantiation only) packs the round's tree rows.
// The warp index is read from lane 0, so the compiler knows the role
// branches are warp-uniform.  At the end each softmax warp stages its O rows
// through the freed operand buffers and writes them coalesced.
// Tensor memory (512 columns): Q [0,128) as the A operand of S = Q K^T;
// S0/S1 [128,192) [192,256), double-buffered, where P (fp16) overwrites S as
// the A operand of O += P V; O [256,512) fp32 accumulators.
// Shared memory: K (64 keys x 256 ch) and V^T (256 ch x 64 keys) fp16
// operands, 128-byte swizzled K-major; K double-buffered, V^T triple-buffered
// (the unpack may store V of tile i while P.V reads tiles i-1 and i-2, which
// measured 4.6 % faster at 262K than two buffers); the raw ring.
// This kernel runs the exact path on the 3-bit cache and both paths on the
// int4 cache (one K scale per key: Q.K over the exact codes, then the score
// times the key's scale, so the int8 path's integer dot is formed exactly in
// the fp32 accumulator).  The int8 path on the 3-bit cache, whose definition
// needs per-group integer dots, runs in verify_i8.cu.
// Softmax is online in fp32 with a stale-maximum threshold: P uses a
// reference maximum that is raised (rescaling O and l) only when a score
// exceeds it by more than 2^8, so P <= 256 in fp16 and O rescales are rare.
// Every wait is bounded; a timeout sets a CTA abort flag, every role stops,
// in-flight copies and MMAs are waited for (bounded) and TMEM is freed.
#include "combine.cuh"
#include "stv_device.cuh"
#include "tc_util.cuh"

namespace stv {
namespace {

constexpr int kThreads = 448;
constexpr int kStages = 4;
constexpr int kStageBytes = kKTileCodeBytes + kKTileScaleBytes + kVTileCodeBytes + kVTileScaleBytes;  // 14336
constexpr int kOperandBytes = 32768;  // one K or V^T fp16 tile
constexpr int kVBuffers = 3;  // V^T tiles in flight: unpack may run two P.V products ahead
constexpr int kSmemBytes = 1024 /*align slack*/ + (2 + kVBuffers) * kOperandBytes + kStages * kStageBytes + 1024 /*barriers etc*/;

// The cache format's tile arrays (include/stv.h): the pages' 3-bit cache, or
// the int4 per-token-head cache, whose larger stage leaves room for 3 stages.
// The int4 K scale is one per key for the whole head, so it factors out of
// Q.K: the K operand holds the exact codes and the softmax multiplies key j's
// score by its scale in fp32 (no fp16 rounding of scale * code on the score
// path).  The unpack warps hand the scales over in slot i % kKScaleSlots:
// unpacking tile i + 4 waits for QK(i + 2) to finish, which the MMA warp
// issues only after the softmax of tile i has arrived on p_full, so a slot is
// never rewritten while it is read.
constexpr int kKScaleSlots = 4;
template <int kFmt>
struct Fmt {  // the 3-bit cache
  static constexpr int stages = kStages;
  static constexpr int head = kHeadBytes;
  static constexpr int off_kc = kOffKCodes, off_ks = kOffKScales, off_vc = kOffVCodes, off_vs = kOffVScales;
  static constexpr int kc = kKTileCodeBytes, ks = kKTileScaleBytes, vc = kVTileCodeBytes, vs = kVTileScaleBytes;
  static constexpr int stage = kStageBytes;
  static constexpr int smem = kSmemBytes;
};
template <>
struct Fmt<kFmtInt4> {
  static constexpr int stages = 3;
  static constexpr int head = kI4HeadBytes;
  static constexpr int off_kc = kI4OffKCodes, off_ks = kI4OffKScales, off_vc = kI4OffVCodes, off_vs = kI4OffVScales;
  static constexpr int kc = kI4KTileCodeBytes, ks = kI4KTileScaleBytes, vc = kI4VTileCodeBytes, vs = kI4VTileScaleBytes;
  static constexpr int stage = kc + ks + vc + vs;  // 16640
  // + the per-key K scales of the last kKScaleSlots tiles, as fp32
  static constexpr int smem = 1024 + (2 + kVBuffers) * kOperandBytes + stages * stage + 1024 + kKScaleSlots * kTileTok * 4;
};
// The K 4 / V 2-bit cache: a tile's arrays take the 3-bit cache's 14,336 bytes.
template <>
struct Fmt<kFmtK4V2> {
  static constexpr int stages = kStages;
  static constexpr int head = kKv2HeadBytes;
  static constexpr int off_kc = kKv2OffKCodes, off_ks = kKv2OffKScales, off_vc = kKv2OffVCodes,
                       off_vs = kKv2OffVScales;
  static constexpr int kc = kKv2KTileCodeBytes, ks = kKv2KTileScaleBytes, vc = kKv2VTileCodeBytes,
                       vs = kKv2VTileScaleBytes;
  static constexpr int stage = kc + ks + vc + vs;  // 14336
  static constexpr int smem = kSmemBytes;
};
static_assert(Fmt<kFmtK4V2>::stage == kStageBytes, "stage");
static_assert(Fmt<kFmtInt4>::stages <= kStages, "barrier arrays");
static_assert(Fmt<kFmtInt4>::smem <= 232448, "shared memory per CTA");
constexpr float kRescaleThreshold = 8.f;  // log2 units

constexpr uint32_t kColQ = 0, kColS0 = 128, kColO = 256, kTmemCols = 512;

constexpr uint32_t kIdescQK = idesc_f16_f32(128, 64);
constexpr uint32_t kIdescPV = idesc_f16_f32(128, 256);

struct Bars {
  uint64_t raw_full[kStages], raw_empty[kStages];
  uint64_t kd_full[2], kd_empty[2], vd_full[kVBuffers], vd_empty[kVBuffers];
  uint64_t s_full[2], p_full[2];
  uint64_t pv_done, q_ready, mma_done;
  uint64_t tree_packed;  // the round's tree rows of this unit are in the cache (fused append)
  uint32_t tmem_base;
  int abort;
};

static_assert(sizeof(Bars) <= 1024, "barrier block");

// Waits suspend (try_wait with a time hint): measured faster here than
// polling, since this kernel's roles mostly wait on the tensor pipe.
__device__ __forceinline__ bool wait1(uint64_t* b, uint32_t parity, volatile int* abort_flag) {
  return stv::wait1<false>(b, parity, abort_flag);
}
__device__ __forceinline__ bool waitw(uint64_t* b, uint32_t parity, volatile int* abort_flag) {
  return stv::waitw<false>(b, parity, abort_flag);
}
__device__ __forceinline__ bool settle(uint64_t* b, uint32_t parity, uint32_t probed, volatile int* abort_flag) {
  return stv::settle<false>(b, parity, probed, abort_flag);
}

// The epilogue's copy of one softmax warp's 32 O rows (TMEM lane quarter
// `quad`) into the workspace, staged through shared memory (`stage`: the
// operand buffers, 128 KiB, free once every MMA has finished).  Each row goes
// TMEM -> shared memory, its 16-byte pieces XOR-swizzled by row mod 8 so the
// warp's stores spread over the banks; then the warp copies the rows out one
// at a time, a lane per 16 bytes: coalesced 512-byte stores instead of 32
// lanes writing 32 rows 1 KiB apart (measured: 262K 119.6 -> 117.2 us per
// layer-round, 32K unchanged).  Out of line, so the tile loop's code does
// not change with it.
__device__ __noinline__ void epilogue_rows_staged(uint32_t lane_addr, uint8_t* stage, float* dst0, int quad, int R) {
  const int lane = threadIdx.x & 31, r = quad * 32 + lane;
  const uint32_t srow = su32(stage) + (uint32_t)r * 1024u;
#pragma unroll 1
  for (int chunk = 0; chunk < 8; ++chunk) {
    uint32_t o[32];
    tmem_ld32(lane_addr + kColO + 32 * chunk, o);
    tmem_wait_ld(o);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      st_shared_v4(srow + chunk * 128u + (uint32_t)((j ^ (r & 7)) << 4), o[4 * j], o[4 * j + 1], o[4 * j + 2],
                   o[4 * j + 3]);
  }
  __syncwarp();
  const int r_end = min(R, quad * 32 + 32);
#pragma unroll 1
  for (int rr = quad * 32; rr < r_end; ++rr) {
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int q = lane + 32 * hf;  // 16-byte piece of the row, 0..63
      const uint4 x = *reinterpret_cast<const uint4*>(stage + rr * 1024 + (q >> 3) * 128 + (((q & 7) ^ (rr & 7)) << 4));
      reinterpret_cast<uint4*>(dst0 + (int64_t)rr * kHeadDim)[q] = x;
    }
  }
}

// kFused: the round's tree rows (a1), packed by one extra warp of each unit
// before the tiles are read: (sequence, row, KV head) pair q goes to unit
// q mod n_units; lane = channel of each 32-channel group in turn, V bits by
// atomics (rows packed by other units may share a V word).  A warp that
// packed arrives once on the launch's counter, after a proxy fence and a
// release.  Out of line, so that none of it enters the other roles' code.
__device__ __noinline__ void fused_pack_tree_rows(const VerifyParams& p) {
  const int lane = threadIdx.x & 31;
  bool packed = false;
  // Start this unit's rows (512 bytes of K and of V each) on their way to L2
  // first: the packing loop loads them one 32-channel group at a time, each
  // group after the previous group's stores, so every load would otherwise
  // wait out a full trip to HBM.
  for (int q = blockIdx.x; q < p.n_pairs; q += p.n_units) {
    const int64_t row = (int64_t)q * kHeadDim;  // pair q = (sequence row, KV head)
    if (lane < 4) asm volatile("prefetch.global.L2 [%0];" ::"l"(p.k_tree + row + lane * 64));
    else if (lane < 8) asm volatile("prefetch.global.L2 [%0];" ::"l"(p.v_tree + row + (lane - 4) * 64));
  }
  for (int q = blockIdx.x; q < p.n_pairs; q += p.n_units) {
    const int h2 = q % p.hkv, si = q / p.hkv, s2 = si / p.T;
    const int64_t pos = (int64_t)p.seq[s2].ctx + si % p.T;
    const int64_t row = ((int64_t)si * p.hkv + h2) * kHeadDim;
    // all eight groups' values in flight at once (read-only loads), then
    // the rolled packing loop over them
    __half2 kv[8];
#pragma unroll
    for (int g = 0; g < 8; ++g)
      kv[g] = __halves2half2(__ldg(p.k_tree + row + g * 32 + lane), __ldg(p.v_tree + row + g * 32 + lane));
    uint8_t* hb = const_cast<uint8_t*>(
        head_block(p.seq[s2], p.pool, p.page_bytes, p.pool_pages, pos, h2, lane == 0 ? p.status : nullptr));
    if (hb) {
#pragma unroll 1
      for (int g = 0; g < 8; ++g)
        append_row_channel(__low2float(kv[g]), __high2float(kv[g]), hb, (int)(pos & (kPageTok - 1)), g * 32 + lane);
    }
    packed = true;
  }
  if (packed) {
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
      __threadfence();
      atomicAdd(p.cnt, 1u);
    }
  }
}

// kFused: a5 inside the verify launch, by every warp of a unit after its
// teardown.  The unit first publishes its partials on its (sequence, KV
// head)'s counter (the softmax warps wrote them before the teardown barrier;
// the release is cumulative over them).  The merge's items, (sequence, KV
// head, row, channel quarter) over the whole launch, are dealt to the units
// in equal contiguous ranges; a warp waits (bounded: the launch is
// cooperative, every unit is resident) until every unit of an item's head has
// published, then merges it with combine_row_quarter_lean (loads from L2),
// whose sums are split_combine's, bit for bit.  A unit that aborted still
// publishes and counts itself done, so no other unit waits for it past its
// bound.  The last unit of the launch to be done zeroes the counters for the
// next launch: every unit has passed every wait of this one by then.
__device__ __noinline__ void fused_merge(const VerifyParams& p, volatile int* abort_flag, int my_s, int my_h) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, n_warps = blockDim.x >> 5;
  // the fused append alone (stv_append_verify_attn): no merge, only the
  // counters' reset below
  const bool merge = p.o_out != nullptr;
  if (merge && tid == 0) {
    __threadfence();
    atomicAdd(p.cnt + 2 + my_s * p.hkv + my_h, 1u);
  }
  const int per_head = 4 * p.R, n_items = merge ? p.n_seqs * p.hkv * per_head : 0;
  const int i0 = (int)((int64_t)blockIdx.x * n_items / p.n_units);
  const int i1 = (int)((int64_t)(blockIdx.x + 1) * n_items / p.n_units);
  int waited = -1;
  bool ok = !*abort_flag;
  for (int it = i0 + warp; ok && it < i1; it += n_warps) {
    const int head = it / per_head, rq = it % per_head;
    const int s = head / p.hkv, h = head % p.hkv;
    if (head != waited) {
      bool w = true;
      if (lane == 0) w = wait_count(p.cnt + 2 + head, (uint32_t)p.seq[s].splits, abort_flag);
      ok = __shfl_sync(0xffffffffu, w, 0);
      waited = head;
      if (!ok) break;
    }
    combine_row_quarter_lean<true>(p.seq[s], s, h, rq >> 2, rq & 3, p.R, p.T, p.hq, p.G, p.o_part, p.ml, p.o_out);
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(p.cnt + 1, 1u) == (uint32_t)p.n_units - 1) {
      p.cnt[0] = 0u;
      p.cnt[1] = 0u;
      for (int i = 0; i < p.n_seqs * p.hkv; ++i) p.cnt[2 + i] = 0u;
      __threadfence();
    }
  }
}

// kAppend: the round's tree rows are packed into the cache by this launch
// (stv_append_verify_attn); the plain instantiation carries none of that code.
// kWithhold (failure-path test only, stv_verify_attn_timeout_test): the
// producer issues no copy, so every wait on one runs out.
// kFused (cooperative launch): a fifteenth warp packs the round's tree rows
// (fused_pack_tree_rows), a unit copies a tile holding tree keys once every
// packing warp of the launch has arrived on a device counter, and after the
// teardown the units merge the splits (fused_merge) -- one launch per layer,
// stv_append_verify_combine -- or, with no output given, leave the partials
// to split_combine (stv_append_verify_attn for one sequence).
template <bool kAppend, int kFmt, bool kWithhold = false, bool kFused = false>
__global__ void __launch_bounds__(kFused ? kThreads + 32 : kThreads, 1)
    verify_tc_kernel(const __grid_constant__ VerifyParams p) {
  using F = Fmt<kFmt>;
  constexpr bool kI4 = kFmt == kFmtInt4;    // one K scale per key, handed to the softmax
  constexpr bool kKv2 = kFmt == kFmtK4V2;  // 4-bit K, 2-bit V, scales per 32-channel group
  constexpr bool kBit3 = !kI4 && !kKv2;    // the 3-bit cache
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment of the operand tiles (the swizzle works on address bits).
  const uint32_t base_u32 = su32(smem_raw);
  uint8_t* smem = smem_raw + ((1024 - (base_u32 & 1023)) & 1023);
  uint8_t* const kdeq0 = smem;                      // K tiles: kdeq0 + b * kOperandBytes
  uint8_t* const vdeq0 = smem + 2 * kOperandBytes;  // V^T tiles: vdeq0 + b * kOperandBytes
  uint8_t* ring = smem + (2 + kVBuffers) * kOperandBytes;
  Bars* bars = reinterpret_cast<Bars*>(ring + F::stages * F::stage);
  float* const kscale = reinterpret_cast<float*>(ring + F::stages * F::stage + 1024);  // int4 only
  volatile int* abort_flag = &bars->abort;

  const int tid = threadIdx.x, lane = tid & 31;
  // The warp index, read from lane 0: the compiler then knows it is the same
  // across the warp, so the role branches below are warp-uniform (derived
  // from threadIdx.x alone they were compiled as possibly divergent: about
  // 7 % slower, and every role's loop changed with any code added to another).
  const int warp = __shfl_sync(0xffffffffu, tid >> 5, 0);

  // ---- locate the work unit ----
  int s = 0;
  while (s + 1 < p.n_seqs && (int)blockIdx.x >= p.seq[s + 1].unit_base) ++s;
  const SeqDesc sd = p.seq[s];
  const int local = blockIdx.x - sd.unit_base;
  const int h = local / sd.splits, split = local % sd.splits;
  const int T = p.T, G = p.G, R = p.R;
  const int tok0 = split * p.tiles_per_split * kTileTok;
  const int tok1 = min(sd.ctx + T, tok0 + p.tiles_per_split * kTileTok);
  const int n_tiles = (tok1 - tok0 + kTileTok - 1) / kTileTok;

  // ---- set-up ----
  if (tid == 0) {
    for (int i = 0; i < F::stages; ++i) {
      mbar_init(&bars->raw_full[i], 1);
      mbar_init(&bars->raw_empty[i], 8);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->kd_full[i], 8);
      mbar_init(&bars->kd_empty[i], 1);
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 4);
    }
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->q_ready, 4);
    mbar_init(&bars->mma_done, 1);
    mbar_init(&bars->tree_packed, 8);
    for (int i = 0; i < kVBuffers; ++i) {
      mbar_init(&bars->vd_full[i], 8);
      mbar_init(&bars->vd_empty[i], 1);
    }
    bars->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // Nothing above touches global memory: the previous kernel may still be running.
  grid_dep_wait();
  // Start the first global reads' trips to L2 before the set-up barrier:
  // the producer's first page-table line and the softmax threads' Q rows.
  if (tid == 0) asm volatile("prefetch.global.L2 [%0];" ::"l"(sd.page_table + (tok0 >> 8)));
  if (warp >= 2 && warp < 6) {
    const int r = (warp & 3) * 32 + lane;
    if (r < R) {
      const char* qr = p.path == STV_PATH_INT8
                           ? reinterpret_cast<const char*>(p.qi + (((int64_t)s * T + r / G) * p.hq + h * G + r % G) * kHeadDim)
                           : reinterpret_cast<const char*>(p.q + (((int64_t)s * T + r / G) * p.hq + h * G + r % G) * kHeadDim);
      const int lines = p.path == STV_PATH_INT8 ? 2 : 4;  // 256 int8 or 512 fp16 bytes
      for (int ln = 0; ln < lines; ++ln) asm volatile("prefetch.global.L2 [%0];" ::"l"(qr + 128 * ln));
    }
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&bars->tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_before();
  __syncthreads();
  tc_after();
  grid_dep_launch();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // =================== producer ===================
    if (lane == 0) {
      int issued = 0;
      bool tree_ready = !kAppend && !kFused;
      for (int i = 0; i < (kWithhold ? 0 : n_tiles); ++i) {
        const int st = i % F::stages;
        if (!wait1(&bars->raw_empty[st], ((i / F::stages) & 1) ^ 1, abort_flag)) break;
        const int key0 = tok0 + i * kTileTok;
        // a tile holding tree keys is copied only after the unpack warps have
        // packed them (their global writes are fenced for the async proxy)
        if (!tree_ready && key0 + kTileTok > sd.ctx && key0 < sd.ctx + T) {
          if constexpr (kFused) {
            if (!wait_count(p.cnt, (uint32_t)p.packed_target, abort_flag)) break;
          } else {
            if (!wait1(&bars->tree_packed, 0, abort_flag)) break;
          }
          tree_ready = true;
        }
        const int64_t lp = key0 >> 8;
        int32_t page = lp < sd.n_pages ? __ldg(sd.page_table + lp) : -1;
        if (page < 0 || page >= p.pool_pages) {
          report(p.status, STV_DEV_BAD_PAGE);
          page = 0;  // read a valid page; the result is flagged as garbage
        }
        const uint8_t* hb = p.pool + (int64_t)page * p.page_bytes + (int64_t)h * F::head;
        const int t = (key0 & (kPageTok - 1)) / kTileTok;
        uint8_t* dst = ring + st * F::stage;
        uint64_t* bar = &bars->raw_full[st];
        mbar_expect_tx(bar, F::stage);
        bulk_g2s(dst, hb + F::off_kc + t * F::kc, F::kc, bar);
        bulk_g2s(dst + F::kc, hb + F::off_ks + t * F::ks, F::ks, bar);
        bulk_g2s(dst + F::kc + F::ks, hb + F::off_vc + t * F::vc, F::vc, bar);
        bulk_g2s(dst + F::kc + F::ks + F::vc, hb + F::off_vs + t * F::vs, F::vs, bar);
        issued = i + 1;
      }
      // No copy may still be landing when the CTA exits.
      for (int i = max(0, issued - F::stages); i < issued; ++i) {
        volatile int never = 0;
        wait1(&bars->raw_full[i % F::stages], (i / F::stages) & 1, &never);
      }
    }
  } else if (warp == 1) {
    // =================== MMA issuer (whole warp, one elected lane issues) ===================
    const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
    bool ok = waitw(&bars->q_ready, 0, abort_flag);
    tc_after();
    // Issue order: QK(0), QK(1), then PV(j), QK(j+2) for j = 0, 1, ...
    // S is double-buffered: QK(j+2) overwrites the columns that held P(j),
    // after PV(j) in the tensor pipe's order, while softmax(j+1) runs.
    // Descriptors are built once; each MMA then only adds a constant to the
    // start-address field (no carry: shared addresses are < 256 KiB).
    // Rebuilding them per MMA made the issue loop, which competes with the
    // unpack and softmax warps for issue slots, slower than the tensor pipe.
    const uint64_t kdesc0 = desc_sw128(su32(kdeq0)), vdesc0 = desc_sw128(su32(vdeq0));
    auto issue_qk = [&](int i) -> bool {
      const int b = i & 1;
      if (!settle(&bars->kd_full[b], (i >> 1) & 1, probe(&bars->kd_full[b], (i >> 1) & 1), abort_flag)) return false;
      tc_after();
      const uint64_t kd = kdesc0 + (uint64_t)(b * (kOperandBytes >> 4));
      const uint32_t d = tm + kColS0 + 64 * b;
#pragma unroll
      for (int kk = 0; kk < 16; ++kk)
        mma_tmemA(d, tm + kColQ + 8 * kk, kd + (uint64_t)((kk >> 2) * 512 + (kk & 3) * 2), kIdescQK, kk > 0);
      tc_commit(&bars->kd_empty[b]);
      tc_commit(&bars->s_full[b]);
      return true;
    };
    for (int i = 0; ok && i < 2 && i < n_tiles; ++i) ok = issue_qk(i);
    for (int j = 0; ok && j < n_tiles; ++j) {
      const int b = j & 1;
      const uint32_t pr_p = probe(&bars->p_full[b], (j >> 1) & 1);
      const int vb = j % kVBuffers;
      const uint32_t pr_v = probe(&bars->vd_full[vb], (j / kVBuffers) & 1);
      if (!(ok = settle(&bars->p_full[b], (j >> 1) & 1, pr_p, abort_flag))) break;
      if (!(ok = settle(&bars->vd_full[vb], (j / kVBuffers) & 1, pr_v, abort_flag))) break;
      tc_after();
      const uint64_t vd = vdesc0 + (uint64_t)(vb * (kOperandBytes >> 4));
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_tmemA(tm + kColO, tm + kColS0 + 64 * b + 8 * kk, vd + (uint64_t)(kk * 2), kIdescPV, (j > 0 || kk > 0));
      tc_commit(&bars->vd_empty[vb]);
      tc_commit(&bars->pv_done);
      if (j + 2 < n_tiles) ok = issue_qk(j + 2);
    }
    // Every MMA issued here has finished before TMEM is freed.
    tc_commit(&bars->mma_done);
    volatile int never = 0;
    waitw(&bars->mma_done, 0, &never);
  } else if (warp < 6) {
    // =================== softmax (thread = row = TMEM lane) ===================
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
    const bool int8 = p.path == STV_PATH_INT8;
    float c = kLog2e / 16.f;
    int node = 0;
    // Q row -> TMEM columns [0, 128)
    {
      int64_t qrow = 0;
      const bool live = r < R;
      if (live) {
        node = r / G;
        qrow = ((int64_t)s * T + node) * p.hq + h * G + r % G;
        if (int8) c *= p.sq[qrow];
      }
#pragma unroll
      for (int chunk = 0; chunk < 4; ++chunk) {
        uint32_t v[32];
        if (!live) {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0u;
        } else if (!int8) {
          const uint4* src = reinterpret_cast<const uint4*>(p.q + qrow * kHeadDim + chunk * 64);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            uint4 x = __ldg(src + e);
            v[4 * e] = x.x;
            v[4 * e + 1] = x.y;
            v[4 * e + 2] = x.z;
            v[4 * e + 3] = x.w;
          }
        } else {
          const int8_t* src = p.qi + qrow * kHeadDim + chunk * 64;
#pragma unroll
          for (int e = 0; e < 32; ++e)
            v[e] = h2u(__halves2half2(__int2half_rn(src[2 * e]), __int2half_rn(src[2 * e + 1])));
        }
        tmem_st32(lane_addr + kColQ + 32 * chunk, v);
      }
      tmem_wait_st();
      tc_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->q_ready);
    }
    // a2: this row's ancestor-or-self mask, from parent[] (only the tiles
    // that hold tree keys use it, so its loads overlap the first tiles)
    uint32_t anc = 1u << node;
    {
      int n = node;
      const int32_t* par = p.parent + (int64_t)s * T;
      for (int st = 0; st < T && n > 0; ++st) {
        const int pa = __ldg(par + n);
        if (pa < 0 || pa >= n) {
          if (split == 0 && h == 0) report(p.status, STV_DEV_BAD_TREE);
          break;
        }
        anc |= 1u << pa;
        n = pa;
      }
      if (r == 0 && __ldg(par) != -1 && split == 0 && h == 0) report(p.status, STV_DEV_BAD_TREE);
    }
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int i = 0; i < n_tiles; ++i) {
      const int b = i & 1;
      if (!(ok = waitw(&bars->s_full[b], (i >> 1) & 1, abort_flag))) break;
      tc_after();
      uint32_t sa[32], sb[32];
      tmem_ld32(lane_addr + kColS0 + 64 * b, sa);
      tmem_ld32(lane_addr + kColS0 + 64 * b + 32, sb);
      tmem_wait_ld(sa);
      tmem_wait_ld(sb);
      if constexpr (kI4) {  // S = (Q.codes) * per-key scale, in fp32
        const float4* ksc = reinterpret_cast<const float4*>(kscale + (i % kKScaleSlots) * kTileTok);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float4 x = ksc[e], y = ksc[8 + e];
          sa[4 * e] = __float_as_uint(__uint_as_float(sa[4 * e]) * x.x);
          sa[4 * e + 1] = __float_as_uint(__uint_as_float(sa[4 * e + 1]) * x.y);
          sa[4 * e + 2] = __float_as_uint(__uint_as_float(sa[4 * e + 2]) * x.z);
          sa[4 * e + 3] = __float_as_uint(__uint_as_float(sa[4 * e + 3]) * x.w);
          sb[4 * e] = __float_as_uint(__uint_as_float(sb[4 * e]) * y.x);
          sb[4 * e + 1] = __float_as_uint(__uint_as_float(sb[4 * e + 1]) * y.y);
          sb[4 * e + 2] = __float_as_uint(__uint_as_float(sb[4 * e + 2]) * y.z);
          sb[4 * e + 3] = __float_as_uint(__uint_as_float(sb[4 * e + 3]) * y.w);
        }
      }
      const int key0 = tok0 + i * kTileTok;
      if (key0 + kTileTok > sd.ctx || key0 + kTileTok > tok1) {
        // Visibility of the tile's 64 keys as one bit mask: context keys,
        // this row's ancestor-or-self tree keys, nothing at or past tok1.
        // Masked keys become -inf by selection (their S may be garbage).
        const int rel_ctx = sd.ctx - key0, rel_end = tok1 - key0;
        const uint64_t ctxm = rel_ctx >= 64 ? ~0ull : (rel_ctx <= 0 ? 0ull : ((1ull << rel_ctx) - 1));
        const uint64_t treem = rel_ctx >= 64 ? 0ull
                               : (rel_ctx >= 0 ? ((uint64_t)anc << rel_ctx) : ((uint64_t)anc >> (-rel_ctx)));
        const uint64_t livem = rel_end >= 64 ? ~0ull : ((1ull << rel_end) - 1);
        const uint64_t vis = (ctxm | treem) & livem;
        const uint32_t va = (uint32_t)vis, vb = (uint32_t)(vis >> 32);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          sa[e] = ((va >> e) & 1u) ? sa[e] : 0xff800000u;
          sb[e] = ((vb >> e) & 1u) ? sb[e] : 0xff800000u;
        }
      }
      // Row maximum: 3-input max, 8 independent chains.
      float mx8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx8[k] = fmaxf(__uint_as_float(sa[k]), __uint_as_float(sb[k]));
#pragma unroll
      for (int e = 8; e < 32; e += 2) {
        mx8[(e >> 1) & 7] = max3(mx8[(e >> 1) & 7], __uint_as_float(sa[e]), __uint_as_float(sa[e + 1]));
        mx8[((e >> 1) + 4) & 7] = max3(mx8[((e >> 1) + 4) & 7], __uint_as_float(sb[e]), __uint_as_float(sb[e + 1]));
      }
      const float mx = fmaxf(max3(mx8[0], mx8[1], mx8[2]), max3(max3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
      const float m_tile = mx * c;
      float corr = 1.f;
      if (m_tile > m_ref + kRescaleThreshold) {
        if (m_ref != -INFINITY) corr = ex2(m_ref - m_tile);
        m_ref = m_tile;
        l *= corr;
      }
      // P = 2^(S c - m_ref) in fp16, packed key pairs, into the S columns.
      // The exponent arguments and the row sum use the paired fp32 FMA and
      // add (two lanes per instruction, each rounded as its scalar form):
      // the softmax warps share their issue slots with the unpack warps.
      const float mref = m_ref == -INFINITY ? 0.f : m_ref;
      const float2 c2 = make_float2(c, c), nm2 = make_float2(-mref, -mref);
      float2 sum4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float2 xa = __ffma2_rn(make_float2(__uint_as_float(sa[2 * e]), __uint_as_float(sa[2 * e + 1])), c2, nm2);
        const float2 xb = __ffma2_rn(make_float2(__uint_as_float(sb[2 * e]), __uint_as_float(sb[2 * e + 1])), c2, nm2);
        const float2 pa = make_float2(ex2(xa.x), ex2(xa.y)), pb = make_float2(ex2(xb.x), ex2(xb.y));
        sum4[e & 3] = __fadd2_rn(sum4[e & 3], __fadd2_rn(pa, pb));
        sa[e] = h2u(__floats2half2_rn(pa.x, pa.y));
        sb[e] = h2u(__floats2half2_rn(pb.x, pb.y));
      }
      const float2 sum2 = __fadd2_rn(__fadd2_rn(sum4[0], sum4[1]), __fadd2_rn(sum4[2], sum4[3]));
      l += sum2.x + sum2.y;
      uint32_t pk[32];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        pk[e] = sa[e];
        pk[16 + e] = sb[e];
      }
      tmem_st32(lane_addr + kColS0 + 64 * b, pk);
      // O may be rescaled only once P.V of the previous tile has finished, so
      // a warp that rescales waits for it; the others go on.  P.V(i-2) is
      // done (QK(i) followed it) and P.V(i) waits for this warp, so pv_done
      // is in phase i-1 or i and the parity wait is unambiguous.
      if (i >= 1 && __any_sync(0xffffffffu, corr != 1.f)) {
        if (!(ok = waitw(&bars->pv_done, (i - 1) & 1, abort_flag))) break;
        tc_after();
        {
#pragma unroll 1
          for (int chunk = 0; chunk < 8; ++chunk) {
            uint32_t o[32];
            tmem_ld32(lane_addr + kColO + 32 * chunk, o);
            tmem_wait_ld(o);
            const float2 corr2 = make_float2(corr, corr);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float2 x = __fmul2_rn(make_float2(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])), corr2);
              o[2 * e] = __float_as_uint(x.x);
              o[2 * e + 1] = __float_as_uint(x.y);
            }
            tmem_st32(lane_addr + kColO + 32 * chunk, o);
          }
        }
      }
      tmem_wait_st();
      tc_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[b]);
    }
    // ---- epilogue: O, m, l of this row into the workspace ----
    // pv_done may be up to three phases behind here, which a parity wait
    // cannot tell apart; mma_done completes once, after every MMA.
    if (ok) ok = waitw(&bars->mma_done, 0, abort_flag);
    if (ok) {
      tc_after();
      epilogue_rows_staged(lane_addr, kdeq0, p.o_part + (int64_t)blockIdx.x * R * kHeadDim, quad, R);
      if (r < R) {
        p.ml[((int64_t)blockIdx.x * R + r) * 2] = m_ref;
        p.ml[((int64_t)blockIdx.x * R + r) * 2 + 1] = l;
      }
    }
  } else if (warp < 14) {
    // =================== unpack (256 threads) ===================
    const int ut = tid - 6 * 32;
    // K: key and 64-channel column block; a warp holds 8 keys x 4 blocks.
    // The 8 lanes of a 128-bit store phase must land on 8 different
    // swizzled 16-byte positions (8 different keys of one block, or 4 keys
    // of two blocks writing opposite halves of their rows).
    // int4: a key's codes are one 128-byte row, so block kcb of every key
    // sits in the same banks; a 128-bit load is served 8 lanes at a time,
    // so the 8 lanes of each group take different blocks (kcb = j/2 + group,
    // mod 4) and start at different halves (j mod 2), which makes the loads
    // conflict-free while the stores keep 8 different keys per group.
    // 3-bit: a key's codes are 96 bytes and a block's 24, so keys four apart
    // share banks; each half-warp takes 4 keys x 4 blocks (its 64-bit loads
    // then cover all 32 banks once), and the lanes of an odd block store the
    // second half of their row first, so that each quarter-warp's (4 keys x
    // 2 blocks) 128-bit stores still land on 8 different swizzled positions.
    const int kj = kBit3 ? (ut >> 5) * 8 + (ut & 3) + 4 * ((ut >> 4) & 1) : (ut >> 5) * 8 + (ut & 7);
    const int kcb = kBit3 ? (ut >> 2) & 3 : (((ut & 7) >> 1) + ((ut >> 3) & 3)) & 3;
    const int vch = ut;  // V: channel
    // ---- fused append: the tree rows whose keys fall in this unit's range ----
    // (a1 for KV head h; thread ut = channel, warp = 32-channel group, the
    // quantizer and bit layout of append_row_k_vscale).  Consecutive rows
    // (T <= 32) touch at most two pages and, for channel ut, at most two
    // 32-token V blocks: both are looked up and loaded once, before the loop,
    // held in registers and written back after it (this thread alone writes
    // channel ut's bits of these rows in this launch; other units hold other
    // tiles).  The loop is rolled (this code runs once per launch, its
    // instructions come cold) and packs two rows per iteration so that their
    // reduction chains overlap; row values are loaded four rows ahead.
    if constexpr (kAppend) {
      const int i0 = max(0, tok0 - sd.ctx), i1 = min(T, tok1 - sd.ctx);
      if (i0 < i1) {
        uint8_t* pool = const_cast<uint8_t*>(p.pool);
        const int64_t pos0 = (int64_t)sd.ctx + i0, pos1 = (int64_t)sd.ctx + i1 - 1;
        uint8_t* hb0 = const_cast<uint8_t*>(
            head_block(sd, pool, p.page_bytes, p.pool_pages, pos0, h, ut == 0 ? p.status : nullptr));
        uint8_t* hb1 = (pos1 >> 8) == (pos0 >> 8)
                           ? hb0
                           : const_cast<uint8_t*>(head_block(sd, pool, p.page_bytes, p.pool_pages, pos1, h,
                                                             ut == 0 ? p.status : nullptr));
        const __half* krow = p.k_tree + (((int64_t)s * T + i0) * p.hkv + h) * kHeadDim + ut;
        const __half* vrow = p.v_tree + (((int64_t)s * T + i0) * p.hkv + h) * kHeadDim + ut;
        const int64_t row_stride = (int64_t)p.hkv * kHeadDim;
        float qk[4], qv[4];  // rows i .. i+3
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          qk[j] = i0 + j < i1 ? __half2float(krow[(int64_t)j * row_stride]) : 0.f;
          qv[j] = i0 + j < i1 ? __half2float(vrow[(int64_t)j * row_stride]) : 0.f;
        }
        // V blocks A (first row's) and B (last row's, if another one)
        int ia, ib;
        uint32_t* wa = hb0 ? v_block_words(hb0, (int)(pos0 & (kPageTok - 1)), ut, &ia) : nullptr;
        uint32_t* wb = hb1 ? v_block_words(hb1, (int)(pos1 & (kPageTok - 1)), ut, &ib) : nullptr;
        if (wb == wa) wb = nullptr;
        uint32_t a0 = 0u, a1 = 0u, a2 = 0u, b0 = 0u, b1 = 0u, b2 = 0u;
        if (wa) { a0 = wa[0]; a1 = wa[1]; a2 = wa[2]; }
        if (wb) { b0 = wb[0]; b1 = wb[1]; b2 = wb[2]; }
        const int64_t blk_a = pos0 >> 5;
#pragma unroll 1
        for (int i = i0; i < i1; i += 2) {
          const bool two = i + 1 < i1;  // warp-uniform
          const float xk0 = qk[0], xv0 = qv[0], xk1 = qk[1], xv1 = qv[1];
          qk[0] = qk[2]; qv[0] = qv[2]; qk[1] = qk[3]; qv[1] = qv[3];
          if (i + 4 < i1) { qk[2] = __half2float(krow[(int64_t)(i + 4 - i0) * row_stride]); qv[2] = __half2float(vrow[(int64_t)(i + 4 - i0) * row_stride]); }
          if (i + 5 < i1) { qk[3] = __half2float(krow[(int64_t)(i + 5 - i0) * row_stride]); qv[3] = __half2float(vrow[(int64_t)(i + 5 - i0) * row_stride]); }
          const int64_t pa = (int64_t)sd.ctx + i, pb = pa + 1;
          uint8_t* ha = (pa >> 8) == (pos0 >> 8) ? hb0 : hb1;
          uint8_t* hbb = (pb >> 8) == (pos0 >> 8) ? hb0 : hb1;
          int ca = 0, cb = 0;
          if (ha) ca = append_row_k_vscale(xk0, xv0, ha, (int)(pa & (kPageTok - 1)), ut);
          if (two && hbb) cb = append_row_k_vscale(xk1, xv1, hbb, (int)(pb & (kPageTok - 1)), ut);
          if (ha) {
            if ((pa >> 5) == blk_a) set_block_code(a0, a1, a2, (int)(pa & 31), ca);
            else set_block_code(b0, b1, b2, (int)(pa & 31), ca);
          }
          if (two && hbb) {
            if ((pb >> 5) == blk_a) set_block_code(a0, a1, a2, (int)(pb & 31), cb);
            else set_block_code(b0, b1, b2, (int)(pb & 31), cb);
          }
        }
        if (wa) { wa[0] = a0; wa[1] = a1; wa[2] = a2; }
        if (wb) { wb[0] = b0; wb[1] = b1; wb[2] = b2; }
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->tree_packed);
      }
    }
    // Per tile: check the three barriers at once, unpack K then V, then one
    // proxy fence and one arrival on each of kd_full, vd_full and raw_empty.
    // (A fence and arrival after K as well cost about 7 % at 262K: the
    // warp's fixed cost per tile is on the critical path.)  Holding K back
    // until V is unpacked cannot deadlock: V(i) needs P.V(i-3), which the
    // MMA warp issues after QK(i-2), whose K arrived one tile earlier.
    for (int i = 0; i < n_tiles; ++i) {
      const int st = i % F::stages, b = i & 1;
      const uint8_t* stage = ring + st * F::stage;
      const uint32_t pr_raw = probe(&bars->raw_full[st], (i / F::stages) & 1);
      const uint32_t pr_kd = probe(&bars->kd_empty[b], ((i >> 1) & 1) ^ 1);
      const int vb = i % kVBuffers;
      const uint32_t pr_vd = probe(&bars->vd_empty[vb], ((i / kVBuffers) & 1) ^ 1);
      if (!settle(&bars->raw_full[st], (i / F::stages) & 1, pr_raw, abort_flag)) break;
      const int key0 = tok0 + i * kTileTok;
      // ---- K: key kj, groups 2*kcb and 2*kcb+1 -> one 128-byte swizzled row ----
      if (!settle(&bars->kd_empty[b], ((i >> 1) & 1) ^ 1, pr_kd, abort_flag)) break;
      if (!settle(&bars->vd_empty[vb], ((i / kVBuffers) & 1) ^ 1, pr_vd, abort_flag)) break;
      if constexpr (kI4) {
        // int4: key kj's 64 channels are 8 words, stored as exact codes; the
        // key's one scale goes to the softmax (zero for keys past the range,
        // whose stale bytes could hold anything)
        const uint4* wq = reinterpret_cast<const uint4*>(stage + kj * 128 + kcb * 32);
        const int hf = kj & 1;  // the half this lane loads first (see the lane mapping)
        const uint4 x0 = wq[hf], x1 = wq[hf ^ 1];
        const uint4 a0 = hf ? x1 : x0, a1 = hf ? x0 : x1;
        if (kcb == 0) {
          const float sk = __half2float(*reinterpret_cast<const __half*>(stage + F::kc + kj * 2));
          kscale[(i % kKScaleSlots) * kTileTok + kj] = key0 + kj < tok1 ? sk : 0.f;
        }
        const uint32_t krow = su32(kdeq0) + b * kOperandBytes + kcb * 8192 + sw128_row(kj);
        __half2 out[16];
        const uint32_t w0[4] = {a0.x, a0.y, a0.z, a0.w}, w1[4] = {a1.x, a1.y, a1.z, a1.w};
        decode_i4_codes_h2(w0, out);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          st_shared_v4(sw128_chunk(krow, q4), out[4 * q4], out[4 * q4 + 1], out[4 * q4 + 2], out[4 * q4 + 3]);
        decode_i4_codes_h2(w1, out);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          st_shared_v4(sw128_chunk(krow, 4 + q4), out[4 * q4], out[4 * q4 + 1], out[4 * q4 + 2], out[4 * q4 + 3]);
      } else if constexpr (kKv2) {
        // 4-bit K: key kj's groups 2 kcb and 2 kcb + 1 are 4 words each (a
        // key's codes are one 128-byte row: the int4 lane mapping keeps the
        // loads conflict-free), times their group scales
        const uint4* wq = reinterpret_cast<const uint4*>(stage + kj * 128 + kcb * 32);
        const int hf = kj & 1;
        const uint4 x0 = wq[hf], x1 = wq[hf ^ 1];
        const uint4 a0 = hf ? x1 : x0, a1 = hf ? x0 : x1;
        const __half2 sc2 = *reinterpret_cast<const __half2*>(stage + F::kc + kj * 16 + kcb * 4);
        const __half2 s0 = __low2half2(sc2), s1 = __high2half2(sc2);
        const uint32_t krow = su32(kdeq0) + b * kOperandBytes + kcb * 8192 + sw128_row(kj);
        __half2 out[16];
        const uint32_t w0[4] = {a0.x, a0.y, a0.z, a0.w}, w1[4] = {a1.x, a1.y, a1.z, a1.w};
        decode_i4_block_h2(w0, [&](int) { return s0; }, out);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          st_shared_v4(sw128_chunk(krow, q4), out[4 * q4], out[4 * q4 + 1], out[4 * q4 + 2], out[4 * q4 + 3]);
        decode_i4_block_h2(w1, [&](int) { return s1; }, out);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          st_shared_v4(sw128_chunk(krow, 4 + q4), out[4 * q4], out[4 * q4 + 1], out[4 * q4 + 2], out[4 * q4 + 3]);
      } else {
        const uint2* wv = reinterpret_cast<const uint2*>(stage + kj * 96 + kcb * 24);
        const uint2 w01 = wv[0], w23 = wv[1], w45 = wv[2];
        const __half2 sc2 = *reinterpret_cast<const __half2*>(stage + kKTileCodeBytes + kj * 16 + kcb * 4);
        const uint32_t krow = su32(kdeq0) + b * kOperandBytes + kcb * 8192 + sw128_row(kj);
        // group 2 kcb (words 0-2, chunks 0-3) and group 2 kcb + 1 (words 3-5,
        // chunks 4-7); an odd block does the second group first
        const bool odd = kcb & 1;
        const uint32_t a0 = odd ? w23.y : w01.x, a1 = odd ? w45.x : w01.y, a2 = odd ? w45.y : w23.x;
        const uint32_t b0 = odd ? w01.x : w23.y, b1 = odd ? w01.y : w45.x, b2 = odd ? w23.x : w45.y;
        const __half2 sa = odd ? __high2half2(sc2) : __low2half2(sc2), sb = odd ? __low2half2(sc2) : __high2half2(sc2);
        const int ca = odd ? 4 : 0;
        __half2 out[16];
        decode_block_h2(a0, a1, a2, [&](int) { return sa; }, out);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          st_shared_v4(sw128_chunk(krow, ca + q4), out[4 * q4], out[4 * q4 + 1], out[4 * q4 + 2], out[4 * q4 + 3]);
        decode_block_h2(b0, b1, b2, [&](int) { return sb; }, out);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          st_shared_v4(sw128_chunk(krow, (ca ^ 4) + q4), out[4 * q4], out[4 * q4 + 1], out[4 * q4 + 2], out[4 * q4 + 3]);
      }
      // ---- V: channel vch, 64 keys -> one 128-byte swizzled row of V^T ----
      if constexpr (kI4) {
        // int4: channel vch's 64 keys are 8 words; the tile's 64 per-token
        // scales, as 32 (key 2m, 2m+1) pairs, are the same for every channel
        // channels 4..7 of each 8 start at the second half: conflict-free
        const uint4* wq = reinterpret_cast<const uint4*>(stage + F::kc + F::ks + vch * 32);
        const int hf = (vch >> 2) & 1;
        const uint4 x0 = wq[hf], x1 = wq[hf ^ 1];
        const uint4 a0 = hf ? x1 : x0, a1 = hf ? x0 : x1;
        const uint4* sp = reinterpret_cast<const uint4*>(stage + F::kc + F::ks + F::vc);
        const int live = tok1 - key0;  // keys at or beyond this are zeroed
        const uint32_t vrow = su32(vdeq0) + vb * kOperandBytes + sw128_row(vch);
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          uint32_t sc[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 x = sp[blk * 4 + q];
            sc[4 * q] = x.x;
            sc[4 * q + 1] = x.y;
            sc[4 * q + 2] = x.z;
            sc[4 * q + 3] = x.w;
          }
          __half2 out[16];
          const uint32_t w[4] = {blk ? a1.x : a0.x, blk ? a1.y : a0.y, blk ? a1.z : a0.z, blk ? a1.w : a0.w};
          decode_i4_block_h2(w, [&](int m) { return u32_as_h2(sc[m]); }, out);
          if (live < 64) {
#pragma unroll
            for (int m = 0; m < 16; ++m) {
              const int k0 = blk * 32 + 2 * m;
              if (k0 >= live) out[m] = __floats2half2_rn(0.f, 0.f);
              else if (k0 + 1 >= live) out[m] = __halves2half2(__low2half(out[m]), __float2half_rn(0.f));
            }
          }
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            st_shared_v4(sw128_chunk(vrow, blk * 4 + q4), out[4 * q4], out[4 * q4 + 1], out[4 * q4 + 2], out[4 * q4 + 3]);
        }
      } else {
        // 3-bit V: channel vch's 64 keys are 2 blocks of 3 words; 2-bit V
        // (K 4 / V 2 cache): 4 words of 16 keys
        uint32_t vw[6];
        if constexpr (kKv2) {
          const uint4 x = *reinterpret_cast<const uint4*>(stage + F::kc + F::ks + vch * 16);
          vw[0] = x.x; vw[1] = x.y; vw[2] = x.z; vw[3] = x.w; vw[4] = vw[5] = 0u;
        } else {
          const uint2* wv = reinterpret_cast<const uint2*>(stage + F::kc + F::ks + vch * 24);
          const uint2 w01 = wv[0], w23 = wv[1], w45 = wv[2];
          vw[0] = w01.x; vw[1] = w01.y; vw[2] = w23.x; vw[3] = w23.y; vw[4] = w45.x; vw[5] = w45.y;
        }
        // this channel's group: 64 key scales, as 32 (key 2m, 2m+1) pairs
        const uint4* sp =
            reinterpret_cast<const uint4*>(stage + F::kc + F::ks + F::vc + (vch >> 5) * (kTileTok * 2));
        const int live = tok1 - key0;  // keys at or beyond this are zeroed
        const uint32_t vrow = su32(vdeq0) + vb * kOperandBytes + sw128_row(vch);
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          uint32_t sc[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 x = sp[blk * 4 + q];
            sc[4 * q] = x.x;
            sc[4 * q + 1] = x.y;
            sc[4 * q + 2] = x.z;
            sc[4 * q + 3] = x.w;
          }
          __half2 out[16];
          if constexpr (kKv2)
            decode_v2_block_h2(vw[2 * blk], vw[2 * blk + 1], [&](int m) { return u32_as_h2(sc[m]); }, out);
          else
            decode_block_h2(vw[3 * blk], vw[3 * blk + 1], vw[3 * blk + 2], [&](int m) { return u32_as_h2(sc[m]); }, out);
          if (live < 64) {
#pragma unroll
            for (int m = 0; m < 16; ++m) {
              const int k0 = blk * 32 + 2 * m;
              if (k0 >= live) out[m] = __floats2half2_rn(0.f, 0.f);
              else if (k0 + 1 >= live) out[m] = __halves2half2(__low2half(out[m]), __float2half_rn(0.f));
            }
          }
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            st_shared_v4(sw128_chunk(vrow, blk * 4 + q4), out[4 * q4], out[4 * q4 + 1], out[4 * q4 + 2], out[4 * q4 + 3]);
        }
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars->kd_full[b]);
        mbar_arrive(&bars->vd_full[vb]);
        mbar_arrive(&bars->raw_empty[st]);
      }
    }
  } else {
    // =================== kFused: the tree rows' packing warp ===================
    if constexpr (kFused) fused_pack_tree_rows(p);
  }

  // ---- teardown ----
  tc_before();
  __syncthreads();
  if (warp == 1) {
    tc_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
  if constexpr (kFused) fused_merge(p, abort_flag, s, h);
  if (tid == 0 && bars->abort) report(p.status, STV_DEV_TIMEOUT);
}

template <bool kAppend, int kFmt, bool kWithhold = false, bool kFused = false>
cudaError_t launch_one(const VerifyParams& p, cudaStream_t s) {
  auto kernel = verify_tc_kernel<kAppend, kFmt, kWithhold, kFused>;
  constexpr int smem = Fmt<kFmt>::smem;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if constexpr (kFused) return launch_pdl_coop(kernel, p.n_units, kThreads + 32, smem, s, p);
  else return launch_pdl(kernel, p.n_units, kThreads, smem, s, p);
}

}  // namespace

cudaError_t launch_verify(const VerifyParams& p, cudaStream_t s) {
  // the int8 path on the 3-bit cache forms per-group integer dots: its own kernel
  if (p.path == STV_PATH_INT8 && p.fmt == kFmtBit3) return launch_verify_i8(p, s);
  // a balanced plan for several sequences: the persistent kernel (exact path, 3-bit cache)
  if (p.persist_ctas > 0) return launch_verify_persistent(p, s);
  // the packing warp: one launch per layer (append, verify, merge), or the
  // fused append alone (exact path, 3-bit cache)
  if (p.o_out || p.pack_warp) return launch_one<false, kFmtBit3, false, true>(p, s);
  if (p.test_withhold_copies)
    return p.fmt == kFmtInt4 ? launch_one<false, kFmtInt4, true>(p, s) : launch_one<false, kFmtBit3, true>(p, s);
  // the fused append packs the 3-bit cache only (the host refuses it for the others)
  const bool append = p.k_tree != nullptr && p.v_tree != nullptr;
  if (p.fmt == kFmtInt4) return launch_one<false, kFmtInt4>(p, s);
  if (p.fmt == kFmtK4V2) return launch_one<false, kFmtK4V2>(p, s);
  if (append) return launch_one<true, kFmtBit3>(p, s);
  return launch_one<false, kFmtBit3>(p, s);
}

}  // namespace stv
