// prefill_tc.cu -- f2, prefill attention over the 3-bit cache (exact path):
// a persistent kernel over (chunk, KV head) units, on the 5th-generation
// tensor cores.  The same kernel, in its verify mode, runs a4 for a batch of
// several sequences (see "Verify mode" below).
//
// Sources: "elpis" README, "Why fast" (prefill over the quantized KV cache:
// int8 Q.K^T 3021c, a double-buffered K/V ring 3022).  The prompt's own K/V
// rows are in the cache already (stv_kv_append_pack); prompt token j attends
// to the ctx0 tokens before the prompt and to prompt tokens 0..j.
//
// Work.  The prompt is cut into chunks of C tokens (C * G <= 128 query rows);
// a unit is (chunk, KV head): the C * G rows that share the KV head, against
// every key up to the chunk's end.  No unit is split, so each row ends with
// O / l, written in fp16 straight into the output: no partials and no merge
// launch, and the whole prompt is one launch.  Units are taken longest first
// and dealt to the CTAs (one per SM) in snake order -- left to right, then
// right to left -- so the CTAs' tile counts differ by about one unit's.
//
// Per CTA: the roles and per-tile pipeline of the verify kernel (warp 0
// producer, warp 1 TMEM owner and MMA issuer, warps 2-5 softmax with thread
// = query row, warps 6-13 unpack of the 3-bit codes into fp16 operand tiles;
// S = Q.K^T and O += P.V as tcgen05 MMAs with Q, S/P and O in TMEM).  The
// pipeline runs on across units: ring stages, operand buffers and barrier
// phases count the CTA's tiles, not a unit's.  At a unit's end the softmax
// warps write the next unit's Q into TMEM (every Q.K^T of the unit is done:
// its last S was consumed), wait for the unit's last P.V (o_ready), write
// O / l, and release O (o_free) before the next unit's first P.V, which
// starts the accumulator afresh.
// Every wait is bounded; a timeout sets a CTA abort flag, every role stops,
// in-flight copies and MMAs are waited for (bounded) and TMEM is freed.
//
// Verify mode (a2..a4, exact path, a batch of several sequences; Reddit
// posts (u/iamMess), second post: split-KV verify).  A unit is one work
// unit of the verify split plan, (sequence, KV head, range of 64-key tiles),
// and writes its partial O, m, l for split_combine as the verify kernel does.
// The plan may hold more units than SMs: the host orders them longest first
// (VerifyParams::order) and the CTAs take them in snake order, so a batch of
// unequal sequences keeps every SM busy to the end (with one unit per CTA,
// the longest sequence's units would set the launch's time).  The mask is
// the sequence's tree mask; the pipeline carries on across units as above.
#include "stv_device.cuh"
#include "tc_util.cuh"

namespace stv {
namespace {

constexpr int kThreads = 448;
constexpr int kStages = 4;
constexpr int kStageBytes = kKTileCodeBytes + kKTileScaleBytes + kVTileCodeBytes + kVTileScaleBytes;  // 14336
constexpr int kOperandBytes = 32768;  // one K or V^T fp16 tile
constexpr int kVBuffers = 3;
constexpr int kSmemBytes = 1024 /*align slack*/ + (2 + kVBuffers) * kOperandBytes + kStages * kStageBytes + 1024;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
constexpr float kRescaleThreshold = 8.f;  // log2 units
constexpr uint32_t kColQ = 0, kColS0 = 128, kColO = 256, kTmemCols = 512;
constexpr uint32_t kIdescQK = idesc_f16_f32(128, 64);
constexpr uint32_t kIdescPV = idesc_f16_f32(128, 256);

struct Bars {
  uint64_t raw_full[kStages], raw_empty[kStages];
  uint64_t kd_full[2], kd_empty[2], vd_full[kVBuffers], vd_empty[kVBuffers];
  uint64_t s_full[2], p_full[2];
  uint64_t pv_done, q_ready, o_ready, o_free, mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 1024, "barrier block");

__device__ __forceinline__ bool wait1(uint64_t* b, uint32_t parity, volatile int* abort_flag) {
  return stv::wait1<false>(b, parity, abort_flag);
}
__device__ __forceinline__ bool waitw(uint64_t* b, uint32_t parity, volatile int* abort_flag) {
  return stv::waitw<false>(b, parity, abort_flag);
}
__device__ __forceinline__ bool settle(uint64_t* b, uint32_t parity, uint32_t probed, volatile int* abort_flag) {
  return stv::settle<false>(b, parity, probed, abort_flag);
}

// The k-th unit of CTA b: units are numbered longest first and dealt in
// snake order.
__device__ __forceinline__ int unit_of(int k, int b) {
  const int n = (int)gridDim.x;
  return k * n + ((k & 1) ? n - 1 - b : b);
}

// Prefill: unit u is (chunk, KV head), chunks longest (last) first.
struct Unit {
  int c, h;      // chunk, KV head
  int t, R;      // tokens of the chunk, query rows (t * G)
  int ctx;       // keys before the chunk
  int tok1;      // keys of the unit: [0, tok1)
  int n_tiles;
};

__device__ __forceinline__ Unit unit_info(const PrefillParams& p, int u) {
  Unit x;
  x.c = p.n_chunks - 1 - u / p.hkv;
  x.h = u % p.hkv;
  x.t = min(p.chunk, p.n_tokens - x.c * p.chunk);
  x.R = x.t * p.G;
  x.ctx = p.ctx0 + x.c * p.chunk;
  x.tok1 = x.ctx + x.t;
  x.n_tiles = (x.tok1 + kTileTok - 1) / kTileTok;
  return x;
}

// Verify: the w-th longest unit of the split plan (units are numbered
// sequence-major, then KV head, then split).
struct VerifyUnit {
  int h;                       // KV head
  int slot;                    // the work unit whose partials this writes
  int s;                       // sequence
  int node0;                   // Q row of the sequence's first node: [node][hq][256]
  int R;                       // query rows (T * G)
  int ctx;                     // keys before the tree
  int tok0, tok1;              // keys of the unit: [tok0, tok1)
  int n_tiles;
  const int32_t* page_table;   // the sequence's pages
  int n_pages;
};

__device__ __forceinline__ VerifyUnit unit_info(const VerifyParams& p, int w) {
  VerifyUnit x;
  const int u = p.order[w];
  int s = 0;
  while (s + 1 < p.n_seqs && u >= p.seq[s + 1].unit_base) ++s;
  const SeqDesc& sd = p.seq[s];
  const int local = u - sd.unit_base;
  x.h = local / sd.splits;
  x.slot = u;
  x.s = s;
  x.node0 = s * p.T;
  x.R = p.R;
  x.ctx = sd.ctx;
  x.tok0 = (local % sd.splits) * p.tiles_per_split * kTileTok;
  x.tok1 = min(sd.ctx + p.T, x.tok0 + p.tiles_per_split * kTileTok);
  x.n_tiles = (x.tok1 - x.tok0 + kTileTok - 1) / kTileTok;
  x.page_table = sd.page_table;
  x.n_pages = sd.n_pages;
  return x;
}

template <bool kVerify>
struct ParamsOf {
  using type = PrefillParams;
  using unit = Unit;
};
template <>
struct ParamsOf<true> {
  using type = VerifyParams;
  using unit = VerifyUnit;
};

// kWithhold (failure-path test only, stv_prefill_attn_timeout_test): the
// producer issues no copy, so every wait on one runs out.
// kVerify: verify mode (VerifyParams; exact path, 3-bit cache).
template <bool kWithhold, bool kVerify>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ typename ParamsOf<kVerify>::type p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment of the operand tiles (the swizzle works on address bits).
  const uint32_t base_u32 = su32(smem_raw);
  uint8_t* smem = smem_raw + ((1024 - (base_u32 & 1023)) & 1023);
  uint8_t* const kdeq0 = smem;                      // K tiles: kdeq0 + b * kOperandBytes
  uint8_t* const vdeq0 = smem + 2 * kOperandBytes;  // V^T tiles: vdeq0 + b * kOperandBytes
  uint8_t* const ring = smem + (2 + kVBuffers) * kOperandBytes;
  Bars* bars = reinterpret_cast<Bars*>(ring + kStages * kStageBytes);
  volatile int* abort_flag = &bars->abort;
  const int tid = threadIdx.x, lane = tid & 31;
  // The warp index, read from lane 0: the compiler then knows it is the same
  // across the warp, so the role branches below are warp-uniform (derived
  // from threadIdx.x alone they were compiled as possibly divergent: about
  // 7 % slower, and every role's loop changed with any code added to another).
  const int warp = __shfl_sync(0xffffffffu, tid >> 5, 0);
  const int cta = blockIdx.x;

  // ---- set-up ----
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bars->raw_full[i], 1);
      mbar_init(&bars->raw_empty[i], 8);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->kd_full[i], 8);
      mbar_init(&bars->kd_empty[i], 1);
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 4);
    }
    for (int i = 0; i < kVBuffers; ++i) {
      mbar_init(&bars->vd_full[i], 8);
      mbar_init(&bars->vd_empty[i], 1);
    }
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->q_ready, 4);
    mbar_init(&bars->o_ready, 1);
    mbar_init(&bars->o_free, 4);
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
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
  // Nothing above touches global memory: the previous kernel may still be running.
  grid_dep_wait();
  grid_dep_launch();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // =================== producer ===================
    if (lane == 0) {
      int g = 0;  // tiles issued by this CTA
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int u = unit_of(k, cta);
        if (u >= p.n_units) break;
        const auto x = unit_info(p, u);
        for (int i = 0; i < (kWithhold ? 0 : x.n_tiles); ++i) {
          const int st = g % kStages;
          if (!wait1(&bars->raw_empty[st], ((g / kStages) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          int key0, lp;
          int32_t page;
          if constexpr (kVerify) {
            key0 = x.tok0 + i * kTileTok;
            lp = key0 >> 8;
            page = lp < x.n_pages ? __ldg(x.page_table + lp) : -1;
          } else {
            key0 = i * kTileTok;
            lp = key0 >> 8;
            page = lp < p.n_pages ? __ldg(p.page_table + lp) : -1;
          }
          if (page < 0 || page >= p.pool_pages) {
            report(p.status, STV_DEV_BAD_PAGE);
            page = 0;  // read a valid page; the result is flagged as garbage
          }
          const uint8_t* hb = p.pool + (int64_t)page * p.page_bytes + (int64_t)x.h * kHeadBytes;
          const int t = (key0 & (kPageTok - 1)) / kTileTok;
          uint8_t* dst = ring + st * kStageBytes;
          uint64_t* bar = &bars->raw_full[st];
          mbar_expect_tx(bar, kStageBytes);
          bulk_g2s(dst, hb + kOffKCodes + t * kKTileCodeBytes, kKTileCodeBytes, bar);
          bulk_g2s(dst + kKTileCodeBytes, hb + kOffKScales + t * kKTileScaleBytes, kKTileScaleBytes, bar);
          bulk_g2s(dst + kKTileCodeBytes + kKTileScaleBytes, hb + kOffVCodes + t * kVTileCodeBytes, kVTileCodeBytes,
                   bar);
          bulk_g2s(dst + kKTileCodeBytes + kKTileScaleBytes + kVTileCodeBytes, hb + kOffVScales + t * kVTileScaleBytes,
                   kVTileScaleBytes, bar);
          ++g;
        }
      }
      // No copy may still be landing when the CTA exits.
      for (int j = max(0, g - kStages); j < g; ++j) {
        volatile int never = 0;
        wait1(&bars->raw_full[j % kStages], (j / kStages) & 1, &never);
      }
    }
  } else if (warp == 1) {
    // =================== MMA issuer (whole warp, one elected lane issues) ===================
    // Per unit: QK(0), QK(1), then PV(j), QK(j+2) for j = 0, 1, ...; tiles
    // are counted over the CTA (g), so S, K and V^T buffers and their
    // barrier phases carry on from one unit to the next.
    const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
    const uint64_t kdesc0 = desc_sw128(su32(kdeq0)), vdesc0 = desc_sw128(su32(vdeq0));
    auto issue_qk = [&](int g) -> bool {
      const int b = g & 1;
      if (!settle(&bars->kd_full[b], (g >> 1) & 1, probe(&bars->kd_full[b], (g >> 1) & 1), abort_flag)) return false;
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
    bool ok = true;
    int g0 = 0;  // tiles of this CTA's earlier units
    for (int k = 0; ok; ++k) {
      const int u = unit_of(k, cta);
      if (u >= p.n_units) break;
      const auto x = unit_info(p, u);
      if (!(ok = waitw(&bars->q_ready, k & 1, abort_flag))) break;
      tc_after();
      for (int i = 0; ok && i < 2 && i < x.n_tiles; ++i) ok = issue_qk(g0 + i);
      for (int j = 0; ok && j < x.n_tiles; ++j) {
        const int g = g0 + j, b = g & 1, vb = g % kVBuffers;
        const uint32_t pr_p = probe(&bars->p_full[b], (g >> 1) & 1);
        const uint32_t pr_v = probe(&bars->vd_full[vb], (g / kVBuffers) & 1);
        if (!(ok = settle(&bars->p_full[b], (g >> 1) & 1, pr_p, abort_flag))) break;
        if (!(ok = settle(&bars->vd_full[vb], (g / kVBuffers) & 1, pr_v, abort_flag))) break;
        // the unit's first P.V restarts O: the previous unit's O has been read
        if (j == 0 && k > 0 && !(ok = waitw(&bars->o_free, (k - 1) & 1, abort_flag))) break;
        tc_after();
        const uint64_t vd = vdesc0 + (uint64_t)(vb * (kOperandBytes >> 4));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_tmemA(tm + kColO, tm + kColS0 + 64 * b + 8 * kk, vd + (uint64_t)(kk * 2), kIdescPV, (j > 0 || kk > 0));
        tc_commit(&bars->vd_empty[vb]);
        tc_commit(&bars->pv_done);
        if (j + 2 < x.n_tiles) ok = issue_qk(g + 2);
      }
      if (ok) tc_commit(&bars->o_ready);
      g0 += x.n_tiles;
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
    const float c = kLog2e / 16.f;
    // Q rows of a unit -> TMEM columns [0, 128): row r = node * G + (Q head
    // within the KV head); rows past t * G are zero.
    using U = typename ParamsOf<kVerify>::unit;
    auto load_q = [&](const U& x) {
      const bool live = r < x.R;
      const int node = live ? r / p.G : 0;
      int64_t qrow = 0;
      if constexpr (kVerify) qrow = live ? ((int64_t)(x.node0 + node) * p.hq + x.h * p.G + r % p.G) : 0;
      else qrow = live ? ((int64_t)(x.c * p.chunk + node) * p.hq + x.h * p.G + r % p.G) : 0;
#pragma unroll
      for (int chunk = 0; chunk < 4; ++chunk) {
        uint32_t v[32];
        if (!live) {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0u;
        } else {
          const uint4* src = reinterpret_cast<const uint4*>(p.q + qrow * kHeadDim + chunk * 64);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            uint4 x4 = __ldg(src + e);
            v[4 * e] = x4.x;
            v[4 * e + 1] = x4.y;
            v[4 * e + 2] = x4.z;
            v[4 * e + 3] = x4.w;
          }
        }
        tmem_st32(lane_addr + kColQ + 32 * chunk, v);
      }
      tmem_wait_st();
      tc_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->q_ready);
    };
    bool ok = true;
    int g0 = 0;
    int u = unit_of(0, cta);
    U x = {};
    if (u < p.n_units) {
      x = unit_info(p, u);
      load_q(x);
    }
    for (int k = 0; ok && u < p.n_units; ++k) {
      const bool live = r < x.R;
      const int node = live ? r / p.G : 0;
      uint32_t anc;
      if constexpr (kVerify) {
        // a2: this row's ancestor-or-self mask, from the sequence's parent[]
        anc = 1u << node;
        const int32_t* par = p.parent + (int64_t)x.s * p.T;
        for (int n = node, st = 0; st < p.T && n > 0; ++st) {
          const int pa = __ldg(par + n);
          if (pa < 0 || pa >= n) {
            report(p.status, STV_DEV_BAD_TREE);
            break;
          }
          anc |= 1u << pa;
          n = pa;
        }
        if (r == 0 && __ldg(par) != -1) report(p.status, STV_DEV_BAD_TREE);
      } else {
        // chain tree: node i sees prompt tokens 0..i of its chunk
        anc = node >= 31 ? 0xffffffffu : ((2u << node) - 1u);
      }
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < x.n_tiles; ++j) {
        const int g = g0 + j, b = g & 1;
        if (!(ok = waitw(&bars->s_full[b], (g >> 1) & 1, abort_flag))) break;
        tc_after();
        uint32_t sa[32], sb[32];
        tmem_ld32(lane_addr + kColS0 + 64 * b, sa);
        tmem_ld32(lane_addr + kColS0 + 64 * b + 32, sb);
        tmem_wait_ld(sa);
        tmem_wait_ld(sb);
        int key0;
        bool edge;
        if constexpr (kVerify) {
          key0 = x.tok0 + j * kTileTok;
          edge = key0 + kTileTok > x.ctx || key0 + kTileTok > x.tok1;
        } else {
          key0 = j * kTileTok;
          edge = key0 + kTileTok > x.ctx;
        }
        if (edge) {
          // Visibility of the tile's 64 keys as one bit mask: keys before the
          // chunk, this row's own and earlier chunk tokens, nothing at or past
          // the chunk's end.  Masked keys become -inf by selection.
          const int rel_ctx = x.ctx - key0, rel_end = x.tok1 - key0;
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
        for (int e = 0; e < 8; ++e) mx8[e] = fmaxf(__uint_as_float(sa[e]), __uint_as_float(sb[e]));
#pragma unroll
        for (int e = 8; e < 32; e += 2) {
          mx8[(e >> 1) & 7] = max3(mx8[(e >> 1) & 7], __uint_as_float(sa[e]), __uint_as_float(sa[e + 1]));
          mx8[((e >> 1) + 4) & 7] =
              max3(mx8[((e >> 1) + 4) & 7], __uint_as_float(sb[e]), __uint_as_float(sb[e + 1]));
        }
        const float mx = fmaxf(max3(mx8[0], mx8[1], mx8[2]), max3(max3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
        const float m_tile = mx * c;
        float corr = 1.f;
        if (m_tile > m_ref + kRescaleThreshold) {
          if (m_ref != -INFINITY) corr = ex2(m_ref - m_tile);
          m_ref = m_tile;
          l *= corr;
        }
        // P = 2^(S c - m_ref) in fp16, packed key pairs, into the S columns
        // (paired fp32 FMA and add for the exponent arguments and the sum).
        const float mref = m_ref == -INFINITY ? 0.f : m_ref;
        const float2 c2 = make_float2(c, c), nm2 = make_float2(-mref, -mref);
        float2 sum4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float2 xa =
              __ffma2_rn(make_float2(__uint_as_float(sa[2 * e]), __uint_as_float(sa[2 * e + 1])), c2, nm2);
          const float2 xb =
              __ffma2_rn(make_float2(__uint_as_float(sb[2 * e]), __uint_as_float(sb[2 * e + 1])), c2, nm2);
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
        // O may be rescaled only once P.V of the previous tile has finished:
        // P.V(g-2) is done (QK(g) followed it) and P.V(g) waits for this warp,
        // so pv_done is in phase g-1 or g and the parity wait is unambiguous.
        // On a unit's first tile O holds nothing to rescale (and corr is 1).
        if (j >= 1 && __any_sync(0xffffffffu, corr != 1.f)) {
          if (!(ok = waitw(&bars->pv_done, (g - 1) & 1, abort_flag))) break;
          tc_after();
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
        tmem_wait_st();
        tc_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[b]);
      }
      if (!ok) break;
      // The next unit's Q: every Q.K^T of this unit has completed.
      const int un = unit_of(k + 1, cta);
      U xn = {};
      if (un < p.n_units) {
        xn = unit_info(p, un);
        load_q(xn);
      }
      if (!(ok = waitw(&bars->o_ready, k & 1, abort_flag))) break;
      tc_after();
      if constexpr (kVerify) {
        // ---- epilogue: O, m, l of this row into the unit's partials ----
        float* dst = p.o_part + ((int64_t)x.slot * x.R + r) * kHeadDim;
#pragma unroll 1
        for (int chunk = 0; chunk < 8; ++chunk) {
          uint32_t o[32];
          tmem_ld32(lane_addr + kColO + 32 * chunk, o);
          tmem_wait_ld(o);
          if (live) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              reinterpret_cast<float4*>(dst + 32 * chunk)[e] =
                  make_float4(__uint_as_float(o[4 * e]), __uint_as_float(o[4 * e + 1]),
                              __uint_as_float(o[4 * e + 2]), __uint_as_float(o[4 * e + 3]));
          }
        }
        if (live) {
          p.ml[((int64_t)x.slot * x.R + r) * 2] = m_ref;
          p.ml[((int64_t)x.slot * x.R + r) * 2 + 1] = l;
        }
      } else {
        // ---- epilogue: O / l of this row, fp16, into the output ----
        __half* dst = p.o + ((int64_t)(x.c * p.chunk + node) * p.hq + x.h * p.G + r % p.G) * kHeadDim;
#pragma unroll 1
        for (int chunk = 0; chunk < 8; ++chunk) {
          uint32_t o[32];
          tmem_ld32(lane_addr + kColO + 32 * chunk, o);
          tmem_wait_ld(o);
          if (live) {  // l >= 1 for a live row: its own key is visible and P(max) >= 2^-8
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              uint4 w;
              w.x = h2u(__floats2half2_rn(__uint_as_float(o[8 * e]) / l, __uint_as_float(o[8 * e + 1]) / l));
              w.y = h2u(__floats2half2_rn(__uint_as_float(o[8 * e + 2]) / l, __uint_as_float(o[8 * e + 3]) / l));
              w.z = h2u(__floats2half2_rn(__uint_as_float(o[8 * e + 4]) / l, __uint_as_float(o[8 * e + 5]) / l));
              w.w = h2u(__floats2half2_rn(__uint_as_float(o[8 * e + 6]) / l, __uint_as_float(o[8 * e + 7]) / l));
              reinterpret_cast<uint4*>(dst + 32 * chunk)[e] = w;
            }
          }
        }
      }
      tc_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->o_free);
      g0 += x.n_tiles;
      u = un;
      x = xn;
    }
  } else {
    // =================== unpack (256 threads) ===================
    const int ut = tid - 6 * 32;
    // K: key and 64-channel column block.  Each group of 8 consecutive lanes
    // takes 8 different keys of one column block, so the 8 lanes of a
    // 128-bit store phase land on 8 different swizzled 16-byte positions.
    const int kj = (ut >> 5) * 8 + (ut & 7);
    const int kcb = (ut >> 3) & 3;
    const int vch = ut;  // V: channel
    int g = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int u = unit_of(k, cta);
      if (u >= p.n_units) break;
      const auto x = unit_info(p, u);
      for (int i = 0; i < x.n_tiles; ++i) {
        const int st = g % kStages, b = g & 1, vb = g % kVBuffers;
        const uint8_t* stage = ring + st * kStageBytes;
        const uint32_t pr_raw = probe(&bars->raw_full[st], (g / kStages) & 1);
        const uint32_t pr_kd = probe(&bars->kd_empty[b], ((g >> 1) & 1) ^ 1);
        const uint32_t pr_vd = probe(&bars->vd_empty[vb], ((g / kVBuffers) & 1) ^ 1);
        if (!settle(&bars->raw_full[st], (g / kStages) & 1, pr_raw, abort_flag) ||
            !settle(&bars->kd_empty[b], ((g >> 1) & 1) ^ 1, pr_kd, abort_flag) ||
            !settle(&bars->vd_empty[vb], ((g / kVBuffers) & 1) ^ 1, pr_vd, abort_flag)) {
          ok = false;
          break;
        }
        // ---- K: key kj, groups 2*kcb and 2*kcb+1 -> one 128-byte swizzled row ----
        {
          const uint2* wv = reinterpret_cast<const uint2*>(stage + kj * 96 + kcb * 24);
          const uint2 w01 = wv[0], w23 = wv[1], w45 = wv[2];
          const __half2 sc2 = *reinterpret_cast<const __half2*>(stage + kKTileCodeBytes + kj * 16 + kcb * 4);
          const uint32_t krow = su32(kdeq0) + b * kOperandBytes + kcb * 8192 + sw128_row(kj);
          const __half2 s0 = __low2half2(sc2), s1 = __high2half2(sc2);
          __half2 out[16];
          decode_block_h2(w01.x, w01.y, w23.x, [&](int) { return s0; }, out);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            st_shared_v4(sw128_chunk(krow, q4), out[4 * q4], out[4 * q4 + 1], out[4 * q4 + 2], out[4 * q4 + 3]);
          decode_block_h2(w23.y, w45.x, w45.y, [&](int) { return s1; }, out);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            st_shared_v4(sw128_chunk(krow, 4 + q4), out[4 * q4], out[4 * q4 + 1], out[4 * q4 + 2], out[4 * q4 + 3]);
        }
        // ---- V: channel vch, 64 keys -> one 128-byte swizzled row of V^T ----
        {
          const uint2* wv = reinterpret_cast<const uint2*>(stage + kKTileCodeBytes + kKTileScaleBytes + vch * 24);
          const uint2 w01 = wv[0], w23 = wv[1], w45 = wv[2];
          const uint32_t vw[6] = {w01.x, w01.y, w23.x, w23.y, w45.x, w45.y};
          // this channel's group: 64 key scales, as 32 (key 2m, 2m+1) pairs
          const uint4* sp = reinterpret_cast<const uint4*>(stage + kKTileCodeBytes + kKTileScaleBytes +
                                                           kVTileCodeBytes + (vch >> 5) * (kTileTok * 2));
          int live;  // keys at or beyond this are zeroed
          if constexpr (kVerify) live = x.tok1 - (x.tok0 + i * kTileTok);
          else live = x.tok1 - i * kTileTok;
          const uint32_t vrow = su32(vdeq0) + vb * kOperandBytes + sw128_row(vch);
#pragma unroll
          for (int blk = 0; blk < 2; ++blk) {
            uint32_t sc[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint4 s4 = sp[blk * 4 + q];
              sc[4 * q] = s4.x;
              sc[4 * q + 1] = s4.y;
              sc[4 * q + 2] = s4.z;
              sc[4 * q + 3] = s4.w;
            }
            __half2 out[16];
            decode_block_h2(vw[3 * blk], vw[3 * blk + 1], vw[3 * blk + 2], [&](int m) { return u32_as_h2(sc[m]); },
                            out);
            zero_dead_keys(out, blk, live);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              st_shared_v4(sw128_chunk(vrow, blk * 4 + q4), out[4 * q4], out[4 * q4 + 1], out[4 * q4 + 2],
                           out[4 * q4 + 3]);
          }
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bars->kd_full[b]);
          mbar_arrive(&bars->vd_full[vb]);
          mbar_arrive(&bars->raw_empty[st]);
        }
        ++g;
      }
    }
  }

  // ---- teardown ----
  tc_before();
  __syncthreads();
  if (warp == 1) {
    tc_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
  if (tid == 0 && bars->abort) report(p.status, STV_DEV_TIMEOUT);
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, int grid, cudaStream_t s, bool withhold_copies) {
  auto kernel = withhold_copies ? prefill_tc_kernel<true, false> : prefill_tc_kernel<false, false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(kernel, grid, kThreads, kSmemBytes, s, p);
}

cudaError_t launch_verify_persistent(const VerifyParams& p, cudaStream_t s) {
  auto kernel = prefill_tc_kernel<false, true>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(kernel, p.persist_ctas, kThreads, kSmemBytes, s, p);
}

}  // namespace stv
