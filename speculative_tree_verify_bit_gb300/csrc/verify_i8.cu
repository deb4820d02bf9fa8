// verify_i8.cu -- a2..a4, the int8 path on the 3-bit cache, on the
// 5th-generation tensor cores: split-KV, tree-masked GQA verify attention
// that forms the pages' per-group integer dots on the tensor cores.
//
// Sources: "elpis" README, "Why fast" (decode verify int8 Q.K^T with the
// 3-bit K codes used as exact int8 values, integer MMA; 8-row token tree
// verified in one pass); Reddit posts (u/iamMess), second post (split-KV
// verify kernel).  The pages' kernel uses the RTX 3090's integer MMA; sm_103a
// has no integer tcgen05 MMA, so the integers ride on the fp16 one: qi
// (|qi| <= 127) and code - 4 (-4..3) are exact in fp16, each product and
// each 32-channel sum (|I_g| <= 32 * 127 * 4 = 16,256) is an integer below
// 2^24, so the fp32 accumulator holds I_g exactly.
//
// Definition: per (node, Q head) row qi = rne(127 q / max|q|), sQ =
// max|q| / 127 (quantize_q_kernel); per key j and 32-channel group g,
// I_g = sum_{c in g} qi_c (code_c - 4); S_j = sQ sum_g sK_{j,g} I_g / 16 in
// fp32.  The exact path and the int4 cache run in verify_tc.cu.
//
// One CTA per work unit (sequence, KV head, range of 64-key tiles), one CTA
// per SM, 16 warps:
//   warp 0      producer: one bulk copy per array per tile into a ring of raw
//               stages.
//   warp 3      TMEM owner and MMA issuer (a lightly loaded sub-partition:
//               its softmax warp holds only padding rows when T * G <= 96).
//   warps 4-7   softmax: thread = query row = TMEM lane of the dots.
//   warps 8-15  unpack: K codes -> exact fp16 codes in shared memory (their
//               group scales, as fp32, to the softmax); V codes -> fp16 V^T
//               straight into tensor memory.
//   warps 1-2   idle.
// Per 64-key tile:
//   I_g[128 rows x 64 keys] = Q_g (shared) . C_g^T (shared), two groups per
//                             round (four per tile), each round's dots in
//                             one of two TMEM blocks of 128 columns (one
//                             block when T * G > 96)
//   O^T[256 ch x NP rows]  += V^T (TMEM, two 128-channel halves) . P^T (shared)
// The second is P.V with the operands swapped (M = the 256 channels, N = the
// NP = ceil16(T*G) real rows), which keeps the accumulator small enough to
// leave room for the per-group dots.  qi (fp16, the A operand of the dots)
// sits in shared memory, so that tensor memory (512 columns) holds two dot
// blocks of two groups each from column 0, one V^T buffer of 64 columns,
// and the O^T halves of NO = ceil32(T*G) columns at the end: every round
// is a hand-off between the MMA warp and the softmax warps, and two groups
// per round halve their number.
// Softmax is online in fp32 with a stale-maximum threshold: P uses a
// reference maximum that is raised (rescaling O and l) only when a score
// exceeds it by more than 2^8, so P <= 256 in fp16 and O rescales are rare.
// Every wait is bounded; a timeout sets a CTA abort flag, every role stops,
// in-flight copies and MMAs are waited for (bounded) and TMEM is freed.
#include "stv_device.cuh"
#include "tc_util.cuh"

namespace stv {
namespace {

constexpr int kThreads = 512;
constexpr int kQBytes = 65536;        // qi as the A operand: 128 rows x 256 channels, fp16
constexpr int kKBuffers = 2;          // decoded K tiles in shared memory
constexpr int kOperandBytes = 32768;  // one fp16 K tile: 64 keys x 256 channels
constexpr int kPBytes = 16384;        // one fp16 P tile: up to 128 rows x 64 keys
constexpr int kCtlBytes = 2048;       // barriers, masks, rescale factors
constexpr int kStages = 3;            // raw ring
constexpr int kStageBytes = kKTileCodeBytes + kKTileScaleBytes + kVTileCodeBytes + kVTileScaleBytes;  // 14336
// Per-(key, group) K scales handed from the unpack warps to the softmax
// warps, as fp32, in rotating slots (one barrier per slot).  Unpacking tile
// j waits for QK(j - 2) to finish, whose rounds reuse dot blocks that the
// softmax warps released while reading tile j - 3's: they are done with
// tile j - 4, so slot j mod 4 is never rewritten while it is read.
constexpr int kSlots = 4;
constexpr int kSlotFloats = kGroups * kTileTok;
constexpr int kSmemBytes = 1024 /*align slack*/ + kQBytes + kKBuffers * kOperandBytes + 2 * kPBytes +
                           kStages * kStageBytes + kCtlBytes + kSlots * kSlotFloats * 4;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
constexpr float kRescaleThreshold = 8.f;  // log2 units
constexpr uint32_t kColS = 0, kTmemCols = 512;

// D (TMEM) = A (shared-memory descriptor) x B (shared-memory descriptor) (+ D
// when acc != 0), issued by one elected lane.
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, e;\n setp.ne.u32 p, %4, 0;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}

struct Ctl {
  uint64_t raw_full[kStages], raw_empty[kStages];
  uint64_t kd_full[kKBuffers], kd_empty[kKBuffers];
  uint64_t vd_full, vd_empty;
  uint64_t ks_full[kSlots];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full[2], p_empty[2];
  uint64_t q_ready, mma_done;
  uint64_t tree_packed;  // the round's tree rows of this unit are in the cache (fused append)
  uint32_t tmem_base;
  int abort;
  uint32_t anc[kMaxT];
  float corr[2][kMaxRows];  // O rescale factor per row, by tile parity (a slow
                            // warp may still read tile i's while others write i + 1's)
};
static_assert(sizeof(Ctl) <= kCtlBytes, "control block");

// Waits suspend (try_wait with a time hint).  Polling waits measured 13 %
// slower at 262K: with a dozen warps polling, the rounds' MMA-to-softmax
// hand-offs (one per group) took longer to complete.
__device__ __forceinline__ bool wait1(uint64_t* b, uint32_t parity, volatile int* abort_flag) {
  return stv::wait1<false>(b, parity, abort_flag);
}
__device__ __forceinline__ bool waitw(uint64_t* b, uint32_t parity, volatile int* abort_flag) {
  return stv::waitw<false>(b, parity, abort_flag);
}
__device__ __forceinline__ bool settle(uint64_t* b, uint32_t parity, uint32_t probed, volatile int* abort_flag) {
  return stv::settle<false>(b, parity, probed, abort_flag);
}

// Named barrier 1 over the four softmax warps, counting the threads whose
// predicate is set.
__device__ __forceinline__ uint32_t softmax_bar_popc(bool pred) {
  uint32_t cnt;
  asm volatile(
      "{\n .reg .pred q;\n setp.ne.u32 q, %1, 0;\n barrier.cta.red.popc.u32 %0, 1, 128, q;\n}\n"
      : "=r"(cnt)
      : "r"((uint32_t)pred)
      : "memory");
  return cnt;
}

// kAppend: the round's tree rows are packed into the cache by this launch
// (stv_append_verify_attn).  kWithhold (failure-path test only,
// stv_verify_attn_timeout_test): the producer issues no copy, so every wait
// on one runs out.
template <bool kAppend, bool kWithhold = false>
__global__ void __launch_bounds__(kThreads, 1) verify_i8_kernel(const __grid_constant__ VerifyParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment of the operand tiles (the swizzle works on address bits).
  const uint32_t base_u32 = su32(smem_raw);
  uint8_t* smem = smem_raw + ((1024 - (base_u32 & 1023)) & 1023);
  uint8_t* const qbuf0 = smem;                              // qi, the A operand of the dot MMAs
  uint8_t* const kbuf0 = smem + kQBytes;                    // K tiles: kbuf0 + b * kOperandBytes
  uint8_t* const pbuf0 = kbuf0 + kKBuffers * kOperandBytes;  // P tiles: pbuf0 + b * kPBytes
  uint8_t* const ring = pbuf0 + 2 * kPBytes;
  Ctl* ctl = reinterpret_cast<Ctl*>(ring + kStages * kStageBytes);
  float* const kscale = reinterpret_cast<float*>(ring + kStages * kStageBytes + kCtlBytes);
  volatile int* abort_flag = &ctl->abort;

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

  // ---- tensor-memory plan (R <= 128 rows) ----
  const int NP = (R + 15) & ~15;  // N of the P.V product
  const int NO = (R + 31) & ~31;  // columns of one O^T half
  // Two groups per QK round (four rounds per tile), their dots in one of nsb
  // TMEM blocks of 128 columns: two (the MMA of round k + 1 overlaps the
  // softmax warps' loads of round k) when the O^T halves leave room.
  const int nsb = NO <= 96 ? 2 : 1;
  const uint32_t s_end = kColS + 128 * nsb;  // the V^T buffer: [s_end, s_end + 64)
  const uint32_t colO = kTmemCols - 2 * NO;

  // ---- set-up ----
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&ctl->raw_full[i], 1);
      mbar_init(&ctl->raw_empty[i], 8);
    }
    for (int i = 0; i < kKBuffers; ++i) {
      mbar_init(&ctl->kd_full[i], 8);
      mbar_init(&ctl->kd_empty[i], 1);
    }
    mbar_init(&ctl->vd_full, 8);
    mbar_init(&ctl->vd_empty, 1);
    for (int i = 0; i < kSlots; ++i) mbar_init(&ctl->ks_full[i], 8);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl->p_full[i], 4);
      mbar_init(&ctl->p_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl->s_full[i], 1);
      mbar_init(&ctl->s_free[i], 4);
    }
    mbar_init(&ctl->q_ready, 4);
    mbar_init(&ctl->mma_done, 1);
    mbar_init(&ctl->tree_packed, 8);
    ctl->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // Nothing above touches global memory: the previous kernel may still be running.
  grid_dep_wait();
  if (tid < T) {  // a2: ancestor-or-self masks
    uint32_t m = 1u << tid;
    int n = tid;
    const int32_t* par = p.parent + (int64_t)s * T;
    for (int st = 0; st < T && n > 0; ++st) {
      int pa = __ldg(par + n);
      if (pa < 0 || pa >= n) {
        if (split == 0 && h == 0) report(p.status, STV_DEV_BAD_TREE);
        break;
      }
      m |= 1u << pa;
      n = pa;
    }
    if (tid == 0 && __ldg(par) != -1 && split == 0 && h == 0) report(p.status, STV_DEV_BAD_TREE);
    ctl->anc[tid] = m;
  }
  if (warp == 3) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&ctl->tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_before();
  __syncthreads();
  tc_after();
  grid_dep_launch();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == 0) {
    // =================== producer ===================
    if (lane == 0) {
      int issued = 0;
      bool tree_ready = !kAppend;
      for (int i = 0; i < (kWithhold ? 0 : n_tiles); ++i) {
        const int st = i % kStages;
        if (!wait1(&ctl->raw_empty[st], ((i / kStages) & 1) ^ 1, abort_flag)) break;
        const int key0 = tok0 + i * kTileTok;
        // a tile holding tree keys is copied only after the unpack warps have
        // packed them (their global writes are fenced for the async proxy)
        if (!tree_ready && key0 + kTileTok > sd.ctx && key0 < sd.ctx + T) {
          if (!wait1(&ctl->tree_packed, 0, abort_flag)) break;
          tree_ready = true;
        }
        const int64_t lp = key0 >> 8;
        int32_t page = lp < sd.n_pages ? __ldg(sd.page_table + lp) : -1;
        if (page < 0 || page >= p.pool_pages) {
          report(p.status, STV_DEV_BAD_PAGE);
          page = 0;  // read a valid page; the result is flagged as garbage
        }
        const uint8_t* hb = p.pool + (int64_t)page * p.page_bytes + (int64_t)h * kHeadBytes;
        const int t = (key0 & (kPageTok - 1)) / kTileTok;
        uint8_t* dst = ring + st * kStageBytes;
        uint64_t* bar = &ctl->raw_full[st];
        mbar_expect_tx(bar, kStageBytes);
        bulk_g2s(dst, hb + kOffKCodes + t * kKTileCodeBytes, kKTileCodeBytes, bar);
        bulk_g2s(dst + kKTileCodeBytes, hb + kOffKScales + t * kKTileScaleBytes, kKTileScaleBytes, bar);
        bulk_g2s(dst + kKTileCodeBytes + kKTileScaleBytes, hb + kOffVCodes + t * kVTileCodeBytes, kVTileCodeBytes, bar);
        bulk_g2s(dst + kKTileCodeBytes + kKTileScaleBytes + kVTileCodeBytes, hb + kOffVScales + t * kVTileScaleBytes, kVTileScaleBytes, bar);
        issued = i + 1;
      }
      // No copy may still be landing when the CTA exits.
      for (int i = max(0, issued - kStages); i < issued; ++i) {
        volatile int never = 0;
        wait1(&ctl->raw_full[i % kStages], (i / kStages) & 1, &never);
      }
    }
  } else if (warp == 3) {
    // =================== MMA issuer (whole warp, one elected lane issues) ===================
    // Issue order: QK(0) (all rounds), then QK(i), PV(i-1) for i = 1, 2, ...,
    // then PV(last).  A QK round reuses a TMEM block once the softmax warps
    // have loaded the dots it held.
    // Descriptors are built once; each MMA then only adds a constant to the
    // start-address field (no carry: shared addresses are < 256 KiB).
    const uint32_t tm = tmem;
    bool ok = waitw(&ctl->q_ready, 0, abort_flag);
    tc_after();
    const uint64_t qdesc0 = desc_sw128(su32(qbuf0)), kdesc0 = desc_sw128(su32(kbuf0)),
                   pdesc0 = desc_sw128(su32(pbuf0));
    const uint32_t idesc_qk = idesc_f16_f32(128, 64), idesc_pv = idesc_f16_f32(128, NP);
    uint32_t rnd = 0;  // QK rounds issued so far
    auto issue_qk = [&](int i) -> bool {
      const int kb = i % kKBuffers;
      if (!settle(&ctl->kd_full[kb], (i / kKBuffers) & 1, probe(&ctl->kd_full[kb], (i / kKBuffers) & 1),
                  abort_flag))
        return false;
      const uint64_t kd = kdesc0 + (uint64_t)(kb * (kOperandBytes >> 4));
      for (int rr = 0; rr < kGroups / 2; ++rr) {
        const int b = rnd % nsb;
        const uint32_t u = rnd / nsb;  // this block's use count
        if (u > 0 && !settle(&ctl->s_free[b], (u - 1) & 1, probe(&ctl->s_free[b], (u - 1) & 1), abort_flag))
          return false;
        tc_after();
        // groups 2 rr and 2 rr + 1, each into its 64 columns of the block;
        // group g's 32 channels are K16 steps 2g and 2g + 1 (qi: 16 KiB per
        // 64-channel block, the K tile: 8 KiB)
#pragma unroll
        for (int gg = 0; gg < 2; ++gg) {
#pragma unroll
          for (int t2 = 0; t2 < 2; ++t2) {
            const int kk = 2 * (2 * rr + gg) + t2;
            mma_ss(tm + kColS + 128 * b + 64 * gg, qdesc0 + (uint64_t)((kk >> 2) * 1024 + (kk & 3) * 2),
                   kd + (uint64_t)((kk >> 2) * 512 + (kk & 3) * 2), idesc_qk, t2 > 0);
          }
        }
        if (rr == kGroups / 2 - 1) tc_commit(&ctl->kd_empty[kb]);
        tc_commit(&ctl->s_full[b]);
        ++rnd;
      }
      return true;
    };
    auto issue_pv = [&](int j) -> bool {
      const int pb = j & 1;
      const uint32_t pr_p = probe(&ctl->p_full[pb], (j >> 1) & 1);
      const uint32_t pr_v = probe(&ctl->vd_full, j & 1);
      if (!settle(&ctl->p_full[pb], (j >> 1) & 1, pr_p, abort_flag)) return false;
      if (!settle(&ctl->vd_full, j & 1, pr_v, abort_flag)) return false;
      tc_after();
      const uint64_t pd = pdesc0 + (uint64_t)(pb * (kPBytes >> 4));
      const uint32_t vt = tm + s_end;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_tmemA(tm + colO + hh * NO, vt + 32 * hh + 8 * kk, pd + (uint64_t)(2 * kk), idesc_pv, (j > 0 || kk > 0));
      tc_commit(&ctl->vd_empty);
      tc_commit(&ctl->p_empty[pb]);
      return true;
    };
    for (int i = 0; ok && i < n_tiles; ++i) {
      ok = issue_qk(i);
      if (ok && i > 0) ok = issue_pv(i - 1);
    }
    if (ok && n_tiles > 0) ok = issue_pv(n_tiles - 1);
    // Every MMA issued here has finished before TMEM is freed.
    tc_commit(&ctl->mma_done);
    volatile int never = 0;
    waitw(&ctl->mma_done, 0, &never);
  } else if (warp < 4) {
    // warps 1 and 2: idle
  } else if (warp < 8) {
    // =================== softmax (thread = row of S = lane of O^T) ===================
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
    const bool live = r < R;
    float c = kLog2e / 16.f;  // S c = sQ sum_g sK_g I_g / 16 in log2 units
    int node = 0;
    // qi row (exact integers in fp16) -> row r of the A operand in shared
    // memory: four 64-channel blocks of 128 rows x 128 bytes, 128-byte swizzle
    {
      int64_t qrow = 0;
      if (live) {
        node = r / G;
        qrow = ((int64_t)s * T + node) * p.hq + h * G + r % G;
        c *= p.sq[qrow];
      }
#pragma unroll
      for (int chunk = 0; chunk < 4; ++chunk) {
        uint32_t v[32];
        if (!live) {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0u;
        } else {
          const int8_t* src = p.qi + qrow * kHeadDim + chunk * 64;
#pragma unroll
          for (int e = 0; e < 32; ++e)
            v[e] = h2u(__halves2half2(__int2half_rn(src[2 * e]), __int2half_rn(src[2 * e + 1])));
        }
        const uint32_t qrow_s = su32(qbuf0) + chunk * (kQBytes / 4) + sw128_row(r);
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8)
          st_shared_v4(sw128_chunk(qrow_s, c8), v[4 * c8], v[4 * c8 + 1], v[4 * c8 + 2], v[4 * c8 + 3]);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->q_ready);
    }
    const uint32_t anc = ctl->anc[node];
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    uint32_t rnd = 0;  // QK rounds consumed so far
    const int64_t nkeys = (int64_t)sd.ctx + T;  // the dump's keys per row
    for (int i = 0; i < n_tiles; ++i) {
      bool fail = !ok;
      uint32_t sv[64];  // S of this row: keys 0..63 (fp32 bits)
      const int key0 = tok0 + i * kTileTok;
      const int pb = i & 1;
      // P tile pb was last read by P.V(i - 2), which the tensor pipe runs
      // before QK(i): complete by the time S(i) is.  Waiting here, before
      // the tile's registers fill up, keeps the wait loop cheap.
      if (!fail) fail = !waitw(&ctl->p_empty[pb], ((i >> 1) & 1) ^ 1, abort_flag);
      // The K group scales of tile i are handed over before K(i) is released
      // to the MMA warp, so before its dots exist.
      if (!fail) fail = !waitw(&ctl->ks_full[i % kSlots], (i / kSlots) & 1, abort_flag);
      {
        // int8 path: S = sum_g sK_g I_g over the rounds' per-group dots
#pragma unroll
        for (int e = 0; e < 64; ++e) sv[e] = 0u;  // fp32 zero
        const float* ksl = kscale + (i % kSlots) * kSlotFloats;
        // a round holds groups 2 rr and 2 rr + 1: four 32-key parts, taken
        // in group order (S sums the groups in order 0..7)
        for (int rr = 0; rr < kGroups / 2 && !fail; ++rr) {
          const int sb = rnd % nsb;
          if (!waitw(&ctl->s_full[sb], (rnd / nsb) & 1, abort_flag)) {
            fail = true;
            break;
          }
          tc_after();
#pragma unroll
          for (int part = 0; part < 4; ++part) {
            const int g = 2 * rr + (part >> 1), half = part & 1;
            uint32_t t[32];
            tmem_ld32(lane_addr + kColS + 128 * sb + 32 * part, t);
            tmem_wait_ld(t);
            if (part == 3) {  // the round's last load: release the block
              tc_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&ctl->s_free[sb]);
            }
            if (p.dots != nullptr && live) {  // inspection: this kernel's own integer dots
              int32_t* drow = p.dots + (((int64_t)h * R + r) * nkeys + key0 + 32 * half) * kGroups + g;
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (key0 + 32 * half + e < tok1) drow[(int64_t)e * kGroups] = __float2int_rn(__uint_as_float(t[e]));
            }
            const float4* sc4 = reinterpret_cast<const float4*>(ksl + g * kTileTok + 32 * half);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float4 x = sc4[e];
              sv[32 * half + 4 * e] = __float_as_uint(fmaf(x.x, __uint_as_float(t[4 * e]), __uint_as_float(sv[32 * half + 4 * e])));
              sv[32 * half + 4 * e + 1] = __float_as_uint(fmaf(x.y, __uint_as_float(t[4 * e + 1]), __uint_as_float(sv[32 * half + 4 * e + 1])));
              sv[32 * half + 4 * e + 2] = __float_as_uint(fmaf(x.z, __uint_as_float(t[4 * e + 2]), __uint_as_float(sv[32 * half + 4 * e + 2])));
              sv[32 * half + 4 * e + 3] = __float_as_uint(fmaf(x.w, __uint_as_float(t[4 * e + 3]), __uint_as_float(sv[32 * half + 4 * e + 3])));
            }
          }
          ++rnd;
        }
      }
      // ---- mask, tile maximum, rescale decision ----
      float corr = 1.f;
      if (!fail && live) {
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
            sv[e] = ((va >> e) & 1u) ? sv[e] : 0xff800000u;
            sv[32 + e] = ((vb >> e) & 1u) ? sv[32 + e] : 0xff800000u;
          }
        }
        // Row maximum: 3-input max, 8 independent chains.
        float mx8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx8[k] = fmaxf(__uint_as_float(sv[k]), __uint_as_float(sv[32 + k]));
#pragma unroll
        for (int e = 8; e < 32; e += 2) {
          mx8[(e >> 1) & 7] = max3(mx8[(e >> 1) & 7], __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]));
          mx8[((e >> 1) + 4) & 7] =
              max3(mx8[((e >> 1) + 4) & 7], __uint_as_float(sv[32 + e]), __uint_as_float(sv[32 + e + 1]));
        }
        const float mx = fmaxf(max3(mx8[0], mx8[1], mx8[2]), max3(max3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
        const float m_tile = mx * c;
        if (m_tile > m_ref + kRescaleThreshold) {
          if (m_ref != -INFINITY) corr = ex2(m_ref - m_tile);
          m_ref = m_tile;
          l *= corr;
        }
      }
      ctl->corr[i & 1][r] = corr;
      // One meeting of the four softmax warps per tile: whether any of them
      // failed a wait (then all leave together) and whether any row needs
      // its O rescaled (then all four rescale their TMEM lanes).
      const bool fail_w = __any_sync(0xffffffffu, fail), need_w = __any_sync(0xffffffffu, corr != 1.f);
      const uint32_t votes = softmax_bar_popc((lane < 5 && fail_w) || (lane == 31 && need_w));
      if (votes >= 5) {
        ok = false;
        break;
      }
      const bool rescale = votes > 0;
      // ---- P = 2^(S c - m_ref) in fp16, packed key pairs ----
      uint32_t pk[32];
      if (live) {
        const float mref = m_ref == -INFINITY ? 0.f : m_ref;
        float sum8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float p0 = ex2(fmaf(__uint_as_float(sv[2 * e]), c, -mref));
          const float p1 = ex2(fmaf(__uint_as_float(sv[2 * e + 1]), c, -mref));
          sum8[e & 7] += p0 + p1;
          pk[e] = h2u(__floats2half2_rn(p0, p1));
        }
        l += ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
      }
      if (!fail && live) {
        const uint32_t prow = su32(pbuf0) + pb * kPBytes + sw128_row(r);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4)
          st_shared_v4(sw128_chunk(prow, c4), pk[4 * c4], pk[4 * c4 + 1], pk[4 * c4 + 2], pk[4 * c4 + 3]);
      }
      fence_async_smem();
      // O^T may be rescaled only once P.V(i - 1) has finished, and before
      // P.V(i) (which waits for this warp's p_full arrival).  Lane = channel:
      // each thread scales column n of its two O^T rows by corr[n].
      if (rescale && i >= 1 && !fail) {
        if (!waitw(&ctl->p_empty[(i - 1) & 1], ((i - 1) >> 1) & 1, abort_flag)) {
          fail = true;
        } else {
          tc_after();
#pragma unroll 1
          for (int hh = 0; hh < 2; ++hh) {
#pragma unroll 1
            for (int n0 = 0; n0 < NO; n0 += 16) {
              uint32_t o[16];
              tmem_ld16(lane_addr + colO + hh * NO + n0, o);
              tmem_wait_ld<16>(o);
              const float4* cr = reinterpret_cast<const float4*>(ctl->corr[i & 1] + n0);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float4 x = cr[e];
                o[4 * e] = __float_as_uint(__uint_as_float(o[4 * e]) * x.x);
                o[4 * e + 1] = __float_as_uint(__uint_as_float(o[4 * e + 1]) * x.y);
                o[4 * e + 2] = __float_as_uint(__uint_as_float(o[4 * e + 2]) * x.z);
                o[4 * e + 3] = __float_as_uint(__uint_as_float(o[4 * e + 3]) * x.w);
              }
              tmem_st16(lane_addr + colO + hh * NO + n0, o);
            }
          }
          tmem_wait_st();
        }
      }
      tc_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->p_full[pb]);
      if (fail) ok = false;  // the next meeting tells the others
    }
    // ---- epilogue: O (from O^T, lane = channel), m, l into the workspace ----
    // pv completion barriers may be several phases behind here, which a
    // parity wait cannot tell apart; mma_done completes once, after every MMA.
    ok = __all_sync(0xffffffffu, ok);
    if (ok) ok = waitw(&ctl->mma_done, 0, abort_flag);
    if (ok) {
      tc_after();
      float* dst = p.o_part + (int64_t)blockIdx.x * R * kHeadDim;
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        const int ch = hh * 128 + r;
#pragma unroll 1
        for (int n0 = 0; n0 < NO; n0 += 32) {
          uint32_t o[32];
          tmem_ld32(lane_addr + colO + hh * NO + n0, o);
          tmem_wait_ld(o);
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (n0 + e < R) dst[(int64_t)(n0 + e) * kHeadDim + ch] = __uint_as_float(o[e]);
        }
      }
      if (live) {
        p.ml[((int64_t)blockIdx.x * R + r) * 2] = m_ref;
        p.ml[((int64_t)blockIdx.x * R + r) * 2 + 1] = l;
      }
    }
  } else {
    // =================== unpack (256 threads) ===================
    const int ut = tid - 8 * 32;
    // K: key and 64-channel column block.  Each group of 8 consecutive lanes
    // takes 8 different keys of one column block, so the 8 lanes of a
    // 128-bit store phase land on 8 different swizzled 16-byte positions.
    const int kj = (ut >> 5) * 8 + (ut & 7);
    const int kcb = (ut >> 3) & 3;
    // V: warp w may only reach TMEM lanes 32 (w mod 4) .. + 31, so channel
    // vch = 128 vh + 32 (w mod 4) + lane lands in V^T half vh at that lane.
    const int vq = warp & 3, vh = (warp - 8) >> 2;
    const int vch = vh * 128 + vq * 32 + lane;
    const uint32_t vt_lane = tmem + ((uint32_t)(vq * 32) << 16) + s_end + 32 * vh;
    // ---- fused append: the tree rows whose keys fall in this unit's range ----
    // (a1 for KV head h; thread ut = channel, warp = 32-channel group, the
    // quantizer and bit layout of append_row_k_vscale).  Consecutive rows
    // (T <= 32) touch at most two pages and, for channel ut, at most two
    // 32-token V blocks: both are looked up and loaded once, before the loop,
    // held in registers and written back after it (this thread alone writes
    // channel ut's bits of these rows in this launch; other units hold other
    // tiles).
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
        if (lane == 0) mbar_arrive(&ctl->tree_packed);
      }
    }
    // K of tile i: raw stage -> the exact codes (code - 4, exact in fp16) in K
    // tile i % kKBuffers (shared memory), once QK(i - kKBuffers) has read that
    // buffer; the key's two group scales go to the softmax as fp32 (zero past
    // the key range, whose stale bytes could hold anything).
    auto unpack_k = [&](int i) -> bool {
      const int st = i % kStages, kb = i % kKBuffers;
      const uint32_t pr_raw = probe(&ctl->raw_full[st], (i / kStages) & 1);
      const uint32_t pr_kd = probe(&ctl->kd_empty[kb], ((i / kKBuffers) & 1) ^ 1);
      if (!settle(&ctl->raw_full[st], (i / kStages) & 1, pr_raw, abort_flag)) return false;
      if (!settle(&ctl->kd_empty[kb], ((i / kKBuffers) & 1) ^ 1, pr_kd, abort_flag)) return false;
      const uint8_t* stage = ring + st * kStageBytes;
      const int key0 = tok0 + i * kTileTok;
      const uint32_t krow = su32(kbuf0) + kb * kOperandBytes + kcb * 8192 + sw128_row(kj);
      // key kj, groups 2 kcb and 2 kcb + 1 -> one 128-byte swizzled row
      const uint2* wv = reinterpret_cast<const uint2*>(stage + kj * 96 + kcb * 24);
      const uint2 w01 = wv[0], w23 = wv[1], w45 = wv[2];
      const __half2 sc2 = *reinterpret_cast<const __half2*>(stage + kKTileCodeBytes + kj * 16 + kcb * 4);
      const bool in = key0 + kj < tok1;
      float* ksl = kscale + (i % kSlots) * kSlotFloats;
      ksl[(2 * kcb) * kTileTok + kj] = in ? __low2float(sc2) : 0.f;
      ksl[(2 * kcb + 1) * kTileTok + kj] = in ? __high2float(sc2) : 0.f;
      __half2 out[16];
      decode_block_raw(w01.x, w01.y, w23.x, out);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
        st_shared_v4(sw128_chunk(krow, q4), out[4 * q4], out[4 * q4 + 1], out[4 * q4 + 2], out[4 * q4 + 3]);
      decode_block_raw(w23.y, w45.x, w45.y, out);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
        st_shared_v4(sw128_chunk(krow, 4 + q4), out[4 * q4], out[4 * q4 + 1], out[4 * q4 + 2], out[4 * q4 + 3]);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&ctl->kd_full[kb]);
        mbar_arrive(&ctl->ks_full[i % kSlots]);
      }
      return true;
    };
    // V of tile i (its raw stage already waited for by unpack_k(i)): channel
    // vch's 64 keys -> 32 fp16 pairs s * (code - 4) in its TMEM lane of V^T,
    // once P.V(i - 1) has read the buffer.  Then the raw stage is free.
    auto unpack_v = [&](int i) -> bool {
      const int st = i % kStages;
      if (!settle(&ctl->vd_empty, (i & 1) ^ 1, probe(&ctl->vd_empty, (i & 1) ^ 1), abort_flag)) return false;
      tc_after();
      const uint8_t* stage = ring + st * kStageBytes;
      const int live = tok1 - (tok0 + i * kTileTok);  // keys at or beyond this are zeroed
      uint32_t vr[32];
      const uint2* wv = reinterpret_cast<const uint2*>(stage + kKTileCodeBytes + kKTileScaleBytes + vch * 24);
      const uint2 w01 = wv[0], w23 = wv[1], w45 = wv[2];
      // this channel's group: 64 key scales, as 32 (key 2m, 2m+1) pairs
      const uint4* sp = reinterpret_cast<const uint4*>(stage + kKTileCodeBytes + kKTileScaleBytes + kVTileCodeBytes +
                                                       (vch >> 5) * (kTileTok * 2));
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
        if (blk == 0)
          decode_block_h2(w01.x, w01.y, w23.x, [&](int m) { return u32_as_h2(sc[m]); }, out);
        else
          decode_block_h2(w23.y, w45.x, w45.y, [&](int m) { return u32_as_h2(sc[m]); }, out);
        zero_dead_keys(out, blk, live);
#pragma unroll
        for (int m = 0; m < 16; ++m) vr[16 * blk + m] = h2u(out[m]);
      }
      tmem_st32(vt_lane, vr);
      tmem_wait_st();
      tc_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&ctl->vd_full);
        mbar_arrive(&ctl->raw_empty[st]);
      }
      return true;
    };
    // K runs one tile ahead of V: K(i + 1) is ready well before QK(i + 1),
    // while V(i) can only start once P.V(i - 1) has released the buffer.
    bool ok = n_tiles > 0 ? unpack_k(0) : true;
    for (int i = 0; ok && i < n_tiles; ++i) {
      if (i + 1 < n_tiles) ok = unpack_k(i + 1);
      if (ok) ok = unpack_v(i);
    }
  }

  // ---- teardown ----
  tc_before();
  __syncthreads();
  if (warp == 3) {
    tc_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
  if (tid == 0 && ctl->abort) report(p.status, STV_DEV_TIMEOUT);
}

template <bool kAppend, bool kWithhold = false>
cudaError_t launch_one(const VerifyParams& p, cudaStream_t s) {
  auto kernel = verify_i8_kernel<kAppend, kWithhold>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(kernel, p.n_units, kThreads, kSmemBytes, s, p);
}

}  // namespace

cudaError_t launch_verify_i8(const VerifyParams& p, cudaStream_t s) {
  const bool append = p.k_tree != nullptr && p.v_tree != nullptr;
  if (p.test_withhold_copies) return launch_one<false, true>(p, s);
  return append ? launch_one<true>(p, s) : launch_one<false>(p, s);
}

}  // namespace stv
