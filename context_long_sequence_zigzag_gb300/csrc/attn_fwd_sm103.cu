// attn_fwd_sm103.cu — fused context-parallel causal attention forward on the
// sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// One CTA computes one 128-row query tile of one head against every key run
// of its plan entry: the KV shards in ring order r, r-1, ..., r-C+1 (mod C),
// fully masked tiles already removed on the host ("超长上下文训练速度翻倍秘籍"
// §2 pitfall 1: the diagonal block is causal, earlier shards unmasked;
// "LLM context parallel production guide", 因果 Attention 会制造 Rank 负载不均:
// blocks above the diagonal are skipped).  The per-block (out, lse) merge of
// "Ulysses与Ring-Attention详解" §4.1-§4.2 happens on chip: a reference row
// maximum and the running row sum rescale the TMEM output accumulator, so
// the result equals merging every block's partial exactly.
//
// S = Q K^T is an SS MMA (Q, loaded once, and the streamed K both K-major in
// shared memory) into one of three TMEM S buffers; P (bf16) overwrites the
// first half of its S buffer, so O += P V is a TS MMA with V read from shared
// memory as an MN-major operand.  TMEM columns: S0, S1, S2 (128 each), O (DV)
// = 512.  S(j+3) reuses buffer j % 3 once PV(j) has completed.  With three
// buffers the S of the next two key tiles is already computed while the
// softmax works on this one, so the softmax never waits for the PV -> S round
// trip of the step before.
//
// Two warps issue the MMAs, one the S products and one the PV products.
// The tensor pipe queues only about two and a half MMAs, so every cycle an
// issuing warp spends on its commits, barrier waits and loop overhead idles
// the pipe unless another warp is issuing meanwhile.
//
// Roles (224 threads):
//   warps 0-3  softmax: thread t owns query row t = TMEM lane t.  Per key
//              tile it loads S, masks, takes the row maximum, exponentiates,
//              writes P back to TMEM, rescales O when the reference maximum
//              moves by more than 2^8, and finally normalises O and writes
//              o / lse.
//   warp 4     TMA producers: lane 0 loads Q, then streams K; lane 1 streams
//              V, each into its own ring.  A gathered key tile (a plan
//              run of kind kRangePacked) arrives as one box per piece.
//   warp 5     TMEM allocator; issues S(j) = Q K(j)^T.
//   warp 6     issues O += P(j) V(j).
#include <cuda.h>
#include <cuda_bf16.h>

#include "internal.h"
#include "plan_check.cuh"
#include "sm103_ptx.cuh"

namespace cpattn {

namespace {

constexpr int BM = 128;  // query rows per CTA
constexpr int BN = 128;  // key rows per step
constexpr uint32_t kSubTile = 128 * 128;  // one 128-row x 64-column bf16 swizzle panel: 16 KiB
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: a new maximum moves the reference past this
constexpr float kLagSum = 1.0995116e12f;    // 2^40: a tile's row sum above this sends it down the full path
constexpr uint64_t kWaitLimitNs = 2000000000ull;

enum WaitSite : int {
  kSiteQ = 1, kSiteKEmpty, kSiteVEmpty, kSiteKFull, kSitePFull, kSiteVFull, kSiteSFull, kSiteOFull,
  kSiteDrain, kSiteAlign,
};

template <int DQK, int DV>
struct FwdCfg {
  static constexpr int kQPanels = DQK / 64;
  static constexpr int kVPanels = DV / 64;
  static constexpr int NSK = DQK <= 128 ? 3 : 2;
  static constexpr int NSV = DQK <= 128 ? 3 : 2;
  static constexpr int NS_S = 3;  // TMEM S buffers
  static constexpr uint32_t kQBytes = kQPanels * kSubTile;
  static constexpr uint32_t kKBytes = kQPanels * kSubTile;
  static constexpr uint32_t kVBytes = kVPanels * kSubTile;
  static constexpr uint32_t offQ = 0;
  static constexpr uint32_t offK = offQ + kQBytes;
  static constexpr uint32_t offV = offK + NSK * kKBytes;
  static constexpr uint32_t offBar = offV + NSV * kVBytes;
  static constexpr int kNumBars = 1 + 2 * NSK + 2 * NSV + 3 * NS_S + 2;
  // the tile's runs and the key masks of its gathered tiles, staged for the
  // softmax warps when the tile has at most kSlots runs
  static constexpr int kSlots = 64;
  static constexpr uint32_t offRanges = (offBar + kNumBars * 8 + 16 + 15) / 16 * 16;
  static constexpr uint32_t offMasks = offRanges + kSlots * 16;
  static constexpr uint32_t kSmem = offMasks + kSlots * 16;
  // TMEM columns
  static constexpr uint32_t tS0 = 0;
  static constexpr uint32_t tO = NS_S * BN;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(tO + DV <= kTmemCols, "TMEM budget");
  static_assert(kSmem <= 232448, "shared memory budget");
};

// Boxes of 8, 16, ..., 120 rows of K and V for the pieces of gathered key
// tiles (kRangePacked runs): a piece of r rows (a multiple of 8) is one box
// per panel (map r / 8 - 1; the 128-row maps for r = 128).  One box per piece
// matters: loading a piece as several boxes of 64, 32, 16 and 8 rows made the
// forward on a 128K-token pack of short sequences 9 % slower.
constexpr int kPieceMaps = 15;

struct FwdParams {
  CUtensorMap tq, tk, tv;
  CUtensorMap tkp[kPieceMaps], tvp[kPieceMaps];  // box rows 8 (i + 1)
  AttnArgs a;
  int32_t* err;
};

// Iterates the key tiles of a plan entry (its runs cut into BN-row steps).
struct KvCursor {
  const RangeDesc* r;
  int count, ri, off;
  RangeDesc cur;
  __device__ void init(const RangeDesc* ranges, int begin, int cnt) {
    r = ranges + begin;
    count = cnt;
    ri = 0;
    off = 0;
    if (count > 0) cur = r[0];
  }
  // Current tile: first row, rows, position of the first row; a gathered
  // tile (packed()) has its pieces from entry row0 and its key mask at pos0.
  __device__ bool packed() const { return (cur.flags & kRangePacked) != 0; }
  __device__ int row() const { return cur.row0 + off; }
  __device__ int n() const { return min(BN, cur.nrows - off); }
  __device__ int pos() const { return cur.pos0 + off; }
  __device__ void next() {
    off += BN;
    if (off >= cur.nrows) {
      off = 0;
      if (++ri < count) cur = r[ri];
    }
  }
};

// Grid order of the query-major kernels: key/value heads outermost, then
// the tiles (heaviest first), then the query heads of the group, so that the
// CTAs resident at one time read the K and V of one key/value head, which
// then stay in L2 (the heads of one tile inside each other instead made the
// resident CTAs stream every head at once: S=256K with 64 heads of 192,
// forward 1.61 s against 0.86 s in this order).
__device__ __forceinline__ void grid_tile_slot(const AttnArgs& a, int& tile_idx, int& slot) {
  const int G = a.hq / a.hkv;
  const unsigned per_kv = unsigned(a.num_tiles) * unsigned(G);
  const int kv = int(blockIdx.x / per_kv);
  const unsigned rem = blockIdx.x - unsigned(kv) * per_kv;
  tile_idx = int(rem / unsigned(G));
  slot = kv * G + int(rem - unsigned(tile_idx) * unsigned(G));
}

__device__ __forceinline__ int head_of_slot(int slot, const AttnArgs& a) {
  const int G = a.hq / a.hkv;
  const int kv = slot / G, g = slot - kv * G;
  return a.gqa_interleaved ? g * a.hkv + kv : kv * G + g;
}

// PACKED: the plan has gathered key tiles (kRangePacked runs).  Plans without
// them run an instantiation without that code: the extra branches slowed the
// S = 64K forward by 2-3 % where they never ran.
template <int DQK, int DV, bool PACKED>
__global__ void __launch_bounds__(224, 1) attn_fwd_tc_kernel(const __grid_constant__ FwdParams p) {
  using Cfg = FwdCfg<DQK, DV>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = ptx::smem_u32(smem);
  const AttnArgs& a = p.a;
  if (sbase & 1023u) {  // the swizzled operand panels need 1024-byte alignment
    if (threadIdx.x == 0 && p.err) atomicCAS(p.err, 0, 0x100 | kSiteAlign);
    return;
  }

  int tile_idx, slot;
  grid_tile_slot(a, tile_idx, slot);
  const int h = head_of_slot(slot, a);
  const int kvh = a.gqa_interleaved ? h % a.hkv : h / (a.hq / a.hkv);
  if (a.debug && !debug_plan_ok(a, tile_idx, h, kvh, false, p.err)) return;
  const TileDesc tile = a.tiles[tile_idx];
  const int n_kv = tile.work;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t bar0 = sbase + Cfg::offBar;
  const uint32_t bar_q = bar0;  // Q tile landed in shared memory
  auto bar_k_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto bar_k_empty = [&](int s) { return bar0 + 8u * (1 + Cfg::NSK + s); };
  auto bar_v_full = [&](int s) { return bar0 + 8u * (1 + 2 * Cfg::NSK + s); };
  auto bar_v_empty = [&](int s) { return bar0 + 8u * (1 + 2 * Cfg::NSK + Cfg::NSV + s); };
  const uint32_t barx = bar0 + 8u * (1 + 2 * Cfg::NSK + 2 * Cfg::NSV);
  // One (S computed, P written, PV done) triple per S buffer b = j % 3: the
  // softmax may run up to two key tiles ahead of the MMA issuer, and a
  // per-buffer barrier is then never more than one phase ahead of a waiter,
  // which is what a parity wait needs.
  auto bar_s_full = [&](int b) { return barx + 8u * b; };
  auto bar_p_full = [&](int b) { return barx + 8u * (Cfg::NS_S + b); };      // 4 softmax warps
  auto bar_o_done = [&](int b) { return barx + 8u * (2 * Cfg::NS_S + b); };  // PV(j) done
  auto bar_drain = [&](int w) { return barx + 8u * (3 * Cfg::NS_S + w); };    // per issuing warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::offBar + Cfg::kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::offBar + Cfg::kNumBars * 8 + 4);

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar_q, 1);
    for (int s = 0; s < Cfg::NSK; ++s) {
      ptx::mbar_init(bar_k_full(s), 1);
      ptx::mbar_init(bar_k_empty(s), 1);
    }
    for (int s = 0; s < Cfg::NSV; ++s) {
      ptx::mbar_init(bar_v_full(s), 1);
      ptx::mbar_init(bar_v_empty(s), 1);
    }
    for (int b = 0; b < Cfg::NS_S; ++b) {
      ptx::mbar_init(bar_s_full(b), 1);
      ptx::mbar_init(bar_p_full(b), 4);
      ptx::mbar_init(bar_o_done(b), 1);
    }
    ptx::mbar_init(bar_drain(0), 1);
    ptx::mbar_init(bar_drain(1), 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 5) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), Cfg::kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    ptx::prefetch_tmap(&p.tq);
    ptx::prefetch_tmap(&p.tk);
    ptx::prefetch_tmap(&p.tv);
  }
  if (PACKED && warp == 4 && lane >= 2)  // the piece maps, one per lane
    ptx::prefetch_tmap(lane < 2 + kPieceMaps ? &p.tkp[lane - 2] : &p.tvp[lane - 2 - kPieceMaps]);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const ptx::WaitCtx wctx{abort_flag, p.err, kWaitLimitNs};

  if (warp == 4) {
    // ------------------------------------------------------------ producers
    // Lane 0 loads Q, then streams K; lane 1 streams V: on GB300 one
    // thread's tiled TMA loads top out near 40 B/cycle, two issuing threads
    // reach about 60.
    if (lane == 0 && n_kv > 0) {
      ptx::mbar_arrive_expect_tx(bar_q, Cfg::kQBytes);
      for (int c = 0; c < Cfg::kQPanels; ++c)
        ptx::tma_load_3d(sbase + Cfg::offQ + c * kSubTile, &p.tq, bar_q, c * 64, h, tile.row0);
    }
    if (lane < 2 && n_kv > 0) {
      const bool kstream = lane == 0;
      const int NS = kstream ? Cfg::NSK : Cfg::NSV;
      const uint32_t bytes = kstream ? Cfg::kKBytes : Cfg::kVBytes;
      const int panels = kstream ? Cfg::kQPanels : Cfg::kVPanels;
      const uint32_t base = sbase + (kstream ? Cfg::offK : Cfg::offV);
      const CUtensorMap* map = kstream ? &p.tk : &p.tv;
      auto full = [&](int st) { return kstream ? bar_k_full(st) : bar_v_full(st); };
      auto empty = [&](int st) { return kstream ? bar_k_empty(st) : bar_v_empty(st); };
      int issued = 0;
      KvCursor cur;
      cur.init(a.ranges, tile.range_begin, tile.range_count);
      for (int j = 0; j < n_kv; ++j, cur.next()) {
        const int st = j % NS;
        if (j >= NS && !ptx::mbar_wait(empty(st), ((j / NS) - 1) & 1, kstream ? kSiteKEmpty : kSiteVEmpty, wctx)) break;
        ptx::mbar_arrive_expect_tx(full(st), bytes);
        if (!PACKED || !cur.packed()) {
          for (int c = 0; c < panels; ++c)
            ptx::tma_load_3d(base + st * bytes + c * kSubTile, map, full(st), c * 64, kvh, cur.row());
        } else {
          // the pieces cover tile rows [0, BN) from 8-row (1 KiB) boundaries,
          // so the boxes land on whole swizzle atoms and fill every row
          const CUtensorMap* maps = kstream ? p.tkp : p.tvp;
          const int count = cur.cur.flags >> kPackCountShift;
          for (int i = 0; i < count; ++i) {
            const PackPiece pc = a.pieces[cur.cur.row0 + i];
            const CUtensorMap* m = pc.rows >= BN ? map : maps + (max(pc.rows, 8) >> 3) - 1;
            for (int c = 0; c < panels; ++c)
              ptx::tma_load_3d(base + st * bytes + c * kSubTile + uint32_t(pc.dst) * 128, m, full(st), c * 64, kvh,
                               pc.src);
          }
        }
        ++issued;
      }
      if (*abort_flag) {
        // Let every copy still in flight land before the CTA exits.
        volatile int no_abort = 0;
        const ptx::WaitCtx drain{&no_abort, nullptr, kWaitLimitNs};
        if (kstream) ptx::mbar_wait(bar_q, 0, kSiteDrain, drain);
        for (int j = max(0, issued - NS); j < issued; ++j) ptx::mbar_wait(full(j % NS), (j / NS) & 1, kSiteDrain, drain);
      }
    }
  } else if (warp == 5 || warp == 6) {
    // ------------------------------------------------------------ MMA issuers (whole warps)
    if (n_kv > 0) {
      bool ok = true;
      if (warp == 5) {
        // S(j) = Q K(j)^T into S buffer j % 3 (A = Q, B = K, both K-major in
        // shared memory), once PV(j-3) has finished reading that buffer
        constexpr uint32_t idS = ptx::idesc_bf16_f32(BM, BN, false, false);
        const uint64_t qd = ptx::sdesc_sw128(sbase + Cfg::offQ, 16, 1024);
        ok = ptx::mbar_wait_w(bar_q, 0, kSiteQ, wctx);
        for (int j = 0; ok && j < n_kv; ++j) {
          const int sk = j % Cfg::NSK, sb = j % Cfg::NS_S;
          if (j >= Cfg::NS_S)
            ok = ptx::mbar_wait_w(bar_o_done(sb), ((j - Cfg::NS_S) / Cfg::NS_S) & 1, kSiteOFull, wctx);
          ok = ok && ptx::mbar_wait_w(bar_k_full(sk), (j / Cfg::NSK) & 1, kSiteKFull, wctx);
          if (!ok) break;
          ptx::tc_fence_after();
          const uint64_t kd = ptx::sdesc_sw128(sbase + Cfg::offK + sk * Cfg::kKBytes, 16, 1024);
          const uint32_t tS = tmem + Cfg::tS0 + BN * sb;
#pragma unroll
          for (int kk = 0; kk < DQK / 16; ++kk) {
            const uint32_t adv = ((kk >> 2) * kSubTile + (kk & 3) * 32) >> 4;
            ptx::mma_ss_w(tS, qd + adv, kd + adv, idS, kk > 0);
          }
          ptx::mma_commit_w(bar_s_full(sb));
          ptx::mma_commit_w(bar_k_empty(sk));
        }
      } else {
        // O += P(j) V(j), P(j) over the first half of S buffer j % 3
        constexpr uint32_t idO = ptx::idesc_bf16_f32(BM, DV, false, true);
        const uint32_t tO = tmem + Cfg::tO;
        for (int j = 0; ok && j < n_kv; ++j) {
          const int sv = j % Cfg::NSV, sb = j % Cfg::NS_S;
          ok = ptx::mbar_wait_w(bar_p_full(sb), (j / Cfg::NS_S) & 1, kSitePFull, wctx) &&
               ptx::mbar_wait_w(bar_v_full(sv), (j / Cfg::NSV) & 1, kSiteVFull, wctx);
          if (!ok) break;
          ptx::tc_fence_after();
          const uint64_t vd = ptx::sdesc_sw128(sbase + Cfg::offV + sv * Cfg::kVBytes, kSubTile, 1024);
          const uint32_t tP = tmem + Cfg::tS0 + BN * sb;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            ptx::mma_ts_w(tO, tP + kk * 8, vd + ((kk * 2048) >> 4), idO, (j > 0 || kk > 0));
          ptx::mma_commit_w(bar_o_done(sb));
          ptx::mma_commit_w(bar_v_empty(sv));
        }
      }
      if (!ok) {
        // Wait for every MMA this warp already issued before TMEM is released.
        volatile int no_abort = 0;
        const ptx::WaitCtx drain{&no_abort, nullptr, kWaitLimitNs};
        ptx::mma_commit_w(bar_drain(warp - 5));
        ptx::mbar_wait_w(bar_drain(warp - 5), 0, kSiteDrain, drain);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int row = threadIdx.x;  // 0..127, TMEM lane
    const uint32_t lane_base = uint32_t(warp * 32) << 16;
    const uint32_t tO = tmem + lane_base + Cfg::tO;
    const float sl2 = a.scale * kLog2e;
    const int qpos = tile.pos0 + row;
    const bool row_ok = row < tile.nrows;
    const int64_t qrow = int64_t(tile.row0) + row;
    // reference maximum of scale*log2e*s (log2 units); rows past the tile use 0
    // so that they never hold their warp on the full path
    float m_ref = row_ok ? -INFINITY : 0.f;
    float l = 0.f;
    bool ok = true;
    // A warp whose 32 rows all lie past a ragged tile only keeps the barrier
    // phases: P of those TMEM lanes feeds only O rows that are never stored.
    const bool idle_warp = __all_sync(0xffffffffu, !row_ok);
    // The tile's runs, and the key masks of its gathered tiles, are staged
    // in shared memory once, so that stepping from one short run to the next
    // costs no global-memory round trip on the softmax's critical path.
    RangeDesc* rtab = reinterpret_cast<RangeDesc*>(smem + Cfg::offRanges);
    uint4* mtab = reinterpret_cast<uint4*>(smem + Cfg::offMasks);
    const bool staged = PACKED && tile.range_count <= Cfg::kSlots;  // the same for the whole CTA
    if (staged) {
      for (int i = row; i < tile.range_count; i += 128) {
        const RangeDesc r = a.ranges[tile.range_begin + i];
        rtab[i] = r;
        if (r.flags & kRangePacked) mtab[i] = *reinterpret_cast<const uint4*>(a.packs[r.pos0].valid);
      }
      ptx::named_barrier(1, 128);  // the four softmax warps, before any wait
    }
    KvCursor cur;
    if (staged) cur.init(rtab, 0, tile.range_count);
    else cur.init(a.ranges, tile.range_begin, tile.range_count);
    for (int j = 0; j < n_kv; ++j, cur.next()) {
      const int sb = j % Cfg::NS_S;
      const uint32_t tS = tmem + lane_base + Cfg::tS0 + BN * sb;
      if (!__all_sync(0xffffffffu, ptx::mbar_wait_poll(bar_s_full(sb), (j / Cfg::NS_S) & 1, kSiteSFull, wctx))) {
        ok = false;
        break;
      }
      if (idle_warp) {
        // arrive only after S(j): one arrival per phase of the buffer's barrier
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar_p_full(sb));
        continue;
      }
      ptx::tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) ptx::tmem_ld32(tS + c * 32, sr[c]);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 4; ++c) ptx::reg_fence32(sr[c]);

      // mask: columns at or beyond `lim` are not visible to this row, nor,
      // in a gathered key tile, the columns that hold no key
      const bool packed = PACKED && cur.packed();
      const int kn = cur.n(), kp = cur.pos();
      int lim = row_ok ? kn : 0;
      if (a.causal && !packed) lim = min(lim, qpos - kp + 1);
      if (!PACKED) {
        if (lim < BN) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (c * 32 + i >= lim) sr[c][i] = __float_as_uint(-INFINITY);
        }
      } else if (lim < BN || packed) {
        uint32_t vm[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
        if (packed) {
          const uint4 vk = staged ? mtab[cur.ri] : *reinterpret_cast<const uint4*>(a.packs[cur.cur.pos0].valid);
          vm[0] = vk.x;
          vm[1] = vk.y;
          vm[2] = vk.z;
          vm[3] = vk.w;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {  // and the columns below lim
          const int t = lim - 32 * c;
          vm[c] &= t >= 32 ? 0xffffffffu : (t <= 0 ? 0u : (1u << t) - 1u);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (!(vm[c] & (1u << i))) sr[c][i] = __float_as_uint(-INFINITY);
      }
      // P = exp2(s * scale * log2e - mref) (bf16, two per column) over the
      // first half of the S buffer (PV(j-3) finished reading it before S(j)
      // was issued); returns the row sum, kept in 8 chains as 4 packed pairs
      const uint64_t sl2x2 = ptx::f32x2(sl2, sl2);
      auto exp_tile = [&](float mref) {
        uint64_t r2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) r2[e] = 0ull;
        const uint64_t nmx2 = ptx::f32x2(-mref, -mref);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint64_t x = ptx::fma_f32x2(
                ptx::f32x2(__uint_as_float(sr[c][2 * i]), __uint_as_float(sr[c][2 * i + 1])), sl2x2, nmx2);
            float x0, x1;
            ptx::f32x2_split(x, x0, x1);
            const float e0 = ptx::ex2(x0), e1 = ptx::ex2(x1);
            r2[i & 3] = ptx::add_f32x2(r2[i & 3], ptx::f32x2(e0, e1));
            pk[i] = ptx::pack_bf16(e0, e1);
          }
          ptx::tmem_st16(tS + c * 16, pk);
        }
        float r8[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) ptx::f32x2_split(r2[e], r8[2 * e], r8[2 * e + 1]);
        return ((r8[0] + r8[1]) + (r8[2] + r8[3])) + ((r8[4] + r8[5]) + (r8[6] + r8[7]));
      };
      // Fast path: exponentiate against the reference maximum as it stands,
      // without this tile's row maximum.  Exact as long as nothing overflows:
      // P and the fp32 sums only need the reference within 2^kLagLimit of
      // the true maximum, which the tile's row sum shows (any element above
      // 2^kLagLimit makes it exceed that; an overflow makes it inf).  A warp
      // with a row past that bound, or without a reference yet, takes the
      // full path: row maximum, rescale when it grew by more than 2^8, and
      // the exponentials again (overwriting the P just stored).
      float alpha = 1.f, rs = 0.f;
      bool full = !__all_sync(0xffffffffu, m_ref != -INFINITY);
      if (!full) {
        rs = exp_tile(m_ref);
        full = __any_sync(0xffffffffu, !(rs <= kLagSum));
      }
      if (full) {
        // row maximum over 8 independent chains (one warp per SMSP: the
        // latency of a single 128-long dependent chain would dominate)
        float m8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) m8[e] = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) m8[i & 7] = fmaxf(m8[i & 7], __uint_as_float(sr[c][i]));
        const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                               fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
        const float m_new = mx * sl2;
        if (m_new > m_ref + kRescaleThreshold) {
          alpha = ptx::ex2(m_ref - m_new);  // 0 when m_ref = -inf
          m_ref = m_new;
        }
        rs = exp_tile(m_ref == -INFINITY ? 0.f : m_ref);
      }
      l = l * alpha + rs;
      // O may be rescaled once PV(j-1) is complete (rare: the reference
      // maximum only moves when a row's maximum grows by more than 2^8)
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        const int jp = j - 1;  // PV(j-1) done implies every earlier PV is (in-order pipe)
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar_o_done(jp % Cfg::NS_S), (jp / Cfg::NS_S) & 1, kSiteOFull,
                                                     wctx))) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < DV / 32; ++c) {
          uint32_t o[32];
          ptx::tmem_ld32(tO + c * 32, o);
          ptx::tmem_ld_wait();
          ptx::reg_fence32(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          ptx::tmem_st32(tO + c * 32, o);
        }
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_p_full(sb));
    }

    // ------------------------------------------------------------ epilogue
    if (ok && n_kv > 0) {
      const int jl = n_kv - 1;
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar_o_done(jl % Cfg::NS_S), (jl / Cfg::NS_S) & 1, kSiteOFull, wctx));
    }
    if (ok) {
      ptx::tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse_blk = l > 0.f ? m_ref * kLn2 + logf(l) : -INFINITY;
      const int64_t orow = a.block_mode ? int64_t(tile.out_row0) + row : qrow;
      // block_mode 2: exact merge of this block's partial (o * inv, lse_blk)
      // into the accumulator ("Ulysses与Ring-Attention详解" §4.2):
      // lse = max + log1p(exp(-|a - b|)), o = e^(a - lse) o_acc + e^(b - lse) o;
      // -inf is the identity on either side.
      float wa = 0.f, wb = inv, lse_out = lse_blk;
      if (a.block_mode == 2 && row_ok) {
        const float la = a.lse[int64_t(h) * a.lse_stride + orow];
        const float mm = fmaxf(la, lse_blk);
        if (mm == -INFINITY) {
          wa = 1.f;
          wb = 0.f;
          lse_out = -INFINITY;
        } else {
          lse_out = mm + log1pf(expf(-fabsf(la - lse_blk)));
          wa = expf(la - lse_out);
          wb = expf(lse_blk - lse_out) * inv;
        }
      }
#pragma unroll 1
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t o[32];
        if (n_kv > 0) {
          ptx::tmem_ld32(tO + c * 32, o);
          ptx::tmem_ld_wait();
          ptx::reg_fence32(o);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        if (row_ok) {
          if (a.block_mode == 2) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + (orow * a.hq + h) * DV + c * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 x = dst[i];
              dst[i] = make_float4(wa * x.x + wb * __uint_as_float(o[4 * i]), wa * x.y + wb * __uint_as_float(o[4 * i + 1]),
                                   wa * x.z + wb * __uint_as_float(o[4 * i + 2]),
                                   wa * x.w + wb * __uint_as_float(o[4 * i + 3]));
            }
          } else if (a.block_mode) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + (orow * a.hq + h) * DV + c * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                   __uint_as_float(o[4 * i + 2]) * inv, __uint_as_float(o[4 * i + 3]) * inv);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + (orow * a.hq + h) * DV + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint4 v;
              v.x = ptx::pack_bf16(__uint_as_float(o[8 * i + 0]) * inv, __uint_as_float(o[8 * i + 1]) * inv);
              v.y = ptx::pack_bf16(__uint_as_float(o[8 * i + 2]) * inv, __uint_as_float(o[8 * i + 3]) * inv);
              v.z = ptx::pack_bf16(__uint_as_float(o[8 * i + 4]) * inv, __uint_as_float(o[8 * i + 5]) * inv);
              v.w = ptx::pack_bf16(__uint_as_float(o[8 * i + 6]) * inv, __uint_as_float(o[8 * i + 7]) * inv);
              dst[i] = v;
            }
          }
        }
      }
      if (row_ok) a.lse[int64_t(h) * a.lse_stride + orow] = lse_out;
    }
  }

  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

}  // namespace

EncodeTiledFn get_encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// 3-D map over a token-major [T, heads, dim] tensor: box = (inner, 1, rows).
bool make_map_3d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elt, int64_t dim, int64_t heads,
                 int64_t T, int box_inner, int box_rows, CUtensorMapSwizzle swz) {
  EncodeTiledFn enc = get_encode_tiled();
  if (enc == nullptr) return false;
  const cuuint64_t gdim[3] = {cuuint64_t(dim), cuuint64_t(heads), cuuint64_t(T)};
  const cuuint64_t gstride[2] = {cuuint64_t(dim * elt), cuuint64_t(heads * dim * elt)};
  const cuuint32_t box[3] = {cuuint32_t(box_inner), 1u, cuuint32_t(box_rows)};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  return enc(map, dt, 3, const_cast<void*>(base), gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_fwd_supported(int32_t d_qk, int32_t d_v) { return (d_qk == 128 || d_qk == 192) && d_v == 128; }

template <int DQK, int DV>
static cudaError_t launch_fwd_impl(const AttnArgs& a, cudaStream_t st) {
  using Cfg = FwdCfg<DQK, DV>;
  FwdParams p;
  p.a = a;
  p.err = device_error_word();
  if (!make_map_3d(&p.tq, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DQK, a.hq, a.T, 64, BM,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_3d(&p.tk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DQK, a.hkv, a.T_kv ? a.T_kv : a.T, 64, BN,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_3d(&p.tv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DV, a.hkv, a.T_kv ? a.T_kv : a.T, 64, BN,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (a.num_packs > 0) {
    for (int m = 0; m < kPieceMaps; ++m)
      if (!make_map_3d(&p.tkp[m], a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DQK, a.hkv, a.T_kv ? a.T_kv : a.T, 64,
                       8 * (m + 1), CU_TENSOR_MAP_SWIZZLE_128B) ||
          !make_map_3d(&p.tvp[m], a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DV, a.hkv, a.T_kv ? a.T_kv : a.T, 64,
                       8 * (m + 1), CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
  }
  auto kernel = a.num_packs > 0 ? attn_fwd_tc_kernel<DQK, DV, true> : attn_fwd_tc_kernel<DQK, DV, false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(Cfg::kSmem));
  if (e != cudaSuccess) return e;
  const int64_t grid = int64_t(a.num_tiles) * a.hq;
  if (grid == 0) return cudaSuccess;
  kernel<<<unsigned(grid), 224, Cfg::kSmem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_tc_fwd(const AttnArgs& a, cudaStream_t st) {
  if (a.d_qk == 128 && a.d_v == 128) return launch_fwd_impl<128, 128>(a, st);
  if (a.d_qk == 192 && a.d_v == 128) return launch_fwd_impl<192, 128>(a, st);
  return cudaErrorInvalidValue;
}

}  // namespace cpattn
