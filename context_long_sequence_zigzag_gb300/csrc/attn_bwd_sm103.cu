// attn_bwd_sm103.cu — context-parallel causal attention backward on the
// sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// "Ulysses与Ring-Attention详解" §4.3: the backward recomputes the attention
// probabilities instead of storing them.  They are rebuilt here from q, k and
// the forward's final lse (never from per-block statistics), with
// D = rowsum(dout * o) computed beforehand:
//     P = exp(scale q.k - lse),  dP = dout . v,  dS = scale P (dP - D)
//     dV = sum P^T dout,  dK = sum dS^T q,  dQ = sum dS k.
//
// Two kernels, neither with atomics (value heads are 128 wide; query/key
// heads 128 or 192 wide):
//
// attn_bwd_dkdv_kernel — key-tile-major.  One CTA owns a 128-row key/value
//   tile of one kv head and visits every query tile that sees it (every
//   virtual rank's runs in ring order, fully masked tiles removed), for all
//   query heads of the GQA group, summing dK and dV in TMEM.  Per step of
//   BNQ query rows (128 for 128-wide heads, 64 for 192-wide so that dK fits),
//   TMEM columns:
//     [0,BNQ)        S^T = K Q^T (SS); then P^T (bf16)
//     [BNQ,2BNQ)     dP^T = V dO^T (SS); then dS^T (bf16)
//     next 128       dV += P^T dO (TS: A read from TMEM)
//     next DQK       dK += dS^T Q (TS)
//   MMA order S(i), dK(i-1), dP(i), dV(i): the tensor pipe computes dK of
//   the previous step and dP while the softmax warps turn S into P, and S of
//   the next step while they turn dP into dS.  Q and dO stream through
//   separate TMA rings (3 and 2 stages for 128-wide heads): a Q stage is
//   released by dK, a dO stage by dV.
//
// attn_bwd_dq_kernel — query-tile-major.  One CTA owns a 128-row query tile
//   of one head and visits the key tiles of the forward plan; dQ accumulates
//   in TMEM over all of them and is written once.  Per step:
//     [0,128)   S = Q K^T (TS with Q in TMEM for 128-wide heads, else SS)
//     [128,256) dP = dO V^T (SS)
//     [256,256+DQK) dQ += dS K (TS)
//     then 64 columns of dS (bf16; one buffer: a second one measured no
//     faster), then Q (bf16, 128-wide heads)
//   S(j+1) is issued as soon as S(j) has been read and dP(j+1) as soon as
//   dP(j) has been read, ahead of dQ(j).
//
// In both kernels two groups of four compute warps split the N columns
// (group g owns the g-th half, thread = TMEM lane); each group writes its
// bf16 result only into TMEM columns it has already read.  Roles: warps 0-7
// compute, warp 8 TMA producers (lanes 0 and 1, one stream each), warp 9
// TMEM allocator + MMA issuer; the dQ
// kernel adds warp 10, which issues the dQ MMAs so that waiting for dS never
// delays S and dP of the next key tile.  MMA-issuing warps run converged and
// elect one lane per instruction.  The P and dS loops use packed f32x2
// arithmetic; dK/dV stages its per-column statistics negated so that a float4
// of them is two packed addends.
//
// Gathered tiles (plan runs of kind kRangePacked; a separate instantiation of
// each kernel): the dQ kernel's key tiles and the dK/dV kernel's query tiles
// may hold the ragged tails of several fully visible runs, one TMA box per
// piece.  dQ masks their key-less columns from a per-tile key mask; dK/dV
// gives a query-less column the statistic -lse = -inf, so that its P and dS
// are exactly zero.
#include <cuda.h>
#include <cuda_bf16.h>

#include "internal.h"
#include "plan_check.cuh"
#include "sm103_ptx.cuh"

namespace cpattn {

bool make_map_3d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elt, int64_t dim, int64_t heads,
                 int64_t T, int box_inner, int box_rows, CUtensorMapSwizzle swz);

namespace {

constexpr int BT = 128;                 // key rows per dK/dV tile, key rows per dQ step
constexpr int DV = 128;                 // value head dim
constexpr uint32_t kPanel = 128 * 128;  // 128 rows x 64 bf16 columns, 128-byte swizzled: 16 KiB
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr int kComputeThreads = 256;
constexpr int kThreads = kComputeThreads + 64;
constexpr int kThreadsDq = kComputeThreads + 96;  // dQ kernel: a second MMA-issuing warp

enum WaitSite : int {
  kSiteKV = 0x21, kSiteQEmpty, kSiteQFull, kSiteSFull, kSiteDPFull, kSitePFull, kSiteDSFull, kSiteFinal,
  kSiteDrain, kSiteAlign, kSiteStat, kSiteKVFull, kSiteKVEmpty, kSiteQ,
};

// Boxes of 8, 16, ..., 120 rows for the pieces of gathered tiles
// (kRangePacked runs): K and V for the dQ kernel's key tiles, Q and dO for
// the dK/dV kernel's query tiles.  A piece of r rows (a multiple of 8) is one
// box per panel (map r / 8 - 1; the 128-row maps for r = 128).
constexpr int kPieceMaps = 15;

struct BwdParams {
  CUtensorMap tq, tk, tv, tdo;
  CUtensorMap tkp[kPieceMaps], tvp[kPieceMaps];  // box rows 8 (i + 1); dQ with gathered tiles only
  CUtensorMap tqp[kPieceMaps], top[kPieceMaps];  // the same for Q and dO; dK/dV with gathered tiles only
  AttnArgs a;
  int32_t* err;
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

// ---------------------------------------------------------------------------
// Shared pieces of the compute warps.
// ---------------------------------------------------------------------------

// NC consecutive TMEM columns of this thread's lane into registers.
template <int NC>
__device__ __forceinline__ void ldcols(uint32_t taddr, uint32_t (&x)[NC / 32][32]) {
#pragma unroll
  for (int c = 0; c < NC / 32; ++c) ptx::tmem_ld32(taddr + 32 * c, x[c]);
  ptx::tmem_ld_wait();
#pragma unroll
  for (int c = 0; c < NC / 32; ++c) ptx::reg_fence32(x[c]);
}

template <int NC>
__device__ __forceinline__ float colv(const uint32_t (&x)[NC / 32][32], int c) {
  return __uint_as_float(x[c >> 5][c & 31]);
}

// Packs NC floats into NC/2 bf16 pairs and stores them into NC/2 TMEM columns.
template <int NC>
__device__ __forceinline__ void st_bf16(uint32_t taddr, const float (&v)[NC]) {
  if constexpr (NC == 64) {
    uint32_t pk[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) pk[j] = ptx::pack_bf16(v[2 * j], v[2 * j + 1]);
    ptx::tmem_st32(taddr, pk);
  } else {
    static_assert(NC == 32, "column count");
    uint32_t pk[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) pk[j] = ptx::pack_bf16(v[2 * j], v[2 * j + 1]);
    ptx::tmem_st16(taddr, pk);
  }
}

// NC FP32 TMEM columns of this lane (from `taddr`) as bf16 into dst[0..NC).
template <int NC>
__device__ __forceinline__ void store_cols_bf16(uint32_t taddr, __nv_bfloat16* dst, bool valid, bool have) {
#pragma unroll 1
  for (int c = 0; c < NC / 32; ++c) {
    uint32_t x[32];
    if (have) {
      ptx::tmem_ld32(taddr + 32 * c, x);
      ptx::tmem_ld_wait();
      ptx::reg_fence32(x);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] = 0u;
    }
    if (valid) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint4 v;
        v.x = ptx::pack_bf16(__uint_as_float(x[8 * k + 0]), __uint_as_float(x[8 * k + 1]));
        v.y = ptx::pack_bf16(__uint_as_float(x[8 * k + 2]), __uint_as_float(x[8 * k + 3]));
        v.z = ptx::pack_bf16(__uint_as_float(x[8 * k + 4]), __uint_as_float(x[8 * k + 5]));
        v.w = ptx::pack_bf16(__uint_as_float(x[8 * k + 6]), __uint_as_float(x[8 * k + 7]));
        reinterpret_cast<uint4*>(dst + 32 * c)[k] = v;
      }
    }
  }
}

// ===========================================================================
// dK / dV
// ===========================================================================

// Walks the query steps of a key tile: for every query head of the GQA
// group, every query run of the plan, cut into BNQ-row tiles.
template <int BNQ>
struct StepCursor {
  const RangeDesc* r;
  int count, G, kvh, hkv, inter;
  int g, ri, off;
  RangeDesc cur;
  __device__ void init(const RangeDesc* ranges, int begin, int cnt, int G_, int kvh_, int hkv_, int inter_) {
    r = ranges + begin;
    count = cnt;
    G = G_;
    kvh = kvh_;
    hkv = hkv_;
    inter = inter_;
    g = 0;
    ri = 0;
    off = 0;
    if (count > 0) cur = r[0];
  }
  __device__ int head() const { return inter ? g * hkv + kvh : kvh * G + g; }
  // a gathered query tile (packed()) has its pieces from entry row0
  __device__ bool packed() const { return (cur.flags & kRangePacked) != 0; }
  __device__ int row() const { return cur.row0 + off; }
  __device__ int n() const { return min(BNQ, cur.nrows - off); }
  __device__ int pos() const { return cur.pos0 + off; }
  __device__ void next() {
    off += BNQ;
    if (off >= cur.nrows) {
      off = 0;
      if (++ri >= count) {
        ri = 0;
        ++g;
      }
      if (count > 0) cur = r[ri];
    }
  }
};

// Number of BNQ-row steps of a tile's query runs (the plan counts 128-row
// steps; 64-row steps are counted here).
template <int BNQ>
__device__ __forceinline__ int count_steps(const RangeDesc* ranges, int begin, int cnt) {
  int n = 0;
  for (int i = 0; i < cnt; ++i) n += (ranges[begin + i].nrows + BNQ - 1) / BNQ;
  return n;
}

// Negated statistic of query column t (0..BNQ-1: -lse * log2e;
// BNQ..2BNQ-1: -D * scale) of the step the cursor points at.  Stored negated
// so that a pair of them is directly the addend of a packed FMA.  In a
// gathered query tile a column that holds no query gets -lse = -inf, so that
// its P = exp2(s * scale * log2e - inf) is exactly 0 and so is its dS.
template <int BNQ, bool PACKED>
__device__ __forceinline__ float load_stat(const AttnArgs& a, const StepCursor<BNQ>& c, int t) {
  const int col = t % BNQ;
  if (t >= 2 * BNQ) return 0.f;
  int64_t row;
  if (PACKED && c.packed()) {
    row = -1;
    const int count = c.cur.flags >> kPackCountShift;
    for (int i = 0; i < count; ++i) {
      const PackPiece pc = a.pieces[c.cur.row0 + i];
      if (col >= pc.dst && col < pc.dst + pc.keys) row = int64_t(pc.src) + (col - pc.dst);
    }
    if (row < 0) return t < BNQ ? -INFINITY : 0.f;
  } else {
    if (col >= c.n()) return 0.f;
    row = c.row() + col;
  }
  const int64_t idx = int64_t(c.head()) * a.T + row;
  return t < BNQ ? -(a.lse_in[idx] * kLog2e) : -(a.dpsum[idx] * a.scale);
}

// v[0..3] = exp2(s[c0..c0+3] * sl2 + nl[0..3]) with two packed FMAs
template <int NC>
__device__ __forceinline__ void exp4(const uint32_t (&x)[NC / 32][32], int c0, uint64_t sl2x2, const float4 nl,
                                     float* v) {
  const uint64_t y0 = ptx::fma_f32x2(ptx::f32x2(colv<NC>(x, c0), colv<NC>(x, c0 + 1)), sl2x2, ptx::f32x2(nl.x, nl.y));
  const uint64_t y1 =
      ptx::fma_f32x2(ptx::f32x2(colv<NC>(x, c0 + 2), colv<NC>(x, c0 + 3)), sl2x2, ptx::f32x2(nl.z, nl.w));
  float t[4];
  ptx::f32x2_split(y0, t[0], t[1]);
  ptx::f32x2_split(y1, t[2], t[3]);
#pragma unroll
  for (int e = 0; e < 4; ++e) v[e] = ptx::ex2(t[e]);
}

// v[0..3] *= s[c0..c0+3] * scale + nd[0..3] with packed FMAs and products
template <int NC>
__device__ __forceinline__ void ds4(const uint32_t (&x)[NC / 32][32], int c0, uint64_t scx2, const float4 nd,
                                    float* v) {
  const uint64_t y0 = ptx::fma_f32x2(ptx::f32x2(colv<NC>(x, c0), colv<NC>(x, c0 + 1)), scx2, ptx::f32x2(nd.x, nd.y));
  const uint64_t y1 = ptx::fma_f32x2(ptx::f32x2(colv<NC>(x, c0 + 2), colv<NC>(x, c0 + 3)), scx2, ptx::f32x2(nd.z, nd.w));
  const uint64_t p0 = ptx::mul_f32x2(ptx::f32x2(v[0], v[1]), y0);
  const uint64_t p1 = ptx::mul_f32x2(ptx::f32x2(v[2], v[3]), y1);
  ptx::f32x2_split(p0, v[0], v[1]);
  ptx::f32x2_split(p1, v[2], v[3]);
}

template <int DQK, int BNQ>
struct DkdvCfg {
  static constexpr int kKPanels = DQK / 64;
  // Q(i) is read by S(i) and, a full step later, by dK(i); dO(i) by dP(i) and
  // dV(i) within the step: Q gets the deeper ring.
  static constexpr int NSQ = DQK == 128 ? 3 : 4;  // stages of Q
  static constexpr int NSO = DQK == 128 ? 2 : 3;  // stages of dO
  static constexpr uint32_t kQPanel = BNQ * 128;  // BNQ rows x 64 bf16 columns
  static constexpr uint32_t kKBytes = kKPanels * kPanel;
  static constexpr uint32_t kVBytes = 2 * kPanel;
  static constexpr uint32_t kQBytes = kKPanels * kQPanel;
  static constexpr uint32_t kOBytes = 2 * kQPanel;
  static constexpr uint32_t offK = 0;
  static constexpr uint32_t offV = offK + kKBytes;
  static constexpr uint32_t offQ = offV + kVBytes;        // NSQ stages
  static constexpr uint32_t offO = offQ + NSQ * kQBytes;  // NSO stages
  static constexpr uint32_t offStat = offO + NSO * kOBytes;  // [2][2*BNQ] floats
  static constexpr uint32_t offBar = offStat + 2 * 2 * BNQ * 4;
  static constexpr int kNumBars = 1 + 2 * NSQ + 2 * NSO + 9;
  static constexpr uint32_t kSmem = offBar + kNumBars * 8 + 16;
  // TMEM columns
  static constexpr uint32_t tS = 0, tDP = BNQ, tDV = 2 * BNQ, tDK = 2 * BNQ + DV;
  static constexpr int kCols = BNQ / 2;                        // columns per compute group
  static constexpr uint32_t kPk1 = BNQ - BNQ / 4;              // packed bf16 of group 1 (group 0 at 0)
  static_assert(tDK + DQK <= 512, "TMEM budget");
  static_assert(kSmem <= 232448, "shared memory budget");
};

// PACKED: the plan has gathered query tiles (kRangePacked runs, 128-row steps
// only); plans without them run an instantiation without that code.
template <int DQK, int BNQ, bool PACKED>
__global__ void __launch_bounds__(kThreads, 1) attn_bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
  using Cfg = DkdvCfg<DQK, BNQ>;
  constexpr int NC = Cfg::kCols;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = ptx::smem_u32(smem);
  const AttnArgs& a = p.a;
  if (sbase & 1023u) {  // the swizzled operand panels need 1024-byte alignment
    if (threadIdx.x == 0 && p.err) atomicCAS(p.err, 0, 0x100 | kSiteAlign);
    return;
  }
  // key/value heads outermost, then the tiles (heaviest first): the CTAs
  // resident at one time read one head's Q and dO
  const int kvh = int(blockIdx.x / unsigned(a.num_tiles));
  const int tile_idx = int(blockIdx.x - unsigned(kvh) * unsigned(a.num_tiles));
  if (a.debug && !debug_plan_ok(a, tile_idx, kvh, kvh, true, p.err)) return;
  const TileDesc tile = a.tiles[tile_idx];
  const int G = a.hq / a.hkv;
  const int n_steps = (BNQ == 128 ? tile.work : count_steps<BNQ>(a.ranges, tile.range_begin, tile.range_count)) * G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t bar0 = sbase + Cfg::offBar;
  const uint32_t bar_kv = bar0;
  auto bar_q_full = [&](int s) { return bar0 + 8u * (1 + s); };                    // Q of stage s landed
  auto bar_q_empty = [&](int s) { return bar0 + 8u * (1 + Cfg::NSQ + s); };        // dK read it
  auto bar_o_full = [&](int s) { return bar0 + 8u * (1 + 2 * Cfg::NSQ + s); };     // dO of stage s landed
  auto bar_o_empty = [&](int s) { return bar0 + 8u * (1 + 2 * Cfg::NSQ + Cfg::NSO + s); };  // dV read it
  const uint32_t bar_s_full = bar0 + 8u * (1 + 2 * Cfg::NSQ + 2 * Cfg::NSO);
  const uint32_t bar_dp_full = bar_s_full + 8;
  const uint32_t bar_p_full = bar_s_full + 16;
  const uint32_t bar_ds_full = bar_s_full + 24;
  const uint32_t bar_final = bar_s_full + 32;
  const uint32_t bar_drain = bar_s_full + 40;
  auto bar_stat = [&](int b) { return bar_s_full + 48 + 8u * b; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::offBar + Cfg::kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::offBar + Cfg::kNumBars * 8 + 4);
  float* stat = reinterpret_cast<float*>(smem + Cfg::offStat);

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar_kv, 1);
    for (int s = 0; s < Cfg::NSQ; ++s) {
      ptx::mbar_init(bar_q_full(s), 1);
      ptx::mbar_init(bar_q_empty(s), 1);
    }
    for (int s = 0; s < Cfg::NSO; ++s) {
      ptx::mbar_init(bar_o_full(s), 1);
      ptx::mbar_init(bar_o_empty(s), 1);
    }
    ptx::mbar_init(bar_s_full, 1);
    ptx::mbar_init(bar_dp_full, 1);
    ptx::mbar_init(bar_p_full, 8);
    ptx::mbar_init(bar_ds_full, 8);
    ptx::mbar_init(bar_final, 1);
    ptx::mbar_init(bar_drain, 1);
    ptx::mbar_init(bar_stat(0), kComputeThreads);
    ptx::mbar_init(bar_stat(1), kComputeThreads);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 9) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 512);
    ptx::tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    ptx::prefetch_tmap(&p.tq);
    ptx::prefetch_tmap(&p.tk);
    ptx::prefetch_tmap(&p.tv);
    ptx::prefetch_tmap(&p.tdo);
  }
  if (PACKED && warp == 8 && lane >= 2)  // the piece maps, one per lane
    ptx::prefetch_tmap(lane < 2 + kPieceMaps ? &p.tqp[lane - 2] : &p.top[lane - 2 - kPieceMaps]);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const ptx::WaitCtx wctx{abort_flag, p.err, kWaitLimitNs};

  if (warp == 8) {
    // ------------------------------------------------------------ producers
    // Lane 0 loads the K/V tile, then streams Q; lane 1 streams dO.  On GB300
    // one thread's tiled TMA loads top out near 40 B/cycle, two reach ~60.
    if (lane < 2 && n_steps > 0) {
      const bool qstream = lane == 0;
      int issued = 0;
      if (qstream) {
        ptx::mbar_arrive_expect_tx(bar_kv, Cfg::kKBytes + Cfg::kVBytes);
        for (int c = 0; c < Cfg::kKPanels; ++c)
          ptx::tma_load_3d(sbase + Cfg::offK + c * kPanel, &p.tk, bar_kv, c * 64, kvh, tile.row0);
        for (int c = 0; c < 2; ++c)
          ptx::tma_load_3d(sbase + Cfg::offV + c * kPanel, &p.tv, bar_kv, c * 64, kvh, tile.row0);
      }
      const int NS = qstream ? Cfg::NSQ : Cfg::NSO;
      auto full = [&](int st) { return qstream ? bar_q_full(st) : bar_o_full(st); };
      auto empty = [&](int st) { return qstream ? bar_q_empty(st) : bar_o_empty(st); };
      StepCursor<BNQ> cur;
      cur.init(a.ranges, tile.range_begin, tile.range_count, G, kvh, a.hkv, a.gqa_interleaved);
      for (int i = 0; i < n_steps; ++i, cur.next()) {
        const int st = i % NS;
        // stage st is free once the last reader of its previous occupant completed
        if (i >= NS && !ptx::mbar_wait(empty(st), ((i / NS) - 1) & 1, kSiteQEmpty, wctx)) break;
        const int h = cur.head();
        const uint32_t dst0 = sbase + (qstream ? Cfg::offQ + st * Cfg::kQBytes : Cfg::offO + st * Cfg::kOBytes);
        const int panels = qstream ? Cfg::kKPanels : 2;
        const CUtensorMap* map = qstream ? &p.tq : &p.tdo;
        ptx::mbar_arrive_expect_tx(full(st), qstream ? Cfg::kQBytes : Cfg::kOBytes);
        if (!PACKED || !cur.packed()) {
          for (int c = 0; c < panels; ++c)
            ptx::tma_load_3d(dst0 + c * Cfg::kQPanel, map, full(st), c * 64, h, cur.row());
        } else {
          // one box per piece; the pieces cover rows [0, BNQ) of the step
          // from 8-row (1 KiB) boundaries
          const CUtensorMap* maps = qstream ? p.tqp : p.top;
          const int count = cur.cur.flags >> kPackCountShift;
          for (int k = 0; k < count; ++k) {
            const PackPiece pc = a.pieces[cur.cur.row0 + k];
            const CUtensorMap* m = pc.rows >= BNQ ? map : maps + (max(pc.rows, 8) >> 3) - 1;
            for (int c = 0; c < panels; ++c)
              ptx::tma_load_3d(dst0 + c * Cfg::kQPanel + uint32_t(pc.dst) * 128, m, full(st), c * 64, h, pc.src);
          }
        }
        ++issued;
      }
      if (*abort_flag) {
        volatile int no_abort = 0;
        const ptx::WaitCtx drain{&no_abort, nullptr, kWaitLimitNs};
        if (qstream) ptx::mbar_wait(bar_kv, 0, kSiteDrain, drain);
        for (int i = max(0, issued - NS); i < issued; ++i) ptx::mbar_wait(full(i % NS), (i / NS) & 1, kSiteDrain, drain);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer (whole warp)
    if (n_steps > 0) {
      constexpr uint32_t idS = ptx::idesc_bf16_f32(BT, BNQ, false, false);
      constexpr uint32_t idDV = ptx::idesc_bf16_f32(BT, DV, false, true);  // B = dO, MN-major
      constexpr uint32_t idDK = ptx::idesc_bf16_f32(BT, DQK, false, true);  // B = Q, MN-major
      const uint32_t tS = tmem + Cfg::tS, tDP = tmem + Cfg::tDP, tDV = tmem + Cfg::tDV, tDK = tmem + Cfg::tDK;
      const uint32_t kb = sbase + Cfg::offK, vb = sbase + Cfg::offV;
      auto qb = [&](int i) { return sbase + Cfg::offQ + (i % Cfg::NSQ) * Cfg::kQBytes; };
      auto ob = [&](int i) { return sbase + Cfg::offO + (i % Cfg::NSO) * Cfg::kOBytes; };
      // D = A (K-major panels of 128 rows) x B^T (K-major panels of BNQ rows)
      auto issue_ss = [&](uint32_t d, uint32_t abase, uint32_t bbase, int ksteps) {
        const uint64_t da = ptx::sdesc_sw128(abase, 16, 1024), db = ptx::sdesc_sw128(bbase, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < ksteps; ++kk)
          ptx::mma_ss_w(d, da + (((kk >> 2) * kPanel + (kk & 3) * 32) >> 4),
                      db + (((kk >> 2) * Cfg::kQPanel + (kk & 3) * 32) >> 4), idS, kk > 0);
      };
      // D += (packed bf16 A in TMEM: group 0 at a0, group 1 at a0 + kPk1) x B (MN-major smem)
      auto issue_ts = [&](uint32_t d, uint32_t a0, uint32_t bbase, uint32_t idesc, bool acc) {
        const uint64_t db = ptx::sdesc_sw128(bbase, Cfg::kQPanel, 1024);
#pragma unroll
        for (int kk = 0; kk < BNQ / 16; ++kk) {
          const uint32_t acol = kk < BNQ / 32 ? kk * 8 : Cfg::kPk1 + (kk - BNQ / 32) * 8;
          ptx::mma_ts_w(d, a0 + acol, db + ((kk * 2048) >> 4), idesc, (acc || kk > 0));
        }
      };
      bool ok = ptx::mbar_wait_w(bar_kv, 0, kSiteKV, wctx) && ptx::mbar_wait_w(bar_q_full(0), 0, kSiteQFull, wctx);
      if (ok) {
        ptx::tc_fence_after();
        issue_ss(tS, kb, qb(0), DQK / 16);
        ptx::mma_commit_w(bar_s_full);
      }
      for (int i = 0; ok && i < n_steps; ++i) {
        // dK(i-1) needs dS(i-1): once it is issued, dP(i) may overwrite tDP
        if (i > 0) {
          if (!ptx::mbar_wait_w(bar_ds_full, (i - 1) & 1, kSiteDSFull, wctx)) { ok = false; break; }
          ptx::tc_fence_after();
          issue_ts(tDK, tDP, qb(i - 1), idDK, i - 1 > 0);
          ptx::mma_commit_w(bar_q_empty((i - 1) % Cfg::NSQ));
        }
        if (!ptx::mbar_wait_w(bar_o_full(i % Cfg::NSO), (i / Cfg::NSO) & 1, kSiteQFull, wctx)) { ok = false; break; }
        ptx::tc_fence_after();
        issue_ss(tDP, vb, ob(i), DV / 16);
        ptx::mma_commit_w(bar_dp_full);
        // dV(i) needs P(i); once it is issued, S(i+1) may overwrite tS
        if (!ptx::mbar_wait_w(bar_p_full, i & 1, kSitePFull, wctx)) { ok = false; break; }
        ptx::tc_fence_after();
        issue_ts(tDV, tS, ob(i), idDV, i > 0);
        ptx::mma_commit_w(bar_o_empty(i % Cfg::NSO));
        if (i + 1 < n_steps) {
          if (!ptx::mbar_wait_w(bar_q_full((i + 1) % Cfg::NSQ), ((i + 1) / Cfg::NSQ) & 1, kSiteQFull, wctx)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          issue_ss(tS, kb, qb(i + 1), DQK / 16);
          ptx::mma_commit_w(bar_s_full);
        }
      }
      if (ok) {
        ok = ptx::mbar_wait_w(bar_ds_full, (n_steps - 1) & 1, kSiteDSFull, wctx);
        if (ok) {
          ptx::tc_fence_after();
          issue_ts(tDK, tDP, qb(n_steps - 1), idDK, n_steps - 1 > 0);
          ptx::mma_commit_w(bar_final);
        }
      }
      if (!ok) {
        volatile int no_abort = 0;
        const ptx::WaitCtx drain{&no_abort, nullptr, kWaitLimitNs};
        ptx::mma_commit_w(bar_drain);
        ptx::mbar_wait_w(bar_drain, 0, kSiteDrain, drain);
      }
    }
  } else {
    // ------------------------------------------------------------ compute warps
    const int grp = warp >> 2;               // query columns NC*grp .. NC*grp+NC-1
    const int r = ((warp & 3) << 5) | lane;  // key row = TMEM lane
    const int t = threadIdx.x;               // 0..255, statistics loader index
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + Cfg::tS, tDP = tmem + lane_base + Cfg::tDP;
    const uint32_t colS = grp * NC;
    const uint32_t colPk = grp ? Cfg::kPk1 : 0;
    const float sl2 = a.scale * kLog2e;
    const uint64_t sl2x2 = ptx::f32x2(sl2, sl2), scx2 = ptx::f32x2(a.scale, a.scale);
    const int kpos = tile.pos0 + r;
    const int nk = tile.nrows;
    bool ok = true;

    StepCursor<BNQ> cur, nxt;
    cur.init(a.ranges, tile.range_begin, tile.range_count, G, kvh, a.hkv, a.gqa_interleaved);
    nxt = cur;
    if (n_steps > 0) {
      if (t < 2 * BNQ) stat[t] = load_stat<BNQ, PACKED>(a, cur, t);
      ptx::mbar_arrive(bar_stat(0));
    }
    nxt.next();
    for (int i = 0; i < n_steps; ++i, cur.next(), nxt.next()) {
      const int nq = cur.n(), qpos0 = cur.pos();
      const float* sL = stat + (i & 1) * 2 * BNQ;
      const float* sD = sL + BNQ;
      // statistics of this step are in place (a buffer is refilled only after
      // every compute warp passed the dS phase of the step in between)
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar_stat(i & 1), (i >> 1) & 1, kSiteStat, wctx))) {
        ok = false;
        break;
      }
      const float nstat = (i + 1 < n_steps) ? load_stat<BNQ, PACKED>(a, nxt, t) : 0.f;
      // a gathered query tile is causally unmasked; its query-less columns
      // have P = 0 through their statistics
      const bool causal = a.causal && !(PACKED && cur.packed());
      const bool need_mask = nq < BNQ || nk < BT || (causal && qpos0 < tile.pos0 + BT - 1);
      const int cmin = (causal ? kpos - qpos0 : 0) - int(colS);  // first visible column (relative)
      const int cmax = (r < nk ? nq : 0) - int(colS);             // columns [cmin, cmax) are visible

      // ---- P^T = exp(S^T * scale - lse)
      if (!__all_sync(0xffffffffu, ptx::mbar_wait_poll(bar_s_full, i & 1, kSiteSFull, wctx))) { ok = false; break; }
      ptx::tc_fence_after();
      uint32_t x[NC / 32][32];
      ldcols<NC>(tS + colS, x);
      float pf[NC];
      // Warp-uniform split: only tiles on the diagonal or at a ragged edge
      // pay for the per-element visibility test.
      if (need_mask) {
#pragma unroll
        for (int j = 0; j < NC; j += 4) {
          exp4<NC>(x, j, sl2x2, *reinterpret_cast<const float4*>(sL + colS + j), pf + j);
#pragma unroll
          for (int e = 0; e < 4; ++e) pf[j + e] = (j + e >= cmin && j + e < cmax) ? pf[j + e] : 0.f;
        }
      } else {
#pragma unroll
        for (int j = 0; j < NC; j += 4) exp4<NC>(x, j, sl2x2, *reinterpret_cast<const float4*>(sL + colS + j), pf + j);
      }
      st_bf16<NC>(tS + colPk, pf);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_p_full);

      // ---- dS^T = P^T (dP^T - D) * scale
      if (!__all_sync(0xffffffffu, ptx::mbar_wait_poll(bar_dp_full, i & 1, kSiteDPFull, wctx))) { ok = false; break; }
      ptx::tc_fence_after();
      ldcols<NC>(tDP + colS, x);
#pragma unroll
      for (int j = 0; j < NC; j += 4) ds4<NC>(x, j, scx2, *reinterpret_cast<const float4*>(sD + colS + j), pf + j);
      st_bf16<NC>(tDP + colPk, pf);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_ds_full);
      if (i + 1 < n_steps) {
        if (t < 2 * BNQ) stat[((i + 1) & 1) * 2 * BNQ + t] = nstat;
        ptx::mbar_arrive(bar_stat((i + 1) & 1));
      }
    }

    // ------------------------------------------------------------ dK, dV epilogue
    if (ok && n_steps > 0) ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar_final, 0, kSiteFinal, wctx));
    if (ok) {
      ptx::tc_fence_after();
      const int64_t krow = int64_t(tile.row0) + r;
      // group 0 writes dV, group 1 writes dK
      if (grp == 0)
        store_cols_bf16<DV>(tmem + lane_base + Cfg::tDV,
                            static_cast<__nv_bfloat16*>(a.dv) + (krow * a.hkv + kvh) * DV, r < nk, n_steps > 0);
      else
        store_cols_bf16<DQK>(tmem + lane_base + Cfg::tDK,
                             static_cast<__nv_bfloat16*>(a.dk) + (krow * a.hkv + kvh) * DQK, r < nk, n_steps > 0);
    }
  }

  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// ===========================================================================
// dQ
// ===========================================================================

// Iterates the key tiles of a query tile's plan entry (runs cut into BT rows).
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
  // a gathered tile (packed()) has its pieces from entry row0 and its key
  // mask at pos0
  __device__ bool packed() const { return (cur.flags & kRangePacked) != 0; }
  __device__ int row() const { return cur.row0 + off; }
  __device__ int n() const { return min(BT, cur.nrows - off); }
  __device__ int pos() const { return cur.pos0 + off; }
  __device__ void next() {
    off += BT;
    if (off >= cur.nrows) {
      off = 0;
      if (++ri < count) cur = r[ri];
    }
  }
};

template <int DQK>
struct DqCfg {
  // 128-wide heads keep Q in TMEM (64 packed columns after the single dS
  // buffer), so S = Q K^T is a TS MMA and Q's shared memory goes to a
  // fourth K stage.  K(j) is read by S(j) and, later, by dQ(j); V(j) only
  // by dP(j): K gets the deeper ring.
  static constexpr bool kQTmem = DQK == 128;
  static constexpr int kKPanels = DQK / 64;
  static constexpr int NSK = DQK == 128 ? 4 : 2;
  static constexpr int NSV = DQK == 128 ? 2 : 1;
  static constexpr int NB = 1;  // dS buffers
  static constexpr uint32_t kKBytes = kKPanels * kPanel;
  static constexpr uint32_t kVBytes = 2 * kPanel;
  static constexpr uint32_t kQBytes = kQTmem ? 0 : kKBytes;  // Q panels in shared memory
  static constexpr uint32_t offQ = 0;
  static constexpr uint32_t offO = offQ + kQBytes;
  static constexpr uint32_t offK = offO + kVBytes;           // NSK stages
  static constexpr uint32_t offV = offK + NSK * kKBytes;     // NSV stages
  static constexpr uint32_t offBar = offV + NSV * kVBytes;
  static constexpr int kNumBars = 1 + 2 * NSK + 2 * NSV + 9 + NB;
  // the tile's runs and the key masks of its gathered tiles, staged for the
  // compute warps when the tile has at most kSlots runs (gathering plans only)
  static constexpr int kSlots = 64;
  static constexpr uint32_t offRanges = (offBar + kNumBars * 8 + 16 + 15) / 16 * 16;
  static constexpr uint32_t offMasks = offRanges + kSlots * 16;
  static constexpr uint32_t kSmem = offMasks + kSlots * 16;
  // TMEM columns
  static constexpr uint32_t tS = 0, tDP = 128, tDQ = 256, tDS = 256 + DQK, tQ = tDS + 64 * NB;
  static_assert(tQ + (kQTmem ? DQK / 2 : 0) <= 512, "TMEM budget");
  static_assert(kSmem <= 232448, "shared memory budget");
};

// PACKED: the plan has gathered key tiles (kRangePacked runs); plans without
// them run an instantiation without that code.
template <int DQK, bool PACKED>
__global__ void __launch_bounds__(kThreadsDq, 1) attn_bwd_dq_kernel(const __grid_constant__ BwdParams p) {
  using Cfg = DqCfg<DQK>;
  constexpr int NB = Cfg::NB;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = ptx::smem_u32(smem);
  const AttnArgs& a = p.a;
  if (sbase & 1023u) {
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
  const uint32_t bar_q = bar0;
  auto bar_k_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto bar_k_empty = [&](int s) { return bar0 + 8u * (1 + Cfg::NSK + s); };
  auto bar_v_full = [&](int s) { return bar0 + 8u * (1 + 2 * Cfg::NSK + s); };
  auto bar_v_empty = [&](int s) { return bar0 + 8u * (1 + 2 * Cfg::NSK + Cfg::NSV + s); };
  const uint32_t bar_s_full = bar0 + 8u * (1 + 2 * Cfg::NSK + 2 * Cfg::NSV);
  const uint32_t bar_dp_full = bar_s_full + 8;
  const uint32_t bar_p_full = bar_s_full + 16;
  const uint32_t bar_ds_full = bar_s_full + 24;
  const uint32_t bar_final = bar_s_full + 32;
  const uint32_t bar_drain = bar_s_full + 40;
  const uint32_t bar_dp_read = bar_s_full + 48;                        // compute warps hold dP(j)
  auto bar_dq_done = [&](int b) { return bar_s_full + 56 + 8u * b; };  // dQ(j) read dS buffer b = j % NB
  const uint32_t bar_drain2 = bar_s_full + 56 + 8u * NB;            // drain of the dQ issuer
  const uint32_t bar_qt = bar_s_full + 64 + 8u * NB;                // Q rows written into TMEM (8 warps)
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
    ptx::mbar_init(bar_s_full, 1);
    ptx::mbar_init(bar_dp_full, 1);
    ptx::mbar_init(bar_p_full, 8);
    ptx::mbar_init(bar_ds_full, 8);
    ptx::mbar_init(bar_final, 1);
    ptx::mbar_init(bar_drain, 1);
    ptx::mbar_init(bar_dp_read, 8);
    for (int b = 0; b < NB; ++b) ptx::mbar_init(bar_dq_done(b), 1);
    ptx::mbar_init(bar_drain2, 1);
    ptx::mbar_init(bar_qt, 8);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 9) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 512);
    ptx::tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    ptx::prefetch_tmap(&p.tq);
    ptx::prefetch_tmap(&p.tk);
    ptx::prefetch_tmap(&p.tv);
    ptx::prefetch_tmap(&p.tdo);
  }
  if (PACKED && warp == 8 && lane >= 2)  // the piece maps, one per lane
    ptx::prefetch_tmap(lane < 2 + kPieceMaps ? &p.tkp[lane - 2] : &p.tvp[lane - 2 - kPieceMaps]);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const ptx::WaitCtx wctx{abort_flag, p.err, kWaitLimitNs};

  if (warp == 8) {
    // ------------------------------------------------------------ producers
    // Lane 0 streams K; lane 1 loads Q / dO, then streams V.  On GB300 one
    // thread's tiled TMA loads top out near 40 B/cycle, two reach about 60.
    if (lane < 2 && n_kv > 0) {
      const bool kstream = lane == 0;
      const int NS = kstream ? Cfg::NSK : Cfg::NSV;
      const uint32_t bytes = kstream ? Cfg::kKBytes : Cfg::kVBytes;
      const int panels = kstream ? Cfg::kKPanels : 2;
      const uint32_t base = sbase + (kstream ? Cfg::offK : Cfg::offV);
      const CUtensorMap* map = kstream ? &p.tk : &p.tv;
      auto full = [&](int st) { return kstream ? bar_k_full(st) : bar_v_full(st); };
      auto empty = [&](int st) { return kstream ? bar_k_empty(st) : bar_v_empty(st); };
      if (!kstream) {
        ptx::mbar_arrive_expect_tx(bar_q, Cfg::kQBytes + Cfg::kVBytes);
        if (!Cfg::kQTmem)
          for (int c = 0; c < Cfg::kKPanels; ++c)
            ptx::tma_load_3d(sbase + Cfg::offQ + c * kPanel, &p.tq, bar_q, c * 64, h, tile.row0);
        for (int c = 0; c < 2; ++c)
          ptx::tma_load_3d(sbase + Cfg::offO + c * kPanel, &p.tdo, bar_q, c * 64, h, tile.row0);
      }
      int issued = 0;
      KvCursor cur;
      cur.init(a.ranges, tile.range_begin, tile.range_count);
      for (int j = 0; j < n_kv; ++j, cur.next()) {
        const int st = j % NS;
        if (j >= NS && !ptx::mbar_wait(empty(st), ((j / NS) - 1) & 1, kSiteKVEmpty, wctx)) break;
        ptx::mbar_arrive_expect_tx(full(st), bytes);
        if (!PACKED || !cur.packed()) {
          for (int c = 0; c < panels; ++c)
            ptx::tma_load_3d(base + st * bytes + c * kPanel, map, full(st), c * 64, kvh, cur.row());
        } else {
          // one box per piece; the pieces cover tile rows [0, BT) from 8-row
          // (1 KiB) boundaries
          const CUtensorMap* maps = kstream ? p.tkp : p.tvp;
          const int count = cur.cur.flags >> kPackCountShift;
          for (int i = 0; i < count; ++i) {
            const PackPiece pc = a.pieces[cur.cur.row0 + i];
            const CUtensorMap* m = pc.rows >= BT ? map : maps + (max(pc.rows, 8) >> 3) - 1;
            for (int c = 0; c < panels; ++c)
              ptx::tma_load_3d(base + st * bytes + c * kPanel + uint32_t(pc.dst) * 128, m, full(st), c * 64, kvh,
                               pc.src);
          }
        }
        ++issued;
      }
      if (*abort_flag) {
        volatile int no_abort = 0;
        const ptx::WaitCtx drain{&no_abort, nullptr, kWaitLimitNs};
        if (!kstream) ptx::mbar_wait(bar_q, 0, kSiteDrain, drain);
        for (int j = max(0, issued - NS); j < issued; ++j) ptx::mbar_wait(full(j % NS), (j / NS) & 1, kSiteDrain, drain);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer of S and dP (whole warp)
    if (n_kv > 0) {
      constexpr uint32_t idS = ptx::idesc_bf16_f32(BT, BT, false, false);
      const uint32_t tS = tmem + Cfg::tS, tDP = tmem + Cfg::tDP;
      const uint32_t qb = sbase + Cfg::offQ, obb = sbase + Cfg::offO;
      auto kb = [&](int j) { return sbase + Cfg::offK + (j % Cfg::NSK) * Cfg::kKBytes; };
      auto vb = [&](int j) { return sbase + Cfg::offV + (j % Cfg::NSV) * Cfg::kVBytes; };
      auto issue_ss = [&](uint32_t d, uint32_t abase, uint32_t bbase, int ksteps) {
        const uint64_t da = ptx::sdesc_sw128(abase, 16, 1024), db = ptx::sdesc_sw128(bbase, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < ksteps; ++kk) {
          const uint32_t off = ((kk >> 2) * kPanel + (kk & 3) * 32) >> 4;
          ptx::mma_ss_w(d, da + off, db + off, idS, kk > 0);
        }
      };
      // S(j) = Q K(j)^T: TS with Q from TMEM (128-wide heads), else SS
      auto issue_s = [&](int j) {
        if constexpr (Cfg::kQTmem) {
          const uint64_t kd = ptx::sdesc_sw128(kb(j), 16, 1024);
#pragma unroll
          for (int kk = 0; kk < DQK / 16; ++kk)
            ptx::mma_ts_w(tS, tmem + Cfg::tQ + kk * 8, kd + (((kk >> 2) * kPanel + (kk & 3) * 32) >> 4), idS, kk > 0);
        } else {
          issue_ss(tS, qb, kb(j), DQK / 16);
        }
      };
      bool ok = ptx::mbar_wait_w(Cfg::kQTmem ? bar_qt : bar_q, 0, kSiteQ, wctx) &&
                ptx::mbar_wait_w(bar_k_full(0), 0, kSiteKVFull, wctx);
      if (ok) {
        ptx::tc_fence_after();
        issue_s(0);
        ptx::mma_commit_w(bar_s_full);
        ok = (!Cfg::kQTmem || ptx::mbar_wait_w(bar_q, 0, kSiteQ, wctx)) &&
             ptx::mbar_wait_w(bar_v_full(0), 0, kSiteKVFull, wctx);
      }
      if (ok) {
        ptx::tc_fence_after();
        issue_ss(tDP, obb, vb(0), DV / 16);
        ptx::mma_commit_w(bar_dp_full);
        ptx::mma_commit_w(bar_v_empty(0));
      }
      for (int j = 0; ok && j + 1 < n_kv; ++j) {
        // S(j+1) as soon as the compute warps have read S(j)
        if (!ptx::mbar_wait_w(bar_p_full, j & 1, kSitePFull, wctx) ||
            !ptx::mbar_wait_w(bar_k_full((j + 1) % Cfg::NSK), ((j + 1) / Cfg::NSK) & 1, kSiteKVFull, wctx)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        issue_s(j + 1);
        ptx::mma_commit_w(bar_s_full);
        // dP(j+1) as soon as they have read dP(j)
        if (!ptx::mbar_wait_w(bar_dp_read, j & 1, kSiteDPFull, wctx) ||
            !ptx::mbar_wait_w(bar_v_full((j + 1) % Cfg::NSV), ((j + 1) / Cfg::NSV) & 1, kSiteKVFull, wctx)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        issue_ss(tDP, obb, vb(j + 1), DV / 16);
        ptx::mma_commit_w(bar_dp_full);
        ptx::mma_commit_w(bar_v_empty((j + 1) % Cfg::NSV));
      }
      if (!ok) {
        volatile int no_abort = 0;
        const ptx::WaitCtx drain{&no_abort, nullptr, kWaitLimitNs};
        ptx::mma_commit_w(bar_drain);
        ptx::mbar_wait_w(bar_drain, 0, kSiteDrain, drain);
      }
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------ MMA issuer of dQ (whole warp)
    // A second issuing warp: dQ(j) waits only for dS(j), so its wait never
    // holds back S and dP of the next key tile.  It reads TMEM columns of its
    // own (the dS buffers) and writes the dQ accumulator, which no MMA of the
    // other warp touches; K(j) was last read by S(j), complete before the
    // compute warps could publish dS(j).
    if (n_kv > 0) {
      constexpr uint32_t idQ = ptx::idesc_bf16_f32(BT, DQK, false, true);  // dQ: B = K as MN-major
      const uint32_t tDQ = tmem + Cfg::tDQ;
      bool ok = true;
      for (int j = 0; j < n_kv; ++j) {
        // dQ(j) += dS(j) K(j), dS(j) in buffer j % NB
        if (!ptx::mbar_wait_w(bar_ds_full, j & 1, kSiteDSFull, wctx)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint64_t kd = ptx::sdesc_sw128(sbase + Cfg::offK + (j % Cfg::NSK) * Cfg::kKBytes, kPanel, 1024);
        const uint32_t tA = tmem + Cfg::tDS + 64 * (j % NB);
#pragma unroll
        for (int kk = 0; kk < BT / 16; ++kk)
          ptx::mma_ts_w(tDQ, tA + kk * 8, kd + ((kk * 2048) >> 4), idQ, (j > 0 || kk > 0));
        ptx::mma_commit_w(bar_dq_done(j % NB));
        ptx::mma_commit_w(bar_k_empty(j % Cfg::NSK));
      }
      if (ok) {
        ptx::mma_commit_w(bar_final);
      } else {
        volatile int no_abort = 0;
        const ptx::WaitCtx drain{&no_abort, nullptr, kWaitLimitNs};
        ptx::mma_commit_w(bar_drain2);
        ptx::mbar_wait_w(bar_drain2, 0, kSiteDrain, drain);
      }
    }
  } else {
    // ------------------------------------------------------------ compute warps
    const int grp = warp >> 2;               // key columns 64*grp .. 64*grp+63
    const int r = ((warp & 3) << 5) | lane;  // query row = TMEM lane
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + Cfg::tS, tDP = tmem + lane_base + Cfg::tDP;
    const uint32_t colS = grp * 64;
    const float sl2 = a.scale * kLog2e;
    const uint64_t sl2x2 = ptx::f32x2(sl2, sl2), scx2 = ptx::f32x2(a.scale, a.scale);
    const bool row_ok = r < tile.nrows;
    const int qpos = tile.pos0 + r;
    const int64_t qrow = int64_t(tile.row0) + r;
    const float lse2 = row_ok ? a.lse_in[int64_t(h) * a.T + qrow] * kLog2e : 0.f;
    const float dsc = row_ok ? a.dpsum[int64_t(h) * a.T + qrow] * a.scale : 0.f;
    if (Cfg::kQTmem && n_kv > 0) {
      // Q row -> TMEM, group g the g-th half (bf16 pairs are the A-operand
      // packing).  Rows past the tile read the following rows (or zeros past
      // the end); they are masked out of P.
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) +
                                                        (qrow * a.hq + h) * DQK) + grp * 8;
      const bool in_range = qrow < a.T;
      uint32_t qr[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 v = in_range ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
        qr[4 * i] = v.x;
        qr[4 * i + 1] = v.y;
        qr[4 * i + 2] = v.z;
        qr[4 * i + 3] = v.w;
      }
      ptx::tmem_st32(tmem + lane_base + Cfg::tQ + grp * 32, qr);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_qt);
    }
    bool ok = true;
    // With gathered tiles the runs and key masks are staged in shared memory
    // once (the mask is needed on the P critical path).
    RangeDesc* rtab = reinterpret_cast<RangeDesc*>(smem + Cfg::offRanges);
    uint4* mtab = reinterpret_cast<uint4*>(smem + Cfg::offMasks);
    const bool staged = PACKED && tile.range_count <= Cfg::kSlots;  // the same for the whole CTA
    if (staged) {
      for (int i = threadIdx.x; i < tile.range_count; i += kComputeThreads) {
        const RangeDesc rd = a.ranges[tile.range_begin + i];
        rtab[i] = rd;
        if (rd.flags & kRangePacked) mtab[i] = *reinterpret_cast<const uint4*>(a.packs[rd.pos0].valid);
      }
      ptx::named_barrier(1, kComputeThreads);  // the eight compute warps, before any wait
    }
    KvCursor cur;
    if (staged) cur.init(rtab, 0, tile.range_count);
    else cur.init(a.ranges, tile.range_begin, tile.range_count);
    for (int j = 0; j < n_kv; ++j, cur.next()) {
      const bool packed = PACKED && cur.packed();
      const int kn = cur.n(), kp = cur.pos();
      const bool need_mask =
          packed || kn < BT || tile.nrows < BT || (a.causal && kp + BT - 1 > tile.pos0);
      int lim = row_ok ? kn : 0;
      if (a.causal && !packed) lim = min(lim, qpos - kp + 1);
      lim -= int(colS);  // columns [0, lim) of this group are visible

      // ---- P = exp(S * scale - lse)
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar_s_full, j & 1, kSiteSFull, wctx))) { ok = false; break; }
      ptx::tc_fence_after();
      uint32_t x[2][32];
      ldcols<64>(tS + colS, x);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_p_full);  // S(j) has been read
      float pf[64];
      const float4 nl4 = make_float4(-lse2, -lse2, -lse2, -lse2);
      if (PACKED && need_mask) {  // the group's 64 columns: below lim and, if gathered, holding a key
        uint32_t vm[2];
#pragma unroll
        for (int w = 0; w < 2; ++w) {
          const int t = lim - 32 * w;
          vm[w] = t >= 32 ? 0xffffffffu : (t <= 0 ? 0u : (1u << t) - 1u);
        }
        if (packed) {
          const uint4 vk = staged ? mtab[cur.ri] : *reinterpret_cast<const uint4*>(a.packs[cur.cur.pos0].valid);
          vm[0] &= grp ? vk.z : vk.x;
          vm[1] &= grp ? vk.w : vk.y;
        }
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
          exp4<64>(x, c, sl2x2, nl4, pf + c);
#pragma unroll
          for (int e = 0; e < 4; ++e) pf[c + e] = (vm[(c + e) >> 5] & (1u << ((c + e) & 31))) ? pf[c + e] : 0.f;
        }
      } else if (need_mask) {  // warp-uniform: diagonal and ragged tiles only
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
          exp4<64>(x, c, sl2x2, nl4, pf + c);
#pragma unroll
          for (int e = 0; e < 4; ++e) pf[c + e] = c + e < lim ? pf[c + e] : 0.f;
        }
      } else {
#pragma unroll
        for (int c = 0; c < 64; c += 4) exp4<64>(x, c, sl2x2, nl4, pf + c);
      }
      // ---- dS = P (dP - D) * scale
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar_dp_full, j & 1, kSiteDPFull, wctx))) { ok = false; break; }
      ptx::tc_fence_after();
      ldcols<64>(tDP + colS, x);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_dp_read);  // dP(j) has been read
      const float4 nd4 = make_float4(-dsc, -dsc, -dsc, -dsc);
#pragma unroll
      for (int c = 0; c < 64; c += 4) ds4<64>(x, c, scx2, nd4, pf + c);
      // dS buffer j % NB was last read by dQ(j - NB)
      if (j >= NB && !__all_sync(0xffffffffu, ptx::mbar_wait(bar_dq_done(j % NB), ((j - NB) / NB) & 1,
                                                             kSiteDSFull, wctx))) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      st_bf16<64>(tmem + lane_base + Cfg::tDS + 64 * (j % NB) + 32 * grp, pf);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_ds_full);
    }

    // ------------------------------------------------------------ dQ epilogue
    if (ok && n_kv > 0) ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar_final, 0, kSiteFinal, wctx));
    if (ok) {
      ptx::tc_fence_after();
      constexpr int half = DQK / 2;  // columns written by each group
      __nv_bfloat16* dqp = static_cast<__nv_bfloat16*>(a.dq) + (qrow * a.hq + h) * DQK + grp * half;
      store_cols_bf16<half>(tmem + lane_base + Cfg::tDQ + grp * half, dqp, row_ok, n_kv > 0);
    }
  }

  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

bool make_maps(BwdParams& p, const AttnArgs& a, int dqk, int qrows) {
  return make_map_3d(&p.tq, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dqk, a.hq, a.T, 64, qrows,
                     CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_map_3d(&p.tk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dqk, a.hkv, a.T, 64, BT,
                     CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_map_3d(&p.tv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DV, a.hkv, a.T, 64, BT,
                     CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_map_3d(&p.tdo, a.dout, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DV, a.hq, a.T, 64, qrows,
                     CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int DQK, int BNQ>
cudaError_t launch_dkdv(const AttnArgs& a, cudaStream_t st) {
  using Cfg = DkdvCfg<DQK, BNQ>;
  BwdParams p;
  p.a = a;
  p.err = device_error_word();
  if (!make_maps(p, a, DQK, BNQ)) return cudaErrorInvalidValue;
  if (a.num_packs > 0) {
    if (BNQ != 128) return cudaErrorInvalidValue;  // gathered query tiles are 128 rows
    for (int m = 0; m < kPieceMaps; ++m)
      if (!make_map_3d(&p.tqp[m], a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DQK, a.hq, a.T, 64, 8 * (m + 1),
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
          !make_map_3d(&p.top[m], a.dout, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DV, a.hq, a.T, 64, 8 * (m + 1),
                       CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
  }
  auto kernel = a.num_packs > 0 ? attn_bwd_dkdv_kernel<DQK, BNQ, true> : attn_bwd_dkdv_kernel<DQK, BNQ, false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(Cfg::kSmem));
  if (e != cudaSuccess) return e;
  const int64_t grid = int64_t(a.num_tiles) * a.hkv;
  if (grid == 0) return cudaSuccess;
  kernel<<<unsigned(grid), kThreads, Cfg::kSmem, st>>>(p);
  return cudaGetLastError();
}

template <int DQK>
cudaError_t launch_dq(const AttnArgs& a, cudaStream_t st) {
  using Cfg = DqCfg<DQK>;
  BwdParams p;
  p.a = a;
  p.err = device_error_word();
  if (!make_maps(p, a, DQK, BT)) return cudaErrorInvalidValue;
  if (a.num_packs > 0) {
    for (int m = 0; m < kPieceMaps; ++m)
      if (!make_map_3d(&p.tkp[m], a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DQK, a.hkv, a.T, 64, 8 * (m + 1),
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
          !make_map_3d(&p.tvp[m], a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DV, a.hkv, a.T, 64, 8 * (m + 1),
                       CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
  }
  auto kernel = a.num_packs > 0 ? attn_bwd_dq_kernel<DQK, true> : attn_bwd_dq_kernel<DQK, false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(Cfg::kSmem));
  if (e != cudaSuccess) return e;
  const int64_t grid = int64_t(a.num_tiles) * a.hq;
  if (grid == 0) return cudaSuccess;
  kernel<<<unsigned(grid), kThreadsDq, Cfg::kSmem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace

bool tc_bwd_supported(int32_t d_qk, int32_t d_v) { return (d_qk == 128 || d_qk == 192) && d_v == 128; }

cudaError_t launch_tc_bwd_dkdv(const AttnArgs& a, cudaStream_t st) {
  if (a.d_v != DV) return cudaErrorInvalidValue;
  if (a.d_qk == 128) return launch_dkdv<128, 128>(a, st);
  if (a.d_qk == 192) return launch_dkdv<192, 64>(a, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_tc_bwd_dq(const AttnArgs& a, cudaStream_t st) {
  if (a.d_v != DV) return cudaErrorInvalidValue;
  if (a.d_qk == 128) return launch_dq<128>(a, st);
  if (a.d_qk == 192) return launch_dq<192>(a, st);
  return cudaErrorInvalidValue;
}

}  // namespace cpattn
