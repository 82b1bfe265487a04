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
// Two kernels, neither with atomics:
//
// attn_bwd_dkdv_kernel — key-tile-major.  One CTA owns a 128-row key/value
//   tile of one kv head and visits every query tile that sees it (every
//   virtual rank's runs in ring order, fully masked tiles removed), for all
//   query heads of the GQA group, summing dK and dV in TMEM.  Per step
//   (M = 128 keys, N = 128 queries), TMEM columns:
//     [0,128)   S^T = K Q^T (SS); then P^T (bf16) of query columns 0-63 in
//               [0,32) and of 64-127 in [96,128)
//     [128,256) dP^T = V dO^T (SS); then dS^T (bf16) in [128,160), [224,256)
//     [256,384) dV += P^T dO (TS: A read from TMEM)
//     [384,512) dK += dS^T Q (TS)
//   MMA order S(i), dK(i-1), dP(i), dV(i): the tensor pipe computes dK of
//   the previous step and dP while the softmax warps turn S into P, and S of
//   the next step while they turn dP into dS.
//
// attn_bwd_dq_kernel — query-tile-major.  One CTA owns a 128-row query tile
//   of one head and visits the key tiles of the forward plan; dQ accumulates
//   in TMEM over all of them and is written once.  Per step:
//     [0,128)   S = Q K^T (SS)
//     [128,256) dP = dO V^T (SS)
//     [256,384) dQ += dS K (TS)
//     [384,448), [448,512)  dS (bf16), double-buffered across steps
//   S(j+1) is issued as soon as S(j) has been read and dP(j+1) as soon as
//   dP(j) has been read, ahead of dQ(j), so the tensor pipe keeps working
//   while the softmax warps turn S into P and dP into dS.
//
// In both kernels two groups of four compute warps split the N = 128 columns
// (group g owns 64g..64g+63, thread = TMEM lane); each group writes its bf16
// result only into TMEM columns it has already read.  Roles (320 threads):
// warps 0-7 compute, warp 8 TMA producer, warp 9 TMEM allocator + MMA issuer.
#include <cuda.h>
#include <cuda_bf16.h>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace cpattn {

bool make_map_3d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elt, int64_t dim, int64_t heads,
                 int64_t T, int box_inner, int box_rows, CUtensorMapSwizzle swz);

namespace {

constexpr int BT = 128;                 // rows per tile, both sides
constexpr uint32_t kPanel = 128 * 128;  // 128 rows x 64 bf16 columns, 128-byte swizzled: 16 KiB
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr int kComputeThreads = 256;
constexpr int kThreads = kComputeThreads + 64;
constexpr int D = 128;                  // head dim (q/k and v)
constexpr uint32_t kTileBytes = (D / 64) * kPanel;  // one 128 x 128 bf16 operand tile: 32 KiB

enum WaitSite : int {
  kSiteKV = 0x21, kSiteQEmpty, kSiteQFull, kSiteSFull, kSiteDPFull, kSitePFull, kSiteDSFull, kSiteFinal,
  kSiteDrain, kSiteAlign, kSiteStat, kSiteKVFull, kSiteKVEmpty, kSiteQ,
};

struct BwdParams {
  CUtensorMap tq, tk, tv, tdo;
  AttnArgs a;
  int32_t* err;
};

__device__ __forceinline__ int head_of_slot(int slot, const AttnArgs& a) {
  const int G = a.hq / a.hkv;
  const int kv = slot / G, g = slot - kv * G;
  return a.gqa_interleaved ? g * a.hkv + kv : kv * G + g;
}

// ---------------------------------------------------------------------------
// Shared pieces of the compute warps.
// ---------------------------------------------------------------------------

// Loads 64 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void ld64(uint32_t taddr, uint32_t (&x0)[32], uint32_t (&x1)[32]) {
  ptx::tmem_ld32(taddr, x0);
  ptx::tmem_ld32(taddr + 32, x1);
  ptx::tmem_ld_wait();
  ptx::reg_fence32(x0);
  ptx::reg_fence32(x1);
}

__device__ __forceinline__ float pick(const uint32_t (&x0)[32], const uint32_t (&x1)[32], int c) {
  return __uint_as_float(c < 32 ? x0[c] : x1[c - 32]);
}

// Packs 64 floats into 32 bf16 pairs and stores them into 32 TMEM columns.
__device__ __forceinline__ void st_bf16_64(uint32_t taddr, const float (&v)[64]) {
  uint32_t pk[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) pk[j] = ptx::pack_bf16(v[2 * j], v[2 * j + 1]);
  ptx::tmem_st32(taddr, pk);
}

// Stores 128 FP32 TMEM columns of this lane (from column `tcol`, 64 of them
// starting at `c0`) as bf16 into dst[c0 .. c0+63].
__device__ __forceinline__ void store_row_bf16(uint32_t taddr, __nv_bfloat16* dst, bool valid, bool have) {
  uint32_t x0[32], x1[32];
  if (have) {
    ld64(taddr, x0, x1);
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) x0[j] = x1[j] = 0u;
  }
  if (!valid) return;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    uint4 v;
    v.x = ptx::pack_bf16(pick(x0, x1, 8 * k + 0), pick(x0, x1, 8 * k + 1));
    v.y = ptx::pack_bf16(pick(x0, x1, 8 * k + 2), pick(x0, x1, 8 * k + 3));
    v.z = ptx::pack_bf16(pick(x0, x1, 8 * k + 4), pick(x0, x1, 8 * k + 5));
    v.w = ptx::pack_bf16(pick(x0, x1, 8 * k + 6), pick(x0, x1, 8 * k + 7));
    reinterpret_cast<uint4*>(dst)[k] = v;
  }
}

// ===========================================================================
// dK / dV
// ===========================================================================

// Walks the query steps of a key tile: for every query head of the GQA
// group, every query run of the plan, cut into BT-row tiles.
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
  __device__ int row() const { return cur.row0 + off; }
  __device__ int n() const { return min(BT, cur.nrows - off); }
  __device__ int pos() const { return cur.pos0 + off; }
  __device__ void next() {
    off += BT;
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

// Statistic of query column t (0..127: lse * log2e; 128..255: D * scale) of
// the step the cursor points at.
__device__ __forceinline__ float load_stat(const AttnArgs& a, const StepCursor& c, int t) {
  const int col = t & 127;
  if (col >= c.n()) return 0.f;
  const int64_t idx = int64_t(c.head()) * a.T + c.row() + col;
  return t < 128 ? a.lse_in[idx] * kLog2e : a.dpsum[idx] * a.scale;
}

struct DkdvCfg {
  static constexpr int NS = 2;  // stages of (Q, dO)
  static constexpr uint32_t offK = 0;
  static constexpr uint32_t offV = offK + kTileBytes;
  static constexpr uint32_t offQ = offV + kTileBytes;       // NS stages
  static constexpr uint32_t offO = offQ + NS * kTileBytes;  // NS stages
  static constexpr uint32_t offStat = offO + NS * kTileBytes;  // [2][256] floats
  static constexpr uint32_t offBar = offStat + 2 * 256 * 4;
  static constexpr int kNumBars = 1 + 2 * NS + 9;
  static constexpr uint32_t kSmem = offBar + kNumBars * 8 + 16;
  static_assert(kSmem <= 232448, "shared memory budget");
};

__global__ void __launch_bounds__(kThreads, 1) attn_bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
  using Cfg = DkdvCfg;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = ptx::smem_u32(smem);
  const AttnArgs& a = p.a;
  if (sbase & 1023u) {  // the swizzled operand panels need 1024-byte alignment
    if (threadIdx.x == 0 && p.err) atomicCAS(p.err, 0, 0x100 | kSiteAlign);
    return;
  }
  const int tile_idx = blockIdx.x / a.hkv;
  const int kvh = blockIdx.x - tile_idx * a.hkv;
  const TileDesc tile = a.tiles[tile_idx];
  const int G = a.hq / a.hkv;
  const int n_steps = tile.work * G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t bar0 = sbase + Cfg::offBar;
  const uint32_t bar_kv = bar0;
  auto bar_q_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto bar_q_empty = [&](int s) { return bar0 + 8u * (1 + Cfg::NS + s); };
  const uint32_t bar_s_full = bar0 + 8u * (1 + 2 * Cfg::NS);
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
    for (int s = 0; s < Cfg::NS; ++s) {
      ptx::mbar_init(bar_q_full(s), 1);
      ptx::mbar_init(bar_q_empty(s), 1);
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
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const ptx::WaitCtx wctx{abort_flag, p.err, kWaitLimitNs};

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_steps > 0) {
      int issued = 0;
      ptx::mbar_arrive_expect_tx(bar_kv, 2 * kTileBytes);
      for (int c = 0; c < 2; ++c) {
        ptx::tma_load_3d(sbase + Cfg::offK + c * kPanel, &p.tk, bar_kv, c * 64, kvh, tile.row0);
        ptx::tma_load_3d(sbase + Cfg::offV + c * kPanel, &p.tv, bar_kv, c * 64, kvh, tile.row0);
      }
      StepCursor cur;
      cur.init(a.ranges, tile.range_begin, tile.range_count, G, kvh, a.hkv, a.gqa_interleaved);
      for (int i = 0; i < n_steps; ++i, cur.next()) {
        const int s = i % Cfg::NS;
        if (i >= Cfg::NS && !ptx::mbar_wait(bar_q_empty(s), ((i / Cfg::NS) - 1) & 1, kSiteQEmpty, wctx)) break;
        ptx::mbar_arrive_expect_tx(bar_q_full(s), 2 * kTileBytes);
        const int h = cur.head();
        for (int c = 0; c < 2; ++c) {
          ptx::tma_load_3d(sbase + Cfg::offQ + s * kTileBytes + c * kPanel, &p.tq, bar_q_full(s), c * 64, h,
                           cur.row());
          ptx::tma_load_3d(sbase + Cfg::offO + s * kTileBytes + c * kPanel, &p.tdo, bar_q_full(s), c * 64, h,
                           cur.row());
        }
        ++issued;
      }
      if (*abort_flag) {
        volatile int no_abort = 0;
        const ptx::WaitCtx drain{&no_abort, nullptr, kWaitLimitNs};
        ptx::mbar_wait(bar_kv, 0, kSiteDrain, drain);
        for (int i = max(0, issued - Cfg::NS); i < issued; ++i)
          ptx::mbar_wait(bar_q_full(i % Cfg::NS), (i / Cfg::NS) & 1, kSiteDrain, drain);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_steps > 0) {
      constexpr uint32_t idS = ptx::idesc_bf16_f32(BT, BT, false, false);
      constexpr uint32_t idG = ptx::idesc_bf16_f32(BT, D, false, true);  // dV, dK: B MN-major
      const uint32_t tS = tmem, tDP = tmem + 128, tDV = tmem + 256, tDK = tmem + 384;
      const uint32_t kb = sbase + Cfg::offK, vb = sbase + Cfg::offV;
      auto qb = [&](int i) { return sbase + Cfg::offQ + (i % Cfg::NS) * kTileBytes; };
      auto ob = [&](int i) { return sbase + Cfg::offO + (i % Cfg::NS) * kTileBytes; };
      auto issue_ss = [&](uint32_t d, uint32_t abase, uint32_t bbase) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
          ptx::mma_ss(d, ptx::sdesc_sw128(abase + off, 16, 1024), ptx::sdesc_sw128(bbase + off, 16, 1024), idS,
                      kk > 0);
        }
      };
      // dst += (packed bf16 A in TMEM at [a0, a0+32) and [a0+96, a0+128)) x B (MN-major smem)
      auto issue_ts = [&](uint32_t d, uint32_t a0, uint32_t bbase, bool acc) {
#pragma unroll
        for (int kk = 0; kk < BT / 16; ++kk)
          ptx::mma_ts(d, a0 + (kk < 4 ? kk * 8 : 96 + (kk - 4) * 8), ptx::sdesc_sw128(bbase + kk * 2048, kPanel, 1024),
                      idG, (acc || kk > 0));
      };
      bool ok = ptx::mbar_wait(bar_kv, 0, kSiteKV, wctx) && ptx::mbar_wait(bar_q_full(0), 0, kSiteQFull, wctx);
      if (ok) {
        ptx::tc_fence_after();
        issue_ss(tS, kb, qb(0));
        ptx::mma_commit(bar_s_full);
      }
      for (int i = 0; ok && i < n_steps; ++i) {
        // dK(i-1) needs dS(i-1): once it is issued, dP(i) may overwrite tDP
        if (i > 0) {
          if (!ptx::mbar_wait(bar_ds_full, (i - 1) & 1, kSiteDSFull, wctx)) { ok = false; break; }
          ptx::tc_fence_after();
          issue_ts(tDK, tDP, qb(i - 1), i - 1 > 0);
          ptx::mma_commit(bar_q_empty((i - 1) % Cfg::NS));
        }
        issue_ss(tDP, vb, ob(i));
        ptx::mma_commit(bar_dp_full);
        // dV(i) needs P(i); once it is issued, S(i+1) may overwrite tS
        if (!ptx::mbar_wait(bar_p_full, i & 1, kSitePFull, wctx)) { ok = false; break; }
        ptx::tc_fence_after();
        issue_ts(tDV, tS, ob(i), i > 0);
        if (i + 1 < n_steps) {
          if (!ptx::mbar_wait(bar_q_full((i + 1) % Cfg::NS), ((i + 1) / Cfg::NS) & 1, kSiteQFull, wctx)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          issue_ss(tS, kb, qb(i + 1));
          ptx::mma_commit(bar_s_full);
        }
      }
      if (ok) {
        ok = ptx::mbar_wait(bar_ds_full, (n_steps - 1) & 1, kSiteDSFull, wctx);
        if (ok) {
          ptx::tc_fence_after();
          issue_ts(tDK, tDP, qb(n_steps - 1), n_steps - 1 > 0);
          ptx::mma_commit(bar_final);
        }
      }
      if (!ok) {
        volatile int no_abort = 0;
        const ptx::WaitCtx drain{&no_abort, nullptr, kWaitLimitNs};
        ptx::mma_commit(bar_drain);
        ptx::mbar_wait(bar_drain, 0, kSiteDrain, drain);
      }
    }
  } else {
    // ------------------------------------------------------------ compute warps
    const int grp = warp >> 2;               // query columns 64*grp .. 64*grp+63
    const int r = ((warp & 3) << 5) | lane;  // key row = TMEM lane
    const int t = threadIdx.x;               // 0..255, statistics loader index
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base, tDP = tmem + lane_base + 128;
    const uint32_t colS = grp * 64;
    const uint32_t colPk = grp ? 96 : 0;
    const float sl2 = a.scale * kLog2e;
    const int kpos = tile.pos0 + r;
    const int nk = tile.nrows;
    bool ok = true;

    StepCursor cur, nxt;
    cur.init(a.ranges, tile.range_begin, tile.range_count, G, kvh, a.hkv, a.gqa_interleaved);
    nxt = cur;
    if (n_steps > 0) {
      stat[t] = load_stat(a, cur, t);
      ptx::mbar_arrive(bar_stat(0));
    }
    nxt.next();
    for (int i = 0; i < n_steps; ++i, cur.next(), nxt.next()) {
      const int nq = cur.n(), qpos0 = cur.pos();
      const float* sL = stat + (i & 1) * 256;
      const float* sD = sL + 128;
      // statistics of this step are in place (a buffer is refilled only after
      // every compute warp passed the dS phase of the step in between)
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar_stat(i & 1), (i >> 1) & 1, kSiteStat, wctx))) {
        ok = false;
        break;
      }
      const float nstat = (i + 1 < n_steps) ? load_stat(a, nxt, t) : 0.f;
      const bool need_mask = nq < BT || nk < BT || (a.causal && qpos0 < tile.pos0 + BT - 1);
      const int cmin = (a.causal ? kpos - qpos0 : 0) - int(colS);  // first visible column (relative)
      const int cmax = (r < nk ? nq : 0) - int(colS);             // columns [cmin, cmax) are visible

      // ---- P^T = exp(S^T * scale - lse)
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar_s_full, i & 1, kSiteSFull, wctx))) { ok = false; break; }
      ptx::tc_fence_after();
      uint32_t x0[32], x1[32];
      ld64(tS + colS, x0, x1);
      float pf[64];
#pragma unroll
      for (int j = 0; j < 64; j += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(sL + colS + j);
        const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = j + e;
          float pv = ptx::ex2(fmaf(pick(x0, x1, c), sl2, -lv[e]));
          if (need_mask) pv = (c >= cmin && c < cmax) ? pv : 0.f;
          pf[c] = pv;
        }
      }
      st_bf16_64(tS + colPk, pf);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_p_full);

      // ---- dS^T = P^T (dP^T - D) * scale
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar_dp_full, i & 1, kSiteDPFull, wctx))) { ok = false; break; }
      ptx::tc_fence_after();
      ld64(tDP + colS, x0, x1);
#pragma unroll
      for (int j = 0; j < 64; j += 4) {
        const float4 d4 = *reinterpret_cast<const float4*>(sD + colS + j);
        const float dv4[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) pf[j + e] *= fmaf(pick(x0, x1, j + e), a.scale, -dv4[e]);
      }
      st_bf16_64(tDP + colPk, pf);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_ds_full);
      if (i + 1 < n_steps) {
        stat[((i + 1) & 1) * 256 + t] = nstat;
        ptx::mbar_arrive(bar_stat((i + 1) & 1));
      }
    }

    // ------------------------------------------------------------ dK, dV epilogue
    if (ok && n_steps > 0) ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar_final, 0, kSiteFinal, wctx));
    if (ok) {
      ptx::tc_fence_after();
      const int64_t krow = int64_t(tile.row0) + r;
      __nv_bfloat16* dvp = static_cast<__nv_bfloat16*>(a.dv) + (krow * a.hkv + kvh) * D + colS;
      __nv_bfloat16* dkp = static_cast<__nv_bfloat16*>(a.dk) + (krow * a.hkv + kvh) * D + colS;
      store_row_bf16(tmem + lane_base + 256 + colS, dvp, r < nk, n_steps > 0);
      store_row_bf16(tmem + lane_base + 384 + colS, dkp, r < nk, n_steps > 0);
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

struct DqCfg {
  // K(j) is read by S(j) and, one step later in issue order, by dQ(j); V(j)
  // only by dP(j): K gets the deeper ring.
  static constexpr int NSK = 3, NSV = 2;
  static constexpr uint32_t offQ = 0;
  static constexpr uint32_t offO = offQ + kTileBytes;
  static constexpr uint32_t offK = offO + kTileBytes;        // NSK stages
  static constexpr uint32_t offV = offK + NSK * kTileBytes;  // NSV stages
  static constexpr uint32_t offBar = offV + NSV * kTileBytes;
  static constexpr int kNumBars = 1 + 2 * NSK + 2 * NSV + 9;
  static constexpr uint32_t kSmem = offBar + kNumBars * 8 + 16;
  static_assert(kSmem <= 232448, "shared memory budget");
};

__global__ void __launch_bounds__(kThreads, 1) attn_bwd_dq_kernel(const __grid_constant__ BwdParams p) {
  using Cfg = DqCfg;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = ptx::smem_u32(smem);
  const AttnArgs& a = p.a;
  if (sbase & 1023u) {
    if (threadIdx.x == 0 && p.err) atomicCAS(p.err, 0, 0x100 | kSiteAlign);
    return;
  }
  const int tile_idx = blockIdx.x / a.hq;
  const int h = head_of_slot(blockIdx.x - tile_idx * a.hq, a);
  const int kvh = a.gqa_interleaved ? h % a.hkv : h / (a.hq / a.hkv);
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
  const uint32_t bar_dp_read = bar_s_full + 48;                   // compute warps hold dP(j)
  auto bar_dq_done = [&](int b) { return bar_s_full + 56 + 8u * b; };  // dQ(j) read dS buffer b = j & 1
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::offBar + Cfg::kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::offBar + Cfg::kNumBars * 8 + 4);

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar_dp_read, 8);
    ptx::mbar_init(bar_dq_done(0), 1);
    ptx::mbar_init(bar_dq_done(1), 1);
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
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const ptx::WaitCtx wctx{abort_flag, p.err, kWaitLimitNs};

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_kv > 0) {
      int issued = 0;
      ptx::mbar_arrive_expect_tx(bar_q, 2 * kTileBytes);
      for (int c = 0; c < 2; ++c) {
        ptx::tma_load_3d(sbase + Cfg::offQ + c * kPanel, &p.tq, bar_q, c * 64, h, tile.row0);
        ptx::tma_load_3d(sbase + Cfg::offO + c * kPanel, &p.tdo, bar_q, c * 64, h, tile.row0);
      }
      int issued_v = 0;
      KvCursor cur;
      cur.init(a.ranges, tile.range_begin, tile.range_count);
      for (int j = 0; j < n_kv; ++j, cur.next()) {
        const int sk = j % Cfg::NSK, sv = j % Cfg::NSV;
        if (j >= Cfg::NSK && !ptx::mbar_wait(bar_k_empty(sk), ((j / Cfg::NSK) - 1) & 1, kSiteKVEmpty, wctx)) break;
        ptx::mbar_arrive_expect_tx(bar_k_full(sk), kTileBytes);
        for (int c = 0; c < 2; ++c)
          ptx::tma_load_3d(sbase + Cfg::offK + sk * kTileBytes + c * kPanel, &p.tk, bar_k_full(sk), c * 64, kvh,
                           cur.row());
        ++issued;
        if (j >= Cfg::NSV && !ptx::mbar_wait(bar_v_empty(sv), ((j / Cfg::NSV) - 1) & 1, kSiteKVEmpty, wctx)) break;
        ptx::mbar_arrive_expect_tx(bar_v_full(sv), kTileBytes);
        for (int c = 0; c < 2; ++c)
          ptx::tma_load_3d(sbase + Cfg::offV + sv * kTileBytes + c * kPanel, &p.tv, bar_v_full(sv), c * 64, kvh,
                           cur.row());
        ++issued_v;
      }
      if (*abort_flag) {
        volatile int no_abort = 0;
        const ptx::WaitCtx drain{&no_abort, nullptr, kWaitLimitNs};
        ptx::mbar_wait(bar_q, 0, kSiteDrain, drain);
        for (int j = max(0, issued - Cfg::NSK); j < issued; ++j)
          ptx::mbar_wait(bar_k_full(j % Cfg::NSK), (j / Cfg::NSK) & 1, kSiteDrain, drain);
        for (int j = max(0, issued_v - Cfg::NSV); j < issued_v; ++j)
          ptx::mbar_wait(bar_v_full(j % Cfg::NSV), (j / Cfg::NSV) & 1, kSiteDrain, drain);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_kv > 0) {
      constexpr uint32_t idS = ptx::idesc_bf16_f32(BT, BT, false, false);
      constexpr uint32_t idQ = ptx::idesc_bf16_f32(BT, D, false, true);  // dQ: B = K as MN-major
      const uint32_t tS = tmem, tDP = tmem + 128, tDQ = tmem + 256;
      const uint32_t qb = sbase + Cfg::offQ, obb = sbase + Cfg::offO;
      auto kb = [&](int j) { return sbase + Cfg::offK + (j % Cfg::NSK) * kTileBytes; };
      auto vb = [&](int j) { return sbase + Cfg::offV + (j % Cfg::NSV) * kTileBytes; };
      auto issue_ss = [&](uint32_t d, uint32_t abase, uint32_t bbase) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
          ptx::mma_ss(d, ptx::sdesc_sw128(abase + off, 16, 1024), ptx::sdesc_sw128(bbase + off, 16, 1024), idS,
                      kk > 0);
        }
      };
      bool ok = ptx::mbar_wait(bar_q, 0, kSiteQ, wctx) && ptx::mbar_wait(bar_k_full(0), 0, kSiteKVFull, wctx);
      if (ok) {
        ptx::tc_fence_after();
        issue_ss(tS, qb, kb(0));
        ptx::mma_commit(bar_s_full);
        ok = ptx::mbar_wait(bar_v_full(0), 0, kSiteKVFull, wctx);
      }
      if (ok) {
        ptx::tc_fence_after();
        issue_ss(tDP, obb, vb(0));
        ptx::mma_commit(bar_dp_full);
        ptx::mma_commit(bar_v_empty(0));
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        if (j + 1 < n_kv) {
          // S(j+1) as soon as the compute warps have read S(j)
          if (!ptx::mbar_wait(bar_p_full, j & 1, kSitePFull, wctx) ||
              !ptx::mbar_wait(bar_k_full((j + 1) % Cfg::NSK), ((j + 1) / Cfg::NSK) & 1, kSiteKVFull, wctx)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          issue_ss(tS, qb, kb(j + 1));
          ptx::mma_commit(bar_s_full);
          // dP(j+1) as soon as they have read dP(j)
          if (!ptx::mbar_wait(bar_dp_read, j & 1, kSiteDPFull, wctx) ||
              !ptx::mbar_wait(bar_v_full((j + 1) % Cfg::NSV), ((j + 1) / Cfg::NSV) & 1, kSiteKVFull, wctx)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          issue_ss(tDP, obb, vb(j + 1));
          ptx::mma_commit(bar_dp_full);
          ptx::mma_commit(bar_v_empty((j + 1) % Cfg::NSV));
        }
        // dQ(j) += dS(j) K(j), dS(j) in buffer j & 1
        if (!ptx::mbar_wait(bar_ds_full, j & 1, kSiteDSFull, wctx)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t kbj = kb(j);
        const uint32_t tA = tmem + 384 + 64 * (j & 1);
#pragma unroll
        for (int kk = 0; kk < BT / 16; ++kk)
          ptx::mma_ts(tDQ, tA + kk * 8, ptx::sdesc_sw128(kbj + kk * 2048, kPanel, 1024), idQ, (j > 0 || kk > 0));
        ptx::mma_commit(bar_dq_done(j & 1));
        ptx::mma_commit(bar_k_empty(j % Cfg::NSK));
      }
      if (ok) ptx::mma_commit(bar_final);
      if (!ok) {
        volatile int no_abort = 0;
        const ptx::WaitCtx drain{&no_abort, nullptr, kWaitLimitNs};
        ptx::mma_commit(bar_drain);
        ptx::mbar_wait(bar_drain, 0, kSiteDrain, drain);
      }
    }
  } else {
    // ------------------------------------------------------------ compute warps
    const int grp = warp >> 2;               // key columns 64*grp .. 64*grp+63
    const int r = ((warp & 3) << 5) | lane;  // query row = TMEM lane
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base, tDP = tmem + lane_base + 128;
    const uint32_t colS = grp * 64;
    const float sl2 = a.scale * kLog2e;
    const bool row_ok = r < tile.nrows;
    const int qpos = tile.pos0 + r;
    const int64_t qrow = int64_t(tile.row0) + r;
    const float lse2 = row_ok ? a.lse_in[int64_t(h) * a.T + qrow] * kLog2e : 0.f;
    const float dsc = row_ok ? a.dpsum[int64_t(h) * a.T + qrow] * a.scale : 0.f;
    bool ok = true;
    KvCursor cur;
    cur.init(a.ranges, tile.range_begin, tile.range_count);
    for (int j = 0; j < n_kv; ++j, cur.next()) {
      const int kn = cur.n(), kp = cur.pos();
      const bool need_mask = kn < BT || tile.nrows < BT || (a.causal && kp + BT - 1 > tile.pos0);
      int lim = row_ok ? kn : 0;
      if (a.causal) lim = min(lim, qpos - kp + 1);
      lim -= int(colS);  // columns [0, lim) of this group are visible

      // ---- P = exp(S * scale - lse)
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar_s_full, j & 1, kSiteSFull, wctx))) { ok = false; break; }
      ptx::tc_fence_after();
      uint32_t x0[32], x1[32];
      ld64(tS + colS, x0, x1);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_p_full);  // S(j) has been read
      float pf[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        float pv = ptx::ex2(fmaf(pick(x0, x1, c), sl2, -lse2));
        if (need_mask) pv = c < lim ? pv : 0.f;
        pf[c] = pv;
      }
      // ---- dS = P (dP - D) * scale
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar_dp_full, j & 1, kSiteDPFull, wctx))) { ok = false; break; }
      ptx::tc_fence_after();
      ld64(tDP + colS, x0, x1);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_dp_read);  // dP(j) has been read
#pragma unroll
      for (int c = 0; c < 64; ++c) pf[c] *= fmaf(pick(x0, x1, c), a.scale, -dsc);
      // dS buffer j & 1 was last read by dQ(j - 2)
      if (j >= 2 &&
          !__all_sync(0xffffffffu, ptx::mbar_wait(bar_dq_done(j & 1), ((j - 2) >> 1) & 1, kSiteDSFull, wctx))) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      st_bf16_64(tmem + lane_base + 384 + 64 * (j & 1) + 32 * grp, pf);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_ds_full);
    }

    // ------------------------------------------------------------ dQ epilogue
    if (ok && n_kv > 0) ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar_final, 0, kSiteFinal, wctx));
    if (ok) {
      ptx::tc_fence_after();
      __nv_bfloat16* dqp = static_cast<__nv_bfloat16*>(a.dq) + (qrow * a.hq + h) * D + colS;
      store_row_bf16(tmem + lane_base + 256 + colS, dqp, row_ok, n_kv > 0);
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

bool make_maps(BwdParams& p, const AttnArgs& a) {
  return make_map_3d(&p.tq, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.hq, a.T, 64, BT,
                     CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_map_3d(&p.tk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.hkv, a.T, 64, BT,
                     CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_map_3d(&p.tv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.hkv, a.T, 64, BT,
                     CU_TENSOR_MAP_SWIZZLE_128B) &&
         make_map_3d(&p.tdo, a.dout, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.hq, a.T, 64, BT,
                     CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

bool tc_bwd_supported(int32_t d_qk, int32_t d_v) { return d_qk == 128 && d_v == 128; }

cudaError_t launch_tc_bwd_dkdv(const AttnArgs& a, cudaStream_t st) {
  if (a.d_qk != D || a.d_v != D) return cudaErrorInvalidValue;
  BwdParams p;
  p.a = a;
  p.err = device_error_word();
  if (!make_maps(p, a)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(DkdvCfg::kSmem));
  if (e != cudaSuccess) return e;
  const int64_t grid = int64_t(a.num_tiles) * a.hkv;
  if (grid == 0) return cudaSuccess;
  attn_bwd_dkdv_kernel<<<unsigned(grid), kThreads, DkdvCfg::kSmem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_tc_bwd_dq(const AttnArgs& a, cudaStream_t st) {
  if (a.d_qk != D || a.d_v != D) return cudaErrorInvalidValue;
  BwdParams p;
  p.a = a;
  p.err = device_error_word();
  if (!make_maps(p, a)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(DqCfg::kSmem));
  if (e != cudaSuccess) return e;
  const int64_t grid = int64_t(a.num_tiles) * a.hq;
  if (grid == 0) return cudaSuccess;
  attn_bwd_dq_kernel<<<unsigned(grid), kThreads, DqCfg::kSmem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace cpattn
