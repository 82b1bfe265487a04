// attn_bwd_sm103.cu — context-parallel causal attention backward on the
// sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// "Ulysses与Ring-Attention详解" §4.3: the backward recomputes the attention
// probabilities instead of storing them.  They are rebuilt here from q, k and
// the forward's final lse (never from per-block statistics), with
// D = rowsum(dout * o) computed beforehand:
//     P = exp(scale q.k - lse),  dP = dout . v,  dS = P (dP - D)
//     dV += P^T dout,  dK += scale dS^T q,  dQ += scale dS k.
//
// Key-tile-major: one CTA owns a 128-row key/value tile of one kv head and
// visits every query tile that can see it (the plan lists the query runs of
// every virtual rank in ring order, fully masked tiles removed), for every
// query head of the GQA group, so dK/dV are summed in TMEM with no atomics.
// dQ contributions are added to an FP32 accumulator in global memory.
//
// Per query tile (M = 128 keys, N = 128 queries), TMEM columns:
//   [0,128)    S^T = K Q^T (SS MMA); then P^T (bf16) of query columns 0-63 in
//              [0,32) and of 64-127 in [96,128)
//   [128,256)  dP^T = V dO^T (SS MMA); then dS^T (bf16) in [128,160) and
//              [224,256)
//   [32,96)    dQ^T[:, 0:64]   = K^T dS^T[:, 0:64]    (SS MMA, N = 64)
//   [160,224)  dQ^T[:, 64:128] = K^T dS^T[:, 64:128]
//   [256,384)  dV += P^T dO    (TS MMA: A read from TMEM)
//   [384,512)  dK += dS^T Q    (TS MMA)
// Two groups of four compute warps split the query columns (group g owns
// columns 64g..64g+63); each writes its bf16 results only into TMEM columns
// it has already read, so the groups never wait for each other.  The MMA
// warp issues dV as soon as P is ready (while dS is being computed) and
// orders dQ^T[:, 0:64] before dK so group 0 reads it out during dK.
//
// Roles (320 threads): warps 0-7 compute (thread = key row = TMEM lane for
// S^T/dP^T, head-dim index for dQ^T), warp 8 TMA producer, warp 9 TMEM
// allocator + MMA issuer.
#include <cuda.h>
#include <cuda_bf16.h>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace cpattn {

bool make_map_3d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elt, int64_t dim, int64_t heads,
                 int64_t T, int box_inner, int box_rows, CUtensorMapSwizzle swz);

namespace {

constexpr int BM = 128;  // key rows per CTA
constexpr int BN = 128;  // query rows per step
constexpr uint32_t kPanel = 128 * 128;  // 128 rows x 64 bf16 columns, 128-byte swizzled: 16 KiB
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr int kComputeThreads = 256;
constexpr int kThreads = kComputeThreads + 64;

enum WaitSite : int {
  kSiteKV = 0x21, kSiteQEmpty, kSiteQFull, kSiteSFree, kSiteDPFree, kSiteSFull, kSiteDPFull, kSitePFull,
  kSiteDSFull, kSiteH0, kSiteH1, kSiteDrain, kSiteAlign, kSiteStat,
};

template <int DQK, int DV>
struct BwdCfg {
  static constexpr int kQPanels = DQK / 64;
  static constexpr int kVPanels = DV / 64;
  static constexpr int NS = 2;  // stages of (Q, dO)
  static constexpr uint32_t kKBytes = kQPanels * kPanel;
  static constexpr uint32_t kVBytes = kVPanels * kPanel;
  static constexpr uint32_t kQBytes = kQPanels * kPanel;
  static constexpr uint32_t kOBytes = kVPanels * kPanel;
  static constexpr uint32_t kDSBytes = (BN / 64) * kPanel;
  static constexpr uint32_t offK = 0;
  static constexpr uint32_t offV = offK + kKBytes;
  static constexpr uint32_t offQ = offV + kVBytes;       // NS stages of Q
  static constexpr uint32_t offO = offQ + NS * kQBytes;  // NS stages of dO
  static constexpr uint32_t offDS = offO + NS * kOBytes;
  static constexpr uint32_t offStat = offDS + kDSBytes;  // [2][256] floats: lse*log2e | D*scale
  static constexpr uint32_t offBar = offStat + 2 * 256 * 4;
  static constexpr int kNumBars = 1 + 2 * NS + 12;
  static constexpr uint32_t kSmem = offBar + kNumBars * 8 + 16;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(DQK == 128 && DV == 128, "TMEM plan is laid out for 128-wide heads");
  static_assert(kSmem <= 232448, "shared memory budget");
};

struct BwdParams {
  CUtensorMap tq, tk, tv, tdo;
  AttnArgs a;
  int32_t* err;
};

// Walks the query steps of a key tile: for every query head of the GQA
// group, every query run of the plan, cut into BN-row tiles.
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
  __device__ int n() const { return min(BN, cur.nrows - off); }
  __device__ int pos() const { return cur.pos0 + off; }
  __device__ void next() {
    off += BN;
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

// Statistic of query column t (0..127: lse * log2e; 128..255: D * scale)
// for the step the cursor points at.
__device__ __forceinline__ float load_stat(const AttnArgs& a, const StepCursor& c, int t) {
  const int col = t & 127;
  if (col >= c.n()) return 0.f;
  const int64_t idx = int64_t(c.head()) * a.T + c.row() + col;
  return t < 128 ? a.lse_in[idx] * kLog2e : a.dpsum[idx] * a.scale;
}

template <int DQK, int DV>
__global__ void __launch_bounds__(kThreads, 1) attn_bwd_tc_kernel(const __grid_constant__ BwdParams p) {
  using Cfg = BwdCfg<DQK, DV>;
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
  const uint32_t bar_h0 = bar_s_full + 32;
  const uint32_t bar_h1 = bar_s_full + 40;
  const uint32_t bar_s_free = bar_s_full + 48;
  const uint32_t bar_dp_free = bar_s_full + 56;
  const uint32_t bar_drain = bar_s_full + 64;
  // statistics double buffer b is full (256 arrivals); its k-th fill is for step 2k + b
  auto bar_stat = [&](int b) { return bar_s_full + 72 + 8u * b; };
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
    ptx::mbar_init(bar_h0, 1);
    ptx::mbar_init(bar_h1, 1);
    ptx::mbar_init(bar_s_free, 4);
    ptx::mbar_init(bar_dp_free, 4);
    ptx::mbar_init(bar_drain, 1);
    ptx::mbar_init(bar_stat(0), kComputeThreads);
    ptx::mbar_init(bar_stat(1), kComputeThreads);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 9) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), Cfg::kTmemCols);
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
      ptx::mbar_arrive_expect_tx(bar_kv, Cfg::kKBytes + Cfg::kVBytes);
      for (int c = 0; c < Cfg::kQPanels; ++c)
        ptx::tma_load_3d(sbase + Cfg::offK + c * kPanel, &p.tk, bar_kv, c * 64, kvh, tile.row0);
      for (int c = 0; c < Cfg::kVPanels; ++c)
        ptx::tma_load_3d(sbase + Cfg::offV + c * kPanel, &p.tv, bar_kv, c * 64, kvh, tile.row0);
      StepCursor cur;
      cur.init(a.ranges, tile.range_begin, tile.range_count, G, kvh, a.hkv, a.gqa_interleaved);
      for (int i = 0; i < n_steps; ++i, cur.next()) {
        const int s = i % Cfg::NS;
        if (i >= Cfg::NS && !ptx::mbar_wait(bar_q_empty(s), ((i / Cfg::NS) - 1) & 1, kSiteQEmpty, wctx)) break;
        ptx::mbar_arrive_expect_tx(bar_q_full(s), Cfg::kQBytes + Cfg::kOBytes);
        const int h = cur.head();
        for (int c = 0; c < Cfg::kQPanels; ++c)
          ptx::tma_load_3d(sbase + Cfg::offQ + s * Cfg::kQBytes + c * kPanel, &p.tq, bar_q_full(s), c * 64, h,
                           cur.row());
        for (int c = 0; c < Cfg::kVPanels; ++c)
          ptx::tma_load_3d(sbase + Cfg::offO + s * Cfg::kOBytes + c * kPanel, &p.tdo, bar_q_full(s), c * 64, h,
                           cur.row());
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
      constexpr uint32_t idS = ptx::idesc_bf16_f32(BM, BN, false, false);
      constexpr uint32_t idDV = ptx::idesc_bf16_f32(BM, DV, false, true);
      constexpr uint32_t idDK = ptx::idesc_bf16_f32(BM, DQK, false, true);
      constexpr uint32_t idDQ = ptx::idesc_bf16_f32(128, 64, true, true);  // M = head dim 128, N = 64 queries
      const uint32_t tS = tmem, tDP = tmem + 128, tDV = tmem + 256, tDK = tmem + 256 + DV;
      const uint32_t kb = sbase + Cfg::offK, vb = sbase + Cfg::offV, dsb = sbase + Cfg::offDS;
      bool ok = ptx::mbar_wait(bar_kv, 0, kSiteKV, wctx);
      for (int i = 0; ok && i < n_steps; ++i) {
        const int s = i % Cfg::NS;
        const uint32_t qb = sbase + Cfg::offQ + s * Cfg::kQBytes;
        const uint32_t ob = sbase + Cfg::offO + s * Cfg::kOBytes;
        ok = ptx::mbar_wait(bar_q_full(s), (i / Cfg::NS) & 1, kSiteQFull, wctx);
        if (ok && i > 0) ok = ptx::mbar_wait(bar_s_free, (i - 1) & 1, kSiteSFree, wctx);
        if (!ok) break;
        ptx::tc_fence_after();
        // S^T = K Q^T
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
          ptx::mma_ss(tS, ptx::sdesc_sw128(kb + off, 16, 1024), ptx::sdesc_sw128(qb + off, 16, 1024), idS, kk > 0);
        }
        ptx::mma_commit(bar_s_full);
        if (i > 0 && !ptx::mbar_wait(bar_dp_free, (i - 1) & 1, kSiteDPFree, wctx)) { ok = false; break; }
        ptx::tc_fence_after();
        // dP^T = V dO^T
#pragma unroll
        for (int kk = 0; kk < DV / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
          ptx::mma_ss(tDP, ptx::sdesc_sw128(vb + off, 16, 1024), ptx::sdesc_sw128(ob + off, 16, 1024), idS, kk > 0);
        }
        ptx::mma_commit(bar_dp_full);
        // dV += P^T dO  (P^T of query columns 0-63 at [0,32), 64-127 at [96,128))
        if (!ptx::mbar_wait(bar_p_full, i & 1, kSitePFull, wctx)) { ok = false; break; }
        ptx::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          ptx::mma_ts(tDV, tS + (kk < 4 ? kk * 8 : 96 + (kk - 4) * 8),
                      ptx::sdesc_sw128(ob + kk * 2048, kPanel, 1024), idDV, (i > 0 || kk > 0));
        if (!ptx::mbar_wait(bar_ds_full, i & 1, kSiteDSFull, wctx)) { ok = false; break; }
        ptx::tc_fence_after();
        // dQ^T[:, 0:64] = K^T dS^T[:, 0:64] -> [32, 96)
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)
          ptx::mma_ss(tS + 32, ptx::sdesc_sw128(kb + kk * 2048, kPanel, 1024),
                      ptx::sdesc_sw128(dsb + kk * 2048, kPanel, 1024), idDQ, kk > 0);
        ptx::mma_commit(bar_h0);
        // dK += dS^T Q  (dS^T of query columns 0-63 at [128,160), 64-127 at [224,256))
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          ptx::mma_ts(tDK, tDP + (kk < 4 ? kk * 8 : 96 + (kk - 4) * 8),
                      ptx::sdesc_sw128(qb + kk * 2048, kPanel, 1024), idDK, (i > 0 || kk > 0));
        // dQ^T[:, 64:128] = K^T dS^T[:, 64:128] -> [160, 224)
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)
          ptx::mma_ss(tDP + 32, ptx::sdesc_sw128(kb + kk * 2048, kPanel, 1024),
                      ptx::sdesc_sw128(dsb + kPanel + kk * 2048, kPanel, 1024), idDQ, kk > 0);
        ptx::mma_commit(bar_h1);
        ptx::mma_commit(bar_q_empty(s));
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
    const int grp = warp >> 2;                    // query columns 64*grp .. 64*grp+63
    const int r = ((warp & 3) << 5) | lane;       // key row = TMEM lane
    const int t = threadIdx.x;                    // 0..255 (statistics loader index)
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base, tDP = tmem + lane_base + 128;
    const uint32_t colS = grp * 64;               // this group's S^T / dP^T columns
    const uint32_t colPk = grp ? 96 : 0;          // where its packed bf16 P^T / dS^T go
    const float sl2 = a.scale * kLog2e;
    const int kpos = tile.pos0 + r;
    const int nk = tile.nrows;
    uint8_t* dsrow = smem + Cfg::offDS + grp * kPanel + r * 128;
    const int sw = r & 7;
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
      const int h = cur.head(), qrow0 = cur.row(), nq = cur.n(), qpos0 = cur.pos();
      const float* sL = stat + (i & 1) * 256;
      const float* sD = sL + 128;
      // this step's statistics are in place (a buffer is refilled only after
      // every compute warp passed the dS phase of the step in between)
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar_stat(i & 1), (i >> 1) & 1, kSiteStat, wctx))) {
        ok = false;
        break;
      }
      // prefetch the next step's statistics (stored at the end of this step)
      const float nstat = (i + 1 < n_steps) ? load_stat(a, nxt, t) : 0.f;

      const bool need_mask = nq < BN || nk < BM || (a.causal && qpos0 < tile.pos0 + BM - 1);
      const int cmin = (a.causal ? kpos - qpos0 : 0) - int(colS);  // relative to this group's columns
      const int cmax = (r < nk ? nq : 0) - int(colS);

      // ---- P^T = exp(S^T * scale - lse)
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar_s_full, i & 1, kSiteSFull, wctx))) { ok = false; break; }
      ptx::tc_fence_after();
      uint32_t x0[32], x1[32];
      ptx::tmem_ld32(tS + colS, x0);
      ptx::tmem_ld32(tS + colS + 32, x1);
      ptx::tmem_ld_wait();
      ptx::reg_fence32(x0);
      ptx::reg_fence32(x1);
      float pf[64];
#pragma unroll
      for (int j = 0; j < 64; j += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(sL + colS + j);
        const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = j + e;
          const float s = __uint_as_float(c < 32 ? x0[c] : x1[c - 32]);
          float pv = ptx::ex2(fmaf(s, sl2, -lv[e]));
          if (need_mask) pv = (c >= cmin && c < cmax) ? pv : 0.f;
          pf[c] = pv;
        }
      }
      uint32_t pk[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) pk[j] = ptx::pack_bf16(pf[2 * j], pf[2 * j + 1]);
      ptx::tmem_st32(tS + colPk, pk);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_p_full);

      // ---- dS^T = P^T (dP^T - D) * scale
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar_dp_full, i & 1, kSiteDPFull, wctx))) { ok = false; break; }
      ptx::tc_fence_after();
      ptx::tmem_ld32(tDP + colS, x0);
      ptx::tmem_ld32(tDP + colS + 32, x1);
      ptx::tmem_ld_wait();
      ptx::reg_fence32(x0);
      ptx::reg_fence32(x1);
#pragma unroll
      for (int j = 0; j < 64; j += 4) {
        const float4 d4 = *reinterpret_cast<const float4*>(sD + colS + j);
        const float dv4[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = j + e;
          const float dp = __uint_as_float(c < 32 ? x0[c] : x1[c - 32]);
          pf[c] = pf[c] * fmaf(dp, a.scale, -dv4[e]);
        }
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) pk[j] = ptx::pack_bf16(pf[2 * j], pf[2 * j + 1]);
      ptx::tmem_st32(tDP + colPk, pk);
      // dS^T row into this group's swizzled [key][query] panel
#pragma unroll
      for (int k = 0; k < 8; ++k)
        *reinterpret_cast<uint4*>(dsrow + ((k ^ sw) << 4)) = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
      ptx::tmem_st_wait();
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_ds_full);

      // ---- dQ^T (lane = head-dim index) for this group's 64 queries -> global
      const uint32_t bar_h = grp ? bar_h1 : bar_h0;
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar_h, i & 1, grp ? kSiteH1 : kSiteH0, wctx))) { ok = false; break; }
      ptx::tc_fence_after();
      const uint32_t tq = (grp ? tDP : tS) + 32;
      ptx::tmem_ld32(tq, x0);
      ptx::tmem_ld32(tq + 32, x1);
      ptx::tmem_ld_wait();
      ptx::reg_fence32(x0);
      ptx::reg_fence32(x1);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(grp ? bar_dp_free : bar_s_free);
      {
        const int64_t qstride = int64_t(a.hq) * DQK;
        float* dqp = a.dq_acc + (int64_t(qrow0 + colS) * a.hq + h) * DQK + r;
        const int lim = nq - int(colS);
#pragma unroll
        for (int j = 0; j < 64; ++j)
          if (j < lim) ptx::red_add_f32(dqp + j * qstride, __uint_as_float(j < 32 ? x0[j] : x1[j - 32]));
      }
      if (i + 1 < n_steps) {
        stat[((i + 1) & 1) * 256 + t] = nstat;
        ptx::mbar_arrive(bar_stat((i + 1) & 1));
      }
    }

    // ------------------------------------------------------------ dK, dV epilogue
    if (ok && n_steps > 0)
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar_h1, (n_steps - 1) & 1, kSiteH1, wctx));
    if (ok) {
      ptx::tc_fence_after();
      const int64_t krow = int64_t(tile.row0) + r;
      // group 0 writes dV, group 1 writes dK
      const int ncols = grp ? DQK : DV;
      const uint32_t tcol = grp ? 256 + DV : 256;
      __nv_bfloat16* dst = grp ? static_cast<__nv_bfloat16*>(a.dk) + (krow * a.hkv + kvh) * DQK
                               : static_cast<__nv_bfloat16*>(a.dv) + (krow * a.hkv + kvh) * DV;
      for (int c = 0; c < ncols / 32; ++c) {
        uint32_t x[32];
        if (n_steps > 0) {
          ptx::tmem_ld32(tmem + lane_base + tcol + c * 32, x);
          ptx::tmem_ld_wait();
          ptx::reg_fence32(x);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) x[j] = 0u;
        }
        if (r < nk) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 v;
            v.x = ptx::pack_bf16(__uint_as_float(x[8 * k + 0]), __uint_as_float(x[8 * k + 1]));
            v.y = ptx::pack_bf16(__uint_as_float(x[8 * k + 2]), __uint_as_float(x[8 * k + 3]));
            v.z = ptx::pack_bf16(__uint_as_float(x[8 * k + 4]), __uint_as_float(x[8 * k + 5]));
            v.w = ptx::pack_bf16(__uint_as_float(x[8 * k + 6]), __uint_as_float(x[8 * k + 7]));
            reinterpret_cast<uint4*>(dst + c * 32)[k] = v;
          }
        }
      }
    }
  }

  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

}  // namespace

bool tc_bwd_supported(int32_t d_qk, int32_t d_v) { return d_qk == 128 && d_v == 128; }

template <int DQK, int DV>
static cudaError_t launch_bwd_impl(const AttnArgs& a, cudaStream_t st) {
  using Cfg = BwdCfg<DQK, DV>;
  BwdParams p;
  p.a = a;
  p.err = device_error_word();
  if (!make_map_3d(&p.tq, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DQK, a.hq, a.T, 64, BN,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_3d(&p.tk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DQK, a.hkv, a.T, 64, BM,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_3d(&p.tv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DV, a.hkv, a.T, 64, BM,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_3d(&p.tdo, a.dout, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DV, a.hq, a.T, 64, BN,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_tc_kernel<DQK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(Cfg::kSmem));
  if (e != cudaSuccess) return e;
  const int64_t grid = int64_t(a.num_tiles) * a.hkv;
  if (grid == 0) return cudaSuccess;
  attn_bwd_tc_kernel<DQK, DV><<<unsigned(grid), kThreads, Cfg::kSmem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_tc_bwd(const AttnArgs& a, cudaStream_t st) {
  if (a.d_qk == 128 && a.d_v == 128) return launch_bwd_impl<128, 128>(a, st);
  return cudaErrorInvalidValue;
}

}  // namespace cpattn
