// attn_fwd_sm103.cu — fused context-parallel causal attention forward on the
// sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// One CTA computes one 128-row query tile of one head against every key run
// of its plan entry: the KV shards in ring order r, r-1, ..., r-C+1 (mod C),
// fully masked tiles already removed on the host ("超长上下文训练速度翻倍秘籍"
// §2 pitfall 1: the diagonal block is causal, earlier shards unmasked;
// "LLM context parallel production guide", 因果 Attention 会制造 Rank 负载不均:
// blocks above the diagonal are skipped).  The per-block (out, lse) merge of
// "Ulysses与Ring-Attention详解" §4.1-§4.2 happens on chip: the running row
// maximum and sum rescale the TMEM output accumulator, so the result equals
// merging every block's partial exactly.
//
// Roles (192 threads):
//   warps 0-3  softmax: thread t owns query row t = TMEM lane t.  Loads S from
//              TMEM, masks, exponentiates, writes P (bf16) to shared memory,
//              rescales O in TMEM when its reference maximum moves, and
//              finally normalises O and writes o / lse.
//   warp 4     TMA producer: Q once, then K and V tiles into two rings.
//   warp 5     TMEM allocator and MMA issuer: S = Q K^T, O += P V.
// Shared memory holds every operand in the 128-byte-swizzled K-major layout
// TMA writes (V is read as an MN-major operand of the same layout).
#include <cuda.h>
#include <cuda_bf16.h>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace cpattn {

namespace {

constexpr int BM = 128;  // query rows per CTA
constexpr int BN = 128;  // key rows per step
constexpr uint32_t kSubTile = 128 * 128;  // one 128-row x 64-column bf16 swizzle panel: 16 KiB
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P stays below 2^8
constexpr uint64_t kWaitLimitNs = 2000000000ull;

enum WaitSite : int {
  kSiteQ = 1, kSiteKEmpty, kSiteVEmpty, kSiteKFull, kSiteSFree, kSitePFull, kSiteVFull,
  kSiteSFull, kSiteOFull, kSiteDrain, kSiteAlign,
};

template <int DQK, int DV>
struct FwdCfg {
  static constexpr int kQPanels = DQK / 64;
  static constexpr int kVPanels = DV / 64;
  static constexpr int NSK = DQK <= 128 ? 2 : 2;
  static constexpr int NSV = DQK <= 128 ? 2 : 1;
  static constexpr uint32_t kQBytes = kQPanels * kSubTile;
  static constexpr uint32_t kKBytes = kQPanels * kSubTile;
  static constexpr uint32_t kVBytes = kVPanels * kSubTile;
  static constexpr uint32_t kPBytes = (BN / 64) * kSubTile;
  static constexpr uint32_t offQ = 0;
  static constexpr uint32_t offK = offQ + kQBytes;
  static constexpr uint32_t offV = offK + NSK * kKBytes;
  static constexpr uint32_t offP = offV + NSV * kVBytes;
  static constexpr uint32_t offBar = offP + kPBytes;
  static constexpr int kNumBars = 1 + 2 * NSK + 2 * NSV + 5;
  static constexpr uint32_t kSmem = offBar + kNumBars * 8 + 16;
  static constexpr uint32_t kSmemAlloc = kSmem + 1024;  // slack to 1024-align the base
  static constexpr uint32_t kTmemCols = 256;           // S: 128 columns, O: DV columns
  static constexpr uint32_t tS = 0;
  static constexpr uint32_t tO = 128;
  static_assert(128 + DV <= kTmemCols, "TMEM budget");
  static_assert(kSmemAlloc <= 232448, "shared memory budget");
};

struct FwdParams {
  CUtensorMap tq, tk, tv;
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
  // Current tile: first row, rows, position of the first row.
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

__device__ __forceinline__ int head_of_slot(int slot, const AttnArgs& a) {
  const int G = a.hq / a.hkv;
  const int kv = slot / G, g = slot - kv * G;
  return a.gqa_interleaved ? g * a.hkv + kv : kv * G + g;
}

template <int DQK, int DV>
__global__ void __launch_bounds__(192, 1) attn_fwd_tc_kernel(const __grid_constant__ FwdParams p) {
  using Cfg = FwdCfg<DQK, DV>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const AttnArgs& a = p.a;

  const int tile_idx = blockIdx.x / a.hq;
  const int h = head_of_slot(blockIdx.x - tile_idx * a.hq, a);
  const int kvh = a.gqa_interleaved ? h % a.hkv : h / (a.hq / a.hkv);
  const TileDesc tile = a.tiles[tile_idx];
  const int n_kv = tile.work;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // barriers
  const uint32_t bar0 = sbase + Cfg::offBar;
  const uint32_t bar_q = bar0;
  auto bar_k_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto bar_k_empty = [&](int s) { return bar0 + 8u * (1 + Cfg::NSK + s); };
  auto bar_v_full = [&](int s) { return bar0 + 8u * (1 + 2 * Cfg::NSK + s); };
  auto bar_v_empty = [&](int s) { return bar0 + 8u * (1 + 2 * Cfg::NSK + Cfg::NSV + s); };
  const uint32_t bar_s_full = bar0 + 8u * (1 + 2 * Cfg::NSK + 2 * Cfg::NSV);
  const uint32_t bar_s_free = bar_s_full + 8;
  const uint32_t bar_p_full = bar_s_full + 16;
  const uint32_t bar_o_full = bar_s_full + 24;
  const uint32_t bar_drain = bar_s_full + 32;
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
    ptx::mbar_init(bar_s_free, 4);
    ptx::mbar_init(bar_p_full, 4);
    ptx::mbar_init(bar_o_full, 1);
    ptx::mbar_init(bar_drain, 1);
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
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const ptx::WaitCtx wctx{abort_flag, p.err, kWaitLimitNs};

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    int issued_k = 0, issued_v = 0;
    if (lane == 0 && n_kv > 0) {
      ptx::mbar_arrive_expect_tx(bar_q, Cfg::kQBytes);
      for (int c = 0; c < Cfg::kQPanels; ++c)
        ptx::tma_load_3d(sbase + Cfg::offQ + c * kSubTile, &p.tq, bar_q, c * 64, h, tile.row0);
      KvCursor cur;
      cur.init(a.ranges, tile.range_begin, tile.range_count);
      for (int j = 0; j < n_kv; ++j, cur.next()) {
        const int sk = j % Cfg::NSK;
        if (j >= Cfg::NSK && !ptx::mbar_wait(bar_k_empty(sk), ((j / Cfg::NSK) - 1) & 1, kSiteKEmpty, wctx)) break;
        ptx::mbar_arrive_expect_tx(bar_k_full(sk), Cfg::kKBytes);
        for (int c = 0; c < Cfg::kQPanels; ++c)
          ptx::tma_load_3d(sbase + Cfg::offK + sk * Cfg::kKBytes + c * kSubTile, &p.tk, bar_k_full(sk), c * 64,
                           kvh, cur.row());
        ++issued_k;
        const int sv = j % Cfg::NSV;
        if (j >= Cfg::NSV && !ptx::mbar_wait(bar_v_empty(sv), ((j / Cfg::NSV) - 1) & 1, kSiteVEmpty, wctx)) break;
        ptx::mbar_arrive_expect_tx(bar_v_full(sv), Cfg::kVBytes);
        for (int c = 0; c < Cfg::kVPanels; ++c)
          ptx::tma_load_3d(sbase + Cfg::offV + sv * Cfg::kVBytes + c * kSubTile, &p.tv, bar_v_full(sv), c * 64,
                           kvh, cur.row());
        ++issued_v;
      }
      if (*abort_flag) {
        // Let every copy still in flight land before the CTA exits.
        volatile int no_abort = 0;
        const ptx::WaitCtx drain{&no_abort, nullptr, kWaitLimitNs};
        ptx::mbar_wait(bar_q, 0, kSiteDrain, drain);
        for (int j = max(0, issued_k - Cfg::NSK); j < issued_k; ++j)
          ptx::mbar_wait(bar_k_full(j % Cfg::NSK), (j / Cfg::NSK) & 1, kSiteDrain, drain);
        for (int j = max(0, issued_v - Cfg::NSV); j < issued_v; ++j)
          ptx::mbar_wait(bar_v_full(j % Cfg::NSV), (j / Cfg::NSV) & 1, kSiteDrain, drain);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_kv > 0) {
      constexpr uint32_t idS = ptx::idesc_bf16_f32(BM, BN, false, false);
      constexpr uint32_t idO = ptx::idesc_bf16_f32(BM, DV, false, true);
      const uint32_t tS = tmem + Cfg::tS, tO = tmem + Cfg::tO;
      auto issue_s = [&](int j) {
        const int sk = j % Cfg::NSK;
        const uint32_t kb = sbase + Cfg::offK + sk * Cfg::kKBytes;
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kSubTile + (kk & 3) * 32;
          ptx::mma_ss(tS, ptx::sdesc_sw128(sbase + Cfg::offQ + off, 16, 1024), ptx::sdesc_sw128(kb + off, 16, 1024),
                      idS, kk > 0);
        }
        ptx::mma_commit(bar_s_full);
        ptx::mma_commit(bar_k_empty(sk));
      };
      bool ok = ptx::mbar_wait(bar_q, 0, kSiteQ, wctx) && ptx::mbar_wait(bar_k_full(0), 0, kSiteKFull, wctx);
      if (ok) {
        ptx::tc_fence_after();
        issue_s(0);
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        if (j + 1 < n_kv) {
          const int sk = (j + 1) % Cfg::NSK;
          ok = ptx::mbar_wait(bar_k_full(sk), ((j + 1) / Cfg::NSK) & 1, kSiteKFull, wctx) &&
               ptx::mbar_wait(bar_s_free, j & 1, kSiteSFree, wctx);
          if (!ok) break;
          ptx::tc_fence_after();
          issue_s(j + 1);
        }
        const int sv = j % Cfg::NSV;
        ok = ptx::mbar_wait(bar_p_full, j & 1, kSitePFull, wctx) &&
             ptx::mbar_wait(bar_v_full(sv), (j / Cfg::NSV) & 1, kSiteVFull, wctx);
        if (!ok) break;
        ptx::tc_fence_after();
        const uint32_t vb = sbase + Cfg::offV + sv * Cfg::kVBytes;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint32_t poff = (kk >> 2) * kSubTile + (kk & 3) * 32;
          ptx::mma_ss(tO, ptx::sdesc_sw128(sbase + Cfg::offP + poff, 16, 1024),
                      ptx::sdesc_sw128(vb + kk * 2048, kSubTile, 1024), idO, (j > 0 || kk > 0));
        }
        ptx::mma_commit(bar_o_full);
        ptx::mma_commit(bar_v_empty(sv));
      }
      if (!ok) {
        // Wait for every MMA already issued before TMEM is released.
        volatile int no_abort = 0;
        const ptx::WaitCtx drain{&no_abort, nullptr, kWaitLimitNs};
        ptx::mma_commit(bar_drain);
        ptx::mbar_wait(bar_drain, 0, kSiteDrain, drain);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int row = threadIdx.x;  // 0..127, TMEM lane
    const uint32_t lane_base = uint32_t(warp * 32) << 16;
    const uint32_t tS = tmem + lane_base + Cfg::tS, tO = tmem + lane_base + Cfg::tO;
    const float sl2 = a.scale * kLog2e;
    const int qpos = tile.pos0 + row;
    float m_ref = -INFINITY;  // reference maximum of scale*log2e*s (log2 units)
    float l = 0.f;
    bool ok = true;
    uint8_t* prow = smem + Cfg::offP + row * 128;
    const int sw = row & 7;
    KvCursor cur;
    cur.init(a.ranges, tile.range_begin, tile.range_count);
    for (int j = 0; j < n_kv; ++j, cur.next()) {
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar_s_full, j & 1, kSiteSFull, wctx))) { ok = false; break; }
      ptx::tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) ptx::tmem_ld32(tS + c * 32, sr[c]);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 4; ++c) ptx::reg_fence32(sr[c]);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_s_free);

      // mask: columns at or beyond `lim` are not visible to this row
      const int kn = cur.n(), kp = cur.pos();
      int lim = kn;
      if (a.causal) lim = min(lim, qpos - kp + 1);
      float mx = -INFINITY;
      if (lim < BN) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float s = c * 32 + i < lim ? __uint_as_float(sr[c][i]) : -INFINITY;
            sr[c][i] = __float_as_uint(s);
            mx = fmaxf(mx, s);
          }
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) mx = fmaxf(mx, __uint_as_float(sr[c][i]));
      }
      const float m_new = mx * sl2;
      float alpha = 1.f;
      if (m_new > m_ref + kRescaleThreshold || (m_ref == -INFINITY && m_new != -INFINITY)) {
        alpha = ptx::ex2(m_ref - m_new);  // 0 when m_ref = -inf
        m_ref = m_new;
      }
      const float mref = m_ref == -INFINITY ? 0.f : m_ref;
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float e = ptx::ex2(fmaf(__uint_as_float(sr[c][i]), sl2, -mref));
          rs += e;
          sr[c][i] = __float_as_uint(e);
        }
      l = l * alpha + rs;

      // O and the P buffer are free once the previous P.V is done.
      if (j > 0) {
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar_o_full, (j - 1) & 1, kSiteOFull, wctx))) { ok = false; break; }
        ptx::tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < DV / 32; ++c) {
            uint32_t o[32];
            ptx::tmem_ld32(tO + c * 32, o);
            ptx::tmem_ld_wait();
            ptx::reg_fence32(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            ptx::tmem_st32(tO + c * 32, o);
          }
          ptx::tmem_st_wait();
        }
      }
      // P (bf16) into the swizzled K-major panels: 16-byte chunk k of this
      // row's 128-byte line sits at chunk position k ^ (row % 8).
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint4 v;
          v.x = ptx::pack_bf16(__uint_as_float(sr[c][8 * k + 0]), __uint_as_float(sr[c][8 * k + 1]));
          v.y = ptx::pack_bf16(__uint_as_float(sr[c][8 * k + 2]), __uint_as_float(sr[c][8 * k + 3]));
          v.z = ptx::pack_bf16(__uint_as_float(sr[c][8 * k + 4]), __uint_as_float(sr[c][8 * k + 5]));
          v.w = ptx::pack_bf16(__uint_as_float(sr[c][8 * k + 6]), __uint_as_float(sr[c][8 * k + 7]));
          const int chunk = (c & 1) * 4 + k;  // chunk inside the 64-column panel
          *reinterpret_cast<uint4*>(prow + (c >> 1) * kSubTile + ((chunk ^ sw) << 4)) = v;
        }
      }
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_p_full);
    }

    // ------------------------------------------------------------ epilogue
    if (ok && n_kv > 0) ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar_o_full, (n_kv - 1) & 1, kSiteOFull, wctx));
    if (ok) {
      ptx::tc_fence_after();
      const bool valid = row < tile.nrows;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int64_t orow = a.block_mode ? int64_t(tile.out_row0) + row : int64_t(tile.row0) + row;
#pragma unroll
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
        if (valid) {
          if (a.block_mode) {
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
      if (valid) a.lse[int64_t(h) * a.lse_stride + orow] = l > 0.f ? m_ref * kLn2 + logf(l) : -INFINITY;
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

// ---------------------------------------------------------------------------
// Head-pair forward: one CTA computes the same 128 query rows for two query
// heads of one GQA group.  Both share every K/V tile (one TMA load feeds two
// QK^T and two PV products), each head has its own softmax warpgroup, and P
// goes back into TMEM over its S columns to be the A operand of a TS MMA
// (no shared-memory round trip).  TMEM: S_A [0,128) (P_A bf16 in [0,64)),
// O_A [128,256), S_B [256,384), O_B [384,512).  MMA order
//   ... PV_A(j), S_A(j+1), PV_B(j), S_B(j+1) ...
// so one warpgroup's softmax always overlaps the other head's MMAs.  S_X(j)
// completing implies PV_X(j-1) completed (one issuing thread, in order), so a
// warpgroup may rescale O_X and overwrite P_X as soon as it sees S_X(j).
// Roles (320 threads): warps 0-3 head A, warps 4-7 head B, warp 8 TMA
// producer, warp 9 TMEM allocator + MMA issuer.
// ---------------------------------------------------------------------------
struct PairCfg {
  static constexpr int NS = 2;                   // K and V stages
  static constexpr uint32_t kT = 2 * kSubTile;   // one 128 x 128 bf16 tile: 32 KiB
  static constexpr uint32_t offQA = 0;
  static constexpr uint32_t offQB = kT;
  static constexpr uint32_t offK = 2 * kT;
  static constexpr uint32_t offV = offK + NS * kT;
  static constexpr uint32_t offBar = offV + NS * kT;
  static constexpr int kNumBars = 1 + 4 * NS + 7;
  static constexpr uint32_t kSmem = offBar + kNumBars * 8 + 16;
  static_assert(kSmem <= 232448, "shared memory budget");
};

__global__ void __launch_bounds__(320, 1) attn_fwd_pair_kernel(const __grid_constant__ FwdParams p) {
  using Cfg = PairCfg;
  constexpr int DV = 128;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = ptx::smem_u32(smem);
  const AttnArgs& a = p.a;
  if (sbase & 1023u) {  // the swizzled operand panels need 1024-byte alignment
    if (threadIdx.x == 0 && p.err) atomicCAS(p.err, 0, 0x100 | kSiteAlign);
    return;
  }
  const int G = a.hq / a.hkv;
  const int npair = a.hq / 2;
  const int tile_idx = blockIdx.x / npair;
  const int slot = blockIdx.x - tile_idx * npair;
  const int kvh = slot / (G / 2), g0 = 2 * (slot - kvh * (G / 2));
  const int hA = a.gqa_interleaved ? g0 * a.hkv + kvh : kvh * G + g0;
  const int hB = a.gqa_interleaved ? (g0 + 1) * a.hkv + kvh : kvh * G + g0 + 1;
  const TileDesc tile = a.tiles[tile_idx];
  const int n_kv = tile.work;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t bar0 = sbase + Cfg::offBar;
  const uint32_t bar_q = bar0;
  auto bar_k_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto bar_k_empty = [&](int s) { return bar0 + 8u * (1 + Cfg::NS + s); };
  auto bar_v_full = [&](int s) { return bar0 + 8u * (1 + 2 * Cfg::NS + s); };
  auto bar_v_empty = [&](int s) { return bar0 + 8u * (1 + 3 * Cfg::NS + s); };
  const uint32_t barx = bar0 + 8u * (1 + 4 * Cfg::NS);
  auto bar_s_full = [&](int x) { return barx + 8u * x; };       // S_X(j) computed
  auto bar_p_full = [&](int x) { return barx + 16 + 8u * x; };  // P_X(j) in TMEM (4 warps)
  auto bar_o_done = [&](int x) { return barx + 32 + 8u * x; };  // PV_X(j) done
  const uint32_t bar_drain = barx + 48;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::offBar + Cfg::kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::offBar + Cfg::kNumBars * 8 + 4);

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar_q, 1);
    for (int s = 0; s < Cfg::NS; ++s) {
      ptx::mbar_init(bar_k_full(s), 1);
      ptx::mbar_init(bar_k_empty(s), 1);
      ptx::mbar_init(bar_v_full(s), 1);
      ptx::mbar_init(bar_v_empty(s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      ptx::mbar_init(bar_s_full(x), 1);
      ptx::mbar_init(bar_p_full(x), 4);
      ptx::mbar_init(bar_o_done(x), 1);
    }
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
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const ptx::WaitCtx wctx{abort_flag, p.err, kWaitLimitNs};

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_kv > 0) {
      int issued_k = 0, issued_v = 0;
      ptx::mbar_arrive_expect_tx(bar_q, 2 * Cfg::kT);
      for (int c = 0; c < 2; ++c) {
        ptx::tma_load_3d(sbase + Cfg::offQA + c * kSubTile, &p.tq, bar_q, c * 64, hA, tile.row0);
        ptx::tma_load_3d(sbase + Cfg::offQB + c * kSubTile, &p.tq, bar_q, c * 64, hB, tile.row0);
      }
      KvCursor cur;
      cur.init(a.ranges, tile.range_begin, tile.range_count);
      for (int j = 0; j < n_kv; ++j, cur.next()) {
        const int s = j % Cfg::NS;
        if (j >= Cfg::NS && !ptx::mbar_wait(bar_k_empty(s), ((j / Cfg::NS) - 1) & 1, kSiteKEmpty, wctx)) break;
        ptx::mbar_arrive_expect_tx(bar_k_full(s), Cfg::kT);
        for (int c = 0; c < 2; ++c)
          ptx::tma_load_3d(sbase + Cfg::offK + s * Cfg::kT + c * kSubTile, &p.tk, bar_k_full(s), c * 64, kvh,
                           cur.row());
        ++issued_k;
        if (j >= Cfg::NS && !ptx::mbar_wait(bar_v_empty(s), ((j / Cfg::NS) - 1) & 1, kSiteVEmpty, wctx)) break;
        ptx::mbar_arrive_expect_tx(bar_v_full(s), Cfg::kT);
        for (int c = 0; c < 2; ++c)
          ptx::tma_load_3d(sbase + Cfg::offV + s * Cfg::kT + c * kSubTile, &p.tv, bar_v_full(s), c * 64, kvh,
                           cur.row());
        ++issued_v;
      }
      if (*abort_flag) {
        volatile int no_abort = 0;
        const ptx::WaitCtx drain{&no_abort, nullptr, kWaitLimitNs};
        ptx::mbar_wait(bar_q, 0, kSiteDrain, drain);
        for (int j = max(0, issued_k - Cfg::NS); j < issued_k; ++j)
          ptx::mbar_wait(bar_k_full(j % Cfg::NS), (j / Cfg::NS) & 1, kSiteDrain, drain);
        for (int j = max(0, issued_v - Cfg::NS); j < issued_v; ++j)
          ptx::mbar_wait(bar_v_full(j % Cfg::NS), (j / Cfg::NS) & 1, kSiteDrain, drain);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_kv > 0) {
      constexpr uint32_t idS = ptx::idesc_bf16_f32(BM, BN, false, false);
      constexpr uint32_t idO = ptx::idesc_bf16_f32(BM, DV, false, true);
      auto issue_s = [&](int x, int j) {
        const uint32_t qb = sbase + (x ? Cfg::offQB : Cfg::offQA);
        const uint32_t kb = sbase + Cfg::offK + (j % Cfg::NS) * Cfg::kT;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kSubTile + (kk & 3) * 32;
          ptx::mma_ss(tmem + 256 * x, ptx::sdesc_sw128(qb + off, 16, 1024), ptx::sdesc_sw128(kb + off, 16, 1024),
                      idS, kk > 0);
        }
        ptx::mma_commit(bar_s_full(x));
      };
      auto issue_pv = [&](int x, int j) {
        const uint32_t vb = sbase + Cfg::offV + (j % Cfg::NS) * Cfg::kT;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          ptx::mma_ts(tmem + 256 * x + 128, tmem + 256 * x + kk * 8,
                      ptx::sdesc_sw128(vb + kk * 2048, kSubTile, 1024), idO, (j > 0 || kk > 0));
        ptx::mma_commit(bar_o_done(x));
      };
      bool ok = ptx::mbar_wait(bar_q, 0, kSiteQ, wctx) && ptx::mbar_wait(bar_k_full(0), 0, kSiteKFull, wctx);
      if (ok) {
        ptx::tc_fence_after();
        issue_s(0, 0);
        issue_s(1, 0);
        ptx::mma_commit(bar_k_empty(0));
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        const int s = j % Cfg::NS;
        ok = ptx::mbar_wait(bar_p_full(0), j & 1, kSitePFull, wctx) &&
             ptx::mbar_wait(bar_v_full(s), (j / Cfg::NS) & 1, kSiteVFull, wctx);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_pv(0, j);
        if (j + 1 < n_kv) {
          ok = ptx::mbar_wait(bar_k_full((j + 1) % Cfg::NS), ((j + 1) / Cfg::NS) & 1, kSiteKFull, wctx);
          if (!ok) break;
          ptx::tc_fence_after();
          issue_s(0, j + 1);
        }
        ok = ptx::mbar_wait(bar_p_full(1), j & 1, kSitePFull, wctx);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_pv(1, j);
        ptx::mma_commit(bar_v_empty(s));
        if (j + 1 < n_kv) {
          issue_s(1, j + 1);
          ptx::mma_commit(bar_k_empty((j + 1) % Cfg::NS));
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
    // ------------------------------------------------------------ softmax (one warpgroup per head)
    const int x = warp >> 2;
    const int h = x ? hB : hA;
    const int row = ((warp & 3) << 5) | lane;  // TMEM lane
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + 256 * x, tO = tS + 128;
    const float sl2 = a.scale * kLog2e;
    const int qpos = tile.pos0 + row;
    const bool row_ok = row < tile.nrows;
    float m_ref = -INFINITY;  // reference maximum of scale*log2e*s (log2 units)
    float l = 0.f;
    bool ok = true;
    KvCursor cur;
    cur.init(a.ranges, tile.range_begin, tile.range_count);
    for (int j = 0; j < n_kv; ++j, cur.next()) {
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar_s_full(x), j & 1, kSiteSFull, wctx))) { ok = false; break; }
      ptx::tc_fence_after();
      const int kn = cur.n(), kp = cur.pos();
      int lim = row_ok ? kn : 0;
      if (a.causal) lim = min(lim, qpos - kp + 1);
      const bool masked = lim < BN;
      // pass 1: row maximum over the visible columns (S read 64 columns at a time)
      float mx = -INFINITY;
#pragma unroll 1
      for (int hlf = 0; hlf < 2; ++hlf) {
        uint32_t s0[32], s1[32];
        ptx::tmem_ld32(tS + hlf * 64, s0);
        ptx::tmem_ld32(tS + hlf * 64 + 32, s1);
        ptx::tmem_ld_wait();
        ptx::reg_fence32(s0);
        ptx::reg_fence32(s1);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int c0 = hlf * 64 + i, c1 = c0 + 32;
          const float v0 = __uint_as_float(s0[i]), v1 = __uint_as_float(s1[i]);
          mx = fmaxf(mx, (!masked || c0 < lim) ? v0 : -INFINITY);
          mx = fmaxf(mx, (!masked || c1 < lim) ? v1 : -INFINITY);
        }
      }
      const float m_new = mx * sl2;
      float alpha = 1.f;
      if (m_new > m_ref + kRescaleThreshold) {
        alpha = ptx::ex2(m_ref - m_new);  // 0 when m_ref = -inf
        m_ref = m_new;
      }
      const float mref = m_ref == -INFINITY ? 0.f : m_ref;
      // PV_X(j-1) is complete (S_X(j) was issued after it): O may be rescaled.
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
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
      // pass 2: P = exp2(s * scale * log2e - m_ref), row sum, and P (bf16, two
      // per column) over columns that have already been read
      float rs = 0.f;
#pragma unroll 1
      for (int hlf = 0; hlf < 2; ++hlf) {
        uint32_t s0[32], s1[32];
        ptx::tmem_ld32(tS + hlf * 64, s0);
        ptx::tmem_ld32(tS + hlf * 64 + 32, s1);
        ptx::tmem_ld_wait();
        ptx::reg_fence32(s0);
        ptx::reg_fence32(s1);
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int c = hlf * 64 + 2 * i;
          const float a0 = __uint_as_float(i < 16 ? s0[2 * i] : s1[2 * i - 32]);
          const float a1 = __uint_as_float(i < 16 ? s0[2 * i + 1] : s1[2 * i + 1 - 32]);
          float e0 = ptx::ex2(fmaf(a0, sl2, -mref));
          float e1 = ptx::ex2(fmaf(a1, sl2, -mref));
          if (masked) {
            e0 = c < lim ? e0 : 0.f;
            e1 = c + 1 < lim ? e1 : 0.f;
          }
          rs += e0 + e1;
          pk[i] = ptx::pack_bf16(e0, e1);
        }
        ptx::tmem_st32(tS + hlf * 32, pk);
      }
      l = l * alpha + rs;
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_p_full(x));
    }

    // ------------------------------------------------------------ epilogue
    if (ok && n_kv > 0)
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar_o_done(x), (n_kv - 1) & 1, kSiteOFull, wctx));
    if (ok) {
      ptx::tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int64_t orow = int64_t(tile.row0) + row;
#pragma unroll
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
      if (row_ok) a.lse[int64_t(h) * a.lse_stride + orow] = l > 0.f ? m_ref * kLn2 + logf(l) : -INFINITY;
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
      !make_map_3d(&p.tk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DQK, a.hkv, a.T, 64, BN,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_3d(&p.tv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DV, a.hkv, a.T, 64, BN,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_tc_kernel<DQK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(Cfg::kSmemAlloc));
  if (e != cudaSuccess) return e;
  const int64_t grid = int64_t(a.num_tiles) * a.hq;
  if (grid == 0) return cudaSuccess;
  attn_fwd_tc_kernel<DQK, DV><<<unsigned(grid), 192, Cfg::kSmemAlloc, st>>>(p);
  return cudaGetLastError();
}

// Head-pair kernel for 128-wide heads when every GQA group has an even number
// of query heads (outside block mode); the one-head kernel otherwise.  The
// pair kernel is MUFU-bound until part of its exponentials move to the FMA
// pipe, so the one-head kernel serves every shape for now.
constexpr bool kUsePairForward = false;
static cudaError_t launch_fwd_pair(const AttnArgs& a, cudaStream_t st) {
  FwdParams p;
  p.a = a;
  p.err = device_error_word();
  if (!make_map_3d(&p.tq, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 128, a.hq, a.T, 64, BM,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_3d(&p.tk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 128, a.hkv, a.T, 64, BN,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_3d(&p.tv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 128, a.hkv, a.T, 64, BN,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(PairCfg::kSmem));
  if (e != cudaSuccess) return e;
  const int64_t grid = int64_t(a.num_tiles) * (a.hq / 2);
  if (grid == 0) return cudaSuccess;
  attn_fwd_pair_kernel<<<unsigned(grid), 320, PairCfg::kSmem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_tc_fwd(const AttnArgs& a, cudaStream_t st) {
  if (kUsePairForward && a.d_qk == 128 && a.d_v == 128 && !a.block_mode && (a.hq / a.hkv) % 2 == 0)
    return launch_fwd_pair(a, st);
  if (a.d_qk == 128 && a.d_v == 128) return launch_fwd_impl<128, 128>(a, st);
  if (a.d_qk == 192 && a.d_v == 128) return launch_fwd_impl<192, 128>(a, st);
  return cudaErrorInvalidValue;
}

}  // namespace cpattn
