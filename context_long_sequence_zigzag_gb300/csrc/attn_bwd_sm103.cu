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
// Per query tile (M = 128 keys, N = 128 queries):
//   S^T  = K Q^T          (SS MMA)           -> TMEM [0, 128)
//   dP^T = V dO^T         (SS MMA)           -> TMEM [128, 256)
//   softmax warps: P^T, dS^T (bf16) back into the low 64 columns of each
//   region, and dS^T into shared memory
//   dV  += P^T dO         (TS MMA, A = TMEM)  TMEM [256, 384)
//   dK  += dS^T Q         (TS MMA)            TMEM [384, 512)
//   dQ^T = K^T dS^T       (SS MMA, two N = 64 halves into the high 64 columns
//                          of the S^T and dP^T regions)
//   softmax warps read dQ^T (lane = head-dim index) and add it to global
//   memory with coalesced reductions.
//
// Roles (192 threads): warps 0-3 softmax / dQ / epilogue (thread = key row
// = TMEM lane), warp 4 TMA producer, warp 5 TMEM allocator + MMA issuer.
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

enum WaitSite : int {
  kSiteKV = 0x21, kSiteQEmpty, kSiteQFull, kSiteTmemFree, kSiteSFull, kSitePFull, kSiteMma2, kSiteDrain,
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
  static constexpr uint32_t offQ = offV + kVBytes;                 // NS stages of Q
  static constexpr uint32_t offO = offQ + NS * kQBytes;            // NS stages of dO
  static constexpr uint32_t offDS = offO + NS * kOBytes;
  static constexpr uint32_t offL = offDS + kDSBytes;               // lse * log2(e), 128 floats
  static constexpr uint32_t offD = offL + BN * 4;                  // D, 128 floats
  static constexpr uint32_t offBar = offD + BN * 4;
  static constexpr int kNumBars = 1 + 2 * NS + 5;
  static constexpr uint32_t kSmem = offBar + kNumBars * 8 + 16;
  static constexpr uint32_t kSmemAlloc = kSmem + 1024;
  static constexpr uint32_t tS = 0, tDP = 128, tDV = 256, tDK = 256 + DV;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(tDK + DQK <= kTmemCols, "TMEM budget");
  static_assert(kSmemAlloc <= 232448, "shared memory budget");
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
  int count, G, kvh, hq, hkv, inter;
  int g, ri, off;
  RangeDesc cur;
  __device__ void init(const RangeDesc* ranges, int begin, int cnt, int G_, int kvh_, int hq_, int hkv_,
                       int inter_) {
    r = ranges + begin;
    count = cnt;
    G = G_;
    kvh = kvh_;
    hq = hq_;
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

template <int DQK, int DV>
__global__ void __launch_bounds__(192, 1) attn_bwd_tc_kernel(const __grid_constant__ BwdParams p) {
  using Cfg = BwdCfg<DQK, DV>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const AttnArgs& a = p.a;

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
  const uint32_t bar_p_full = bar_s_full + 8;
  const uint32_t bar_mma2 = bar_s_full + 16;
  const uint32_t bar_tmem_free = bar_s_full + 24;
  const uint32_t bar_drain = bar_s_full + 32;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::offBar + Cfg::kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::offBar + Cfg::kNumBars * 8 + 4);

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar_kv, 1);
    for (int s = 0; s < Cfg::NS; ++s) {
      ptx::mbar_init(bar_q_full(s), 1);
      ptx::mbar_init(bar_q_empty(s), 1);
    }
    ptx::mbar_init(bar_s_full, 1);
    ptx::mbar_init(bar_p_full, 4);
    ptx::mbar_init(bar_mma2, 1);
    ptx::mbar_init(bar_tmem_free, 4);
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
    ptx::prefetch_tmap(&p.tdo);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const ptx::WaitCtx wctx{abort_flag, p.err, kWaitLimitNs};

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_steps > 0) {
      int issued = 0;
      ptx::mbar_arrive_expect_tx(bar_kv, Cfg::kKBytes + Cfg::kVBytes);
      for (int c = 0; c < Cfg::kQPanels; ++c)
        ptx::tma_load_3d(sbase + Cfg::offK + c * kPanel, &p.tk, bar_kv, c * 64, kvh, tile.row0);
      for (int c = 0; c < Cfg::kVPanels; ++c)
        ptx::tma_load_3d(sbase + Cfg::offV + c * kPanel, &p.tv, bar_kv, c * 64, kvh, tile.row0);
      StepCursor cur;
      cur.init(a.ranges, tile.range_begin, tile.range_count, G, kvh, a.hq, a.hkv, a.gqa_interleaved);
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
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_steps > 0) {
      constexpr uint32_t idS = ptx::idesc_bf16_f32(BM, BN, false, false);
      constexpr uint32_t idDV = ptx::idesc_bf16_f32(BM, DV, false, true);
      constexpr uint32_t idDK = ptx::idesc_bf16_f32(BM, DQK, false, true);
      constexpr uint32_t idDQ = ptx::idesc_bf16_f32(128, 64, true, true);  // M = head dim 128
      const uint32_t tS = tmem + Cfg::tS, tDP = tmem + Cfg::tDP;
      const uint32_t tDV = tmem + Cfg::tDV, tDK = tmem + Cfg::tDK;
      const uint32_t kb = sbase + Cfg::offK, vb = sbase + Cfg::offV, dsb = sbase + Cfg::offDS;
      bool ok = ptx::mbar_wait(bar_kv, 0, kSiteKV, wctx);
      for (int i = 0; ok && i < n_steps; ++i) {
        const int s = i % Cfg::NS;
        ok = ptx::mbar_wait(bar_q_full(s), (i / Cfg::NS) & 1, kSiteQFull, wctx);
        if (ok && i > 0) ok = ptx::mbar_wait(bar_tmem_free, (i - 1) & 1, kSiteTmemFree, wctx);
        if (!ok) break;
        ptx::tc_fence_after();
        const uint32_t qb = sbase + Cfg::offQ + s * Cfg::kQBytes;
        const uint32_t ob = sbase + Cfg::offO + s * Cfg::kOBytes;
        // S^T = K Q^T, dP^T = V dO^T
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
          ptx::mma_ss(tS, ptx::sdesc_sw128(kb + off, 16, 1024), ptx::sdesc_sw128(qb + off, 16, 1024), idS, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < DV / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kPanel + (kk & 3) * 32;
          ptx::mma_ss(tDP, ptx::sdesc_sw128(vb + off, 16, 1024), ptx::sdesc_sw128(ob + off, 16, 1024), idS, kk > 0);
        }
        ptx::mma_commit(bar_s_full);
        ok = ptx::mbar_wait(bar_p_full, i & 1, kSitePFull, wctx);
        if (!ok) break;
        ptx::tc_fence_after();
        // dV += P^T dO ; dQ^T[:, 0:64] = K^T dS^T[:, 0:64]
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          ptx::mma_ts(tDV, tS + kk * 8, ptx::sdesc_sw128(ob + kk * 2048, kPanel, 1024), idDV, (i > 0 || kk > 0));
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)
          ptx::mma_ss(tS + 64, ptx::sdesc_sw128(kb + kk * 2048, kPanel, 1024), ptx::sdesc_sw128(dsb + kk * 2048, kPanel, 1024),
                      idDQ, kk > 0);
        // dK += dS^T Q ; dQ^T[:, 64:128] = K^T dS^T[:, 64:128]
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          ptx::mma_ts(tDK, tDP + kk * 8, ptx::sdesc_sw128(qb + kk * 2048, kPanel, 1024), idDK, (i > 0 || kk > 0));
#pragma unroll
        for (int kk = 0; kk < BM / 16; ++kk)
          ptx::mma_ss(tDP + 64, ptx::sdesc_sw128(kb + kk * 2048, kPanel, 1024),
                      ptx::sdesc_sw128(dsb + kPanel + kk * 2048, kPanel, 1024), idDQ, kk > 0);
        ptx::mma_commit(bar_mma2);
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
    // ------------------------------------------------------------ softmax / dQ / epilogue
    const int r = threadIdx.x;  // key row = TMEM lane (and head-dim index for dQ^T)
    const uint32_t lane_base = uint32_t(warp * 32) << 16;
    const uint32_t tS = tmem + lane_base + Cfg::tS, tDP = tmem + lane_base + Cfg::tDP;
    const float sl2 = a.scale * kLog2e;
    const int kpos = tile.pos0 + r;
    const bool row_ok = r < tile.nrows;
    float* sL = reinterpret_cast<float*>(smem + Cfg::offL);
    float* sD = reinterpret_cast<float*>(smem + Cfg::offD);
    uint8_t* dsrow = smem + Cfg::offDS + r * 128;
    const int sw = r & 7;
    bool ok = true;
    StepCursor cur;
    cur.init(a.ranges, tile.range_begin, tile.range_count, G, kvh, a.hq, a.hkv, a.gqa_interleaved);
    for (int i = 0; i < n_steps; ++i, cur.next()) {
      const int h = cur.head(), qrow0 = cur.row(), nq = cur.n(), qpos0 = cur.pos();
      // statistics of this step's query rows
      const float lv = r < nq ? a.lse_in[int64_t(h) * a.T + qrow0 + r] * kLog2e : 0.f;
      const float dv = r < nq ? a.dpsum[int64_t(h) * a.T + qrow0 + r] : 0.f;
      ptx::named_barrier(1, 128);  // previous step's readers are done
      sL[r] = lv;
      sD[r] = dv;
      ptx::named_barrier(1, 128);
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar_s_full, i & 1, kSiteSFull, wctx))) { ok = false; break; }
      ptx::tc_fence_after();
      // first visible query column of this key row
      const int cmin = a.causal ? kpos - qpos0 : 0;
      const int cmax = row_ok ? nq : 0;  // columns [cmin, cmax) are visible
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t sr[32], dr[32];
        ptx::tmem_ld32(tS + c * 32, sr);
        ptx::tmem_ld32(tDP + c * 32, dr);
        ptx::tmem_ld_wait();
        ptx::reg_fence32(sr);
        ptx::reg_fence32(dr);
        uint32_t pp[16], dd[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float pv[2], dsv[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int col = c * 32 + 2 * j + e;
            const bool vis = col >= cmin && col < cmax;
            const float pr = ptx::ex2(fmaf(__uint_as_float(sr[2 * j + e]), sl2, -sL[col]));
            pv[e] = vis ? pr : 0.f;
            dsv[e] = pv[e] * (__uint_as_float(dr[2 * j + e]) - sD[col]) * a.scale;
          }
          pp[j] = ptx::pack_bf16(pv[0], pv[1]);
          dd[j] = ptx::pack_bf16(dsv[0], dsv[1]);
        }
        ptx::tmem_st16(tS + c * 16, pp);
        ptx::tmem_st16(tDP + c * 16, dd);
        // dS^T row into the swizzled [key][query] panels (query = K-major)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int chunk = (c & 1) * 4 + k;
          *reinterpret_cast<uint4*>(dsrow + (c >> 1) * kPanel + ((chunk ^ sw) << 4)) =
              make_uint4(dd[4 * k], dd[4 * k + 1], dd[4 * k + 2], dd[4 * k + 3]);
        }
      }
      ptx::tmem_st_wait();
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_p_full);

      // dQ^T (lane = head-dim index) -> global FP32 accumulator
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar_mma2, i & 1, kSiteMma2, wctx))) { ok = false; break; }
      ptx::tc_fence_after();
      float* dqp = a.dq_acc + (int64_t(qrow0) * a.hq + h) * DQK + r;
      const int64_t qstride = int64_t(a.hq) * DQK;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        const uint32_t base = (half ? tDP : tS) + 64;
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t qr[32];
          ptx::tmem_ld32(base + cc * 32, qr);
          ptx::tmem_ld_wait();
          ptx::reg_fence32(qr);
          const int col0 = half * 64 + cc * 32;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (col0 + j < nq) ptx::red_add_f32(dqp + int64_t(col0 + j) * qstride, __uint_as_float(qr[j]));
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_tmem_free);
    }

    // ------------------------------------------------------------ dK, dV epilogue
    if (ok && n_steps > 0)
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar_mma2, (n_steps - 1) & 1, kSiteMma2, wctx));
    if (ok) {
      ptx::tc_fence_after();
      const int64_t krow = int64_t(tile.row0) + r;
      __nv_bfloat16* dkp = static_cast<__nv_bfloat16*>(a.dk) + (krow * a.hkv + kvh) * DQK;
      __nv_bfloat16* dvp = static_cast<__nv_bfloat16*>(a.dv) + (krow * a.hkv + kvh) * DV;
      auto store_row = [&](uint32_t tcol, __nv_bfloat16* dst, int ncols) {
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
          if (row_ok) {
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
      };
      store_row(Cfg::tDV, dvp, DV);
      store_row(Cfg::tDK, dkp, DQK);
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
                                       int(Cfg::kSmemAlloc));
  if (e != cudaSuccess) return e;
  const int64_t grid = int64_t(a.num_tiles) * a.hkv;
  if (grid == 0) return cudaSuccess;
  attn_bwd_tc_kernel<DQK, DV><<<unsigned(grid), 192, Cfg::kSmemAlloc, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_tc_bwd(const AttnArgs& a, cudaStream_t st) {
  if (a.d_qk == 128 && a.d_v == 128) return launch_bwd_impl<128, 128>(a, st);
  return cudaErrorInvalidValue;
}

}  // namespace cpattn
