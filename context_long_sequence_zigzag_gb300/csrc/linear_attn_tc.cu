// linear_attn_tc.cu — the block-state and block-output passes of decayed
// linear attention with AllGather context parallelism on the sm_103a tensor
// cores, for bf16 tensors with 128-wide heads ("超长上下文训练速度翻倍秘籍":
// the recurrence h_t = alpha h_{t-1} + K_t^T V_t, O_t = Q_t h_t, and the
// AllGather CP section: rank-local states, the decayed prefix over the
// gathered states, and the output correction (q * decay) @ init_state).
//
// A block of at most kLinBlock tokens is processed in chunks of 128 tokens,
// the chunked form of the recurrence with alpha = exp(g):
//   A'[t][s] = (q_t . k_s) alpha^(t-s) for s <= t, else 0
//   O_c      = scale (A' V_c + diag(alpha^(t+1)) Q_c H)
//   H       <- alpha^n H + sum_s alpha^(n-1-s) k_s^T v_s        (n tokens)
// Every product is a tcgen05 MMA with a 128 x 128 fp32 TMEM accumulator:
//   Q K^T   SS, Q and K K-major (as loaded by TMA)
//   Q H     SS, H staged as bf16 in shared memory (MN-major: row d holds j)
//   A' V    TS, A' written back to TMEM as bf16 by the threads, V MN-major
//   K'^T V  SS, both MN-major: K' is K with row s scaled by alpha^(n-1-s),
//           done in place in shared memory once Q K^T has read K
// H lives in TMEM in fp32 across the chunks of a block.
#include <cuda.h>
#include <cuda_bf16.h>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace cpattn {

bool make_map_3d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elt, int64_t dim, int64_t heads,
                 int64_t T, int box_inner, int box_rows, CUtensorMapSwizzle swz);

namespace {

constexpr int kC = 128;                   // tokens per chunk
constexpr int kD = 128;                   // head dim (Dk = Dv)
constexpr uint32_t kPanel = 128 * 128;    // 128 rows x 64 bf16 (128 B, 128B-swizzled): 16 KiB
constexpr uint32_t kTile = 2 * kPanel;    // 128 rows x 128 bf16
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

enum LinSite : int {
  kLinSiteFull = 32, kLinSiteEmpty, kLinSiteHb, kLinSiteQk, kLinSiteAp, kLinSiteXh, kLinSiteScaled, kLinSiteMma,
  kLinSiteDrain, kLinSiteAlign,
};

struct LinTcParams {
  CUtensorMap tq, tk, tv;
  const LinBlock* blocks;
  const float* g;
  const float* init;  // [nblocks, H, D, D] carried-in state (output pass)
  float* states;      // [nblocks, H, D, D] block states (state pass)
  __nv_bfloat16* o;
  int32_t H;
  float scale;
  int32_t* err;
};

// Scales the 128 bf16 of row r of a [128 x 128] 128B-swizzled tile by w in
// place.  The swizzle only permutes 16-byte chunks inside a row, so the row
// is the same 2 x 128 bytes whatever the permutation.  Thread r starts at
// chunk r % 8: the rows of a warp are 128 bytes apart, so visiting the same
// chunk index in every row would put all 32 lanes on the same four banks.
__device__ __forceinline__ void scale_row_bf16(uint8_t* tile, int r, float w) {
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    uint4* row = reinterpret_cast<uint4*>(tile + p * kPanel + r * 128);
#pragma unroll
    for (int qq = 0; qq < 8; ++qq) {
      const int q = (qq + r) & 7;
      uint4 u = row[q];
      uint32_t* w32 = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&w32[e]);
        const float2 f = __bfloat1622float2(b);
        w32[e] = ptx::pack_bf16(f.x * w, f.y * w);
      }
      row[q] = u;
    }
  }
}

// TMEM row (this thread's lane) of 128 fp32 columns -> row r of a [128 x 128]
// bf16 tile in the 128B-swizzled layout (16-byte chunk q of row r sits at
// chunk q ^ (r % 8) of its 128-byte row).
__device__ __forceinline__ void tmem_row_to_swizzled_bf16(uint32_t taddr, uint8_t* tile, int r) {
  // all 128 columns in flight at once: one TMEM round trip, not four
  uint32_t x[4][32];
#pragma unroll
  for (int c = 0; c < 4; ++c) ptx::tmem_ld32(taddr + c * 32, x[c]);
  ptx::tmem_ld_wait();
#pragma unroll
  for (int c = 0; c < 4; ++c) ptx::reg_fence32(x[c]);
#pragma unroll
  for (int c = 0; c < 4; ++c) {  // 32 columns = 4 chunks of 8
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int col = c * 32 + k * 8;
      const int p = col >> 6, q = (col & 63) >> 3;
      uint4 u;
      u.x = ptx::pack_bf16(__uint_as_float(x[c][8 * k + 0]), __uint_as_float(x[c][8 * k + 1]));
      u.y = ptx::pack_bf16(__uint_as_float(x[c][8 * k + 2]), __uint_as_float(x[c][8 * k + 3]));
      u.z = ptx::pack_bf16(__uint_as_float(x[c][8 * k + 4]), __uint_as_float(x[c][8 * k + 5]));
      u.w = ptx::pack_bf16(__uint_as_float(x[c][8 * k + 6]), __uint_as_float(x[c][8 * k + 7]));
      *reinterpret_cast<uint4*>(tile + p * kPanel + r * 128 + ((q ^ (r & 7)) << 4)) = u;
    }
  }
}

// 16 MMAs-worth of K-steps over a 128-deep contraction: descriptor advance
// for a K-major operand (32 B per 16 elements inside a panel, a panel per 64)
__device__ __forceinline__ uint32_t kmajor_adv(int kk) { return ((kk >> 2) * kPanel + (kk & 3) * 32) >> 4; }
// ... and for an MN-major operand (16 rows of 128 B per step)
__device__ __forceinline__ uint32_t mnmajor_adv(int kk) { return (kk * 2048) >> 4; }

// ============================================================================
// Block states: S_b = sum_s alpha^(len-1-s) k_s^T v_s from a zero start, one
// CTA per (block, head).  160 threads: warps 0-3 scale K rows (thread = token
// row of the chunk) and write the state out (thread = state row d); warp 4
// loads (lane 0) and issues the MMAs.  Single-buffered: several CTAs share an
// SM and hide each other's latency.
// ============================================================================
constexpr int kStateThreads = 160;
constexpr uint32_t kStateSmem = 2 * kTile + 8 * 4 + 16;  // K, V tiles; 4 barriers; TMEM slot, abort flag

__global__ void __launch_bounds__(kStateThreads) lin_state_tc_kernel(const __grid_constant__ LinTcParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = ptx::smem_u32(smem);
  if (sbase & 1023u) {
    if (threadIdx.x == 0 && p.err) atomicCAS(p.err, 0, 0x100 | kLinSiteAlign);
    return;
  }
  uint8_t* Ks = smem;
  const uint32_t bar0 = sbase + 2 * kTile;
  const uint32_t bar_full = bar0, bar_scaled = bar0 + 8, bar_mma = bar0 + 16, bar_drain = bar0 + 24;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 2 * kTile + 32);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 2 * kTile + 36);
  const int b = blockIdx.x / p.H, h = blockIdx.x - (blockIdx.x / p.H) * p.H;
  const LinBlock bl = p.blocks[b];
  const int nch = (bl.len + kC - 1) / kC;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar_full, 1);
    ptx::mbar_init(bar_scaled, 4);
    ptx::mbar_init(bar_mma, 1);
    ptx::mbar_init(bar_drain, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 4) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 128);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const ptx::WaitCtx wctx{abort_flag, p.err, kWaitLimitNs};
  const float gl2 = p.g[h] * kLog2e;  // log2(alpha)

  if (warp == 4) {
    constexpr uint32_t idH = ptx::idesc_bf16_f32(kD, kD, true, true);
    bool ok = true;
    int loaded = 0;  // chunks whose load was issued
    for (int c = 0; ok && c < nch; ++c) {
      ++loaded;
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(bar_full, 2 * kTile);
        for (int q = 0; q < 2; ++q) {
          ptx::tma_load_3d(sbase + q * kPanel, &p.tk, bar_full, q * 64, h, bl.row0 + c * kC);
          ptx::tma_load_3d(sbase + kTile + q * kPanel, &p.tv, bar_full, q * 64, h, bl.row0 + c * kC);
        }
      }
      __syncwarp();
      ok = ptx::mbar_wait_w(bar_scaled, c & 1, kLinSiteScaled, wctx);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint64_t kd = ptx::sdesc_sw128(sbase, kPanel, 1024), vd = ptx::sdesc_sw128(sbase + kTile, kPanel, 1024);
#pragma unroll
      for (int kk = 0; kk < kC / 16; ++kk)
        ptx::mma_ss_w(tmem, kd + mnmajor_adv(kk), vd + mnmajor_adv(kk), idH, (c > 0 || kk > 0));
      ptx::mma_commit_w(bar_mma);
      ok = ptx::mbar_wait_w(bar_mma, c & 1, kLinSiteMma, wctx);  // the tile is free again
    }
    if (!ok) {
      // let the last load land and every issued MMA finish before the CTA exits
      volatile int no_abort = 0;
      const ptx::WaitCtx drain{&no_abort, nullptr, kWaitLimitNs};
      ptx::mbar_wait_w(bar_full, (loaded - 1) & 1, kLinSiteDrain, drain);
      ptx::mma_commit_w(bar_drain);
      ptx::mbar_wait_w(bar_drain, 0, kLinSiteDrain, drain);
    }
  } else {
    const int r = threadIdx.x;  // token row of the chunk / state row d (TMEM lane)
    bool ok = true;
    for (int c = 0; c < nch; ++c) {
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar_full, c & 1, kLinSiteFull, wctx));
      if (!ok) break;
      const int n = min(kC, bl.len - c * kC);
      // alpha^(len-1-s) for token s of the block, 0 past the chunk's end
      const float w = r < n ? ptx::ex2(gl2 * float(bl.len - 1 - (c * kC + r))) : 0.f;
      scale_row_bf16(Ks, r, w);
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_scaled);
      // the next chunk's load waits for the MMA; wait here too so the
      // scaled rows are not touched before the MMA read them
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar_mma, c & 1, kLinSiteMma, wctx));
      if (!ok) break;
    }
    if (ok && nch > 0) {
      ptx::tc_fence_after();
      float* out = p.states + ((int64_t(b) * p.H + h) * kD + r) * kD;
      const uint32_t trow = tmem + (uint32_t((warp & 3) * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t x[32];
        ptx::tmem_ld32(trow + c * 32, x);
        ptx::tmem_ld_wait();
        ptx::reg_fence32(x);
        float4* dst = reinterpret_cast<float4*>(out + c * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          dst[i] = make_float4(__uint_as_float(x[4 * i]), __uint_as_float(x[4 * i + 1]), __uint_as_float(x[4 * i + 2]),
                               __uint_as_float(x[4 * i + 3]));
      }
    } else if (ok) {
      float4* dst = reinterpret_cast<float4*>(p.states + ((int64_t(b) * p.H + h) * kD + r) * kD);
      for (int i = 0; i < kD / 4; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 128);
  }
}

// ============================================================================
// Block outputs from the carried-in state, one CTA per (block, head).
// 192 threads: warps 0-3 compute (thread = chunk row t and state row d, the
// TMEM lane), warp 4 issues the MMAs and owns TMEM, warp 5 lane 0 loads
// Q, K, V of the chunks into two stages.
// TMEM: A (Q K^T, then A' as bf16) [0,128), Y = Q H [128,256),
//       X = A' V [256,384), H [384,512).
// Per chunk c:  MMA warp: Q K^T, Q H           -> bar_qk
//               threads:  A', K' in place, H *= alpha^n -> bar_ap
//               MMA warp: A' V, H += K'^T V     -> bar_xh (+ stage free)
//               threads:  o rows, H -> bf16 for the next chunk -> bar_hb
// ============================================================================
constexpr int kOutThreads = 192;
constexpr uint32_t kStage = 3 * kTile;  // Q, K, V
constexpr uint32_t offHb = 2 * kStage;
constexpr uint32_t offBarO = offHb + kTile;
constexpr int kNumBarsO = 2 + 2 + 5;
constexpr uint32_t offTabO = offBarO + kNumBarsO * 8 + 16;  // alpha^d, d = 0..127 (fp32)
constexpr uint32_t kOutSmem = offTabO + kC * 4;
static_assert(kOutSmem <= 232448, "shared memory budget");

__global__ void __launch_bounds__(kOutThreads, 1) lin_output_tc_kernel(const __grid_constant__ LinTcParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = ptx::smem_u32(smem);
  if (sbase & 1023u) {
    if (threadIdx.x == 0 && p.err) atomicCAS(p.err, 0, 0x100 | kLinSiteAlign);
    return;
  }
  const uint32_t bar0 = sbase + offBarO;
  auto bar_full = [&](int s) { return bar0 + 8u * s; };
  auto bar_empty = [&](int s) { return bar0 + 16u + 8u * s; };
  const uint32_t bar_hb = bar0 + 32, bar_qk = bar0 + 40, bar_ap = bar0 + 48, bar_xh = bar0 + 56,
                 bar_drain = bar0 + 64;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + offBarO + kNumBarsO * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + offBarO + kNumBarsO * 8 + 4);
  const int b = blockIdx.x / p.H, h = blockIdx.x - (blockIdx.x / p.H) * p.H;
  const LinBlock bl = p.blocks[b];
  const int nch = (bl.len + kC - 1) / kC;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(bar_full(s), 1);
      ptx::mbar_init(bar_empty(s), 1);
    }
    ptx::mbar_init(bar_hb, 4);
    ptx::mbar_init(bar_qk, 1);
    ptx::mbar_init(bar_ap, 4);
    ptx::mbar_init(bar_xh, 1);
    ptx::mbar_init(bar_drain, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 4) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), 512);
    ptx::tmem_relinquish();
  }
  if (warp == 5 && lane == 0) {
    ptx::prefetch_tmap(&p.tq);
    ptx::prefetch_tmap(&p.tk);
    ptx::prefetch_tmap(&p.tv);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tA = tmem, tY = tmem + 128, tX = tmem + 256, tH = tmem + 384;
  const ptx::WaitCtx wctx{abort_flag, p.err, kWaitLimitNs};
  const float gl2 = p.g[h] * kLog2e;  // log2(alpha)

  if (warp == 5) {
    // ------------------------------------------------------------ loads
    if (lane == 0) {
      int issued = 0;
      for (int c = 0; c < nch; ++c) {
        const int st = c & 1;
        if (c >= 2 && !ptx::mbar_wait(bar_empty(st), ((c >> 1) - 1) & 1, kLinSiteEmpty, wctx)) break;
        ptx::mbar_arrive_expect_tx(bar_full(st), kStage);
        const uint32_t dst = sbase + st * kStage;
        const int row = bl.row0 + c * kC;
        for (int q = 0; q < 2; ++q) {
          ptx::tma_load_3d(dst + q * kPanel, &p.tq, bar_full(st), q * 64, h, row);
          ptx::tma_load_3d(dst + kTile + q * kPanel, &p.tk, bar_full(st), q * 64, h, row);
          ptx::tma_load_3d(dst + 2 * kTile + q * kPanel, &p.tv, bar_full(st), q * 64, h, row);
        }
        ++issued;
      }
      if (*abort_flag) {
        volatile int no_abort = 0;
        const ptx::WaitCtx drain{&no_abort, nullptr, kWaitLimitNs};
        for (int c = max(0, issued - 2); c < issued; ++c) ptx::mbar_wait(bar_full(c & 1), (c >> 1) & 1, kLinSiteDrain, drain);
      }
    }
  } else if (warp == 4) {
    // ------------------------------------------------------------ MMA issuer (whole warp)
    constexpr uint32_t idQK = ptx::idesc_bf16_f32(kC, kC, false, false);   // K-major x K-major
    constexpr uint32_t idQH = ptx::idesc_bf16_f32(kC, kD, false, true);    // K-major x MN-major
    constexpr uint32_t idAV = ptx::idesc_bf16_f32(kC, kD, false, true);    // TMEM x MN-major
    constexpr uint32_t idKV = ptx::idesc_bf16_f32(kD, kD, true, true);     // MN-major x MN-major
    // Q K^T of chunk c+1 needs only that chunk's loads: it is issued right
    // after chunk c's A' V (which it overwrites in TMEM after, in pipe
    // order), so it runs while the threads write chunk c's output.  Q H has
    // to wait for the restaged state.
    auto issue_qk = [&](int c) {
      const uint32_t sQ = sbase + (c & 1) * kStage;
      const uint64_t qd = ptx::sdesc_sw128(sQ, 16, 1024), kdk = ptx::sdesc_sw128(sQ + kTile, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk) ptx::mma_ss_w(tA, qd + kmajor_adv(kk), kdk + kmajor_adv(kk), idQK, kk > 0);
    };
    bool ok = true;
    if (nch > 0) {
      ok = ptx::mbar_wait_w(bar_full(0), 0, kLinSiteFull, wctx);
      if (ok) {
        ptx::tc_fence_after();
        issue_qk(0);
      }
    }
    for (int c = 0; ok && c < nch; ++c) {
      const int st = c & 1;
      const uint32_t sQ = sbase + st * kStage, sK = sQ + kTile, sV = sQ + 2 * kTile;
      ok = ptx::mbar_wait_w(bar_hb, c & 1, kLinSiteHb, wctx);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint64_t qd = ptx::sdesc_sw128(sQ, 16, 1024);
      const uint64_t hd = ptx::sdesc_sw128(sbase + offHb, kPanel, 1024);
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk) ptx::mma_ss_w(tY, qd + kmajor_adv(kk), hd + mnmajor_adv(kk), idQH, kk > 0);
      ptx::mma_commit_w(bar_qk);
      ok = ptx::mbar_wait_w(bar_ap, c & 1, kLinSiteAp, wctx);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint64_t vd = ptx::sdesc_sw128(sV, kPanel, 1024), kdm = ptx::sdesc_sw128(sK, kPanel, 1024);
#pragma unroll
      for (int kk = 0; kk < kC / 16; ++kk) ptx::mma_ts_w(tX, tA + kk * 8, vd + mnmajor_adv(kk), idAV, kk > 0);
#pragma unroll
      for (int kk = 0; kk < kC / 16; ++kk) ptx::mma_ss_w(tH, kdm + mnmajor_adv(kk), vd + mnmajor_adv(kk), idKV, 1);
      ptx::mma_commit_w(bar_xh);
      ptx::mma_commit_w(bar_empty(st));
      if (c + 1 < nch) {
        ok = ptx::mbar_wait_w(bar_full((c + 1) & 1), ((c + 1) >> 1) & 1, kLinSiteFull, wctx);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_qk(c + 1);
      }
    }
    if (!ok) {
      volatile int no_abort = 0;
      const ptx::WaitCtx drain{&no_abort, nullptr, kWaitLimitNs};
      ptx::mma_commit_w(bar_drain);
      ptx::mbar_wait_w(bar_drain, 0, kLinSiteDrain, drain);
    }
  } else {
    // ------------------------------------------------------------ compute (thread = TMEM lane)
    const int r = threadIdx.x;  // chunk row t / state row d
    const uint32_t lane_base = uint32_t(warp * 32) << 16;
    uint8_t* Hb = smem + offHb;
    bool ok = true;
    // alpha^d for every distance d inside a chunk, computed once: the decay
    // mask then takes a table entry per element instead of an exponential
    float* dec = reinterpret_cast<float*>(smem + offTabO);
    dec[r] = ptx::ex2(gl2 * float(r));
    ptx::named_barrier(1, 128);
    // carried-in state -> TMEM (fp32) and the bf16 copy for the first Q H;
    // all 32 loads of the row are issued before any is used
    {
      const float4* src = reinterpret_cast<const float4*>(p.init + ((int64_t(b) * p.H + h) * kD + r) * kD);
      float4 v4[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v4[i] = __ldcs(src + i);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t x[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 v = v4[c * 8 + i];
          x[4 * i] = __float_as_uint(v.x);
          x[4 * i + 1] = __float_as_uint(v.y);
          x[4 * i + 2] = __float_as_uint(v.z);
          x[4 * i + 3] = __float_as_uint(v.w);
        }
        ptx::tmem_st32(tH + lane_base + c * 32, x);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int col = c * 32 + k * 8;
          const int pn = col >> 6, q = (col & 63) >> 3;
          uint4 u;
          u.x = ptx::pack_bf16(__uint_as_float(x[8 * k + 0]), __uint_as_float(x[8 * k + 1]));
          u.y = ptx::pack_bf16(__uint_as_float(x[8 * k + 2]), __uint_as_float(x[8 * k + 3]));
          u.z = ptx::pack_bf16(__uint_as_float(x[8 * k + 4]), __uint_as_float(x[8 * k + 5]));
          u.w = ptx::pack_bf16(__uint_as_float(x[8 * k + 6]), __uint_as_float(x[8 * k + 7]));
          *reinterpret_cast<uint4*>(Hb + pn * kPanel + r * 128 + ((q ^ (r & 7)) << 4)) = u;
        }
      }
      ptx::tmem_st_wait();
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_hb);
    }
    for (int c = 0; c < nch; ++c) {
      const int st = c & 1;
      const int n = min(kC, bl.len - c * kC);
      ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar_qk, c & 1, kLinSiteQk, wctx));
      if (!ok) break;
      ptx::tc_fence_after();
      // ---- A'[t][s] = A[t][s] alpha^(t-s) for s <= t, s < n (bf16 into TMEM A).
      // All 128 columns are loaded first (one TMEM round trip); the packed
      // chunk k then lands in columns [16k, 16k+16).
      {
        const int lim = min(r + 1, n);  // visible columns [0, lim)
        uint32_t x[4][32];
#pragma unroll
        for (int k = 0; k < 4; ++k) ptx::tmem_ld32(tA + lane_base + k * 32, x[k]);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 4; ++k) ptx::reg_fence32(x[k]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int s0 = k * 32 + 2 * i;
            const float d0 = s0 < lim ? dec[r - s0] : 0.f;
            const float d1 = s0 + 1 < lim ? dec[r - s0 - 1] : 0.f;
            pk[i] = ptx::pack_bf16(__uint_as_float(x[k][2 * i]) * d0, __uint_as_float(x[k][2 * i + 1]) * d1);
          }
          ptx::tmem_st16(tA + lane_base + k * 16, pk);
        }
      }
      // ---- H *= alpha^n, its TMEM loads in flight while K' = K with row s
      // scaled by alpha^(n-1-s) (0 past the chunk) is formed in place
      {
        uint32_t x[4][32];
#pragma unroll
        for (int k = 0; k < 4; ++k) ptx::tmem_ld32(tH + lane_base + k * 32, x[k]);
        const float w = r < n ? ptx::ex2(gl2 * float(n - 1 - r)) : 0.f;
        scale_row_bf16(smem + st * kStage + kTile, r, w);
        const float an = ptx::ex2(gl2 * float(n));
        ptx::tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 4; ++k) ptx::reg_fence32(x[k]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
#pragma unroll
          for (int i = 0; i < 32; ++i) x[k][i] = __float_as_uint(__uint_as_float(x[k][i]) * an);
          ptx::tmem_st32(tH + lane_base + k * 32, x[k]);
        }
      }
      ptx::tmem_st_wait();
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar_ap);

      ok = __all_sync(0xffffffffu, ptx::mbar_wait(bar_xh, c & 1, kLinSiteXh, wctx));
      if (!ok) break;
      ptx::tc_fence_after();
      // ---- o[t] = scale (X[t] + alpha^(t+1) Y[t])
      {
        const float dy = ptx::ex2(gl2 * float(r + 1));
        __nv_bfloat16* dst = p.o + ((int64_t(bl.row0) + c * kC + r) * p.H + h) * kD;
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {  // 64 columns of X and Y per TMEM round trip
          uint32_t x[2][32], y[2][32];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            ptx::tmem_ld32(tX + lane_base + (2 * hh + k) * 32, x[k]);
            ptx::tmem_ld32(tY + lane_base + (2 * hh + k) * 32, y[k]);
          }
          ptx::tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            ptx::reg_fence32(x[k]);
            ptx::reg_fence32(y[k]);
          }
          if (r < n) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              uint4* d4 = reinterpret_cast<uint4*>(dst + (2 * hh + k) * 32);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                float v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                  v[e] = p.scale * fmaf(dy, __uint_as_float(y[k][8 * i + e]), __uint_as_float(x[k][8 * i + e]));
                uint4 u;
                u.x = ptx::pack_bf16(v[0], v[1]);
                u.y = ptx::pack_bf16(v[2], v[3]);
                u.z = ptx::pack_bf16(v[4], v[5]);
                u.w = ptx::pack_bf16(v[6], v[7]);
                d4[i] = u;
              }
            }
          }
        }
      }
      // ---- H -> bf16 operand of the next chunk's Q H
      if (c + 1 < nch) {
        tmem_row_to_swizzled_bf16(tH + lane_base, Hb, r);
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar_hb);
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool lin_tc_supported(int32_t dtype, int32_t Dk, int32_t Dv) { return dtype == CP_DT_BF16 && Dk == kD && Dv == kD; }

cudaError_t launch_lin_state_tc(const LinBlock* blocks, int32_t nblocks, int32_t H, int64_t T, const void* k,
                                const void* v, const float* g, float* states, cudaStream_t st) {
  LinTcParams p{};
  if (!make_map_3d(&p.tk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kD, H, T, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_3d(&p.tv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kD, H, T, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  p.blocks = blocks;
  p.g = g;
  p.states = states;
  p.H = H;
  p.err = device_error_word();
  const unsigned grid = unsigned(int64_t(nblocks) * H);
  if (grid == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(lin_state_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(kStateSmem));
  if (e != cudaSuccess) return e;
  lin_state_tc_kernel<<<grid, kStateThreads, kStateSmem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_lin_output_tc(const LinBlock* blocks, int32_t nblocks, int32_t H, int64_t T, float scale,
                                 const void* q, const void* k, const void* v, const float* g, const float* init,
                                 void* o, cudaStream_t st) {
  LinTcParams p{};
  if (!make_map_3d(&p.tq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kD, H, T, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_3d(&p.tk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kD, H, T, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_3d(&p.tv, v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kD, H, T, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  p.blocks = blocks;
  p.g = g;
  p.init = init;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.H = H;
  p.scale = scale;
  p.err = device_error_word();
  const unsigned grid = unsigned(int64_t(nblocks) * H);
  if (grid == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(lin_output_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(kOutSmem));
  if (e != cudaSuccess) return e;
  lin_output_tc_kernel<<<grid, kOutThreads, kOutSmem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace cpattn
