// simple_kernels.cu — bandwidth-bound kernels (shard permutation, LSE merge,
// backward pre/post-processing) and the CUDA-core attention path used for
// FP32 inputs and for head dims the tensor-core kernels do not cover.
#include <cuda_bf16.h>

#include <cmath>

#include "internal.h"
#include "plan_check.cuh"

namespace cpattn {
namespace {

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

// ----------------------------------------------------------------------------
// Shard permutation ("Ulysses与Ring-Attention详解" §4.2; "LLM context parallel
// production guide", 位置编码必须跟序列分片一起走).  The map is a list of
// contiguous chunk copies; every CTA copies 32 KiB pieces with 16-byte
// streaming loads, all loads of a piece issued before its stores.
// ----------------------------------------------------------------------------
constexpr int kPermThreads = 256;
constexpr int kPermUnroll = int(kPermutePiece / (16 * kPermThreads));  // 8

__global__ void __launch_bounds__(kPermThreads) permute_kernel(const CopySeg* __restrict__ segs,
                                                               int32_t nseg, int64_t npieces,
                                                               const char* __restrict__ in,
                                                               char* __restrict__ out) {
  for (int64_t piece = blockIdx.x; piece < npieces; piece += gridDim.x) {
    int lo = 0, hi = nseg - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (segs[mid].piece0 <= piece) lo = mid; else hi = mid - 1;
    }
    const CopySeg s = segs[lo];
    const int64_t off = (piece - s.piece0) * kPermutePiece;
    const int64_t n = s.bytes - off < kPermutePiece ? s.bytes - off : kPermutePiece;
    const int nv = int(n >> 4);
    const int4* src = reinterpret_cast<const int4*>(in + s.src + off);
    int4* dst = reinterpret_cast<int4*>(out + s.dst + off);
    int4 buf[kPermUnroll];
#pragma unroll
    for (int u = 0; u < kPermUnroll; ++u) {
      const int i = threadIdx.x + u * kPermThreads;
      if (i < nv) buf[u] = __ldcs(src + i);
    }
#pragma unroll
    for (int u = 0; u < kPermUnroll; ++u) {
      const int i = threadIdx.x + u * kPermThreads;
      if (i < nv) __stcs(dst + i, buf[u]);
    }
  }
}

// ----------------------------------------------------------------------------
// Ulysses all-to-all on one GPU ("Ulysses Context Parallelism 的工程取舍全记录"
// §1.2): sequence shards of every head <-> the whole sequence of H/C heads
// per virtual rank.  A sharded row s (token perm[s] in global order) holds C
// consecutive head groups of chunk16 16-byte words; group r goes to row
// perm[s] of rank r's [T, H/C, ...] block.  One warp per sharded row; the
// direction only swaps which side is read.
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(256) ulysses_a2a_kernel(const int32_t* __restrict__ perm, int64_t T,
                                                          int32_t C, int64_t chunk16,
                                                          const int4* __restrict__ in, int4* __restrict__ out,
                                                          int32_t inverse) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = int64_t(gridDim.x) * (blockDim.x >> 5);
  for (int64_t s = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; s < T; s += nwarps) {
    const int64_t g = perm[s];
    const int64_t srow = s * C * chunk16;
    for (int r = 0; r < C; ++r) {
      const int64_t sh = srow + int64_t(r) * chunk16;    // sharded side
      const int64_t uh = (int64_t(r) * T + g) * chunk16;  // head-sharded side
      const int64_t src = inverse ? uh : sh, dst = inverse ? sh : uh;
      for (int64_t i0 = 0; i0 < chunk16; i0 += 128) {
        int4 buf[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t i = i0 + lane + 32 * u;
          if (i < chunk16) buf[u] = __ldcs(in + src + i);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t i = i0 + lane + 32 * u;
          if (i < chunk16) __stcs(out + dst + i, buf[u]);
        }
      }
    }
  }
}

// Statistics [H, T] (sharded token order) <-> [H/C, C*T] (head h = r*H/C + j
// of rank r at row j, column r*T + perm[s]): the layout of the unsharded
// per-rank problem's lse.
__global__ void __launch_bounds__(256) ulysses_lse_kernel(const int32_t* __restrict__ perm, int64_t T,
                                                          int32_t C, int32_t H, const float* __restrict__ in,
                                                          float* __restrict__ out, int32_t inverse) {
  const int64_t n = int64_t(H) * T;
  const int32_t hc = H / C;
  for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < n; e += int64_t(gridDim.x) * blockDim.x) {
    const int64_t h = e / T, s = e - h * T;
    const int64_t r = h / hc, j = h - r * hc;
    const int64_t u = j * (C * T) + r * T + perm[s];
    if (inverse)
      out[e] = in[u];
    else
      out[u] = in[e];
  }
}

// ----------------------------------------------------------------------------
// LSE merge ("Ulysses与Ring-Attention详解" §4.1 update step, §4.2 lse formula).
// One warp per (row, head): lse = max + log1p(exp(-|a-b|)), weights
// exp(a - lse), exp(b - lse); -inf is the identity.
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(256) lse_merge_kernel(int64_t rows, int32_t hq, int32_t dv,
                                                        float* __restrict__ o_acc,
                                                        float* __restrict__ lse_acc,
                                                        const float* __restrict__ o_part,
                                                        const float* __restrict__ lse_part) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = int64_t(gridDim.x) * (blockDim.x >> 5);
  const int64_t total = rows * hq;
  for (int64_t w = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; w < total; w += nwarps) {
    const int64_t h = w / rows, t = w - h * rows;
    const float a = lse_acc[h * rows + t];
    const float b = __ldcs(lse_part + h * rows + t);
    const float m = fmaxf(a, b);
    if (m == -INFINITY) continue;  // both empty: accumulator stays (0, -inf)
    const float lse = m + log1pf(expf(-fabsf(a - b)));
    const float wa = expf(a - lse), wb = expf(b - lse);
    float4* oa = reinterpret_cast<float4*>(o_acc + (t * hq + h) * dv);
    const float4* ob = reinterpret_cast<const float4*>(o_part + (t * hq + h) * dv);
    for (int c = lane; c < (dv >> 2); c += 32) {
      float4 x = oa[c];
      const float4 y = __ldcs(ob + c);
      x.x = wa * x.x + wb * y.x;
      x.y = wa * x.y + wb * y.y;
      x.z = wa * x.z + wb * y.z;
      x.w = wa * x.w + wb * y.w;
      oa[c] = x;
    }
    if (lane == 0) lse_acc[h * rows + t] = lse;
  }
}

// ----------------------------------------------------------------------------
// Element access helpers for the CUDA-core path.
// ----------------------------------------------------------------------------
template <typename E> __device__ __forceinline__ float ldf(const E* p);
template <> __device__ __forceinline__ float ldf<float>(const float* p) { return *p; }
template <> __device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <typename E> __device__ __forceinline__ void stf(E* p, float x);
template <> __device__ __forceinline__ void stf<float>(float* p, float x) { *p = x; }
template <> __device__ __forceinline__ void stf<__nv_bfloat16>(__nv_bfloat16* p, float x) {
  *p = __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Query heads sharing one key/value head get adjacent block indices.
__device__ __forceinline__ int head_of_slot(int slot, const AttnArgs& a) {
  const int G = a.hq / a.hkv;
  const int kv = slot / G, g = slot - kv * G;
  return a.gqa_interleaved ? g * a.hkv + kv : kv * G + g;
}
__device__ __forceinline__ int kv_of_head(int h, const AttnArgs& a) {
  return a.gqa_interleaved ? h % a.hkv : h / (a.hq / a.hkv);
}

constexpr int kMaxPerLane = 8;  // head dims up to 256 spread over a warp

// Forward, one warp per query row, online softmax over the visible keys of
// the tile's runs (exact in real arithmetic; FP32 throughout).
template <typename E>
__global__ void __launch_bounds__(256) simt_fwd_kernel(const AttnArgs a) {
  const int tile_idx = blockIdx.x / a.hq;
  const int h = head_of_slot(blockIdx.x - tile_idx * a.hq, a);
  const int kvh = kv_of_head(h, a);
  if (a.debug && !debug_plan_ok(a, tile_idx, h, kvh, false, a.err)) return;
  const TileDesc t = a.tiles[tile_idx];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const E* q = static_cast<const E*>(a.q);
  const E* k = static_cast<const E*>(a.k);
  const E* v = static_cast<const E*>(a.v);
  for (int r = warp; r < t.nrows; r += (blockDim.x >> 5)) {
    const int64_t qrow = int64_t(t.row0) + r;
    const int qpos = t.pos0 + r;
    float qv[kMaxPerLane], acc[kMaxPerLane];
#pragma unroll
    for (int e = 0; e < kMaxPerLane; ++e) {
      const int c = lane + 32 * e;
      qv[e] = c < a.d_qk ? ldf(q + (qrow * a.hq + h) * a.d_qk + c) : 0.f;
      acc[e] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    for (int ri = 0; ri < t.range_count; ++ri) {
      const RangeDesc R = a.ranges[t.range_begin + ri];
      int lim = R.nrows;
      if (a.causal) lim = min(lim, qpos - R.pos0 + 1);
      for (int j = 0; j < lim; ++j) {
        const int64_t krow = int64_t(R.row0) + j;
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < kMaxPerLane; ++e) {
          const int c = lane + 32 * e;
          if (c < a.d_qk) s += qv[e] * ldf(k + (krow * a.hkv + kvh) * a.d_qk + c);
        }
        s = warp_sum(s) * a.scale;
        const float mn = fmaxf(m, s);
        const float alpha = expf(m - mn);
        const float p = expf(s - mn);
        l = l * alpha + p;
#pragma unroll
        for (int e = 0; e < kMaxPerLane; ++e) {
          const int c = lane + 32 * e;
          if (c < a.d_v) acc[e] = acc[e] * alpha + p * ldf(v + (krow * a.hkv + kvh) * a.d_v + c);
        }
        m = mn;
      }
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    float lse = l > 0.f ? m + logf(l) : -INFINITY;
    const int64_t orow = a.block_mode ? int64_t(t.out_row0) + r : qrow;
    // block_mode 2: merge into the fp32 accumulator (the lse merge of
    // "Ulysses与Ring-Attention详解" §4.2, -inf the identity)
    float wa = 0.f, wb = inv;
    if (a.block_mode == 2) {
      const float la = a.lse[int64_t(h) * a.lse_stride + orow];
      const float mm = fmaxf(la, lse);
      if (mm == -INFINITY) {
        wa = 1.f;
        wb = 0.f;
      } else {
        const float lo = mm + log1pf(expf(-fabsf(la - lse)));
        wa = expf(la - lo);
        wb = expf(lse - lo) * inv;
        lse = lo;
      }
      __syncwarp();  // every lane has read the old lse before lane 0 overwrites it
    }
#pragma unroll
    for (int e = 0; e < kMaxPerLane; ++e) {
      const int c = lane + 32 * e;
      if (c < a.d_v) {
        float* of = static_cast<float*>(a.out) + (orow * a.hq + h) * a.d_v + c;
        if (a.block_mode == 2)
          *of = wa * *of + wb * acc[e];
        else if (a.block_mode)
          *of = acc[e] * inv;
        else
          stf(static_cast<E*>(a.out) + (orow * a.hq + h) * a.d_v + c, acc[e] * inv);
      }
    }
    if (lane == 0) a.lse[int64_t(h) * a.lse_stride + orow] = lse;
  }
}

// D = rowsum(dout * o) in FP32, one warp per (row, head); rows of one token
// are adjacent in memory, so consecutive warps read consecutive bytes.
template <typename E>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const AttnArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = int64_t(gridDim.x) * (blockDim.x >> 5);
  const int64_t total = a.T * a.hq;
  const E* o = static_cast<const E*>(a.o);
  const E* dout = static_cast<const E*>(a.dout);
  for (int64_t w = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; w < total; w += nwarps) {
    const int64_t t = w / a.hq, h = w - t * a.hq;
    const E* po = o + w * a.d_v;
    const E* pd = dout + w * a.d_v;
    float s = 0.f;
    for (int c = lane; c < a.d_v; c += 32) s += ldf(po + c) * ldf(pd + c);
    s = warp_sum(s);
    if (lane == 0) a.dpsum[h * a.T + t] = s;
  }
}

// The same for bf16 rows of 8*DV8 values: DV8 lanes per row, one 16-byte
// load of o and of dout each, so a warp covers 32/DV8 rows at a time.  Rows
// are taken in (head, token) order, so the D values a warp writes sit next
// to each other.
template <int DV8>
__global__ void __launch_bounds__(256) bwd_preprocess_bf16_kernel(const AttnArgs a) {
  constexpr int kRows = 32 / DV8;  // rows per warp
  const int lane = threadIdx.x & 31, sub = lane / DV8, part = lane - sub * DV8;
  const int64_t nrows = a.T * a.hq;
  const int64_t step = int64_t(gridDim.x) * (blockDim.x >> 5) * kRows;
  for (int64_t i0 = (int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5)) * kRows; i0 < nrows; i0 += step) {
    const int64_t i = i0 + sub;  // (head, token) pair of this lane group
    float s = 0.f;
    int64_t h = 0, t = 0;
    if (i < nrows) {
      h = i / a.T;
      t = i - h * a.T;
      const int64_t off = (t * a.hq + h) * (8 * DV8) + 8 * part;
      const uint4 ov = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.o) + off);
      const uint4 dv = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.dout) + off);
      const uint32_t* o32 = reinterpret_cast<const uint32_t*>(&ov);
      const uint32_t* d32 = reinterpret_cast<const uint32_t*>(&dv);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&o32[e]));
        const float2 df = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&d32[e]));
        s = fmaf(of.x, df.x, s);
        s = fmaf(of.y, df.y, s);
      }
    }
#pragma unroll
    for (int m = DV8 / 2; m > 0; m >>= 1) s += __shfl_xor_sync(0xffffffffu, s, m);
    if (part == 0 && i < nrows) a.dpsum[h * a.T + t] = s;
  }
}

// dq for one query row per warp (query-major plan).
template <typename E>
__global__ void __launch_bounds__(256) simt_bwd_dq_kernel(const AttnArgs a) {
  const int tile_idx = blockIdx.x / a.hq;
  const int h = head_of_slot(blockIdx.x - tile_idx * a.hq, a);
  const int kvh = kv_of_head(h, a);
  if (a.debug && !debug_plan_ok(a, tile_idx, h, kvh, false, a.err)) return;
  const TileDesc t = a.tiles[tile_idx];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const E* q = static_cast<const E*>(a.q);
  const E* k = static_cast<const E*>(a.k);
  const E* v = static_cast<const E*>(a.v);
  const E* dout = static_cast<const E*>(a.dout);
  for (int r = warp; r < t.nrows; r += (blockDim.x >> 5)) {
    const int64_t qrow = int64_t(t.row0) + r;
    const int qpos = t.pos0 + r;
    const float lse = a.lse_in[int64_t(h) * a.T + qrow];
    const float Di = a.dpsum[int64_t(h) * a.T + qrow];
    float qv[kMaxPerLane], dov[kMaxPerLane], acc[kMaxPerLane];
#pragma unroll
    for (int e = 0; e < kMaxPerLane; ++e) {
      const int c = lane + 32 * e;
      qv[e] = c < a.d_qk ? ldf(q + (qrow * a.hq + h) * a.d_qk + c) : 0.f;
      dov[e] = c < a.d_v ? ldf(dout + (qrow * a.hq + h) * a.d_v + c) : 0.f;
      acc[e] = 0.f;
    }
    for (int ri = 0; ri < t.range_count; ++ri) {
      const RangeDesc R = a.ranges[t.range_begin + ri];
      int lim = R.nrows;
      if (a.causal) lim = min(lim, qpos - R.pos0 + 1);
      for (int j = 0; j < lim; ++j) {
        const int64_t krow = int64_t(R.row0) + j;
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int e = 0; e < kMaxPerLane; ++e) {
          const int c = lane + 32 * e;
          if (c < a.d_qk) s += qv[e] * ldf(k + (krow * a.hkv + kvh) * a.d_qk + c);
          if (c < a.d_v) dp += dov[e] * ldf(v + (krow * a.hkv + kvh) * a.d_v + c);
        }
        s = warp_sum(s) * a.scale;
        dp = warp_sum(dp);
        const float p = expf(s - lse);
        const float ds = p * (dp - Di);
#pragma unroll
        for (int e = 0; e < kMaxPerLane; ++e) {
          const int c = lane + 32 * e;
          if (c < a.d_qk) acc[e] += ds * ldf(k + (krow * a.hkv + kvh) * a.d_qk + c);
        }
      }
    }
#pragma unroll
    for (int e = 0; e < kMaxPerLane; ++e) {
      const int c = lane + 32 * e;
      if (c < a.d_qk) stf(static_cast<E*>(a.dq) + (qrow * a.hq + h) * a.d_qk + c, acc[e] * a.scale);
    }
  }
}

// dk, dv for one key row per warp (key-major plan), summed over the query
// heads of the key's GQA group.
template <typename E>
__global__ void __launch_bounds__(256) simt_bwd_dkdv_kernel(const AttnArgs a) {
  const int tile_idx = blockIdx.x / a.hkv;
  const int kvh = blockIdx.x - tile_idx * a.hkv;
  const int G = a.hq / a.hkv;
  if (a.debug && !debug_plan_ok(a, tile_idx, kvh, kvh, true, a.err)) return;
  const TileDesc t = a.tiles[tile_idx];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const E* q = static_cast<const E*>(a.q);
  const E* k = static_cast<const E*>(a.k);
  const E* v = static_cast<const E*>(a.v);
  const E* dout = static_cast<const E*>(a.dout);
  for (int r = warp; r < t.nrows; r += (blockDim.x >> 5)) {
    const int64_t krow = int64_t(t.row0) + r;
    const int kpos = t.pos0 + r;
    float kv_[kMaxPerLane], vv[kMaxPerLane], dk[kMaxPerLane], dv[kMaxPerLane];
#pragma unroll
    for (int e = 0; e < kMaxPerLane; ++e) {
      const int c = lane + 32 * e;
      kv_[e] = c < a.d_qk ? ldf(k + (krow * a.hkv + kvh) * a.d_qk + c) : 0.f;
      vv[e] = c < a.d_v ? ldf(v + (krow * a.hkv + kvh) * a.d_v + c) : 0.f;
      dk[e] = 0.f;
      dv[e] = 0.f;
    }
    for (int g = 0; g < G; ++g) {
      const int h = a.gqa_interleaved ? g * a.hkv + kvh : kvh * G + g;
      for (int ri = 0; ri < t.range_count; ++ri) {
        const RangeDesc R = a.ranges[t.range_begin + ri];
        const int i0 = a.causal ? max(0, kpos - R.pos0) : 0;
        for (int i = i0; i < R.nrows; ++i) {
          const int64_t qrow = int64_t(R.row0) + i;
          const float lse = a.lse_in[int64_t(h) * a.T + qrow];
          const float Di = a.dpsum[int64_t(h) * a.T + qrow];
          float s = 0.f, dp = 0.f;
          float qv[kMaxPerLane], dov[kMaxPerLane];
#pragma unroll
          for (int e = 0; e < kMaxPerLane; ++e) {
            const int c = lane + 32 * e;
            qv[e] = c < a.d_qk ? ldf(q + (qrow * a.hq + h) * a.d_qk + c) : 0.f;
            dov[e] = c < a.d_v ? ldf(dout + (qrow * a.hq + h) * a.d_v + c) : 0.f;
            s += qv[e] * kv_[e];
            dp += dov[e] * vv[e];
          }
          s = warp_sum(s) * a.scale;
          dp = warp_sum(dp);
          const float p = expf(s - lse);
          const float ds = p * (dp - Di);
#pragma unroll
          for (int e = 0; e < kMaxPerLane; ++e) {
            dk[e] += ds * qv[e];
            dv[e] += p * dov[e];
          }
        }
      }
    }
#pragma unroll
    for (int e = 0; e < kMaxPerLane; ++e) {
      const int c = lane + 32 * e;
      if (c < a.d_qk) stf(static_cast<E*>(a.dk) + (krow * a.hkv + kvh) * a.d_qk + c, dk[e] * a.scale);
      if (c < a.d_v) stf(static_cast<E*>(a.dv) + (krow * a.hkv + kvh) * a.d_v + c, dv[e]);
    }
  }
}

int64_t grid_for(int64_t work_items, int per_block) {
  int64_t g = (work_items + per_block - 1) / per_block;
  const int64_t cap = int64_t(sm_count()) * 16;
  if (g > cap) g = cap;
  return g < 1 ? 1 : g;
}

}  // namespace

cudaError_t launch_permute(const CopySeg* segs, int32_t nseg, int64_t npieces, const void* in,
                           void* out, cudaStream_t st, int32_t ctas_per_sm) {
  if (npieces == 0) return cudaSuccess;
  int64_t grid = npieces;
  const int64_t cap = int64_t(sm_count()) * ctas_per_sm;
  if (grid > cap) grid = cap;
  permute_kernel<<<unsigned(grid), kPermThreads, 0, st>>>(segs, nseg, npieces,
                                                          static_cast<const char*>(in),
                                                          static_cast<char*>(out));
  return cudaGetLastError();
}

cudaError_t launch_ulysses_a2a(const int32_t* perm, int64_t T, int32_t C, int64_t chunk_bytes, const void* in,
                               void* out, int32_t inverse, cudaStream_t st) {
  const int64_t grid = grid_for(T, 8);
  ulysses_a2a_kernel<<<unsigned(grid), 256, 0, st>>>(perm, T, C, chunk_bytes / 16, static_cast<const int4*>(in),
                                                     static_cast<int4*>(out), inverse);
  return cudaGetLastError();
}

cudaError_t launch_ulysses_lse(const int32_t* perm, int64_t T, int32_t C, int32_t H, const float* in, float* out,
                               int32_t inverse, cudaStream_t st) {
  const int64_t grid = grid_for(int64_t(H) * T, 256);
  ulysses_lse_kernel<<<unsigned(grid), 256, 0, st>>>(perm, T, C, H, in, out, inverse);
  return cudaGetLastError();
}

// fp32 -> bf16 (round to nearest even), 8 elements per thread and step.
__global__ void __launch_bounds__(256) cast_bf16_kernel(const float4* __restrict__ in, uint4* __restrict__ out,
                                                        int64_t n8) {
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += int64_t(gridDim.x) * blockDim.x) {
    const float4 x = __ldcs(in + 2 * i), y = __ldcs(in + 2 * i + 1);
    uint4 r;
    __nv_bfloat162 b;
    b = __floats2bfloat162_rn(x.x, x.y);
    r.x = *reinterpret_cast<uint32_t*>(&b);
    b = __floats2bfloat162_rn(x.z, x.w);
    r.y = *reinterpret_cast<uint32_t*>(&b);
    b = __floats2bfloat162_rn(y.x, y.y);
    r.z = *reinterpret_cast<uint32_t*>(&b);
    b = __floats2bfloat162_rn(y.z, y.w);
    r.w = *reinterpret_cast<uint32_t*>(&b);
    out[i] = r;
  }
}

cudaError_t launch_cast_bf16(const float* in, void* out, int64_t n, cudaStream_t st) {
  const int64_t n8 = n / 8;
  if (n8 == 0) return cudaSuccess;
  const int64_t grid = grid_for(n8, 256);
  cast_bf16_kernel<<<unsigned(grid), 256, 0, st>>>(reinterpret_cast<const float4*>(in), static_cast<uint4*>(out), n8);
  return cudaGetLastError();
}

cudaError_t launch_lse_merge(int64_t rows, int32_t hq, int32_t dv, float* o_acc, float* lse_acc,
                             const float* o_part, const float* lse_part, cudaStream_t st) {
  const int64_t grid = grid_for(rows * hq, 8);
  lse_merge_kernel<<<unsigned(grid), 256, 0, st>>>(rows, hq, dv, o_acc, lse_acc, o_part, lse_part);
  return cudaGetLastError();
}

cudaError_t launch_simt_fwd(const AttnArgs& args, int32_t dtype, cudaStream_t st) {
  AttnArgs a = args;
  a.err = device_error_word();
  const int64_t grid = int64_t(a.num_tiles) * a.hq;
  if (grid == 0) return cudaSuccess;
  if (dtype == CP_DT_F32)
    simt_fwd_kernel<float><<<unsigned(grid), 256, 0, st>>>(a);
  else
    simt_fwd_kernel<__nv_bfloat16><<<unsigned(grid), 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_bwd_preprocess(const AttnArgs& a, int32_t dtype, cudaStream_t st) {
  if (dtype != CP_DT_F32 && a.d_v == 128 && ((reinterpret_cast<uintptr_t>(a.o) | reinterpret_cast<uintptr_t>(a.dout)) & 15) == 0) {
    bwd_preprocess_bf16_kernel<16><<<unsigned(grid_for(a.T * a.hq, 16)), 256, 0, st>>>(a);
    return cudaGetLastError();
  }
  const int64_t grid = grid_for(a.T * a.hq, 8);
  if (dtype == CP_DT_F32)
    bwd_preprocess_kernel<float><<<unsigned(grid), 256, 0, st>>>(a);
  else
    bwd_preprocess_kernel<__nv_bfloat16><<<unsigned(grid), 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_simt_bwd_dq(const AttnArgs& args, int32_t dtype, cudaStream_t st) {
  AttnArgs a = args;
  a.err = device_error_word();
  const int64_t grid = int64_t(a.num_tiles) * a.hq;
  if (grid == 0) return cudaSuccess;
  if (dtype == CP_DT_F32)
    simt_bwd_dq_kernel<float><<<unsigned(grid), 256, 0, st>>>(a);
  else
    simt_bwd_dq_kernel<__nv_bfloat16><<<unsigned(grid), 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_simt_bwd_dkdv(const AttnArgs& args, int32_t dtype, cudaStream_t st) {
  AttnArgs a = args;
  a.err = device_error_word();
  const int64_t grid = int64_t(a.num_tiles) * a.hkv;
  if (grid == 0) return cudaSuccess;
  if (dtype == CP_DT_F32)
    simt_bwd_dkdv_kernel<float><<<unsigned(grid), 256, 0, st>>>(a);
  else
    simt_bwd_dkdv_kernel<__nv_bfloat16><<<unsigned(grid), 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace cpattn
