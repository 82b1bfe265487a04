// linear_attn.cu — decayed linear attention with AllGather context
// parallelism on one GPU ("超长上下文训练速度翻倍秘籍": the recurrence
// h_t = alpha h_{t-1} + K_t^T V_t, O_t = Q_t h_t; the AllGather CP section:
// rank-local hidden states and outputs, the gathered states ([B, H, D, D])
// combined by the decayed prefix kv_state = kv_state * decay + cur into every
// rank's initial state, and the output correction (q * decay) @ init_state,
// made a vectorised prefix and a fused correction instead of per-rank and
// per-sub-sequence loops).
//
// With alpha = exp(g) per head, every rank piece is cut into blocks of at most
// kLinBlock tokens (the unit of parallel work), and three kernels run:
//   lin_state_kernel  — per (block, head): S = sum_s alpha^(n-1-s) k_s^T v_s,
//                        the hidden state at the block end from a zero start;
//   lin_prefix_kernel — per (sequence, head): the decayed prefix over the
//                        gathered states in sequence order (ranks in order,
//                        blocks in order inside a rank): init_b = cur,
//                        cur = alpha^(n_b) cur + S_b; at rank granularity this
//                        is the page's state recovery;
//   lin_output_kernel — per (block, head): chunked decayed attention of the
//                        block started from init_b, i.e. the local output plus
//                        the page's correction, in one pass.
// Here: FP32 CUDA-core arithmetic, register-tiled (head dims multiples of 8,
// up to 128), bf16 or fp32 tensors.  bf16 with 128-wide heads takes the
// tensor-core state and output passes of linear_attn_tc.cu instead.
#include <cuda_bf16.h>

#include "internal.h"

namespace cpattn {
namespace {

constexpr int kLinB = 64;      // tokens per chunk
constexpr int kLinThreads = 256;
constexpr int kLdPad = 1;      // Q/K rows padded to an odd stride (bank spread)

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Rows [row0, row0 + n) of a [T, H, D] tensor, head h, into smem rows of
// `ld` floats as fp32, each row times w(row); zeros past n.
template <typename T, typename W>
__device__ __forceinline__ void load_rows(float* dst, int ld, const T* src, int64_t row0, int n, int H, int h, int D,
                                          W w) {
  for (int e = threadIdx.x; e < kLinB * D; e += blockDim.x) {
    const int t = e / D, d = e - t * D;
    dst[t * ld + d] = t < n ? to_f(src[((row0 + t) * H + h) * D + d]) * w(t) : 0.f;
  }
}

// acc[8][8] += sum_s (w_s K[s][d_i]) V[s][j_jj], thread tile rows ty*8.., cols tx*8..
__device__ __forceinline__ void kv_outer(float (&acc)[8][8], const float* Ks, int ldk, const float* Vs, int ldv,
                                         const float* Ws, int n, int ty, int tx, int Dk, int Dv) {
  const int d0 = ty * 8, j0 = tx * 8;
  if (d0 >= Dk || j0 >= Dv) return;
  for (int s = 0; s < n; ++s) {
    const float w = Ws ? Ws[s] : 1.f;
    float kr[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) kr[i] = Ks[s * ldk + d0 + i] * w;
    const float4 v0 = *reinterpret_cast<const float4*>(Vs + s * ldv + j0);
    const float4 v1 = *reinterpret_cast<const float4*>(Vs + s * ldv + j0 + 4);
    const float vr[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(kr[i], vr[j], acc[i][j]);
  }
}

template <typename T>
__global__ void __launch_bounds__(kLinThreads) lin_state_kernel(const LinBlock* __restrict__ blocks, int32_t H,
                                                                 int32_t Dk, int32_t Dv, const T* __restrict__ k,
                                                                 const T* __restrict__ v, const float* __restrict__ g,
                                                                 float* __restrict__ states) {
  extern __shared__ __align__(16) float lsm[];
  const int ldk = Dk + kLdPad;
  float* Ks = lsm;                 // [kLinB][Dk + 1]
  float* Vs = Ks + kLinB * ldk;    // [kLinB][Dv]  (offset rounded to 4 floats below)
  Vs = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(Vs) + 15) & ~uintptr_t(15));
  const int b = blockIdx.x / H, h = blockIdx.x - (blockIdx.x / H) * H;
  const LinBlock bl = blocks[b];
  const float gh = g[h];
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  float acc[8][8] = {};
  for (int c0 = 0; c0 < bl.len; c0 += kLinB) {
    const int n = min(kLinB, bl.len - c0);
    const int last = bl.len - 1 - c0;  // exponent of chunk row 0
    __syncthreads();
    load_rows(Ks, ldk, k, bl.row0 + c0, n, H, h, Dk, [&](int t) { return __expf(gh * float(last - t)); });
    load_rows(Vs, Dv, v, bl.row0 + c0, n, H, h, Dv, [](int) { return 1.f; });
    __syncthreads();
    kv_outer(acc, Ks, ldk, Vs, Dv, nullptr, n, ty, tx, Dk, Dv);
  }
  float* out = states + (int64_t(b) * H + h) * Dk * Dv;
  if (ty * 8 < Dk && tx * 8 < Dv)
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) out[(ty * 8 + i) * Dv + tx * 8 + j] = acc[i][j];
}

// One thread per (sequence, head, state element): blocks of sequence s in
// order are [seq_begin[s], seq_begin[s+1]); the scan over them is serial per
// element, the elements are spread over the whole grid.
constexpr int kPrefixThreads = 256;
__global__ void __launch_bounds__(kPrefixThreads) lin_prefix_kernel(const LinBlock* __restrict__ blocks,
                                                                     const int32_t* __restrict__ seq_begin, int32_t H,
                                                                     int32_t DD, const float* __restrict__ g,
                                                                     const float* __restrict__ states,
                                                                     float* __restrict__ init) {
  const int per_sh = (DD + kPrefixThreads - 1) / kPrefixThreads;  // CTAs per (sequence, head)
  const int sh = blockIdx.x / per_sh;
  const int e = (blockIdx.x - sh * per_sh) * kPrefixThreads + threadIdx.x;
  if (e >= DD) return;
  const int s = sh / H, h = sh - (sh / H) * H;
  const float gh = g[h];
  const int b0 = seq_begin[s], b1 = seq_begin[s + 1];
  float cur = 0.f;
  for (int b = b0; b < b1; ++b) {
    const int64_t idx = (int64_t(b) * H + h) * DD + e;
    init[idx] = cur;
    cur = __expf(gh * float(blocks[b].len)) * cur + __ldcs(states + idx);
  }
}

template <typename T>
__global__ void __launch_bounds__(kLinThreads) lin_output_kernel(const LinBlock* __restrict__ blocks, int32_t H,
                                                                  int32_t Dk, int32_t Dv, float scale,
                                                                  const T* __restrict__ q, const T* __restrict__ k,
                                                                  const T* __restrict__ v, const float* __restrict__ g,
                                                                  const float* __restrict__ init, T* __restrict__ o) {
  extern __shared__ __align__(16) float lsm[];
  const int ldq = Dk + 4;              // 16-byte rows, rows ty*4 and ty*4+4 on different banks
  const int ldk = Dk + kLdPad;
  constexpr int lda = kLinB + 4;
  float* Hs = lsm;                     // [Dk][Dv] carried state
  float* Vs = Hs + Dk * Dv;            // [kLinB][Dv]
  float* Qs = Vs + kLinB * Dv;         // [kLinB][Dk + 4]
  float* As = Qs + kLinB * ldq;        // [kLinB][kLinB + 4], A transposed: As[s][t]
  float* Ws = As + kLinB * lda;        // [kLinB] alpha^(n-1-s)
  float* Ds = Ws + kLinB;              // [kLinB] alpha^(t+1)
  float* Ks = Ds + kLinB;              // [kLinB][Dk + 1]
  const int b = blockIdx.x / H, h = blockIdx.x - (blockIdx.x / H) * H;
  const LinBlock bl = blocks[b];
  const float gh = g[h];
  const int DD = Dk * Dv;
  const float* h0 = init + (int64_t(b) * H + h) * DD;
  for (int e = threadIdx.x; e < DD; e += blockDim.x) Hs[e] = h0[e];
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  for (int c0 = 0; c0 < bl.len; c0 += kLinB) {
    const int n = min(kLinB, bl.len - c0);
    __syncthreads();  // the previous chunk is finished with every buffer
    load_rows(Qs, ldq, q, bl.row0 + c0, n, H, h, Dk, [](int) { return 1.f; });
    load_rows(Ks, ldk, k, bl.row0 + c0, n, H, h, Dk, [](int) { return 1.f; });
    load_rows(Vs, Dv, v, bl.row0 + c0, n, H, h, Dv, [](int) { return 1.f; });
    for (int t = threadIdx.x; t < kLinB; t += blockDim.x) {
      Ws[t] = t < n ? __expf(gh * float(n - 1 - t)) : 0.f;
      Ds[t] = __expf(gh * float(t + 1));
    }
    __syncthreads();
    // ---- A[t][s] = (q_t . k_s) alpha^(t-s), s <= t (4x4 tile: t = ty*4+i, s = tx*4+j)
    {
      float a[4][4] = {};
      for (int d = 0; d < Dk; ++d) {
        float qv[4], kv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          qv[i] = Qs[(ty * 4 + i) * ldq + d];
          kv[i] = Ks[(tx * 4 + i) * ldk + d];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) a[i][j] = fmaf(qv[i], kv[j], a[i][j]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int t = ty * 4 + i, s = tx * 4 + j;
          As[s * lda + t] = (s <= t) ? a[i][j] * __expf(gh * float(t - s)) : 0.f;
        }
    }
    __syncthreads();
    // ---- O[t][j] = scale (sum_s A[t][s] V[s][j] + alpha^(t+1) sum_d Q[t][d] H[d][j])
    //      (4x8 tile: t = ty*4+i, j = tx*8+jj)
    if (tx * 8 < Dv) {
      const int j0 = tx * 8;
      float x[4][8] = {}, y[4][8] = {};
      for (int s = 0; s < kLinB; ++s) {
        const float4 av = *reinterpret_cast<const float4*>(As + s * lda + ty * 4);
        const float ar[4] = {av.x, av.y, av.z, av.w};
        const float4 v0 = *reinterpret_cast<const float4*>(Vs + s * Dv + j0);
        const float4 v1 = *reinterpret_cast<const float4*>(Vs + s * Dv + j0 + 4);
        const float vr[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) x[i][jj] = fmaf(ar[i], vr[jj], x[i][jj]);
      }
      for (int d = 0; d < Dk; ++d) {
        float qr[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) qr[i] = Qs[(ty * 4 + i) * ldq + d];
        const float4 h0v = *reinterpret_cast<const float4*>(Hs + d * Dv + j0);
        const float4 h1v = *reinterpret_cast<const float4*>(Hs + d * Dv + j0 + 4);
        const float hr[8] = {h0v.x, h0v.y, h0v.z, h0v.w, h1v.x, h1v.y, h1v.z, h1v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) y[i][jj] = fmaf(qr[i], hr[jj], y[i][jj]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = ty * 4 + i;
        if (t < n) {
          T* dst = o + ((bl.row0 + c0 + t) * int64_t(H) + h) * Dv + j0;
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) dst[jj] = from_f<T>(scale * (x[i][jj] + Ds[t] * y[i][jj]));
        }
      }
    }
    __syncthreads();  // every thread read Hs before it is updated
    // ---- H = alpha^n H + sum_s alpha^(n-1-s) k_s^T v_s (8x8 tile: d = ty*8+i, j = tx*8+jj)
    {
      float acc[8][8] = {};
      kv_outer(acc, Ks, ldk, Vs, Dv, Ws, n, ty, tx, Dk, Dv);
      const float an = __expf(gh * float(n));
      if (ty * 8 < Dk && tx * 8 < Dv)
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            float* p = Hs + (ty * 8 + i) * Dv + tx * 8 + jj;
            *p = an * *p + acc[i][jj];
          }
    }
  }
}

size_t state_smem(int32_t Dk, int32_t Dv) {
  return sizeof(float) * (size_t(kLinB) * (Dk + kLdPad) + 4 + size_t(kLinB) * Dv);
}

}  // namespace

size_t lin_output_smem(int32_t Dk, int32_t Dv) {
  return sizeof(float) * (size_t(Dk) * Dv + size_t(kLinB) * Dv + size_t(kLinB) * (Dk + 4) +
                          size_t(kLinB) * (kLinB + 4) + 2 * kLinB + size_t(kLinB) * (Dk + kLdPad));
}

cudaError_t launch_lin_attn(const LinBlock* blocks, int32_t nblocks, const int32_t* seq_begin, int32_t S, int32_t H,
                            int64_t T, int32_t Dk, int32_t Dv, float scale, int32_t dtype, const void* q,
                            const void* k, const void* v, const float* g, float* states, float* init, void* o,
                            cudaStream_t st) {
  if (Dk > 128 || Dv > 128 || Dk % 8 || Dv % 8) return cudaErrorInvalidValue;
  const unsigned grid = unsigned(int64_t(nblocks) * H);
  if (grid == 0) return cudaSuccess;
  const int per_sh = (Dk * Dv + kPrefixThreads - 1) / kPrefixThreads;
  if (lin_tc_supported(dtype, Dk, Dv)) {
    cudaError_t e = launch_lin_state_tc(blocks, nblocks, H, T, k, v, g, states, st);
    if (e != cudaSuccess) return e;
    lin_prefix_kernel<<<unsigned(int64_t(S) * H * per_sh), kPrefixThreads, 0, st>>>(blocks, seq_begin, H, Dk * Dv, g,
                                                                                   states, init);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return launch_lin_output_tc(blocks, nblocks, H, T, scale, q, k, v, g, init, o, st);
  }
  const size_t sm_state = state_smem(Dk, Dv), sm_out = lin_output_smem(Dk, Dv);
  auto run = [&](auto ks, auto ko, auto tag) -> cudaError_t {
    using E = decltype(tag);
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sm_state))) != cudaSuccess ||
        (e = cudaFuncSetAttribute(ko, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sm_out))) != cudaSuccess)
      return e;
    ks<<<grid, kLinThreads, sm_state, st>>>(blocks, H, Dk, Dv, static_cast<const E*>(k), static_cast<const E*>(v), g,
                                            states);
    lin_prefix_kernel<<<unsigned(int64_t(S) * H * per_sh), kPrefixThreads, 0, st>>>(blocks, seq_begin, H, Dk * Dv, g,
                                                                                   states, init);
    ko<<<grid, kLinThreads, sm_out, st>>>(blocks, H, Dk, Dv, scale, static_cast<const E*>(q),
                                          static_cast<const E*>(k), static_cast<const E*>(v), g, init,
                                          static_cast<E*>(o));
    return cudaGetLastError();
  };
  if (dtype == CP_DT_BF16)
    return run(lin_state_kernel<__nv_bfloat16>, lin_output_kernel<__nv_bfloat16>, __nv_bfloat16{});
  return run(lin_state_kernel<float>, lin_output_kernel<float>, float{});
}

}  // namespace cpattn
