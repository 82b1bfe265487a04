// linear_attn.cu — decayed linear attention with AllGather context
// parallelism on one GPU ("超长上下文训练速度翻倍秘籍": the recurrence
// h_t = alpha h_{t-1} + K_t^T V_t, O_t = Q_t h_t; the AllGather CP section:
// rank-local hidden states and outputs, the gathered states ([B, H, D, D])
// combined by the decayed prefix kv_state = kv_state * decay + cur into every
// rank's initial state, and the output correction (q * decay) @ init_state,
// made a vectorised prefix and a fused correction instead of per-rank and
// per-sub-sequence loops).
//
// With alpha = exp(g) per head, three kernels:
//   lin_state_kernel  — per (piece, head): S = sum_s alpha^(n-1-s) k_s^T v_s,
//                        the hidden state at the piece end from a zero start
//                        (one decay-weighted K^T V product);
//   lin_prefix_kernel — per (sequence, head): init_0 = 0,
//                        init_{r+1} = alpha^(n_r) init_r + S_r;
//   lin_output_kernel — per (piece, head): chunked decayed attention of the
//                        piece started from init_r, which equals the local
//                        output plus the page's correction, in one pass.
// FP32 CUDA-core arithmetic (head dims up to 128); bf16 or fp32 in and out.
#include <cuda_bf16.h>

#include "internal.h"

namespace cpattn {
namespace {

constexpr int kLinB = 64;      // tokens per chunk
constexpr int kLinMaxD = 128;  // head dims up to 128
constexpr int kLinThreads = 256;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Rows [row0, row0 + n) of a [T, H, D] tensor, head h, into smem rows of
// `ld` floats (ld >= D) as fp32, each row multiplied by w(row), zero past n.
template <typename T, typename W>
__device__ __forceinline__ void load_rows(float* dst, int ld, const T* src, int64_t row0, int n, int H, int h, int D,
                                          W w) {
  for (int e = threadIdx.x; e < kLinB * D; e += blockDim.x) {
    const int t = e / D, d = e - t * D;
    dst[t * ld + d] = t < n ? to_f(src[((row0 + t) * H + h) * D + d]) * w(t) : 0.f;
  }
}

template <typename T>
__global__ void __launch_bounds__(kLinThreads) lin_state_kernel(const LinPiece* __restrict__ pieces, int32_t H,
                                                                 int32_t Dk, int32_t Dv, const T* __restrict__ k,
                                                                 const T* __restrict__ v, const float* __restrict__ g,
                                                                 float* __restrict__ states) {
  extern __shared__ float lsm[];
  float* Ks = lsm;                  // [kLinB][Dk]
  float* Vs = lsm + kLinB * Dk;     // [kLinB][Dv]
  const int p = blockIdx.x / H, h = blockIdx.x - (blockIdx.x / H) * H;
  const LinPiece pc = pieces[p];
  const float gh = g[h];
  // thread (ty, tx) owns S rows ty*8.. and columns tx*8..
  const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
  float acc[8][8] = {};
  for (int c0 = 0; c0 < pc.len; c0 += kLinB) {
    const int n = min(kLinB, pc.len - c0);
    const int last = pc.len - 1 - c0;  // exponent of row 0 of this chunk
    load_rows(Ks, Dk, k, pc.row0 + c0, n, H, h, Dk, [&](int t) { return __expf(gh * float(last - t)); });
    load_rows(Vs, Dv, v, pc.row0 + c0, n, H, h, Dv, [](int) { return 1.f; });
    __syncthreads();
    for (int s = 0; s < n; ++s) {
      float kr[8], vr[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        kr[i] = (ty * 8 + i < Dk) ? Ks[s * Dk + ty * 8 + i] : 0.f;
        vr[i] = (tx * 8 + i < Dv) ? Vs[s * Dv + tx * 8 + i] : 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(kr[i], vr[j], acc[i][j]);
    }
    __syncthreads();
  }
  float* out = states + (int64_t(p) * H + h) * Dk * Dv;
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (ty * 8 + i < Dk && tx * 8 + j < Dv) out[(ty * 8 + i) * Dv + tx * 8 + j] = acc[i][j];
}

// pieces are rank-major: piece (r, s) = r * S + s
__global__ void __launch_bounds__(kLinThreads) lin_prefix_kernel(const LinPiece* __restrict__ pieces, int32_t S,
                                                                  int32_t C, int32_t H, int32_t DD,
                                                                  const float* __restrict__ g,
                                                                  const float* __restrict__ states,
                                                                  float* __restrict__ init) {
  const int s = blockIdx.x / H, h = blockIdx.x - (blockIdx.x / H) * H;
  const float gh = g[h];
  for (int e = threadIdx.x; e < DD; e += blockDim.x) {
    float cur = 0.f;
    for (int r = 0; r < C; ++r) {
      const int64_t p = int64_t(r) * S + s;
      const int64_t idx = (p * H + h) * DD + e;
      init[idx] = cur;
      cur = __expf(gh * float(pieces[p].len)) * cur + states[idx];
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(kLinThreads) lin_output_kernel(const LinPiece* __restrict__ pieces, int32_t H,
                                                                  int32_t Dk, int32_t Dv, float scale,
                                                                  const T* __restrict__ q, const T* __restrict__ k,
                                                                  const T* __restrict__ v, const float* __restrict__ g,
                                                                  const float* __restrict__ init, T* __restrict__ o) {
  extern __shared__ float lsm[];
  const int ldk = Dk + 1;              // padded K rows: lanes walking s hit distinct banks
  float* Hs = lsm;                     // [Dk][Dv] carried state
  float* Qs = Hs + Dk * Dv;            // [kLinB][Dk]
  float* Ks = Qs + kLinB * Dk;         // [kLinB][Dk + 1]
  float* Vs = Ks + kLinB * ldk;        // [kLinB][Dv]
  float* As = Vs + kLinB * Dv;         // [kLinB][kLinB] decayed causal scores
  float* Ws = As + kLinB * kLinB;      // [kLinB] alpha^(n-1-s) of the state update
  float* Ds = Ws + kLinB;              // [kLinB] alpha^(t+1) of the initial-state term
  const int p = blockIdx.x / H, h = blockIdx.x - (blockIdx.x / H) * H;
  const LinPiece pc = pieces[p];
  const float gh = g[h];
  const int DD = Dk * Dv;
  const float* h0 = init + (int64_t(p) * H + h) * DD;
  for (int e = threadIdx.x; e < DD; e += blockDim.x) Hs[e] = h0[e];
  for (int c0 = 0; c0 < pc.len; c0 += kLinB) {
    const int n = min(kLinB, pc.len - c0);
    __syncthreads();  // previous chunk's readers of Qs/Ks/Vs/As and writers of Hs are done
    load_rows(Qs, Dk, q, pc.row0 + c0, n, H, h, Dk, [](int) { return 1.f; });
    load_rows(Ks, ldk, k, pc.row0 + c0, n, H, h, Dk, [](int) { return 1.f; });
    load_rows(Vs, Dv, v, pc.row0 + c0, n, H, h, Dv, [](int) { return 1.f; });
    for (int t = threadIdx.x; t < kLinB; t += blockDim.x) {
      Ws[t] = t < n ? __expf(gh * float(n - 1 - t)) : 0.f;
      Ds[t] = __expf(gh * float(t + 1));
    }
    __syncthreads();
    // A[t][s] = (q_t . k_s) alpha^(t-s) for s <= t
    for (int e = threadIdx.x; e < kLinB * kLinB; e += blockDim.x) {
      const int t = e / kLinB, s = e - t * kLinB;
      float a = 0.f;
      if (s <= t && t < n) {
        for (int d = 0; d < Dk; ++d) a = fmaf(Qs[t * Dk + d], Ks[s * ldk + d], a);
        a *= __expf(gh * float(t - s));
      }
      As[e] = a;
    }
    __syncthreads();
    // O[t][j] = scale (sum_s A[t][s] V[s][j] + alpha^(t+1) sum_d Q[t][d] H[d][j])
    for (int e = threadIdx.x; e < kLinB * Dv; e += blockDim.x) {
      const int t = e / Dv, j = e - t * Dv;
      if (t >= n) continue;
      float x = 0.f, y = 0.f;
      for (int s = 0; s <= t; ++s) x = fmaf(As[t * kLinB + s], Vs[s * Dv + j], x);
      for (int d = 0; d < Dk; ++d) y = fmaf(Qs[t * Dk + d], Hs[d * Dv + j], y);
      o[((pc.row0 + c0 + t) * int64_t(H) + h) * Dv + j] = from_f<T>(scale * (x + Ds[t] * y));
    }
    __syncthreads();
    // H = alpha^n H + sum_s alpha^(n-1-s) k_s^T v_s
    const float an = __expf(gh * float(n));
    for (int e = threadIdx.x; e < DD; e += blockDim.x) {
      const int d = e / Dv, j = e - d * Dv;
      float x = 0.f;
      for (int s = 0; s < n; ++s) x = fmaf(Ws[s] * Ks[s * ldk + d], Vs[s * Dv + j], x);
      Hs[e] = an * Hs[e] + x;
    }
  }
}

}  // namespace

size_t lin_output_smem(int32_t Dk, int32_t Dv) {
  return sizeof(float) * (size_t(Dk) * Dv + kLinB * Dk + kLinB * (Dk + 1) + kLinB * Dv + kLinB * kLinB + 2 * kLinB);
}

cudaError_t launch_lin_attn(const LinPiece* pieces, int32_t npieces, int32_t S, int32_t C, int32_t H, int32_t Dk,
                            int32_t Dv, float scale, int32_t dtype, const void* q, const void* k, const void* v,
                            const float* g, float* states, float* init, void* o, cudaStream_t st) {
  if (Dk > kLinMaxD || Dv > kLinMaxD) return cudaErrorInvalidValue;
  const unsigned grid = unsigned(int64_t(npieces) * H);
  if (grid == 0) return cudaSuccess;
  const size_t sm_state = sizeof(float) * size_t(kLinB) * (Dk + Dv);
  const size_t sm_out = lin_output_smem(Dk, Dv);
  cudaError_t e;
  if (dtype == CP_DT_BF16) {
    auto ks = lin_state_kernel<__nv_bfloat16>;
    auto ko = lin_output_kernel<__nv_bfloat16>;
    if ((e = cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sm_state))) != cudaSuccess ||
        (e = cudaFuncSetAttribute(ko, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sm_out))) != cudaSuccess)
      return e;
    ks<<<grid, kLinThreads, sm_state, st>>>(pieces, H, Dk, Dv, static_cast<const __nv_bfloat16*>(k),
                                            static_cast<const __nv_bfloat16*>(v), g, states);
    lin_prefix_kernel<<<unsigned(S * H), kLinThreads, 0, st>>>(pieces, S, C, H, Dk * Dv, g, states, init);
    ko<<<grid, kLinThreads, sm_out, st>>>(pieces, H, Dk, Dv, scale, static_cast<const __nv_bfloat16*>(q),
                                          static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v),
                                          g, init, static_cast<__nv_bfloat16*>(o));
  } else {
    auto ks = lin_state_kernel<float>;
    auto ko = lin_output_kernel<float>;
    if ((e = cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sm_state))) != cudaSuccess ||
        (e = cudaFuncSetAttribute(ko, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sm_out))) != cudaSuccess)
      return e;
    ks<<<grid, kLinThreads, sm_state, st>>>(pieces, H, Dk, Dv, static_cast<const float*>(k),
                                            static_cast<const float*>(v), g, states);
    lin_prefix_kernel<<<unsigned(S * H), kLinThreads, 0, st>>>(pieces, S, C, H, Dk * Dv, g, states, init);
    ko<<<grid, kLinThreads, sm_out, st>>>(pieces, H, Dk, Dv, scale, static_cast<const float*>(q),
                                          static_cast<const float*>(k), static_cast<const float*>(v), g, init,
                                          static_cast<float*>(o));
  }
  return cudaGetLastError();
}

}  // namespace cpattn
