// device_status.cu — the device error word written by bounded waits that
// ran out, its host read-back, and a self-check kernel that makes one wait
// run out on purpose (a barrier nothing completes) to prove that the waits
// return instead of hanging.
#include "internal.h"
#include "sm103_ptx.cuh"

namespace cpattn {

namespace {
__device__ int32_t g_error_word;

__global__ void wait_selftest_kernel(int64_t limit_ns, int32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bar), 1);
    ptx::fence_barrier_init();
    abort_flag = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    ptx::WaitCtx ctx{&abort_flag, err, uint64_t(limit_ns)};
    // Phase 0 never completes: no thread arrives on the barrier.
    (void)ptx::mbar_wait(ptx::smem_u32(&bar), 0, /*site=*/0x7f, ctx);
  }
  __syncthreads();
}
}  // namespace

int32_t* device_error_word() {
  static int32_t* ptrs[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (ptrs[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int32_t*>(p);
  }
  return ptrs[dev];
}

cudaError_t read_and_clear_device_status(int32_t* code, cudaStream_t st) {
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return e;
  int32_t* w = device_error_word();
  if (w == nullptr) return cudaErrorInvalidSymbol;
  e = cudaMemcpy(code, w, sizeof(int32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return e;
  const int32_t zero = 0;
  return cudaMemcpy(w, &zero, sizeof(int32_t), cudaMemcpyHostToDevice);
}

cudaError_t launch_wait_selftest(int64_t timeout_ns, cudaStream_t st) {
  int32_t* w = device_error_word();
  if (w == nullptr) return cudaErrorInvalidSymbol;
  wait_selftest_kernel<<<1, 32, 0, st>>>(timeout_ns, w);
  return cudaGetLastError();
}

}  // namespace cpattn
