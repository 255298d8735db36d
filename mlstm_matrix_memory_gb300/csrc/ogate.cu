// The output gate of "xLSTM: Extended Long Short-Term Memory", part 17/30
// eq (27) and part 28/30 eq (78), h = sigmoid(o~) (.) H~, applied in place to
// a finished H~ for the forward kernels that do not fuse it into their
// epilogue (the CTA-pair kernel does).  A streaming elementwise pass.
#include "internal.h"

namespace mlstm {
namespace {

template <typename T>
__global__ void apply_ogate_kernel(T* __restrict__ h, const T* __restrict__ og, long long n) {
  for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < n; x += (long long)gridDim.x * blockDim.x)
    Elem<T>::store(h, x, Elem<T>::load(h, x) * sigmoid(Elem<T>::load(og, x)));
}

}  // namespace

cudaError_t launch_apply_ogate(void* h, const void* og, long long n, int dtype, cudaStream_t stream) {
  if (n <= 0 || !og) return cudaSuccess;
  const int threads = 256;
  const long long want = (n + threads - 1) / threads;
  const unsigned grid = (unsigned)(want < 65536 ? want : 65536);
  if (dtype == kF32)
    apply_ogate_kernel<float><<<grid, threads, 0, stream>>>((float*)h, (const float*)og, n);
  else
    apply_ogate_kernel<__nv_bfloat16><<<grid, threads, 0, stream>>>((__nv_bfloat16*)h, (const __nv_bfloat16*)og, n);
  return cudaGetLastError();
}

}  // namespace mlstm
