// The output gate of "xLSTM: Extended Long Short-Term Memory", part 17/30
// eq (27) and part 28/30 eq (78), h = sigmoid(o~) (.) H~, applied in place to
// a finished H~ for the forward kernels that do not fuse it into their
// epilogue (the CTA-pair kernel does), and its two backward passes (the
// chain rule of eq 78, with sigmoid' = sigmoid (1 - sigmoid), the output-gate
// gradient of eq 70): dL/dH~ = dL/dh (.) sigmoid(o~) and
// dL/do~ = dL/dh (.) H~ (.) sigmoid(o~) (1 - sigmoid(o~)).  Streaming
// elementwise passes.
#include "internal.h"

namespace mlstm {
namespace {

template <typename T>
__global__ void apply_ogate_kernel(T* __restrict__ h, const T* __restrict__ og, long long n) {
  for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < n; x += (long long)gridDim.x * blockDim.x)
    Elem<T>::store(h, x, Elem<T>::load(h, x) * sigmoid(Elem<T>::load(og, x)));
}

// dHt = dh (.) sigmoid(o~)
template <typename T>
__global__ void ogate_bwd_in_kernel(const T* __restrict__ dh, const T* __restrict__ og, T* __restrict__ dht,
                                    long long n) {
  for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < n; x += (long long)gridDim.x * blockDim.x)
    Elem<T>::store(dht, x, Elem<T>::load(dh, x) * sigmoid(Elem<T>::load(og, x)));
}

// dog = dh (.) H~ (.) sigmoid(o~) (1 - sigmoid(o~))
template <typename T>
__global__ void ogate_bwd_out_kernel(const T* __restrict__ dh, const T* __restrict__ og, const T* __restrict__ ht,
                                     T* __restrict__ dog, long long n) {
  for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < n; x += (long long)gridDim.x * blockDim.x) {
    const float sg = sigmoid(Elem<T>::load(og, x));
    Elem<T>::store(dog, x, Elem<T>::load(dh, x) * Elem<T>::load(ht, x) * sg * (1.0f - sg));
  }
}

unsigned grid_for(long long n, int threads) {
  const long long want = (n + threads - 1) / threads;
  return (unsigned)(want < 65536 ? want : 65536);
}

}  // namespace

cudaError_t launch_ogate_bwd_in(const void* dh, const void* og, void* dht, long long n, int dtype,
                                cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  if (dtype == kF32)
    ogate_bwd_in_kernel<float><<<grid_for(n, 256), 256, 0, stream>>>((const float*)dh, (const float*)og, (float*)dht, n);
  else
    ogate_bwd_in_kernel<__nv_bfloat16><<<grid_for(n, 256), 256, 0, stream>>>(
        (const __nv_bfloat16*)dh, (const __nv_bfloat16*)og, (__nv_bfloat16*)dht, n);
  return cudaGetLastError();
}

cudaError_t launch_ogate_bwd_out(const void* dh, const void* og, const void* ht, void* dog, long long n, int dtype,
                                 cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  if (dtype == kF32)
    ogate_bwd_out_kernel<float><<<grid_for(n, 256), 256, 0, stream>>>((const float*)dh, (const float*)og,
                                                                      (const float*)ht, (float*)dog, n);
  else
    ogate_bwd_out_kernel<__nv_bfloat16><<<grid_for(n, 256), 256, 0, stream>>>(
        (const __nv_bfloat16*)dh, (const __nv_bfloat16*)og, (const __nv_bfloat16*)ht, (__nv_bfloat16*)dog, n);
  return cudaGetLastError();
}

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
