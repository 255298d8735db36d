// Shared device helpers of libmlstm.so: element loads/stores, the gate
// activations, the bounded-wait status protocol and block reductions.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace mlstm {

// Status codes, identical to mlstm_status in include/mlstm.h.
enum Status : int {
  kOk = 0,
  kInval = -1,
  kAlign = -2,
  kDtype = -3,
  kCuda = -4,
  kTimeout = -5,
  kUnsupported = -6,
  kWorkspace = -7,
};

enum Dtype : int { kF32 = 0, kBF16 = 1 };

// Where a kernel may give up a bounded wait.  The device status word is
// {code, site}: the first failure wins.
struct DevStatus {
  int* word;             // 2 ints in device memory: [0] = status, [1] = site
  long long spin_limit;  // polling iterations per wait before giving up
};

__device__ __forceinline__ void report_timeout(const DevStatus& st, int site) {
  if (atomicCAS(st.word, 0, (int)kTimeout) == 0) atomicExch(st.word + 1, site);
}

// log(sigmoid(x)) = min(x, 0) - log1p(exp(-|x|)); exact 0 at +inf, -inf at -inf.
__device__ __forceinline__ float log_sigmoid(float x) {
  return fminf(x, 0.0f) - log1pf(expf(-fabsf(x)));
}

__device__ __forceinline__ float sigmoid(float x) { return 1.0f / (1.0f + expf(-x)); }

template <typename T> struct Elem;
template <> struct Elem<float> {
  static __device__ __forceinline__ float load(const float* p, size_t i) { return p[i]; }
  static __device__ __forceinline__ void store(float* p, size_t i, float v) { p[i] = v; }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float load(const __nv_bfloat16* p, size_t i) {
    return __bfloat162float(p[i]);
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, size_t i, float v) {
    p[i] = __float2bfloat16_rn(v);
  }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide sum; `red` holds >= 32 floats of shared memory.  All threads
// receive the total.
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = lane < nw ? red[lane] : 0.0f;
  t = warp_sum(t);
  return t;
}

constexpr float kLog2e = 1.4426950408889634f;

}  // namespace mlstm
