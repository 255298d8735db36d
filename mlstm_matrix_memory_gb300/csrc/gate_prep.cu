// Gate preprocessing for the parallel mLSTM forward pass.
//
// "xLSTM: Extended Long Short-Term Memory", part 28/30, eqs (79)-(81) and
// (101): with cs_t = sum_{k<=t} log sigmoid(f~_k) (inclusive prefix sum),
//   Fbar_ij = cs_i - cs_j  (j <= i)   and   D~_ij = cs_i + (i~_j - cs_j),
// so the row maximum of eq (80) is a prefix maximum,
//   m_i = cs_i + max_{j<=i} (i~_j - cs_j),
// and the stabilized gate of eq (81) factors into a column and a row term:
//   D'_ij = exp(D~_ij - m_i) = exp2(a2_j - p2_i),
//   a2_j = (i~_j - cs_j) log2(e),   p2_i = max_{j<=i} a2_j.
// p2 is the running max of the *stored* a2 values, so a2_j - p2_i <= 0 holds
// exactly for every j <= i and D' never exceeds 1.
//
// One CTA per (b, h) sequence.  Each thread owns a contiguous segment of the
// sequence; the sum runs in fp64 (the differences cs_i - cs_j must stay
// accurate over 16k tokens) and the segment totals are combined with a
// block-wide scan built from warp shuffles.
#include "internal.h"

namespace mlstm {
namespace {

constexpr int kThreads = 256;

template <typename T, typename Op>
__device__ T block_exclusive_scan(T v, T identity, Op op, T* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // inclusive scan within the warp
  T x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x = op(y, x);
  }
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  if (warp == 0) {
    T w = lane < kThreads / 32 ? sh[lane] : identity;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      T y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w = op(y, w);
    }
    if (lane < kThreads / 32) sh[lane] = w;   // inclusive scan of warp totals
  }
  __syncthreads();
  T warp_prefix = warp > 0 ? sh[warp - 1] : identity;
  T excl = __shfl_up_sync(0xffffffffu, x, 1);
  if (lane == 0) excl = identity;
  T r = op(warp_prefix, excl);
  __syncthreads();   // sh may be reused by the caller
  return r;
}

struct AddD { __device__ double operator()(double a, double b) const { return a + b; } };
struct MaxD { __device__ double operator()(double a, double b) const { return fmax(a, b); } };

__global__ void __launch_bounds__(kThreads)
gate_prep_kernel(const float* __restrict__ ig, const float* __restrict__ fg, float* __restrict__ a2,
                 float* __restrict__ p2, float* __restrict__ mrow, int T) {
  __shared__ double sh[32];
  const size_t base = (size_t)blockIdx.x * T;
  const int seg = (T + kThreads - 1) / kThreads;
  const int t0 = min(T, (int)threadIdx.x * seg), t1 = min(T, t0 + seg);

  double local = 0.0;
  for (int t = t0; t < t1; ++t) local += (double)log_sigmoid(fg[base + t]);
  const double cs0 = block_exclusive_scan(local, 0.0, AddD(), sh);

  // second walk: the maximum of a_j = i~_j - cs_j over this segment
  double cs = cs0, segmax = -INFINITY;
  for (int t = t0; t < t1; ++t) {
    cs += (double)log_sigmoid(fg[base + t]);
    segmax = fmax(segmax, (double)ig[base + t] - cs);
  }
  double pm = block_exclusive_scan(segmax, -(double)INFINITY, MaxD(), sh);

  // third walk: column term a2, prefix max p2, row max m (eq 80).  float(x *
  // log2e) is monotone in x, so p2 equals the running max of the stored a2.
  cs = cs0;
  for (int t = t0; t < t1; ++t) {
    cs += (double)log_sigmoid(fg[base + t]);
    const double a = (double)ig[base + t] - cs;
    pm = fmax(pm, a);
    a2[base + t] = (float)(a * 1.4426950408889634);
    p2[base + t] = (float)(pm * 1.4426950408889634);
    mrow[base + t] = (float)(cs + pm);
  }
}

}  // namespace

cudaError_t launch_gate_prep(const float* ig, const float* fg, GateTerms g, int BH, int T,
                             cudaStream_t stream) {
  if (BH <= 0 || T <= 0) return cudaSuccess;
  gate_prep_kernel<<<BH, kThreads, 0, stream>>>(ig, fg, g.a2, g.p2, g.m, T);
  return cudaGetLastError();
}

}  // namespace mlstm
