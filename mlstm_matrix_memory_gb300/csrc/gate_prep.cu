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
// p2 is the running max of the *stored* a2 values (float(x * log2 e) is
// monotone in x), so a2_j - p2_i <= 0 holds exactly for every j <= i and D'
// never exceeds 1.
//
// One CTA of 1024 threads per (b, h) sequence, one pass: each thread keeps
// its contiguous segment in registers, and the segment totals are combined by
// block-wide scans built from warp shuffles.  The running sum cs must keep the
// differences cs_i - cs_j accurate over 16k tokens, so it is carried as an
// unevaluated pair hi + lo of fp32 values with error-free (two-sum) additions;
// fp64 throughput on this part is far too low to use for it.
#include "internal.h"

namespace mlstm {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxSeg = 16;            // tokens per thread held in registers (T <= 16384)

// hi + lo, with |lo| below half an ulp of hi.
struct F2 {
  float hi, lo;
};

// Knuth's two-sum: s + e == a + b exactly.
__device__ __forceinline__ F2 two_sum(float a, float b) {
  const float s = a + b;
  const float bb = s - a;
  const float e = (a - (s - bb)) + (b - bb);
  return {s, e};
}
__device__ __forceinline__ F2 add2(F2 a, F2 b) {
  F2 s = two_sum(a.hi, b.hi);
  s.lo += a.lo + b.lo;
  return two_sum(s.hi, s.lo);
}
__device__ __forceinline__ F2 add2(F2 a, float b) {
  F2 s = two_sum(a.hi, b);
  s.lo += a.lo;
  return two_sum(s.hi, s.lo);
}

// Running maximum of a_j = i~_j - cs_j together with the argmax's i~ and cs,
// so that m_i = i~_* + (cs_i - cs_*) is formed from a small difference
// instead of two cancelling large terms.
struct MaxRec {
  float a, ig;
  F2 cs;
};

struct AddF2 { __device__ F2 operator()(F2 a, F2 b) const { return add2(a, b); } };
struct MaxR { __device__ MaxRec operator()(MaxRec a, MaxRec b) const { return b.a > a.a ? b : a; } };

__device__ __forceinline__ F2 shfl_up(F2 v, int o) {
  return {__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
}
__device__ __forceinline__ MaxRec shfl_up(MaxRec v, int o) {
  return {__shfl_up_sync(0xffffffffu, v.a, o), __shfl_up_sync(0xffffffffu, v.ig, o), shfl_up(v.cs, o)};
}

template <typename T, typename Op>
__device__ __forceinline__ T warp_inclusive(T x, Op op) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T y = shfl_up(x, o);
    if (lane >= o) x = op(y, x);
  }
  return x;
}

// Exclusive block scan; `sh` holds kWarps entries.
template <typename T, typename Op>
__device__ __forceinline__ T block_exclusive(T v, T identity, Op op, T* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T x = warp_inclusive(v, op);
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  if (warp == 0) sh[lane] = warp_inclusive(sh[lane], op);   // kWarps == 32
  __syncthreads();
  T excl = shfl_up(x, 1);
  if (lane == 0) excl = identity;
  T r = op(warp > 0 ? sh[warp - 1] : identity, excl);
  __syncthreads();
  return r;
}

__device__ __forceinline__ MaxRec rec(float a, float ig, F2 cs) { return MaxRec{a, ig, cs}; }

// Writes the three gate terms of token t given its a_t, cs_t and the running
// max record over j <= t.
__device__ __forceinline__ void emit(float* a2, float* p2, float* mrow, size_t idx, float a, const MaxRec& pm,
                                     F2 cs) {
  a2[idx] = a * kLog2e;                // fp32 product: monotone in a, so p2 = max of stored a2
  p2[idx] = pm.a * kLog2e;
  F2 d = two_sum(cs.hi, -pm.cs.hi);    // cs_t - cs_* (log forget product from * to t)
  d.lo += cs.lo - pm.cs.lo;
  mrow[idx] = pm.ig + (d.hi + d.lo);
}

// log of the forget gate: log sigmoid(f~) (default) or f~ (exponential activation)
__device__ __forceinline__ float log_forget(float x, int forget_exp) { return forget_exp ? x : log_sigmoid(x); }

template <int SEG>
__global__ void __launch_bounds__(kThreads)
gate_prep_kernel(const float* __restrict__ ig, const float* __restrict__ fg, float* __restrict__ a2,
                 float* __restrict__ p2, float* __restrict__ mrow, int T, int forget_exp) {
  __shared__ F2 shs[kWarps];
  __shared__ MaxRec shm[kWarps];
  // the fused kernel that follows may start its prologue (it waits for this
  // grid before reading any gate term)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const size_t base = (size_t)blockIdx.x * T;
  const int t0 = threadIdx.x * SEG;
  float lf[SEG], iv[SEG];
  F2 local = {0.0f, 0.0f};
#pragma unroll
  for (int s = 0; s < SEG; ++s) {
    const int t = t0 + s;
    lf[s] = t < T ? log_forget(fg[base + t], forget_exp) : 0.0f;
    iv[s] = t < T ? ig[base + t] : 0.0f;
    local = add2(local, lf[s]);
  }
  const F2 cs0 = block_exclusive(local, F2{0.0f, 0.0f}, AddF2(), shs);
  const MaxRec none = {-INFINITY, 0.0f, {0.0f, 0.0f}};
  F2 cs = cs0;
  MaxRec segmax = none;
#pragma unroll
  for (int s = 0; s < SEG; ++s) {
    cs = add2(cs, lf[s]);
    if (t0 + s < T) segmax = MaxR()(segmax, rec((iv[s] - cs.hi) - cs.lo, iv[s], cs));
  }
  MaxRec pm = block_exclusive(segmax, none, MaxR(), shm);
  cs = cs0;
#pragma unroll
  for (int s = 0; s < SEG; ++s) {
    cs = add2(cs, lf[s]);
    const float a = (iv[s] - cs.hi) - cs.lo;
    pm = MaxR()(pm, rec(a, iv[s], cs));
    if (t0 + s < T) emit(a2, p2, mrow, base + t0 + s, a, pm, cs);
  }
}

// Sequences longer than kThreads * kMaxSeg: the same computation in strided
// passes over global memory.
__global__ void __launch_bounds__(kThreads)
gate_prep_long_kernel(const float* __restrict__ ig, const float* __restrict__ fg, float* __restrict__ a2,
                      float* __restrict__ p2, float* __restrict__ mrow, int T, int forget_exp) {
  __shared__ F2 shs[kWarps];
  __shared__ MaxRec shm[kWarps];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const size_t base = (size_t)blockIdx.x * T;
  const int seg = (T + kThreads - 1) / kThreads;
  const int t0 = min(T, (int)threadIdx.x * seg), t1 = min(T, t0 + seg);
  F2 local = {0.0f, 0.0f};
  for (int t = t0; t < t1; ++t) local = add2(local, log_forget(fg[base + t], forget_exp));
  const F2 cs0 = block_exclusive(local, F2{0.0f, 0.0f}, AddF2(), shs);
  const MaxRec none = {-INFINITY, 0.0f, {0.0f, 0.0f}};
  F2 cs = cs0;
  MaxRec segmax = none;
  for (int t = t0; t < t1; ++t) {
    cs = add2(cs, log_forget(fg[base + t], forget_exp));
    const float iv = ig[base + t];
    segmax = MaxR()(segmax, rec((iv - cs.hi) - cs.lo, iv, cs));
  }
  MaxRec pm = block_exclusive(segmax, none, MaxR(), shm);
  cs = cs0;
  for (int t = t0; t < t1; ++t) {
    cs = add2(cs, log_forget(fg[base + t], forget_exp));
    const float iv = ig[base + t];
    const float a = (iv - cs.hi) - cs.lo;
    pm = MaxR()(pm, rec(a, iv, cs));
    emit(a2, p2, mrow, base + t, a, pm, cs);
  }
}

}  // namespace

cudaError_t launch_gate_prep(const float* ig, const float* fg, GateTerms g, int BH, int T, int forget_exp,
                             cudaStream_t stream) {
  if (BH <= 0 || T <= 0) return cudaSuccess;
  const int seg = (T + kThreads - 1) / kThreads;
  if (seg <= 2)
    gate_prep_kernel<2><<<BH, kThreads, 0, stream>>>(ig, fg, g.a2, g.p2, g.m, T, forget_exp);
  else if (seg <= 4)
    gate_prep_kernel<4><<<BH, kThreads, 0, stream>>>(ig, fg, g.a2, g.p2, g.m, T, forget_exp);
  else if (seg <= kMaxSeg)
    gate_prep_kernel<kMaxSeg><<<BH, kThreads, 0, stream>>>(ig, fg, g.a2, g.p2, g.m, T, forget_exp);
  else
    gate_prep_long_kernel<<<BH, kThreads, 0, stream>>>(ig, fg, g.a2, g.p2, g.m, T, forget_exp);
  return cudaGetLastError();
}

}  // namespace mlstm
