// Final recurrent state of a sequence from its parallel-form gate terms: the
// hand-off from the parallel forward (prefill) to the recurrent step
// (generation).
//
// "xLSTM: Extended Long Short-Term Memory", part 28/30: unrolling the
// stabilized recurrence (eqs 59-70) over t = 1..T from C = 0, n = 0,
// m = -inf gives
//   m_T = max_j D~_Tj                      (the last row's max, eq 80),
//   C_T = sum_j exp(D~_Tj - m_T) v_j (s k_j)^T,   n_T = sum_j exp(D~_Tj - m_T) s k_j,
// with D~_Tj = cs_T - cs_j + i~_j (eqs 79, 101): the weights are the last row
// of the stabilized gate matrix D' of eq (81).  From the gate pass's terms,
// D'_Tj = exp2(a2_j - p2_T), so the state is one weighted product V^T W K per
// head: a GEMM over the T tokens with a per-token weight.
//
// CUDA-core version: each CTA computes a 64 x 64 tile of C (d_v rows x d_qk
// columns) over a range of tokens, staging 32 weighted tokens of V and K in
// shared memory at a time; each thread owns a 4 x 4 block of the tile.  When
// there are too few tiles to fill the GPU, the token range is split and the
// partial tiles are added into C (zeroed first) with atomic adds.
#include <algorithm>

#include "internal.h"

namespace mlstm {
namespace {

constexpr int kTile = 64, kTok = 32, kThreads = 256;

template <typename E>
__global__ void __launch_bounds__(kThreads)
final_state_kernel(const E* __restrict__ k, const E* __restrict__ v, GateTerms g, float* __restrict__ C,
                   float* __restrict__ n, float* __restrict__ m, int T, int dqk, int dv, int ntr, int ntc,
                   int ksplit, float scale) {
  __shared__ float Vs[kTok][kTile + 4];
  __shared__ float Ks[kTok][kTile + 4];
  const int per_head = ntr * ntc * ksplit;
  const int bh = blockIdx.x / per_head;
  int rem = blockIdx.x % per_head;
  const int split = rem % ksplit;
  rem /= ksplit;
  const int tr = rem / ntc, tc = rem % ntc;
  const int r0 = tr * kTile, c0 = tc * kTile;
  const int tpb = (T + ksplit - 1) / ksplit;
  const int j0 = split * tpb, j1 = min(T, j0 + tpb);
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;   // 16 x 16 threads, 4 x 4 each
  const size_t hb = (size_t)bh * T;
  const float p2T = g.p2[hb + T - 1];

  float acc[4][4] = {};
  float nacc[4] = {};
  for (int jb = j0; jb < j1; jb += kTok) {
    // weighted tokens: V rows scaled by w_j, K columns by s (the weight once)
    for (int e = threadIdx.x; e < kTok * kTile; e += kThreads) {
      const int jj = e / kTile, x = e % kTile, j = jb + jj;
      float w = 0.0f;
      if (j < j1) w = exp2f(g.a2[hb + j] - p2T);
      const int r = r0 + x, c = c0 + x;
      Vs[jj][x] = (j < j1 && r < dv) ? w * Elem<E>::load(v, (hb + j) * dv + r) : 0.0f;
      Ks[jj][x] = (j < j1 && c < dqk) ? scale * Elem<E>::load(k, (hb + j) * dqk + c) : 0.0f;
    }
    __syncthreads();
#pragma unroll 8
    for (int jj = 0; jj < kTok; ++jj) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = Vs[jj][ty * 4 + i];
        b[i] = Ks[jj][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int l = 0; l < 4; ++l) acc[i][l] = fmaf(a[i], b[l], acc[i][l]);
    }
    if (tr == 0 && ty == 0) {
      // n = sum_j w_j s k_j: the weight is not in Ks, so apply it here
      for (int jj = 0; jj < kTok && jb + jj < j1; ++jj) {
        const float w = exp2f(g.a2[hb + jb + jj] - p2T);
#pragma unroll
        for (int l = 0; l < 4; ++l) nacc[l] = fmaf(w, Ks[jj][tx * 4 + l], nacc[l]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = r0 + ty * 4 + i;
    if (r >= dv) continue;
#pragma unroll
    for (int l = 0; l < 4; ++l) {
      const int c = c0 + tx * 4 + l;
      if (c >= dqk) continue;
      float* dst = C + ((size_t)bh * dv + r) * dqk + c;
      if (ksplit > 1) atomicAdd(dst, acc[i][l]);
      else *dst = acc[i][l];
    }
  }
  if (tr == 0 && ty == 0) {
#pragma unroll
    for (int l = 0; l < 4; ++l) {
      const int c = c0 + tx * 4 + l;
      if (c >= dqk) continue;
      if (ksplit > 1) atomicAdd(n + (size_t)bh * dqk + c, nacc[l]);
      else n[(size_t)bh * dqk + c] = nacc[l];
    }
  }
  if (tr == 0 && tc == 0 && split == 0 && threadIdx.x == 0) m[bh] = g.m[hb + T - 1];
}

}  // namespace

cudaError_t launch_final_state(const void* k, const void* v, GateTerms g, float* C, float* n, float* m, int BH,
                               int T, int dqk, int dv, int dtype, float scale, cudaStream_t stream) {
  if (BH <= 0 || T <= 0) return cudaSuccess;
  const int ntr = (dv + kTile - 1) / kTile, ntc = (dqk + kTile - 1) / kTile;
  const long long tiles = (long long)BH * ntr * ntc;
  int sms = 148, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // enough CTAs for a few per SM, but at least 256 tokens per split
  int ksplit = (int)std::max<long long>(1, (4LL * sms + tiles - 1) / tiles);
  ksplit = std::max(1, std::min(ksplit, T / 256));
  const long long grid = tiles * ksplit;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  if (ksplit > 1) {
    cudaError_t e = cudaMemsetAsync(C, 0, (size_t)BH * dv * dqk * sizeof(float), stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(n, 0, (size_t)BH * dqk * sizeof(float), stream);
    if (e != cudaSuccess) return e;
  }
  if (dtype == kF32)
    final_state_kernel<float><<<(unsigned)grid, kThreads, 0, stream>>>(
        (const float*)k, (const float*)v, g, C, n, m, T, dqk, dv, ntr, ntc, ksplit, scale);
  else
    final_state_kernel<__nv_bfloat16><<<(unsigned)grid, kThreads, 0, stream>>>(
        (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, g, C, n, m, T, dqk, dv, ntr, ntc, ksplit, scale);
  return cudaGetLastError();
}

}  // namespace mlstm
