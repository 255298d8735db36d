// Stabilized parallel mLSTM forward on CUDA cores in fp32.
//
// "xLSTM: Extended Long Short-Term Memory", part 28/30, eqs (79)-(86).  Used
// for fp32 inputs (tensor-core operands cannot hold fp32 accuracy) and for
// bf16 head sizes the tensor-core kernel does not tile.  Any d_qk, d_v <= 512.
//
// One CTA owns 32 query rows of one head and walks the causal key tiles of 32
// keys.  For each tile it forms S = Q K_j^T in shared memory, applies the gate
// D'_ij = exp2(a2_j - p2_i) (zero above the diagonal), accumulates the signed
// row sum b_i of C'_ij (eq 83) in fp32 and O += C' V_j in registers.  The
// epilogue divides by n_i = max(|b_i|, exp(-m_i)) (eq 84).
#include "internal.h"

namespace mlstm {
namespace {

constexpr int kBM = 32, kBN = 32, kThreads = 256, kMaxD = 512;
constexpr int kAcc = kMaxD / 8;   // O accumulators per thread (8 threads per row)

template <typename T>
__global__ void __launch_bounds__(kThreads)
fwd_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                const float* __restrict__ a2, const float* __restrict__ p2,
                const float* __restrict__ mrow, T* __restrict__ h, float* __restrict__ m_out, float* __restrict__ b_out,
                float* __restrict__ n_out, int T_, int dqk, int dv, float scale) {
  extern __shared__ float smem[];
  const int ldk = dqk + 1;                  // padded row: conflict-free column reads
  float* Qs = smem;                         // [kBM][dqk]
  float* Ks = Qs + kBM * dqk;               // [kBN][dqk+1]
  float* Vs = Ks + kBN * ldk;               // [kBN][dv]
  float* Ps = Vs + kBN * dv;                // [kBM][kBN+1]
  float* colg = Ps + kBM * (kBN + 1);       // [kBN] column terms a2 of the tile

  // all heads' last (longest) query tiles are scheduled first
  const int nqt = (T_ + kBM - 1) / kBM;
  const int BH = (int)(gridDim.x / nqt);
  const int qt = nqt - 1 - (int)(blockIdx.x / BH);
  const int bh = (int)(blockIdx.x % BH);
  const int i0 = qt * kBM;
  const size_t hq = (size_t)bh * T_;

  const int tid = threadIdx.x;
  const int r = tid >> 3;          // row of this thread within the tile
  const int c8 = tid & 7;          // column phase
  const int gi = i0 + r;           // global query row

  for (int e = tid; e < kBM * dqk; e += kThreads) {
    const int rr = e / dqk, cc = e % dqk;
    Qs[e] = (i0 + rr < T_) ? Elem<T>::load(q, (hq + i0 + rr) * dqk + cc) : 0.0f;
  }
  const float rowp = gi < T_ ? p2[hq + gi] : 0.0f;

  float acc[kAcc];
#pragma unroll
  for (int u = 0; u < kAcc; ++u) acc[u] = 0.0f;
  float bsum = 0.0f;

  const int nkt = (min(T_, i0 + kBM) + kBN - 1) / kBN;
  for (int kt = 0; kt < nkt; ++kt) {
    const int j0 = kt * kBN;
    __syncthreads();   // previous tile fully consumed
    for (int e = tid; e < kBN * dqk; e += kThreads) {
      const int rr = e / dqk, cc = e % dqk;
      Ks[rr * ldk + cc] = (j0 + rr < T_) ? Elem<T>::load(k, (hq + j0 + rr) * dqk + cc) : 0.0f;
    }
    for (int e = tid; e < kBN * dv; e += kThreads) {
      const int rr = e / dv, cc = e % dv;
      Vs[e] = (j0 + rr < T_) ? Elem<T>::load(v, (hq + j0 + rr) * dv + cc) : 0.0f;
    }
    if (tid < kBN) colg[tid] = (j0 + tid < T_) ? a2[hq + j0 + tid] : -INFINITY;
    __syncthreads();

    // S and gated C' for 4 columns per thread
#pragma unroll
    for (int u = 0; u < kBN / 8; ++u) {
      const int c = c8 + 8 * u, gj = j0 + c;
      float s = 0.0f;
      for (int d = 0; d < dqk; ++d) s = fmaf(Qs[r * dqk + d], Ks[c * ldk + d], s);
      float cp = 0.0f;
      if (gi < T_ && gj <= gi) cp = s * scale * exp2f(colg[c] - rowp);   // eqs (81)-(82)
      Ps[r * (kBN + 1) + c] = cp;
      bsum += cp;                                                          // eq (83)
    }
    __syncthreads();

    // O[r][c8 + 8w] += sum_c P[r][c] V[c][c8 + 8w]
    for (int c = 0; c < kBN; ++c) {
      const float p = Ps[r * (kBN + 1) + c];
#pragma unroll
      for (int w = 0; w < kAcc; ++w) {
        const int col = c8 + 8 * w;
        if (col < dv) acc[w] = fmaf(p, Vs[c * dv + col], acc[w]);
      }
    }
  }

  // the 8 threads of a row hold partial row sums: combine them
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) bsum += __shfl_xor_sync(0xffffffffu, bsum, o);
  if (gi >= T_) return;
  const float m = mrow[hq + gi];
  const float nrm = fmaxf(fabsf(bsum), expf(-m));                          // eq (84)
  const float inv = nrm > 0.0f ? 1.0f / nrm : 0.0f;
#pragma unroll
  for (int w = 0; w < kAcc; ++w) {
    const int col = c8 + 8 * w;
    if (col < dv) Elem<T>::store(h, (hq + gi) * dv + col, acc[w] * inv);     // eqs (85)-(86)
  }
  if (c8 == 0) {
    if (m_out) m_out[hq + gi] = m;
    if (n_out) n_out[hq + gi] = nrm;
    if (b_out) b_out[hq + gi] = bsum;
  }
}

size_t simt_smem_bytes(int dqk, int dv) {
  return sizeof(float) * ((size_t)kBM * dqk + (size_t)kBN * (dqk + 1) + (size_t)kBN * dv +
                          (size_t)kBM * (kBN + 1) + kBN);
}

template <typename T>
cudaError_t launch_t(const FwdArgs& a, cudaStream_t stream) {
  const size_t smem = simt_smem_bytes(a.dqk, a.dv);
  cudaError_t e = cudaFuncSetAttribute(fwd_simt_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const long long nqt = (a.T + kBM - 1) / kBM;
  const long long grid = nqt * a.BH;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  fwd_simt_kernel<T><<<(unsigned)grid, kThreads, smem, stream>>>(
      (const T*)a.q, (const T*)a.k, (const T*)a.v, a.g.a2, a.g.p2, a.g.m, (T*)a.h, a.m_out, a.b_out, a.n_out,
      a.T, a.dqk, a.dv, a.scale);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_simt(const FwdArgs& a, cudaStream_t stream) {
  if (a.BH <= 0 || a.T <= 0) return cudaSuccess;
  if (a.dqk > kMaxD || a.dv > kMaxD) return cudaErrorInvalidValue;
  return a.dtype == kF32 ? launch_t<float>(a, stream) : launch_t<__nv_bfloat16>(a, stream);
}

}  // namespace mlstm
