// One stabilized recurrent mLSTM step over a batch of heads (generation).
//
// The recurrence differentiated by "xLSTM: Extended Long Short-Term Memory",
// part 28/30, eqs (59)-(70), with the output gate of part 17/30 eq (27):
//   m' = max(log sigmoid(f~) + m, i~),  f' = exp(log sigmoid(f~) + m - m'),
//   i' = exp(i~ - m'),  C <- f'C + i' v (s k)^T,  n <- f'n + i' s k,
//   h  = sigmoid(o) * (C q) / max(|n.q|, exp(-m')),     s = 1/sqrt(d_qk).
//
// The step is a single streaming pass over the matrix memory C, so it is
// bound by HBM bandwidth.  A cluster of R CTAs owns one head: CTA r updates
// rows [r*dv/R, (r+1)*dv/R) of C with 128-bit streaming loads and stores,
// one warp per row, and folds C_new q into the numerator of h as it goes.  It
// also updates the slice r of n and its partial dot product with q.  The
// partials meet through distributed shared memory after a cluster barrier, so
// n and m are updated in place with no second pass and no global scratch.
#include "internal.h"

namespace mlstm {
namespace {

constexpr int kThreads = 256, kWarps = kThreads / 32, kMaxD = 512;

__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_peer_smem(const float* local, unsigned rank) {
  unsigned a = (unsigned)__cvta_generic_to_shared(local), ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}

// NV = float4 chunks per lane per row (d_qk <= 128 * NV).
template <typename T, int NV>
__global__ void __launch_bounds__(kThreads)
step_kernel(float* __restrict__ C, float* __restrict__ n, float* __restrict__ m,
            const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
            const T* __restrict__ o, const float* __restrict__ ig, const float* __restrict__ fg,
            T* __restrict__ h, int dqk, int dv, int R, float scale, int forget_exp) {
  __shared__ __align__(16) float ks[kMaxD];   // s * k
  __shared__ __align__(16) float qs[kMaxD];
  __shared__ float hs[kMaxD];                 // numerators (C_new q) of this CTA's rows
  __shared__ float red[32];
  __shared__ float partial;                   // this CTA's share of n_new . q

  const unsigned rank = cluster_rank();
  const int bh = (int)(blockIdx.x / R);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // gate scalars (every CTA of the cluster reads the old m before the barrier)
  const float lf = forget_exp ? fg[bh] : log_sigmoid(fg[bh]);    // exponential or sigmoid forget
  const float igv = ig[bh];
  const float m_old = m[bh];
  const float m_new = fmaxf(lf + m_old, igv);
  const float fp = expf(lf + m_old - m_new);
  const float ip = expf(igv - m_new);

  for (int j = tid; j < dqk; j += kThreads) {
    ks[j] = Elem<T>::load(k, (size_t)bh * dqk + j) * scale;
    qs[j] = Elem<T>::load(q, (size_t)bh * dqk + j);
  }
  __syncthreads();

  // slice of n owned by this CTA, and its contribution to n_new . q
  const int ns = dqk / R, nj0 = (int)rank * ns;
  float pq = 0.0f;
  for (int j = nj0 + tid; j < nj0 + ns; j += kThreads) {
    const float nn = fp * n[(size_t)bh * dqk + j] + ip * ks[j];
    n[(size_t)bh * dqk + j] = nn;
    pq += nn * qs[j];
  }
  pq = block_sum(pq, red);
  if (tid == 0) partial = pq;
  cluster_arrive_release();          // publishes `partial` to the cluster

  // stream this CTA's rows of C: C_new = f' C + (i' v_r) (s k); h_r = C_new . q
  float4 kr[NV], qr[NV];
#pragma unroll
  for (int u = 0; u < NV; ++u) {
    const int c = (lane + 32 * u) * 4;
    kr[u] = c < dqk ? *reinterpret_cast<const float4*>(&ks[c]) : make_float4(0.f, 0.f, 0.f, 0.f);
    qr[u] = c < dqk ? *reinterpret_cast<const float4*>(&qs[c]) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const int rows = dv / R, r0 = (int)rank * rows;
  for (int lr = warp; lr < rows; lr += kWarps) {
    const int row = r0 + lr;
    float4* crow = reinterpret_cast<float4*>(C + ((size_t)bh * dv + row) * dqk);
    const float iv = ip * Elem<T>::load(v, (size_t)bh * dv + row);
    float4 x[NV];
#pragma unroll
    for (int u = 0; u < NV; ++u)
      if ((lane + 32 * u) * 4 < dqk) x[u] = __ldcs(crow + lane + 32 * u);
    float dot = 0.0f;
#pragma unroll
    for (int u = 0; u < NV; ++u) {
      if ((lane + 32 * u) * 4 < dqk) {
        float4 y;
        y.x = fmaf(fp, x[u].x, iv * kr[u].x);
        y.y = fmaf(fp, x[u].y, iv * kr[u].y);
        y.z = fmaf(fp, x[u].z, iv * kr[u].z);
        y.w = fmaf(fp, x[u].w, iv * kr[u].w);
        __stcs(crow + lane + 32 * u, y);
        dot = fmaf(y.x, qr[u].x, dot);
        dot = fmaf(y.y, qr[u].y, dot);
        dot = fmaf(y.z, qr[u].z, dot);
        dot = fmaf(y.w, qr[u].w, dot);
      }
    }
    dot = warp_sum(dot);
    if (lane == 0) hs[lr] = dot;
  }

  cluster_wait_acquire();            // every CTA has read m_old and published its partial
  float nq = 0.0f;
  for (int r = 0; r < R; ++r) nq += ld_peer_smem(&partial, (unsigned)r);
  __syncthreads();                   // hs complete
  if (rank == 0 && tid == 0) m[bh] = m_new;
  const float nrm = fmaxf(fabsf(nq), expf(-m_new));
  const float inv = nrm > 0.0f ? 1.0f / nrm : 0.0f;
  for (int lr = tid; lr < rows; lr += kThreads) {
    const int row = r0 + lr;
    float hv = hs[lr] * inv;
    if (o) hv *= sigmoid(Elem<T>::load(o, (size_t)bh * dv + row));
    Elem<T>::store(h, (size_t)bh * dv + row, hv);
  }
  // keep this CTA's shared memory alive until every peer has read `partial`
  cluster_arrive_release();
  cluster_wait_acquire();
}

template <typename T, int NV>
cudaError_t launch_nv(const StepArgs& a, int R, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.BH * R));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)R;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, step_kernel<T, NV>, a.C, a.n, a.m, (const T*)a.q, (const T*)a.k,
                            (const T*)a.v, (const T*)a.o, a.ig, a.fg, (T*)a.h, a.dqk, a.dv, R, a.scale,
                            a.forget_exp);
}

template <typename T>
cudaError_t launch_t(const StepArgs& a, int R, cudaStream_t stream) {
  const int nv = (a.dqk + 127) / 128;
  switch (nv) {
    case 1: return launch_nv<T, 1>(a, R, stream);
    case 2: return launch_nv<T, 2>(a, R, stream);
    case 3: return launch_nv<T, 3>(a, R, stream);
    default: return launch_nv<T, 4>(a, R, stream);
  }
}

}  // namespace

cudaError_t launch_step(const StepArgs& a, cudaStream_t stream) {
  if (a.BH <= 0) return cudaSuccess;
  if (a.dqk > kMaxD || a.dv > kMaxD || a.dqk % 4 != 0) return cudaErrorInvalidValue;
  // cluster size: 8 CTAs per head when rows and the n vector split evenly
  const int R = (a.dv % 8 == 0 && a.dqk % 8 == 0 && a.dv >= 64) ? 8 : 1;
  if ((long long)a.BH * R > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaError_t e = a.dtype == kF32 ? launch_t<float>(a, R, stream) : launch_t<__nv_bfloat16>(a, R, stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mlstm
