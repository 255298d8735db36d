// Stabilized parallel mLSTM backward pass.
//
// "xLSTM: Extended Long Short-Term Memory", part 28/30, "Parallel mLSTM
// Backward Pass", eqs (87)-(105), for one head with S = Q K^T / sqrt(d):
//   dC    = dH~ V^T                                              (87)
//   dn_i  = -(sum_j C~'_ij dC_ij) / n_i^2                         (88)-(89)
//   db_i  = sign(b_i) dn_i  if |b_i| > exp(-m_i), else 0          (90)
//   dC~'  = dC / n + db  (both broadcast along the row)           (91)-(93)
//   G     = D' (.) dC~',   dD~ = S (.) G                           (94)-(95)
//   dQ    = G K / sqrt(d),  dK = G^T Q / sqrt(d),  dV = (C~'/n)^T dH~   (98)-(100)
//   d i~_k = sum_{i>=k} dD~_ik,   d f~_k = sigma(-f~_k) sum_{j<k} sum_{i>=k} dD~_ij   (102)-(105)
// (eq 90 prints sign(n); the derivative of max(|b|, e^-m) is sign(b)).  The
// stabilizer m is a constant, as on the pages.  S and dC stay in fp32 (in
// bf16 the cancellation in dC/n + db costs dq about 3 % at T = 300: measured).
//
// The five T x T products are plain batched GEMMs (cuBLAS, tensor cores for
// bf16); the elementwise work between them is one kernel of this file: a warp
// per query row recomputes D' from the gate terms, forms C~', b, n, dn, db,
// writes G and P = C~'/n (zero above the diagonal), the row sums of dD~ and
// per-block column sums.  A last kernel turns the row and column sums into
// the gate gradients with suffix sums.  Every T x T matrix is materialised in
// the workspace, for all heads at once.
#include <cublas_v2.h>

#include <algorithm>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "internal.h"
#include "mlstm.h"

namespace mlstm {
namespace {

constexpr int kRowsPerCta = 32;            // one warp per row
constexpr int kMaxBwdT = 16384;            // column sums of a block live in shared memory

size_t r256(size_t x) { return (x + 255) & ~(size_t)255; }

struct BwdLayout {
  size_t gate, S, dC, G, P, R, Cpart, Ccol, total;
  int nblk;
};

BwdLayout bwd_layout(long long BH, int T, int dtype) {
  BwdLayout L;
  const size_t es = dtype == kF32 ? 4 : 2;
  const size_t tt = (size_t)BH * T * T;
  L.nblk = (T + kRowsPerCta - 1) / kRowsPerCta;
  L.gate = mlstm_parallel_fwd_workspace(1, (int)BH, T);
  L.S = r256(tt * 4);
  L.dC = r256(tt * 4);
  L.G = r256(tt * es);
  L.P = r256(tt * es);
  L.R = r256((size_t)BH * T * 4);
  L.Cpart = r256((size_t)BH * L.nblk * T * 4);
  L.Ccol = r256((size_t)BH * T * 4);
  L.total = L.gate + L.S + L.dC + L.G + L.P + L.R + L.Cpart + L.Ccol;
  return L;
}

template <typename E>
__device__ __forceinline__ void put(E* p, size_t i, float x) { Elem<E>::store(p, i, x); }

// One warp per query row i of one head: D', C~', b, n, dn, db, then G, P,
// the row sum of dD~ and this block's column sums of dD~.
template <typename E>
__global__ void __launch_bounds__(kRowsPerCta * 32)
bwd_rows_kernel(const float* __restrict__ S, const float* __restrict__ dC, GateTerms g, E* __restrict__ G,
                E* __restrict__ P, float* __restrict__ R, float* __restrict__ Cpart, int T, int nblk) {
  extern __shared__ float colsum[];          // [T]
  const int bh = blockIdx.x / nblk, blk = blockIdx.x % nblk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i0 = blk * kRowsPerCta;
  const int jmax = min(T, i0 + kRowsPerCta);  // columns this block can touch
  for (int j = threadIdx.x; j < jmax; j += blockDim.x) colsum[j] = 0.0f;
  __syncthreads();
  const int i = i0 + warp;
  const size_t hb = (size_t)bh * T;
  if (i < T) {
    const size_t row = ((size_t)bh * T + i) * T;
    const float p2i = g.p2[hb + i], mi = g.m[hb + i];
    float b = 0.0f, r = 0.0f;
    for (int j = lane; j <= i; j += 32) {
      const float ct = S[row + j] * exp2f(g.a2[hb + j] - p2i);           // C~' = S (.) D'
      b += ct;
      r = fmaf(ct, dC[row + j], r);
    }
    b = warp_sum(b);
    r = warp_sum(r);
    const float floor = expf(-mi);
    const float n = fmaxf(fabsf(b), floor);
    const float inv = 1.0f / n;
    const float dn = -r * inv * inv;                                       // (89)
    const float db = fabsf(b) > floor ? (b > 0.0f ? dn : (b < 0.0f ? -dn : 0.0f)) : 0.0f;   // (90)
    float rs = 0.0f;
    for (int j = lane; j < T; j += 32) {
      if (j <= i) {
        const float s = S[row + j];
        const float dp = exp2f(g.a2[hb + j] - p2i);
        const float gv = dp * fmaf(dC[row + j], inv, db);                   // D' (.) dC~'
        const float dd = s * gv;                                           // dD~
        put(G, row + j, gv);
        put(P, row + j, s * dp * inv);                                     // C~' / n
        rs += dd;
        atomicAdd(&colsum[j], dd);
      } else {
        put(G, row + j, 0.0f);
        put(P, row + j, 0.0f);
      }
    }
    rs = warp_sum(rs);
    if (lane == 0) R[hb + i] = rs;
  }
  __syncthreads();
  float* out = Cpart + ((size_t)bh * nblk + blk) * T;
  for (int j = threadIdx.x; j < T; j += blockDim.x) out[j] = j < jmax ? colsum[j] : 0.0f;
}

// Column sums of dD~: Ccol[bh][t] = sum over the row blocks of the partials
// (blocks whose rows all lie above column t contribute nothing).
__global__ void bwd_colsum_kernel(const float* __restrict__ Cpart, float* __restrict__ Ccol, int T, int nblk,
                                  long long n) {
  const long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= n) return;
  const int bh = (int)(x / T), t = (int)(x % T);
  float c = 0.0f;
  for (int b2 = t / kRowsPerCta; b2 < nblk; ++b2) c += Cpart[((size_t)bh * nblk + b2) * T + t];
  Ccol[x] = c;
}

// Gate gradients of one head (one CTA): column sums from the block partials,
// then d i~_k = Ccol_k and d fbar_k = sum_{i>=k} R_i - sum_{j>=k} Ccol_j
// (the rows >= k minus the columns >= k of the lower triangle), in fp64.
__global__ void __launch_bounds__(1024)
bwd_gates_kernel(const float* __restrict__ R, const float* __restrict__ Ccol, const float* __restrict__ fg,
                 float* __restrict__ dig, float* __restrict__ dfg, int T) {
  __shared__ double sh[32];
  const int bh = blockIdx.x;
  const size_t hb = (size_t)bh * T;
  const int per = (T + blockDim.x - 1) / blockDim.x;
  const int t0 = min(T, (int)threadIdx.x * per), t1 = min(T, t0 + per);
  // local totals of (R - Ccol) over this thread's segment
  double seg = 0.0;
  for (int t = t0; t < t1; ++t) seg += (double)R[hb + t] - (double)Ccol[hb + t];
  // exclusive suffix sum of the segment totals over threads (reverse scan)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  double x = seg;
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_down_sync(0xffffffffu, x, o);
    if (lane + o < 32) x += y;
  }
  if (lane == 0) sh[warp] = x;
  __syncthreads();
  if (warp == 0) {
    double w = lane < (int)(blockDim.x >> 5) ? sh[lane] : 0.0;
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_down_sync(0xffffffffu, w, o);
      if (lane + o < 32) w += y;
    }
    sh[lane] = w;                      // inclusive suffix over warps
  }
  __syncthreads();
  double after = (warp + 1 < (int)(blockDim.x >> 5) ? sh[warp + 1] : 0.0) + (x - seg);   // totals of later threads
  for (int t = t1 - 1; t >= t0; --t) {
    const double c = Ccol[hb + t];
    after += (double)R[hb + t] - c;    // now the suffix from t
    dig[hb + t] = (float)c;
    dfg[hb + t] = (float)(after * (double)sigmoid(-fg[hb + t]));    // sigma(-f~) d fbar (eq 104)
  }
}

struct Blas {
  cublasHandle_t h = nullptr;
};
Blas g_blas[64];
std::mutex g_blas_mu;

cublasHandle_t blas_handle() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(g_blas_mu);
  if (!g_blas[dev].h && cublasCreate(&g_blas[dev].h) != CUBLAS_STATUS_SUCCESS) g_blas[dev].h = nullptr;
  return g_blas[dev].h;
}

// Column-major batched GEMM C = op(A) op(B) (the row-major products of this
// file are expressed through their transposes).
bool gemm(cublasHandle_t h, cublasOperation_t ta, cublasOperation_t tb, int m, int n, int k, float alpha,
          const void* A, cudaDataType ta_t, int lda, long long sa, const void* B, cudaDataType tb_t, int ldb,
          long long sb, void* C, cudaDataType tc_t, int ldc, long long sc, int batch) {
  const float beta = 0.0f;
  return cublasGemmStridedBatchedEx(h, ta, tb, m, n, k, &alpha, A, ta_t, lda, sa, B, tb_t, ldb, sb, &beta, C, tc_t,
                                    ldc, sc, batch, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT) == CUBLAS_STATUS_SUCCESS;
}

int bwd_tc_path(const void* q, const void* k, const void* v, const float* igate_pre, const float* fgate_pre,
                const void* dh, void* dq, void* dk, void* dv, float* d_igate, float* d_fgate, int BH, int T, int d_qk,
                int d_v, void* workspace, cudaStream_t st, const void* h_saved = nullptr,
                const float* n_saved = nullptr, const float* b_saved = nullptr);

// Workspace of the tensor-core path: gate terms, the forward's H~ (d_v
// columns) and row statistics, bf16 G and P with rows of ldT = T rounded up
// to 8 (16-byte pitch for TMA), the tiles' row and column sums of dD~, R,
// Ccol.
struct TcLayout {
  size_t gate, hf, rowv, G, P, part, R, Ccol, total;
  int ldT, nb;
};

TcLayout tc_layout(long long BH, int T, int dv) {
  TcLayout L;
  L.ldT = (T + 7) & ~7;
  L.nb = (T + 127) / 128;
  L.gate = mlstm_parallel_fwd_workspace(1, (int)BH, T);
  L.hf = r256((size_t)BH * T * dv * 2);
  L.rowv = r256((size_t)BH * T * 4);                // one of: n, b, 1/n, db
  L.G = r256((size_t)BH * T * L.ldT * 2);
  L.P = L.G;
  L.part = r256((size_t)BH * L.nb * T * 4);         // one of: Rpart, Cpart
  L.R = r256((size_t)BH * T * 4);
  L.Ccol = L.R;
  L.total = L.gate + L.hf + 4 * L.rowv + L.G + L.P + 2 * L.part + L.R + L.Ccol;
  return L;
}

// The tensor-core path runs for bf16 on the sm_100 family unless
// MLSTM_BWD_PATH=blas in the environment selects the cuBLAS path (tests).
bool use_tc_path(int T, int dqk, int dv, int dtype) {
  static const char* force = getenv("MLSTM_BWD_PATH");
  if (force && force[0] == 'b') return false;
  return bwd_tc_supported(T, dqk, dv, dtype) && device_is_sm100_family();
}

}  // namespace
}  // namespace mlstm

using namespace mlstm;

extern "C" {

size_t mlstm_parallel_bwd_workspace_ex(int B, int H, int T, int d_qk, int d_v, int dtype) {
  if (B <= 0 || H <= 0 || T <= 0 || T > kMaxBwdT || d_qk < 1 || d_v < 1 || d_qk > 512 || d_v > 512) return 0;
  if (dtype != MLSTM_F32 && dtype != MLSTM_BF16) return 0;
  if (use_tc_path(T, d_qk, d_v, dtype)) return tc_layout((long long)B * H, T, d_v).total;
  return bwd_layout((long long)B * H, T, dtype).total;
}

size_t mlstm_parallel_bwd_workspace(int B, int H, int T, int dtype) {
  if (B <= 0 || H <= 0 || T <= 0 || T > kMaxBwdT) return 0;
  if (dtype != MLSTM_F32 && dtype != MLSTM_BF16) return 0;
  return bwd_layout((long long)B * H, T, dtype).total;
}

int mlstm_parallel_bwd(const void* q, const void* k, const void* v, const float* igate_pre, const float* fgate_pre,
                       const void* dh, void* dq, void* dk, void* dv, float* d_igate, float* d_fgate, int B, int H,
                       int T, int d_qk, int d_v, int dtype, void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || H < 0 || T < 0 || T > kMaxBwdT) return MLSTM_EINVAL;
  if (d_qk < 1 || d_v < 1 || d_qk > 512 || d_v > 512) return MLSTM_EINVAL;
  if (dtype != MLSTM_F32 && dtype != MLSTM_BF16) return MLSTM_EDTYPE;
  const long long BH = (long long)B * H;
  if (BH > (1 << 20)) return MLSTM_EINVAL;
  if (BH == 0 || T == 0) return MLSTM_OK;
  if (!q || !k || !v || !igate_pre || !fgate_pre || !dh || !dq || !dk || !dv || !d_igate || !d_fgate)
    return MLSTM_EINVAL;
  if (!workspace) return MLSTM_EWORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return MLSTM_EALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (use_tc_path(T, d_qk, d_v, dtype) && workspace_bytes >= tc_layout(BH, T, d_v).total)
    return bwd_tc_path(q, k, v, igate_pre, fgate_pre, dh, dq, dk, dv, d_igate, d_fgate, (int)BH, T, d_qk, d_v,
                       workspace, st);
  if (workspace_bytes < mlstm_parallel_bwd_workspace(B, H, T, dtype)) return MLSTM_EWORKSPACE;
  const BwdLayout L = bwd_layout(BH, T, dtype);
  char* w = static_cast<char*>(workspace);
  char* gate_ws = w;
  char* S = w + L.gate;
  char* dC = w + L.gate + L.S;
  char* G = w + L.gate + L.S + L.dC;
  char* P = G + L.G;
  float* R = reinterpret_cast<float*>(P + L.P);
  float* Cpart = reinterpret_cast<float*>(reinterpret_cast<char*>(R) + L.R);
  float* Ccol = reinterpret_cast<float*>(reinterpret_cast<char*>(Cpart) + L.Cpart);

  // gate terms of eqs (79)-(81): a2, p2, m
  int rc = mlstm_gate_prep(igate_pre, fgate_pre, 1, (int)BH, T, gate_ws, L.gate, stream);
  if (rc != MLSTM_OK) return rc;
  const long long BHT = BH * T;
  const size_t arr = (L.gate) / 3;           // three arrays of equal, 256-aligned size
  GateTerms g{reinterpret_cast<float*>(gate_ws), reinterpret_cast<float*>(gate_ws + arr),
              reinterpret_cast<float*>(gate_ws + 2 * arr)};
  (void)BHT;

  cublasHandle_t h = blas_handle();
  if (!h || cublasSetStream(h, st) != CUBLAS_STATUS_SUCCESS) return MLSTM_ECUDA;
  const cudaDataType et = dtype == MLSTM_F32 ? CUDA_R_32F : CUDA_R_16BF;
  const float s = (float)(1.0 / sqrt((double)d_qk));
  const long long TT = (long long)T * T, Tq = (long long)T * d_qk, Tv = (long long)T * d_v;
  const int nb = (int)BH;
  // row-major S = s Q K^T  <=>  col-major S^T = s K Q^T
  if (!gemm(h, CUBLAS_OP_T, CUBLAS_OP_N, T, T, d_qk, s, k, et, d_qk, Tq, q, et, d_qk, Tq, S, CUDA_R_32F, T, TT, nb))
    return MLSTM_ECUDA;
  // row-major dC = dH V^T  (87)
  if (!gemm(h, CUBLAS_OP_T, CUBLAS_OP_N, T, T, d_v, 1.0f, v, et, d_v, Tv, dh, et, d_v, Tv, dC, CUDA_R_32F, T, TT, nb))
    return MLSTM_ECUDA;
  const int nblk = L.nblk;
  const size_t smem = (size_t)T * sizeof(float);
  if (dtype == MLSTM_F32) {
    if (cudaFuncSetAttribute(bwd_rows_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return MLSTM_ECUDA;
    bwd_rows_kernel<float><<<(unsigned)(BH * nblk), kRowsPerCta * 32, smem, st>>>(
        reinterpret_cast<const float*>(S), reinterpret_cast<const float*>(dC), g, reinterpret_cast<float*>(G),
        reinterpret_cast<float*>(P), R, Cpart, T, nblk);
  } else {
    if (cudaFuncSetAttribute(bwd_rows_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return MLSTM_ECUDA;
    bwd_rows_kernel<__nv_bfloat16><<<(unsigned)(BH * nblk), kRowsPerCta * 32, smem, st>>>(
        reinterpret_cast<const float*>(S), reinterpret_cast<const float*>(dC), g,
        reinterpret_cast<__nv_bfloat16*>(G), reinterpret_cast<__nv_bfloat16*>(P), R, Cpart, T, nblk);
  }
  if (cudaGetLastError() != cudaSuccess) return MLSTM_ECUDA;
  // row-major dQ = s G K  <=>  col-major dQ^T = s K^T G^T          (98)
  if (!gemm(h, CUBLAS_OP_N, CUBLAS_OP_N, d_qk, T, T, s, k, et, d_qk, Tq, G, et, T, TT, dq, et, d_qk, Tq, nb))
    return MLSTM_ECUDA;
  // row-major dK = s G^T Q  <=>  col-major dK^T = s Q^T G          (99)
  if (!gemm(h, CUBLAS_OP_N, CUBLAS_OP_T, d_qk, T, T, s, q, et, d_qk, Tq, G, et, T, TT, dk, et, d_qk, Tq, nb))
    return MLSTM_ECUDA;
  // row-major dV = P^T dH  <=>  col-major dV^T = dH^T P            (100)
  if (!gemm(h, CUBLAS_OP_N, CUBLAS_OP_T, d_v, T, T, 1.0f, dh, et, d_v, Tv, P, et, T, TT, dv, et, d_v, Tv, nb))
    return MLSTM_ECUDA;
  const long long ncol = BH * T;
  bwd_colsum_kernel<<<(unsigned)((ncol + 255) / 256), 256, 0, st>>>(Cpart, Ccol, T, nblk, ncol);
  bwd_gates_kernel<<<(unsigned)BH, 1024, 0, st>>>(R, Ccol, fgate_pre, d_igate, d_fgate, T);
  return cudaGetLastError() == cudaSuccess ? MLSTM_OK : MLSTM_ECUDA;
}

int mlstm_parallel_bwd_saved(const void* q, const void* k, const void* v, const float* igate_pre,
                             const float* fgate_pre, const void* dh, const void* h, const float* n, const float* b,
                             void* dq, void* dk, void* dv, float* d_igate, float* d_fgate, int B, int H, int T,
                             int d_qk, int d_v, int dtype, void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || H < 0 || T < 0 || T > kMaxBwdT) return MLSTM_EINVAL;
  if (d_qk < 1 || d_v < 1 || d_qk > 512 || d_v > 512) return MLSTM_EINVAL;
  if (dtype != MLSTM_F32 && dtype != MLSTM_BF16) return MLSTM_EDTYPE;
  const long long BH = (long long)B * H;
  if (BH > (1 << 20)) return MLSTM_EINVAL;
  if (BH == 0 || T == 0) return MLSTM_OK;
  if (!h || !n || !b) return MLSTM_EINVAL;
  if (!q || !k || !v || !igate_pre || !fgate_pre || !dh || !dq || !dk || !dv || !d_igate || !d_fgate)
    return MLSTM_EINVAL;
  if (!workspace) return MLSTM_EWORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return MLSTM_EALIGN;
  if (use_tc_path(T, d_qk, d_v, dtype) && workspace_bytes >= tc_layout(BH, T, d_v).total)
    return bwd_tc_path(q, k, v, igate_pre, fgate_pre, dh, dq, dk, dv, d_igate, d_fgate, (int)BH, T, d_qk, d_v,
                       workspace, static_cast<cudaStream_t>(stream), h, n, b);
  return mlstm_parallel_bwd(q, k, v, igate_pre, fgate_pre, dh, dq, dk, dv, d_igate, d_fgate, B, H, T, d_qk, d_v,
                            dtype, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace mlstm {
namespace {

// Tensor-core path: gate pass, forward (H~, n, signed b), the tile kernel
// (G, P, row and column sums of dD~), the three products dQ, dK, dV over the
// lower triangle of G and P, the gate gradients.
int bwd_tc_path(const void* q, const void* k, const void* v, const float* igate_pre, const float* fgate_pre,
                const void* dh, void* dq, void* dk, void* dv, float* d_igate, float* d_fgate, int BH, int T, int d_qk,
                int d_v, void* workspace, cudaStream_t st, const void* h_saved, const float* n_saved,
                const float* b_saved) {
  const TcLayout L = tc_layout(BH, T, d_v);
  char* w = static_cast<char*>(workspace);
  char* gate_ws = w;
  char* hf = gate_ws + L.gate;
  float* nrow = reinterpret_cast<float*>(hf + L.hf);
  float* brow = reinterpret_cast<float*>(reinterpret_cast<char*>(nrow) + L.rowv);
  float* invn = reinterpret_cast<float*>(reinterpret_cast<char*>(brow) + L.rowv);
  float* dbv = reinterpret_cast<float*>(reinterpret_cast<char*>(invn) + L.rowv);
  char* G = reinterpret_cast<char*>(dbv) + L.rowv;
  char* P = G + L.G;
  float* Rpart = reinterpret_cast<float*>(P + L.P);
  float* Cpart = reinterpret_cast<float*>(reinterpret_cast<char*>(Rpart) + L.part);
  float* R = reinterpret_cast<float*>(reinterpret_cast<char*>(Cpart) + L.part);
  float* Ccol = reinterpret_cast<float*>(reinterpret_cast<char*>(R) + L.R);

  int rc = mlstm_gate_prep(igate_pre, fgate_pre, 1, BH, T, gate_ws, L.gate, st);
  if (rc != MLSTM_OK) return rc;
  const size_t arr = L.gate / 3;
  GateTerms g{reinterpret_cast<float*>(gate_ws), reinterpret_cast<float*>(gate_ws + arr),
              reinterpret_cast<float*>(gate_ws + 2 * arr)};
  DevStatus ds;
  if (!current_status(&ds)) return MLSTM_ECUDA;
  const float s = (float)(1.0 / sqrt((double)d_qk));
  const bool saved = h_saved && n_saved && b_saved;
  if (!saved) {
    // forward: H~, n and the signed row sums b (eqs 79-86)
    FwdArgs fa;
    fa.q = q; fa.k = k; fa.v = v; fa.h = hf; fa.m_out = nullptr; fa.n_out = nrow; fa.b_out = brow;
    fa.g = g; fa.BH = BH; fa.T = T; fa.dqk = d_qk; fa.dv = d_v; fa.dtype = kBF16; fa.scale = s; fa.st = ds;
    rc = launch_fwd_tc(fa, st);
    if (rc == kUnsupported) rc = launch_fwd_simt(fa, st) == cudaSuccess ? kOk : kCuda;
    if (rc != kOk) return rc;
  }
  BwdTileArgs ta;
  ta.q = q; ta.k = k; ta.v = v; ta.dh = dh; ta.g = g;
  ta.h = saved ? h_saved : hf;
  ta.nrow = saved ? n_saved : nrow;
  ta.brow = saved ? b_saved : brow;
  ta.invn = invn; ta.db = dbv; ta.G = G; ta.P = P; ta.Rpart = Rpart; ta.Cpart = Cpart; ta.R = R; ta.Ccol = Ccol;
  ta.BH = BH; ta.T = T; ta.ldT = L.ldT; ta.dqk = d_qk; ta.dv = d_v; ta.scale = s; ta.st = ds;
  rc = launch_bwd_tiles(ta, st);
  if (rc != kOk) return rc;

  // dQ, dK, dV over the lower triangle on the tensor cores            (98)-(100)
  BwdProdArgs pa;
  pa.q = q; pa.k = k; pa.dh = dh; pa.G = G; pa.P = P; pa.dq = dq; pa.dk = dk; pa.dvo = dv;
  pa.BH = BH; pa.T = T; pa.ldT = L.ldT; pa.dqk = d_qk; pa.dv = d_v; pa.scale = s; pa.st = ds;
  rc = launch_bwd_products(pa, st);
  if (rc != kOk) return rc;
  bwd_gates_kernel<<<(unsigned)BH, 1024, 0, st>>>(R, Ccol, fgate_pre, d_igate, d_fgate, T);
  return cudaGetLastError() == cudaSuccess ? MLSTM_OK : MLSTM_ECUDA;
}

}  // namespace
}  // namespace mlstm
