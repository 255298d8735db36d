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
// CUDA-core path (fp32, and bf16 shapes the tensor-core kernels do not
// tile): the five T x T products run in one batched GEMM kernel of this file
// (fp32 accumulation), each over its causal part only; the elementwise work
// between them is a second kernel: a warp per query row recomputes D' from
// the gate terms, forms C~', b, n, dn, db, writes G and P = C~'/n (zero above
// the diagonal), the row sums of dD~ and per-block column sums.  A last
// kernel turns the row and column sums into the gate gradients with suffix
// sums.  Every T x T matrix is materialised in the workspace, for all heads
// at once.

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

// An unevaluated sum hi + lo of fp32 values, added with error-free (two-sum)
// steps: suffix sums over 16k tokens as accurate as fp64 at fp32 speed (the
// fp64 rate of this part is a small fraction of its fp32 rate).
struct Sum2 {
  float hi, lo;
};
__device__ __forceinline__ Sum2 sum2_add(Sum2 a, float b) {
  const float s = a.hi + b, bb = s - a.hi;
  const float e = (a.hi - (s - bb)) + (b - bb);        // a.hi + b == s + e exactly
  const float lo = a.lo + e, hi = s + lo;
  return {hi, lo - (hi - s)};
}
__device__ __forceinline__ Sum2 sum2_add(Sum2 a, Sum2 b) { return sum2_add(sum2_add(a, b.hi), b.lo); }
__device__ __forceinline__ Sum2 sum2_shfl_down(Sum2 v, int o) {
  return {__shfl_down_sync(0xffffffffu, v.hi, o), __shfl_down_sync(0xffffffffu, v.lo, o)};
}

// Gate gradients of one head (one CTA): d i~_k = Ccol_k and d log f_k =
// sum_{i>=k} R_i - sum_{j>=k} Ccol_j (the rows >= k minus the columns >= k of
// the lower triangle), in two-sum fp32 arithmetic, times d log f / d f~.
__global__ void __launch_bounds__(1024)
bwd_gates_kernel(const float* __restrict__ R, const float* __restrict__ Ccol, const float* __restrict__ fg,
                 float* __restrict__ dig, float* __restrict__ dfg, int T, int forget_exp) {
  __shared__ Sum2 sh[32];
  const int bh = blockIdx.x;
  const size_t hb = (size_t)bh * T;
  const int per = (T + blockDim.x - 1) / blockDim.x;
  const int t0 = min(T, (int)threadIdx.x * per), t1 = min(T, t0 + per);
  // local totals of (R - Ccol) over this thread's segment
  Sum2 seg = {0.0f, 0.0f};
  for (int t = t0; t < t1; ++t) seg = sum2_add(sum2_add(seg, R[hb + t]), -Ccol[hb + t]);
  // exclusive suffix sum of the segment totals over threads (reverse scan)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  Sum2 x = seg;
  for (int o = 1; o < 32; o <<= 1) {
    const Sum2 y = sum2_shfl_down(x, o);
    if (lane + o < 32) x = sum2_add(x, y);
  }
  if (lane == 0) sh[warp] = x;
  __syncthreads();
  if (warp == 0) {
    Sum2 w = lane < (int)(blockDim.x >> 5) ? sh[lane] : Sum2{0.0f, 0.0f};
    for (int o = 1; o < 32; o <<= 1) {
      const Sum2 y = sum2_shfl_down(w, o);
      if (lane + o < 32) w = sum2_add(w, y);
    }
    sh[lane] = w;                      // inclusive suffix over warps
  }
  __syncthreads();
  // totals of later threads: the later warps', then this warp's later lanes
  // (x minus seg: this lane's inclusive suffix without its own segment)
  Sum2 after = warp + 1 < (int)(blockDim.x >> 5) ? sh[warp + 1] : Sum2{0.0f, 0.0f};
  after = sum2_add(after, sum2_add(x, Sum2{-seg.hi, -seg.lo}));
  for (int t = t1 - 1; t >= t0; --t) {
    const float c = Ccol[hb + t];
    after = sum2_add(sum2_add(after, R[hb + t]), -c);   // now the suffix from t
    dig[hb + t] = c;
    // d f~ = (d log f / d f~) d log f: sigma(-f~) for log f = log sigmoid(f~)
    // (eq 104), 1 for the exponential activation log f = f~ (eq 70's gamma = exp)
    dfg[hb + t] = (after.hi + after.lo) * (forget_exp ? 1.0f : sigmoid(-fg[hb + t]));
  }
}

// ---------------------------------------------------------------- batched GEMM (CUDA cores)
// Row-major C[m][n] = alpha sum_k opA(m, k) opB(k, n) for every head b of a
// batch, fp32 accumulation: opA(m, k) = A[m][k] (TA: A[k][m]), opB(k, n) =
// B[k][n] (TB: B[n][k]).  The products of eqs (82), (87), (98)-(100) use only
// the causal part of a T x T operand, which `causal` restricts to:
//   kLowerOut  output tiles with some n <= m (S, dC: read for j <= i only;
//              tiles wholly above the diagonal are not written),
//   kKUpToM    k <= m (dQ = s G K: G[i][j] = 0 for j > i),
//   kKFromM    k >= m (dK = s G^T Q, dV = P^T dH: G, P zero above the diagonal).
// 64 x 64 output tiles, 16-deep k steps through shared memory, 256 threads,
// a 4 x 4 block of outputs per thread.
enum Causal : int { kFull = 0, kLowerOut = 1, kKUpToM = 2, kKFromM = 3 };
constexpr int kGBM = 64, kGBN = 64, kGBK = 16;

template <typename EA, typename EB, typename EC, bool TA, bool TB, int CAUSAL>
__global__ void __launch_bounds__(256)
gemm_kernel(const EA* __restrict__ A, const EB* __restrict__ B, EC* __restrict__ C, int M, int N, int K, int lda,
            int ldb, int ldc, long long sA, long long sB, long long sC, float alpha, int tiles_m, int tiles_n) {
  __shared__ float As[kGBK][kGBM + 4];
  __shared__ float Bs[kGBK][kGBN + 4];
  const long long tiles = (long long)tiles_m * tiles_n;
  const long long bid = blockIdx.x;
  const int b = (int)(bid / tiles);
  const int tile = (int)(bid % tiles);
  const int m0 = (tile / tiles_n) * kGBM, n0 = (tile % tiles_n) * kGBN;
  if (CAUSAL == kLowerOut && n0 > m0 + kGBM - 1) return;          // wholly above the diagonal
  const int k_lo = CAUSAL == kKFromM ? (m0 / kGBK) * kGBK : 0;
  const int k_hi = CAUSAL == kKUpToM ? min(K, m0 + kGBM) : K;
  A += (size_t)b * sA;
  B += (size_t)b * sB;
  C += (size_t)b * sC;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;          // 16 x 16 threads, 4 x 4 outputs each
  float acc[4][4] = {};
  for (int k0 = k_lo; k0 < k_hi; k0 += kGBK) {
    // stage a 16 x 64 slab of opA (k x m) and of opB (k x n): 1024 values each, 4 per thread
    for (int e = threadIdx.x; e < kGBK * kGBM; e += 256) {
      int kk, mm;
      if (TA) { mm = e % kGBM; kk = e / kGBM; } else { kk = e % kGBK; mm = e / kGBK; }
      const int gk = k0 + kk, gm = m0 + mm;
      float x = 0.0f;
      if (gk < k_hi && gm < M) x = Elem<EA>::load(A, TA ? (size_t)gk * lda + gm : (size_t)gm * lda + gk);
      As[kk][mm] = x;
    }
    for (int e = threadIdx.x; e < kGBK * kGBN; e += 256) {
      int kk, nn;
      if (TB) { kk = e % kGBK; nn = e / kGBK; } else { nn = e % kGBN; kk = e / kGBN; }
      const int gk = k0 + kk, gn = n0 + nn;
      float x = 0.0f;
      if (gk < k_hi && gn < N) x = Elem<EB>::load(B, TB ? (size_t)gn * ldb + gk : (size_t)gk * ldb + gn);
      Bs[kk][nn] = x;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kGBK; ++kk) {
      float a[4], bb[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) a[r] = As[kk][ty * 4 + r];
#pragma unroll
      for (int c = 0; c < 4; ++c) bb[c] = Bs[kk][tx * 4 + c];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(a[r], bb[c], acc[r][c]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int gm = m0 + ty * 4 + r;
    if (gm >= M) continue;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int gn = n0 + tx * 4 + c;
      if (gn < N) Elem<EC>::store(C, (size_t)gm * ldc + gn, alpha * acc[r][c]);
    }
  }
}

template <typename EA, typename EB, typename EC, bool TA, bool TB, int CAUSAL>
bool gemm(const void* A, const void* B, void* C, int M, int N, int K, int lda, int ldb, int ldc, long long sA,
          long long sB, long long sC, float alpha, int batch, cudaStream_t st) {
  const int tm = (M + kGBM - 1) / kGBM, tn = (N + kGBN - 1) / kGBN;
  const long long blocks = (long long)batch * tm * tn;
  if (blocks > 0x7fffffffLL) return false;
  gemm_kernel<EA, EB, EC, TA, TB, CAUSAL><<<(unsigned)blocks, 256, 0, st>>>(
      static_cast<const EA*>(A), static_cast<const EB*>(B), static_cast<EC*>(C), M, N, K, lda, ldb, ldc, sA, sB, sC,
      alpha, tm, tn);
  return cudaGetLastError() == cudaSuccess;
}

// The five products of the CUDA-core path for element type E (q, k, v, dh,
// G, P, dq, dk, dv), S and dC in fp32.
template <typename E>
bool bwd_products_simt(const void* q, const void* k, const void* v, const void* dh, float* S, float* dC,
                       const void* G, const void* P, void* dq, void* dk, void* dv, int BH, int T, int d_qk, int d_v,
                       float s, cudaStream_t st, bool first_half) {
  const long long TT = (long long)T * T, Tq = (long long)T * d_qk, Tv = (long long)T * d_v;
  if (first_half) {
    // S = s Q K^T (82) and dC = dH V^T (87), their lower triangles
    return gemm<E, E, float, false, true, kLowerOut>(q, k, S, T, T, d_qk, d_qk, d_qk, T, Tq, Tq, TT, s, BH, st) &&
           gemm<E, E, float, false, true, kLowerOut>(dh, v, dC, T, T, d_v, d_v, d_v, T, Tv, Tv, TT, 1.0f, BH, st);
  }
  // dQ = s G K (98), dK = s G^T Q (99), dV = P^T dH (100) over the lower triangle of G, P
  return gemm<E, E, E, false, false, kKUpToM>(G, k, dq, T, d_qk, T, T, d_qk, d_qk, TT, Tq, Tq, s, BH, st) &&
         gemm<E, E, E, true, false, kKFromM>(G, q, dk, T, d_qk, T, T, d_qk, d_qk, TT, Tq, Tq, s, BH, st) &&
         gemm<E, E, E, true, false, kKFromM>(P, dh, dv, T, d_v, T, T, d_v, d_v, TT, Tv, Tv, 1.0f, BH, st);
}

// The tensor-core path (defined at the end of this file).  Gate terms are in
// `gate_ws` already; dh is dL/dH~; the forward's H~ goes to (or, saved, is
// read from) `*hf_out`.
int bwd_tc_path(const void* q, const void* k, const void* v, const float* fgate_pre, const void* dh, void* dq,
                void* dk, void* dv, float* d_igate, float* d_fgate, int BH, int T, int d_qk, int d_v,
                void* workspace, cudaStream_t st, int forget_exp, const void* h_saved, const float* n_saved,
                const float* b_saved, const void** hf_out);

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

namespace {

// Extra workspace of the options, after the path's own layout: dL/dH~ of an
// output gate, and (CUDA-core path) the forward's H~, which the output-gate
// gradient needs.
size_t og_extra(long long BH, int T, int d_v, int dtype, bool tc, const mlstm_options* opt) {
  if (!opt || !opt->ogate_pre) return 0;
  const size_t es = dtype == MLSTM_F32 ? 4 : 2;
  const size_t one = r256((size_t)BH * T * d_v * es);
  return tc ? one : 2 * one;
}

// Workspace of the path that will run for these sizes and options, and
// whether it is the tensor-core path.
size_t bwd_need(long long BH, int T, int d_qk, int d_v, int dtype, const mlstm_options* opt, bool* tc) {
  *tc = use_tc_path(T, d_qk, d_v, dtype);
  const size_t base = *tc ? tc_layout(BH, T, d_v).total : bwd_layout(BH, T, dtype).total;
  return base + og_extra(BH, T, d_v, dtype, *tc, opt);
}

// The parallel backward for every entry point (part 28/30 eqs 87-105; the
// output gate of eq 78 and the forget activation of eq 70 from `opt`).
int bwd_impl(const void* q, const void* k, const void* v, const float* igate_pre, const float* fgate_pre,
             const void* dh, const void* h_saved, const float* n_saved, const float* b_saved, void* dq, void* dk,
             void* dv, float* d_igate, float* d_fgate, void* d_ogate, int B, int H, int T, int d_qk, int d_v,
             int dtype, void* workspace, size_t workspace_bytes, const mlstm_options* opt, void* stream) {
  if (B < 0 || H < 0 || T < 0 || T > kMaxBwdT) return MLSTM_EINVAL;
  if (d_qk < 1 || d_v < 1 || d_qk > 512 || d_v > 512) return MLSTM_EINVAL;
  if (dtype != MLSTM_F32 && dtype != MLSTM_BF16) return MLSTM_EDTYPE;
  const long long BH = (long long)B * H;
  if (BH > (1 << 20)) return MLSTM_EINVAL;
  if (BH == 0 || T == 0) return MLSTM_OK;
  if (!q || !k || !v || !igate_pre || !fgate_pre || !dh || !dq || !dk || !dv || !d_igate || !d_fgate)
    return MLSTM_EINVAL;
  const void* og = opt ? opt->ogate_pre : nullptr;
  if (og && !d_ogate) return MLSTM_EINVAL;
  const int fexp = opt ? opt->forget_exp : 0;
  if (!workspace) return MLSTM_EWORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return MLSTM_EALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  bool tc = false;
  size_t need = bwd_need(BH, T, d_qk, d_v, dtype, opt, &tc);
  if (tc && workspace_bytes < need) {            // too small for the tensor-core path: the CUDA-core one
    tc = false;
    need = bwd_layout(BH, T, dtype).total + og_extra(BH, T, d_v, dtype, false, opt);
  }
  if (workspace_bytes < need) return MLSTM_EWORKSPACE;
  char* w = static_cast<char*>(workspace);
  const size_t base = tc ? tc_layout(BH, T, d_v).total : bwd_layout(BH, T, dtype).total;
  const size_t es = dtype == MLSTM_F32 ? 4 : 2;
  const size_t vbytes = r256((size_t)BH * T * d_v * es);
  const long long nv = BH * T * d_v;

  // output gate: the core works on dL/dH~ = dL/dh (.) sigmoid(o~)     (78)
  const void* dht = dh;
  if (og) {
    if (launch_ogate_bwd_in(dh, og, w + base, nv, dtype, st) != cudaSuccess) return MLSTM_ECUDA;
    dht = w + base;
  }
  // gate terms of eqs (79)-(81) with the chosen forget activation: a2, p2, m
  const size_t gate_bytes = mlstm_parallel_fwd_workspace(1, (int)BH, T);
  int rc = mlstm_gate_prep_opt(igate_pre, fgate_pre, 1, (int)BH, T, w, gate_bytes, opt, stream);
  if (rc != MLSTM_OK) return rc;
  const size_t arr = gate_bytes / 3;           // three arrays of equal, 256-aligned size
  GateTerms g{reinterpret_cast<float*>(w), reinterpret_cast<float*>(w + arr), reinterpret_cast<float*>(w + 2 * arr)};
  const bool saved = h_saved && n_saved && b_saved;
  const void* ht = saved ? h_saved : nullptr;   // H~ of the forward, for the output-gate gradient

  if (tc) {
    rc = bwd_tc_path(q, k, v, fgate_pre, dht, dq, dk, dv, d_igate, d_fgate, (int)BH, T, d_qk, d_v, workspace, st,
                     fexp, saved ? h_saved : nullptr, saved ? n_saved : nullptr, saved ? b_saved : nullptr, &ht);
    if (rc != MLSTM_OK) return rc;
  } else {
    const BwdLayout L = bwd_layout(BH, T, dtype);
    char* S = w + L.gate;
    char* dC = S + L.S;
    char* G = dC + L.dC;
    char* P = G + L.G;
    float* R = reinterpret_cast<float*>(P + L.P);
    float* Cpart = reinterpret_cast<float*>(reinterpret_cast<char*>(R) + L.R);
    float* Ccol = reinterpret_cast<float*>(reinterpret_cast<char*>(Cpart) + L.Cpart);
    const float s = (float)(1.0 / sqrt((double)d_qk));
    const bool f32 = dtype == MLSTM_F32;
    // S = s Q K^T (82) and dC = dH~ V^T (87) over the lower triangle
    if (!(f32 ? bwd_products_simt<float>(q, k, v, dht, (float*)S, (float*)dC, G, P, dq, dk, dv, (int)BH, T, d_qk,
                                         d_v, s, st, true)
              : bwd_products_simt<__nv_bfloat16>(q, k, v, dht, (float*)S, (float*)dC, G, P, dq, dk, dv, (int)BH, T,
                                                 d_qk, d_v, s, st, true)))
      return MLSTM_ECUDA;
    const int nblk = L.nblk;
    const size_t smem = (size_t)T * sizeof(float);
    if (f32) {
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
    // dQ = s G K (98), dK = s G^T Q (99), dV = P^T dH~ (100) over the lower triangle of G, P
    if (!(f32 ? bwd_products_simt<float>(q, k, v, dht, (float*)S, (float*)dC, G, P, dq, dk, dv, (int)BH, T, d_qk,
                                         d_v, s, st, false)
              : bwd_products_simt<__nv_bfloat16>(q, k, v, dht, (float*)S, (float*)dC, G, P, dq, dk, dv, (int)BH, T,
                                                 d_qk, d_v, s, st, false)))
      return MLSTM_ECUDA;
    const long long ncol = BH * T;
    bwd_colsum_kernel<<<(unsigned)((ncol + 255) / 256), 256, 0, st>>>(Cpart, Ccol, T, nblk, ncol);
    bwd_gates_kernel<<<(unsigned)BH, 1024, 0, st>>>(R, Ccol, fgate_pre, d_igate, d_fgate, T, fexp);
    if (cudaGetLastError() != cudaSuccess) return MLSTM_ECUDA;
    if (og && !ht) {
      // the forward's H~ (eqs 79-86) for the output-gate gradient
      FwdArgs fa;
      fa.q = q; fa.k = k; fa.v = v; fa.h = w + base + vbytes; fa.m_out = nullptr; fa.n_out = nullptr;
      fa.g = g; fa.BH = (int)BH; fa.T = T; fa.dqk = d_qk; fa.dv = d_v; fa.dtype = dtype; fa.scale = s;
      if (!current_status(&fa.st)) return MLSTM_ECUDA;
      rc = launch_fwd_tc(fa, st);
      if (rc == kUnsupported) rc = launch_fwd_simt(fa, st) == cudaSuccess ? kOk : kCuda;
      if (rc != kOk) return rc;
      ht = fa.h;
    }
  }
  // dL/do~ = dL/dh (.) H~ (.) sigmoid'(o~)                              (78), (70)
  if (og && launch_ogate_bwd_out(dh, og, ht, d_ogate, nv, dtype, st) != cudaSuccess) return MLSTM_ECUDA;
  return MLSTM_OK;
}

}  // namespace

extern "C" {

size_t mlstm_parallel_bwd_workspace_opt(int B, int H, int T, int d_qk, int d_v, int dtype, const mlstm_options* opt) {
  if (B <= 0 || H <= 0 || T <= 0 || T > kMaxBwdT || d_qk < 1 || d_v < 1 || d_qk > 512 || d_v > 512) return 0;
  if (dtype != MLSTM_F32 && dtype != MLSTM_BF16) return 0;
  bool tc = false;
  return bwd_need((long long)B * H, T, d_qk, d_v, dtype, opt, &tc);
}

size_t mlstm_parallel_bwd_workspace_ex(int B, int H, int T, int d_qk, int d_v, int dtype) {
  return mlstm_parallel_bwd_workspace_opt(B, H, T, d_qk, d_v, dtype, nullptr);
}

size_t mlstm_parallel_bwd_workspace(int B, int H, int T, int dtype) {
  if (B <= 0 || H <= 0 || T <= 0 || T > kMaxBwdT) return 0;
  if (dtype != MLSTM_F32 && dtype != MLSTM_BF16) return 0;
  return bwd_layout((long long)B * H, T, dtype).total;
}

int mlstm_parallel_bwd(const void* q, const void* k, const void* v, const float* igate_pre, const float* fgate_pre,
                       const void* dh, void* dq, void* dk, void* dv, float* d_igate, float* d_fgate, int B, int H,
                       int T, int d_qk, int d_v, int dtype, void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(q, k, v, igate_pre, fgate_pre, dh, nullptr, nullptr, nullptr, dq, dk, dv, d_igate, d_fgate, nullptr,
                  B, H, T, d_qk, d_v, dtype, workspace, workspace_bytes, nullptr, stream);
}

int mlstm_parallel_bwd_saved(const void* q, const void* k, const void* v, const float* igate_pre,
                             const float* fgate_pre, const void* dh, const void* h, const float* n, const float* b,
                             void* dq, void* dk, void* dv, float* d_igate, float* d_fgate, int B, int H, int T,
                             int d_qk, int d_v, int dtype, void* workspace, size_t workspace_bytes, void* stream) {
  if (!h || !n || !b) return MLSTM_EINVAL;
  return bwd_impl(q, k, v, igate_pre, fgate_pre, dh, h, n, b, dq, dk, dv, d_igate, d_fgate, nullptr, B, H, T, d_qk,
                  d_v, dtype, workspace, workspace_bytes, nullptr, stream);
}

int mlstm_parallel_bwd_opt(const void* q, const void* k, const void* v, const float* igate_pre,
                           const float* fgate_pre, const void* dh, const void* h_saved, const float* n_saved,
                           const float* b_saved, void* dq, void* dk, void* dv, float* d_igate, float* d_fgate,
                           void* d_ogate, int B, int H, int T, int d_qk, int d_v, int dtype, void* workspace,
                           size_t workspace_bytes, const mlstm_options* opt, void* stream) {
  const int nsaved = (h_saved != nullptr) + (n_saved != nullptr) + (b_saved != nullptr);
  if (nsaved != 0 && nsaved != 3) return MLSTM_EINVAL;
  return bwd_impl(q, k, v, igate_pre, fgate_pre, dh, h_saved, n_saved, b_saved, dq, dk, dv, d_igate, d_fgate,
                  d_ogate, B, H, T, d_qk, d_v, dtype, workspace, workspace_bytes, opt, stream);
}

}  // extern "C"

namespace mlstm {
namespace {

// Tensor-core path: the forward (H~, n, signed b) unless given, the tile
// kernel (G, P, row and column sums of dD~), the three products dQ, dK, dV
// over the lower triangle of G and P, the gate gradients.
int bwd_tc_path(const void* q, const void* k, const void* v, const float* fgate_pre, const void* dh, void* dq,
                void* dk, void* dv, float* d_igate, float* d_fgate, int BH, int T, int d_qk, int d_v,
                void* workspace, cudaStream_t st, int forget_exp, const void* h_saved, const float* n_saved,
                const float* b_saved, const void** hf_out) {
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

  // the gate terms are in the workspace already (the caller's gate pass)
  const size_t arr = L.gate / 3;
  GateTerms g{reinterpret_cast<float*>(gate_ws), reinterpret_cast<float*>(gate_ws + arr),
              reinterpret_cast<float*>(gate_ws + 2 * arr)};
  DevStatus ds;
  if (!current_status(&ds)) return MLSTM_ECUDA;
  const float s = (float)(1.0 / sqrt((double)d_qk));
  const bool saved = h_saved && n_saved && b_saved;
  int rc;
  if (!saved) {
    // forward: H~, n and the signed row sums b (eqs 79-86)
    FwdArgs fa;
    fa.q = q; fa.k = k; fa.v = v; fa.h = hf; fa.m_out = nullptr; fa.n_out = nrow; fa.b_out = brow;
    fa.g = g; fa.BH = BH; fa.T = T; fa.dqk = d_qk; fa.dv = d_v; fa.dtype = kBF16; fa.scale = s; fa.st = ds;
    rc = launch_fwd_tc(fa, st);
    if (rc == kUnsupported) rc = launch_fwd_simt(fa, st) == cudaSuccess ? kOk : kCuda;
    if (rc != kOk) return rc;
  }
  *hf_out = saved ? h_saved : hf;
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
  bwd_gates_kernel<<<(unsigned)BH, 1024, 0, st>>>(R, Ccol, fgate_pre, d_igate, d_fgate, T, forget_exp);
  return cudaGetLastError() == cudaSuccess ? MLSTM_OK : MLSTM_ECUDA;
}

}  // namespace
}  // namespace mlstm
