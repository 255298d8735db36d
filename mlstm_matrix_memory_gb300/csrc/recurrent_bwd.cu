// Backward pass of the recurrent mLSTM form (backpropagation through time),
// "xLSTM: Extended Long Short-Term Memory", part 28/30 eqs (59)-(70), with
// the output gate of part 17/30 eq (27) and the gate activations of the
// recurrent step:
//   C_t = f_t C_{t-1} + i_t v_t (s k_t)^T,  n_t = f_t n_{t-1} + i_t s k_t,
//   h~_t = C_t q_t / N_t,  N_t = max(|n_t^T q_t|, 1),  h_t = sigma(o~_t) (.) h~_t,
// i_t = exp(i~_t), f_t = sigma(f~_t) (or exp(f~_t)), s = 1/sqrt(d_qk).
//
// Four passes, each state-carrying pass holding its matrix in registers the
// way step_seq.cu does (a CTA owns 64 rows of one head, a warp 8 rows, a lane
// every 32nd column pair):
//
// 1. forward sweep (stabilized: running max m, states C' = e^-m C, n' = e^-m n,
//    so C/N = C'/N' with N' = max(|n'.q|, e^-m)).  Per token it forms h~, the
//    output-gate gradient (eq 70), and this CTA's share of
//        dq_t = (C'_t^T dh~_t - (h~_t . dh~_t) Omega_t n'_t) / N'_t        (eq 64)
//    (the share of h~.dh~ over its rows goes into the second term, so the
//    shares add up), and of h~.dh~ Omega, and log N_t.
// 2. backward sweep over t = T-1..0 of dC_t, dn_t, eqs (60)-(61), kept as
//    dC^ = e^-nu dC, dn^ = e^-nu dn with nu_t = max(log f_{t+1} + nu_{t+1},
//    -log N_t): both recurrence coefficients are then at most 1.  Per token
//        dv_t = i_t dC_t (s k_t),  dk_t = s i_t (dC_t^T v_t + dn_t)        (eqs 62-63)
//    (dv rows are complete in the CTA; dk is a per-CTA share).
// 3. per token: the shares summed into dq, dk; d i~_t = k_t . dk_t, which is
//    eq (69) (i_t scales k_t wherever k_t enters), and r_t = q_t.dq_t - k_t.dk_t.
// 4. per head: d f~_t = act'(f~_t) sum_{u >= t} r_u.  This is eq (68): adding a
//    to log f_t changes the cell exactly as scaling q_u by e^a and k_u by e^-a
//    for every u >= t does (the normalizer included, since n_u.q_u scales with
//    C_u q_u), so dL/dlog f_t is that suffix sum; act' = dlog f/df~ is
//    sigma(-f~) (eq 104) or 1 for the exponential activation.
//
// Work per token and head: 3 d_v d_qk fused multiply-adds in each sweep.
#include <cmath>

#include "internal.h"
#include "mlstm.h"

namespace mlstm {
namespace {

constexpr int kRW = 8;                      // rows per warp
constexpr int kChunk = 16;                  // tokens staged in shared memory at a time
constexpr int kGroup = 4;                   // tokens per cross-warp reduction
constexpr int kMaxR = 8;                    // CTAs per head (d_v <= 512, 64 rows a CTA at least)
constexpr float kRenorm = 1.0f / 16777216.0f;   // 2^-24: fold the scale into the state below this

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// One chunk of tokens in shared memory; the row arrays hold the CTA's RPC
// rows.  Sweep 2 also stages every CTA's share of h~.dh~ Omega and log N.
template <typename T>
struct Chunk {
  T* q;        // [kChunk][qs]
  T* k;        // [kChunk][qs]
  T* v;        // [kChunk][RPC]
  T* o;        // [kChunk][RPC]
  T* dh;       // [kChunk][RPC]
  float* ig;   // [kChunk]
  float* fg;   // [kChunk]
  float* lnN;  // [kChunk]
  float* sp;   // [kMaxR][kChunk]
};

// q and k rows are qs elements apart: d_qk for bf16 (widened to fp32 rows of
// PADC columns per chunk), PADC for fp32 (staged straight into padded rows).
template <typename T>
__host__ __device__ constexpr size_t chunk_bytes(int qs, int rpc) {
  return (size_t)kChunk * (2 * qs + 3 * rpc) * sizeof(T) + (size_t)kChunk * (3 + kMaxR) * sizeof(float);
}

template <typename T>
__device__ __forceinline__ Chunk<T> chunk_at(uint8_t* base, int qs, int rpc) {
  Chunk<T> b;
  b.q = reinterpret_cast<T*>(base);
  b.k = b.q + kChunk * qs;
  b.v = b.k + kChunk * qs;
  b.o = b.v + kChunk * rpc;
  b.dh = b.o + kChunk * rpc;
  b.ig = reinterpret_cast<float*>(b.dh + kChunk * rpc);
  b.fg = b.ig + kChunk;
  b.lnN = b.fg + kChunk;
  b.sp = b.lnN + kChunk;
  return b;
}

struct Inputs {
  const void* q;
  const void* k;
  const void* v;
  const void* o;       // may be null
  const void* dh;
  const float* ig;
  const float* fg;
};

// Shared scratch besides the two staging buffers (PADC = 32 NC columns):
//  qf, kf  the chunk's q and k rows as fp32, zero past d_qk     [kChunk][PADC]
//          (bf16 only: fp32 rows are staged padded in the chunk buffer)
//  vf, dhf the chunk's v and dh~ = sigma(o~) dh rows as fp32, zero past the
//          CTA's rows                                              [kChunk][RPC]
//          (bf16 only: fp32 rows are used, and dh turned into dh~, in place)
//  tsc     per-token scalars of the chunk, four arrays of kChunk
//          (sweep 1: f', i', e^-m, m; sweep 2: alpha, beta, i e^nu, h~.dh~ Omega)
//  col     per token of a reduction group, every warp's column share [G][NW][PADC]
//  vec     per token, n' (sweep 1) or dn^ (sweep 2), in the warps' scaled form
//  gbuf    per token, the CTA's row sums (C' q or dC^ k), unscaled   [G][RPC]
//  sc      per token, eight scalars;  tok  its token index within the chunk
struct Scratch {
  float* qf;
  float* kf;
  float* vf;
  float* dhf;
  float* tsc;
  float* col;
  float* vec;
  float* gbuf;
  float* sc;
  int* tok;
};

__host__ __device__ constexpr size_t scratch_bytes(int padc, int nw, bool wide) {
  return (wide ? 0 : (size_t)2 * kChunk * (padc + nw * kRW) * sizeof(float)) + (size_t)4 * kChunk * sizeof(float) +
         (size_t)kGroup * (nw + 1) * padc * sizeof(float) + (size_t)kGroup * nw * kRW * sizeof(float) +
         (size_t)kGroup * 8 * sizeof(float) + kGroup * sizeof(int);
}

__device__ __forceinline__ Scratch scratch_at(uint8_t* base, int padc, int nw, bool wide) {
  Scratch r;
  r.qf = reinterpret_cast<float*>(base);
  r.kf = r.qf + (wide ? 0 : kChunk * padc);
  r.vf = r.kf + (wide ? 0 : kChunk * padc);
  r.dhf = r.vf + (wide ? 0 : kChunk * nw * kRW);
  r.tsc = r.dhf + (wide ? 0 : kChunk * nw * kRW);
  r.col = r.tsc + 4 * kChunk;
  r.vec = r.col + kGroup * nw * padc;
  r.gbuf = r.vec + kGroup * padc;
  r.sc = r.gbuf + kGroup * nw * kRW;
  r.tok = reinterpret_cast<int*>(r.sc + kGroup * 8);
  return r;
}

// bf16: the staged chunk's q and k rows converted to fp32 into qf, kf (rows of
// PADC columns, zeros past d_qk and past the chunk's last token), and v and
// dh~ = sigma(o~) dh into vf, dhf (zeros past the CTA's rows).  fp32: dh turned
// into dh~ in place (the other rows are used as staged).
template <typename T, int PADC, int RPC>
__device__ __forceinline__ void widen(const Scratch& sx, const Chunk<T>& b, int cnt, int dqk, int nrows, bool has_o) {
  if constexpr (sizeof(T) == 4) {
    if (has_o)
      for (int idx = threadIdx.x; idx < cnt * nrows; idx += blockDim.x) {
        const int t = idx / nrows, r = idx - t * nrows;
        float* d = reinterpret_cast<float*>(b.dh) + t * RPC + r;
        *d *= sigmoid(Elem<T>::load(b.o, (size_t)t * RPC + r));
      }
  } else {
    for (int idx = threadIdx.x; idx < kChunk * PADC; idx += blockDim.x) {
      const int t = idx / PADC, c = idx - t * PADC;
      const bool on = t < cnt && c < dqk;
      sx.qf[idx] = on ? Elem<T>::load(b.q, (size_t)t * dqk + c) : 0.0f;
      sx.kf[idx] = on ? Elem<T>::load(b.k, (size_t)t * dqk + c) : 0.0f;
    }
    for (int idx = threadIdx.x; idx < kChunk * RPC; idx += blockDim.x) {
      const int t = idx / RPC, r = idx - t * RPC;
      const bool on = t < cnt && r < nrows;
      sx.vf[idx] = on ? Elem<T>::load(b.v, (size_t)idx) : 0.0f;
      const float dhv = on ? Elem<T>::load(b.dh, (size_t)idx) : 0.0f;
      sx.dhf[idx] = on && has_o ? sigmoid(Elem<T>::load(b.o, (size_t)idx)) * dhv : dhv;
    }
  }
}

// Copies of tokens [tok, tok+cnt) into `b` (all nthreads threads).  `sweep2`
// also fetches the R CTAs' shares of h~.dh~ Omega and log N.
template <typename T>
__device__ __forceinline__ void stage(const Chunk<T>& b, const Inputs& in, size_t tok, int cnt, int dqk, int qs,
                                      int dv, int rpc, int r0, int nrows, bool vec_rows, bool sweep2, const float* sp,
                                      const float* lnN, int R, long long BHT) {
  constexpr int E = 16 / sizeof(T);
  const int nthreads = blockDim.x;
  const T* q = static_cast<const T*>(in.q);
  const T* k = static_cast<const T*>(in.k);
  const T* v = static_cast<const T*>(in.v);
  const T* o = static_cast<const T*>(in.o);
  const T* dh = static_cast<const T*>(in.dh);
  const int per_row = dqk / E;
  for (int p = threadIdx.x; p < cnt * per_row; p += nthreads) {
    const int t = p / per_row, e = (p - t * per_row) * E;
    cp_async16(b.q + t * qs + e, q + (tok + t) * dqk + e);
    cp_async16(b.k + t * qs + e, k + (tok + t) * dqk + e);
  }
  if (vec_rows) {
    const int per = nrows / E;
    for (int p = threadIdx.x; p < cnt * per; p += nthreads) {
      const int t = p / per, e = (p % per) * E;
      cp_async16(b.v + t * rpc + e, v + (tok + t) * dv + r0 + e);
      cp_async16(b.dh + t * rpc + e, dh + (tok + t) * dv + r0 + e);
      if (o) cp_async16(b.o + t * rpc + e, o + (tok + t) * dv + r0 + e);
    }
  } else {
    for (int p = threadIdx.x; p < cnt * nrows; p += nthreads) {
      const int t = p / nrows, e = p % nrows;
      b.v[t * rpc + e] = v[(tok + t) * dv + r0 + e];
      b.dh[t * rpc + e] = dh[(tok + t) * dv + r0 + e];
      if (o) b.o[t * rpc + e] = o[(tok + t) * dv + r0 + e];
    }
  }
  for (int t = threadIdx.x; t < cnt; t += nthreads) {
    cp_async4(b.ig + t, in.ig + tok + t);
    cp_async4(b.fg + t, in.fg + tok + t);
    if (sweep2) cp_async4(b.lnN + t, lnN + tok + t);
  }
  if (sweep2)
    for (int p = threadIdx.x; p < R * cnt; p += nthreads) {
      const int r = p / cnt, t = p % cnt;
      cp_async4(b.sp + r * kChunk + t, sp + (size_t)r * BHT + tok + t);
    }
}

// The eight per-lane row partial sums of a warp reduced in halving steps:
// afterwards lane l (l % 4 == 0) holds the full sum of row myrow(l).
__device__ __forceinline__ float reduce_rows(const float (&dot)[kRW], int lane) {
  float e[4], f2[2], g;
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    e[j] = (b4 ? dot[j + 4] : dot[j]) + __shfl_xor_sync(0xffffffffu, b4 ? dot[j] : dot[j + 4], 16);
#pragma unroll
  for (int j = 0; j < 2; ++j)
    f2[j] = (b3 ? e[j + 2] : e[j]) + __shfl_xor_sync(0xffffffffu, b3 ? e[j] : e[j + 2], 8);
  g = (b2 ? f2[1] : f2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? f2[0] : f2[1], 4);
  g += __shfl_xor_sync(0xffffffffu, g, 2);
  g += __shfl_xor_sync(0xffffffffu, g, 1);
  return g;
}

// Eight consecutive fp32 row values (16-byte aligned), the same for every lane.
__device__ __forceinline__ void load_rows(const float* p, float (&x)[kRW]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// Inclusive scans over the 32 lanes.
__device__ __forceinline__ float scan_add(float x, int lane) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  return x;
}
__device__ __forceinline__ float scan_max(float x, int lane) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x = fmaxf(x, y);
  }
  return x;
}

// x_t = max(g_t + x_{t-1}, h_t) over the lanes, from x_{-1} = x0, in closed
// form: x_t = cs_t + max(x0, max_{j<=t}(h_j - cs_j)), cs the prefix sum of g.
// Returns x_t; *xprev gets x_{t-1}.
__device__ __forceinline__ float maxplus_scan(float g, float h, float x0, int lane, float* xprev) {
  const float cs = scan_add(g, lane);
  const float x = cs + fmaxf(x0, scan_max(h - cs, lane));
  const float up = __shfl_up_sync(0xffffffffu, x, 1);
  *xprev = lane == 0 ? x0 : up;
  return x;
}

// The state of a warp is S * c^ with one scale S for all its entries, so a
// decay multiplies S alone and the rank-one term is one fused multiply-add
// per entry; when S falls below 2^-24 it is folded into the entries.
template <int NC>
__device__ __forceinline__ void fold_scale(float (&c)[kRW][NC], float (&vecs)[NC], float& S, float decay) {
  const float s2 = S * decay;
  if (s2 < kRenorm) {
#pragma unroll
    for (int i = 0; i < kRW; ++i)
#pragma unroll
      for (int u = 0; u < NC; ++u) c[i][u] *= s2;
#pragma unroll
    for (int u = 0; u < NC; ++u) vecs[u] *= s2;
    S = 1.0f;
  } else {
    S = s2;
  }
}

// Sweep 1 (forward in time).  Grid: BH * R CTAs of NW warps; CTA (bh, r)
// owns rows [r RPC, (r+1) RPC) of head bh, RPC = 8 NW.  Per token a warp
// updates its 8 rows and its copy of n', and leaves its rows' C'q and its
// column share of C'^T dh~ in shared memory; every kGroup tokens the CTA
// forms n'.q, h~, d o~ and h~.dh~ (one warp per token) and then the dq share.
template <typename T, int NC, int NW>
__global__ void __launch_bounds__(NW * 32, 1)
rbwd_forward_kernel(Inputs in, T* __restrict__ dog, float* __restrict__ qpart, float* __restrict__ spart,
                    float* __restrict__ lnN, int Tn, int dqk, int dv, int R, float scale, int forget_exp,
                    long long BHT) {
  constexpr int NP = NC / 2, RPC = NW * kRW, PADC = 32 * NC;
  extern __shared__ __align__(16) uint8_t smem[];
  const int bh = (int)(blockIdx.x / R), rank = (int)(blockIdx.x % R);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r0 = rank * RPC;
  const int nrows = max(0, min(RPC, dv - r0));
  const int wrow = warp * kRW;
  const bool has_o = in.o != nullptr;
  const bool vec_rows = (dv * (int)sizeof(T)) % 16 == 0 && (nrows * (int)sizeof(T)) % 16 == 0 &&
                        (reinterpret_cast<uintptr_t>(in.v) & 15) == 0 &&
                        (reinterpret_cast<uintptr_t>(in.o) & 15) == 0 &&
                        (reinterpret_cast<uintptr_t>(in.dh) & 15) == 0;
  const size_t tok0 = (size_t)bh * Tn;
  constexpr bool kWide = sizeof(T) == 4;
  const int qs = kWide ? PADC : dqk;
  const size_t cb = chunk_bytes<T>(qs, RPC);
  const Scratch sx = scratch_at(smem + 2 * cb, PADC, NW, kWide);
  if constexpr (kWide) {              // what staging never writes stays zero in both chunk buffers:
    for (int idx = threadIdx.x; idx < 4 * kChunk * (PADC - dqk); idx += NW * 32) {   // q, k columns past d_qk
      const int row = idx / (PADC - dqk), cc = dqk + idx - row * (PADC - dqk);
      reinterpret_cast<float*>(smem + (row / (2 * kChunk)) * cb)[(row % (2 * kChunk)) * PADC + cc] = 0.0f;
    }
    for (int idx = threadIdx.x; idx < 4 * kChunk * (RPC - nrows); idx += NW * 32) {  // v, dh rows past the CTA's
      const int row = idx / (RPC - nrows), r = nrows + idx - row * (RPC - nrows);
      const int buf = row / (2 * kChunk), arr = (row / kChunk) & 1, t = row % kChunk;
      const Chunk<T> cbuf = chunk_at<T>(smem + buf * cb, qs, RPC);
      (arr ? cbuf.dh : cbuf.v)[t * RPC + r] = 0.0f;
    }
  }
  const int nchunks = (Tn + kChunk - 1) / kChunk;
  const int myrow = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
  const bool writer = (lane & 3) == 0;

  stage(chunk_at<T>(smem, qs, RPC), in, tok0, min(kChunk, Tn), dqk, qs, dv, RPC, r0, nrows, vec_rows, false, nullptr,
        nullptr, R, BHT);
  cp_async_commit();

  float c[kRW][NC], nn[NC];
#pragma unroll
  for (int i = 0; i < kRW; ++i)
#pragma unroll
    for (int u = 0; u < NC; ++u) c[i][u] = 0.0f;
#pragma unroll
  for (int u = 0; u < NC; ++u) nn[u] = 0.0f;
  float S = 1.0f;
  float m_carry = -INFINITY;          // warp 0: m after the last processed chunk
  int slot = 0;

  for (int ch = 0; ch < nchunks; ++ch) {
    const int t0 = ch * kChunk, cnt = min(kChunk, Tn - t0);
    if (ch + 1 < nchunks) {
      stage(chunk_at<T>(smem + ((ch + 1) & 1) * cb, qs, RPC), in, tok0 + t0 + kChunk,
            min(kChunk, Tn - t0 - kChunk), dqk, qs, dv, RPC, r0, nrows, vec_rows, false, nullptr, nullptr, R, BHT);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const Chunk<T> b = chunk_at<T>(smem + (ch & 1) * cb, qs, RPC);
    widen<T, PADC, RPC>(sx, b, cnt, dqk, nrows, has_o);
    const float* qf = kWide ? reinterpret_cast<const float*>(b.q) : sx.qf;
    const float* kf = kWide ? reinterpret_cast<const float*>(b.k) : sx.kf;
    const float* vf = kWide ? reinterpret_cast<const float*>(b.v) : sx.vf;
    const float* dhf = kWide ? reinterpret_cast<const float*>(b.dh) : sx.dhf;
    if (warp == 0) {
      // the stabilizer over the chunk: m_t = max(log f_t + m_{t-1}, i~_t)
      const bool on = lane < cnt;
      const float lf = on ? (forget_exp ? b.fg[lane] : log_sigmoid(b.fg[lane])) : 0.0f;
      const float ig = on ? b.ig[lane] : -INFINITY;
      float mprev;
      const float m = maxplus_scan(lf, ig, m_carry, lane, &mprev);
      if (on) {
        sx.tsc[lane] = expf(lf + mprev - m);              // f'
        sx.tsc[kChunk + lane] = expf(ig - m);             // i'
        sx.tsc[2 * kChunk + lane] = expf(-m);             // normalizer floor
        sx.tsc[3 * kChunk + lane] = m;
      }
      m_carry = __shfl_sync(0xffffffffu, m, cnt - 1);
    }
    __syncthreads();
    for (int tt = 0; tt < cnt; ++tt) {
      fold_scale(c, nn, S, sx.tsc[tt]);
      const float a = __fdividef(sx.tsc[kChunk + tt] * scale, S);   // k's coefficient in the scaled update
      float vr[kRW], dr[kRW];
      load_rows(vf + tt * RPC + wrow, vr);
      load_rows(dhf + tt * RPC + wrow, dr);
      float dot[kRW];
#pragma unroll
      for (int i = 0; i < kRW; ++i) dot[i] = 0.0f;
      const float* qrow = qf + tt * PADC + 2 * lane;
      const float* krow = kf + tt * PADC + 2 * lane;
      float* colw = sx.col + (slot * NW + warp) * PADC + 2 * lane;
#pragma unroll
      for (int u = 0; u < NP; ++u) {
        const float2 kx = *reinterpret_cast<const float2*>(krow + 64 * u);
        const float2 qx = *reinterpret_cast<const float2*>(qrow + 64 * u);
        const float k0 = kx.x * a, k1 = kx.y * a;
        nn[2 * u] += k0;
        nn[2 * u + 1] += k1;
        float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
        for (int i = 0; i < kRW; ++i) {
          c[i][2 * u] = fmaf(vr[i], k0, c[i][2 * u]);
          c[i][2 * u + 1] = fmaf(vr[i], k1, c[i][2 * u + 1]);
          dot[i] = fmaf(c[i][2 * u], qx.x, dot[i]);
          dot[i] = fmaf(c[i][2 * u + 1], qx.y, dot[i]);
          s0 = fmaf(c[i][2 * u], dr[i], s0);
          s1 = fmaf(c[i][2 * u + 1], dr[i], s1);
        }
        *reinterpret_cast<float2*>(colw + 64 * u) = make_float2(s0, s1);
      }
      if (warp == 0) {
        float* vw = sx.vec + slot * PADC + 2 * lane;
#pragma unroll
        for (int u = 0; u < NP; ++u) *reinterpret_cast<float2*>(vw + 64 * u) = make_float2(nn[2 * u], nn[2 * u + 1]);
      }
      const float g = reduce_rows(dot, lane);
      if (writer) sx.gbuf[slot * RPC + wrow + myrow] = g;
      if (threadIdx.x == 0) {
        sx.sc[slot * 8 + 0] = S;
        sx.tok[slot] = tt;
      }
      ++slot;
      if (slot == kGroup || tt == cnt - 1) {
        __syncthreads();
        if (warp < slot) {
          // token j = warp: n'.q, the normalizer, h~ of the CTA's rows, d o~ (70), h~.dh~
          const int j = warp, tj = sx.tok[j];
          const float Sj = sx.sc[j * 8 + 0];
          float nq = 0.0f;
          for (int cc = lane; cc < PADC; cc += 32) nq = fmaf(sx.vec[j * PADC + cc], qf[tj * PADC + cc], nq);
          nq = warp_sum(nq) * Sj;
          const float fl = sx.tsc[2 * kChunk + tj];
          const float nrm = fmaxf(fabsf(nq), fl);
          const float hs = nrm > 0.0f ? Sj / nrm : 0.0f;
          float share = 0.0f;
          for (int r = lane; r < nrows; r += 32) {
            const float hv = hs * sx.gbuf[j * RPC + r];
            const float dht = dhf[tj * RPC + r];
            share = fmaf(hv, dht, share);
            if (has_o)   // (70): h~ sigma'(o~) dh = h~ (1 - sigma(o~)) dh~
              Elem<T>::store(dog, (tok0 + t0 + tj) * dv + r0 + r,
                             hv * (1.0f - sigmoid(Elem<T>::load(b.o, (size_t)tj * RPC + r))) * dht);
          }
          share = warp_sum(share);
          if (lane == 0) {
            const float om = fabsf(nq) > fl ? (nq > 0.0f ? 1.0f : -1.0f) : 0.0f;                // Omega
            sx.sc[j * 8 + 1] = hs;
            sx.sc[j * 8 + 2] = share * om;
            sx.sc[j * 8 + 3] = fmaxf(sx.tsc[3 * kChunk + tj] + logf(fabsf(nq)), 0.0f);          // log N
          }
        }
        __syncthreads();
        for (int j = 0; j < slot; ++j) {
          const float hs = sx.sc[j * 8 + 1], so = sx.sc[j * 8 + 2];
          const size_t tokj = tok0 + t0 + sx.tok[j];
          const size_t orow = ((size_t)rank * BHT + tokj) * dqk;
          for (int cc = threadIdx.x; cc < dqk; cc += NW * 32) {
            float acc = 0.0f;
#pragma unroll
            for (int w = 0; w < NW; ++w) acc += sx.col[(j * NW + w) * PADC + cc];
            qpart[orow + cc] = (acc - so * sx.vec[j * PADC + cc]) * hs;                     // (64)
          }
          if (threadIdx.x == 0) {
            spart[(size_t)rank * BHT + tokj] = so;
            if (rank == 0) lnN[tokj] = sx.sc[j * 8 + 3];
          }
        }
        __syncthreads();
        slot = 0;
      }
    }
    __syncthreads();                  // buffer ch&1 may be refilled by the next stage
  }
}

// Sweep 2 (backward in time), same CTA layout as sweep 1.  Per token a warp
// updates its 8 rows of dC^ and its copy of dn^, and leaves its rows' dC^ k
// and its column share of dC^T v; every kGroup tokens the CTA writes the dv
// rows and the dk share.
template <typename T, int NC, int NW>
__global__ void __launch_bounds__(NW * 32, 1)
rbwd_backward_kernel(Inputs in, const float* __restrict__ spart, const float* __restrict__ lnN,
                     T* __restrict__ dvout, float* __restrict__ kpart, int Tn, int dqk, int dv, int R, float scale,
                     int forget_exp, long long BHT) {
  constexpr int NP = NC / 2, RPC = NW * kRW, PADC = 32 * NC;
  extern __shared__ __align__(16) uint8_t smem[];
  const int bh = (int)(blockIdx.x / R), rank = (int)(blockIdx.x % R);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r0 = rank * RPC;
  const int nrows = max(0, min(RPC, dv - r0));
  const int wrow = warp * kRW;
  const bool has_o = in.o != nullptr;
  const bool vec_rows = (dv * (int)sizeof(T)) % 16 == 0 && (nrows * (int)sizeof(T)) % 16 == 0 &&
                        (reinterpret_cast<uintptr_t>(in.v) & 15) == 0 &&
                        (reinterpret_cast<uintptr_t>(in.o) & 15) == 0 &&
                        (reinterpret_cast<uintptr_t>(in.dh) & 15) == 0;
  const size_t tok0 = (size_t)bh * Tn;
  constexpr bool kWide = sizeof(T) == 4;
  const int qs = kWide ? PADC : dqk;
  const size_t cb = chunk_bytes<T>(qs, RPC);
  const Scratch sx = scratch_at(smem + 2 * cb, PADC, NW, kWide);
  if constexpr (kWide) {              // what staging never writes stays zero in both chunk buffers:
    for (int idx = threadIdx.x; idx < 4 * kChunk * (PADC - dqk); idx += NW * 32) {   // q, k columns past d_qk
      const int row = idx / (PADC - dqk), cc = dqk + idx - row * (PADC - dqk);
      reinterpret_cast<float*>(smem + (row / (2 * kChunk)) * cb)[(row % (2 * kChunk)) * PADC + cc] = 0.0f;
    }
    for (int idx = threadIdx.x; idx < 4 * kChunk * (RPC - nrows); idx += NW * 32) {  // v, dh rows past the CTA's
      const int row = idx / (RPC - nrows), r = nrows + idx - row * (RPC - nrows);
      const int buf = row / (2 * kChunk), arr = (row / kChunk) & 1, t = row % kChunk;
      const Chunk<T> cbuf = chunk_at<T>(smem + buf * cb, qs, RPC);
      (arr ? cbuf.dh : cbuf.v)[t * RPC + r] = 0.0f;
    }
  }
  const int nchunks = (Tn + kChunk - 1) / kChunk;
  const int myrow = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
  const bool writer = (lane & 3) == 0;

  {
    const int t0 = (nchunks - 1) * kChunk;
    stage(chunk_at<T>(smem, qs, RPC), in, tok0 + t0, Tn - t0, dqk, qs, dv, RPC, r0, nrows, vec_rows, true, spart, lnN,
          R, BHT);
  }
  cp_async_commit();

  float dc[kRW][NC], dn[NC];
#pragma unroll
  for (int i = 0; i < kRW; ++i)
#pragma unroll
    for (int u = 0; u < NC; ++u) dc[i][u] = 0.0f;
#pragma unroll
  for (int u = 0; u < NC; ++u) dn[u] = 0.0f;
  float S = 1.0f;
  float nu_carry = -INFINITY, lf_carry = 0.0f;       // warp 0: nu and log f of the last processed token
  int slot = 0;

  for (int ch = 0; ch < nchunks; ++ch) {
    const int ci = nchunks - 1 - ch;
    const int t0 = ci * kChunk, cnt = min(kChunk, Tn - t0);
    if (ch + 1 < nchunks) {
      stage(chunk_at<T>(smem + ((ch + 1) & 1) * cb, qs, RPC), in, tok0 + t0 - kChunk, kChunk, dqk, qs, dv, RPC, r0,
            nrows, vec_rows, true, spart, lnN, R, BHT);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const Chunk<T> b = chunk_at<T>(smem + (ch & 1) * cb, qs, RPC);
    widen<T, PADC, RPC>(sx, b, cnt, dqk, nrows, has_o);
    const float* qf = kWide ? reinterpret_cast<const float*>(b.q) : sx.qf;
    const float* kf = kWide ? reinterpret_cast<const float*>(b.k) : sx.kf;
    const float* vf = kWide ? reinterpret_cast<const float*>(b.v) : sx.vf;
    const float* dhf = kWide ? reinterpret_cast<const float*>(b.dh) : sx.dhf;
    if (warp == 0) {
      // lane p takes the p-th token in processing order, tt = cnt-1-p:
      // nu_t = max(log f_{t+1} + nu_{t+1}, -log N_t)
      const bool on = lane < cnt;
      const int tt = cnt - 1 - lane;
      const float lf_own = on ? (forget_exp ? b.fg[tt] : log_sigmoid(b.fg[tt])) : 0.0f;
      const float up = __shfl_up_sync(0xffffffffu, lf_own, 1);
      const float g = lane == 0 ? lf_carry : up;                  // log f of token t+1
      const float h = on ? -b.lnN[tt] : -INFINITY;
      float nprev;
      const float nu = maxplus_scan(on ? g : 0.0f, h, nu_carry, lane, &nprev);
      if (on) {
        float so = 0.0f;
        for (int r = 0; r < R; ++r) so += b.sp[r * kChunk + tt];
        sx.tsc[tt] = expf(g + nprev - nu);                        // alpha = f_{t+1} e^(nu_{t+1} - nu_t)
        sx.tsc[kChunk + tt] = expf(h - nu);                       // beta = e^-nu_t / N_t
        sx.tsc[2 * kChunk + tt] = expf(b.ig[tt] + nu);            // i_t e^nu_t
        sx.tsc[3 * kChunk + tt] = so;                             // h~.dh~ Omega of the head
      }
      nu_carry = __shfl_sync(0xffffffffu, nu, cnt - 1);
      lf_carry = __shfl_sync(0xffffffffu, lf_own, cnt - 1);
    }
    __syncthreads();
    for (int tt = cnt - 1; tt >= 0; --tt) {
      fold_scale(dc, dn, S, sx.tsc[tt]);
      const float bs = __fdividef(sx.tsc[kChunk + tt], S);
      float vr[kRW], dr[kRW];
      load_rows(vf + tt * RPC + wrow, vr);
      load_rows(dhf + tt * RPC + wrow, dr);
#pragma unroll
      for (int i = 0; i < kRW; ++i) dr[i] *= bs;
      const float cn = -bs * sx.tsc[3 * kChunk + tt];
      float dot[kRW];
#pragma unroll
      for (int i = 0; i < kRW; ++i) dot[i] = 0.0f;
      const float* qrow = qf + tt * PADC + 2 * lane;
      const float* krow = kf + tt * PADC + 2 * lane;
      float* colw = sx.col + (slot * NW + warp) * PADC + 2 * lane;
#pragma unroll
      for (int u = 0; u < NP; ++u) {
        const float2 kx = *reinterpret_cast<const float2*>(krow + 64 * u);
        const float2 qx = *reinterpret_cast<const float2*>(qrow + 64 * u);
        dn[2 * u] = fmaf(cn, qx.x, dn[2 * u]);                    // (61)
        dn[2 * u + 1] = fmaf(cn, qx.y, dn[2 * u + 1]);
        float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
        for (int i = 0; i < kRW; ++i) {
          dc[i][2 * u] = fmaf(dr[i], qx.x, dc[i][2 * u]);         // (60)
          dc[i][2 * u + 1] = fmaf(dr[i], qx.y, dc[i][2 * u + 1]);
          dot[i] = fmaf(dc[i][2 * u], kx.x, dot[i]);
          dot[i] = fmaf(dc[i][2 * u + 1], kx.y, dot[i]);
          s0 = fmaf(dc[i][2 * u], vr[i], s0);
          s1 = fmaf(dc[i][2 * u + 1], vr[i], s1);
        }
        *reinterpret_cast<float2*>(colw + 64 * u) = make_float2(s0, s1);
      }
      if (warp == 0) {
        float* vw = sx.vec + slot * PADC + 2 * lane;
#pragma unroll
        for (int u = 0; u < NP; ++u) *reinterpret_cast<float2*>(vw + 64 * u) = make_float2(dn[2 * u], dn[2 * u + 1]);
      }
      const float g = reduce_rows(dot, lane);
      if (writer) sx.gbuf[slot * RPC + wrow + myrow] = g;
      if (threadIdx.x == 0) {
        sx.sc[slot * 8 + 0] = scale * sx.tsc[2 * kChunk + tt] * S;    // s i_t e^nu_t S
        sx.tok[slot] = tt;
      }
      ++slot;
      if (slot == kGroup || tt == 0) {
        __syncthreads();
        for (int j = 0; j < slot; ++j) {
          const float f = sx.sc[j * 8 + 0];
          const size_t tokj = tok0 + t0 + sx.tok[j];
          const size_t orow = ((size_t)rank * BHT + tokj) * dqk;
          for (int cc = threadIdx.x; cc < dqk; cc += NW * 32) {
            float acc = rank == 0 ? sx.vec[j * PADC + cc] : 0.0f;
#pragma unroll
            for (int w = 0; w < NW; ++w) acc += sx.col[(j * NW + w) * PADC + cc];
            kpart[orow + cc] = f * acc;                                                      // (63)
          }
          for (int r = threadIdx.x; r < nrows; r += NW * 32)
            Elem<T>::store(dvout, tokj * dv + r0 + r, f * sx.gbuf[j * RPC + r]);            // (62)
        }
        __syncthreads();
        slot = 0;
      }
    }
    __syncthreads();
  }
}

// Sweep 3: one warp per token sums the R shares of dq and dk (four columns a
// lane at a time), writes them, d i~ = k.dk, and r = q.dq - k.dk.
template <typename T>
__device__ __forceinline__ float4 load4(const T* p);
template <>
__device__ __forceinline__ float4 load4<float>(const float* p) { return *reinterpret_cast<const float4*>(p); }
template <>
__device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

template <typename T>
__global__ void __launch_bounds__(256)
rbwd_combine_kernel(const T* __restrict__ q, const T* __restrict__ k, const float* __restrict__ qpart,
                    const float* __restrict__ kpart, T* __restrict__ dq, T* __restrict__ dk,
                    float* __restrict__ dig, float* __restrict__ rr, int dqk, int R, long long BHT) {
  const long long tok = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (tok >= BHT) return;
  float qd = 0.0f, kd = 0.0f;
  for (int c = 4 * lane; c < dqk; c += 128) {      // d_qk is a multiple of 8
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
    for (int r = 0; r < R; ++r) {
      const float4 x = *reinterpret_cast<const float4*>(qpart + ((size_t)r * BHT + tok) * dqk + c);
      const float4 y = *reinterpret_cast<const float4*>(kpart + ((size_t)r * BHT + tok) * dqk + c);
      a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
      b.x += y.x; b.y += y.y; b.z += y.z; b.w += y.w;
    }
    const size_t o = (size_t)tok * dqk + c;
    Elem<T>::store(dq, o, a.x); Elem<T>::store(dq, o + 1, a.y);
    Elem<T>::store(dq, o + 2, a.z); Elem<T>::store(dq, o + 3, a.w);
    Elem<T>::store(dk, o, b.x); Elem<T>::store(dk, o + 1, b.y);
    Elem<T>::store(dk, o + 2, b.z); Elem<T>::store(dk, o + 3, b.w);
    const float4 qv = load4<T>(q + o), kv = load4<T>(k + o);
    qd = fmaf(qv.x, a.x, fmaf(qv.y, a.y, fmaf(qv.z, a.z, fmaf(qv.w, a.w, qd))));
    kd = fmaf(kv.x, b.x, fmaf(kv.y, b.y, fmaf(kv.z, b.z, fmaf(kv.w, b.w, kd))));
  }
  qd = warp_sum(qd);
  kd = warp_sum(kd);
  if (lane == 0) {
    dig[tok] = kd;            // (69)
    rr[tok] = qd - kd;
  }
}

// Sweep 4: one CTA of 256 threads per head.  Each thread sums its run of
// consecutive tokens in fp64, the CTA scans the 256 run sums (suffix
// direction), and each thread then walks its run from the end.
constexpr int kScanThreads = 256;

__global__ void __launch_bounds__(kScanThreads)
rbwd_forget_kernel(const float* __restrict__ rr, const float* __restrict__ fg, float* __restrict__ dfg, int Tn,
                   int forget_exp) {
  __shared__ double part[kScanThreads];
  const size_t base = (size_t)blockIdx.x * Tn;
  const int tid = threadIdx.x;
  const int per = (Tn + kScanThreads - 1) / kScanThreads;
  const int lo = min(Tn, tid * per), hi = min(Tn, lo + per);
  double run = 0.0;
  for (int t = lo; t < hi; ++t) run += (double)rr[base + t];
  part[tid] = run;
  __syncthreads();
  // suffix scan over the run sums: after it, part[i] = sum of runs i..255
  for (int off = 1; off < kScanThreads; off <<= 1) {
    const double y = tid + off < kScanThreads ? part[tid + off] : 0.0;
    __syncthreads();
    part[tid] += y;
    __syncthreads();
  }
  double acc = tid + 1 < kScanThreads ? part[tid + 1] : 0.0;   // tokens after this run
  for (int t = hi - 1; t >= lo; --t) {
    acc += (double)rr[base + t];
    const float f = fg[base + t];
    const double act = forget_exp ? 1.0 : (double)sigmoid(-f);   // dlog f / df~ (eq 104)
    dfg[base + t] = (float)(acc * act);
  }
}

size_t r256(size_t x) { return (x + 255) & ~(size_t)255; }

// The workspace is sized for 64-row CTAs, the most CTAs per head any launch
// uses.
struct RbLayout {
  int R;
  size_t qpart, kpart, spart, lnN, rr, total;
};

RbLayout rb_layout(long long BHT, int dqk, int dv) {
  RbLayout L;
  L.R = (dv + 63) / 64;
  L.qpart = r256((size_t)L.R * BHT * dqk * sizeof(float));
  L.kpart = L.qpart;
  L.spart = r256((size_t)L.R * BHT * sizeof(float));
  L.lnN = r256((size_t)BHT * sizeof(float));
  L.rr = L.lnN;
  L.total = L.qpart + L.kpart + L.spart + L.lnN + L.rr;
  return L;
}

constexpr size_t kMaxSmem = 232448;

template <typename T, int NC, int NW>
size_t sweep_smem(int dqk) {
  constexpr bool wide = sizeof(T) == 4;
  return 2 * chunk_bytes<T>(wide ? 32 * NC : dqk, NW * kRW) + scratch_bytes(32 * NC, NW, wide);
}

template <typename T, int NC, int NW>
cudaError_t launch_sweeps(const Inputs& in, void* dog, void* dvout, float* qpart, float* kpart, float* spart,
                          float* lnN, int BH, int Tn, int dqk, int dv, float scale, int forget_exp,
                          cudaStream_t st) {
  const long long BHT = (long long)BH * Tn;
  const int R = (dv + NW * kRW - 1) / (NW * kRW);
  const size_t smem = sweep_smem<T, NC, NW>(dqk);
  if (smem > kMaxSmem) return cudaErrorInvalidValue;
  if (cudaFuncSetAttribute(rbwd_forward_kernel<T, NC, NW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess ||
      cudaFuncSetAttribute(rbwd_backward_kernel<T, NC, NW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return cudaErrorInvalidValue;
  const unsigned grid = (unsigned)(BH * R);
  rbwd_forward_kernel<T, NC, NW><<<grid, NW * 32, smem, st>>>(in, static_cast<T*>(dog), qpart, spart, lnN, Tn, dqk,
                                                              dv, R, scale, forget_exp, BHT);
  rbwd_backward_kernel<T, NC, NW><<<grid, NW * 32, smem, st>>>(in, spart, lnN, static_cast<T*>(dvout), kpart, Tn,
                                                               dqk, dv, R, scale, forget_exp, BHT);
  return cudaGetLastError();
}

// CTAs of 8 warps (64 rows) or 12 warps (96 rows), whichever finishes the
// heads sooner with one CTA per SM: waves of CTAs times rows per CTA.
template <typename T, int NC>
int pick_warps(int BH, int dqk, int dv) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms < 1) sms = 1;
  // 12 warps leave 168 registers a thread: enough for 8 x 12 state columns,
  // not for 8 x 16 (d_qk > 384)
  if (NC > 12 || sweep_smem<T, NC, 12>(dqk) > kMaxSmem) return 8;
  auto cost = [&](int nw) {
    const long long ctas = (long long)BH * ((dv + 8 * nw - 1) / (8 * nw));
    return ((ctas + sms - 1) / sms) * 8 * nw;
  };
  return cost(12) < cost(8) ? 12 : 8;
}

template <typename T, int NC>
cudaError_t launch_nc(int* nw, const Inputs& in, void* dog, void* dvout, float* qpart, float* kpart, float* spart,
                      float* lnN, int BH, int Tn, int dqk, int dv, float scale, int forget_exp, cudaStream_t st) {
  *nw = pick_warps<T, NC>(BH, dqk, dv);
  if constexpr (NC <= 12) {
    if (*nw == 12)
      return launch_sweeps<T, NC, 12>(in, dog, dvout, qpart, kpart, spart, lnN, BH, Tn, dqk, dv, scale, forget_exp,
                                      st);
  }
  return launch_sweeps<T, NC, 8>(in, dog, dvout, qpart, kpart, spart, lnN, BH, Tn, dqk, dv, scale, forget_exp, st);
}

template <typename T>
cudaError_t launch_all(const Inputs& in, void* dq, void* dk, void* dvout, float* dig, float* dfg, void* dog,
                       const RbLayout& L, char* ws, int BH, int Tn, int dqk, int dv, int forget_exp,
                       cudaStream_t st) {
  float* qpart = reinterpret_cast<float*>(ws);
  float* kpart = reinterpret_cast<float*>(ws + L.qpart);
  float* spart = reinterpret_cast<float*>(ws + L.qpart + L.kpart);
  float* lnN = reinterpret_cast<float*>(ws + L.qpart + L.kpart + L.spart);
  float* rr = reinterpret_cast<float*>(ws + L.qpart + L.kpart + L.spart + L.lnN);
  const float scale = (float)(1.0 / sqrt((double)dqk));
  const int nc = (dqk + 31) / 32;
  int nw = 8;
  cudaError_t e;
  if (nc <= 4)
    e = launch_nc<T, 4>(&nw, in, dog, dvout, qpart, kpart, spart, lnN, BH, Tn, dqk, dv, scale, forget_exp, st);
  else if (nc <= 8)
    e = launch_nc<T, 8>(&nw, in, dog, dvout, qpart, kpart, spart, lnN, BH, Tn, dqk, dv, scale, forget_exp, st);
  else if (nc <= 12)
    e = launch_nc<T, 12>(&nw, in, dog, dvout, qpart, kpart, spart, lnN, BH, Tn, dqk, dv, scale, forget_exp, st);
  else
    e = launch_nc<T, 16>(&nw, in, dog, dvout, qpart, kpart, spart, lnN, BH, Tn, dqk, dv, scale, forget_exp, st);
  if (e != cudaSuccess) return e;
  const long long BHT = (long long)BH * Tn;
  const int R = (dv + 8 * nw - 1) / (8 * nw);
  rbwd_combine_kernel<T><<<(unsigned)((BHT + 7) / 8), 256, 0, st>>>(
      static_cast<const T*>(in.q), static_cast<const T*>(in.k), qpart, kpart, static_cast<T*>(dq),
      static_cast<T*>(dk), dig, rr, dqk, R, BHT);
  rbwd_forget_kernel<<<(unsigned)BH, kScanThreads, 0, st>>>(rr, in.fg, dfg, Tn, forget_exp);
  return cudaGetLastError();
}

bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace
}  // namespace mlstm

using namespace mlstm;

extern "C" {

size_t mlstm_recurrent_bwd_workspace(int B, int H, int T, int d_qk, int d_v) {
  if (B <= 0 || H <= 0 || T <= 0 || d_qk <= 0 || d_v <= 0 || d_qk > 512 || d_v > 512) return 0;
  return rb_layout((long long)B * H * T, d_qk, d_v).total;
}

int mlstm_recurrent_bwd(const void* q, const void* k, const void* v, const float* igate_pre, const float* fgate_pre,
                        const void* dh, void* dq, void* dk, void* dv, float* d_igate, float* d_fgate, void* d_ogate,
                        int B, int H, int T, int d_qk, int d_v, int dtype, void* workspace, size_t workspace_bytes,
                        const mlstm_options* opt, void* stream) {
  if (B < 0 || H < 0 || T < 0) return MLSTM_EINVAL;
  if (d_qk < 1 || d_v < 1 || d_qk > 512 || d_v > 512 || d_qk % 8 != 0) return MLSTM_EINVAL;
  if (dtype != MLSTM_F32 && dtype != MLSTM_BF16) return MLSTM_EDTYPE;
  const long long BH = (long long)B * H;
  const long long BHT = BH * T;
  const long long R = (d_v + 63) / 64;
  if (BH * R > 0x7fffffffLL || BHT > (1LL << 40) || (BHT + 7) / 8 > 0x7fffffffLL) return MLSTM_EINVAL;
  if (BH == 0 || T == 0) return MLSTM_OK;
  const void* og = opt ? opt->ogate_pre : nullptr;
  if (!q || !k || !v || !igate_pre || !fgate_pre || !dh || !dq || !dk || !dv || !d_igate || !d_fgate)
    return MLSTM_EINVAL;
  if (og && !d_ogate) return MLSTM_EINVAL;
  if (!a16(q) || !a16(k)) return MLSTM_EALIGN;
  if (!workspace || workspace_bytes < mlstm_recurrent_bwd_workspace(B, H, T, d_qk, d_v)) return MLSTM_EWORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return MLSTM_EALIGN;
  const RbLayout L = rb_layout(BHT, d_qk, d_v);
  Inputs in{q, k, v, og, dh, igate_pre, fgate_pre};
  const int fe = opt ? opt->forget_exp : 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const cudaError_t e =
      dtype == MLSTM_F32
          ? launch_all<float>(in, dq, dk, dv, d_igate, d_fgate, d_ogate, L, ws, (int)BH, T, d_qk, d_v, fe, st)
          : launch_all<__nv_bfloat16>(in, dq, dk, dv, d_igate, d_fgate, d_ogate, L, ws, (int)BH, T, d_qk, d_v, fe,
                                      st);
  return e == cudaSuccess ? MLSTM_OK : MLSTM_ECUDA;
}

}  // extern "C"
