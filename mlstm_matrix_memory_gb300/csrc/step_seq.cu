// L consecutive stabilized recurrent mLSTM steps per head in one pass
// (recurrent prefill, or several generated tokens at once).
//
// The recurrence differentiated by "xLSTM: Extended Long Short-Term Memory",
// part 28/30, eqs (59)-(70), with the output gate of part 17/30 eq (27); the
// same step as step.cu, applied for t = 0..L-1:
//   m' = max(log sigmoid(f~_t) + m, i~_t),  f' = exp(log sigmoid(f~_t) + m - m'),
//   i' = exp(i~_t - m'),  C <- f'C + i' v_t (s k_t)^T,  n <- f'n + i' s k_t,
//   h_t = sigmoid(o_t) * (C q_t) / max(|n.q_t|, exp(-m')),     s = 1/sqrt(d_qk).
//
// The state is read once and written once; in between each head's C lives in
// registers.  A cluster of R <= 8 CTAs owns one head: CTA r holds rows
// [64r, 64r+64) of C, eight rows per warp, each row spread over the 32 lanes
// (lane l holds columns l, l+32, ...).  Every warp keeps its own copy of n and
// m: per token a warp updates its rows and n, and reduces n.q and its rows'
// C q within the warp.  The token operands come through shared memory in
// chunks of 16 tokens, loaded by asynchronous copies one chunk ahead.  The
// cluster only makes every CTA read the initial n and m before CTA 0 writes
// the final ones.  Per token the work is 4 d_v d_qk flops per head on
// the CUDA cores (a rank-one update and a matrix-vector product).
#include "internal.h"

namespace mlstm {
namespace {

constexpr int kThreads = 256, kWarps = kThreads / 32;
constexpr int kRW = 8;                      // rows of C per warp
constexpr int kRowsPerCta = kWarps * kRW;   // 64

__device__ __forceinline__ unsigned cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

constexpr int kChunk = 16;                  // tokens staged in shared memory at a time

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

// One chunk of tokens in shared memory: q and k rows of all d_qk columns, v
// and o of this CTA's 64 rows, and the two gates.
template <typename T>
struct ChunkBuf {
  T* q;        // [kChunk][dqk]
  T* k;        // [kChunk][dqk]
  T* v;        // [kChunk][kRowsPerCta]
  T* o;        // [kChunk][kRowsPerCta]
  float* ig;   // [kChunk]
  float* fg;   // [kChunk]
};

template <typename T>
__device__ __forceinline__ ChunkBuf<T> chunk_buf(uint8_t* base, int dqk) {
  ChunkBuf<T> b;
  b.q = reinterpret_cast<T*>(base);
  b.k = b.q + kChunk * dqk;
  b.v = b.k + kChunk * dqk;
  b.o = b.v + kChunk * kRowsPerCta;
  b.ig = reinterpret_cast<float*>(b.o + kChunk * kRowsPerCta);
  b.fg = b.ig + kChunk;
  return b;
}

// Bytes of one chunk buffer (each array starts on a 16-byte boundary because
// d_qk is a multiple of 8 and kRowsPerCta of 8).
template <typename T>
__host__ __device__ constexpr size_t chunk_bytes(int dqk) {
  return (size_t)kChunk * (2 * dqk + 2 * kRowsPerCta) * sizeof(T) + 2 * kChunk * sizeof(float);
}

// Issues the copies of tokens [t0, t0+cnt) into `b` (all threads).  q, k and,
// when rows are 16-byte multiples, v and o go by 16-byte asynchronous copies;
// otherwise v and o are copied element by element.
template <typename T>
__device__ __forceinline__ void stage_chunk(const ChunkBuf<T>& b, const T* __restrict__ q, const T* __restrict__ k,
                                            const T* __restrict__ v, const T* __restrict__ o,
                                            const float* __restrict__ ig, const float* __restrict__ fg,
                                            size_t tok, int cnt, int dqk, int dv, int r0, int nrows, bool vec_rows) {
  constexpr int E = 16 / sizeof(T);                       // elements per 16-byte piece
  const int nq = cnt * dqk / E;
  for (int p = threadIdx.x; p < nq; p += kThreads) {
    cp_async16(b.q + p * E, q + tok * dqk + (size_t)p * E);
    cp_async16(b.k + p * E, k + tok * dqk + (size_t)p * E);
  }
  if (vec_rows) {
    const int per = nrows / E;                             // pieces per token row segment
    for (int p = threadIdx.x; p < cnt * per; p += kThreads) {
      const int t = p / per, e = (p % per) * E;
      cp_async16(b.v + t * kRowsPerCta + e, v + (tok + t) * dv + r0 + e);
      if (o) cp_async16(b.o + t * kRowsPerCta + e, o + (tok + t) * dv + r0 + e);
    }
  } else {
    for (int p = threadIdx.x; p < cnt * nrows; p += kThreads) {
      const int t = p / nrows, e = p % nrows;
      b.v[t * kRowsPerCta + e] = v[(tok + t) * dv + r0 + e];
      if (o) b.o[t * kRowsPerCta + e] = o[(tok + t) * dv + r0 + e];
    }
  }
  for (int t = threadIdx.x; t < cnt; t += kThreads) {
    cp_async4(b.ig + t, ig + tok + t);
    cp_async4(b.fg + t, fg + tok + t);
  }
}

// Two consecutive elements of a shared or global array as floats.
__device__ __forceinline__ float2 ld2(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ float2 ld2(const __nv_bfloat16* p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}

// Eight consecutive row values (16-byte aligned), the same for every lane.
__device__ __forceinline__ void load8(const float* p, float (&x)[kRW]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&x)[kRW]) {
  const uint4 a = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

// Inclusive max-plus scan over the lanes: x_t = max(g_t + x_{t-1}, h_t) from
// x_{-1} = x0, in closed form x_t = cs_t + max(x0, max_{j<=t}(h_j - cs_j))
// with cs the prefix sum of g.  Returns x_t; *xprev gets x_{t-1}.
__device__ __forceinline__ float maxplus_scan(float g, float h, float x0, int lane, float* xprev) {
  float cs = g;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, cs, off);
    if (lane >= off) cs += y;
  }
  float mx = h - cs;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, mx, off);
    if (lane >= off) mx = fmaxf(mx, y);
  }
  const float x = cs + fmaxf(x0, mx);
  const float up = __shfl_up_sync(0xffffffffu, x, 1);
  *xprev = lane == 0 ? x0 : up;
  return x;
}

constexpr float kRenorm = 1.0f / 16777216.0f;   // 2^-24

// NC = columns per lane (d_qk <= 32 * NC, NC even).  Lane l holds the column
// pairs (2l + 64u, 2l + 64u + 1), u < NC/2, so every load moves a pair.  Each
// warp keeps its rows of C and its copy of n as S * (C^, n^) with one scale
// S: the decay f' multiplies S alone and the rank-one term is one fused
// multiply-add per entry; S is folded back into the entries when it falls
// below 2^-24.  The chunk's f', i' and e^-m come from one warp (a max-plus
// scan of the stabilizer recurrence) before its tokens are processed.
template <typename T, int NC>
__global__ void __launch_bounds__(kThreads, 1)
step_seq_kernel(float* __restrict__ C, float* __restrict__ n, float* __restrict__ m,
                const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                const T* __restrict__ o, const float* __restrict__ ig, const float* __restrict__ fg,
                T* __restrict__ h, int L, int dqk, int dv, int R, float scale, int forget_exp) {
  constexpr int NP = NC / 2;
  extern __shared__ __align__(16) uint8_t smem[];
  const unsigned rank = cluster_rank();
  const int bh = (int)(blockIdx.x / R);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r0 = (int)rank * kRowsPerCta;                  // this CTA's first row
  const int nrows = max(0, min(kRowsPerCta, dv - r0));
  const int wrow = warp * kRW;                              // this warp's first row within the CTA
  const bool vec_rows = (dv * (int)sizeof(T)) % 16 == 0 && (nrows * (int)sizeof(T)) % 16 == 0 &&
                        (reinterpret_cast<uintptr_t>(v) & 15) == 0 && (reinterpret_cast<uintptr_t>(o) & 15) == 0;
  const size_t tok0 = (size_t)bh * L;
  const size_t cb = chunk_bytes<T>(dqk);
  float* tsc = reinterpret_cast<float*>(smem + 2 * cb);     // [3][kChunk]: f', i', e^-m of the chunk
  const int nchunks = (L + kChunk - 1) / kChunk;
  // after the in-warp reduction, lane l (l % 4 == 0) holds row `myrow` of the warp
  const int myrow = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
  const bool writer = (lane & 3) == 0 && wrow + myrow < nrows;

  stage_chunk(chunk_buf<T>(smem, dqk), q, k, v, o, ig, fg, tok0, min(kChunk, L), dqk, dv, r0, nrows, vec_rows);
  cp_async_commit();
  // rows of v and o that staging never writes (past this CTA's rows) stay zero
  for (int idx = threadIdx.x; idx < 2 * kChunk * (kRowsPerCta - nrows); idx += kThreads) {
    const int row = idx / (kRowsPerCta - nrows), r = nrows + idx - row * (kRowsPerCta - nrows);
    const ChunkBuf<T> cbuf = chunk_buf<T>(smem + (row / kChunk) * cb, dqk);
    Elem<T>::store(cbuf.v, (size_t)(row % kChunk) * kRowsPerCta + r, 0.0f);
  }

  float c[kRW][NC], nn[NC];
#pragma unroll
  for (int i = 0; i < kRW; ++i) {
    const int row = r0 + wrow + i;
#pragma unroll
    for (int u = 0; u < NP; ++u) {
      const int col = 2 * lane + 64 * u;
      const float2 x = (row < dv && col < dqk) ? ld2(C + ((size_t)bh * dv + row) * dqk + col) : make_float2(0.f, 0.f);
      c[i][2 * u] = x.x;
      c[i][2 * u + 1] = x.y;
    }
  }
#pragma unroll
  for (int u = 0; u < NP; ++u) {
    const int col = 2 * lane + 64 * u;
    const float2 x = col < dqk ? ld2(n + (size_t)bh * dqk + col) : make_float2(0.f, 0.f);
    nn[2 * u] = x.x;
    nn[2 * u + 1] = x.y;
  }
  float m_carry = m[bh];              // warp 0: m after the last processed chunk
  float S = 1.0f;
  cluster_sync();                     // every CTA of the head has read n and m

  for (int ch = 0; ch < nchunks; ++ch) {
    const int t0 = ch * kChunk, cnt = min(kChunk, L - t0);
    if (ch + 1 < nchunks) {
      stage_chunk(chunk_buf<T>(smem + ((ch + 1) & 1) * cb, dqk), q, k, v, o, ig, fg, tok0 + t0 + kChunk,
                  min(kChunk, L - t0 - kChunk), dqk, dv, r0, nrows, vec_rows);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();                  // chunk ch is in shared memory for every thread
    const ChunkBuf<T> b = chunk_buf<T>(smem + (ch & 1) * cb, dqk);
    if (warp == 0) {
      // m_t = max(log f_t + m_{t-1}, i~_t) over the chunk
      const bool on = lane < cnt;
      const float lf = on ? (forget_exp ? b.fg[lane] : log_sigmoid(b.fg[lane])) : 0.0f;
      const float igv = on ? b.ig[lane] : -INFINITY;
      float mprev;
      const float mt = maxplus_scan(lf, igv, m_carry, lane, &mprev);
      if (on) {
        tsc[lane] = expf(lf + mprev - mt);                 // f'
        tsc[kChunk + lane] = expf(igv - mt);               // i'
        tsc[2 * kChunk + lane] = expf(-mt);                // normalizer floor
      }
      m_carry = __shfl_sync(0xffffffffu, mt, cnt - 1);
    }
    __syncthreads();
    for (int tt = 0; tt < cnt; ++tt) {
      const float s2 = S * tsc[tt];
      if (s2 < kRenorm) {             // fold the scale into the entries
#pragma unroll
        for (int i = 0; i < kRW; ++i)
#pragma unroll
          for (int u = 0; u < NC; ++u) c[i][u] *= s2;
#pragma unroll
        for (int u = 0; u < NC; ++u) nn[u] *= s2;
        S = 1.0f;
      } else {
        S = s2;
      }
      const float a = __fdividef(tsc[kChunk + tt] * scale, S);   // k's coefficient in the scaled update
      float vr[kRW];
      load8(b.v + (size_t)tt * kRowsPerCta + wrow, vr);
      float dot[kRW];
#pragma unroll
      for (int i = 0; i < kRW; ++i) dot[i] = 0.0f;
      float nq = 0.0f;
#pragma unroll
      for (int u = 0; u < NP; ++u) {
        const int col = 2 * lane + 64 * u;
        const float2 kx = col < dqk ? ld2(b.k + (size_t)tt * dqk + col) : make_float2(0.f, 0.f);
        const float2 qx = col < dqk ? ld2(b.q + (size_t)tt * dqk + col) : make_float2(0.f, 0.f);
        const float k0 = kx.x * a, k1 = kx.y * a;
        nn[2 * u] += k0;
        nn[2 * u + 1] += k1;
        nq = fmaf(nn[2 * u], qx.x, nq);
        nq = fmaf(nn[2 * u + 1], qx.y, nq);
#pragma unroll
        for (int i = 0; i < kRW; ++i) {
          c[i][2 * u] = fmaf(vr[i], k0, c[i][2 * u]);
          c[i][2 * u + 1] = fmaf(vr[i], k1, c[i][2 * u + 1]);
          dot[i] = fmaf(c[i][2 * u], qx.x, dot[i]);
          dot[i] = fmaf(c[i][2 * u + 1], qx.y, dot[i]);
        }
      }
      nq = warp_sum(nq);
      // reduce the eight row sums across the warp in halving steps: after the
      // xor-16, -8 and -4 exchanges each lane holds one row's partial sum
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
      if (writer) {
        const float nrm = fmaxf(fabsf(nq * S), tsc[2 * kChunk + tt]);
        float hv = nrm > 0.0f ? g * S / nrm : 0.0f;
        if (o) hv *= sigmoid(Elem<T>::load(b.o, (size_t)tt * kRowsPerCta + wrow + myrow));
        Elem<T>::store(h, (tok0 + t0 + tt) * dv + r0 + wrow + myrow, hv);
      }
    }
    __syncthreads();                  // buffer ch&1 may be refilled by the next stage
  }

#pragma unroll
  for (int i = 0; i < kRW; ++i) {
    const int row = r0 + wrow + i;
#pragma unroll
    for (int u = 0; u < NP; ++u) {
      const int col = 2 * lane + 64 * u;
      if (row < dv && col < dqk)
        *reinterpret_cast<float2*>(C + ((size_t)bh * dv + row) * dqk + col) =
            make_float2(c[i][2 * u] * S, c[i][2 * u + 1] * S);
    }
  }
  if (rank == 0 && warp == 0) {
#pragma unroll
    for (int u = 0; u < NP; ++u) {
      const int col = 2 * lane + 64 * u;
      if (col < dqk)
        *reinterpret_cast<float2*>(n + (size_t)bh * dqk + col) = make_float2(nn[2 * u] * S, nn[2 * u + 1] * S);
    }
    if (lane == 0) m[bh] = m_carry;
  }
}

template <typename T, int NC>
cudaError_t launch_nc(const StepArgs& a, int L, int R, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.BH * R));
  cfg.blockDim = dim3(kThreads);
  const size_t smem = 2 * chunk_bytes<T>(a.dqk) + 3 * kChunk * sizeof(float);
  if (cudaFuncSetAttribute(step_seq_kernel<T, NC>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return cudaErrorInvalidValue;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)R;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, step_seq_kernel<T, NC>, a.C, a.n, a.m, (const T*)a.q, (const T*)a.k,
                            (const T*)a.v, (const T*)a.o, a.ig, a.fg, (T*)a.h, L, a.dqk, a.dv, R, a.scale,
                            a.forget_exp);
}

template <typename T>
cudaError_t launch_t(const StepArgs& a, int L, int R, cudaStream_t stream) {
  const int nc = (a.dqk + 31) / 32;
  if (nc <= 4) return launch_nc<T, 4>(a, L, R, stream);
  if (nc <= 8) return launch_nc<T, 8>(a, L, R, stream);
  if (nc <= 12) return launch_nc<T, 12>(a, L, R, stream);
  return launch_nc<T, 16>(a, L, R, stream);
}

}  // namespace

cudaError_t launch_step_seq(const StepArgs& a, int L, cudaStream_t stream) {
  if (a.BH <= 0 || L <= 0) return cudaSuccess;
  if (a.dqk > 512 || a.dv > 512) return cudaErrorInvalidValue;
  // one token: the single-step kernel (same layouts, no state kept on chip)
  if (L == 1) return launch_step(a, stream);
  const int R = (a.dv + kRowsPerCta - 1) / kRowsPerCta;   // <= 8
  if ((long long)a.BH * R > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaError_t e = a.dtype == kF32 ? launch_t<float>(a, L, R, stream) : launch_t<__nv_bfloat16>(a, L, R, stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mlstm
