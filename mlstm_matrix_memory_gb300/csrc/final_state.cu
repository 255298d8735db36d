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
// Tensor-core version (bf16, d_qk and d_v multiples of 64): one CTA owns 128
// rows of C (d_v) and all d_qk columns, accumulated in TMEM over a range of
// tokens.  Per 64-token stage a TMA thread loads V [64 x 128] and K
// [64 x d_qk] (128-byte swizzle); eight warps (two per SM sub-partition, so
// that one hides the other's shared-memory latency) scale each V row by its
// token's weight s*D'_Tj in shared memory and sum their slice of the weighted
// K columns into n (the head's tile CTAs share the columns); one
// thread issues tcgen05.mma with both operands MN-major (M = d_v rows,
// N = d_qk columns, K = tokens).  CUDA-core version (fp32, other sizes): 64 x
// 64 tiles of C in registers, 32 weighted tokens staged at a time.  Both
// split the token range when there are too few tiles to fill the GPU and add
// the partial results into C and n (zeroed first).
#include <algorithm>
#include <cstdlib>

#include "internal.h"
#include "tc_ptx.cuh"

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


// ---------------------------------------------------------------- tensor cores
using namespace tc;
constexpr int kTcTok = 64, kTcM = 128, kTcThreads = 384;
constexpr int kTcScaleWarps = 8;            // warps 2..5 and 8..11: weights, n, epilogue
constexpr int kTcProducers = 3;             // warps 0, 6, 7: one issuing thread moves only ~30 B/clk
constexpr int kTcMaxStages = 4;
enum : int { kFsFull = 0, kFsScaled = kTcMaxStages, kFsEmpty = 2 * kTcMaxStages, kFsAcc = 3 * kTcMaxStages,
             kFsBars = 3 * kTcMaxStages + 1 };

struct FsTcParams {
  GateTerms g;
  float* C;
  float* n;
  float* m;
  int T, dqk, dv, ntr, ksplit, nst;
  uint32_t tmem_cols;
  float scale;
  DevStatus st;
};

__global__ void __launch_bounds__(kTcThreads, 1)
final_state_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                      const FsTcParams p) {
  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t bars[kFsBars];
  __shared__ uint32_t tmem_holder;
  __shared__ float w_s[kTcMaxStages][kTcTok];
  __shared__ int issued_s[kTcProducers];     // stages each producer has issued (settled after an abort)
  __shared__ int abort_flag;
  volatile int* abort = &abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per_head = p.ntr * p.ksplit;
  const int bh = blockIdx.x / per_head;
  const int tr = (blockIdx.x % per_head) / p.ksplit, split = blockIdx.x % p.ksplit;
  const int r0 = tr * kTcM;
  const int nchunk_all = (p.T + kTcTok - 1) / kTcTok;
  const int cps = (nchunk_all + p.ksplit - 1) / p.ksplit;        // chunks per split
  const int c0 = split * cps, c1 = min(nchunk_all, c0 + cps);
  const int nkb = p.dqk / 64;
  const uint32_t stage_bytes = 16384u + (uint32_t)nkb * 8192u;
  const uint32_t base = (smem_u32(dsmem) + 1023u) & ~1023u;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const size_t hb = (size_t)bh * p.T;
  const long long spin = p.st.spin_limit;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int q = 0; q < kTcProducers; ++q) issued_s[q] = 0;
    for (int s2 = 0; s2 < kTcMaxStages; ++s2) {
      mbar_init(bar(kFsFull + s2), 1);
      mbar_init(bar(kFsScaled + s2), kTcScaleWarps);
      mbar_init(bar(kFsEmpty + s2), 1);
    }
    mbar_init(bar(kFsAcc), 1);
    fence_barrier_init();
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_v);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_holder), p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_holder;

  if ((warp == 0 || warp == 6 || warp == 7) && lane == 0) {
    // ---- TMA producers: the stage's 2 + nkb boxes dealt round-robin; the
    // bytes of all of them are posted by warp 0
    const int pi = warp == 0 ? 0 : warp - 5;
    for (int c = c0, i = 0; c < c1; ++c, ++i) {
      const int s2 = i % p.nst;
      const uint32_t u = (uint32_t)(i / p.nst);
      if (!mbar_wait(bar(kFsEmpty + s2), (u & 1u) ^ 1u, spin, abort, p.st, 21)) break;
      const uint32_t dst = base + (uint32_t)s2 * stage_bytes;
      if (pi == 0) mbar_arrive_expect_tx(bar(kFsFull + s2), stage_bytes);
      for (int b = pi; b < 2 + nkb; b += kTcProducers) {
        if (b < 2) tma_load_3d(dst + b * 8192u, &tmap_v, bar(kFsFull + s2), r0 + 64 * b, c * kTcTok, bh);
        else tma_load_3d(dst + 16384u + (b - 2) * 8192u, &tmap_k, bar(kFsFull + s2), 64 * (b - 2), c * kTcTok, bh);
      }
      issued_s[pi] = i + 1;
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer: C[128 x d_qk] += (w V)^T K over the stage's 64 tokens
    bool ok = true, first = true;
    for (int c = c0, i = 0; c < c1 && ok; ++c, ++i) {
      const int s2 = i % p.nst;
      const uint32_t u = (uint32_t)(i / p.nst);
      ok = mbar_wait(bar(kFsScaled + s2), u & 1u, spin, abort, p.st, 22);
      if (!ok) break;
      tc_fence_after();
      const uint32_t sb = base + (uint32_t)s2 * stage_bytes;
      const uint64_t dA = smem_desc_sw128(sb, 8192, 1024);
      for (int nb = 0; nb < nkb; nb += 4) {
        const int nbox = min(4, nkb - nb);
        const uint32_t idesc = idesc_bf16_f32(kTcM, 64 * nbox, 1, 1);
        const uint64_t dB = smem_desc_sw128(sb + 16384u + (uint32_t)nb * 8192u, 8192, 1024);
#pragma unroll
        for (int kk = 0; kk < kTcTok / 16; ++kk)
          mma_bf16_ss(tmem + 64 * nb, dA + kk * 128, dB + kk * 128, idesc, (first && kk == 0) ? 0u : 1u);
      }
      first = false;
      mma_commit(bar(kFsEmpty + s2));
    }
    if (ok) mma_commit(bar(kFsAcc));
  } else if ((warp >= 2 && warp < 6) || warp >= 8) {
    // ---- weights, V scaling, n, then the epilogue (eight warps: each TMEM
    // lane quarter twice, one per half of the columns)
    const int t2 = warp < 6 ? threadIdx.x - 64 : threadIdx.x - 128;   // 0..255, a warp's lanes consecutive
    const float p2T = p.g.p2[hb + p.T - 1];
    // n = sum_j w_j k_j: the tile CTAs of a head share the columns (slice
    // [ncol0, ncol1), a multiple of 64).  A thread sums one 8-column chunk
    // over one group of tokens (16-byte loads); the groups of a chunk are
    // neighbouring lanes and meet by shuffles.
    const int cs = ((p.dqk / 64 + p.ntr - 1) / p.ntr) * 64;
    const int ncol0 = min(p.dqk, tr * cs), ncol1 = min(p.dqk, ncol0 + cs);
    const int nchk = (ncol1 - ncol0) / 8;                     // 8-column chunks in the slice (<= 64)
    int groups = 1;                                          // token groups per chunk: a power of 2 <= 16
    while (groups < 16 && 2 * groups * nchk <= 256) groups *= 2;
    const int chunk = t2 / groups, tg = t2 % groups;
    const bool n_thread = chunk < nchk;
    const int tpg = kTcTok / groups;                         // tokens per group
    float nacc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float a2_next = 0.0f;                                    // gate term two stages ahead
    auto load_a2 = [&](int c) {
      const int j = c * kTcTok + (t2 & 63);
      return (t2 < kTcTok && c < c1 && j < p.T) ? p.g.a2[hb + j] : -INFINITY;
    };
    auto weights = [&](float a2v, int s2) {
      if (t2 < kTcTok) w_s[s2][t2] = a2v == -INFINITY ? 0.0f : exp2f(a2v - p2T) * p.scale;
    };
    if (c0 < c1) weights(load_a2(c0), 0);
    a2_next = load_a2(c0 + 1);
    // The loop is the hot path of this kernel; its wait and exit are kept in
    // their plainest form (per-lane wait, early exit), which measured fastest:
    // a warp-level vote or a reducing barrier per stage cost 6-10 us of the
    // 49 us 125M-scale hand-off.  A warp that leaves early (its wait gave up,
    // raising the abort flag) then arrives on the barriers of the stages it
    // skipped, so every stage's barrier still counts all eight warps, and the
    // group agrees on the result once, after the loop.  The 32 lanes of a warp
    // poll the same barrier with the same instructions and take the same exit.
    bool ok = true;
    int done = 0;
    for (int c = c0, i = 0; c < c1 && ok; ++c, ++i) {
      const int s2 = i % p.nst;
      const uint32_t u = (uint32_t)(i / p.nst);
      ok = mbar_wait(bar(kFsFull + s2), u & 1u, spin, abort, p.st, 23);
      if (!ok) break;
      named_bar_sync(1, 256);                        // w_s[s2] written by every thread
      ++done;
      const uint32_t sb = base + (uint32_t)s2 * stage_bytes;
      {
        // V row (token) t2 % 64 of box (t2 / 64) % 2: four of its eight
        // 16-byte chunks (the half t2 / 128), taken in an order rotated by the
        // row so that neighbouring lanes (rows 128 bytes apart) hit different banks
        const int j = t2 & 63;
        const float w = w_s[s2][j];
        const uint32_t row = sb + (uint32_t)((t2 >> 6) & 1) * 8192u + (uint32_t)j * 128u;
#pragma unroll
        for (int q0 = 0; q0 < 4; ++q0) {
          const uint32_t q = (uint32_t)((4 * (t2 >> 7) + q0 + j) & 7);
          uint32_t x[4];
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]) : "r"(row + q * 16u));
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x[e]));
            x[e] = pack_bf16x2(f.x * w, f.y * w);
          }
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + q * 16u), "r"(x[0]), "r"(x[1]),
                       "r"(x[2]), "r"(x[3])
                       : "memory");
        }
      }
      if (n_thread) {
        const int col = ncol0 + chunk * 8;
        const uint32_t kb = sb + 16384u + (uint32_t)(col >> 6) * 8192u;
        const int cq = (col & 63) >> 3;
        for (int jj = 0; jj < tpg; ++jj) {
          const int j = jj * groups + tg;       // neighbouring lanes: neighbouring rows, distinct swizzled chunks
          uint32_t x[4];
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3])
                       : "r"(kb + (uint32_t)j * 128u + (uint32_t)((cq ^ (j & 7)) << 4)));
          const float w = w_s[s2][j];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x[e]));
            nacc[2 * e] = fmaf(w, f.x, nacc[2 * e]);
            nacc[2 * e + 1] = fmaf(w, f.y, nacc[2 * e + 1]);
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kFsScaled + s2));
      if (c + 1 < c1) {
        weights(a2_next, (i + 1) % p.nst);
        a2_next = load_a2(c + 2);
      }
    }
    for (int c = c0 + done; c < c1; ++c) named_bar_sync(1, 256);   // stages this warp skipped
    ok = bar_red_and(1, 256, ok);
    // the token groups of each chunk meet (neighbouring lanes)
#pragma unroll
    for (int e = 0; e < 8; ++e)
      for (int o = 1; o < groups; o <<= 1) nacc[e] += __shfl_xor_sync(0xffffffffu, nacc[e], o);
    // epilogue: row r0 + 32*(warp%4) + lane of C from TMEM, the column half
    // of this warp group
    if (ok && c1 > c0) ok = mbar_wait_warp(bar(kFsAcc), 0, spin, abort, p.st, 24);
    tc_fence_after();
    const int qd = warp & 3, hc = p.dqk / 2;
    const int r = r0 + 32 * qd + lane;
    if (ok && c1 > c0) {
      for (int cb = warp < 6 ? 0 : hc; cb < (warp < 6 ? hc : p.dqk); cb += 32) {
        uint32_t o[32];
        tmem_ld32(tmem + ((uint32_t)(32 * qd) << 16) + cb, o);
        tmem_wait_ld();
        if (r < p.dv) {
          float* dst = p.C + ((size_t)bh * p.dv + r) * p.dqk + cb;
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 val = make_float4(__uint_as_float(o[e]), __uint_as_float(o[e + 1]), __uint_as_float(o[e + 2]),
                                           __uint_as_float(o[e + 3]));
            if (p.ksplit > 1) atomicAdd(reinterpret_cast<float4*>(dst + e), val);
            else *reinterpret_cast<float4*>(dst + e) = val;
          }
        }
      }
      if (n_thread && tg == 0) {
        float* dst = p.n + (size_t)bh * p.dqk + ncol0 + chunk * 8;
        const float4 v0 = make_float4(nacc[0], nacc[1], nacc[2], nacc[3]);
        const float4 v1 = make_float4(nacc[4], nacc[5], nacc[6], nacc[7]);
        if (p.ksplit > 1) {
          atomicAdd(reinterpret_cast<float4*>(dst), v0);
          atomicAdd(reinterpret_cast<float4*>(dst + 4), v1);
        } else {
          *reinterpret_cast<float4*>(dst) = v0;
          *reinterpret_cast<float4*>(dst + 4) = v1;
        }
      }
    }
    if (tr == 0 && split == 0 && t2 == 0) p.m[bh] = p.g.m[hb + p.T - 1];
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 0 && lane == 0 && abort_flag) {
    // After an abort the producers may have stopped at different stages (they
    // are at most nst stages apart, as each waits for the stage nst back to be
    // consumed, so only the last nst stages can be partial): make each of those
    // phases complete when the boxes that were issued for it land, and wait.
    int f = 0;
    for (int q = 0; q < kTcProducers; ++q) f = max(f, issued_s[q]);
    for (int i = max(0, f - p.nst); i < f; ++i) {
      uint32_t land = 0;
      for (int q = 0; q < kTcProducers; ++q)
        if (issued_s[q] > i)
          for (int b = q; b < 2 + nkb; b += kTcProducers) land += 8192u;
      settle_last_phase(bar(kFsFull + i % p.nst), i / p.nst + 1, issued_s[0] > i, stage_bytes, land, 1LL << 22);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

}  // namespace

namespace {

cudaError_t launch_final_state_tc(const void* k, const void* v, GateTerms g, float* C, float* n, float* m, int BH,
                                  int T, int dqk, int dv, float scale, DevStatus st, int sms, cudaStream_t stream) {
  FsTcParams p;
  p.g = g; p.C = C; p.n = n; p.m = m; p.T = T; p.dqk = dqk; p.dv = dv; p.scale = scale; p.st = st;
  p.ntr = (dv + kTcM - 1) / kTcM;
  p.tmem_cols = 32;
  while ((int)p.tmem_cols < dqk) p.tmem_cols <<= 1;
  const size_t stage = 16384 + (size_t)(dqk / 64) * 8192;
  const int smem_limit = 232448 - 4096;                         // room for static shared memory
  p.nst = (int)std::min<size_t>(kTcMaxStages, (smem_limit - 1024) / stage);
  if (p.nst < 2) return cudaErrorInvalidValue;
  const size_t smem = 1024 + (size_t)p.nst * stage;
  const long long tiles = (long long)BH * p.ntr;
  const int nchunks = (T + kTcTok - 1) / kTcTok;
  // one wave: split the tokens only as far as whole waves of tiles fit on the
  // SMs (measured: the atomic adds of a split cost more than idle SMs), with
  // at least 4 stages per split
  int ksplit = (int)std::max<long long>(1, sms / tiles);
  ksplit = std::max(1, std::min(ksplit, nchunks / 4));
  if (const char* e = getenv("MLSTM_FS_KSPLIT")) ksplit = std::max(1, std::min(atoi(e), nchunks));  // tuning
  p.ksplit = ksplit;
  const long long grid = tiles * ksplit;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  CUtensorMap mk, mv;
  if (!make_map(&mk, k, dqk, T, BH, kTcTok) || !make_map(&mv, v, dv, T, BH, kTcTok)) return cudaErrorInvalidValue;
  if (ksplit > 1) {
    cudaError_t e = cudaMemsetAsync(C, 0, (size_t)BH * dv * dqk * sizeof(float), stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(n, 0, (size_t)BH * dqk * sizeof(float), stream);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = cudaFuncSetAttribute(final_state_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  final_state_tc_kernel<<<(unsigned)grid, kTcThreads, smem, stream>>>(mk, mv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_final_state(const void* k, const void* v, GateTerms g, float* C, float* n, float* m, int BH,
                               int T, int dqk, int dv, int dtype, float scale, DevStatus st, cudaStream_t stream) {
  if (BH <= 0 || T <= 0) return cudaSuccess;
  const int ntr = (dv + kTile - 1) / kTile, ntc = (dqk + kTile - 1) / kTile;
  const long long tiles = (long long)BH * ntr * ntc;
  int sms = 148, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (dtype == kBF16 && dqk % 64 == 0 && dv % 64 == 0 && device_is_sm100_family())
    return launch_final_state_tc(k, v, g, C, n, m, BH, T, dqk, dv, scale, st, sms, stream);
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
