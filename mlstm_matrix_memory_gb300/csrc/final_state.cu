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
// Tensor-core version (bf16, d_qk and d_v multiples of 64): a CTA owns 128
// rows of C (one row tile of a head) and all d_qk columns, accumulated in TMEM
// over 64-token chunks.  The CTAs form one group per row tile; the groups walk
// the same sequence of (head, chunk) units side by side, each CTA a contiguous
// range of it (whole heads when they spread evenly over the SMs, else an even
// share of units, so that every SM has work).  Per unit, TMA threads load V
// [64 x 128] and K [64 x d_qk] (128-byte swizzle); eight V warps (two per SM
// sub-partition) scale each V row by its token's weight s*D'_Tj into the
// MMA's A operand (in TMEM, or in place in shared memory at d_qk = 512); four
// n warps sum their slice of the weighted K columns into n (the row tiles of
// a head share the columns) and two of them prepare the next unit's weights;
// one thread issues tcgen05.mma (M = d_v rows, N = d_qk columns, K = tokens).
// At the end of each piece (the part of a head a CTA holds) the V warps move C
// out of TMEM through 128 x 32 boxes in shared memory to TMA stores (a whole
// head) or TMA adds (a head cut between CTAs, into C and n zeroed by a pass
// launched just before).
// CUDA-core version (fp32, other sizes): 64 x 64 tiles of C in registers, 32
// weighted tokens staged at a time, the token range split when there are too
// few tiles to fill the GPU and the partial results added into C and n
// (zeroed first).
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
constexpr int kTcTok = 64, kTcM = 128, kTcThreads = 512;
constexpr int kSmemLimit = 232448;         // opt-in shared memory per block on sm_100-family
constexpr int kTcScaleWarps = 8;            // warps 2..5 and 8..11: weighted V, C epilogue
constexpr int kTcNWarps = 4;                // warps 12..15: n (and, 12..13, the weights)
constexpr int kTcProducers = 3;             // warps 0, 6, 7: one issuing thread moves only ~30 B/clk
constexpr int kTcMaxStages = 4;
constexpr uint32_t kCBoxBytes = 16384;      // one 128 x 32 fp32 box of C (128-byte swizzle)
constexpr uint32_t kStagingBytes = 2 * kCBoxBytes;
enum : int { kFsFull = 0, kFsScaled = kTcMaxStages, kFsEmpty = 2 * kTcMaxStages, kFsAccFull = 3 * kTcMaxStages,
             kFsAccEmpty = 3 * kTcMaxStages + 1, kFsDrain = 3 * kTcMaxStages + 2, kFsBars = 3 * kTcMaxStages + 3 };

struct FsTcParams {
  GateTerms g;
  float* n;
  float* m;
  long long ug;               // units of a row tile's group: heads x chunks (chunk = 64 tokens)
  int T, dqk, dv, ntr, nchunk, nst;
  int gt;                     // CTAs per group; the grid is gt x ntr
  int whole;                  // 1: each CTA takes whole heads
  uint32_t acol;              // first TMEM column of the A slots (AT)
  int kbox;                   // K's 64-column blocks per TMA box (divides d_qk / 64)
  int split;                  // 1: some tile is shared by CTAs; C and n were zeroed and are added into
  uint32_t tmem_cols;
  float scale;
  DevStatus st;
};

// The CTAs form one group per 128-row tile of C (tr = blockIdx % ntr); the
// groups walk the same (head, chunk) sequence side by side, so that the row
// tiles of a head read each K chunk at about the same time (from L2 after the
// first).  CTA k of a group takes a contiguous range of that sequence,
// rounded to whole heads when p.whole.
__device__ __forceinline__ void unit_range(const FsTcParams& p, long long& va, long long& vb) {
  const long long k = blockIdx.x / p.ntr;
  if (p.whole) {
    const long long heads = p.ug / p.nchunk;
    va = k * heads / p.gt * p.nchunk;
    vb = (k + 1) * heads / p.gt * p.nchunk;
  } else {
    va = k * p.ug / p.gt;
    vb = (k + 1) * p.ug / p.gt;
  }
}

// Next unit of the sequence.
__device__ __forceinline__ void next_unit(int& bh, int& c, int nchunk) {
  if (++c == nchunk) {
    c = 0;
    ++bh;
  }
}

// The units of a CTA form pieces: maximal runs inside one head.  A piece is
// accumulated in TMEM over its chunks, then written out (the whole head: a
// store; part of it: an add into C, which the zero pass cleared).
// AT: the weighted V^T (the MMA's A operand) goes to TMEM columns beside the
// accumulator (one 32-column slot per stage) instead of back to shared memory,
// which takes the A reads of every MMA and the write-back of V off the shared
// memory port (d_qk + 32 nst <= 512).
template <bool AT>
__global__ void __launch_bounds__(kTcThreads, 1)
final_state_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                      const __grid_constant__ CUtensorMap tmap_c, const FsTcParams p) {
  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t bars[kFsBars];
  __shared__ uint32_t tmem_holder;
  __shared__ __align__(16) float w_s[kTcMaxStages][kTcTok];
  __shared__ int issued_s[kTcProducers];     // stages each producer has issued (settled after an abort)
  __shared__ int abort_flag;
  volatile int* abort = &abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tr = blockIdx.x % p.ntr, r0 = tr * kTcM;
  long long va, vb;
  unit_range(p, va, vb);
  const int nu = (int)(vb - va);
  const int bh0 = (int)(va / p.nchunk), cc0 = (int)(va % p.nchunk);   // first unit
  const int nkb = p.dqk / 64;
  const uint32_t stage_bytes = 16384u + (uint32_t)nkb * 8192u;
  const uint32_t base = (smem_u32(dsmem) + 1023u) & ~1023u;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const long long spin = p.st.spin_limit;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int q = 0; q < kTcProducers; ++q) issued_s[q] = 0;
    for (int s2 = 0; s2 < kTcMaxStages; ++s2) {
      mbar_init(bar(kFsFull + s2), 1);
      mbar_init(bar(kFsScaled + s2), kTcScaleWarps);
      mbar_init(bar(kFsEmpty + s2), 1 + kTcNWarps);   // the MMA commit and the n warps' reads of K
    }
    mbar_init(bar(kFsAccFull), 1);
    mbar_init(bar(kFsAccEmpty), kTcScaleWarps);
    mbar_init(bar(kFsDrain), 1);
    fence_barrier_init();
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_v);
    tma_prefetch_desc(&tmap_c);
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
    // ---- TMA producers: the stage's boxes (V's two 64-row blocks in one, K's
    // nkb 64-column blocks in nkb / kbox) dealt round-robin; the bytes of all
    // of them are posted by warp 0.  One issuing thread moves about one box
    // per ~600 cycles whatever its size, so few large boxes on three threads
    // land a stage sooner than many small ones.
    const int pi = warp == 0 ? 0 : warp - 5;
    int bh = bh0, c = cc0;
    for (int i = 0; i < nu; ++i, next_unit(bh, c, p.nchunk)) {
      const int s2 = i % p.nst;
      const uint32_t u = (uint32_t)(i / p.nst);
      if (!mbar_wait(bar(kFsEmpty + s2), (u & 1u) ^ 1u, spin, abort, p.st, 21)) break;
      const uint32_t dst = base + (uint32_t)s2 * stage_bytes;
      if (pi == 0) mbar_arrive_expect_tx(bar(kFsFull + s2), stage_bytes);
      for (int b = pi; b < 1 + nkb / p.kbox; b += kTcProducers) {
        if (b == 0) tma_load_4d(dst, &tmap_v, bar(kFsFull + s2), 0, c * kTcTok, r0 / 64, bh);
        else
          tma_load_4d(dst + 16384u + (uint32_t)((b - 1) * p.kbox) * 8192u, &tmap_k, bar(kFsFull + s2), 0, c * kTcTok,
                      (b - 1) * p.kbox, bh);
      }
      issued_s[pi] = i + 1;
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer: C[128 x d_qk] += (w V)^T K over the stage's 64 tokens;
    // a piece's first MMAs overwrite the accumulator once the previous
    // piece's epilogue has read it
    bool ok = true;
    int piece = 0, bh = bh0, c = cc0;
    for (int i = 0; i < nu && ok; ++i, next_unit(bh, c, p.nchunk)) {
      const int s2 = i % p.nst;
      const uint32_t u = (uint32_t)(i / p.nst);
      const bool pstart = i == 0 || c == 0, pend = i == nu - 1 || c == p.nchunk - 1;
      ok = mbar_wait(bar(kFsScaled + s2), u & 1u, spin, abort, p.st, 22);
      if (!ok) break;
      if (pstart && piece > 0) {
        ok = mbar_wait(bar(kFsAccEmpty), (uint32_t)(piece - 1) & 1u, spin, abort, p.st, 25);
        if (!ok) break;
      }
      tc_fence_after();
      const uint32_t sb = base + (uint32_t)s2 * stage_bytes;
      const uint64_t dA = smem_desc_sw128(sb, 8192, 1024);
      const uint32_t aT = tmem + p.acol + 32u * (uint32_t)s2;
      for (int nb = 0; nb < nkb; nb += 4) {
        const int nbox = min(4, nkb - nb);
        const uint32_t idesc = idesc_bf16_f32(kTcM, 64 * nbox, AT ? 0 : 1, 1);
        const uint64_t dB = smem_desc_sw128(sb + 16384u + (uint32_t)nb * 8192u, 8192, 1024);
#pragma unroll
        for (int kk = 0; kk < kTcTok / 16; ++kk) {
          if (AT) mma_bf16_ts(tmem + 64 * nb, aT + 8u * kk, dB + kk * 128, idesc, (pstart && kk == 0) ? 0u : 1u);
          else mma_bf16_ss(tmem + 64 * nb, dA + kk * 128, dB + kk * 128, idesc, (pstart && kk == 0) ? 0u : 1u);
        }
      }
      mma_commit(bar(kFsEmpty + s2));
      if (pend) {
        mma_commit(bar(kFsAccFull));
        ++piece;
      }
    }
    // every MMA this thread issued has finished before the CTA frees TMEM and
    // its stages (on an abort nobody else waits for the last ones)
    // (a bounded wait that does not give up on the abort flag)
    mma_commit(bar(kFsDrain));
    for (long long it = 0; it < (1LL << 22) && !mbar_try_wait(bar(kFsDrain), 0); ++it) {
    }
  } else if (warp >= 2 && warp != 6 && warp != 7) {
    // ---- twelve warps share the stage loop:
    //  - V warps (2..5, 8..11): the weighted V and each piece's C epilogue,
    //    each TMEM lane quarter twice (one per token half, then per half of
    //    the columns);
    //  - n warps (12..15): n over their slice of K, and (12, 13) the next
    //    unit's weights.
    // No warp does two of these per unit: the stage barrier waits for the
    // slowest, and two weighting warps per sub-partition hid too little
    // latency.
    const bool vw = warp < 12;
    const int t2 = vw ? (warp < 6 ? threadIdx.x - 64 : threadIdx.x - 128) : -1;   // V warps: 0..255
    const int tn = vw ? -1 : threadIdx.x - 384;                                   // n warps: 0..127
    const int qd = warp & 3;
    // n = sum_j w_j k_j: the row tiles of a head share the columns (slice
    // [ncol0, ncol0 + 8 nchk) of row tile tr, a multiple of 64).  A thread sums
    // one 8-column chunk over one group of tokens (16-byte loads); the groups
    // of a chunk are neighbouring lanes and meet by shuffles.
    const int cs = ((p.dqk / 64 + p.ntr - 1) / p.ntr) * 64;
    const int ncol0 = min(p.dqk, tr * cs);
    const int nchk = (min(p.dqk, ncol0 + cs) - ncol0) / 8;  // 8-column chunks in the slice (<= 64)
    int groups = 1;                                        // token groups per chunk: a power of 2 <= 16
    while (groups < 16 && 2 * groups * nchk <= 128) groups *= 2;   // the 128 n threads cover every chunk
    const int chunk = max(tn, 0) / groups, tg = max(tn, 0) % groups;
    const bool n_thread = tn >= 0 && chunk < nchk;
    const int tpg = kTcTok / groups;                       // tokens per group: 4..64, a multiple of 4
    float nacc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    // Gate terms of token tk = tn of a unit (warps 12 and 13): a2_j and p2_T
    // (the row of the head's last token), weight exp2(a2_j - p2_T) s.  Unit u's are fetched four
    // units before their use into register pair u % 4 (a switch picks the
    // pair, so no register holding a load in flight is ever copied, which
    // would wait for it), so that a load from DRAM (microseconds under load)
    // never holds up the stage loop.
    constexpr int kAhead = 4;
    const int tk = tn;
    const bool gate_thread = tk >= 0 && tk < kTcTok;
    auto load_gate = [&](int bh, int c, bool valid, float& a, float& q) {
      const int j = c * kTcTok + tk;
      const size_t hb = (size_t)bh * p.T;
      const bool v = valid && gate_thread && j < p.T;
      a = v ? p.g.a2[hb + j] : -INFINITY;
      q = v ? p.g.p2[hb + p.T - 1] : 0.0f;
    };
    auto weights = [&](float a, float q, int s2) {
      if (gate_thread) w_s[s2][tk] = a == -INFINITY ? 0.0f : exp2f(a - q) * p.scale;
    };
    int bh2 = bh0, c2 = cc0;                       // the unit kAhead + 1 ahead of the loop
    float ga0, gq0, ga1, gq1, ga2, gq2, ga3, gq3;  // gate terms of unit u in pair u % 4
    {
      float a, q;
      load_gate(bh2, c2, nu > 0, a, q);
      if (nu > 0) weights(a, q, 0);
    }
    next_unit(bh2, c2, p.nchunk);
    load_gate(bh2, c2, 1 < nu, ga1, gq1);
    next_unit(bh2, c2, p.nchunk);
    load_gate(bh2, c2, 2 < nu, ga2, gq2);
    next_unit(bh2, c2, p.nchunk);
    load_gate(bh2, c2, 3 < nu, ga3, gq3);
    next_unit(bh2, c2, p.nchunk);
    load_gate(bh2, c2, 4 < nu, ga0, gq0);
    next_unit(bh2, c2, p.nchunk);
    bool waited_zero = false;
    // The stage loop's wait and exit are kept in their plainest form (per-lane
    // wait, early exit), which measured fastest: a warp-level vote or a
    // reducing barrier per stage cost 6-10 us of the 49 us 125M-scale
    // hand-off.  A warp that leaves early (its wait gave up, raising the abort
    // flag) then arrives on the barriers of the stages it skipped, so every
    // stage's barrier still counts all twelve warps, and the group agrees on
    // the result once, after the loop.  The 32 lanes of a warp poll the same
    // barrier with the same instructions and take the same exit.
    bool ok = true;
    int done = 0, piece = 0, pc0 = 0, bh = bh0, c = cc0;
    for (int i = 0; i < nu && ok; ++i, next_unit(bh, c, p.nchunk)) {
      const int s2 = i % p.nst;
      const uint32_t u = (uint32_t)(i / p.nst);
      const bool pstart = i == 0 || c == 0, pend = i == nu - 1 || c == p.nchunk - 1;
      if (pstart) {
        pc0 = c;
        if (tr == 0 && c == 0 && t2 == 0) p.m[bh] = p.g.m[(size_t)bh * p.T + p.T - 1];
      }
      ok = mbar_wait(bar(kFsFull + s2), u & 1u, spin, abort, p.st, 23);
      if (!ok) break;
      named_bar_sync(1, 384);                        // w_s[s2] written
      ++done;
      const uint32_t sb = base + (uint32_t)s2 * stage_bytes;
      if (!vw) {
        // (n warps: below)
      } else if (AT) {
        // A = (w V)^T into TMEM slot s2: this warp's lane quarter (d_v rows
        // 32 qd ..) and token half (32 th ..), as 2 x 2 blocks of 16 rows x 16
        // tokens.  ldmatrix.trans turns 8 x 8 blocks of the token-major V
        // stage into (row, token pair) elements in the mma fragment layout,
        // which the 16x256b store takes as is: register 0 (1) of a thread holds
        // tokens 4 (t % 4) + 0, 1 (+ 2, 3) of a block, i.e. TMEM columns
        // 2 (t % 4) and 2 (t % 4) + 1; matrices 2 and 3 the rows 8 further on.
        const int th = warp < 6 ? 0 : 1;
        uint32_t x[4][4];
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
          const int m0 = 32 * qd + 16 * (blk >> 1), k0 = 32 * th + 16 * (blk & 1);
          const int mi = lane >> 3, mj = lane & 7;
          const int k = k0 + 4 * (mj >> 1) + (mj & 1) + 2 * (mi & 1), m = m0 + 8 * (mi >> 1);
          ldmatrix_x4_trans(sb + (uint32_t)(m >> 6) * 8192u + (uint32_t)k * 128u +
                                (uint32_t)((((m & 63) >> 3) ^ (k & 7)) << 4),
                            x[blk]);
        }
        // the two token blocks' weights, loaded before the first TMEM store
        // (an asm statement that the compiler does not move loads across)
        const float4 wb0 = *reinterpret_cast<const float4*>(&w_s[s2][32 * th + 4 * (lane & 3)]);
        const float4 wb1 = *reinterpret_cast<const float4*>(&w_s[s2][32 * th + 16 + 4 * (lane & 3)]);
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
          const int m0 = 32 * qd + 16 * (blk >> 1), k0 = 32 * th + 16 * (blk & 1);
          const float4 w = (blk & 1) ? wb1 : wb0;
          uint32_t y[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x[blk][e]));
            y[e] = (e & 1) ? pack_bf16x2(f.x * w.z, f.y * w.w) : pack_bf16x2(f.x * w.x, f.y * w.y);
          }
          tmem_st16x256b(tmem + ((uint32_t)m0 << 16) + p.acol + 32u * (uint32_t)s2 + (uint32_t)(k0 >> 1), y[0], y[1],
                         y[2], y[3]);
        }
      } else {
        // V row (token) t2 % 64 of box (t2 / 64) % 2: four of its eight
        // 16-byte chunks (the half t2 / 128), taken in an order rotated by the
        // row so that neighbouring lanes (rows 128 bytes apart) hit different
        // banks; all four loads are issued before the first store
        const int j = t2 & 63;
        const float w = w_s[s2][j];
        const uint32_t row = sb + (uint32_t)((t2 >> 6) & 1) * 8192u + (uint32_t)j * 128u;
        uint32_t x[4][4];
#pragma unroll
        for (int q0 = 0; q0 < 4; ++q0) {
          const uint32_t q = (uint32_t)((4 * (t2 >> 7) + q0 + j) & 7);
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(x[q0][0]), "=r"(x[q0][1]), "=r"(x[q0][2]), "=r"(x[q0][3]) : "r"(row + q * 16u));
        }
#pragma unroll
        for (int q0 = 0; q0 < 4; ++q0) {
          const uint32_t q = (uint32_t)((4 * (t2 >> 7) + q0 + j) & 7);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x[q0][e]));
            x[q0][e] = pack_bf16x2(f.x * w, f.y * w);
          }
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + q * 16u), "r"(x[q0][0]),
                       "r"(x[q0][1]), "r"(x[q0][2]), "r"(x[q0][3])
                       : "memory");
        }
      }
      if (n_thread) {
        const int col = ncol0 + chunk * 8;
        const uint32_t kb = sb + 16384u + (uint32_t)(col >> 6) * 8192u;
        const int cq = (col & 63) >> 3;
        for (int jj = 0; jj < tpg; jj += 4) {
          // four tokens' loads in flight at once; neighbouring lanes take
          // neighbouring rows (distinct swizzled chunks)
          uint32_t x[4][4];
          float w[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int j = (jj + r) * groups + tg;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(x[r][0]), "=r"(x[r][1]), "=r"(x[r][2]), "=r"(x[r][3])
                         : "r"(kb + (uint32_t)j * 128u + (uint32_t)((cq ^ (j & 7)) << 4)));
            w[r] = w_s[s2][j];
          }
#pragma unroll
          for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x[r][e]));
              nacc[2 * e] = fmaf(w[r], f.x, nacc[2 * e]);
              nacc[2 * e + 1] = fmaf(w[r], f.y, nacc[2 * e + 1]);
            }
        }
      }
      if (!vw) {
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kFsEmpty + s2));   // this warp has read the stage's K
      } else {
        if (AT) {
          tmem_wait_st();                            // this thread's A stores are in TMEM
          tc_fence_before();
        } else {
          fence_proxy_async_smem();                  // the scaled V is visible to the tensor core
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kFsScaled + s2));
      }
      if (gate_thread && i + 1 < nu) {
        // unit i + 1's weights, then unit i + 1 + kAhead's gate terms into the same pair
        const bool more = i + 1 + kAhead < nu;
        switch ((i + 1) & 3) {
          case 0: weights(ga0, gq0, (i + 1) % p.nst); load_gate(bh2, c2, more, ga0, gq0); break;
          case 1: weights(ga1, gq1, (i + 1) % p.nst); load_gate(bh2, c2, more, ga1, gq1); break;
          case 2: weights(ga2, gq2, (i + 1) % p.nst); load_gate(bh2, c2, more, ga2, gq2); break;
          default: weights(ga3, gq3, (i + 1) % p.nst); load_gate(bh2, c2, more, ga3, gq3); break;
        }
        next_unit(bh2, c2, p.nchunk);
      }
      if (!pend) continue;
      // ---- the piece's epilogue: n, then C rows r0 + 32*qd + lane from
      // TMEM, this warp's half of the columns
      const bool whole_tile = pc0 == 0 && c == p.nchunk - 1;   // no other CTA adds into this tile
      if (p.split && !waited_zero) {
        asm volatile("griddepcontrol.wait;" ::: "memory");   // C and n zeroed by the preceding pass
        fence_proxy_async_global();
        waited_zero = true;
      }
      if (!vw)
#pragma unroll
        for (int e = 0; e < 8; ++e)
          for (int o = 1; o < groups; o <<= 1) nacc[e] += __shfl_xor_sync(0xffffffffu, nacc[e], o);
      if (n_thread && tg == 0) {
        float* dst = p.n + (size_t)bh * p.dqk + ncol0 + chunk * 8;
        const float4 v0 = make_float4(nacc[0], nacc[1], nacc[2], nacc[3]);
        const float4 v1 = make_float4(nacc[4], nacc[5], nacc[6], nacc[7]);
        if (!whole_tile) {
          atomicAdd(reinterpret_cast<float4*>(dst), v0);
          atomicAdd(reinterpret_cast<float4*>(dst + 4), v1);
        } else {
          *reinterpret_cast<float4*>(dst) = v0;
          *reinterpret_cast<float4*>(dst + 4) = v1;
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) nacc[e] = 0.0f;
      // the eight warps agree that the piece's accumulator is complete before
      // any of them enters the epilogue's group barriers
      ok = bar_red_and(4, 384, mbar_wait_warp(bar(kFsAccFull), (uint32_t)piece & 1u, spin, abort, p.st, 24));
      if (!ok) break;                                // (this unit's barriers are done)
      if (!vw) {
        ++piece;
        continue;
      }
      tc_fence_after();
      // C leaves TMEM in 128-row x 32-column boxes (16 KB, 128-byte swizzle):
      // the four warps of a column half each write their 32 rows of a box, one
      // thread issues its TMA store (the whole head's tile) or add.  After the
      // CTA's last piece the stage ring is idle (every load has landed and
      // every MMA has read its stage), so a half takes half of the ring and the
      // staging area and keeps its boxes in flight; before then a half has one
      // box of the staging area.
      const bool last = i == nu - 1;
      const int h = warp < 6 ? 0 : 1, hc = p.dqk / 2;
      const bool issuer = qd == 0 && lane == 0;
      const int nbuf = last ? (int)(((uint32_t)p.nst * stage_bytes + kStagingBytes) / 2u / kCBoxBytes) : 1;
      const uint32_t region = last ? base + (uint32_t)(h * nbuf) * kCBoxBytes
                                   : base + (uint32_t)p.nst * stage_bytes + (uint32_t)h * kCBoxBytes;
      for (int bi = 0; bi < hc / 32; ++bi) {
        const int cb = h * hc + 32 * bi;
        const uint32_t box = region + (uint32_t)(bi % nbuf) * kCBoxBytes;
        uint32_t o[32];
        tmem_ld32(tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)cb, o);
        tmem_wait_ld();
        if (piece > 0 || bi >= nbuf) {
          if (issuer) tma_store_wait_read();         // the buffer's previous box has been read out
          named_bar_sync(2 + h, 128);
        }
        const uint32_t rp = box + (uint32_t)(32 * qd + lane) * 128u;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(rp + ((uint32_t)(q ^ (lane & 7)) << 4)),
                       "r"(o[4 * q]), "r"(o[4 * q + 1]), "r"(o[4 * q + 2]), "r"(o[4 * q + 3])
                       : "memory");
        fence_proxy_async_smem();
        named_bar_sync(2 + h, 128);
        if (issuer) {
          if (whole_tile) tma_store_3d(&tmap_c, box, cb, r0, bh);
          else tma_reduce_add_3d(&tmap_c, box, cb, r0, bh);
          tma_store_commit();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kFsAccEmpty));
      ++piece;
    }
    // A warp that left early makes up the barriers of the units it skipped, in
    // order: each unit's stage barrier and, at a piece end, the piece's
    // agreement (reporting failure), so that the other warps' barriers count
    // all eight warps and they leave at the next piece end.
    for (int j = done; j < nu; ++j) {
      named_bar_sync(1, 384);
      if (j == nu - 1 || (int)((va + j) % p.nchunk) == p.nchunk - 1) bar_red_and(4, 384, false);
    }
    ok = bar_red_and(1, 384, ok);
    if (lane == 0) tma_store_wait_read();            // staging boxes read out before the CTA exits
    __syncwarp();
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
          for (int b = q; b < 1 + nkb / p.kbox; b += kTcProducers) land += b == 0 ? 16384u : (uint32_t)p.kbox * 8192u;
      settle_last_phase(bar(kFsFull + i % p.nst), i / p.nst + 1, issued_s[0] > i, stage_bytes, land, 1LL << 22);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

// Zeroes C and n for a launch whose heads are shared by CTAs; the hand-off
// kernel is launched as its programmatic dependent and waits for it before its
// first add.
__global__ void __launch_bounds__(256) fs_zero_kernel(float4* __restrict__ C, long long nC4, float4* __restrict__ n,
                                                      long long nn4) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < nC4; x += stride) C[x] = z;
  for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < nn4; x += stride) n[x] = z;
}

}  // namespace

namespace {

// Static shared memory of the tensor-core kernel, read once.
size_t fs_static_smem() {
  static const size_t bytes = [] {
    cudaFuncAttributes fa;
    size_t b = 4096;
    if (cudaFuncGetAttributes(&fa, final_state_tc_kernel<true>) == cudaSuccess) b = fa.sharedSizeBytes;
    if (cudaFuncGetAttributes(&fa, final_state_tc_kernel<false>) == cudaSuccess) b = std::max(b, fa.sharedSizeBytes);
    cudaGetLastError();
    return b;
  }();
  return bytes;
}

cudaError_t launch_final_state_tc(const void* k, const void* v, GateTerms g, float* C, float* n, float* m, int BH,
                                  int T, int dqk, int dv, float scale, DevStatus st, int sms, cudaStream_t stream) {
  FsTcParams p;
  p.g = g; p.n = n; p.m = m; p.T = T; p.dqk = dqk; p.dv = dv; p.scale = scale; p.st = st;
  p.ntr = (dv + kTcM - 1) / kTcM;
  p.nchunk = (T + kTcTok - 1) / kTcTok;
  const size_t stage = 16384 + (size_t)(dqk / 64) * 8192;
  const long long room = (long long)kSmemLimit - (long long)fs_static_smem() - 1024 - (long long)kStagingBytes;
  p.nst = (int)std::min<long long>(kTcMaxStages, room / (long long)stage);
  if (p.nst < 2) return cudaErrorInvalidValue;
  const size_t smem = 1024 + (size_t)p.nst * stage + kStagingBytes;
  // A in TMEM when its slots fit beside the accumulator (512 columns)
  const bool at = dqk + 32 * p.nst <= 512 && getenv("MLSTM_FS_ASMEM") == nullptr;   // (variable: tuning)
  p.acol = (uint32_t)dqk;
  const int cols = at ? dqk + 32 * p.nst : dqk;
  p.tmem_cols = 32;
  while ((int)p.tmem_cols < cols) p.tmem_cols <<= 1;
  // One group of CTAs per row tile; whole heads per CTA when they spread over
  // a group's SMs within 10 %, otherwise the (head, chunk) units are dealt
  // evenly (at least 4 per CTA) and the heads cut between CTAs are added
  // together in C.
  p.ug = (long long)BH * p.nchunk;
  const int gmax = std::max(1, sms / p.ntr);
  const long long per = ((long long)BH + gmax - 1) / gmax;   // heads on the busiest CTA
  p.whole = per * gmax * 10 <= (long long)BH * 11 ? 1 : 0;
  if (const char* e = getenv("MLSTM_FS_WHOLE")) p.whole = atoi(e) != 0;   // tuning
  p.gt = (int)(p.whole ? std::min<long long>(gmax, BH) : std::max<long long>(1, std::min<long long>(gmax, p.ug / 4)));
  p.split = 0;
  if (!p.whole)
    for (long long kk = 1; kk < p.gt; ++kk)
      if ((kk * p.ug / p.gt) % p.nchunk != 0) p.split = 1;
  const long long G = (long long)p.gt * p.ntr;
  CUtensorMap mk, mv, mc;
  const int nkb = dqk / 64;
  p.kbox = nkb % 4 == 0 && nkb > 4 ? 4 : nkb % 3 == 0 && nkb > 3 ? 3 : nkb % 2 == 0 && nkb > 2 ? 2 : nkb <= 4 ? nkb : 1;
  if (!make_map_blocks(&mk, k, dqk, T, BH, kTcTok, p.kbox) || !make_map_blocks(&mv, v, dv, T, BH, kTcTok, 2) ||
      !make_map_f32(&mc, C, dqk, dv, BH, 32, kTcM))
    return cudaErrorInvalidValue;
  const auto kern = at ? final_state_tc_kernel<true> : final_state_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)G);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 0;
  if (p.split) {
    const long long nC4 = (long long)BH * dv * dqk / 4, nn4 = (long long)BH * dqk / 4;
    fs_zero_kernel<<<(unsigned)std::max(1, std::min(sms, (int)((nC4 + 255) / 256))), 256, 0, stream>>>(
        reinterpret_cast<float4*>(C), nC4, reinterpret_cast<float4*>(n), nn4);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    cfg.numAttrs = 1;
  }
  if ((e = cudaLaunchKernelEx(&cfg, kern, mk, mv, mc, p)) != cudaSuccess) return e;
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
