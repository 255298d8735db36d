// Fused causal mLSTM forward on the Blackwell tensor cores (tcgen05 + TMEM + TMA).
//
// "xLSTM: Extended Long Short-Term Memory", part 28/30, stabilized parallel
// forward, eqs (79)-(86).  bf16 q, k, v; fp32 accumulation; fp32 gates.
//
// One CTA computes 128 query rows (one TMEM lane per row) of one head for a
// slice of d_v.  Per causal key tile j (BN keys):
//   S_j  = Q K_j^T                       tcgen05.mma, A = Q, B = K_j (both K-major,
//                                        TMA-staged with 128-byte swizzle), D in TMEM
//   P_j  = S_j * s * D'_j                gating warps: tcgen05.ld of S, the gate
//                                        D'_ij = exp2(a2_j - p2_i) (eq 81; zero above
//                                        the diagonal), signed row sum b_i in fp32
//                                        (eq 83), bf16 P written to shared memory
//   O   += P_j V_j                       tcgen05.mma, A = P (K-major), B = V_j (MN-major)
// The row max m_i of eq (80) is known before the loop (prefix max from the gate
// pass), so the online rescaling of O and b that softmax attention needs never
// fires here and is not performed.  Off-diagonal tiles use the rank-one form
// D'_ij = 2^(a2_j - A) * 2^(A - p2_i) with A the tile's max column term (both
// factors <= 1): one exponential per row and per column instead of per entry.
// The epilogue divides O by n_i = max(|b_i|, exp(-m_i)) (eq 84) and stores H~.
//
// Warp roles (384 threads): warps 0, 2, 3 TMA producers (warp 2 also
// allocates TMEM), warp 1 MMA issuer, warps 4..11 gating + epilogue (two warps per TMEM lane
// quarter, each owning half of the tile's columns).  S is double-buffered in
// TMEM so the MMA of tile j+1 overlaps the gating of tile j.  Every wait is
// bounded; a wait that runs out records its site, raises a CTA-wide abort flag,
// drains in-flight copies and MMAs, frees TMEM and returns.
#include <algorithm>
#include <cstdlib>
#include <mutex>

#include "internal.h"
#include "tc_ptx.cuh"

namespace mlstm {
namespace {

using namespace tc;

constexpr int kBM = 128;           // query rows per CTA (TMEM lanes)
constexpr int kBN = 128;           // keys per tile
constexpr int kThreads = 384;
constexpr int kStageBytes = 32768;   // one ring slot: a [128 keys x 128 columns] K or V chunk
constexpr int kMaxStages = 8;
constexpr int kProducers = 3;      // warps 0, 2, 3 issue the tensor loads
constexpr uint32_t kTmemCols = 512;
constexpr int kSmemLimit = 232448;      // opt-in shared memory per block on sm_100-family
constexpr long long kDrainSpin = 1LL << 22;

#ifdef MLSTM_TRACE
// Per-event clock64 stamps of one CTA (trace builds only): [event][tile].
constexpr int kTraceTiles = 64;
__device__ long long g_trace[24 * kTraceTiles];
__device__ int g_trace_block;
#define TRACE(ev, j)                                                                  \
  do {                                                                                \
    if (trace_on && (j) < kTraceTiles) g_trace[(ev) * kTraceTiles + (j)] = clock64(); \
  } while (0)
#else
#define TRACE(ev, j) \
  do {               \
  } while (0)
#endif

// barrier slots
enum : int {
  kBarQFull = 0,
  kBarSFull = 1,    // 2 buffers
  kBarSEmpty = 3,   // 2 buffers
  kBarPFull = 5,
  kBarPEmpty = 6,
  kBarOFull = 7,
  kBarDrain = 8,
  kBarFull = 9,                   // kMaxStages
  kBarEmpty = 9 + kMaxStages,     // kMaxStages
  kNumBars = 9 + 2 * kMaxStages,
};

// wait-site codes recorded in the status word
enum : int { kSiteProducer = 1, kSiteMma = 2, kSiteGate = 3, kSiteEpilogue = 4 };

struct TcParams {
  const float* a2;
  const float* p2;
  const float* mrow;
  __nv_bfloat16* h;
  float* m_out;
  float* n_out;
  float* b_out;
  int T, BH, dqk, dv;
  int nsplit;      // CTAs per query tile along d_v (1 or 2)
  int dv_slice;    // d_v columns of the first slice (the second gets the rest)
  int nst;         // ring stages
  int vk;          // keys per V stage
  int nqt;         // query tiles per head
  float log2_scale;
  DevStatus st;
};

template <int BN, int NSBUF>
__global__ void __launch_bounds__(kThreads, 1)
fwd_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
              const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_h,
              const TcParams p) {
  constexpr int HALF = BN / 2;           // columns of a tile owned by one gating warp
  constexpr uint32_t SOFF = kTmemCols - NSBUF * BN;   // TMEM column of S buffer 0
  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t bars[kNumBars];
  __shared__ uint32_t tmem_holder;
  __shared__ int abort_flag;
  __shared__ int last_it_s[kMaxStages];     // last ring iteration loaded into each slot
  volatile int* last_it = last_it_s;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &abort_flag;
#ifdef MLSTM_TRACE
  const bool trace_on = (int)blockIdx.x == g_trace_block;   // read once
#endif

  // ---- work item: longest query tiles of all heads first
  const int per_rank = p.BH * p.nsplit;
  const int qt = p.nqt - 1 - (int)(blockIdx.x / per_rank);
  const int rem = (int)(blockIdx.x % per_rank);
  const int bh = rem / p.nsplit, split = rem % p.nsplit;
  const int i0 = qt * kBM;
  const int dv_off = split * p.dv_slice;
  const int dv_cta = split == 0 ? p.dv_slice : p.dv - p.dv_slice;
  const int i_last = min(p.T, i0 + kBM) - 1;
  const int nkv = i_last / BN + 1;
  const int nkc = (p.dqk + 127) / 128;   // K stages per key tile (128 d-columns each)
  const int nvc = (dv_cta + 127) / 128;  // V stages per key tile (128 d_v columns each)
  const size_t hbase = (size_t)bh * p.T;

  const uint32_t base = (smem_u32(dsmem) + 1023u) & ~1023u;
  const uint32_t sQ = base;                                  // dqk/64 boxes of [128 x 64] bf16
  const uint32_t sP = sQ + (uint32_t)p.dqk * kBM * 2;        // BN/64 boxes of [128 x 64] bf16
  const uint32_t sRing = sP + (uint32_t)BN * kBM * 2;        // nst stages of 16 KB
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  if (threadIdx.x < kMaxStages) last_it_s[threadIdx.x] = -1;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(bar(kBarQFull), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kBarSFull + b), 1);
      mbar_init(bar(kBarSEmpty + b), 8);   // one arrival per gating warp
    }
    mbar_init(bar(kBarPFull), 8);
    mbar_init(bar(kBarPEmpty), 1);
    mbar_init(bar(kBarOFull), 1);
    mbar_init(bar(kBarDrain), 1);
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(bar(kBarFull + s), 1);
      mbar_init(bar(kBarEmpty + s), 1);
    }
    fence_barrier_init();
    tma_prefetch_desc(&tmap_q);
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_v);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(&tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_holder;
  const long long spin = p.st.spin_limit;
  if (threadIdx.x == 0) TRACE(14, 0);

  if ((warp == 0 || warp == 2 || warp == 3) && lane == 0) {
    // ------------------------------------------------------------ TMA producers
    // Three producer warps share the ring.  Each slot has one owner, producer
    // slot % kProducers, which handles every round of that slot in order, so
    // no producer ever waits more than one phase ahead on a slot's barrier
    // (parity waits cannot tell phase k from phase k+2).  Several issuing
    // warps keep more tensor loads in flight than one.  Ring order per key
    // tile j: K_j (nkc slots), then V_{j-1} (nvc slots).
    const int pi = warp == 0 ? 0 : warp - 1;
    if (pi == 0) mbar_arrive_expect_tx(bar(kBarQFull), (uint32_t)p.dqk * kBM * 2);
    for (int b2 = pi; b2 < p.dqk / 64; b2 += kProducers)
      tma_load_3d(sQ + b2 * 16384u, &tmap_q, bar(kBarQFull), b2 * 64, i0, bh);
    int st = 0, it = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int j = 0; j <= nkv && ok; ++j) {
      if (j < nkv) {
        for (int c = 0; c < nkc; ++c, ++it) {
          if (st % kProducers == pi) {
            ok = mbar_wait(bar(kBarEmpty + st), ph ^ 1, spin, abort, p.st, kSiteProducer);
            if (!ok) break;
            if (c == 0) TRACE(4, j);
            TRACE(16, it);
            const int kb = min(2, (p.dqk - c * 128) / 64);     // 64-column boxes in this chunk
            mbar_arrive_expect_tx(bar(kBarFull + st), (uint32_t)kb * BN * 128);
            for (int b2 = 0; b2 < kb; ++b2)
              tma_load_3d(sRing + st * kStageBytes + b2 * (BN * 128u), &tmap_k, bar(kBarFull + st),
                          c * 128 + b2 * 64, j * BN, bh);
            last_it[st] = it;
          }
          if (++st == p.nst) { st = 0; ph ^= 1; }
        }
      }
      if (j >= 1 && ok) {
        for (int e = 0; e < nvc; ++e, ++it) {
          if (st % kProducers == pi) {
            ok = mbar_wait(bar(kBarEmpty + st), ph ^ 1, spin, abort, p.st, kSiteProducer);
            if (!ok) break;
            if (e == 0) TRACE(5, j - 1);
            TRACE(16, it);
            const uint32_t dst = sRing + st * kStageBytes;
            const int vb = min(2, (dv_cta - e * 128) / 64);   // 64-column boxes in this chunk
            mbar_arrive_expect_tx(bar(kBarFull + st), (uint32_t)vb * BN * 128);
            for (int s2 = 0; s2 < vb; ++s2)
              tma_load_3d(dst + s2 * (BN * 128u), &tmap_v, bar(kBarFull + st), dv_off + e * 128 + s2 * 64,
                          (j - 1) * BN, bh);
            last_it[st] = it;
          }
          if (++st == p.nst) { st = 0; ph ^= 1; }
        }
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    // Descriptors are built once; per MMA only the start-address field moves
    // (16-byte units in the low bits, no carry: shared addresses < 256 KB).
    const uint32_t idS = idesc_bf16_f32(kBM, BN, 0, 0);
    const uint64_t dQ = smem_desc_sw128(sQ, 16, 1024);
    const uint64_t dK = smem_desc_sw128(sRing, 16, 1024);
    const uint64_t dP = smem_desc_sw128(sP, 16, 1024);
    // V chunk: [128 keys x 128 d_v] as two 64-column boxes (MN-major atoms
    // BN*128 bytes apart); O[:, chunk] += P V_chunk over 8 k-steps of 16 keys.
    const uint64_t dV = smem_desc_sw128(sRing, BN * 128u, 1024);
    const uint32_t idO128 = idesc_bf16_f32(kBM, 128, 0, 1), idO64 = idesc_bf16_f32(kBM, 64, 0, 1);
    bool ok = mbar_wait(bar(kBarQFull), 0, spin, abort, p.st, kSiteMma);
    tc_fence_after();
    int st = 0, mit = 0;
    uint32_t ph = 0;
    for (int j = 0; j <= nkv && ok; ++j) {
      if (j < nkv) {
        const int buf = j % NSBUF, u = j / NSBUF;
        TRACE(0, j);
        ok = mbar_wait(bar(kBarSEmpty + buf), (u & 1) ^ 1, spin, abort, p.st, kSiteMma);
        if (!ok) break;
        // no tcgen05 fence: the gating warps finished their TMEM reads (wait::ld)
        // and made P visible to the async proxy before arriving
        const uint32_t d_s = tmem + SOFF + buf * BN;
        for (int c = 0; c < nkc; ++c, ++mit) {
          TRACE(17, mit);
          ok = mbar_wait(bar(kBarFull + st), ph, spin, abort, p.st, kSiteMma);
          if (!ok) break;
          TRACE(18, mit);
          if (c == 0) TRACE(13, j);
          const uint64_t aq = dQ + (uint64_t)(c * 2048);            // Q boxes 2c, 2c+1 (16 KB each)
          const uint64_t bk = dK + (uint64_t)(st * (kStageBytes >> 4));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            if (j == 5) TRACE(20, c * 8 + kk);
            mma_bf16_ss(d_s, aq + 2 * kk, bk + 2 * kk, idS, (c | kk) != 0);
          }
          if (p.dqk - c * 128 > 64) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              if (j == 5) TRACE(20, c * 8 + 4 + kk);
              mma_bf16_ss(d_s, aq + 1024 + 2 * kk, bk + (BN * 128 >> 4) + 2 * kk, idS, 1);
            }
          }
          mma_commit(bar(kBarEmpty + st));
          TRACE(19, mit);
          if (++st == p.nst) { st = 0; ph ^= 1; }
        }
        if (!ok) break;
        mma_commit(bar(kBarSFull + buf));
        TRACE(1, j);
      }
      if (j >= 1) {
        const int jj = j - 1;
        ok = mbar_wait(bar(kBarPFull), jj & 1, spin, abort, p.st, kSiteMma);
        if (!ok) break;
        // no tcgen05 fence: the gating warps finished their TMEM reads (wait::ld)
        // and made P visible to the async proxy before arriving
        TRACE(2, jj);
        for (int e = 0; e < nvc; ++e, ++mit) {
          TRACE(17, mit);
          ok = mbar_wait(bar(kBarFull + st), ph, spin, abort, p.st, kSiteMma);
          if (!ok) break;
          TRACE(18, mit);
          if (e == 0) TRACE(15, jj);
          const uint64_t bv = dV + (uint64_t)(st * (kStageBytes >> 4));
          const uint32_t d_o = tmem + e * 128;
          const uint32_t acc0 = jj != 0;
          // keys 16kk..16kk+15: P box kk/4 at +32 B per step; V rows at +2 KB per 16 keys
          if (dv_cta - e * 128 >= 128) {
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk) {
              if (jj == 5) TRACE(21, e * 8 + kk);
              mma_bf16_ss(d_o, dP + (kk >> 2) * 1024 + (kk & 3) * 2, bv + kk * 128, idO128, acc0 | (kk != 0));
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              mma_bf16_ss(d_o, dP + (kk >> 2) * 1024 + (kk & 3) * 2, bv + kk * 128, idO64, acc0 | (kk != 0));
          }
          mma_commit(bar(kBarEmpty + st));
          TRACE(19, mit);
          if (jj == 5) TRACE(22, e);
          if (++st == p.nst) { st = 0; ph ^= 1; }
        }
        if (!ok) break;
        mma_commit(bar(kBarPEmpty));
        TRACE(3, jj);
      }
    }
    if (ok) mma_commit(bar(kBarOFull));
    // drain: every MMA issued above has completed before TMEM is released
    mma_commit(bar(kBarDrain));
    for (long long w = 0; w < kDrainSpin; ++w)
      if (mbar_try_wait(bar(kBarDrain), 0)) break;
  } else if (warp >= 4) {
    // ------------------------------------------------------------ gating + epilogue
    const int gw = warp - 4, qd = gw & 3, half = gw >> 2;
    // gate terms come from the preceding gate pass: wait for that grid (a no-op
    // unless this kernel was launched as its programmatic dependent)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int rl = 32 * qd + lane;                  // row within the tile = TMEM lane
    const int i = i0 + rl;
    const bool row_ok = i < p.T;
    const float rr = row_ok ? p.p2[hbase + i] - p.log2_scale : 0.0f;   // P = S * 2^(a2_j - rr)
    const uint32_t lane_addr = (uint32_t)(32 * qd) << 16;
    float bsum = 0.0f;
    bool ok = true;
    // column terms of the next tile are loaded one tile ahead (latency hiding)
    float av_next[HALF / 32];
#pragma unroll
    for (int t = 0; t < HALF / 32; ++t) {
      const int col = half * HALF + lane + 32 * t;
      av_next[t] = col < p.T ? p.a2[hbase + col] : -INFINITY;
    }
    // A warp whose wait gives up (raising the abort flag) leaves the tile loop,
    // which has no group barrier; the gating warps agree on the result at the
    // reducing barrier of the epilogue, which every one of them reaches.
    for (int j = 0; j < nkv && ok; ++j) {
      const int j0 = j * BN, cbase = j0 + half * HALF;
      const int buf = j % NSBUF, u = j / NSBUF;
      float av[HALF / 32];
#pragma unroll
      for (int t = 0; t < HALF / 32; ++t) {
        av[t] = av_next[t];
        const int col = cbase + BN + lane + 32 * t;
        av_next[t] = (j + 1 < nkv && col < p.T) ? p.a2[hbase + col] : -INFINITY;
      }
      const bool diag = j0 + BN - 1 > i0;
      float A = -INFINITY;
      if (!diag) {
#pragma unroll
        for (int t = 0; t < HALF / 32; ++t) A = fmaxf(A, av[t]);
        A = warp_max(A);
#pragma unroll
        for (int t = 0; t < HALF / 32; ++t) av[t] = A == -INFINITY ? 0.0f : exp2f(av[t] - A);
      }
      ok = mbar_wait(bar(kBarSFull + buf), u & 1, spin, abort, p.st, kSiteGate);
      if (!ok) break;
      tc_fence_after();
      if (gw == 0 && lane == 0) TRACE(6, j);
      uint32_t sv[HALF];
#pragma unroll
      for (int t = 0; t < HALF / 32; ++t)
        tmem_ld32(tmem + lane_addr + SOFF + buf * BN + half * HALF + 32 * t,
                  *reinterpret_cast<uint32_t(*)[32]>(&sv[32 * t]));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarSEmpty + buf));
      if (gw == 0 && lane == 0) TRACE(7, j);

      uint32_t pk[HALF / 2];
      if (!diag) {
        const float r = (A == -INFINITY || !row_ok) ? 0.0f : exp2f(A - rr);
#pragma unroll
        for (int c = 0; c < HALF; c += 2) {
          const float c0 = __shfl_sync(0xffffffffu, av[c / 32], c & 31);
          const float c1 = __shfl_sync(0xffffffffu, av[(c + 1) / 32], (c + 1) & 31);
          const float x0 = __uint_as_float(sv[c]) * c0 * r;
          const float x1 = __uint_as_float(sv[c + 1]) * c1 * r;
          bsum += x0 + x1;
          pk[c / 2] = pack_bf16x2(x0, x1);
        }
      } else {
#pragma unroll
        for (int c = 0; c < HALF; c += 2) {
          const float a0 = __shfl_sync(0xffffffffu, av[c / 32], c & 31);
          const float a1 = __shfl_sync(0xffffffffu, av[(c + 1) / 32], (c + 1) & 31);
          const int col = cbase + c;
          const float e0 = (row_ok && col <= i) ? exp2f(a0 - rr) : 0.0f;
          const float e1 = (row_ok && col + 1 <= i) ? exp2f(a1 - rr) : 0.0f;
          const float x0 = __uint_as_float(sv[c]) * e0;
          const float x1 = __uint_as_float(sv[c + 1]) * e1;
          bsum += x0 + x1;
          pk[c / 2] = pack_bf16x2(x0, x1);
        }
      }
      // the previous tile's O MMA must be done reading P before it is overwritten
      if (gw == 0 && lane == 0) TRACE(8, j);
      ok = mbar_wait(bar(kBarPEmpty), (j & 1) ^ 1, spin, abort, p.st, kSiteGate);
      if (!ok) break;
      if (gw == 0 && lane == 0) TRACE(9, j);
#pragma unroll
      for (int g = 0; g < HALF / 8; ++g) {
        const int c = half * HALF + 8 * g;           // column within the tile
        const uint32_t addr = sP + (c >> 6) * 16384u + rl * 128u + ((((c & 63) >> 3) ^ (rl & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * g]),
                     "r"(pk[4 * g + 1]), "r"(pk[4 * g + 2]), "r"(pk[4 * g + 3])
                     : "memory");
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPFull));
      if (gw == 0 && lane == 0) TRACE(10, j);
    }

    // ---- epilogue: n = max(|b|, exp(-m)), H~ = O / n
    if (ok) ok = mbar_wait(bar(kBarOFull), 0, spin, abort, p.st, kSiteEpilogue);
    tc_fence_after();
    if (gw == 0 && lane == 0) TRACE(11, 0);
    // After the last O MMA no operand is read any more: the P tile combines the
    // two half row sums, and Q/P/ring space stages the bf16 output tile (128
    // rows x dv_cta in 64-column boxes with the 128-byte swizzle) for TMA stores.
    float* bpart = reinterpret_cast<float*>(dsmem + (sP - smem_u32(dsmem)));
    if (ok) bpart[half * kBM + rl] = bsum;
    // every gating warp arrives here whatever its waits returned; all of them
    // take the result of the whole group from here on
    ok = bar_red_and(1, 256, ok);
    float nrm = 0.0f, m = 0.0f, bsig = 0.0f;
    if (ok) {
      const float b = bpart[rl] + bpart[kBM + rl];
      bsig = b;
      m = row_ok ? p.mrow[hbase + i] : 0.0f;
      nrm = fmaxf(fabsf(b), expf(-m));
    }
    named_bar_sync(1, 256);              // bpart reads done before the tile overwrites P
    if (ok) {
      const float inv = nrm > 0.0f ? 1.0f / nrm : 0.0f;
      const int cols = dv_cta / 2, c0 = half * cols;
      for (int ch = 0; ch < cols / 32; ++ch) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_addr + c0 + 32 * ch, o);
        tmem_wait_ld();
        const int col = c0 + 32 * ch;                    // first of this thread's 32 columns
        const uint32_t box = sQ + (uint32_t)(col >> 6) * 16384u + rl * 128u;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint32_t w[4];
#pragma unroll
          for (int t = 0; t < 4; ++t)
            w[t] = pack_bf16x2(__uint_as_float(o[8 * g + 2 * t]) * inv, __uint_as_float(o[8 * g + 2 * t + 1]) * inv);
          const int chunk = ((col & 63) >> 3) + g;     // 16-byte chunk within the 128-byte row
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(box + ((chunk ^ (rl & 7)) << 4)), "r"(w[0]),
                       "r"(w[1]), "r"(w[2]), "r"(w[3])
                       : "memory");
        }
      }
      if (row_ok && split == 0 && half == 0) {
        if (p.m_out) p.m_out[hbase + i] = m;
        if (p.n_out) p.n_out[hbase + i] = nrm;
        if (p.b_out) p.b_out[hbase + i] = bsig;
      }
      fence_proxy_async_smem();
    }
    named_bar_sync(1, 256);
    if (ok && gw == 0 && lane == 0) {
      for (int b2 = 0; b2 < dv_cta / 64; ++b2)
        tma_store_3d(&tmap_h, sQ + b2 * 16384u, dv_off + b2 * 64, i0, bh);
      tma_store_commit();
      tma_store_wait_read();
    }
    tc_fence_before();
    if (gw == 0 && lane == 0) TRACE(12, 0);
  }

  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // After an abort some loads may never have been consumed: wait (bounded)
  // until none of them can still write this CTA's shared memory.
  if (threadIdx.x == 0 && abort_flag) {
    for (long long w = 0; w < kDrainSpin; ++w)
      if (mbar_try_wait(bar(kBarQFull), 0)) break;
    for (int s2 = 0; s2 < p.nst; ++s2)
      if (last_it[s2] >= 0) {
        const uint32_t par = (uint32_t)(last_it[s2] / p.nst) & 1u;
        for (long long w = 0; w < kDrainSpin; ++w)
          if (mbar_try_wait(bar(kBarFull + s2), par)) break;
      }
  }
}

// ---------------------------------------------------------------- host side
struct Plan {
  int nsbuf, nsplit, dv_slice, vk, nst;
  size_t smem;
};

// Tiling: 128 query rows x 128 keys.  TMEM (512 columns) holds O (dv_slice
// columns) and NSBUF S buffers of 128 columns: dv <= 256 double-buffers S;
// dv <= 384 single-buffers it (the gating warps release S as soon as they have
// read it); larger dv is split over two CTAs of 256 + the rest.
Plan plan_for(int dqk, int dv) {
  Plan pl;
  if (dv <= 256) {
    pl.nsbuf = 2; pl.nsplit = 1; pl.dv_slice = dv;
  } else if (dv <= 384) {
    pl.nsbuf = 1; pl.nsplit = 1; pl.dv_slice = dv;
  } else {
    pl.nsbuf = 2; pl.nsplit = 2; pl.dv_slice = 256;
  }
  pl.vk = kBN;   // V boxes cover a whole key tile
  const size_t fixed = 1024 + (size_t)dqk * kBM * 2 + (size_t)kBN * kBM * 2;
  const size_t static_smem = 1024;  // barriers, TMEM address, abort flag (rounded up)
  long long room = (long long)kSmemLimit - (long long)static_smem - (long long)fixed;
  pl.nst = (int)std::min<long long>(kMaxStages, room / kStageBytes);
  static const char* force_st = getenv("MLSTM_TC_STAGES");   // tuning: fewer ring stages
  if (force_st && atoi(force_st) >= 2 && atoi(force_st) < pl.nst) pl.nst = atoi(force_st);
  pl.smem = fixed + (size_t)pl.nst * kStageBytes;
  return pl;
}

template <int NSBUF>
int launch_ns(const FwdArgs& a, const Plan& pl, const CUtensorMap& mq, const CUtensorMap& mk,
              const CUtensorMap& mv, const CUtensorMap& mh, cudaStream_t stream) {
  if (cudaFuncSetAttribute(fwd_tc_kernel<kBN, NSBUF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)pl.smem) != cudaSuccess)
    return kCuda;
  TcParams p;
  p.a2 = a.g.a2; p.p2 = a.g.p2; p.mrow = a.g.m;
  p.h = (__nv_bfloat16*)a.h; p.m_out = a.m_out; p.n_out = a.n_out; p.b_out = a.b_out;
  p.T = a.T; p.BH = a.BH; p.dqk = a.dqk; p.dv = a.dv;
  p.nsplit = pl.nsplit; p.dv_slice = pl.dv_slice; p.nst = pl.nst; p.vk = pl.vk;
  p.nqt = (a.T + kBM - 1) / kBM;
  p.log2_scale = log2f(a.scale);
  p.st = a.st;
  const long long grid = (long long)p.nqt * a.BH * pl.nsplit;
  if (grid > 0x7fffffffLL) return kInval;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.after_gate_prep ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, fwd_tc_kernel<kBN, NSBUF>, mq, mk, mv, mh, p) != cudaSuccess) return kCuda;
  return cudaGetLastError() == cudaSuccess ? kOk : kCuda;
}

}  // namespace

int device_is_sm100_family() {
  int dev = 0, major = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return 0;
  return major == 10;
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
  static std::once_flag once;
  static EncodeTiled fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(ptr);
  });
  return fn;
}

// [BH, T, d] bf16 viewed as a 3-D tensor (d fastest); box = 64 x rows x 1 with
// 128-byte swizzle.  Rows past T read as zeros.
bool make_map(CUtensorMap* m, const void* base, int d, int T, int BH, int rows) {
  EncodeTiled enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)T, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)d * 2 * T};
  cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [BH, T, d] bf16 viewed as a 4-D tensor (64 columns, T, d / 64 column
// blocks, BH), so that one box (64 x rows x blocks x 1, 128-byte swizzle)
// lands as `blocks` consecutive 64-column tiles of rows x 128 bytes: the layout
// of that many separate 64-column boxes, in one copy.  Rows past T and blocks
// past d read as zeros.
bool make_map_blocks(CUtensorMap* m, const void* base, int d, int T, int BH, int rows, int blocks) {
  EncodeTiled enc = encode_fn();
  if (!enc || d % 64 != 0) return false;
  cuuint64_t dims[4] = {64, (cuuint64_t)T, (cuuint64_t)(d / 64), (cuuint64_t)BH};
  cuuint64_t strides[3] = {(cuuint64_t)d * 2, 128, (cuuint64_t)d * 2 * T};
  cuuint32_t box[4] = {64, (cuuint32_t)rows, (cuuint32_t)blocks, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [BH, rows, cols] bf16 with row pitch ld (ld*2 a multiple of 16) viewed as
// 4-D (64 columns, rows, cols / 64 column blocks, BH): one box (64 x box_rows x
// blocks x 1, 128-byte swizzle) lands as `blocks` consecutive 64-column tiles.
// cols must be a multiple of 64 (a partial last block would read the pitch
// padding instead of zeros).
bool make_map_ld_blocks(CUtensorMap* m, const void* base, int cols, int rows, int BH, int ld, int box_rows,
                        int blocks) {
  EncodeTiled enc = encode_fn();
  if (!enc || (ld * 2) % 16 != 0 || cols % 64 != 0) return false;
  cuuint64_t dims[4] = {64, (cuuint64_t)rows, (cuuint64_t)(cols / 64), (cuuint64_t)BH};
  cuuint64_t strides[3] = {(cuuint64_t)ld * 2, 128, (cuuint64_t)ld * 2 * rows};
  cuuint32_t box[4] = {64, (cuuint32_t)box_rows, (cuuint32_t)blocks, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [BH, rows, cols] fp32 viewed as a 3-D tensor (cols fastest); box = box_cols
// x box_rows x 1 with 128-byte swizzle (box_cols * 4 <= 128).
bool make_map_f32(CUtensorMap* m, float* base, int cols, int rows, int BH, int box_cols, int box_rows) {
  EncodeTiled enc = encode_fn();
  if (!enc || (cols * 4) % 16 != 0 || box_cols * 4 > 128) return false;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)cols * 4, (cuuint64_t)cols * 4 * rows};
  cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_ld(CUtensorMap* m, const void* base, int cols, int rows, int BH, int ld, int box_rows) {
  EncodeTiled enc = encode_fn();
  if (!enc || (ld * 2) % 16 != 0) return false;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)ld * 2, (cuuint64_t)ld * 2 * rows};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

#ifdef MLSTM_TRACE
extern "C" int mlstm_trace_set_block(int b) {
  return cudaMemcpyToSymbol(g_trace_block, &b, sizeof(int)) == cudaSuccess ? 0 : -4;
}
extern "C" int mlstm_trace_read(long long* host) {
  return cudaMemcpyFromSymbol(host, g_trace, sizeof(g_trace)) == cudaSuccess ? 0 : -4;
}
#endif

bool fwd_tc_supported(int dqk, int dv, int dtype) {
  return dtype == kBF16 && dqk % 64 == 0 && dv % 64 == 0 && dqk >= 64 && dv >= 64 && dqk <= 512 &&
         dv <= 512;
}

int launch_fwd_tc(const FwdArgs& a, cudaStream_t stream) {
  if (a.BH <= 0 || a.T <= 0) return kOk;
  if (!fwd_tc_supported(a.dqk, a.dv, a.dtype)) return kUnsupported;
  if (!device_is_sm100_family()) return kUnsupported;
  // CTA-pair kernel when the shape allows it; MLSTM_TC_VARIANT=single or
  // =pair in the environment forces one variant (tuning and tests).
  const char* var = getenv("MLSTM_TC_VARIANT");
  const bool force_single = var && var[0] == 's', force_pair = var && var[0] == 'p';
  // The pair halves each SM's K/V traffic and runs persistently; it is as fast
  // or faster from T = 512 on (measured), and the only choice for d_v = 512.
  const bool pair_pays = a.T > 256 || a.dv > 384;
  if (!force_single && fwd_tc2_supported(a.dqk, a.dv) && (pair_pays || force_pair))
    return launch_fwd_tc2(a, stream);
  if (force_pair) return kUnsupported;
  const Plan pl = plan_for(a.dqk, a.dv);
  if (pl.nst < 2) return kUnsupported;
  CUtensorMap mq, mk, mv, mh;
  if (!make_map(&mq, a.q, a.dqk, a.T, a.BH, kBM) || !make_map(&mk, a.k, a.dqk, a.T, a.BH, kBN) ||
      !make_map(&mv, a.v, a.dv, a.T, a.BH, pl.vk) || !make_map(&mh, a.h, a.dv, a.T, a.BH, kBM))
    return kCuda;
  const int rc = pl.nsbuf == 1 ? launch_ns<1>(a, pl, mq, mk, mv, mh, stream)
                               : launch_ns<2>(a, pl, mq, mk, mv, mh, stream);
  // this kernel does not fuse the output gate: apply it in a separate pass
  if (rc == kOk && a.og &&
      launch_apply_ogate(a.h, a.og, (long long)a.BH * a.T * a.dv, a.dtype, stream) != cudaSuccess)
    return kCuda;
  return rc;
}

}  // namespace mlstm
