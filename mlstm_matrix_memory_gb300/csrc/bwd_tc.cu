// Tiles of the stabilized parallel mLSTM backward on the tensor cores.
//
// "xLSTM: Extended Long Short-Term Memory", part 28/30, "Parallel mLSTM
// Backward Pass", eqs (87)-(95), (100), for bf16 q, k, v, dH~:
//   dC     = dH~ V^T                                         (87)
//   dn_i   = -(sum_j C~'_ij dC_ij) / n_i^2                    (89)
//   db_i   = sign(b_i) dn_i where |b_i| > exp(-m_i), else 0   (90)
//   G      = D' (.) (dC / n + db),   dD~ = S (.) G            (91)-(95)
//   P      = C~' / n                                         (operand of eq 100)
// with S = Q K^T / sqrt(d) and C~' = S (.) D'.  The row sum in eq (89) needs
// no pass over the keys: sum_j C~'_ij dC_ij = dH~_i . (sum_j C~'_ij v_j)
// = n_i dH~_i . h~_i, with h~ and n (and the signed b) from the forward.
//
// Per 128 x 128 tile (query block ib, key block jb <= ib) of one head:
//   S  = Q_ib K_jb^T      tcgen05.mma into a TMEM buffer's columns 0..127
//   dC = dH_ib V_jb^T     tcgen05.mma into its columns 128..255
// both contractions streamed through a ring of 64-column chunks (TMA, 128-byte
// swizzle, zero fill past d).  The kernel is persistent, one CTA per SM,
// tiles taken round robin in head-major order; two TMEM buffers let the
// products of one tile run while eight epilogue warps (two per TMEM lane
// quarter, 64 columns each) turn the previous one into G and P: fp32 from
// the TMEM rows, bf16 staging, TMA stores, and the tile's row and column sums
// of dD~ (the column sums by a shuffle reduce-scatter, so every partial is
// formed in a fixed order).
// Within the diagonal tile G and P are stored as zero above the diagonal;
// nothing above it is ever stored or read.
#include <algorithm>
#include <cmath>
#include <cstdlib>

#include "internal.h"
#include "tc_ptx.cuh"

namespace mlstm {
namespace {

using namespace tc;

constexpr int kTile = 128;            // query rows and keys of a tile
constexpr int kThreads = 320;         // warp 0 TMA, warp 1 MMA + TMEM, warps 2..9 epilogue
constexpr int kNst = 4;               // ring stages
constexpr uint32_t kStage = 32768;    // a stage: [128 rows x 64 columns] of A and of B
constexpr uint32_t kStaging = 65536;  // bf16 G and P of a tile: four [128 x 64] boxes
constexpr long long kDrainSpin = 1LL << 22;

enum : int {
  kBarFull = 0, kBarEmpty = kNst, kBarAccFull = 2 * kNst, kBarAccEmpty = 2 * kNst + 2, kBarDrain = 2 * kNst + 4,
  kNumBars = 2 * kNst + 5
};
enum : int { kSiteTProducer = 41, kSiteTMma = 42, kSiteTEpi = 43 };

struct TileParams {
  int wide;                  // two 64-column chunks a stage through 4-D views (d_qk, d_v multiples of 64)
  const float* a2;
  const float* p2;
  const float* invn;
  const float* db;
  float* Rpart;
  float* Cpart;
  int T, BH, dqk, dv, nb, nitems;
  float scale;
  DevStatus st;
};

// 16-byte chunk q (8 bf16) of row r of a [128 x 64] box with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz(uint32_t box, int r, int q) {
  return box + (uint32_t)r * 128u + ((uint32_t)(q ^ (r & 7)) << 4);
}

// G, P and dD~/s of 32 consecutive columns (first key j0c) of one row i from
// the TMEM words of S/s and dC.  DIAG: the diagonal tile, D' = 2^(a2_j - p2_i)
// for j <= i (ct holds a2); otherwise D' = ct_j rowf (ct holds 2^(a2_j - A)).
template <bool DIAG>
__device__ __forceinline__ void tile_values(const uint32_t (&sv)[32], const uint32_t (&cv)[32], const float* ct,
                                            int j0c, int i, bool row_ok, float p2i, float rowf, float invn,
                                            float dbi, float pscale, float (&dd)[32], uint32_t (&gw)[16],
                                            uint32_t (&pw)[16], float& rs) {
  // column pairs in packed fp32 (each element rounded as in scalar fp32; the
  // row sum runs in two lanes, added at the end)
  const f32x2 rowf2 = f2_make(rowf, rowf), invn2 = f2_make(invn, invn), dbi2 = f2_make(dbi, dbi);
  const f32x2 ps2 = f2_make(pscale, pscale);
  f32x2 rs2 = f2_make(0.0f, 0.0f);
#pragma unroll
  for (int c = 0; c < 32; c += 4) {
    const float4 c4 = *reinterpret_cast<const float4*>(ct + c);
#pragma unroll
    for (int e = 0; e < 4; e += 2) {
      f32x2 dp;
      if (DIAG) {
        const float ca = e == 0 ? c4.x : c4.z, cb = e == 0 ? c4.y : c4.w;
        dp = f2_make((row_ok && j0c + c + e <= i) ? exp2f(ca - p2i) : 0.0f,
                     (row_ok && j0c + c + e + 1 <= i) ? exp2f(cb - p2i) : 0.0f);
      } else {
        dp = f2_mul(e == 0 ? f2_make(c4.x, c4.y) : f2_make(c4.z, c4.w), rowf2);
      }
      const f32x2 sr = f2_make(__uint_as_float(sv[c + e]), __uint_as_float(sv[c + e + 1]));   // S / s
      const f32x2 cc = f2_make(__uint_as_float(cv[c + e]), __uint_as_float(cv[c + e + 1]));
      const f32x2 g = f2_mul(dp, f2_fma(cc, invn2, dbi2));         // D' (.) dC~'
      const f32x2 pv = f2_mul(f2_mul(sr, ps2), dp);                // C~' / n
      const f32x2 d2 = f2_mul(sr, g);                              // dD~ / s
      rs2 = f2_add(rs2, d2);
      const float2 gf = f2_split(g), pf = f2_split(pv), df = f2_split(d2);
      dd[c + e] = df.x;
      dd[c + e + 1] = df.y;
      gw[(c + e) / 2] = pack_bf16x2(gf.x, gf.y);
      pw[(c + e) / 2] = pack_bf16x2(pf.x, pf.y);
    }
  }
  const float2 r2 = f2_split(rs2);
  rs += r2.x + r2.y;
}

// Item it -> head and tile: t = ib (ib + 1) / 2 + jb, jb <= ib.
__device__ __forceinline__ void tile_of(int it, int nb, int* bh, int* ib, int* jb) {
  const int ntri = nb * (nb + 1) / 2;
  *bh = it / ntri;
  const int t = it - *bh * ntri;
  int i = (int)((sqrtf(8.0f * (float)t + 1.0f) - 1.0f) * 0.5f);
  while (i * (i + 1) / 2 > t) --i;
  while ((i + 1) * (i + 2) / 2 <= t) ++i;
  *ib = i;
  *jb = t - i * (i + 1) / 2;
}

__global__ void __launch_bounds__(kThreads, 1)
bwd_tile_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                const __grid_constant__ CUtensorMap tmap_dh, const __grid_constant__ CUtensorMap tmap_v,
                const __grid_constant__ CUtensorMap tmap_g, const __grid_constant__ CUtensorMap tmap_p,
                const __grid_constant__ CUtensorMap tmap_q4, const __grid_constant__ CUtensorMap tmap_k4,
                const __grid_constant__ CUtensorMap tmap_dh4, const __grid_constant__ CUtensorMap tmap_v4,
                const TileParams p) {
  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t bars[kNumBars];
  __shared__ uint32_t tmem_holder;
  __shared__ int abort_flag;
  __shared__ int issued_s;                    // chunks whose loads the producer issued
  __shared__ int epi_stop;
  __shared__ __align__(16) float col_term[kTile];   // a2_j (diagonal tile) or 2^(a2_j - A); read as float4
  __shared__ float col_red[4][kTile];         // per lane quarter: column sums of dD~ over its 32 rows
  __shared__ float row_red[2][kTile];         // per column half: row sums of dD~
  __shared__ float amax_red[4];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &abort_flag;
  const int nb = p.nb;
  const uint32_t base = (smem_u32(dsmem) + 1023u) & ~1023u;
  const uint32_t sStage = base + kNst * kStage;            // staging of G (boxes 0, 1) and P (2, 3)
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  // ring stages: four of one 64-column chunk of A and of B, or (p.wide: d_qk
  // and d_v multiples of 64) two of two chunks, each operand one 4-D box
  const int nst = p.wide ? 2 : kNst;
  const uint32_t stage = p.wide ? 2u * kStage : kStage;
  const int cw = p.wide ? 128 : 64;
  const int nq = (p.dqk + cw - 1) / cw, nch = nq + (p.dv + cw - 1) / cw;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    issued_s = 0;
    for (int s = 0; s < kNst; ++s) {
      mbar_init(bar(kBarFull + s), 1);
      mbar_init(bar(kBarEmpty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kBarAccFull + b), 1);
      mbar_init(bar(kBarAccEmpty + b), 8);      // one arrival per epilogue warp
    }
    mbar_init(bar(kBarDrain), 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_holder;
  const long long spin = p.st.spin_limit;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    tma_prefetch_desc(&tmap_q);
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_dh);
    tma_prefetch_desc(&tmap_v);
    int cc = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < p.nitems && ok; it += gridDim.x) {
      int bh, ib, jb;
      tile_of(it, nb, &bh, &ib, &jb);
      const int i0 = ib * kTile, j0 = jb * kTile;
      for (int c = 0; c < nch; ++c, ++cc) {
        const int s = cc % nst, u = cc / nst;
        ok = mbar_wait(bar(kBarEmpty + s), (uint32_t)(u & 1) ^ 1u, spin, abort, p.st, kSiteTProducer);
        if (!ok) break;
        const uint32_t dst = base + (uint32_t)s * stage;
        mbar_arrive_expect_tx(bar(kBarFull + s), stage);
        if (p.wide) {
          // two 64-column chunks per operand, each operand one 4-D box
          if (c < nq) {
            tma_load_4d(dst, &tmap_q4, bar(kBarFull + s), 0, i0, 2 * c, bh);
            tma_load_4d(dst + stage / 2, &tmap_k4, bar(kBarFull + s), 0, j0, 2 * c, bh);
          } else {
            tma_load_4d(dst, &tmap_dh4, bar(kBarFull + s), 0, i0, 2 * (c - nq), bh);
            tma_load_4d(dst + stage / 2, &tmap_v4, bar(kBarFull + s), 0, j0, 2 * (c - nq), bh);
          }
        } else if (c < nq) {
          tma_load_3d(dst, &tmap_q, bar(kBarFull + s), 64 * c, i0, bh);
          tma_load_3d(dst + stage / 2, &tmap_k, bar(kBarFull + s), 64 * c, j0, bh);
        } else {
          tma_load_3d(dst, &tmap_dh, bar(kBarFull + s), 64 * (c - nq), i0, bh);
          tma_load_3d(dst + stage / 2, &tmap_v, bar(kBarFull + s), 64 * (c - nq), j0, bh);
        }
        issued_s = cc + 1;
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = idesc_bf16_f32(kTile, kTile, 0, 0);
    int cc = 0, li = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < p.nitems && ok; it += gridDim.x, ++li) {
      const int b = li & 1, ub = li >> 1;
      // the epilogue has read this buffer's previous tile
      ok = mbar_wait(bar(kBarAccEmpty + b), (uint32_t)(ub & 1) ^ 1u, spin, abort, p.st, kSiteTMma);
      if (!ok) break;
      tc_fence_after();
      for (int c = 0; c < nch && ok; ++c, ++cc) {
        const int s = cc % nst, u = cc / nst;
        ok = mbar_wait(bar(kBarFull + s), (uint32_t)(u & 1), spin, abort, p.st, kSiteTMma);
        if (!ok) break;
        tc_fence_after();
        const uint32_t a_addr = base + (uint32_t)s * stage;
        const uint32_t d = tmem + 256u * (uint32_t)b + (c < nq ? 0u : 128u);
        const bool first = c == 0 || c == nq;
        // one or two K-major 128-byte-swizzle atoms (64 columns each, 16 KB apart)
        for (int at = 0; at < (p.wide ? 2 : 1); ++at) {
          const uint64_t da = smem_desc_sw128(a_addr + (uint32_t)at * 16384u, 16, 1024);
          const uint64_t db = smem_desc_sw128(a_addr + stage / 2 + (uint32_t)at * 16384u, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ss(d, da + 2 * kk, db + 2 * kk, idesc, (first && at == 0 && kk == 0) ? 0u : 1u);
        }
        mma_commit(bar(kBarEmpty + s));
      }
      if (ok) mma_commit(bar(kBarAccFull + b));
    }
    mma_commit(bar(kBarDrain));
    for (long long w = 0; w < kDrainSpin; ++w)
      if (mbar_try_wait(bar(kBarDrain), 0)) break;
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    // eight warps: warp w reads TMEM lane quarter w % 4 (rows 32 (w % 4) ..),
    // columns 64 h .. 64 h + 63 with h = (w - 2) / 4
    const int et = threadIdx.x - 64;               // 0..255; et < 128: a column of the column terms
    const int qd = warp & 3, hf = (warp - 2) >> 2;
    const int r = 32 * qd + lane;                  // tile row = TMEM lane
    const uint32_t lane_addr = (uint32_t)(32 * qd) << 16;
    int li = 0;
    for (int it = blockIdx.x;; it += gridDim.x, ++li) {
      // every thread of the group passes each barrier of an item, abort or not
      if (et == 0) {
        tma_store_wait_read();                      // the staging buffer is free again
        epi_stop = it >= p.nitems || *abort;
      }
      named_bar_sync(1, 256);
      if (epi_stop) break;
      int bh, ib, jb;
      tile_of(it, nb, &bh, &ib, &jb);
      const int i0 = ib * kTile, j0 = jb * kTile;
      const int i = i0 + r;
      const bool row_ok = i < p.T;
      const size_t hb = (size_t)bh * p.T;
      const bool diag = jb == ib;
      const int jc = j0 + (et & 127);
      const float a2c = (et < 128 && jc < p.T) ? p.a2[hb + jc] : -INFINITY;
      const float p2i = row_ok ? p.p2[hb + i] : 0.0f;
      const float invn = row_ok ? p.invn[hb + i] : 0.0f;
      const float dbi = row_ok ? p.db[hb + i] : 0.0f;
      const float pscale = invn * p.scale;           // P = S_raw s D' / n
      float rowf = 0.0f;
      if (diag) {
        if (et < 128) col_term[et] = a2c;
      } else {
        // rank-one gate factor: D'_ij = 2^(a2_j - A) 2^(A - p2_i), A the tile's
        // largest column term (every key of the tile precedes every query row)
        const float m = warp_max(a2c);
        if (lane == 0 && et < 128) amax_red[warp - 2] = m;
        named_bar_sync(1, 256);
        const float A = fmaxf(fmaxf(amax_red[0], amax_red[1]), fmaxf(amax_red[2], amax_red[3]));
        if (et < 128) col_term[et] = exp2f(a2c - A);
        rowf = row_ok ? exp2f(A - p2i) : 0.0f;
      }
      named_bar_sync(1, 256);                        // column terms visible
      const int b = li & 1, ub = li >> 1;
      // warp-uniform: the TMEM loads and shuffles below are warp-collective
      const bool ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarAccFull + b), (uint32_t)(ub & 1), spin, abort,
                                                        p.st, kSiteTEpi));
      tc_fence_after();
      float rs = 0.0f;                               // S_raw (.) G over this warp's columns
      if (ok) {
        uint32_t sv[2][32], cv[2][32];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          tmem_ld32(tmem + lane_addr + 256u * (uint32_t)b + 64 * hf + 32 * u, sv[u]);
          tmem_ld32(tmem + lane_addr + 256u * (uint32_t)b + 128 + 64 * hf + 32 * u, cv[u]);
        }
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarAccEmpty + b));   // the buffer is read: the products may reuse it
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int ch = 2 * hf + u;                 // 32-column chunk of the tile
          float dd[32];
          uint32_t gw[16], pw[16];
          if (diag)
            tile_values<true>(sv[u], cv[u], col_term + 32 * ch, j0 + 32 * ch, i, row_ok, p2i, rowf, invn, dbi,
                              pscale, dd, gw, pw, rs);
          else
            tile_values<false>(sv[u], cv[u], col_term + 32 * ch, j0 + 32 * ch, i, row_ok, p2i, rowf, invn, dbi,
                               pscale, dd, gw, pw, rs);
          // stage: columns 32ch..32ch+31 = 16-byte chunks 4(ch&1)..4(ch&1)+3 of box ch>>1
          const uint32_t gbox = sStage + (uint32_t)(ch >> 1) * 16384u;
          const uint32_t pbox = sStage + 32768u + (uint32_t)(ch >> 1) * 16384u;
#pragma unroll
          for (int g4 = 0; g4 < 4; ++g4) {
            const int q = 4 * (ch & 1) + g4;
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(swz(gbox, r, q)), "r"(gw[4 * g4]),
                         "r"(gw[4 * g4 + 1]), "r"(gw[4 * g4 + 2]), "r"(gw[4 * g4 + 3])
                         : "memory");
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(swz(pbox, r, q)), "r"(pw[4 * g4]),
                         "r"(pw[4 * g4 + 1]), "r"(pw[4 * g4 + 2]), "r"(pw[4 * g4 + 3])
                         : "memory");
          }
          // column sums over the warp's 32 rows: halving reduce-scatter; lane l
          // ends with column 32ch + l
#pragma unroll
          for (int o = 16, n = 32; o >= 1; o >>= 1, n >>= 1) {
            const bool hi = lane & o;
            if (n >= 4) {
#pragma unroll
              for (int k2 = 0; k2 < n / 2; k2 += 2) {       // two columns per packed add
                const f32x2 keep = hi ? f2_make(dd[k2 + n / 2], dd[k2 + 1 + n / 2]) : f2_make(dd[k2], dd[k2 + 1]);
                const float s0 = hi ? dd[k2] : dd[k2 + n / 2], s1 = hi ? dd[k2 + 1] : dd[k2 + 1 + n / 2];
                const float2 sum = f2_split(f2_add(keep, f2_make(__shfl_xor_sync(0xffffffffu, s0, o),
                                                                 __shfl_xor_sync(0xffffffffu, s1, o))));
                dd[k2] = sum.x;
                dd[k2 + 1] = sum.y;
              }
            } else {
              const float keep = hi ? dd[1] : dd[0];
              const float send = hi ? dd[0] : dd[1];
              dd[0] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
          }
          col_red[qd][32 * ch + lane] = dd[0];
        }
        row_red[hf][r] = rs;
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 256);                        // staging and partial sums complete
      if (ok) {
        if (et < 128) {
          if (jc < p.T)
            p.Cpart[((size_t)bh * nb + ib) * p.T + jc] =
                p.scale * (col_red[0][et] + col_red[1][et] + col_red[2][et] + col_red[3][et]);
          if (i0 + et < p.T) p.Rpart[((size_t)bh * nb + jb) * p.T + i0 + et] = p.scale * (row_red[0][et] + row_red[1][et]);
        }
        if (et == 0) {
          for (int b2 = 0; b2 < 2 && j0 + 64 * b2 < p.T; ++b2) {   // boxes that start inside the matrix
            tma_store_3d(&tmap_g, sStage + (uint32_t)b2 * 16384u, j0 + 64 * b2, i0, bh);
            tma_store_3d(&tmap_p, sStage + 32768u + (uint32_t)b2 * 16384u, j0 + 64 * b2, i0, bh);
          }
          tma_store_commit();
        }
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  // after an abort, loads may still be landing: wait (bounded) for the last
  // round of every slot
  if (threadIdx.x == 0 && abort_flag) {
    const int issued = issued_s;
    for (int c = max(0, issued - nst); c < issued; ++c)
      for (long long w = 0; w < kDrainSpin; ++w)
        if (mbar_try_wait(bar(kBarFull + c % nst), (uint32_t)((c / nst) & 1))) break;
  }
}

// ---------------------------------------------------------------- products
// The three products of eqs (98)-(100) over the lower triangle of G and P,
// one CTA per (product, head, 128-row output block g):
//   dQ_g = s sum_{kb <= g} G[g, kb] K[kb]       A = G block, K-major
//   dK_g = s sum_{ib >= g} G[ib, g]^T Q[ib]     A = G^T block, MN-major
//   dV_g =   sum_{ib >= g} P[ib, g]^T dH[ib]    A = P^T block, MN-major
// B (K, Q or dH rows) is MN-major.  The 128 x d accumulator sits in TMEM
// (d <= 512 columns); A blocks come through a two-slot ring, B through a
// four-slot ring of 128-column chunks.  CTAs run head by head, longest first
// within a head.
constexpr int kPThreads = 192;          // warp 0 TMA, warp 1 MMA + TMEM, warps 2..5 epilogue
constexpr int kANst = 2, kBNst = 4;
constexpr uint32_t kABytes = 32768, kBBytes = 32768;
enum : int {
  kPBarAFull = 0, kPBarAEmpty = kANst, kPBarBFull = 2 * kANst, kPBarBEmpty = 2 * kANst + kBNst,
  kPBarDone = 2 * kANst + 2 * kBNst, kPBarDrain = kPBarDone + 1, kPNumBars = kPBarDone + 2
};
enum : int { kSitePProducer = 44, kSitePMma = 45, kSitePEpi = 46 };

struct ProdParams {
  int T, BH, nb, dqk, dv;
  int a4;                    // CTA pairs: A blocks load through their 4-D view (T a multiple of 64)
  float scale;
  DevStatus st;
};

__global__ void __launch_bounds__(kPThreads, 1)
bwd_prod_kernel(const __grid_constant__ CUtensorMap tmap_g, const __grid_constant__ CUtensorMap tmap_p,
                const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
                const __grid_constant__ CUtensorMap tmap_dh, const __grid_constant__ CUtensorMap tmap_dq,
                const __grid_constant__ CUtensorMap tmap_dk, const __grid_constant__ CUtensorMap tmap_dv,
                const ProdParams p) {
  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t bars[kPNumBars];
  __shared__ uint32_t tmem_holder;
  __shared__ int abort_flag;
  __shared__ int a_issued_s, b_issued_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &abort_flag;

  // work item: head-major (the CTAs in flight share a few heads' G, P, K, Q,
  // dH in L2), within a head longest first: rank w sums nb - w blocks
  const int bh = (int)(blockIdx.x / (3u * (unsigned)p.nb));
  const int w = (int)((blockIdx.x % (3u * (unsigned)p.nb)) / 3u);
  const int prod = (int)(blockIdx.x % 3u);
  const int nkb = p.nb - w;                                  // blocks in the sum
  const int g = prod == 0 ? p.nb - 1 - w : w;                // output row block
  const int kb0 = prod == 0 ? 0 : g;                         // first summed block
  const int r0 = g * kTile;
  const int d = prod == 2 ? p.dv : p.dqk;
  const int nbox = (d + 63) / 64, nchunk = (nbox + 1) / 2;   // 64-column boxes, 128-column chunks
  const CUtensorMap* ma = prod == 2 ? &tmap_p : &tmap_g;
  const CUtensorMap* mb = prod == 0 ? &tmap_k : (prod == 1 ? &tmap_q : &tmap_dh);
  const CUtensorMap* mo = prod == 0 ? &tmap_dq : (prod == 1 ? &tmap_dk : &tmap_dv);
  const float alpha = prod == 2 ? 1.0f : p.scale;
  const uint32_t base = (smem_u32(dsmem) + 1023u) & ~1023u;
  const uint32_t sA = base, sB = base + kANst * kABytes;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  if (threadIdx.x == 0) {
    abort_flag = 0;
    a_issued_s = 0;
    b_issued_s = 0;
    for (int s2 = 0; s2 < kANst; ++s2) {
      mbar_init(bar(kPBarAFull + s2), 1);
      mbar_init(bar(kPBarAEmpty + s2), 1);
    }
    for (int s2 = 0; s2 < kBNst; ++s2) {
      mbar_init(bar(kPBarBFull + s2), 1);
      mbar_init(bar(kPBarBEmpty + s2), 1);
    }
    mbar_init(bar(kPBarDone), 1);
    mbar_init(bar(kPBarDrain), 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_holder;
  const long long spin = p.st.spin_limit;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    tma_prefetch_desc(ma);
    tma_prefetch_desc(mb);
    int bi = 0;
    bool ok = true;
    for (int t = 0; t < nkb && ok; ++t) {
      const int kb = kb0 + t;
      const int as = t % kANst, au = t / kANst;
      ok = mbar_wait(bar(kPBarAEmpty + as), (uint32_t)(au & 1) ^ 1u, spin, abort, p.st, kSitePProducer);
      if (!ok) break;
      mbar_arrive_expect_tx(bar(kPBarAFull + as), kABytes);
      const uint32_t adst = sA + (uint32_t)as * kABytes;
      for (int h = 0; h < 2; ++h) {
        if (prod == 0)   // G[g rows, kb keys]: keys 128kb + 64h ..
          tma_load_3d(adst + h * 16384u, ma, bar(kPBarAFull + as), kb * kTile + 64 * h, r0, bh);
        else             // G[kb rows, g keys]^T: keys r0 + 64h .. as the M half h
          tma_load_3d(adst + h * 16384u, ma, bar(kPBarAFull + as), r0 + 64 * h, kb * kTile, bh);
      }
      a_issued_s = t + 1;
      for (int c = 0; c < nchunk && ok; ++c, ++bi) {
        const int bs = bi % kBNst, bu = bi / kBNst;
        ok = mbar_wait(bar(kPBarBEmpty + bs), (uint32_t)(bu & 1) ^ 1u, spin, abort, p.st, kSitePProducer);
        if (!ok) break;
        const int nb2 = min(2, nbox - 2 * c);
        mbar_arrive_expect_tx(bar(kPBarBFull + bs), (uint32_t)nb2 * 16384u);
        for (int h = 0; h < nb2; ++h)
          tma_load_3d(sB + (uint32_t)bs * kBBytes + h * 16384u, mb, bar(kPBarBFull + bs), 64 * (2 * c + h),
                      kb * kTile, bh);
        b_issued_s = bi + 1;
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t a_mn = prod == 0 ? 0u : 1u;
    const uint32_t id128 = idesc_bf16_f32(kTile, 128, (int)a_mn, 1), id64 = idesc_bf16_f32(kTile, 64, (int)a_mn, 1);
    int bi = 0;
    bool ok = true;
    for (int t = 0; t < nkb && ok; ++t) {
      const int as = t % kANst, au = t / kANst;
      ok = mbar_wait(bar(kPBarAFull + as), (uint32_t)(au & 1), spin, abort, p.st, kSitePMma);
      if (!ok) break;
      tc_fence_after();
      const uint32_t aaddr = sA + (uint32_t)as * kABytes;
      // K-major A: two 64-key boxes, 32 B per 16-key step within a box;
      // MN-major A: two 64-row M halves 16 KB apart, 2 KB per 16-key step
      const uint64_t da = prod == 0 ? smem_desc_sw128(aaddr, 16, 1024) : smem_desc_sw128(aaddr, 16384, 1024);
      for (int c = 0; c < nchunk && ok; ++c, ++bi) {
        const int bs = bi % kBNst, bu = bi / kBNst;
        ok = mbar_wait(bar(kPBarBFull + bs), (uint32_t)(bu & 1), spin, abort, p.st, kSitePMma);
        if (!ok) break;
        tc_fence_after();
        const uint64_t dbd = smem_desc_sw128(sB + (uint32_t)bs * kBBytes, 16384, 1024);
        const uint32_t idesc = nbox - 2 * c >= 2 ? id128 : id64;
        const uint32_t dcol = tmem + 128u * (uint32_t)c;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ak = prod == 0 ? da + (uint64_t)((kk >> 2) * 1024 + (kk & 3) * 2) : da + (uint64_t)(kk * 128);
          mma_bf16_ss(dcol, ak, dbd + (uint64_t)(kk * 128), idesc, (t | kk) != 0 ? 1u : 0u);
        }
        mma_commit(bar(kPBarBEmpty + bs));
      }
      if (ok) mma_commit(bar(kPBarAEmpty + as));
    }
    if (ok) mma_commit(bar(kPBarDone));
    mma_commit(bar(kPBarDrain));
    for (long long w2 = 0; w2 < kDrainSpin; ++w2)
      if (mbar_try_wait(bar(kPBarDrain), 0)) break;
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    const int qd = warp & 3, r = 32 * qd + lane;
    const uint32_t lane_addr = (uint32_t)(32 * qd) << 16;
    // warp-uniform: the TMEM loads below are warp-collective
    const bool ok = __all_sync(0xffffffffu, mbar_wait(bar(kPBarDone), 0, spin, abort, p.st, kSitePEpi));
    tc_fence_after();
    if (ok) {
      // stage the bf16 block in 64-column boxes over the (now idle) rings
      for (int c32 = 0; c32 < 2 * nbox; ++c32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_addr + 32 * c32, v);
        tmem_wait_ld();
        const uint32_t box = base + (uint32_t)(c32 >> 1) * 16384u;
#pragma unroll
        for (int g4 = 0; g4 < 4; ++g4) {
          uint32_t wv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            wv[e] = pack_bf16x2(__uint_as_float(v[8 * g4 + 2 * e]) * alpha, __uint_as_float(v[8 * g4 + 2 * e + 1]) * alpha);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(swz(box, r, 4 * (c32 & 1) + g4)),
                       "r"(wv[0]), "r"(wv[1]), "r"(wv[2]), "r"(wv[3])
                       : "memory");
        }
      }
      fence_proxy_async_smem();
    }
    tc_fence_before();
    named_bar_sync(1, 128);
    if (ok && threadIdx.x == 64) {
      for (int b2 = 0; b2 < nbox; ++b2) tma_store_3d(mo, base + (uint32_t)b2 * 16384u, 64 * b2, r0, bh);
      tma_store_commit();
      tma_store_wait_read();
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && abort_flag) {
    // loads may still be landing: wait (bounded) for the last round of every slot
    const int ai = a_issued_s, bi = b_issued_s;
    for (int c = max(0, ai - kANst); c < ai; ++c)
      for (long long w2 = 0; w2 < kDrainSpin; ++w2)
        if (mbar_try_wait(bar(kPBarAFull + c % kANst), (uint32_t)((c / kANst) & 1))) break;
    for (int c = max(0, bi - kBNst); c < bi; ++c)
      for (long long w2 = 0; w2 < kDrainSpin; ++w2)
        if (mbar_try_wait(bar(kPBarBFull + c % kBNst), (uint32_t)((c / kBNst) & 1))) break;
  }
}

// ---------------------------------------------------------------- products on CTA pairs
// The same three products with M = 256 on a cluster of two CTAs (tcgen05
// cta_group::2): CTA rank r owns output block 2 gp + r of a block pair gp and
// holds its own A blocks; the B chunk (K, Q or dH rows) is split by columns
// between the two CTAs, so each SM loads half of the B bytes a single-CTA
// block needs.  A pair sums over the union of its two blocks' ranges; the
// extra block reads the tile (2 gp, 2 gp + 1) above the diagonal, which
// the row-statistics launch stores as zeros.  Requires d_qk and d_v multiples of
// 128 (a B chunk is 256 columns, or 128 for the last, split in halves).
__global__ void __launch_bounds__(kPThreads, 1)
bwd_prod2_kernel(const __grid_constant__ CUtensorMap tmap_g, const __grid_constant__ CUtensorMap tmap_p,
                 const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
                 const __grid_constant__ CUtensorMap tmap_dh, const __grid_constant__ CUtensorMap tmap_dq,
                 const __grid_constant__ CUtensorMap tmap_dk, const __grid_constant__ CUtensorMap tmap_dv,
                 const __grid_constant__ CUtensorMap tmap_g4, const __grid_constant__ CUtensorMap tmap_p4,
                 const __grid_constant__ CUtensorMap tmap_k4, const __grid_constant__ CUtensorMap tmap_q4,
                 const __grid_constant__ CUtensorMap tmap_dh4, const ProdParams p) {
  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t bars[kPNumBars];
  __shared__ uint32_t tmem_holder;
  __shared__ int abort_flag;
  __shared__ int a_issued_s, b_issued_s;
  __shared__ int peer_s[3];                  // (leader) the peer's A and B load counts and abort flag, sent at exit
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &abort_flag;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  // work item of the pair: head-major, longest first within a head
  const int np = (p.nb + 1) / 2;
  const int cid = (int)(blockIdx.x >> 1);
  const int bh = cid / (3 * np);
  const int w = (cid % (3 * np)) / 3;
  const int prod = cid % 3;
  const int gp = prod == 0 ? np - 1 - w : w;
  const int g0 = 2 * gp, gr = g0 + (int)rank;                // this CTA's output block
  const int kb0 = prod == 0 ? 0 : g0;
  const int nkb = prod == 0 ? min(g0 + 2, p.nb) : p.nb - g0;
  const int r0 = gr * kTile;
  const int d = prod == 2 ? p.dv : p.dqk;
  const int nbox = d / 64;                                   // a multiple of 2
  const int nchunk = (nbox + 3) / 4;                         // 256-column chunks (the last may be 128)
  const CUtensorMap* ma = prod == 2 ? &tmap_p : &tmap_g;
  const CUtensorMap* mb = prod == 0 ? &tmap_k : (prod == 1 ? &tmap_q : &tmap_dh);
  const CUtensorMap* mo = prod == 0 ? &tmap_dq : (prod == 1 ? &tmap_dk : &tmap_dv);
  const float alpha = prod == 2 ? 1.0f : p.scale;
  // the A and B operands as 4-D views: one box of two 64-column blocks (the A
  // view only when T is a multiple of 64, p.a4)
  const CUtensorMap* ma4 = prod == 2 ? &tmap_p4 : &tmap_g4;
  const CUtensorMap* mb4 = prod == 0 ? &tmap_k4 : (prod == 1 ? &tmap_q4 : &tmap_dh4);
  const uint32_t base = (smem_u32(dsmem) + 1023u) & ~1023u;
  const uint32_t sA = base, sB = base + kANst * kABytes;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  auto lbar = [&](int i) { return mapa_shared(smem_u32(&bars[i]), 0); };   // the leader's barrier

  if (threadIdx.x == 0) {
    abort_flag = 0;
    a_issued_s = 0;
    b_issued_s = 0;
    for (int s2 = 0; s2 < kANst; ++s2) {
      mbar_init(bar(kPBarAFull + s2), 1);
      mbar_init(bar(kPBarAEmpty + s2), 1);
    }
    for (int s2 = 0; s2 < kBNst; ++s2) {
      mbar_init(bar(kPBarBFull + s2), 1);
      mbar_init(bar(kPBarBEmpty + s2), 1);
    }
    mbar_init(bar(kPBarDone), 1);
    mbar_init(bar(kPBarDrain), 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&tmem_holder), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();                        // peer barriers initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = tmem_holder;
  const long long spin = p.st.spin_limit;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producers (both CTAs)
    // Each CTA loads its own A blocks and its half of every B chunk into its
    // own buffers; completion is counted on the leader's full barriers, whose
    // expected bytes (both CTAs) only the leader posts.
    tma_prefetch_desc(ma);
    tma_prefetch_desc(mb);
    tma_prefetch_desc(ma4);
    tma_prefetch_desc(mb4);
    int bi = 0;
    bool ok = true;
    for (int t = 0; t < nkb && ok; ++t) {
      const int kb = kb0 + t;
      const int as = t % kANst, au = t / kANst;
      ok = mbar_wait(bar(kPBarAEmpty + as), (uint32_t)(au & 1) ^ 1u, spin, abort, p.st, kSitePProducer);
      if (!ok) break;
      if (leader) mbar_arrive_expect_tx(bar(kPBarAFull + as), 2u * kABytes);
      const uint32_t adst = sA + (uint32_t)as * kABytes;
      if (p.a4) {        // the block's two 64-column halves in one copy
        if (prod == 0) tma_load_4d_pair(adst, ma4, lbar(kPBarAFull + as), 0, r0, 2 * kb, bh);
        else tma_load_4d_pair(adst, ma4, lbar(kPBarAFull + as), 0, kb * kTile, r0 / 64, bh);
      } else {
        for (int h = 0; h < 2; ++h) {
          if (prod == 0)   // G[gr rows, kb keys]
            tma_load_3d_pair(adst + h * 16384u, ma, lbar(kPBarAFull + as), kb * kTile + 64 * h, r0, bh);
          else             // G[kb rows, gr keys]^T
            tma_load_3d_pair(adst + h * 16384u, ma, lbar(kPBarAFull + as), r0 + 64 * h, kb * kTile, bh);
        }
      }
      a_issued_s = t + 1;
      for (int c = 0; c < nchunk && ok; ++c, ++bi) {
        const int bs = bi % kBNst, bu = bi / kBNst;
        ok = mbar_wait(bar(kPBarBEmpty + bs), (uint32_t)(bu & 1) ^ 1u, spin, abort, p.st, kSitePProducer);
        if (!ok) break;
        const bool wide = nbox - 4 * c >= 4;            // 256 columns: two boxes a CTA, else one
        const int col0 = 256 * c;
        if (leader) mbar_arrive_expect_tx(bar(kPBarBFull + bs), 2u * (wide ? 32768u : 16384u));
        if (wide) {       // this CTA's two 64-column blocks in one copy
          tma_load_4d_pair(sB + (uint32_t)bs * kBBytes, mb4, lbar(kPBarBFull + bs), 0, kb * kTile,
                           (col0 + 128 * (int)rank) / 64, bh);
        } else {
          tma_load_3d_pair(sB + (uint32_t)bs * kBBytes, mb, lbar(kPBarBFull + bs), col0 + 64 * (int)rank,
                           kb * kTile, bh);
        }
        b_issued_s = bi + 1;
      }
    }
  } else if (warp == 1 && lane == 0 && leader) {
    // ------------------------------------------------------------ MMA issuer (leader)
    const uint32_t a_mn = prod == 0 ? 0u : 1u;
    const uint32_t id256 = idesc_bf16_f32(2 * kTile, 256, (int)a_mn, 1), id128 = idesc_bf16_f32(2 * kTile, 128, (int)a_mn, 1);
    int bi = 0;
    bool ok = true;
    for (int t = 0; t < nkb && ok; ++t) {
      const int as = t % kANst, au = t / kANst;
      ok = mbar_wait(bar(kPBarAFull + as), (uint32_t)(au & 1), spin, abort, p.st, kSitePMma);
      if (!ok) break;
      tc_fence_after();
      const uint32_t aaddr = sA + (uint32_t)as * kABytes;
      const uint64_t da = prod == 0 ? smem_desc_sw128(aaddr, 16, 1024) : smem_desc_sw128(aaddr, 16384, 1024);
      for (int c = 0; c < nchunk && ok; ++c, ++bi) {
        const int bs = bi % kBNst, bu = bi / kBNst;
        ok = mbar_wait(bar(kPBarBFull + bs), (uint32_t)(bu & 1), spin, abort, p.st, kSitePMma);
        if (!ok) break;
        tc_fence_after();
        const uint64_t dbd = smem_desc_sw128(sB + (uint32_t)bs * kBBytes, 16384, 1024);
        const uint32_t idesc = nbox - 4 * c >= 4 ? id256 : id128;
        const uint32_t dcol = tmem + 256u * (uint32_t)c;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ak = prod == 0 ? da + (uint64_t)((kk >> 2) * 1024 + (kk & 3) * 2) : da + (uint64_t)(kk * 128);
          mma_bf16_ss_pair(dcol, ak, dbd + (uint64_t)(kk * 128), idesc, (t | kk) != 0 ? 1u : 0u);
        }
        mma_commit_pair_mc(bar(kPBarBEmpty + bs), 0x3);
      }
      if (ok) mma_commit_pair_mc(bar(kPBarAEmpty + as), 0x3);
    }
    if (ok) mma_commit_pair_mc(bar(kPBarDone), 0x3);
    mma_commit_pair(bar(kPBarDrain));
    for (long long w2 = 0; w2 < kDrainSpin; ++w2)
      if (mbar_try_wait(bar(kPBarDrain), 0)) break;
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue (both CTAs, own rows)
    const int qd = warp & 3, r = 32 * qd + lane;
    const uint32_t lane_addr = (uint32_t)(32 * qd) << 16;
    // warp-uniform: the TMEM loads below are warp-collective
    const bool ok = __all_sync(0xffffffffu, mbar_wait(bar(kPBarDone), 0, spin, abort, p.st, kSitePEpi));
    tc_fence_after();
    const bool store = ok && r0 < p.T;
    if (store) {
      // stage the bf16 block in 64-column boxes over the (now idle) rings
      for (int c32 = 0; c32 < 2 * nbox; ++c32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_addr + 32 * c32, v);
        tmem_wait_ld();
        const uint32_t box = base + (uint32_t)(c32 >> 1) * 16384u;
#pragma unroll
        for (int g4 = 0; g4 < 4; ++g4) {
          uint32_t wv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            wv[e] = pack_bf16x2(__uint_as_float(v[8 * g4 + 2 * e]) * alpha, __uint_as_float(v[8 * g4 + 2 * e + 1]) * alpha);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(swz(box, r, 4 * (c32 & 1) + g4)),
                       "r"(wv[0]), "r"(wv[1]), "r"(wv[2]), "r"(wv[3])
                       : "memory");
        }
      }
      fence_proxy_async_smem();
    }
    tc_fence_before();
    named_bar_sync(1, 128);
    if (store && threadIdx.x == 64) {
      for (int b2 = 0; b2 < nbox; ++b2) tma_store_3d(mo, base + (uint32_t)b2 * 16384u, 64 * b2, r0, bh);
      tma_store_commit();
      tma_store_wait_read();
    }
  }

  __syncthreads();
  // Every issuer of both CTAs has stopped.  The peer sends the leader its
  // load counts and abort flag; after an abort in either CTA the leader makes
  // the last phase of every slot complete exactly when the loads issued for
  // it (by either CTA; the two counts differ by at most one round, as every
  // round waits for the previous one to be consumed) have landed, and waits
  // (bounded), so no copy can still write shared memory once the pair exits.
  if (!leader && threadIdx.x < 3) {
    const int v = threadIdx.x == 0 ? a_issued_s : (threadIdx.x == 1 ? b_issued_s : abort_flag);
    st_shared_cluster_u32(mapa_shared(smem_u32(&peer_s[threadIdx.x]), 0), (uint32_t)v);
  }
  cluster_sync_all();
  if (threadIdx.x == 0 && leader && (abort_flag || peer_s[2])) {
    const int ai[2] = {a_issued_s, peer_s[0]}, bi[2] = {b_issued_s, peer_s[1]};
    // rounds of slot s among the first n loads of a ring of ns slots
    auto rounds = [](int n, int s, int ns) { return n > s ? (n - 1 - s) / ns + 1 : 0; };
    for (int s2 = 0; s2 < kANst; ++s2) {
      const int fl = rounds(ai[0], s2, kANst), fp = rounds(ai[1], s2, kANst), f = max(fl, fp);
      settle_last_phase(bar(kPBarAFull + s2), f, fl == f, 2u * kABytes,
                        (fl == f ? kABytes : 0u) + (fp == f ? kABytes : 0u), kDrainSpin);
    }
    for (int s2 = 0; s2 < kBNst; ++s2) {
      const int fl = rounds(bi[0], s2, kBNst), fp = rounds(bi[1], s2, kBNst), f = max(fl, fp);
      if (f == 0) continue;
      const int c = ((f - 1) * kBNst + s2) % nchunk;           // the chunk of the last round
      const uint32_t half = nbox - 4 * c >= 4 ? 32768u : 16384u;
      settle_last_phase(bar(kPBarBFull + s2), f, fl == f, 2u * half, (fl == f ? half : 0u) + (fp == f ? half : 0u),
                        kDrainSpin);
    }
  }
  // both CTAs are done with TMEM and with each other's shared memory
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

// G and P tiles (ib, ib + 1) for even ib, above the diagonal: zeros (the
// extra block a product pair reads).  One block per tile.
__device__ void bwd_zero_tile(__nv_bfloat16* __restrict__ G, __nv_bfloat16* __restrict__ P, int T, int ldT, int nb,
                              int tile) {
  const int np = nb / 2;                     // tiles (2 gp, 2 gp + 1) with 2 gp + 1 < nb
  const int bh = tile / np, gp = tile % np;
  const int i0 = 2 * gp * kTile, j0 = i0 + kTile;
  const int rows = min(kTile, T - i0), cols8 = (min(kTile, ldT - j0) + 7) / 8;
  for (int x = threadIdx.x; x < rows * cols8; x += blockDim.x) {
    const int rr = x / cols8, c8 = x % cols8;
    const size_t off = ((size_t)bh * T + i0 + rr) * ldT + j0 + 8 * c8;
    *reinterpret_cast<uint4*>(G + off) = make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint4*>(P + off) = make_uint4(0u, 0u, 0u, 0u);
  }
}

// Per row: 1/n_i and db_i (eqs 89-90) from the forward's H~, n, signed b and
// the row max m.  Sixteen threads per row, every load of a row issued before
// the first product (16-byte loads of bf16 where rows allow).  Blocks past
// the rows' (zero_base and on) instead zero the tiles above the diagonal that
// a product pair reads (one tile each; see bwd_zero_tile).
template <typename E>
__global__ void __launch_bounds__(256)
bwd_rowstat_kernel(const E* __restrict__ dh, const E* __restrict__ h, const float* __restrict__ nrow,
                   const float* __restrict__ brow, const float* __restrict__ mrow, float* __restrict__ invn,
                   float* __restrict__ db, int dv, long long BHT, unsigned zero_base, __nv_bfloat16* G,
                   __nv_bfloat16* P, int T, int ldT, int nb) {
  if (blockIdx.x >= zero_base) {
    bwd_zero_tile(G, P, T, ldT, nb, (int)(blockIdx.x - zero_base));
    return;
  }
  const long long row = (long long)blockIdx.x * 16 + (threadIdx.x >> 4);
  const int l16 = threadIdx.x & 15;
  const bool live = row < BHT;
  float dot = 0.0f;
  if (sizeof(E) == 2 && dv % 8 == 0 && dv <= 512 && (((uintptr_t)dh | (uintptr_t)h) & 15u) == 0) {
    const uint4* a = reinterpret_cast<const uint4*>(dh + (size_t)(live ? row : 0) * dv);
    const uint4* b = reinterpret_cast<const uint4*>(h + (size_t)(live ? row : 0) * dv);
    uint4 xa[4], xb[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c8 = l16 + 16 * u;
      const bool in = live && c8 < dv / 8;
      xa[u] = in ? a[c8] : make_uint4(0u, 0u, 0u, 0u);
      xb[u] = in ? b[c8] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t xs[4] = {xa[u].x, xa[u].y, xa[u].z, xa[u].w}, ys[4] = {xb[u].x, xb[u].y, xb[u].z, xb[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fx = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xs[e]));
        const float2 fy = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ys[e]));
        dot = fmaf(fx.x, fy.x, dot);
        dot = fmaf(fx.y, fy.y, dot);
      }
    }
  } else if (live) {
    for (int c = l16; c < dv; c += 16)
      dot = fmaf(Elem<E>::load(dh, (size_t)row * dv + c), Elem<E>::load(h, (size_t)row * dv + c), dot);
  }
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);   // within the 16 lanes of a row
  if (live && l16 == 0) {
    const float n = nrow[row], b = brow[row];
    const float inv = n > 0.0f ? 1.0f / n : 0.0f;
    const float dn = -dot * inv;                                  // -(dH~ . h~) / n = -(sum C~' dC) / n^2
    invn[row] = inv;
    db[row] = fabsf(b) > expf(-mrow[row]) ? (b > 0.0f ? dn : (b < 0.0f ? -dn : 0.0f)) : 0.0f;
  }
}

// R_i = sum over key blocks jb <= ib(i) of the tile row sums; Ccol_j = sum
// over query blocks ib >= jb(j) of the tile column sums (fixed order).
__global__ void bwd_tile_sums_kernel(const float* __restrict__ Rpart, const float* __restrict__ Cpart,
                                     float* __restrict__ R, float* __restrict__ Ccol, int T, int nb, long long n) {
  const long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= n) return;
  const int bh = (int)(x / T), t = (int)(x % T);
  const int blk = t / kTile;
  float rsum = 0.0f, csum = 0.0f;
  // four loads in flight at a time; the additions keep the block order
  const float* rp = Rpart + (size_t)bh * nb * T + t;
  const float* cp = Cpart + (size_t)bh * nb * T + t;
  for (int b2 = 0; b2 <= blk; b2 += 4) {
    float v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = b2 + u <= blk ? rp[(size_t)(b2 + u) * T] : 0.0f;
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (b2 + u <= blk) rsum += v[u];
  }
  for (int b2 = blk; b2 < nb; b2 += 4) {
    float v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = b2 + u < nb ? cp[(size_t)(b2 + u) * T] : 0.0f;
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (b2 + u < nb) csum += v[u];
  }
  R[x] = rsum;
  Ccol[x] = csum;
}

}  // namespace

// The products run on CTA pairs when d_qk and d_v are multiples of 128
// (MLSTM_BWD_PROD=single forces one CTA per block, for the tests).
bool bwd_prod_pairs(int dqk, int dv) {
  static const char* force = getenv("MLSTM_BWD_PROD");
  return dqk % 128 == 0 && dv % 128 == 0 && !(force && force[0] == 's');
}

int launch_bwd_products(const BwdProdArgs& a, cudaStream_t stream) {
  if (a.BH <= 0 || a.T <= 0) return kOk;
  const int nb = (a.T + kTile - 1) / kTile;
  const long long grid = 3LL * a.BH * nb;
  if (grid > 0x7fffffffLL) return kInval;
  CUtensorMap mg, mp, mk, mq, mdh, mdq, mdk, mdv;
  if (!make_map_ld(&mg, a.G, a.T, a.T, a.BH, a.ldT, kTile) || !make_map_ld(&mp, a.P, a.T, a.T, a.BH, a.ldT, kTile) ||
      !make_map(&mk, a.k, a.dqk, a.T, a.BH, kTile) || !make_map(&mq, a.q, a.dqk, a.T, a.BH, kTile) ||
      !make_map(&mdh, a.dh, a.dv, a.T, a.BH, kTile) || !make_map(&mdq, a.dq, a.dqk, a.T, a.BH, kTile) ||
      !make_map(&mdk, a.dk, a.dqk, a.T, a.BH, kTile) || !make_map(&mdv, a.dvo, a.dv, a.T, a.BH, kTile))
    return kCuda;
  ProdParams p;
  p.T = a.T; p.BH = a.BH; p.nb = nb; p.dqk = a.dqk; p.dv = a.dv; p.scale = a.scale; p.st = a.st; p.a4 = 0;
  const size_t smem = (size_t)kANst * kABytes + (size_t)kBNst * kBBytes + 1024;
  if (bwd_prod_pairs(a.dqk, a.dv)) {
    // CTA pairs (the tiles above the diagonal that a pair's extra block reads
    // were zeroed with the row statistics)
    if (cudaFuncSetAttribute(bwd_prod2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return kCuda;
    // 4-D views: A blocks and wide B chunks as one box of two 64-column blocks
    // (an issuing thread handles its copies one after another)
    CUtensorMap mg4 = mg, mp4 = mp, mk4, mq4, mdh4;
    p.a4 = a.T % 64 == 0 && make_map_ld_blocks(&mg4, a.G, a.T, a.T, a.BH, a.ldT, kTile, 2) &&
           make_map_ld_blocks(&mp4, a.P, a.T, a.T, a.BH, a.ldT, kTile, 2);
    if (!p.a4) { mg4 = mg; mp4 = mp; }
    if (!make_map_blocks(&mk4, a.k, a.dqk, a.T, a.BH, kTile, 2) || !make_map_blocks(&mq4, a.q, a.dqk, a.T, a.BH, kTile, 2) ||
        !make_map_blocks(&mdh4, a.dh, a.dv, a.T, a.BH, kTile, 2))
      return kCuda;
    const long long pairs = 3LL * a.BH * ((nb + 1) / 2);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * pairs));
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, bwd_prod2_kernel, mg, mp, mk, mq, mdh, mdq, mdk, mdv, mg4, mp4, mk4, mq4, mdh4, p) !=
        cudaSuccess)
      return kCuda;
    return cudaGetLastError() == cudaSuccess ? kOk : kCuda;
  }
  if (cudaFuncSetAttribute(bwd_prod_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return kCuda;
  bwd_prod_kernel<<<(unsigned)grid, kPThreads, smem, stream>>>(mg, mp, mk, mq, mdh, mdq, mdk, mdv, p);
  return cudaGetLastError() == cudaSuccess ? kOk : kCuda;
}

bool bwd_tc_supported(int T, int dqk, int dv, int dtype) {
  return dtype == kBF16 && T >= 1 && dqk % 8 == 0 && dv % 8 == 0 && dqk <= 512 && dv <= 512;
}

int launch_bwd_tiles(const BwdTileArgs& a, cudaStream_t stream) {
  if (a.BH <= 0 || a.T <= 0) return kOk;
  if (!bwd_tc_supported(a.T, a.dqk, a.dv, kBF16) || !device_is_sm100_family()) return kUnsupported;
  const int nb = (a.T + kTile - 1) / kTile;
  const long long BHT = (long long)a.BH * a.T;
  const long long nitems = (long long)a.BH * (nb * (nb + 1) / 2);
  if (nitems > 0x7fffffffLL || (BHT + 7) / 8 > 0x7fffffffLL) return kInval;
  CUtensorMap mq, mk, mdh, mv, mg, mp;
  if (!make_map(&mq, a.q, a.dqk, a.T, a.BH, kTile) || !make_map(&mk, a.k, a.dqk, a.T, a.BH, kTile) ||
      !make_map(&mdh, a.dh, a.dv, a.T, a.BH, kTile) || !make_map(&mv, a.v, a.dv, a.T, a.BH, kTile) ||
      !make_map_ld(&mg, a.G, a.T, a.T, a.BH, a.ldT, kTile) || !make_map_ld(&mp, a.P, a.T, a.T, a.BH, a.ldT, kTile))
    return kCuda;
  // row statistics, plus (CTA-pair products) one block per tile above the
  // diagonal that a pair's extra block reads, zeroed
  const long long row_blocks = (BHT + 15) / 16;
  const long long zero_blocks = bwd_prod_pairs(a.dqk, a.dv) && nb >= 2 ? (long long)a.BH * (nb / 2) : 0;
  if (row_blocks + zero_blocks > 0x7fffffffLL) return kInval;
  bwd_rowstat_kernel<__nv_bfloat16><<<(unsigned)(row_blocks + zero_blocks), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(a.dh), static_cast<const __nv_bfloat16*>(a.h), a.nrow, a.brow, a.g.m,
      a.invn, a.db, a.dv, BHT, (unsigned)row_blocks, static_cast<__nv_bfloat16*>(a.G), static_cast<__nv_bfloat16*>(a.P),
      a.T, a.ldT, nb);
  if (cudaGetLastError() != cudaSuccess) return kCuda;
  TileParams p;
  p.a2 = a.g.a2; p.p2 = a.g.p2; p.invn = a.invn; p.db = a.db;
  p.Rpart = a.Rpart; p.Cpart = a.Cpart;
  p.T = a.T; p.BH = a.BH; p.dqk = a.dqk; p.dv = a.dv; p.nb = nb; p.nitems = (int)nitems;
  p.scale = a.scale; p.st = a.st;
  // 4-D views for two-chunk stages: one box per operand and stage instead of
  // two (an issuing thread handles its copies one after another)
  CUtensorMap mq4 = mq, mk4 = mk, mdh4 = mdh, mv4 = mv;
  p.wide = a.dqk % 64 == 0 && a.dv % 64 == 0 && make_map_blocks(&mq4, a.q, a.dqk, a.T, a.BH, kTile, 2) &&
           make_map_blocks(&mk4, a.k, a.dqk, a.T, a.BH, kTile, 2) && make_map_blocks(&mdh4, a.dh, a.dv, a.T, a.BH, kTile, 2) &&
           make_map_blocks(&mv4, a.v, a.dv, a.T, a.BH, kTile, 2);
  if (const char* e = getenv("MLSTM_BWD_TILE_NARROW")) p.wide = p.wide && e[0] == '0';   // (tuning)
  const size_t smem = (size_t)kNst * kStage + kStaging + 1024;
  if (cudaFuncSetAttribute(bwd_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return kCuda;
  int dev = 0, sms = 1;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return kCuda;
  const int grid = (int)std::min<long long>(nitems, sms);   // persistent: one CTA per SM
  bwd_tile_kernel<<<(unsigned)grid, kThreads, smem, stream>>>(mq, mk, mdh, mv, mg, mp, mq4, mk4, mdh4, mv4, p);
  if (cudaGetLastError() != cudaSuccess) return kCuda;
  bwd_tile_sums_kernel<<<(unsigned)((BHT + 255) / 256), 256, 0, stream>>>(a.Rpart, a.Cpart, a.R, a.Ccol, a.T, nb,
                                                                            BHT);
  return cudaGetLastError() == cudaSuccess ? kOk : kCuda;
}

}  // namespace mlstm
