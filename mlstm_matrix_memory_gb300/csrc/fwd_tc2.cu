// Fused causal mLSTM forward on a pair of SMs (tcgen05 cta_group::2).
//
// "xLSTM: Extended Long Short-Term Memory", part 28/30, stabilized parallel
// forward, eqs (79)-(86); same arithmetic as fwd_tc.cu (see there), different
// decomposition.  A cluster of two CTAs owns 256 consecutive query rows of one
// head (CTA rank r: rows 128r..128r+127 of the pair) and a slice of d_v.  The
// leader (rank 0) issues M=256 MMAs: each CTA holds its own 128 rows of Q, P,
// S and O, and one half of every K and V tile (K: 64 of the 128 keys; V: half
// of the d_v columns).  Each SM therefore loads half of the K/V bytes a
// single-CTA tile needs.
//
// K and V stream through two rings of 16 KB granules, every granule full: a K
// granule is [64 keys x 128 d] (one 8-MMA burst of the S product), a V
// granule [128 keys x 64 d_v].  One producer thread fills each ring and one
// MMA thread drains it: warp 1 issues S = Q K^T, warp 2 issues O += P V, so
// the tensor pipe stays fed while either thread waits on a barrier.
//
// Synchronisation: every tensor load of both CTAs completes on the leader's
// `full` barrier; the leader's MMA commits are multicast to both CTAs'
// `empty`, `s_full`, `p_empty` and `o_full` barriers; the gating warps of
// both CTAs arrive on the leader's `s_empty` and `p_full`.  Waits are bounded
// as in fwd_tc.cu.
//
// d_v = 512 (QUAD): O of 128 rows x 512 columns would fill a CTA's whole
// TMEM, so a cluster of four CTAs runs two pairs over the same 256 query rows,
// pair q owning d_v columns [256 q, 256 q + 256).  Key tiles alternate between
// the pairs over the cluster's whole sequence of tiles, and S is formed once,
// by the pair whose turn it is.  Its gating warps write the bf16 P tile twice:
// into their own TMEM, over the S columns they have just read (the A operand
// of their own pair's O product, which then frees that S buffer), and into the
// shared-memory P buffer of the other pair's CTA of the same rows, where the
// other pair's O product reads it (16-byte remote stores into a K-major layout
// without swizzle, so that each warp store covers 512 contiguous bytes).  The
// row sums b of eq (83) are split the same way and exchanged before the
// epilogue.  Each pair thus issues the S product of every other tile only, and
// its own O product never waits for the other pair's buffer.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "internal.h"
#include "tc_ptx.cuh"

namespace mlstm {
namespace {

using namespace tc;

constexpr int kBM = 128;                 // query rows per CTA (256 per pair)
constexpr int kBN = 128;                 // keys per tile
constexpr int kThreads = 384;
constexpr int kSlotBytes = 16384;        // ring granule per CTA: 2 K boxes [64 keys x 64 d] or 1 V box [128 keys x 64 d_v]
constexpr int kMaxSlots = 16;
constexpr int kQuadSlots = 8;            // ring granules of the four-CTA form (4 fit at d_qk = 512 beside Q and P)
constexpr int kProducers = 2;
constexpr uint32_t kTmemCols = 512;
constexpr int kSmemLimit = 232448;
constexpr long long kDrainSpin = 1LL << 22;

enum : int {
  kBarQFull = 0,
  kBarSFull = 1,
  kBarSEmpty = 3,                         // QUAD: freed by the own-tile O product that read P from it
  kBarPFull = 5,                          // QUAD: this pair's P of its own tile in S buffer 0 is in TMEM
  kBarPEmpty = 6,                         // QUAD: the other pair has consumed this CTA's last P sent to it
  kBarOFull = 7,
  kBarDrain = 8,                          // two: S issuer, O issuer
  kBarQEmpty = 10,                        // Q of the current item read by its last S product
  kBarFull = 11,                          // then the rings' empty barriers, then (QUAD) the ones below
};
// QUAD only, after the rings' barriers (offsets from kBarFull + 2 x slots)
enum : int {
  kQBarPFull1 = 0,                        // this pair's P of its own tile in S buffer 1 is in TMEM
  kQBarBxFull = 1,                        // the other pair's row sums written here
  kQBarEpiDone = 2,                       // the other pair's CTA of these rows finished its epilogue
  kQBarODrained = 3,                      // (pair leader) the pair's epilogue has read O out of TMEM
  kQBarPRx = 4,                           // (pair leader) the other pair's P tile is in this pair's buffers
  kQBars = 5,
};
enum : int { kSiteProducer = 11, kSiteMma = 12, kSiteGate = 13, kSiteEpilogue = 14 };

#ifdef MLSTM_TRACE
// clock64 stamps of both CTAs of one cluster (trace builds only): [cta][event][tile]
__device__ long long g_trace2[2 * 16 * 64];
__device__ int g_trace2_cluster;
__device__ int g_trace2_item;                     // which item of the cluster is traced
__device__ unsigned long long g_trace2_wall[2 * 512];   // per cluster: %globaltimer at start and end
#define TRACE2(ev, j)                                                                             \
  do {                                                                                            \
    if (trace_on && (j) < 64 && trace_rank < 2) g_trace2[(trace_rank * 16 + (ev)) * 64 + (j)] = clock64(); \
  } while (0)
#else
#define TRACE2(ev, j) \
  do {                \
  } while (0)
#endif

struct Tc2Params {
  const float* a2;
  const float* p2;
  const float* mrow;
  float* m_out;
  float* n_out;
  float* b_out;
  const __nv_bfloat16* og;                // output-gate pre-activations (eq 78), or null
  int T, BH, dqk, dv;
  int nsplit, dv_slice, nk, nv, npairs;   // nk + nv ring granules (K ring, then V ring)
  int n_items, nclusters;                 // work items (query-row pairs x d_v splits); clusters launched
  int l2_prefetch;                        // the next key tile's K/V boxes brought into L2 one tile ahead
  float log2_scale;
  DevStatus st;
};

// MMA bursts with compile-time trip counts: every descriptor is the slot base
// plus a constant, so the issuing thread sends the MMAs back to back.
// S += Q K^T over KB boxes of 64 d-columns (4 k-steps each).
template <int KB>
__device__ __forceinline__ void issue_s(uint32_t d_s, uint64_t aq, uint64_t bk, uint32_t idS, bool first) {
#pragma unroll
  for (int b2 = 0; b2 < KB; ++b2)
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_bf16_ss_pair(d_s, aq + b2 * 1024 + 2 * kk, bk + b2 * 512 + 2 * kk, idS, first ? ((b2 | kk) != 0) : 1u);
}
// O[:, cols] += P V[:, cols] over the 128 keys of a tile (8 k-steps of 16 keys):
// N = 256 columns (each CTA holds one whole 128-column chunk: two MN atoms
// 16 KB apart) or N = 128 (each CTA holds 64 columns: one atom).
__device__ __forceinline__ void issue_o(uint32_t d_o, uint64_t dP, uint64_t bv, uint32_t idO, bool first) {
#pragma unroll
  for (int kk = 0; kk < kBN / 16; ++kk)
    mma_bf16_ss_pair(d_o, dP + (kk >> 2) * 1024 + (kk & 3) * 2, bv + kk * 128, idO, first ? (kk != 0) : 1u);
}

// The same over the other pair's P, received without swizzle: row R's keys
// 8c..8c+7 at byte 2048 c + 16 R (core matrices 128 bytes apart along the
// rows, 2 KB apart along the keys), so a k-step of 16 keys is 4 KB on.
__device__ __forceinline__ void issue_o_rx(uint32_t d_o, uint64_t dPx, uint64_t bv, uint32_t idO, bool first) {
#pragma unroll
  for (int kk = 0; kk < kBN / 16; ++kk)
    mma_bf16_ss_pair(d_o, dPx + (uint64_t)(256 * kk), bv + kk * 128, idO, first ? (kk != 0) : 1u);
}
// The same over A in TMEM (the pair's own P, over the S buffer it came from):
// a warp wrote the P of its 64 keys into the first 32 columns of its 64-column
// half of the buffer, so keys 16 kk.. sit at column 64 (kk / 4) + 8 (kk % 4).
__device__ __forceinline__ void issue_o_ts(uint32_t d_o, uint32_t a_p, uint64_t bv, uint32_t idO, bool first) {
#pragma unroll
  for (int kk = 0; kk < kBN / 16; ++kk)
    mma_bf16_ts_pair(d_o, a_p + 64u * (kk >> 2) + 8u * (kk & 3), bv + kk * 128, idO, first ? (kk != 0) : 1u);
}

// One work item: a pair of 128-row query blocks of one head and one d_v slice.
struct Item {
  int bh, split, i0, dv_off, dv_cta, nkv;
};

// Items in longest-first order over all heads; cluster c takes, in round r,
// item r*G + c (r even) or r*G + G-1-c (r odd).  This serpentine order
// balances the clusters as well as greedy list scheduling does here, and
// every role of every CTA derives the same sequence without communicating.
// prank: the CTA's rank in its pair (its 128 rows); pr: with QUAD, the pair's
// d_v half (the item's split), else -1.
__device__ __forceinline__ bool item_at(const Tc2Params& p, int r, int c, uint32_t prank, int pr, Item& it) {
  const int G = p.nclusters;
  const int w = r * G + ((r & 1) ? G - 1 - c : c);
  if (w >= p.n_items) return false;
  const int per_rank = p.BH * p.nsplit;
  const int pair = p.npairs - 1 - w / per_rank;
  const int rem = w % per_rank;
  it.bh = rem / p.nsplit;
  it.split = pr >= 0 ? pr : rem % p.nsplit;
  it.i0 = (2 * pair + (int)prank) * kBM;
  it.dv_off = it.split * p.dv_slice;
  it.dv_cta = (pr >= 0 || it.split == 0) ? p.dv_slice : p.dv - p.dv_slice;
  it.nkv = (min(p.T, (2 * pair + 2) * kBM) - 1) / kBN + 1;       // key tiles, same in both CTAs
  return true;
}

// OG: the output gate is applied in the epilogue (a separate instantiation,
// so that the kernel without it keeps its register allocation).  QUAD: the
// four-CTA form for d_v = 512 described at the top of this file.
template <int NSBUF, bool OG, bool QUAD>
__global__ void __launch_bounds__(kThreads, 1)
fwd_tc2_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
               const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_h,
               const Tc2Params p) {
  static_assert(!QUAD || NSBUF == 2, "the four-CTA form double-buffers S");
  constexpr int HALF = kBN / 2;
  constexpr uint32_t SOFF = kTmemCols - NSBUF * kBN;
  constexpr int kCluster = QUAD ? 4 : 2;
  constexpr int kSlots = QUAD ? kQuadSlots : kMaxSlots;
  constexpr int kBarEmpty = kBarFull + kSlots;
  constexpr int kBarQuad = kBarFull + 2 * kSlots;
  constexpr int kBarPFull1 = kBarQuad + kQBarPFull1, kBarBxFull = kBarQuad + kQBarBxFull;
  constexpr int kBarEpiDone = kBarQuad + kQBarEpiDone, kBarODrained = kBarQuad + kQBarODrained;
  constexpr int kBarPRx = kBarQuad + kQBarPRx;
  constexpr int kNumBars = kBarQuad + (QUAD ? kQBars : 0);
  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t bars[kNumBars];
  __shared__ uint32_t tmem_holder;
  __shared__ int abort_flag;
  __shared__ int s_issued_s;                // key tile of the last fully issued S product (read by the two-CTA form only)
  // Loads each producer of this CTA issued (ring granules, written once at
  // its exit; Q fills) and, in the pair leader, the peer's counts and abort
  // flag, sent at exit: after an abort the leader settles every load of the pair.
  __shared__ int loads_s[kProducers];
  __shared__ int qfills_s[kProducers];
  __shared__ int peer_loads_s[kProducers];
  __shared__ int peer_qfills_s[kProducers];
  __shared__ int peer_abort_s;
  // row sums of the two column halves; with QUAD a third slot holds those of
  // the other pair's CTA of the same rows (its key tiles)
  __shared__ float bpart[(QUAD ? 3 : 2) * kBM];
  volatile int* abort = &abort_flag;
  volatile int* s_issued = &s_issued_s;
  volatile int* qfills = qfills_s;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t prank = rank & 1u;                          // rank in the pair: which 128 rows
  const int pr = QUAD ? (int)(rank >> 1) : -1;               // QUAD: the pair (d_v half)
  const uint32_t lead = rank & ~1u;                          // the pair's leader
  const bool leader = prank == 0;
  const uint16_t pmask = (uint16_t)(0x3u << lead);           // this pair's CTAs
  const uint16_t xmask = (uint16_t)(0x3u << (lead ^ 2u));    // QUAD: the other pair's CTAs
  const int cid = (int)(blockIdx.x / kCluster);
#ifdef MLSTM_TRACE
  const bool trace_cluster = cid == g_trace2_cluster;   // read once; the first item is traced
  bool trace_on = trace_cluster;
  const int trace_rank = (int)rank;
#define TRACE_ITEM(q) (trace_on = trace_cluster && (q) == g_trace2_item)
#else
#define TRACE_ITEM(q) ((void)0)
#endif
  // QUAD: key tile g of the cluster's whole sequence belongs to pair g & 1
  auto own = [&](int g) { return !QUAD || (g & 1) == pr; };

  const int nkg = p.dqk / 128;                               // K granules per key tile
  const uint32_t base = (smem_u32(dsmem) + 1023u) & ~1023u;
  const uint32_t sQ = base;
  const uint32_t sP = sQ + (uint32_t)p.dqk * kBM * 2;
  const uint32_t sRing = sP + (uint32_t)kBN * kBM * 2;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  auto lbar = [&](int i) { return mapa_shared(smem_u32(&bars[i]), lead); };   // the pair leader's barrier

  if (threadIdx.x < kProducers) {
    loads_s[threadIdx.x] = 0;
    qfills_s[threadIdx.x] = 0;
    peer_loads_s[threadIdx.x] = 0;
    peer_qfills_s[threadIdx.x] = 0;
  }
  if (threadIdx.x == 0) {
    abort_flag = 0;
    peer_abort_s = 0;
    s_issued_s = -1;
    mbar_init(bar(kBarQFull), 1);
    mbar_init(bar(kBarQEmpty), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kBarSFull + b), 1);
      mbar_init(bar(kBarSEmpty + b), QUAD ? 1 : 16);   // QUAD: the own-tile O product; else both CTAs' gating warps
    }
    // QUAD: a P barrier per S buffer.  One barrier for both could complete
    // two phases before the O issuer, held up by the other pair's tile, waits
    // for the first, and a parity wait cannot tell that from none; the next
    // use of a buffer waits for the O product that read its last P.
    mbar_init(bar(kBarPFull), 16);          // both CTAs' gating warps
    mbar_init(bar(kBarPEmpty), 1);
    mbar_init(bar(kBarOFull), 1);
    mbar_init(bar(kBarDrain), 1);
    mbar_init(bar(kBarDrain + 1), 1);
    if (QUAD) {
      mbar_init(bar(kBarPFull1), 16);        // both CTAs' gating warps
      mbar_init(bar(kBarBxFull), 4);         // the other pair's half-0 gating warps of these rows
      mbar_init(bar(kBarEpiDone), 1);        // one gating thread of the other pair's CTA of these rows
      mbar_init(bar(kBarODrained), 2);       // one gating thread of each CTA of this pair
      mbar_init(bar(kBarPRx), 16);           // the other pair's gating warps (both its CTAs)
    }
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bar(kBarFull + s), 1);
      mbar_init(bar(kBarEmpty + s), 1);
    }
    fence_barrier_init();
    tma_prefetch_desc(&tmap_q);
    tma_prefetch_desc(&tmap_k);
    tma_prefetch_desc(&tmap_v);
    tma_prefetch_desc(&tmap_h);
  }
  if (warp == 2) {
    tmem_alloc_pair(smem_u32(&tmem_holder), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();                       // every CTA's barriers initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = tmem_holder;
  const long long spin = p.st.spin_limit;
  if (threadIdx.x == 0) TRACE2(0, 0);
#ifdef MLSTM_TRACE
  if (threadIdx.x == 0 && rank == 0 && cid < 512) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    g_trace2_wall[2 * cid] = t;
  }
#endif
  Item it;

  if ((warp == 0 || warp == 3) && lane == 0) {
    // ------------------------------------------------------------ TMA producers (every CTA)
    // Warp 0 fills the K ring, warp 3 the V ring; both load half of each
    // item's Q once the previous item's S products have read the old Q.  Each
    // CTA loads its own halves into its own buffers; completion is counted on
    // the pair leader's full barriers, whose expected bytes (both halves) only
    // the leader posts.  With QUAD the K ring carries only this pair's key tiles.
    const int pi = warp == 0 ? 0 : 1;
    const int base_slot = pi == 0 ? 0 : p.nk, n = pi == 0 ? p.nk : p.nv;
    int st = 0, nloads = 0;                  // nloads: granules filled (round-robin over the ring)
    uint32_t ph = 0;
    bool ok = true;
    // loads the ring's next granule; with pf_dy > 0, first asks L2 for the
    // same boxes pf_dy keys further on (the ring's next key tile), so that
    // their own loads, a tile later, hit L2.  kblk > 0: the granule is one 4-D
    // box of kblk 64-column blocks starting at block x0 / 64 (one copy instead
    // of kblk: each issuing thread handles its copies one after another);
    // otherwise nbox 3-D boxes.
    auto load = [&](const CUtensorMap* map, int nbox, int kblk, uint32_t box_bytes, int x0, int dx, int y,
                    int pf_dy) {
      if (!ok) return;
      const int g = base_slot + st;
      if (pf_dy > 0) {
        if (kblk > 0) tma_prefetch_l2_4d(map, 0, y + pf_dy, x0 / 64, it.bh);
        else
          for (int b2 = 0; b2 < nbox; ++b2) tma_prefetch_l2_3d(map, x0 + b2 * dx, y + pf_dy, it.bh);
      }
      ok = mbar_wait(bar(kBarEmpty + g), ph ^ 1, spin, abort, p.st, kSiteProducer);
      if (!ok) return;
      if (leader) mbar_arrive_expect_tx(bar(kBarFull + g), 2u * kSlotBytes);
      if (kblk > 0) tma_load_4d_pair(sRing + g * kSlotBytes, map, lbar(kBarFull + g), 0, y, x0 / 64, it.bh);
      else
        for (int b2 = 0; b2 < nbox; ++b2)
          tma_load_3d_pair(sRing + g * kSlotBytes + b2 * box_bytes, map, lbar(kBarFull + g), x0 + b2 * dx, y, it.bh);
      ++nloads;
      if (++st == n) { st = 0; ph ^= 1; }
    };
    constexpr int kstep = QUAD ? 2 : 1;      // key tiles between two of this ring's K tiles
    int qi = 0, g0 = 0;                      // items so far; key tiles of the sequence before this item
    for (int r = 0; r * p.nclusters < p.n_items && ok; ++r) {
      if (!item_at(p, r, cid, prank, pr, it)) continue;
      if (qi > 0) ok = mbar_wait(bar(kBarQEmpty), (uint32_t)(qi - 1) & 1u, spin, abort, p.st, kSiteProducer);
      if (!ok) break;
      if (leader && pi == 0) mbar_arrive_expect_tx(bar(kBarQFull), 2u * (uint32_t)p.dqk * kBM * 2);
      {
        // each producer loads its half of Q's 64-column blocks as one 4-D box
        const int qb = p.dqk / 64 / kProducers;
        tma_load_4d_pair(sQ + (uint32_t)(pi * qb) * 16384u, &tmap_q, lbar(kBarQFull), 0, it.i0, pi * qb, it.bh);
      }
      ++qi;
      qfills[pi] = qi;
      const int nch = it.dv_cta / 128, nvc = (nch + 1) / 2;
      if (pi == 0) {
        for (int j = 0; j < it.nkv && ok; ++j) {
          if (!own(g0 + j)) continue;
          const int pf = (p.l2_prefetch && j + kstep < it.nkv) ? kstep * kBN : 0;
          for (int c = 0; c < nkg; ++c) load(&tmap_k, 1, 2, 0u, c * 128, 0, j * kBN + (int)prank * 64, pf);
        }
      } else {
        for (int j = 0; j < it.nkv && ok; ++j) {
          const int pf = (p.l2_prefetch && j + 1 < it.nkv) ? kBN : 0;
          for (int e = 0; e < nvc; ++e) {
            // a pair of 128-column chunks in two adjacent granules takes one N=256
            // MMA burst (this CTA holds chunk 2e+rank whole); otherwise each chunk
            // is its own N=128 burst over one granule (this CTA holds 64 columns)
            if (2 * e + 1 < nch && st + 1 < n) {
              const int col = it.dv_off + (2 * e + (int)prank) * 128;
              load(&tmap_v, 1, 0, 0u, col, 0, j * kBN, pf);
              load(&tmap_v, 1, 0, 0u, col + 64, 0, j * kBN, pf);
            } else {
              for (int q = 2 * e; q < min(2 * e + 2, nch); ++q)
                load(&tmap_v, 1, 0, 0u, it.dv_off + q * 128 + (int)prank * 64, 0, j * kBN, pf);
            }
          }
        }
      }
      g0 += it.nkv;
    }
    loads_s[pi] = nloads;
  } else if ((warp == 1 || warp == 2) && lane == 0 && leader) {
    // ------------------------------------------------------------ MMA issuers (pair leader)
    // Warp 1 issues S = Q K^T, warp 2 issues O += P V.  The two products use
    // disjoint TMEM columns and rings, so the threads need no ordering between
    // them beyond the gating handshake; with two issuing threads the tensor
    // pipe stays fed while either one waits on a barrier.
    const bool s_role = warp == 1;
    const uint32_t idS = idesc_bf16_f32(2 * kBM, kBN, 0, 0);       // M=256 rows over the pair, N=128 keys
    const uint32_t idO = idesc_bf16_f32(2 * kBM, 128, 0, 1);       // N=128 d_v columns, V MN-major
    const uint32_t idO2 = idesc_bf16_f32(2 * kBM, 256, 0, 1);      // N=256: two chunks
    const uint64_t dQ = smem_desc_sw128(sQ, 16, 1024);
    const uint64_t dK = smem_desc_sw128(sRing, 16, 1024);
    const uint64_t dP = smem_desc_sw128(sP, 16, 1024);
    const uint64_t dPx = smem_desc_noswz(sP, 2048, 128);           // QUAD: the other pair's P
    const uint64_t dV = smem_desc_sw128(sRing + (uint32_t)p.nk * kSlotBytes, 16384, 1024);
    const int base_slot = s_role ? 0 : p.nk, n = s_role ? p.nk : p.nv;
    int st = 0;
    uint32_t ph = 0;
    bool ok = true;
    auto full = [&](int s2) { return mbar_wait(bar(kBarFull + base_slot + s2), ph, spin, abort, p.st, kSiteMma); };
    auto release = [&](int s2) { mma_commit_pair_mc(bar(kBarEmpty + base_slot + s2), pmask); };
    auto next = [&]() { if (++st == n) { st = 0; ph ^= 1; } };
    // items; key tiles of the sequence; this pair's S tiles; the other pair's tiles
    int qi = 0, gt = 0, gs = 0, go = 0;
    for (int r = 0; r * p.nclusters < p.n_items && ok; ++r) {
      if (!item_at(p, r, cid, prank, pr, it)) continue;
      TRACE_ITEM(qi);
      if (s_role) {
        ok = mbar_wait(bar(kBarQFull), (uint32_t)qi & 1u, spin, abort, p.st, kSiteMma);
        for (int j = 0; j < it.nkv && ok; ++j, ++gt) {
          if (!own(gt)) continue;
          const int buf = gs % NSBUF, u = gs / NSBUF;
          TRACE2(1, j);
          ok = mbar_wait(bar(kBarSEmpty + buf), (u & 1) ^ 1, spin, abort, p.st, kSiteMma);
          if (!ok) break;
          // no tcgen05 fence: the gating warps finished their TMEM reads (wait::ld)
          // before arriving; with QUAD the buffer was freed by an MMA commit
          TRACE2(2, j);
          const uint32_t d_s = tmem + SOFF + buf * kBN;
          for (int c = 0; c < nkg; ++c) {
            ok = full(st);
            if (!ok) break;
            issue_s<2>(d_s, dQ + (uint64_t)(2 * c * 1024), dK + (uint64_t)(st * (kSlotBytes >> 4)), idS, c == 0);
            release(st);
            next();
          }
          if (!ok) break;
          mma_commit_pair_mc(bar(kBarSFull + buf), pmask);
          *s_issued = gs;
          ++gs;
          TRACE2(3, j);
        }
        // this item's Q may be replaced once its S products complete
        if (ok) mma_commit_pair_mc(bar(kBarQEmpty), pmask);
      } else {
        const int nch = it.dv_cta / 128, nvc = (nch + 1) / 2;
        if constexpr (QUAD) {
          // the pair's epilogue has read the previous item's O out of TMEM (the
          // first P of an item may come from the other pair's gating warps)
          if (qi > 0) ok = mbar_wait_cluster(bar(kBarODrained), (uint32_t)(qi - 1) & 1u, spin, abort, p.st, kSiteMma);
        }
        for (int j = 0; j < it.nkv && ok; ++j, ++gt) {
          // QUAD: this pair's tile has its P in TMEM, over S buffer `buf`; the
          // other pair's tile has it in this pair's shared-memory P buffers
          const bool mine = own(gt);
          int buf = 0;
          if constexpr (QUAD) {
            if (mine) {
              buf = gs % NSBUF;
              ok = mbar_wait_cluster(bar(buf == 0 ? kBarPFull : kBarPFull1), (uint32_t)(gs / NSBUF) & 1u, spin, abort,
                                     p.st, kSiteMma);
              ++gs;
            } else {
              ok = mbar_wait_cluster(bar(kBarPRx), (uint32_t)go & 1u, spin, abort, p.st, kSiteMma);
              ++go;
            }
          } else {
            ok = mbar_wait(bar(kBarPFull), (uint32_t)gt & 1u, spin, abort, p.st, kSiteMma);
          }
          if (!ok) break;
          // P is in shared memory, made visible to the async proxy before the
          // gating warps arrived, or (QUAD, own tile) in TMEM, stored before
          // they arrived.  Before the first tile of an item they also finished
          // reading the previous item's O (wait::ld), which these MMAs overwrite.
          if (QUAD || j == 0) tc_fence_after();
          TRACE2(4, j);
          const uint32_t a_p = tmem + SOFF + buf * kBN;
          for (int e = 0; e < nvc && ok; ++e) {
            if (2 * e + 1 < nch && st + 1 < n) {
              // granules st, st+1: this CTA's two MN atoms 16 KB apart, N=256
              const int s0 = st;
              ok = full(s0);
              next();
              ok = ok && full(st);
              if (!ok) break;
              const uint64_t bv = dV + (uint64_t)(s0 * (kSlotBytes >> 4));
              if (QUAD && mine) issue_o_ts(tmem + 256 * e, a_p, bv, idO2, j == 0);
              else if (QUAD) issue_o_rx(tmem + 256 * e, dPx, bv, idO2, j == 0);
              else issue_o(tmem + 256 * e, dP, bv, idO2, j == 0);
              release(s0);
              release(st);
              next();
            } else {
              for (int q = 2 * e; q < min(2 * e + 2, nch); ++q) {
                // within an item, the tile's last (narrow) chunk waits until the
                // next S product is issued: queued behind it, it keeps the pipe
                // busy while the gating warps hand the S buffer back (bounded)
                if (!QUAD && q == nch - 1 && nch > 1 && j + 1 < it.nkv)
                  for (long long w2 = 0; *s_issued < gt + 1 && w2 < spin && !*abort; ++w2) {
                  }
                ok = full(st);
                if (!ok) break;
                const uint64_t bv = dV + (uint64_t)(st * (kSlotBytes >> 4));
                if (QUAD && mine) issue_o_ts(tmem + 128 * q, a_p, bv, idO, j == 0);
                else if (QUAD) issue_o_rx(tmem + 128 * q, dPx, bv, idO, j == 0);
                else issue_o(tmem + 128 * q, dP, bv, idO, j == 0);
                release(st);
                next();
              }
            }
          }
          if (!ok) break;
          if constexpr (QUAD) {
            // own tile: its S buffer (holding P) is free for the S product two
            // own tiles on; other tile: the sender's next P may replace this one
            if (mine) mma_commit_pair_mc(bar(kBarSEmpty + buf), pmask);
            else mma_commit_pair_mc(bar(kBarPEmpty), xmask);
          } else {
            mma_commit_pair_mc(bar(kBarPEmpty), pmask);
          }
          TRACE2(5, j);
        }
        if (ok) mma_commit_pair_mc(bar(kBarOFull), pmask);
      }
      ++qi;
    }
    if (s_role) *s_issued = 0x7fffffff;     // no further S products
    // every MMA this thread issued has completed before TMEM is released
    const int drain = kBarDrain + (s_role ? 0 : 1);
    mma_commit_pair(bar(drain));
    for (long long w = 0; w < kDrainSpin; ++w)
      if (mbar_try_wait(bar(drain), 0)) break;
  } else if (warp >= 4) {
    // ------------------------------------------------------------ gating + epilogue (every CTA)
    const int gw = warp - 4, qd = gw & 3, half = gw >> 2;
    asm volatile("griddepcontrol.wait;" ::: "memory");        // gate terms from the preceding gate pass
    const int rl = 32 * qd + lane;
    const uint32_t lane_addr = (uint32_t)(32 * qd) << 16;
    const uint32_t l_sempty0 = lbar(kBarSEmpty), l_sempty1 = lbar(kBarSEmpty + 1), l_pfull = lbar(kBarPFull);
    const uint32_t l_pfull1 = QUAD ? lbar(kBarPFull1) : 0u;
    // QUAD: the CTA of the other pair that holds these rows: its P buffer and
    // the other pair leader's barrier for its arrival
    const uint32_t xrank = rank ^ 2u;
    const uint32_t x_sP = QUAD ? mapa_shared(sP, xrank) : 0u;
    const uint32_t x_prx = QUAD ? mapa_shared(bar(kBarPRx), lead ^ 2u) : 0u;
    // Exit rule: a warp whose wait gives up (raising the abort flag, after
    // which every wait returns at once) leaves the item's tile loop; the tile
    // loop has no group barrier.  The eight warps of the CTA then meet once
    // per item at the reducing barrier after the O wait (twice with QUAD:
    // again after the row-sum exchange), and all of them go on with the
    // epilogue or all leave.  So every named barrier below is reached by all
    // 256 threads (or all 128 of a half) on every path.  The 32 lanes of a
    // warp poll the same barrier with the same instructions and take the same
    // exit; the waits are kept in this plainest form because a warp vote per
    // wait measured slower.
    bool ok = true;
    int qi = 0, gt = 0, gs = 0;              // items; key tiles of the sequence; this pair's tiles
    for (int r = 0; r * p.nclusters < p.n_items && ok; ++r) {
      if (!item_at(p, r, cid, prank, pr, it)) continue;
      TRACE_ITEM(qi);
      const int i = it.i0 + rl;
      const bool row_ok = i < p.T;
      const size_t hbase = (size_t)it.bh * p.T;
      const float rr = row_ok ? p.p2[hbase + i] - p.log2_scale : 0.0f;
      const float m = row_ok ? p.mrow[hbase + i] : 0.0f;      // for the epilogue
      float bsum = 0.0f;
      // this pair's key tiles of the item: every tile, or (QUAD) every other one
      const int jfirst = own(gt) ? 0 : 1, jstep = QUAD ? 2 : 1;
      // QUAD: P goes into the other pair's P buffer, which its epilogue of the
      // previous item stages output through: wait until that is done
      bool partner_free = !QUAD || qi == 0;
      float av_next[HALF / 32];
#pragma unroll
      for (int t = 0; t < HALF / 32; ++t) {
        const int col = jfirst * kBN + half * HALF + lane + 32 * t;
        av_next[t] = (jfirst < it.nkv && col < p.T) ? p.a2[hbase + col] : -INFINITY;
      }
      for (int j = jfirst; j < it.nkv && ok; j += jstep, ++gs) {
        const int j0 = j * kBN, cbase = j0 + half * HALF;
        const int buf = gs % NSBUF, u = gs / NSBUF;
        float av[HALF / 32];
#pragma unroll
        for (int t = 0; t < HALF / 32; ++t) {
          av[t] = av_next[t];
          const int col = cbase + jstep * kBN + lane + 32 * t;
          av_next[t] = (j + jstep < it.nkv && col < p.T) ? p.a2[hbase + col] : -INFINITY;
        }
        const bool diag = j0 + kBN - 1 > it.i0;                 // some column of the tile lies above a row
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
        if (gw == 0 && lane == 0) TRACE2(6, j);
        uint32_t sv[HALF];
#pragma unroll
        for (int t = 0; t < HALF / 32; ++t)
          tmem_ld32(tmem + lane_addr + SOFF + buf * kBN + half * HALF + 32 * t,
                    *reinterpret_cast<uint32_t(*)[32]>(&sv[32 * t]));
        tmem_wait_ld();
        if constexpr (!QUAD) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(buf == 0 ? l_sempty0 : l_sempty1);
        }

        uint32_t pk[HALF / 2];
        if (!diag) {
          const float rfac = (A == -INFINITY || !row_ok) ? 0.0f : exp2f(A - rr);
#pragma unroll
          for (int c = 0; c < HALF; c += 2) {
            const float c0 = __shfl_sync(0xffffffffu, av[c / 32], c & 31);
            const float c1 = __shfl_sync(0xffffffffu, av[(c + 1) / 32], (c + 1) & 31);
            const float x0 = __uint_as_float(sv[c]) * c0 * rfac;
            const float x1 = __uint_as_float(sv[c + 1]) * c1 * rfac;
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
        if (gw == 0 && lane == 0) TRACE2(7, j);
        if constexpr (QUAD) {
          // this pair's copy: into TMEM over the first 32 columns of the 64
          // this warp has just read (the other half-warp's 64 are disjoint)
          tmem_st32(tmem + lane_addr + SOFF + buf * kBN + half * HALF, pk);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_release_cluster(buf == 0 ? l_pfull : l_pfull1);
          // the other pair's copy: once its CTA of these rows has finished its
          // previous epilogue (first tile of an item) and its O product has
          // read the last P this CTA sent (every phase is seen in order: one
          // send per tile of this pair)
          if (!partner_free) {
            ok = mbar_wait_cluster(bar(kBarEpiDone), (uint32_t)(qi - 1) & 1u, spin, abort, p.st, kSiteGate);
            if (!ok) break;
            partner_free = true;
          }
          ok = mbar_wait_cluster(bar(kBarPEmpty), ((uint32_t)gs & 1u) ^ 1u, spin, abort, p.st, kSiteGate);
          if (!ok) break;
          if (gw == 0 && lane == 0) TRACE2(8, j);
          // without swizzle: keys 8c..8c+7 of row rl at 2048 c + 16 rl, so each
          // store of the warp covers 512 contiguous bytes (remote stores of
          // scattered 16-byte pieces measured about half as fast)
#pragma unroll
          for (int g = 0; g < HALF / 8; ++g) {
            const uint32_t off = (uint32_t)(half * (HALF / 8) + g) * 2048u + rl * 16u;
            st_shared_cluster_v4(x_sP + off, pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
          }
          fence_proxy_async_cluster();
          __syncwarp();
          if (lane == 0) mbar_arrive_release_cluster(x_prx);
        } else {
          ok = mbar_wait(bar(kBarPEmpty), ((uint32_t)gs & 1u) ^ 1u, spin, abort, p.st, kSiteGate);
          if (!ok) break;
          if (gw == 0 && lane == 0) TRACE2(8, j);
#pragma unroll
          for (int g = 0; g < HALF / 8; ++g) {
            const int c = half * HALF + 8 * g;
            const uint32_t addr = sP + (c >> 6) * 16384u + rl * 128u + ((((c & 63) >> 3) ^ (rl & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * g]),
                         "r"(pk[4 * g + 1]), "r"(pk[4 * g + 2]), "r"(pk[4 * g + 3])
                         : "memory");
          }
          fence_proxy_async_smem();
          // also orders this warp's earlier TMEM reads of O before the next
          // item's first O product (which waits on this arrival)
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(l_pfull);
        }
        if (gw == 0 && lane == 0) TRACE2(9, j);
      }
      if constexpr (QUAD) {
        // an item with none of this pair's tiles still waits, once, for the
        // other pair's previous epilogue (every phase is seen in order)
        if (ok && !partner_free) ok = mbar_wait_cluster(bar(kBarEpiDone), (uint32_t)(qi - 1) & 1u, spin, abort,
                                                        p.st, kSiteGate);
      }
      gt += it.nkv;
      if constexpr (!QUAD) {
        // the next item's gate terms (its rows' p2 and m, the first two key
        // tiles' a2) into L2 while this epilogue runs: read at its start, they
        // otherwise wait on DRAM (up to ~4,000 cycles, clock traces).  125M-
        // scale layer 105.9 -> 104.7 us; in the four-CTA form, whose first
        // tile of an item waits on the other pair anyway, it measured 0.7 %
        // slower, so it is left out there.
        Item nx;
        if (item_at(p, r + 1, cid, prank, pr, nx)) {
          const size_t nb = (size_t)nx.bh * p.T;
          const int ni = nx.i0 + rl;
          if (ni < p.T) {
            prefetch_l2(p.p2 + nb + ni);
            prefetch_l2(p.mrow + nb + ni);
          }
#pragma unroll
          for (int t = 0; t < 2 * (HALF / 32); ++t) {
            const int col = (t / (HALF / 32)) * kBN + half * HALF + lane + 32 * (t % (HALF / 32));
            if (col < p.T) prefetch_l2(p.a2 + nb + col);
          }
        }
      }

      if constexpr (QUAD) {
        bpart[half * kBM + rl] = bsum;
        // this pair's row sums are final once its tiles are gated: send them
        // to the other pair's CTA of these rows now, ahead of the O wait (the
        // pair without the item's last tile finishes its O products later).
        // Its slot was read before its last epilogue ended, which the waits
        // above have seen.
        ok = bar_red_and(1, 256, ok);        // all eight warps leave together, or none
        if (!ok) break;
        if (half == 0) {
          st_shared_cluster_f32(mapa_shared(smem_u32(&bpart[2 * kBM + rl]), xrank), bpart[rl] + bpart[kBM + rl]);
          __syncwarp();
          if (lane == 0) mbar_arrive_release_cluster(mapa_shared(bar(kBarBxFull), xrank));
        }
      }

      // ---- epilogue: n = max(|b|, exp(-m)), H~ = O / n.  Each half stages its
      // 64-column boxes one at a time in its 16 KB of the P buffer (free until
      // the next item's first P) and stores each by TMA as soon as it is written.
      if (ok) ok = mbar_wait(bar(kBarOFull), (uint32_t)qi & 1u, spin, abort, p.st, kSiteEpilogue);
      if (QUAD && ok) ok = mbar_wait_cluster(bar(kBarBxFull), (uint32_t)qi & 1u, spin, abort, p.st, kSiteEpilogue);
      tc_fence_after();
      if (gw == 0 && lane == 0) TRACE2(10, 0);
      if constexpr (!QUAD) bpart[half * kBM + rl] = bsum;
      ok = bar_red_and(1, 256, ok);          // all eight warps leave together, or none
      if (!ok) break;
      float b = bpart[rl] + bpart[kBM + rl];
      if constexpr (QUAD) b += bpart[2 * kBM + rl];   // the other pair's key tiles
      const float nrm = fmaxf(fabsf(b), expf(-m));
      const float inv = nrm > 0.0f ? 1.0f / nrm : 0.0f;
      if (row_ok && it.split == 0 && half == 0) {
        if (p.m_out) p.m_out[hbase + i] = m;
        if (p.n_out) p.n_out[hbase + i] = nrm;
        if (p.b_out) p.b_out[hbase + i] = b;
      }
      if (gw == 0 && lane == 0) TRACE2(12, 0);
      const int cols = it.dv_cta / 2, c0 = half * cols;      // a multiple of 64
      const uint32_t stage = sP + (uint32_t)half * 16384u;
      const bool issuer = qd == 0 && lane == 0 && it.i0 < p.T;
      const bool use_og = OG && row_ok;
      for (int ch = 0; ch < cols / 64; ++ch) {
        // the output gate's 64 values of this row and box (eq 78), loaded
        // while the accumulator comes out of TMEM
        uint4 og4[OG ? 8 : 1];
        if (OG && use_og) {
          const uint4* src = reinterpret_cast<const uint4*>(p.og + (hbase + i) * (size_t)p.dv + it.dv_off + c0 + 64 * ch);
#pragma unroll
          for (int g = 0; g < 8; ++g) og4[g] = __ldg(src + g);
        }
        uint32_t o[64];
        tmem_ld32(tmem + lane_addr + c0 + 64 * ch, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
        tmem_ld32(tmem + lane_addr + c0 + 64 * ch + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
        tmem_wait_ld();
        // the half's previous box must have been read out by its store (and
        // bpart read by everyone, for the first box)
        if (issuer) tma_store_wait_read();
        named_bar_sync(2 + half, 128);
        const uint32_t row = stage + rl * 128u;
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          uint32_t w[4];
          const uint32_t* ow = reinterpret_cast<const uint32_t*>(&og4[OG ? g : 0]);
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            float x0 = __uint_as_float(o[8 * g + 2 * t]) * inv, x1 = __uint_as_float(o[8 * g + 2 * t + 1]) * inv;
            if (OG && use_og) {
              const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[t]));
              x0 *= sigmoid(f.x);
              x1 *= sigmoid(f.y);
            }
            w[t] = pack_bf16x2(x0, x1);
          }
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + ((g ^ (rl & 7)) << 4)), "r"(w[0]),
                       "r"(w[1]), "r"(w[2]), "r"(w[3])
                       : "memory");
        }
        fence_proxy_async_smem();
        named_bar_sync(2 + half, 128);
        if (issuer) {
          tma_store_3d(&tmap_h, stage, it.dv_off + c0 + 64 * ch, it.i0, it.bh);
          tma_store_commit();
        }
      }
      if (gw == 0 && lane == 0) TRACE2(14, 0);
      // the P buffer is free again once both halves' last stores read it out
      if (issuer) tma_store_wait_read();
      if constexpr (QUAD) tc_fence_before();   // this thread's TMEM reads of O, before the barrier
      named_bar_sync(1, 256);
      if constexpr (QUAD) {
        // O is read out and the P buffer free: one thread tells this pair's
        // leader (its next O product) and the other pair's CTA of these rows
        // (its next P write into this CTA, its next row-sum write).  It is a
        // thread of a warp that stored nothing to global memory, whose
        // cluster-scope release has no outstanding writes of its own to wait for.
        if (gw == 0 && lane == 0) TRACE2(15, 0);
        if (gw == 5 && lane == 0) {
          mbar_arrive_release_cluster(lbar(kBarODrained));
          mbar_arrive_release_cluster(mapa_shared(bar(kBarEpiDone), xrank));
        }
      }
      if (gw == 0 && lane == 0) TRACE2(11, 0);
      ++qi;
    }
    tc_fence_before();
  }

  __syncthreads();
  // Every issuer of the cluster's CTAs has stopped.  The peer sends its pair
  // leader its load counts and abort flag; after an abort in either CTA the
  // leader makes the last phase of Q and of every granule complete exactly
  // when the loads that were issued for it (by either CTA) have landed, and
  // waits for that (bounded), so no copy can still write shared memory once
  // the pair exits.  (The P tiles sent between the pairs are plain stores,
  // complete before the cluster barrier below.)
  if (!leader) {
    const int t = threadIdx.x;
    if (t < kProducers) st_shared_cluster_u32(mapa_shared(smem_u32(&peer_loads_s[t]), lead), (uint32_t)loads_s[t]);
    else if (t < 2 * kProducers)
      st_shared_cluster_u32(mapa_shared(smem_u32(&peer_qfills_s[t - kProducers]), lead),
                            (uint32_t)qfills_s[t - kProducers]);
    else if (t == 2 * kProducers)
      st_shared_cluster_u32(mapa_shared(smem_u32(&peer_abort_s), lead), (uint32_t)abort_flag);
  }
  cluster_sync_all();
  if (leader && threadIdx.x == 0 && (abort_flag || peer_abort_s)) {
    const uint32_t qhalf = (uint32_t)p.dqk * kBM;          // Q bytes of one producer (half a CTA's rows x d)
    int fq = 0;
    for (int pi = 0; pi < kProducers; ++pi) fq = max(fq, max(qfills_s[pi], peer_qfills_s[pi]));
    uint32_t qland = 0;
    for (int pi = 0; pi < kProducers; ++pi)
      qland += (qfills_s[pi] == fq ? qhalf : 0u) + (peer_qfills_s[pi] == fq ? qhalf : 0u);
    settle_last_phase(bar(kBarQFull), fq, qfills_s[0] == fq, 4u * qhalf, qland, kDrainSpin);
    // granule s of a ring of n has had one fill per round of loads reaching it
    auto rounds = [](int loads, int s, int n) { return loads > s ? (loads - 1 - s) / n + 1 : 0; };
    for (int pi = 0; pi < kProducers; ++pi) {
      const int base_slot = pi == 0 ? 0 : p.nk, n = pi == 0 ? p.nk : p.nv;
      for (int s2 = 0; s2 < n; ++s2) {
        const int fl = rounds(loads_s[pi], s2, n), fp = rounds(peer_loads_s[pi], s2, n), f = max(fl, fp);
        const uint32_t land = (fl == f ? (uint32_t)kSlotBytes : 0u) + (fp == f ? (uint32_t)kSlotBytes : 0u);
        settle_last_phase(bar(kBarFull + base_slot + s2), f, fl == f, 2u * kSlotBytes, land, kDrainSpin);
      }
    }
  }
  // every CTA is done with TMEM and with the others' shared memory
  tc_fence_before();
  cluster_sync_all();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
  if (threadIdx.x == 0) TRACE2(13, 0);
#ifdef MLSTM_TRACE
  if (threadIdx.x == 0 && rank == 0 && cid < 512) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    g_trace2_wall[2 * cid + 1] = t;
  }
#endif
}

#ifdef MLSTM_TRACE
}  // namespace
extern "C" int mlstm_trace2_set_cluster(int c) {
  return cudaMemcpyToSymbol(g_trace2_cluster, &c, sizeof(int)) == cudaSuccess ? 0 : -4;
}
extern "C" int mlstm_trace2_read(long long* host) {
  return cudaMemcpyFromSymbol(host, g_trace2, sizeof(g_trace2)) == cudaSuccess ? 0 : -4;
}
extern "C" int mlstm_trace2_set_item(int q) {
  return cudaMemcpyToSymbol(g_trace2_item, &q, sizeof(int)) == cudaSuccess ? 0 : -4;
}
extern "C" int mlstm_trace2_read_wall(unsigned long long* host) {
  return cudaMemcpyFromSymbol(host, g_trace2_wall, sizeof(g_trace2_wall)) == cudaSuccess ? 0 : -4;
}
namespace {
#endif

// Static shared memory of the kernel's instantiations (two CTAs or four), read once.
template <bool QUAD>
size_t static_smem() {
  static const size_t bytes = [] {
    size_t mx = 0;
    cudaFuncAttributes fa;
    if (!QUAD) {
      if (cudaFuncGetAttributes(&fa, fwd_tc2_kernel<1, false, false>) == cudaSuccess) mx = std::max(mx, fa.sharedSizeBytes);
      if (cudaFuncGetAttributes(&fa, fwd_tc2_kernel<1, true, false>) == cudaSuccess) mx = std::max(mx, fa.sharedSizeBytes);
    }
    if (cudaFuncGetAttributes(&fa, fwd_tc2_kernel<2, false, QUAD>) == cudaSuccess) mx = std::max(mx, fa.sharedSizeBytes);
    if (cudaFuncGetAttributes(&fa, fwd_tc2_kernel<2, true, QUAD>) == cudaSuccess) mx = std::max(mx, fa.sharedSizeBytes);
    cudaGetLastError();
    return mx > 0 ? mx : (size_t)4096;
  }();
  return bytes;
}

// Clusters that fit on the device at once with this shared-memory size
// (queried once per size and cluster size; SMs / cluster size if the query fails).
template <bool QUAD>
int resident_clusters(size_t smem) {
  constexpr int kCluster = QUAD ? 4 : 2;
  static std::mutex mu;
  static size_t last_smem = 0;
  static int last_dev = -1, last = 0;
  std::lock_guard<std::mutex> lock(mu);
  int dev = 0, sms = 0, n = 0;
  cudaGetDevice(&dev);
  if (last_smem == smem && last_dev == dev && last > 0) return last;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaFuncSetAttribute(fwd_tc2_kernel<2, false, QUAD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kCluster);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaOccupancyMaxActiveClusters(&n, fwd_tc2_kernel<2, false, QUAD>, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = std::max(1, sms / kCluster);
  }
  last_smem = smem;
  last_dev = dev;
  last = n;
  return n;
}

// The device's L2 size in bytes (queried once per device).
size_t l2_bytes() {
  static std::mutex mu;
  static int last_dev = -1;
  static size_t last = 0;
  std::lock_guard<std::mutex> lock(mu);
  int dev = 0, v = 0;
  cudaGetDevice(&dev);
  if (dev != last_dev) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) != cudaSuccess) {
      cudaGetLastError();
      v = 0;
    }
    last_dev = dev;
    last = (size_t)v;
  }
  return last;
}

template <int NSBUF, bool OG, bool QUAD>
int launch_pair(const FwdArgs& a, const Tc2Params& p, size_t smem, const CUtensorMap& mq, const CUtensorMap& mk,
                const CUtensorMap& mv, const CUtensorMap& mh, cudaStream_t stream) {
  constexpr int kCluster = QUAD ? 4 : 2;
  if (cudaFuncSetAttribute(fwd_tc2_kernel<NSBUF, OG, QUAD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return kCuda;
  const long long grid = (long long)kCluster * p.nclusters;   // persistent: each cluster loops over its items
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.after_gate_prep ? 2 : 1;
  if (cudaLaunchKernelEx(&cfg, fwd_tc2_kernel<NSBUF, OG, QUAD>, mq, mk, mv, mh, p) != cudaSuccess) return kCuda;
  return cudaGetLastError() == cudaSuccess ? kOk : kCuda;
}

// Fills the ring split and the grid of one form (two CTAs or four) and
// launches it; kUnsupported when its operands do not fit in shared memory.
template <bool QUAD>
int plan_and_launch(const FwdArgs& a, Tc2Params p, int nsbuf, cudaStream_t stream) {
  constexpr int kSlots = QUAD ? kQuadSlots : kMaxSlots;
  const size_t fixed = 1024 + (size_t)a.dqk * kBM * 2 + (size_t)kBN * kBM * 2;
  const long long room = (long long)kSmemLimit - (long long)static_smem<QUAD>() - (long long)fixed;
  const int total = (int)std::min<long long>(kSlots, room / kSlotBytes);
  if (total < (QUAD ? 4 : 2)) return kUnsupported;
  // split the granules between the rings in proportion to the bytes a key
  // tile needs from each (QUAD: K for every other tile only); two V granules
  // at least when chunks pair up (N=256)
  const int nkg = a.dqk / 128, nch = p.dv_slice / 128;
  p.nv = (int)lround((double)total * nch / ((QUAD ? 0.5 : 1.0) * nkg + nch));
  if (nch >= 2 && total >= 4) p.nv = std::max(p.nv, 2);
  p.nv = std::min(std::max(p.nv, 1), total - 1);
  p.nk = total - p.nv;
  const size_t smem = fixed + (size_t)total * kSlotBytes;
  const long long items = (long long)p.npairs * a.BH * p.nsplit;
  if (items > 0x7fffffffLL) return kInval;
  p.n_items = (int)items;
  p.nclusters = std::min(p.n_items, resident_clusters<QUAD>(smem));
#ifdef MLSTM_TRACE
  fprintf(stderr, "fwd_tc2: %d-CTA clusters %d (resident %d), items %d, rings K %d V %d, smem %zu\n", QUAD ? 4 : 2,
          p.nclusters, resident_clusters<QUAD>(smem), p.n_items, p.nk, p.nv, smem);
#endif
  CUtensorMap mq, mk, mv, mh;
  // K granules (64 keys x 128 d_qk) load as one 4-D box of two 64-column blocks
  if (!make_map_blocks(&mq, a.q, a.dqk, a.T, a.BH, kBM, a.dqk / 64 / kProducers) ||
      !make_map_blocks(&mk, a.k, a.dqk, a.T, a.BH, 64, 2) ||
      !make_map(&mv, a.v, a.dv, a.T, a.BH, kBN) || !make_map(&mh, a.h, a.dv, a.T, a.BH, kBM))
    return kCuda;
  if constexpr (QUAD) {
    return p.og ? launch_pair<2, true, true>(a, p, smem, mq, mk, mv, mh, stream)
                : launch_pair<2, false, true>(a, p, smem, mq, mk, mv, mh, stream);
  } else {
    if (p.og)
      return nsbuf == 1 ? launch_pair<1, true, false>(a, p, smem, mq, mk, mv, mh, stream)
                        : launch_pair<2, true, false>(a, p, smem, mq, mk, mv, mh, stream);
    return nsbuf == 1 ? launch_pair<1, false, false>(a, p, smem, mq, mk, mv, mh, stream)
                      : launch_pair<2, false, false>(a, p, smem, mq, mk, mv, mh, stream);
  }
}

}  // namespace

// The pair splits each 128-column V chunk and each 128-key K tile in halves
// of 64 (one swizzle atom), so d_qk and every d_v slice are multiples of 128.
bool fwd_tc2_supported(int dqk, int dv) {
  if (dqk % 128 != 0 || dqk > 512) return false;
  if (dv <= 384) return dv % 128 == 0;
  return dv == 512;
}

int launch_fwd_tc2(const FwdArgs& a, cudaStream_t stream) {
  Tc2Params p;
  p.a2 = a.g.a2; p.p2 = a.g.p2; p.mrow = a.g.m;
  p.m_out = a.m_out; p.n_out = a.n_out; p.b_out = a.b_out;
  p.og = static_cast<const __nv_bfloat16*>(a.og);
  p.T = a.T; p.BH = a.BH; p.dqk = a.dqk; p.dv = a.dv;
  const int nqt = (a.T + kBM - 1) / kBM;
  p.npairs = (nqt + 1) / 2;
  p.log2_scale = log2f(a.scale);
  p.st = a.st;
  // L2 prefetch of the ring's next key tile.  With d_v split over two CTA
  // pairs that both form S (two slices of a query block read the same K/V) it
  // measured 114.0 -> 107.7 us on the 350M-scale layer and 1150 -> 1116 us on
  // the T = 16384 workload (d = 512).  With one slice (d_v <= 384) it measured
  // ~1 us slower on the 125M-scale layer (109.4 against 110.9 us, three
  // alternating runs), so it is off there.  MLSTM_TC_L2PF=0 or 1 in the
  // environment overrides the choice.
  static const char* pf_env = getenv("MLSTM_TC_L2PF");
  if (a.dv == 512) {
    // four-CTA clusters forming S once and sending P across; MLSTM_TC_XCH=0
    // in the environment keeps the two-CTA form that forms S in both d_v
    // halves (comparison and tests)
    const char* xch = getenv("MLSTM_TC_XCH");   // read per call: tests switch it
    p.dv_slice = 256;
    if (!(xch && xch[0] == '0')) {
      // The four-CTA form prefetches where the layer's K and V take at most
      // three quarters of L2: on the 350M-scale layer (64 MiB) it measured
      // 102.4 -> 101.4 us, on the T = 16384 workload (128 MiB, all of L2)
      // 938 -> 991 us.
      const double kv = (double)a.BH * a.T * (a.dqk + a.dv) * 2.0;
      p.nsplit = 1;
      p.l2_prefetch = pf_env ? (pf_env[0] == '0' ? 0 : 1) : (kv <= 0.75 * (double)l2_bytes() ? 1 : 0);
      const int rc = plan_and_launch<true>(a, p, 2, stream);
      if (rc != kUnsupported) return rc;
    }
    p.nsplit = 2;
    p.l2_prefetch = pf_env ? (pf_env[0] == '0' ? 0 : 1) : 1;
    return plan_and_launch<false>(a, p, 2, stream);
  }
  p.nsplit = 1;
  p.dv_slice = a.dv;
  p.l2_prefetch = pf_env ? (pf_env[0] == '0' ? 0 : 1) : 0;
  return plan_and_launch<false>(a, p, a.dv <= 256 ? 2 : 1, stream);
}

}  // namespace mlstm
