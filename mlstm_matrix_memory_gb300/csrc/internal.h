// Host-side launch interfaces between the C-ABI layer (api.cu) and the
// kernels.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace mlstm {

// Per-token gate terms of one sequence set, produced by gate_prep, each
// [B*H*T] fp32 (see gate_prep.cu):
//   a2[t] = (i~_t - cs_t) * log2(e)                 column term of D~ - m
//   p2[t] = max_{j<=t} a2[j]                        row term of D~ - m
//   m[t]  = cs_t + max_{j<=t}(i~_j - cs_j)          row max of D~ (eq 80)
// with cs_t = sum_{k<=t} log sigmoid(f~_k).  Then for j <= i:
//   D~_ij - m_i = (a2[j] - p2[i]) / log2(e)  <= 0.
struct GateTerms {
  float* a2;
  float* p2;
  float* m;
};

struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  void* h;
  float* m_out;   // may be null
  float* n_out;   // may be null
  float* b_out = nullptr;   // signed row sums b (eq 83), or null (used by the backward)
  GateTerms g;
  int BH, T, dqk, dv;
  int dtype;      // kF32 / kBF16
  float scale;    // 1/sqrt(dqk)
  DevStatus st;
  const void* og = nullptr;       // output-gate pre-activations [BH,T,dv] (dtype), or null
  bool after_gate_prep = false;   // launched right after gate_prep on the same stream:
                                  // may overlap its prologue with it (programmatic
                                  // dependent launch; gate terms are read after the wait)
};

struct StepArgs {
  float* C;
  float* n;
  float* m;
  const void* q;
  const void* k;
  const void* v;
  const void* o;  // may be null
  const float* ig;
  const float* fg;
  void* h;
  int BH, dqk, dv;
  int dtype;
  float scale;
  int forget_exp = 0;   // 1: log f = f~ (exponential forget activation)
};

cudaError_t launch_gate_prep(const float* ig, const float* fg, GateTerms g, int BH, int T, int forget_exp,
                             cudaStream_t stream);
cudaError_t launch_fwd_simt(const FwdArgs& a, cudaStream_t stream);
bool fwd_tc_supported(int dqk, int dv, int dtype);
int launch_fwd_tc(const FwdArgs& a, cudaStream_t stream);   // returns a Status
cudaError_t launch_step(const StepArgs& a, cudaStream_t stream);
// L steps per head; q/k/v/o/gates/h carry a token axis of length L.
cudaError_t launch_step_seq(const StepArgs& a, int L, cudaStream_t stream);
// (C, n, m) after the last token, from the gate terms of the whole sequence.
cudaError_t launch_final_state(const void* k, const void* v, GateTerms g, float* C, float* n, float* m, int BH,
                               int T, int dqk, int dv, int dtype, float scale, DevStatus st, cudaStream_t stream);
// h *= sigmoid(o) elementwise (the output gate, eq 78), for the kernels that
// do not apply it in their epilogue.
cudaError_t launch_apply_ogate(void* h, const void* og, long long n, int dtype, cudaStream_t stream);
// Backward of the output gate (ogate.cu): dht = dh (.) sigmoid(og), and
// dog = dh (.) ht (.) sigmoid'(og), n elements of dtype each.
cudaError_t launch_ogate_bwd_in(const void* dh, const void* og, void* dht, long long n, int dtype,
                                cudaStream_t stream);
cudaError_t launch_ogate_bwd_out(const void* dh, const void* og, const void* ht, void* dog, long long n, int dtype,
                                 cudaStream_t stream);
// 1 when the current device runs tcgen05 code (sm_100 family).
int device_is_sm100_family();

// CTA-pair (cta_group::2) variant of the tensor-core forward (fwd_tc2.cu).
bool fwd_tc2_supported(int dqk, int dv);
int launch_fwd_tc2(const FwdArgs& a, cudaStream_t stream);

// The device status word and the current spin limit (false: no status word).
bool current_status(DevStatus* out);

// Tiles of the parallel backward on the tensor cores (bwd_tc.cu): from the
// gate terms and the forward's row statistics, writes G = D' (.) dC~' and
// P = C~'/n (bf16, [BH, T, ldT]: the tiles on and below the diagonal, zero
// above it within the diagonal tiles) and the row and column sums R, Ccol of
// dD~ = S (.) G.  Returns a Status.
struct BwdTileArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* dh;
  const void* h;        // H~ of the forward [BH, T, dv]
  const float* nrow;    // n_i of the forward
  const float* brow;    // signed b_i of the forward
  GateTerms g;
  float* invn;          // scratch [BH*T]
  float* db;            // scratch [BH*T]
  void* G;
  void* P;
  float* Rpart;         // scratch [BH][nb][T]
  float* Cpart;         // scratch [BH][nb][T]
  float* R;             // out [BH*T]
  float* Ccol;          // out [BH*T]
  int BH, T, ldT, dqk, dv;
  float scale;
  DevStatus st;
};
// dQ = s G K, dK = s G^T Q, dV = P^T dH over the lower triangle of G and P
// (bf16, [BH, T, ldT]), tensor cores (bwd_tc.cu).  Returns a Status.
struct BwdProdArgs {
  const void* q;
  const void* k;
  const void* dh;
  const void* G;
  const void* P;
  void* dq;
  void* dk;
  void* dvo;
  int BH, T, ldT, dqk, dv;
  float scale;
  DevStatus st;
};
int launch_bwd_products(const BwdProdArgs& a, cudaStream_t stream);
bool bwd_tc_supported(int T, int dqk, int dv, int dtype);
int launch_bwd_tiles(const BwdTileArgs& a, cudaStream_t stream);

// 3-D TMA map over [BH, rows, cols] bf16 with row pitch ld elements (ld*2 a
// multiple of 16), box 64 x box_rows x 1, 128-byte swizzle (fwd_tc.cu).
bool make_map_ld(CUtensorMap* m, const void* base, int cols, int rows, int BH, int ld, int box_rows);

// 3-D TMA map over a [BH, T, d] bf16 tensor, box 64 x rows x 1, 128-byte
// swizzle; rows past T read as zeros and are clipped on stores (fwd_tc.cu).
bool make_map(CUtensorMap* m, const void* base, int d, int T, int BH, int rows);
// [BH, T, d] bf16 as 4-D (64 columns, T, d / 64 blocks, BH): one box is
// `blocks` consecutive 64-column x rows tiles (128-byte swizzle).
bool make_map_blocks(CUtensorMap* m, const void* base, int d, int T, int BH, int rows, int blocks);
// [BH, rows, cols] bf16 with row pitch ld as 4-D (64 columns, rows, cols / 64
// blocks, BH); cols a multiple of 64.
bool make_map_ld_blocks(CUtensorMap* m, const void* base, int cols, int rows, int BH, int ld, int box_rows,
                        int blocks);
// [BH, rows, cols] fp32 (cols fastest), box box_cols x box_rows x 1, 128-byte swizzle.
bool make_map_f32(CUtensorMap* m, float* base, int cols, int rows, int BH, int box_cols, int box_rows);

}  // namespace mlstm
