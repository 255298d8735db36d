// C-ABI entry points of libmlstm.so (declared in include/mlstm.h): argument
// checks on the host, workspace carving, kernel choice and launch.  Nothing
// here computes on the host; every step of the path runs in the kernels.
#include <atomic>
#include <mutex>
#include <stdint.h>
#include <math.h>

#include "../../include/mlstm.h"
#include "internal.h"

namespace mlstm {

// Device status word {code, site}, one per device (a __device__ variable is
// instantiated on every device that loads the library).
__device__ int g_status[2];

namespace {

constexpr long long kDefaultSpin = 1LL << 22;
std::atomic<long long> g_spin_limit{kDefaultSpin};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_status_ptr[kMaxDevices] = {};

// Device address of g_status on the current device (looked up once per device).
int status_ptr(int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return kCuda;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return kCuda;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  *out = g_status_ptr[dev];
  return kOk;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

size_t gate_array_bytes(long long BHT) { return round256((size_t)BHT * sizeof(float)); }

}  // namespace

bool current_status(DevStatus* out) {
  int* status = nullptr;
  if (status_ptr(&status) != kOk) return false;
  out->word = status;
  out->spin_limit = g_spin_limit.load();
  return true;
}

}  // namespace mlstm

using namespace mlstm;

extern "C" {

int mlstm_version(void) { return 100; }

const char* mlstm_status_str(int s) {
  switch (s) {
    case MLSTM_OK: return "ok";
    case MLSTM_EINVAL: return "invalid argument";
    case MLSTM_EALIGN: return "pointer not 16-byte aligned";
    case MLSTM_EDTYPE: return "unsupported dtype";
    case MLSTM_ECUDA: return "CUDA call failed";
    case MLSTM_ETIMEOUT: return "a kernel's bounded wait ran out";
    case MLSTM_EUNSUPPORTED: return "shape, dtype or device not supported by the chosen kernel";
    case MLSTM_EWORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

long long mlstm_set_spin_limit(long long limit) {
  return g_spin_limit.exchange(limit > 0 ? limit : kDefaultSpin);
}

size_t mlstm_parallel_fwd_workspace(int B, int H, int T) {
  if (B < 0 || H < 0 || T < 0) return 0;
  const long long BHT = (long long)B * H * T;
  return 3 * gate_array_bytes(BHT);
}

namespace {

int check_sizes(int B, int H, int T) {
  if (B < 0 || H < 0 || T < 0) return MLSTM_EINVAL;
  const long long BH = (long long)B * H;
  if (BH > 0x7fffffffLL || BH * T > (1LL << 40)) return MLSTM_EINVAL;
  return MLSTM_OK;
}

GateTerms carve(const void* workspace, long long BHT) {
  const size_t arr = gate_array_bytes(BHT);
  char* ws = static_cast<char*>(const_cast<void*>(workspace));
  return GateTerms{reinterpret_cast<float*>(ws), reinterpret_cast<float*>(ws + arr),
                   reinterpret_cast<float*>(ws + 2 * arr)};
}

}  // namespace

int mlstm_gate_prep_opt(const float* igate_pre, const float* fgate_pre, int B, int H, int T, void* workspace,
                        size_t workspace_bytes, const mlstm_options* opt, void* stream) {
  int rc = check_sizes(B, H, T);
  if (rc != MLSTM_OK) return rc;
  const long long BH = (long long)B * H, BHT = BH * T;
  if (BHT == 0) return MLSTM_OK;
  if (!igate_pre || !fgate_pre) return MLSTM_EINVAL;
  if (!workspace || workspace_bytes < mlstm_parallel_fwd_workspace(B, H, T)) return MLSTM_EWORKSPACE;
  if (!aligned16(workspace)) return MLSTM_EALIGN;
  return launch_gate_prep(igate_pre, fgate_pre, carve(workspace, BHT), (int)BH, T, opt ? opt->forget_exp : 0,
                          static_cast<cudaStream_t>(stream)) == cudaSuccess ? MLSTM_OK : MLSTM_ECUDA;
}

int mlstm_gate_prep(const float* igate_pre, const float* fgate_pre, int B, int H, int T, void* workspace,
                    size_t workspace_bytes, void* stream) {
  return mlstm_gate_prep_opt(igate_pre, fgate_pre, B, H, T, workspace, workspace_bytes, nullptr, stream);
}

namespace {

int fwd_gated(const void* q, const void* k, const void* v, void* h, float* m_out, float* n_out, int B, int H,
              int T, int d_qk, int d_v, int dtype, const void* workspace, size_t workspace_bytes, int algo,
              bool after_gate_prep, const void* og, void* stream, float* b_out = nullptr) {
  int rc = check_sizes(B, H, T);
  if (rc != MLSTM_OK) return rc;
  if (d_qk < 1 || d_v < 1 || d_qk > 512 || d_v > 512) return MLSTM_EINVAL;
  if (dtype != MLSTM_F32 && dtype != MLSTM_BF16) return MLSTM_EDTYPE;
  const int vec = dtype == MLSTM_F32 ? 4 : 8;   // 16-byte rows
  if (d_qk % vec != 0 || d_v % vec != 0) return MLSTM_EINVAL;
  if (algo < MLSTM_ALGO_AUTO || algo > MLSTM_ALGO_TC) return MLSTM_EINVAL;
  const long long BH = (long long)B * H, BHT = BH * T;
  if (BHT == 0) return MLSTM_OK;
  if (!q || !k || !v || !h) return MLSTM_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(h)) return MLSTM_EALIGN;
  if (og && !aligned16(og)) return MLSTM_EALIGN;
  if (!workspace || workspace_bytes < mlstm_parallel_fwd_workspace(B, H, T)) return MLSTM_EWORKSPACE;
  if (!aligned16(workspace)) return MLSTM_EALIGN;

  const bool tc_ok = fwd_tc_supported(d_qk, d_v, dtype);
  bool use_tc;
  if (algo == MLSTM_ALGO_TC) {
    if (!tc_ok) return MLSTM_EUNSUPPORTED;
    use_tc = true;
  } else {
    use_tc = algo == MLSTM_ALGO_AUTO && tc_ok;
  }
  int* status = nullptr;
  if (status_ptr(&status) != kOk) return MLSTM_ECUDA;
  FwdArgs a;
  a.q = q; a.k = k; a.v = v; a.h = h; a.m_out = m_out; a.n_out = n_out; a.g = carve(workspace, BHT);
  a.BH = (int)BH; a.T = T; a.dqk = d_qk; a.dv = d_v; a.dtype = dtype;
  a.scale = (float)(1.0 / sqrt((double)d_qk));
  a.st.word = status;
  a.st.spin_limit = g_spin_limit.load();
  a.after_gate_prep = after_gate_prep;
  a.og = og;
  a.b_out = b_out;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (use_tc) return launch_fwd_tc(a, s);
  if (launch_fwd_simt(a, s) != cudaSuccess) return MLSTM_ECUDA;
  // the CUDA-core kernel does not fuse the output gate
  return launch_apply_ogate(h, og, BHT * d_v, dtype, s) == cudaSuccess ? MLSTM_OK : MLSTM_ECUDA;
}

}  // namespace

int mlstm_parallel_fwd_gated(const void* q, const void* k, const void* v, void* h, float* m_out, float* n_out,
                             int B, int H, int T, int d_qk, int d_v, int dtype, const void* workspace,
                             size_t workspace_bytes, int algo, void* stream) {
  return fwd_gated(q, k, v, h, m_out, n_out, B, H, T, d_qk, d_v, dtype, workspace, workspace_bytes, algo, false,
                   nullptr, stream);
}

int mlstm_parallel_fwd_opt(const void* q, const void* k, const void* v, const float* igate_pre,
                           const float* fgate_pre, void* h, float* m_out, float* n_out, int B, int H, int T,
                           int d_qk, int d_v, int dtype, void* workspace, size_t workspace_bytes,
                           const mlstm_options* opt, void* stream) {
  const int algo = opt ? opt->algo : MLSTM_ALGO_AUTO;
  const void* og = opt ? opt->ogate_pre : nullptr;
  int rc = check_sizes(B, H, T);
  if (rc != MLSTM_OK) return rc;
  if (d_qk < 1 || d_v < 1 || d_qk > 512 || d_v > 512) return MLSTM_EINVAL;
  if (dtype != MLSTM_F32 && dtype != MLSTM_BF16) return MLSTM_EDTYPE;
  const int vec = dtype == MLSTM_F32 ? 4 : 8;
  if (d_qk % vec != 0 || d_v % vec != 0) return MLSTM_EINVAL;
  if (algo < MLSTM_ALGO_AUTO || algo > MLSTM_ALGO_TC) return MLSTM_EINVAL;
  if ((long long)B * H * T == 0) return MLSTM_OK;
  if (!q || !k || !v || !igate_pre || !fgate_pre || !h) return MLSTM_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(h)) return MLSTM_EALIGN;
  if (og && !aligned16(og)) return MLSTM_EALIGN;          // before the gate pass writes the workspace
  if (!workspace || workspace_bytes < mlstm_parallel_fwd_workspace(B, H, T)) return MLSTM_EWORKSPACE;
  if (!aligned16(workspace)) return MLSTM_EALIGN;
  if (algo == MLSTM_ALGO_TC && !fwd_tc_supported(d_qk, d_v, dtype)) return MLSTM_EUNSUPPORTED;
  rc = mlstm_gate_prep_opt(igate_pre, fgate_pre, B, H, T, workspace, workspace_bytes, opt, stream);
  if (rc != MLSTM_OK) return rc;
  return fwd_gated(q, k, v, h, m_out, n_out, B, H, T, d_qk, d_v, dtype, workspace, workspace_bytes, algo, true,
                   og, stream, opt ? opt->b_out : nullptr);
}

int mlstm_parallel_fwd_ex(const void* q, const void* k, const void* v, const float* igate_pre,
                          const float* fgate_pre, void* h, float* m_out, float* n_out, int B, int H, int T,
                          int d_qk, int d_v, int dtype, void* workspace, size_t workspace_bytes, int algo,
                          void* stream) {
  mlstm_options o = {};
  o.algo = algo;
  return mlstm_parallel_fwd_opt(q, k, v, igate_pre, fgate_pre, h, m_out, n_out, B, H, T, d_qk, d_v, dtype,
                                workspace, workspace_bytes, &o, stream);
}

int mlstm_parallel_fwd(const void* q, const void* k, const void* v, const float* igate_pre,
                       const float* fgate_pre, void* h, float* m_out, float* n_out, int B, int H, int T,
                       int d_qk, int d_v, int dtype, void* workspace, size_t workspace_bytes,
                       void* stream) {
  return mlstm_parallel_fwd_ex(q, k, v, igate_pre, fgate_pre, h, m_out, n_out, B, H, T, d_qk, d_v, dtype,
                               workspace, workspace_bytes, MLSTM_ALGO_AUTO, stream);
}

int mlstm_parallel_final_state(const void* k, const void* v, const void* workspace, size_t workspace_bytes,
                               float* C, float* n, float* m, int B, int H, int T, int d_qk, int d_v, int dtype,
                               void* stream) {
  int rc = check_sizes(B, H, T);
  if (rc != MLSTM_OK) return rc;
  if (d_qk < 1 || d_v < 1 || d_qk > 512 || d_v > 512) return MLSTM_EINVAL;
  if (dtype != MLSTM_F32 && dtype != MLSTM_BF16) return MLSTM_EDTYPE;
  const long long BH = (long long)B * H, BHT = BH * T;
  if (BH == 0) return MLSTM_OK;
  if (T < 1) return MLSTM_EINVAL;
  if (!k || !v || !C || !n || !m) return MLSTM_EINVAL;
  if (!aligned16(C) || !aligned16(n) || !aligned16(k) || !aligned16(v)) return MLSTM_EALIGN;
  if (!workspace || workspace_bytes < mlstm_parallel_fwd_workspace(B, H, T)) return MLSTM_EWORKSPACE;
  if (!aligned16(workspace)) return MLSTM_EALIGN;
  int* status = nullptr;
  if (status_ptr(&status) != kOk) return MLSTM_ECUDA;
  DevStatus st;
  st.word = status;
  st.spin_limit = g_spin_limit.load();
  return launch_final_state(k, v, carve(workspace, BHT), C, n, m, (int)BH, T, d_qk, d_v, dtype,
                            (float)(1.0 / sqrt((double)d_qk)), st, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MLSTM_OK
             : MLSTM_ECUDA;
}

int mlstm_step(float* C, float* n, float* m, const void* q, const void* k, const void* v, const void* o,
               const float* igate_pre, const float* fgate_pre, void* h, int B, int H, int d_qk, int d_v,
               int dtype, void* stream) {
  if (B < 0 || H < 0) return MLSTM_EINVAL;
  if (d_qk < 1 || d_v < 1 || d_qk > 512 || d_v > 512 || d_qk % 8 != 0) return MLSTM_EINVAL;
  if (dtype != MLSTM_F32 && dtype != MLSTM_BF16) return MLSTM_EDTYPE;
  const long long BH = (long long)B * H;
  if (BH > (1LL << 28)) return MLSTM_EINVAL;
  if (BH == 0) return MLSTM_OK;
  if (!C || !n || !m || !q || !k || !v || !igate_pre || !fgate_pre || !h) return MLSTM_EINVAL;
  if (!aligned16(C) || !aligned16(n) || !aligned16(q) || !aligned16(k)) return MLSTM_EALIGN;
  StepArgs a;
  a.C = C; a.n = n; a.m = m; a.q = q; a.k = k; a.v = v; a.o = o; a.ig = igate_pre; a.fg = fgate_pre;
  a.h = h; a.BH = (int)BH; a.dqk = d_qk; a.dv = d_v; a.dtype = dtype;
  a.scale = (float)(1.0 / sqrt((double)d_qk));
  return launch_step(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? MLSTM_OK : MLSTM_ECUDA;
}

int mlstm_step_seq_opt(float* C, float* n, float* m, const void* q, const void* k, const void* v, const void* o,
                       const float* igate_pre, const float* fgate_pre, void* h, int B, int H, int L, int d_qk,
                       int d_v, int dtype, const mlstm_options* opt, void* stream) {
  if (B < 0 || H < 0 || L < 0) return MLSTM_EINVAL;
  if (d_qk < 1 || d_v < 1 || d_qk > 512 || d_v > 512 || d_qk % 8 != 0) return MLSTM_EINVAL;
  if (dtype != MLSTM_F32 && dtype != MLSTM_BF16) return MLSTM_EDTYPE;
  const long long BH = (long long)B * H;
  if (BH > (1LL << 28) || BH * (long long)L > (1LL << 40)) return MLSTM_EINVAL;
  if (BH == 0 || L == 0) return MLSTM_OK;
  if (!C || !n || !m || !q || !k || !v || !igate_pre || !fgate_pre || !h) return MLSTM_EINVAL;
  if (!aligned16(C) || !aligned16(n) || !aligned16(q) || !aligned16(k)) return MLSTM_EALIGN;
  StepArgs a;
  a.C = C; a.n = n; a.m = m; a.q = q; a.k = k; a.v = v; a.o = o; a.ig = igate_pre; a.fg = fgate_pre;
  a.h = h; a.BH = (int)BH; a.dqk = d_qk; a.dv = d_v; a.dtype = dtype;
  a.scale = (float)(1.0 / sqrt((double)d_qk));
  a.forget_exp = opt ? opt->forget_exp : 0;
  return launch_step_seq(a, L, static_cast<cudaStream_t>(stream)) == cudaSuccess ? MLSTM_OK : MLSTM_ECUDA;
}

int mlstm_step_seq(float* C, float* n, float* m, const void* q, const void* k, const void* v, const void* o,
                   const float* igate_pre, const float* fgate_pre, void* h, int B, int H, int L, int d_qk,
                   int d_v, int dtype, void* stream) {
  return mlstm_step_seq_opt(C, n, m, q, k, v, o, igate_pre, fgate_pre, h, B, H, L, d_qk, d_v, dtype, nullptr,
                            stream);
}

int mlstm_last_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MLSTM_ECUDA;
  int* status = nullptr;
  if (status_ptr(&status) != kOk) return MLSTM_ECUDA;
  int host[2] = {0, 0};
  if (cudaMemcpy(host, status, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess) return MLSTM_ECUDA;
  if (host[0] != 0) {
    const int zero[2] = {0, 0};
    if (cudaMemcpy(status, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return MLSTM_ECUDA;
  }
  return host[0];
}

}  // extern "C"
