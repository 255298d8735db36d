// Allocation-free variant of the parallel forward pass.
//
// Some callers cannot call cudaMalloc: code running where the allocator is
// off limits (inside a custom memory pool's own callbacks, on a stream being
// captured by another library that forbids new allocations, in plug-ins whose
// host application owns all device memory, or under a strict memory budget
// that counts every allocation).  For them, mlstm_parallel_fwd_noalloc keeps
// the gate-term scratch of the parallel forward in a fixed array compiled
// into this library, so the caller passes only inputs and outputs.
//
// The array lives in device memory on every GPU that loads the library and
// stays there until the process exits.  Host code cannot use the array's name
// as a device address; the address is looked up once per device with
// cudaGetSymbolAddress and cached.
#include <mutex>
#include <stdint.h>

#include "../../include/mlstm.h"
#include "internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[MLSTM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device; looked up the
// first time each device is used.
int scratch_ptr(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLSTM_ECUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MLSTM_ECUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MLSTM_OK;
}

}  // namespace

extern "C" int mlstm_parallel_fwd_noalloc(const void* q, const void* k, const void* v, const float* igate_pre,
                                          const float* fgate_pre, void* h, float* m_out, float* n_out, int B,
                                          int H, int T, int d_qk, int d_v, int dtype, void* stream) {
  // the shape checks of mlstm_parallel_fwd (the same bounds on B*H and
  // B*H*T, so no product below can overflow), before the scratch is touched
  if (B < 0 || H < 0 || T < 0) return MLSTM_EINVAL;
  const long long BH = (long long)B * H;
  if (BH > 0x7fffffffLL || BH * T > (1LL << 40)) return MLSTM_EINVAL;
  if (d_qk < 1 || d_v < 1 || d_qk > 512 || d_v > 512) return MLSTM_EINVAL;
  if (dtype != MLSTM_F32 && dtype != MLSTM_BF16) return MLSTM_EDTYPE;
  const int vec = dtype == MLSTM_F32 ? 4 : 8;
  if (d_qk % vec != 0 || d_v % vec != 0) return MLSTM_EINVAL;
  if (BH * T == 0) return MLSTM_OK;
  const size_t need = mlstm_parallel_fwd_workspace(B, H, T);
  if (need == 0 || need > (size_t)MLSTM_NOALLOC_SCRATCH_BYTES) return MLSTM_EWORKSPACE;
  void* scratch = nullptr;
  const int rc = scratch_ptr(&scratch);
  if (rc != MLSTM_OK) return rc;
  // The gate pass overwrites every scratch entry the fused pass reads, so the
  // previous call's contents never need clearing.
  return mlstm_parallel_fwd(q, k, v, igate_pre, fgate_pre, h, m_out, n_out, B, H, T, d_qk, d_v, dtype, scratch,
                            need, stream);
}
