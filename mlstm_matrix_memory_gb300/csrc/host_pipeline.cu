// The parallel forward on inputs and an output that live in host memory: the
// heads are processed in chunks whose uploads, compute and downloads overlap
// on three streams (the caller's stream computes; two cached streams copy),
// with two device buffers per operand taking turns.  The arithmetic is that
// of mlstm_parallel_fwd (each head is independent, so chunking by heads
// changes nothing in the result).
#include <algorithm>
#include <mutex>

#include "internal.h"
#include "mlstm.h"

namespace mlstm {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kChunks = 8;       // chunks of heads per call (at most)

size_t r256(size_t x) { return (x + 255) & ~(size_t)255; }

struct Slot {
  char* q;
  char* k;
  char* v;
  float* ig;
  float* fg;
  char* h;
  char* gate_ws;
};

struct Layout {
  int hc;                        // heads per chunk
  size_t q, k, v, g, h, ws;      // bytes of each per-slot array
  size_t slot;                   // bytes of one slot
};

Layout layout(int BH, int T, int dqk, int dv, int dtype) {
  Layout L;
  const int nc = BH < kChunks ? BH : kChunks;
  L.hc = (BH + nc - 1) / nc;
  const size_t es = dtype == MLSTM_F32 ? 4 : 2;
  const size_t tok = (size_t)L.hc * T;
  L.q = r256(tok * dqk * es);
  L.k = L.q;
  L.v = r256(tok * dv * es);
  L.g = r256(tok * sizeof(float));
  L.h = L.v;
  L.ws = r256(mlstm_parallel_fwd_workspace(1, L.hc, T));
  L.slot = L.q + L.k + L.v + 2 * L.g + L.h + L.ws;
  return L;
}

Slot slot_at(void* ws, const Layout& L, int s) {
  char* p = static_cast<char*>(ws) + (size_t)s * L.slot;
  Slot o;
  o.q = p;
  o.k = o.q + L.q;
  o.v = o.k + L.k;
  o.ig = reinterpret_cast<float*>(o.v + L.v);
  o.fg = reinterpret_cast<float*>(reinterpret_cast<char*>(o.ig) + L.g);
  o.h = reinterpret_cast<char*>(o.fg) + L.g;
  o.gate_ws = o.h + L.h;
  return o;
}

// Two copy streams and the events of the two slots, created once per device.
struct Engine {
  cudaStream_t up = nullptr, down = nullptr;
  cudaEvent_t entry = nullptr, up_done[2] = {}, comp_done[2] = {}, down_done[2] = {};
  bool ready = false;
};
Engine g_engine[kMaxDevices];
std::mutex g_engine_mu;

bool engine_init(Engine& e) {
  if (e.ready) return true;
  const unsigned fl = cudaEventDisableTiming;
  if (cudaStreamCreateWithFlags(&e.up, cudaStreamNonBlocking) != cudaSuccess) return false;
  if (cudaStreamCreateWithFlags(&e.down, cudaStreamNonBlocking) != cudaSuccess) return false;
  if (cudaEventCreateWithFlags(&e.entry, fl) != cudaSuccess) return false;
  for (int s = 0; s < 2; ++s)
    if (cudaEventCreateWithFlags(&e.up_done[s], fl) != cudaSuccess ||
        cudaEventCreateWithFlags(&e.comp_done[s], fl) != cudaSuccess ||
        cudaEventCreateWithFlags(&e.down_done[s], fl) != cudaSuccess)
      return false;
  e.ready = true;
  return true;
}

}  // namespace
}  // namespace mlstm

using namespace mlstm;

extern "C" {

size_t mlstm_parallel_fwd_host_workspace(int B, int H, int T, int d_qk, int d_v, int dtype) {
  if (B <= 0 || H <= 0 || T <= 0 || d_qk <= 0 || d_v <= 0) return 0;
  if (dtype != MLSTM_F32 && dtype != MLSTM_BF16) return 0;
  return 2 * layout(B * H, T, d_qk, d_v, dtype).slot;
}

int mlstm_parallel_fwd_host(const void* q, const void* k, const void* v, const float* igate_pre,
                            const float* fgate_pre, void* h, int B, int H, int T, int d_qk, int d_v, int dtype,
                            void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || H < 0 || T < 0) return MLSTM_EINVAL;
  if (d_qk < 1 || d_v < 1 || d_qk > 512 || d_v > 512) return MLSTM_EINVAL;
  if (dtype != MLSTM_F32 && dtype != MLSTM_BF16) return MLSTM_EDTYPE;
  const long long BH = (long long)B * H;
  if (BH > 0x7fffffffLL || BH * T > (1LL << 40)) return MLSTM_EINVAL;
  if (BH == 0 || T == 0) return MLSTM_OK;
  if (!q || !k || !v || !igate_pre || !fgate_pre || !h) return MLSTM_EINVAL;
  if (!workspace || workspace_bytes < mlstm_parallel_fwd_host_workspace(B, H, T, d_qk, d_v, dtype))
    return MLSTM_EWORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return MLSTM_EALIGN;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLSTM_ECUDA;

  std::lock_guard<std::mutex> lock(g_engine_mu);   // the cached events are shared per device
  Engine& e = g_engine[dev];
  if (!engine_init(e)) return MLSTM_ECUDA;
  cudaStream_t comp = static_cast<cudaStream_t>(stream);
  const Layout L = layout((int)BH, T, d_qk, d_v, dtype);
  const size_t es = dtype == MLSTM_F32 ? 4 : 2;
  const int nchunks = (int)((BH + L.hc - 1) / L.hc);
  auto ck = [](cudaError_t r) { return r == cudaSuccess; };

  // the uploads start after whatever the caller queued before this call
  if (!ck(cudaEventRecord(e.entry, comp)) || !ck(cudaStreamWaitEvent(e.up, e.entry, 0))) return MLSTM_ECUDA;
  for (int c = 0; c < nchunks; ++c) {
    const int s = c & 1;
    const Slot sl = slot_at(workspace, L, s);
    const long long h0 = (long long)c * L.hc;
    const int hn = (int)std::min<long long>(L.hc, BH - h0);
    const size_t tok0 = (size_t)h0 * T, ntok = (size_t)hn * T;
    // upload: the slot's inputs were last read by the compute of chunk c-2
    if (c >= 2 && !ck(cudaStreamWaitEvent(e.up, e.comp_done[s], 0))) return MLSTM_ECUDA;
    if (!ck(cudaMemcpyAsync(sl.q, static_cast<const char*>(q) + tok0 * d_qk * es, ntok * d_qk * es,
                            cudaMemcpyHostToDevice, e.up)) ||
        !ck(cudaMemcpyAsync(sl.k, static_cast<const char*>(k) + tok0 * d_qk * es, ntok * d_qk * es,
                            cudaMemcpyHostToDevice, e.up)) ||
        !ck(cudaMemcpyAsync(sl.v, static_cast<const char*>(v) + tok0 * d_v * es, ntok * d_v * es,
                            cudaMemcpyHostToDevice, e.up)) ||
        !ck(cudaMemcpyAsync(sl.ig, igate_pre + tok0, ntok * sizeof(float), cudaMemcpyHostToDevice, e.up)) ||
        !ck(cudaMemcpyAsync(sl.fg, fgate_pre + tok0, ntok * sizeof(float), cudaMemcpyHostToDevice, e.up)) ||
        !ck(cudaEventRecord(e.up_done[s], e.up)))
      return MLSTM_ECUDA;
    // compute: needs the uploads, and the slot's output read out (chunk c-2)
    if (!ck(cudaStreamWaitEvent(comp, e.up_done[s], 0))) return MLSTM_ECUDA;
    if (c >= 2 && !ck(cudaStreamWaitEvent(comp, e.down_done[s], 0))) return MLSTM_ECUDA;
    const int rc = mlstm_parallel_fwd(sl.q, sl.k, sl.v, sl.ig, sl.fg, sl.h, nullptr, nullptr, 1, hn, T, d_qk, d_v,
                                      dtype, sl.gate_ws, L.ws, comp);
    if (rc != MLSTM_OK) return rc;
    if (!ck(cudaEventRecord(e.comp_done[s], comp))) return MLSTM_ECUDA;
    // download
    if (!ck(cudaStreamWaitEvent(e.down, e.comp_done[s], 0)) ||
        !ck(cudaMemcpyAsync(static_cast<char*>(h) + tok0 * d_v * es, sl.h, ntok * d_v * es, cudaMemcpyDeviceToHost,
                            e.down)) ||
        !ck(cudaEventRecord(e.down_done[s], e.down)))
      return MLSTM_ECUDA;
  }
  // the caller's stream completes after every download
  for (int s = 0; s < 2 && s < nchunks; ++s)
    if (!ck(cudaStreamWaitEvent(comp, e.down_done[s], 0))) return MLSTM_ECUDA;
  return MLSTM_OK;
}

}  // extern "C"
