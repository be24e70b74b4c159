// Allocation-free speculative-sampling verification.
//
// Some callers cannot allocate device memory at the point where they verify:
// an allocator-less runtime embedding this library, code running inside an
// arena it does not own, or a serving loop that forbids cudaMalloc on its hot
// path because it synchronises the device. For them, dlite_verify_sample_static
// runs the same verification kernel as dlite_verify_sample without a handle and
// without any allocation: the one scratch buffer that kernel needs (the
// fixed-point residual row of the rare exact fallback draw) is this file's
// static device array below. The caller passes every input and output.
#include <math.h>

#include <mutex>

#include "kernels.h"

namespace {

// Residual scratch: B * V fixed-point entries at most (8 MiB). Every GPU that
// loads the library holds this array until the process exits.
constexpr size_t kResidCap = (size_t)1 << 20;
static __device__ __align__(256) unsigned long long g_resid_scratch[kResidCap];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device; looked up once
// per device (host code cannot use the symbol itself as a device pointer).
// The cached address belongs to the device's context of that first call: it
// does not survive cudaDeviceReset (the header says so).
int scratch_for_current_device(unsigned long long** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DLITE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_resid_scratch) != cudaSuccess || !p) return DLITE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = (unsigned long long*)g_scratch_addr[dev];
  return DLITE_OK;
}

}  // namespace

extern "C" int dlite_verify_sample_static(int B, int K, int V, int D, const int32_t* candidates,
                                          const dlite_qstats* qstats, const float* hs,
                                          const float* E, const float* target_probs,
                                          float temperature, uint64_t seed, const int64_t* pos,
                                          int32_t* accepted, int32_t* commits, int32_t* n_commit,
                                          int32_t* next_anchor, dlite_stream_t stream) {
  if (!candidates || !qstats || !hs || !E || !target_probs || !pos || !accepted || !commits ||
      !n_commit || !next_anchor)
    return DLITE_ERR_INVALID_ARG;
  if (B < 1 || K < 1 || K > 31 || V < 8 || V % 8 || V > 262144 || D < 4 || D % 4)
    return DLITE_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || isinf(temperature)) return DLITE_ERR_INVALID_ARG;
  // E, hs and the probability rows are read with 16-byte vector loads
  if (((uintptr_t)E | (uintptr_t)hs | (uintptr_t)target_probs) & 15) return DLITE_ERR_INVALID_ARG;
  if ((size_t)B * (size_t)V > kResidCap) return DLITE_ERR_UNSUPPORTED_SHAPE;  // scratch too small
  unsigned long long* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc) return rc;
  dlite::VerifyArgs v;
  v.B = B;
  v.K = K;
  v.V = V;
  v.D = D;
  v.cand = candidates;
  v.qs = qstats;
  v.hs = hs;
  v.probs = target_probs;
  v.Ef = E;
  v.resid = scratch;  // fully written before it is read: nothing to clear between calls
  v.counters = nullptr;
  v.T = (double)temperature;
  v.k0 = (uint32_t)(seed & 0xffffffffu);
  v.k1 = (uint32_t)(seed >> 32);
  v.pos = pos;
  v.accepted = accepted;
  v.commits = commits;
  v.n_commit = n_commit;
  v.next_anchor = next_anchor;
  v.status = nullptr;  // no handle, so no status word: see the header on out-of-range candidates
  if (dlite::launch_verify_sample(v, (cudaStream_t)stream) != cudaSuccess) return DLITE_ERR_CUDA;
  return DLITE_OK;
}
