// noalloc.cu -- greedy verification for callers that cannot allocate device memory.
//
// Some hosts of this library have no way to hand it a workspace: a plug-in running inside an
// inference engine that reserves all device memory up front and forbids later allocation, a
// real-time loop in which the implicit synchronisation of cudaMalloc would stall the pipeline,
// or a caller whose memory belongs to another framework's allocator that it cannot reach from
// this call site. spec_verify_greedy_noalloc serves them: its scratch (one status word and one
// argmax per target row) lives in a file-scope device array that every GPU loading the library
// holds until the process exits, so the call itself allocates nothing.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "spec_markov.h"

namespace spec {
namespace {

constexpr size_t kStatusBytes = 256;  // the status word, padded to keep the argmax aligned
constexpr size_t kScratchBytes = kStatusBytes + (size_t)SPEC_NOALLOC_MAX_ROWS * sizeof(int);

// Device scratch shared by every call on a device. In host code this name only stands in for
// the array; kernels receive the device address that cudaGetSymbolAddress returns.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPEC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();  // the failure is reported through the return code alone
      return SPEC_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SPEC_OK;
}

bool valid_sizes(int R, int gamma, int V) {
  if (R < 0 || gamma < 0 || V < 1) return false;
  if ((long long)R * (gamma + 1) * V > (1LL << 46)) return false;
  return true;
}

bool vec_loads(const void* target, int dtype, int V) {
  const size_t es = dtype == SPEC_BF16 ? 2 : 4;
  return (reinterpret_cast<uintptr_t>(target) & 15) == 0 && ((size_t)V * es) % 16 == 0;
}

}  // namespace
}  // namespace spec

using namespace spec;

extern "C" int spec_verify_greedy_noalloc(const void* target, int t_dtype,
                                          const int32_t* draft_tokens, const int32_t* lengths,
                                          int R, int gamma, int V, int32_t* accept_len,
                                          int32_t* out_tokens, int32_t* next_anchor,
                                          uint32_t* device_status, void* stream) {
  if (!valid_sizes(R, gamma, V)) return SPEC_ERR_INVALID_ARG;
  if (t_dtype != SPEC_F32 && t_dtype != SPEC_BF16) return SPEC_ERR_UNSUPPORTED_DTYPE;
  if ((long long)R * (gamma + 1) > SPEC_NOALLOC_MAX_ROWS) return SPEC_ERR_TOO_LARGE;
  if (R == 0) return SPEC_OK;
  if (!target || !accept_len || (gamma > 0 && !draft_tokens)) return SPEC_ERR_INVALID_ARG;
  void* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc != SPEC_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* status = static_cast<uint32_t*>(scratch);
  int* amax = reinterpret_cast<int*>(static_cast<unsigned char*>(scratch) + kStatusBytes);
  // the status word keeps the previous call's bits: start this call from zero
  if (cudaMemsetAsync(status, 0, sizeof(uint32_t), s) != cudaSuccess) return SPEC_ERR_CUDA;
  RowJob j;
  memset(&j, 0, sizeof j);
  j.rows = R * (gamma + 1);
  j.map = MAP_TARGET;
  j.mode = MODE_STATS;
  j.R = R;
  j.gamma = gamma;
  j.V = V;
  j.scale = 1.0f;
  j.T = target;
  j.lengths = lengths;
  j.status = status;
  launch_row_stats(j, t_dtype, vec_loads(target, t_dtype, V), nullptr, amax, s);
  launch_greedy_scan(R, gamma, amax, draft_tokens, lengths, nullptr, accept_len, out_tokens,
                     next_anchor, status, s);
  if (device_status &&
      cudaMemcpyAsync(device_status, status, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s) !=
          cudaSuccess)
    return SPEC_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
