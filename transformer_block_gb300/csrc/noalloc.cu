// noalloc.cu — the stream-K GEMM for callers that cannot allocate device memory.
//
// pb_gemm_bf16 splits the last waves of tiles along K and needs a scratch buffer from
// its caller for the partial tiles. Some callers have no way to provide one: plugins
// inside an inference engine or framework whose device memory all belongs to the host
// program's own allocator (they are handed inputs and outputs, nothing else), and
// latency-bound paths where a cudaMalloc could synchronise the device or block on the
// driver. pb_gemm_bf16_static runs the same GEMM with its scratch in a fixed array that
// lives in this library's own device memory, so the caller passes only A, B and C.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/pb.h"
#include "kernels.h"

namespace {

// Partial tiles and flags for up to kSkMaxClusters CTA pairs (25,171,968 bytes). Every GPU
// on which this library's device code is loaded holds it until the process exits, and it
// keeps what the last call left. Only the flags must start at zero: the array is
// zero-initialised when the module loads, and the GEMM clears every flag it consumed before
// it ends (the partial tiles are always written before they are read).
static __device__ __align__(256) uint8_t g_sk_scratch[pb::kSkScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_setup_mutex;
// Device address of g_sk_scratch, per device ordinal, looked up once in the device's
// primary context (the context the runtime API uses); the entry point assumes that context
// stays alive for the rest of the process (no cudaDeviceReset in between).
void* g_scratch_ptr[kMaxDevices];

}  // namespace

namespace pb {
pb_status record_error(pb_status s, const char* message);
}

extern "C" pb_status pb_gemm_bf16_static(int32_t M, int32_t N, int32_t K, const void* A,
                                         const void* B, void* C, int* status, void* stream) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return pb::record_error(PB_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return pb::record_error(PB_ERR_UNSUPPORTED, "device ordinal beyond the static table");
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return pb::record_error(PB_ERR_CUDA, cudaGetErrorString(e));
  if (sms / 2 > pb::kSkMaxClusters) {
    char msg[160];
    snprintf(msg, sizeof msg,
             "the static stream-K array holds partial tiles for %d CTA pairs; this GPU has "
             "%d SMs (%d pairs)",
             pb::kSkMaxClusters, sms, sms / 2);
    return pb::record_error(PB_ERR_UNSUPPORTED, msg);
  }
  void* scratch = nullptr;
  {
    // Once per device, with that device current: the array's device address. (In host
    // code the name g_sk_scratch is only a host-side stand-in, not a device address.)
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_sk_scratch);
      if (e != cudaSuccess) return pb::record_error(PB_ERR_CUDA, cudaGetErrorString(e));
      g_scratch_ptr[dev] = p;
    }
    scratch = g_scratch_ptr[dev];
  }
  return pb_gemm_bf16(M, N, K, A, B, C, scratch, pb::kSkScratchBytes, status, stream);
}
