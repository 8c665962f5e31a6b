// ttt_mlp_fwd_noalloc: TTT-MLP forward for callers that cannot allocate
// device memory.
//
// ttt_mlp_fwd needs a caller-provided workspace: a status word plus, when the
// fp32 SIMT kernel serves the call, a copy of the chunk-start weights W1, W2
// per (batch row, head) that the kernel keeps while it walks a chunk. Some
// callers have no way to get that memory: code that runs where cudaMalloc is
// not allowed or not wise (inside a region that must not synchronise the
// device, under a memory pool that hands out only the tensors it manages, or
// from a plain C host that owns just its input and output buffers). This entry
// point takes the workspace from a fixed array in this file instead, so the
// caller passes only inputs and outputs and nothing is allocated.
//
// Limits and sharing:
//  - The array holds kNoAllocScratchBytes (8 MiB) of snapshot space after a
//    256-byte status block. The tensor-core kernel (bf16, d = 64, b % 16 == 0)
//    keeps its chunk-start copies on chip and uses the status block alone, so
//    it takes any number of units. The fp32 SIMT kernel needs 2 * d * 4d
//    floats per unit: at d = 64 up to 64 (batch row, head) units. Larger
//    requests return TTT_ERR_UNSUPPORTED before anything is enqueued.
//  - Every GPU that loads this library holds the array until the process exits.
//  - All calls on a device share the one array and it keeps what the last call
//    left there. The status word is cleared at the start of every call; the
//    snapshot needs no clearing, the kernel writes it before reading it. Calls
//    whose kernels overlap on the GPU (different streams, no ordering between
//    them) race on the array and give wrong results; order them on one stream
//    or make them wait for each other.
//  - A kernel that gives up a bounded wait records TTT_ERR_TIMEOUT in the
//    array's status block; ttt_mlp_noalloc_last_device_status reads it.
//  - The first call on a device looks up the array's device address
//    (cudaGetSymbolAddress, with that device current) and caches it; make that
//    first call before any stream capture begins.
#include <cuda_runtime.h>

#include <mutex>

#include "ttt.h"
#include "kernels.h"

namespace {

constexpr size_t kNoAllocStatusBytes = 256;
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
constexpr int kMaxDevices = 64;

}  // namespace

// The scratch array. Host code must not use this name as a device address:
// on the host it names a stand-in object; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_ttt_mlp_noalloc_scratch[kNoAllocStatusBytes + kNoAllocScratchBytes];

namespace {

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
ttt_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return TTT_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return TTT_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_ttt_mlp_noalloc_scratch) != cudaSuccess || p == nullptr) return TTT_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return TTT_OK;
}

}  // namespace

extern "C" ttt_status ttt_mlp_fwd_noalloc(const void* Q, const void* K, const void* V, ttt_dtype dt,
                                          const float* eta, const float* W1_0, const float* W2_0, int B, int H,
                                          int T, int d, int b, void* Z, float* W1_out, float* W2_out,
                                          void* stream) {
  if (dt != TTT_F32 && dt != TTT_BF16) return TTT_ERR_ARG;
  // Size by the kernel that will serve the call: the status block alone for the
  // tensor-core kernel, plus the per-unit snapshot for the SIMT kernel.
  const size_t need = ttt::mlp_workspace_bytes_for_path(B, H, T, d, b, dt, nullptr);
  if (need == 0) return TTT_ERR_ARG;
  if (need > sizeof(g_ttt_mlp_noalloc_scratch)) return TTT_ERR_UNSUPPORTED;
  void* ws = nullptr;
  const ttt_status st = scratch_address(&ws);
  if (st != TTT_OK) return st;
  return ttt::mlp_forward(Q, K, V, dt, eta, W1_0, W2_0, B, H, T, d, b, Z, W1_out, W2_out, ws,
                          sizeof(g_ttt_mlp_noalloc_scratch), stream, nullptr, true);
}

extern "C" ttt_status ttt_mlp_noalloc_last_device_status(void* stream) {
  void* ws = nullptr;
  const ttt_status st = scratch_address(&ws);
  if (st != TTT_OK) return st;
  return ttt_last_device_status(ws, stream);
}
