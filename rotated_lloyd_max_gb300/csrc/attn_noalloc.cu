// tq_decode_attn_noalloc: the decode attention with its split-K workspace in a
// fixed, library-owned device array instead of caller-provided memory.
//
// For callers that cannot allocate device memory when they run attention:
// code whose device memory is reserved up front by a host framework or a
// pooling allocator that does not expose raw allocation, plugins whose enqueue
// step is forbidden to allocate, and latency-critical loops that cannot afford
// cudaMalloc's implicit device synchronisation.  The array is
// TQ_NOALLOC_WORKSPACE_BYTES large and lives as long as the library is loaded,
// on every GPU that loads it.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/tq.h"

namespace {

static __device__ __align__(256) unsigned char g_attn_scratch[TQ_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the array on the current device; looked up once per
// device (with that device current) and cached for the life of the process
// (a cudaDeviceReset invalidates it; the header tells callers not to call
// again after one).  In host code the symbol itself is only a host-side
// stand-in and must never be passed to a kernel.
tq_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TQ_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) return TQ_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return TQ_OK;
}

}  // namespace

extern "C" tq_status tq_decode_attn_noalloc(const tq_attn_args* args, const tq_codec* k_codec,
                                            const tq_codec* v_codec, void* stream) {
  tq_attn_plan plan;  // the planner's own status: invalid vs unsupported arguments
  const tq_status ps = tq_decode_attn_plan(args, k_codec, v_codec, &plan);
  if (ps != TQ_OK) return ps;
  if (plan.workspace_bytes > (uint64_t)TQ_NOALLOC_WORKSPACE_BYTES) return TQ_ERR_WORKSPACE;
  void* ws = nullptr;
  const tq_status st = scratch_address(&ws);
  if (st != TQ_OK) return st;
  return tq_decode_attn(args, k_codec, v_codec, ws, (size_t)TQ_NOALLOC_WORKSPACE_BYTES, stream);
}
