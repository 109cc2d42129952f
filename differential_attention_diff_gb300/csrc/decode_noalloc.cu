// decode_noalloc.cu — diffattn_v2_decode_noalloc: the V2 decode for callers
// that cannot allocate device memory.
//
// Some callers of a decode step have no way to hand the library a workspace:
// an inference runtime whose device memory is carved up once at start-up and
// that forbids allocations on the token loop, a host program that drives the
// GPU through someone else's context and has no allocator of its own, or a
// plugin whose host framework exposes inputs and outputs but no scratch
// buffers.  For them this entry point runs the same split-KV decode as
// diffattn_v2_decode, with the split partials (and the gate, when it is
// computed from X) placed in a fixed array that lives in this file:
//
//   static __device__ __align__(256) uint8_t g_decode_scratch[16 MiB]
//
// Every GPU that loads the library reserves those 16 MiB until the process
// exits.  The first call on a device looks up the array's device address
// (cudaGetSymbolAddress, with that device current) and caches it; later calls
// reuse it.  The cached address belongs to the device's primary context as it
// was at that first call: after a cudaDeviceReset the array lives at a new
// address in a new context, so the library (this entry point, and the device
// status word every entry point uses, which is cached the same way) must not
// be used again in a process that has reset the device.  All calls share the
// one array: calls that overlap on the GPU (different streams, or several
// host threads) race on it and must be serialised by the caller.  Nothing in
// the array needs to start at zero: every call overwrites every partial it
// later reads.
#include <cuda_runtime.h>

#include <mutex>

#include "diffattn.h"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = DIFFATTN_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device (looked up once
// per device).
da_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
      return DA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return DA_OK;
}

}  // namespace

extern "C" da_status diffattn_v2_decode_noalloc(const da_v2_decode_params* p, void* stream) {
  // the shape checks of diffattn_v2_decode first, so that a malformed problem
  // is reported as such and not as one that does not fit the scratch
  const da_status chk = da::check_v2_decode_args(p);
  if (chk != DA_OK) return chk;
  const int gate_given = p->gate != nullptr;
  auto need = [&](int splits) {
    return diffattn_v2_decode_workspace_size(p->B, p->h, p->h_kv, p->d, p->L_max, splits,
                                             gate_given);
  };
  int splits = p->num_splits;
  if (splits > 0) {
    if (need(splits) > kScratchBytes) return DA_ERR_WORKSPACE;
  } else {
    // the library's usual split count, lowered until the partials fit
    splits = diffattn_v2_decode_num_splits(p->B, p->h_kv, p->L_max);
    while (splits > 1 && need(splits) > kScratchBytes) --splits;
    if (need(splits) > kScratchBytes) return DA_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  const da_status st = scratch_address(&scratch);
  if (st != DA_OK) return st;
  da_v2_decode_params q = *p;
  q.num_splits = splits;
  q.workspace = scratch;
  q.workspace_bytes = kScratchBytes;
  return diffattn_v2_decode(&q, stream);
}
