// Backward pass for callers that cannot allocate device memory.
//
// attn_bwd needs scratch memory (the fp32 dQ accumulator, D = rowsum(dO o O)
// and, in deterministic mode, the ordering semaphores) and expects the caller to
// pass it in. Some callers have no way to get that memory at the point where they
// run the backward pass: a plugin inside a host program that owns every byte of
// device memory through its own pool and hands out no allocator, or a
// latency-critical loop in which cudaMalloc / cudaFree would stall on an implicit
// device synchronisation. attn_bwd_noalloc serves them from a buffer that is part
// of the library itself: a file-scope __device__ array of fixed size, created
// when the library's device code is loaded on a GPU and held until the process
// exits. The entry point allocates nothing, neither directly nor through a
// library routine.
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/attn.h"

namespace {

// Every GPU that loads this library holds this buffer until process exit.
static __device__ __align__(256) uint8_t g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

// Device address of the buffer on the current device. In host code the array's
// name only stands in for the symbol; the real address comes from the runtime,
// with the device current. It is looked up on every call rather than cached:
// the lookup allocates nothing and is cheap, and a cached address would go stale
// if the device's context were torn down and created again (cudaDeviceReset),
// which reloads the library's device code and may move the buffer. The first
// lookup on a device loads the library's device code there (this is where the
// buffer comes into existence), so make the first call on a device before any
// stream capture.
int noalloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return ATTN_ERR_NO_DEVICE;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
    return ATTN_ERR_CUDA;
  *out = p;
  return ATTN_OK;
}

}  // namespace

extern "C" int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                int B, int H_q, int H_kv, int N_q, int N_k, int d, int causal,
                                const int* seqlens, float scale, int deterministic,
                                attn_stream_t stream) {
  // Reject oversize problems before touching the device.
  const size_t need = attn_bwd_workspace_bytes(B, H_q, H_kv, N_q, N_k, d, seqlens != nullptr,
                                               deterministic);
  if (need > ATTN_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_WORKSPACE;
  if (B == 0 || N_q == 0 || N_k == 0 || need == 0) {
    // nothing needs scratch (empty problem) or the arguments are invalid:
    // attn_bwd reports either case without using the workspace
    return attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H_q, H_kv, N_q, N_k, d, causal, seqlens,
                    scale, deterministic, nullptr, 0, stream);
  }
  void* scratch = nullptr;
  const int st = noalloc_scratch(&scratch);
  if (st != ATTN_OK) return st;
  // attn_bwd clears everything in the scratch that has to start at zero, so the
  // contents left by an earlier call do not matter.
  return attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H_q, H_kv, N_q, N_k, d, causal, seqlens,
                  scale, deterministic, scratch, ATTN_NOALLOC_SCRATCH_BYTES, stream);
}
