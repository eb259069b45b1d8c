// attn_bwd_noalloc.cu -- the fixed device scratch behind attn_bwd_noalloc.
//
// attn_bwd needs a workspace (each row's Delta and lse * log2(e)) that its caller allocates.
// Some callers cannot allocate device memory at the point where they run the backward pass:
// an engine that hands nearly all of the GPU's memory to its own pool at start-up, or a host
// program that forbids allocation inside its per-step calls, has no way to obtain a fresh
// buffer there.  For them the library carries the workspace itself, as one statically sized
// device array per GPU: it is part of the library's device image, so every GPU that loads the
// library holds these bytes until the process exits, and no call allocates or frees memory.
//
// The array is shared by every call on a device and keeps the last call's contents.  Nothing
// in it has to start at zero: each backward pass first rewrites every entry it will read (the
// Delta kernel writes the whole [B*H][2][S rounded up to 128] region, padding included).
// Calls whose kernels overlap on the GPU (two streams, or two host threads, at once) race on
// the array and may produce wrong gradients; serialise them.
#include <cuda_runtime.h>

#include "internal.h"

namespace ea46 {

namespace {

// The scratch itself: NOALLOC_BWD_SCRATCH_BYTES (16 MiB) per GPU.
static __device__ __align__(256) float g_bwd_scratch[NOALLOC_BWD_SCRATCH_BYTES / sizeof(float)];

}  // namespace

// The device address of the current GPU's scratch.  In host code g_bwd_scratch names a host
// stand-in, not device memory, so the address comes from cudaGetSymbolAddress, with the
// caller's device current.  It is looked up on every call rather than kept: the lookup is a
// host-side query (no stream work), and an address kept from an earlier context -- before a
// device reset reloaded the module -- would point at memory that no longer exists.
cudaError_t noalloc_bwd_scratch(float** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_bwd_scratch);
  if (e != cudaSuccess) return e;
  *out = static_cast<float*>(p);
  return cudaSuccess;
}

}  // namespace ea46
