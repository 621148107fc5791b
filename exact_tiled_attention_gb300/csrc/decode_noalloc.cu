// decode_noalloc.cu -- split-KV decode for callers that cannot allocate
// device memory.
//
// attn_decode_splitkv needs a caller-provided scratch buffer for the
// per-chunk partial states.  Some callers have no way to provide one: code
// embedded in a host framework that owns every device allocation and forbids
// plugins from calling cudaMalloc, memory-capped or real-time services that
// must never enter the allocator (cudaMalloc may synchronise the device), and
// C callers that only receive pointers to their inputs and outputs.  For
// them, attn_decode_splitkv_noalloc runs the same two kernels with the
// scratch taken from a fixed array in the library's own device memory.
//
// The array is a file-scope static __device__ object: every GPU that loads
// the library holds kNoallocScratchBytes of it until the process exits.
// CUDA loads a library's device code lazily by default, so the array itself
// comes into being when the first call on a device looks up its address
// (cudaGetSymbolAddress, with that device current): that first call loads
// the module and may allocate and synchronise inside the runtime.  Callers
// that must never reach the allocator make one call at initialisation,
// outside any stream capture.  The address is cached per device together
// with the id of the CUDA context it belongs to, and looked up again when
// the context changes (after cudaDeviceReset the old address is dead).
// All calls share the one array and it keeps the previous call's contents;
// the partial kernel overwrites every partial state it later reads, so
// nothing needs clearing, but two calls whose kernels overlap on the GPU
// (different streams without ordering) race on the array and must be
// serialised by the caller.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/gbattn.h"
#include "gbattn_internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = 32u << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device and CUDA context), or nullptr if the runtime could not provide it.
void* scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  const unsigned long long ctx = gbattn::current_context_id();
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_ptr[dev] == nullptr || ctx != g_scratch_ctx[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_ptr[dev] = ptr;
    g_scratch_ctx[dev] = gbattn::current_context_id();  // the lookup made the primary context current
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" {

size_t attn_decode_noalloc_scratch_bytes(void) { return kNoallocScratchBytes; }

int attn_decode_splitkv_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                const int* seqlens, void* o, float* lse, int B, int Hq, int Hkv,
                                int Sk_max, int d, float scale, int n_split, int dtype,
                                void* stream) {
  // The same argument checks as attn_decode_splitkv (less the workspace
  // pair), before the capacity check, so that a bad argument reports its
  // own code and not GBATTN_EWORKSPACE.
  const int check = gbattn::check_decode_args(q, k_cache, v_cache, seqlens, o, lse, B, Hq, Hkv, Sk_max, d,
                                              n_split, dtype);
  if (check != GBATTN_OK) return check;
  const size_t need = attn_decode_workspace_bytes(B, Hq, n_split, d);
  if (need > kNoallocScratchBytes) return GBATTN_EWORKSPACE;  // problem too large for the array
  void* scratch = scratch_for_current_device();
  if (scratch == nullptr) return GBATTN_EUNSUPPORTED;
  return attn_decode_splitkv(q, k_cache, v_cache, seqlens, o, lse, B, Hq, Hkv, Sk_max, d, scale,
                             n_split, scratch, kNoallocScratchBytes, dtype, stream);
}

}  // extern "C"
