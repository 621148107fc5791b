// gbattn_internal.h -- host-side declarations shared by the library's
// translation units (not part of the public C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

namespace gbattn {

// Arguments of one prefill launch (already validated by the C-ABI layer).
struct PrefillArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, H, Hkv, Sq, Sk, d;
  float scale;
  int causal;
  bool bf16;
  cudaStream_t stream;
  int* status;                     // device status word
  int num_sms;                     // SMs of the device (CTAs resident at once)
  unsigned long long* timeline;    // per-CTA records (gbattn_timeline_set), or null
  long long timeline_capacity;     // records the buffer holds
};

// Arguments of one split-KV decode (partial + merge) launch.
struct DecodeArgs {
  const void* q;
  const void* k;
  const void* v;
  const int* seqlens;
  void* o;
  float* lse;
  int B, Hq, Hkv, Sk_max, d;
  float scale;
  int n_split;
  float* workspace;
  bool bf16;
  cudaStream_t stream;
  int* status;
};

// Arguments of one backward (preprocess + main + dQ conversion).
struct BackwardArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const float* lse;
  const void* dout;
  void* dq;
  void* dk;
  void* dv;
  int B, H, Hkv, Sq, Sk, d;
  float scale;
  int causal;
  float* Dvec;    // workspace: [B*H*Sq] fp32 row scalars D
  float* dq_acc = nullptr;  // atomic variant: workspace [B*H*Sq*d] fp32 dQ accumulator
  bool bf16;
  cudaStream_t stream;
  int* status;
};

// Arguments of one FP8 (E4M3) forward launch.
struct PrefillFp8Args {
  const void* q;   // E4M3 [B,H,Sq,d]
  const void* k;   // E4M3 [B,Hkv,Sk,d]
  const void* v;   // E4M3 [B,Hkv,Sk,d]
  const float* q_descale;  // [B,Hkv] or nullptr (1.0)
  const float* k_descale;
  const float* v_descale;
  void* o;         // bf16 [B,H,Sq,d]
  float* lse;
  int B, H, Hkv, Sq, Sk, d;
  float scale;
  int causal;
  void* vt;        // workspace: E4M3 [B,Hkv,d,Sk_pad], Sk_pad = Sk rounded up to 128
  cudaStream_t stream;
  int* status;
  int num_sms;                     // SMs of the device (CTAs resident at once)
  unsigned long long* timeline;    // per-CTA records (gbattn_timeline_set), or null
  long long timeline_capacity;     // records the buffer holds
};

// Each returns a cudaError_t / CUresult folded into 0 (ok) or -1 (launch or
// tensor-map failure).
int launch_prefill(const PrefillArgs& a);
// Non-causal d = 128 forward on a tcgen05 CTA pair (prefill_pair.cu); -1 if
// the arguments are outside that case or a launch failed.
int launch_prefill_pair(const PrefillArgs& a);
int launch_decode(const DecodeArgs& a);
int launch_backward(const BackwardArgs& a);
// Column owner with fp32 atomic dQ (backward_atomic.cu); d = 128 and a.dq_acc
// set, else -1.
int launch_backward_atomic(const BackwardArgs& a);
int launch_prefill_fp8(const PrefillFp8Args& a);

// Checks the scalar and pointer arguments of a split-KV decode (everything
// attn_decode_splitkv checks except the workspace); GBATTN_OK or the error.
int check_decode_args(const void* q, const void* k_cache, const void* v_cache, const int* seqlens,
                      const void* o, const float* lse, int B, int Hq, int Hkv, int Sk_max, int d,
                      int n_split, int dtype);

// Unique id of the CUDA context current on the calling thread (cuCtxGetId,
// through the runtime's driver entry points), or 0 when no context is current
// or the driver does not provide the calls.  A cached device address (a
// __device__ symbol's) is valid only within the context it was looked up in:
// after cudaDeviceReset the device's next primary context has a new id.
unsigned long long current_context_id();

// cuTensorMapEncodeTiled fetched once through the runtime's driver entry
// point (no link-time dependency on libcuda).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

// Heads per L2 scheduling group.  The launchers order their CTAs in groups of
// heads whose K/V (or whatever per-head data the kernel re-reads) stay resident
// in L2 while the group runs: at most hg_max heads, a multiple of `step` (whole
// KV-head groups), and groups of equal size -- the largest such size, down to
// half of hg_max, that divides `heads`, else near-equal groups.  A short last
// group would start its heaviest (causal) units last and leave a tail: at 64
// heads of 4 MB, groups of 12 (five of 12, one of 4) measured 5 % slower on the
// causal 8192-token forward than groups of 8.
inline int balanced_head_group(long long hg_max, long long heads, long long step) {
  if (step < 1) step = 1;
  if (hg_max < step) hg_max = step;
  if (hg_max > heads) hg_max = heads;
  for (long long c = hg_max - hg_max % step; c >= step && 2 * c >= hg_max; c -= step)
    if (heads % c == 0) return static_cast<int>(c);
  const long long n_groups = (heads + hg_max - 1) / hg_max;
  long long hg = (heads + n_groups - 1) / n_groups;
  hg = (hg + step - 1) / step * step;
  return static_cast<int>(hg < heads ? hg : heads);
}

// Raises `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device, once per device for each call site (`done` holds one bit per device
// ordinal; devices past 63 set it on every call).  The attribute belongs to
// the device's context, so a process that launches on several GPUs needs it
// on each; concurrent host threads may both set it, which is harmless.
template <typename Kernel>
inline bool set_smem_limit_once(Kernel kernel, int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
  done.fetch_or(bit, std::memory_order_release);
  return true;
}

// 3-D tensor map over a contiguous [outer, rows, d] 16-bit tensor with a
// (64 x box_rows x 1) box and 128-byte swizzle; rows past `rows` read as 0.
bool make_tmap_3d(CUtensorMap* map, const void* base, bool bf16, int d, int rows, long long outer,
                  int box_rows);

// 3-D tensor map over a contiguous [outer, rows, inner] fp32 tensor with a
// (box_inner x box_rows x 1) box, box_inner * 4 <= 128 bytes, and 128-byte
// swizzle; rows past `rows` are not read or written.
bool make_tmap_3d_f32(CUtensorMap* map, void* base, int inner, int rows, long long outer, int box_inner,
                      int box_rows);

// 3-D tensor map over a contiguous [outer, rows, inner] byte tensor with a
// (128 x box_rows x 1) box and 128-byte swizzle; rows past `rows` and bytes
// past `inner` read as 0.  inner must be a multiple of 16.
bool make_tmap_3d_u8(CUtensorMap* map, const void* base, long long inner, int rows, long long outer,
                     int box_rows);

}  // namespace gbattn
