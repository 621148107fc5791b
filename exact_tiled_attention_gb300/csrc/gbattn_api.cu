// gbattn_api.cu -- the C ABI (include/gbattn.h): argument validation, host
// planning helpers, tensor-map encoding and dispatch to the kernels.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include <mutex>

#include "../../include/gbattn.h"
#include "gbattn_internal.h"
#include "gbattn_ptx.cuh"

namespace gbattn {

// Device status word written by the kernels' bounded waits (0 = ok).
__device__ int g_device_status;

namespace {

std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

// Device status pointer per device (looked up once per context, then cached).
constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices] = {};
unsigned long long g_status_ctx[kMaxDevices] = {};
int g_sm_major[kMaxDevices] = {};
int g_sm_minor[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};
std::mutex g_dev_mutex;

// Per-CTA timeline of attn_fwd launches (gbattn_timeline_set).
std::mutex g_timeline_mutex;
unsigned long long* g_timeline = nullptr;
long long g_timeline_capacity = 0;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Returns GBATTN_OK and the status pointer (and, if asked, the SM count) of
// the current device, or an error.
int current_device(int** status, int* sm_count = nullptr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return GBATTN_EUNSUPPORTED;
  }
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (g_status_ptr[dev] == nullptr || ctx != g_status_ctx[dev]) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return GBATTN_EUNSUPPORTED;
    }
    g_sm_major[dev] = major;
    g_sm_minor[dev] = minor;
    g_sm_count[dev] = sms;
    if (major != 10 || minor != 3) return GBATTN_EUNSUPPORTED;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_device_status) != cudaSuccess) {
      cudaGetLastError();
      return GBATTN_ELAUNCH;
    }
    g_status_ptr[dev] = static_cast<int*>(ptr);
    g_status_ctx[dev] = current_context_id();  // the lookup made the primary context current
  }
  if (g_sm_major[dev] != 10 || g_sm_minor[dev] != 3) return GBATTN_EUNSUPPORTED;
  *status = g_status_ptr[dev];
  if (sm_count != nullptr) *sm_count = g_sm_count[dev];
  return GBATTN_OK;
}

}  // namespace

unsigned long long current_context_id() {
  using GetCurrentFn = CUresult (*)(CUcontext*);
  using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(fn);
    cudaGetLastError();
  });
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

int check_decode_args(const void* q, const void* k_cache, const void* v_cache, const int* seqlens,
                      const void* o, const float* lse, int B, int Hq, int Hkv, int Sk_max, int d,
                      int n_split, int dtype) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Sk_max < 1) return GBATTN_EBADSHAPE;
  if (B > 65535) return GBATTN_EBADSHAPE;
  if (Hq % Hkv != 0) return GBATTN_EHEADS;
  if (d != 64 && d != 128) return GBATTN_EHEADDIM;
  if (dtype != GBATTN_F16 && dtype != GBATTN_BF16) return GBATTN_EDTYPE;
  if (n_split < 1 || n_split > 256) return GBATTN_ESPLIT;
  if (!q || !k_cache || !v_cache || !seqlens || !o || !aligned16(q) || !aligned16(k_cache) ||
      !aligned16(v_cache) || !aligned16(o) || (reinterpret_cast<uintptr_t>(seqlens) & 3u) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return GBATTN_EPOINTER;
  return GBATTN_OK;
}

EncodeTiledFn encode_tiled_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    else
      cudaGetLastError();
  });
  return g_encode;
}

bool make_tmap_3d(CUtensorMap* map, const void* base, bool bf16, int d, int rows, long long outer,
                  int box_rows) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(outer)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(rows) * static_cast<cuuint64_t>(d) * 2};
  const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_rows), 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r =
      enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
          const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_3d_f32(CUtensorMap* map, void* base, int inner, int rows, long long outer, int box_inner,
                      int box_rows) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr || box_inner * 4 > 128) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(outer)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner) * 4,
                                 static_cast<cuuint64_t>(rows) * static_cast<cuuint64_t>(inner) * 4};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_rows), 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Both exp2 paths of the kernels on n values: y_poly = ex2_poly3_x2 (FMA
// pipe), y_hw = ex2.approx (MUFU).  n is even.
__global__ void ex2_paths_kernel(const float* __restrict__ x, float* __restrict__ y_poly,
                                 float* __restrict__ y_hw, long long n2) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n2) return;
  const float2 v = reinterpret_cast<const float2*>(x)[i];
  reinterpret_cast<float2*>(y_poly)[i] = ex2_poly3_x2(v);
  reinterpret_cast<float2*>(y_hw)[i] = make_float2(ex2_approx(v.x), ex2_approx(v.y));
}

bool make_tmap_3d_u8(CUtensorMap* map, const void* base, long long inner, int rows, long long outer,
                     int box_rows) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr || (inner % 16) != 0) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(outer)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner),
                                 static_cast<cuuint64_t>(rows) * static_cast<cuuint64_t>(inner)};
  const cuuint32_t box[3] = {128u, static_cast<cuuint32_t>(box_rows), 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace gbattn

using namespace gbattn;

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
             int Hkv, int Sq, int Sk, int d, float scale, int causal, int dtype, void* stream) {
  if (B < 1 || H < 1 || Hkv < 1 || Sq < 1 || Sk < 1) return GBATTN_EBADSHAPE;
  if (H % Hkv != 0) return GBATTN_EHEADS;
  if (d != 64 && d != 128) return GBATTN_EHEADDIM;
  if (dtype != GBATTN_F16 && dtype != GBATTN_BF16) return GBATTN_EDTYPE;
  if (!q || !k || !v || !o || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return GBATTN_EPOINTER;
  // Tensor-map extents are 32-bit per dimension except the outermost.
  if (static_cast<long long>(B) * H > 0x7FFFFFFFLL || static_cast<long long>(B) * Hkv > 0x7FFFFFFFLL)
    return GBATTN_EBADSHAPE;
  int* status = nullptr;
  int sms = 0;
  int rc = current_device(&status, &sms);
  if (rc != GBATTN_OK) return rc;
  PrefillArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.H = H;
  a.Hkv = Hkv;
  a.Sq = Sq;
  a.Sk = Sk;
  a.d = d;
  a.scale = scale;
  a.causal = causal ? 1 : 0;
  a.bf16 = dtype == GBATTN_BF16;
  a.stream = static_cast<cudaStream_t>(stream);
  a.status = status;
  a.num_sms = sms;
  {
    std::lock_guard<std::mutex> lock(g_timeline_mutex);
    a.timeline = g_timeline;
    a.timeline_capacity = g_timeline_capacity;
  }
  return launch_prefill(a) == 0 ? GBATTN_OK : GBATTN_ELAUNCH;
}

int attn_fwd_pair(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv, int Sq,
                  int Sk, int d, float scale, int dtype, void* stream) {
  if (B < 1 || H < 1 || Hkv < 1 || Sq < 1 || Sk < 1) return GBATTN_EBADSHAPE;
  if (H % Hkv != 0) return GBATTN_EHEADS;
  if (d != 128) return GBATTN_EHEADDIM;
  if (dtype != GBATTN_F16 && dtype != GBATTN_BF16) return GBATTN_EDTYPE;
  if (!q || !k || !v || !o || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return GBATTN_EPOINTER;
  if (static_cast<long long>(B) * H > 0x7FFFFFFFLL || static_cast<long long>(B) * Hkv > 0x7FFFFFFFLL)
    return GBATTN_EBADSHAPE;
  int* status = nullptr;
  int sms = 0;
  int rc = current_device(&status, &sms);
  if (rc != GBATTN_OK) return rc;
  PrefillArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.H = H;
  a.Hkv = Hkv;
  a.Sq = Sq;
  a.Sk = Sk;
  a.d = d;
  a.scale = scale;
  a.causal = 0;
  a.bf16 = dtype == GBATTN_BF16;
  a.stream = static_cast<cudaStream_t>(stream);
  a.status = status;
  a.num_sms = sms;
  {
    std::lock_guard<std::mutex> lock(g_timeline_mutex);
    a.timeline = g_timeline;
    a.timeline_capacity = g_timeline_capacity;
  }
  return launch_prefill_pair(a) == 0 ? GBATTN_OK : GBATTN_ELAUNCH;
}

size_t attn_decode_workspace_bytes(int B, int Hq, int n_split, int d) {
  if (B < 1 || Hq < 1 || n_split < 1 || d < 1) return 0;
  return static_cast<size_t>(B) * Hq * n_split * (static_cast<size_t>(d) + 2) * sizeof(float);
}

int attn_decode_splitkv(const void* q, const void* k_cache, const void* v_cache, const int* seqlens,
                        void* o, float* lse, int B, int Hq, int Hkv, int Sk_max, int d, float scale,
                        int n_split, void* workspace, size_t workspace_bytes, int dtype,
                        void* stream) {
  const int check = check_decode_args(q, k_cache, v_cache, seqlens, o, lse, B, Hq, Hkv, Sk_max, d,
                                      n_split, dtype);
  if (check != GBATTN_OK) return check;
  if (!workspace || !aligned16(workspace)) return GBATTN_EPOINTER;
  if (workspace_bytes < attn_decode_workspace_bytes(B, Hq, n_split, d)) return GBATTN_EWORKSPACE;
  int* status = nullptr;
  int rc = current_device(&status);
  if (rc != GBATTN_OK) return rc;
  DecodeArgs a;
  a.q = q;
  a.k = k_cache;
  a.v = v_cache;
  a.seqlens = seqlens;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Sk_max = Sk_max;
  a.d = d;
  a.scale = scale;
  a.n_split = n_split;
  a.workspace = static_cast<float*>(workspace);
  a.bf16 = dtype == GBATTN_BF16;
  a.stream = static_cast<cudaStream_t>(stream);
  a.status = status;
  return launch_decode(a) == 0 ? GBATTN_OK : GBATTN_ELAUNCH;
}

size_t attn_bwd_workspace_bytes(int B, int H, int Sq, int d) {
  if (B < 1 || H < 1 || Sq < 1 || d < 1) return 0;
  // the fp32 row scalars D, rounded up to 256 bytes
  return ((static_cast<size_t>(B) * H * Sq * sizeof(float)) + 255) & ~static_cast<size_t>(255);
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dout, void* dq, void* dk, void* dv, int B, int H, int Hkv, int Sq, int Sk,
             int d, float scale, int causal, void* workspace, size_t workspace_bytes, int dtype,
             void* stream) {
  if (B < 1 || H < 1 || Hkv < 1 || Sq < 1 || Sk < 1) return GBATTN_EBADSHAPE;
  if (H % Hkv != 0) return GBATTN_EHEADS;
  if (d != 64 && d != 128) return GBATTN_EHEADDIM;
  if (dtype != GBATTN_F16 && dtype != GBATTN_BF16) return GBATTN_EDTYPE;
  const void* ptrs[] = {q, k, v, o, dout, dq, dk, dv, workspace};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return GBATTN_EPOINTER;
  if (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u)) return GBATTN_EPOINTER;
  if (static_cast<long long>(B) * H > 0x7FFFFFFFLL || static_cast<long long>(B) * Hkv > 0x7FFFFFFFLL)
    return GBATTN_EBADSHAPE;
  if (workspace_bytes < attn_bwd_workspace_bytes(B, H, Sq, d)) return GBATTN_EWORKSPACE;
  int* status = nullptr;
  int rc = current_device(&status);
  if (rc != GBATTN_OK) return rc;
  BackwardArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.dout = dout;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.B = B;
  a.H = H;
  a.Hkv = Hkv;
  a.Sq = Sq;
  a.Sk = Sk;
  a.d = d;
  a.scale = scale;
  a.causal = causal ? 1 : 0;
  a.Dvec = static_cast<float*>(workspace);
  a.bf16 = dtype == GBATTN_BF16;
  a.stream = static_cast<cudaStream_t>(stream);
  a.status = status;
  return launch_backward(a) == 0 ? GBATTN_OK : GBATTN_ELAUNCH;
}

size_t attn_bwd_atomic_workspace_bytes(int B, int H, int Sq, int d) {
  const size_t dbytes = attn_bwd_workspace_bytes(B, H, Sq, d);
  if (dbytes == 0) return 0;
  // the row scalars D, then the fp32 dQ accumulator [B, H, Sq, d]
  return dbytes + static_cast<size_t>(B) * H * Sq * d * sizeof(float);
}

int attn_bwd_atomic(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dout, void* dq, void* dk, void* dv, int B, int H, int Hkv, int Sq, int Sk,
                    int d, float scale, int causal, void* workspace, size_t workspace_bytes, int dtype,
                    void* stream) {
  if (B < 1 || H < 1 || Hkv < 1 || Sq < 1 || Sk < 1) return GBATTN_EBADSHAPE;
  if (H % Hkv != 0) return GBATTN_EHEADS;
  if (d != 64 && d != 128) return GBATTN_EHEADDIM;
  if (dtype != GBATTN_F16 && dtype != GBATTN_BF16) return GBATTN_EDTYPE;
  const void* ptrs[] = {q, k, v, o, dout, dq, dk, dv, workspace};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return GBATTN_EPOINTER;
  if (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u)) return GBATTN_EPOINTER;
  if (static_cast<long long>(B) * H > 0x7FFFFFFFLL || static_cast<long long>(B) * Hkv > 0x7FFFFFFFLL)
    return GBATTN_EBADSHAPE;
  if (workspace_bytes < attn_bwd_atomic_workspace_bytes(B, H, Sq, d)) return GBATTN_EWORKSPACE;
  int* status = nullptr;
  int rc = current_device(&status);
  if (rc != GBATTN_OK) return rc;
  BackwardArgs a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.dout = dout;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.B = B;
  a.H = H;
  a.Hkv = Hkv;
  a.Sq = Sq;
  a.Sk = Sk;
  a.d = d;
  a.scale = scale;
  a.causal = causal ? 1 : 0;
  a.Dvec = static_cast<float*>(workspace);
  a.dq_acc = reinterpret_cast<float*>(static_cast<char*>(workspace) + attn_bwd_workspace_bytes(B, H, Sq, d));
  a.bf16 = dtype == GBATTN_BF16;
  a.stream = static_cast<cudaStream_t>(stream);
  a.status = status;
  return launch_backward_atomic(a) == 0 ? GBATTN_OK : GBATTN_ELAUNCH;
}

size_t attn_fwd_fp8_workspace_bytes(int B, int Hkv, int Sk, int d) {
  if (B < 1 || Hkv < 1 || Sk < 1 || d < 1) return 0;
  const size_t sk_pad = (static_cast<size_t>(Sk) + 127) / 128 * 128;
  return static_cast<size_t>(B) * Hkv * d * sk_pad;
}

int attn_fwd_fp8(const void* q, const void* k, const void* v, const float* q_descale, const float* k_descale,
                 const float* v_descale, void* o, float* lse, int B, int H, int Hkv, int Sq, int Sk, int d,
                 float scale, int causal, void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 1 || H < 1 || Hkv < 1 || Sq < 1 || Sk < 1) return GBATTN_EBADSHAPE;
  if (H % Hkv != 0) return GBATTN_EHEADS;
  if (d != 128) return GBATTN_EHEADDIM;
  const void* ptrs[] = {q, k, v, o, workspace};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return GBATTN_EPOINTER;
  const void* opt[] = {q_descale, k_descale, v_descale, lse};
  for (const void* ptr : opt)
    if (ptr && (reinterpret_cast<uintptr_t>(ptr) & 3u)) return GBATTN_EPOINTER;
  if (static_cast<long long>(B) * H > 0x7FFFFFFFLL || static_cast<long long>(B) * Hkv > 65535)
    return GBATTN_EBADSHAPE;
  if (workspace_bytes < attn_fwd_fp8_workspace_bytes(B, Hkv, Sk, d)) return GBATTN_EWORKSPACE;
  int* status = nullptr;
  int sms = 0;
  int rc = current_device(&status, &sms);
  if (rc != GBATTN_OK) return rc;
  PrefillFp8Args a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.q_descale = q_descale;
  a.k_descale = k_descale;
  a.v_descale = v_descale;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.H = H;
  a.Hkv = Hkv;
  a.Sq = Sq;
  a.Sk = Sk;
  a.d = d;
  a.scale = scale;
  a.causal = causal ? 1 : 0;
  a.vt = workspace;
  a.stream = static_cast<cudaStream_t>(stream);
  a.status = status;
  a.num_sms = sms;
  {
    std::lock_guard<std::mutex> lock(g_timeline_mutex);
    a.timeline = g_timeline;
    a.timeline_capacity = g_timeline_capacity;
  }
  return launch_prefill_fp8(a) == 0 ? GBATTN_OK : GBATTN_ELAUNCH;
}

int gbattn_causal_tile_counts(int Sq, int Sk, int Br, int Bc, long long* full, long long* partial,
                              long long* skipped, long long* allowed_cells,
                              long long* visited_cells) {
  if (Sq < 1 || Sk < 1 || Br < 1 || Bc < 1) return GBATTN_EBADSHAPE;
  const long long delta = static_cast<long long>(Sk) - Sq;
  long long nf = 0, np = 0, ns = 0, allowed = 0, visited = 0;
  const int tq = (Sq + Br - 1) / Br, tk = (Sk + Bc - 1) / Bc;
  for (int i = 0; i < tq; ++i) {
    const long long q0 = static_cast<long long>(i) * Br;
    const long long q1 = q0 + Br < Sq ? q0 + Br : Sq;
    for (int j = 0; j < tk; ++j) {
      const long long k0 = static_cast<long long>(j) * Bc;
      const long long k1 = k0 + Bc < Sk ? k0 + Bc : Sk;
      if (k0 > (q1 - 1) + delta) {
        ++ns;
        continue;
      }
      if (k1 - 1 <= q0 + delta)
        ++nf;
      else
        ++np;
      visited += (q1 - q0) * (k1 - k0);
    }
  }
  for (long long i = 0; i < Sq; ++i) {
    long long last = i + delta;  // largest visible key of row i
    if (last >= Sk) last = Sk - 1;
    if (last >= 0) allowed += last + 1;
  }
  if (full) *full = nf;
  if (partial) *partial = np;
  if (skipped) *skipped = ns;
  if (allowed_cells) *allowed_cells = allowed;
  if (visited_cells) *visited_cells = visited;
  return GBATTN_OK;
}

int gbattn_exp2_paths(const float* x, float* y_poly, float* y_hw, long long n, void* stream) {
  if (n < 0 || (n & 1)) return GBATTN_EBADSHAPE;
  if (n == 0) return GBATTN_OK;
  if (!x || !y_poly || !y_hw || (reinterpret_cast<uintptr_t>(x) & 7u) ||
      (reinterpret_cast<uintptr_t>(y_poly) & 7u) || (reinterpret_cast<uintptr_t>(y_hw) & 7u))
    return GBATTN_EPOINTER;
  int* status = nullptr;
  int rc = current_device(&status);
  if (rc != GBATTN_OK) return rc;
  const long long n2 = n / 2, blocks = (n2 + 255) / 256;
  if (blocks > 0x7FFFFFFFLL) return GBATTN_EBADSHAPE;
  ex2_paths_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(x, y_poly, y_hw,
                                                                                                 n2);
  return cudaGetLastError() == cudaSuccess ? GBATTN_OK : GBATTN_ELAUNCH;
}

// One warp: thread 0 waits (bounded) on an mbarrier that completes only if
// `arrive` is set -- the wait every kernel role performs on its producer.
__global__ void selftest_wait_kernel(int arrive, int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (arrive) mbar_arrive(&bar);
    bounded_wait(&bar, 0, &abort_flag, status, kStatusSelftest);
  }
}

int gbattn_selftest_bounded_wait(int arrive, void* stream) {
  int* status = nullptr;
  int rc = current_device(&status);
  if (rc != GBATTN_OK) return rc;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(arrive ? 1 : 0, status);
  return cudaGetLastError() == cudaSuccess ? GBATTN_OK : GBATTN_ELAUNCH;
}

int gbattn_timeline_set(unsigned long long* records, long long capacity) {
  if (records != nullptr) {
    if ((reinterpret_cast<uintptr_t>(records) & 7u) != 0) return GBATTN_EPOINTER;
    if (capacity < 1) return GBATTN_EBADSHAPE;
  }
  std::lock_guard<std::mutex> lock(g_timeline_mutex);
  g_timeline = records;
  g_timeline_capacity = records != nullptr ? capacity : 0;
  return GBATTN_OK;
}

int gbattn_device_status(void) {
  int* status = nullptr;
  int rc = current_device(&status);
  if (rc != GBATTN_OK) return rc;
  if (cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    return GBATTN_ELAUNCH;
  }
  int value = 0;
  if (cudaMemcpyFromSymbol(&value, g_device_status, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return GBATTN_ELAUNCH;
  }
  if (value != 0) {
    const int zero = 0;
    cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int));
    return GBATTN_EDEVICE_TIMEOUT;
  }
  return GBATTN_OK;
}

const char* gbattn_error_string(int code) {
  switch (code) {
    case GBATTN_OK: return "ok";
    case GBATTN_EBADSHAPE: return "bad shape (a size is < 1 or too large)";
    case GBATTN_EHEADS: return "query heads are not a multiple of KV heads";
    case GBATTN_EHEADDIM: return "unsupported head dimension (only 64 and 128)";
    case GBATTN_EDTYPE: return "unsupported dtype (only fp16 and bf16)";
    case GBATTN_EPOINTER: return "null or misaligned pointer";
    case GBATTN_EWORKSPACE: return "workspace too small (or problem beyond a fixed scratch size)";
    case GBATTN_ELAUNCH: return "CUDA launch or tensor-map encoding failed";
    case GBATTN_EDEVICE_TIMEOUT: return "a kernel gave up on the device (bounded wait timed out or shared memory misaligned)";
    case GBATTN_ESPLIT: return "n_split out of range (1..256)";
    case GBATTN_EUNSUPPORTED: return "no sm_103 device is current";
    default: return "unknown status code";
  }
}

const char* gbattn_version(void) { return "gbattn 0.1.0 sm_103a"; }

}  // extern "C"
