// decode_splitkv.cu -- one-query decode over a padded KV cache, split-KV.
//
// Partial kernel: one CTA per (chunk c, KV head, group of <= 16 query heads,
// batch b).  The chunk [floor(c*L_b/n), floor((c+1)*L_b/n)) of the KV head is
// streamed through a shared-memory ring by TMA (64 keys of K and V per slot,
// 128-byte swizzle) and every K/V row is read once for all the query heads
// that share it (M4.4 0x06A head map; 0x06D grouped reuse).  Four consumer
// warps each take 16 keys of a slot; scores and P.V use warp-level
// m16n8k16 tensor-core MMAs with fp32 accumulation (the query heads fill the
// 16-row A operand).  Each warp keeps an online (m, l, o) state per query
// head with the same conditional rescaling as the prefill kernel; the four
// warp states are merged in shared memory with the common-maximum merge of
// M4.3 0x08B and written to the workspace in natural-log units:
//     ws_o [B, Hq, n, d]  unnormalised o  (o / l = the chunk's output)
//     ws_ml[B, Hq, n, 2]  (m, l); an empty chunk is (-inf, 0) with o = 0.
//
// Merge kernel: one warp per (b, query head) folds the n partial states
// (M4.3 0x08B with the 0x08C validity branch): M = max m_c,
// l = sum e^(m_c - M) l_c, o = sum e^(m_c - M) o_c; O = o / l,
// LSE = M + log l.  This is the split-KV tower's outer bracket ("Learning
// FlashAttention the Hard Way — Part 2", Move 6; M4.4 0x01 Flash-Decoding).
#include <cuda_runtime.h>

#include "gbattn_internal.h"
#include "gbattn_ptx.cuh"

namespace gbattn {
namespace {

constexpr int kKeysPerSlot = 64;
constexpr int kConsumerWarps = 4;
constexpr int kDecThreads = (kConsumerWarps + 1) * 32;
constexpr int kSlots = 3;
constexpr int kMaxGroup = 16;  // query heads per CTA (rows of the m16 A operand)
constexpr float kRescaleThreshold = 8.0f;

template <int D>
struct DCfg {
  static constexpr int kColBlocks = D / 64;
  static constexpr int kBlockBytes = kKeysPerSlot * 128;       // 64 keys x 128 B
  static constexpr int kTileBytes = kColBlocks * kBlockBytes;  // K (or V) of one slot
  static constexpr int kSlotBytes = 2 * kTileBytes;            // K then V
  static constexpr int kRingBytes = kSlots * kSlotBytes;
  // After the key loop the ring is dead and holds the four warp states.
  static constexpr int kCombineBytes = kConsumerWarps * kMaxGroup * (D + 2) * 4;
  static_assert(kCombineBytes <= kRingBytes, "warp states must fit in the ring");
  static constexpr int kBarOff = kRingBytes;
  static constexpr int kSmemBytes = 1024 + kBarOff + 256;
};

struct DecParams {
  const uint16_t* q;
  const int* seqlens;
  float* ws_o;
  float* ws_ml;
  int B, Hq, Hkv, Sk_max, g, n_groups, n_split;
  float scale_log2;
  int* status;
};

struct __align__(8) DecBars {
  uint64_t full[kSlots];
  uint64_t empty[kSlots];
  int abort_flag;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

template <bool BF16>
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (BF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// Byte offset of 16-byte chunk `chunk` (0..7 within a 128-byte row) of key
// row `key` inside one 64-key block written by TMA with 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128(int key, int chunk) {
  return static_cast<uint32_t>(key * 128 + ((chunk ^ (key & 7)) << 4));
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kDecThreads)
    decode_partial_kernel(const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_v, const DecParams p) {
  using C = DCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  float* comb = reinterpret_cast<float*>(smem);  // aliases the ring after the loop
  DecBars* bars = reinterpret_cast<DecBars*>(smem + C::kBarOff);
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int c = blockIdx.x;
  const int kvh = blockIdx.y / p.n_groups;
  const int grp = blockIdx.y % p.n_groups;
  const int b = blockIdx.z;
  const int h_begin = kvh * p.g + grp * kMaxGroup;
  const int n_rows = min(kMaxGroup, p.g - grp * kMaxGroup);  // query heads in this CTA

  int L = p.seqlens[b];
  L = max(1, min(L, p.Sk_max));
  const int lo = static_cast<int>((static_cast<long long>(c) * L) / p.n_split);
  const int hi = static_cast<int>((static_cast<long long>(c + 1) * L) / p.n_split);
  const int n_keys = hi - lo;
  const int n_slots = (n_keys + kKeysPerSlot - 1) / kKeysPerSlot;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], kConsumerWarps);
    }
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // Per-thread online state of the consumer warps (unused by the producer).
  float o[D / 8][4];
  float m[2] = {-INFINITY, -INFINITY};  // retained reference (raw units), rows r0, r0+8
  float l[2] = {0.f, 0.f};              // this thread's share of the row sums
#pragma unroll
  for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  const int r0 = lane >> 2;  // A/C fragment rows owned: r0 and r0 + 8
  const int quad = lane & 3;

  if (warp == kConsumerWarps) {
    // ================================================================ producer
    if (lane == 0 && n_slots > 0) {
      prefetch_tensormap(&tmap_k);
      prefetch_tensormap(&tmap_v);
      const uint64_t stream_once = policy_evict_first();
      int issued = 0;
      for (int i = 0; i < n_slots; ++i) {
        const int s = i % kSlots;
        const uint32_t ph = (i / kSlots) & 1;
        if (!bounded_wait(&bars->empty[s], ph ^ 1, abort_flag, p.status, kStatusTimeoutDecode)) break;
        uint8_t* slot = smem + s * C::kSlotBytes;
        mbar_arrive_expect_tx(&bars->full[s], C::kSlotBytes);
        const int y = lo + i * kKeysPerSlot;
        const int z = b * p.Hkv + kvh;
        for (int cb = 0; cb < C::kColBlocks; ++cb) {
          tma_load_3d(slot + cb * C::kBlockBytes, &tmap_k, &bars->full[s], cb * 64, y, z, stream_once);
          tma_load_3d(slot + C::kTileBytes + cb * C::kBlockBytes, &tmap_v, &bars->full[s], cb * 64, y,
                      z, stream_once);
        }
        issued = i + 1;
      }
      for (int i = max(0, issued - kSlots); i < issued; ++i) {
        int dummy = 0;
        bounded_wait(&bars->full[i % kSlots], (i / kSlots) & 1, reinterpret_cast<volatile int*>(&dummy),
                     p.status, kStatusTimeoutDrain);
      }
    }
    __syncwarp();
  } else {
    // ================================================================ consumers
    const float lam = p.scale_log2;
    // Q A-fragments for all D/16 k-steps (rows >= n_rows are zero).
    uint32_t qa[D / 16][4];
    {
      const uint16_t* qb = p.q + (static_cast<size_t>(b) * p.Hq + h_begin) * D;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int d0 = ks * 16 + quad * 2;
        qa[ks][0] = r0 < n_rows ? *reinterpret_cast<const uint32_t*>(qb + r0 * D + d0) : 0u;
        qa[ks][1] = r0 + 8 < n_rows ? *reinterpret_cast<const uint32_t*>(qb + (r0 + 8) * D + d0) : 0u;
        qa[ks][2] = r0 < n_rows ? *reinterpret_cast<const uint32_t*>(qb + r0 * D + d0 + 8) : 0u;
        qa[ks][3] = r0 + 8 < n_rows ? *reinterpret_cast<const uint32_t*>(qb + (r0 + 8) * D + d0 + 8) : 0u;
      }
    }
    const uint32_t smem_base = smem_u32(smem);

    for (int i = 0; i < n_slots; ++i) {
      const int s = i % kSlots;
      bool ok = bounded_wait(&bars->full[s], (i / kSlots) & 1, abort_flag, p.status, kStatusTimeoutDecode);
      if (!__all_sync(0xffffffffu, ok)) break;
      const uint32_t kbase = smem_base + s * C::kSlotBytes;
      const uint32_t vbase = kbase + C::kTileBytes;
      const int kw = warp * 16;  // this warp's first key within the slot
      // ---- S = Q K^T for 16 keys (two n8 tiles)
      float sc[2][4];
#pragma unroll
      for (int t = 0; t < 2; ++t) sc[t][0] = sc[t][1] = sc[t][2] = sc[t][3] = 0.f;
      {
        const int mi = lane >> 3, rr = lane & 7;
        const int key = kw + rr + (mi >= 2 ? 8 : 0);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const int d = ks * 16 + (mi & 1) * 8;
          const uint32_t addr = kbase + (d / 64) * C::kBlockBytes + sw128(key, (d % 64) / 8);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(addr, b0, b1, b2, b3);
          mma16816<BF16>(sc[0], qa[ks], b0, b1);
          mma16816<BF16>(sc[1], qa[ks], b2, b3);
        }
      }
      // ---- mask keys outside [lo, hi)
      const int key_base = lo + i * kKeysPerSlot + kw;
      const bool partial = key_base + 16 > hi;
      if (partial) {
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (key_base + t * 8 + quad * 2 + (e & 1) >= hi) sc[t][e] = -INFINITY;
      }
      // ---- online softmax with conditional rescaling, per row
      float gamma[2];
#pragma unroll
      for (int rh = 0; rh < 2; ++rh) {
        float mx = fmaxf(fmaxf(sc[0][2 * rh], sc[0][2 * rh + 1]), fmaxf(sc[1][2 * rh], sc[1][2 * rh + 1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float cand = fmaxf(m[rh], mx);
        gamma[rh] = 1.f;
        if ((cand - m[rh]) * lam > kRescaleThreshold) {
          gamma[rh] = ex2_approx((m[rh] - cand) * lam);
          m[rh] = cand;
        }
        l[rh] *= gamma[rh];
        const float ms = (m[rh] == -INFINITY) ? 0.f : m[rh] * lam;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          sc[t][2 * rh] = ex2_approx(fmaf(sc[t][2 * rh], lam, -ms));
          sc[t][2 * rh + 1] = ex2_approx(fmaf(sc[t][2 * rh + 1], lam, -ms));
          l[rh] += sc[t][2 * rh] + sc[t][2 * rh + 1];
        }
      }
      if (gamma[0] != 1.f || gamma[1] != 1.f) {
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
          o[n][0] *= gamma[0];
          o[n][1] *= gamma[0];
          o[n][2] *= gamma[1];
          o[n][3] *= gamma[1];
        }
      }
      // ---- O += P V  (P from the score fragments, V via transposed ldmatrix)
      uint32_t pa[4];
      pa[0] = pack2<BF16>(sc[0][0], sc[0][1]);
      pa[1] = pack2<BF16>(sc[0][2], sc[0][3]);
      pa[2] = pack2<BF16>(sc[1][0], sc[1][1]);
      pa[3] = pack2<BF16>(sc[1][2], sc[1][3]);
      // V rows past the chunk end may be padding (any bit pattern, NaN
      // included): zero the operand halves of invalid keys so 0 * NaN never
      // enters the accumulator.
      uint32_t vmask0 = 0xFFFFFFFFu, vmask1 = 0xFFFFFFFFu;
      if (partial) {
        const int k_a = key_base + quad * 2;      // keys of b0/b1 halves
        const int k_b = key_base + 8 + quad * 2;  // keys of b2/b3 halves
        vmask0 = (k_a < hi ? 0x0000FFFFu : 0u) | (k_a + 1 < hi ? 0xFFFF0000u : 0u);
        vmask1 = (k_b < hi ? 0x0000FFFFu : 0u) | (k_b + 1 < hi ? 0xFFFF0000u : 0u);
      }
      {
        const int mi = lane >> 3, rr = lane & 7;
        const int key = kw + rr + (mi & 1) * 8;
#pragma unroll
        for (int np = 0; np < D / 16; ++np) {
          const int d = np * 16 + (mi >> 1) * 8;
          const uint32_t addr = vbase + (d / 64) * C::kBlockBytes + sw128(key, (d % 64) / 8);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(addr, b0, b1, b2, b3);
          mma16816<BF16>(o[2 * np], pa, b0 & vmask0, b1 & vmask1);
          mma16816<BF16>(o[2 * np + 1], pa, b2 & vmask0, b3 & vmask1);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->empty[s]);
    }
  }
  __syncthreads();  // every slot consumed and every copy landed: the ring is free

  if (warp < kConsumerWarps) {
    // ---- per-warp state -> shared memory (rows r0, r0+8; quad-reduced l)
#pragma unroll
    for (int rh = 0; rh < 2; ++rh) {
      l[rh] += __shfl_xor_sync(0xffffffffu, l[rh], 1);
      l[rh] += __shfl_xor_sync(0xffffffffu, l[rh], 2);
    }
    float* wst = comb + warp * kMaxGroup * (D + 2);
#pragma unroll
    for (int rh = 0; rh < 2; ++rh) {
      const int row = r0 + rh * 8;
      float* rowp = wst + row * (D + 2);
      if (quad == 0) {
        rowp[D] = m[rh];
        rowp[D + 1] = l[rh];
      }
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        rowp[n * 8 + quad * 2] = o[n][2 * rh];
        rowp[n * 8 + quad * 2 + 1] = o[n][2 * rh + 1];
      }
    }
  }
  __syncthreads();

  // ---- merge the four warp states (M4.3 0x08B) and write the chunk state
  if (threadIdx.x < kConsumerWarps * 32) {
    const float lam = p.scale_log2;
    const float inv_log2e = 0.69314718055994531f;  // converts lambda-frame to natural units
    for (int idx = threadIdx.x; idx < n_rows * D; idx += kConsumerWarps * 32) {
      const int row = idx / D;
      const int dd = idx % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float* rp = comb + (w * kMaxGroup + row) * (D + 2);
        if (rp[D + 1] > 0.f) M = fmaxf(M, rp[D]);
      }
      float acc = 0.f, lsum = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float* rp = comb + (w * kMaxGroup + row) * (D + 2);
          if (rp[D + 1] > 0.f) {
            const float a = ex2_approx((rp[D] - M) * lam);
            acc += a * rp[dd];
            lsum += a * rp[D + 1];
          }
        }
      }
      const size_t st = (static_cast<size_t>(b) * p.Hq + h_begin + row) * p.n_split + c;
      p.ws_o[st * D + dd] = acc;
      if (dd == 0) {
        p.ws_ml[2 * st] = (M == -INFINITY) ? -INFINITY : M * lam * inv_log2e;
        p.ws_ml[2 * st + 1] = lsum;
      }
    }
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(128)
    decode_merge_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_ml,
                        uint16_t* __restrict__ out, float* __restrict__ lse, int rows, int n_split) {
  const int warp = blockIdx.x * 4 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (warp >= rows) return;
  const float* ml = ws_ml + static_cast<size_t>(warp) * n_split * 2;
  const float* po = ws_o + static_cast<size_t>(warp) * n_split * D;
  float M = -INFINITY;
  for (int c = lane; c < n_split; c += 32)
    if (ml[2 * c + 1] > 0.f) M = fmaxf(M, ml[2 * c]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  constexpr int kPer = D / 32;
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  float lsum = 0.f;
  if (M != -INFINITY) {
    for (int c = 0; c < n_split; ++c) {
      const float lc = ml[2 * c + 1];
      if (!(lc > 0.f)) continue;  // identity (empty chunk)
      const float a = __expf(ml[2 * c] - M);
      lsum += a * lc;
      const float* oc = po + static_cast<size_t>(c) * D + lane * kPer;
#pragma unroll
      for (int e = 0; e < kPer; ++e) acc[e] += a * oc[e];
    }
  }
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  uint16_t* orow = out + static_cast<size_t>(warp) * D + lane * kPer;
#pragma unroll
  for (int e = 0; e < kPer; e += 2) {
    const uint32_t pk = pack2<BF16>(acc[e] * inv, acc[e + 1] * inv);
    *reinterpret_cast<uint32_t*>(orow + e) = pk;
  }
  if (lane == 0 && lse != nullptr) lse[warp] = lsum > 0.f ? M + __logf(lsum) : -INFINITY;
}

template <int D, bool BF16>
int launch_decode_t(const DecodeArgs& a) {
  using C = DCfg<D>;
  CUtensorMap tk, tv;
  const long long outer = static_cast<long long>(a.B) * a.Hkv;
  if (!make_tmap_3d(&tk, a.k, BF16, D, a.Sk_max, outer, kKeysPerSlot) ||
      !make_tmap_3d(&tv, a.v, BF16, D, a.Sk_max, outer, kKeysPerSlot))
    return -1;
  auto kern = decode_partial_kernel<D, BF16>;
  static std::atomic<unsigned long long> attr_done{0};  // per instantiation
  if (!set_smem_limit_once(kern, C::kSmemBytes, attr_done)) return -1;
  DecParams p;
  p.q = static_cast<const uint16_t*>(a.q);
  p.seqlens = a.seqlens;
  const size_t n_states = static_cast<size_t>(a.B) * a.Hq * a.n_split;
  p.ws_o = a.workspace;
  p.ws_ml = a.workspace + n_states * D;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.Sk_max = a.Sk_max;
  p.g = a.Hq / a.Hkv;
  p.n_groups = (p.g + kMaxGroup - 1) / kMaxGroup;
  p.n_split = a.n_split;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.status = a.status;
  if (static_cast<long long>(a.Hkv) * p.n_groups > 65535 || a.B > 65535) return -1;
  dim3 grid(a.n_split, a.Hkv * p.n_groups, a.B);
  kern<<<grid, kDecThreads, C::kSmemBytes, a.stream>>>(tk, tv, p);
  if (cudaGetLastError() != cudaSuccess) return -1;
  const int rows = a.B * a.Hq;
  decode_merge_kernel<D, BF16><<<(rows + 3) / 4, 128, 0, a.stream>>>(
      p.ws_o, p.ws_ml, static_cast<uint16_t*>(a.o), a.lse, rows, a.n_split);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

int launch_decode(const DecodeArgs& a) {
  if (a.d == 128) return a.bf16 ? launch_decode_t<128, true>(a) : launch_decode_t<128, false>(a);
  return a.bf16 ? launch_decode_t<64, true>(a) : launch_decode_t<64, false>(a);
}

}  // namespace gbattn
