// backward.cu -- exact attention backward on sm_103a.
//
// Gradients (M4.4 "FlashAttention-2 Work Partitioning and the Decode
// Boundary", 0x06.1A), with tau the score scale and the forward's saved O and
// natural-log LSE:
//     P_ij  = exp(tau q_i.k_j - LSE_i)          (0 where masked)
//     dP_ij = dO_i . v_j,    D_i = dO_i . O_i
//     dS_ij = P_ij (dP_ij - D_i)
//     dQ = tau dS K,   dK = tau dS^T Q,   dV = P^T dO
//
// Three kernels in stream order (the producer graph of 0x06.1D):
//   1. bwd_preprocess_kernel: D = rowsum(dO * O) in fp32 and a zeroed fp32
//      dQ accumulator;
//   2. bwd_main_kernel: one CTA owns a 128-key tile of one (batch, KV head)
//      -- the column owner of 0x06.1B -- and loops over every visible 64-row
//      query block of EVERY query head that reads this KV head.  dK and dV of
//      the tile accumulate in tensor memory across the whole loop, so the
//      grouped-query sum of 0x06.1H happens in the accumulator and no
//      expanded per-query-head dK/dV buffers or group-sum pass exist.  Each
//      block's dQ contribution is added to the fp32 accumulator in global
//      memory with one bulk asynchronous reduce-add (atomic per element, no
//      fixed order: 0x06.1F);
//   3. bwd_dq_convert_kernel: dQ accumulator (already scaled by tau) -> dtype.
//
// Main kernel, per query block t (64 rows of query head h), all five
// contractions on tcgen05 with fp32 accumulation in tensor memory; the key
// axis is the TMEM lane axis, so each thread of the "P" warpgroup owns one
// key row of the transposed score tile:
//     S^T  = K Q_t^T          M=128 keys, N=64 rows, K=d     (SS, K-major)
//     dP^T = V dO_t^T         M=128 keys, N=64 rows, K=d     (SS, K-major)
//     dV  += P^T dO_t         M=128 keys, N=d, K=64 rows     (A K-major, B MN-major)
//     dK  += dS^T Q_t         M=128 keys, N=d, K=64 rows     (A K-major, B MN-major)
//     dQ_t^T = K^T dS^T       M=d, N=64 rows, K=128 keys     (A and B MN-major)
// P^T and dS^T are rounded to the input dtype and staged in shared memory
// (K-major for dV/dK, read MN-major by the dQ^T product -- one buffer serves
// both).  Tensor memory (512 columns): dV [0,128), dK [128,256),
// S^T two buffers [256,320) [320,384), dP^T [384,448), dQ^T [448,512).
//
// Roles (320 threads):
//   warps 0-3  "P" warpgroup: thread = key row; P^T, dS^T; then dV epilogue
//   warps 4-7  "Q" warpgroup: thread = column d of dQ^T; dQ drain through a
//              shared staging tile + bulk reduce-add; then dK epilogue
//   warp  8    loader: K, V once (TMA), Q_t/dO_t per block (TMA, 3 stages),
//              per-row LSE (in base 2) and D (plain loads by all 32 lanes)
//   warp  9    TMEM allocation; lane 0 issues every MMA and commit
//
// Causal (bottom-right delta = Sk - Sq): query rows that cannot see the tile's
// first key are never visited; blocks crossing the diagonal and the key /
// query tails are masked element-wise before the exponential.
#include <cuda_runtime.h>

#include "gbattn_internal.h"
#include "gbattn_ptx.cuh"

namespace gbattn {
namespace {

constexpr int kD = 128;       // head dimension of this kernel
constexpr int kBN = 128;      // keys per CTA (TMEM lanes)
constexpr int kBM = 64;       // query rows per block
constexpr int kStages = 3;    // Q/dO stages
constexpr int kThreads = 320;
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr float kLog2e = 1.4426950408889634f;

// Shared memory (offsets from a 1024-byte aligned base).
constexpr int kKBytes = kBN * kD * 2;        // 32 KiB: two 128-row x 128-byte column blocks
constexpr int kKBlock = kBN * 128;           // 16 KiB
constexpr int kQBytes = kBM * kD * 2;        // 16 KiB: two 64-row x 128-byte column blocks
constexpr int kQBlock = kBM * 128;           // 8 KiB
constexpr int kPBytes = kBN * kBM * 2;       // 16 KiB: 128 key rows x 128 bytes
constexpr int kStageBytes = kBM * kD * 4;    // 32 KiB fp32 dQ staging tile
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kKBytes;
constexpr int kOffQ = kOffV + kKBytes;                 // kStages tiles
constexpr int kOffDO = kOffQ + kStages * kQBytes;      // kStages tiles
constexpr int kOffP = kOffDO + kStages * kQBytes;
constexpr int kOffDS = kOffP + kPBytes;
constexpr int kOffStage = kOffDS + kPBytes;
constexpr int kOffStats = kOffStage + kStageBytes;     // kStages x (64 lse2 + 64 D) floats
constexpr int kOffBars = kOffStats + kStages * 2 * kBM * 4;
constexpr int kSmemBytes = 1024 + kOffBars + 256;
static_assert(kSmemBytes <= 232448, "shared memory budget");

// TMEM columns
constexpr uint32_t kColDV = 0, kColDK = 128, kColS0 = 256, kColDP = 384, kColDQ = 448;

struct BwdParams {
  const float* lse;   // [B,H,Sq] natural log
  const float* Dvec;  // [B,H,Sq]
  float* dq_acc;      // [B,H,Sq,D] fp32
  void* dk;           // [B,Hkv,Sk,D]
  void* dv;
  int B, H, Hkv, Sq, Sk, g;
  int n_ktiles, head_group, delta;
  float scale, scale_log2;
  int* status;
};

struct __align__(8) BwdBars {
  uint64_t kv_full;
  uint64_t qd_full[kStages];
  uint64_t qd_empty[kStages];
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t dp_full, dp_free;
  uint64_t p_full, p_free;
  uint64_t ds_full, ds_free;
  uint64_t dq_full, dq_free;
  uint64_t acc_done;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         int* status) {
  return bounded_wait(bar, parity, abort_flag, status, kStatusTimeoutBwd);
}

template <bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v,
                    const __grid_constant__ CUtensorMap tmap_do, const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem + kOffBars);
  float* stats = reinterpret_cast<float*>(smem + kOffStats);  // [stage][lse2 64 | D 64]
  volatile int* abort_flag = &bars->abort_flag;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  // ---- work unit: (batch * Hkv + kv head, key tile).  CTAs run in groups of
  // p.head_group KV heads (their Q/dO/dQ working set stays in L2); inside a
  // group, key tiles ascend (causal: the tiles with the most query blocks
  // first) and heads vary fastest.
  const int BHkv = p.B * p.Hkv;
  const int group = blockIdx.x / (p.head_group * p.n_ktiles);
  const int heads_here = min(p.head_group, BHkv - group * p.head_group);
  const int r_in = blockIdx.x - group * p.head_group * p.n_ktiles;
  const int bkv = group * p.head_group + r_in % heads_here;
  const int jt = r_in / heads_here;
  const int b = bkv / p.Hkv;
  const int kvh = bkv % p.Hkv;
  const int k0 = jt * kBN;
  const int nqb = (p.Sq + kBM - 1) / kBM;
  int i_start = 0;
  if (CAUSAL) {
    const int q_min = k0 - p.delta;  // first query row that sees key k0
    i_start = q_min <= 0 ? 0 : (q_min >= p.Sq ? nqb : q_min / kBM);
  }
  const int n_blk = nqb - i_start;
  const int T = p.g * n_blk;  // query blocks this CTA visits

  // ---- setup
  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->qd_full[s], 1 + 32);  // TMA arrive + 32 lanes' stat stores
      mbar_init(&bars->qd_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars->s_full[x], 1);
      mbar_init(&bars->s_free[x], 128);
    }
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->dp_free, 128);
    mbar_init(&bars->p_full, 128);
    mbar_init(&bars->p_free, 1);
    mbar_init(&bars->ds_full, 128);
    mbar_init(&bars->ds_free, 1);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_free, 128);
    mbar_init(&bars->acc_done, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kLoadWarp && lane == 0) {
    prefetch_tensormap(&tmap_q);
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
    prefetch_tensormap(&tmap_do);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  auto block_coords = [&](int t, int& h, int& q0) {
    const int hh = t / n_blk;
    h = kvh * p.g + hh;
    q0 = (i_start + (t - hh * n_blk)) * kBM;
  };

  if (warp == kLoadWarp) {
    // ================================================================ loader
    int issued = 0;
    if (T > 0) {
      if (lane == 0) {
        const uint64_t keep = policy_evict_first();  // K/V: read by this CTA only
        mbar_arrive_expect_tx(&bars->kv_full, 2 * kKBytes);
        for (int cb = 0; cb < 2; ++cb) {
          tma_load_3d(smem + kOffK + cb * kKBlock, &tmap_k, &bars->kv_full, cb * 64, k0, bkv, keep);
          tma_load_3d(smem + kOffV + cb * kKBlock, &tmap_v, &bars->kv_full, cb * 64, k0, bkv, keep);
        }
      }
      const uint64_t reuse = policy_evict_last();  // Q/dO: re-read by every key tile
      for (int t = 0; t < T; ++t) {
        const int s = t % kStages;
        const uint32_t ph = (t / kStages) & 1;
        bool ok = wait_bar(&bars->qd_empty[s], ph ^ 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) break;
        int h, q0;
        block_coords(t, h, q0);
        const long long row0 = (static_cast<long long>(b) * p.H + h) * p.Sq;
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars->qd_full[s], 2 * kQBytes);
          for (int cb = 0; cb < 2; ++cb) {
            tma_load_3d(smem + kOffQ + s * kQBytes + cb * kQBlock, &tmap_q, &bars->qd_full[s], cb * 64,
                        q0, b * p.H + h, reuse);
            tma_load_3d(smem + kOffDO + s * kQBytes + cb * kQBlock, &tmap_do, &bars->qd_full[s],
                        cb * 64, q0, b * p.H + h, reuse);
          }
        }
        // per-row statistics: LSE in base 2 (+inf for rows past Sq or rows
        // with no visible key, so that their P is exactly 0) and D
        float* st = stats + s * 2 * kBM;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int c = lane + 32 * u;
          const int row = q0 + c;
          float l2 = INFINITY, dv = 0.f;
          if (row < p.Sq) {
            const float lse = p.lse[row0 + row];
            if (lse != -INFINITY) l2 = lse * kLog2e;
            dv = p.Dvec[row0 + row];
          }
          st[c] = l2;
          st[kBM + c] = dv;
        }
        mbar_arrive(&bars->qd_full[s]);
        issued = t + 1;
      }
    }
    if (lane == 0 && T > 0) {
      // Drain: every copy this thread issued must land before exit.
      int dummy = 0;
      volatile int* no_abort = reinterpret_cast<volatile int*>(&dummy);
      bounded_wait(&bars->kv_full, 0, no_abort, p.status, kStatusTimeoutDrain);
      for (int t = max(0, issued - kStages); t < issued; ++t)
        bounded_wait(&bars->qd_full[t % kStages], (t / kStages) & 1, no_abort, p.status,
                     kStatusTimeoutDrain);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ================================================================ MMA issuer
    if (lane == 0 && T > 0) {
      constexpr uint32_t kIdS = idesc_f16(BF16, false, false, kBN, kBM);   // S^T, dP^T
      constexpr uint32_t kIdAcc = idesc_f16(BF16, false, true, kBN, kD);   // dV, dK
      constexpr uint32_t kIdDQ = idesc_f16(BF16, true, true, kD, kBM);     // dQ^T
      const uint32_t aK = smem_u32(smem + kOffK), aV = smem_u32(smem + kOffV);
      const uint32_t aP = smem_u32(smem + kOffP), aDS = smem_u32(smem + kOffDS);
      // K-major descriptors (K, V as A; Q, dO as B of the score products; P,
      // dS as A of the accumulations): a K-step of 16 elements adds 32 bytes
      // inside a 128-byte row, or jumps a column block.
      const uint64_t dK_A = smem_desc_sw128(aK, 16, 1024);
      const uint64_t dV_A = smem_desc_sw128(aV, 16, 1024);
      const uint64_t dP_A = smem_desc_sw128(aP, 16, 1024);
      const uint64_t dDS_A = smem_desc_sw128(aDS, 16, 1024);
      // MN-major descriptors: leading offset = stride between 64-element
      // column blocks, stride offset = 8 rows of 128 bytes; a K-step of 16
      // rows adds 2048 bytes.
      const uint64_t dKT_A = smem_desc_sw128(aK, kKBlock, 1024);  // K^T for dQ^T
      const uint64_t dDS_B = smem_desc_sw128(aDS, kKBlock, 1024); // dS^T as B of dQ^T

      auto issue_scores = [&](uint32_t d_col, uint64_t a_desc, uint32_t b_base) {
        const uint64_t bd = smem_desc_sw128(b_base, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint64_t ao = ((kk / 4) * kKBlock + (kk % 4) * 32) >> 4;
          const uint64_t bo = ((kk / 4) * kQBlock + (kk % 4) * 32) >> 4;
          mma_f16_ss(tmem + d_col, a_desc + ao, bd + bo, kIdS, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_acc = [&](uint32_t d_col, uint64_t a_desc, uint32_t b_base, bool accumulate) {
        const uint64_t bd = smem_desc_sw128(b_base, kQBlock, 1024);
#pragma unroll
        for (int kk = 0; kk < kBM / 16; ++kk)
          mma_f16_ss(tmem + d_col, a_desc + ((kk * 32) >> 4), bd + ((kk * 2048) >> 4), kIdAcc,
                     (accumulate || kk > 0) ? 1u : 0u);
      };
      auto issue_dq = [&]() {
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_f16_ss(tmem + kColDQ, dKT_A + ((kk * 2048) >> 4), dDS_B + ((kk * 2048) >> 4), kIdDQ,
                     kk > 0 ? 1u : 0u);
      };
      const uint32_t aQ0 = smem_u32(smem + kOffQ), aDO0 = smem_u32(smem + kOffDO);

      bool ok = wait_bar(&bars->kv_full, 0, abort_flag, p.status) &&
                wait_bar(&bars->qd_full[0], 0, abort_flag, p.status);
      if (ok) {
        tc_fence_after();
        issue_scores(kColS0, dK_A, aQ0);
        mma_commit(&bars->s_full[0]);
        issue_scores(kColDP, dV_A, aDO0);
        mma_commit(&bars->dp_full);
      }
      for (int t = 0; ok && t < T; ++t) {
        const int s = t % kStages;
        if (t + 1 < T) {
          const int s1 = (t + 1) % kStages;
          const int sb = (t + 1) & 1;  // S buffer
          if (!(ok = wait_bar(&bars->qd_full[s1], ((t + 1) / kStages) & 1, abort_flag, p.status))) break;
          if (t + 1 >= 2 &&
              !(ok = wait_bar(&bars->s_free[sb], (((t + 1) >> 1) - 1) & 1, abort_flag, p.status)))
            break;
          tc_fence_after();
          issue_scores(kColS0 + sb * kBM, dK_A, aQ0 + s1 * kQBytes);
          mma_commit(&bars->s_full[sb]);
        }
        // dV += P^T dO_t
        if (!(ok = wait_bar(&bars->p_full, t & 1, abort_flag, p.status))) break;
        tc_fence_after();
        issue_acc(kColDV, dP_A, aDO0 + s * kQBytes, t > 0);
        mma_commit(&bars->p_free);
        // dP^T of the next block as soon as dP^T(t) is in registers, so the
        // P warpgroup can form dS(t+1) while dK(t) and dQ(t) run
        if (t + 1 < T) {
          if (!(ok = wait_bar(&bars->dp_free, t & 1, abort_flag, p.status))) break;
          tc_fence_after();
          issue_scores(kColDP, dV_A, aDO0 + ((t + 1) % kStages) * kQBytes);
          mma_commit(&bars->dp_full);
        }
        // dK += dS^T Q_t ; dQ_t^T = K^T dS^T
        if (!(ok = wait_bar(&bars->ds_full, t & 1, abort_flag, p.status))) break;
        tc_fence_after();
        issue_acc(kColDK, dDS_A, aQ0 + s * kQBytes, t > 0);
        mma_commit(&bars->qd_empty[s]);  // last reader of Q_t and dO_t
        if (t >= 1 && !(ok = wait_bar(&bars->dq_free, (t - 1) & 1, abort_flag, p.status))) break;
        tc_fence_after();
        issue_dq();
        mma_commit(&bars->dq_full);
        mma_commit(&bars->ds_free);
      }
      mma_commit(&bars->acc_done);
      // Every MMA issued must complete before TMEM is released.
      int dummy = 0;
      bounded_wait(&bars->acc_done, 0, reinterpret_cast<volatile int*>(&dummy), p.status,
                   kStatusTimeoutDrain);
    }
    __syncwarp();
  } else if (warp < 4) {
    // ================================================================ P warpgroup
    const int kl = warp * 32 + lane;  // key row within the tile (= TMEM lane)
    const int key = k0 + kl;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    uint8_t* p_row = smem + kOffP + kl * 128;
    uint8_t* ds_row = smem + kOffDS + kl * 128;
    const float lam = p.scale_log2;
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      const int s = t % kStages;
      const int sb = t & 1;
      int h, q0;
      block_coords(t, h, q0);
      (void)h;
      // S^T(t) in TMEM; the block's row statistics (plain stores by the
      // loader, published through qd_full) in shared memory
      ok = wait_bar(&bars->s_full[sb], (t >> 1) & 1, abort_flag, p.status) &&
           wait_bar(&bars->qd_full[s], (t / kStages) & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t u[kBM];
      tmem_ld32(tmem + lane_off + kColS0 + sb * kBM, *reinterpret_cast<uint32_t(*)[32]>(&u[0]));
      tmem_ld32(tmem + lane_off + kColS0 + sb * kBM + 32, *reinterpret_cast<uint32_t(*)[32]>(&u[32]));
      tmem_wait_ld();
      reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&u[0]));
      reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&u[32]));
      tc_fence_before();
      mbar_arrive(&bars->s_free[sb]);
      const float* st = stats + s * 2 * kBM;
      // P = 2^(lambda s - LSE log2 e); rows past Sq carry LSE = +inf (P = 0).
      // Masked: keys past Sk, and (causal) column c with q0 + c + delta < key.
      const bool need_mask = (k0 + kBN > p.Sk) || (CAUSAL && (k0 + kBN - 1 > q0 + p.delta));
      const int first_c = (key >= p.Sk) ? kBM : (CAUSAL ? key - p.delta - q0 : 0);
      float pr[kBM];
      const float4* sl4 = reinterpret_cast<const float4*>(st);
#pragma unroll
      for (int c4 = 0; c4 < kBM / 4; ++c4) {
        const float4 l4 = sl4[c4];  // base-2 LSE of rows 4c4 .. 4c4+3 (broadcast read)
        const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = 4 * c4 + i;
          float x = ex2_approx(fmaf(__uint_as_float(u[c]), lam, -lv[i]));
          if (need_mask && c < first_c) x = 0.f;
          pr[c] = x;
        }
      }
      if (t >= 1) {
        ok = wait_bar(&bars->p_free, (t - 1) & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
      }
#pragma unroll
      for (int ch = 0; ch < kBM / 8; ++ch) {
        const uint32_t w0 = pack2<BF16>(pr[ch * 8 + 0], pr[ch * 8 + 1]);
        const uint32_t w1 = pack2<BF16>(pr[ch * 8 + 2], pr[ch * 8 + 3]);
        const uint32_t w2 = pack2<BF16>(pr[ch * 8 + 4], pr[ch * 8 + 5]);
        const uint32_t w3 = pack2<BF16>(pr[ch * 8 + 6], pr[ch * 8 + 7]);
        *reinterpret_cast<uint4*>(p_row + ((ch ^ (kl & 7)) << 4)) = make_uint4(w0, w1, w2, w3);
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars->p_full);
      // dP^T row -> dS^T row
      ok = wait_bar(&bars->dp_full, t & 1, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      tmem_ld32(tmem + lane_off + kColDP, *reinterpret_cast<uint32_t(*)[32]>(&u[0]));
      tmem_ld32(tmem + lane_off + kColDP + 32, *reinterpret_cast<uint32_t(*)[32]>(&u[32]));
      tmem_wait_ld();
      reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&u[0]));
      reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&u[32]));
      tc_fence_before();
      mbar_arrive(&bars->dp_free);
      const float4* st4 = reinterpret_cast<const float4*>(st + kBM);
#pragma unroll
      for (int c4 = 0; c4 < kBM / 4; ++c4) {
        const float4 dd = st4[c4];  // D of rows 4c4 .. 4c4+3 (broadcast read)
        pr[4 * c4 + 0] *= __uint_as_float(u[4 * c4 + 0]) - dd.x;
        pr[4 * c4 + 1] *= __uint_as_float(u[4 * c4 + 1]) - dd.y;
        pr[4 * c4 + 2] *= __uint_as_float(u[4 * c4 + 2]) - dd.z;
        pr[4 * c4 + 3] *= __uint_as_float(u[4 * c4 + 3]) - dd.w;
      }
      if (t >= 1) {
        ok = wait_bar(&bars->ds_free, (t - 1) & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
      }
#pragma unroll
      for (int ch = 0; ch < kBM / 8; ++ch) {
        const uint32_t w0 = pack2<BF16>(pr[ch * 8 + 0], pr[ch * 8 + 1]);
        const uint32_t w1 = pack2<BF16>(pr[ch * 8 + 2], pr[ch * 8 + 3]);
        const uint32_t w2 = pack2<BF16>(pr[ch * 8 + 4], pr[ch * 8 + 5]);
        const uint32_t w3 = pack2<BF16>(pr[ch * 8 + 6], pr[ch * 8 + 7]);
        *reinterpret_cast<uint4*>(ds_row + ((ch ^ (kl & 7)) << 4)) = make_uint4(w0, w1, w2, w3);
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars->ds_full);
    }
    // ---- dV epilogue: this thread's key row, 128 columns
    bool have = ok && T > 0;
    if (have) {
      have = wait_bar(&bars->acc_done, 0, abort_flag, p.status);
      have = __all_sync(0xffffffffu, have);
      tc_fence_after();
    }
    uint16_t* dst = reinterpret_cast<uint16_t*>(p.dv) + (static_cast<long long>(bkv) * p.Sk + key) * kD;
#pragma unroll 1
    for (int c = 0; c < kD / 32; ++c) {
      uint32_t w[32];
      if (have) {
        tmem_ld32(tmem + lane_off + kColDV + c * 32, w);
        tmem_wait_ld();
        reg_fence32(w);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = 0u;
      }
      if (key < p.Sk) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack2<BF16>(__uint_as_float(w[2 * i]), __uint_as_float(w[2 * i + 1]));
        uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
      }
    }
  } else {
    // ================================================================ Q warpgroup
    const int wq = warp - 4;
    const int dl = wq * 32 + lane;  // column of dQ (= TMEM lane of dQ^T)
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    float* stage = reinterpret_cast<float*>(smem + kOffStage);
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      int h, q0;
      block_coords(t, h, q0);
      ok = wait_bar(&bars->dq_full, t & 1, abort_flag, p.status);
      ok = named_bar_and(1, 128, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t u[kBM];
      tmem_ld32(tmem + lane_off + kColDQ, *reinterpret_cast<uint32_t(*)[32]>(&u[0]));
      tmem_ld32(tmem + lane_off + kColDQ + 32, *reinterpret_cast<uint32_t(*)[32]>(&u[32]));
      tmem_wait_ld();
      reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&u[0]));
      reg_fence32(*reinterpret_cast<uint32_t(*)[32]>(&u[32]));
      tc_fence_before();
      mbar_arrive(&bars->dq_free);
      // the previous reduce must have finished reading the staging tile
      if (dl == 0) bulk_wait_group_read0();
      named_bar_sync(1, 128);
#pragma unroll
      for (int c = 0; c < kBM; ++c) stage[c * kD + dl] = __uint_as_float(u[c]) * p.scale;
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (dl == 0) {
        const int rows = min(kBM, p.Sq - q0);
        float* dst = p.dq_acc + ((static_cast<long long>(b) * p.H + h) * p.Sq + q0) * kD;
        bulk_reduce_add_f32(dst, stage, static_cast<uint32_t>(rows) * kD * 4u);
        bulk_commit_group();
      }
    }
    if (dl == 0) bulk_wait_group0();
    // ---- dK epilogue: key row = TMEM lane, scaled by tau
    const int kl = dl;
    const int key = k0 + kl;
    bool have = ok && T > 0;
    if (have) {
      have = wait_bar(&bars->acc_done, 0, abort_flag, p.status);
      have = __all_sync(0xffffffffu, have);
      tc_fence_after();
    }
    uint16_t* dst = reinterpret_cast<uint16_t*>(p.dk) + (static_cast<long long>(bkv) * p.Sk + key) * kD;
#pragma unroll 1
    for (int c = 0; c < kD / 32; ++c) {
      uint32_t w[32];
      if (have) {
        tmem_ld32(tmem + lane_off + kColDK + c * 32, w);
        tmem_wait_ld();
        reg_fence32(w);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = 0u;
      }
      if (key < p.Sk) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack2<BF16>(__uint_as_float(w[2 * i]) * p.scale, __uint_as_float(w[2 * i + 1]) * p.scale);
        uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
      }
    }
  }

  // ---- teardown: all TMEM traffic done before the allocator warp frees it
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

// D[row] = sum_t dO[row,t] * O[row,t] (fp32) and dq_acc[row, :] = 0.
// 16 threads per row, 8 elements (16 bytes) each.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const uint16_t* __restrict__ o,
                                                             const uint16_t* __restrict__ dout,
                                                             float* __restrict__ Dvec,
                                                             float* __restrict__ dq_acc, long long n_rows) {
  constexpr int kTpr = D / 8;  // threads per row
  const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long row = tid / kTpr;
  const int part = static_cast<int>(tid % kTpr);
  float acc = 0.f;
  if (row < n_rows) {
    const uint4 a = *reinterpret_cast<const uint4*>(o + row * D + part * 8);
    const uint4 c = *reinterpret_cast<const uint4*>(dout + row * D + part * 8);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float a0, a1, c0, c1;
      if constexpr (BF16) {
        a0 = __uint_as_float(aw[i] << 16), a1 = __uint_as_float(aw[i] & 0xffff0000u);
        c0 = __uint_as_float(cw[i] << 16), c1 = __uint_as_float(cw[i] & 0xffff0000u);
      } else {
        const __half2 ha = *reinterpret_cast<const __half2*>(&aw[i]);
        const __half2 hc = *reinterpret_cast<const __half2*>(&cw[i]);
        a0 = __low2float(ha), a1 = __high2float(ha), c0 = __low2float(hc), c1 = __high2float(hc);
      }
      acc = fmaf(a0, c0, acc);
      acc = fmaf(a1, c1, acc);
    }
    float4* z = reinterpret_cast<float4*>(dq_acc + row * D + part * 8);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int off = kTpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < n_rows && part == 0) Dvec[row] = acc;
}

// dq[i] = dtype(dq_acc[i]), 8 elements per thread.
template <bool BF16>
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const float* __restrict__ dq_acc,
                                                             uint16_t* __restrict__ dq, long long n8) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const float4 a = reinterpret_cast<const float4*>(dq_acc)[2 * i];
  const float4 c = reinterpret_cast<const float4*>(dq_acc)[2 * i + 1];
  reinterpret_cast<uint4*>(dq)[i] =
      make_uint4(pack2<BF16>(a.x, a.y), pack2<BF16>(a.z, a.w), pack2<BF16>(c.x, c.y), pack2<BF16>(c.z, c.w));
}

template <bool BF16, bool CAUSAL>
int launch_bwd_t(const BackwardArgs& a) {
  CUtensorMap tq, tk, tv, tdo;
  if (!make_tmap_3d(&tq, a.q, BF16, kD, a.Sq, static_cast<long long>(a.B) * a.H, kBM) ||
      !make_tmap_3d(&tdo, a.dout, BF16, kD, a.Sq, static_cast<long long>(a.B) * a.H, kBM) ||
      !make_tmap_3d(&tk, a.k, BF16, kD, a.Sk, static_cast<long long>(a.B) * a.Hkv, kBN) ||
      !make_tmap_3d(&tv, a.v, BF16, kD, a.Sk, static_cast<long long>(a.B) * a.Hkv, kBN))
    return -1;
  const long long n_rows = static_cast<long long>(a.B) * a.H * a.Sq;
  {
    const long long threads = n_rows * (kD / 8);
    const long long blocks = (threads + 255) / 256;
    if (blocks > 0x7FFFFFFFLL) return -1;
    bwd_preprocess_kernel<kD, BF16><<<static_cast<unsigned>(blocks), 256, 0, a.stream>>>(
        static_cast<const uint16_t*>(a.o), static_cast<const uint16_t*>(a.dout), a.Dvec, a.dq_acc, n_rows);
  }
  auto kern = bwd_main_kernel<BF16, CAUSAL>;
  static bool attr_set = false;  // per instantiation
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
      return -1;
    attr_set = true;
  }
  BwdParams p;
  p.lse = a.lse;
  p.Dvec = a.Dvec;
  p.dq_acc = a.dq_acc;
  p.dk = a.dk;
  p.dv = a.dv;
  p.B = a.B;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.Sq = a.Sq;
  p.Sk = a.Sk;
  p.g = a.H / a.Hkv;
  p.n_ktiles = (a.Sk + kBN - 1) / kBN;
  {
    // KV heads per scheduling group: about 48 MB of Q, dO (16-bit) and the
    // fp32 dQ accumulator of their query heads in flight (L2 is 129 MB).
    const long long per_kv = static_cast<long long>(p.g) * a.Sq * kD * (2 + 2 + 4);
    long long hg = (48LL << 20) / (per_kv > 0 ? per_kv : 1);
    if (hg < 1) hg = 1;
    const long long BHkv = static_cast<long long>(a.B) * a.Hkv;
    p.head_group = static_cast<int>(hg < BHkv ? hg : BHkv);
  }
  p.delta = a.Sk - a.Sq;
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  p.status = a.status;
  const long long grid = static_cast<long long>(a.B) * a.Hkv * p.n_ktiles;
  if (grid > 0x7FFFFFFFLL) return -1;
  kern<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, a.stream>>>(tq, tk, tv, tdo, p);
  {
    const long long n8 = n_rows * kD / 8;
    const long long blocks = (n8 + 255) / 256;
    bwd_dq_convert_kernel<BF16><<<static_cast<unsigned>(blocks), 256, 0, a.stream>>>(
        a.dq_acc, static_cast<uint16_t*>(a.dq), n8);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

int launch_backward(const BackwardArgs& a) {
  if (a.d != kD) return -1;
  if (a.bf16) return a.causal ? launch_bwd_t<true, true>(a) : launch_bwd_t<true, false>(a);
  return a.causal ? launch_bwd_t<false, true>(a) : launch_bwd_t<false, false>(a);
}

}  // namespace gbattn
